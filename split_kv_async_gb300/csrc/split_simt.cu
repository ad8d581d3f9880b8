// split_simt.cu -- per-split kernel on CUDA cores (fp32 or bf16 K/V, head_dim 64/128, G <= 16).
//
// One CTA (4 warps) handles one unit (sequence b, kv head g, split j) at a time and loops over
// the units of a persistent grid. A warp reads the K and V rows of head g coalesced and forms the
// dot products with shuffle butterflies, accumulating in fp32 registers:
//   up to 8 query rows per kv head: 16 bytes per lane, so a token row takes D * sizeof(T) / 16
//              lanes and one load instruction serves 32 / that many tokens, two loads in flight
//              per lane group; each group (token slot) keeps its own frame, merged at the end;
//   up to 16 rows: a token at a time per warp, 32 lanes x D / 32 elements;
//   fast pass  (opt.ai.kr "FlashDecoding++ async softmax -- theory", s3, unified max):
//              p = exp(s - phi), l += p, o += p v; no running max, nothing shared between splits;
//   detection  every valid score is tested against lo <= s - phi <= hi (same page, s3: a score
//              past the phi criterion sends the block back to online softmax);
//   recompute  when a head of the unit was flagged, the whole split is read again with the
//              ordinary online softmax (running max m, rescale by exp(m_old - m)) and the
//              partials of the flagged heads are replaced.
// The 4 warps' partials are merged through shared memory (a plain sum in the phi frame).
#include <cuda_bf16.h>

#include <type_traits>

#include "device_common.cuh"

namespace fdpp {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    // E consecutive fp32 values (E = 2 or 4) -> registers.
    template <int E>
    __device__ static __forceinline__ void load(const float* p, float (&x)[E])
    {
        if constexpr (E == 4) {
            float4 v = __ldg(reinterpret_cast<const float4*>(p));
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else {
            float2 v = __ldg(reinterpret_cast<const float2*>(p));
            x[0] = v.x; x[1] = v.y;
        }
    }
};

template <>
struct Elem<__nv_bfloat16> {
    template <int E>
    __device__ static __forceinline__ void load(const __nv_bfloat16* p, float (&x)[E])
    {
        if constexpr (E == 4) {
            uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
            float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.x));
            float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.y));
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else {
            unsigned v = __ldg(reinterpret_cast<const unsigned*>(p));
            float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
            x[0] = a.x; x[1] = a.y;
        }
    }
};

// 16 bytes of T as fp32 registers (8 bf16 or 4 fp32 elements).
template <typename T>
struct Vec16;

template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ static __forceinline__ void load(const float* p, float (&x)[4])
    {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
};

template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static __forceinline__ void load(const __nv_bfloat16* p, float (&x)[8])
    {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            x[2 * i] = f.x; x[2 * i + 1] = f.y;
        }
    }
};

template <int E, int GM>
struct SimtShared {
    long long red[32];
    float o[kWarps][GM][128];
    float l[kWarps][GM];
    float m[kWarps][GM];
    unsigned f[kWarps][GM];
    unsigned unit_flags[GM];
    int flagged_any;
};

// Element offset of the K/V row (b, t, g), or -1 when the block table entry is outside the pool.
__device__ __forceinline__ long long kv_row(const KernelArgs& a, int b, int t, int g)
{
    const long long hd = (long long)a.Hkv * a.D;
    if (!a.block_table) return ((long long)b * a.max_seq_len + t) * hd + (long long)g * a.D;
    int blk = a.block_table[(long long)b * a.max_blocks + t / a.block_size];
    if (blk < 0 || blk >= a.num_blocks) return -1;
    return ((long long)blk * a.block_size + (t % a.block_size)) * hd + (long long)g * a.D;
}

// One pass of one warp over its tokens of split [t0, t1). ONLINE selects the running-max
// softmax; otherwise the phi frame. Results stay in the warp's registers.
template <typename T, int E, int GM, bool ONLINE>
__device__ __forceinline__ void warp_pass(const KernelArgs& a, int b, int g, int t0, int t1,
                                          const float (&qr)[GM][E], const float (&ph)[GM],
                                          const int (&lim)[GM], float (&o)[GM][E], float (&l)[GM],
                                          float (&m)[GM], unsigned (&fl)[GM], bool& bad_block)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T* K = static_cast<const T*>(a.k);
    const T* V = static_cast<const T*>(a.v);
#pragma unroll
    for (int h = 0; h < GM; ++h) {
        l[h] = 0.f;
        m[h] = ONLINE ? -INFINITY : ph[h];
        fl[h] = 0u;
#pragma unroll
        for (int e = 0; e < E; ++e) o[h][e] = 0.f;
    }
    for (int t = t0 + warp; t < t1; t += kWarps) {
        const long long row = kv_row(a, b, t, g);
        if (row < 0) { bad_block = true; continue; }
        float kx[E], vx[E];
        Elem<T>::template load<E>(K + row + lane * E, kx);
        Elem<T>::template load<E>(V + row + lane * E, vx);
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            if (h >= a.R) break;
            if (t >= lim[h]) continue;             // past this query row's keys (warp-uniform)
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) part = fmaf(qr[h][e], kx[e], part);
            part = warp_sum(part);
            const float s = __fmul_rn(part, a.scale);
            const float x = __fsub_rn(s, ph[h]);
            fl[h] |= classify(x, a.lo, a.hi);
            if (ONLINE) {
                const float mn = fmaxf(m[h], s);
                const float corr = (m[h] == -INFINITY) ? 0.f : __expf(m[h] - mn);
                const float p = __expf(s - mn);
                l[h] = fmaf(l[h], corr, p);
#pragma unroll
                for (int e = 0; e < E; ++e) o[h][e] = fmaf(o[h][e], corr, p * vx[e]);
                m[h] = mn;
            } else {
                const float p = __expf(x);
                l[h] += p;
#pragma unroll
                for (int e = 0; e < E; ++e) o[h][e] = fmaf(p, vx[e], o[h][e]);
            }
        }
    }
}

// The same pass with 16-byte lanes (at most GM = 4 rows per kv head): LPT = D / N lanes per token
// row (N elements of T in 16 bytes), TPI = 32 / LPT token slots per load, U loads in flight per
// slot. Lanes of slot `slot` take tokens tb + u TPI + slot of each step; every slot keeps its own
// sums and running max, and the slots are merged at the end (weighted into a common frame), after
// which lanes 0 .. LPT - 1 hold the warp's o for columns lane N .. lane N + N - 1.
template <typename T, int D, int GM, bool ONLINE>
__device__ __forceinline__ void warp_pass_v(const KernelArgs& a, int b, int g, int t0, int t1,
                                            const float (&qr)[GM][Vec16<T>::N], const float (&ph)[GM],
                                            const int (&lim)[GM], float (&o)[GM][Vec16<T>::N],
                                            float (&l)[GM], float (&m)[GM], unsigned (&fl)[GM],
                                            bool& bad_block)
{
    constexpr int N = Vec16<T>::N;
    constexpr int LPT = D / N;
    constexpr int TPI = 32 / LPT;
    constexpr int U = 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = lane / LPT, li = lane - slot * LPT;
    const T* K = static_cast<const T*>(a.k);
    const T* V = static_cast<const T*>(a.v);
#pragma unroll
    for (int h = 0; h < GM; ++h) {
        l[h] = 0.f;
        m[h] = ONLINE ? -INFINITY : ph[h];
        fl[h] = 0u;
#pragma unroll
        for (int e = 0; e < N; ++e) o[h][e] = 0.f;
    }
    for (int tb = t0 + warp * U * TPI; tb < t1; tb += kWarps * U * TPI) {
        float kx[U][N], vx[U][N];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = tb + u * TPI + slot;
            ok[u] = t < t1;
            const long long row = ok[u] ? kv_row(a, b, t, g) : -1;
            if (ok[u] && row < 0) { bad_block = true; ok[u] = false; }
            if (ok[u]) {
                Vec16<T>::load(K + row + li * N, kx[u]);
                Vec16<T>::load(V + row + li * N, vx[u]);
            } else {
#pragma unroll
                for (int e = 0; e < N; ++e) { kx[u][e] = 0.f; vx[u][e] = 0.f; }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = tb + u * TPI + slot;
#pragma unroll
            for (int h = 0; h < GM; ++h) {
                if (h >= a.R) break;
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < N; ++e) part = fmaf(qr[h][e], kx[u][e], part);
#pragma unroll
                for (int sh = 1; sh < LPT; sh <<= 1) part += __shfl_xor_sync(0xffffffffu, part, sh);
                const bool valid = ok[u] && t < lim[h];
                const float s = __fmul_rn(part, a.scale);
                const float x = __fsub_rn(s, ph[h]);
                if (valid) fl[h] |= classify(x, a.lo, a.hi);
                if (ONLINE) {
                    const float mn = valid ? fmaxf(m[h], s) : m[h];
                    const float corr = (m[h] == mn) ? 1.f : (m[h] == -INFINITY ? 0.f : __expf(m[h] - mn));
                    const float p = valid ? __expf(s - mn) : 0.f;
                    l[h] = fmaf(l[h], corr, p);
#pragma unroll
                    for (int e = 0; e < N; ++e) o[h][e] = fmaf(o[h][e], corr, p * vx[u][e]);
                    m[h] = mn;
                } else {
                    const float p = valid ? __expf(x) : 0.f;
                    l[h] += p;
#pragma unroll
                    for (int e = 0; e < N; ++e) o[h][e] = fmaf(p, vx[u][e], o[h][e]);
                }
            }
        }
    }
    // the token slots of the warp into one frame (a plain sum in the phi frame)
#pragma unroll
    for (int sh = LPT; sh < 32; sh <<= 1) {
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            if (h >= a.R) break;
            const float mo = __shfl_xor_sync(0xffffffffu, m[h], sh);
            const float M = fmaxf(m[h], mo);
            const float ws = frame_weight(m[h], M), wo = frame_weight(mo, M);
            l[h] = fmaf(wo, __shfl_xor_sync(0xffffffffu, l[h], sh), ws * l[h]);
#pragma unroll
            for (int e = 0; e < N; ++e) o[h][e] = fmaf(wo, __shfl_xor_sync(0xffffffffu, o[h][e], sh), ws * o[h][e]);
            m[h] = M;
            fl[h] |= __shfl_xor_sync(0xffffffffu, fl[h], sh);
        }
    }
}

// Merges the warps' partials of unit (b, g, j) and writes them. Heads are written when
// `write_mask` has their bit; flags are OR-ed with `extra_flag` for written heads.
template <int E, int GM, int LPT = 32>
__device__ __forceinline__ void merge_and_store(const KernelArgs& a, SimtShared<E, GM>& sh, int b,
                                                int g, int j, const float (&o)[GM][E],
                                                const float (&l)[GM], const float (&m)[GM],
                                                const unsigned (&fl)[GM], unsigned write_mask,
                                                unsigned extra_flag, bool store_flags)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int D = a.D;
    __syncthreads();   // previous readers of sh are done
#pragma unroll
    for (int h = 0; h < GM; ++h) {
        if (h >= a.R) break;
        if (lane < LPT) {
#pragma unroll
            for (int e = 0; e < E; ++e) sh.o[warp][h][lane * E + e] = o[h][e];
        }
        if (lane == 0) { sh.l[warp][h] = l[h]; sh.m[warp][h] = m[h]; sh.f[warp][h] = fl[h]; }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < a.R * D; idx += kThreads) {
        const int h = idx / D, d = idx - h * D;
        if (!((write_mask >> h) & 1u)) continue;
        float M = sh.m[0][h];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) M = fmaxf(M, sh.m[w][h]);
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc = fmaf(frame_weight(sh.m[w][h], M), sh.o[w][h][d], acc);
        a.o_part[unit_row_slot(a, b, g, h, j) * D + d] = acc;
    }
    if (threadIdx.x < a.R && ((write_mask >> threadIdx.x) & 1u)) {
        const int h = threadIdx.x;
        float M = sh.m[0][h];
        unsigned f = sh.f[0][h];
        for (int w = 1; w < kWarps; ++w) { M = fmaxf(M, sh.m[w][h]); f |= sh.f[w][h]; }
        float lsum = 0.f;
        for (int w = 0; w < kWarps; ++w) lsum = fmaf(frame_weight(sh.m[w][h], M), sh.l[w][h], lsum);
        const long long r = unit_row_slot(a, b, g, h, j);
        a.l_part[r] = lsum;
        a.m_part[r] = M;
        if (store_flags) a.flags[r] = (uint8_t)(f | extra_flag);
        else a.flags[r] = (uint8_t)(a.flags[r] | extra_flag);
        sh.unit_flags[h] = f;
    }
    __syncthreads();
}

// VEC: the 16-byte-lane pass (E = elements per 16 bytes, at most GM = 4 rows, D a template
// parameter); else a token per warp, E = D / 32 elements per lane.
template <typename T, int E, int GM, bool VEC = false, int DV = 128>
__global__ void __launch_bounds__(kThreads) split_simt_kernel(KernelArgs a)
{
    constexpr int LPT = VEC ? DV / E : 32;      // lanes holding the warp's columns
    __shared__ SimtShared<E, GM> sh;
    int S, n_units;
    block_plan(a, sh.red, S, n_units);

    const int lane = threadIdx.x & 31;
    const T* Q = static_cast<const T*>(a.q);
    UnitCursor cur;
    cur.reset();
    bool bad_block = false;
    const unsigned all_heads = (a.R >= 32) ? 0xffffffffu : ((1u << a.R) - 1u);

    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        int b, g, j, L;
        cur.seek(a, a.Hkv, S, u, b, g, j, L);
        const int t0 = j * S, t1 = min(t0 + S, L);

        // the unit's R = Tq G query rows: row h is head g G + h % G of query token h / G
        float qr[GM][E];
        float ph[GM];                               // each row's unified max (its head's)
        int lim[GM];                                // each row's key limit
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            const int i = h / a.G, hh = h - i * a.G;
            if (h < a.R) {
                const T* qrow = Q + (((long long)b * a.Tq + i) * a.Hq + (long long)g * a.G + hh) * a.D;
                if constexpr (VEC)
                    Vec16<T>::load(qrow + (lane % LPT) * E, qr[h]);
                else
                    Elem<T>::template load<E>(qrow + lane * E, qr[h]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) qr[h][e] = 0.f;
            }
            ph[h] = h < a.R ? phi_of(a, g * a.G + hh) : a.phi;
            lim[h] = h < a.R ? key_limit(a, L, i) : 0;
        }
        float o[GM][E], l[GM], m[GM];
        unsigned fl[GM];
        auto pass = [&](auto online_c) {
            constexpr bool ONLINE = decltype(online_c)::value;
            if constexpr (VEC)
                warp_pass_v<T, DV, GM, ONLINE>(a, b, g, t0, t1, qr, ph, lim, o, l, m, fl, bad_block);
            else
                warp_pass<T, E, GM, ONLINE>(a, b, g, t0, t1, qr, ph, lim, o, l, m, fl, bad_block);
        };
        if (a.mode == FDPP_MODE_FORCE_ONLINE) {
            pass(std::true_type{});
            merge_and_store<E, GM, LPT>(a, sh, b, g, j, o, l, m, fl, all_heads, FDPP_FLAG_RECOMPUTED, true);
            continue;
        }
        pass(std::false_type{});
        merge_and_store<E, GM, LPT>(a, sh, b, g, j, o, l, m, fl, all_heads, 0u, true);
        if (a.mode != FDPP_MODE_NORMAL) continue;
        unsigned redo = 0u;
        for (int h = 0; h < a.R; ++h)
            if (sh.unit_flags[h] & FDPP_FLAG_OUT) redo |= 1u << h;
        if (!redo) continue;
        // the split left the safe window: read it again with the ordinary online softmax
        pass(std::true_type{});
        merge_and_store<E, GM, LPT>(a, sh, b, g, j, o, l, m, fl, redo, FDPP_FLAG_RECOMPUTED, false);
    }
    if (bad_block) set_error(a, FDPP_ERRBIT_BLOCK_TABLE);
}

// Score ranges for choosing phi in advance (opt.ai.kr "FlashDecoding++ async softmax -- theory",
// s3: phi is set by observing the distribution beforehand): for every unit, the least and greatest
// scaled score of each of its G heads over the split's tokens, the least into l_part and the
// greatest into m_part. Only K is read. Same plan and unit walk as the split kernel.
template <typename T, int E, int GM>
__global__ void __launch_bounds__(kThreads) score_range_kernel(KernelArgs a)
{
    __shared__ long long red[32];
    __shared__ float s_lo[kWarps][GM], s_hi[kWarps][GM];
    int S, n_units;
    block_plan(a, red, S, n_units);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T* Q = static_cast<const T*>(a.q);
    const T* K = static_cast<const T*>(a.k);
    UnitCursor cur;
    cur.reset();
    bool bad_block = false;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        int b, g, j, L;
        cur.seek(a, a.Hkv, S, u, b, g, j, L);
        const int t0 = j * S, t1 = min(t0 + S, L);
        float qr[GM][E];
        int lim[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            const int i = h / a.G, hh = h - i * a.G;
            if (h < a.R) {
                Elem<T>::template load<E>(Q + (((long long)b * a.Tq + i) * a.Hq + (long long)g * a.G + hh) * a.D + lane * E, qr[h]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) qr[h][e] = 0.f;
            }
            lim[h] = h < a.R ? key_limit(a, L, i) : 0;
        }
        float lo[GM], hi[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) { lo[h] = INFINITY; hi[h] = -INFINITY; }
        for (int t = t0 + warp; t < t1; t += kWarps) {
            const long long row = kv_row(a, b, t, g);
            if (row < 0) { bad_block = true; continue; }
            float kx[E];
            Elem<T>::template load<E>(K + row + lane * E, kx);
#pragma unroll
            for (int h = 0; h < GM; ++h) {
                if (h >= a.R) break;
                if (t >= lim[h]) continue;         // past this query row's keys (warp-uniform)
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) part = fmaf(qr[h][e], kx[e], part);
                part = warp_sum(part);
                const float s = __fmul_rn(part, a.scale);
                lo[h] = fminf(lo[h], s);
                hi[h] = fmaxf(hi[h], s);
            }
        }
        __syncthreads();                           // the previous unit's readers are done
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GM; ++h) { s_lo[warp][h] = lo[h]; s_hi[warp][h] = hi[h]; }
        }
        __syncthreads();
        if (threadIdx.x < a.R) {
            const int h = threadIdx.x;
            float mn = s_lo[0][h], mx = s_hi[0][h];
            for (int w = 1; w < kWarps; ++w) { mn = fminf(mn, s_lo[w][h]); mx = fmaxf(mx, s_hi[w][h]); }
            const long long r = unit_row_slot(a, b, g, h, j);
            a.l_part[r] = mn;
            a.m_part[r] = mx;
        }
    }
    if (bad_block) set_error(a, FDPP_ERRBIT_BLOCK_TABLE);
}

template <typename T, int E, int GM, bool VEC = false, int DV = 128>
cudaError_t launch_t(const KernelArgs& a, int grid, cudaStream_t s)
{
    split_simt_kernel<T, E, GM, VEC, DV><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

// up to 4 rows per kv head: 16-byte lanes; more: a token per warp
template <typename T>
cudaError_t launch_dtype(const KernelArgs& a, int grid, cudaStream_t s)
{
    constexpr int N = Vec16<T>::N;
    const bool e4 = (a.D == 128);
    if (a.R <= 4) return e4 ? launch_t<T, N, 4, true, 128>(a, grid, s) : launch_t<T, N, 4, true, 64>(a, grid, s);
    return e4 ? launch_t<T, 4, 16>(a, grid, s) : launch_t<T, 2, 16>(a, grid, s);
}

template <typename T, int E, int GM, bool VEC = false, int DV = 128>
int occ_t()
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, split_simt_kernel<T, E, GM, VEC, DV>, kThreads, 0) !=
        cudaSuccess)
        return 0;
    return n;
}

template <typename T>
int occ_dtype(const KernelArgs& a)
{
    constexpr int N = Vec16<T>::N;
    const bool e4 = (a.D == 128);
    if (a.R <= 4) return e4 ? occ_t<T, N, 4, true, 128>() : occ_t<T, N, 4, true, 64>();
    return e4 ? occ_t<T, 4, 16>() : occ_t<T, 2, 16>();
}

}  // namespace

cudaError_t launch_split_simt(const KernelArgs& a, int dtype, int grid, cudaStream_t s)
{
    return dtype == FDPP_F32 ? launch_dtype<float>(a, grid, s)
                             : launch_dtype<__nv_bfloat16>(a, grid, s);
}

int split_simt_ctas_per_sm(const KernelArgs& a, int dtype)
{
    return dtype == FDPP_F32 ? occ_dtype<float>(a) : occ_dtype<__nv_bfloat16>(a);
}

namespace {

template <typename T>
cudaError_t launch_ranges_dtype(const KernelArgs& a, int grid, cudaStream_t s)
{
    const bool e4 = (a.D == 128);
    if (a.R <= 4) {
        if (e4) score_range_kernel<T, 4, 4><<<grid, kThreads, 0, s>>>(a);
        else score_range_kernel<T, 2, 4><<<grid, kThreads, 0, s>>>(a);
    } else {
        if (e4) score_range_kernel<T, 4, 16><<<grid, kThreads, 0, s>>>(a);
        else score_range_kernel<T, 2, 16><<<grid, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

template <typename T>
int ranges_occ_dtype(const KernelArgs& a)
{
    int n = 0;
    const bool e4 = (a.D == 128);
    cudaError_t e;
    if (a.R <= 4)
        e = e4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_range_kernel<T, 4, 4>, kThreads, 0)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_range_kernel<T, 2, 4>, kThreads, 0);
    else
        e = e4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_range_kernel<T, 4, 16>, kThreads, 0)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, score_range_kernel<T, 2, 16>, kThreads, 0);
    return e == cudaSuccess ? n : 0;
}

}  // namespace

cudaError_t launch_score_ranges(const KernelArgs& a, int dtype, int grid, cudaStream_t s)
{
    return dtype == FDPP_F32 ? launch_ranges_dtype<float>(a, grid, s)
                             : launch_ranges_dtype<__nv_bfloat16>(a, grid, s);
}

int score_ranges_ctas_per_sm(const KernelArgs& a, int dtype)
{
    return dtype == FDPP_F32 ? ranges_occ_dtype<float>(a) : ranges_occ_dtype<__nv_bfloat16>(a);
}

}  // namespace fdpp
