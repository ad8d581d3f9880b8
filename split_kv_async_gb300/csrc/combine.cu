// combine.cu -- cross-split combine: one CTA (8 warps) per softmax row (sequence b, query head h).
//
// opt.ai.kr "FlashDecoding++ async softmax -- theory", s3: with a unified max every split's
// partial (o_j, l_j) is already in the same frame, so only a plain sum remains. A split that
// was recomputed with online softmax carries its own max m_j, so the general form is
//     M = max_j m_j,  out = sum_j w_j o_j / sum_j w_j l_j,  w_j = exp(m_j - M)
// with w_j = 1 exactly when m_j == M: if no split of the row fell back (all m_j = phi) this is
// exactly the plain sum.
//
// The row's partials (its n_b splits, then its extra slots) are divided into contiguous ranges,
// one per warp of the row (each lane owns 4 or 2 output columns), read 4 at a time per lane; the
// warp sums are then added in warp order. A row gets up to 32 warps while the rows fit on the
// GPU at that width, and fewer when there are many rows, so that all rows are in flight. The
// order is fixed, so results are deterministic. The result is rounded to nearest even into the
// output dtype.
//
// Extra slots. The tensor kernel cuts the 64-token tiles of all units (order b, g, j) into P
// equal parts, part c = tiles [floor(c T / P), floor((c + 1) T / P)). A part that starts inside
// a split (not on its first tile) computed that split's partial over its own tiles only and left
// it in extra slot c, in the phi frame or, if recomputed, in its own max frame. Partials of
// disjoint token sets of one split add up like those of different splits, so the combine adds
// each extra slot in with the same weights, and ORs its flag byte into the split's flag byte.
//
// Launched as a programmatic dependent of the split kernel: it may start while the split kernel
// finishes, and waits (griddepcontrol.wait) before touching the partials. It lets the kernel
// after it launch early in turn (the next call's split kernel is a programmatic dependent too).
#include <cuda_bf16.h>

#include "device_common.cuh"

namespace fdpp {
namespace {

constexpr int CW = 8;                 // warps per CTA of the many-rows build
constexpr int CW_WIDE = 32;           // warps per CTA when a few long rows take 16 or 32 warps each

template <typename T>
__device__ __forceinline__ void store_out(T* p, float x);

template <>
__device__ __forceinline__ void store_out<float>(float* p, float x) { *p = x; }

template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float x)
{
    *p = __float2bfloat16_rn(x);
}

template <typename T, int D, int NW>
__global__ void __launch_bounds__(NW * 32, NW == CW ? 3 : 1) combine_kernel(KernelArgs a, int wpr)
{
    constexpr int E = D / 32;                       // output columns per lane
    __shared__ float s_acc[NW][D];
    __shared__ float s_lam[NW];
    __shared__ float s_max[NW];
    // the next call's split kernel may launch now; it waits for this grid to complete before
    // it touches global memory
    grid_launch_dependents();
    grid_dependency_wait();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rpc = NW / wpr;                       // rows of this CTA, wpr warps each
    const int rl = warp / wpr, wr = warp - rl * wpr;
    const int row = blockIdx.x * rpc + rl;          // (b Tq + i) Hq + h: head h of query token i
    const bool live = row < a.B * a.Tq * a.Hq;
    // the split kernel has finished: its fallback-list counters go back to zero for the next call
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int i = 0; i < 2 * REDO_NLISTS; ++i) a.hdr[HDR_REDO_LISTS + i] = 0;
    }
    const int bi = live ? row / a.Hq : 0;           // query row of the batch: b Tq + i
    const int b = bi / a.Tq;
    const int h = live ? row - bi * a.Hq : 0;
    // the row's place in the tensor kernel's units: kv-head row rr, in row group rr / 8 (the
    // virtual head kvh NRG + group) as row rr % 8 (the extra-slot row)
    const int rr = (bi - b * a.Tq) * a.G + h % a.G;
    const int grp = a.NRG == 1 ? 0 : rr / TC_MAX_GROUP;
    const int rr8 = rr - grp * TC_MAX_GROUP;
    const int n = live ? a.nsplit[b] : 0;

    // Parts that may start inside this row's units: the row's kv head (and row group) owns tiles
    // [W, W + nt). The split kernel orders its tiles (row group, b, kv head, j).
    const int P = a.hdr[HDR_PARTS];
    long long W = 0, tiles = 1;
    int nt = 0, TS = 1, c_lo = 0, c_hi = -1;
    if (P > 0 && n > 0) {
        tiles = a.hdr[HDR_TILES];
        TS = (a.hdr[HDR_SPLIT] + 63) / 64;
        nt = a.tstart[b + 1] - a.tstart[b];
        W = (long long)grp * a.Hkv * a.tstart[a.B] + (long long)a.Hkv * a.tstart[b] +
            (long long)(h / a.G) * nt;
        c_lo = (int)(((W + 1) * P + tiles - 1) / tiles);   // first part starting after tile W
        c_hi = (int)(((W + nt) * P - 1) / tiles);           // last part starting before W + nt
    }
    // extra slot of part c belongs to split jx of this row, or c left none here. Part c starts at
    // floor(c tiles / P) = c q + floor(c r / P) with tiles = q P + r (32-bit arithmetic per part).
    const long long q_p = P > 0 ? tiles / P : 0;
    const int r_p = P > 0 ? (int)(tiles - q_p * P) : 0;
    auto extra_split = [&](int c) -> int {
        const long long k = (long long)c * q_p + (c * r_p) / P - W;
        if (k <= 0 || k >= nt) return -1;
        const int ki = (int)k;
        const int jx = ki / TS;
        return ki == jx * TS ? -1 : jx;
    };
    const float* xm = a.xm + rr8;
    const float* xl = a.xl + rr8;
    const float* xo = a.xo + (long long)rr8 * D;
    const long long base = (long long)row * a.max_splits;
    const float* m = a.m_part + base;
    const float* l = a.l_part + base;
    const float* o = a.o_part + base * D;

    // The row's entries: its n splits, then the candidate extra slots c_lo .. c_hi (those that
    // are not extra slots of this row are skipped). Entry e < n is split e.
    const int n_c = c_hi >= c_lo ? c_hi - c_lo + 1 : 0;
    const int n_e = n + n_c;

    // M = max over the row's partials; the extra slots' flag bytes are ORed into their splits'
    float M = -INFINITY;
    for (int e = wr * 32 + lane; e < n_e; e += wpr * 32) {
        if (e < n) {
            M = fmaxf(M, m[e]);
            continue;
        }
        const int c = c_lo + (e - n);
        const int jx = extra_split(c);
        if (jx >= 0) {
            M = fmaxf(M, xm[(long long)c * a.Rg]);
            // the split's flag byte also covers the extra slot's tokens
            uint8_t* fb = a.flags + (long long)row * a.max_splits + jx;
            const uintptr_t addr = reinterpret_cast<uintptr_t>(fb);
            const unsigned sh = (unsigned)(addr & 3u) * 8u;
            atomicOr(reinterpret_cast<unsigned*>(addr & ~uintptr_t(3)),
                     (unsigned)a.xf[(long long)c * a.Rg + rr8] << sh);
        }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
    if (lane == 0) s_max[warp] = M;
    __syncthreads();
    M = s_max[rl * wpr];
    for (int w = 1; w < wpr; ++w) M = fmaxf(M, s_max[rl * wpr + w]);

    // this warp's contiguous range of the row's entries, ascending, U loads in flight per lane
    const int per = (n_e + wpr - 1) / wpr;
    const int e0 = wr * per, e1 = min(n_e, e0 + per);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float lam = 0.f;
    constexpr int U = 4;
    for (int eb = e0; eb < e1; eb += U) {
        float mv[U], lv[U], ov[U][E];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = eb + u;
            ok[u] = false;
            const float *pm = m, *pl = l, *po = o;
            if (e < e1) {
                if (e < n) {
                    pm = m + e; pl = l + e; po = o + (long long)e * D;
                    ok[u] = true;
                } else {
                    const int c = c_lo + (e - n);
                    if (extra_split(c) >= 0) {
                        pm = xm + (long long)c * a.Rg; pl = xl + (long long)c * a.Rg;
                        po = xo + (long long)c * a.Rg * D;
                        ok[u] = true;
                    }
                }
            }
            if (ok[u]) {
                mv[u] = *pm;
                lv[u] = *pl;
                const float* oj = po + lane * E;
                if constexpr (E == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(oj);
                    ov[u][0] = v.x; ov[u][1] = v.y; ov[u][2] = v.z; ov[u][3] = v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(oj);
                    ov[u][0] = v.x; ov[u][1] = v.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (ok[u]) {
                const float w = frame_weight(mv[u], M);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(w, ov[u][e], acc[e]);
                lam = fmaf(w, lv[u], lam);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc[e];
    if (lane == 0) s_lam[warp] = lam;
    __syncthreads();
    // the row's warp sums in warp order; the first warp of the row writes the output
    if (live && wr == 0) {
        T* out = static_cast<T*>(a.out) + (long long)row * D;
        float ltot = 0.f;
        for (int w = 0; w < wpr; ++w) ltot += s_lam[rl * wpr + w];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane + 32 * e;
            float total = 0.f;
            for (int w = 0; w < wpr; ++w) total += s_acc[rl * wpr + w][d];
            // a query row that sees no key (or a sequence without keys) is a zero row
            store_out<T>(out + d, (n > 0 && ltot != 0.f) ? __fdiv_rn(total, ltot) : 0.f);
        }
    }
}

// Warps per row: up to 32 while the rows fit on the GPU at that width (a long row's partials
// are then read by many warps at once), fewer for many rows, so that all rows are in flight
// together.
int warps_per_row(long long rows, int num_sms)
{
    const long long resident = (long long)num_sms * 3 * CW;     // 3 CTAs of 8 warps per SM
    int w = CW_WIDE;
    while (w > 1 && rows * w > resident) w >>= 1;
    return w;
}

template <typename T, int D>
cudaError_t launch_t(const KernelArgs& a, cudaStream_t s)
{
    const long long rows = (long long)a.B * a.Tq * a.Hq;
    const int wpr = warps_per_row(rows, a.num_sms);
    const int nw = wpr > CW ? CW_WIDE : CW;
    const int rpc = nw / wpr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + rpc - 1) / rpc));
    cfg.blockDim = dim3((unsigned)(nw * 32));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (nw == CW_WIDE) return cudaLaunchKernelEx(&cfg, combine_kernel<T, D, CW_WIDE>, a, wpr);
    return cudaLaunchKernelEx(&cfg, combine_kernel<T, D, CW>, a, wpr);
}

}  // namespace

cudaError_t launch_combine(const KernelArgs& a, int dtype, cudaStream_t s)
{
    cudaError_t e;
    if (dtype == FDPP_F32)
        e = a.D == 128 ? launch_t<float, 128>(a, s) : launch_t<float, 64>(a, s);
    else
        e = a.D == 128 ? launch_t<__nv_bfloat16, 128>(a, s) : launch_t<__nv_bfloat16, 64>(a, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace fdpp
