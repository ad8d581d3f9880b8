// combine.cu -- cross-split combine: for every softmax row (sequence b, query head h) the sum of
// its split partials.
//
// opt.ai.kr "FlashDecoding++ async softmax -- theory", s3: with a unified max every split's
// partial (o_j, l_j) is already in the same frame, so only a plain sum remains. A split that
// was recomputed with online softmax carries its own max m_j, so the general form is
//     M = max_j m_j,  out = sum_j w_j o_j / sum_j w_j l_j,  w_j = exp(m_j - M)
// with w_j = 1 exactly when m_j == M: if no split of the row fell back (all m_j = phi) this is
// exactly the plain sum.
//
// Entries of a row. A split kernel that cut its work into parts (the tensor kernel, header
// HDR_PARTS = P > 0) leaves one partial per run: part c's share of one (row group, sequence,
// kv head) u, in run slot c + u. A run covers whole splits and pieces of splits in the phi frame;
// its rows whose scores left the window in one of its splits hold an empty partial there, and the
// fallback rewrote those rows piece by piece: a first piece that starts inside a split into the
// run slot, every other piece into its split's own slot, marked FDPP_FLAG_SLOT. So the row's
// entries are its head's run slots (the parts overlapping its tiles) and the own slots of its
// splits marked FDPP_FLAG_SLOT. A run that starts inside a split also carries that piece's window
// decisions (edge flags), which are ORed into the split's flag byte. A split kernel without parts
// (P = 0: the SIMT kernel, and very large batches) leaves one partial per split in its own slot.
//
// One pass. A warp owns a row (or, with ES warps per row for rows with many runs, a contiguous
// share of its runs and splits); each lane owns D/32 output columns, and the warp reads up to U
// entries at a time (each entry's columns in one coalesced load per lane, with its m and l),
// keeping a running max that is the same in every lane (the sums are rescaled only when the max
// grows, so phi-frame partials add with weight 1). The flag bytes are scanned 32 at a time. The
// slices of a row are added in warp order through shared memory. Every order is fixed, so results
// are deterministic. The result is rounded to nearest even into the output dtype.
//
// Launched as a programmatic dependent of the split kernel: it may start while the split kernel
// finishes, and waits (griddepcontrol.wait) before touching the partials. It lets the kernel
// after it launch early in turn (the next call's split kernel is a programmatic dependent too).
#include <cuda_bf16.h>

#include "device_common.cuh"

namespace fdpp {
namespace {

constexpr int NWC = 8;                // warps per CTA
constexpr int U = 8;                  // entries in flight per warp

template <typename T>
__device__ __forceinline__ void store_out(T* p, float x);

template <>
__device__ __forceinline__ void store_out<float>(float* p, float x) { *p = x; }

template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float x)
{
    *p = __float2bfloat16_rn(x);
}

// Running sums of one warp: acc (this lane's columns) and lam, in the frame of the max mrun.
template <int E>
struct Sums {
    float acc[E];
    float lam, mrun;

    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int c = 0; c < E; ++c) acc[c] = 0.f;
        lam = 0.f;
        mrun = -INFINITY;
    }
    __device__ __forceinline__ void add(float mv, float lv, const float (&ov)[E])
    {
        if (mv > mrun) {                             // a larger max: earlier sums shrink
            const float r = mrun == -INFINITY ? 0.f : __expf(mrun - mv);
#pragma unroll
            for (int c = 0; c < E; ++c) acc[c] *= r;
            lam *= r;
            mrun = mv;
        }
        const float w = frame_weight(mv, mrun);
#pragma unroll
        for (int c = 0; c < E; ++c) acc[c] = fmaf(w, ov[c], acc[c]);
        lam = fmaf(w, lv, lam);
    }
};

template <int E>
__device__ __forceinline__ void load_cols(const float* oj, float (&ov)[E])
{
    if constexpr (E == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(oj));
        ov[0] = v.x; ov[1] = v.y; ov[2] = v.z; ov[3] = v.w;
    } else {
        const float2 v = __ldg(reinterpret_cast<const float2*>(oj));
        ov[0] = v.x; ov[1] = v.y;
    }
}

// ES warps per row, NWC / ES rows per CTA.
template <typename T, int D, int ES>
__global__ void __launch_bounds__(NWC * 32) combine_kernel(KernelArgs a)
{
    constexpr int RPC = NWC / ES;
    constexpr int E = D / 32;                       // output columns per lane
    __shared__ float s_acc[ES > 1 ? NWC : 1][D];
    __shared__ float s_lam[NWC];
    __shared__ float s_max[NWC];
    // the next call's split kernel may launch now; it waits for this grid to complete before
    // it touches global memory
    grid_launch_dependents();
    grid_dependency_wait();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rw = warp / ES, slice = warp - rw * ES;
    // the split kernel has finished: its fallback-list counters go back to zero for the next call
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int i = 0; i < 2 * REDO_NLISTS; ++i) a.hdr[HDR_REDO_LISTS + i] = 0;
    }
    const long long rows = (long long)a.B * a.Tq * a.Hq;
    const long long row_ll = (long long)blockIdx.x * RPC + rw;
    const bool live = row_ll < rows;
    const int row = live ? (int)row_ll : 0;         // (b Tq + i) Hq + h: head h of query token i
    const int bi = row / a.Hq;                      // query row of the batch: b Tq + i
    const int b = bi / a.Tq;
    const int h = row - bi * a.Hq;
    // the row's place in the tensor kernel's units: kv-head row rr, in row group rr / 8 (the
    // virtual head kvh NRG + group) as row rr % 8 (the run-slot row)
    const int rr = (bi - b * a.Tq) * a.G + h % a.G;
    const int grp = a.NRG == 1 ? 0 : rr / TC_MAX_GROUP;
    const int rr8 = rr - grp * TC_MAX_GROUP;
    const int kvh = h / a.G;
    const int n = live ? a.nsplit[b] : 0;
    const long long fbase = (long long)row * a.max_splits;   // the row's flag bytes and split slots

    // Runs of the row's head u = (grp, b, kvh): it owns tiles [W, W + nt) of the split kernel's
    // order (row group, b, kv head, j), at [V, V + nt) in the cut stream that counts K phantom
    // tiles between heads (V = W + K u); part c = [floor(c T / P), floor((c + 1) T / P)) of that
    // stream (T with the phantoms).
    const int P = a.hdr[HDR_PARTS];
    long long W = 0, tiles = 1;
    int nt = 0, TS = 1, c_first = 0, n_r = 0, u = 0;
    if (P > 0 && n > 0) {
        tiles = a.hdr[HDR_TILES];
        TS = (a.hdr[HDR_SPLIT] + 63) / 64;
        nt = a.tstart[b + 1] - a.tstart[b];
        W = (long long)grp * a.Hkv * a.tstart[a.B] + (long long)a.Hkv * a.tstart[b] + (long long)kvh * nt;
        u = (grp * a.B + b) * a.Hkv + kvh;
        W += (long long)a.hdr[HDR_SEGK] * u;
        // the parts holding tiles W and W + nt - 1
        c_first = (int)(((W + 1) * P - 1) / tiles);
        n_r = (int)(((W + nt) * P - 1) / tiles) - c_first + 1;
    }
    const long long q_p = P > 0 ? tiles / P : 0;
    const int r_p = P > 0 ? (int)(tiles - q_p * P) : 0;

    Sums<E> sm;
    sm.zero();
    // the slice's splits j_lo .. j_hi - 1; the first 32 flag bytes are read together with the runs
    const int jper = (n + ES - 1) / ES;
    const int j_lo = slice * jper, j_hi = min(n, j_lo + jper);
    const unsigned f_first = (P > 0 && j_lo + lane < j_hi) ? __ldg(a.flags + fbase + j_lo + lane) : 0u;
    // the slice's runs, U at a time
    {
        const int per = (n_r + ES - 1) / ES;
        const int e_lo = slice * per, e_hi = min(n_r, e_lo + per);
        for (int eb = e_lo; eb < e_hi; eb += U) {
            float mv[U], lv[U], ov[U][E];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                if (eb + k >= e_hi) continue;
                const int c = c_first + eb + k;
                const long long rs = (long long)(c + u) * a.Rg + rr8;
                mv[k] = __ldg(a.xm + rs);
                lv[k] = __ldg(a.xl + rs);
                load_cols<E>(a.xo + rs * D + lane * E, ov[k]);
                // a run that starts inside a split: its edge flags go into the split's byte
                if (lane == 0) {
                    const long long ks = (long long)c * q_p + (c * r_p) / P - W;   // part start
                    if (ks > 0 && ks < nt) {
                        const int kt = (int)ks, jx = kt / TS;
                        if (kt != jx * TS) {
                            uint8_t* fb = a.flags + fbase + jx;
                            const uintptr_t addr = reinterpret_cast<uintptr_t>(fb);
                            const unsigned sh = (unsigned)(addr & 3u) * 8u;
                            atomicOr(reinterpret_cast<unsigned*>(addr & ~uintptr_t(3)),
                                     (unsigned)a.xf[rs] << sh);
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k)
                if (eb + k < e_hi) sm.add(mv[k], lv[k], ov[k]);
        }
    }
    // the slice's splits: with parts, only those whose own slot holds a recomputed piece
    {
        for (int jb = j_lo; jb < j_hi; jb += 32) {
            const int j = jb + lane;
            bool take = false;
            if (j < j_hi)
                take = P == 0 || ((jb == j_lo ? f_first : (unsigned)__ldg(a.flags + fbase + j)) & FDPP_FLAG_SLOT);
            unsigned mask = __ballot_sync(0xffffffffu, take);
            while (mask != 0u) {
                float mv[U], lv[U], ov[U][E];
                int cnt = 0;
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    if (mask == 0u) continue;
                    const int jj = jb + __ffs(mask) - 1;
                    mask &= mask - 1u;
                    mv[k] = __ldg(a.m_part + fbase + jj);
                    lv[k] = __ldg(a.l_part + fbase + jj);
                    load_cols<E>(a.o_part + (fbase + jj) * D + lane * E, ov[k]);
                    cnt = k + 1;
                }
#pragma unroll
                for (int k = 0; k < U; ++k)
                    if (k < cnt) sm.add(mv[k], lv[k], ov[k]);
            }
        }
    }
    if constexpr (ES > 1) {
        // the row's slices in warp order, each weighted to the row's max
#pragma unroll
        for (int c = 0; c < E; ++c) s_acc[warp][lane * E + c] = sm.acc[c];
        if (lane == 0) { s_lam[warp] = sm.lam; s_max[warp] = sm.mrun; }
        __syncthreads();
        if (slice != 0) return;
        const int w0 = rw * ES;
        float Mr = s_max[w0];
#pragma unroll
        for (int w = 1; w < ES; ++w) Mr = fmaxf(Mr, s_max[w0 + w]);
        sm.zero();
#pragma unroll
        for (int w = 0; w < ES; ++w) {
            const float wt = frame_weight(s_max[w0 + w], Mr);
#pragma unroll
            for (int c = 0; c < E; ++c) sm.acc[c] = fmaf(wt, s_acc[w0 + w][lane * E + c], sm.acc[c]);
            sm.lam = fmaf(wt, s_lam[w0 + w], sm.lam);
        }
    }
    if (live) {
        // a query row that sees no key (or a sequence without keys) is a zero row
        T* out = static_cast<T*>(a.out) + (long long)row * D + lane * E;
#pragma unroll
        for (int c = 0; c < E; ++c)
            store_out<T>(out + c, (n > 0 && sm.lam != 0.f) ? __fdiv_rn(sm.acc[c], sm.lam) : 0.f);
    }
}

// Warps per row: enough that a warp reads about U entries of a row at once. With parts a head's
// runs number about P / (its share of the heads) + 1 (the split kernel's grid bounds P; heads of
// equal length share the tiles evenly); without, a row has up to max_splits entries.
int slices_for(const KernelArgs& a, int split_grid)
{
    long long entries = a.max_splits;
    if (a.kernel_id == FDPP_KERNEL_TENSOR && a.B <= TC_PLAN_SMEM_MAX_B) {
        const long long heads = (long long)a.B * a.Hkv * a.NRG;
        entries = split_grid / heads + 2;
    }
    int es = 1;
    while (es < NWC && entries > (long long)U * es) es *= 2;
    return es;
}

template <typename T, int D, int ES>
cudaError_t launch_es(const KernelArgs& a, cudaStream_t s)
{
    const long long rows = (long long)a.B * a.Tq * a.Hq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + NWC / ES - 1) / (NWC / ES)));
    cfg.blockDim = dim3(NWC * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel<T, D, ES>, a);
}

template <typename T, int D>
cudaError_t launch_t(const KernelArgs& a, int split_grid, cudaStream_t s)
{
    switch (slices_for(a, split_grid)) {
    case 1: return launch_es<T, D, 1>(a, s);
    case 2: return launch_es<T, D, 2>(a, s);
    case 4: return launch_es<T, D, 4>(a, s);
    default: return launch_es<T, D, 8>(a, s);
    }
}

}  // namespace

cudaError_t launch_combine(const KernelArgs& a, int dtype, int split_grid, cudaStream_t s)
{
    cudaError_t e;
    if (dtype == FDPP_F32)
        e = a.D == 128 ? launch_t<float, 128>(a, split_grid, s) : launch_t<float, 64>(a, split_grid, s);
    else
        e = a.D == 128 ? launch_t<__nv_bfloat16, 128>(a, split_grid, s)
                       : launch_t<__nv_bfloat16, 64>(a, split_grid, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace fdpp
