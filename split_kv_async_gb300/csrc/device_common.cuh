// device_common.cuh -- device helpers shared by the kernels of libfdpp.
//
//  * the split scheduler (block-cooperative, run by every CTA so no plan launch is needed);
//  * the unit cursor that maps a unit index to (sequence b, kv head g, split j);
//  * inline-PTX wrappers for mbarrier, TMA (cp.async.bulk[.tensor]), ldmatrix and mma.sync;
//  * bounded waits: every wait gives up after FDPP_WAIT_NS nanoseconds of global time.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fdpp_internal.h"

namespace fdpp {

#ifndef FDPP_WAIT_NS
#define FDPP_WAIT_NS 2000000000ull   // 2 s of %globaltimer per wait
#endif

// ------------------------------------------------------------------------------------------
// split scheduler
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// Split length: the caller's S when > 0, otherwise spread sum_b L_b * Hkv over
// auto_units * num_sms units, rounded up to the granule and clamped to [auto_min, max_seq_len
// rounded up] (auto_units and auto_min from the dataflow table, else the defaults).
__device__ __forceinline__ int auto_split_len(long long total_tokens, const KernelArgs& a)
{
    if (a.split_req > 0) return a.split_req;
    long long units = (long long)a.auto_units * (long long)a.num_sms;
    if (units < 1) units = 1;
    long long gran = FDPP_AUTO_GRANULE;
    if (a.block_table && a.block_size > gran) gran = a.block_size;
    long long pairs = total_tokens * (long long)a.Hkv;
    long long S = (pairs + units - 1) / units;
    S = (S + gran - 1) / gran * gran;
    long long hi = ((long long)a.max_seq_len + gran - 1) / gran * gran;
    const long long lo = a.auto_min;
    if (hi < lo) hi = lo;
    if (S < lo) S = lo;
    if (S > hi) S = hi;
    return (int)S;
}

template <typename V>
__device__ __forceinline__ V warp_sum(V x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Block-wide sum of a 64-bit value. `red` is shared scratch of >= 32 long longs. All threads of
// the block call it; the result is returned to every thread.
__device__ __forceinline__ long long block_sum_ll(long long x, long long* red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    x = warp_sum(x);
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    long long t = 0;
    for (int w = 0; w < nw; ++w) t += red[w];
    return t;
}

// Every CTA computes the same plan: S and the unit count. CTA 0 also publishes the plan
// (nsplit[b] and the header) and reports out-of-range seq_lens. Called by all threads.
__device__ __forceinline__ void block_plan(const KernelArgs& a, long long* red, int& S_out,
                                           int& units_out)
{
    long long total = 0, bad = 0;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        int L = a.seq_lens[b];
        bad += (L < 0 || L > a.max_seq_len) ? 1 : 0;
        total += clamp_len(L, a.max_seq_len);
    }
    total = block_sum_ll(total, red);
    const int S = auto_split_len(total, a);
    long long n = 0;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        int nb = ceil_div_i(clamp_len(a.seq_lens[b], a.max_seq_len), S);
        if (nb > a.max_splits) nb = a.max_splits;       // cannot happen for valid S; keeps writes in bounds
        n += nb;
        if (blockIdx.x == 0) a.nsplit[b] = nb;
    }
    n = block_sum_ll(n, red);
    bad = block_sum_ll(bad, red);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        a.hdr[HDR_SPLIT] = S;
        a.hdr[HDR_UNITS] = (int)(n * a.Hkv);
        a.hdr[HDR_KERNEL] = a.kernel_id;
        a.hdr[HDR_BATCH] = a.B;
        a.hdr[HDR_MAXSPLITS] = a.max_splits;
        a.hdr[HDR_PARTS] = 0;                           // whole units only: no extra slots
        if (bad) atomicOr((unsigned*)&a.hdr[HDR_ERR], (unsigned)FDPP_ERRBIT_SEQ_LEN);
    }
    S_out = S;
    units_out = (int)(n * a.Hkv);
}

// Walks units in increasing order: unit u -> (b, g, j). Units are b-major, then kv head g,
// then split j; sequence b owns Hkv * n_b consecutive units.
struct UnitCursor {
    int b;
    int nb;
    long long base;

    __device__ __forceinline__ void reset() { b = -1; nb = 0; base = 0; }

    // heads: the heads of a sequence's units (Hkv, or the tensor kernel's virtual heads Hv)
    __device__ __forceinline__ void seek(const KernelArgs& a, int heads, int S, long long u, int& ub,
                                         int& ug, int& uj, int& L)
    {
        while (b < 0 || u >= base + (long long)heads * nb) {
            if (b >= 0) base += (long long)heads * nb;
            ++b;
            int n = ceil_div_i(clamp_len(a.seq_lens[b], a.max_seq_len), S);
            nb = n > a.max_splits ? a.max_splits : n;
        }
        long long r = u - base;
        ub = b;
        ug = (int)(r / nb);
        uj = (int)(r % nb);
        L = clamp_len(a.seq_lens[b], a.max_seq_len);
    }
};

__device__ __forceinline__ void set_error(const KernelArgs& a, unsigned bit)
{
    atomicOr((unsigned*)&a.hdr[HDR_ERR], bit);
}

// ------------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `parity` to complete; false after FDPP_WAIT_NS without completion.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && global_ns() - t0 > FDPP_WAIT_NS) return false;
    }
}

// 3-D tiled TMA load into shared memory, completing `bytes` on mbarrier `bar`. The K/V cache is
// read once per step, so its lines are marked first to go from L2 (evict_first): the split
// partials, the next step's prefetched tiles and the small per-call arrays stay there instead.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar)
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
        : "memory");
}

// 4-D tiled TMA load into shared memory (default L2 policy), completing on mbarrier `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// L2 prefetch of a 3-D tiled box (no destination, no completion signal).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Plain bulk copy global -> shared (size and both addresses multiples of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Brings the 128-byte line holding p into L2 (no register result, no completion).
__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transposes an 8x8 matrix of 16-bit elements held across the warp in the mma fragment layout
// (lane 4r + c holds row r, columns 2c and 2c+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// GPU-scope acquire/release atomics (one thread publishes or observes a whole CTA's writes; a
// CTA barrier before the release, or after the acquire, carries them to the other threads).
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_release_gpu(long long* p, long long v)
{
    asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ long long ld_acquire_gpu(const long long* p)
{
    long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Orders this thread's generic-proxy shared-memory accesses before later async-proxy (TMA)
// accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: allow the next kernel in the stream to start launching, and
// (in that kernel) wait until the previous one has completed and its memory is visible.
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Window decision for x = s - phi (closed window; NaN is outside).
__device__ __forceinline__ unsigned classify(float x, float lo, float hi)
{
    if (x >= lo && x <= hi) return 0u;
    if (x != x) return FDPP_FLAG_OUT | FDPP_FLAG_NAN;
    return x > hi ? (FDPP_FLAG_OUT | FDPP_FLAG_ABOVE) : (FDPP_FLAG_OUT | FDPP_FLAG_BELOW);
}

// Partial slot of query row rr of unit (b, g): query token i = rr / G of sequence b, head
// g G + rr % G, split j. Partial arrays are [B][Tq][Hq][max_splits].
__device__ __forceinline__ long long unit_row_slot(const KernelArgs& a, int b, int g, int rr, int j)
{
    const int i = rr / a.G, hh = rr - i * a.G;
    return (((long long)b * a.Tq + i) * a.Hq + (long long)g * a.G + hh) * a.max_splits + j;
}

// Keys query token i of a sequence with L keys sees: t < L - Tq + 1 + i (causal over the last
// Tq positions; all L keys for Tq = 1).
__device__ __forceinline__ int key_limit(const KernelArgs& a, int L, int i)
{
    const int lim = L - a.Tq + 1 + i;
    return lim < 0 ? 0 : lim;
}

// Unified max of query head h: its own value when the caller gave one per head.
__device__ __forceinline__ float phi_of(const KernelArgs& a, int h)
{
    return a.phi_heads ? __ldg(a.phi_heads + h) : a.phi;
}

// exp(m_w - M) with the exact 1 when the frames agree (so phi-frame partials add plainly).
__device__ __forceinline__ float frame_weight(float m, float M)
{
    return m == M ? 1.0f : __expf(m - M);
}

}  // namespace fdpp
