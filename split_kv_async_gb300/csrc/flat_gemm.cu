// flat_gemm.cu -- the flat GEMM of decode-time linear layers, y = x W^T, on tcgen05 tensor cores.
//
// opt.ai.kr "FlashDecoding++ async softmax -- theory", s2 (2) and s4: the matrices of decoding's
// linear layers are flat (M, the batch's query tokens, is tiny; the weight N x K is fixed and
// large). Libraries pad M to a large tile with zeros, so most of their arithmetic is wasted; the
// remedy is to pad as little as possible and to double-buffer, computing while the next data
// arrives.
//
// GB300 form. The work is the stream of W (N K bf16), so the kernel is a weight-streaming
// pipeline:
//   - y^T = W x^T: 128 weight rows are the MMA's M, the M activation rows its N, padded only to
//     Mp = the next multiple of 16 (the smallest N of a 128-row MMA);
//   - one CTA per (128-row weight tile, K range); warp 0 streams 64-wide K slices of W and x with
//     TMA (128-byte swizzle) into a ring of shared-memory stages, warp 1 issues tcgen05.mma from
//     each stage into a TMEM accumulator (128 lanes x Mp fp32 columns) and returns the stage to
//     the producer through tcgen05.commit, warps 2-5 read the accumulator (tcgen05.ld) and write y;
//   - when the weight tiles alone are too few for the GPU, K is cut into split_k ranges, and the
//     split_k CTAs of a weight tile form one thread-block cluster: each leaves its fp32 partial
//     in its own shared memory, and after a cluster barrier each adds its share of the tile's
//     outputs from every member's shared memory (distributed shared memory), in range order, so
//     the result does not depend on timing and no partial goes through global memory.
// Every wait is bounded: on a timeout the CTA records FDPP_ERRBIT_TIMEOUT, lets its copies and
// MMAs land, frees its tensor memory and exits.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>

#include "device_common.cuh"
#include "fdpp_gemm.h"
#include "tcgen05.cuh"

namespace fdpp {
namespace {

constexpr int GB_N = 128;                // weight rows per tile (the MMA's M)
constexpr int GB_K = 64;                 // K elements per stage (one 128-byte swizzle row)
constexpr int GW_BYTES = GB_N * GB_K * 2;   // W slice of a stage
constexpr int G_THREADS = 192;           // producer warp, MMA warp, 4 epilogue warps
constexpr int G_MAX_STAGES = 8;
constexpr int G_MAX_SPLIT = 8;            // K ranges per weight tile (a portable cluster)

struct GemmArgs {
    __nv_bfloat16* y;
    unsigned* err;                       // sticky FDPP_ERRBIT_*
    int M, N, K, Mp;
    int split_k, kb_total, n_tiles, nstage;
    uint32_t idesc;                      // tcgen05 instruction descriptor
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void gemm_error(const GemmArgs& g, unsigned bit) { atomicOr(g.err, bit); }

// Barrier of every thread of the cluster; the arrive releases and the wait acquires this
// thread's (and, through them, the CTA's) shared-memory writes at cluster scope.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in cluster member `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// ---- the kernel ---------------------------------------------------------------------------

// Shared memory (dynamic, 1024-byte aligned base): nstage stages of [W slice 16 KB | x slice
// Mp x 128 B], then full[nstage], empty[nstage], the accumulator barrier, the TMEM address and
// the abort flag. Once every MMA has completed, the stages hold this CTA's fp32 partial
// [M][128] for the cluster reduction.
__global__ void __launch_bounds__(G_THREADS, 2)
    flat_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const GemmArgs g)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int xbytes = g.Mp * GB_K * 2;
    const int stage_bytes = GW_BYTES + xbytes;
    const uint32_t bars = sbase + g.nstage * stage_bytes;
    const uint32_t full = bars, empty = bars + 8 * g.nstage, accf = bars + 16 * g.nstage;
    volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(sm + g.nstage * stage_bytes + 16 * g.nstage + 8);
    volatile int* abort_ = reinterpret_cast<volatile int*>(sm + g.nstage * stage_bytes + 16 * g.nstage + 16);

    // a cluster per weight tile: its split_k CTAs take the K ranges in rank order
    const int tile = blockIdx.x / g.split_k;
    const int ks = g.split_k > 1 ? (int)cluster_rank() : 0;
    const int n0 = tile * GB_N;
    const int kb0 = (int)((long long)ks * g.kb_total / g.split_k);
    const int kb1 = (int)((long long)(ks + 1) * g.kb_total / g.split_k);
    const int nkb = kb1 - kb0;
    uint32_t ncols = 32;
    while ((int)ncols < g.Mp) ncols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < g.nstage; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        mbar_init(accf, 1);
        *abort_ = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32((const void*)tslot), ncols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    int issued = 0;                      // producer: slices issued
    if (warp == 0) {
        // ---- producer: W and x slices of this CTA's K range into the ring ----
        if (lane == 0) {
            // The weights are not written by the kernel before this one on the stream (a
            // programmatic dependency): the first ring's worth of W slices streams while that
            // kernel finishes; x, the workspace and y wait for it.
            const int pre = nkb < g.nstage ? nkb : g.nstage;
            for (int i = 0; i < pre; ++i) {
                const uint32_t dst = sbase + i * stage_bytes;
                mbar_arrive_expect_tx(full + 8 * i, (uint32_t)stage_bytes);
                tma_load_2d(dst, &tmW, (kb0 + i) * GB_K, n0, full + 8 * i);
            }
            grid_dependency_wait();
            for (int i = 0; i < pre; ++i)
                tma_load_2d(sbase + i * stage_bytes + GW_BYTES, &tmX, (kb0 + i) * GB_K, 0, full + 8 * i);
            issued = pre;
            for (int i = pre; i < nkb; ++i) {
                const int s = i % g.nstage;
                const uint32_t par = (uint32_t)(i / g.nstage) & 1u;
                if (*abort_ || !mbar_wait(empty + 8 * s, par ^ 1u)) {
                    gemm_error(g, FDPP_ERRBIT_TIMEOUT);
                    *abort_ = 1;
                    break;
                }
                const uint32_t dst = sbase + s * stage_bytes;
                const int k = (kb0 + i) * GB_K;
                mbar_arrive_expect_tx(full + 8 * s, (uint32_t)stage_bytes);
                tma_load_2d(dst, &tmW, k, n0, full + 8 * s);
                tma_load_2d(dst + GW_BYTES, &tmX, k, 0, full + 8 * s);
                ++issued;
            }
            // every load of this CTA is issued: the next kernel on the stream may launch
            grid_launch_dependents();
        } else {
            grid_dependency_wait();
        }
    } else if (warp == 1) {
        grid_dependency_wait();
        // ---- MMA issuer: four K=16 steps per slice, the stage returned when they complete ----
        if (lane == 0) {
            int done = 0;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % g.nstage;
                const uint32_t par = (uint32_t)(i / g.nstage) & 1u;
                if (*abort_ || !mbar_wait(full + 8 * s, par)) {
                    gemm_error(g, FDPP_ERRBIT_TIMEOUT);
                    *abort_ = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = sbase + s * stage_bytes, b0 = a0 + GW_BYTES;
#pragma unroll
                for (int kk = 0; kk < GB_K / 16; ++kk)
                    umma_bf16(tmem, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32), g.idesc,
                              (i > 0 || kk > 0) ? 1u : 0u);
                umma_commit(empty + 8 * s);
                ++done;
            }
            // the accumulator is complete (or, after an abort, every issued MMA has landed)
            umma_commit(accf);
            if (*abort_ && !mbar_wait(accf, 0)) gemm_error(g, FDPP_ERRBIT_TIMEOUT);
            (void)done;
        }
    } else {
        grid_dependency_wait();
        // ---- epilogue: TMEM lanes 32 (warp % 4) .. hold weight rows n0 + that lane ----
        const int q = warp & 3;
        const int n = n0 + 32 * q + lane;
        bool ok = mbar_wait(accf, 0);
        if (!ok) {
            gemm_error(g, FDPP_ERRBIT_TIMEOUT);
            *abort_ = 1;
        }
        ok = ok && !*abort_;
        tc_fence_after();
        // the tensor cores' reads of the stages are complete (accumulator barrier); the partial
        // of a split tile reuses that memory
        fence_proxy_async_smem();
        float* red = reinterpret_cast<float*>(sm);
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        if (ok) {
            for (int c = 0; c < g.Mp / 16; ++c) {
                float v[16];
                tmem_ld16(trow + 16 * c, v);
                if (n < g.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = 16 * c + j;
                        if (m >= g.M) break;
                        if (g.split_k == 1)
                            g.y[(long long)m * g.N + n] = __float2bfloat16_rn(v[j]);
                        else
                            red[m * GB_N + (n - n0)] = v[j];
                    }
                }
            }
        }
        tc_fence_before();
    }

    // ---- split tile: every member adds its share of the outputs from all members' partials ----
    __syncthreads();
    if (g.split_k > 1) {
        // every thread of every member passes both cluster barriers, whatever happened before
        cluster_sync_all();
        if (!*abort_) {
            // (m, 4-column group) pairs of the tile; member ks takes [ks P / S, (ks + 1) P / S)
            const int P = g.M * (GB_N / 4);
            const int p0 = (int)((long long)ks * P / g.split_k), p1 = (int)((long long)(ks + 1) * P / g.split_k);
            const uint32_t rbase = smem_u32(sm);
            for (int pidx = p0 + (int)threadIdx.x; pidx < p1; pidx += G_THREADS) {
                const int m = pidx / (GB_N / 4), c4 = pidx - m * (GB_N / 4);
                const int nn = n0 + 4 * c4;
                if (nn >= g.N) continue;
                const uint32_t off = rbase + (uint32_t)((m * GB_N + 4 * c4) * 4);
                float4 t[G_MAX_SPLIT];
#pragma unroll
                for (int r = 0; r < G_MAX_SPLIT; ++r)
                    if (r < g.split_k) t[r] = ld_dsmem_f4(dsmem_addr(off, (uint32_t)r));
                float4 acc = t[0];
#pragma unroll
                for (int r = 1; r < G_MAX_SPLIT; ++r)
                    if (r < g.split_k) {
                        acc.x += t[r].x; acc.y += t[r].y; acc.z += t[r].z; acc.w += t[r].w;
                    }
                __nv_bfloat16* yp = g.y + (long long)m * g.N + nn;
                const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
                if (nn + 3 < g.N && ((reinterpret_cast<uintptr_t>(yp) & 7u) == 0)) {
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(a4[0], a4[1]);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(a4[2], a4[3]);
                    uint2 pk;
                    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(yp) = pk;
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (nn + u < g.N) yp[u] = __float2bfloat16_rn(a4[u]);
                }
            }
        }
        // no member leaves (releasing its shared memory) while another still reads it
        cluster_sync_all();
    }

    // ---- teardown: copies and MMAs landed, tensor memory freed ----
    if (*abort_ && warp == 0 && lane == 0) {
        // let every slice still in flight land before the CTA's shared memory is released
        for (int i = issued > g.nstage ? issued - g.nstage : 0; i < issued; ++i) {
            const int s = i % g.nstage;
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(full + 8 * s, (uint32_t)(i / g.nstage) & 1u) && global_ns() - t0 < 100000000ull) {
            }
        }
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, ncols);
}

// ---- host ---------------------------------------------------------------------------------

fdpp_status gfail(fdpp_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_last_error(buf);
    return s;
}

bool shape_ok(int M, int N, int K) { return M >= 1 && M <= FDPP_GEMM_MAX_M && N >= 1 && K >= 8 && K % 8 == 0; }

int padded_m(int M) { return (M + 15) / 16 * 16; }

// Ring depth for two CTAs per SM.
int gemm_stages(int Mp, int smem_per_sm, int smem_per_block)
{
    const int stage = GW_BYTES + Mp * GB_K * 2;
    const int budget = std::min(smem_per_sm / 2 - 1024, smem_per_block) - 1024 - 256;
    return std::max(2, std::min(G_MAX_STAGES, budget / stage));
}

int gemm_smem_bytes(int Mp, int nstage) { return nstage * (GW_BYTES + Mp * GB_K * 2) + 16 * nstage + 32 + 1024; }

// Clusters of `split` CTAs the GPU holds at once for this ring (0 if the query fails); cached.
int max_active_clusters(int split, int Mp, int nstage)
{
    static std::mutex mu;
    static std::map<long long, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const long long key = ((long long)dev << 32) | ((long long)split << 16) | ((long long)Mp << 4) | nstage;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const int smem = gemm_smem_bytes(Mp, nstage);
    int n = 0;
    if (cudaFuncSetAttribute(flat_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)split);
        cfg.blockDim = dim3(G_THREADS);
        cfg.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)split;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, flat_gemm_kernel, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache[key] = n;
    return n;
}

// Heuristic split: the largest number of K ranges (at most G_MAX_SPLIT, at least two K slices
// each) whose clusters all fit on the GPU at once; one range when even the tiles alone do not.
int heuristic_split(int N, int K, int Mp, int nstage)
{
    const int tiles = (N + GB_N - 1) / GB_N;
    const int kb = (K + GB_K - 1) / GB_K;
    const int smax = std::max(1, std::min(G_MAX_SPLIT, kb / 2));
    for (int s = smax; s > 1; --s)
        if (tiles <= max_active_clusters(s, Mp, nstage)) return s;
    return 1;
}

struct LutEntry {
    int m_max, N, K, split_k;
};
// Lookup table of measured choices (fdpp_flat_gemm_set_lut), by (N, K) and the smallest M bucket
// that holds M.
LutEntry g_lut[64];
int g_lut_n = 0;

int choose_split(int M, int N, int K, int Mp, int nstage, int req)
{
    const int kb = (K + GB_K - 1) / GB_K;
    if (req > 0) return std::min(req, kb);   // checked against G_MAX_SPLIT by the caller
    int best = -1, best_m = 1 << 30;
    for (int i = 0; i < g_lut_n; ++i)
        if (g_lut[i].N == N && g_lut[i].K == K && M <= g_lut[i].m_max && g_lut[i].m_max < best_m) {
            best = i;
            best_m = g_lut[i].m_max;
        }
    if (best >= 0) return std::max(1, std::min(std::min(g_lut[best].split_k, kb), G_MAX_SPLIT));
    return heuristic_split(N, K, Mp, nstage);
}

// The workspace holds the sticky error word only (partials stay in the clusters' shared memory).
size_t ws_bytes(int, int, int) { return 256; }

fdpp_status encode_2d(CUtensorMap* map, const void* base, int rows, int K, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    fdpp_status st = get_tensor_map_encoder(&enc);
    if (st != FDPP_OK) return st;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {GB_K, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return gfail(FDPP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FDPP_OK;
}

}  // namespace
}  // namespace fdpp

using namespace fdpp;

extern "C" {

int fdpp_flat_gemm_split_k(int M, int N, int K, int split_k_req)
{
    if (!shape_ok(M, N, K) || split_k_req < 0) return 0;
    int sms = 0, smem_sm = 0, smem_blk = 0;
    if (query_device(&sms, &smem_sm, &smem_blk) != FDPP_OK) return 0;
    const int Mp = padded_m(M);
    return choose_split(M, N, K, Mp, gemm_stages(Mp, smem_sm, smem_blk), split_k_req);
}

size_t fdpp_flat_gemm_workspace_size(int M, int N, int K, int split_k_req)
{
    const int s = fdpp_flat_gemm_split_k(M, N, K, split_k_req);
    return s > 0 ? ws_bytes(M, N, s) : 0;
}

fdpp_status fdpp_flat_gemm_set_lut(const int32_t* entries, int n_entries)
{
    if (n_entries < 0 || n_entries > 64 || (n_entries > 0 && !entries))
        return gfail(FDPP_ERR_INVALID_ARG, "lookup table of %d entries (0 .. 64, 4 ints each)", n_entries);
    for (int i = 0; i < n_entries; ++i) {
        const int32_t* e = entries + 4 * i;
        if (e[0] < 1 || e[1] < 1 || e[2] < 8 || e[3] < 1)
            return gfail(FDPP_ERR_INVALID_ARG, "lookup table entry %d is not (m_max, N, K, split_k) >= (1, 1, 8, 1)", i);
    }
    for (int i = 0; i < n_entries; ++i) g_lut[i] = LutEntry{entries[4 * i], entries[4 * i + 1], entries[4 * i + 2], entries[4 * i + 3]};
    g_lut_n = n_entries;
    return FDPP_OK;
}

fdpp_status fdpp_flat_gemm(const void* x, const void* w, void* y, int M, int N, int K, int split_k, void* workspace,
                           size_t workspace_bytes, fdpp_stream stream)
{
    if (!shape_ok(M, N, K))
        return gfail(FDPP_ERR_INVALID_ARG, "flat GEMM shape M=%d N=%d K=%d (1 <= M <= %d, N >= 1, K >= 8, K %% 8 == 0)",
                     M, N, K, FDPP_GEMM_MAX_M);
    if (!x || !w || !y || !workspace) return gfail(FDPP_ERR_INVALID_ARG, "null pointer");
    if (((uintptr_t)x | (uintptr_t)w) % 16 != 0) return gfail(FDPP_ERR_INVALID_ARG, "x and w must be 16-byte aligned");
    if ((uintptr_t)workspace % 256 != 0) return gfail(FDPP_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    const int kb = (K + GB_K - 1) / GB_K;
    const int kmax = std::min(kb, G_MAX_SPLIT);
    if (split_k < 0 || split_k > kmax) return gfail(FDPP_ERR_INVALID_ARG, "split_k %d outside 0 .. %d", split_k, kmax);
    int sms = 0, smem_sm = 0, smem_blk = 0;
    fdpp_status st = query_device(&sms, &smem_sm, &smem_blk);
    if (st != FDPP_OK) return st;
    const int Mp = padded_m(M), nstage = gemm_stages(Mp, smem_sm, smem_blk);
    const int split = choose_split(M, N, K, Mp, nstage, split_k);
    const size_t need = ws_bytes(M, N, split);
    if (workspace_bytes < need)
        return gfail(FDPP_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);

    GemmArgs g{};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    g.err = reinterpret_cast<unsigned*>(ws);
    g.y = static_cast<__nv_bfloat16*>(y);
    g.M = M;
    g.N = N;
    g.K = K;
    g.Mp = Mp;
    g.split_k = split;
    g.kb_total = kb;
    g.n_tiles = (N + GB_N - 1) / GB_N;
    g.nstage = nstage;
    // kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1), both K-major,
    // N = Mp (bits 17-22 = N / 8), M = 128 (bits 24-28 = M / 16)
    g.idesc = umma_idesc_bf16(GB_N, g.Mp, false);

    CUtensorMap tw, tx;
    if ((st = encode_2d(&tw, w, N, K, GB_N)) != FDPP_OK) return st;
    if ((st = encode_2d(&tx, x, M, K, g.Mp)) != FDPP_OK) return st;
    const int smem = gemm_smem_bytes(Mp, nstage);
    cudaError_t e = cudaFuncSetAttribute(flat_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return gfail(FDPP_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    // a programmatic dependent of the kernel before it on the stream (see the producer)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(g.n_tiles * split));
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // the split_k CTAs of a weight tile are one cluster (consecutive block indices)
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, flat_gemm_kernel, tw, tx, g);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return gfail(FDPP_ERR_CUDA, "flat GEMM launch: %s", cudaGetErrorString(e));
    return FDPP_OK;
}

fdpp_status fdpp_flat_gemm_read_error(const void* workspace, uint32_t* error_bits)
{
    if (!workspace || !error_bits) return gfail(FDPP_ERR_INVALID_ARG, "null pointer");
    cudaError_t e = cudaMemcpy(error_bits, workspace, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return gfail(FDPP_ERR_CUDA, "cudaMemcpy: %s", cudaGetErrorString(e));
    return FDPP_OK;
}

}  // extern "C"
