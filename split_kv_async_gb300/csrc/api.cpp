// api.cpp -- the C ABI of libfdpp: argument checks, workspace layout, kernel choice, TMA
// descriptors and launches. Every entry point here is declared and documented in fdpp.h.
//
// A decode step is two stream-ordered launches:
//   1. the split kernel (tensor-core or SIMT variant), persistent over the (b, g, j) units: split
//      plan, phi-frame partials, window test and fallback recompute. Kernels plan the splits
//      themselves from seq_lens on the device, so no plan launch and no host sync is needed;
//   2. the combine kernel, one CTA per (b, h) row, launched as a programmatic dependent so its
//      launch overlaps the split kernel's tail.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fdpp.h"
#include "fdpp_internal.h"

using namespace fdpp;

namespace {

thread_local std::string g_last_error;

fdpp_status fail(fdpp_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int q_tokens_of(const fdpp_params& p) { return p.q_tokens > 1 ? p.q_tokens : 1; }

int max_splits_of(const fdpp_params& p)
{
    const long long S = p.split_len > 0 ? p.split_len : FDPP_AUTO_MIN_SPLIT;
    return (int)((p.max_seq_len + S - 1) / S);
}

// Host-only checks shared by every entry point (no CUDA call).
fdpp_status check_params(const fdpp_params* p)
{
    if (!p) return fail(FDPP_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1) return fail(FDPP_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", p->batch);
    if (p->num_q_heads < 1 || p->num_kv_heads < 1)
        return fail(FDPP_ERR_INVALID_ARG, "head counts must be >= 1");
    if (p->num_q_heads % p->num_kv_heads)
        return fail(FDPP_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                    p->num_q_heads, p->num_kv_heads);
    if (p->dtype != FDPP_F32 && p->dtype != FDPP_BF16)
        return fail(FDPP_ERR_INVALID_ARG, "dtype must be FDPP_F32 or FDPP_BF16 (got %d)", p->dtype);
    if (p->head_dim != 64 && p->head_dim != 128)
        return fail(FDPP_ERR_UNSUPPORTED, "head_dim %d: only 64 and 128 are built", p->head_dim);
    if (p->max_seq_len < 1) return fail(FDPP_ERR_INVALID_ARG, "max_seq_len must be >= 1");
    if (p->split_len < 0) return fail(FDPP_ERR_INVALID_ARG, "split_len must be >= 0");
    if (!std::isfinite(p->scale) || !std::isfinite(p->phi) || !std::isfinite(p->lo) ||
        !std::isfinite(p->hi))
        return fail(FDPP_ERR_INVALID_ARG, "scale, phi, lo and hi must be finite");
    if (!(p->lo <= p->hi)) return fail(FDPP_ERR_INVALID_ARG, "window needs lo <= hi");
    if (!(p->scale > 0.f)) return fail(FDPP_ERR_INVALID_ARG, "scale must be positive (got %g)", (double)p->scale);
    if (p->mode < FDPP_MODE_NORMAL || p->mode > FDPP_MODE_FORCE_ONLINE)
        return fail(FDPP_ERR_INVALID_ARG, "unknown mode %d", p->mode);
    if (p->kernel < FDPP_KERNEL_AUTO || p->kernel > FDPP_KERNEL_SIMT)
        return fail(FDPP_ERR_INVALID_ARG, "unknown kernel %d", p->kernel);
    if (p->tc_stages < 0 || p->tc_stages == 1 || p->tc_stages > 12)
        return fail(FDPP_ERR_INVALID_ARG, "tc_stages must be 0 or in [2, 12]");
    if (p->tc_ctas_per_sm < 0 || p->tc_ctas_per_sm > 2)
        return fail(FDPP_ERR_INVALID_ARG, "tc_ctas_per_sm must be 0, 1 or 2");
    if (p->tc_prefetch < -1 || p->tc_prefetch > 32)
        return fail(FDPP_ERR_INVALID_ARG, "tc_prefetch must be -1, 0 or in [1, 32]");
    if (p->phi_heads && ((uintptr_t)p->phi_heads % 4) != 0)
        return fail(FDPP_ERR_INVALID_ARG, "phi_heads must be 4-byte aligned");
    if (p->q_tokens < 0 || p->q_tokens > 64)
        return fail(FDPP_ERR_INVALID_ARG, "q_tokens must be in [0, 64] (got %d)", p->q_tokens);
    if (p->tc_mma < FDPP_TC_MMA_AUTO || p->tc_mma > FDPP_TC_MMA_TCGEN05)
        return fail(FDPP_ERR_INVALID_ARG, "unknown tc_mma %d", p->tc_mma);
    const int G = p->num_q_heads / p->num_kv_heads;
    const int R = q_tokens_of(*p) * G;
    if (R > TC_MAX_ROWS)
        return fail(FDPP_ERR_UNSUPPORTED, "query rows per kv head (q_tokens x heads per kv head) %d > %d",
                    R, TC_MAX_ROWS);
    // sizes stay far from overflow: partials below 2^50 bytes, unit indices below 2^31
    const long double o_bytes = (long double)p->batch * q_tokens_of(*p) * p->num_q_heads *
                                max_splits_of(*p) * p->head_dim * 4.0L;
    const long double units = (long double)p->batch * p->num_kv_heads * max_splits_of(*p);
    if (o_bytes > 1e15L || units > 2e9L)
        return fail(FDPP_ERR_INVALID_ARG, "problem too large for one workspace");
    return FDPP_OK;
}

fdpp_status check_paged(const fdpp_params* p)
{
    if (!is_pow2(p->block_size) || p->block_size < 16 || p->block_size > 256)
        return fail(FDPP_ERR_INVALID_ARG, "block_size must be a power of two in [16, 256] (got %d)",
                    p->block_size);
    if (p->max_blocks_per_seq < 1) return fail(FDPP_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
    if (p->num_kv_blocks < 1) return fail(FDPP_ERR_INVALID_ARG, "num_kv_blocks must be >= 1");
    if ((long long)p->max_seq_len > (long long)p->max_blocks_per_seq * p->block_size)
        return fail(FDPP_ERR_INVALID_ARG, "max_seq_len exceeds max_blocks_per_seq * block_size");
    if (p->split_len > 0 && p->split_len % p->block_size)
        return fail(FDPP_ERR_INVALID_ARG, "split_len (%d) must be a multiple of block_size (%d)",
                    p->split_len, p->block_size);
    return FDPP_OK;
}

// Entries of one fallback list: one per split piece a run may push.
// Row groups of the tensor kernel: each (kv head, group of up to 8 query rows) is a unit head.
int row_groups_of(const fdpp_params& p)
{
    const int R = q_tokens_of(p) * (p.num_q_heads / p.num_kv_heads);
    return (R + TC_MAX_GROUP - 1) / TC_MAX_GROUP;
}

// The tcgen05 build can take the call: bf16, d = 128, more than 8 query rows per kv head.
bool um_applies(const fdpp_params& p)
{
    const int R = q_tokens_of(p) * (p.num_q_heads / p.num_kv_heads);
    return p.dtype == FDPP_BF16 && p.head_dim == 128 && R > TC_MAX_GROUP && R <= TC_MAX_ROWS;
}

// The tcgen05 build's ring depth for short parts (measured on a GB300: 4 stages beat 5 at 27
// tiles per CTA, tie at 54, lose at 108).
constexpr int UM_SHORT_STAGES = 4;
constexpr int UM_SHORT_TILES = 48;

// The tcgen05 build's cost of a run boundary inside a CTA's part (the epilogue of one run and the
// start of the next, while its stream waits), in 64-token tiles at the copy rate: the partition
// counts that many phantom tiles between units, so a part that holds a boundary takes fewer tiles.
// Measured best on a GB300 over 134 MB caches at 16, 32 and 64 rows per kv head.
int um_seg_tiles(int R) { return R > 32 ? 9 : 6; }

// The tensor kernel of this call is the tcgen05 build (tc_mma, and the geometry asked for).
bool um_selected(const fdpp_params& p)
{
    if (!um_applies(p) || p.tc_mma == FDPP_TC_MMA_SYNC) return false;
    return p.tc_mma == FDPP_TC_MMA_TCGEN05 || p.tc_ctas_per_sm <= 1;
}

size_t redo_capacity(const fdpp_params& p)
{
    // split pieces: every split once, plus one more per run boundary (parts + heads)
    const size_t heads = (size_t)p.batch * p.num_kv_heads * row_groups_of(p);
    return heads * max_splits_of(p) + TC_MAX_PARTS + heads;
}

WsLayout layout_of(const fdpp_params& p)
{
    WsLayout w{};
    w.max_splits = max_splits_of(p);
    const size_t rows = (size_t)p.batch * q_tokens_of(p) * p.num_q_heads;
    const size_t slots = rows * (size_t)w.max_splits;
    size_t off = 0;
    w.header = off;  off = align256(off + HDR_WORDS * 4);
    w.nsplit = off;  off = align256(off + (size_t)p.batch * 4);
    w.tstart = off;  off = align256(off + ((size_t)p.batch + 1) * 4);
    // a fallback entry per unit, plus one per part for units cut in two
    const size_t entries = redo_capacity(p);
    w.redo = off;    off = align256(off + REDO_NLISTS * entries * REDO_WORDS * 8);
    w.hint = off;    off = align256(off + (size_t)TC_MAX_PARTS * HINT_WORDS * 4);
    w.flags = off;   off = align256(off + slots);
    w.m_part = off;  off = align256(off + slots * 4);
    w.l_part = off;  off = align256(off + slots * 4);
    w.o_part = off;  off = align256(off + slots * (size_t)p.head_dim * 4);
    // run slots of the tensor kernel: a run is a part's share of one (row group, sequence, kv
    // head), so there are fewer than parts + (row groups x sequences x kv heads) of them, each
    // of min(R, 8) rows; the tcgen05 build's runs hold all R rows, with at most TC_UM_MAX_CTAS
    // parts
    const size_t R = (size_t)q_tokens_of(p) * (size_t)(p.num_q_heads / p.num_kv_heads);
    const size_t runs = (size_t)TC_MAX_PARTS + (size_t)p.batch * p.num_kv_heads * row_groups_of(p);
    size_t xrows = runs * (R < TC_MAX_GROUP ? R : TC_MAX_GROUP);
    if (um_applies(p)) {
        const size_t um_rows = ((size_t)TC_UM_MAX_CTAS + (size_t)p.batch * p.num_kv_heads) * R;
        if (um_rows > xrows) xrows = um_rows;
    }
    w.xf = off;      off = align256(off + xrows);
    w.xm = off;      off = align256(off + xrows * 4);
    w.xl = off;      off = align256(off + xrows * 4);
    w.xo = off;      off = align256(off + xrows * (size_t)p.head_dim * 4);
    w.total = off;
    return w;
}

bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

// The heuristic dataflow table of decode attention (fdpp_attn_set_lut): process-wide, copied in.
std::mutex g_lut_mutex;
std::vector<fdpp_attn_lut_row> g_lut;

struct AutoChoice {
    int kernel, units, min_split;
};

// The kernel and split-scheduler parameters a call with `p` uses: the first table row whose
// ranges hold the shape, else the defaults; a kernel named by the table that cannot take the
// call (dtype, rows per kv head) leaves the default rule.
AutoChoice auto_choice(const fdpp_params& p)
{
    const int R = q_tokens_of(p) * (p.num_q_heads / p.num_kv_heads);
    const bool tc_ok = p.dtype == FDPP_BF16 && R <= TC_MAX_ROWS;
    const bool simt_ok = R <= SIMT_MAX_GROUP;
    AutoChoice c{p.kernel, FDPP_AUTO_UNITS_PER_SM, FDPP_AUTO_MIN_SPLIT};
    int lut_kernel = FDPP_KERNEL_AUTO;
    {
        std::lock_guard<std::mutex> lk(g_lut_mutex);
        for (const fdpp_attn_lut_row& r : g_lut) {
            if (p.batch <= r.max_batch && p.max_seq_len <= r.max_seq_len && R <= r.max_rows) {
                lut_kernel = r.kernel;
                c.units = r.units_per_sm;
                c.min_split = r.min_split;
                break;
            }
        }
    }
    if (c.kernel == FDPP_KERNEL_AUTO) {
        if ((lut_kernel == FDPP_KERNEL_TENSOR && tc_ok) || (lut_kernel == FDPP_KERNEL_SIMT && simt_ok))
            c.kernel = lut_kernel;
        else
            c.kernel = tc_ok ? FDPP_KERNEL_TENSOR : FDPP_KERNEL_SIMT;
    }
    return c;
}

struct DeviceInfo {
    bool valid = false;
    int sms = 0, smem_per_sm = 0, smem_per_block = 0;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

fdpp_status device_info(DeviceInfo& out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FDPP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(FDPP_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.valid) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail(FDPP_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        if (major != 10 || minor != 3)
            return fail(FDPP_ERR_UNSUPPORTED, "libfdpp is built for sm_103a only (device is sm_%d%d)",
                        major, minor);
        d.valid = true;
    }
    out = d;
    return FDPP_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

fdpp_status tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000& fn)
{
    std::call_once(g_encode_once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    if (!g_encode) return fail(FDPP_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    fn = g_encode;
    return FDPP_OK;
}

// 3-D bf16 tensor map over a K or V cache with 128-byte swizzle and 64-element-wide boxes.
//   contiguous: dims {Hkv*d, Lmax, B},          box {64, 64, 1}
//   paged:      dims {Hkv*d, block_size, nblk}, box {64, min(block_size, 64), 1}
fdpp_status encode_kv_map(CUtensorMap* map, const void* base, const fdpp_params& p, bool paged)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    fdpp_status st = tensor_map_encoder(enc);
    if (st != FDPP_OK) return st;
    const cuuint64_t row = (cuuint64_t)p.num_kv_heads * p.head_dim;
    const cuuint64_t d1 = paged ? (cuuint64_t)p.block_size : (cuuint64_t)p.max_seq_len;
    const cuuint64_t d2 = paged ? (cuuint64_t)p.num_kv_blocks : (cuuint64_t)p.batch;
    cuuint64_t dims[3] = {row, d1, d2};
    cuuint64_t strides[2] = {row * 2, row * 2 * d1};
    const cuuint32_t box_rows =
        (cuuint32_t)(paged ? (p.block_size < TC_TILE_TOKENS ? p.block_size : TC_TILE_TOKENS)
                           : TC_TILE_TOKENS);
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FDPP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FDPP_OK;
}

// 4-D bf16 tensor map over q for the tcgen05 build: dims {d, Hq, Tq, B}, box {64, G, Tq, 1}, so
// one load lands the R = Tq G query rows of a kv head (row i G + h = head g G + h of query token
// i) as R rows of 128 bytes, 128-byte swizzled: the K-major B operand of S^T = K Q^T.
fdpp_status encode_q_map(CUtensorMap* map, const void* q, const fdpp_params& p)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    fdpp_status st = tensor_map_encoder(enc);
    if (st != FDPP_OK) return st;
    const cuuint64_t D = (cuuint64_t)p.head_dim, Hq = (cuuint64_t)p.num_q_heads;
    const cuuint64_t Tq = (cuuint64_t)q_tokens_of(p);
    cuuint64_t dims[4] = {D, Hq, Tq, (cuuint64_t)p.batch};
    cuuint64_t strides[3] = {D * 2, Hq * D * 2, Tq * Hq * D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)(p.num_q_heads / p.num_kv_heads), (cuuint32_t)Tq, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FDPP_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
    return FDPP_OK;
}

// Everything the kernels of one call need: pointers into the caller's buffers and workspace,
// and the shape.
KernelArgs kernel_args(const fdpp_params& P, const WsLayout& w, void* workspace, const void* q,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* seq_lens, void* out, int num_sms, int kernel, bool um = false)
{
    const fdpp_params* p = &P;
    const bool paged = block_table != nullptr;
    const int G = p->num_q_heads / p->num_kv_heads;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    KernelArgs a{};
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = out;
    a.hdr = reinterpret_cast<int32_t*>(ws + w.header);
    a.nsplit = reinterpret_cast<int32_t*>(ws + w.nsplit);
    a.tstart = reinterpret_cast<int32_t*>(ws + w.tstart);
    a.redo = reinterpret_cast<long long*>(ws + w.redo);
    a.hint = reinterpret_cast<int32_t*>(ws + w.hint);
    a.redo_cap = (int)redo_capacity(*p);
    a.flags = ws + w.flags;
    a.m_part = reinterpret_cast<float*>(ws + w.m_part);
    a.l_part = reinterpret_cast<float*>(ws + w.l_part);
    a.o_part = reinterpret_cast<float*>(ws + w.o_part);
    a.xf = ws + w.xf;
    a.xm = reinterpret_cast<float*>(ws + w.xm);
    a.xl = reinterpret_cast<float*>(ws + w.xl);
    a.xo = reinterpret_cast<float*>(ws + w.xo);
    a.B = p->batch;
    a.Hq = p->num_q_heads;
    a.Hkv = p->num_kv_heads;
    a.G = G;
    a.Tq = q_tokens_of(*p);
    a.R = a.Tq * G;
    // the tcgen05 build takes all R rows of a kv head in one unit: one row group of R rows
    a.NRG = um ? 1 : row_groups_of(*p);
    a.Rg = um ? a.R : (a.R < TC_MAX_GROUP ? a.R : TC_MAX_GROUP);
    a.Hv = p->num_kv_heads * a.NRG;
    a.D = p->head_dim;
    a.max_seq_len = p->max_seq_len;
    a.block_size = paged ? p->block_size : 0;
    a.max_blocks = paged ? p->max_blocks_per_seq : 0;
    a.num_blocks = paged ? p->num_kv_blocks : 0;
    a.split_req = p->split_len;
    a.max_splits = w.max_splits;
    a.num_sms = num_sms;
    a.scale = p->scale;
    a.phi = p->phi;
    a.phi_heads = p->phi_heads;
    a.lo = p->lo;
    a.hi = p->hi;
    a.mode = p->mode;
    a.kernel_id = kernel;
    const AutoChoice ch = auto_choice(*p);
    a.auto_units = ch.units;
    a.auto_min = ch.min_split;
    a.seg_tiles = um ? um_seg_tiles(a.R) : 0;
    return a;
}

}  // namespace

namespace fdpp {

fdpp_status query_device(int* sms, int* smem_per_sm, int* smem_per_block)
{
    DeviceInfo d;
    const fdpp_status st = device_info(d);
    if (st != FDPP_OK) return st;
    if (sms) *sms = d.sms;
    if (smem_per_sm) *smem_per_sm = d.smem_per_sm;
    if (smem_per_block) *smem_per_block = d.smem_per_block;
    return FDPP_OK;
}

fdpp_status get_tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn)
{
    return tensor_map_encoder(*fn);
}
// Bytes at the start of a workspace for `p` that hold the state which must be zero before a call:
// header, plan and the fallback list (everything before the flag bytes).
size_t workspace_zero_prefix(const fdpp_params& p) { return layout_of(p).flags; }
// Offset of the start-up hint region: everything before it (header, plan, fallback lists) is
// the state that a call must find zeroed or written by the call before it.
size_t workspace_hint_offset(const fdpp_params& p) { return layout_of(p).hint; }
// Sets the reason fdpp_last_error() reports on this thread.
void set_last_error(const char* what) { g_last_error = what; }
}  // namespace fdpp

extern "C" {

const char* fdpp_status_str(fdpp_status s)
{
    switch (s) {
    case FDPP_OK: return "FDPP_OK";
    case FDPP_ERR_INVALID_ARG: return "FDPP_ERR_INVALID_ARG";
    case FDPP_ERR_UNSUPPORTED: return "FDPP_ERR_UNSUPPORTED";
    case FDPP_ERR_WORKSPACE: return "FDPP_ERR_WORKSPACE";
    case FDPP_ERR_CUDA: return "FDPP_ERR_CUDA";
    }
    return "FDPP_UNKNOWN_STATUS";
}

const char* fdpp_last_error(void) { return g_last_error.c_str(); }

fdpp_status fdpp_attn_set_lut(const fdpp_attn_lut_row* rows, int n)
{
    if (n < 0 || (n > 0 && !rows)) return fail(FDPP_ERR_INVALID_ARG, "rows is NULL or n < 0");
    if (n > 4096) return fail(FDPP_ERR_INVALID_ARG, "at most 4096 table rows (got %d)", n);
    for (int i = 0; i < n; ++i) {
        const fdpp_attn_lut_row& r = rows[i];
        if (r.max_batch < 1 || r.max_seq_len < 1 || r.max_rows < 1)
            return fail(FDPP_ERR_INVALID_ARG, "table row %d: ranges must be >= 1", i);
        if (r.kernel < FDPP_KERNEL_AUTO || r.kernel > FDPP_KERNEL_SIMT)
            return fail(FDPP_ERR_INVALID_ARG, "table row %d: unknown kernel %d", i, r.kernel);
        if (r.units_per_sm < 1 || r.units_per_sm > 64)
            return fail(FDPP_ERR_INVALID_ARG, "table row %d: units_per_sm must be in [1, 64]", i);
        if (r.min_split < FDPP_AUTO_MIN_SPLIT || r.min_split > (1 << 20) || r.min_split % FDPP_AUTO_GRANULE)
            return fail(FDPP_ERR_INVALID_ARG,
                        "table row %d: min_split must be a multiple of %d in [%d, %d]", i,
                        FDPP_AUTO_GRANULE, FDPP_AUTO_MIN_SPLIT, 1 << 20);
    }
    std::lock_guard<std::mutex> lk(g_lut_mutex);
    g_lut.assign(rows, rows + n);
    return FDPP_OK;
}

fdpp_status fdpp_attn_auto_choice(const fdpp_params* p, int* kernel, int* units_per_sm, int* min_split)
{
    const fdpp_status st = check_params(p);
    if (st != FDPP_OK) return st;
    const AutoChoice c = auto_choice(*p);
    if (kernel) *kernel = c.kernel;
    if (units_per_sm) *units_per_sm = c.units;
    if (min_split) *min_split = c.min_split;
    return FDPP_OK;
}

int fdpp_max_splits(const fdpp_params* p)
{
    if (check_params(p) != FDPP_OK) return -1;
    return max_splits_of(*p);
}

fdpp_status fdpp_workspace_size(const fdpp_params* p, size_t* bytes)
{
    fdpp_status st = check_params(p);
    if (st != FDPP_OK) return st;
    if (!bytes) return fail(FDPP_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = layout_of(*p).total;
    return FDPP_OK;
}

fdpp_status fdpp_workspace_init(void* workspace, size_t workspace_bytes, fdpp_stream stream)
{
    if (!workspace) return fail(FDPP_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(workspace, 256)) return fail(FDPP_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(FDPP_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return FDPP_OK;
}

fdpp_status fdpp_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const fdpp_params* p, void* workspace, size_t workspace_bytes,
                             void* out, fdpp_stream stream)
{
    return fdpp_decode_attn_timed(q, k_cache, v_cache, block_table, seq_lens, p, workspace,
                                  workspace_bytes, out, stream, nullptr, nullptr);
}

fdpp_status fdpp_decode_attn_timed(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   const fdpp_params* p, void* workspace, size_t workspace_bytes,
                                   void* out, fdpp_stream stream, void* ev_split_begin,
                                   void* ev_split_end)
{
    fdpp_status st = check_params(p);
    if (st != FDPP_OK) return st;
    const bool paged = block_table != nullptr;
    if (paged && (st = check_paged(p)) != FDPP_OK) return st;
    if (!q || !k_cache || !v_cache || !seq_lens || !out)
        return fail(FDPP_ERR_INVALID_ARG, "q, k_cache, v_cache, seq_lens and out must be non-NULL");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return fail(FDPP_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (!aligned(seq_lens, 4) || (paged && !aligned(block_table, 4)))
        return fail(FDPP_ERR_INVALID_ARG, "seq_lens and block_table must be 4-byte aligned");
    if (!workspace) return fail(FDPP_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(workspace, 256)) return fail(FDPP_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    const WsLayout w = layout_of(*p);
    if (workspace_bytes < w.total)
        return fail(FDPP_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, w.total);

    const int G = p->num_q_heads / p->num_kv_heads;
    const int R = q_tokens_of(*p) * G;
    const bool tc_ok = p->dtype == FDPP_BF16 && R <= TC_MAX_ROWS;
    const int kernel = auto_choice(*p).kernel;
    if (kernel == FDPP_KERNEL_SIMT && R > SIMT_MAX_GROUP)
        return fail(FDPP_ERR_UNSUPPORTED, "SIMT kernel needs at most %d query rows per kv head (got %d)",
                    SIMT_MAX_GROUP, R);
    if (kernel == FDPP_KERNEL_TENSOR && !tc_ok)
        return fail(FDPP_ERR_UNSUPPORTED, "tensor kernel needs bf16 and at most %d query rows per kv head",
                    TC_MAX_ROWS);
    if (kernel == FDPP_KERNEL_TENSOR && p->tc_mma == FDPP_TC_MMA_TCGEN05 && !um_applies(*p))
        return fail(FDPP_ERR_UNSUPPORTED,
                    "tcgen05 build needs bf16, head_dim 128 and 9..%d query rows per kv head", TC_MAX_ROWS);
    if (kernel == FDPP_KERNEL_TENSOR && p->tc_mma == FDPP_TC_MMA_TCGEN05 && p->tc_ctas_per_sm > 1)
        return fail(FDPP_ERR_UNSUPPORTED, "tcgen05 build runs one CTA per SM");
    const bool um = kernel == FDPP_KERNEL_TENSOR && um_selected(*p);

    DeviceInfo dev;
    if ((st = device_info(dev)) != FDPP_OK) return st;

    KernelArgs a = kernel_args(*p, w, workspace, q, k_cache, v_cache, block_table, seq_lens, out,
                               dev.sms, kernel, um);

    const long long units_max = (long long)p->batch * p->num_kv_heads * w.max_splits;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    int split_grid = 0;
    if (ev_split_begin && (e = cudaEventRecord((cudaEvent_t)ev_split_begin, s)) != cudaSuccess)
        return fail(FDPP_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
    if (um) {
        // tcgen05 build: one CTA per SM with the deepest ring that fits (or the depth asked for),
        // but UM_SHORT_STAGES when every CTA streams few tiles (at most UM_SHORT_TILES, counted at
        // max_seq_len): at the start each CTA asks for its whole ring at once, and a shallower
        // ring lands its first tile sooner, which only short parts do not win back.
        const int budget = std::min(dev.smem_per_block, dev.smem_per_sm - 1024);
        const long long tiles_max = (long long)((p->max_seq_len + 63) / 64) * p->batch * p->num_kv_heads;
        const bool short_parts = tiles_max <= (long long)UM_SHORT_TILES * dev.sms;
        int ns = p->tc_stages > 0 ? p->tc_stages : (short_parts ? UM_SHORT_STAGES : 8);
        while (ns >= 2 && split_um_smem_bytes(R, ns, p->batch) > budget) --ns;
        if (ns < 2 || (p->tc_stages > 0 && ns != p->tc_stages))
            return fail(FDPP_ERR_UNSUPPORTED, "no tcgen05 geometry fits (stages %d)", p->tc_stages);
        a.nstage = ns;
        a.pf_tiles = p->tc_prefetch > 0 ? p->tc_prefetch : 0;
        CUtensorMap tk, tv, tq;
        if ((st = encode_kv_map(&tk, k_cache, *p, paged)) != FDPP_OK) return st;
        if ((st = encode_kv_map(&tv, v_cache, *p, paged)) != FDPP_OK) return st;
        if ((st = encode_q_map(&tq, q, *p)) != FDPP_OK) return st;
        long long grid = std::min<long long>(dev.sms, TC_UM_MAX_CTAS);
        if (p->batch > TC_PLAN_SMEM_MAX_B && grid > units_max) grid = units_max;
        split_grid = (int)grid;
        e = launch_split_um(a, tk, tv, tq, (int)grid, split_um_smem_bytes(R, ns, p->batch), s);
    } else if (kernel == FDPP_KERNEL_TENSOR) {
        const TcPlan plan = split_tc_plan(p->head_dim, R < TC_MAX_GROUP ? R : TC_MAX_GROUP, p->batch, p->tc_stages,
                                          p->tc_ctas_per_sm, dev.smem_per_sm, dev.smem_per_block);
        if (plan.nstage == 0)
            return fail(FDPP_ERR_UNSUPPORTED, "no tensor-kernel geometry fits (stages %d, CTAs/SM %d)",
                        p->tc_stages, p->tc_ctas_per_sm);
        a.nstage = plan.nstage;
        // L2 prefetch ahead of the ring measured slower on every workload here: off unless asked
        a.pf_tiles = p->tc_prefetch > 0 ? p->tc_prefetch : 0;
        CUtensorMap tk, tv;
        if ((st = encode_kv_map(&tk, k_cache, *p, paged)) != FDPP_OK) return st;
        if ((st = encode_kv_map(&tv, v_cache, *p, paged)) != FDPP_OK) return st;
        // persistent grid: every SM busy (SMs x resident CTAs). Batches whose plan fits in shared
        // memory are cut into equal parts of tiles, one per CTA (the kernel uses at most
        // TC_MAX_PARTS); larger ones are dealt out as whole units, no more CTAs than units.
        long long grid = (long long)dev.sms * plan.ctas_per_sm;
        if (grid > TC_MAX_PARTS) grid = TC_MAX_PARTS;
        const long long vunits = units_max * row_groups_of(*p);
        if (p->batch > TC_PLAN_SMEM_MAX_B && grid > vunits) grid = vunits;
        split_grid = (int)grid;
        e = launch_split_tc(a, tk, tv, (int)grid, plan.smem_bytes, plan.ctas_per_sm, s);
    } else {
        const int occ = split_simt_ctas_per_sm(a, p->dtype);
        long long grid = (long long)dev.sms * (occ > 0 ? occ : 1);
        if (grid > units_max) grid = units_max;
        split_grid = (int)grid;
        e = launch_split_simt(a, p->dtype, (int)grid, s);
    }
    if (e != cudaSuccess) return fail(FDPP_ERR_CUDA, "split kernel launch: %s", cudaGetErrorString(e));
    if (ev_split_end && (e = cudaEventRecord((cudaEvent_t)ev_split_end, s)) != cudaSuccess)
        return fail(FDPP_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
    e = launch_combine(a, p->dtype, split_grid, s);
    if (e != cudaSuccess) return fail(FDPP_ERR_CUDA, "combine kernel launch: %s", cudaGetErrorString(e));
    return FDPP_OK;
}

fdpp_status fdpp_score_ranges(const void* q, const void* k_cache, const int32_t* block_table,
                              const int32_t* seq_lens, const fdpp_params* p, void* workspace,
                              size_t workspace_bytes, float* smin_host, float* smax_host,
                              int32_t* nsplit_host, fdpp_stream stream)
{
    fdpp_status st = check_params(p);
    if (st != FDPP_OK) return st;
    if (q_tokens_of(*p) * (p->num_q_heads / p->num_kv_heads) > SIMT_MAX_GROUP)
        return fail(FDPP_ERR_UNSUPPORTED, "score ranges take at most %d query rows per kv head", SIMT_MAX_GROUP);
    const bool paged = block_table != nullptr;
    if (paged && (st = check_paged(p)) != FDPP_OK) return st;
    if (!q || !k_cache || !seq_lens || !smin_host || !smax_host)
        return fail(FDPP_ERR_INVALID_ARG, "q, k_cache, seq_lens, smin_host and smax_host must be non-NULL");
    if (!aligned(q, 16) || !aligned(k_cache, 16))
        return fail(FDPP_ERR_INVALID_ARG, "q and k_cache must be 16-byte aligned");
    if (!aligned(seq_lens, 4) || (paged && !aligned(block_table, 4)))
        return fail(FDPP_ERR_INVALID_ARG, "seq_lens and block_table must be 4-byte aligned");
    if (!workspace) return fail(FDPP_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(workspace, 256)) return fail(FDPP_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    const WsLayout w = layout_of(*p);
    if (workspace_bytes < w.total)
        return fail(FDPP_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, w.total);
    DeviceInfo dev;
    if ((st = device_info(dev)) != FDPP_OK) return st;

    KernelArgs a = kernel_args(*p, w, workspace, q, k_cache, nullptr, block_table, seq_lens, nullptr,
                               dev.sms, FDPP_KERNEL_SIMT);
    const long long units_max = (long long)p->batch * p->num_kv_heads * w.max_splits;
    const int occ = score_ranges_ctas_per_sm(a, p->dtype);
    long long grid = (long long)dev.sms * (occ > 0 ? occ : 1);
    if (grid > units_max) grid = units_max;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_score_ranges(a, p->dtype, (int)grid, s);
    if (e != cudaSuccess) return fail(FDPP_ERR_CUDA, "score range kernel launch: %s", cudaGetErrorString(e));
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess)
        return fail(FDPP_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));

    const size_t B = (size_t)p->batch, Tq = (size_t)q_tokens_of(*p), Hq = (size_t)p->num_q_heads,
                 ms = (size_t)w.max_splits, rows = B * Tq * Hq;
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    std::string nsb(B * 4, '\0');
    if ((e = cudaMemcpy(&nsb[0], ws + w.nsplit, nsb.size(), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(smin_host, ws + w.l_part, rows * ms * 4, cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(smax_host, ws + w.m_part, rows * ms * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail(FDPP_ERR_CUDA, "cudaMemcpy: %s", cudaGetErrorString(e));
    const int32_t* ns = reinterpret_cast<const int32_t*>(nsb.data());
    for (size_t r = 0; r < rows; ++r) {
        const size_t b = r / (Tq * Hq);
        const size_t n = ns[b] < 0 ? 0 : (ns[b] > (int)ms ? ms : (size_t)ns[b]);
        for (size_t j = 0; j < ms; ++j) {
            float& lo = smin_host[r * ms + j];
            float& hi = smax_host[r * ms + j];
            // past the sequence's splits, or a split holding none of this query row's keys
            if (j >= n || !std::isfinite(lo) || !std::isfinite(hi)) { lo = NAN; hi = NAN; }
        }
    }
    if (nsplit_host)
        for (size_t b = 0; b < B; ++b)
            for (size_t i = 0; i < Tq; ++i) nsplit_host[b * Tq + i] = ns[b];
    return FDPP_OK;
}

fdpp_status fdpp_pick_phi(const float* smin, const float* smax, const int32_t* nsplit, int batch,
                          int num_q_heads, int max_splits, float lo, float hi, float fallback,
                          float* phi_out, int32_t* kept_out)
{
    if (!smin || !smax || !nsplit || !phi_out)
        return fail(FDPP_ERR_INVALID_ARG, "smin, smax, nsplit and phi_out must be non-NULL");
    if (batch < 1 || num_q_heads < 1 || max_splits < 1)
        return fail(FDPP_ERR_INVALID_ARG, "batch, num_q_heads and max_splits must be >= 1");
    if (!std::isfinite(lo) || !std::isfinite(hi) || !(lo <= hi) || !std::isfinite(fallback))
        return fail(FDPP_ERR_INVALID_ARG, "lo <= hi and fallback must be finite");
    // Sweep per head. The kept count is constant on each distinct endpoint and on each open gap
    // between two consecutive ones: element 2i is endpoint x_i, element 2i+1 the gap after it. A
    // split's phi interval [a, b] covers elements 2 idx(a) .. 2 idx(b), counted with a difference
    // array. The best count's widest run of elements (ties: the first) gives phi (its middle).
    std::vector<double> a, b, x;
    std::vector<int> diff;
    for (int h = 0; h < num_q_heads; ++h) {
        a.clear();
        b.clear();
        for (int s = 0; s < batch; ++s) {
            const int n = nsplit[s] < 0 ? 0 : (nsplit[s] > max_splits ? max_splits : nsplit[s]);
            for (int j = 0; j < n; ++j) {
                const size_t r = ((size_t)s * num_q_heads + h) * (size_t)max_splits + j;
                const double lo_phi = (double)smax[r] - hi, hi_phi = (double)smin[r] - lo;
                if (std::isfinite(lo_phi) && std::isfinite(hi_phi) && lo_phi <= hi_phi) {
                    a.push_back(lo_phi);
                    b.push_back(hi_phi);
                }
            }
        }
        if (a.empty()) {
            phi_out[h] = fallback;
            if (kept_out) kept_out[h] = 0;
            continue;
        }
        x.assign(a.begin(), a.end());
        x.insert(x.end(), b.begin(), b.end());
        std::sort(x.begin(), x.end());
        x.erase(std::unique(x.begin(), x.end()), x.end());
        const size_t ne = 2 * x.size() - 1;
        diff.assign(ne + 1, 0);
        for (size_t i = 0; i < a.size(); ++i) {
            const size_t ia = std::lower_bound(x.begin(), x.end(), a[i]) - x.begin();
            const size_t ib = std::lower_bound(x.begin(), x.end(), b[i]) - x.begin();
            diff[2 * ia] += 1;
            diff[2 * ib + 1] -= 1;
        }
        int best = 0, run = 0;
        std::vector<int> cnt(ne);
        for (size_t e = 0; e < ne; ++e) {
            run += diff[e];
            cnt[e] = run;
            best = std::max(best, run);
        }
        double best_w = -1.0, best_mid = 0.0;
        for (size_t e = 0; e < ne;) {
            if (cnt[e] != best) { ++e; continue; }
            size_t f = e;
            while (f + 1 < ne && cnt[f + 1] == best) ++f;
            const double left = x[e / 2], right = x[(f + 1) / 2];
            if (right - left > best_w) { best_w = right - left; best_mid = 0.5 * (left + right); }
            e = f + 1;
        }
        phi_out[h] = (float)best_mid;
        if (kept_out) kept_out[h] = best;
    }
    return FDPP_OK;
}

fdpp_status fdpp_read_diag(const void* workspace, size_t workspace_bytes, const fdpp_params* p,
                           fdpp_diag* diag, uint8_t* flags_host, int32_t* nsplit_host)
{
    fdpp_status st = check_params(p);
    if (st != FDPP_OK) return st;
    if (!diag) return fail(FDPP_ERR_INVALID_ARG, "diag is NULL");
    if (!workspace) return fail(FDPP_ERR_WORKSPACE, "workspace is NULL");
    const WsLayout w = layout_of(*p);
    if (workspace_bytes < w.total)
        return fail(FDPP_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, w.total);
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    int32_t hdr[HDR_WORDS];
    cudaError_t e = cudaMemcpy(hdr, ws + w.header, sizeof hdr, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(FDPP_ERR_CUDA, "cudaMemcpy: %s", cudaGetErrorString(e));
    const size_t B = (size_t)p->batch, Tq = (size_t)q_tokens_of(*p), Hq = (size_t)p->num_q_heads,
                 ms = (size_t)w.max_splits;
    std::string nsb(B * 4, '\0');
    std::string flb(B * Tq * Hq * ms, '\0');
    if ((e = cudaMemcpy(&nsb[0], ws + w.nsplit, nsb.size(), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(&flb[0], ws + w.flags, flb.size(), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail(FDPP_ERR_CUDA, "cudaMemcpy: %s", cudaGetErrorString(e));
    const int32_t* ns = reinterpret_cast<const int32_t*>(nsb.data());
    const uint8_t* fl = reinterpret_cast<const uint8_t*>(flb.data());
    std::memset(diag, 0, sizeof *diag);
    diag->split_len = hdr[HDR_SPLIT];
    diag->max_splits = w.max_splits;
    diag->n_units = hdr[HDR_UNITS];
    diag->error_bits = (uint32_t)hdr[HDR_ERR];
    diag->kernel = hdr[HDR_KERNEL];
    diag->tc_build = hdr[HDR_KERNEL] == FDPP_KERNEL_TENSOR ? hdr[HDR_TC_BUILD] : 0;
    diag->tc_parts = hdr[HDR_KERNEL] == FDPP_KERNEL_TENSOR ? hdr[HDR_PARTS] : 0;
    diag->tc_seg_tiles = hdr[HDR_KERNEL] == FDPP_KERNEL_TENSOR && hdr[HDR_PARTS] > 0 ? hdr[HDR_SEGK] : 0;
    const size_t G = Hq / (size_t)p->num_kv_heads;
    for (size_t b = 0; b < B; ++b) {
        const int n = ns[b] < 0 ? 0 : (ns[b] > (int)ms ? (int)ms : ns[b]);
        for (int j = 0; j < n; ++j) {
            for (size_t g = 0; g < (size_t)p->num_kv_heads; ++g) {
                bool any = false;
                for (size_t i = 0; i < Tq; ++i)
                    for (size_t hh = 0; hh < G; ++hh) {
                        const uint8_t f = fl[(((b * Tq + i) * Hq) + g * G + hh) * ms + (size_t)j];
                        if (f & FDPP_FLAG_OUT) { ++diag->n_flagged_row_splits; any = true; }
                        if (f & FDPP_FLAG_RECOMPUTED) ++diag->n_recomputed_row_splits;
                    }
                if (any) ++diag->n_flagged_units;
            }
        }
    }
    if (flags_host) std::memcpy(flags_host, fl, flb.size());
    if (nsplit_host) std::memcpy(nsplit_host, ns, B * 4);
    return FDPP_OK;
}

}  // extern "C"
