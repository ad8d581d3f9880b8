// fdpp_internal.h -- types shared by the host API and the kernels of libfdpp (not installed).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fdpp.h"

namespace fdpp {

// Workspace header words (int32 each).
enum {
    HDR_SPLIT = 0,      // S used by the last call
    HDR_UNITS = 1,      // (b, g, j) units of the last call
    HDR_KERNEL = 2,     // fdpp_kernel that ran
    HDR_ERR = 3,        // sticky FDPP_ERRBIT_* (atomicOr)
    HDR_BATCH = 4,      // B of the last call
    HDR_MAXSPLITS = 5,  // partial slots per row
    HDR_REDO_LISTS = 16, // fallback lists: words 16 + 2i / 17 + 2i = entries pushed to / claimed
                         //   from list i (read together as one 8-byte word), i < REDO_NLISTS;
                         //   zeroed by the combine kernel
    HDR_PARTS = 11,     // tensor kernel: parts P of the tile-balanced partition (0: none)
    HDR_TILES = 12,     // tensor kernel: 64-token tiles T of all units together, with phantoms
    HDR_TC_BUILD = 13,  // tensor kernel build that ran: 1 mma.sync, 2 tcgen05 (split_um.cu)
    HDR_SEGK = 14,      // tensor kernel: phantom tiles between units in the partition (HDR_TILES
                        //   counts them)
    HDR_WORDS = 64
};

// Byte offsets of the workspace regions (each 256-byte aligned).
struct WsLayout {
    size_t header, nsplit, tstart, redo, hint, flags, m_part, l_part, o_part, xf, xm, xl, xo, total;
    int max_splits;
};

// The tensor kernel cuts the tiles of all units into at most this many equal parts, one per
// CTA. A part's share of one (row group, sequence, kv head) is a run, which leaves one partial
// in its run slot c + u (u: that head's index in tile order), which the combine adds in.
constexpr int TC_MAX_PARTS = FDPP_TC_MAX_PARTS;
// Batches up to this size keep their split plan in the tensor kernel's shared memory (and are
// cut into parts); larger batches are dealt out to the CTAs as whole units.
constexpr int TC_PLAN_SMEM_MAX_B = 1024;
// Fallback list entry: 4 x int64 = {(b + 1) | (g * max_splits + j) << 32,
// t0 | t1 << 32 (token range of the segment), dest (-1: split slot j, else run slot), the
// segment's rows whose scores left the window (one bit per row of its row group)}.
constexpr int REDO_WORDS = 4;
// The fallback list is this many lists (CTA c pushes to list c % REDO_NLISTS), each with room for
// every entry of a call.
constexpr int REDO_NLISTS = 8;
// A claimed fallback entry that spans several splits is cut into one entry per split, shared
// by the free CTAs, while fewer than this many entries wait to be claimed.
constexpr int REDO_SPLIT_BELOW = 64;
// Start-up hint of the tensor kernel (contiguous caches): per CTA, the TMA coordinates (x, y, z)
// of the first HINT_TILES tiles it streamed in the last call, after a count; prefetched into L2
// before the kernel waits for the previous one. HINT_WORDS int32 per CTA.
constexpr int HINT_TILES = 5;
constexpr int HINT_WORDS = 16;

// Everything a kernel of this library needs about one call. Plain pointers and sizes.
struct KernelArgs {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* block_table;   // nullptr: contiguous cache
    const int32_t* seq_lens;
    void* out;
    int32_t* hdr;
    int32_t* nsplit;              // [B], written by CTA 0 of the split kernel
    int32_t* tstart;              // [B + 1] tile prefix of the sequences (tensor kernel, CTA 0)
    long long* redo;              // fallback lists, REDO_WORDS per entry (tensor kernel)
    int32_t* hint;                // [TC_MAX_PARTS][HINT_WORDS] start-up hint (tensor kernel)
    int redo_cap;                 // entries per fallback list
    uint8_t* flags;               // [B][Tq][Hq][max_splits]
    float* m_part;                // [B][Tq][Hq][max_splits]
    float* l_part;                // [B][Tq][Hq][max_splits]
    float* o_part;                // [B][Tq][Hq][max_splits][D]
    uint8_t* xf;                  // run slots [TC_MAX_PARTS + B Hkv NRG][min(R, 8)]: edge flags,
    float* xm;                    //   m,
    float* xl;                    //   l,
    float* xo;                    //   o [..][min(R, 8)][D]
    int B, Hq, Hkv, G, D;
    int Tq;                       // query tokens per sequence (the last Tq positions, causal)
    int R;                        // query rows per kv head and sequence: Tq * G
    int max_seq_len, block_size, max_blocks, num_blocks;
    int split_req, max_splits, num_sms;
    float scale, phi, lo, hi;
    const float* phi_heads;       // [Hq] per-head unified max, or nullptr (phi for every head)
    int mode;
    int kernel_id;
    int nstage;                   // tensor kernel: TMA ring depth
    int pf_tiles;                 // tensor kernel: L2 prefetch distance in tiles (0 = off)
    // Tensor kernel: the R rows of a kv head are cut into NRG groups of up to Rg = min(R, 8)
    // rows; each (kv head, group) is a virtual head of the plan, Hv = Hkv * NRG of them. (Kept
    // last: fields added in the middle move the others' parameter offsets and change the
    // kernels' code.)
    int NRG, Rg, Hv;
    // split_len == 0: the split scheduler's units per SM and least split length (dataflow table)
    int auto_units, auto_min;
    // Tensor kernel partition: phantom tiles counted between consecutive units (row group,
    // sequence, kv head) of the tile order, the time a run boundary inside a part costs (0: none)
    int seg_tiles;
};

// Query rows per kv head (R = Tq * G): the tensor kernel takes 8 rows per unit (the columns of one
// m16n8k16 tile) and up to TC_MAX_ROWS in groups of 8; the SIMT kernel holds 16 register rows.
constexpr int TC_MAX_GROUP = 8;
// Window decisions of split pieces in flight in one CTA of the tensor kernel (a power of two
// above the deepest TMA ring: no consumer warp runs more pieces ahead of another).
constexpr int TC_FSLOTS = 16;
constexpr int TC_MAX_ROWS = 64;
constexpr int SIMT_MAX_GROUP = 16;

// Launchers (each returns the launch status). `grid` is the persistent CTA count. Either split
// kernel is followed by launch_combine (a programmatic dependent launch).
cudaError_t launch_split_simt(const KernelArgs& a, int dtype, int grid, cudaStream_t s);
cudaError_t launch_split_tc(const KernelArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, int smem_bytes, int ctas_per_sm, cudaStream_t s);
// split_grid: CTAs of the split kernel before it (bounds the tensor kernel's runs per row).
cudaError_t launch_combine(const KernelArgs& a, int dtype, int split_grid, cudaStream_t s);
// Score range of every row-split (least into l_part, greatest into m_part) and the split plan.
cudaError_t launch_score_ranges(const KernelArgs& a, int dtype, int grid, cudaStream_t s);
int score_ranges_ctas_per_sm(const KernelArgs& a, int dtype);

// The current device's SM count and shared-memory limits (sm_103a checked; cached per device).
fdpp_status query_device(int* sms, int* smem_per_sm, int* smem_per_block);
// The driver's cuTensorMapEncodeTiled (looked up once).
fdpp_status get_tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn);

// Bytes at the front of a workspace for `p` that must be zero when a call starts.
size_t workspace_zero_prefix(const fdpp_params& p);
// Offset of the start-up hint region (the zero prefix minus the hint, which may stay stale).
size_t workspace_hint_offset(const fdpp_params& p);
// Sets the reason fdpp_last_error() reports on this thread.
void set_last_error(const char* what);

// Resident CTAs per SM of the SIMT split kernel for this shape (0 if it cannot launch).
int split_simt_ctas_per_sm(const KernelArgs& a, int dtype);

// Tensor-core kernel geometry for one call: ring depth, CTAs per SM and dynamic shared memory.
struct TcPlan {
    int nstage;
    int ctas_per_sm;
    int smem_bytes;
};
// Chooses the geometry (requested values when > 0) from the per-SM and per-block shared
// memory limits of the device. nstage == 0 in the result means no geometry fits.
TcPlan split_tc_plan(int head_dim, int group, int batch, int req_stages, int req_ctas,
                     int smem_per_sm, int smem_per_block);
// Tokens per TMA tile of the tensor-core kernel (box height of the contiguous tensor maps).
constexpr int TC_TILE_TOKENS = 64;

// tcgen05 build of the tensor kernel (split_um.cu): bf16, d = 128, more than 8 and at most
// TC_MAX_ROWS query rows per kv head, all of them in one unit; one CTA per SM, at most
// TC_UM_MAX_CTAS CTAs (so at most that many parts), rows padded to split_um_rows_padded(R).
constexpr int TC_UM_MAX_CTAS = FDPP_TC_UM_MAX_CTAS;
int split_um_rows_padded(int R);
// Dynamic shared memory of one CTA with an `nstage`-deep ring (alignment slack included).
int split_um_smem_bytes(int R, int nstage, int batch);
// tq: the query tensor map ({d, Hq, Tq, B} bf16, box {64, G, Tq, 1}, 128-byte swizzle).
cudaError_t launch_split_um(const KernelArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tq, int grid, int smem_bytes, cudaStream_t s);

}  // namespace fdpp
