/*
 * fdpp.h -- C ABI of libfdpp: unified-max split-KV decode attention for GB300 (sm_103a).
 *
 * The operation. In the decode step, one query token per sequence attends to that sequence's
 * K/V cache, which keeps growing (opt.ai.kr "FlashDecoding++ async softmax -- theory",
 * section 1). For sequence b, query head h and kv head g = floor(h / G), G = Hq / Hkv:
 *
 *     s_t   = scale * <q[b,h,:], k[b,t,g,:]>                      for t < L_b = seq_lens[b]
 *     out   = sum_t exp(s_t - mu) v[b,t,g,:] / sum_t exp(s_t - mu),  mu any finite shift
 *
 * How it is computed (same page, section 3). The cache of each sequence is cut into splits of
 * S tokens. Every split works alone against a unified max phi fixed in advance: it forms
 * o_j = sum exp(s_t - phi) v_t and l_j = sum exp(s_t - phi), with no communication between
 * splits. A split in which some score leaves the safe window, i.e. NOT (lo <= s_t - phi <= hi),
 * gets the ordinary online softmax's partial (running max m_j): the tensor kernel's mma.sync build
 * continues it with the running max from the first tile holding such a score (the tiles before
 * were inside the window, so their phi-frame sums stand), its tcgen05 build and the SIMT kernel
 * compute it again. The final combine is
 * out = sum_j exp(m_j - M) o_j / sum_j exp(m_j - M) l_j with M = max_j m_j, which is the plain
 * sum of the page whenever no split fell back (every m_j = phi).
 *
 * Conventions for every call below:
 *   - Pointers marked DEVICE are device memory owned by the caller. The library allocates and
 *     frees nothing, keeps no pointer after a call returns, and writes only `out` and the
 *     caller's workspace.
 *   - Calls that take a stream only enqueue work on it (no host synchronisation) and return
 *     before the GPU runs it. Two calls that share one workspace must not overlap on the GPU.
 *   - Argument errors are reported synchronously, before anything is enqueued, as a status code;
 *     fdpp_last_error() then gives a one-line reason (thread-local). A CUDA launch error returns
 *     FDPP_ERR_CUDA. Problems found on the device (a seq_len out of range, a bad block table
 *     entry, a pipeline wait that ran out) never trap: they set sticky bits read by
 *     fdpp_read_diag().
 *   - Every kernel is bounded: each wait gives up after about two seconds, sets
 *     FDPP_ERRBIT_TIMEOUT and lets the launch finish.
 */
#ifndef FDPP_H
#define FDPP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* fdpp_stream;

typedef enum {
    FDPP_OK = 0,
    FDPP_ERR_INVALID_ARG = 1,   /* a pointer, size or parameter violates the contract */
    FDPP_ERR_UNSUPPORTED = 2,   /* valid, but no kernel here handles it (e.g. head_dim 96) */
    FDPP_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or smaller than required */
    FDPP_ERR_CUDA = 4           /* a CUDA runtime call or a launch failed */
} fdpp_status;

typedef enum { FDPP_F32 = 0, FDPP_BF16 = 1 } fdpp_dtype;

typedef enum {
    FDPP_MODE_NORMAL = 0,        /* phi frame, fallback recompute of out-of-window splits */
    FDPP_MODE_FORCE_FAST = 1,    /* phi frame, never recompute (negative control: results of
                                    flagged splits may be inf/NaN) */
    FDPP_MODE_FORCE_ONLINE = 2   /* every split with the ordinary online softmax (the
                                    running-max baseline the unified max replaces) */
} fdpp_mode;

typedef enum {
    FDPP_KERNEL_AUTO = 0,        /* tensor-core kernel when it applies, else the SIMT kernel */
    FDPP_KERNEL_TENSOR = 1,      /* TMA-fed kernel, q.K^T and P.V on tensor cores: bf16,
                                    head_dim 64/128, G <= 8 */
    FDPP_KERNEL_SIMT = 2         /* CUDA-core kernel with warp-shuffle reductions: f32 or bf16,
                                    head_dim 64/128, G <= 16 */
} fdpp_kernel;

/* Flag byte per (b, h, j), readable through fdpp_read_diag. */
enum {
    FDPP_FLAG_OUT = 1,           /* some score of the split left the window */
    FDPP_FLAG_ABOVE = 2,         /* ... above phi + hi (the overflow side) */
    FDPP_FLAG_BELOW = 4,         /* ... below phi + lo */
    FDPP_FLAG_NAN = 8,           /* ... was NaN */
    FDPP_FLAG_RECOMPUTED = 16,   /* the partial of this row-split came from online softmax */
    FDPP_FLAG_SLOT = 32          /* tensor kernel (tcgen05 build): this row-split's own partial
                                    slot holds a recomputed piece (its run's phi-frame partial
                                    left it out) */
};

/* Sticky device error bits (cleared by fdpp_workspace_init). */
enum {
    FDPP_ERRBIT_SEQ_LEN = 1,     /* a seq_lens entry was < 0 or > max_seq_len (clamped) */
    FDPP_ERRBIT_BLOCK_TABLE = 2, /* a block table entry of a valid token was outside the pool
                                    (that block was not read; its row is wrong) */
    FDPP_ERRBIT_TIMEOUT = 4      /* a pipeline wait ran out; results of that call are invalid */
};

typedef struct fdpp_params {
    int batch;               /* B >= 1 sequences, one query token each */
    int num_q_heads;         /* Hq >= 1 */
    int num_kv_heads;        /* Hkv >= 1, Hq % Hkv == 0 */
    int head_dim;            /* d: 64 or 128 */
    int dtype;               /* fdpp_dtype of q, k_cache, v_cache and out */
    int max_seq_len;         /* contiguous cache: its token dimension Lmax. Paged cache: an
                                upper bound on every seq_len, <= max_blocks_per_seq*block_size.
                                Sizes the workspace. */
    int block_size;          /* paged only: tokens per block, a power of two in [16, 256] */
    int max_blocks_per_seq;  /* paged only: row length of block_table */
    int num_kv_blocks;       /* paged only: number of blocks in the K (and V) pool */
    float scale;             /* score scale, positive and finite, usually 1/sqrt(d) */
    float phi;               /* unified max, in units of the scaled score s */
    float lo, hi;            /* safe window: a score is inside iff lo <= s - phi <= hi */
    int split_len;           /* S > 0: tokens per split (paged: a multiple of block_size).
                                0: chosen per call from sum_b L_b, Hkv and the SM count */
    int mode;                /* fdpp_mode */
    int kernel;              /* fdpp_kernel */
    int tc_stages;           /* tensor kernel: depth of the TMA ring (2..12), 0 = automatic */
    int tc_ctas_per_sm;      /* tensor kernel: resident CTAs per SM (1 or 2), 0 = automatic */
    int tc_prefetch;         /* tensor kernel: L2 prefetch distance in 64-token tiles ahead of the
                                TMA ring (1..32); 0 = automatic (off), -1 = off */
    const float* phi_heads;  /* DEVICE float32 [Hq], 4-byte aligned: the unified max of each query
                                head (e.g. from fdpp_pick_phi), used in place of `phi`; NULL = the
                                scalar `phi` for every head */
    int q_tokens;            /* Tq query tokens per sequence (0 or 1: one, the decode step): the
                                sequence's last Tq positions, whose keys are already in the cache,
                                so query token i sees the keys t < L_b - Tq + 1 + i (a short
                                prefill chunk or a speculative-decoding step). q and out are then
                                [B][Tq][Hq][d]. Query rows per kv head, R = Tq * Hq / Hkv: at
                                most 64 for the tensor kernel, at most 16 for the SIMT kernel and
                                for fdpp_score_ranges; more is FDPP_ERR_UNSUPPORTED. */
    int tc_mma;              /* tensor kernel with more than 8 query rows per kv head (fdpp_tc_mma):
                                which build takes them */
} fdpp_params;

/* Builds of the tensor kernel for more than 8 query rows per kv head. */
typedef enum fdpp_tc_mma {
    FDPP_TC_MMA_AUTO = 0,        /* TCGEN05 where it applies (bf16, d = 128, tc_ctas_per_sm 0 or
                                    1), else MMA_SYNC */
    FDPP_TC_MMA_SYNC = 1,        /* mma.sync m16n8k16: the rows in groups of 8, each group a unit
                                    that streams the kv head's K/V (the groups' reads of a tile
                                    mostly meet in L2); two CTAs per SM */
    FDPP_TC_MMA_TCGEN05 = 2      /* tcgen05 tensor cores, accumulators in tensor memory: all R
                                    rows in one unit, K/V streamed once; one CTA per SM; bf16 and
                                    d = 128 only (else FDPP_ERR_UNSUPPORTED) */
} fdpp_tc_mma;

/* Split length chosen by split_len == 0: spread sum_b L_b * Hkv over units_per_sm * num_sms
 * units, round up to a multiple of FDPP_AUTO_GRANULE (or of block_size when larger), clamp to
 * [min_split, max_seq_len rounded up]. units_per_sm and min_split come from the dataflow table
 * (fdpp_attn_set_lut) for the call's shape, else FDPP_AUTO_UNITS_PER_SM and FDPP_AUTO_MIN_SPLIT. */
#define FDPP_AUTO_UNITS_PER_SM 4
#define FDPP_AUTO_GRANULE 64
#define FDPP_AUTO_MIN_SPLIT 256

/* One row of the heuristic dataflow table for decode attention (opt.ai.kr "FlashDecoding++
 * async softmax -- theory", sections 2(3) and 4: the configuration is taken per shape range
 * from a table measured offline, instead of one static choice for every shape). A call uses the
 * first row whose ranges hold its shape: batch <= max_batch, max_seq_len <= max_seq_len and
 * rows per kv head (q_tokens * Hq / Hkv) <= max_rows. */
typedef struct fdpp_attn_lut_row {
    int max_batch;           /* >= 1 */
    int max_seq_len;         /* >= 1 */
    int max_rows;            /* >= 1 */
    int kernel;              /* fdpp_kernel for calls with kernel == FDPP_KERNEL_AUTO; AUTO keeps
                                the default rule, and a kernel that cannot take the call too */
    int units_per_sm;        /* split_len == 0: units per SM the split length aims at, in [1, 64] */
    int min_split;           /* split_len == 0: least split length, a multiple of
                                FDPP_AUTO_GRANULE in [FDPP_AUTO_MIN_SPLIT, 1 << 20] */
} fdpp_attn_lut_row;

typedef struct fdpp_diag {
    int32_t split_len;            /* S used by the last call on this workspace */
    int32_t max_splits;           /* partial slots per (b, h) in this workspace */
    int64_t n_units;              /* (b, g, j) units of the last call */
    int64_t n_flagged_row_splits; /* (b, h, j) with FDPP_FLAG_OUT */
    int64_t n_flagged_units;      /* (b, g, j) with at least one flagged head */
    int64_t n_recomputed_row_splits; /* (b, h, j) with FDPP_FLAG_RECOMPUTED */
    uint32_t error_bits;          /* FDPP_ERRBIT_* since the last fdpp_workspace_init */
    int32_t kernel;               /* fdpp_kernel that ran last (1 tensor, 2 SIMT) */
    int32_t tc_build;             /* tensor kernel: the build that ran (FDPP_TC_MMA_SYNC, or
                                     FDPP_TC_MMA_TCGEN05); 0 for the SIMT kernel */
    int32_t tc_parts;             /* tensor kernel: parts P its tiles were cut into (one per CTA;
                                     0: whole units, no run slots); 0 for the SIMT kernel */
    int32_t tc_seg_tiles;         /* tensor kernel: phantom tiles counted after each (sequence,
                                     kv head) unit in that cut (a part holding a run boundary
                                     takes that many tiles fewer); 0 for the SIMT kernel */
} fdpp_diag;

/* Partial slots per (b, h) that a workspace for `p` holds: ceil(max_seq_len / S) for a fixed
 * S, ceil(max_seq_len / FDPP_AUTO_MIN_SPLIT) for S == 0. Returns -1 on invalid params. */
int fdpp_max_splits(const fdpp_params* p);

/* The tensor kernel cuts the 64-token tiles of all (b, g, j) units into at most this many
 * equal parts, one per CTA, so that every CTA streams about the same number of bytes. A part's
 * share of one sequence's kv head is a run, which leaves one partial (in the phi frame, summed
 * across its splits) in a run slot of the workspace; window decisions stay per split. The
 * tcgen05 build cuts a stream that counts a few phantom tiles after each (sequence, kv head), so
 * that a part holding a run boundary, which costs time, takes fewer real tiles (fdpp_diag's
 * tc_seg_tiles). */
#define FDPP_TC_MAX_PARTS 512

/* The tensor kernel's tcgen05 build (more than 8 query rows per kv head, bf16, d = 128) runs at
 * most this many CTAs, one per SM, so at most this many parts; its run slots hold all R rows of a
 * kv head. */
#define FDPP_TC_UM_MAX_CTAS 256

/* Bytes of device workspace fdpp_decode_attn needs for `p` (written to *bytes). The workspace
 * holds the split plan, the per-split partials (o: fp32 [B][Tq][Hq][max_splits][d]; l, m: fp32
 * [B][Tq][Hq][max_splits]), the flag bytes [B][Tq][Hq][max_splits], the tensor kernel's run
 * slots (FDPP_TC_MAX_PARTS + B * Hkv * ceil(Tq * Hq / Hkv / 8) of them, min(Tq * Hq / Hkv, 8)
 * rows each: o, l, m and edge flags, like a split's; a run is one CTA's share of one sequence's
 * kv head, across split boundaries), the fallback lists and a small header. */
fdpp_status fdpp_workspace_size(const fdpp_params* p, size_t* bytes);

/* Zeroes a workspace (stream-ordered). Call once after allocating it; it also clears the
 * sticky error bits. workspace: DEVICE, 256-byte aligned. */
fdpp_status fdpp_workspace_init(void* workspace, size_t workspace_bytes, fdpp_stream stream);

/* One decode-attention step for B sequences (enqueued on `stream`).
 *   q           DEVICE [B][Tq][Hq][d] of dtype, 16-byte aligned (Tq = q_tokens, 1 by default).
 *   k_cache,    DEVICE, 16-byte aligned, dtype. Contiguous (block_table == NULL):
 *   v_cache       [B][max_seq_len][Hkv][d]. Paged: pools [num_kv_blocks][block_size][Hkv][d];
 *                 token t of sequence b is slot t % block_size of block
 *                 block_table[b][t / block_size].
 *   block_table DEVICE int32 [B][max_blocks_per_seq] or NULL (contiguous cache).
 *   seq_lens    DEVICE int32 [B]: L_b, 0 <= L_b <= max_seq_len. L_b == 0 gives a zero row.
 *   workspace   DEVICE, 256-byte aligned, >= fdpp_workspace_size bytes, zeroed once by
 *               fdpp_workspace_init. Not shared by overlapping calls.
 *   out         DEVICE [B][Tq][Hq][d] of dtype (rounded to nearest even from fp32). A query token
 *               that sees no key (L_b < Tq) gives a zero row.
 * Tokens t >= L_b are never part of a score, a window test or a sum (they may hold anything,
 * NaN included). */
fdpp_status fdpp_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const fdpp_params* p, void* workspace, size_t workspace_bytes,
                             void* out, fdpp_stream stream);

/* fdpp_decode_attn, and also records two caller-owned CUDA events (cudaEvent_t, either may be
 * NULL) on `stream`: ev_split_begin right before the split kernel (steps: split plan, phi-frame
 * partials, window test, recompute) and ev_split_end right after it, before the combine kernel.
 * Lets a caller time the dominant kernel alone; results are identical to fdpp_decode_attn. */
fdpp_status fdpp_decode_attn_timed(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   const fdpp_params* p, void* workspace, size_t workspace_bytes,
                                   void* out, fdpp_stream stream, void* ev_split_begin,
                                   void* ev_split_end);

/* Size in bytes of the device array behind fdpp_decode_attn_noalloc (16 MiB per GPU). */
#define FDPP_NOALLOC_WORKSPACE_BYTES (16u << 20)

/* fdpp_decode_attn for callers that cannot allocate device memory: a plugin inside a runtime
 * that owns every device allocation and offers no allocator, or a serving loop whose memory is
 * fixed at start-up and may not call cudaMalloc (or any allocating library) afterwards. The
 * pages have no counterpart to this entry point; it is a deployment convenience.
 * It needs no workspace: its scratch is one library-owned device array of
 * FDPP_NOALLOC_WORKSPACE_BYTES that every GPU loading the library keeps until the process
 * exits. It allocates nothing and frees nothing. Arguments are those of fdpp_decode_attn.
 *   - Problems whose fdpp_workspace_size exceeds FDPP_NOALLOC_WORKSPACE_BYTES are rejected
 *     with FDPP_ERR_WORKSPACE before anything is enqueued (fdpp_last_error() says by how much).
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress, on the host). The first call on a device also loads the array
 *     there, so make that first call before any stream capture on that device.
 *   - Each call clears, on `stream`, the array's header, split plan and fallback lists, then
 *     runs the same kernels as fdpp_decode_attn on the same inputs, with the same results bit
 *     for bit. All calls share the array and it keeps the last call's contents: calls that
 *     overlap on the GPU (unordered streams or threads) race on it and produce wrong results.
 *     Calls ordered on one stream are safe, whatever shapes they have.
 *   - What the last call found on the device (error bits, fallback flags, the split plan) is
 *     read with fdpp_read_diag_noalloc, after that call's stream has been synchronised; the
 *     error bits there are that call's alone, not sticky across calls. */
fdpp_status fdpp_decode_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     const fdpp_params* p, void* out, fdpp_stream stream);

/* fdpp_read_diag for the array behind fdpp_decode_attn_noalloc on the current device: what the
 * last no-alloc call with parameters `p` left there (synchronous device-to-host copies; call after
 * that call's stream has been synchronised). Arguments and results as for fdpp_read_diag.
 * Problems beyond FDPP_NOALLOC_WORKSPACE_BYTES are rejected with FDPP_ERR_WORKSPACE. This reader
 * has no counterpart in the pages either; it exists so that a caller of the no-alloc step can see
 * device-side problems (FDPP_ERRBIT_*) and the fallback decisions, as a workspace caller can. */
fdpp_status fdpp_read_diag_noalloc(const fdpp_params* p, fdpp_diag* diag, uint8_t* flags_host,
                                   int32_t* nsplit_host);

/* Installs the dataflow table (copied; process-wide, for every device; n == 0 removes it, and
 * the defaults apply again). Host only, no CUDA call. FDPP_ERR_INVALID_ARG for a row outside the
 * ranges documented in fdpp_attn_lut_row (the table is then left as it was). */
fdpp_status fdpp_attn_set_lut(const fdpp_attn_lut_row* rows, int n);

/* What a call with `p` would use (host only, no CUDA call): the kernel (FDPP_KERNEL_TENSOR or
 * FDPP_KERNEL_SIMT, after the table and the default rule), and the units_per_sm and min_split of
 * the split scheduler (used when p->split_len == 0). Any output pointer may be NULL. */
fdpp_status fdpp_attn_auto_choice(const fdpp_params* p, int* kernel, int* units_per_sm,
                                  int* min_split);

/* Score range of every row-split, for choosing phi in advance (opt.ai.kr "FlashDecoding++ async
 * softmax -- theory", section 3: phi is set by observing the score distribution beforehand).
 * On sample inputs laid out as for fdpp_decode_attn (q, k_cache, block_table, seq_lens, p,
 * workspace), writes for each query row (b, i), head h and split j < nsplit[b] the least and
 * greatest scaled score s = scale <q, k_t> over the split's tokens that row sees:
 *   smin_host, smax_host  HOST float [B][Tq][Hq][max_splits] (NaN past a sequence's splits, and
 *                         for a split that holds none of the row's keys);
 *   nsplit_host           HOST int32 [B][Tq] (each query row's split count, its sequence's) or
 *                         NULL.
 * V is not read. Enqueues one kernel on `stream` and waits for it (synchronous). Uses the
 * workspace's partial arrays; phi, lo, hi, mode and kernel in p are ignored. */
fdpp_status fdpp_score_ranges(const void* q, const void* k_cache, const int32_t* block_table,
                              const int32_t* seq_lens, const fdpp_params* p, void* workspace,
                              size_t workspace_bytes, float* smin_host, float* smax_host,
                              int32_t* nsplit_host, fdpp_stream stream);

/* Per-head unified max from score ranges (host only, no CUDA call). A row-split stays on the
 * fast path for phi iff lo <= s - phi <= hi for all its scores, i.e. iff phi lies in
 * [smax - hi, smin - lo]. For each head h, phi_out[h] is a value inside the most such intervals
 * of the row-splits j < nsplit[b] over all sequences b; of all values that reach that count, the
 * middle of the widest closed run of them. A head with no split that any phi keeps gets
 * `fallback`. smin, smax: HOST float [batch][Hq][max_splits] as written by fdpp_score_ranges
 * (batch = B * Tq query rows); nsplit: HOST int32 [batch]; phi_out: HOST float [Hq];
 * kept_out: HOST int32 [Hq] (the row-splits each phi_out keeps) or NULL. */
fdpp_status fdpp_pick_phi(const float* smin, const float* smax, const int32_t* nsplit, int batch,
                          int num_q_heads, int max_splits, float lo, float hi, float fallback,
                          float* phi_out, int32_t* kept_out);

/* Reads what the last call left in `workspace` (synchronous device-to-host copies; call after
 * that call's stream has been synchronised). diag: HOST, required. flags_host: HOST uint8
 * [B][Tq][Hq][max_splits] or NULL. nsplit_host: HOST int32 [B] (splits per sequence) or NULL.
 * Entries with j >= nsplit[b] are stale. */
fdpp_status fdpp_read_diag(const void* workspace, size_t workspace_bytes, const fdpp_params* p,
                           fdpp_diag* diag, uint8_t* flags_host, int32_t* nsplit_host);

/* Static name of a status code. */
const char* fdpp_status_str(fdpp_status s);

/* Reason for the last non-OK status returned on this thread ("" if none). */
const char* fdpp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FDPP_H */
