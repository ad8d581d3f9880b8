// split_tc.cu -- per-split kernel for bf16 K/V: TMA-fed ring, tensor-core q.K^T and P.V, and the
// fallback recompute, in one persistent launch; combine.cu then sums the split partials.
//
// What it computes (opt.ai.kr "FlashDecoding++ async softmax -- theory", s1 and s3). For one unit
// (sequence b, kv head g, split j) and the G query heads that share kv head g:
//     s_t = scale <q_h, k_t>, p_t = exp(s_t - phi), l = sum p_t, o = sum p_t v_t    (fast pass)
// against the unified max phi, with no communication between splits; every score is tested
// against lo <= s - phi <= hi. A segment (see below) with a head outside the window goes on a
// device-wide list and is streamed again with the ordinary online softmax (running max) by
// whichever CTA is free first; its flagged heads' partials are replaced by ones in their own
// max frame.
//
// How. One CTA = 1 producer warp + 4 consumer warps, persistent over an equal share of tiles.
//   work      the 64-token tiles of all units, in unit order (b, g, j), are cut into P equal
//             parts, one per CTA, so every CTA streams the same bytes whatever the unit count
//             (whole units dealt round-robin would leave a last wave of few CTAs). A part is a
//             run of segments, each the part's share of one (sequence, kv head): a segment may
//             span several splits and begin or end inside one. Its phi-frame sums run across
//             the splits into one partial (a run slot, which combine.cu adds in), while the
//             window decisions are taken split by split.
//   producer  plans the splits in shared memory (prefixes of n_b = ceil(L_b / S) and of the
//             tiles per sequence), then for each segment writes a small header into a Q-ring
//             slot and bulk-copies the unit's G query rows there (this slot is also how
//             consumers learn which segment comes next), and
//             streams 64-token K and V tiles of head g with 3-D TMA loads (128-byte swizzle)
//             into a ring of `nstage` stages (mbarriers: full = bytes landed, empty = the four
//             consumer warps released the stage). A paged cache is read one block per box,
//             block-table entries fetched 32 at a time by the warp. After its own part it
//             claims fallback segments from the list until it is empty, then sends a sentinel.
//   consumers each own 16 tokens of a tile and compute it transposed (tokens on M, heads on N):
//             S^T = K Q^T            mma.m16n8k16 bf16 -> fp32, columns = the G heads, so each
//                                    K byte read from HBM feeds all G heads once;
//             P = exp(S - phi), window test;
//             O^T += V^T P^T         P carried as bf16 hi + lo parts (~16 mantissa bits).
//             The four warps merge their fp32 partials through shared memory of their own, as a
//             tree (w0 + w2) + (w1 + w3) (a plain sum in the phi frame), and warp 0 writes o, l,
//             m and the flag byte of each query row; every stage goes back to the producer as
//             soon as its tile is read.
// When a CTA starts its last own segment it allows the dependent combine launch to begin
// (programmatic dependent launch), so that launch overlaps the tail of this one. This kernel is
// a programmatic dependent too: before it waits for the previous kernel, each CTA prefetches
// into L2 the tiles it streamed first in the previous call (a hint kept in the workspace).
// Several query tokens per sequence (MQ builds): R = Tq G query rows per kv head, each with its
// causal key limit. More than 8 rows (RG builds, a prefill chunk): the rows are cut into groups
// of 8, each (kv head, group) a virtual head with its own units, and the tiles are ordered
// group-major so that the groups' reads of one K/V tile fall at about the same time and all but
// the first hit L2. The one-group builds compile exactly as without row groups.
// Every wait is bounded; a wait that runs out sets FDPP_ERRBIT_TIMEOUT and the CTA stops.
// (A fused last-arriver combine was measured here and removed: under full HBM load its
// latency-bound reads of the partials stalled the consumer warps for several microseconds per
// combine, more than the TMA ring can hide.)
#include <cuda_bf16.h>

#include <type_traits>

#include "device_common.cuh"

namespace fdpp {
namespace {

constexpr int NCW = 4;                  // consumer warps
constexpr int TPW = 16;                 // tokens per consumer warp and tile
constexpr int TILE = NCW * TPW;         // tokens per tile
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int PLAN_SMEM_MAX_B = TC_PLAN_SMEM_MAX_B;
constexpr int QHDR_BYTES = 64;          // unit header at the start of each Q-ring slot
static_assert(TILE == TC_TILE_TOKENS, "tile height is part of the tensor-map contract");

// unit kinds carried in the Q-ring header
enum { KIND_OWN = 0, KIND_LAST_OWN = 1, KIND_REDO = 2, KIND_END = 3 };
// header words: a segment is tokens [T0, T1) of sequence B, virtual head G, starting in split J
// (split length S); DEST is its partial slot (a run slot, or -1: the split's own slot J). A
// redo segment lies in one split: F0/F1 carry its rows' flag bytes (four per word), MASK the rows
// it rewrites, ONL the rows it recomputes with online softmax (the others stay in the phi frame).
enum { H_KIND = 0, H_B, H_G, H_J, H_T0, H_T1, H_DEST, H_F0, H_F1, H_MASK, H_L, H_S, H_ONL, H_WORDS };
static_assert(H_WORDS * 4 <= QHDR_BYTES, "segment header fits its slot");

// Shared-memory layout of one CTA (byte offsets from a 1024-byte aligned base). The merge has
// scratch of its own, so a unit's last stage goes back to the producer like any other:
//   xchg: two slots of one warp's O^T fragments (d/16 float4 per lane) for the warp-sum tree;
//   xrow: l, m and flag word per consumer warp and query row, two buffers (by unit parity);
//   fslot: the window decisions of split pieces (TC_FSLOTS 64-bit words), then the taint words of
//   two segments (by parity).
struct TcLayout {
    int stage_bytes, kv_bytes, qslot_bytes;
    int stages, qring, xchg, xrow, fslot, plan, bars, misc, total;

    __host__ __device__ static constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

    __host__ __device__ TcLayout(int D, int G, int nstage, int B)
        : stage_bytes(2 * TILE * D * 2), kv_bytes(TILE * D * 2),
          qslot_bytes(round_up(QHDR_BYTES + G * D * 2, 128)), stages(0), qring(0), xchg(0),
          xrow(0), fslot(0), plan(0), bars(0), misc(0), total(0)
    {
        qring = stages + nstage * stage_bytes;
        xchg = qring + 2 * qslot_bytes;
        xrow = xchg + 2 * (D / 16) * 32 * 16;
        fslot = xrow + 2 * 3 * NCW * TC_MAX_GROUP * 4;
        plan = fslot + TC_FSLOTS * 8 + 16;
        const int plan_ints = (B <= PLAN_SMEM_MAX_B ? 2 * B + 1 : 0) + 1;
        bars = round_up(plan + plan_ints * 4, 8);
        misc = bars + (2 * nstage + 8) * 8;
        total = misc + 16;
    }
};

struct Ring {
    uint32_t full, empty, qfull, qempty;   // shared addresses of the barrier arrays
    uint32_t cbar;                         // merge: every consumer warp wrote its partial (4 arrivals)
    uint32_t own_done;                     // consumers finished the CTA's own units
    uint32_t mhand;                        // merge: warp 1's sum is in exchange slot 1
    uint32_t mdone;                        // merge: warp 0 has read both exchange slots
    int nstage;
};

// All lanes wait; any lane that runs out of time aborts the CTA (warp-uniform result).
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, volatile int* misc,
                                          const KernelArgs& a)
{
    bool ok = (misc[0] == 0) && mbar_wait(bar, parity);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) {
        misc[0] = 1;
        set_error(a, FDPP_ERRBIT_TIMEOUT);
    }
    return ok;
}

// ------------------------------------------------------------------------------------------
// producer warp
// ------------------------------------------------------------------------------------------
// The unit the producer streams after the current one (for L2 prefetch across units).
struct NextUnit {
    int valid, b, g, t0, t1, win_base, ent;
};

// RG: row-group build (R > 8 rows per kv head): each unit head is a virtual head g = kvh NRG +
// group. Other builds fold heads() to Hkv and kv_head(g) to g.
template <bool RG>
struct Producer {
    const CUtensorMap* tmK;
    const CUtensorMap* tmV;
    const KernelArgs* a;
    const TcLayout* lay;
    Ring rg;
    uint32_t sbase;
    uint8_t* smp;              // generic pointer to the same shared-memory base
    volatile int* misc;
    int* tplan;                // smem (B <= PLAN_SMEM_MAX_B): prefix of the tiles of each sequence [B + 1],
    int* lplan;                //   clamped L_b [B] (n_b = min(ceil(L_b / S), max_splits))
    int S = 0, TS = 0;         // split length, tiles of a full split
    uint32_t stage = 0, phase = 0, qiter = 0;
    int hint_n = 0;            // tiles recorded in this CTA's start-up hint
    bool bad_block = false;

    __device__ __forceinline__ int heads() const { if constexpr (RG) return a->Hv; else return a->Hkv; }
    __device__ __forceinline__ int kv_head(int g) const { if constexpr (RG) return g / a->NRG; else return g; }

    // Split plan: S, the n_b and tile prefixes in smem (or a global walk for large batches),
    // the unit count; T = 64-token tiles of all units.
    __device__ __forceinline__ int make_plan(long long& T)
    {
        const KernelArgs& A = *a;
        const int lane = threadIdx.x & 31;
        const bool in_smem = A.B <= PLAN_SMEM_MAX_B;
        long long sum = 0;
        bool bad = false;
        for (int b = lane; b < A.B; b += 32) {
            const int L = A.seq_lens[b];
            bad |= (L < 0 || L > A.max_seq_len);
            const int Lc = clamp_len(L, A.max_seq_len);
            sum += Lc;
            if (in_smem) lplan[b] = Lc;
        }
        sum = warp_sum(sum);
        bad = __any_sync(0xffffffffu, bad);
        S = auto_split_len(sum, A);
        TS = ceil_div_i(S, TILE);
        int run = 0;
        long long trun = 0;
        __syncwarp();
        for (int base = 0; base < A.B; base += 32) {
            const int b = base + lane;
            int nb = 0;
            long long nt = 0;
            if (b < A.B) {
                const int Lc = in_smem ? lplan[b] : clamp_len(A.seq_lens[b], A.max_seq_len);
                nb = min(ceil_div_i(Lc, S), A.max_splits);
                if (nb > 0)
                    nt = (long long)(nb - 1) * TS + ceil_div_i(min(Lc - (nb - 1) * S, S), TILE);
            }
            int incl = nb;
            long long tincl = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                const long long ty = __shfl_up_sync(0xffffffffu, tincl, o);
                if (lane >= o) { incl += y; tincl += ty; }
            }
            __syncwarp();
            if (b < A.B) {
                const int tfirst = (int)(trun + tincl - nt);
                if (in_smem) tplan[b] = tfirst;
                if (blockIdx.x == 0) { A.nsplit[b] = nb; A.tstart[b] = tfirst; }
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
            trun += __shfl_sync(0xffffffffu, tincl, 31);
        }
        if (lane == 0) {
            if (in_smem) tplan[A.B] = (int)trun;
            if (blockIdx.x == 0) A.tstart[A.B] = (int)trun;
        }
        __syncwarp();
        // units and tiles over the virtual heads (kv head, row group); the diag reports the
        // (b, g, j) units
        T = trun * heads();
        const int n_units = run * heads();
        if (blockIdx.x == 0) {
            if (lane == 0) {
                A.hdr[HDR_SPLIT] = S;
                A.hdr[HDR_UNITS] = run * A.Hkv;
                A.hdr[HDR_KERNEL] = A.kernel_id;
                A.hdr[HDR_BATCH] = A.B;
                A.hdr[HDR_MAXSPLITS] = A.max_splits;
                if (bad) set_error(A, FDPP_ERRBIT_SEQ_LEN);
            }
            // rows of empty sequences are zero (no unit will write them)
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(A.out);
            for (int b = 0; b < A.B; ++b) {
                const int Lc = in_smem ? lplan[b] : clamp_len(A.seq_lens[b], A.max_seq_len);
                if (Lc != 0) continue;
                for (int i = lane; i < A.Tq * A.Hq * A.D; i += 32)
                    out[(long long)b * A.Tq * A.Hq * A.D + i] = __float2bfloat16_rn(0.f);
            }
        }
        return n_units;
    }

    // L2 prefetch of one 64-token tile of kv head g (no shared memory, no barrier): the tile's
    // DRAM reads start before a ring stage is free for it, so the ring's own TMA load hits L2.
    // Paged: only blocks inside the given block-table window are prefetched.
    template <int D, bool PAGED>
    __device__ __forceinline__ void prefetch_tile(int b, int g, int tt, int t1, int win_base, int ent)
    {
        constexpr int HALVES = D / 64;
        constexpr int PER_BLK = 2 * HALVES;
        const KernelArgs& A = *a;
        const int lane = threadIdx.x & 31;
        const int nvalid = min(TILE, t1 - tt);
        if (nvalid <= 0) return;
        if (!PAGED) {
            if (lane < PER_BLK) {
                const int hv = lane >> 1;
                tma_prefetch_3d((lane & 1) ? tmV : tmK, kv_head(g) * D + hv * 64, tt, b);
            }
        } else {
            const int bs = A.block_size;
            const int lb0 = tt / bs;
            const int nbk = (bs <= TILE) ? ceil_div_i(nvalid, bs) : 1;
            if (lb0 < win_base || lb0 + nbk > win_base + 32) return;
            const int k = min(lane / PER_BLK, TILE / 16 - 1), r = lane % PER_BLK, hv = r >> 1;
            const int e = __shfl_sync(0xffffffffu, ent, min(lb0 + k - win_base, 31));
            if (lane < nbk * PER_BLK && e >= 0 && e < A.num_blocks)
                tma_prefetch_3d((r & 1) ? tmV : tmK, kv_head(g) * D + hv * 64,
                                (bs <= TILE) ? 0 : (tt % bs), e);
        }
    }

    // Emits one segment: tokens [t0, t1) of sequence b, virtual head g, starting in split j,
    // whose partial goes to `dest` (-1: split j's own slot, else run slot `dest`); hw: a redo
    // piece's flag words, rewritten rows and online rows. Header + Q rows go into the Q ring, then
    // the K/V tiles into the stage ring, prefetching into L2 the tile `pf` places ahead (in this
    // segment, or in `nx`, the next one).
    // pre_base/pre_ent: a block-table window (entries pre_base + lane) loaded ahead of time.
    template <int D, bool PAGED>
    __device__ __forceinline__ bool emit(int kind, int b, int g, int j, int t0, int t1, int L,
                                         int dest, const int (&hw)[4], int pre_base = -(1 << 30),
                                         int pre_ent = -1, const NextUnit* nx = nullptr,
                                         bool first = false)
    {
        constexpr int HALVES = D / 64;
        const KernelArgs& A = *a;
        const int lane = threadIdx.x & 31;
        const uint32_t qs = qiter & 1u;
        if (!ring_wait(rg.qempty + 8 * qs, ((qiter >> 1) & 1u) ^ 1u, misc, A)) return false;
        const uint32_t slot = sbase + lay->qring + qs * lay->qslot_bytes;
        if (lane == 0) {
            int* hdr = reinterpret_cast<int*>(smp + lay->qring + qs * lay->qslot_bytes);
            hdr[H_KIND] = kind; hdr[H_B] = b; hdr[H_G] = g; hdr[H_J] = j;
            hdr[H_T0] = t0; hdr[H_T1] = t1; hdr[H_DEST] = dest;
            hdr[H_F0] = hw[0]; hdr[H_F1] = hw[1]; hdr[H_MASK] = hw[2]; hdr[H_L] = L;
            hdr[H_S] = S; hdr[H_ONL] = hw[3];
            if (kind == KIND_END) {
                mbar_arrive(rg.qfull + 8 * qs);
            } else {
                // The unit's query rows: row rr of the kv head's R = Tq G rows is head
                // kvh G + rr % G of query token rr / G. Virtual head g = kvh NRG + group takes
                // rows group * 8 .. (up to Rg of them).
                const int kvh = kv_head(g);
                const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(A.q);
                if constexpr (!RG) {
                    const uint32_t bytes = (uint32_t)(A.G * D * 2);
                    mbar_arrive_expect_tx(rg.qfull + 8 * qs, bytes * (uint32_t)A.Tq);
                    for (int i = 0; i < A.Tq; ++i)
                        bulk_load(slot + QHDR_BYTES + i * bytes,
                                  q + (((long long)b * A.Tq + i) * A.Hq + (long long)kvh * A.G) * D, bytes,
                                  rg.qfull + 8 * qs);
                } else {
                    const int rbase = (g - kvh * A.NRG) * TC_MAX_GROUP;
                    const int nrow = min(A.Rg, A.R - rbase);
                    const uint32_t bytes = (uint32_t)(D * 2);
                    mbar_arrive_expect_tx(rg.qfull + 8 * qs, bytes * (uint32_t)nrow);
                    for (int rr = 0; rr < nrow; ++rr) {
                        const int row = rbase + rr, i = row / A.G;
                        bulk_load(slot + QHDR_BYTES + rr * bytes,
                                  q + (((long long)b * A.Tq + i) * A.Hq + (long long)kvh * A.G + (row - i * A.G)) * D,
                                  bytes, rg.qfull + 8 * qs);
                    }
                }
            }
        }
        ++qiter;
        if (kind == KIND_END) return true;

        const int gk = kv_head(g);
        const int bs = PAGED ? A.block_size : TILE;
        const int rows_box = bs < TILE ? bs : TILE;
        const uint32_t box_bytes = 128u * (uint32_t)rows_box;
        // 64-token tiles of the segment, never across a split boundary (counted only for the
        // L2 prefetch, which is off by default)
        int ntiles = 0;
        if (A.pf_tiles > 0)
            for (int x = t0; x < t1;) {
                const int e = min((x / S + 1) * S, t1);
                ntiles += ceil_div_i(e - x, TILE);
                x = e;
            }
        int win_base = pre_base, ent = pre_ent;    // paged: 32 block-table entries per window
        const int nblk_seq = PAGED ? ceil_div_i(L, bs) : 0;
        constexpr int PER_BLK = 2 * HALVES;        // boxes per block: K and V, each half
        const int pf = A.pf_tiles;
        if (PAGED && pf > 0 && win_base == -(1 << 30)) {   // the segment's first window, now
            win_base = t0 / bs;
            const int lb = win_base + lane;
            ent = (lb < nblk_seq) ? __ldg(A.block_table + (long long)b * A.max_blocks + lb) : -1;
        }
        if (first && pf > 0)                       // the CTA's first segment: nothing prefetched
            for (int ti = 1; ti <= pf && ti < ntiles; ++ti)
                prefetch_tile<D, PAGED>(b, g, t0 + ti * TILE, t1, win_base, ent);
        int tt = t0, se = (t0 / S + 1) * S;        // tile start, end of its split
        for (int i = 0; tt < t1; ++i) {
            const int tend = min(min(tt + TILE, se), t1);
            const int nvalid = tend - tt;
            if (!ring_wait(rg.empty + 8 * stage, phase ^ 1u, misc, A)) return false;
            const uint32_t kdst = sbase + lay->stages + stage * lay->stage_bytes;
            const uint32_t vdst = kdst + lay->kv_bytes;
            const uint32_t fb = rg.full + 8 * stage;
            if (!PAGED) {
                // one lane per box: K and V, each 128-byte half of the head row
                if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)lay->stage_bytes);
                __syncwarp();
                if (lane < PER_BLK) {
                    const int hv = lane >> 1;
                    tma_load_3d(((lane & 1) ? vdst : kdst) + hv * TILE * 128, (lane & 1) ? tmV : tmK,
                                gk * D + hv * 64, tt, b, fb);
                }
                // the first tiles of this call are the next call's start-up hint
                if (lane == 0 && hint_n < HINT_TILES && kind != KIND_REDO && blockIdx.x < TC_MAX_PARTS) {
                    int* h = A.hint + (long long)blockIdx.x * HINT_WORDS;
                    h[1 + 3 * hint_n] = gk * D;
                    h[2 + 3 * hint_n] = tt;
                    h[3 + 3 * hint_n] = b;
                    h[0] = ++hint_n;
                }
            } else {
                const int lb0 = tt / bs;
                const int nbk = (bs <= TILE) ? ceil_div_i(nvalid, bs) : 1;
                if (lb0 < win_base || lb0 + nbk > win_base + 32) {
                    win_base = lb0;
                    const int lb = lb0 + lane;
                    ent = (lb < nblk_seq) ? __ldg(A.block_table + (long long)b * A.max_blocks + lb) : -1;
                }
                uint32_t bytes = 0;
#pragma unroll
                for (int k = 0; k < TILE / 16; ++k) {
                    if (k < nbk) {
                        const int e = __shfl_sync(0xffffffffu, ent, lb0 + k - win_base);
                        if (e >= 0 && e < A.num_blocks) bytes += PER_BLK * box_bytes;
                        else bad_block = true;
                    }
                }
                if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
                __syncwarp();
                // one lane per (block, K/V, half) box
                const int k = min(lane / PER_BLK, TILE / 16 - 1), r = lane % PER_BLK, hv = r >> 1;
                const int e = __shfl_sync(0xffffffffu, ent, min(lb0 + k - win_base, 31));
                if (lane < nbk * PER_BLK && e >= 0 && e < A.num_blocks) {
                    const int y = (bs <= TILE) ? 0 : (tt % bs);
                    const uint32_t off = hv * TILE * 128 + k * rows_box * 128;
                    tma_load_3d(((r & 1) ? vdst : kdst) + off, (r & 1) ? tmV : tmK, gk * D + hv * 64, y,
                                e, fb);
                }
            }
            if (pf > 0) {
                const int ti = i + pf;
                if (ti < ntiles) {
                    prefetch_tile<D, PAGED>(b, g, t0 + ti * TILE, t1, win_base, ent);
                } else if (nx && nx->valid) {
                    const int tn = nx->t0 + (ti - ntiles) * TILE;
                    if (tn < nx->t1) prefetch_tile<D, PAGED>(nx->b, nx->g, tn, nx->t1, nx->win_base, nx->ent);
                }
            }
            if (++stage == (uint32_t)rg.nstage) { stage = 0; phase ^= 1u; }
            tt = tend;
            if (tt == se) se += S;
        }
        return true;
    }

    // The first block-table window (32 entries from the block holding token t0) of a segment
    // that will be emitted next, loaded one segment ahead.
    __device__ __forceinline__ int window_entry(int b, int t0, int L) const
    {
        const KernelArgs& A = *a;
        const int lb = t0 / A.block_size + (int)(threadIdx.x & 31);
        return lb < ceil_div_i(L, A.block_size) ? __ldg(A.block_table + (long long)b * A.max_blocks + lb)
                                                : -1;
    }

    // Own work, tile-balanced: the T tiles of all units (in unit order b, g, j) are cut into P
    // equal parts and CTA c streams part c, [c T / P, (c + 1) T / P). A part is a sequence of
    // runs, one per (sequence, virtual head) it touches; a run may cover several splits and
    // begin or end inside one. Each run leaves one phi-frame partial, in run slot c + u (u: the
    // index of the (row group, sequence, kv head) in tile order; the slots of all runs are
    // distinct), and the flag bytes split by split.
    // RG builds order the tiles group-major, (row group, b, kv head, j): the groups' ranges
    // have the same shape, so parts c, c + P / NRG, ... read the same K/V tiles at about the
    // same time and all but the first find them in L2.
    template <int D, bool PAGED>
    __device__ __forceinline__ bool run_parts(long long T, int P, bool& had_own)
    {
        const KernelArgs& A = *a;
        const int c = blockIdx.x;
        if (c >= P) return true;
        // floor(c T / P) = c q + floor(c r / P) with T = q P + r: no 64-bit division
        const long long q = T / P;
        const int r = (int)(T - q * P);
        const long long tb = (long long)c * q + (c * r) / P;
        const long long te = (long long)(c + 1) * q + ((c + 1) * r) / P;
        const int zero4[4] = {0, 0, 0, 0};
        struct Seg { int b, g, j, t0, t1, L, ntile, dest; };
        const int nseq = A.B;
        int cb = 0, cgrp = 0;
        auto seg_at = [&](long long t, Seg& s) {
            long long tg = t;                        // tile index within the row group
            int grp = 0;
            if constexpr (RG) {
                const long long TG = (long long)A.Hkv * tplan[A.B];
                grp = (int)(t / TG);
                tg = t - grp * TG;
                if (grp != cgrp) { cgrp = grp; cb = 0; }
            }
            while ((long long)A.Hkv * tplan[cb + 1] <= tg) ++cb;
            const int ntb = tplan[cb + 1] - tplan[cb];
            const int r = (int)(tg - (long long)A.Hkv * tplan[cb]);
            s.b = cb;
            const int kvh = r / ntb;
            s.g = RG ? kvh * A.NRG + grp : kvh;
            const int k = r - kvh * ntb;             // tile of sequence cb, kv head kvh
            // the run: tiles k .. kend - 1 of the sequence's ntb (split j has tiles j TS .. j TS +
            // TS - 1, the last split fewer), tokens t0 .. t1
            const int kend = (int)min((long long)ntb, k + (te - t));
            s.j = k / TS;
            s.L = lplan[cb];
            s.t0 = s.j * S + (k - s.j * TS) * TILE;
            if (kend >= ntb) {
                s.t1 = s.L;
            } else {
                const int je = kend / TS;
                s.t1 = je * S + (kend - je * TS) * TILE;
            }
            s.ntile = kend - k;
            s.dest = c + (grp * nseq + cb) * A.Hkv + kvh;
        };
        Seg cur, nxt;
        long long t = tb;
        seg_at(t, cur);
        int cur_ent = PAGED ? window_entry(cur.b, cur.t0, cur.L) : -1;
        for (;;) {
            const long long tn = t + cur.ntile;
            const bool last = tn >= te;
            // The next segment is located after this one is issued (its block-table window is
            // loaded while the ring holds this segment's tiles), unless the L2 prefetch wants
            // its first tiles now.
            NextUnit nx{0, 0, 0, 0, 0, -(1 << 30), -1};
            int nxt_ent = -1;
            const bool ahead = !last && A.pf_tiles > 0;
            if (ahead) {
                seg_at(tn, nxt);
                if (PAGED) nxt_ent = window_entry(nxt.b, nxt.t0, nxt.L);
                nx = NextUnit{1, nxt.b, nxt.g, nxt.t0, nxt.t1,
                              PAGED ? nxt.t0 / A.block_size : -(1 << 30), nxt_ent};
            }
            if (last) grid_launch_dependents();
            if (!emit<D, PAGED>(last ? KIND_LAST_OWN : KIND_OWN, cur.b, cur.g, cur.j, cur.t0, cur.t1,
                                cur.L, cur.dest, zero4,
                                PAGED ? cur.t0 / A.block_size : -(1 << 30), cur_ent, &nx, !had_own))
                return false;
            had_own = true;
            if (last) break;
            if (!ahead) {
                seg_at(tn, nxt);
                if (PAGED) nxt_ent = window_entry(nxt.b, nxt.t0, nxt.L);
            }
            t = tn;
            cur = nxt;
            cur_ent = nxt_ent;
        }
        return true;
    }

    // Own work for batches whose plan is not kept in shared memory: whole units
    // u = blockIdx.x + k * gridDim.x, found by a walk over seq_lens.
    template <int D, bool PAGED>
    __device__ __forceinline__ bool run_units(int n_units, bool& had_own)
    {
        const KernelArgs& A = *a;
        const int zero4[4] = {0, 0, 0, 0};
        UnitCursor cur;
        cur.reset();
        for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
            int b, g, j, L;
            cur.seek(A, heads(), S, u, b, g, j, L);
            const int kind = (u + gridDim.x >= n_units) ? KIND_LAST_OWN : KIND_OWN;
            if (kind == KIND_LAST_OWN) grid_launch_dependents();
            const int t0 = j * S, t1 = min(t0 + S, L);
            if (!emit<D, PAGED>(kind, b, g, j, t0, t1, L, -1, zero4, -(1 << 30), -1, nullptr, !had_own))
                return false;
            had_own = true;
        }
        return true;
    }

    template <int D, bool PAGED>
    __device__ __forceinline__ void run()
    {
        const KernelArgs& A = *a;
        const int lane = threadIdx.x & 31;
        long long T = 0;
        const int n_units = make_plan(T);
        const bool in_smem = A.B <= PLAN_SMEM_MAX_B;
        const int P = (in_smem && T > 0 && T < (1ll << 31))
                          ? (int)min(min((long long)gridDim.x, T), (long long)TC_MAX_PARTS) : 0;
        if (blockIdx.x == 0 && lane == 0) {
            A.hdr[HDR_PARTS] = P;
            A.hdr[HDR_TILES] = P > 0 ? (int)T : 0;
        }
        bool had_own = false;
        const bool ok = P > 0 ? run_parts<D, PAGED>(T, P, had_own) : run_units<D, PAGED>(n_units, had_own);
        if (!ok) return;

        if (A.mode == FDPP_MODE_NORMAL) {
            // The consumers push this CTA's flagged segments before they report the own work done.
            // The list is REDO_NLISTS lists, CTA c pushing to list c % REDO_NLISTS: a CTA drains
            // its own list first, then the others in turn, so that few CTAs contend for one
            // list's claim word.
            if (had_own && !ring_wait(rg.own_done, 0u, misc, A)) return;
            for (;;) {
                // every list's (count, taken) in one read, a lane per list starting at this CTA's
                const int my = (int)((blockIdx.x + lane) % REDO_NLISTS);
                bool pending = false;
                int waiting = 0;
                if (lane < REDO_NLISTS) {
                    const unsigned long long both = ld_relaxed_gpu_u64(
                        reinterpret_cast<const unsigned long long*>(&A.hdr[HDR_REDO_LISTS + 2 * my]));
                    waiting = (int)(unsigned)(both & 0xffffffffull) - (int)(unsigned)(both >> 32);
                    pending = waiting > 0;
                }
                waiting = warp_sum(max(waiting, 0));      // entries not yet claimed, all lists
                const unsigned lists = __ballot_sync(0xffffffffu, pending);
                if (lists == 0u) break;
                const int list = (int)((blockIdx.x + (__ffs(lists) - 1)) % REDO_NLISTS);
                int* cnt = &A.hdr[HDR_REDO_LISTS + 2 * list];
                int* taken = cnt + 1;
                int k = 0;
                bool got = false;
                if (lane == 0) {
                    for (;;) {
                        // count and taken (the next word) in one read
                        const unsigned long long both = ld_relaxed_gpu_u64(
                            reinterpret_cast<const unsigned long long*>(cnt));
                        const int c = (int)(unsigned)(both & 0xffffffffull);
                        const int t = (int)(unsigned)(both >> 32);
                        if (t >= c) break;
                        if (atomicCAS(taken, t, t + 1) == t) { k = t; got = true; break; }
                    }
                }
                got = __shfl_sync(0xffffffffu, got, 0);
                k = __shfl_sync(0xffffffffu, k, 0);
                if (!got) continue;
                // the pusher reserved entry k before storing it: read it with a bounded wait
                long long e = 0, rng = 0, dst = 0, tnt = 0;
                if (lane == 0) {
                    long long* ent = A.redo + ((long long)list * A.redo_cap + k) * REDO_WORDS;
                    const uint64_t t0 = global_ns();
                    while ((e = ld_acquire_gpu(ent)) == 0 && global_ns() - t0 < FDPP_WAIT_NS) {
                    }
                    if (e != 0) {
                        rng = __ldcg(ent + 1);
                        dst = __ldcg(ent + 2);
                        tnt = __ldcg(ent + 3);
                        ent[0] = 0;                    // leave the list zeroed for the next call
                    }
                }
                e = __shfl_sync(0xffffffffu, e, 0);
                rng = __shfl_sync(0xffffffffu, rng, 0);
                dst = __shfl_sync(0xffffffffu, dst, 0);
                tnt = __shfl_sync(0xffffffffu, tnt, 0);
                if (e == 0) {
                    if (lane == 0) { misc[0] = 1; set_error(A, FDPP_ERRBIT_TIMEOUT); }
                    return;
                }
                const int rb = (int)(e & 0xffffffffll) - 1;
                const int gj = (int)(e >> 32);
                const int rg_ = gj / A.max_splits;
                const int st0 = (int)(rng & 0xffffffffll), st1 = (int)(rng >> 32);
                const int dest = (int)dst;
                const unsigned taint = (unsigned)tnt;     // the run's rows to recompute
                const int L = clamp_len(A.seq_lens[rb], A.max_seq_len);
                const int rkvh = kv_head(rg_);
                const int rrow = RG ? (rg_ - rkvh * A.NRG) * TC_MAX_GROUP + lane : lane;
                const int rows = RG ? A.Rg : A.R;        // rows of a unit (run-slot stride)
                // The tainted run again, split by split: each piece's tainted rows are rewritten,
                // with online softmax where that split's scores left the window (its own flag
                // bytes, written by the pushing CTA before its push), else in the phi frame. A
                // first piece that starts inside a split goes back to the run slot (its flags are
                // the slot's edge flags); every other piece to its split's own slot. An entry of
                // several pieces keeps its first piece here and goes back on this CTA's list for
                // the rest, which another free CTA cuts again (while fewer than REDO_SPLIT_BELOW
                // entries wait).
                int st1_own = st1;
                {
                    const int pe = min((st0 / S + 1) * S, st1);   // end of the first piece
                    // only while few entries wait: with many, every free CTA has one already
                    if (pe < st1 && waiting < REDO_SPLIT_BELOW) {
                        st1_own = pe;
                        if (lane == 0) {
                            const int ml = (int)(blockIdx.x % REDO_NLISTS);
                            const int kk = atomicAdd(&A.hdr[HDR_REDO_LISTS + 2 * ml], 1);
                            long long* ent = A.redo + ((long long)ml * A.redo_cap + kk) * REDO_WORDS;
                            ent[1] = (long long)(unsigned)pe | ((long long)(unsigned)st1 << 32);
                            ent[2] = -1;
                            ent[3] = (long long)taint;
                            st_release_gpu(ent, ((long long)(rg_ * A.max_splits + pe / S) << 32) |
                                                    (long long)(unsigned)(rb + 1));
                        }
                    }
                }
                for (int tp0 = st0; tp0 < st1_own;) {
                    const int rj = tp0 / S;
                    const int tp1 = min((rj + 1) * S, st1_own);
                    const int dp = (tp0 == st0 && dest >= 0 && tp0 != rj * S) ? dest : -1;
                    int hw[4] = {0, 0, (int)taint, 0};
                    if (lane < rows && rrow < A.R) {
                        const unsigned f = dp < 0 ? __ldcg(A.flags + unit_row_slot(A, rb, rkvh, rrow, rj))
                                                  : __ldcg(A.xf + (long long)dp * rows + lane);
                        const unsigned sh = (unsigned)(lane & 3) * 8u;
                        hw[0] = (int)(lane < 4 ? (f << sh) : 0u);
                        hw[1] = (int)(lane >= 4 ? (f << sh) : 0u);
                        hw[3] = (int)(((f & FDPP_FLAG_OUT) && ((taint >> lane) & 1u)) ? (1u << lane) : 0u);
                    }
    #pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        hw[0] |= __shfl_xor_sync(0xffffffffu, hw[0], o);
                        hw[1] |= __shfl_xor_sync(0xffffffffu, hw[1], o);
                        hw[3] |= __shfl_xor_sync(0xffffffffu, hw[3], o);
                    }
                    if (!emit<D, PAGED>(KIND_REDO, rb, rg_, rj, tp0, tp1, L, dp, hw)) return;
                    tp0 = tp1;
                }
            }
        }
        const int zeros[4] = {0, 0, 0, 0};
        emit<D, PAGED>(KIND_END, 0, 0, 0, 0, 0, 0, -1, zeros);
    }
};

// ------------------------------------------------------------------------------------------
// consumer warps
// ------------------------------------------------------------------------------------------
template <int D, bool MQ, bool RG>
__device__ __forceinline__ void consume(const KernelArgs& a, const TcLayout& lay, uint8_t* sm,
                                        uint32_t sbase, const Ring& rg, volatile int* misc)
{
    // The tile is computed transposed, tokens on the MMA's M dimension and heads on N:
    //   S^T[16 tok x 8 heads] = K[16 x d] Q^T[d x 8]      (d/16 MMAs)
    //   O^T[d x 8 heads]     += V^T[d x 16 tok] P^T[16 x 8] (d/16 MMAs, d on M)
    // Fragment roles for lane = 4 r + qd: S^T and O^T rows r and r+8 (a token, resp. a d),
    // columns 2qd and 2qd+1 (two heads). P^T is turned into the B operand of the second MMA
    // with movmatrix.trans. P is carried as bf16 hi + lo: for G <= 4 the lo part rides in head
    // columns 4..7 (unused otherwise), so P.V costs d/16 MMAs; for G > 4 hi and lo go through
    // two MMAs into the same accumulator.
    // A segment is a run of tiles of one (sequence, virtual head) that may cover several splits:
    // the phi-frame sums run across them, and the window decisions are taken split by split.
    constexpr int KS = D / 16;           // k-steps of S^T, and m-tiles of O^T
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, qd = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;      // ldmatrix: matrix and row of this lane
    const bool pack_lo = a.R <= 4;
    const uint32_t k_row = warp * TPW + (mi & 1) * 8 + r8;
    const uint32_t v_row = warp * TPW + (mi >> 1) * 8 + r8;
    const int tok_r = warp * TPW + r;             // this lane's tokens: tok_r and tok_r + 8
    const int tok_q = warp * TPW + 2 * qd;        // tokens of this lane's V^T fragment columns
    const int head0 = 2 * qd;                     // this lane's heads: head0, head0 + 1
    uint32_t stage = 0, phase = 0, qiter = 0, un = 0;   // un: segments merged so far
    uint32_t portion = 0;                         // split pieces of own segments finished
    unsigned long long* fslot = reinterpret_cast<unsigned long long*>(sm + lay.fslot);
    unsigned* taint_s = reinterpret_cast<unsigned*>(sm + lay.fslot + TC_FSLOTS * 8);

    for (;;) {
        // ---- next segment from the producer ----
        const uint32_t qs = qiter & 1u;
        if (!ring_wait(rg.qfull + 8 * qs, (qiter >> 1) & 1u, misc, a)) return;
        const uint8_t* slot = sm + lay.qring + qs * lay.qslot_bytes;
        const int* hdr = reinterpret_cast<const int*>(slot);
        const int kind = hdr[H_KIND];
        if (kind == KIND_END) return;
        const int b = hdr[H_B], g = hdr[H_G], j0 = hdr[H_J];
        const int t0 = hdr[H_T0], t1 = hdr[H_T1], dest = hdr[H_DEST], seq_len = hdr[H_L];
        const int S = hdr[H_S];
        const unsigned fw0 = (unsigned)hdr[H_F0], fw1 = (unsigned)hdr[H_F1];
        const unsigned redo_mask = (unsigned)hdr[H_MASK];
        const unsigned onl_mask = (unsigned)hdr[H_ONL];
        const bool redo = kind == KIND_REDO;
        // a redo piece keeps the phi frame for rows whose own split stayed in the window
        const bool online = (redo && onl_mask != 0u) || (a.mode == FDPP_MODE_FORCE_ONLINE);
        const uint32_t upar = un & 1u;
        // RG builds: virtual head g = kv head kvh, row group of rows rbase .. rbase + nrow() - 1
        // of the kv head (rows() = the unit's row stride in the run slots); else g is the kv
        // head. Both are read at each use: a kernel parameter holds no register between uses.
        const int kvh = RG ? g / a.NRG : g;
        const int rbase = RG ? (g - kvh * a.NRG) * TC_MAX_GROUP : 0;
        auto nrow = [&]() { return RG ? min(a.Rg, a.R - rbase) : a.R; };
        auto rows = [&]() { return RG ? a.Rg : a.R; };
        const bool q_ok = r < nrow();              // this lane supplies Q row r of the group

        uint32_t qb[KS][2];                        // B operand of S^T: Q^T, column r = head r
        {
            const uint8_t* qp = slot + QHDR_BYTES;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qb[ks][0] = q_ok ? *reinterpret_cast<const uint32_t*>(qp + (r * D + ks * 16 + 2 * qd) * 2) : 0u;
                qb[ks][1] = q_ok ? *reinterpret_cast<const uint32_t*>(qp + (r * D + ks * 16 + 8 + 2 * qd) * 2) : 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rg.qempty + 8 * qs);
            ++qiter;
        }

        float o[KS][4];                            // O^T rows 16mt + r (+8), heads head0, head0+1
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float lsum[2] = {0.f, 0.f};
        // this lane's two query rows head0, head0 + 1 of the group: kv-head row rr = rbase + head0
        // (+ 1) is head kvh G + rr % G of query token rr / G, which sees the keys
        // t < L - Tq + 1 + rr / G
        const bool hv[2] = {head0 < nrow(), head0 + 1 < nrow()};
        const float phv[2] = {hv[0] ? phi_of(a, kvh * a.G + (rbase + head0) % a.G) : a.phi,
                              hv[1] ? phi_of(a, kvh * a.G + (rbase + head0 + 1) % a.G) : a.phi};
        // several query tokens: keys of the segment each row sees, counted from t0 (none for a
        // lane without a row); one query token sees every key of the segment
        int kseg[2] = {0, 0};
        if constexpr (MQ) {
            kseg[0] = hv[0] ? key_limit(a, seq_len, (rbase + head0) / a.G) - t0 : 0;
            kseg[1] = hv[1] ? key_limit(a, seq_len, (rbase + head0 + 1) / a.G) - t0 : 0;
        }
        // rows kept in the phi frame inside an online segment (a redo piece's clean rows)
        const bool frz[2] = {redo && !((onl_mask >> head0) & 1u), redo && !((onl_mask >> (head0 + 1)) & 1u)};
        float mrun[2] = {online && !frz[0] ? -INFINITY : phv[0], online && !frz[1] ? -INFINITY : phv[1]};
        unsigned fl[2] = {0u, 0u};

        // End of one split piece of an own segment: the four warps' window decisions for it,
        // combined by whichever warp arrives last (one atomic OR on a 64-bit shared word: 4 bits
        // per row, an arrival bit per warp), which writes the rows' flag bytes (the split's own,
        // or the run slot's edge byte for a first piece that starts inside a split) and marks
        // the rows with a score outside the window as the segment's taint. Pieces cycle through
        // TC_FSLOTS words: no warp runs more than a ring's depth of tiles ahead of another.
        auto finish_piece = [&](int jp, bool first_piece) {
            unsigned f0 = fl[0], f1 = fl[1];
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                f0 |= __shfl_xor_sync(0xffffffffu, f0, sh);
                f1 |= __shfl_xor_sync(0xffffffffu, f1, sh);
            }
            fl[0] = fl[1] = 0u;
            if (redo) return;                      // a redo piece's flag bytes come with it
            unsigned word = ((f0 & 15u) << (8 * qd)) | ((f1 & 15u) << (8 * qd + 4));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            const uint32_t ks = portion++ & (uint32_t)(TC_FSLOTS - 1);
            unsigned long long old = 0ull;
            if (lane == 0) old = atomicOr(&fslot[ks], (1ull << (32 + warp)) | (unsigned long long)word);
            old = __shfl_sync(0xffffffffu, old, 0);
            if ((((unsigned)(old >> 32)) | (1u << warp)) != (1u << NCW) - 1u) return;
            const unsigned full = (unsigned)old | word;
            if (lane == 0) {
                fslot[ks] = 0ull;
                unsigned out_rows = 0u;
#pragma unroll
                for (int hh = 0; hh < TC_MAX_GROUP; ++hh)
                    if ((full >> (4 * hh)) & FDPP_FLAG_OUT) out_rows |= 1u << hh;
                if (out_rows) atomicOr(&taint_s[upar], out_rows);
            }
            if (lane < nrow()) {
                const uint8_t fb = (uint8_t)(((full >> (4 * lane)) & 15u) |
                                             (a.mode == FDPP_MODE_FORCE_ONLINE ? FDPP_FLAG_RECOMPUTED : 0u));
                if (first_piece && dest >= 0 && t0 != jp * S)
                    a.xf[(long long)dest * rows() + lane] = fb;
                else
                    a.flags[MQ ? unit_row_slot(a, b, kvh, rbase + lane, jp)
                               : ((long long)b * a.Hq + kvh * a.G + rbase + lane) * a.max_splits + jp] = fb;
            }
        };

        // The tile loop, built once for the phi frame and once for the running max (redo pieces
        // and forced online mode), so the hot phi-frame loop stays compact. Tiles are 64 tokens
        // and never cross a split boundary.
        auto run_tiles = [&](auto online_c) -> bool {
            constexpr bool ONLINE = decltype(online_c)::value;
            int tt = t0, se = (t0 / S + 1) * S, jp = j0;
            bool first_piece = true;
            while (tt < t1) {
                const int tend = min(min(tt + TILE, se), t1);
                const int nvalid = tend - tt;
                if (!ring_wait(rg.full + 8 * stage, phase, misc, a)) return false;
                const uint32_t kb = sbase + lay.stages + stage * lay.stage_bytes;
                const uint32_t vb = kb + lay.kv_bytes;

                // S^T = K Q^T for this warp's 16 tokens, two accumulation chains
                float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int chunk = 2 * ks + (mi >> 1);
                    const uint32_t addr = kb + (chunk >> 3) * (TILE * 128) + k_row * 128 + (((chunk & 7) ^ r8) << 4);
                    uint32_t k0, k1, k2, k3;
                    ldsm_x4(addr, k0, k1, k2, k3);
                    mma_16816(sa[ks & 1], k0, k1, k2, k3, qb[ks][0], qb[ks][1]);
                }
                // element e of sa: token tok_r + 8 (e >> 1), head head0 + (e & 1)
                float sv[4];
                bool valid[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sv[e] = __fmul_rn(sa[0][e] + sa[1][e], a.scale);
                    const int tok = tok_r + 8 * (e >> 1);
                    if constexpr (MQ)
                        valid[e] = tok < min(nvalid, kseg[e & 1] - (tt - t0));   // the row's tokens of the tile
                    else
                        valid[e] = hv[e & 1] && tok < nvalid;
                    if (valid[e]) fl[e & 1] |= classify(__fsub_rn(sv[e], phv[e & 1]), a.lo, a.hi);
                }

                float p[4];
                if constexpr (!ONLINE) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) p[e] = valid[e] ? __expf(__fsub_rn(sv[e], phv[e & 1])) : 0.f;
                } else {
                    float corr[2];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        float tmax = -INFINITY;
                        if (valid[c]) tmax = sv[c];
                        if (valid[c + 2]) tmax = fmaxf(tmax, sv[c + 2]);
                        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
                        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
                        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
                        const float mnew = frz[c] ? mrun[c] : fmaxf(mrun[c], tmax);
                        corr[c] = (mrun[c] == mnew) ? 1.f : (mrun[c] == -INFINITY ? 0.f : __expf(mrun[c] - mnew));
                        mrun[c] = mnew;
                        lsum[c] *= corr[c];
                        p[c] = valid[c] ? __expf(sv[c] - mnew) : 0.f;
                        p[c + 2] = valid[c + 2] ? __expf(sv[c + 2] - mnew) : 0.f;
                    }
                    // columns 4..7 of lanes qd >= 2 hold the lo part of heads 0..3 (G <= 4)
                    float oc[2] = {corr[0], corr[1]};
                    if (pack_lo) {
                        const float x0 = __shfl_xor_sync(0xffffffffu, corr[0], 2);
                        const float x1 = __shfl_xor_sync(0xffffffffu, corr[1], 2);
                        if (qd >= 2) { oc[0] = x0; oc[1] = x1; }
                    }
                    if (oc[0] != 1.f || oc[1] != 1.f) {
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            o[mt][0] *= oc[0]; o[mt][2] *= oc[0];
                            o[mt][1] *= oc[1]; o[mt][3] *= oc[1];
                        }
                    }
                }
                lsum[0] += p[0] + p[2];
                lsum[1] += p[1] + p[3];

                // P^T as the B operand of O^T += V^T P^T (tokens x heads), hi and lo bf16 parts
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(p[0], p[1]);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(p[2], p[3]);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                uint32_t x_hi0 = *reinterpret_cast<const uint32_t*>(&h01);
                uint32_t x_hi1 = *reinterpret_cast<const uint32_t*>(&h23);
                const uint32_t x_lo0 = pack_bf16x2(p[0] - f01.x, p[1] - f01.y);
                const uint32_t x_lo1 = pack_bf16x2(p[2] - f23.x, p[3] - f23.y);
                uint32_t b_hi0, b_hi1, b_lo0 = 0u, b_lo1 = 0u;
                if (pack_lo) {
                    const uint32_t y0 = __shfl_xor_sync(0xffffffffu, x_lo0, 2);
                    const uint32_t y1 = __shfl_xor_sync(0xffffffffu, x_lo1, 2);
                    if (qd >= 2) { x_hi0 = y0; x_hi1 = y1; }
                    b_hi0 = movmatrix_trans(x_hi0);
                    b_hi1 = movmatrix_trans(x_hi1);
                } else {
                    b_hi0 = movmatrix_trans(x_hi0);
                    b_hi1 = movmatrix_trans(x_hi1);
                    b_lo0 = movmatrix_trans(x_lo0);
                    b_lo1 = movmatrix_trans(x_lo1);
                }

                // V rows past the valid tokens may hold anything (NaN included): mask them to zero
                uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
                if (nvalid < TILE) {
                    vm_lo = (tok_q < nvalid ? 0x0000ffffu : 0u) | (tok_q + 1 < nvalid ? 0xffff0000u : 0u);
                    vm_hi = (tok_q + 8 < nvalid ? 0x0000ffffu : 0u) | (tok_q + 9 < nvalid ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    const int chunk = 2 * mt + (mi & 1);
                    const uint32_t addr = vb + (chunk >> 3) * (TILE * 128) + v_row * 128 + (((chunk & 7) ^ r8) << 4);
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(addr, v0, v1, v2, v3);
                    v0 &= vm_lo; v1 &= vm_lo; v2 &= vm_hi; v3 &= vm_hi;
                    mma_16816(o[mt], v0, v1, v2, v3, b_hi0, b_hi1);
                    if (!pack_lo) mma_16816(o[mt], v0, v1, v2, v3, b_lo0, b_lo1);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(rg.empty + 8 * stage);
                if (++stage == (uint32_t)rg.nstage) { stage = 0; phase ^= 1u; }
                tt = tend;
                if (tt == se || tt == t1) {            // a split piece ends here
                    finish_piece(jp, first_piece);
                    first_piece = false;
                    ++jp;
                    se += S;
                }
            }
            return true;
        };
        if (!(online ? run_tiles(std::true_type{}) : run_tiles(std::false_type{}))) return;
        // ---- this warp's partial: reduce over its 16 tokens (lanes r), fold in the lo part ----
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) lsum[c] += __shfl_xor_sync(0xffffffffu, lsum[c], sh);
        }
        if (pack_lo) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(0xffffffffu, o[mt][e], 2);
        }

        // ---- merge of the four warp partials: (w0 + w2) + (w1 + w3) ----
        // Warps 2 and 3 leave their O^T fragments in exchange slots 0 and 1 (after warp 0 has read
        // the previous segment's), every warp its rows' l and m; warps 0 and 1 add the slot of
        // their partner, warp 1 hands its sum to warp 0 through slot 1, and warp 0 writes the
        // rows' partial. In the phi frame every warp's m is phi and each weight is exactly 1, so
        // the sums need no exponentials.
        float4* xs = reinterpret_cast<float4*>(sm + lay.xchg);
        float* xl_s = reinterpret_cast<float*>(sm + lay.xrow) + upar * 3 * NCW * TC_MAX_GROUP;
        float* xm_s = xl_s + NCW * TC_MAX_GROUP;
        if (warp >= 2) {
            if (un > 0 && !ring_wait(rg.mdone, upar ^ 1u, misc, a)) return;
            float4* xslot = xs + (warp - 2) * KS * 32;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) xslot[mt * 32 + lane] = make_float4(o[mt][0], o[mt][1], o[mt][2], o[mt][3]);
        }
        if (r == 0) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!hv[c]) continue;
                xl_s[warp * TC_MAX_GROUP + head0 + c] = lsum[c];
                xm_s[warp * TC_MAX_GROUP + head0 + c] = mrun[c];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(rg.cbar);
        ++un;
        if (warp >= 2) continue;                   // warps 2 and 3 go on to the next segment
        if (!ring_wait(rg.cbar, upar, misc, a)) return;

        // this warp and its partner (warp + 2), each weighted into the rows' common frame
        {
            float ws[2] = {1.f, 1.f}, wp[2] = {1.f, 1.f};
            if (online) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (!hv[c]) continue;
                    const int hh = head0 + c;
                    float M = xm_s[hh];
#pragma unroll
                    for (int w = 1; w < NCW; ++w) M = fmaxf(M, xm_s[w * TC_MAX_GROUP + hh]);
                    ws[c] = frame_weight(xm_s[warp * TC_MAX_GROUP + hh], M);
                    wp[c] = frame_weight(xm_s[(warp + 2) * TC_MAX_GROUP + hh], M);
                }
            }
            const float4* xslot = xs + warp * KS * 32;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const float4 v = xslot[mt * 32 + lane];
                if (!online) {
                    o[mt][0] += v.x; o[mt][1] += v.y; o[mt][2] += v.z; o[mt][3] += v.w;
                } else {
                    o[mt][0] = fmaf(wp[0], v.x, ws[0] * o[mt][0]);
                    o[mt][1] = fmaf(wp[1], v.y, ws[1] * o[mt][1]);
                    o[mt][2] = fmaf(wp[0], v.z, ws[0] * o[mt][2]);
                    o[mt][3] = fmaf(wp[1], v.w, ws[1] * o[mt][3]);
                }
            }
        }
        if (warp == 1) {
            // warp 1 has read slot 1 (warp 3's); its own sum takes the slot for warp 0
            float4* xslot = xs + KS * 32;
            __syncwarp();
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) xslot[mt * 32 + lane] = make_float4(o[mt][0], o[mt][1], o[mt][2], o[mt][3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(rg.mhand);
            continue;
        }

        // ---- warp 0: l and m of every row (lane hh for row hh) ----
        // Rows whose scores left the window in some split of an own segment (its taint, complete
        // once all four warps have merged) get an empty partial here in normal mode: the fallback
        // recomputes them piece by piece. A redo piece rewrites its tainted rows only and writes
        // their flag bytes.
        const unsigned write_mask = redo ? redo_mask : 0xffffffffu;
        const unsigned taint = redo ? 0u : taint_s[upar];
        const bool refill = !redo && a.mode == FDPP_MODE_NORMAL;
        {
            const int hh = lane;
            float M = 0.f, lam = 0.f;
            if (hh < nrow()) {
                M = xm_s[hh];
#pragma unroll
                for (int w = 1; w < NCW; ++w) M = fmaxf(M, xm_s[w * TC_MAX_GROUP + hh]);
#pragma unroll
                for (int w = 0; w < NCW; ++w)
                    lam = online ? fmaf(frame_weight(xm_s[w * TC_MAX_GROUP + hh], M), xl_s[w * TC_MAX_GROUP + hh], lam)
                                 : lam + xl_s[w * TC_MAX_GROUP + hh];
            }
            if (hh < nrow() && ((write_mask >> hh) & 1u)) {
                const long long rs = dest >= 0 ? (long long)dest * rows() + hh
                                     : MQ ? unit_row_slot(a, b, kvh, rbase + hh, j0)
                                          : ((long long)b * a.Hq + kvh * a.G + rbase + hh) * a.max_splits + j0;
                float* lp = dest < 0 ? a.l_part : a.xl;
                float* mp = dest < 0 ? a.m_part : a.xm;
                const bool empty = refill && ((taint >> hh) & 1u);
                lp[rs] = empty ? 0.f : lam;
                mp[rs] = empty ? -INFINITY : M;
                if (redo) {
                    const unsigned f0 = ((hh < 4 ? fw0 : fw1) >> ((hh & 3) * 8)) & 0xffu;
                    const unsigned rc = ((onl_mask >> hh) & 1u) ? FDPP_FLAG_RECOMPUTED : 0u;
                    if (dest < 0) a.flags[rs] = (uint8_t)(f0 | rc | FDPP_FLAG_SLOT);
                    else a.xf[rs] = (uint8_t)(f0 | rc);
                }
            }
        }
        if (!redo && lane == 0) taint_s[upar] = 0u;   // ready for the segment after next
        // the partial rows of this lane: head0 and head0 + 1, the run slot or the split's own
        float* orow[2] = {nullptr, nullptr};
        bool oempty[2] = {false, false};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int hh = head0 + c;
            if (!hv[c] || !((write_mask >> hh) & 1u)) continue;
            oempty[c] = refill && ((taint >> hh) & 1u);
            orow[c] = dest >= 0 ? a.xo + ((long long)dest * rows() + hh) * D
                                : a.o_part + (MQ ? unit_row_slot(a, b, kvh, rbase + hh, j0)
                                                 : ((long long)b * a.Hq + kvh * a.G + rbase + hh) * a.max_splits + j0) * D;
        }
        if (!ring_wait(rg.mhand, upar, misc, a)) return;
        {
            const float4* xslot = xs + KS * 32;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const float4 v = xslot[mt * 32 + lane];
                o[mt][0] += v.x; o[mt][1] += v.y; o[mt][2] += v.z; o[mt][3] += v.w;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(rg.mdone);      // both slots read: warps 2 and 3 may refill them
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            if (orow[c] == nullptr) continue;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                orow[c][16 * mt + r] = oempty[c] ? 0.f : o[mt][c];
                orow[c][16 * mt + r + 8] = oempty[c] ? 0.f : o[mt][c + 2];
            }
        }
        // ---- a segment with rows outside the window goes on the device-wide fallback list ----
        // (every flag byte of its pieces, and warp 0's stores, are ordered before the release
        // store that publishes the entry)
        __syncwarp();
        if (!redo && taint != 0u && a.mode == FDPP_MODE_NORMAL && lane == 0) {
            const int list = (int)(blockIdx.x % REDO_NLISTS);
            const int k = atomicAdd(&a.hdr[HDR_REDO_LISTS + 2 * list], 1);
            long long* ent = a.redo + ((long long)list * a.redo_cap + k) * REDO_WORDS;
            ent[1] = (long long)(unsigned)t0 | ((long long)(unsigned)t1 << 32);
            ent[2] = dest;
            ent[3] = (long long)taint;
            st_release_gpu(ent, ((long long)(g * a.max_splits + j0) << 32) | (long long)(unsigned)(b + 1));
        }
        if (lane == 0 && kind == KIND_LAST_OWN) mbar_arrive(rg.own_done);
    }
}

// ------------------------------------------------------------------------------------------
// kernel
// ------------------------------------------------------------------------------------------
// MINB = CTAs per SM the build is register-limited for: 2 caps a thread at 168 registers (two
// 5-warp CTAs, warps allocated in pairs), 1 leaves the compiler free (~240) and pairs with a
// deeper TMA ring. MQ: several query tokens per sequence (rows R = Tq G with causal key limits);
// the one-token build keeps the plain row addressing. RG (with MQ): more than 8 rows per kv head,
// taken as row groups of 8 by virtual heads.
template <int D, bool PAGED, int MINB, bool MQ, bool RG>
__global__ void __launch_bounds__(NTHREADS, MINB)
    split_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const KernelArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const TcLayout lay(D, RG ? a.Rg : a.R, a.nstage, a.B);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* misc = reinterpret_cast<volatile int*>(sm + lay.misc);   // [0] abort, [1] last
    Ring rg;
    rg.nstage = a.nstage;
    rg.full = sbase + lay.bars;
    rg.empty = rg.full + 8 * a.nstage;
    rg.qfull = rg.empty + 8 * a.nstage;
    rg.qempty = rg.qfull + 16;
    rg.cbar = rg.qempty + 16;
    rg.own_done = rg.cbar + 8;
    rg.mhand = rg.own_done + 8;
    rg.mdone = rg.mhand + 8;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nstage; ++s) {
            mbar_init(rg.full + 8 * s, 1);
            mbar_init(rg.empty + 8 * s, NCW);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(rg.qfull + 8 * s, 1);
            mbar_init(rg.qempty + 8 * s, NCW);
        }
        mbar_init(rg.cbar, NCW);
        mbar_init(rg.own_done, 1);
        mbar_init(rg.mhand, 1);
        mbar_init(rg.mdone, 1);
        misc[0] = 0;
        misc[1] = 0;
        unsigned long long* fs = reinterpret_cast<unsigned long long*>(sm + lay.fslot);
        for (int i = 0; i < TC_FSLOTS + 2; ++i) fs[i] = 0ull;
        fence_mbar_init();
    }
    __syncthreads();
    // Launched as a programmatic dependent: nothing is read into the CTA or written before the
    // previous kernel on the stream has completed. Before that, while it finishes, the tiles this
    // CTA streamed first in the last call (contiguous caches) are prefetched into L2: the split
    // plan changes little from one decode step to the next. A stale hint costs a useless
    // prefetch only (L2 is where the previous kernel's writes land).
    if (!PAGED && warp == NCW && lane == 0 && blockIdx.x < TC_MAX_PARTS) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        const volatile int* h = a.hint + (long long)blockIdx.x * HINT_WORDS;
        const int n = min(max(h[0], 0), HINT_TILES);
        for (int i = 0; i < n; ++i) {
            const int x = h[1 + 3 * i], y = h[2 + 3 * i], z = h[3 + 3 * i];
            if (x < 0 || (x & 63) != 0) continue;
#pragma unroll
            for (int hv = 0; hv < D / 64; ++hv) {
                tma_prefetch_3d(&tmK, x + 64 * hv, y, z);
                tma_prefetch_3d(&tmV, x + 64 * hv, y, z);
            }
        }
    }
    grid_dependency_wait();

    int* plan = reinterpret_cast<int*>(sm + lay.plan);
    Producer<RG> pr{&tmK, &tmV, &a, &lay, rg, sbase, sm, misc, plan, plan + (a.B + 1)};
    if (warp == NCW) {
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
        pr.template run<D, PAGED>();
        if (pr.bad_block && lane == 0) set_error(a, FDPP_ERRBIT_BLOCK_TABLE);
    } else {
        consume<D, MQ, RG>(a, lay, sm, sbase, rg, misc);
    }
    __syncthreads();
    if (warp == NCW && lane == 0) {
        if (misc[0] != 0) {
            // Aborted: let every copy this CTA issued land before it exits (bounded waits). The
            // latest issue into stage s had phase `phase` when s < stage, else phase ^ 1.
            for (int s = 0; s < a.nstage; ++s) {
                const uint32_t par = (uint32_t)s < pr.stage ? pr.phase : (pr.phase ^ 1u);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(rg.full + 8 * s, par) && global_ns() - t0 < 100000000ull) {
                }
            }
            for (uint32_t k = 0; k < 2 && k < pr.qiter; ++k) {
                const uint32_t it = pr.qiter - 1 - k, qs = it & 1u, par = (it >> 1) & 1u;
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(rg.qfull + 8 * qs, par) && global_ns() - t0 < 100000000ull) {
                }
            }
        }
    }
}

template <int D, bool PAGED>
cudaError_t launch_t(const KernelArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                     int smem, int ctas_per_sm, cudaStream_t s)
{
    // several query tokens per sequence take their own build (causal row limits, row addressing),
    // and more than 8 rows per kv head another (row groups)
    const bool two = ctas_per_sm >= 2;
    auto kern = a.NRG > 1 ? (two ? split_tc_kernel<D, PAGED, 2, true, true> : split_tc_kernel<D, PAGED, 1, true, true>)
              : a.Tq > 1  ? (two ? split_tc_kernel<D, PAGED, 2, true, false> : split_tc_kernel<D, PAGED, 1, true, false>)
                          : (two ? split_tc_kernel<D, PAGED, 2, false, false> : split_tc_kernel<D, PAGED, 1, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the previous kernel on the stream (the previous call's combine
    // lets it launch early): its CTAs start while that kernel finishes and wait for it to
    // complete before touching global memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

TcPlan split_tc_plan(int head_dim, int group, int batch, int req_stages, int req_ctas,
                     int smem_per_sm, int smem_per_block)
{
    TcPlan p{0, 0, 0};
    const int reserve = 1024;                         // per-CTA system reservation
    auto bytes = [&](int ns) { return TcLayout(head_dim, group, ns, batch).total + 1024; };
    const int cands[2] = {2, 1};
    for (int ci = 0; ci < 2; ++ci) {
        const int ctas = req_ctas > 0 ? req_ctas : cands[ci];
        const int budget = smem_per_sm / ctas - reserve;
        int ns = req_stages > 0 ? req_stages : 12;
        while (ns >= 2 && (bytes(ns) > budget || bytes(ns) > smem_per_block)) --ns;
        if (req_stages > 0 && ns != req_stages) ns = 0;
        if (ns >= 2) {
            p.nstage = ns;
            p.ctas_per_sm = ctas;
            p.smem_bytes = bytes(ns);
            return p;
        }
        if (req_ctas > 0) break;
    }
    return p;
}

cudaError_t launch_split_tc(const KernelArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, int smem_bytes, int ctas_per_sm, cudaStream_t s)
{
    const bool paged = a.block_table != nullptr;
    if (a.D == 128)
        return paged ? launch_t<128, true>(a, tk, tv, grid, smem_bytes, ctas_per_sm, s)
                     : launch_t<128, false>(a, tk, tv, grid, smem_bytes, ctas_per_sm, s);
    return paged ? launch_t<64, true>(a, tk, tv, grid, smem_bytes, ctas_per_sm, s)
                 : launch_t<64, false>(a, tk, tv, grid, smem_bytes, ctas_per_sm, s);
}

}  // namespace fdpp
