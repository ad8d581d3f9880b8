// split_tc_common.cuh -- what the two tensor-core split kernels share: the tile and segment
// constants, the shared-memory layout of the mma.sync build, the ring barriers and the producer
// warp (split plan, tile-balanced parts, TMA streaming of K/V tiles, fallback-list drain).
// split_tc.cu holds the mma.sync consumer (up to 8 query rows per unit, row groups beyond);
// split_um.cu the tcgen05 consumer (up to 64 query rows per unit, accumulators in tensor memory).
#pragma once

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
// The tcgen05 build (rows up to 64) takes MASK/MASK_HI and ONL/ONL_HI as 64-bit row masks, reads a
// redo piece's flag bytes itself, and streams a segment twice when PASS says so: first for the
// rows' maxima (PASS_MAX), then for the sums in that frame (PASS_SUM).
enum { H_KIND = 0, H_B, H_G, H_J, H_T0, H_T1, H_DEST, H_F0, H_F1, H_MASK, H_L, H_S, H_ONL,
       H_MASK_HI, H_ONL_HI, H_PASS, H_WORDS };
enum { PASS_SUM = 0, PASS_MAX = 1 };
static_assert(H_WORDS * 4 <= QHDR_BYTES, "segment header fits its slot");

// Shared-memory layout of one CTA (byte offsets from a 1024-byte aligned base). The merge has
// scratch of its own, so a unit's last stage goes back to the producer like any other:
//   xchg: two slots of one warp's O^T fragments (d/16 float4 per lane) for the warp-sum tree;
//   xrow: l, m and flag word per consumer warp and query row, two buffers (by unit parity);
//   fslot: the window decisions of split pieces (TC_FSLOTS 64-bit words), then the taint words of
//   two segments (by parity).
struct TcLayout {
    static constexpr bool UM = false;      // the mma.sync build's layout
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

// The start-up hint, by one whole warp before the programmatic dependency wait: the K/V tiles this
// CTA streamed first in the last call go into L2 (contiguous caches; the plan changes little from
// one decode step to the next, and a stale hint costs a useless prefetch only). The hint's words
// arrive in one read, and each lane prefetches one tile.
template <int D>
__device__ __forceinline__ void prefetch_hint(const KernelArgs& a, const CUtensorMap* tmK, const CUtensorMap* tmV)
{
    static_assert(HINT_WORDS <= 32 && 1 + 3 * HINT_TILES <= HINT_WORDS, "hint layout");
    const int lane = threadIdx.x & 31;
    const int* h = a.hint + (long long)blockIdx.x * HINT_WORDS;
    const int w = lane < HINT_WORDS ? __ldcg(h + lane) : 0;
    const int n = min(max(__shfl_sync(0xffffffffu, w, 0), 0), HINT_TILES);
    const int i = min(lane, HINT_TILES - 1);
    const int x = __shfl_sync(0xffffffffu, w, 1 + 3 * i);
    const int y = __shfl_sync(0xffffffffu, w, 2 + 3 * i);
    const int z = __shfl_sync(0xffffffffu, w, 3 + 3 * i);
    if (lane < n && x >= 0 && (x & 63) == 0) {
#pragma unroll
        for (int hv = 0; hv < D / 64; ++hv) {
            tma_prefetch_3d(tmK, x + 64 * hv, y, z);
            tma_prefetch_3d(tmV, x + 64 * hv, y, z);
        }
    }
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
// Lay: TcLayout (mma.sync build: the header and the query rows share a Q-ring slot) or the tcgen05
// build's layout (Lay::UM: headers apart, query rows landed by a 4-D TMA load in 128-byte swizzle).
template <bool RG, typename Lay = TcLayout>
struct Producer {
    const CUtensorMap* tmK;
    const CUtensorMap* tmV;
    const KernelArgs* a;
    const Lay* lay;
    Ring rg;
    uint32_t sbase;
    uint8_t* smp;              // generic pointer to the same shared-memory base
    volatile int* misc;
    int* tplan;                // smem (B <= PLAN_SMEM_MAX_B): prefix of the tiles of each sequence [B + 1],
    int* lplan;                //   clamped L_b [B] (n_b = min(ceil(L_b / S), max_splits))
    const CUtensorMap* tmQ = nullptr;   // Lay::UM: q as {d, Hq, Tq, B}, box {64, G, Tq, 1}
    int S = 0, TS = 0;         // split length, tiles of a full split
    int K = 0;                 // phantom tiles after each unit in the cut of own work
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
                A.hdr[HDR_TC_BUILD] = Lay::UM ? 2 : 1;
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
    // piece's flag words, rewritten rows and online rows (Lay::UM: the rewritten and the online
    // rows as two 64-bit masks, low word first; pass: PASS_SUM or PASS_MAX). Header + Q rows go
    // into the Q ring, then
    // the K/V tiles into the stage ring, prefetching into L2 the tile `pf` places ahead (in this
    // segment, or in `nx`, the next one).
    // pre_base/pre_ent: a block-table window (entries pre_base + lane) loaded ahead of time.
    template <int D, bool PAGED>
    __device__ __forceinline__ bool emit(int kind, int b, int g, int j, int t0, int t1, int L,
                                         int dest, const int (&hw)[4], int pre_base = -(1 << 30),
                                         int pre_ent = -1, const NextUnit* nx = nullptr,
                                         bool first = false, int pass = PASS_SUM)
    {
        constexpr int HALVES = D / 64;
        const KernelArgs& A = *a;
        const int lane = threadIdx.x & 31;
        const uint32_t qs = qiter & 1u;
        if (!ring_wait(rg.qempty + 8 * qs, ((qiter >> 1) & 1u) ^ 1u, misc, A)) return false;
        const uint32_t slot = sbase + lay->qring + qs * lay->qslot_bytes;
        if (lane == 0) {
            int* hdr;
            if constexpr (Lay::UM) hdr = reinterpret_cast<int*>(smp + lay->qhdr + qs * QHDR_BYTES);
            else hdr = reinterpret_cast<int*>(smp + lay->qring + qs * lay->qslot_bytes);
            hdr[H_KIND] = kind; hdr[H_B] = b; hdr[H_G] = g; hdr[H_J] = j;
            hdr[H_T0] = t0; hdr[H_T1] = t1; hdr[H_DEST] = dest;
            if constexpr (Lay::UM) {
                hdr[H_MASK] = hw[0]; hdr[H_MASK_HI] = hw[1]; hdr[H_ONL] = hw[2]; hdr[H_ONL_HI] = hw[3];
                hdr[H_PASS] = pass;
            } else {
                hdr[H_F0] = hw[0]; hdr[H_F1] = hw[1]; hdr[H_MASK] = hw[2]; hdr[H_ONL] = hw[3];
            }
            hdr[H_L] = L;
            hdr[H_S] = S;
            if (kind == KIND_END) {
                mbar_arrive(rg.qfull + 8 * qs);
            } else if constexpr (Lay::UM) {
                // the R = Tq G query rows of kv head g land as R rows of 128 bytes per 64-wide
                // half of d (128-byte swizzle): row rr = i G + h is head g G + h of query token i
                const uint32_t bytes = (uint32_t)A.R * 128u;
                mbar_arrive_expect_tx(rg.qfull + 8 * qs, bytes * (uint32_t)HALVES);
#pragma unroll
                for (int hv = 0; hv < HALVES; ++hv)
                    tma_load_4d(slot + hv * lay->qhalf_bytes, tmQ, hv * 64, g * A.G, 0, b, rg.qfull + 8 * qs);
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
    // distinct), and the flag bytes split by split. With K > 0 the cut is made in a stream where
    // K phantom tiles follow each unit (T counts them; unit u's tiles start at W_u + K u): a part
    // that holds a run boundary, which costs the CTA about K tiles' time, takes K tiles fewer. A
    // phantom position starts the next unit.
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
        struct Seg { int b, g, kvh, j, t0, t1, L, ntile, dest; };
        const int nseq = A.B;
        int cb = 0, cgrp = 0;
        // The run at virtual tile v (moved past phantoms to the next unit's first tile); false
        // once the part holds no more real tiles. (K is 0 outside the tcgen05 build.)
        auto seg_at = [&](long long& v, Seg& s) -> bool {
            const int K = Lay::UM ? this->K : 0;
            for (;;) {
                if (v >= te) return false;
                long long vg = v;                    // virtual tile within the row group
                int grp = 0;
                if constexpr (RG) {
                    const long long TG = (long long)A.Hkv * (tplan[A.B] + (long long)K * A.B);
                    grp = (int)(v / TG);
                    vg = v - grp * TG;
                    if (grp != cgrp) { cgrp = grp; cb = 0; }
                }
                while ((long long)A.Hkv * (tplan[cb + 1] + (long long)K * (cb + 1)) <= vg) ++cb;
                const int ntb = tplan[cb + 1] - tplan[cb];
                const int r = (int)(vg - (long long)A.Hkv * (tplan[cb] + (long long)K * cb));
                const int kvh = r / (ntb + K);
                const int k = r - kvh * (ntb + K);   // tile of sequence cb, kv head kvh
                if (Lay::UM && k >= ntb) {           // a phantom: the next unit's first tile
                    v += ntb + K - k;
                    continue;
                }
                s.b = cb;
                s.g = RG ? kvh * A.NRG + grp : kvh;
                s.kvh = kvh;
                // the run: tiles k .. kend - 1 of the sequence's ntb (split j has tiles j TS .. j TS +
                // TS - 1, the last split fewer), tokens t0 .. t1
                const int kend = (int)min((long long)ntb, k + (te - v));
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
                return true;
            }
        };
        Seg cur, nxt;
        long long t = tb;
        if (!seg_at(t, cur)) return true;            // phantoms only
        int cur_ent = PAGED ? window_entry(cur.b, cur.t0, cur.L) : -1;
        for (;;) {
            long long tn = t + cur.ntile;
            // Whether a real tile remains: a run that ends before te ends at its unit's last tile,
            // and the next unit (past K phantoms) is the sequence's next kv head, which has tiles,
            // or the next sequence's first, which may have none. The look ahead leaves the
            // sequence cursor where it was: the walk from tn starts inside this sequence.
            bool last = tn >= te;
            if (Lay::UM && !last && K > 0) {
                if (te <= tn + K) {
                    last = true;
                } else if (cur.kvh + 1 >= A.Hkv) {
                    const int cb_keep = cb, cgrp_keep = cgrp;
                    long long v = tn;
                    Seg probe;
                    last = !seg_at(v, probe);
                    cb = cb_keep;
                    cgrp = cgrp_keep;
                }
            }
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
            // tcgen05 build, forced online softmax: the segment's row maxima first
            if constexpr (Lay::UM)
                if (A.mode == FDPP_MODE_FORCE_ONLINE &&
                    !emit<D, PAGED>(KIND_OWN, cur.b, cur.g, cur.j, cur.t0, cur.t1, cur.L, cur.dest, zero4,
                                    PAGED ? cur.t0 / A.block_size : -(1 << 30), cur_ent, nullptr, !had_own,
                                    PASS_MAX))
                    return false;
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
            if constexpr (Lay::UM)
                if (A.mode == FDPP_MODE_FORCE_ONLINE &&
                    !emit<D, PAGED>(KIND_OWN, b, g, j, t0, t1, L, -1, zero4, -(1 << 30), -1, nullptr, !had_own,
                                    PASS_MAX))
                    return false;
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
        // The cut stream (tcgen05 build): the real tiles and K phantoms after each unit. None where
        // the equal cut already ends parts at unit boundaries only (units of equal length, U
        // dividing P). The mma.sync builds cut the real tiles (their run boundaries cost little).
        const long long U = (long long)A.NRG * A.B * A.Hkv;      // units (runs' heads)
        const int P = (in_smem && T > 0 && T + (Lay::UM ? (long long)A.seg_tiles * U : 0ll) < (1ll << 31))
                          ? (int)min(min((long long)gridDim.x, T), (long long)TC_MAX_PARTS) : 0;
        if constexpr (Lay::UM) {
            bool eq = true;
            if (in_smem)
                for (int b = lane; b < A.B; b += 32) eq = eq && tplan[b + 1] - tplan[b] == tplan[1] - tplan[0];
            eq = __all_sync(0xffffffffu, eq);
            K = (eq && P > 0 && P % (int)U == 0) ? 0 : A.seg_tiles;
        }
        const long long TV = T + (long long)K * U;
        if (blockIdx.x == 0 && lane == 0) {
            A.hdr[HDR_PARTS] = P;
            A.hdr[HDR_TILES] = P > 0 ? (int)TV : 0;
            A.hdr[HDR_SEGK] = K;
        }
        bool had_own = false;
        const bool ok = P > 0 ? run_parts<D, PAGED>(TV, P, had_own) : run_units<D, PAGED>(n_units, had_own);
        if (!ok) return;

        // The fallback lists. Only the tcgen05 build pushes (the mma.sync builds finish an
        // out-of-window row-split in place), and there every CTA that pushed drains the lists after
        // its push, so no entry is left behind; a CTA that pushed nothing helps only if entries
        // were waiting when its last own tiles had been issued (read now, while they stream).
        // The consumers push this CTA's flagged segments (misc[1]) before they report the own
        // work done. The list is REDO_NLISTS lists, CTA c pushing to list c % REDO_NLISTS: a CTA
        // drains its own list first, then the others in turn, so that few CTAs contend for one
        // list's claim word.
        if (Lay::UM && A.mode == FDPP_MODE_NORMAL) {
            bool help = false;
            if (lane < REDO_NLISTS) {
                const unsigned long long both = ld_relaxed_gpu_u64(
                    reinterpret_cast<const unsigned long long*>(&A.hdr[HDR_REDO_LISTS + 2 * lane]));
                help = (int)(unsigned)(both & 0xffffffffull) > (int)(unsigned)(both >> 32);
            }
            help = __any_sync(0xffffffffu, help);
            if (had_own && !ring_wait(rg.own_done, 0u, misc, A)) return;
            help = help || misc[1] != 0;
            while (help) {
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
                            if constexpr (Lay::UM) ent[3] = tnt;
                            else ent[3] = (long long)taint;
                            st_release_gpu(ent, ((long long)(rg_ * A.max_splits + pe / S) << 32) |
                                                    (long long)(unsigned)(rb + 1));
                        }
                    }
                }
                if constexpr (Lay::UM) {
                    // tcgen05 build: a unit holds all R <= 64 rows (64-bit masks); a piece with
                    // rows to recompute online is streamed twice, for their maxima and then for
                    // the sums in that frame
                    for (int tp0 = st0; tp0 < st1_own;) {
                        const int rj = tp0 / S;
                        const int tp1 = min((rj + 1) * S, st1_own);
                        const int dp = (tp0 == st0 && dest >= 0 && tp0 != rj * S) ? dest : -1;
                        unsigned onl[2] = {0u, 0u};
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int rr = lane + 32 * hf;
                            bool o = false;
                            if (rr < A.R && ((tnt >> rr) & 1ll)) {
                                const unsigned f = dp < 0 ? __ldcg(A.flags + unit_row_slot(A, rb, rkvh, rr, rj))
                                                          : __ldcg(A.xf + (long long)dp * A.R + rr);
                                o = (f & FDPP_FLAG_OUT) != 0u;
                            }
                            onl[hf] = __ballot_sync(0xffffffffu, o);
                        }
                        const int hw[4] = {(int)(unsigned)tnt, (int)(unsigned)(tnt >> 32), (int)onl[0], (int)onl[1]};
                        if ((onl[0] | onl[1]) != 0u &&
                            !emit<D, PAGED>(KIND_REDO, rb, rg_, rj, tp0, tp1, L, dp, hw, -(1 << 30), -1, nullptr,
                                            false, PASS_MAX))
                            return;
                        if (!emit<D, PAGED>(KIND_REDO, rb, rg_, rj, tp0, tp1, L, dp, hw)) return;
                        tp0 = tp1;
                    }
                } else {
                    const int rrow = RG ? (rg_ - rkvh * A.NRG) * TC_MAX_GROUP + lane : lane;
                    const int rows = RG ? A.Rg : A.R;        // rows of a unit (run-slot stride)
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
        }
        const int zeros[4] = {0, 0, 0, 0};
        emit<D, PAGED>(KIND_END, 0, 0, 0, 0, 0, 0, -1, zeros);
    }
};

}  // namespace
}  // namespace fdpp
