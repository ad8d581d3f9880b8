// split_um.cu -- per-split kernel for many query rows per kv head (a prefill chunk, a
// speculative-decoding step, a wide GQA group: up to 64 rows) with bf16 K/V and d = 128, on the
// tcgen05 tensor cores with the accumulators in tensor memory. combine.cu then sums the partials.
//
// What it computes is what split_tc.cu computes (opt.ai.kr "FlashDecoding++ async softmax --
// theory", s1 and s3): for one unit (sequence b, kv head g, split j) and its R = Tq G query rows,
//     s = scale <q_r, k_t>, p = exp(s - phi_r), l = sum p, o = sum p v_t      (fast pass)
// in the unified-max frame, each score tested against lo <= s - phi <= hi, and a segment with a
// row outside the window goes on the device-wide fallback list, whose pieces are computed again
// in the rows' own max frame. Query token i of a sequence with L keys sees the keys
// t < L - Tq + 1 + i. The partial of a segment (a part's share of one (sequence, kv head), see
// split_tc_common.cuh) goes to a run slot or to the split's own slot, exactly as in split_tc.cu,
// with all R rows of the kv head in one unit.
//
// Why another kernel. At R = 64 every 512 bytes of K and V read from HBM carry 49,152 FLOP
// (q.K^T, and P.V with P split into bf16 hi and lo parts): 0.64 PFLOP/s at the copy rate, beyond
// what m16n8k16 mma.sync issue keeps up with, well inside the tcgen05 rate.
//
// How. One CTA per SM, eleven warps:
//   warp 8    the producer of split_tc_common.cuh: split plan, tile-balanced parts, 64-token K/V
//             tiles by TMA into a ring of stages (128-byte swizzle), fallback-list drain. The
//             unit's R query rows arrive by one 4-D TMA load per 64-wide half of d.
//   warps 9, 10  one thread each issues MMAs (warp 9 also owns the tensor memory):
//               warp 9:  S^T = K Q^T      M = 64 tokens, N = NP (R rounded up to 16, 32 or 64),
//                                         K = d, for every tile;
//               warp 10: O^T += V^T P^T   M = d = 128, N = 2 NP, K = 64 tokens: P's bf16 hi
//                                         parts are rows 0 .. NP - 1 of the B operand and its lo
//                                         parts (what hi leaves out, ~16 mantissa bits together)
//                                         rows NP .. 2 NP - 1, so one MMA per 16 tokens reads
//                                         V^T once for both;
//             V^T is read MN-major straight from the TMA-landed V tile. S^T has UM_NSB buffers in
//             tensor memory (used in turn by the tiles), O^T two (segment parity). Two issuing warps keep
//             either's waits (a stage, an S^T buffer, a P buffer) from holding the other's MMAs
//             back, and descriptors are built once and offset per MMA: the issuing threads'
//             own work, not the tensor core, set the pace before. tcgen05.commit arrives on
//             mbarriers that release the K/V stage, the P buffer and the Q slot and wake the
//             softmax warps.
//   warps 0-7 softmax, two warps per tensor-memory lane quadrant: warp w holds tokens
//             16 (w % 4) .. + 15 of a tile (the 64-row accumulator puts token t in lane
//             (t mod 16) + 32 floor(t / 16)) and rows NP/2 floor(w / 4) .. + NP/2 - 1; tcgen05.ld
//             16x256b gives each thread 2 tokens x NP/8 rows in the mma.sync fragment order, so
//             stmatrix.trans writes P^T as the K-major swizzled B operand, 16 bytes per row.
//             The window test keeps per row and split the max, min and a NaN marker of q.k, and
//             classifies once per split (scale > 0 and the rounding of s = scale q.k and of
//             s - phi are monotone, so this is exactly the per-score test). At a segment's end
//             each thread reads one d of O^T (hi plus lo) and writes it for its warp's rows.
// Rows recomputed with online softmax (fallback pieces, and every segment in forced-online mode)
// are streamed twice: first for the rows' maxima M, then for the sums in the frame M (the
// accumulator in tensor memory is never rescaled). The result is the online softmax's up to
// rounding.
// Every wait is bounded; a wait that runs out sets FDPP_ERRBIT_TIMEOUT, the CTA lets its
// copies and MMAs land, frees its tensor memory and exits.
#include "split_tc_common.cuh"
#include "tcgen05.cuh"

namespace fdpp {
namespace {

constexpr int UM_D = 128;                 // head dim of this kernel
constexpr int UM_NSW = 8;                 // softmax warps: two per tensor-memory lane quadrant
constexpr int UM_PROD_WARP = UM_NSW;      // then the producer
constexpr int UM_MMA_WARP = UM_NSW + 1;   // the q.K^T warp (owns the tensor memory)
constexpr int UM_PV_WARP = UM_NSW + 2;    // the P.V warp
constexpr int UM_THREADS = (UM_NSW + 3) * 32;
constexpr int UM_FSLOTS = 8;              // window decisions of split pieces in flight
constexpr int UM_MAX_ROWS = 64;
constexpr int UM_NBARS = 23;              // barriers besides the stage ring's
// P^T buffers. One: the softmax warps compute a tile's P while the P.V of the tile before runs and
// wait only to store it; the shared memory of a second goes to another K/V stage instead.
constexpr int UM_NPB = 1;
// S^T buffers in tensor memory (q.K^T runs up to this many tiles ahead of the softmax), then the
// two O^T buffers: UM_NSB NP + 4 NP columns.
constexpr int UM_NSB = 3;

// Shared-memory layout (byte offsets from a 1024-byte aligned base).
//   stages   nstage x (K tile, V tile), each two [64 token][64 d] boxes of 128-byte rows
//   qring    2 slots x two [NP row][64 d] halves (the B operand of S^T)
//   pbuf     UM_NPB buffers x (hi, lo) [NP row][64 token] (the B operand of O^T), used in turn by
//            the tiles that have a P.V
//   qhdr     2 segment headers
//   fsw/fcnt per split piece in flight: each lane quadrant's flag nibble of every row (the two
//            warps of a quadrant hold different rows), arrival count
//   taint    the rows with a score outside the window, per segment parity (64-bit)
//   xl/xm    per lane quadrant and row: the l sum of a segment (per segment parity), the max of
//            a max pass
//   rowoff   per row n = i G + h: its offset (i Hq + h) max_splits in the split-slot order
struct UmLayout {
    static constexpr bool UM = true;
    int stage_bytes, kv_bytes, qslot_bytes, qhalf_bytes, p_bytes;
    int stages, qring, pbuf, qhdr, fsw, fcnt, taint, xl, xm, rowoff, plan, bars, misc, tslot, total;

    __host__ __device__ static constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

    __host__ __device__ UmLayout(int NP, int nstage, int B)
        : stage_bytes(2 * TILE * UM_D * 2), kv_bytes(TILE * UM_D * 2), qslot_bytes(2 * NP * 128),
          qhalf_bytes(NP * 128), p_bytes(NP * 128), stages(0), qring(0), pbuf(0), qhdr(0), fsw(0),
          fcnt(0), taint(0), xl(0), xm(0), rowoff(0), plan(0), bars(0), misc(0), tslot(0), total(0)
    {
        qring = stages + nstage * stage_bytes;
        pbuf = qring + 2 * qslot_bytes;
        qhdr = pbuf + UM_NPB * 2 * p_bytes;
        fsw = qhdr + 2 * QHDR_BYTES;
        fcnt = fsw + UM_FSLOTS * 4 * UM_MAX_ROWS;
        taint = fcnt + UM_FSLOTS * 4;
        xl = taint + 2 * 8;
        xm = xl + 2 * 4 * UM_MAX_ROWS * 4;
        rowoff = xm + 4 * UM_MAX_ROWS * 4;
        plan = rowoff + UM_MAX_ROWS * 8;
        const int plan_ints = (B <= PLAN_SMEM_MAX_B ? 2 * B + 1 : 0) + 1;
        bars = round_up(plan + plan_ints * 4, 8);
        misc = bars + (2 * nstage + UM_NBARS) * 8;
        tslot = misc + 16;
        total = tslot + 16;
    }
};

// The barriers besides the producer's ring (shared addresses). Arrival counts: sfull, pfree and
// ofull one commit, drain one commit from each MMA warp; sfree, pready, ofree and wsync the
// softmax warps.
struct UmBars {
    uint32_t sfull, sfree;     // [UM_NSB] S^T buffer written / read out (used in turn by the tiles)
    uint32_t pready, pfree;    // [UM_NPB] P^T buffer written / consumed by its MMAs (used in
                               //     turn by the tiles that have a P.V: max passes have none)
    uint32_t ofull, ofree;     // [2] O^T buffer complete / read out (segment parity)
    uint32_t drain;            // every MMA of the CTA has completed
    uint32_t wsync;            // the softmax warps meet (a bounded barrier among them)
};

// hi = bf16(p0, p1) rounded to nearest, lo = bf16 of what hi leaves out (p ~ hi + lo to ~16 bits)
__device__ __forceinline__ void split_bf16x2(float p0, float p1, uint32_t& hi, uint32_t& lo)
{
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
    hi = *reinterpret_cast<const uint32_t*>(&h2);
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16x2(p0 - h0, p1 - h1);
}

// 2^x (ex2.approx, flushing results below 2^-126 to zero)
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two ring waits whose barriers usually have completed already: both are tested at once (their
// latencies overlap), and only a phase still open takes the bounded wait.
__device__ __forceinline__ bool ring_wait2(uint32_t bar1, uint32_t par1, uint32_t bar2, uint32_t par2,
                                           volatile int* misc, const KernelArgs& a)
{
    const bool d1 = mbar_try_wait(bar1, par1);
    const bool d2 = mbar_try_wait(bar2, par2);
    if (__all_sync(0xffffffffu, d1 && d2)) return true;
    return ring_wait(bar1, par1, misc, a) && ring_wait(bar2, par2, misc, a);
}

__device__ __forceinline__ float max_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// ------------------------------------------------------------------------------------------
// MMA warps: one issues q.K^T for every tile, the other P.V for every tile that has one, so that
// neither's waits hold the other's MMAs back
// ------------------------------------------------------------------------------------------
// Descriptors are built once per stage, Q slot and P buffer; an MMA adds a constant to the
// start-address field (addr / 16 in its low 14 bits; shared addresses stay below 256 KB, so the
// field never carries).
struct UmDescs {
    uint64_t k0, v0, q0, p0;
    uint32_t stage16, qslot16, qhalf16, pbuf16;

    __device__ __forceinline__ UmDescs(const UmLayout& lay, uint32_t sbase)
        : k0(sw128_kmajor_desc(sbase + lay.stages)),
          v0(sw128_mnmajor_desc(sbase + lay.stages + lay.kv_bytes, TILE * 128, 1024)),
          q0(sw128_kmajor_desc(sbase + lay.qring)), p0(sw128_kmajor_desc(sbase + lay.pbuf)),
          stage16((uint32_t)lay.stage_bytes >> 4), qslot16((uint32_t)lay.qslot_bytes >> 4),
          qhalf16((uint32_t)lay.qhalf_bytes >> 4), pbuf16((uint32_t)(2 * lay.p_bytes) >> 4)
    {
    }
};

// Every MMA the calling thread issued has landed (before the tensor memory and the stages are
// released); the drain barrier takes one commit from each MMA warp.
__device__ __forceinline__ void mma_drain(const KernelArgs& a, const UmBars& ub, volatile int* misc)
{
    const int lane = threadIdx.x & 31;
    if (lane == 0) umma_commit(ub.drain);
    __syncwarp();
    if (!mbar_wait(ub.drain, 0u) && lane == 0) {
        misc[0] = 1;
        set_error(a, FDPP_ERRBIT_TIMEOUT);
    }
    __syncwarp();
}

// q.K^T of every tile: S^T = K Q^T, M = 64 tokens, N = NP rows, into the S^T buffer of the tile's
// parity once the softmax warps have read the tile two before out of it. The stage goes back to
// the producer here for a max pass (no P.V follows); the Q slot after a segment's last tile.
template <int NP>
__device__ __forceinline__ void mma_s_warp(const KernelArgs& a, const UmLayout& lay, const uint8_t* sm,
                                           uint32_t sbase, const Ring& rg, const UmBars& ub, uint32_t tmem,
                                           volatile int* misc)
{
    const int lane = threadIdx.x & 31;
    constexpr uint32_t IDESC_S = umma_idesc_bf16(64, NP, false);
    const UmDescs ds(lay, sbase);
    uint32_t stage = 0, phase = 0, qiter = 0, it = 0;
    for (;;) {
        const uint32_t qs = qiter & 1u;
        if (!ring_wait(rg.qfull + 8 * qs, (qiter >> 1) & 1u, misc, a)) break;
        const int* hdr = reinterpret_cast<const int*>(sm + lay.qhdr + qs * QHDR_BYTES);
        const int kind = hdr[H_KIND];
        if (kind == KIND_END) break;
        const int t0 = hdr[H_T0], t1 = hdr[H_T1], S = hdr[H_S];
        const bool maxpass = hdr[H_PASS] == PASS_MAX;
        ++qiter;
        const uint64_t qd = ds.q0 + qs * ds.qslot16;
        int tt = t0, se = (t0 / S + 1) * S;
        bool ok = true;
        while (tt < t1) {
            const int tend = min(min(tt + TILE, se), t1);
            const uint32_t sb = it % UM_NSB, suse = it / UM_NSB;
            if (!ring_wait2(rg.full + 8 * stage, phase, ub.sfree + 8 * sb, (suse & 1u) ^ 1u, misc, a)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint64_t kd = ds.k0 + stage * ds.stage16;
                const uint32_t sd = tmem + sb * NP;
#pragma unroll
                for (int ks = 0; ks < UM_D / 16; ++ks) {
                    // K and Q^T: K-major, 32 bytes per 16 of d, the second half of d in its own box
                    umma_bf16(sd, kd + (ks >> 2) * ((TILE * 128) >> 4) + (ks & 3) * (32 >> 4),
                              qd + (ks >> 2) * ds.qhalf16 + (ks & 3) * (32 >> 4), IDESC_S, ks > 0 ? 1u : 0u);
                }
                umma_commit(ub.sfull + 8 * sb);
                if (tend == t1) umma_commit(rg.qempty + 8 * qs);   // the segment's Q slot is read
                if (maxpass) umma_commit(rg.empty + 8 * stage);
            }
            __syncwarp();
            ++it;
            if (++stage == (uint32_t)rg.nstage) { stage = 0; phase ^= 1u; }
            tt = tend;
            if (tt == se) se += S;
        }
        if (!ok) break;
    }
    mma_drain(a, ub, misc);
}

// P.V of every tile of a sums pass: O^T += V^T P^T, M = d, N = 2 NP (P's bf16 hi parts are the
// B operand's rows 0 .. NP - 1, its lo parts rows NP .. 2 NP - 1, so one MMA per 16 tokens reads
// V^T once for both), into the O^T buffer of the segment's parity. Commits release the P buffer
// and the stage, and after a segment's last tile wake the epilogue.
template <int NP>
__device__ __forceinline__ void mma_o_warp(const KernelArgs& a, const UmLayout& lay, const uint8_t* sm,
                                           uint32_t sbase, const Ring& rg, const UmBars& ub, uint32_t tmem,
                                           volatile int* misc)
{
    const int lane = threadIdx.x & 31;
    constexpr uint32_t IDESC_O = umma_idesc_bf16(128, 2 * NP, true);
    const UmDescs ds(lay, sbase);
    uint32_t stage = 0, qiter = 0, pit = 0, obn = 0;
    for (;;) {
        const uint32_t qs = qiter & 1u;
        if (!ring_wait(rg.qfull + 8 * qs, (qiter >> 1) & 1u, misc, a)) break;
        const int* hdr = reinterpret_cast<const int*>(sm + lay.qhdr + qs * QHDR_BYTES);
        const int kind = hdr[H_KIND];
        if (kind == KIND_END) break;
        const int t0 = hdr[H_T0], t1 = hdr[H_T1], S = hdr[H_S];
        const bool maxpass = hdr[H_PASS] == PASS_MAX;
        __syncwarp();
        if (lane == 0) mbar_arrive(rg.qempty + 8 * qs);    // header read
        ++qiter;
        int tt = t0, se = (t0 / S + 1) * S;
        bool ok = true, first = true;
        const uint32_t ob = obn & 1u;
        while (tt < t1) {
            const int tend = min(min(tt + TILE, se), t1);
            if (!maxpass) {
                const uint32_t pb = pit % UM_NPB, puse = pit / UM_NPB;
                if (!ring_wait(ub.pready + 8 * pb, puse & 1u, misc, a) ||
                    (first && !ring_wait(ub.ofree + 8 * ob, ((obn >> 1) & 1u) ^ 1u, misc, a))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t vd = ds.v0 + stage * ds.stage16;
                    const uint64_t pd = ds.p0 + pb * ds.pbuf16;
                    const uint32_t od = tmem + UM_NSB * NP + ob * (2 * NP);
#pragma unroll
                    for (int kt = 0; kt < TILE / 16; ++kt) {
                        // V^T: d on M (two 64-wide halves TILE * 128 bytes apart), 16 tokens
                        // (2048 bytes) per k-step; P^T: 32 bytes per 16 tokens
                        umma_bf16(od, vd + kt * (2048 >> 4), pd + kt * (32 >> 4), IDESC_O,
                                  (first && kt == 0) ? 0u : 1u);
                    }
                    umma_commit(ub.pfree + 8 * pb);
                    umma_commit(rg.empty + 8 * stage);
                    if (tend == t1) umma_commit(ub.ofull + 8 * ob);
                }
                __syncwarp();
                ++pit;
                first = false;
            }
            if (++stage == (uint32_t)rg.nstage) stage = 0;
            tt = tend;
            if (tt == se) se += S;
        }
        if (!ok) break;
        if (!maxpass) ++obn;
    }
    mma_drain(a, ub, misc);
}

// ------------------------------------------------------------------------------------------
// softmax warps
// ------------------------------------------------------------------------------------------
// Softmax warp w: tensor-memory quadrant w % 4 (tokens 16 (w % 4) .. + 15 of a tile), row half
// w / 4 (rows NP/2 (w / 4) .. + NP/2 - 1). A thread holds NPC = NP / 8 rows of 2 tokens.
template <int NP>
__device__ __forceinline__ void softmax_warps(const KernelArgs& a, const UmLayout& lay, uint8_t* sm,
                                              uint32_t sbase, const Ring& rg, const UmBars& ub,
                                              uint32_t tmem, volatile int* misc)
{
    constexpr int NGW = NP / 16;         // 8-column groups of S^T per warp
    constexpr int NV = 4 * NGW;          // S^T values per thread and tile
    constexpr int NPC = 2 * NGW;         // rows (columns) per thread
    constexpr float LOG2E = 1.4426950408889634f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qw = warp & 3, hw = warp >> 2;
    const int q = lane & 3, a4 = lane >> 2;
    const int tokA = qw * 16 + a4;       // this thread's tokens in a tile: tokA, tokA + 8
    const int g0 = hw * NGW;             // first 8-column group of this warp
    const uint32_t lane_base = (uint32_t)(32 * qw) << 16;
    uint8_t* fsw = sm + lay.fsw;
    int* fcnt = reinterpret_cast<int*>(sm + lay.fcnt);
    unsigned long long* taint_s = reinterpret_cast<unsigned long long*>(sm + lay.taint);
    float* xl_s = reinterpret_cast<float*>(sm + lay.xl);
    float* xm_s = reinterpret_cast<float*>(sm + lay.xm);
    const long long* rowoff_s = reinterpret_cast<const long long*>(sm + lay.rowoff);
    uint32_t stage = 0, phase = 0, qiter = 0, it = 0, pit = 0, obn = 0, portion = 0, un = 0, nsync = 0;
    const int R = a.R;
    const float c_exp = a.scale * LOG2E;          // p = 2^(acc scale log2e - frame log2e)
    // row n of column c of this thread
    auto row_of = [&](int c) { return 8 * (g0 + (c >> 1)) + 2 * q + (c & 1); };
    // the softmax warps meet (bounded: a warp that gave up lets the others time out)
    auto warps_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(ub.wsync);
        const bool ok = ring_wait(ub.wsync, nsync & 1u, misc, a);
        ++nsync;
        return ok;
    };

    for (;;) {
        // ---- next segment ----
        const uint32_t qs = qiter & 1u;
        if (!ring_wait(rg.qfull + 8 * qs, (qiter >> 1) & 1u, misc, a)) return;
        const int* hdr = reinterpret_cast<const int*>(sm + lay.qhdr + qs * QHDR_BYTES);
        const int kind = hdr[H_KIND];
        if (kind == KIND_END) return;
        const int b = hdr[H_B], g = hdr[H_G], j0 = hdr[H_J];
        const int t0 = hdr[H_T0], t1 = hdr[H_T1], dest = hdr[H_DEST], L = hdr[H_L], S = hdr[H_S];
        const bool maxpass = hdr[H_PASS] == PASS_MAX;
        const unsigned long long redo_mask =
            (unsigned long long)(unsigned)hdr[H_MASK] | ((unsigned long long)(unsigned)hdr[H_MASK_HI] << 32);
        const unsigned long long onl_mask =
            (unsigned long long)(unsigned)hdr[H_ONL] | ((unsigned long long)(unsigned)hdr[H_ONL_HI] << 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(rg.qempty + 8 * qs);
        ++qiter;
        const bool redo = kind == KIND_REDO;
        const bool force_online = a.mode == FDPP_MODE_FORCE_ONLINE;
        const uint32_t upar = un & 1u;
        // causal limit of the query token with the fewest keys (row 0): a tile wholly below it
        // needs no per-row mask
        const int lim0 = key_limit(a, L, 0);
        // split j0's slot of row 0; row n of split j is at slot0 + (j - j0) + rowoff_s[n]
        const long long slot0 = (((long long)b * a.Tq) * a.Hq + (long long)g * a.G) * a.max_splits + j0;

        // Per row of this thread: the frame of the sums (phi, or the max pass's M) times log2 e,
        // the causal key limit (absolute token index), the window trackers on the raw q.k
        // (scale > 0 and each rounding is monotone, so the max, min and NaN of q.k decide the
        // test of every s - phi exactly), and the l sum.
        float frl[NPC], amax[NPC], amin[NPC], anan[NPC], lsum[NPC];
        int lim[NPC];
#pragma unroll
        for (int c = 0; c < NPC; ++c) {
            const int n = row_of(c);
            const bool live = n < R;
            lim[c] = live ? key_limit(a, L, n / a.G) : 0;
            const bool onl = !maxpass && ((redo && ((onl_mask >> n) & 1ull)) || (!redo && force_online));
            float fr = live ? phi_of(a, g * a.G + n % a.G) : a.phi;
            if (onl) {
                fr = xm_s[n];
#pragma unroll
                for (int w = 1; w < 4; ++w) fr = fmaxf(fr, xm_s[w * UM_MAX_ROWS + n]);
            }
            frl[c] = fr * LOG2E;
            amax[c] = -INFINITY;
            amin[c] = INFINITY;
            anan[c] = -INFINITY;
            lsum[c] = 0.f;
        }

        // Window decisions of split pieces. A piece's trackers give each row's nibble (ORed over
        // the warp's tokens; the trackers restart), which the warp puts in the piece's slot for
        // its quadrant; a row is out when any quadrant's nibble says so.
        auto piece_nibbles = [&]() -> unsigned {
            unsigned nb = 0u;
#pragma unroll
            for (int c = 0; c < NPC; ++c) {
                const int n = row_of(c);
                const float ph = n < R ? phi_of(a, g * a.G + n % a.G) : a.phi;
                unsigned f = 0u;
                if (__fsub_rn(__fmul_rn(amax[c], a.scale), ph) > a.hi) f |= FDPP_FLAG_OUT | FDPP_FLAG_ABOVE;
                if (__fsub_rn(__fmul_rn(amin[c], a.scale), ph) < a.lo) f |= FDPP_FLAG_OUT | FDPP_FLAG_BELOW;
                if (anan[c] != anan[c]) f |= FDPP_FLAG_OUT | FDPP_FLAG_NAN;
                nb |= f << (4 * c);
                amax[c] = -INFINITY;
                amin[c] = INFINITY;
                anan[c] = -INFINITY;
            }
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) nb |= __shfl_xor_sync(0xffffffffu, nb, sh);
            return nb;
        };
        auto publish = [&](uint32_t ks, unsigned nb) {
            uint8_t* mine = fsw + (ks * 4 + qw) * UM_MAX_ROWS;
            if (lane < 4) {
#pragma unroll
                for (int c = 0; c < NPC; ++c) mine[row_of(c)] = (uint8_t)((nb >> (4 * c)) & 15u);
            }
        };
        // The out rows of slot ks once every quadrant's nibbles are in; `write`: this warp also
        // writes the piece's flag bytes (split jp's own, or the run slot's edge byte for a first
        // piece that starts inside a split).
        auto piece_rows = [&](uint32_t ks, int jp, bool first_piece, bool write) -> unsigned long long {
            const uint8_t* all = fsw + ks * 4 * UM_MAX_ROWS;
            unsigned long long out_rows = 0ull;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int n = lane + 32 * hf;
                bool out = false;
                if (n < R && n < NP) {
                    const unsigned f = all[n] | all[UM_MAX_ROWS + n] | all[2 * UM_MAX_ROWS + n] |
                                       all[3 * UM_MAX_ROWS + n];
                    out = (f & FDPP_FLAG_OUT) != 0u;
                    if (write) {
                        const uint8_t fb = (uint8_t)(f | (force_online ? FDPP_FLAG_RECOMPUTED : 0u));
                        if (first_piece && dest >= 0 && t0 != jp * S)
                            a.xf[(long long)dest * R + n] = fb;
                        else
                            a.flags[slot0 + (jp - j0) + rowoff_s[n]] = fb;
                    }
                }
                out_rows |= (unsigned long long)__ballot_sync(0xffffffffu, out) << (32 * hf);
            }
            return out_rows;
        };
        // A piece that ends inside the segment: the warp that arrives last (a shared count) decides
        // it and marks the segment's taint. The segment's last piece is decided by every warp after
        // the epilogue's barrier instead.
        auto finish_piece = [&](int jp, bool first_piece) {
            const unsigned nb = piece_nibbles();
            const uint32_t ks = portion++ & (uint32_t)(UM_FSLOTS - 1);
            publish(ks, nb);
            __syncwarp();
            int old = 0;
            if (lane == 0) {
                __threadfence_block();
                old = atomicAdd(&fcnt[ks], 1);
            }
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old != UM_NSW - 1) return;
            __threadfence_block();
            const unsigned long long out_rows = piece_rows(ks, jp, first_piece, true);
            if (lane == 0) {
                fcnt[ks] = 0;
                if (out_rows) atomicOr(&taint_s[upar], out_rows);
            }
        };

        // ---- the segment's tiles ----
        int tt = t0, se = (t0 / S + 1) * S, jp = j0, last_jp = j0;
        bool first_piece = true, last_first = false;
        int last_ks = -1;
        while (tt < t1) {
            const int tend = min(min(tt + TILE, se), t1);
            const int nvalid = tend - tt;
            const uint32_t sb = it % UM_NSB, suse = it / UM_NSB;
            if (!ring_wait(ub.sfull + 8 * sb, suse & 1u, misc, a)) return;
            tc_fence_after();
            uint32_t v[NV];
            tmem_ld_16x256b<NGW>(tmem + sb * NP + lane_base + 8 * g0, v);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ub.sfree + 8 * sb);
            // every score of the tile counts: no ragged tail and every row sees every key
            const bool whole = nvalid == TILE && tt + TILE <= lim0;
            // element e: row column c = 2 (e / 4) + e % 2, token tokA + 8 ((e / 2) % 2)
            auto valid_at = [&](int e) {
                const int c = 2 * (e >> 2) + (e & 1);
                const int tok = tokA + 8 * ((e >> 1) & 1);
                return tok < nvalid && tt + tok < lim[c];
            };
            if (maxpass) {
                if (whole) {
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        const int c = 2 * (e >> 2) + (e & 1);
                        amax[c] = fmaxf(amax[c], __uint_as_float(v[e]));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        const int c = 2 * (e >> 2) + (e & 1);
                        amax[c] = fmaxf(amax[c], valid_at(e) ? __uint_as_float(v[e]) : -INFINITY);
                    }
                }
            } else {
                float p[NV];
                if (whole) {
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        const int c = 2 * (e >> 2) + (e & 1);
                        const float x = __uint_as_float(v[e]);
                        amax[c] = fmaxf(amax[c], x);
                        amin[c] = fminf(amin[c], x);
                        anan[c] = max_nan(anan[c], x);
                        p[e] = ex2_approx(fmaf(x, c_exp, -frl[c]));
                        lsum[c] += p[e];
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        const int c = 2 * (e >> 2) + (e & 1);
                        const float x = __uint_as_float(v[e]);
                        const bool ok = valid_at(e);
                        amax[c] = fmaxf(amax[c], ok ? x : -INFINITY);
                        amin[c] = fminf(amin[c], ok ? x : INFINITY);
                        anan[c] = max_nan(anan[c], ok ? x : -INFINITY);
                        p[e] = ok ? ex2_approx(fmaf(x, c_exp, -frl[c])) : 0.f;
                        lsum[c] += p[e];
                    }
                    // V rows past the valid tokens may hold anything (NaN included): zero them
                    // before the tensor core reads the tile (the stage has landed: its barrier
                    // is waited on); the first row half's warps take the quadrant's 16 rows
                    if (nvalid < TILE && hw == 0) {
                        if (!ring_wait(rg.full + 8 * stage, phase, misc, a)) return;
                        const int tok = qw * 16 + (lane & 15);
                        if (tok >= nvalid) {
                            uint4* row = reinterpret_cast<uint4*>(sm + lay.stages + stage * lay.stage_bytes +
                                                                  lay.kv_bytes + (lane >> 4) * TILE * 128 + tok * 128);
#pragma unroll
                            for (int i = 0; i < 8; ++i) row[i] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                // P^T (hi, lo) into the next P buffer, once the MMAs that last read it are done:
                // stored row n holds the tile's 64 tokens (16-byte chunk k = tokens 8k .. 8k + 7
                // at chunk k ^ (n % 8), 128-byte swizzle), 8-row groups 1024 bytes apart
                const uint32_t pbi = pit % UM_NPB, puse = pit / UM_NPB;
                if (!ring_wait(ub.pfree + 8 * pbi, (puse & 1u) ^ 1u, misc, a)) return;
                const uint32_t pb = sbase + lay.pbuf + pbi * 2 * lay.p_bytes;
                {
                    const int jm = lane >> 3, r = lane & 7;
                    if constexpr (NGW >= 2) {
#pragma unroll
                        for (int u = 0; u < NGW / 2; ++u) {
                            const int gg = g0 + 2 * u + (jm >> 1), th = jm & 1;
                            const uint32_t addr = pb + gg * 1024 + r * 128 + ((uint32_t)((2 * qw + th) ^ r) << 4);
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) split_bf16x2(p[8 * u + 2 * j], p[8 * u + 2 * j + 1], hi[j], lo[j]);
                            stmatrix_x4_trans(addr, hi[0], hi[1], hi[2], hi[3]);
                            stmatrix_x4_trans(addr + lay.p_bytes, lo[0], lo[1], lo[2], lo[3]);
                        }
                    } else {
                        // one group per warp: two matrices (the token halves), addresses from lanes 0-15
                        const int th = jm & 1;
                        const uint32_t addr = pb + g0 * 1024 + r * 128 + ((uint32_t)((2 * qw + th) ^ r) << 4);
                        uint32_t hi[2], lo[2];
#pragma unroll
                        for (int j = 0; j < 2; ++j) split_bf16x2(p[2 * j], p[2 * j + 1], hi[j], lo[j]);
                        stmatrix_x2_trans(addr, hi[0], hi[1]);
                        stmatrix_x2_trans(addr + lay.p_bytes, lo[0], lo[1]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(ub.pready + 8 * pbi);
                ++pit;
            }
            ++it;
            if (++stage == (uint32_t)rg.nstage) { stage = 0; phase ^= 1u; }
            tt = tend;
            if (tt == se || tt == t1) {            // a split piece ends here
                if (!maxpass && !redo) {
                    if (tt < t1) {
                        finish_piece(jp, first_piece);
                    } else {
                        last_ks = (int)(portion++ & (uint32_t)(UM_FSLOTS - 1));
                        publish((uint32_t)last_ks, piece_nibbles());
                        last_jp = jp;
                        last_first = first_piece;
                    }
                }
                first_piece = false;
                ++jp;
                se += S;
            }
        }

        if (maxpass) {
            // ---- the rows' maxima over the segment (scaled): per quadrant, read by every warp ----
#pragma unroll
            for (int c = 0; c < NPC; ++c) {
#pragma unroll
                for (int sh = 4; sh < 32; sh <<= 1) amax[c] = fmaxf(amax[c], __shfl_xor_sync(0xffffffffu, amax[c], sh));
            }
            if (lane < 4) {
#pragma unroll
                for (int c = 0; c < NPC; ++c) xm_s[qw * UM_MAX_ROWS + row_of(c)] = __fmul_rn(amax[c], a.scale);
            }
            if (!warps_sync()) return;
            continue;
        }

        // ---- epilogue: l of every row, then O^T out of tensor memory ----
#pragma unroll
        for (int c = 0; c < NPC; ++c) {
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) lsum[c] += __shfl_xor_sync(0xffffffffu, lsum[c], sh);
        }
        float* xl_p = xl_s + upar * 4 * UM_MAX_ROWS;     // by segment parity: no barrier before reuse
        if (lane < 4) {
#pragma unroll
            for (int c = 0; c < NPC; ++c) xl_p[qw * UM_MAX_ROWS + row_of(c)] = lsum[c];
        }
        // every warp's l, and every piece's window decisions, are in
        if (!warps_sync()) return;
        // the taint: the rows out of the window in any piece (the last one decided here, its flag
        // bytes written by the last warp). Every warp read the previous segment's taint word
        // before this barrier: it is cleared for the segment after this one.
        unsigned long long taint = 0ull;
        if (!redo) {
            taint = taint_s[upar];
            if (last_ks >= 0) taint |= piece_rows((uint32_t)last_ks, last_jp, last_first, warp == UM_NSW - 1);
        }
        if (warp == 0 && lane == 0) taint_s[upar ^ 1u] = 0ull;
        const unsigned long long write_mask = redo ? redo_mask : ~0ull;
        const bool refill = !redo && a.mode == FDPP_MODE_NORMAL;
        const unsigned long long zero_rows = refill ? taint : 0ull;
        const bool push = refill && taint != 0ull;
        const uint32_t ob = obn & 1u;
        if (!ring_wait(ub.ofull + 8 * ob, (obn >> 1) & 1u, misc, a)) return;
        ++obn;
        tc_fence_after();
        {
            // d = 32 (w % 4) + lane; the quadrant's two warps take a half of the 16-column chunks
            // each (NP = 16: the first warp the one chunk). All loads, then one wait.
            constexpr int NCH = NP / 16, CPW = NCH >= 2 ? NCH / 2 : 1;
            if (hw * CPW < NCH) {
                const int d = 32 * qw + lane;
                uint32_t oh[CPW][16], olo[CPW][16];
#pragma unroll
                for (int u = 0; u < CPW; ++u) {
                    const uint32_t col = UM_NSB * NP + ob * (2 * NP) + 16 * (hw * CPW + u);
                    tmem_ld16_async(tmem + col + lane_base, oh[u]);
                    tmem_ld16_async(tmem + col + NP + lane_base, olo[u]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < CPW; ++u) {
                    reg_fence16(oh[u]);
                    reg_fence16(olo[u]);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int n = 16 * (hw * CPW + u) + k;
                        if (n >= R || !((write_mask >> n) & 1ull)) continue;
                        const float o = __uint_as_float(oh[u][k]) + __uint_as_float(olo[u][k]);
                        float* orow = dest >= 0 ? a.xo + ((long long)dest * R + n) * UM_D
                                                : a.o_part + (slot0 + rowoff_s[n]) * UM_D;
                        orow[d] = ((zero_rows >> n) & 1ull) ? 0.f : o;
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ub.ofree + 8 * ob);
        // l and m: warp w writes rows 8 w .. 8 w + 7
        if (lane < 8) {
            const int n = 8 * warp + lane;
            if (n < R && n < NP && ((write_mask >> n) & 1ull)) {
                const float lam = ((xl_p[n] + xl_p[UM_MAX_ROWS + n]) + xl_p[2 * UM_MAX_ROWS + n]) +
                                  xl_p[3 * UM_MAX_ROWS + n];
                const bool onl = (redo && ((onl_mask >> n) & 1ull)) || (!redo && force_online);
                float M = phi_of(a, g * a.G + n % a.G);
                if (onl) {
                    M = xm_s[n];
#pragma unroll
                    for (int w = 1; w < 4; ++w) M = fmaxf(M, xm_s[w * UM_MAX_ROWS + n]);
                }
                const long long rs = dest >= 0 ? (long long)dest * R + n : slot0 + rowoff_s[n];
                float* lp = dest < 0 ? a.l_part : a.xl;
                float* mp = dest < 0 ? a.m_part : a.xm;
                const bool empty = (zero_rows >> n) & 1ull;
                lp[rs] = empty ? 0.f : lam;
                mp[rs] = empty ? -INFINITY : M;
                if (redo) {
                    // the piece's flag byte (written by the pushing CTA) gains its marks
                    uint8_t* fp = dest < 0 ? a.flags + rs : a.xf + rs;
                    const unsigned f0 = __ldcg(fp);
                    const unsigned rc = onl ? FDPP_FLAG_RECOMPUTED : 0u;
                    *fp = (uint8_t)(f0 | rc | (dest < 0 ? FDPP_FLAG_SLOT : 0u));
                }
            }
        }
        // Only where needed, the warps meet again: every warp's stores before the fallback push (a
        // release by warp 0), and a redo or forced-online segment's maxima read before the next
        // max pass writes them.
        if (push || redo || force_online) {
            if (!warps_sync()) return;
        }
        ++un;
        if (warp == 0 && lane == 0) {
            if (push) {
                const int list = (int)(blockIdx.x % REDO_NLISTS);
                const int k = atomicAdd(&a.hdr[HDR_REDO_LISTS + 2 * list], 1);
                long long* ent = a.redo + ((long long)list * a.redo_cap + k) * REDO_WORDS;
                ent[1] = (long long)(unsigned)t0 | ((long long)(unsigned)t1 << 32);
                ent[2] = dest;
                ent[3] = (long long)taint;
                st_release_gpu(ent, ((long long)(g * a.max_splits + j0) << 32) | (long long)(unsigned)(b + 1));
                misc[1] = 1;                        // the producer drains the lists after its own work
            }
            if (kind == KIND_LAST_OWN) mbar_arrive(rg.own_done);
        }
    }
}

// ------------------------------------------------------------------------------------------
// kernel
// ------------------------------------------------------------------------------------------
template <int NP, bool PAGED>
__global__ void __launch_bounds__(UM_THREADS, 1)
    split_um_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmQ, const KernelArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const UmLayout lay(NP, a.nstage, a.B);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* misc = reinterpret_cast<volatile int*>(sm + lay.misc);   // [0] abort
    Ring rg{};
    rg.nstage = a.nstage;
    rg.full = sbase + lay.bars;
    rg.empty = rg.full + 8 * a.nstage;
    rg.qfull = rg.empty + 8 * a.nstage;
    rg.qempty = rg.qfull + 16;
    rg.own_done = rg.qempty + 16;
    UmBars ub;
    ub.sfull = rg.own_done + 8;
    ub.sfree = ub.sfull + 8 * 4;
    ub.pready = ub.sfree + 8 * 4;
    ub.pfree = ub.pready + 16;
    ub.ofull = ub.pfree + 16;
    ub.ofree = ub.ofull + 16;
    ub.drain = ub.ofree + 16;
    ub.wsync = ub.drain + 8;
    static_assert(UM_NSB <= 4 && UM_NPB <= 2, "barrier slots");
    static_assert(UM_NBARS * 8 >= 16 + 16 + 8 + 2 * 32 + 4 * 16 + 8 + 8, "barrier region");
    // S^T x UM_NSB (NP each), O^T x 2 (2 NP each), rounded up to a power of two
    constexpr uint32_t NCOLS_USED = (UM_NSB + 4) * NP;
    constexpr uint32_t NCOLS = NCOLS_USED <= 64 ? 64 : NCOLS_USED <= 128 ? 128 : NCOLS_USED <= 256 ? 256 : 512;
    static_assert(NCOLS_USED <= 512, "tensor memory holds 512 columns");
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + lay.tslot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nstage; ++s) {
            mbar_init(rg.full + 8 * s, 1);
            mbar_init(rg.empty + 8 * s, 1);
        }
        for (int s = 0; s < UM_NSB; ++s) {
            mbar_init(ub.sfull + 8 * s, 1);
            mbar_init(ub.sfree + 8 * s, UM_NSW);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(rg.qfull + 8 * s, 1);
            mbar_init(rg.qempty + 8 * s, 2 + UM_NSW);   // q.K^T commit, P.V warp, softmax warps
            mbar_init(ub.pready + 8 * s, UM_NSW);
            mbar_init(ub.pfree + 8 * s, 1);
            mbar_init(ub.ofull + 8 * s, 1);
            mbar_init(ub.ofree + 8 * s, UM_NSW);
        }
        mbar_init(rg.own_done, 1);
        mbar_init(ub.drain, 2);
        mbar_init(ub.wsync, UM_NSW);
        misc[0] = 0;
        misc[1] = 0;
        int* fc = reinterpret_cast<int*>(sm + lay.fcnt);
        for (int i = 0; i < UM_FSLOTS; ++i) fc[i] = 0;
        unsigned long long* ts = reinterpret_cast<unsigned long long*>(sm + lay.taint);
        ts[0] = ts[1] = 0ull;
        fence_mbar_init();
    }
    if (threadIdx.x < UM_MAX_ROWS) {
        const int n = (int)threadIdx.x;
        reinterpret_cast<long long*>(sm + lay.rowoff)[n] =
            ((long long)(n / a.G) * a.Hq + n % a.G) * a.max_splits;
    }
    if (warp == UM_MMA_WARP) tmem_alloc(smem_u32(tslot), NCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // a programmatic dependent: while the previous kernel finishes, the P.V warp (idle until the
    // first tiles land) brings into L2 the sequence lengths the plan starts from and the tiles
    // this CTA streamed first in the last call (contiguous caches), then every warp waits for it
    if (warp == UM_PV_WARP && lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmQ);
        for (int b = 0; b < a.B && b < 32 * 8; b += 32) prefetch_l2(a.seq_lens + b);
    }
    if (!PAGED && warp == UM_PV_WARP && blockIdx.x < TC_MAX_PARTS) prefetch_hint<UM_D>(a, &tmK, &tmV);
    grid_dependency_wait();

    int* plan = reinterpret_cast<int*>(sm + lay.plan);
    if (warp == UM_PROD_WARP) {
        Producer<false, UmLayout> pr{&tmK, &tmV, &a, &lay, rg, sbase, sm, misc, plan, plan + (a.B + 1), &tmQ};
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            prefetch_tensormap(&tmQ);
        }
        pr.template run<UM_D, PAGED>();
        if (pr.bad_block && lane == 0) set_error(a, FDPP_ERRBIT_BLOCK_TABLE);
        if (lane == 0 && misc[0] != 0) {
            // aborted: let every copy this CTA issued land before it exits (bounded waits); the
            // latest issue into stage s had phase `phase` when s < stage, else phase ^ 1
            for (int s = 0; s < a.nstage; ++s) {
                const uint32_t par = (uint32_t)s < pr.stage ? pr.phase : (pr.phase ^ 1u);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(rg.full + 8 * s, par) && global_ns() - t0 < 100000000ull) {
                }
            }
            for (uint32_t k = 0; k < 2 && k < pr.qiter; ++k) {
                const uint32_t itq = pr.qiter - 1 - k, qs = itq & 1u, par = (itq >> 1) & 1u;
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(rg.qfull + 8 * qs, par) && global_ns() - t0 < 100000000ull) {
                }
            }
        }
    } else if (warp == UM_MMA_WARP) {
        mma_s_warp<NP>(a, lay, sm, sbase, rg, ub, tmem, misc);
    } else if (warp == UM_PV_WARP) {
        mma_o_warp<NP>(a, lay, sm, sbase, rg, ub, tmem, misc);
    } else {
        softmax_warps<NP>(a, lay, sm, sbase, rg, ub, tmem, misc);
        tc_fence_before();
    }
    __syncthreads();
    if (warp == UM_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, NCOLS);
    }
}

template <int NP, bool PAGED>
cudaError_t launch_np(const KernelArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                      int grid, int smem, cudaStream_t s)
{
    auto kern = split_um_kernel<NP, PAGED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(UM_THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tk, tv, tq, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int split_um_rows_padded(int R) { return R <= 16 ? 16 : (R <= 32 ? 32 : 64); }

int split_um_smem_bytes(int R, int nstage, int batch)
{
    return UmLayout(split_um_rows_padded(R), nstage, batch).total + 1024;
}

cudaError_t launch_split_um(const KernelArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tq, int grid, int smem_bytes, cudaStream_t s)
{
    const bool paged = a.block_table != nullptr;
    switch (split_um_rows_padded(a.R)) {
    case 16: return paged ? launch_np<16, true>(a, tk, tv, tq, grid, smem_bytes, s)
                          : launch_np<16, false>(a, tk, tv, tq, grid, smem_bytes, s);
    case 32: return paged ? launch_np<32, true>(a, tk, tv, tq, grid, smem_bytes, s)
                          : launch_np<32, false>(a, tk, tv, tq, grid, smem_bytes, s);
    default: return paged ? launch_np<64, true>(a, tk, tv, tq, grid, smem_bytes, s)
                          : launch_np<64, false>(a, tk, tv, tq, grid, smem_bytes, s);
    }
}

}  // namespace fdpp
