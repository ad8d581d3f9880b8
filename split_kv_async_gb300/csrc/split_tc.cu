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
#include "split_tc_common.cuh"

namespace fdpp {
namespace {

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
    // per segment parity: a warp switched to the running max (the merge weighs the frames)
    unsigned* mixed_s = reinterpret_cast<unsigned*>(sm + lay.fslot + TC_FSLOTS * 8);

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
        // a redo piece keeps the phi frame for rows whose own split stayed in the window; a
        // segment switches to the running max at its first score outside the window (below)
        bool online = (redo && onl_mask != 0u) || (a.mode == FDPP_MODE_FORCE_ONLINE);
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
        bool frz[2] = {redo && !((onl_mask >> head0) & 1u), redo && !((onl_mask >> (head0 + 1)) & 1u)};
        float mrun[2] = {online && !frz[0] ? -INFINITY : phv[0], online && !frz[1] ? -INFINITY : phv[1]};
        unsigned fl[2] = {0u, 0u};

        // End of one split piece of an own segment: the four warps' window decisions for it,
        // combined by whichever warp arrives last (one atomic OR on a 64-bit shared word: 4 bits
        // per row, an arrival bit per warp), which writes the rows' flag bytes (the split's own,
        // or the run slot's edge byte for a first piece that starts inside a split). In normal
        // mode a row-split with a score outside the window was finished with the running max
        // (the switch below) and is marked recomputed. Pieces cycle through TC_FSLOTS words: no
        // warp runs more than a ring's depth of tiles ahead of another.
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
            if (lane == 0) fslot[ks] = 0ull;
            if (lane < nrow()) {
                const unsigned f = (full >> (4 * lane)) & 15u;
                const bool rc = a.mode == FDPP_MODE_FORCE_ONLINE ||
                                (a.mode == FDPP_MODE_NORMAL && (f & FDPP_FLAG_OUT));
                const uint8_t fb = (uint8_t)(f | (rc ? FDPP_FLAG_RECOMPUTED : 0u));
                if (first_piece && dest >= 0 && t0 != jp * S)
                    a.xf[(long long)dest * rows() + lane] = fb;
                else
                    a.flags[MQ ? unit_row_slot(a, b, kvh, rbase + lane, jp)
                               : ((long long)b * a.Hq + kvh * a.G + rbase + lane) * a.max_splits + jp] = fb;
            }
        };

        // The tile loop, built once for the phi frame and once for the running max (redo pieces,
        // forced online mode, and a segment after its first score outside the window), so the
        // hot phi-frame loop stays compact. Tiles are 64 tokens and never cross a split boundary.
        int tt = t0, se = (t0 / S + 1) * S, jp = j0;
        bool first_piece = true, to_online = false;
        auto run_tiles = [&](auto online_c) -> bool {
            constexpr bool ONLINE = decltype(online_c)::value;
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
                // Normal mode, phi frame: a score of this warp outside the window ends the
                // phi-frame loop before the tile is used; the running-max loop takes the segment
                // on from this tile (the tiles before were inside the window, so their sums are
                // those of the online softmax in the frame phi).
                if constexpr (!ONLINE) {
                    if (a.mode == FDPP_MODE_NORMAL &&
                        __any_sync(0xffffffffu, ((fl[0] | fl[1]) & FDPP_FLAG_OUT) != 0u)) {
                        to_online = true;
                        return true;
                    }
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
        if (to_online) {
            // Each row of this warp continues with its running max: the frame phi if the warp
            // already holds some of the row's sum, else none yet. The merge then weighs the
            // four warps' frames (the segment's mixed-frame mark).
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float lw = lsum[c];
#pragma unroll
                for (int sh = 4; sh < 32; sh <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, sh);
                mrun[c] = lw > 0.f ? phv[c] : -INFINITY;
                frz[c] = false;
            }
            online = true;
            if (lane == 0) mixed_s[upar] = 1u;
            if (!run_tiles(std::true_type{})) return;
        }
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
        // the sums need no exponentials; a segment in which some warp switched to the running
        // max weighs each warp's sums into the rows' common frame.
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
        const bool mix = online || mixed_s[upar] != 0u;

        // this warp and its partner (warp + 2), each weighted into the rows' common frame
        {
            float ws[2] = {1.f, 1.f}, wp[2] = {1.f, 1.f};
            if (mix) {
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
                if (!mix) {
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
        // A redo piece (pushed by the tcgen05 build's protocol; this build finishes a row-split
        // with the running max in place and pushes none) rewrites its tainted rows only and
        // writes their flag bytes.
        const unsigned write_mask = redo ? redo_mask : 0xffffffffu;
        {
            const int hh = lane;
            float M = 0.f, lam = 0.f;
            if (hh < nrow()) {
                M = xm_s[hh];
#pragma unroll
                for (int w = 1; w < NCW; ++w) M = fmaxf(M, xm_s[w * TC_MAX_GROUP + hh]);
#pragma unroll
                for (int w = 0; w < NCW; ++w)
                    lam = mix ? fmaf(frame_weight(xm_s[w * TC_MAX_GROUP + hh], M), xl_s[w * TC_MAX_GROUP + hh], lam)
                              : lam + xl_s[w * TC_MAX_GROUP + hh];
            }
            if (hh < nrow() && ((write_mask >> hh) & 1u)) {
                const long long rs = dest >= 0 ? (long long)dest * rows() + hh
                                     : MQ ? unit_row_slot(a, b, kvh, rbase + hh, j0)
                                          : ((long long)b * a.Hq + kvh * a.G + rbase + hh) * a.max_splits + j0;
                float* lp = dest < 0 ? a.l_part : a.xl;
                float* mp = dest < 0 ? a.m_part : a.xm;
                lp[rs] = lam;
                mp[rs] = M;
                if (redo) {
                    const unsigned f0 = ((hh < 4 ? fw0 : fw1) >> ((hh & 3) * 8)) & 0xffu;
                    const unsigned rc = ((onl_mask >> hh) & 1u) ? FDPP_FLAG_RECOMPUTED : 0u;
                    if (dest < 0) a.flags[rs] = (uint8_t)(f0 | rc | FDPP_FLAG_SLOT);
                    else a.xf[rs] = (uint8_t)(f0 | rc);
                }
            }
        }
        // the partial rows of this lane: head0 and head0 + 1, the run slot or the split's own
        float* orow[2] = {nullptr, nullptr};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int hh = head0 + c;
            if (!hv[c] || !((write_mask >> hh) & 1u)) continue;
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
        // warp 1 has read the mark (mhand): clear it for the segment after next before warps 2
        // and 3 may go on to it
        if (lane == 0) mixed_s[upar] = 0u;
        __syncwarp();
        if (lane == 0) mbar_arrive(rg.mdone);      // both slots read: warps 2 and 3 may refill them
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            if (orow[c] == nullptr) continue;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                orow[c][16 * mt + r] = o[mt][c];
                orow[c][16 * mt + r + 8] = o[mt][c + 2];
            }
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
    // previous kernel on the stream has completed. Before that, consumer warp 0 (idle until the
    // first tiles land) brings into L2 the sequence lengths the producer's plan starts from and
    // the start-up hint's tiles.
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        for (int b = 0; b < a.B && b < 32 * 8; b += 32) prefetch_l2(a.seq_lens + b);
    }
    if (!PAGED && warp == 0 && blockIdx.x < TC_MAX_PARTS) prefetch_hint<D>(a, &tmK, &tmV);
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
