// split_tc.cu -- per-split kernel for bf16 K/V: TMA-fed ring, tensor-core q.K^T and P.V.
//
// What it computes (opt.ai.kr "FlashDecoding++ async softmax -- theory", s1 and s3): for one
// unit (sequence b, kv head g, split j) and the G query heads that share kv head g,
//     s_t = scale <q_h, k_t>, p_t = exp(s_t - phi), l = sum p_t, o = sum p_t v_t   (fast pass)
// against the unified max phi, with no communication between splits; every score is tested
// against lo <= s - phi <= hi; a unit with a head outside the window is streamed again at the
// end of the CTA's work and recomputed with the ordinary online softmax (running max).
//
// How. One CTA = 4 consumer warps + 1 producer warp, persistent over units. The producer streams
// 64-token K and V tiles of head g with 3-D TMA loads (128-byte swizzle) into a ring of
// `nstage` shared-memory stages guarded by mbarriers (full: TMA bytes landed; empty: 4 consumer
// warps released the stage); for a paged cache it issues one box per 16..64-token block, using
// the block table. Each consumer warp owns 16 tokens of a tile:
//   S[16 x 16] = Q[16 x d] K^T        mma.m16n8k16 (bf16 in, fp32 accumulate); rows 0..G-1 are
//                                     the G query heads (zero padded), so each K byte read from
//                                     HBM feeds all G heads;
//   P = exp(S - phi), detect window
//   O[16 x d] += [P_hi ; P_lo] V      P is split into bf16 hi + lo parts stacked in the 16 rows
//                                     of the A tile (G <= 8), so P.V keeps ~16 mantissa bits;
//                                     row h + row h+8 is head h's output.
// Warps merge their fp32 partials through shared memory (a plain sum in the phi frame) and
// write o, l, m = phi and the flag byte of each head of the unit.
#include <cuda_bf16.h>

#include "device_common.cuh"

namespace fdpp {
namespace {

constexpr int NCW = 4;                  // consumer warps
constexpr int TPW = 16;                 // tokens per consumer warp and tile
constexpr int TILE = NCW * TPW;         // tokens per tile
constexpr int NTHREADS = (NCW + 1) * 32;
static_assert(TILE == TC_TILE_TOKENS, "tile height is part of the tensor-map contract");

// Shared-memory layout of one CTA (byte offsets from a 1024-byte aligned base).
struct TcLayout {
    int stage_bytes, kv_bytes, q_bytes, scr_row;
    int stages, qbuf, scr_o, scr_l, scr_m, scr_f, bars, misc, red, total;

    __host__ __device__ static constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

    __host__ __device__ TcLayout(int D, int G, int nstage)
        : stage_bytes(2 * TILE * D * 2), kv_bytes(TILE * D * 2), q_bytes(round_up(G * D * 2, 128)),
          scr_row(D + 8), stages(0), qbuf(0), scr_o(0), scr_l(0), scr_m(0), scr_f(0), bars(0),
          misc(0), red(0), total(0)
    {
        qbuf = stages + nstage * stage_bytes;
        scr_o = qbuf + 2 * q_bytes;
        scr_l = scr_o + NCW * G * scr_row * 4;
        scr_m = scr_l + NCW * G * 4;
        scr_f = scr_m + NCW * G * 4;
        bars = round_up(scr_f + NCW * G * 4, 8);
        misc = bars + (2 * nstage + 5) * 8;
        red = round_up(misc + 16, 8);
        total = red + 32 * 8;
    }
};

struct Ring {
    uint32_t full, empty, qfull, qempty;   // shared addresses of the barrier arrays
    uint32_t cbar;                         // consumer-warps barrier (128 arrivals per phase)
    int nstage;
};

// All lanes wait; any lane that runs out of time aborts the CTA (warp-uniform result).
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, volatile int* misc,
                                          const KernelArgs& a)
{
    bool ok = (misc[1] == 0) && mbar_wait(bar, parity);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        if ((threadIdx.x & 31) == 0) {
            misc[1] = 1;
            set_error(a, FDPP_ERRBIT_TIMEOUT);
        }
    }
    return ok;
}

// Barrier of the 4 consumer warps with a bounded wait (a bar.sync could not give up).
__device__ __forceinline__ bool consumer_sync(const Ring& rg, uint32_t& parity, volatile int* misc,
                                              const KernelArgs& a)
{
    mbar_arrive(rg.cbar);
    const bool ok = ring_wait(rg.cbar, parity, misc, a);
    parity ^= 1u;
    return ok;
}

// Heads of unit (b, g, j) whose fast pass left the window (bit h for head g*G + h).
__device__ __forceinline__ unsigned unit_redo_mask(const KernelArgs& a, int b, int g, int j)
{
    unsigned mask = 0u;
    for (int h = 0; h < a.G; ++h) {
        const long long r = ((long long)b * a.Hq + (long long)g * a.G + h) * a.max_splits + j;
        if (a.flags[r] & FDPP_FLAG_OUT) mask |= 1u << h;
    }
    return mask;
}

// ------------------------------------------------------------------------------------------
// producer warp
// ------------------------------------------------------------------------------------------
template <int D, bool PAGED>
__device__ __forceinline__ void produce(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                        const KernelArgs& a, const TcLayout& lay, uint32_t sbase,
                                        const Ring& rg, volatile int* misc, int S, int n_units,
                                        bool recompute, uint32_t& p_stage, uint32_t& p_phase,
                                        uint32_t& pq_iter)
{
    constexpr int HALVES = D / 64;
    const int lane = threadIdx.x & 31;
    const int bs = PAGED ? a.block_size : TILE;
    const int rows_box = bs < TILE ? bs : TILE;
    const uint32_t box_bytes = 128u * (uint32_t)rows_box;
    UnitCursor cur;
    cur.reset();
    bool bad_block = false;

    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        int b, g, j, L;
        cur.seek(a, S, u, b, g, j, L);
        if (recompute && unit_redo_mask(a, b, g, j) == 0u) continue;
        const int t0 = j * S, t1 = min(t0 + S, L);
        const int ntiles = ceil_div_i(t1 - t0, TILE);

        // query rows of the unit's G heads: one bulk copy into the Q ring
        {
            const uint32_t qs = pq_iter & 1u, quse = pq_iter >> 1;
            if (!ring_wait(rg.qempty + 8 * qs, (quse & 1u) ^ 1u, misc, a)) return;
            if (lane == 0) {
                const uint32_t bytes = (uint32_t)(a.G * D * 2);
                const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.q) +
                                           ((long long)b * a.Hq + (long long)g * a.G) * D;
                mbar_arrive_expect_tx(rg.qfull + 8 * qs, bytes);
                bulk_load(sbase + lay.qbuf + qs * lay.q_bytes, src, bytes, rg.qfull + 8 * qs);
            }
            ++pq_iter;
        }

        int win_base = -(1 << 30), ent = -1;           // paged: 32 block-table entries per window
        const int nblk_seq = PAGED ? ceil_div_i(L, bs) : 0;
        for (int i = 0; i < ntiles; ++i) {
            const int tt = t0 + i * TILE;
            const int nvalid = min(TILE, t1 - tt);
            if (!ring_wait(rg.empty + 8 * p_stage, p_phase ^ 1u, misc, a)) return;
            const uint32_t kdst = sbase + lay.stages + p_stage * lay.stage_bytes;
            const uint32_t vdst = kdst + lay.kv_bytes;
            const uint32_t fb = rg.full + 8 * p_stage;
            if (!PAGED) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, (uint32_t)lay.stage_bytes);
#pragma unroll
                    for (int hv = 0; hv < HALVES; ++hv) {
                        tma_load_3d(kdst + hv * TILE * 128, tmK, g * D + hv * 64, tt, b, fb);
                        tma_load_3d(vdst + hv * TILE * 128, tmV, g * D + hv * 64, tt, b, fb);
                    }
                }
            } else {
                // logical blocks touched by the valid tokens of this tile
                const int lb0 = tt / bs;
                const int nb = (bs <= TILE) ? ceil_div_i(nvalid, bs) : 1;
                if (lb0 < win_base || lb0 + nb > win_base + 32) {
                    win_base = lb0;
                    const int lb = lb0 + lane;
                    ent = (lb < nblk_seq) ? __ldg(a.block_table + (long long)b * a.max_blocks + lb)
                                          : -1;
                }
                int blk[TILE / 16];
                uint32_t bytes = 0;
#pragma unroll
                for (int k = 0; k < TILE / 16; ++k) {
                    blk[k] = -1;
                    if (k < nb) {
                        const int e = __shfl_sync(0xffffffffu, ent, lb0 + k - win_base);
                        if (e >= 0 && e < a.num_blocks) {
                            blk[k] = e;
                            bytes += 2u * HALVES * box_bytes;
                        } else {
                            bad_block = true;
                        }
                    }
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, bytes);
                    const int y = (bs <= TILE) ? 0 : (tt % bs);
#pragma unroll
                    for (int k = 0; k < TILE / 16; ++k) {
                        if (blk[k] < 0) continue;
#pragma unroll
                        for (int hv = 0; hv < HALVES; ++hv) {
                            const uint32_t off = hv * TILE * 128 + k * rows_box * 128;
                            tma_load_3d(kdst + off, tmK, g * D + hv * 64, y, blk[k], fb);
                            tma_load_3d(vdst + off, tmV, g * D + hv * 64, y, blk[k], fb);
                        }
                    }
                }
            }
            if (++p_stage == (uint32_t)rg.nstage) { p_stage = 0; p_phase ^= 1u; }
        }
    }
    if (bad_block && lane == 0) set_error(a, FDPP_ERRBIT_BLOCK_TABLE);
}

// ------------------------------------------------------------------------------------------
// consumer warps
// ------------------------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void consume(const KernelArgs& a, const TcLayout& lay, uint8_t* sm,
                                        uint32_t sbase, const Ring& rg, volatile int* misc, int S,
                                        int n_units, bool recompute, uint32_t& c_stage,
                                        uint32_t& c_phase, uint32_t& cq_iter, uint32_t& cparity)
{
    constexpr int KS = D / 16;           // k-steps of q.K^T, and column pairs of P.V
    constexpr int NT = D / 8;            // n-tiles of the output
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, ctid = threadIdx.x;
    const int h = lane >> 2, qd = lane & 3;       // head row and column pair of this lane
    const int mi = lane >> 3, r8 = lane & 7;      // ldmatrix: matrix and row of this lane
    const bool head_ok = h < a.G;
    const bool online = recompute || (a.mode == FDPP_MODE_FORCE_ONLINE);
    const uint32_t k_row = warp * TPW + (mi >> 1) * 8 + r8;
    const uint32_t v_row = warp * TPW + (mi & 1) * 8 + r8;
    const int tok_lo = warp * TPW + 2 * qd;       // this lane's first token in n-tile 0
    float* scr_o = reinterpret_cast<float*>(sm + lay.scr_o);
    float* scr_l = reinterpret_cast<float*>(sm + lay.scr_l);
    float* scr_m = reinterpret_cast<float*>(sm + lay.scr_m);
    unsigned* scr_f = reinterpret_cast<unsigned*>(sm + lay.scr_f);
    UnitCursor cur;
    cur.reset();

    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        int b, g, j, L;
        cur.seek(a, S, u, b, g, j, L);
        const unsigned redo = recompute ? unit_redo_mask(a, b, g, j) : 0u;
        if (recompute && redo == 0u) continue;
        const int t0 = j * S, t1 = min(t0 + S, L);
        const int ntiles = ceil_div_i(t1 - t0, TILE);

        // Q fragments (A operand rows 0..7 = heads; rows 8..15 zero)
        uint32_t qa[KS][2];
        {
            const uint32_t qs = cq_iter & 1u;
            if (!ring_wait(rg.qfull + 8 * qs, (cq_iter >> 1) & 1u, misc, a)) return;
            const uint8_t* qb = sm + lay.qbuf + qs * lay.q_bytes;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qa[ks][0] = head_ok ? *reinterpret_cast<const uint32_t*>(qb + (h * D + ks * 16 + 2 * qd) * 2) : 0u;
                qa[ks][1] = head_ok ? *reinterpret_cast<const uint32_t*>(qb + (h * D + ks * 16 + 8 + 2 * qd) * 2) : 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rg.qempty + 8 * qs);
            ++cq_iter;
        }

        float o[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float lsum = 0.f;
        float mrun = online ? -INFINITY : a.phi;
        unsigned fl = 0u;

        for (int i = 0; i < ntiles; ++i) {
            const int nvalid = min(TILE, t1 - (t0 + i * TILE));
            if (!ring_wait(rg.full + 8 * c_stage, c_phase, misc, a)) return;
            const uint32_t kb = sbase + lay.stages + c_stage * lay.stage_bytes;
            const uint32_t vb = kb + lay.kv_bytes;

            // S = Q K^T for this warp's 16 tokens (two n-tiles of 8 tokens), two chains each
            float sa[2][2][4];
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) sa[c][nt][0] = sa[c][nt][1] = sa[c][nt][2] = sa[c][nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int chunk = 2 * ks + (mi & 1);
                const uint32_t addr = kb + (chunk >> 3) * (TILE * 128) + k_row * 128 + (((chunk & 7) ^ r8) << 4);
                uint32_t k0, k1, k2, k3;
                ldsm_x4(addr, k0, k1, k2, k3);
                mma_16816(sa[ks & 1][0], qa[ks][0], 0u, qa[ks][1], 0u, k0, k1);
                mma_16816(sa[ks & 1][1], qa[ks][0], 0u, qa[ks][1], 0u, k2, k3);
            }

            // scores of head h at tokens tok_lo + 8*nt + e
            float s[2][2];
            bool valid[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[nt][e] = __fmul_rn(sa[0][nt][e] + sa[1][nt][e], a.scale);
                    valid[nt][e] = head_ok && (tok_lo + 8 * nt + e < nvalid);
                    if (valid[nt][e]) fl |= classify(__fsub_rn(s[nt][e], a.phi), a.lo, a.hi);
                }

            float p[2][2];
            if (!online) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        p[nt][e] = valid[nt][e] ? __expf(__fsub_rn(s[nt][e], a.phi)) : 0.f;
            } else {
                float tmax = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (valid[nt][e]) tmax = fmaxf(tmax, s[nt][e]);
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
                const float mnew = fmaxf(mrun, tmax);
                const float corr = (mrun == mnew) ? 1.f : (mrun == -INFINITY ? 0.f : __expf(mrun - mnew));
                if (corr != 1.f) {
                    lsum *= corr;
#pragma unroll
                    for (int n = 0; n < NT; ++n) { o[n][0] *= corr; o[n][1] *= corr; o[n][2] *= corr; o[n][3] *= corr; }
                }
                mrun = mnew;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        p[nt][e] = valid[nt][e] ? __expf(s[nt][e] - mnew) : 0.f;
            }
            lsum += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);

            // A operand of P.V: rows 0..7 = bf16(p), rows 8..15 = bf16(p - bf16(p))
            uint32_t pa[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const __nv_bfloat162 hi = __floats2bfloat162_rn(p[nt][0], p[nt][1]);
                const float2 hf = __bfloat1622float2(hi);
                pa[2 * nt] = *reinterpret_cast<const uint32_t*>(&hi);
                pa[2 * nt + 1] = pack_bf16x2(p[nt][0] - hf.x, p[nt][1] - hf.y);
            }

            // masks for V rows past the valid tokens (their shared-memory rows may hold NaN)
            uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
            if (nvalid < TILE) {
                vm_lo = (tok_lo < nvalid ? 0x0000ffffu : 0u) | (tok_lo + 1 < nvalid ? 0xffff0000u : 0u);
                vm_hi = (tok_lo + 8 < nvalid ? 0x0000ffffu : 0u) | (tok_lo + 9 < nvalid ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int c2 = 0; c2 < KS; ++c2) {
                const int chunk = 2 * c2 + (mi >> 1);
                const uint32_t addr = vb + (chunk >> 3) * (TILE * 128) + v_row * 128 + (((chunk & 7) ^ r8) << 4);
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(addr, v0, v1, v2, v3);
                v0 &= vm_lo; v2 &= vm_lo; v1 &= vm_hi; v3 &= vm_hi;
                mma_16816(o[2 * c2], pa[0], pa[1], pa[2], pa[3], v0, v1);
                mma_16816(o[2 * c2 + 1], pa[0], pa[1], pa[2], pa[3], v2, v3);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rg.empty + 8 * c_stage);
            if (++c_stage == (uint32_t)rg.nstage) { c_stage = 0; c_phase ^= 1u; }
        }

        // ---- merge the 4 warps' partials of this unit and write them ----
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
        fl |= __shfl_xor_sync(0xffffffffu, fl, 1);
        fl |= __shfl_xor_sync(0xffffffffu, fl, 2);
        if (!consumer_sync(rg, cparity, misc, a)) return;   // scratch of the previous unit is free
        if (head_ok) {
            float* row = scr_o + (warp * a.G + h) * lay.scr_row;
#pragma unroll
            for (int n = 0; n < NT; ++n)
                *reinterpret_cast<float2*>(row + 8 * n + 2 * qd) = make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
            if (qd == 0) {
                scr_l[warp * a.G + h] = lsum;
                scr_m[warp * a.G + h] = mrun;
                scr_f[warp * a.G + h] = fl;
            }
        }
        if (!consumer_sync(rg, cparity, misc, a)) return;
        const unsigned write_mask = recompute ? redo : 0xffffffffu;
        for (int idx = ctid; idx < a.G * D; idx += NCW * 32) {
            const int hh = idx / D, d = idx - hh * D;
            if (!((write_mask >> hh) & 1u)) continue;
            float M = scr_m[hh];
#pragma unroll
            for (int w = 1; w < NCW; ++w) M = fmaxf(M, scr_m[w * a.G + hh]);
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w)
                acc = fmaf(frame_weight(scr_m[w * a.G + hh], M), scr_o[(w * a.G + hh) * lay.scr_row + d], acc);
            const long long r = ((long long)b * a.Hq + (long long)g * a.G + hh) * a.max_splits + j;
            a.o_part[r * D + d] = acc;
        }
        if (ctid < a.G && ((write_mask >> ctid) & 1u)) {
            const int hh = ctid;
            float M = scr_m[hh];
            unsigned f = scr_f[hh];
            for (int w = 1; w < NCW; ++w) { M = fmaxf(M, scr_m[w * a.G + hh]); f |= scr_f[w * a.G + hh]; }
            float lam = 0.f;
            for (int w = 0; w < NCW; ++w) lam = fmaf(frame_weight(scr_m[w * a.G + hh], M), scr_l[w * a.G + hh], lam);
            const long long r = ((long long)b * a.Hq + (long long)g * a.G + hh) * a.max_splits + j;
            a.l_part[r] = lam;
            a.m_part[r] = M;
            if (recompute) {
                a.flags[r] = (uint8_t)(a.flags[r] | FDPP_FLAG_RECOMPUTED);
            } else {
                a.flags[r] = (uint8_t)(f | (online ? FDPP_FLAG_RECOMPUTED : 0u));
                if ((f & FDPP_FLAG_OUT) && a.mode == FDPP_MODE_NORMAL) misc[0] = 1;
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// kernel
// ------------------------------------------------------------------------------------------
template <int D, bool PAGED>
__global__ void __launch_bounds__(NTHREADS, 2)
    split_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const KernelArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const TcLayout lay(D, a.G, a.nstage);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* misc = reinterpret_cast<volatile int*>(sm + lay.misc);   // [0] refetch needed, [1] abort
    Ring rg;
    rg.nstage = a.nstage;
    rg.full = sbase + lay.bars;
    rg.empty = rg.full + 8 * a.nstage;
    rg.qfull = rg.empty + 8 * a.nstage;
    rg.qempty = rg.qfull + 16;
    rg.cbar = rg.qempty + 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nstage; ++s) {
            mbar_init(rg.full + 8 * s, 1);
            mbar_init(rg.empty + 8 * s, NCW);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(rg.qfull + 8 * s, 1);
            mbar_init(rg.qempty + 8 * s, NCW);
        }
        mbar_init(rg.cbar, NCW * 32);
        misc[0] = 0;
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == NCW && lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    int S, n_units;
    block_plan(a, reinterpret_cast<long long*>(sm + lay.red), S, n_units);   // syncs the block

    uint32_t stage = 0, phase = 0, qiter = 0, cparity = 0;
    if (warp == NCW)
        produce<D, PAGED>(&tmK, &tmV, a, lay, sbase, rg, misc, S, n_units, false, stage, phase, qiter);
    else
        consume<D>(a, lay, sm, sbase, rg, misc, S, n_units, false, stage, phase, qiter, cparity);
    __syncthreads();
    // splits that left the safe window: stream them again and recompute with online softmax
    if (a.mode == FDPP_MODE_NORMAL && misc[0] != 0 && misc[1] == 0) {
        if (warp == NCW)
            produce<D, PAGED>(&tmK, &tmV, a, lay, sbase, rg, misc, S, n_units, true, stage, phase, qiter);
        else
            consume<D>(a, lay, sm, sbase, rg, misc, S, n_units, true, stage, phase, qiter, cparity);
    }
    __syncthreads();
    if (misc[1] != 0 && warp == NCW && lane == 0) {
        // Aborted: let every copy this CTA issued land before the CTA exits (bounded waits).
        // The latest issue into stage s had phase `phase` when s < stage, else phase ^ 1 (a
        // stage never issued waits on the completed phase before its first and passes at once).
        for (int s = 0; s < a.nstage; ++s) {
            const uint32_t par = (uint32_t)s < stage ? phase : (phase ^ 1u);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(rg.full + 8 * s, par) && global_ns() - t0 < 100000000ull) {
            }
        }
        for (uint32_t k = 0; k < 2 && k < qiter; ++k) {
            const uint32_t it = qiter - 1 - k, qs = it & 1u, par = (it >> 1) & 1u;
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(rg.qfull + 8 * qs, par) && global_ns() - t0 < 100000000ull) {
            }
        }
    }
}

template <int D, bool PAGED>
cudaError_t launch_t(const KernelArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                     int smem, cudaStream_t s)
{
    auto kern = split_tc_kernel<D, PAGED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NTHREADS, smem, s>>>(tk, tv, a);
    return cudaGetLastError();
}

}  // namespace

TcPlan split_tc_plan(int head_dim, int group, int req_stages, int req_ctas, int smem_per_sm,
                     int smem_per_block)
{
    TcPlan p{0, 0, 0};
    const int reserve = 1024;                         // per-CTA system reservation
    auto bytes = [&](int ns) { return TcLayout(head_dim, group, ns).total + 1024; };
    const int cands[4] = {2, 1, 3, 4};
    for (int ci = 0; ci < 4; ++ci) {
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
                            int grid, int smem_bytes, cudaStream_t s)
{
    const bool paged = a.block_table != nullptr;
    if (a.D == 128)
        return paged ? launch_t<128, true>(a, tk, tv, grid, smem_bytes, s)
                     : launch_t<128, false>(a, tk, tv, grid, smem_bytes, s);
    return paged ? launch_t<64, true>(a, tk, tv, grid, smem_bytes, s)
                 : launch_t<64, false>(a, tk, tv, grid, smem_bytes, s);
}

}  // namespace fdpp
