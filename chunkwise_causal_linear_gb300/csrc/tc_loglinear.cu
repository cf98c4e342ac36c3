// tc_loglinear.cu -- tensor-core path for the log-linear (Fenwick) mask (sm_103a).
//
// "論文紹介：Log Linear Attention" (slides 15-17, 20-21): query t weighs key s <= t by
// lambda_t^(l), l = 0 if s == t else 1 + floor(log2(t XOR s)).  With chunks of C = 64 rows
// aligned on multiples of 64, a same-chunk pair has l <= 6 (the intra-chunk mask), and a pair
// in chunks c_s < c_t has l = 7 + floor(log2(c_t XOR c_s)): the earlier chunks split into
// dyadic blocks, one per set bit j of c_t (block B_j(c_t) = the 2^j chunks below c_t that
// share c_t's bits above j, with bit j cleared).  So
//     o_t = sum_{s in chunk, s <= t} lambda_t^(l(t,s)) (q_t.k_s) v_s
//         + sum_{j : bit j of c_t} lambda_t^(7+j) q_t T_j(c_t),   T_j = sum_{s in B_j} k_s^T v_s.
// Shapes here: identity feature map, d_k = d_v = 64, C = 64, bf16 storage, no normaliser.
//
// Work split.  A head's chunks are cut into segments of 2^p chunks (one CTA each).  Inside a
// segment starting at chunk a, the bits j >= p of every chunk index equal those of a, so
// the levels j >= p are fixed for the whole segment: each is a sum of whole earlier segments,
// built at the CTA's start from per-segment totals (a first, totals-only launch writes them).
// The levels j < p lie inside the segment and follow the Fenwick recurrence.  The running
// state PS(i) = sum of the segment's chunks before local chunk i accumulates in TMEM, and
// the block that closes after chunk i (r = ctz(i + 1)) is T_r = PS(i + 1) - PS(i + 1 - 2^r).
// The fp32 snapshots PS(x) at the binary prefixes x of the current position form a stack
// (depth = popcount(x)) kept in the workspace, where it stays in L2.
//
// Per chunk (all MMAs M = 64 rows, K = 64 as 4 x K16; bf16 in, fp32 accumulate):
//   scores  A   = Q K^T                 (A K-major, B K-major)
//   state   PS += K^T V                 (A = K MN-major, B = V MN-major)
//   intra   O   = P V,  P = lambda-masked A
//   levels  R_j = Q T_j                 per set bit j
// Both kinds of product go, in that order, through one ring of 6 TMEM slots, and the output
// rows o_t = O[t] + sum_j lambda_t^(7+j) R_j[t] are formed in fp32 by the output warps, so
// the level weights never pass through a bf16 operand.
// Warps: 0 TMA producer, 1 MMA issuer, 4-7 turn scores into P, 8-11 close the Fenwick
// blocks, 12-15 combine and store the output rows.  A group of four consecutive warps
// covers the four TMEM lane quadrants (warp % 4).
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace la {

using namespace ptx;
using namespace tcc;

namespace {

constexpr int LL_THREADS = 512;  // 16 warps
constexpr int LL_D = 64, LL_C = 64, LL_LOG2C = 6;
constexpr int LL_RING = 6;       // TMEM slots for the products P V and R_j
constexpr int LL_MAXLEV = 12;    // inter levels: up to 4096 chunks per head
constexpr int LL_MAXNL = 32;     // lambda entries per row held in shared memory
constexpr int LL_TILE = LL_C * 128;
constexpr int LL_STAGES_MAIN = 3;   // Q, K, V, lambda (32 KB each)
constexpr int LL_STAGES_TOT = 6;    // K, V (16 KB each)
constexpr int LL_STAGE_AREA = LL_STAGES_MAIN * 4 * LL_TILE;
static_assert(LL_STAGES_TOT * 2 * LL_TILE <= LL_STAGE_AREA, "stage area");
static_assert(LL_C * LL_MAXNL * 4 <= LL_TILE, "lambda tile");
constexpr int LL_N_BAR = 2 * LL_STAGES_TOT + 2 * LL_RING + 16;   // all used

// TMEM columns (M = 64 layout: row m at lane (m % 16) + 32 (m / 16))
constexpr uint32_t LT_PS = 0;     // running segment state PS [d_k rows][d_v]
constexpr uint32_t LT_A = 64;     // scores
constexpr uint32_t LT_R = 128;    // products P V and R_j, LL_RING slots of 64 columns
static_assert(LT_R + 64 * LL_RING <= 512, "TMEM columns");

struct LlLayout {
    int off_T, off_P, off_bar, bytes, alloc;
};

inline LlLayout ll_layout(int nlev)
{
    LlLayout l;
    l.off_T = LL_STAGE_AREA;
    // nlev block tiles, plus a second tile for level 0 (the block of one chunk closes after
    // every other chunk, and is written while the previous one may still be read)
    l.off_P = l.off_T + (nlev + 1) * LL_TILE;   // two P tiles (chunk parity)
    l.off_bar = l.off_P + 2 * LL_TILE;
    l.bytes = l.off_bar + LL_N_BAR * 8 + 16;
    l.alloc = l.bytes + 1024;
    return l;
}

struct LlArgs {
    CUtensorMap tm_q, tm_k, tm_v;
    const float *lam;        // [BH][L][NL]
    __nv_bfloat16 *out;      // [BH][L][64]
    int L, nch, NL;
    int p, seg_chunks, nseg, nlev;
    int totals, grid_seg, BH;
    LlLayout lay;
    float *ws_G;             // [nseg - 1][BH][64][64] segment totals
    float *ws_stack;         // [BH * nseg][p][64][64] prefix snapshots
    int *err;
    unsigned long long timeout_ns;
};

__global__ void __launch_bounds__(LL_THREADS, 1) tc_loglinear_kernel(const __grid_constant__ LlArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = (uint64_t *)(sm + a.lay.off_bar);
    uint64_t *full = bars;                           // [stages]
    uint64_t *stage_free = full + LL_STAGES_TOT;     // [stages]
    uint64_t *r_full = stage_free + LL_STAGES_TOT;   // [RING]
    uint64_t *r_free = r_full + LL_RING;             // [RING]
    uint64_t *scores_done = r_free + LL_RING;
    uint64_t *a_free = scores_done + 1;
    // p_ready alternates by chunk parity, t_formed and c_done by chunk mod 4: their producers
    // may run one (p_ready) or two chunks (t_formed, c_done) ahead of the waiter, and one
    // barrier must never be two phases ahead of it.
    uint64_t *p_ready = a_free + 1;                  // [2]
    uint64_t *state_done = p_ready + 2;
    uint64_t *ps_read = state_done + 1;              // PS copied out by the block-closing warps
    uint64_t *t_formed = ps_read + 1;                // [4] the block closed after a chunk is in smem
    uint64_t *c_done = t_formed + 4;                 // [4] every product of a chunk is in TMEM
    uint64_t *drain = c_done + 4;
    uint64_t *totals_done = drain + 1;
    uint32_t *tmem_slot = (uint32_t *)(sm + a.lay.off_bar + LL_N_BAR * 8);
    volatile int *abort_flag = (volatile int *)(sm + a.lay.off_bar + LL_N_BAR * 8 + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x / a.grid_seg, seg = blockIdx.x % a.grid_seg;
    const int tile0 = seg * a.seg_chunks;               // first chunk of the segment
    const int nloc = min(a.seg_chunks, a.nch - tile0);  // chunks in this segment
    const bool totals = a.totals != 0;
    const int NL = a.NL;
    const int nst = totals ? LL_STAGES_TOT : LL_STAGES_MAIN;
    const int sbytes = totals ? 2 * LL_TILE : 4 * LL_TILE;
    Ctl ctl{abort_flag, a.err, a.timeout_ns};
    if (totals) pdl_trigger();  // the main pass may be scheduled now
    else pdl_wait();            // the totals pass (if any) has completed
    // stage layout: main [Q | K | V | lambda], totals [K | V]
    auto stage_q = [&](int s) { return sm + s * sbytes; };
    auto stage_k = [&](int s) { return sm + s * sbytes + (totals ? 0 : LL_TILE); };
    auto stage_v = [&](int s) { return stage_k(s) + LL_TILE; };
    auto stage_l = [&](int s) { return (const float *)(sm + s * sbytes + 3 * LL_TILE); };
    auto tbuf = [&](int j) { return sm + a.lay.off_T + j * LL_TILE; };

    if (tid == 0) {
        for (int i = 0; i < nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&stage_free[i], totals ? 1 : 2);  // MMA commit (+ output warps, main)
        }
        for (int i = 0; i < LL_RING; ++i) {
            mbar_init(&r_full[i], 1);
            mbar_init(&r_free[i], 4);
        }
        mbar_init(scores_done, 1);
        mbar_init(a_free, 4);
        mbar_init(&p_ready[0], 1);
        mbar_init(&p_ready[1], 1);
        mbar_init(state_done, 1);
        mbar_init(ps_read, 4);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&t_formed[i], 1);
            mbar_init(&c_done[i], 1);
        }
        mbar_init(drain, 1);
        mbar_init(totals_done, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);

    // ---- fixed levels j >= p: sums of whole earlier segments (main pass) ----
    if (!totals && warp >= 8 && warp < 12) {
        const int tt = tid - 256, m = tt >> 1, h = tt & 1;
        for (int j = a.p; j < a.nlev; ++j) {
            if (!((tile0 >> j) & 1)) continue;
            const int b = j - a.p;
            const int g0 = (seg >> (b + 1)) << (b + 1), cnt = 1 << b;
            float acc[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = 0.f;
            for (int g = g0; g < g0 + cnt; ++g) {
                const float4 *src = (const float4 *)(a.ws_G + (((size_t)g * a.BH + head) * LL_D + m) * LL_D + 32 * h);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v4 = src[q];
                    acc[4 * q] += v4.x; acc[4 * q + 1] += v4.y; acc[4 * q + 2] += v4.z; acc[4 * q + 3] += v4.w;
                }
            }
            uint8_t *row = tbuf(j) + m * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ck = 4 * h + q;
                *(uint4 *)(row + ((ck ^ (m & 7)) << 4)) =
                    make_uint4(pack_bf16x2(acc[8 * q], acc[8 * q + 1]), pack_bf16x2(acc[8 * q + 2], acc[8 * q + 3]),
                               pack_bf16x2(acc[8 * q + 4], acc[8 * q + 5]), pack_bf16x2(acc[8 * q + 6], acc[8 * q + 7]));
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0, s = 0, ph = 0;
            for (int i = 0; i < nloc; ++i) {
                if (i >= nst && !wait_phase(&stage_free[s], ph ^ 1, ctl)) break;
                const int row = (tile0 + i) * LL_C;
                const int rows = min(LL_C, a.L - row);
                const uint32_t lam_bytes = totals ? 0u : (uint32_t)(rows * NL * 4);
                mbar_arrive_expect_tx(&full[s], (totals ? 2 : 3) * LL_TILE + lam_bytes);
                if (!totals) {
                    tma_load_3d(stage_q(s), &a.tm_q, 0, row, head, &full[s]);
                    bulk_load((void *)stage_l(s), a.lam + ((size_t)head * a.L + row) * NL, lam_bytes, &full[s]);
                }
                tma_load_3d(stage_k(s), &a.tm_k, 0, row, head, &full[s]);
                tma_load_3d(stage_v(s), &a.tm_v, 0, row, head, &full[s]);
                issued = i + 1;
                if (++s == nst) { s = 0; ph ^= 1; }
            }
            for (int i = (issued > nst ? issued - nst : 0); i < issued; ++i) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_sleep(&full[i % nst], (i / nst) & 1, 200000u))
                    if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Main pass, software-pipelined by one chunk: iteration i issues the scores and the
        // state update of chunk i + 1 before the level products and P V of chunk i, so the
        // P and block-closing warps work a chunk ahead of the output warps.
        if (lane == 0) {
            constexpr uint32_t ID_SC = idesc_bf16_f32(64, 64, 0, 0);
            constexpr uint32_t ID_ST = idesc_bf16_f32(64, 64, 1, 1);
            constexpr uint32_t ID_AB = idesc_bf16_f32(64, 64, 0, 1);
            const uint64_t dP0 = smem_desc(smem_u32(sm + a.lay.off_P), 16, 1024);
            const uint64_t dT0 = smem_desc(smem_u32(tbuf(0)), LL_TILE, 1024);
            // descriptor start addresses advance 16 bytes per unit: +2 is one K16 step of a
            // K-major tile (32 bytes), +128 one of an MN-major tile (2048 bytes)
            auto dK_k = [&](int s) { return smem_desc(smem_u32(stage_k(s)), 16, 1024); };
            auto dK_m = [&](int s) { return smem_desc(smem_u32(stage_k(s)), LL_TILE, 1024); };
            auto dV_m = [&](int s) { return smem_desc(smem_u32(stage_v(s)), LL_TILE, 1024); };
            auto dQ_k = [&](int s) { return smem_desc(smem_u32(stage_q(s)), 16, 1024); };
            bool ok = true;
            if (totals) {
                int s = 0, ph = 0;
                for (int i = 0; i < nloc && ok; ++i) {
                    if (!wait_phase(&full[s], ph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dKm = dK_m(s), dVm = dV_m(s);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tmem + LT_PS, dKm + 128 * ks, dVm + 128 * ks, ID_ST, (i > 0) || (ks > 0));
                    mma_commit(&stage_free[s]);
                    if (++s == nst) { s = 0; ph ^= 1; }
                }
                mma_commit(totals_done);
            } else {
                // scores and state of chunk i (stage sl, phase pl)
                auto front = [&](int i, int sl, int pl) -> bool {
                    if (!wait_phase(&full[sl], pl, ctl)) return false;
                    tc_fence_after();
                    const uint64_t dQ = dQ_k(sl), dKk = dK_k(sl), dKm = dK_m(sl), dVm = dV_m(sl);
                    if (i >= 1 && !wait_phase(a_free, (i - 1) & 1, ctl)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) mma_ss(tmem + LT_A, dQ + 2 * ks, dKk + 2 * ks, ID_SC, ks > 0);
                    mma_commit(scores_done);
                    if (i >= 1 && !wait_phase(ps_read, (i - 1) & 1, ctl)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tmem + LT_PS, dKm + 128 * ks, dVm + 128 * ks, ID_ST, (i > 0) || (ks > 0));
                    mma_commit(state_done);
                    return true;
                };
                int s = 0;                           // stage of chunk i
                int s1 = 1 % nst, ph1 = (1 == nst) ? 1 : 0;  // stage of chunk i + 1
                int kr = 0, slot = 0;                // ring uses so far, next slot
                // one product into the next ring slot (4 x K16 MMAs), its slot known to be free
                auto issue = [&](uint64_t dA, uint64_t dB) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tmem + LT_R + 64 * slot, dA + 2 * ks, dB + 128 * ks, ID_AB, ks > 0);
                    mma_commit(&r_full[slot]);
                    ++kr;
                    if (++slot == LL_RING) slot = 0;
                };
                // wait until the slots of the next n products are free: the output warps free
                // the slots in order, so the last one being free means all of them are
                auto slots_free = [&](int n) -> bool {
                    const int kl = kr + n - 1;
                    if (kl >= LL_RING && !wait_phase(&r_free[kl % LL_RING], ((kl / LL_RING) - 1) & 1, ctl))
                        return false;
                    tc_fence_after();
                    return true;
                };
                ok = front(0, 0, 0);
                for (int i = 0; i < nloc && ok; ++i) {
                    const int b = i & 1;
                    if (i + 1 < nloc && !front(i + 1, s1, ph1)) { ok = false; break; }
                    const uint64_t dQ = dQ_k(s), dVm = dV_m(s);
                    // P V first: its P was written a chunk ahead
                    if (!wait_phase(&p_ready[b], (i >> 1) & 1, ctl)) { ok = false; break; }
                    if (!slots_free(1)) { ok = false; break; }
                    issue(dP0 + (uint64_t)(b * (LL_TILE >> 4)), dVm);
                    if (i >= 1 && !wait_phase(&t_formed[(i - 1) & 3], ((i - 1) >> 2) & 1, ctl)) { ok = false; break; }
                    // set bits of the chunk index, lowest first (one product each), in batches of
                    // up to LL_RING behind one wait; the block of level 0 (chunk i - 1, i odd)
                    // sits in its second tile when bit 1 of i is set
                    uint32_t bits = (uint32_t)(tile0 + i) & ((1u << a.nlev) - 1u);
                    while (bits && ok) {
                        const int nb = min(__popc(bits), LL_RING);
                        if (!slots_free(nb)) { ok = false; break; }
                        for (int n = 0; n < nb; ++n, bits &= bits - 1u) {
                            const int j = __ffs(bits) - 1;
                            const int jt = (j == 0 && ((i >> 1) & 1)) ? a.nlev : j;
                            issue(dQ, dT0 + (uint64_t)(jt * (LL_TILE >> 4)));
                        }
                    }
                    if (!ok) break;
                    mma_commit(&c_done[i & 3]);
                    mma_commit(&stage_free[s]);
                    s = s1;
                    if (++s1 == nst) { s1 = 0; ph1 ^= 1; }
                }
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_sleep(drain, 0, 200000u))
                if (globaltimer() - t0 > ctl.timeout_ns) break;
        }
    } else if (warp >= 4 && warp < 8 && !totals) {
        // ------------------------------------------------------------ scores -> P (intra mask)
        // Each thread owns half of two rows, ta = 16 q4 + lane/4 and tb = ta + 8: columns
        // 8k + 2 (lane % 4) and the next one (k = 0..7), as a 16x256b TMEM load delivers them.
        const int q4 = warp & 3, pt = tid - 128;
        const int cpos = lane & 3;
        const int trow[2] = {16 * q4 + (lane >> 2), 16 * q4 + 8 + (lane >> 2)};
        const uint32_t tA = tmem + LT_A + ((uint32_t)(32 * q4) << 16);
        int s = 0, ph = 0;
        for (int i = 0; i < nloc; ++i) {
            if (!group_wait(pt == 0, 2, scores_done, i & 1, &full[s], ph, true, ctl)) break;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld16x256_x8(tA, r);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_free);
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                // lambda_t^(l) for the intra levels 0..6.  Column block k (8 keys) against row
                // block t8: below the diagonal the level is 4 + floor(log2(k ^ t8)), on it
                // 1 + floor(log2(e ^ t7)) (0 on the diagonal element).
                const int t = trow[hr], t8 = t >> 3, t7 = t & 7;
                const bool valid = (tile0 + i) * LL_C + t < a.L;
                const float *lrow = stage_l(s) + t * NL;
                float lw[LL_LOG2C + 1];
#pragma unroll
                for (int l = 0; l <= LL_LOG2C; ++l) lw[l] = valid ? lrow[l] : 0.f;
                uint8_t *prow = sm + a.lay.off_P + (i & 1) * LL_TILE + t * 128 + 4 * cpos;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float x0 = __uint_as_float(r[4 * k + 2 * hr]), x1 = __uint_as_float(r[4 * k + 2 * hr + 1]);
                    float v0 = 0.f, v1 = 0.f;
                    if (k < t8) {
                        const int x = k ^ t8;
                        const float w = x >= 4 ? lw[6] : (x >= 2 ? lw[5] : lw[4]);
                        v0 = x0 * w;
                        v1 = x1 * w;
                    } else if (k == t8) {
                        const int e0 = 2 * cpos, e1 = e0 + 1;
                        const int y0 = e0 ^ t7, y1 = e1 ^ t7;
                        const float w0 = y0 == 0 ? lw[0] : (y0 >= 4 ? lw[3] : (y0 >= 2 ? lw[2] : lw[1]));
                        const float w1 = y1 == 0 ? lw[0] : (y1 >= 4 ? lw[3] : (y1 >= 2 ? lw[2] : lw[1]));
                        v0 = e0 <= t7 ? x0 * w0 : 0.f;
                        v1 = e1 <= t7 ? x1 * w1 : 0.f;
                    }
                    *(uint32_t *)(prow + ((k ^ (t & 7)) << 4)) = pack_bf16x2(v0, v1);
                }
            }
            fence_async_smem();
            named_bar(2, 128);
            if (pt == 0) mbar_arrive(&p_ready[i & 1]);
            if (++s == nst) { s = 0; ph ^= 1; }
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ close Fenwick blocks
        const int q4 = warp & 3, ct = tid - 256;
        const int m = 16 * q4 + (lane & 15);
        const bool row_lane = lane < 16;
        const uint32_t tP = tmem + LT_PS + ((uint32_t)(32 * q4) << 16);
        if (totals) {
            if (group_wait(ct == 0, 4, totals_done, 0, nullptr, 0, false, ctl)) {
                tc_fence_after();
                uint32_t r0[32], r1[32];
                tmem_ld32(tP, r0);
                tmem_ld32(tP + 32, r1);
                tmem_wait_ld();
                if (row_lane) {
                    float4 *dst = (float4 *)(a.ws_G + (((size_t)seg * a.BH + head) * LL_D + m) * LL_D);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1]),
                                             __uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3]));
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[8 + q] = make_float4(__uint_as_float(r1[4 * q]), __uint_as_float(r1[4 * q + 1]),
                                                 __uint_as_float(r1[4 * q + 2]), __uint_as_float(r1[4 * q + 3]));
                }
            }
        } else {
            // each thread: half of rows ma = 16 q4 + lane/4 and mb = ma + 8 (16x256b loads)
            const int cpos = lane & 3;
            const int mrow[2] = {16 * q4 + (lane >> 2), 16 * q4 + 8 + (lane >> 2)};
            for (int i = 0; i < nloc; ++i) {
                if (!group_wait(ct == 0, 4, state_done, i & 1, nullptr, 0, false, ctl)) break;
                tc_fence_after();
                uint32_t r[32];
                tmem_ld16x256_x8(tP, r);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ps_read);
                const int x = i + 1;  // position after this chunk
                // The tile about to be overwritten was last read by the level products of chunk
                // x - 2^r - 1 <= i - 2 (r >= 1), or, for level 0 with its two tiles, of chunk
                // i - 3: wait until chunk i - 2's products are done.  (Waiting on every chunk also
                // keeps t_formed at most two chunks ahead of the MMA issuer, which its four
                // barriers allow.)
                if (i >= 2 &&
                    !group_wait(ct == 0, 4, &c_done[(i - 2) & 3], ((i - 2) >> 2) & 1, nullptr, 0, false, ctl))
                    break;
                if (x < nloc) {
                    const int d = __popc(x), r_ = __ffs(x) - 1;
                    // T_r = PS(x) - PS(x - 2^r); PS(x - 2^r) is the snapshot at depth d - 1.
                    // PS(x) becomes the snapshot at depth d: a later block reads it back when
                    // it closes at a position one level below x (none does if x is odd).
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int m = mrow[hr];
                        const float *stk = a.ws_stack + (size_t)blockIdx.x * a.p * LL_D * LL_D + (size_t)m * LL_D + 2 * cpos;
                        const float *src = stk + (size_t)(d >= 2 ? d - 2 : 0) * LL_D * LL_D;
                        float *dst = (float *)stk + (size_t)(d - 1) * LL_D * LL_D;
                        // level 0 alternates between its two tiles (bit 1 of x)
                        uint8_t *row = tbuf((r_ == 0 && ((x >> 1) & 1)) ? a.nlev : r_) + m * 128 + 4 * cpos;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float v0 = __uint_as_float(r[4 * k + 2 * hr]), v1 = __uint_as_float(r[4 * k + 2 * hr + 1]);
                            if (r_ >= 1) *(float2 *)(dst + 8 * k) = make_float2(v0, v1);
                            if (d >= 2) {
                                const float2 u = *(const float2 *)(src + 8 * k);
                                v0 -= u.x;
                                v1 -= u.y;
                            }
                            *(uint32_t *)(row + ((k ^ (m & 7)) << 4)) = pack_bf16x2(v0, v1);
                        }
                    }
                }
                fence_async_smem();
                named_bar(4, 128);
                if (ct == 0) mbar_arrive(&t_formed[i & 3]);
            }
        }
    } else if (warp >= 12 && !totals) {
        // ------------------------------------------------------------ combine + store rows
        // Each thread owns half of two rows, ta = 16 q4 + lane/4 and tb = ta + 8: columns
        // 8k + 2 (lane % 4) and the next one (k = 0..7), as a 16x256b TMEM load delivers them.
        const int q4 = warp & 3, ot = tid - 384;
        const int cpos = lane & 3;
        const int trow[2] = {16 * q4 + (lane >> 2), 16 * q4 + 8 + (lane >> 2)};
        const uint32_t lq = (uint32_t)(32 * q4) << 16;
        int slot = 0, rph = 0, s = 0, ph = 0;
        for (int i = 0; i < nloc; ++i) {
            const int c = tile0 + i;
            bool valid[2];
            const float *lrow[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) valid[hr] = c * LL_C + trow[hr] < a.L;
            // the stage holds this chunk's lambda rows
            if (!group_wait(ot == 0, 3, &full[s], ph, nullptr, 0, false, ctl)) break;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) lrow[hr] = stage_l(s) + trow[hr] * NL + 1 + LL_LOG2C;  // lambda_t^(7 + j) at [j]
            float acc[32];  // register 4k + 2 hr + e of the loads: row trow[hr], column 8k + 2 cpos + e
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = 0.f;
            bool ok = true;
            // products in issue order: P V (weight 1), then R_j for the set bits j of c
            uint32_t bits = (uint32_t)c & ((1u << a.nlev) - 1u);
            for (int j = -1;;) {  // j = -1: P V
                if (!group_wait(ot == 0, 3, &r_full[slot], rph, nullptr, 0, false, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float wa = j < 0 ? 1.f : (valid[0] ? lrow[0][j] : 0.f);
                const float wb = j < 0 ? 1.f : (valid[1] ? lrow[1][j] : 0.f);
                uint32_t r[32];
                tmem_ld16x256_x8(tmem + LT_R + 64 * slot + lq, r);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&r_free[slot]);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    acc[4 * k] = fmaf(wa, __uint_as_float(r[4 * k]), acc[4 * k]);
                    acc[4 * k + 1] = fmaf(wa, __uint_as_float(r[4 * k + 1]), acc[4 * k + 1]);
                    acc[4 * k + 2] = fmaf(wb, __uint_as_float(r[4 * k + 2]), acc[4 * k + 2]);
                    acc[4 * k + 3] = fmaf(wb, __uint_as_float(r[4 * k + 3]), acc[4 * k + 3]);
                }
                if (++slot == LL_RING) { slot = 0; rph ^= 1; }
                if (!bits) break;
                j = __ffs(bits) - 1;
                bits &= bits - 1u;
            }
            if (!ok) break;
            // every output thread is past its lambda reads: the stage may be refilled
            named_bar(3, 128);
            if (ot == 0) mbar_arrive(&stage_free[s]);
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                if (!valid[hr]) continue;
                uint32_t *dst = (uint32_t *)(a.out + ((size_t)head * a.L + c * LL_C + trow[hr]) * LL_D) + cpos;
#pragma unroll
                for (int k = 0; k < 8; ++k) dst[4 * k] = pack_bf16x2(acc[4 * k + 2 * hr], acc[4 * k + 2 * hr + 1]);
            }
            if (++s == nst) { s = 0; ph ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int ll_levels(int nch)
{
    int n = 0;
    while ((1 << n) < nch) ++n;
    return n;
}

// segment = 2^p chunks: as few CTAs per head as fill the GPU, at most 32 segments per head
void ll_split(int BH, int nch, int num_sms, int *p_out, int *nseg_out)
{
    const int nlev = ll_levels(nch);
    const int maxseg = max(1, min(32, num_sms / BH));
    int p = 0;
    while (p < nlev && ((nch + (1 << p) - 1) >> p) > maxseg) ++p;
    *p_out = p;
    *nseg_out = (nch + (1 << p) - 1) >> p;
}

size_t ll_workspace(int BH, int nseg, int p)
{
    const size_t st = (size_t)LL_D * LL_D * sizeof(float);
    return (size_t)(nseg - 1) * BH * st + (size_t)BH * nseg * p * st;
}

}  // namespace

bool tcl_supported(const Problem &p)
{
    if (!(p.dtype == LA_BF16 && p.lam && p.fm == LA_FM_IDENTITY && !p.normalize && p.dk == LL_D &&
          p.dv == LL_D && p.C == LL_C && p.L >= 2 * LL_C))
        return false;
    const int nch = (p.L + LL_C - 1) / LL_C;
    if (ll_levels(nch) > LL_MAXLEV) return false;
    // lambda rows are copied in bulk: every chunk's rows must start and end on 16 bytes
    if (p.nl > LL_MAXNL || ((long long)p.L * p.nl) % 4 != 0) return false;
    return true;
}

int tcl_plan(const Problem &p, int num_sms, la_plan_info *info)
{
    const int nch = (p.L + LL_C - 1) / LL_C, BH = p.B * p.H;
    int pp = 0, nseg = 1;
    ll_split(BH, nch, num_sms, &pp, &nseg);
    info->grid_x = BH * nseg;
    info->grid_y = 1;
    info->block = LL_THREADS;
    info->smem_bytes = ll_layout(ll_levels(nch)).alloc;
    info->n_launches = nseg > 1 ? 2 : 1;
    info->workspace_bytes = ll_workspace(BH, nseg, pp);
    return LA_OK;
}

int tcl_launch(const Problem &p, int num_sms)
{
    if (!tcl_supported(p)) return LA_ERR_UNSUPPORTED;
    if (((uintptr_t)p.lam & 15) != 0) return LA_ERR_UNSUPPORTED;
    LlArgs a;
    memset(&a, 0, sizeof(a));
    const int BH = p.B * p.H;
    if (!make_map(&a.tm_q, p.q, BH, p.L, LL_D, LL_C) || !make_map(&a.tm_k, p.k, BH, p.L, LL_D, LL_C) ||
        !make_map(&a.tm_v, p.v, BH, p.L, LL_D, LL_C))
        return LA_ERR_CUDA;
    a.lam = p.lam;
    a.out = (__nv_bfloat16 *)p.out;
    a.L = p.L;
    a.nch = (p.L + LL_C - 1) / LL_C;
    a.NL = p.nl;
    a.nlev = ll_levels(a.nch);
    ll_split(BH, a.nch, num_sms, &a.p, &a.nseg);
    a.seg_chunks = 1 << a.p;
    a.BH = BH;
    a.lay = ll_layout(a.nlev);
    a.err = p.err;
    a.timeout_ns = 2000000000ull;
    const char *e = getenv("LA_DEBUG_TIMEOUT_NS");
    if (e && *e) a.timeout_ns = strtoull(e, nullptr, 10);
    const size_t need = ll_workspace(BH, a.nseg, a.p);
    if (need) {
        if (!p.workspace || p.workspace_bytes < need) return LA_ERR_WORKSPACE;
        a.ws_G = (float *)p.workspace;
        a.ws_stack = a.ws_G + (size_t)(a.nseg - 1) * BH * LL_D * LL_D;
    }
    if (cudaFuncSetAttribute(tc_loglinear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, a.lay.alloc) !=
        cudaSuccess)
        return LA_ERR_CUDA;
    if (a.nseg > 1) {
        a.totals = 1;
        a.grid_seg = a.nseg - 1;
        tc_loglinear_kernel<<<BH * (a.nseg - 1), LL_THREADS, a.lay.alloc, p.stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    a.totals = 0;
    a.grid_seg = a.nseg;
    if (a.nseg > 1) {
        // starts while the totals pass drains
        if (launch_dependent(tc_loglinear_kernel, BH * a.nseg, LL_THREADS, a.lay.alloc, p.stream, a) != cudaSuccess)
            return LA_ERR_CUDA;
        return LA_OK;
    }
    tc_loglinear_kernel<<<BH * a.nseg, LL_THREADS, a.lay.alloc, p.stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace la
