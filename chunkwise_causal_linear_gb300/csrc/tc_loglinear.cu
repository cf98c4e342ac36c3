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
// Per chunk (all MMAs M = 64, N = 64, K = 64 as 4 x K16; bf16 in, fp32 accumulate):
//   scores  A   = Q K^T                      (A K-major, B K-major)
//   state   PS += K^T V                      (A = K MN-major, B = V MN-major)
//   inter   O  += (lambda^(7+j) . Q) T_j     per set bit j (A K-major from a ring, B MN-major)
//   intra   O  += P V,  P = lambda-masked A  (A K-major, B = V MN-major)
// Warps: 0 TMA producer, 1 MMA issuer, 2-3 write the lambda-scaled copies of Q into a ring
// of 4 tiles, 4-7 turn scores into P, 8-11 close the Fenwick blocks, 12-15 store output
// rows.  A group of four consecutive warps covers the four TMEM lane quadrants (warp % 4).
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
constexpr int LL_STAGES = 2;
constexpr int LL_D = 64, LL_C = 64, LL_LOG2C = 6;
constexpr int LL_RING = 4;
constexpr int LL_MAXLEV = 12;   // inter levels: up to 4096 chunks per head
constexpr int LL_MAXNL = 32;    // lambda entries per row held in shared memory
constexpr int LL_TILE = LL_C * 128;
constexpr int LL_LAMBUF = LL_C * LL_MAXNL * 4;            // 8 KB
constexpr int LL_STAGE_BYTES = 3 * LL_TILE + LL_LAMBUF;   // Q, K, V, lambda
constexpr int LL_N_BAR = 2 * LL_STAGES + 2 * LL_RING + 12;

// TMEM columns (M = 64 layout: row m at lane (m % 16) + 32 (m / 16))
constexpr uint32_t LT_PS = 0;     // running segment state PS [d_k rows][d_v]
constexpr uint32_t LT_A = 64;     // scores
constexpr uint32_t LT_O = 128;    // output, two buffers of 64 columns

struct LlLayout {
    int off_T, off_ring, off_P, off_bar, bytes, alloc;
};

inline LlLayout ll_layout(int nlev)
{
    LlLayout l;
    l.off_T = LL_STAGES * LL_STAGE_BYTES;
    l.off_ring = l.off_T + nlev * LL_TILE;
    l.off_P = l.off_ring + LL_RING * LL_TILE;
    l.off_bar = l.off_P + LL_TILE;
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
    uint64_t *full = bars;                        // [STAGES]
    uint64_t *stage_free = full + LL_STAGES;      // [STAGES]
    uint64_t *ring_full = stage_free + LL_STAGES; // [RING]
    uint64_t *ring_free = ring_full + LL_RING;    // [RING]
    uint64_t *scores_done = ring_free + LL_RING;
    uint64_t *a_free = scores_done + 1;
    uint64_t *p_ready = a_free + 1;
    uint64_t *state_done = p_ready + 1;
    uint64_t *ps_read = state_done + 1;           // PS copied out by the block-closing group
    uint64_t *t_formed = ps_read + 1;             // the block closed after a chunk is in smem
    uint64_t *o_done = t_formed + 1;              // [2]
    uint64_t *o_free = o_done + 2;                // [2]
    uint64_t *drain = o_free + 2;
    uint64_t *totals_done = drain + 1;
    uint32_t *tmem_slot = (uint32_t *)(sm + a.lay.off_bar + LL_N_BAR * 8);
    volatile int *abort_flag = (volatile int *)(sm + a.lay.off_bar + LL_N_BAR * 8 + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x / a.grid_seg, seg = blockIdx.x % a.grid_seg;
    const int tile0 = seg * a.seg_chunks;               // first chunk of the segment
    const int nloc = min(a.seg_chunks, a.nch - tile0);  // chunks in this segment
    const bool totals = a.totals != 0;
    const int NL = a.NL;
    Ctl ctl{abort_flag, a.err, a.timeout_ns};
    auto stage_q = [&](int s) { return sm + s * LL_STAGE_BYTES; };
    auto stage_k = [&](int s) { return stage_q(s) + LL_TILE; };
    auto stage_v = [&](int s) { return stage_q(s) + 2 * LL_TILE; };
    auto stage_l = [&](int s) { return (const float *)(stage_q(s) + 3 * LL_TILE); };
    auto tbuf = [&](int j) { return sm + a.lay.off_T + j * LL_TILE; };
    auto ring = [&](int r) { return sm + a.lay.off_ring + r * LL_TILE; };

    if (tid == 0) {
        for (int i = 0; i < LL_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&stage_free[i], 1);
        }
        for (int i = 0; i < LL_RING; ++i) {
            mbar_init(&ring_full[i], 1);
            mbar_init(&ring_free[i], 1);
        }
        mbar_init(scores_done, 1);
        mbar_init(a_free, 4);
        mbar_init(p_ready, 1);
        mbar_init(state_done, 1);
        mbar_init(ps_read, 4);
        mbar_init(t_formed, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&o_done[i], 1);
            mbar_init(&o_free[i], 4);
        }
        mbar_init(drain, 1);
        mbar_init(totals_done, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 256);

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
            int issued = 0;
            for (int i = 0; i < nloc; ++i) {
                const int s = i % LL_STAGES;
                if (i >= LL_STAGES && !wait_phase(&stage_free[s], ((i / LL_STAGES) - 1) & 1, ctl)) break;
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
            }
            for (int i = (issued > LL_STAGES ? issued - LL_STAGES : 0); i < issued; ++i) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_sleep(&full[i % LL_STAGES], (i / LL_STAGES) & 1, 200000u))
                    if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_SC = idesc_bf16_f32(64, 64, 0, 0);
            constexpr uint32_t ID_ST = idesc_bf16_f32(64, 64, 1, 1);
            constexpr uint32_t ID_AB = idesc_bf16_f32(64, 64, 0, 1);
            const uint32_t pa = smem_u32(sm + a.lay.off_P);
            int kq = 0;  // ring uses so far
            for (int i = 0; i < nloc; ++i) {
                const int s = i % LL_STAGES, b = i & 1;
                if (!wait_phase(&full[s], (i / LL_STAGES) & 1, ctl)) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(stage_q(s)), ka = smem_u32(stage_k(s)), va = smem_u32(stage_v(s));
                if (!totals) {
                    if (i >= 1 && !wait_phase(a_free, (i - 1) & 1, ctl)) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tmem + LT_A, smem_desc(qa + ks * 32, 16, 1024), smem_desc(ka + ks * 32, 16, 1024),
                               ID_SC, ks > 0);
                    mma_commit(scores_done);
                    if (i >= 1 && !wait_phase(ps_read, (i - 1) & 1, ctl)) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem + LT_PS, smem_desc(ka + ks * 2048, LL_TILE, 1024),
                           smem_desc(va + ks * 2048, LL_TILE, 1024), ID_ST, (i > 0) || (ks > 0));
                if (totals) {
                    mma_commit(&stage_free[s]);
                    continue;
                }
                mma_commit(state_done);
                if (i >= 1 && !wait_phase(t_formed, (i - 1) & 1, ctl)) break;
                if (i >= 2 && !wait_phase(&o_free[b], ((i >> 1) - 1) & 1, ctl)) break;
                tc_fence_after();
                const uint32_t tO = tmem + LT_O + 64 * b;
                const int c = tile0 + i;
                bool first = true, ok = true;
                for (int j = 0; j < a.nlev; ++j) {
                    if (!((c >> j) & 1)) continue;
                    const int slot = kq % LL_RING;
                    if (!wait_phase(&ring_full[slot], (kq / LL_RING) & 1, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ra = smem_u32(ring(slot)), tb = smem_u32(tbuf(j));
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tO, smem_desc(ra + ks * 32, 16, 1024), smem_desc(tb + ks * 2048, LL_TILE, 1024),
                               ID_AB, (!first) || (ks > 0));
                    mma_commit(&ring_free[slot]);
                    ++kq;
                    first = false;
                }
                if (!ok) break;
                if (!wait_phase(p_ready, i & 1, ctl)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tO, smem_desc(pa + ks * 32, 16, 1024), smem_desc(va + ks * 2048, LL_TILE, 1024), ID_AB,
                           (!first) || (ks > 0));
                mma_commit(&o_done[b]);
                mma_commit(&stage_free[s]);
            }
            if (totals) mma_commit(totals_done);
            mma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_sleep(drain, 0, 200000u))
                if (globaltimer() - t0 > ctl.timeout_ns) break;
        }
    } else if (warp >= 2 && warp < 4 && !totals) {
        // ------------------------------------------------------------ lambda-scaled copies of Q
        const int st = tid - 64, t = st;  // one row per thread
        int kq = 0;
        for (int i = 0; i < nloc; ++i) {
            const int c = tile0 + i, s = i % LL_STAGES;
            if (c == 0) continue;  // chunk 0 has no earlier blocks
            if (!group_wait(st == 0, 5, &full[s], (i / LL_STAGES) & 1, nullptr, 0, false, ctl, 64)) break;
            const bool valid = c * LL_C + t < a.L;
            const uint8_t *qrow = stage_q(s) + t * 128;
            const float *lrow = stage_l(s) + t * NL;
            bool ok = true;
            for (int j = 0; j < a.nlev; ++j) {
                if (!((c >> j) & 1)) continue;
                const int slot = kq % LL_RING;
                if (kq >= LL_RING &&
                    !group_wait(st == 0, 5, &ring_free[slot], ((kq / LL_RING) - 1) & 1, nullptr, 0, false, ctl, 64)) {
                    ok = false;
                    break;
                }
                const float w = valid ? lrow[1 + LL_LOG2C + j] : 0.f;
                uint8_t *dst = ring(slot) + t * 128;
#pragma unroll
                for (int ck = 0; ck < 8; ++ck) {
                    const int off = (ck ^ (t & 7)) << 4;
                    const uint4 x = *(const uint4 *)(qrow + off);
                    *(uint4 *)(dst + off) = make_uint4(pack_bf16x2(bf_lo(x.x) * w, bf_hi(x.x) * w),
                                                       pack_bf16x2(bf_lo(x.y) * w, bf_hi(x.y) * w),
                                                       pack_bf16x2(bf_lo(x.z) * w, bf_hi(x.z) * w),
                                                       pack_bf16x2(bf_lo(x.w) * w, bf_hi(x.w) * w));
                }
                fence_async_smem();
                named_bar(5, 64);
                if (st == 0) mbar_arrive(&ring_full[slot]);
                ++kq;
            }
            if (!ok) break;
        }
    } else if (warp >= 4 && warp < 8 && !totals) {
        // ------------------------------------------------------------ scores -> P (intra mask)
        const int q4 = warp & 3, pt = tid - 128;
        const int t = 16 * q4 + (lane & 15);
        const bool row_lane = lane < 16;
        const uint32_t tA = tmem + LT_A + ((uint32_t)(32 * q4) << 16);
        for (int i = 0; i < nloc; ++i) {
            const int s = i % LL_STAGES;
            if (!group_wait(pt == 0, 2, scores_done, i & 1, &full[s], (i / LL_STAGES) & 1, true, ctl)) break;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tA, r0);
            tmem_ld32(tA + 32, r1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_free);
            if (row_lane) {
                const bool valid = (tile0 + i) * LL_C + t < a.L;
                const float *lrow = stage_l(s) + t * NL;  // lambda_t^(0..6) by level
                uint8_t *prow = sm + a.lay.off_P + t * 128;
#pragma unroll
                for (int ck = 0; ck < 8; ++ck) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s0 = 8 * ck + 2 * e, s1 = s0 + 1;
                        const uint32_t *rr = s0 < 32 ? r0 : r1;
                        const float l0 = lrow[fenwick_level(t, s0)], l1 = lrow[fenwick_level(t, s1)];
                        const float v0 = (valid && s0 <= t) ? __uint_as_float(rr[s0 & 31]) * l0 : 0.f;
                        const float v1 = (valid && s1 <= t) ? __uint_as_float(rr[s1 & 31]) * l1 : 0.f;
                        w[e] = pack_bf16x2(v0, v1);
                    }
                    *(uint4 *)(prow + ((ck ^ (t & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_async_smem();
            named_bar(2, 128);
            if (pt == 0) mbar_arrive(p_ready);
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ close Fenwick blocks
        const int q4 = warp & 3, ct = tid - 256;
        const int m = 16 * q4 + (lane & 15);
        const bool row_lane = lane < 16;
        const uint32_t tP = tmem + LT_PS + ((uint32_t)(32 * q4) << 16);
        float *stack = a.ws_stack + (size_t)blockIdx.x * a.p * LL_D * LL_D + (size_t)m * LL_D;
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
            for (int i = 0; i < nloc; ++i) {
                if (!group_wait(ct == 0, 4, state_done, i & 1, nullptr, 0, false, ctl)) break;
                tc_fence_after();
                uint32_t r0[32], r1[32];
                tmem_ld32(tP, r0);
                tmem_ld32(tP + 32, r1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ps_read);
                const int x = i + 1;  // position after this chunk
                if (x < nloc && row_lane) {
                    const int d = __popc(x), r = __ffs(x) - 1;
                    // T_r = PS(x) - PS(x - 2^r); PS(x - 2^r) is the snapshot at depth d - 1.
                    // PS(x) becomes the snapshot at depth d: a later block reads it back when
                    // it closes at a position one level below x (none does if x is odd).
                    const float4 *src = (const float4 *)(stack + (size_t)(d >= 2 ? d - 2 : 0) * LL_D * LL_D);
                    float4 *dst = (float4 *)(stack + (size_t)(d - 1) * LL_D * LL_D);
                    uint8_t *row = tbuf(r) + m * 128;
#pragma unroll
                    for (int ck = 0; ck < 8; ++ck) {
                        const uint32_t *rr = ck < 4 ? r0 : r1;
                        const int i0 = (8 * ck) & 31;
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(rr[i0 + e]);
                        if (r >= 1) {
                            dst[2 * ck] = make_float4(v[0], v[1], v[2], v[3]);
                            dst[2 * ck + 1] = make_float4(v[4], v[5], v[6], v[7]);
                        }
                        if (d >= 2) {
                            const float4 u0 = src[2 * ck], u1 = src[2 * ck + 1];
                            v[0] -= u0.x; v[1] -= u0.y; v[2] -= u0.z; v[3] -= u0.w;
                            v[4] -= u1.x; v[5] -= u1.y; v[6] -= u1.z; v[7] -= u1.w;
                        }
                        *(uint4 *)(row + ((ck ^ (m & 7)) << 4)) =
                            make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                       pack_bf16x2(v[6], v[7]));
                    }
                }
                fence_async_smem();
                named_bar(4, 128);
                if (ct == 0) mbar_arrive(t_formed);
            }
        }
    } else if (warp >= 12 && !totals) {
        // ------------------------------------------------------------ output rows -> global
        const int q4 = warp & 3, ot = tid - 384;
        const int t = 16 * q4 + (lane & 15);
        const bool row_lane = lane < 16;
        for (int i = 0; i < nloc; ++i) {
            const int b = i & 1;
            const int row = (tile0 + i) * LL_C + t;
            if (!group_wait(ot == 0, 3, &o_done[b], (i >> 1) & 1, nullptr, 0, false, ctl)) break;
            tc_fence_after();
            const uint32_t tO = tmem + LT_O + 64 * b + ((uint32_t)(32 * q4) << 16);
            uint32_t r0[32], r1[32];
            tmem_ld32(tO, r0);
            tmem_ld32(tO + 32, r1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[b]);
            if (row_lane && row < a.L) {
                uint4 *dst = (uint4 *)(a.out + ((size_t)head * a.L + row) * LL_D);
#pragma unroll
                for (int ck = 0; ck < 8; ++ck) {
                    const uint32_t *rr = ck < 4 ? r0 : r1;
                    const int i0 = (8 * ck) & 31;
                    dst[ck] = make_uint4(pack_bf16x2(__uint_as_float(rr[i0]), __uint_as_float(rr[i0 + 1])),
                                         pack_bf16x2(__uint_as_float(rr[i0 + 2]), __uint_as_float(rr[i0 + 3])),
                                         pack_bf16x2(__uint_as_float(rr[i0 + 4]), __uint_as_float(rr[i0 + 5])),
                                         pack_bf16x2(__uint_as_float(rr[i0 + 6]), __uint_as_float(rr[i0 + 7])));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
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
    tc_loglinear_kernel<<<BH * a.nseg, LL_THREADS, a.lay.alloc, p.stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace la
