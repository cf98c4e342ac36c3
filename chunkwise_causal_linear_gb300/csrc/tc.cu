// tc.cu -- single-pass tensor-core path for chunkwise causal linear attention (sm_103a).
//
// One CTA per (b, h) head sweeps the head's chunks in order ("attention と線形の間",
// section 2, Chunked): for chunk c the output is the carried state read by the chunk's
// queries (inter) plus the causally masked in-chunk scores times the chunk's values
// (intra); then the chunk's phi(K)^T V joins the state.  The normaliser of "Linear
// Attention / Performerの理論と実装" (y_t = phi(q_t)^T S_t / phi(q_t)^T z_t) is carried
// beside it: z_c = sum of phi(k) over the chunks before c, kept in fp32.
//
// GB300 mapping (everything stays on chip except q, k, v in and out):
//   * warp 0       TMA producer: Q_c, K_c, V_c tiles (128-byte swizzled) into a ring of four
//                  stages (three where four do not fit in shared memory).
//   * warp 1       one thread issues every tcgen05.mma; the warp owns the TMEM allocation.
//   * warps 2-4, 6-8, 10-11 (not on the MMA issuer's sub-partition)
//                  feature map phi applied in place in shared memory; with the normaliser,
//                  the fp32 column sums of phi(K_c) update z, and z_c is written (as a bf16
//                  hi/lo pair) into two extra rows after the chunk's 64 key rows, so the
//                  scores MMA also returns phi(q_t).z_c in fp32.
//   * warps 12-15  scores -> P: read the scores row from TMEM, causal mask (diagonal kept),
//                  fp32 row sum, 1 / (phi(q_t).z_c + row sum) for the normaliser, bf16 P
//                  into one of two shared-memory P tiles; after each state update, S^T (fp32
//                  in TMEM) -> its bf16 copy in TMEM.
//   * warps 16-19  output epilogue: O^T from TMEM, normaliser, bf16 rows stored from
//                  registers (a warp writes 64 contiguous bytes of a row per store).
// With dv = 64 the dv-row accumulators use the M = 64 lane layout (row m in lane
// m%16 + 32*(m/16)), which is also where an M = 64 A operand is read from in TMEM.
// TMEM (512 columns): S^T fp32 [dv lanes x D] | S^T bf16 [dv x D/2] | O^T x2 [dv x C] |
// scores x2 [C x (C + 8)].  The state is accumulated in fp32 by the MMA and never leaves
// TMEM; the inter-chunk product reads its bf16 copy as the A operand straight from TMEM.
//
// Rows move in 64-row tiles (TMA box, MMA tile).  The chunk size CH is 16, 32 or 64: a tile
// holds 64/CH chunks, each with its own inter product (from the state at the chunk's start),
// its own state update and its own bf16 state copy, while the intra part of the tile uses
// a block-diagonal causal mask at CH granularity.  The normaliser does not depend on CH: it
// is phi(q_t).z at the tile start plus the causal row sum inside the tile.
//
// MMAs per tile (bf16 in, fp32 accumulate), D = feature dim, T = 64:
//   scores  A     = phi(Q_T) [phi(K_T); z]^T     M=T   N=T(+8)  K=D   once per tile
//   inter   O^T_j = bf16(S_j)^T phi(Q_j)^T       M=dv  N=CH     K=D   per chunk j (A in TMEM)
//   state   S^T  += V_j^T phi(K_j)               M=dv  N=D      K=CH  per chunk j
//   intra   O^T  += V_T^T P_T^T                  M=dv  N=T      K=T   once per tile
// The MMA thread issues, per tile c: inter and state of c, the scores of c+1, the intra product
// of c (with four chunks per tile, the scores of c first).  The P warps then find the next
// scores ready when they finish a tile, so the chain scores -> P -> intra does not wait for
// each intra product to be issued; the fourth ring stage absorbs the longer hold of a stage
// (its stage is released when the intra product completes, after the next tile's phi).
//
// Decay (the Retention update S_t = gamma S_{t-1} + phi(k_t) v_t^T of "Linear Attention /
// Performerの理論と実装", one chunk per tile): with i, j the rows of the chunk,
//     y_i = gamma^(i+1) phi(q_i) S + sum_{j<=i} gamma^(i-j) (phi(q_i).phi(k_j)) v_j.
// The feature-map group writes K~_j = gamma^(C-1-j) phi(k_j), so the unmasked scores carry
// gamma^(C-1-j); the state copy that the inter product reads is gamma^C S, so the sum that
// lands in O^T is gamma^(C-1-i) y_i and the epilogue multiplies by gamma^(i+1-C) (with the
// normaliser the factor cancels: z rides along as gamma^C z, and den gets the same
// factor).  The fp32 accumulator A is rescaled in TMEM (load, scale, store back) only
// once every P chunks.  Inside a period, chunk m = 0..P-1 scales its keys by a further
// gamma^(-C m); so that its scores, its inter product and its normaliser share that
// factor, it reads the state copy gamma^(C (1-m)) S and the z rows gamma^(C (1-m)) z, and
// the unnormalised epilogue multiplies by gamma^(i+1-C+C m).  After the update of chunk m,
// A = gamma^(-C m) S_m, which is exactly the copy chunk m+1 needs; at the period's end the
// readback scales A by gamma^(C P) (= gamma^C S), stores it back and copies it.  P is the
// largest period with gamma^(C P) >= 2^-64 (at least 1, as gamma^C >= 2^-64), so every
// factor used here, gamma^(C P) included, is a normal fp32 number (the factors come from
// the flush-to-zero hardware ex2), and every scaled key, A and the copy stay well inside
// the fp32 / bf16 range.  The totals pass scales each
// key by gamma^(segment end - s) instead and needs no rescaling of the accumulator; a
// segment starts from sum_g gamma^(rows after segment g) T_g.
//
// Every mbarrier wait is bounded (wall-clock limit); on expiry the CTA records
// LA_ERR_TIMEOUT in the device error word, raises a shared abort flag that the other roles
// poll, drains its own async copies / MMAs, frees TMEM and exits.
#include <stdio.h>
#include <stdlib.h>

#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace la {

using namespace ptx;
using namespace tcc;

namespace {

constexpr int TC_THREADS = 640;
constexpr int TC_FWARPS = 8;  // warps in the feature-map group

// The feature-map group is warps 2, 3, 4, 6, 7, 8, 10, 11: none shares a sub-partition
// (warp % 4) with the MMA issuer (warp 1), whose single issuing thread would otherwise
// compete with two busy feature-map warps for issue slots.  Returns the warp's rank in
// the group, or -1.
__device__ __forceinline__ int phi_rank(int warp)
{
    if (warp < 2 || warp >= 12 || (warp & 3) == 1) return -1;
    return warp - 2 - (warp > 5) - (warp > 9);
}
constexpr int TC_DEN = 4;  // ring of per-chunk 1/den vectors

struct TcArgs {
    CUtensorMap tm_q, tm_k, tm_v;
    void *out;   // [BH][L][DV], bf16 (fp32 in the fp32-output mode); rows stored from registers
    int L, nch;  // nch: number of 64-row tiles of a head
    int nsub;    // number of chunks of CH rows of a head
    // Sequence split: a head's tiles are cut into segments of seg_tiles tiles, one CTA each.
    // The totals pass writes each segment's sum of phi(K)^T V (as S^T rows) and of phi(K);
    // the main pass starts segment g from the sum of the totals of segments 0..g-1.
    int seg_tiles;
    int grid_seg;    // segments per head in this launch's grid
    int totals;      // 1: totals pass
    int BH;
    float *ws_T;     // [segments-1][BH][dv][D]
    float *ws_z;     // [segments-1][BH][D]
    int *err;
    unsigned long long timeout_ns;
    int debug_stall;  // test knob: the feature-map group never signals (forces a timeout)
    // Non-causal (bidirectional) main pass: every segment starts from the sum of all nseg_all
    // segments' totals, the state is never updated, and P is zero, so each row gets exactly
    // phi(q) S_total (/ phi(q) z_total).
    int noncausal, nseg_all;
    float l2g;  // decay: log2(gamma)
    int anti;   // anti-causal pass (identity features, no normaliser, C = 64): see the kernel
    int esyn;   // q = k = e (1, 0, ..., 0) rows: constant tiles, only V loaded (see the kernel)
    const float *S0, *z0;  // NULL, or the state before row 0 ([BH][D][DV], [BH][D])
    int period; // decay: chunks between rescalings of the fp32 state accumulator (P)
};

// kernel modes (TC_F32OUT: causal, output stored as fp32 rows; TC_DECAY_F32OUT: both, for the
// backward pass of the decayed forward)
constexpr int TC_CAUSAL = 0, TC_NONCAUSAL = 1, TC_DECAY = 2, TC_F32OUT = 3, TC_DECAY_F32OUT = 4;

template <int D, int DV, int C, bool NORM, bool F32O = false>
struct TcLayout {
    static constexpr int KROWS = NORM ? C + 8 : C;    // key rows (+ z hi/lo + zero rows)
    static constexpr int NSC = KROWS;                 // N of the scores MMA
    static constexpr int K_BLK = KROWS * 128;         // one 64-feature block of the K tile
    static constexpr int Q_BYTES = C * D * 2;
    static constexpr int K_BYTES = (D / 64) * K_BLK;
    static constexpr int V_BYTES = C * DV * 2;
    static constexpr int STAGE_BYTES = Q_BYTES + K_BYTES + V_BYTES;
    static constexpr int STAGE_TX = Q_BYTES + C * D * 2 + V_BYTES;  // bytes TMA delivers
    static constexpr int P_BYTES = C * C * 2;
    // P is double-buffered (tile c in buffer c & 1): the scores of tile c+1 are issued before
    // the intra product of tile c, and the commit after them also covers the intra product
    // of tile c-1, the last reader of buffer (c+1) & 1.  fp32-output mode: each buffer holds
    // a bf16 hi tile and a lo tile (P - hi).
    static constexpr int P_SET = (F32O ? 2 : 1) * P_BYTES;
    // floats: rden[TC_DEN][C], z[D], zpart[TC_FWARPS][D]
    static constexpr int N_F32 = TC_DEN * C + D + TC_FWARPS * D;
    static constexpr int F32_BYTES = ((N_F32 * 4 + 15) / 16) * 16;
    // everything but the stage ring: P, floats, barriers (at most 4 stages), misc, slack for
    // the 1024-byte alignment of the swizzled tiles
    static constexpr int FIXED = 2 * P_SET + F32_BYTES + (3 * 4 + 2 * 4 + 2 * TC_DEN + 3) * 8 + 16 + 1024;
    // the TMA ring: four stages where they fit in shared memory, else three
    static constexpr int STAGES = (4 * STAGE_BYTES + FIXED <= 232448) ? 4 : 3;
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_P = STAGES * STAGE_BYTES;
    static constexpr int OFF_F32 = OFF_P + 2 * P_SET;
    static constexpr int OFF_BAR = OFF_F32 + F32_BYTES;
    static constexpr int N_BAR = 3 * STAGES + 2 * 4 + 2 * TC_DEN + 3;
    static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
    // TMEM columns
    // fp32-output mode (no normaliser: scores are C = 64 columns): the state copy is a bf16
    // hi / lo pair, S^T fp32 | hi | lo | O^T x2 | scores x2 fills the 512 columns
    static constexpr uint32_t T_S = 0, T_SB = 128, T_SL = 192, T_O = F32O ? 256 : 192,
                              T_A = F32O ? 384 : 320, A_STRIDE = F32O ? 64 : 80;
    static_assert(D <= 128 && (DV == 64 || DV == 128), "tensor-core path: D <= 128, dv 64 or 128");
    static_assert(C == 64, "tensor-core path: 64-row tiles");
    static_assert(K_BLK % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms stay aligned");
    static_assert(ALLOC <= 232448, "shared memory budget");
};

// 2^x on the SFU (hardware ex2, relative error ~2^-22, flush-to-zero): the decay factors
__device__ __forceinline__ float ex2(float x)
{
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x));
    return e;
}

template <int D, int DV, int CH, int FM, bool NORM, int MODE>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_chunked_kernel(const __grid_constant__ TcArgs a)
{
    constexpr int C = 64;           // rows per tile
    constexpr int NSUB = C / CH;    // chunks per tile
    constexpr bool NC = MODE == TC_NONCAUSAL;
    constexpr bool DK = MODE == TC_DECAY || MODE == TC_DECAY_F32OUT;
    constexpr bool FO = MODE == TC_F32OUT || MODE == TC_DECAY_F32OUT;
    static_assert(!DK || CH == C, "decay: one chunk per tile");
    static_assert(!FO || (FM == LA_FM_IDENTITY && !NORM), "fp32 output: identity features, no normaliser");
    // Anti-causal pass (row t reads the rows s >= t; used by the backward pass).  It is the
    // causal pass over the mirrored sequence v = L-1-t, run in mirrored order: virtual tile c
    // is the box of rows L - 64 (c+1) .. L - 64 c - 1 (a negative start reads zeros), and
    // smem row r of a tile is virtual row 63 - r of it.  Segments, totals, their prefix and the
    // decay periods all stay in virtual order; only the loads, the causal mask (s >= t in smem
    // order), the decay's in-tile factors and the rows stored change.
    const bool anti = FM == LA_FM_IDENTITY && !NORM && !NC && CH == C && a.anti != 0;
    // Constant rows e = (1, 0, ..., 0) as both Q and K (the backward pass's prefix and suffix
    // sums, sum_{s<=t} v_s): written once into every stage, never loaded.  No decay (its
    // feature-map warps would rescale the K tiles in place).
    const bool esyn = FM == LA_FM_IDENTITY && !NORM && !NC && !DK && a.esyn != 0;
    using Lay = TcLayout<D, DV, C, NORM, FO>;
    constexpr int ST = Lay::STAGES;  // TMA ring depth
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the 128B-swizzled tiles (offset taken in the shared window)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *f32 = (float *)(sm + Lay::OFF_F32);
    float *rden = f32;                   // [TC_DEN][C]  1 / den per row of a chunk
    float *zs = rden + TC_DEN * C;       // [D]
    float *zpart = zs + D;               // [TC_FWARPS][D]
    uint64_t *bars = (uint64_t *)(sm + Lay::OFF_BAR);
    uint64_t *full = bars;                           // [S] TMA -> feature map
    uint64_t *phi_ready = full + ST;          // [S] feature map -> MMA
    uint64_t *stage_free = phi_ready + ST;    // [S] MMA -> TMA
    uint64_t *scores_done = stage_free + ST;  // [2]
    uint64_t *p_ready = scores_done + 2;             // [2]
    uint64_t *o_done = p_ready + 2;                  // [2]
    uint64_t *o_free = o_done + 2;                   // [2]
    uint64_t *den_full = o_free + 2;                 // [TC_DEN]
    uint64_t *den_empty = den_full + TC_DEN;         // [TC_DEN]
    uint64_t *state_done = den_empty + TC_DEN;       // [1]
    uint64_t *s_ready = state_done + 1;              // [1]
    uint64_t *drain = s_ready + 1;                   // [1] abort path: MMA drain
    uint32_t *tmem_slot = (uint32_t *)(sm + Lay::OFF_MISC);
    volatile int *abort_flag = (volatile int *)(sm + Lay::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x / a.grid_seg, seg = blockIdx.x % a.grid_seg;
    const int tile0 = seg * a.seg_tiles;                 // first tile of this CTA
    const int nch = min(a.seg_tiles, a.nch - tile0);     // tiles of this CTA
    const bool totals = a.totals != 0;
    Ctl ctl{abort_flag, a.err, a.timeout_ns};
    const float gC = DK ? ex2(a.l2g * (float)C) : 1.f;  // gamma^C
    // decay: weight of earlier segment g's total at this segment's start
    auto seg_w = [&](int g) { return DK ? ex2(a.l2g * (float)((seg - 1 - g) * a.seg_tiles * C)) : 1.f; };

    auto stage_q = [&](int s) { return sm + Lay::OFF_STAGE + s * Lay::STAGE_BYTES; };
    auto stage_k = [&](int s) { return stage_q(s) + Lay::Q_BYTES; };
    auto stage_v = [&](int s) { return stage_k(s) + Lay::K_BYTES; };
    uint8_t *const p_tile = sm + Lay::OFF_P;  // P buffer b at p_tile + b * Lay::P_SET

    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&phi_ready[i], 1);
            mbar_init(&stage_free[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&scores_done[i], 1);
            mbar_init(&p_ready[i], 1);
            mbar_init(&o_done[i], 1);
            mbar_init(&o_free[i], 4);
        }
        for (int i = 0; i < TC_DEN; ++i) {
            mbar_init(&den_full[i], 1);
            mbar_init(&den_empty[i], 1);
        }
        mbar_init(state_done, 1);
        mbar_init(s_ready, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    // Segments after the first start from the (decay-weighted) sum of the earlier segments'
    // totals, plus a given initial state.  Every thread takes part: the sums go through an
    // fp32 scratch in the stage ring (unused until the producer starts), with independent,
    // coalesced loads, so the start-up does not wait on one serial chain of global loads.
    const int nprev = totals ? 0 : (NC ? a.nseg_all : seg);
    const bool has_prefix = !totals && (nprev > 0 || a.S0 != nullptr);
    if (totals) pdl_trigger();  // the main pass may be scheduled now
    else pdl_wait();            // the totals pass (if any) has completed
    constexpr int SCR_LD = D + 4;  // scratch row stride in floats (padding against bank conflicts)
    float *const scr = (float *)(sm + Lay::OFF_STAGE);
    static_assert(DV * (D + 4) * 4 <= ST * Lay::STAGE_BYTES, "prefix scratch fits the stage ring");
    if (has_prefix) {
        for (int e4 = tid; e4 < DV * D / 4; e4 += TC_THREADS) {
            const int j = e4 / (D / 4), i = 4 * (e4 % (D / 4));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int g = 0; g < nprev; ++g) {
                const float4 v4 = __ldcg((const float4 *)(a.ws_T + ((size_t)g * a.BH + head) * DV * D) + e4);
                const float w = seg_w(g);
                acc.x += w * v4.x; acc.y += w * v4.y; acc.z += w * v4.z; acc.w += w * v4.w;
            }
            if (a.S0) {
                // the given state before row 0 (S[i][j] at S0 + (head D + i) DV + j), decayed
                // over the rows of the earlier segments
                const float w = seg_w(-1);
                const float *s0 = a.S0 + ((size_t)head * D + i) * DV + j;
                acc.x += w * s0[0]; acc.y += w * s0[DV]; acc.z += w * s0[2 * DV]; acc.w += w * s0[3 * DV];
            }
            *(float4 *)(scr + j * SCR_LD + i) = acc;
        }
    }
    if (NORM)
        for (int i = tid; i < D; i += TC_THREADS) {
            float z0 = 0.f;
            if (!totals) {
#pragma unroll 4
                for (int g = 0; g < nprev; ++g) z0 += seg_w(g) * __ldcg(a.ws_z + ((size_t)g * a.BH + head) * D + i);
                if (a.z0) z0 += seg_w(-1) * a.z0[(size_t)head * D + i];  // the given state
            }
            zs[i] = z0;
        }
    if (DK && !NORM)
        for (int i = tid; i < C; i += TC_THREADS)  // gamma^(i'+1-C), i' the row's in-tile virtual index
            rden[i] = ex2(a.l2g * (float)(anti ? -i : i + 1 - C));
    if (CH == C)
        // P rows 0-31, columns 32-63: always zero (causal mask), written once in every P tile
        // (both buffers; hi and lo tiles in the fp32-output mode)
        for (int e = tid; e < 2 * (FO ? 2 : 1) * 32 * 4; e += TC_THREADS) {
            const int t = (e >> 2) & 31, chn = 4 + (e & 3);
            *(uint4 *)(p_tile + (e >> 7) * Lay::P_BYTES + t * 128 + ((chn ^ (t & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
        }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem + Lay::T_S, tSB = tmem + Lay::T_SB, tSL = tmem + Lay::T_SL;
    // fp32-output mode: bf16 hi / lo split of fp32 values (x = hi + lo to ~2^-16 relative)
    auto lo_of = [](float x) { return x - __bfloat162float(__float2bfloat16_rn(x)); };
    if (warp >= 4 + TC_FWARPS && warp < 8 + TC_FWARPS) {
        // the state and its bf16 copy start at the prefix in the scratch (zero for the first
        // segment and for the totals pass)
        const uint32_t lo = (uint32_t)(32 * (warp & 3)) << 16;
        const int jr = (DV == 128) ? 32 * (warp & 3) + lane : 16 * (warp & 3) + (lane & 15);
        const bool live = (DV == 128) || lane < 16;
#pragma unroll 1
        for (int col = 0; col < D; col += 16) {
            float acc[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = 0.f;
            if (live && has_prefix)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v4 = *(const float4 *)(scr + jr * SCR_LD + col + 4 * q);
                    acc[4 * q] = v4.x; acc[4 * q + 1] = v4.y; acc[4 * q + 2] = v4.z; acc[4 * q + 3] = v4.w;
                }
            if (DK)  // the first chunk reads gamma^C S and accumulates onto it
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] *= gC;
            uint32_t w32[16], w16[8];
#pragma unroll
            for (int e = 0; e < 16; ++e) w32[e] = __float_as_uint(acc[e]);
#pragma unroll
            for (int e = 0; e < 8; ++e) w16[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
            tmem_st16(tS + lo + col, w32);
            tmem_st8(tSB + lo + col / 2, w16);
            if (FO) {
#pragma unroll
                for (int e = 0; e < 8; ++e) w16[e] = pack_bf16x2(lo_of(acc[2 * e]), lo_of(acc[2 * e + 1]));
                tmem_st8(tSL + lo + col / 2, w16);
            }
        }
        tmem_wait_st();
    }
    // the scratch has been read: the stage ring's z rows can now be written
    __syncthreads();
    if (NORM) {
        // the z rows of every stage's K tile: rows C, C+1 rewritten per chunk, the rest zero
        for (int e = tid; e < ST * (D / 64) * 8 * 8; e += TC_THREADS) {
            const int st = e / ((D / 64) * 64), r = e % ((D / 64) * 64);
            const int kb = r / 64, row = C + (r % 64) / 8, chn = r % 8;
            *(uint4 *)(stage_k(st) + kb * Lay::K_BLK + row * 128 + chn * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    if (NC && NORM && !totals) {
        // non-causal main pass: z of the whole sequence as a bf16 hi / lo pair in key rows C and
        // C+1 of every stage (no keys are loaded in this pass, so they stay); written after the
        // zero rows above
        __syncthreads();
        for (int e = tid; e < ST * (D / 8) * 2; e += TC_THREADS) {
            const int st = e / ((D / 8) * 2), zr = e & 1, cg = (e >> 1) % (D / 8);
            const int zkb = cg >> 3, zch = cg & 7, row = C + zr;
            uint32_t pk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float z0 = zs[8 * cg + 2 * u], z1 = zs[8 * cg + 2 * u + 1];
                const float h0 = __bfloat162float(__float2bfloat16_rn(z0));
                const float h1 = __bfloat162float(__float2bfloat16_rn(z1));
                pk[u] = zr ? pack_bf16x2(z0 - h0, z1 - h1) : pack_bf16x2(h0, h1);
            }
            *(uint4 *)(stage_k(st) + zkb * Lay::K_BLK + row * 128 + ((zch ^ (row & 7)) << 4)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
    }
    if (esyn)
        // e in every row of every stage's Q and K tiles: element 0 lies in the row's first
        // 16-byte chunk, which the 128B swizzle puts at chunk position row % 8
        for (int e = tid; e < ST * 2 * (D / 64) * C * 8; e += TC_THREADS) {
            const int chn = e & 7, row = (e >> 3) % C, blk = (e >> 3) / C;
            const int kb = blk % (D / 64), isk = (blk / (D / 64)) & 1, st = blk / (2 * (D / 64));
            uint8_t *const t = isk ? stage_k(st) + kb * Lay::K_BLK : stage_q(st) + kb * C * 128;
            *(uint4 *)(t + row * 128 + ((chn ^ (row & 7)) << 4)) =
                make_uint4((kb == 0 && chn == 0) ? 0x3F80u : 0u, 0u, 0u, 0u);  // bf16 1.0
        }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            // the non-causal main pass reads the whole sequence's state: only Q is loaded
            const bool qonly = NC && !totals;
            for (int c = 0; c < nch; ++c) {
                const int s = c % ST;
                if (c >= ST && !wait_phase(&stage_free[s], ((c / ST) - 1) & 1, ctl))
                    break;
                const int row = anti ? a.L - (tile0 + c + 1) * C : (tile0 + c) * C;
                mbar_arrive_expect_tx(&full[s], esyn ? Lay::V_BYTES
                                                : totals ? Lay::STAGE_TX - Lay::Q_BYTES
                                                         : (qonly ? Lay::Q_BYTES : Lay::STAGE_TX));
                for (int kb = 0; kb < D / 64 && !esyn; ++kb) {
                    if (!totals)
                        tma_load_3d(stage_q(s) + kb * C * 128, &a.tm_q, kb * 64, row, head, &full[s]);
                    if (!qonly)
                        tma_load_3d(stage_k(s) + kb * Lay::K_BLK, &a.tm_k, kb * 64, row, head, &full[s]);
                }
                for (int jb = 0; jb < DV / 64 && !qonly; ++jb)
                    tma_load_3d(stage_v(s) + jb * C * 128, &a.tm_v, jb * 64, row, head, &full[s]);
                issued = c + 1;
            }
            // never leave the CTA with loads in flight: wait for every issued stage to land
            for (int c = (issued > ST ? issued - ST : 0); c < issued; ++c) {
                const int s = c % ST;
                const uint64_t t0 = globaltimer();
                while (!mbar_try_sleep(&full[s], (c / ST) & 1, 200000u))
                    if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_SC = idesc_bf16_f32(C, Lay::NSC, 0, 0);
            constexpr uint32_t ID_INTER = idesc_bf16_f32(DV, CH, 0, 0);
            constexpr uint32_t ID_STATE = idesc_bf16_f32(DV, D, 1, 1);
            constexpr uint32_t ID_INTRA = idesc_bf16_f32(DV, C, 1, 0);
            const int nsub = a.nsub;
            bool ok = true;
            if (totals) {
                // totals pass: only the state, over whole tiles
                for (int c = 0; c < nch; ++c) {
                    const int s = c % ST;
                    uint64_t *ph = (FM == LA_FM_IDENTITY && !NORM && !DK) ? &full[s] : &phi_ready[s];
                    if (!wait_phase(ph, (c / ST) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ka = smem_u32(stage_k(s)), va = smem_u32(stage_v(s));
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_ss(tS, smem_desc(va + ks * 2048, C * 128, 1024),
                               smem_desc(ka + ks * 2048, Lay::K_BLK, 1024), ID_STATE, 1);
                    mma_commit(&stage_free[s]);
                }
                if (ok) mma_commit(state_done);
                ok = false;  // skip the main loop
            }
            if constexpr (NC) {
                // non-causal main pass: every row reads the whole sequence's state, so a tile
                // needs only the inter product and (normaliser) phi(Q) z, from the z rows of
                // the K tile alone; no scores over keys, no intra product
                constexpr uint32_t ID_Z = idesc_bf16_f32(C, 8, 0, 0);  // rows C .. C+7 of a block
                auto dadd = [](uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); };
                for (int c = 0; ok && c < nch; ++c) {
                    const int s = c % ST, b = c & 1;
                    uint64_t *ph = (FM == LA_FM_IDENTITY) ? &full[s] : &phi_ready[s];
                    if (!wait_phase(ph, (c / ST) & 1, ctl)) break;
                    // scores buffer b: the P warps are done with tile c-2
                    if (NORM && c >= 2 && !wait_phase(&p_ready[b], ((c >> 1) - 1) & 1, ctl)) break;
                    if (c >= 2 && !wait_phase(&o_free[b], ((c >> 1) - 1) & 1, ctl)) break;
                    tc_fence_after();
                    const uint64_t dQ = smem_desc(smem_u32(stage_q(s)), 16, 1024);
                    const uint32_t tA = tmem + Lay::T_A + b * Lay::A_STRIDE, tO = tmem + Lay::T_O + b * C;
                    if (NORM) {
                        // z hi / lo in rows C, C+1 of each 64-feature block (then six zero
                        // rows): TMEM columns C, C+1
                        const uint64_t dZ = smem_desc(smem_u32(stage_k(s)) + C * 128, 16, 1024);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            mma_ss(tA + C, dadd(dQ, (ks >> 2) * C * 128 + (ks & 3) * 32),
                                   dadd(dZ, (ks >> 2) * Lay::K_BLK + (ks & 3) * 32), ID_Z, ks > 0);
                        mma_commit(&scores_done[b]);
                    }
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ts(tO, tSB + ks * 8, dadd(dQ, (ks >> 2) * C * 128 + (ks & 3) * 32), ID_INTER, ks > 0);
                    mma_commit(&o_done[b]);
                    mma_commit(&stage_free[s]);
                }
                ok = false;
            }
            // Software-pipelined order (one or two chunks per tile): inter and state of tile
            // c, then the scores of tile c+1, then the intra product of tile c.  The P warps
            // find the scores of tile c+1 complete when they finish tile c, so the loop-carried
            // chain scores -> P -> intra no longer waits for each intra product to be issued.
            // With four chunks per tile the chain of state updates and their bf16 copies binds
            // instead, and the scores of tile c go first in its own iteration.
            constexpr bool EARLY = NSUB <= 2;
            auto dadd = [](uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); };
            auto issue_scores = [&](int c) -> bool {
                const int s = c % ST, b = c & 1;
                uint64_t *ph = (FM == LA_FM_IDENTITY && !NORM && !DK) ? &full[s] : &phi_ready[s];
                if (!wait_phase(ph, (c / ST) & 1, ctl)) return false;
                // Scores buffer b was last read by the P warps for tile c-2.  No wait is
                // needed: this thread already waited for p_ready of tile c-2 (before its
                // intra product), which the P warps raise after fencing their TMEM loads
                // (fence::before_thread_sync before the barrier that precedes the arrive).
                tc_fence_after();
                // Descriptors: one per operand and tile; a constant byte offset goes into the
                // address field (addr >> 4), which never carries since shared addresses stay
                // below 256 KB.  This keeps the issuing thread's work per MMA to one add.
                const uint64_t dQ = smem_desc(smem_u32(stage_q(s)), 16, 1024);
                const uint64_t dK = smem_desc(smem_u32(stage_k(s)), 16, 1024);
                const uint32_t tA = tmem + Lay::T_A + b * Lay::A_STRIDE;
                // scores of the tile: phi(Q) [phi(K); z]^T, both K-major, K = D in steps of 16
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t qo = (ks >> 2) * C * 128 + (ks & 3) * 32;
                    const uint32_t ko = (ks >> 2) * Lay::K_BLK + (ks & 3) * 32;
                    mma_ss(tA, dadd(dQ, qo), dadd(dK, ko), ID_SC, ks > 0);
                }
                mma_commit(&scores_done[b]);
                return true;
            };
            if (EARLY && ok && nch > 0) ok = issue_scores(0);
            for (int c = 0; ok && c < nch; ++c) {
                const int s = c % ST, b = c & 1;
                if (!EARLY && !issue_scores(c)) break;
                const uint32_t qa = smem_u32(stage_q(s)), ka = smem_u32(stage_k(s)),
                               va = smem_u32(stage_v(s)), pa = smem_u32(p_tile + b * Lay::P_SET);
                const uint32_t tO = tmem + Lay::T_O + b * C;
                const uint64_t dQ = smem_desc(qa, 16, 1024);
                const uint64_t dVmn = smem_desc(va, C * 128, 1024), dKmn = smem_desc(ka, Lay::K_BLK, 1024);
                const uint64_t dP = smem_desc(pa, 16, 1024);
                if (c >= 2 && !wait_phase(&o_free[b], ((c >> 1) - 1) & 1, ctl)) break;
                for (int j = 0; j < NSUB; ++j) {
                    const int g = (tile0 + c) * NSUB + j;  // chunk index in the sequence
                    const int lg = c * NSUB + j;           // chunk index in this CTA
                    if (g >= nsub) break;
                    if (!NC && lg >= 1 && !wait_phase(s_ready, (lg - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // inter: bf16(S_g)^T (TMEM) x phi(Q_g)^T, the chunk's CH rows, K = D
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t qo = (ks >> 2) * C * 128 + (ks & 3) * 32 + j * CH * 128;
                        mma_ts(tO + j * CH, tSB + ks * 8, dadd(dQ, qo), ID_INTER, ks > 0);
                    }
                    if (FO)  // the state copy's lo part
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t qo = (ks >> 2) * C * 128 + (ks & 3) * 32 + j * CH * 128;
                            mma_ts(tO + j * CH, tSL + ks * 8, dadd(dQ, qo), ID_INTER, 1);
                        }
                    // state: S^T += V_g^T phi(K_g), both MN-major, K = CH in steps of 16 rows
                    if (g + 1 < nsub && !NC) {
#pragma unroll
                        for (int ks = 0; ks < CH / 16; ++ks) {
                            const uint32_t ro = (j * CH + 16 * ks) * 128;
                            mma_ss(tS, dadd(dVmn, ro), dadd(dKmn, ro), ID_STATE, 1);
                        }
                        mma_commit(state_done);
                    }
                }
                if (!ok) break;
                if (EARLY && c + 1 < nch && !issue_scores(c + 1)) break;
                if (!wait_phase(&p_ready[b], (c >> 1) & 1, ctl)) break;
                tc_fence_after();
                // intra: V^T (MN-major A) x P^T (K-major B) over the tile, K = 64
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tO, dadd(dVmn, ks * 2048), dadd(dP, ks * 32), ID_INTRA, 1);
                if (FO)  // P's lo tile
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_ss(tO, dadd(dVmn, ks * 2048), dadd(dP, Lay::P_BYTES + ks * 32), ID_INTRA, 1);
                mma_commit(&o_done[b]);
                mma_commit(&stage_free[s]);
            }
            // drain: every MMA issued above has completed before TMEM is released
            mma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_sleep(drain, 0, 200000u))
                if (globaltimer() - t0 > ctl.timeout_ns) break;
        }
    } else if (phi_rank(warp) >= 0) {
        // ------------------------------------------------------------ feature map / z
        // Thread (rg, g) owns 16-byte chunk g (8 features) of rows rg, rg + RG, ...: it
        // loads all its Q and K chunks at once, transforms them in registers and stores
        // them back in place (same swizzled slot).
        const int ft = 32 * phi_rank(warp) + lane;
        constexpr int NF = 32 * TC_FWARPS;  // threads in the group
        constexpr int G = D / 8;            // 16-byte chunks per row
        constexpr int RG = NF / G;          // row groups
        constexpr int NR = C / RG;          // rows per thread
        const int g = ft % G, rg = ft / G;
        const int kb = g >> 3, ch = g & 7;
        const int q_swz = kb * C * 128 + ((ch ^ (rg & 7)) << 4) + rg * 128;
        const int k_swz = kb * Lay::K_BLK + ((ch ^ (rg & 7)) << 4) + rg * 128;
        // non-causal main pass: no keys; the z rows were written once at the start, so only
        // phi(Q) is formed (nothing at all for identity features)
        const bool qonly = NC && !totals;
        if ((FM != LA_FM_IDENTITY || NORM || DK) && !(qonly && FM == LA_FM_IDENTITY)) {
            // decay: key row r of chunk c is weighted by gamma^(C-1-r) (rowf, fixed) times
            // gamma^(-C m) with m = c's place in the rescale period (main pass), or times
            // gamma^(C (nch-1-c)) (totals pass)
            float rowf[NR];
#pragma unroll
            for (int n = 0; n < NR; ++n)  // (the in-tile virtual index is C-1-r in the anti-causal pass)
                rowf[n] = DK ? ex2(a.l2g * (float)(anti ? rg + n * RG : C - 1 - rg - n * RG)) : 1.f;
            int pm = 0;  // c mod period
            for (int c = 0; c < nch; ++c, pm = (pm + 1 == a.period) ? 0 : pm + 1) {
                const int s = c % ST;
                const float chf = DK ? ex2(a.l2g * (float)(totals ? (nch - 1 - c) * C : -C * pm)) : 1.f;
                if (!group_wait(ft == 0, 1, &full[s], (c / ST) & 1, nullptr, 0, false, ctl,
                                NF))
                    break;
                uint4 *qp = (uint4 *)(stage_q(s) + q_swz);
                uint4 *kp = (uint4 *)(stage_k(s) + k_swz);
                uint4 wq[NR], wk[NR];
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    if (FM != LA_FM_IDENTITY && !totals) wq[n] = qp[n * RG * 8];
                    if (!qonly) wk[n] = kp[n * RG * 8];
                }
                if (NORM && !totals && !NC && ft < 8 * (D / 64) * 2) {
                    // z_c (before this chunk) as a bf16 hi/lo pair in key rows C and C+1
                    const int zkb = ft / 16, zr = (ft / 8) & 1, zch = ft & 7;
                    const float4 z0 = ((const float4 *)zs)[(64 * zkb + 8 * zch) / 4];
                    const float4 z1 = ((const float4 *)zs)[(64 * zkb + 8 * zch) / 4 + 1];
                    // decay: gamma^(C (1-m)) z, matching the state copy the inter product reads
                    const float zf = DK ? ex2(a.l2g * (float)(C * (1 - pm))) : 1.f;
                    const float zz[8] = {zf * z0.x, zf * z0.y, zf * z0.z, zf * z0.w,
                                         zf * z1.x, zf * z1.y, zf * z1.z, zf * z1.w};
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float h0 = __bfloat162float(__float2bfloat16_rn(zz[2 * e]));
                        float h1 = __bfloat162float(__float2bfloat16_rn(zz[2 * e + 1]));
                        pk[e] = zr ? pack_bf16x2(zz[2 * e] - h0, zz[2 * e + 1] - h1) : pack_bf16x2(h0, h1);
                    }
                    const int row = C + zr;
                    *(uint4 *)(stage_k(s) + zkb * Lay::K_BLK + row * 128 + ((zch ^ (row & 7)) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                if (FM != LA_FM_IDENTITY && !totals) {
#pragma unroll
                    for (int n = 0; n < NR; ++n) {
                        uint32_t *wv = (uint32_t *)&wq[n];
#pragma unroll
                        for (int e = 0; e < 4; ++e) wv[e] = elu1_bf16x2(wv[e]);
                    }
                }
                float colsum[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) colsum[e] = 0.f;
#pragma unroll
                for (int n = 0; n < NR && !qonly; ++n) {
                    uint32_t *wv = (uint32_t *)&wk[n];
                    // rows past L are TMA zero fill and phi(0) may be nonzero (elu+1): keep them out
                    // of z where z is used after the last tile (the non-causal totals)
                    const bool in_seq = !NC || (tile0 + c) * C + rg + n * RG < a.L;
                    // decay: key row r weighted by gamma^(C-1-r), or by gamma^(segment end - row)
                    // in the totals pass
                    const float rf = rowf[n] * chf;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // elu+1 in bf16x2; the decay scales the bf16 features in fp32
                        if (FM == LA_FM_ELU1) wv[e] = elu1_bf16x2(wv[e]);
                        if (DK) {
                            const float x0 = bf_lo(wv[e]) * rf, x1 = bf_hi(wv[e]) * rf;
                            if (NORM && in_seq) {
                                colsum[2 * e] += x0;
                                colsum[2 * e + 1] += x1;
                            }
                            wv[e] = pack_bf16x2(x0, x1);
                        } else if (NORM && in_seq) {
                            add_bf16x2_to_f32(colsum[2 * e], colsum[2 * e + 1], wv[e]);
                        }
                    }
                }
                if (FM != LA_FM_IDENTITY || DK) {
#pragma unroll
                    for (int n = 0; n < NR; ++n) {
                        if (FM != LA_FM_IDENTITY && !totals) qp[n * RG * 8] = wq[n];
                        if (!qonly) kp[n * RG * 8] = wk[n];
                    }
                }
                fence_async_smem();
                const bool zupd = NORM && (totals || (c + 1 < nch && !NC));
                if (zupd) {
                    // column sums over the row groups: lanes g, g+G, ... of a warp, then the
                    // group's warps through shared memory
#pragma unroll
                    for (int o = G; o < 32; o <<= 1)
#pragma unroll
                        for (int e = 0; e < 8; ++e) colsum[e] += __shfl_xor_sync(0xffffffffu, colsum[e], o);
                    if (lane < G) {
                        float4 *zp = (float4 *)(zpart + (ft >> 5) * D + 8 * g);
                        zp[0] = make_float4(colsum[0], colsum[1], colsum[2], colsum[3]);
                        zp[1] = make_float4(colsum[4], colsum[5], colsum[6], colsum[7]);
                    }
                }
                named_bar(1, NF);
                if (ft == 0 && !a.debug_stall) mbar_arrive(&phi_ready[s]);
                if (zupd) {
                    for (int i = ft; i < D; i += NF) {
                        float acc = 0.f;
#pragma unroll
                        for (int w = 0; w < TC_FWARPS; ++w) acc += zpart[w * D + i];
                        // decay: the keys carried gamma^(-C m) of the state's period
                        zs[i] = (DK && !totals) ? gC * zs[i] + ex2(a.l2g * (float)(C * pm)) * acc
                                                : zs[i] + acc;
                    }
                    // no barrier here: the next tile's group wait (a barrier of the whole
                    // group) orders these zs writes before its z rows are formed, and the
                    // zpart reads before zpart is written again
                }
            }
            if (totals && NORM)
                for (int i = ft; i < D; i += NF) a.ws_z[((size_t)seg * a.BH + head) * D + i] = zs[i];
        }
    } else if (warp >= 4 + TC_FWARPS && warp < 8 + TC_FWARPS) {
        // ------------------------------------------------------------ scores -> P, S readback
        const int q4 = warp & 3;
        const int pt = tid - 32 * (4 + TC_FWARPS);
        const int t = 16 * q4 + (lane & 15);  // M = 64 TMEM layout: row t at lane t%16 of quadrant t/16
        const bool row_lane = lane < 16;
        const int ta = 16 * q4 + (lane >> 2), tb = ta + 8, cpos = lane & 3;  // 16x256b loads
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        if (totals) {
            // this segment's total: S^T rows (fp32) to the workspace
            const int jr = (DV == 128) ? 32 * q4 + lane : 16 * q4 + (lane & 15);
            const bool live = (DV == 128) || lane < 16;
            if (group_wait(pt == 0, 2, state_done, 0, nullptr, 0, false, ctl)) {
                tc_fence_after();
                float *dst = a.ws_T + (((size_t)seg * a.BH + head) * DV + jr) * D;
#pragma unroll 1
                for (int cb = 0; cb < D / 32; ++cb) {
                    uint32_t sv[32];
                    tmem_ld32(tS + lane_off + cb * 32, sv);
                    tmem_wait_ld();
                    if (live) {
                        float4 *d4 = (float4 *)(dst + cb * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            d4[q] = make_float4(__uint_as_float(sv[4 * q]), __uint_as_float(sv[4 * q + 1]),
                                                __uint_as_float(sv[4 * q + 2]), __uint_as_float(sv[4 * q + 3]));
                    }
                }
            }
        }
        // non-causal main pass (normaliser): den = phi(q_t).z (hi + lo) of the whole sequence
        for (int c = 0; NC && NORM && c < nch && !totals; ++c) {
            const int b = c & 1, slot = c % TC_DEN;
            if (!group_wait(pt == 0, 2, &scores_done[b], (c >> 1) & 1, &den_empty[slot],
                            ((c / TC_DEN) - 1) & 1, c >= TC_DEN, ctl))
                break;
            tc_fence_after();
            uint32_t rz[8];
            tmem_ld8(tmem + Lay::T_A + b * Lay::A_STRIDE + lane_off + C, rz);
            tmem_wait_ld();
            tc_fence_before();  // scores buffer b read
            if (row_lane) rden[slot * C + t] = __fdividef(1.f, __uint_as_float(rz[0]) + __uint_as_float(rz[1]));
            named_bar(2, 128);
            if (pt == 0) {
                mbar_arrive(&p_ready[b]);
                mbar_arrive(&den_full[slot]);
            }
        }
        for (int c = 0; c < nch && !totals && !NC; ++c) {
            const int b = c & 1, slot = c % TC_DEN;
            if (!group_wait(pt == 0, 2, &scores_done[b], (c >> 1) & 1, &den_empty[slot],
                            ((c / TC_DEN) - 1) & 1, NORM && c >= TC_DEN, ctl))
                break;
            tc_fence_after();
            // Each thread owns half of two rows: ta = 16 q4 + lane/4 and tb = ta + 8, columns
            // 8k + 2 (lane % 4) and the next one, as a 16x256b TMEM load delivers them; the four
            // threads of a row pool their row sums with shuffles.  With one chunk per tile,
            // rows 0-31 (warps 0, 1 of the group) keep nothing from columns 32-63: their P there
            // is the zero block written at the start, and they load only the first half.
            const uint32_t tA = tmem + Lay::T_A + b * Lay::A_STRIDE + lane_off;
            const int nh = (CH == C && q4 < 2 && !anti) ? 1 : 2;  // 32-column halves to read
            float rsa[2] = {0.f, 0.f}, rsb[2] = {0.f, 0.f};  // this thread's part of the row sums
            uint32_t rz[4];
            uint8_t *pa = p_tile + b * Lay::P_SET + ta * 128 + 4 * cpos;
            uint8_t *pb = p_tile + b * Lay::P_SET + tb * 128 + 4 * cpos;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h >= nh) break;
                uint32_t r[32];  // r[0..15]: columns 32h .. 32h+31
                tmem_ld16x256_x4(tA + 32 * h, r);
                if (NORM && h == 0) tmem_ld16x256_x1(tA + C, rz);  // columns C, C+1: phi(q_t).z_c (hi, lo)
                tmem_wait_ld();
                if (h == nh - 1) tc_fence_before();  // scores buffer b read (see the MMA issuer)
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    // P keeps s in t's chunk with s <= t (block-diagonal causal mask at CH); the
                    // normaliser's row sum keeps every s <= t of the tile
                    const int k = 4 * h + k4, s0 = 8 * k + 2 * cpos, s1 = s0 + 1;
                    // (anti-causal: s >= t in smem order, which is s <= t in virtual rows)
                    const float a0 = (anti ? s0 >= ta : s0 <= ta) ? __uint_as_float(r[4 * k4]) : 0.f;
                    const float a1 = (anti ? s1 >= ta : s1 <= ta) ? __uint_as_float(r[4 * k4 + 1]) : 0.f;
                    const float b0 = (anti ? s0 >= tb : s0 <= tb) ? __uint_as_float(r[4 * k4 + 2]) : 0.f;
                    const float b1 = (anti ? s1 >= tb : s1 <= tb) ? __uint_as_float(r[4 * k4 + 3]) : 0.f;
                    rsa[k4 & 1] += a0 + a1;
                    rsb[k4 & 1] += b0 + b1;
                    uint32_t wa, wb;
                    if (CH == C) {
                        wa = pack_bf16x2(a0, a1);
                        wb = pack_bf16x2(b0, b1);
                    } else {
                        const int la = ta & ~(CH - 1), lb = tb & ~(CH - 1);
                        wa = pack_bf16x2(s0 >= la ? a0 : 0.f, s1 >= la ? a1 : 0.f);
                        wb = pack_bf16x2(s0 >= lb ? b0 : 0.f, s1 >= lb ? b1 : 0.f);
                    }
                    const int oa = (k ^ (ta & 7)) << 4, ob = (k ^ (tb & 7)) << 4;
                    *(uint32_t *)(pa + oa) = wa;
                    *(uint32_t *)(pb + ob) = wb;
                    if (FO) {
                        // P's lo tile: the rounding residue of each kept score (CH == C here)
                        *(uint32_t *)(pa + Lay::P_BYTES + oa) = pack_bf16x2(lo_of(a0), lo_of(a1));
                        *(uint32_t *)(pb + Lay::P_BYTES + ob) = pack_bf16x2(lo_of(b0), lo_of(b1));
                    }
                }
            }
            // den = phi(q_t).z_c + masked row sum
            // (fast division: 1/den only scales the fp32 row before its bf16 rounding)
            if (NORM) {
                float sa = rsa[0] + rsa[1], sb = rsb[0] + rsb[1];
                sa += __shfl_xor_sync(0xffffffffu, sa, 1);
                sb += __shfl_xor_sync(0xffffffffu, sb, 1);
                sa += __shfl_xor_sync(0xffffffffu, sa, 2);
                sb += __shfl_xor_sync(0xffffffffu, sb, 2);
                if (cpos == 0) {
                    rden[slot * C + ta] = __fdividef(1.f, __uint_as_float(rz[0]) + __uint_as_float(rz[1]) + sa);
                    rden[slot * C + tb] = __fdividef(1.f, __uint_as_float(rz[2]) + __uint_as_float(rz[3]) + sb);
                }
            }
            fence_async_smem();
            named_bar(2, 128);
            if (pt == 0) {
                mbar_arrive(&p_ready[b]);
                if (NORM) mbar_arrive(&den_full[slot]);
            }
            // bf16 copy of the state for each next chunk's inter product
            bool rb_ok = true;
            const int pm = DK ? c % a.period : 0;  // once per tile (NSUB = 1 under decay)
            for (int j = 0; j < NSUB; ++j) {
                const int g = (tile0 + c) * NSUB + j;  // chunk index in the sequence
                const int lg = c * NSUB + j;           // chunk index in this CTA
                if (NC || g + 1 >= a.nsub) break;  // no state update after the last chunk
                if (!group_wait(pt == 0, 2, state_done, lg & 1, nullptr, 0, false, ctl)) {
                    rb_ok = false;
                    break;
                }
                tc_fence_after();
                // decay: chunk m of the period leaves A = gamma^(-C m) S, the copy chunk m+1
                // reads; at the period's end A becomes gamma^(C P) A = gamma^C S
                const bool restore = DK && pm == a.period - 1;
                const float cf = restore ? ex2(a.l2g * (float)(C * a.period)) : 1.f;
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) {
                    uint32_t sv[32], pk[16];
                    tmem_ld32(tS + lane_off + cb * 32, sv);
                    tmem_wait_ld();
                    if (restore) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) sv[e] = __float_as_uint(cf * __uint_as_float(sv[e]));
                        tmem_st16(tS + lane_off + cb * 32, *reinterpret_cast<const uint32_t(*)[16]>(sv));
                        tmem_st16(tS + lane_off + cb * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(sv + 16));
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]));
                    tmem_st16(tSB + lane_off + cb * 16, pk);
                    if (FO) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16x2(lo_of(__uint_as_float(sv[2 * e])), lo_of(__uint_as_float(sv[2 * e + 1])));
                        tmem_st16(tSL + lane_off + cb * 16, pk);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_ready);
            }
            if (!rb_ok) break;
        }
    } else if (warp >= 8 + TC_FWARPS) {
        // ------------------------------------------------------------ output epilogue
        // Rows go from registers straight to global memory: for each token a warp writes 32
        // neighbouring output columns (64 contiguous bytes in bf16, 128 in fp32), so no
        // shared-memory staging tile is needed; rows past L are skipped.
        const int q4 = warp & 3;
        const int ot = tid - 32 * (8 + TC_FWARPS);
        // row j of O^T: lane j (dv = 128), or lane j%16 of quadrant j/16 (dv = 64)
        const int j = (DV == 128) ? 32 * q4 + lane : 16 * q4 + (lane & 15);
        const bool live = (DV == 128) || lane < 16;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const bool odd = lane & 1;
        for (int c = 0; c < nch && !totals; ++c) {
            const int b = c & 1, slot = c % TC_DEN;
            if (!group_wait(ot == 0, 3, &o_done[b], (c >> 1) & 1, &den_full[slot], (c / TC_DEN) & 1,
                            NORM, ctl))
                break;
            tc_fence_after();
            // rows of this tile inside the sequence: smem rows tlo .. thi-1 at rows row0 + tt
            const int row0 = anti ? a.L - (tile0 + c + 1) * C : (tile0 + c) * C;
            const int tlo = anti ? max(0, -row0) : 0, thi = anti ? C : min(C, a.L - row0);
            const long rbase = (long)head * a.L + row0;
            const uint32_t tO = tmem + Lay::T_O + b * C + lane_off;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
                tmem_ld32(tO + 32 * h, r);
                tmem_wait_ld();
                if (h == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&o_free[b]);
                }
                // 1 / den per row, or (decay, no normaliser) gamma^(i+1-C) gamma^(C m), read
                // per pair of rows from shared memory
                const float2 *rp = (const float2 *)(rden + (NORM ? slot * C : 0) + 32 * h);
                const float mf = (DK && !NORM) ? ex2(a.l2g * (float)(C * (c % a.period))) : 1.f;
                if constexpr (FO) {
                    // fp32 rows: column j of token tt (decay: times gamma^(i+1-C) gamma^(C m))
                    const float *rf = (const float *)rp;
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const int tt = 32 * h + u;
                        const float x = DK ? __uint_as_float(r[u]) * (mf * rf[u]) : __uint_as_float(r[u]);
                        if (live && tt >= tlo && tt < thi) ((float *)a.out)[(rbase + tt) * DV + j] = x;
                    }
                } else {
                    // Lanes j, j^1 swap one value per pair of rows so that each writes two
                    // neighbouring columns of one row as a single 32-bit word.
                    uint32_t *const o = (uint32_t *)a.out + (j >> 1);  // column pair j & ~1
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        float a0 = __uint_as_float(r[2 * u]), a1 = __uint_as_float(r[2 * u + 1]);
                        if (NORM || DK) {
                            const float2 f = rp[u];
                            a0 *= mf * f.x;
                            a1 *= mf * f.y;
                        }
                        const float recv = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
                        const int tt = 32 * h + 2 * u + (odd ? 1 : 0);
                        const uint32_t wv = odd ? pack_bf16x2(recv, a1) : pack_bf16x2(a0, recv);
                        if (live && tt >= tlo && tt < thi) o[(rbase + tt) * (DV / 2)] = wv;
                    }
                }
            }
            if (NORM) {
                // every thread has read this chunk's 1/den
                named_bar(3, 128);
                if (ot == 0) mbar_arrive(&den_empty[slot]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------- host side
// Segments per head: split the sequence when the heads alone leave most SMs idle, keeping
// at least 4 tiles (256 rows) per segment.
int tc_segments(const Problem &p, int num_sms, int *seg_tiles)
{
    return split_segments(p.B * p.H, (p.L + 63) / 64, num_sms, 4, seg_tiles);
}

size_t tc_workspace(const Problem &p, int nseg)
{
    if (nseg <= 1) return 0;
    return (size_t)(nseg - 1) * p.B * p.H * ((size_t)p.dv * p.D + p.D) * sizeof(float);
}

template <int D, int DV, int CH, int FM, bool NORM>
int launch_t(const Problem &p, int num_sms, int mode = TC_CAUSAL)
{
    const bool noncausal = mode == TC_NONCAUSAL;
    constexpr int C = 64;  // rows per tile
    using Lay = TcLayout<D, DV, C, NORM>;
    TcArgs a;
    memset(&a, 0, sizeof(a));
    const int BH = p.B * p.H;
    if (!make_map(&a.tm_q, p.q, BH, p.L, p.dk, C) || !make_map(&a.tm_k, p.k, BH, p.L, p.dk, C) ||
        !make_map(&a.tm_v, p.v, BH, p.L, p.dv, C))
        return LA_ERR_CUDA;
    a.out = p.out;
    a.L = p.L;
    a.nch = (p.L + C - 1) / C;
    a.nsub = (p.L + CH - 1) / CH;
    const int nseg = tc_segments(p, num_sms, &a.seg_tiles);
    a.BH = BH;
    // segments with a total: all but the last (causal); all of them (non-causal)
    const int ntot = noncausal ? nseg : nseg - 1;
    if (ntot > 0) {
        const size_t need = (size_t)ntot * BH * ((size_t)DV * D + D) * sizeof(float);
        if (!p.workspace || p.workspace_bytes < need) return LA_ERR_WORKSPACE;
        a.ws_T = (float *)p.workspace;
        a.ws_z = a.ws_T + (size_t)ntot * BH * DV * D;
    }
    a.noncausal = noncausal ? 1 : 0;
    a.nseg_all = nseg;
    a.l2g = (mode == TC_DECAY || mode == TC_DECAY_F32OUT) ? p.l2g : 0.f;
    a.anti = p.rev ? 1 : 0;
    a.esyn = p.esyn;
    a.S0 = p.S0;
    a.z0 = p.z0;
    // largest period P with C P |log2 gamma| <= 64 (gamma^(C P) >= 2^-64); tc_supported keeps
    // gamma^C >= 2^-64, so P >= 1
    a.period = 1 << 20;
    if (a.l2g < 0.f) a.period = (int)fmax(1.0, fmin((double)(1 << 20), floor(64.0 / (C * -(double)a.l2g))));
    a.err = p.err;
    a.timeout_ns = 2000000000ull;
    const char *e = getenv("LA_DEBUG_TIMEOUT_NS");
    if (e && *e) a.timeout_ns = strtoull(e, nullptr, 10);
    const char *st = getenv("LA_DEBUG_STALL");
    a.debug_stall = (st && *st && *st != '0') ? 1 : 0;
    auto kern = tc_chunked_kernel<D, DV, CH, FM, NORM, TC_CAUSAL>;
    int alloc = Lay::ALLOC;
    if constexpr (CH == C) {
        if (mode == TC_NONCAUSAL) kern = tc_chunked_kernel<D, DV, CH, FM, NORM, TC_NONCAUSAL>;
        if (mode == TC_DECAY) kern = tc_chunked_kernel<D, DV, CH, FM, NORM, TC_DECAY>;
        if (mode == TC_F32OUT || mode == TC_DECAY_F32OUT) {
            if constexpr (FM == LA_FM_IDENTITY && !NORM) {
                kern = mode == TC_F32OUT ? tc_chunked_kernel<D, DV, CH, FM, NORM, TC_F32OUT>
                                         : tc_chunked_kernel<D, DV, CH, FM, NORM, TC_DECAY_F32OUT>;
                alloc = TcLayout<D, DV, C, NORM, true>::ALLOC;
            } else {
                return LA_ERR_UNSUPPORTED;
            }
        }
    } else if (mode != TC_CAUSAL) {
        return LA_ERR_UNSUPPORTED;
    }
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, alloc) != cudaSuccess)
        return LA_ERR_CUDA;
    if (ntot > 0) {
        // totals of segments 0..ntot-1, then the main pass over all segments
        a.totals = 1;
        a.grid_seg = ntot;
        kern<<<BH * ntot, TC_THREADS, alloc, p.stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    a.totals = 0;
    a.grid_seg = nseg;
    if (ntot > 0) {
        // starts its set-up while the totals pass drains
        if (launch_dependent(kern, BH * nseg, TC_THREADS, alloc, p.stream, a) != cudaSuccess) return LA_ERR_CUDA;
        return LA_OK;
    }
    kern<<<BH * nseg, TC_THREADS, alloc, p.stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

template <int D, int DV, int CH>
int launch_dc(const Problem &p, int sms, int mode = TC_CAUSAL)
{
    const bool n = p.normalize != 0;
    if (p.fm == LA_FM_IDENTITY)
        return n ? launch_t<D, DV, CH, LA_FM_IDENTITY, true>(p, sms, mode)
                 : launch_t<D, DV, CH, LA_FM_IDENTITY, false>(p, sms, mode);
    return n ? launch_t<D, DV, CH, LA_FM_ELU1, true>(p, sms, mode)
             : launch_t<D, DV, CH, LA_FM_ELU1, false>(p, sms, mode);
}

template <int D, int DV>
int launch_d(const Problem &p, int sms)
{
    if (p.decay) return launch_dc<D, DV, 64>(p, sms, p.out_f32 ? TC_DECAY_F32OUT : TC_DECAY);
    if (p.out_f32) return launch_dc<D, DV, 64>(p, sms, TC_F32OUT);
    if (p.C == 16) return launch_dc<D, DV, 16>(p, sms);
    if (p.C == 32) return launch_dc<D, DV, 32>(p, sms);
    return launch_dc<D, DV, 64>(p, sms);
}

}  // namespace

bool tcf_supported(const Problem &p);
int tcf_plan(const Problem &p, int num_sms, la_plan_info *info);
int tcf_launch(const Problem &p, int num_sms);
bool tcl_supported(const Problem &p);
int tcl_plan(const Problem &p, int num_sms, la_plan_info *info);
int tcl_launch(const Problem &p, int num_sms);
bool tcw_supported(const Problem &p);
bool tcf_nc_supported(const Problem &p);
size_t tcf_nc_workspace(const Problem &p, int num_sms);
int tcf_nc_launch(const Problem &p, int num_sms);
int tcw_plan(const Problem &p, int num_sms, la_plan_info *info);
int tcw_launch(const Problem &p, int num_sms);

bool tc_supported(const Problem &p, int num_sms)
{
    (void)num_sms;
    // the anti-causal pass: identity features, no normaliser, one 64-row chunk per tile
    if (p.rev && (p.fm != LA_FM_IDENTITY || p.normalize || p.lam || p.C != 64 || p.S0 || p.z0)) return false;
    // constant e rows: dk = 64, identity, no normaliser, no decay
    if (p.esyn && (p.dk != 64 || p.fm != LA_FM_IDENTITY || p.normalize || p.lam || p.decay || p.C != 64))
        return false;
    if (p.decay) {
        // one 64-row chunk per tile; gamma^64 >= 2^-64 keeps the scaled keys and the
        // output factor gamma^(i+1-64) well inside the fp32 / bf16 range
        if (p.lam || p.C != 64 || p.l2g < -1.f) return false;
        if (p.fm != LA_FM_IDENTITY && p.fm != LA_FM_ELU1) return false;
    }
    if (p.out_f32 && (p.lam || p.C != 64 || p.fm != LA_FM_IDENTITY || p.normalize))
        return false;
    // a given initial state: the identity / elu+1 kernel with C <= 64 (or the decay mode)
    if ((p.S0 || p.z0) && (p.lam || p.fm == LA_FM_FAVOR || p.C > 64)) return false;
    if (p.lam) return tcl_supported(p);
    if (p.fm == LA_FM_FAVOR) return tcf_supported(p);
    if (p.C == 128 || p.C == 256) return tcw_supported(p);
    if (p.dtype != LA_BF16) return false;
    if (p.fm != LA_FM_IDENTITY && p.fm != LA_FM_ELU1) return false;
    if (p.dk != p.D) return false;
    // (D, dv) in {(64, 64), (64, 128), (128, 128)}; (128, 64) for the fp32-output mode
    // without the decay (the backward pass's FAVOR+ route)
    const bool d128v64 = p.D == 128 && p.dv == 64 && p.out_f32 && !p.decay;
    if (!((p.D == 64 && (p.dv == 64 || p.dv == 128)) || (p.D == 128 && p.dv == 128) || d128v64)) return false;
    if (p.C != 16 && p.C != 32 && p.C != 64) return false;
    if (p.L < 2 * 64) return false;  // short sequences: the generic path is as fast
    return true;
}

int tc_plan(const Problem &p, int num_sms, la_plan_info *info)
{
    if (p.lam) return tcl_plan(p, num_sms, info);
    if (p.fm == LA_FM_FAVOR) return tcf_plan(p, num_sms, info);
    if (p.C == 128 || p.C == 256) return tcw_plan(p, num_sms, info);
    int seg_tiles = 0;
    const int nseg = tc_segments(p, num_sms, &seg_tiles);
    info->grid_x = p.B * p.H * nseg;
    info->grid_y = 1;
    info->block = TC_THREADS;
    auto alloc = [&](auto d, auto dv) {
        constexpr int D = decltype(d)::value, DV = decltype(dv)::value;
        return p.normalize ? TcLayout<D, DV, 64, true>::ALLOC : TcLayout<D, DV, 64, false>::ALLOC;
    };
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    info->smem_bytes = p.D == 128 ? (p.dv == 128 ? alloc(I128{}, I128{}) : TcLayout<128, 64, 64, false, true>::ALLOC)
                                  : (p.dv == 128 ? alloc(I64{}, I128{}) : alloc(I64{}, I64{}));
    info->n_launches = nseg > 1 ? 2 : 1;
    info->workspace_bytes = tc_workspace(p, nseg);
    return LA_OK;
}

int tc_launch(const Problem &p, int num_sms)
{
    if (!tc_supported(p, num_sms)) return LA_ERR_UNSUPPORTED;
    if (p.lam) return tcl_launch(p, num_sms);
    if (p.fm == LA_FM_FAVOR) return tcf_launch(p, num_sms);
    if (p.C == 128 || p.C == 256) return tcw_launch(p, num_sms);
    if (p.D == 128 && p.dv == 64)  // the fp32-output mode only (tc_supported)
        return launch_t<128, 64, 64, LA_FM_IDENTITY, false>(p, num_sms, TC_F32OUT);
    if (p.D == 128) return launch_d<128, 128>(p, num_sms);
    return p.dv == 128 ? launch_d<64, 128>(p, num_sms) : launch_d<64, 64>(p, num_sms);
}

// ---- non-causal (bidirectional) on the tensor cores: totals of every segment, then a main
// pass that only reads the summed state (64-row tiles; C plays no part)
bool tc_nc_supported(const Problem &p)
{
    if (p.fm == LA_FM_FAVOR) return tcf_nc_supported(p);
    if (p.dtype != LA_BF16 || p.lam) return false;
    if (p.fm != LA_FM_IDENTITY && p.fm != LA_FM_ELU1) return false;
    if (p.dk != p.D) return false;
    if (!((p.D == 64 && (p.dv == 64 || p.dv == 128)) || (p.D == 128 && p.dv == 128))) return false;
    return p.L >= 2 * 64;
}

size_t tc_nc_workspace(const Problem &p, int num_sms)
{
    if (p.fm == LA_FM_FAVOR) return tcf_nc_workspace(p, num_sms);
    const int nseg = tc_segments(p, num_sms, nullptr);
    return (size_t)nseg * p.B * p.H * ((size_t)p.dv * p.D + p.D) * sizeof(float);
}

int tc_nc_launch(const Problem &p, int num_sms)
{
    if (!tc_nc_supported(p)) return LA_ERR_UNSUPPORTED;
    if (p.fm == LA_FM_FAVOR) return tcf_nc_launch(p, num_sms);
    auto go = [&](auto d, auto dv) -> int {
        constexpr int D = decltype(d)::value, DV = decltype(dv)::value;
        const bool n = p.normalize != 0;
        if (p.fm == LA_FM_IDENTITY)
            return n ? launch_t<D, DV, 64, LA_FM_IDENTITY, true>(p, num_sms, TC_NONCAUSAL)
                     : launch_t<D, DV, 64, LA_FM_IDENTITY, false>(p, num_sms, TC_NONCAUSAL);
        return n ? launch_t<D, DV, 64, LA_FM_ELU1, true>(p, num_sms, TC_NONCAUSAL)
                 : launch_t<D, DV, 64, LA_FM_ELU1, false>(p, num_sms, TC_NONCAUSAL);
    };
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    if (p.D == 128) return go(I128{}, I128{});
    return p.dv == 128 ? go(I64{}, I128{}) : go(I64{}, I64{});
}

}  // namespace la
