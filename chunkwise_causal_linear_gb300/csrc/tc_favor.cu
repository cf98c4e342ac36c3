// tc_favor.cu -- tensor-core path for FAVOR+ positive random features (sm_103a).
//
// The chunked order of "attention と線形の間" section 2, with the FAVOR+ feature map of
// "Linear Attention / Performerの理論と実装" (positive random features, with the Performer
// implementation's input scaling):
//     x^ = x dk^{-1/4},   phi(x)_l = exp(omega_l . x^ - |x^|^2 / 2) / sqrt(m),
// and its normalised output y_t = phi(q_t)^T S_t / phi(q_t)^T z_t.  Shapes: dk = 64 inputs,
// m = 256 features, dv = 64, chunks of 64 rows.
//
// Layout (TMEM 512 columns, ~222 KB shared memory, 640 threads):
//   * projection, transposed: P^T = omega' [Q; K]^T (M = 128 features per half, N = 128: the
//     chunk's 64 query rows and 64 key rows, contiguous in the stage, in one product; K = dk),
//     omega' = omega dk^{-1/4} held as bf16 hi + lo (two accumulated MMAs: a single bf16 copy
//     of omega' misses the tolerance).  TMEM lanes are features, so each of the 256
//     feature-map threads owns one feature l: it exponentiates its 64 query and 64 key
//     tokens, writes row l of phi(Q)^T and phi(K)^T ([l][t], t contiguous: one 128-byte row)
//     and keeps z_l as a private fp32 sum.
//   * the phi^T tiles are MN-major A (scores, inter: M = t, K = l), MN-major B (scores: N = s)
//     and K-major A (state: M = l, K = s) -- the same bytes serve all three.
//   * state S (256 x 64) not transposed: two M = 128 halves in TMEM, 128 columns, all lanes.
//     Its bf16 copy S~ is a K-major B operand [j][l] in shared memory with two extra rows
//     j = 64, 65 holding z_hi, z_lo, so the inter MMA (N = 72) also returns phi(q_t).z.
//   * output O (M = 64 tokens, N = 72) in TMEM; each output thread owns one row and stores it
//     straight to global memory (128 contiguous bytes).  The scores share the projection's
//     columns: the projection is read before the scores are written, and the next chunk's
//     projection waits for the scores to be read.
//
// MMAs per chunk (bf16 in, fp32 accumulate):
//   proj    P^T  = omega'(hi+lo) [Q;K]^T  M=128 x2  N=128 K=64  (x2 for hi, lo)
//   scores  A    = phi(Q) phi(K)^T      M=64      N=64  K=256
//   inter   O'   = phi(Q) [S~ | z]      M=64      N=72  K=256
//   state   S   += phi(K)^T V           M=128 x2  N=64  K=64
//   intra   O   += P V                  M=64      N=64  K=64
//
// Long sequences with few heads are split into segments (one CTA each): a totals pass
// (projK, phi(K), state only) writes each segment's S and z; the main pass starts segment g
// from the sum of the earlier totals.  Every wait is bounded as in the other tensor-core
// kernel.
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace la {

using namespace ptx;
using namespace tcc;

namespace {

constexpr int FV_THREADS = 640;
constexpr int FV_STAGES = 2;      // main pass: Q, K, V per stage
constexpr int FV_STAGES_TOT = 3;  // totals pass: K, V per stage, in the same bytes
constexpr int FV_DK = 64, FV_M = 256, FV_DV = 64, FV_C = 64;
constexpr int FV_DEN = 4;

// shared memory (bytes, 1024-aligned tiles)
constexpr int FV_OMEGA = 0;                          // [2 (hi, lo)][256 l][64 dk] bf16 K-major
constexpr int FV_OMEGA_BYTES = 2 * FV_M * 128;       // 64 KB
constexpr int FV_STAGE = FV_OMEGA + FV_OMEGA_BYTES;  // stages: Q, K, V raw tiles [64][64]
constexpr int FV_TILE = FV_C * 128;                  // 8 KB
constexpr int FV_STAGE_BYTES = 3 * FV_TILE;
constexpr int FV_PHIQ = FV_STAGE + FV_STAGES * FV_STAGE_BYTES;  // phi(Q)^T [256 l][64 t]
constexpr int FV_PHIK = FV_PHIQ + FV_M * 128;                   // phi(K)^T [256 l][64 s]
constexpr int FV_SROWS = FV_DV + 8;                             // S~ rows: 64 j + z hi, lo, 6 zero
constexpr int FV_SBLK = FV_SROWS * 128;                         // one 64-feature block
constexpr int FV_SBAR = FV_PHIK + FV_M * 128;                   // S~ [72 j][256 l] K-major
constexpr int FV_P = FV_SBAR + (FV_M / 64) * FV_SBLK;           // P [64 t][64 s]
constexpr int FV_F32 = FV_P + FV_TILE;
constexpr int FV_N_F32 = 2 * FV_C /*nrm q,k*/ + FV_DEN * FV_C /*den_intra*/;
constexpr int FV_BAR = FV_F32 + FV_N_F32 * 4;
constexpr int FV_N_BAR = 2 * FV_STAGES_TOT + 17 + 2 * FV_DEN;
static_assert(FV_STAGES_TOT * 2 * FV_C * 128 <= FV_STAGES * 3 * FV_C * 128, "totals stages fit the stage area");
constexpr int FV_MISC = FV_BAR + FV_N_BAR * 8;
constexpr int FV_BYTES = FV_MISC + 16;
constexpr int FV_ALLOC = FV_BYTES + 1024;
static_assert(FV_ALLOC <= 232448, "shared memory budget");
static_assert(FV_SBLK % 1024 == 0, "swizzle atoms stay aligned");

// TMEM columns
constexpr uint32_t FT_S = 0;      // S: half h at columns 64h (lanes = features 128h..)
constexpr uint32_t FT_P = 128;    // projection: half h at 128 + 128h, Q tokens then K tokens
constexpr uint32_t FT_A = 128;    // scores (M = 64 layout, 64 columns), inside the projection's
constexpr uint32_t FT_O = 384;    // O' (M = 64 layout, 72 columns)

struct FvArgs {
    CUtensorMap tm_q, tm_k, tm_v;
    const float *omega;      // [256][64] fp32
    __nv_bfloat16 *out;      // [BH][L][64]
    int L, nch;              // tiles (= chunks) of a head
    int seg_tiles, grid_seg, totals, BH;
    float *ws_S;             // [segments-1][BH][256][64]  (S rows l)
    float *ws_z;             // [segments-1][BH][256]
    int *err;
    unsigned long long timeout_ns;
    int nseg_all;            // non-causal: segments whose totals make the state
};

// NC: the bidirectional (non-causal) form.  The totals pass then covers every segment; the
// main pass starts from the sum of all of them, never updates the state, and zeroes P, so
// each row gets phi(q) S_total (/ phi(q) z_total).
template <bool NORM, bool NC>
__global__ void __launch_bounds__(FV_THREADS, 1) tc_favor_kernel(const __grid_constant__ FvArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *nrm = (float *)(sm + FV_F32);           // [2][64]: |x^|^2 of the Q rows, K rows
    float *den_intra = nrm + 2 * FV_C;             // [FV_DEN][64]
    uint64_t *bars = (uint64_t *)(sm + FV_BAR);
    uint64_t *full = bars;                         // [S]
    uint64_t *stage_free = full + FV_STAGES_TOT;   // [S]
    uint64_t *p_done = stage_free + FV_STAGES_TOT; // projection of the chunk in TMEM (totals
                                                   // pass: [2] by chunk parity)
    uint64_t *phi_ready = p_done + 3;              // phi(Q), phi(K), z rows written (and the
                                                   // projection read); totals pass: [2]
    uint64_t *scores_done = phi_ready + 2;
    uint64_t *a_free = scores_done + 1;            // scores read (their columns reusable)
    uint64_t *p_ready = a_free + 1;
    uint64_t *state_done = p_ready + 1;
    uint64_t *sbar_ready = state_done + 1;         // S~ rows for the next chunk written
    uint64_t *o_done = sbar_ready + 1;             // [1] (slot 2 spare)
    uint64_t *o_free = o_done + 2;                 // [1] (slot 2 spare)
    uint64_t *drain = o_free + 2;
    uint64_t *totals_done = drain + 1;
    uint64_t *den_full = totals_done + 2;          // [FV_DEN]
    uint64_t *den_empty = den_full + FV_DEN;       // [FV_DEN]
    uint32_t *tmem_slot = (uint32_t *)(sm + FV_MISC);
    volatile int *abort_flag = (volatile int *)(sm + FV_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x / a.grid_seg, seg = blockIdx.x % a.grid_seg;
    const int tile0 = seg * a.seg_tiles;
    const int nch = min(a.seg_tiles, a.nch - tile0);
    const bool totals = a.totals != 0;
    Ctl ctl{abort_flag, a.err, a.timeout_ns};
    if (totals) pdl_trigger();  // the main pass may be scheduled now
    else pdl_wait();            // the totals pass (if any) has completed
    // stages: main pass [Q | K | V] x 2, totals pass [K | V] x 3 (no Q), in the same bytes
    const int NST = totals ? FV_STAGES_TOT : FV_STAGES;
    auto stage_q = [&](int s) { return sm + FV_STAGE + s * FV_STAGE_BYTES; };
    auto stage_k = [&](int s) { return totals ? sm + FV_STAGE + s * 2 * FV_TILE : stage_q(s) + FV_TILE; };
    auto stage_v = [&](int s) { return stage_k(s) + FV_TILE; };

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&stage_free[i], 1);
        }
        mbar_init(&p_done[0], 1);
        mbar_init(&p_done[1], 1);
        mbar_init(&phi_ready[0], 1);
        mbar_init(&phi_ready[1], 1);
        mbar_init(scores_done, 1);
        mbar_init(a_free, 4);
        mbar_init(p_ready, 1);
        mbar_init(state_done, 1);
        mbar_init(sbar_ready, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&o_done[i], 1);
            mbar_init(&o_free[i], 4);
        }
        mbar_init(drain, 1);
        mbar_init(totals_done, 1);
        for (int i = 0; i < FV_DEN; ++i) {
            mbar_init(&den_full[i], 1);
            mbar_init(&den_empty[i], 1);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    // omega' = omega dk^{-1/4} as bf16 hi and lo parts, K-major 128B-swizzled [l][dk]
    const float sc = 0.35355339059327373f;  // 64^{-1/4}
    for (int e = tid; e < FV_M * FV_DK; e += FV_THREADS) {
        const int l = e / FV_DK, d = e % FV_DK;
        const float w = __ldg(a.omega + e) * sc;
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
        const int off = l * 128 + (((d >> 3) ^ (l & 7)) << 4) + (d & 7) * 2;
        *(__nv_bfloat16 *)(sm + FV_OMEGA + off) = hi;
        *(__nv_bfloat16 *)(sm + FV_OMEGA + FV_M * 128 + off) = lo;
    }
    // S~ starts at zero (rows 66..71 stay zero for good)
    for (int e = tid; e < (FV_M / 64) * FV_SBLK / 16; e += FV_THREADS)
        ((uint4 *)(sm + FV_SBAR))[e] = make_uint4(0, 0, 0, 0);
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- initial state of this CTA: zero, or the sum of the earlier segments' totals ----
    float zreg = 0.f;  // feature-map threads: z_l (fp32) of their feature
    if (warp >= 4 && warp < 12) {
        const int l = tid - 128;                       // feature of this thread
        const uint32_t lo = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tS = tmem + FT_S + 64 * (l >> 7) + lo;
        const int nprev = totals ? 0 : (NC ? a.nseg_all : seg);
        for (int g = 0; g < nprev; ++g) zreg += a.ws_z[((size_t)g * a.BH + head) * FV_M + l];
#pragma unroll 1
        for (int col = 0; col < FV_DV; col += 16) {
            float acc[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = 0.f;
            for (int g = 0; g < nprev; ++g) {
                const float4 *src = (const float4 *)(a.ws_S + (((size_t)g * a.BH + head) * FV_M + l) * FV_DV + col);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v4 = src[q];
                    acc[4 * q] += v4.x; acc[4 * q + 1] += v4.y; acc[4 * q + 2] += v4.z; acc[4 * q + 3] += v4.w;
                }
            }
            uint32_t w32[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w32[e] = __float_as_uint(acc[e]);
            tmem_st16(tS + col, w32);
            // S~ rows j = col..col+15 at column l (K-major [j][l] B operand)
            uint8_t *blk = sm + FV_SBAR + (l >> 6) * FV_SBLK + ((l & 7) << 1);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = col + e;
                *(__nv_bfloat16 *)(blk + j * 128 + ((((l & 63) >> 3) ^ (j & 7)) << 4)) = __float2bfloat16_rn(acc[e]);
            }
        }
        tmem_wait_st();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c % NST;
                if (c >= NST && !wait_phase(&stage_free[s], ((c / NST) - 1) & 1, ctl)) break;
                const int row = (tile0 + c) * FV_C;
                mbar_arrive_expect_tx(&full[s], totals ? 2 * FV_TILE : 3 * FV_TILE);
                if (!totals) tma_load_3d(stage_q(s), &a.tm_q, 0, row, head, &full[s]);
                tma_load_3d(stage_k(s), &a.tm_k, 0, row, head, &full[s]);
                tma_load_3d(stage_v(s), &a.tm_v, 0, row, head, &full[s]);
                issued = c + 1;
            }
            for (int c = (issued > NST ? issued - NST : 0); c < issued; ++c) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_sleep(&full[c % NST], (c / NST) & 1, 200000u))
                    if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_PROJ = idesc_bf16_f32(128, 64, 0, 0);    // K rows only
            constexpr uint32_t ID_PROJ2 = idesc_bf16_f32(128, 128, 0, 0);  // Q and K rows
            constexpr uint32_t ID_SC = idesc_bf16_f32(64, 64, 1, 1);
            constexpr uint32_t ID_INTER = idesc_bf16_f32(64, FV_SROWS, 1, 0);
            constexpr uint32_t ID_STATE = idesc_bf16_f32(128, 64, 0, 1);
            constexpr uint32_t ID_INTRA = idesc_bf16_f32(64, 64, 0, 1);
            const uint32_t om = smem_u32(sm + FV_OMEGA), phq = smem_u32(sm + FV_PHIQ),
                           phk = smem_u32(sm + FV_PHIK), sb = smem_u32(sm + FV_SBAR),
                           pa = smem_u32(sm + FV_P);
            // one descriptor per operand, constant offsets added (desc_add)
            const uint64_t dOm = smem_desc(om, 16, 1024), dPhqMN = smem_desc(phq, FV_M * 128, 1024),
                           dPhkMN = smem_desc(phk, FV_M * 128, 1024), dPhk = smem_desc(phk, 16, 1024),
                           dSb = smem_desc(sb, 16, 1024), dPa = smem_desc(pa, 16, 1024);
            // projection of raw rows into TMEM (features on lanes), omega hi + lo: the 128 rows
            // Q, K of the stage (main pass) or the 64 K rows (totals pass)
            auto project = [&](uint32_t xa, uint32_t idesc, uint32_t col) {
                const uint64_t dX = smem_desc(xa, 16, 1024);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ss(tmem + FT_P + 128 * h + col,
                                   desc_add(dOm, part * FV_M * 128 + h * 128 * 128 + ks * 32),
                                   desc_add(dX, ks * 32), idesc, (part | ks) != 0);
            };
            if (totals) {
                // Totals pass, pipelined over two buffers (chunk parity b): the projection of K
                // into TMEM columns FT_P + 128 h + 64 b, phi(K)^T into the phi(K) tile (b = 0) or
                // the otherwise idle phi(Q) tile (b = 1).  The projection of chunk c is issued
                // before the state update of chunk c-1 waits for its phi, so the feature-map
                // warps exponentiate one chunk while the next one is projected.
                bool tok = true;
                auto state_of = [&](int c) -> bool {
                    const int b = c & 1, s = c % NST;
                    if (!wait_phase(&phi_ready[b], (c >> 1) & 1, ctl)) return false;
                    tc_fence_after();
                    const uint64_t dPh = smem_desc(b ? phq : phk, 16, 1024);
                    const uint64_t dV = smem_desc(smem_u32(stage_v(s)), FV_C * 128, 1024);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ss(tmem + FT_S + 64 * h, desc_add(dPh, h * 128 * 128 + ks * 32),
                                   desc_add(dV, ks * 2048), ID_STATE, (c > 0) || (ks > 0));
                    mma_commit(&stage_free[s]);
                    return true;
                };
                for (int c = 0; tok && c < nch; ++c) {
                    const int s = c % NST, b = c & 1;
                    if (!wait_phase(&full[s], (c / NST) & 1, ctl)) {
                        tok = false;
                        break;
                    }
                    // TMEM buffer b was read for chunk c-2: its phi_ready was waited on below
                    tc_fence_after();
                    project(smem_u32(stage_k(s)), ID_PROJ, 64u * b);
                    mma_commit(&p_done[b]);
                    if (c >= 1) tok = state_of(c - 1);
                }
                if (tok && nch > 0 && state_of(nch - 1)) mma_commit(totals_done);
            }
            for (int c = 0; c < nch && !totals; ++c) {
                const int s = c % FV_STAGES;
                const int g = tile0 + c;  // chunk index in the sequence
                if (!wait_phase(&full[s], (c / FV_STAGES) & 1, ctl)) break;
                // the projection's columns hold the previous chunk's scores until the P warps
                // have read them; the previous projection itself was read before phi_ready
                if (!totals && c >= 1 && !wait_phase(a_free, (c - 1) & 1, ctl)) break;
                const uint32_t qa = smem_u32(stage_q(s)), va = smem_u32(stage_v(s));
                const uint64_t dVmn = smem_desc(va, FV_C * 128, 1024);
                tc_fence_after();
                project(qa, ID_PROJ2, 0);  // K follows Q in the stage: rows 0-63 Q, 64-127 K
                mma_commit(&p_done[0]);
                if (!wait_phase(&phi_ready[0], c & 1, ctl)) break;
                tc_fence_after();
                // scores: phi(Q) (MN-major A) x phi(K)^T (MN-major B), K = 256 features, into
                // the projection's columns (read by now: phi_ready)
#pragma unroll
                for (int ks = 0; ks < FV_M / 16; ++ks)
                    mma_ss(tmem + FT_A, desc_add(dPhqMN, ks * 2048), desc_add(dPhkMN, ks * 2048), ID_SC, ks > 0);
                mma_commit(scores_done);
                if (!NC && c >= 1 && !wait_phase(sbar_ready, (c - 1) & 1, ctl)) break;
                if (c >= 1 && !wait_phase(o_free, (c - 1) & 1, ctl)) break;
                tc_fence_after();
                const uint32_t tO = tmem + FT_O;
                // inter: phi(Q) (MN-major A) x [S~ | z] (K-major B, 72 rows), K = 256
#pragma unroll
                for (int ks = 0; ks < FV_M / 16; ++ks)
                    mma_ss(tO, desc_add(dPhqMN, ks * 2048), desc_add(dSb, (ks >> 2) * FV_SBLK + (ks & 3) * 32),
                           ID_INTER, ks > 0);
                // state: S += phi(K)^T (K-major A, features on M) x V (MN-major B), K = 64
                if (g + 1 < a.nch && !NC) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ss(tmem + FT_S + 64 * h, desc_add(dPhk, h * 128 * 128 + ks * 32),
                                   desc_add(dVmn, ks * 2048), ID_STATE, 1);
                    mma_commit(state_done);
                }
                if (!wait_phase(p_ready, c & 1, ctl)) break;
                tc_fence_after();
                // intra: P (K-major A) x V (MN-major B), K = 64
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tO, desc_add(dPa, ks * 32), desc_add(dVmn, ks * 2048), ID_INTRA, 1);
                mma_commit(o_done);
                mma_commit(&stage_free[s]);
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_sleep(drain, 0, 200000u))
                if (globaltimer() - t0 > ctl.timeout_ns) break;
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ feature map (one feature per thread)
        const int l = tid - 128;
        const int half = l >> 7;
        const uint32_t lo = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tP = tmem + FT_P + 128 * half + lo;  // Q tokens at +0, K tokens at +64
        const float inv_sqrt_m = 0.0625f;      // 1 / sqrt(256)
        const float log2e = 1.4426950408889634f;
        uint8_t *rowq = sm + FV_PHIQ + l * 128;
        uint8_t *rowk = sm + FV_PHIK + l * 128;
        // S~ column l: K-major [j][l], block l/64
        uint8_t *sblk = sm + FV_SBAR + (l >> 6) * FV_SBLK + ((l & 7) << 1);
        const int lch = (l & 63) >> 3;
        // phi of this thread's feature for the 64 tokens of a projected tile
        // sum_z: the z sum over the tile's tokens; in the non-causal totals the zero-filled
        // rows past L (whose phi is not zero) are left out, since z is used after them
        // (tokens at TMEM columns col .. col+63 of this thread's projection row)
        auto phi_row = [&](uint32_t col, const float *nr, uint8_t *dst, bool sum_z, int valid) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tP + col, r0);
            tmem_ld32(tP + col + 32, r1);
            tmem_wait_ld();
            tc_fence_before();  // the projection read, before the barrier ahead of phi_ready
            float zs = 0.f;
#pragma unroll
            for (int ck = 0; ck < 8; ++ck) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t0 = 8 * ck + 2 * e;
                    const uint32_t *rr = t0 < 32 ? r0 : r1;
                    const int i0 = t0 & 31;
                    float e0, e1;
                    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"((__uint_as_float(rr[i0]) - 0.5f * nr[t0]) * log2e));
                    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"((__uint_as_float(rr[i0 + 1]) - 0.5f * nr[t0 + 1]) * log2e));
                    e0 *= inv_sqrt_m;
                    e1 *= inv_sqrt_m;
                    if (sum_z) zs += (!NC || t0 < valid ? e0 : 0.f) + (!NC || t0 + 1 < valid ? e1 : 0.f);
                    w[e] = pack_bf16x2(e0, e1);
                }
                *(uint4 *)(dst + ((ck ^ (l & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            return zs;
        };
        for (int c = 0; c < nch; ++c) {
            const int s = c % NST;
            const int g = tile0 + c;
            if (!group_wait(l == 0, 1, &full[s], (c / NST) & 1, nullptr, 0, false, ctl, 256)) break;
            // |x^|^2 = |x|^2 / sqrt(dk) of the Q and K rows: two threads per row
            {
                const int r = l >> 1, part = l & 1;
                const bool isq = r < 64;
                if (!totals || !isq) {
                    const uint8_t *rowp = (isq ? stage_q(s) : stage_k(s)) + (r & 63) * 128;
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int ch = 4 * part + q;
                        const uint4 wv = *(const uint4 *)(rowp + ((ch ^ (r & 7)) << 4));
                        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = __uint_as_float(ww[e] << 16), x1 = __uint_as_float(ww[e] & 0xFFFF0000u);
                            acc += x0 * x0 + x1 * x1;
                        }
                    }
                    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                    if (part == 0) nrm[r] = acc * 0.125f;  // 1/sqrt(64)
                }
            }
            named_bar(1, 256);
            // totals pass: projection buffer and phi(K) tile by chunk parity
            const int tb = totals ? (c & 1) : 0;
            if (!group_wait(l == 0, 1, &p_done[tb], totals ? (c >> 1) & 1 : c & 1, nullptr, 0, false, ctl, 256))
                break;
            tc_fence_after();
            if (!totals) {
                phi_row(0, nrm, rowq, false, 0);
                // z_c (before this chunk) as bf16 hi / lo in S~ rows 64, 65 at column l
                const __nv_bfloat16 zh = __float2bfloat16_rn(zreg);
                const __nv_bfloat16 zl = __float2bfloat16_rn(zreg - __bfloat162float(zh));
                *(__nv_bfloat16 *)(sblk + 64 * 128 + ((lch ^ 0) << 4)) = zh;
                *(__nv_bfloat16 *)(sblk + 65 * 128 + ((lch ^ 1) << 4)) = zl;
            }
            {
                const float zk = phi_row(totals ? 64 * tb : 64, nrm + 64, tb ? rowq : rowk, totals || !NC,
                                         a.L - g * FV_C);
                if (totals || !NC) zreg += zk;
            }
            fence_async_smem();
            named_bar(1, 256);
            if (l == 0) mbar_arrive(&phi_ready[tb]);
            // bf16 copy of the state (S~ rows 0..63, column l) for the next chunk
            if (!totals && !NC && g + 1 < a.nch) {
                if (!group_wait(l == 0, 1, state_done, c & 1, nullptr, 0, false, ctl, 256)) break;
                tc_fence_after();
                const uint32_t tS = tmem + FT_S + 64 * half + lo;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t sv[32];
                    tmem_ld32(tS + 32 * h, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int j = 32 * h + e;
                        *(__nv_bfloat16 *)(sblk + j * 128 + ((lch ^ (j & 7)) << 4)) =
                            __float2bfloat16_rn(__uint_as_float(sv[e]));
                    }
                }
                fence_async_smem();
                named_bar(1, 256);
                if (l == 0) mbar_arrive(sbar_ready);
            }
        }
        if (totals) {
            // this segment's totals: S rows l and z_l
            if (group_wait(l == 0, 1, totals_done, 0, nullptr, 0, false, ctl, 256)) {
                tc_fence_after();
                const uint32_t tS = tmem + FT_S + 64 * half + lo;
                float *dst = a.ws_S + (((size_t)seg * a.BH + head) * FV_M + l) * FV_DV;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t sv[32];
                    tmem_ld32(tS + 32 * h, sv);
                    tmem_wait_ld();
                    float4 *d4 = (float4 *)(dst + 32 * h);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        d4[q] = make_float4(__uint_as_float(sv[4 * q]), __uint_as_float(sv[4 * q + 1]),
                                            __uint_as_float(sv[4 * q + 2]), __uint_as_float(sv[4 * q + 3]));
                }
                a.ws_z[((size_t)seg * a.BH + head) * FV_M + l] = zreg;
            }
        }
    } else if (warp >= 12 && warp < 16 && !totals) {
        // ------------------------------------------------------------ scores -> P (M = 64 rows)
        // Each thread owns half of two rows: ta = 16 q4 + lane/4 and tb = ta + 8, columns
        // 8k + 2 (lane % 4) and the next one, as a 16x256b TMEM load delivers them; the four
        // threads of a row pool their row sums with shuffles.
        const int q4 = warp & 3, pt = tid - 384;
        const int ta = 16 * q4 + (lane >> 2), tb = ta + 8, cpos = lane & 3;
        const uint32_t tA = tmem + FT_A + ((uint32_t)(32 * q4) << 16);
        for (int c = 0; c < nch; ++c) {
            const int slot = c % FV_DEN;
            if (!group_wait(pt == 0, 2, scores_done, c & 1, &den_empty[slot], ((c / FV_DEN) - 1) & 1,
                            NORM && c >= FV_DEN, ctl))
                break;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld16x256_x8(tA, r);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_free);
            float rsa[2] = {0.f, 0.f}, rsb[2] = {0.f, 0.f};  // row sums: two short chains each
            uint8_t *pa = sm + FV_P + ta * 128 + 4 * cpos, *pb = sm + FV_P + tb * 128 + 4 * cpos;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int s0 = 8 * k + 2 * cpos, s1 = s0 + 1;
                const float a0 = (!NC && s0 <= ta) ? __uint_as_float(r[4 * k]) : 0.f;
                const float a1 = (!NC && s1 <= ta) ? __uint_as_float(r[4 * k + 1]) : 0.f;
                const float b0 = (!NC && s0 <= tb) ? __uint_as_float(r[4 * k + 2]) : 0.f;
                const float b1 = (!NC && s1 <= tb) ? __uint_as_float(r[4 * k + 3]) : 0.f;
                rsa[k & 1] += a0 + a1;
                rsb[k & 1] += b0 + b1;
                *(uint32_t *)(pa + ((k ^ (ta & 7)) << 4)) = pack_bf16x2(a0, a1);
                *(uint32_t *)(pb + ((k ^ (tb & 7)) << 4)) = pack_bf16x2(b0, b1);
            }
            if (NORM) {
                float sa = rsa[0] + rsa[1], sb = rsb[0] + rsb[1];
                sa += __shfl_xor_sync(0xffffffffu, sa, 1);
                sb += __shfl_xor_sync(0xffffffffu, sb, 1);
                sa += __shfl_xor_sync(0xffffffffu, sa, 2);
                sb += __shfl_xor_sync(0xffffffffu, sb, 2);
                if (cpos == 0) {
                    den_intra[slot * FV_C + ta] = sa;
                    den_intra[slot * FV_C + tb] = sb;
                }
            }
            fence_async_smem();
            named_bar(2, 128);
            if (pt == 0) {
                mbar_arrive(p_ready);
                if (NORM) mbar_arrive(&den_full[slot]);
            }
        }
    } else if (warp >= 16 && !totals) {
        // ------------------------------------------------------------ output rows -> global
        // Each thread owns half of two rows, ta = 16 q4 + lane/4 and tb = ta + 8 (columns
        // 8k + 2 (lane % 4) and the next one), as a 16x256b TMEM load delivers them.
        const int q4 = warp & 3, ot = tid - 512;
        const int ta = 16 * q4 + (lane >> 2), tb = ta + 8, cpos = lane & 3;
        for (int c = 0; c < nch; ++c) {
            const int slot = c % FV_DEN;
            const int row0 = (tile0 + c) * FV_C;
            if (!group_wait(ot == 0, 3, o_done, c & 1, &den_full[slot], (c / FV_DEN) & 1, NORM, ctl))
                break;
            tc_fence_after();
            const uint32_t tO = tmem + FT_O + ((uint32_t)(32 * q4) << 16);
            uint32_t r[32], rz[4];
            tmem_ld16x256_x8(tO, r);
            if (NORM) tmem_ld16x256_x1(tO + 64, rz);  // columns 64, 65: phi(q_t).z (hi, lo)
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            float inva = 1.f, invb = 1.f;
            if (NORM) {
                // fast division: 1/den only scales the fp32 row before its bf16 rounding; the
                // thread with the z columns (lane % 4 == 0) shares it with its row's others
                if (cpos == 0) {
                    inva = __fdividef(1.f, __uint_as_float(rz[0]) + __uint_as_float(rz[1]) + den_intra[slot * FV_C + ta]);
                    invb = __fdividef(1.f, __uint_as_float(rz[2]) + __uint_as_float(rz[3]) + den_intra[slot * FV_C + tb]);
                }
                inva = __shfl_sync(0xffffffffu, inva, lane & ~3);
                invb = __shfl_sync(0xffffffffu, invb, lane & ~3);
            }
            named_bar(3, 128);
            if (NORM && ot == 0) mbar_arrive(&den_empty[slot]);
            uint32_t *da = (uint32_t *)(a.out + ((size_t)head * a.L + row0 + ta) * FV_DV) + cpos;
            uint32_t *db = (uint32_t *)(a.out + ((size_t)head * a.L + row0 + tb) * FV_DV) + cpos;
            const bool va = row0 + ta < a.L, vb = row0 + tb < a.L;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (va) da[4 * k] = pack_bf16x2(__uint_as_float(r[4 * k]) * inva, __uint_as_float(r[4 * k + 1]) * inva);
                if (vb) db[4 * k] = pack_bf16x2(__uint_as_float(r[4 * k + 2]) * invb, __uint_as_float(r[4 * k + 3]) * invb);
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

template <bool NORM>
int launch_fv(const Problem &p, int num_sms, bool noncausal = false)
{
    FvArgs a;
    memset(&a, 0, sizeof(a));
    const int BH = p.B * p.H;
    if (!make_map(&a.tm_q, p.q, BH, p.L, FV_DK, FV_C) || !make_map(&a.tm_k, p.k, BH, p.L, FV_DK, FV_C) ||
        !make_map(&a.tm_v, p.v, BH, p.L, FV_DV, FV_C))
        return LA_ERR_CUDA;
    a.omega = p.omega;
    a.out = (__nv_bfloat16 *)p.out;
    a.L = p.L;
    a.nch = (p.L + FV_C - 1) / FV_C;
    a.BH = BH;
    a.err = p.err;
    a.timeout_ns = 2000000000ull;
    const char *e = getenv("LA_DEBUG_TIMEOUT_NS");
    if (e && *e) a.timeout_ns = strtoull(e, nullptr, 10);
    const int nseg = split_segments(BH, a.nch, num_sms, 4, &a.seg_tiles);
    const int ntot = noncausal ? nseg : nseg - 1;  // segments with a totals pass
    if (ntot > 0) {
        const size_t need = (size_t)ntot * BH * ((size_t)FV_M * FV_DV + FV_M) * sizeof(float);
        if (!p.workspace || p.workspace_bytes < need) return LA_ERR_WORKSPACE;
        a.ws_S = (float *)p.workspace;
        a.ws_z = a.ws_S + (size_t)ntot * BH * FV_M * FV_DV;
    }
    a.nseg_all = nseg;
    auto kern = noncausal ? tc_favor_kernel<NORM, true> : tc_favor_kernel<NORM, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FV_ALLOC) != cudaSuccess)
        return LA_ERR_CUDA;
    if (ntot > 0) {
        a.totals = 1;
        a.grid_seg = ntot;
        kern<<<BH * ntot, FV_THREADS, FV_ALLOC, p.stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    a.totals = 0;
    a.grid_seg = nseg;
    if (ntot > 0) {
        // starts while the totals pass drains
        if (launch_dependent(kern, BH * nseg, FV_THREADS, FV_ALLOC, p.stream, a) != cudaSuccess) return LA_ERR_CUDA;
        return LA_OK;
    }
    kern<<<BH * nseg, FV_THREADS, FV_ALLOC, p.stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace

bool tcf_supported(const Problem &p)
{
    return p.dtype == LA_BF16 && !p.lam && p.fm == LA_FM_FAVOR && p.dk == FV_DK && p.m == FV_M &&
           p.dv == FV_DV && p.C == FV_C && p.L >= 2 * FV_C;
}

int tcf_plan(const Problem &p, int num_sms, la_plan_info *info)
{
    int seg_tiles = 0;
    const int nch = (p.L + FV_C - 1) / FV_C;
    const int nseg = split_segments(p.B * p.H, nch, num_sms, 4, &seg_tiles);
    info->grid_x = p.B * p.H * nseg;
    info->grid_y = 1;
    info->block = FV_THREADS;
    info->smem_bytes = FV_ALLOC;
    info->n_launches = nseg > 1 ? 2 : 1;
    info->workspace_bytes =
        nseg > 1 ? (size_t)(nseg - 1) * p.B * p.H * ((size_t)FV_M * FV_DV + FV_M) * sizeof(float) : 0;
    return LA_OK;
}

int tcf_launch(const Problem &p, int num_sms)
{
    if (!tcf_supported(p)) return LA_ERR_UNSUPPORTED;
    return p.normalize ? launch_fv<true>(p, num_sms) : launch_fv<false>(p, num_sms);
}

// non-causal FAVOR+ (the Performer's bidirectional form), C plays no part
bool tcf_nc_supported(const Problem &p)
{
    return p.dtype == LA_BF16 && !p.lam && p.fm == LA_FM_FAVOR && p.dk == FV_DK && p.m == FV_M &&
           p.dv == FV_DV && p.L >= 2 * FV_C;
}

size_t tcf_nc_workspace(const Problem &p, int num_sms)
{
    const int nch = (p.L + FV_C - 1) / FV_C;
    const int nseg = split_segments(p.B * p.H, nch, num_sms, 4, nullptr);
    return (size_t)nseg * p.B * p.H * ((size_t)FV_M * FV_DV + FV_M) * sizeof(float);
}

int tcf_nc_launch(const Problem &p, int num_sms)
{
    if (!tcf_nc_supported(p)) return LA_ERR_UNSUPPORTED;
    return p.normalize ? launch_fv<true>(p, num_sms, true) : launch_fv<false>(p, num_sms, true);
}

}  // namespace la
