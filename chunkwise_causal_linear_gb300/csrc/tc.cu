// tc.cu -- single-pass tensor-core path for chunkwise causal linear attention (sm_103a).
//
// One CTA per (b, h) head sweeps the head's chunks in order ("attention と線形の間",
// section 2, Chunked): for chunk c the output is the carried state read by the chunk's
// queries (inter) plus the causally masked in-chunk scores times the chunk's values
// (intra); then the chunk's phi(K)^T V joins the state.  The normaliser of "Linear
// Attention / Performerの理論と実装" (y_t = phi(q_t)^T S_t / phi(q_t)^T z_t) is carried in
// fp32 beside it.
//
// GB300 mapping (everything stays on chip except q, k, v in and out):
//   * warp 0       TMA producer: Q_c, K_c, V_c tiles (128-byte swizzled) into a 3-stage ring.
//   * warp 1       one thread issues every tcgen05.mma; the warp owns the TMEM allocation.
//   * warps 4-7    feature map phi applied in place in shared memory; fp32 normaliser
//                  terms: z += colsum(phi(K_c)) and phi(q_t).z for the chunk's rows.
//   * warps 8-11   scores -> P: read phi(Q_c)phi(K_c)^T from TMEM, causal mask (diagonal
//                  kept), fp32 row sums for the normaliser, bf16 P into shared memory; and
//                  after each state update, S^T (fp32 in TMEM) -> bf16 copy in TMEM.
//   * warps 12-15  output epilogue: O^T from TMEM, normaliser division, bf16, swizzled
//                  shared-memory tile, TMA store.
// TMEM (512 columns): S^T fp32 [dv lanes x D] | S^T bf16 [dv x D/2] | O^T x2 [dv x C] |
// scores x2 [C x C].  The state is accumulated in fp32 by the MMA and never leaves TMEM;
// the inter-chunk product reads its bf16 copy as the A operand straight from TMEM.
//
// MMAs per chunk (bf16 in, fp32 accumulate), D = feature dim, C = chunk:
//   scores  A_c   = phi(Q_c) phi(K_c)^T         M=C   N=C  K=D
//   inter   O^T   = bf16(S)^T phi(Q_c)^T        M=dv  N=C  K=D   (A from TMEM)
//   state   S^T  += V_c^T phi(K_c)              M=dv  N=D  K=C
//   intra   O^T  += V_c^T P_c^T                 M=dv  N=C  K=C
//
// Every mbarrier wait is bounded (wall-clock limit); on expiry the CTA records
// LA_ERR_TIMEOUT in the device error word, raises a shared abort flag that the other roles
// poll, drains its own async copies / MMAs, frees TMEM and exits.
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace la {

using namespace ptx;

namespace {

constexpr int TC_THREADS = 512;
constexpr int TC_STAGES = 3;

struct TcArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    int L, nch;
    int *err;
    unsigned long long timeout_ns;
    int debug_stall;  // test knob: the feature-map group never signals (forces a timeout)
};

template <int D, int DV, int C>
struct TcLayout {
    static constexpr int Q_BYTES = C * D * 2;
    static constexpr int K_BYTES = C * D * 2;
    static constexpr int V_BYTES = C * DV * 2;
    static constexpr int STAGE_BYTES = Q_BYTES + K_BYTES + V_BYTES;
    static constexpr int P_BYTES = C * C * 2;
    static constexpr int O_BYTES = C * DV * 2;
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_P = TC_STAGES * STAGE_BYTES;
    static constexpr int OFF_O = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_F32 = OFF_O + 2 * O_BYTES;              // float area
    // floats: den_inter[2][C], den_intra[2][C], rden[C], z[D], zpart[4][D]
    static constexpr int N_F32 = 2 * C + 2 * C + C + D + 4 * D;
    static constexpr int OFF_BAR = OFF_F32 + ((N_F32 * 4 + 15) / 16) * 16;
    static constexpr int N_BAR = 3 * TC_STAGES + 2 * 6 + 2 + 2 * 2;
    static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
    // TMEM columns
    static constexpr uint32_t T_S = 0, T_SB = 128, T_O = 256, T_A = 384;
    static_assert(D <= 128 && DV == 128, "tensor-core path: D <= 128, dv == 128");
    static_assert(C == 64, "tensor-core path: C == 64");
    static_assert(ALLOC <= 232448, "shared memory budget");
};

struct Ctl {
    volatile int *abort;
    int *err;
    unsigned long long timeout_ns;
};

// Bounded wait on an mbarrier phase.  False when this CTA is aborting (timeout here or
// elsewhere); the first timeout records LA_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, const Ctl &ctl)
{
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 255) == 0) {
            if (*ctl.abort) return false;
            if (globaltimer() - t0 > ctl.timeout_ns) {
                *ctl.abort = 1;
                record_error(ctl.err, LA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// bf16 (raw 16-bit) -> fp32 for the two halves of a 32-bit word
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int FM>
__device__ __forceinline__ float phi1(float x)
{
    if (FM == LA_FM_ELU1) return x >= 0.f ? x + 1.f : __expf(x);
    return x;
}

template <int D, int DV, int C, int FM, bool NORM>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_chunked_kernel(const __grid_constant__ TcArgs a)
{
    using Lay = TcLayout<D, DV, C>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *f32 = (float *)(sm + Lay::OFF_F32);
    float *den_inter = f32;              // [2][C]
    float *den_intra = den_inter + 2 * C;  // [2][C]
    float *rden = den_intra + 2 * C;     // [C]
    float *zs = rden + C;                // [D]
    float *zpart = zs + D;               // [4][D]
    uint64_t *bars = (uint64_t *)(sm + Lay::OFF_BAR);
    uint64_t *full = bars;                       // [S] TMA -> feature map
    uint64_t *phi_ready = full + TC_STAGES;      // [S] feature map -> MMA
    uint64_t *stage_free = phi_ready + TC_STAGES;  // [S] MMA -> TMA
    uint64_t *scores_done = stage_free + TC_STAGES;  // [2]
    uint64_t *a_free = scores_done + 2;          // [2]
    uint64_t *p_ready = a_free + 2;              // [2]
    uint64_t *o_done = p_ready + 2;              // [2]
    uint64_t *o_free = o_done + 2;               // [2]
    uint64_t *den_full = o_free + 2;             // [2]
    uint64_t *state_done = den_full + 2;         // [1]
    uint64_t *s_ready = state_done + 1;          // [1]
    uint64_t *den_empty = s_ready + 1;           // [2]
    uint64_t *drain = den_empty + 2;             // [1] abort path: MMA drain
    uint32_t *tmem_slot = (uint32_t *)(sm + Lay::OFF_MISC);
    volatile int *abort_flag = (volatile int *)(sm + Lay::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x;
    const int nch = a.nch;
    Ctl ctl{abort_flag, a.err, a.timeout_ns};

    if (tid == 0) {
        for (int i = 0; i < TC_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&phi_ready[i], 1);
            mbar_init(&stage_free[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&scores_done[i], 1);
            mbar_init(&a_free[i], 4);
            mbar_init(&p_ready[i], 1);
            mbar_init(&o_done[i], 1);
            mbar_init(&o_free[i], 4);
            mbar_init(&den_full[i], 2);
            mbar_init(&den_empty[i], 1);
        }
        mbar_init(state_done, 1);
        mbar_init(s_ready, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem + Lay::T_S, tSB = tmem + Lay::T_SB;

    auto stage_q = [&](int s) { return sm + Lay::OFF_STAGE + s * Lay::STAGE_BYTES; };
    auto stage_k = [&](int s) { return stage_q(s) + Lay::Q_BYTES; };
    auto stage_v = [&](int s) { return stage_k(s) + Lay::K_BYTES; };
    auto p_buf = [&](int b) { return sm + Lay::OFF_P + b * Lay::P_BYTES; };
    auto o_buf = [&](int b) { return sm + Lay::OFF_O + b * Lay::O_BYTES; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c % TC_STAGES;
                if (c >= TC_STAGES && !wait_phase(&stage_free[s], ((c / TC_STAGES) - 1) & 1, ctl))
                    break;
                mbar_arrive_expect_tx(&full[s], Lay::STAGE_BYTES);
                for (int kb = 0; kb < D / 64; ++kb) {
                    tma_load_3d(stage_q(s) + kb * C * 128, &a.tm_q, kb * 64, c * C, head, &full[s]);
                    tma_load_3d(stage_k(s) + kb * C * 128, &a.tm_k, kb * 64, c * C, head, &full[s]);
                }
                for (int jb = 0; jb < DV / 64; ++jb)
                    tma_load_3d(stage_v(s) + jb * C * 128, &a.tm_v, jb * 64, c * C, head, &full[s]);
                issued = c + 1;
            }
            // never leave the CTA with loads in flight: wait for every issued stage to land
            for (int c = (issued > TC_STAGES ? issued - TC_STAGES : 0); c < issued; ++c) {
                const int s = c % TC_STAGES;
                const uint64_t t0 = globaltimer();
                while (!mbar_try(&full[s], (c / TC_STAGES) & 1))
                    if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_SC = idesc_bf16_f32(C, C, 0, 0);
            constexpr uint32_t ID_INTER = idesc_bf16_f32(DV, C, 0, 0);
            constexpr uint32_t ID_STATE = idesc_bf16_f32(DV, D, 1, 1);
            constexpr uint32_t ID_INTRA = idesc_bf16_f32(DV, C, 1, 0);
            for (int c = 0; c < nch; ++c) {
                const int s = c % TC_STAGES, b = c & 1;
                uint64_t *ph = (FM == LA_FM_IDENTITY && !NORM) ? &full[s] : &phi_ready[s];
                if (!wait_phase(ph, (c / TC_STAGES) & 1, ctl)) break;
                if (c >= 2 && !wait_phase(&a_free[b], ((c >> 1) - 1) & 1, ctl)) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(stage_q(s)), ka = smem_u32(stage_k(s)),
                               va = smem_u32(stage_v(s)), pa = smem_u32(p_buf(b));
                const uint32_t tA = tmem + Lay::T_A + b * C, tO = tmem + Lay::T_O + b * C;
                // scores: phi(Q_c) phi(K_c)^T, both K-major, K = D in steps of 16
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C * 128 + (ks & 3) * 32;
                    mma_ss(tA, smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024), ID_SC,
                           ks > 0);
                }
                mma_commit(&scores_done[b]);
                if (c >= 1 && !wait_phase(s_ready, (c - 1) & 1, ctl)) break;
                if (c >= 2 && !wait_phase(&o_free[b], ((c >> 1) - 1) & 1, ctl)) break;
                tc_fence_after();
                // inter: bf16(S)^T (TMEM) x phi(Q_c)^T (K-major B), K = D
                if (c >= 1) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * C * 128 + (ks & 3) * 32;
                        mma_ts(tO, tSB + ks * 8, smem_desc(qa + off, 16, 1024), ID_INTER, ks > 0);
                    }
                }
                // state: S^T += V_c^T phi(K_c), both MN-major, K = C in steps of 16 rows
                if (c + 1 < nch) {
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks)
                        mma_ss(tS, smem_desc(va + ks * 2048, C * 128, 1024),
                               smem_desc(ka + ks * 2048, C * 128, 1024), ID_STATE, (c > 0) || (ks > 0));
                    mma_commit(state_done);
                }
                if (!wait_phase(&p_ready[b], (c >> 1) & 1, ctl)) break;
                tc_fence_after();
                // intra: V_c^T (MN-major A) x P_c^T (K-major B), K = C
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tO, smem_desc(va + ks * 2048, C * 128, 1024),
                           smem_desc(pa + ks * 32, 16, 1024), ID_INTRA, (c > 0) || (ks > 0));
                mma_commit(&o_done[b]);
                mma_commit(&stage_free[s]);
            }
            // drain: every MMA issued above has completed before TMEM is released
            mma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try(drain, 0))
                if (globaltimer() - t0 > ctl.timeout_ns) break;
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ feature map / normaliser
        const int ft = tid - 128;
        constexpr int G = D / 8;          // 16-byte chunks per row
        constexpr int RG = 128 / G;       // row groups
        const int g = ft % G, rg = ft / G;
        const int kb = g >> 3, ch = g & 7;
        const int swz = ((ch ^ (rg & 7)) << 4);
        if (NORM)
            for (int i = ft; i < D; i += 128) zs[i] = 0.f;
        named_bar(1, 128);
        if (FM != LA_FM_IDENTITY || NORM) {
            for (int c = 0; c < nch; ++c) {
                const int s = c % TC_STAGES, slot = c & 1;
                bool ok = wait_phase(&full[s], (c / TC_STAGES) & 1, ctl);
                if (NORM && c >= 2) ok = ok && wait_phase(&den_empty[slot], ((c >> 1) - 1) & 1, ctl);
                if (!named_bar_and(1, 128, ok)) break;  // one decision for the whole group
                float zc[8];
                if (NORM) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) zc[e] = zs[8 * g + e];
                }
                // Q: phi in place, phi(q_t).z for the normaliser
                uint8_t *qb = stage_q(s) + kb * C * 128 + swz;
#pragma unroll 2
                for (int n = 0; n < C / RG; ++n) {
                    const int t = rg + RG * n;
                    uint4 *p = (uint4 *)(qb + t * 128);
                    uint4 w = *p;
                    uint32_t *wv = (uint32_t *)&w;
                    float dpart = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float x0 = phi1<FM>(bf_lo(wv[e])), x1 = phi1<FM>(bf_hi(wv[e]));
                        if (NORM) dpart += x0 * zc[2 * e] + x1 * zc[2 * e + 1];
                        if (FM != LA_FM_IDENTITY) wv[e] = pack_bf16x2(x0, x1);
                    }
                    if (FM != LA_FM_IDENTITY) *p = w;
                    if (NORM) {
#pragma unroll
                        for (int o = G / 2; o > 0; o >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, o);
                        if (g == 0) den_inter[slot * C + t] = dpart;
                    }
                }
                // K: phi in place, column sums for z
                float colsum[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) colsum[e] = 0.f;
                uint8_t *kbp = stage_k(s) + kb * C * 128 + swz;
#pragma unroll 2
                for (int n = 0; n < C / RG; ++n) {
                    const int t = rg + RG * n;
                    uint4 *p = (uint4 *)(kbp + t * 128);
                    uint4 w = *p;
                    uint32_t *wv = (uint32_t *)&w;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float x0 = phi1<FM>(bf_lo(wv[e])), x1 = phi1<FM>(bf_hi(wv[e]));
                        colsum[2 * e] += x0;
                        colsum[2 * e + 1] += x1;
                        if (FM != LA_FM_IDENTITY) wv[e] = pack_bf16x2(x0, x1);
                    }
                    if (FM != LA_FM_IDENTITY) *p = w;
                }
                fence_async_smem();
                if (NORM && c + 1 < nch) {
                    // reduce the column sums over the row groups: lanes g, g+G, ... of a
                    // warp, then the four warps through shared memory
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        for (int o = G; o < 32; o <<= 1) colsum[e] += __shfl_xor_sync(0xffffffffu, colsum[e], o);
                    if (lane < G)
#pragma unroll
                        for (int e = 0; e < 8; ++e) zpart[(ft >> 5) * D + 8 * g + e] = colsum[e];
                }
                named_bar(1, 128);
                if (ft == 0 && !a.debug_stall) {
                    mbar_arrive(&phi_ready[s]);
                    if (NORM) mbar_arrive(&den_full[slot]);
                }
                if (NORM && c + 1 < nch) {
                    for (int i = ft; i < D; i += 128)
                        zs[i] += zpart[i] + zpart[D + i] + zpart[2 * D + i] + zpart[3 * D + i];
                    named_bar(1, 128);
                }
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ scores -> P, S readback
        const int q4 = warp & 3;
        const int pt = tid - 256;
        const int t = 16 * q4 + (lane & 15);  // M = 64 TMEM layout: row t at lane t%16 of quadrant t/16
        const bool row_lane = lane < 16;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1, slot = c & 1;
            bool ok = wait_phase(&scores_done[b], (c >> 1) & 1, ctl);
            if (NORM && c >= 2) ok = ok && wait_phase(&den_empty[slot], ((c >> 1) - 1) & 1, ctl);
            if (!named_bar_and(2, 128, ok)) break;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            const uint32_t tA = tmem + Lay::T_A + b * C + lane_off;
            tmem_ld32(tA, r0);
            tmem_ld32(tA + 32, r1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_free[b]);
            if (row_lane) {
                float rs = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int s0 = 2 * e, s1 = 2 * e + 1;
                    float v0 = s0 <= t ? __uint_as_float(r0[s0]) : 0.f;
                    float v1 = s1 <= t ? __uint_as_float(r0[s1]) : 0.f;
                    rs += v0 + v1;
                    pk[e] = pack_bf16x2(v0, v1);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int s0 = 32 + 2 * e, s1 = 33 + 2 * e;
                    float v0 = s0 <= t ? __uint_as_float(r1[2 * e]) : 0.f;
                    float v1 = s1 <= t ? __uint_as_float(r1[2 * e + 1]) : 0.f;
                    rs += v0 + v1;
                    pk[16 + e] = pack_bf16x2(v0, v1);
                }
                uint8_t *prow = p_buf(b) + t * 128;
#pragma unroll
                for (int chn = 0; chn < 8; ++chn)
                    *(uint4 *)(prow + ((chn ^ (t & 7)) << 4)) =
                        make_uint4(pk[4 * chn], pk[4 * chn + 1], pk[4 * chn + 2], pk[4 * chn + 3]);
                if (NORM) den_intra[slot * C + t] = rs;
            }
            fence_async_smem();
            named_bar(2, 128);
            if (pt == 0) {
                mbar_arrive(&p_ready[b]);
                if (NORM) mbar_arrive(&den_full[slot]);
            }
            // bf16 copy of the state for the next chunk's inter product
            if (c + 1 < nch) {
                if (!named_bar_and(2, 128, wait_phase(state_done, c & 1, ctl))) break;
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) {
                    uint32_t sv[32], pk[16];
                    tmem_ld32(tS + lane_off + cb * 32, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]));
                    tmem_st16(tSB + lane_off + cb * 16, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_ready);
            }
        }
        (void)pt;
    } else if (warp >= 12) {
        // ------------------------------------------------------------ output epilogue
        const int q4 = warp & 3;
        const int ot = tid - 384;
        const int j = 32 * q4 + lane;  // M = dv = 128: row j at lane j
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1, slot = c & 1;
            bool ok = wait_phase(&o_done[b], (c >> 1) & 1, ctl);
            if (NORM) ok = ok && wait_phase(&den_full[slot], (c >> 1) & 1, ctl);
            if (!named_bar_and(3, 128, ok)) break;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            const uint32_t tO = tmem + Lay::T_O + b * C + lane_off;
            tmem_ld32(tO, r0);
            tmem_ld32(tO + 32, r1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[b]);
            if (NORM && ot < C) rden[ot] = 1.f / (den_inter[slot * C + ot] + den_intra[slot * C + ot]);
            // the staging buffer of chunk c-2 must have been read by its TMA store
            if (ot == 0 && c >= 2) tma_wait_read_le1();
            named_bar(3, 128);
            if (NORM && ot == 0) mbar_arrive(&den_empty[slot]);
            uint8_t *ob = o_buf(b) + (j >> 6) * C * 128 + ((j & 7) << 1);
            const int jc = (j & 63) >> 3;
#pragma unroll
            for (int tt = 0; tt < 32; ++tt) {
                float v0 = __uint_as_float(r0[tt]), v1 = __uint_as_float(r1[tt]);
                if (NORM) {
                    v0 *= rden[tt];
                    v1 *= rden[tt + 32];
                }
                *(__nv_bfloat16 *)(ob + tt * 128 + ((jc ^ (tt & 7)) << 4)) = __float2bfloat16_rn(v0);
                *(__nv_bfloat16 *)(ob + (tt + 32) * 128 + ((jc ^ (tt & 7)) << 4)) =
                    __float2bfloat16_rn(v1);
            }
            fence_async_smem();
            named_bar(3, 128);
            if (ot == 0) {
                for (int jb = 0; jb < DV / 64; ++jb)
                    tma_store_3d(&a.tm_o, o_buf(b) + jb * C * 128, jb * 64, c * C, head);
                tma_commit_group();
            }
        }
        if (ot == 0) tma_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = (EncodeTiledFn)p;
    }
    return fn;
}

// [BH, L, d] bf16 viewed as a 3-D tensor (d innermost); box = 64 columns x C rows x 1 head,
// 128-byte swizzle, rows past L read as zero (loads) or are dropped (stores).
bool make_map(CUtensorMap *m, const void *ptr, int BH, int L, int d, int C)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)C, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int DV, int C, int FM, bool NORM>
int launch_t(const Problem &p)
{
    using Lay = TcLayout<D, DV, C>;
    TcArgs a;
    memset(&a, 0, sizeof(a));
    const int BH = p.B * p.H;
    if (!make_map(&a.tm_q, p.q, BH, p.L, p.dk, C) || !make_map(&a.tm_k, p.k, BH, p.L, p.dk, C) ||
        !make_map(&a.tm_v, p.v, BH, p.L, p.dv, C) || !make_map(&a.tm_o, p.out, BH, p.L, p.dv, C))
        return LA_ERR_CUDA;
    a.L = p.L;
    a.nch = (p.L + C - 1) / C;
    a.err = p.err;
    a.timeout_ns = 2000000000ull;
    const char *e = getenv("LA_DEBUG_TIMEOUT_NS");
    if (e && *e) a.timeout_ns = strtoull(e, nullptr, 10);
    const char *st = getenv("LA_DEBUG_STALL");
    a.debug_stall = (st && *st && *st != '0') ? 1 : 0;
    auto kern = tc_chunked_kernel<D, DV, C, FM, NORM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC) !=
        cudaSuccess)
        return LA_ERR_CUDA;
    kern<<<BH, TC_THREADS, Lay::ALLOC, p.stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

template <int D>
int launch_d(const Problem &p)
{
    const bool n = p.normalize != 0;
    if (p.fm == LA_FM_IDENTITY)
        return n ? launch_t<D, 128, 64, LA_FM_IDENTITY, true>(p)
                 : launch_t<D, 128, 64, LA_FM_IDENTITY, false>(p);
    return n ? launch_t<D, 128, 64, LA_FM_ELU1, true>(p) : launch_t<D, 128, 64, LA_FM_ELU1, false>(p);
}

}  // namespace

bool tc_supported(const Problem &p, int num_sms)
{
    (void)num_sms;
    if (p.dtype != LA_BF16) return false;
    if (p.lam) return false;
    if (p.fm != LA_FM_IDENTITY && p.fm != LA_FM_ELU1) return false;
    if (p.dk != p.D) return false;
    if (!(p.D == 64 || p.D == 128) || p.dv != 128) return false;
    if (p.C != 64) return false;
    if (p.L < 2 * 64) return false;  // short sequences: the generic path is as fast
    return true;
}

int tc_plan(const Problem &p, int num_sms, la_plan_info *info)
{
    (void)num_sms;
    info->grid_x = p.B * p.H;
    info->grid_y = 1;
    info->block = TC_THREADS;
    info->smem_bytes = p.D == 128 ? TcLayout<128, 128, 64>::ALLOC : TcLayout<64, 128, 64>::ALLOC;
    info->n_launches = 1;
    info->workspace_bytes = 0;
    return LA_OK;
}

int tc_launch(const Problem &p, int num_sms)
{
    if (!tc_supported(p, num_sms)) return LA_ERR_UNSUPPORTED;
    return p.D == 128 ? launch_d<128>(p) : launch_d<64>(p);
}

}  // namespace la
