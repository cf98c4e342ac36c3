// tc_wide.cu -- tensor-core path for chunks wider than one tile: C = 128 or 256 (sm_103a).
//
// The chunked order of "attention と線形の間" section 2 with C = 64 R rows per chunk (R = 2 or
// 4): a query row reads the state carried from the chunks before its own (inter), plus the
// causally masked scores of every key of its own chunk (intra); the normaliser of "Linear
// Attention / Performerの理論と実装" rides along as in the one-tile kernel.
//
// Rows still move in 64-row tiles.  Query tile r of a chunk (r = 0 .. R-1) is processed as
// 1 + r score blocks against the key tiles of its chunk:
//   * the diagonal block (its own keys, causal mask, plus the z rows for phi(q).z), from the
//     tile's own stage;
//   * the r blocks against the chunk's earlier key tiles, unmasked; those K, V tiles are
//     fetched again (from L2, where they were read a few tiles earlier) into a two-slot key
//     ring, and phi is applied to them again.
// The inter product reads the bf16 state copy made at the chunk start; the fp32 state takes
// every tile's update, and its bf16 copy is refreshed once per chunk, after the chunk's last
// tile.  z (phi(q).z in the denominator) is likewise the value at the chunk start.  So the
// intra work per row grows with C and the state work per row shrinks with 1/C, as in the
// page's cost model (section 3).
//
// Warp roles (as in the one-tile kernel): 0 TMA producer, 1 MMA issuer, 4-11 feature map,
// 12-15 scores -> P (+ bf16 state copy), 16-19 output epilogue.
//
// MMAs per query tile (bf16 in, fp32 accumulate), D = feature dim, T = 64:
//   scores  A_k   = phi(Q) [phi(K_k); z]^T       M=T   N=T(+8)  K=D   per block k
//   inter   O^T   = bf16(S_chunk)^T phi(Q)^T     M=dv  N=T      K=D   (A in TMEM)
//   state   S^T  += V^T phi(K)                   M=dv  N=D      K=T
//   intra   O^T  += V_k^T P_k^T                  M=dv  N=T      K=T   per block k
// Every wait is bounded as in the one-tile kernel.
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

constexpr int TW_THREADS = 640;
constexpr int TW_FWARPS = 8;
constexpr int TW_STAGES = 2;   // main stages (Q, K, V of a query tile)
constexpr int TW_KR = 2;       // key ring (K, V of an earlier tile of the chunk)
constexpr int TW_DEN = 4;

struct TwArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    int L, nch;          // nch: 64-row tiles of a head
    int seg_tiles;       // a multiple of R: segments start on chunk edges
    int grid_seg, totals, BH;
    float *ws_T;         // [segments-1][BH][dv][D]
    float *ws_z;         // [segments-1][BH][D]
    int *err;
    unsigned long long timeout_ns;
};

template <int D, int DV, bool NORM>
struct TwLayout {
    static constexpr int T = 64;
    static constexpr int KROWS = NORM ? T + 8 : T;
    static constexpr int NSC = KROWS;
    static constexpr int K_BLK = KROWS * 128;        // 64-feature block of a stage's K tile
    static constexpr int Q_BYTES = T * D * 2;
    static constexpr int K_BYTES = (D / 64) * K_BLK;
    static constexpr int V_BYTES = T * DV * 2;
    static constexpr int STAGE_BYTES = Q_BYTES + K_BYTES + V_BYTES;
    static constexpr int STAGE_TX = Q_BYTES + T * D * 2 + V_BYTES;
    static constexpr int RK_BYTES = T * D * 2;       // key ring: K (64-row blocks), V
    static constexpr int RING_BYTES = RK_BYTES + V_BYTES;
    static constexpr int P_BYTES = T * T * 2;
    static constexpr int O_BYTES = T * DV * 2;
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_RING = TW_STAGES * STAGE_BYTES;
    static constexpr int OFF_P = OFF_RING + TW_KR * RING_BYTES;   // two P tiles
    static constexpr int OFF_O = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_F32 = OFF_O + O_BYTES;
    // floats: rden[TW_DEN][T], z (running), z at the chunk start, zpart[TW_FWARPS][D]
    static constexpr int N_F32 = TW_DEN * T + 2 * D + TW_FWARPS * D;
    static constexpr int OFF_BAR = OFF_F32 + ((N_F32 * 4 + 15) / 16) * 16;
    static constexpr int N_BAR = 3 * TW_STAGES + 3 * TW_KR + 2 * 3 + 2 * 2 + 2 * TW_DEN + 3;
    static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;
    static constexpr uint32_t T_S = 0, T_SB = 128, T_O = 192, T_A = 320, A_STRIDE = 80;
    static_assert(D <= 128 && (DV == 64 || DV == 128), "D <= 128, dv 64 or 128");
    static_assert(K_BLK % 1024 == 0 && STAGE_BYTES % 1024 == 0 && RING_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(ALLOC <= 232448, "shared memory budget");
};

template <int D, int DV, int R, int FM, bool NORM>
__global__ void __launch_bounds__(TW_THREADS, 1) tc_wide_kernel(const __grid_constant__ TwArgs a)
{
    using Lay = TwLayout<D, DV, NORM>;
    constexpr int T = Lay::T;
    constexpr bool PHI = FM != LA_FM_IDENTITY;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *f32 = (float *)(sm + Lay::OFF_F32);
    float *rden = f32;                  // [TW_DEN][T]
    float *zs = rden + TW_DEN * T;      // [D] running z
    float *zcs = zs + D;                // [D] z at the chunk start
    float *zpart = zcs + D;             // [TW_FWARPS][D]
    uint64_t *bars = (uint64_t *)(sm + Lay::OFF_BAR);
    uint64_t *full = bars;                          // [S] TMA -> feature map
    uint64_t *phi_ready = full + TW_STAGES;         // [S] feature map -> MMA
    uint64_t *stage_free = phi_ready + TW_STAGES;   // [S] MMA -> TMA
    uint64_t *kfull = stage_free + TW_STAGES;       // [KR] TMA -> feature map
    uint64_t *kready = kfull + TW_KR;               // [KR] feature map -> MMA
    uint64_t *kfree = kready + TW_KR;               // [KR] MMA -> TMA
    uint64_t *scores_done = kfree + TW_KR;          // [2] by block parity
    uint64_t *a_free = scores_done + 2;             // [2]
    uint64_t *p_ready = a_free + 2;                 // [2]
    uint64_t *o_done = p_ready + 2;                 // [2] by tile parity
    uint64_t *o_free = o_done + 2;                  // [2]
    uint64_t *den_full = o_free + 2;                // [TW_DEN]
    uint64_t *den_empty = den_full + TW_DEN;        // [TW_DEN]
    uint64_t *state_done = den_empty + TW_DEN;      // chunk end: fp32 state complete
    uint64_t *s_ready = state_done + 1;             // bf16 state copy of the new chunk
    uint64_t *drain = s_ready + 1;
    uint32_t *tmem_slot = (uint32_t *)(sm + Lay::OFF_MISC);
    volatile int *abort_flag = (volatile int *)(sm + Lay::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x / a.grid_seg, seg = blockIdx.x % a.grid_seg;
    const int tile0 = seg * a.seg_tiles;
    const int nt = min(a.seg_tiles, a.nch - tile0);   // tiles of this CTA
    const bool totals = a.totals != 0;
    Ctl ctl{abort_flag, a.err, a.timeout_ns};
    if (totals) pdl_trigger();  // the main pass may be scheduled now
    else pdl_wait();            // the totals pass (if any) has completed

    auto stage_q = [&](int s) { return sm + Lay::OFF_STAGE + s * Lay::STAGE_BYTES; };
    auto stage_k = [&](int s) { return stage_q(s) + Lay::Q_BYTES; };
    auto stage_v = [&](int s) { return stage_k(s) + Lay::K_BYTES; };
    auto ring_k = [&](int k) { return sm + Lay::OFF_RING + k * Lay::RING_BYTES; };
    auto ring_v = [&](int k) { return ring_k(k) + Lay::RK_BYTES; };
    auto p_tile = [&](int bb) { return sm + Lay::OFF_P + bb * Lay::P_BYTES; };
    uint8_t *const o_tile = sm + Lay::OFF_O;

    if (tid == 0) {
        for (int i = 0; i < TW_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&phi_ready[i], 1);
            mbar_init(&stage_free[i], 1);
        }
        for (int i = 0; i < TW_KR; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kready[i], 1);
            mbar_init(&kfree[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&scores_done[i], 1);
            mbar_init(&a_free[i], 4);
            mbar_init(&p_ready[i], 1);
            mbar_init(&o_done[i], 1);
            mbar_init(&o_free[i], 4);
        }
        for (int i = 0; i < TW_DEN; ++i) {
            mbar_init(&den_full[i], 1);
            mbar_init(&den_empty[i], 1);
        }
        mbar_init(state_done, 1);
        mbar_init(s_ready, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (NORM) {
        for (int e = tid; e < TW_STAGES * (D / 64) * 8 * 8; e += TW_THREADS) {
            const int st = e / ((D / 64) * 64), r = e % ((D / 64) * 64);
            const int kb = r / 64, row = T + (r % 64) / 8, chn = r % 8;
            *(uint4 *)(stage_k(st) + kb * Lay::K_BLK + row * 128 + chn * 16) = make_uint4(0, 0, 0, 0);
        }
        for (int i = tid; i < D; i += TW_THREADS) {
            float z0 = 0.f;
            if (!totals)
                for (int g = 0; g < seg; ++g) z0 += a.ws_z[((size_t)g * a.BH + head) * D + i];
            zs[i] = z0;
            zcs[i] = z0;
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem + Lay::T_S, tSB = tmem + Lay::T_SB;
    if (warp >= 4 + TW_FWARPS && warp < 8 + TW_FWARPS) {
        // state and its bf16 copy start at the sum of the earlier segments' totals
        const uint32_t lo = (uint32_t)(32 * (warp & 3)) << 16;
        const int jr = (DV == 128) ? 32 * (warp & 3) + lane : 16 * (warp & 3) + (lane & 15);
        const bool live = (DV == 128) || lane < 16;
        const int nprev = totals ? 0 : seg;
#pragma unroll 1
        for (int col = 0; col < D; col += 16) {
            float acc[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = 0.f;
            if (live)
                for (int g = 0; g < nprev; ++g) {
                    const float4 *src = (const float4 *)(a.ws_T + (((size_t)g * a.BH + head) * DV + jr) * D + col);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 v4 = src[q];
                        acc[4 * q] += v4.x; acc[4 * q + 1] += v4.y; acc[4 * q + 2] += v4.z; acc[4 * q + 3] += v4.w;
                    }
                }
            uint32_t w32[16], w16[8];
#pragma unroll
            for (int e = 0; e < 16; ++e) w32[e] = __float_as_uint(acc[e]);
#pragma unroll
            for (int e = 0; e < 8; ++e) w16[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
            tmem_st16(tS + lo + col, w32);
            tmem_st8(tSB + lo + col / 2, w16);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0, sph = 0, kslot = 0, kuse = 0;
            bool ok = true;
            for (int c = 0; c < nt && ok; ++c) {
                if (c >= TW_STAGES && !wait_phase(&stage_free[s], sph ^ 1, ctl)) break;
                const int row = (tile0 + c) * T;
                mbar_arrive_expect_tx(&full[s], totals ? Lay::STAGE_TX - Lay::Q_BYTES : Lay::STAGE_TX);
                for (int kb = 0; kb < D / 64; ++kb) {
                    if (!totals) tma_load_3d(stage_q(s) + kb * T * 128, &a.tm_q, kb * 64, row, head, &full[s]);
                    tma_load_3d(stage_k(s) + kb * Lay::K_BLK, &a.tm_k, kb * 64, row, head, &full[s]);
                }
                for (int jb = 0; jb < DV / 64; ++jb)
                    tma_load_3d(stage_v(s) + jb * T * 128, &a.tm_v, jb * 64, row, head, &full[s]);
                if (++s == TW_STAGES) { s = 0; sph ^= 1; }
                if (totals) continue;
                // the chunk's earlier key tiles, for this query tile's off-diagonal blocks
                const int r = c % R;
                for (int k = c - r; k < c; ++k) {
                    if (kuse >= TW_KR && !wait_phase(&kfree[kslot], ((kuse / TW_KR) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    const int krow = (tile0 + k) * T;
                    mbar_arrive_expect_tx(&kfull[kslot], Lay::RK_BYTES + Lay::V_BYTES);
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_3d(ring_k(kslot) + kb * T * 128, &a.tm_k, kb * 64, krow, head, &kfull[kslot]);
                    for (int jb = 0; jb < DV / 64; ++jb)
                        tma_load_3d(ring_v(kslot) + jb * T * 128, &a.tm_v, jb * 64, krow, head, &kfull[kslot]);
                    ++kuse;
                    if (++kslot == TW_KR) kslot = 0;
                }
            }
            // never leave with loads in flight: the last uses of every stage and ring slot
            const uint64_t t0 = globaltimer();
            for (int i = 0; i < TW_STAGES; ++i) {
                // stage i was used ceil((nt - i) / S) times; wait for its last completion
                const int uses = nt > i ? (nt - i + TW_STAGES - 1) / TW_STAGES : 0;
                if (uses > 0)
                    while (!mbar_try_sleep(&full[i], (uses - 1) & 1, 200000u))
                        if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
            for (int i = 0; i < TW_KR; ++i) {
                const int uses = kuse > i ? (kuse - i + TW_KR - 1) / TW_KR : 0;
                if (uses > 0)
                    while (!mbar_try_sleep(&kfull[i], (uses - 1) & 1, 200000u))
                        if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_SCD = idesc_bf16_f32(T, Lay::NSC, 0, 0);   // diagonal block (+ z rows)
            constexpr uint32_t ID_SCO = idesc_bf16_f32(T, T, 0, 0);          // earlier key tile
            constexpr uint32_t ID_INTER = idesc_bf16_f32(DV, T, 0, 0);
            constexpr uint32_t ID_STATE = idesc_bf16_f32(DV, D, 1, 1);
            constexpr uint32_t ID_INTRA = idesc_bf16_f32(DV, T, 1, 0);
            bool ok = true;
            int s = 0, sph = 0;
            if (totals) {
                for (int c = 0; c < nt; ++c) {
                    uint64_t *ph = (!PHI && !NORM) ? &full[s] : &phi_ready[s];
                    if (!wait_phase(ph, sph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ka = smem_u32(stage_k(s)), va = smem_u32(stage_v(s));
#pragma unroll
                    for (int ks = 0; ks < T / 16; ++ks)
                        mma_ss(tS, desc_add(smem_desc(va, T * 128, 1024), ks * 2048),
                               desc_add(smem_desc(ka, Lay::K_BLK, 1024), ks * 2048), ID_STATE, 1);
                    mma_commit(&stage_free[s]);
                    if (++s == TW_STAGES) { s = 0; sph ^= 1; }
                }
                if (ok) mma_commit(state_done);
                ok = false;
            }
            int kb = 0;                   // score blocks issued so far (A / P parity)
            int kuse = 0;                 // key-ring loads consumed so far
            int nref = 0;                 // bf16 state refreshes consumed
            for (int c = 0; ok && c < nt; ++c) {
                const int b = c & 1, r = c % R, gt = tile0 + c;
                uint64_t *ph = (!PHI && !NORM) ? &full[s] : &phi_ready[s];
                if (!wait_phase(ph, sph, ctl)) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(stage_q(s)), ka = smem_u32(stage_k(s)), va = smem_u32(stage_v(s));
                const uint32_t tO = tmem + Lay::T_O + b * T;
                // blocks: n = 0 is the diagonal, n = 1..r the key tiles c - r .. c - 1 (ring)
                const int nblk = 1 + r;
                // scores of block n into A[(kb + n) & 1]
                auto scores = [&](int n) -> bool {
                    const int bb = (kb + n) & 1, use = (kb + n) >> 1;
                    if (kb + n >= 2 && !wait_phase(&a_free[bb], (use - 1) & 1, ctl)) return false;
                    const uint32_t tA = tmem + Lay::T_A + bb * Lay::A_STRIDE;
                    if (n == 0) {
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t qo = (ks >> 2) * T * 128 + (ks & 3) * 32;
                            const uint32_t ko = (ks >> 2) * Lay::K_BLK + (ks & 3) * 32;
                            mma_ss(tA, desc_add(smem_desc(qa, 16, 1024), qo), desc_add(smem_desc(ka, 16, 1024), ko),
                                   ID_SCD, ks > 0);
                        }
                    } else {
                        const int slot = (kuse + n - 1) % TW_KR, u = (kuse + n - 1) / TW_KR;
                        uint64_t *kr = PHI ? &kready[slot] : &kfull[slot];
                        if (!wait_phase(kr, u & 1, ctl)) return false;
                        tc_fence_after();
                        const uint32_t rk = smem_u32(ring_k(slot));
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t qo = (ks >> 2) * T * 128 + (ks & 3) * 32;
                            mma_ss(tA, desc_add(smem_desc(qa, 16, 1024), qo), desc_add(smem_desc(rk, 16, 1024), qo),
                                   ID_SCO, ks > 0);
                        }
                    }
                    mma_commit(&scores_done[bb]);
                    return true;
                };
                // intra of block n: O^T += V_n^T P^T
                auto intra = [&](int n) -> bool {
                    const int bb = (kb + n) & 1, use = (kb + n) >> 1;
                    if (!wait_phase(&p_ready[bb], use & 1, ctl)) return false;
                    tc_fence_after();
                    const uint32_t pa = smem_u32(p_tile(bb));
                    const uint32_t vv = n == 0 ? va : smem_u32(ring_v((kuse + n - 1) % TW_KR));
#pragma unroll
                    for (int ks = 0; ks < T / 16; ++ks)
                        mma_ss(tO, desc_add(smem_desc(vv, T * 128, 1024), ks * 2048), desc_add(smem_desc(pa, 16, 1024), ks * 32),
                               ID_INTRA, 1);
                    if (n > 0) mma_commit(&kfree[(kuse + n - 1) % TW_KR]);
                    return true;
                };
                if (!scores(0)) break;
                // inter from the chunk-start state copy (refreshed after the previous chunk)
                if (c >= 2 && !wait_phase(&o_free[b], ((c >> 1) - 1) & 1, ctl)) break;
                if (r == 0 && c >= 1) {
                    if (!wait_phase(s_ready, nref & 1, ctl)) break;
                    ++nref;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t qo = (ks >> 2) * T * 128 + (ks & 3) * 32;
                    mma_ts(tO, tSB + ks * 8, desc_add(smem_desc(qa, 16, 1024), qo), ID_INTER, ks > 0);
                }
                // state: every tile joins the fp32 state; the copy is refreshed at chunk ends
                if (gt + 1 < a.nch) {
#pragma unroll
                    for (int ks = 0; ks < T / 16; ++ks)
                        mma_ss(tS, desc_add(smem_desc(va, T * 128, 1024), ks * 2048),
                               desc_add(smem_desc(ka, Lay::K_BLK, 1024), ks * 2048), ID_STATE, 1);
                    if (r == R - 1) mma_commit(state_done);
                }
                // scores run one block ahead of the intra products (P is double-buffered)
                bool bok = true;
                for (int n = 0; n < nblk && bok; ++n) {
                    if (n + 1 < nblk) bok = scores(n + 1);
                    if (bok) bok = intra(n);
                }
                if (!bok) break;
                kb += nblk;
                kuse += r;
                mma_commit(&o_done[b]);
                mma_commit(&stage_free[s]);
                if (++s == TW_STAGES) { s = 0; sph ^= 1; }
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_sleep(drain, 0, 200000u))
                if (globaltimer() - t0 > ctl.timeout_ns) break;
        }
    } else if (warp >= 4 && warp < 4 + TW_FWARPS) {
        // ------------------------------------------------------------ feature map / z
        const int ft = tid - 128;
        constexpr int NF = 32 * TW_FWARPS;
        constexpr int G = D / 8;
        constexpr int RG = NF / G;
        constexpr int NR = T / RG;
        const int g = ft % G, rg = ft / G;
        const int kbk = g >> 3, ch = g & 7;
        const int q_swz = kbk * T * 128 + ((ch ^ (rg & 7)) << 4) + rg * 128;
        const int k_swz = kbk * Lay::K_BLK + ((ch ^ (rg & 7)) << 4) + rg * 128;
        int s = 0, sph = 0, kuse = 0;
        if (PHI || NORM) {
            for (int c = 0; c < nt; ++c) {
                const int r = c % R;
                if (!group_wait(ft == 0, 1, &full[s], sph, nullptr, 0, false, ctl, NF)) break;
                if (NORM && !totals && r == 0) {
                    // a new chunk: its phi(q).z uses z at the chunk start
                    for (int i = ft; i < D; i += NF) zcs[i] = zs[i];
                    named_bar(1, NF);
                }
                uint4 *qp = (uint4 *)(stage_q(s) + q_swz);
                uint4 *kp = (uint4 *)(stage_k(s) + k_swz);
                uint4 wq[NR], wk[NR];
#pragma unroll
                for (int n = 0; n < NR; ++n) {
                    if (PHI && !totals) wq[n] = qp[n * RG * 8];
                    wk[n] = kp[n * RG * 8];
                }
                if (NORM && !totals && ft < 8 * (D / 64) * 2) {
                    const int zkb = ft / 16, zr = (ft / 8) & 1, zch = ft & 7;
                    const float4 z0 = ((const float4 *)zcs)[(64 * zkb + 8 * zch) / 4];
                    const float4 z1 = ((const float4 *)zcs)[(64 * zkb + 8 * zch) / 4 + 1];
                    const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float h0 = __bfloat162float(__float2bfloat16_rn(zz[2 * e]));
                        float h1 = __bfloat162float(__float2bfloat16_rn(zz[2 * e + 1]));
                        pk[e] = zr ? pack_bf16x2(zz[2 * e] - h0, zz[2 * e + 1] - h1) : pack_bf16x2(h0, h1);
                    }
                    const int row = T + zr;
                    *(uint4 *)(stage_k(s) + zkb * Lay::K_BLK + row * 128 + ((zch ^ (row & 7)) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                if (PHI && !totals) {
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
                for (int n = 0; n < NR; ++n) {
                    uint32_t *wv = (uint32_t *)&wk[n];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (PHI) wv[e] = elu1_bf16x2(wv[e]);
                        if (NORM) add_bf16x2_to_f32(colsum[2 * e], colsum[2 * e + 1], wv[e]);
                    }
                }
                if (PHI) {
#pragma unroll
                    for (int n = 0; n < NR; ++n) {
                        if (!totals) qp[n * RG * 8] = wq[n];
                        kp[n * RG * 8] = wk[n];
                    }
                }
                fence_async_smem();
                const bool zupd = NORM && (c + 1 < nt || totals);
                if (zupd) {
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
                if (ft == 0) mbar_arrive(&phi_ready[s]);
                if (zupd) {
                    for (int i = ft; i < D; i += NF) {
                        float acc = 0.f;
#pragma unroll
                        for (int w = 0; w < TW_FWARPS; ++w) acc += zpart[w * D + i];
                        zs[i] += acc;
                    }
                    named_bar(1, NF);
                }
                if (++s == TW_STAGES) { s = 0; sph ^= 1; }
                // phi of the chunk's earlier key tiles, fetched again into the key ring
                if (PHI && !totals) {
                    bool ok = true;
                    for (int k = 0; k < r; ++k, ++kuse) {
                        const int slot = kuse % TW_KR;
                        if (!group_wait(ft == 0, 1, &kfull[slot], (kuse / TW_KR) & 1, nullptr, 0, false, ctl, NF)) {
                            ok = false;
                            break;
                        }
                        uint4 *rp = (uint4 *)(ring_k(slot) + q_swz);
#pragma unroll
                        for (int n = 0; n < NR; ++n) {
                            uint4 w = rp[n * RG * 8];
                            uint32_t *wv = (uint32_t *)&w;
#pragma unroll
                            for (int e = 0; e < 4; ++e) wv[e] = elu1_bf16x2(wv[e]);
                            rp[n * RG * 8] = w;
                        }
                        fence_async_smem();
                        named_bar(1, NF);
                        if (ft == 0) mbar_arrive(&kready[slot]);
                    }
                    if (!ok) break;
                }
            }
            if (totals && NORM)
                for (int i = ft; i < D; i += NF) a.ws_z[((size_t)seg * a.BH + head) * D + i] = zs[i];
        }
    } else if (warp >= 4 + TW_FWARPS && warp < 8 + TW_FWARPS) {
        // ------------------------------------------------------------ scores -> P, state copy
        const int q4 = warp & 3;
        const int pt = tid - 32 * (4 + TW_FWARPS);
        const int t = 16 * q4 + (lane & 15);
        const bool row_lane = lane < 16;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        if (totals) {
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
        int kb = 0, nref = 0;
        for (int c = 0; c < nt && !totals; ++c) {
            const int slot = c % TW_DEN, r = c % R, gt = tile0 + c;
            float rsa[4] = {0.f, 0.f, 0.f, 0.f}, dz = 0.f;  // row sum: four short chains
            bool ok = true;
            for (int n = 0; n <= r && ok; ++n, ++kb) {
                const int bb = kb & 1;
                const bool need_den = NORM && n == 0 && c >= TW_DEN;
                if (!group_wait(pt == 0, 2, &scores_done[bb], (kb >> 1) & 1, &den_empty[slot],
                                ((c / TW_DEN) - 1) & 1, need_den, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tA = tmem + Lay::T_A + bb * Lay::A_STRIDE + lane_off;
                if (NORM && n == 0) {
                    uint32_t rz[8];
                    tmem_ld8(tA + T, rz);
                    tmem_wait_ld();
                    dz = __uint_as_float(rz[0]) + __uint_as_float(rz[1]);  // phi(q_t).z at the chunk start
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t rr[32];
                    tmem_ld32(tA + 32 * h, rr);
                    tmem_wait_ld();
                    if (h == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&a_free[bb]);
                    }
                    if (row_lane) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            // diagonal block: keys s <= t; earlier key tiles: all keys
                            const int s0 = 32 * h + 2 * e, s1 = s0 + 1;
                            const float v0 = (n > 0 || s0 <= t) ? __uint_as_float(rr[2 * e]) : 0.f;
                            const float v1 = (n > 0 || s1 <= t) ? __uint_as_float(rr[2 * e + 1]) : 0.f;
                            rsa[e & 3] += v0 + v1;
                            pk[e] = pack_bf16x2(v0, v1);
                        }
                        uint8_t *prow = p_tile(bb) + t * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int chn = 4 * h + q;
                            *(uint4 *)(prow + ((chn ^ (t & 7)) << 4)) =
                                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                        }
                    }
                }
                // fast division: 1/den only scales the fp32 row before its bf16 rounding
                if (NORM && n == r && row_lane)
                    rden[slot * T + t] = __fdividef(1.f, dz + ((rsa[0] + rsa[1]) + (rsa[2] + rsa[3])));
                fence_async_smem();
                named_bar(2, 128);
                if (pt == 0) {
                    mbar_arrive(&p_ready[bb]);
                    if (NORM && n == r) mbar_arrive(&den_full[slot]);
                }
            }
            if (!ok) break;
            // at a chunk end: bf16 copy of the state for the next chunk's inter products
            if (r == R - 1 && gt + 1 < a.nch) {
                if (!group_wait(pt == 0, 2, state_done, nref & 1, nullptr, 0, false, ctl)) break;
                ++nref;
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
    } else if (warp >= 8 + TW_FWARPS) {
        // ------------------------------------------------------------ output epilogue
        const int q4 = warp & 3;
        const int ot = tid - 32 * (8 + TW_FWARPS);
        const int j = (DV == 128) ? 32 * q4 + lane : 16 * q4 + (lane & 15);
        const bool live = (DV == 128) || lane < 16;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const bool odd = lane & 1;
        uint8_t *const ob = o_tile + (j >> 6) * T * 128 + (((j & 7) & ~1) << 1);
        const int jc = (j & 63) >> 3;
        for (int c = 0; c < nt && !totals; ++c) {
            const int b = c & 1, slot = c % TW_DEN;
            if (!group_wait(ot == 0, 3, &o_done[b], (c >> 1) & 1, &den_full[slot], (c / TW_DEN) & 1, NORM, ctl))
                break;
            tc_fence_after();
            if (ot == 0 && c >= 1) tma_wait_read_all();
            named_bar(3, 128);
            const uint32_t tO = tmem + Lay::T_O + b * T + lane_off;
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
                float rd[32];
                if (NORM) {
                    const float4 *rp = (const float4 *)(rden + slot * T + 32 * h);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 v = rp[q];
                        rd[4 * q] = v.x; rd[4 * q + 1] = v.y; rd[4 * q + 2] = v.z; rd[4 * q + 3] = v.w;
                    }
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    float a0 = __uint_as_float(r[2 * u]), a1 = __uint_as_float(r[2 * u + 1]);
                    if (NORM) {
                        a0 *= rd[2 * u];
                        a1 *= rd[2 * u + 1];
                    }
                    const float recv = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
                    const int tt = 32 * h + 2 * u + (odd ? 1 : 0);
                    const uint32_t wv = odd ? pack_bf16x2(recv, a1) : pack_bf16x2(a0, recv);
                    if (live) *(uint32_t *)(ob + tt * 128 + ((jc ^ (tt & 7)) << 4)) = wv;
                }
            }
            fence_async_smem();
            named_bar(3, 128);
            if (ot == 0) {
                for (int jb = 0; jb < DV / 64; ++jb)
                    tma_store_3d(&a.tm_o, o_tile + jb * T * 128, jb * 64, (tile0 + c) * T, head);
                tma_commit_group();
                if (NORM) mbar_arrive(&den_empty[slot]);
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

// segments of a multiple of R tiles (chunk edges), at least 4 tiles
int tw_segments(const Problem &p, int R, int num_sms, int *seg_tiles)
{
    const int tiles = (p.L + 63) / 64;
    int st = 0;
    split_segments(p.B * p.H, tiles, num_sms, 4, &st);
    st = ((st + R - 1) / R) * R;
    if (seg_tiles) *seg_tiles = st;
    return (tiles + st - 1) / st;
}

size_t tw_workspace(const Problem &p, int nseg)
{
    if (nseg <= 1) return 0;
    return (size_t)(nseg - 1) * p.B * p.H * ((size_t)p.dv * p.D + p.D) * sizeof(float);
}

template <int D, int DV, int R, int FM, bool NORM>
int launch_w(const Problem &p, int num_sms)
{
    using Lay = TwLayout<D, DV, NORM>;
    TwArgs a;
    memset(&a, 0, sizeof(a));
    const int BH = p.B * p.H;
    if (!make_map(&a.tm_q, p.q, BH, p.L, p.dk, 64) || !make_map(&a.tm_k, p.k, BH, p.L, p.dk, 64) ||
        !make_map(&a.tm_v, p.v, BH, p.L, p.dv, 64) || !make_map(&a.tm_o, p.out, BH, p.L, p.dv, 64))
        return LA_ERR_CUDA;
    a.L = p.L;
    a.nch = (p.L + 63) / 64;
    const int nseg = tw_segments(p, R, num_sms, &a.seg_tiles);
    a.BH = BH;
    if (nseg > 1) {
        if (!p.workspace || p.workspace_bytes < tw_workspace(p, nseg)) return LA_ERR_WORKSPACE;
        a.ws_T = (float *)p.workspace;
        a.ws_z = a.ws_T + (size_t)(nseg - 1) * BH * DV * D;
    }
    a.err = p.err;
    a.timeout_ns = 2000000000ull;
    const char *e = getenv("LA_DEBUG_TIMEOUT_NS");
    if (e && *e) a.timeout_ns = strtoull(e, nullptr, 10);
    auto kern = tc_wide_kernel<D, DV, R, FM, NORM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC) != cudaSuccess)
        return LA_ERR_CUDA;
    if (nseg > 1) {
        a.totals = 1;
        a.grid_seg = nseg - 1;
        kern<<<BH * (nseg - 1), TW_THREADS, Lay::ALLOC, p.stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    a.totals = 0;
    a.grid_seg = nseg;
    if (nseg > 1) {
        // starts while the totals pass drains
        if (launch_dependent(kern, BH * nseg, TW_THREADS, Lay::ALLOC, p.stream, a) != cudaSuccess) return LA_ERR_CUDA;
        return LA_OK;
    }
    kern<<<BH * nseg, TW_THREADS, Lay::ALLOC, p.stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

template <int D, int DV, int R>
int launch_wr(const Problem &p, int sms)
{
    const bool n = p.normalize != 0;
    if (p.fm == LA_FM_IDENTITY)
        return n ? launch_w<D, DV, R, LA_FM_IDENTITY, true>(p, sms) : launch_w<D, DV, R, LA_FM_IDENTITY, false>(p, sms);
    return n ? launch_w<D, DV, R, LA_FM_ELU1, true>(p, sms) : launch_w<D, DV, R, LA_FM_ELU1, false>(p, sms);
}

template <int D, int DV>
int launch_wd(const Problem &p, int sms)
{
    return p.C == 128 ? launch_wr<D, DV, 2>(p, sms) : launch_wr<D, DV, 4>(p, sms);
}

}  // namespace

bool tcw_supported(const Problem &p)
{
    if (p.dtype != LA_BF16 || p.lam) return false;
    if (p.fm != LA_FM_IDENTITY && p.fm != LA_FM_ELU1) return false;
    if (p.dk != p.D) return false;
    if (!((p.D == 64 && (p.dv == 64 || p.dv == 128)) || (p.D == 128 && p.dv == 128))) return false;
    if (p.C != 128 && p.C != 256) return false;
    return p.L >= 2 * 64;
}

int tcw_plan(const Problem &p, int num_sms, la_plan_info *info)
{
    int seg_tiles = 0;
    const int nseg = tw_segments(p, p.C / 64, num_sms, &seg_tiles);
    info->grid_x = p.B * p.H * nseg;
    info->grid_y = 1;
    info->block = TW_THREADS;
    auto alloc = [&](auto d, auto dv) {
        constexpr int D = decltype(d)::value, DV = decltype(dv)::value;
        return p.normalize ? TwLayout<D, DV, true>::ALLOC : TwLayout<D, DV, false>::ALLOC;
    };
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    info->smem_bytes = p.D == 128 ? alloc(I128{}, I128{}) : (p.dv == 128 ? alloc(I64{}, I128{}) : alloc(I64{}, I64{}));
    info->n_launches = nseg > 1 ? 2 : 1;
    info->workspace_bytes = tw_workspace(p, nseg);
    return LA_OK;
}

int tcw_launch(const Problem &p, int num_sms)
{
    if (!tcw_supported(p)) return LA_ERR_UNSUPPORTED;
    if (p.D == 128) return launch_wd<128, 128>(p, num_sms);
    return p.dv == 128 ? launch_wd<64, 128>(p, num_sms) : launch_wd<64, 64>(p, num_sms);
}

}  // namespace la
