// tc_wide.cu -- tensor-core path for chunks wider than one tile: C = 128 or 256 (sm_103a).
//
// The chunked order of "attention と線形の間" section 2 with C = 64 R rows per chunk (R = 2 or
// 4): a query row reads the state carried from the chunks before its own (inter), plus the
// causally masked scores of every key of its own chunk (intra); the normaliser of "Linear
// Attention / Performerの理論と実装" rides along as in the one-tile kernel.
//
// Rows still move in 64-row tiles.  Query tile r of a chunk (r = 0 .. R-1) is processed as
// 1 + r score blocks against the key tiles of its chunk:
//   * the diagonal block (its own keys, causal mask, plus the z rows for phi(q).z);
//   * the r blocks against the chunk's earlier key tiles, unmasked.
// Q tiles and (K, V) tiles live in two shared-memory rings.  A Q slot is released as soon as
// its tile's scores and inter product are done; a K/V slot holds phi(K) and V until the last
// tile of its chunk is done, so the earlier key tiles are read from HBM once and phi is
// applied to them once.  The K/V ring has room for more than one chunk (2R slots where they
// fit, else R + 1), so the next chunk's tiles load while the current one computes.
// The inter product reads the bf16 state copy made at the chunk start; the fp32 state takes
// every tile's update, and its bf16 copy is refreshed once per chunk, after the chunk's last
// tile.  z (phi(q).z in the denominator) is likewise the value at the chunk start.  So the
// intra work per row grows with C and the state work per row shrinks with 1/C, as in the
// page's cost model (section 3).
//
// Warp roles (as in the one-tile kernel): 0 TMA producer (K, V; and Q unless warp 5 loads
// it), 5 TMA producer of Q when the Q ring is shorter than the K/V ring, 1 MMA issuer, 2-4,
// 6-8, 10-11 feature map, 12-15 scores -> P (+ bf16 state copy), 16-19 output epilogue (rows
// stored from registers).
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

// The feature-map group is warps 2, 3, 4, 6, 7, 8, 10, 11, so that none shares a
// sub-partition (warp % 4) with the MMA issuer (warp 1) and takes its issue slots.
// Returns the warp's rank in the group, or -1.
__device__ __forceinline__ int tw_phi_rank(int warp)
{
    if (warp < 2 || warp >= 12 || (warp & 3) == 1) return -1;
    return warp - 2 - (warp > 5) - (warp > 9);
}
constexpr int TW_DEN = 4;
constexpr int TW_SMEM = 232448 - 1024;   // opt-in shared memory less the alignment slack

struct TwArgs {
    CUtensorMap tm_q, tm_k, tm_v;
    void *out;           // bf16 [BH][L][dv]
    int L, nch;          // nch: 64-row tiles of a head
    int seg_tiles;       // a multiple of R: segments start on chunk edges
    int grid_seg, totals, BH;
    float *ws_T;         // [segments-1][BH][dv][D]
    float *ws_z;         // [segments-1][BH][D]
    int *err;
    unsigned long long timeout_ns;
};

// K/V slots: 2R (a whole chunk ahead) where that fits beside two Q slots, else fewer, at
// least R + 1; then as many Q slots (2 to 4) as the rest allows.
constexpr int tw_pick_nkv(int R, int kv, int q, int fixed)
{
    int n = 2 * R;
    while (n > R + 1 && n * kv + 2 * q + fixed > TW_SMEM) --n;
    return n;
}

constexpr int tw_pick_nq(int nkv, int kv, int q, int fixed)
{
    int n = 4;
    while (n > 2 && nkv * kv + n * q + fixed > TW_SMEM) --n;
    return n;
}

template <int D, int DV, int R, bool NORM>
struct TwLayout {
    static constexpr int T = 64;
    static constexpr int KROWS = NORM ? T + 8 : T;
    static constexpr int NSC = KROWS;
    static constexpr int K_BLK = KROWS * 128;        // 64-feature block of a slot's K tile
    static constexpr int Q_BYTES = T * D * 2;
    static constexpr int K_BYTES = (D / 64) * K_BLK;
    static constexpr int V_BYTES = T * DV * 2;
    static constexpr int KV_BYTES = K_BYTES + V_BYTES;
    static constexpr int KV_TX = T * D * 2 + V_BYTES;   // bytes TMA writes into a K/V slot
    static constexpr int P_BYTES = T * T * 2;
    // floats: rden[TW_DEN][T], z (running), z at the chunk start, zpart[TW_FWARPS][D]
    static constexpr int N_F32 = TW_DEN * T + 2 * D + TW_FWARPS * D;
    static constexpr int F32_BYTES = ((N_F32 * 4 + 15) / 16) * 16;
    static constexpr int MAX_BAR = 3 * 2 * R + 4 + 2 * 5 + 2 * TW_DEN + 3;
    static constexpr int FIXED = 2 * P_BYTES + F32_BYTES + MAX_BAR * 8 + 16;
    static constexpr int NKV = tw_pick_nkv(R, KV_BYTES, Q_BYTES, FIXED);
    static constexpr int NQ = tw_pick_nq(NKV, KV_BYTES, Q_BYTES, FIXED);
    static constexpr int OFF_KV = 0;
    static constexpr int OFF_Q = OFF_KV + NKV * KV_BYTES;
    static constexpr int OFF_P = OFF_Q + NQ * Q_BYTES;     // two P tiles
    static constexpr int OFF_F32 = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_BAR = OFF_F32 + F32_BYTES;
    static constexpr int N_BAR = 3 * NKV + NQ + 2 * 5 + 2 * TW_DEN + 3;
    static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;
    static constexpr uint32_t T_S = 0, T_SB = 128, T_O = 192, T_A = 320, A_STRIDE = 80;
    static_assert(D <= 128 && (DV == 64 || DV == 128), "D <= 128, dv 64 or 128");
    static_assert(K_BLK % 1024 == 0 && KV_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(NKV > R && N_BAR <= MAX_BAR && BYTES <= TW_SMEM, "shared memory budget");
    static_assert(NQ <= NKV, "a Q load must not reach a K/V barrier's previous phase");
};

template <int D, int DV, int R, int FM, bool NORM>
__global__ void __launch_bounds__(TW_THREADS, 1) tc_wide_kernel(const __grid_constant__ TwArgs a)
{
    using Lay = TwLayout<D, DV, R, NORM>;
    constexpr int T = Lay::T;
    constexpr int NKV = Lay::NKV, NQ = Lay::NQ;
    constexpr bool QP = NQ < NKV;  // Q loads from their own producer thread
    constexpr bool PHI = FM != LA_FM_IDENTITY;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *f32 = (float *)(sm + Lay::OFF_F32);
    float *rden = f32;                  // [TW_DEN][T]
    float *zs = rden + TW_DEN * T;      // [D] running z
    float *zcs = zs + D;                // [D] z at the chunk start
    float *zpart = zcs + D;             // [TW_FWARPS][D]
    uint64_t *bars = (uint64_t *)(sm + Lay::OFF_BAR);
    uint64_t *kv_full = bars;                       // [NKV] TMA -> feature map (Q, K, V of a tile)
    uint64_t *phi_ready = kv_full + NKV;            // [NKV] feature map -> MMA
    uint64_t *kv_free = phi_ready + NKV;            // [NKV] MMA -> TMA, at the end of the slot's chunk
    uint64_t *q_free = kv_free + NKV;               // [NQ] MMA -> TMA
    uint64_t *scores_done = q_free + NQ;            // [2] by block parity
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

    // local tile c: Q in slot c % NQ, K and V in slot c % NKV
    auto q_tile = [&](int s) { return sm + Lay::OFF_Q + s * Lay::Q_BYTES; };
    auto k_tile = [&](int s) { return sm + Lay::OFF_KV + s * Lay::KV_BYTES; };
    auto v_tile = [&](int s) { return k_tile(s) + Lay::K_BYTES; };
    auto p_tile = [&](int bb) { return sm + Lay::OFF_P + bb * Lay::P_BYTES; };

    if (tid == 0) {
        for (int i = 0; i < NKV; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&phi_ready[i], 1);
            mbar_init(&kv_free[i], 1);
        }
        for (int i = 0; i < NQ; ++i) mbar_init(&q_free[i], 1);
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
        // rows T .. T+7 of every K block: z hi, z lo, then zeros (TMA writes rows 0 .. T-1)
        for (int e = tid; e < NKV * (D / 64) * 8 * 8; e += TW_THREADS) {
            const int st = e / ((D / 64) * 64), r = e % ((D / 64) * 64);
            const int kb = r / 64, row = T + (r % 64) / 8, chn = r % 8;
            *(uint4 *)(k_tile(st) + kb * Lay::K_BLK + row * 128 + chn * 16) = make_uint4(0, 0, 0, 0);
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
        // With a Q ring shorter than the K/V ring (QP), a tile's K and V load as soon as its
        // K/V slot is free and its Q (main pass) is loaded by warp 5 once its Q slot is free,
        // completing on the same barrier, which this thread arms with the bytes of all three.
        // (The Q bytes may land before the arming: the transaction count goes negative
        // meanwhile.  The Q slot of tile c frees only after tile c - NQ is done, NQ <= NKV, so
        // the barrier's previous phase is complete by then.)  Otherwise this thread loads all
        // three when both slots are free.
        if (lane == 0) {
            for (int c = 0; c < nt; ++c) {
                const int ks = c % NKV, qs = c % NQ;
                // the slot's previous tile: its chunk is done (K/V), its own products are done (Q)
                if (c >= NKV && !wait_phase(&kv_free[ks], ((c / NKV) - 1) & 1, ctl)) break;
                if (!QP && !totals && c >= NQ && !wait_phase(&q_free[qs], ((c / NQ) - 1) & 1, ctl)) break;
                const int row = (tile0 + c) * T;
                mbar_arrive_expect_tx(&kv_full[ks], totals ? Lay::KV_TX : Lay::KV_TX + Lay::Q_BYTES);
                for (int kb = 0; kb < D / 64; ++kb) {
                    if (!QP && !totals) tma_load_3d(q_tile(qs) + kb * T * 128, &a.tm_q, kb * 64, row, head, &kv_full[ks]);
                    tma_load_3d(k_tile(ks) + kb * Lay::K_BLK, &a.tm_k, kb * 64, row, head, &kv_full[ks]);
                }
                for (int jb = 0; jb < DV / 64; ++jb)
                    tma_load_3d(v_tile(ks) + jb * T * 128, &a.tm_v, jb * 64, row, head, &kv_full[ks]);
            }
            // never leave with loads in flight: slot i was filled ceil((nt - i) / NKV) times
            const uint64_t t0 = globaltimer();
            for (int i = 0; i < NKV; ++i) {
                const int uses = nt > i ? (nt - i + NKV - 1) / NKV : 0;
                if (uses > 0)
                    while (!mbar_try_sleep(&kv_full[i], (uses - 1) & 1, 200000u))
                        if (globaltimer() - t0 > ctl.timeout_ns) break;
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ TMA producer (Q, QP only)
        // (warp 5 is otherwise idle: it shares a sub-partition with the MMA issuer, so it does
        // no feature-map work, and this thread mostly sleeps in its waits)
        if (QP && lane == 0 && !totals) {
            for (int c = 0; c < nt; ++c) {
                const int qs = c % NQ;
                // the slot's previous tile: its scores and inter product are done
                if (c >= NQ && !wait_phase(&q_free[qs], ((c / NQ) - 1) & 1, ctl)) break;
                const int row = (tile0 + c) * T;
                for (int kb = 0; kb < D / 64; ++kb)
                    tma_load_3d(q_tile(qs) + kb * T * 128, &a.tm_q, kb * 64, row, head, &kv_full[c % NKV]);
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
            if (totals) {
                for (int c = 0; c < nt; ++c) {
                    const int ks = c % NKV;
                    uint64_t *ph = (!PHI && !NORM) ? &kv_full[ks] : &phi_ready[ks];
                    if (!wait_phase(ph, (c / NKV) & 1, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ka = smem_u32(k_tile(ks)), va = smem_u32(v_tile(ks));
#pragma unroll
                    for (int kk = 0; kk < T / 16; ++kk)
                        mma_ss(tS, desc_add(smem_desc(va, T * 128, 1024), kk * 2048),
                               desc_add(smem_desc(ka, Lay::K_BLK, 1024), kk * 2048), ID_STATE, 1);
                    mma_commit(&kv_free[ks]);
                }
                if (ok) mma_commit(state_done);
                ok = false;
            }
            // Issue order of tile c: the first off-diagonal block's scores (the P warps need
            // them next), inter, state, then the intra products, each block's scores issued
            // ahead of the previous block's intra (the score accumulator and P are
            // double-buffered); after the tile's commits, the next tile's diagonal scores.
            // (Issuing those before this tile's last intra product, as the one-tile kernel
            // does, measured slower here: it delays the commits that free K/V slots.)
            auto wait_phi = [&](int c) {
                uint64_t *ph = (!PHI && !NORM) ? &kv_full[c % NKV] : &phi_ready[c % NKV];
                return wait_phase(ph, (c / NKV) & 1, ctl);
            };
            // scores of block n of local tile c into A[g & 1], g = the block's running index
            auto scores = [&](int c, int n, int g) -> bool {
                const int bb = g & 1, use = g >> 1;
                if (g >= 2 && !wait_phase(&a_free[bb], (use - 1) & 1, ctl)) return false;
                const uint32_t tA = tmem + Lay::T_A + bb * Lay::A_STRIDE;
                const int ksn = n == 0 ? c % NKV : (c - c % R + n - 1) % NKV;
                const uint32_t qa = smem_u32(q_tile(c % NQ)), kk = smem_u32(k_tile(ksn));
                tc_fence_after();
#pragma unroll
                for (int ki = 0; ki < D / 16; ++ki) {
                    const uint32_t qo = (ki >> 2) * T * 128 + (ki & 3) * 32;
                    const uint32_t ko = (ki >> 2) * Lay::K_BLK + (ki & 3) * 32;
                    mma_ss(tA, desc_add(smem_desc(qa, 16, 1024), qo), desc_add(smem_desc(kk, 16, 1024), ko),
                           n == 0 ? ID_SCD : ID_SCO, ki > 0);
                }
                mma_commit(&scores_done[bb]);
                return true;
            };
            int kb = 0;                   // score blocks of the tiles before this one
            int nref = 0;                 // bf16 state refreshes consumed
            if (ok && nt > 0) ok = wait_phi(0) && scores(0, 0, 0);
            for (int c = 0; ok && c < nt; ++c) {
                const int b = c & 1, r = c % R, gt = tile0 + c, ks = c % NKV, qs = c % NQ;
                tc_fence_after();
                const uint32_t qa = smem_u32(q_tile(qs)), ka = smem_u32(k_tile(ks)), va = smem_u32(v_tile(ks));
                const uint32_t tO = tmem + Lay::T_O + b * T;
                // blocks: n = 0 is the diagonal, n = 1..r the key tiles c - r .. c - 1, still resident
                const int nblk = 1 + r;
                // intra of block n: O^T += V_n^T P^T
                auto intra = [&](int n) -> bool {
                    const int bb = (kb + n) & 1, use = (kb + n) >> 1;
                    if (!wait_phase(&p_ready[bb], use & 1, ctl)) return false;
                    tc_fence_after();
                    const uint32_t pa = smem_u32(p_tile(bb));
                    const uint32_t vv = smem_u32(v_tile(n == 0 ? ks : (c - r + n - 1) % NKV));
#pragma unroll
                    for (int ki = 0; ki < T / 16; ++ki)
                        mma_ss(tO, desc_add(smem_desc(vv, T * 128, 1024), ki * 2048),
                               desc_add(smem_desc(pa, 16, 1024), ki * 32), ID_INTRA, 1);
                    return true;
                };
                if (r >= 1 && !scores(c, 1, kb + 1)) break;
                // inter from the chunk-start state copy (refreshed after the previous chunk)
                if (c >= 2 && !wait_phase(&o_free[b], ((c >> 1) - 1) & 1, ctl)) break;
                if (r == 0 && c >= 1) {
                    if (!wait_phase(s_ready, nref & 1, ctl)) break;
                    ++nref;
                }
                tc_fence_after();
#pragma unroll
                for (int ki = 0; ki < D / 16; ++ki) {
                    const uint32_t qo = (ki >> 2) * T * 128 + (ki & 3) * 32;
                    mma_ts(tO, tSB + ki * 8, desc_add(smem_desc(qa, 16, 1024), qo), ID_INTER, ki > 0);
                }
                // state: every tile joins the fp32 state; the copy is refreshed at chunk ends
                if (gt + 1 < a.nch) {
#pragma unroll
                    for (int ki = 0; ki < T / 16; ++ki)
                        mma_ss(tS, desc_add(smem_desc(va, T * 128, 1024), ki * 2048),
                               desc_add(smem_desc(ka, Lay::K_BLK, 1024), ki * 2048), ID_STATE, 1);
                    if (r == R - 1) mma_commit(state_done);
                }
                bool bok = true;
                for (int n = 0; n < nblk && bok; ++n) {
                    if (n >= 1 && n + 1 < nblk) bok = scores(c, n + 1, kb + n + 1);
                    if (bok) bok = intra(n);
                    // the chunk's last tile: key tile n - 1 of the chunk has had its last use
                    if (bok && r == R - 1 && n >= 1) mma_commit(&kv_free[(c - r + n - 1) % NKV]);
                }
                if (!bok) break;
                kb += nblk;
                mma_commit(&o_done[b]);
                mma_commit(&q_free[qs]);
                if (r == R - 1) mma_commit(&kv_free[ks]);
                if (c + 1 < nt && !(wait_phi(c + 1) && scores(c + 1, 0, kb))) break;
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_sleep(drain, 0, 200000u))
                if (globaltimer() - t0 > ctl.timeout_ns) break;
        }
    } else if (tw_phi_rank(warp) >= 0) {
        // ------------------------------------------------------------ feature map / z
        const int ft = 32 * tw_phi_rank(warp) + lane;
        constexpr int NF = 32 * TW_FWARPS;
        constexpr int G = D / 8;
        constexpr int RG = NF / G;
        constexpr int NR = T / RG;
        const int g = ft % G, rg = ft / G;
        const int kbk = g >> 3, ch = g & 7;
        const int q_swz = kbk * T * 128 + ((ch ^ (rg & 7)) << 4) + rg * 128;
        const int k_swz = kbk * Lay::K_BLK + ((ch ^ (rg & 7)) << 4) + rg * 128;
        if (PHI || NORM) {
            for (int c = 0; c < nt; ++c) {
                const int r = c % R, ks = c % NKV, qs = c % NQ;
                if (!group_wait(ft == 0, 1, &kv_full[ks], (c / NKV) & 1, nullptr, 0, false, ctl, NF)) break;
                if (NORM && !totals && r == 0) {
                    // a new chunk: its phi(q).z uses z at the chunk start
                    for (int i = ft; i < D; i += NF) zcs[i] = zs[i];
                    named_bar(1, NF);
                }
                uint4 *qp = (uint4 *)(q_tile(qs) + q_swz);
                uint4 *kp = (uint4 *)(k_tile(ks) + k_swz);
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
                    *(uint4 *)(k_tile(ks) + zkb * Lay::K_BLK + row * 128 + ((zch ^ (row & 7)) << 4)) =
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
                if (ft == 0) mbar_arrive(&phi_ready[ks]);
                if (zupd) {
                    for (int i = ft; i < D; i += NF) {
                        float acc = 0.f;
#pragma unroll
                        for (int w = 0; w < TW_FWARPS; ++w) acc += zpart[w * D + i];
                        zs[i] += acc;
                    }
                    named_bar(1, NF);
                }
            }
            if (totals && NORM)
                for (int i = ft; i < D; i += NF) a.ws_z[((size_t)seg * a.BH + head) * D + i] = zs[i];
        }
    } else if (warp >= 4 + TW_FWARPS && warp < 8 + TW_FWARPS) {
        // ------------------------------------------------------------ scores -> P, state copy
        const int q4 = warp & 3;
        const int pt = tid - 32 * (4 + TW_FWARPS);
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
        // Each thread owns half of two rows of the block: rows ta = 16 q4 + lane/4 and tb = ta + 8,
        // columns 8k + 2 (lane % 4) and the next one (k = 0..7), as a 16x256b TMEM load
        // delivers them; the four threads of a row pool their row sums with shuffles.
        const int ta = 16 * q4 + (lane >> 2), tb = ta + 8, cpos = lane & 3;
        int kb = 0, nref = 0;
        for (int c = 0; c < nt && !totals; ++c) {
            const int slot = c % TW_DEN, r = c % R, gt = tile0 + c;
            float rsa[2] = {0.f, 0.f}, rsb[2] = {0.f, 0.f};  // this thread's part of the row sums
            float dza = 0.f, dzb = 0.f;                      // phi(q).z at the chunk start (cpos 0)
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
                    uint32_t rz[4];
                    tmem_ld16x256_x1(tA + T, rz);  // columns T, T+1: the z rows (hi, lo)
                    tmem_wait_ld();
                    dza = __uint_as_float(rz[0]) + __uint_as_float(rz[1]);
                    dzb = __uint_as_float(rz[2]) + __uint_as_float(rz[3]);
                }
                uint32_t rr[32];
                tmem_ld16x256_x8(tA, rr);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_free[bb]);
                uint8_t *pa = p_tile(bb) + ta * 128 + 4 * cpos, *pb = p_tile(bb) + tb * 128 + 4 * cpos;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    // diagonal block: keys s <= t; earlier key tiles: all keys
                    const int s0 = 8 * k + 2 * cpos, s1 = s0 + 1;
                    const float a0 = (n > 0 || s0 <= ta) ? __uint_as_float(rr[4 * k]) : 0.f;
                    const float a1 = (n > 0 || s1 <= ta) ? __uint_as_float(rr[4 * k + 1]) : 0.f;
                    const float b0 = (n > 0 || s0 <= tb) ? __uint_as_float(rr[4 * k + 2]) : 0.f;
                    const float b1 = (n > 0 || s1 <= tb) ? __uint_as_float(rr[4 * k + 3]) : 0.f;
                    rsa[k & 1] += a0 + a1;
                    rsb[k & 1] += b0 + b1;
                    *(uint32_t *)(pa + ((k ^ (ta & 7)) << 4)) = pack_bf16x2(a0, a1);
                    *(uint32_t *)(pb + ((k ^ (tb & 7)) << 4)) = pack_bf16x2(b0, b1);
                }
                if (NORM && n == r) {
                    float sa = rsa[0] + rsa[1], sb = rsb[0] + rsb[1];
                    sa += __shfl_xor_sync(0xffffffffu, sa, 1);
                    sb += __shfl_xor_sync(0xffffffffu, sb, 1);
                    sa += __shfl_xor_sync(0xffffffffu, sa, 2);
                    sb += __shfl_xor_sync(0xffffffffu, sb, 2);
                    // fast division: 1/den only scales the fp32 row before its bf16 rounding
                    if (cpos == 0) {
                        rden[slot * T + ta] = __fdividef(1.f, dza + sa);
                        rden[slot * T + tb] = __fdividef(1.f, dzb + sb);
                    }
                }
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
        // For each token a warp writes 32 neighbouring output columns (64 contiguous bytes)
        // straight from registers; rows past L are skipped.
        const int q4 = warp & 3;
        const int ot = tid - 32 * (8 + TW_FWARPS);
        // row j of O^T: lane j (dv = 128), or lane j%16 of quadrant j/16 (dv = 64)
        const int j = (DV == 128) ? 32 * q4 + lane : 16 * q4 + (lane & 15);
        const bool live = (DV == 128) || lane < 16;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const bool odd = lane & 1;
        for (int c = 0; c < nt && !totals; ++c) {
            const int b = c & 1, slot = c % TW_DEN;
            if (!group_wait(ot == 0, 3, &o_done[b], (c >> 1) & 1, &den_full[slot], (c / TW_DEN) & 1, NORM, ctl))
                break;
            tc_fence_after();
            const int row0 = (tile0 + c) * T;
            const int nrow = min(T, a.L - row0);   // rows of this tile inside the sequence
            uint32_t *const o = (uint32_t *)((__nv_bfloat16 *)a.out + ((size_t)head * a.L + row0) * DV + (j & ~1));
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
                const float2 *rp = (const float2 *)(rden + slot * T + 32 * h);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    float a0 = __uint_as_float(r[2 * u]), a1 = __uint_as_float(r[2 * u + 1]);
                    if (NORM) {
                        const float2 f = rp[u];
                        a0 *= f.x;
                        a1 *= f.y;
                    }
                    // lanes j, j^1 swap one value per pair of rows: each writes two neighbouring
                    // columns of one row as a 32-bit word
                    const float recv = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
                    const int tt = 32 * h + 2 * u + (odd ? 1 : 0);
                    const uint32_t wv = odd ? pack_bf16x2(recv, a1) : pack_bf16x2(a0, recv);
                    if (live && tt < nrow) o[(size_t)tt * (DV / 2)] = wv;
                }
            }
            if (NORM) {
                // every thread has read this tile's 1/den
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
    using Lay = TwLayout<D, DV, R, NORM>;
    TwArgs a;
    memset(&a, 0, sizeof(a));
    const int BH = p.B * p.H;
    if (!make_map(&a.tm_q, p.q, BH, p.L, p.dk, 64) || !make_map(&a.tm_k, p.k, BH, p.L, p.dk, 64) ||
        !make_map(&a.tm_v, p.v, BH, p.L, p.dv, 64))
        return LA_ERR_CUDA;
    a.out = p.out;
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
        if (p.C == 128) return p.normalize ? TwLayout<D, DV, 2, true>::ALLOC : TwLayout<D, DV, 2, false>::ALLOC;
        return p.normalize ? TwLayout<D, DV, 4, true>::ALLOC : TwLayout<D, DV, 4, false>::ALLOC;
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
