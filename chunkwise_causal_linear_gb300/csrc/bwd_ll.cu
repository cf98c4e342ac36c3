// bwd_ll.cu -- the anti-causal sums of the log-linear mask's backward pass (generic fp32 path).
//
// Under the mask M_ts = lambda_t^(l(t,s)) of "論文紹介：Log Linear Attention" (slide 17;
// l = 0 if s = t else 1 + floor(log2(t XOR s))), the gradients of the keys and values sum over
// the later rows t >= s with the weight of the LATER row:
//     out_s = sum_{t >= s} lambda_t^(l(t,s)) (a_s . b_t) c_t,
// with (a, b, c) = (v', D', phi(q)) for dphi(k) and (phi(k), phi(q), D) for dv.  The weight
// belongs to the summed index, so the carried states of the forward recurrence (whose
// blocks merge as they age) cannot hold it.  This file uses the level structure directly:
// with chunks of C = 2^c rows, a pair in chunks c_t > c_s has level 1 + c + m, m = the
// highest bit in which c_t and c_s differ, so c_s lies in the lower half and c_t in the upper
// half of the aligned block of 2^(m+1) chunks that contains both.  Each such block therefore
// needs one state, built from its upper half with that level's weights,
//     W_m(beta) = sum_{t in upper half of block beta} b_t (lambda_t^(1+c+m) c_t)^T,
// and a row s of chunk c_s reads a_s . W_m(c_s >> (m+1)) for every bit m of c_s that is 0
// (when that upper half exists), plus the pairs inside its own chunk (levels 0 .. c)
// explicitly.  The sum over t is the same set of pairs as the definition, grouped by block.
//
// Rows are fp32 [BH][L][width]; lambda is [BH][L][nl].  Two kernels: the states (one CTA
// per head, block and 64 x 64 tile of W), then the rows (one CTA per head, chunk and
// 32-column slice of out).
#include <stdint.h>

#include "common.cuh"

namespace la {

namespace {

constexpr int LLB_THREADS = 256;
constexpr int LLB_R = 16;    // rows per tile
constexpr int LLB_TW = 64;   // W tile edge (states kernel)
constexpr int LLB_WC = 32;   // output columns per CTA (rows kernel)

// number of chunk-block levels m (blocks of 2^(m+1) chunks whose upper half can be non-empty)
__host__ __device__ inline int llb_levels(int nch)
{
    int m = 0;
    while ((1 << m) < nch) ++m;
    return m;  // m = 0 .. levels-1 have 2^m < nch
}

// blocks at level m: ceil(nch / 2^(m+1))
__host__ __device__ inline int llb_blocks(int nch, int m) { return (nch + (2 << m) - 1) >> (m + 1); }

__device__ inline int llb_level_of(int nch, int y, int *beta)
{
    int m = 0;
    for (;; ++m) {
        const int nb = llb_blocks(nch, m);
        if (y < nb) break;
        y -= nb;
    }
    *beta = y;
    return m;
}

// W_m(beta)[i][j] for one 64 x 64 tile (i0, j0): rows of the block's upper half
__global__ void __launch_bounds__(LLB_THREADS) llb_states_kernel(const float *b, const float *c,
                                                                  const float *lam, float *W, int L,
                                                                  int C, int log2C, int Da, int Wc,
                                                                  int nl, size_t w_stride)
{
    __shared__ float sb[LLB_R][LLB_TW];
    __shared__ float sc[LLB_R][LLB_TW];
    const int head = blockIdx.x;
    const int nch = (L + C - 1) / C;
    int beta;
    const int m = llb_level_of(nch, blockIdx.y, &beta);
    const int ti = blockIdx.z / ((Wc + LLB_TW - 1) / LLB_TW), tj = blockIdx.z % ((Wc + LLB_TW - 1) / LLB_TW);
    const int i0 = ti * LLB_TW, j0 = tj * LLB_TW;
    const long r0 = (long)((2 * beta + 1) << m) * C;  // first row of the upper half
    const long r1 = min((long)L, (long)((2 * beta + 2) << m) * C);
    if (r0 >= r1) return;  // no upper half: never read
    const int level = 1 + log2C + m;
    const float *bh = b + (size_t)head * L * Da, *ch = c + (size_t)head * L * Wc;
    const float *lh = lam + (size_t)head * L * nl;
    // each thread: 16 elements of the tile, rows ib + 16 u and columns jb + 16 w (u, w < 4)
    const int tid = threadIdx.x, ib = tid / 16, jb = tid % 16;
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[u][w] = 0.f;
    for (long t0 = r0; t0 < r1; t0 += LLB_R) {
        const int nr = (int)min((long)LLB_R, r1 - t0);
        for (int e = tid; e < LLB_R * LLB_TW; e += LLB_THREADS) {
            const int r = e / LLB_TW, x = e % LLB_TW;
            const long t = t0 + r;
            const bool in = r < nr;
            sb[r][x] = (in && i0 + x < Da) ? bh[t * Da + i0 + x] : 0.f;
            sc[r][x] = (in && j0 + x < Wc) ? ch[t * Wc + j0 + x] * lh[t * nl + level] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < LLB_R; ++r) {
            float bv[4], cv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) bv[u] = sb[r][ib + 16 * u];
#pragma unroll
            for (int w = 0; w < 4; ++w) cv[w] = sc[r][jb + 16 * w];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(bv[u], cv[w], acc[u][w]);
        }
        __syncthreads();
    }
    // W layout per head: [state index][Da][Wc]; state index = blockIdx.y
    float *Wh = W + (size_t)head * w_stride + (size_t)blockIdx.y * Da * Wc;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int i = i0 + ib + 16 * u, j = j0 + jb + 16 * w;
            if (i < Da && j < Wc) Wh[(size_t)i * Wc + j] = acc[u][w];
        }
}

// out rows of one chunk, 32-column slice: the blocks above the chunk, then the pairs inside it
__global__ void __launch_bounds__(LLB_THREADS) llb_rows_kernel(const float *a, const float *b, const float *c,
                                                                const float *lam, const float *W, float *out,
                                                                int L, int C, int log2C, int Da, int Wc,
                                                                int nl, size_t w_stride)
{
    extern __shared__ float smf[];
    float *sa = smf;                        // [R][Da]
    float *sb = sa + LLB_R * Da;            // [R][Da]
    float *sc = sb + LLB_R * Da;            // [R][WC]
    float *sP = sc + LLB_R * LLB_WC;        // [R][R]
    float *sW = sP + LLB_R * LLB_R;         // [64][WC]
    const int head = blockIdx.x, cs = blockIdx.y, j0 = blockIdx.z * LLB_WC;
    const int tid = threadIdx.x, r = tid / LLB_WC, j = tid % LLB_WC;  // rows r and r + 8
    const int nch = (L + C - 1) / C, levels = llb_levels(nch);
    const long c0 = (long)cs * C, c1 = min((long)L, c0 + C);
    const float *ah = a + (size_t)head * L * Da, *bh = b + (size_t)head * L * Da;
    const float *ch = c + (size_t)head * L * Wc, *lh = lam + (size_t)head * L * nl;
    const float *Wh = W + (size_t)head * w_stride;
    float *oh = out + (size_t)head * L * Wc;
    for (long s0 = c0; s0 < c1; s0 += LLB_R) {
        const int ns = (int)min((long)LLB_R, c1 - s0);
        for (int e = tid; e < LLB_R * Da; e += LLB_THREADS) {
            const int rr = e / Da, i = e % Da;
            sa[e] = rr < ns ? ah[(s0 + rr) * Da + i] : 0.f;
        }
        float acc0 = 0.f, acc1 = 0.f;
        // ---- blocks above the chunk: a_s . W_m(cs >> (m+1)) for every 0 bit m of cs
        int ybase = 0;
        for (int m = 0; m < levels; ++m) {
            const int beta = cs >> (m + 1);
            if (!((cs >> m) & 1) && ((2 * beta + 1) << m) < nch) {
                const float *Wp = Wh + (size_t)(ybase + beta) * Da * Wc;
                for (int i0 = 0; i0 < Da; i0 += 64) {
                    __syncthreads();
                    for (int e = tid; e < 64 * LLB_WC; e += LLB_THREADS) {
                        const int ii = e / LLB_WC, jj = e % LLB_WC;
                        sW[e] = (i0 + ii < Da && j0 + jj < Wc) ? Wp[(size_t)(i0 + ii) * Wc + j0 + jj] : 0.f;
                    }
                    __syncthreads();
                    const int ni = min(64, Da - i0);
                    for (int ii = 0; ii < ni; ++ii) {
                        const float w = sW[ii * LLB_WC + j];
                        acc0 = fmaf(sa[r * Da + i0 + ii], w, acc0);
                        acc1 = fmaf(sa[(r + 8) * Da + i0 + ii], w, acc1);
                    }
                }
            }
            ybase += llb_blocks(nch, m);
        }
        // ---- pairs inside the chunk: rows t >= s, weight lambda_t^(l(t,s))
        for (long t0 = s0; t0 < c1; t0 += LLB_R) {
            const int nt = (int)min((long)LLB_R, c1 - t0);
            __syncthreads();
            for (int e = tid; e < LLB_R * Da; e += LLB_THREADS) {
                const int u = e / Da, i = e % Da;
                sb[e] = u < nt ? bh[(t0 + u) * Da + i] : 0.f;
            }
            for (int e = tid; e < LLB_R * LLB_WC; e += LLB_THREADS) {
                const int u = e / LLB_WC, jj = e % LLB_WC;
                sc[e] = (u < nt && j0 + jj < Wc) ? ch[(t0 + u) * Wc + j0 + jj] : 0.f;
            }
            __syncthreads();
            {
                const int rr = tid / LLB_R, u = tid % LLB_R;  // 256 = 16 x 16 pairs
                const long s = s0 + rr, t = t0 + u;
                float sc_ = 0.f;
                if (rr < ns && u < nt && t >= s) {
                    for (int i = 0; i < Da; ++i) sc_ = fmaf(sa[rr * Da + i], sb[u * Da + i], sc_);
                    sc_ *= lh[t * nl + fenwick_level(t, s)];
                }
                sP[rr * LLB_R + u] = sc_;
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < LLB_R; ++u) {
                const float cv = sc[u * LLB_WC + j];
                acc0 = fmaf(sP[r * LLB_R + u], cv, acc0);
                acc1 = fmaf(sP[(r + 8) * LLB_R + u], cv, acc1);
            }
        }
        if (j0 + j < Wc) {
            if (r < ns) oh[(s0 + r) * Wc + j0 + j] = acc0;
            if (r + 8 < ns) oh[(s0 + r + 8) * Wc + j0 + j] = acc1;
        }
        __syncthreads();
    }
}

}  // namespace

// fp32 elements of the block states for heads of L rows (chunks of C rows), per head
size_t ll_anti_state_floats(int L, int C, int Da, int Wc)
{
    const int nch = (L + C - 1) / C;
    size_t n = 0;
    for (int m = 0; m < llb_levels(nch); ++m) n += (size_t)llb_blocks(nch, m);
    return n * (size_t)Da * Wc;
}

// out_s = sum_{t >= s} lambda_t^(l(t,s)) (a_s . b_t) c_t for BH heads of L fp32 rows: a, b
// [BH][L][Da], c and out [BH][L][Wc], lam [BH][L][nl]; W: ll_anti_state_floats(L, C, Da, Wc)
// floats per head.  C: a power of two; nl must cover the levels of L rows.
int ll_anti_pass(int BH, int L, int C, const float *a, const float *b, const float *c,
                 const float *lam, int nl, float *out, int Da, int Wc, float *W, cudaStream_t st)
{
    if (C <= 0 || (C & (C - 1)) || Da > 520 || Wc <= 0) return LA_ERR_UNSUPPORTED;
    const int log2C = ilog2(C);
    const int nch = (L + C - 1) / C;
    const size_t w_stride = ll_anti_state_floats(L, C, Da, Wc);
    int nstates = 0;
    for (int m = 0; m < llb_levels(nch); ++m) nstates += llb_blocks(nch, m);
    if (nstates > 0) {
        const int tiles = ((Da + LLB_TW - 1) / LLB_TW) * ((Wc + LLB_TW - 1) / LLB_TW);
        llb_states_kernel<<<dim3(BH, nstates, tiles), LLB_THREADS, 0, st>>>(b, c, lam, W, L, C, log2C, Da, Wc,
                                                                           nl, w_stride);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    const size_t smem = sizeof(float) * ((size_t)2 * LLB_R * Da + LLB_R * LLB_WC + LLB_R * LLB_R + 64 * LLB_WC);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(llb_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LA_ERR_CUDA;
    llb_rows_kernel<<<dim3(BH, nch, (Wc + LLB_WC - 1) / LLB_WC), LLB_THREADS, smem, st>>>(
        a, b, c, lam, W, out, L, C, log2C, Da, Wc, nl, w_stride);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace la
