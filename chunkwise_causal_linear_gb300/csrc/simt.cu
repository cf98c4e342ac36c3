// simt.cu -- generic chunkwise causal linear attention on the CUDA cores (fp32).
//
// One CTA per ((b,h) head, slice of WV value columns).  The CTA walks the chunks of its
// head in order, as "attention と線形の間" section 2 (Chunked) describes: for every chunk,
// each output row reads the carried state for the part of the past before the chunk
// (inter) and the causally masked scores for the part inside the chunk (intra, diagonal
// kept); then the chunk's phi(K)^T V is added to the state.  The normaliser rides along
// ("Linear Attention / Performerの理論と実装", normalised output y_t): z = sum phi(k)
// carried the same way, masked score row sums inside the chunk.
//
// Log-linear mask ("論文紹介：Log Linear Attention", slides 34-35): with C = 2^c, a pair
// (t, s) in the same chunk has level 1 + floor(log2(t ^ s)) <= c and is weighted inside
// the chunk; a pair in chunks c_t != c_s has level 1 + c + floor(log2(c_t ^ c_s)), so the
// past chunks group into dyadic blocks of chunks, one per level.  The CTA keeps one
// state per inter-chunk level and updates them after each chunk with the Fenwick rule at
// chunk granularity (slide 22): with r = trailing zeros of (chunk + 1), level r receives
// the chunk plus every lower level, and the lower levels are emptied.  These level
// states live in the caller's workspace (global memory).
//
// Decay (the Retention update S_t = gamma S_{t-1} + phi(k_t) v_t^T of "Linear Attention /
// Performerの理論と実装", z decaying alike): with i, j rows of the chunk, the inter part is
// weighted by gamma^(i+1), the in-chunk scores by gamma^(i-j), and the chunk joins the
// state as S <- gamma^len S + sum_j gamma^(len-1-j) phi(k_j) v_j^T.  Powers are exp2 of
// log2(gamma) times the integer exponent.
//
// Anti-causal (used by the backward pass): every row index t of q, k, v and out is read as
// L-1-t, so the causal sweep over the reversed sequence gives row t the rows s >= t.
//
// Every product accumulates in fp32 in a fixed order; on small-integer inputs whose
// partial sums stay below 2^24 the result is exact.  Rows are handled in tiles of R, so
// any chunk size C >= 1 works (tiles never straddle a chunk boundary).
#include "common.cuh"

namespace la {

constexpr int SIMT_R = 16;    // rows per tile
constexpr int SIMT_WV = 32;   // value columns per CTA
constexpr int SIMT_NT = 256;  // threads per CTA

struct SimtArgs {
    Problem p;
    int n_slices;
    int log2C;                // log-linear only
    int n_inter;              // log-linear: inter-chunk levels kept in the workspace
    float *levels;            // log-linear: [heads][slices][n_inter][D*WV + D]
};

size_t simt_smem_bytes(int D, int dk, int fm)
{
    const int R = SIMT_R, WV = SIMT_WV;
    size_t f = (size_t)2 * R * D + R * WV + (size_t)D * WV + D + R * R + R * WV + R;
    if (fm == LA_FM_FAVOR) f += (size_t)R * dk + R;
    return f * sizeof(float);
}

int simt_inter_levels(int L, int C)
{
    int nch = (L + C - 1) / C;
    if (nch <= 1) return 0;
    return 1 + ilog2(nch - 1);
}

size_t simt_workspace_bytes(int B, int H, int L, int D, int dv, int C, bool loglinear)
{
    if (!loglinear) return 0;
    int ni = simt_inter_levels(L, C);
    if (ni == 0) return 0;
    int ns = (dv + SIMT_WV - 1) / SIMT_WV;
    return (size_t)B * H * ns * ni * ((size_t)D * SIMT_WV + D) * sizeof(float);
}

// storage row of sweep position t (reversed for the anti-causal pass)
__device__ __forceinline__ int srow(const Problem &p, int t) { return p.rev ? p.L - 1 - t : t; }

// phi of rows [row0, row0 + n) of x ([L, dk], storage T) into dst [R][D] (fp32);
// rows >= n are zero.  Ends with __syncthreads().
template <typename T>
__device__ void load_phi_rows(const T *x, int row0, int n, const SimtArgs &a, float *dst,
                              float *sX, float *sNrm)
{
    const Problem &p = a.p;
    const int D = p.D, dk = p.dk, tid = threadIdx.x;
    if (p.fm != LA_FM_FAVOR) {
        for (int e = tid; e < SIMT_R * D; e += SIMT_NT) {
            int r = e / D, i = e - r * D;
            float val = 0.f;
            if (r < n) {
                val = to_f32(x[(long)srow(p, row0 + r) * dk + i]);
                if (p.fm == LA_FM_ELU1) val = phi_elu1(val);
            }
            dst[e] = val;
        }
        __syncthreads();
        return;
    }
    // FAVOR+: x^ = x dk^{-1/4}; phi_l = exp(omega_l . x^ - |x^|^2 / 2) / sqrt(m)
    const float s = rsqrtf(sqrtf((float)dk));
    for (int e = tid; e < SIMT_R * dk; e += SIMT_NT) {
        int r = e / dk, j = e - r * dk;
        sX[e] = (r < n) ? to_f32(x[(long)srow(p, row0 + r) * dk + j]) * s : 0.f;
    }
    __syncthreads();
    for (int r = tid; r < SIMT_R; r += SIMT_NT) {
        float acc = 0.f;
        for (int j = 0; j < dk; ++j) acc += sX[r * dk + j] * sX[r * dk + j];
        sNrm[r] = acc;
    }
    __syncthreads();
    const float inv_sqrt_m = rsqrtf((float)p.m);
    for (int e = tid; e < SIMT_R * D; e += SIMT_NT) {
        int r = e / D, l = e - r * D;
        float val = 0.f;
        if (r < n) {
            const float *w = p.omega + (long)l * dk;
            float acc = 0.f;
            for (int j = 0; j < dk; ++j) acc += __ldg(w + j) * sX[r * dk + j];
            val = expf(acc - 0.5f * sNrm[r]) * inv_sqrt_m;
        }
        dst[e] = val;
    }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(SIMT_NT) simt_chunked_kernel(SimtArgs a)
{
    extern __shared__ float smem[];
    const Problem &p = a.p;
    const int R = SIMT_R, WV = SIMT_WV, NT = SIMT_NT;
    const int D = p.D, dk = p.dk, dv = p.dv, L = p.L, C = p.C, tid = threadIdx.x;
    const bool ll = p.lam != nullptr;

    float *sQ = smem;               // [R][D]
    float *sK = sQ + R * D;         // [R][D]
    float *sV = sK + R * D;         // [R][WV]
    float *sS = sV + R * WV;        // [D][WV]
    float *sz = sS + D * WV;        // [D]
    float *sP = sz + D;             // [R][R]
    float *sAcc = sP + R * R;       // [R][WV]
    float *sDen = sAcc + R * WV;    // [R]
    float *sX = sDen + R;           // [R][dk]  (FAVOR+)
    float *sNrm = sX + R * dk;      // [R]      (FAVOR+)

    const int head = blockIdx.x;
    const int j0 = blockIdx.y * WV;
    const int wv = min(WV, dv - j0);
    const T *q = (const T *)p.q + (long)head * L * dk;
    const T *k = (const T *)p.k + (long)head * L * dk;
    const T *v = (const T *)p.v + (long)head * L * dv;
    T *out = (T *)p.out + (long)head * L * dv;
    const float *lam = ll ? p.lam + (long)head * L * p.nl : nullptr;
    const size_t lvl_stride = (size_t)D * WV + D;
    float *Lv = (ll && a.n_inter > 0)
                    ? a.levels + ((size_t)head * a.n_slices + blockIdx.y) * a.n_inter * lvl_stride
                    : nullptr;

    // the state before row 0: zero, or the given one (columns j0 .. j0 + WV of S0)
    for (int e = tid; e < D * WV; e += NT) {
        const int i = e / WV, j = e - i * WV;
        sS[e] = (p.S0 && j < wv) ? p.S0[((size_t)head * D + i) * dv + j0 + j] : 0.f;
    }
    for (int i = tid; i < D; i += NT) sz[i] = p.z0 ? p.z0[(size_t)head * D + i] : 0.f;
    if (Lv)
        for (size_t e = tid; e < (size_t)a.n_inter * lvl_stride; e += NT) Lv[e] = 0.f;
    __syncthreads();

    const int nch = (L + C - 1) / C;
    for (int cc = 0; cc < nch; ++cc) {
        const int c0 = cc * C, cl = min(C, L - c0);
        for (int qt = 0; qt < cl; qt += R) {
            const int nq = min(R, cl - qt);
            load_phi_rows<T>(q, c0 + qt, nq, a, sQ, sX, sNrm);
            // ---- inter: the part of the past before this chunk, from the state(s)
            for (int e = tid; e < R * WV; e += NT) {
                const int r = e / WV, j = e - r * WV;
                float acc = 0.f;
                if (r < nq && j < wv) {
                    if (!ll) {
                        for (int i = 0; i < D; ++i) acc += sQ[r * D + i] * sS[i * WV + j];
                    } else {
                        const int t = c0 + qt + r;
                        for (int jl = 0; jl < a.n_inter; ++jl) {
                            const float *Sl = Lv + jl * lvl_stride;
                            float part = 0.f;
                            for (int i = 0; i < D; ++i) part += sQ[r * D + i] * Sl[i * WV + j];
                            acc += lam[(long)t * p.nl + 1 + a.log2C + jl] * part;
                        }
                    }
                }
                if (p.decay) acc *= exp2f(p.l2g * (float)(qt + r + 1));
                sAcc[e] = acc;
            }
            for (int r = tid; r < R; r += NT) {
                float den = 0.f;
                if (p.normalize && r < nq) {
                    if (!ll) {
                        for (int i = 0; i < D; ++i) den += sQ[r * D + i] * sz[i];
                    } else {
                        const int t = c0 + qt + r;
                        for (int jl = 0; jl < a.n_inter; ++jl) {
                            const float *zl = Lv + jl * lvl_stride + (size_t)D * WV;
                            float part = 0.f;
                            for (int i = 0; i < D; ++i) part += sQ[r * D + i] * zl[i];
                            den += lam[(long)t * p.nl + 1 + a.log2C + jl] * part;
                        }
                    }
                    if (p.decay) den *= exp2f(p.l2g * (float)(qt + r + 1));
                }
                sDen[r] = den;
            }
            __syncthreads();
            // ---- intra: masked scores inside the chunk, key tiles up to the query tile
            for (int kt = 0; kt <= qt; kt += R) {
                const int nk = min(R, cl - kt);
                load_phi_rows<T>(k, c0 + kt, nk, a, sK, sX, sNrm);
                for (int e = tid; e < R * WV; e += NT) {
                    const int s = e / WV, j = e - s * WV;
                    sV[e] = (s < nk && j < wv) ? to_f32(v[(long)srow(p, c0 + kt + s) * dv + j0 + j]) : 0.f;
                }
                for (int e = tid; e < R * R; e += NT) {
                    const int r = e / R, s = e - r * R;
                    const int t = qt + r, u = kt + s;  // chunk-relative rows
                    float sc = 0.f;
                    if (r < nq && s < nk && u <= t) {
                        for (int i = 0; i < D; ++i) sc += sQ[r * D + i] * sK[s * D + i];
                        if (ll) sc *= lam[(long)(c0 + t) * p.nl + fenwick_level(c0 + t, c0 + u)];
                        if (p.decay) sc *= exp2f(p.l2g * (float)(t - u));
                    }
                    sP[e] = sc;
                }
                __syncthreads();
                for (int e = tid; e < R * WV; e += NT) {
                    const int r = e / WV, j = e - r * WV;
                    float acc = sAcc[e];
                    for (int s = 0; s < R; ++s) acc += sP[r * R + s] * sV[s * WV + j];
                    sAcc[e] = acc;
                }
                if (p.normalize)
                    for (int r = tid; r < R; r += NT) {
                        float den = sDen[r];
                        for (int s = 0; s < R; ++s) den += sP[r * R + s];
                        sDen[r] = den;
                    }
                __syncthreads();
            }
            for (int e = tid; e < R * WV; e += NT) {
                const int r = e / WV, j = e - r * WV;
                if (r < nq && j < wv) {
                    float val = sAcc[e];
                    if (p.normalize) val = val / sDen[r];
                    out[(long)srow(p, c0 + qt + r) * dv + j0 + j] = from_f32<T>(val);
                }
            }
            __syncthreads();
        }
        if (cc + 1 == nch) break;
        // ---- carry the chunk into the state
        float *tS = sS, *tz = sz;
        if (ll) {
            // Fenwick update at chunk granularity: level r gets the lower levels, which
            // empty; the chunk's own phi(K)^T V is added to level r below.
            const int r = __ffs(cc + 1) - 1;
            tS = Lv + r * lvl_stride;
            tz = tS + (size_t)D * WV;
            for (size_t e = tid; e < lvl_stride; e += NT) {
                float acc = 0.f;
                for (int jl = 0; jl < r; ++jl) {
                    acc += Lv[jl * lvl_stride + e];
                    Lv[jl * lvl_stride + e] = 0.f;
                }
                tS[e] = acc;
            }
            __syncthreads();
        }
        // decay: the state so far fades by gamma^cl over the chunk (each thread scales the
        // elements it updates below, before their first update)
        const float gl = p.decay ? exp2f(p.l2g * (float)cl) : 1.f;
        for (int kt = 0; kt < cl; kt += R) {
            const int nk = min(R, cl - kt);
            load_phi_rows<T>(k, c0 + kt, nk, a, sK, sX, sNrm);
            for (int e = tid; e < R * WV; e += NT) {
                const int s = e / WV, j = e - s * WV;
                sV[e] = (s < nk && j < wv) ? to_f32(v[(long)srow(p, c0 + kt + s) * dv + j0 + j]) : 0.f;
            }
            if (p.decay) {
                // key row kt + s of the chunk weighted by gamma^(cl - 1 - kt - s)
                for (int e = tid; e < nk * D; e += NT) sK[e] *= exp2f(p.l2g * (float)(cl - 1 - kt - e / D));
            }
            __syncthreads();
            for (int e = tid; e < D * WV; e += NT) {
                const int i = e / WV, j = e - i * WV;
                float acc = 0.f;
                for (int s = 0; s < nk; ++s) acc += sK[s * D + i] * sV[s * WV + j];
                tS[e] = (kt == 0 ? gl * tS[e] : tS[e]) + acc;
            }
            if (p.normalize)
                for (int i = tid; i < D; i += NT) {
                    float acc = 0.f;
                    for (int s = 0; s < nk; ++s) acc += sK[s * D + i];
                    tz[i] = (kt == 0 ? gl * tz[i] : tz[i]) + acc;
                }
            __syncthreads();
        }
    }
}

// Host launcher.  Returns LA_OK or LA_ERR_CUDA.
int simt_launch(const Problem &p, int n_inter, int log2C)
{
    SimtArgs a;
    a.p = p;
    a.n_slices = (p.dv + SIMT_WV - 1) / SIMT_WV;
    a.log2C = log2C;
    a.n_inter = n_inter;
    a.levels = (float *)p.workspace;
    const size_t smem = simt_smem_bytes(p.D, p.dk, p.fm);
    dim3 grid(p.B * p.H, a.n_slices);
    cudaError_t e;
    if (p.dtype == LA_F32) {
        e = cudaFuncSetAttribute(simt_chunked_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return LA_ERR_CUDA;
        simt_chunked_kernel<float><<<grid, SIMT_NT, smem, p.stream>>>(a);
    } else {
        e = cudaFuncSetAttribute(simt_chunked_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return LA_ERR_CUDA;
        simt_chunked_kernel<__nv_bfloat16><<<grid, SIMT_NT, smem, p.stream>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace la
