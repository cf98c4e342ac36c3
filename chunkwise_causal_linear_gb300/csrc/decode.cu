// decode.cu -- one recurrent decoding step per (b, h) head (sm_103a).
//
// The recurrent form of "Linear Attention / Performerの理論と実装" ("再帰的な状態更新"): with
// the carried state S (d x dv) and normaliser z (d), token t updates
//     S += phi(k_t) v_t^T,   z += phi(k_t),   out_t = phi(q_t)^T S / phi(q_t)^T z
// (the current token included, as in the causal mask).  With log-linear level weights
// ("論文紹介：Log Linear Attention", slides 17-22) the state is one S^(l) per Fenwick level
// l >= 1, the output is
//     out_t = lambda^(0) (q_t.k_t) v_t + sum_{l>=1} lambda^(l) q_t^T S^(l)
// from the states before the update, and then, with r = trailing zeros of t+1, level r+1
// becomes k_t v_t^T + sum_{l<=r} S^(l) and levels 1..r are emptied (the normaliser levels
// z^(l) alike).  With the Retention decay of the first page (S_t = gamma S_{t-1} + phi(k_t)
// v_t^T) the old state and normaliser are scaled by gamma before the token joins them.
//
// A decoding step moves the whole state through the SM once (read and write), so it is
// bandwidth-bound; it runs on the CUDA cores.  Grid: one CTA per head (so z is read and
// rewritten by one CTA); 256 threads = 8 row groups x 32 columns, walking dv in 32-column
// slices; rows i = group, group + 8, ..., so every warp reads and writes one contiguous
// 128-byte row segment of S, and every state element is read and rewritten by one thread.
#include <stdio.h>

#include "common.cuh"

namespace la {

namespace {

constexpr int DEC_THREADS = 256;
constexpr int DEC_COLS = 32;
constexpr int DEC_RG = DEC_THREADS / DEC_COLS;  // row groups

struct DecArgs {
    const void *q, *k, *v;
    void *out;
    float *S;            // plain: [BH][D][dv]; log-linear: [BH][NL-1][D][dv]
    float *z;            // plain: [BH][D];     log-linear: [BH][NL-1][D]; NULL without norm
    int dk, dv, D, fm, m, normalize;
    const float *omega;  // FAVOR+: [m][dk]
    const float *lam;    // log-linear: [BH][NL] for this token, else NULL
    int nl, r;           // log-linear: levels, trailing zeros of t+1
    float gamma;         // decay of the plain state (1: none)
};

template <typename T>
__global__ void __launch_bounds__(DEC_THREADS) decode_kernel(const DecArgs a)
{
    extern __shared__ float dsm[];
    const int D = a.D;
    float *fq = dsm;                 // [D]  phi(q)
    float *fk = fq + D;              // [D]  phi(k)
    float *xq = fk + D;              // [dk] raw q, then k (FAVOR+ scratch)
    float *xk = xq + a.dk;           // [dk]
    float *part = xk + a.dk;         // [DEC_RG][DEC_COLS + 1] column partial sums
    float *dpart = part + DEC_RG * (DEC_COLS + 1);  // [DEC_THREADS] denominator partials
    __shared__ float red[4];
    const int head = blockIdx.x, tid = threadIdx.x;
    const int j = tid % DEC_COLS, rg = tid / DEC_COLS;
    const T *q = (const T *)a.q + (size_t)head * a.dk;
    const T *k = (const T *)a.k + (size_t)head * a.dk;
    const T *v = (const T *)a.v + (size_t)head * a.dv;

    for (int i = tid; i < a.dk; i += DEC_THREADS) {
        xq[i] = to_f32(q[i]);
        xk[i] = to_f32(k[i]);
    }
    __syncthreads();
    if (a.fm == LA_FM_FAVOR) {
        // x^ = x dk^{-1/4}; phi_l = exp(omega_l . x^ - |x^|^2 / 2) / sqrt(m)
        if (tid < 64) {
            float sq = 0.f, sk = 0.f;
            for (int i = tid; i < a.dk; i += 64) {
                sq += xq[i] * xq[i];
                sk += xk[i] * xk[i];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if ((tid & 31) == 0) {
                red[tid >> 5] = sq;
                red[2 + (tid >> 5)] = sk;
            }
        }
        __syncthreads();
        const float s = rsqrtf(sqrtf((float)a.dk));  // dk^{-1/4}
        const float hq = 0.5f * (red[0] + red[1]) * s * s, hk = 0.5f * (red[2] + red[3]) * s * s;
        const float inv = rsqrtf((float)a.m);
        for (int l = tid; l < D; l += DEC_THREADS) {
            const float *w = a.omega + (size_t)l * a.dk;
            float pq = 0.f, pk = 0.f;
            for (int i = 0; i < a.dk; ++i) {
                const float wi = __ldg(w + i);
                pq = fmaf(wi, xq[i], pq);
                pk = fmaf(wi, xk[i], pk);
            }
            fq[l] = expf(pq * s - hq) * inv;
            fk[l] = expf(pk * s - hk) * inv;
        }
    } else {
        for (int i = tid; i < D; i += DEC_THREADS) {
            fq[i] = a.fm == LA_FM_ELU1 ? phi_elu1(xq[i]) : xq[i];
            fk[i] = a.fm == LA_FM_ELU1 ? phi_elu1(xk[i]) : xk[i];
        }
    }
    __syncthreads();
    const size_t sz = (size_t)D * a.dv;
    const int nls = a.nl - 1;  // log-linear: stored levels 1 .. nl-1
    const float *lam = a.lam ? a.lam + (size_t)head * a.nl : nullptr;
    float a0 = 0.f;            // log-linear: lambda^(0) (q.k)
    if (lam) {
        if (tid < 32) {
            float qk = 0.f;
            for (int i = tid; i < D; i += 32) qk = fmaf(fq[i], fk[i], qk);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o);
            if (tid == 0) red[0] = qk;
        }
        __syncthreads();
        a0 = lam[0] * red[0];
    }
    const int r = a.r;
    // ---- denominator, and the normaliser update (each z element by one thread)
    float den = 0.f;
    if (a.normalize) {
        if (!lam) {
            float *z = a.z + (size_t)head * D;
            for (int i = tid; i < D; i += DEC_THREADS) {
                const float zi = a.gamma * z[i] + fk[i];
                z[i] = zi;
                den = fmaf(fq[i], zi, den);
            }
        } else {
            float *z = a.z + (size_t)head * nls * D;
            for (int i = tid; i < D; i += DEC_THREADS) {
                float merged = fk[i], acc = 0.f;
                for (int l = 1; l <= nls; ++l) {
                    float *p = z + (size_t)(l - 1) * D + i;
                    const float zl = *p;
                    acc = fmaf(lam[l], zl, acc);
                    if (l <= r) {
                        merged += zl;
                        *p = 0.f;
                    }
                }
                z[(size_t)r * D + i] = merged;
                den = fmaf(fq[i], acc, den);
            }
            if (tid == 0) den += a0;
        }
    }
    dpart[tid] = den;
    __syncthreads();
    for (int st = DEC_THREADS / 2; st > 0; st >>= 1) {
        if (tid < st) dpart[tid] += dpart[tid + st];
        __syncthreads();
    }
    const float den_all = dpart[0];
    // ---- numerator, 32 columns at a time (each state element by one thread)
    for (int jb = 0; jb < a.dv; jb += DEC_COLS) {
        const int jj = jb + j;
        const bool col = jj < a.dv;
        const float vj = col ? to_f32(v[jj]) : 0.f;
        float num = 0.f;
        if (col) {
            if (!lam) {
                // S += phi(k) v^T, then phi(q) S
                float *S = a.S + (size_t)head * sz;
                for (int i = rg; i < D; i += DEC_RG) {
                    const float sv = a.gamma * S[(size_t)i * a.dv + jj] + fk[i] * vj;
                    S[(size_t)i * a.dv + jj] = sv;
                    num = fmaf(fq[i], sv, num);
                }
            } else {
                // outputs from the levels before the update; then level r+1 = k v^T plus
                // levels 1..r, which are emptied
                float *S = a.S + (size_t)head * nls * sz;
                for (int i = rg; i < D; i += DEC_RG) {
                    float merged = fk[i] * vj, acc = 0.f;
                    for (int l = 1; l <= nls; ++l) {
                        float *p = S + (size_t)(l - 1) * sz + (size_t)i * a.dv + jj;
                        const float sv = *p;
                        acc = fmaf(lam[l], sv, acc);
                        if (l <= r) {
                            merged += sv;
                            *p = 0.f;
                        }
                    }
                    S[(size_t)r * sz + (size_t)i * a.dv + jj] = merged;
                    num = fmaf(fq[i], acc, num);
                }
                if (rg == 0) num = fmaf(a0, vj, num);
            }
        }
        part[rg * (DEC_COLS + 1) + j] = num;
        __syncthreads();
        if (rg == 0 && col) {
            float acc = 0.f;
#pragma unroll
            for (int g = 0; g < DEC_RG; ++g) acc += part[g * (DEC_COLS + 1) + j];
            const float o = a.normalize ? acc / den_all : acc;
            ((T *)a.out)[(size_t)head * a.dv + jj] = from_f32<T>(o);
        }
        __syncthreads();
    }
}

// Plain (no level weights) step with float4 columns: dv % 4 == 0, dv <= 512.  512 threads =
// RG row groups x dv/4 column quads.  The step is a chain of memory latencies, so every
// global read that depends on nothing (the thread's first RGI state rows, q, k, z) is issued
// at the start, and the denominator is reduced with warp shuffles.
constexpr int DV_THREADS = 512;

template <typename T>
__global__ void __launch_bounds__(DV_THREADS) decode_vec_kernel(const DecArgs a)
{
    extern __shared__ float dsm[];
    const int D = a.D, dv = a.dv;
    const int nq = dv / 4;                   // column quads per row
    const int RG = DV_THREADS / nq;          // row groups
    float *fq = dsm;                         // [D]
    float *fk = fq + D;                      // [D]
    float *part = fk + D;                    // [RG][dv] column partial sums
    float *wden = part + RG * dv;            // [DV_THREADS / 32] per-warp denominator sums
    const int head = blockIdx.x, tid = threadIdx.x;
    const int cq = tid % nq, rg = tid / nq;  // column quad, row group
    const bool active = rg < RG;
    constexpr int RGI = 8;                   // rows in flight per thread
    float4 *S = (float4 *)(a.S + (size_t)head * D * dv) + cq;
    float4 sv[RGI];
    if (active)
#pragma unroll
        for (int u = 0; u < RGI; ++u) {
            const int i = rg + u * RG;
            if (i < D) sv[u] = S[(size_t)i * nq];
        }
    const T *q = (const T *)a.q + (size_t)head * a.dk;
    const T *k = (const T *)a.k + (size_t)head * a.dk;
    float *z = a.normalize ? a.z + (size_t)head * D : nullptr;
    // this thread's normaliser entries (i = tid, tid + 512, ...): z and phi(q) kept for den
    float den = 0.f;
    for (int i = tid; i < D; i += DV_THREADS) {
        const float xq = to_f32(q[i]), xk = to_f32(k[i]);
        const float zo = a.normalize ? z[i] : 0.f;
        const float gq = a.fm == LA_FM_ELU1 ? phi_elu1(xq) : xq;
        const float gk = a.fm == LA_FM_ELU1 ? phi_elu1(xk) : xk;
        fq[i] = gq;
        fk[i] = gk;
        if (a.normalize) {
            const float zi = a.gamma * zo + gk;
            z[i] = zi;
            den = fmaf(gq, zi, den);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if ((tid & 31) == 0) wden[tid >> 5] = den;
    __syncthreads();
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) {
        const T *v = (const T *)a.v + (size_t)head * dv + 4 * cq;
        const float v0 = to_f32(v[0]), v1 = to_f32(v[1]), v2 = to_f32(v[2]), v3 = to_f32(v[3]);
        const float gm = a.gamma;
        for (int i0 = rg; i0 < D; i0 += RG * RGI) {
            if (i0 != rg)  // later rounds (D > RG * RGI): load here
#pragma unroll
                for (int u = 0; u < RGI; ++u) {
                    const int i = i0 + u * RG;
                    if (i < D) sv[u] = S[(size_t)i * nq];
                }
#pragma unroll
            for (int u = 0; u < RGI; ++u) {
                const int i = i0 + u * RG;
                if (i < D) {
                    const float f = fk[i], g = fq[i];
                    float4 x = sv[u];
                    x.x = fmaf(f, v0, gm * x.x);
                    x.y = fmaf(f, v1, gm * x.y);
                    x.z = fmaf(f, v2, gm * x.z);
                    x.w = fmaf(f, v3, gm * x.w);
                    S[(size_t)i * nq] = x;
                    num.x = fmaf(g, x.x, num.x);
                    num.y = fmaf(g, x.y, num.y);
                    num.z = fmaf(g, x.z, num.z);
                    num.w = fmaf(g, x.w, num.w);
                }
            }
        }
        *(float4 *)(part + rg * dv + 4 * cq) = num;
    }
    __syncthreads();
    float den_all = 0.f;
    if (a.normalize)
#pragma unroll
        for (int w = 0; w < DV_THREADS / 32; ++w) den_all += wden[w];
    for (int c = tid; c < dv; c += DV_THREADS) {
        float acc = 0.f;
        for (int g = 0; g < RG; ++g) acc += part[g * dv + c];
        const float o = a.normalize ? acc / den_all : acc;
        ((T *)a.out)[(size_t)head * dv + c] = from_f32<T>(o);
    }
}

}  // namespace

int decode_check(int B, int H, int dk, int dv, const la_feature_map *fm, int normalize,
                 int num_levels, long long t, bool loglinear, int *D_out, int *r_out)
{
    if (B <= 0 || H <= 0 || dk <= 0 || dv <= 0) return LA_ERR_SHAPE;
    const int kind = fm ? fm->kind : LA_FM_IDENTITY;
    if (kind != LA_FM_IDENTITY && kind != LA_FM_ELU1 && kind != LA_FM_FAVOR) return LA_ERR_UNSUPPORTED;
    int D = dk;
    if (kind == LA_FM_FAVOR) {
        if (fm->m <= 0) return LA_ERR_SHAPE;
        if (!fm->omega) return LA_ERR_NULL;
        D = fm->m;
    }
    if (D > 4096 || dk > 4096) return LA_ERR_UNSUPPORTED;
    int r = 0;
    if (loglinear) {
        if (t < 0 || num_levels < 2) return LA_ERR_SHAPE;
        unsigned long long x = (unsigned long long)t + 1ull;
        while (!((x >> r) & 1ull)) ++r;
        if (r + 1 >= num_levels) return LA_ERR_SHAPE;  // the levels do not reach position t+1
    }
    *D_out = D;
    *r_out = r;
    return LA_OK;
}

int decode_launch(const void *q, const void *k, const void *v, void *out, float *S, float *z, int B,
                  int H, int dk, int dv, const la_feature_map *fm, int normalize, const float *lam,
                  int num_levels, long long t, int dtype, cudaStream_t stream, float gamma)
{
    int D = 0, r = 0;
    int rc = decode_check(B, H, dk, dv, fm, normalize, num_levels, t, lam != nullptr, &D, &r);
    if (rc != LA_OK) return rc;
    if (dtype != LA_BF16 && dtype != LA_F32) return LA_ERR_UNSUPPORTED;
    DecArgs a;
    a.q = q; a.k = k; a.v = v; a.out = out;
    a.S = S; a.z = z;
    a.dk = dk; a.dv = dv; a.D = D;
    a.fm = fm ? fm->kind : LA_FM_IDENTITY;
    a.m = a.fm == LA_FM_FAVOR ? fm->m : 0;
    a.omega = a.fm == LA_FM_FAVOR ? fm->omega : nullptr;
    a.normalize = normalize ? 1 : 0;
    a.lam = lam;
    a.nl = lam ? num_levels : 0;
    a.r = r;
    a.gamma = gamma;
    if (!lam && a.fm != LA_FM_FAVOR && dv % 4 == 0 && dv <= 512) {
        const int RG = DV_THREADS / (dv / 4);
        const size_t vsm = sizeof(float) * ((size_t)2 * D + (size_t)RG * dv + DV_THREADS / 32);
        if (vsm <= 200 * 1024) {
            dim3 vgrid((unsigned)(B * H));
            if (dtype == LA_BF16) {
                auto kern = decode_vec_kernel<__nv_bfloat16>;
                if (vsm > 48 * 1024 &&
                    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vsm) != cudaSuccess)
                    return LA_ERR_CUDA;
                kern<<<vgrid, DV_THREADS, vsm, stream>>>(a);
            } else {
                auto kern = decode_vec_kernel<float>;
                if (vsm > 48 * 1024 &&
                    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vsm) != cudaSuccess)
                    return LA_ERR_CUDA;
                kern<<<vgrid, DV_THREADS, vsm, stream>>>(a);
            }
            return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
        }
    }
    const size_t smem = sizeof(float) * ((size_t)2 * D + 2 * dk + DEC_RG * (DEC_COLS + 1) + DEC_THREADS);
    if (smem > 200 * 1024) return LA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)(B * H));
    if (dtype == LA_BF16) {
        auto kern = decode_kernel<__nv_bfloat16>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LA_ERR_CUDA;
        kern<<<grid, DEC_THREADS, smem, stream>>>(a);
    } else {
        auto kern = decode_kernel<float>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LA_ERR_CUDA;
        kern<<<grid, DEC_THREADS, smem, stream>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace la
