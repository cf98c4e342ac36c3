// bwd.cu -- backward pass of causal linear attention (generic fp32 path).
//
// The pages give no backward formulas; they follow from the chain rule on the causal
// definition out_t = sum_{s<=t} M_ts a_ts v_s (/ den_t), a_ts = phi(q_t).phi(k_s), M = 1 or
// gamma^(t-s) ("Linear Attention / Performerの理論と実装": normalised output y_t and the
// Retention decay).  With G_ts = M_ts (dout_t . v_s) unnormalised, or
// M_ts (dout_t . v_s - dout_t . out_t) / den_t normalised:
//   dphi(q)_t = sum_{s<=t} G_ts phi(k_s)                     causal pass
//   dphi(k)_s = sum_{t>=s} G_ts phi(q_t)                     anti-causal pass
//   dv_s      = sum_{t>=s} M_ts a_ts dout_t (/ den_t)        anti-causal pass
// Each is a linear-attention pass with the roles swapped.  Writing D_t = dout_t (/ den_t),
// g_t = D_t . out_t (normalised) and the widened rows D'_t = [D_t, -g_t], v'_s = [v_s, 1],
// G_ts = M_ts D'_t . v'_s, so:
//   dphi(q) = causal(q = D', k = v', v = phi(k)),   dphi(k) = anticausal(q = v', k = D', v = phi(q)),
//   dv = anticausal(q = phi(k), k = phi(q), v = D)
// with identity features and no normaliser, on the generic chunked kernel in fp32 (the
// anti-causal pass is its sweep over the reversed sequence).  den_t itself is one more
// causal pass, causal(q = phi(q), k = phi(k), v = 1).  Finally dq = dphi(q) through the
// feature map's derivative (elu+1: 1 or e^x; FAVOR+: s sum_l dphi_l phi_l (omega_l - s x)),
// likewise dk, and the gradients are stored in the input dtype.
//
// Workspace (fp32, per (b, h) head, rows of L): phi(q), phi(k) [D]; den [1]; ones [1];
// D' [w = dv + normalise]; v' [w]; D [dv]; dphi(q), dphi(k) [D]; dv [dv].
#include <math.h>
#include <stdio.h>

#include "common.cuh"

namespace la {

int simt_launch(const Problem &p, int n_inter, int log2C);

namespace {

constexpr int BW_THREADS = 256;

struct BwdBufs {
    float *fq, *fk, *den, *ones, *dw, *vw, *dn, *dfq, *dfk, *dvf;
};

size_t bwd_floats(long rows, int D, int dv, int normalize, float *base, BwdBufs *b)
{
    const int w = dv + (normalize ? 1 : 0);
    size_t off = 0;
    auto take = [&](float **ptr, size_t n) {
        if (b) *ptr = base + off;
        off += (n + 63) / 64 * 64;  // 256-byte aligned pieces
    };
    BwdBufs dummy;
    BwdBufs *t = b ? b : &dummy;
    take(&t->fq, (size_t)rows * D);
    take(&t->fk, (size_t)rows * D);
    take(&t->den, normalize ? (size_t)rows : 0);
    take(&t->ones, normalize ? (size_t)rows : 0);
    take(&t->dw, (size_t)rows * w);
    take(&t->vw, (size_t)rows * w);
    take(&t->dn, (size_t)rows * dv);
    take(&t->dfq, (size_t)rows * D);
    take(&t->dfk, (size_t)rows * D);
    take(&t->dvf, (size_t)rows * dv);
    return off;
}

// phi of every row of x [rows, dk] (storage T) into f [rows, D] fp32
template <typename T>
__global__ void __launch_bounds__(BW_THREADS) bw_phi_kernel(const T *x, float *f, long rows, int dk, int D,
                                                          int fm, const float *omega, int m)
{
    const long r = blockIdx.x;
    if (r >= rows) return;
    const T *xr = x + r * dk;
    float *fr = f + r * D;
    if (fm != LA_FM_FAVOR) {
        for (int i = threadIdx.x; i < dk; i += BW_THREADS) {
            const float v = to_f32(xr[i]);
            fr[i] = fm == LA_FM_ELU1 ? phi_elu1(v) : v;
        }
        return;
    }
    __shared__ float xs[512];
    __shared__ float red[BW_THREADS / 32];
    const float s = rsqrtf(sqrtf((float)dk));
    float n2 = 0.f;
    for (int i = threadIdx.x; i < dk; i += BW_THREADS) {
        const float v = to_f32(xr[i]) * s;
        xs[i] = v;
        n2 += v * v;
    }
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = n2;
    __syncthreads();
    float nrm2 = 0.f;
    for (int wi = 0; wi < BW_THREADS / 32; ++wi) nrm2 += red[wi];
    const float inv = rsqrtf((float)m);
    for (int l = threadIdx.x; l < m; l += BW_THREADS) {
        const float *w = omega + (size_t)l * dk;
        float acc = 0.f;
        for (int i = 0; i < dk; ++i) acc = fmaf(__ldg(w + i), xs[i], acc);
        fr[l] = expf(acc - 0.5f * nrm2) * inv;
    }
}

// per row: D = dout (/ den), D' = [D, -D . out], v' = [v, 1] (normalised) or D' = D, v' = v
template <typename T>
__global__ void __launch_bounds__(BW_THREADS) bw_prep_kernel(const T *dout, const T *out, const T *v,
                                                           const float *den, float *dn, float *dw,
                                                           float *vw, long rows, int dv, int normalize)
{
    const long r = blockIdx.x;
    if (r >= rows) return;
    const int w = dv + (normalize ? 1 : 0);
    const float inv = normalize ? 1.f / den[r] : 1.f;
    __shared__ float red[BW_THREADS / 32];
    float g = 0.f;
    for (int j = threadIdx.x; j < dv; j += BW_THREADS) {
        const float d = to_f32(dout[r * dv + j]) * inv;
        dn[r * dv + j] = d;
        dw[r * w + j] = d;
        vw[r * w + j] = to_f32(v[r * dv + j]);
        if (normalize) g = fmaf(d, to_f32(out[r * dv + j]), g);
    }
    if (!normalize) return;
    for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = g;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int wi = 0; wi < BW_THREADS / 32; ++wi) t += red[wi];
        dw[r * w + dv] = -t;
        vw[r * w + dv] = 1.f;
    }
}

__global__ void bw_fill_kernel(float *x, long n, float v)
{
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) x[i] = v;
}

// dx = dphi through the feature map, stored as T.  x [rows, dk] raw input, df [rows, D].
template <typename T>
__global__ void __launch_bounds__(BW_THREADS) bw_chain_kernel(const T *x, const float *df, T *dx, long rows,
                                                            int dk, int D, int fm, const float *omega,
                                                            int m)
{
    const long r = blockIdx.x;
    if (r >= rows) return;
    const T *xr = x + r * dk;
    const float *dr = df + r * D;
    if (fm != LA_FM_FAVOR) {
        for (int i = threadIdx.x; i < dk; i += BW_THREADS) {
            const float xv = to_f32(xr[i]);
            const float d = fm == LA_FM_ELU1 && xv < 0.f ? dr[i] * expf(xv) : dr[i];
            dx[r * dk + i] = from_f32<T>(d);
        }
        return;
    }
    // FAVOR+: u_l = dphi_l phi_l (recomputed); dx_i = s (sum_l u_l omega_li - xs_i sum_l u_l)
    __shared__ float xs[512];
    __shared__ float u[512];
    __shared__ float red[BW_THREADS / 32];
    const float s = rsqrtf(sqrtf((float)dk));
    float n2 = 0.f;
    for (int i = threadIdx.x; i < dk; i += BW_THREADS) {
        const float v = to_f32(xr[i]) * s;
        xs[i] = v;
        n2 += v * v;
    }
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = n2;
    __syncthreads();
    float nrm2 = 0.f;
    for (int wi = 0; wi < BW_THREADS / 32; ++wi) nrm2 += red[wi];
    __syncthreads();
    const float inv = rsqrtf((float)m);
    float usum = 0.f;
    for (int l = threadIdx.x; l < m; l += BW_THREADS) {
        const float *w = omega + (size_t)l * dk;
        float acc = 0.f;
        for (int i = 0; i < dk; ++i) acc = fmaf(__ldg(w + i), xs[i], acc);
        const float ul = dr[l] * expf(acc - 0.5f * nrm2) * inv;
        u[l] = ul;
        usum += ul;
    }
    for (int o = 16; o > 0; o >>= 1) usum += __shfl_xor_sync(0xffffffffu, usum, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = usum;
    __syncthreads();
    float tot = 0.f;
    for (int wi = 0; wi < BW_THREADS / 32; ++wi) tot += red[wi];
    for (int i = threadIdx.x; i < dk; i += BW_THREADS) {
        float acc = 0.f;
        for (int l = 0; l < m; ++l) acc = fmaf(u[l], __ldg(omega + (size_t)l * dk + i), acc);
        dx[r * dk + i] = from_f32<T>(s * (acc - xs[i] * tot));
    }
}

template <typename T>
__global__ void bw_cast_kernel(const float *x, T *y, long n)
{
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
        y[i] = from_f32<T>(x[i]);
}

// one identity-feature, unnormalised pass of the generic kernel over fp32 rows
int pass(const Problem &base, const float *q, const float *k, const float *v, float *out, int dk,
         int dv, int rev)
{
    Problem p = base;
    p.q = q; p.k = k; p.v = v; p.out = out;
    p.dk = dk; p.dv = dv; p.D = dk;
    p.fm = LA_FM_IDENTITY; p.m = 0; p.omega = nullptr;
    p.normalize = 0;
    p.lam = nullptr; p.nl = 0;
    p.dtype = LA_F32;
    p.rev = rev;
    p.workspace = nullptr; p.workspace_bytes = 0;
    return simt_launch(p, 0, 0);
}

template <typename T>
int bwd_t(const Problem &p, const void *out, const void *dout, void *dq, void *dk_, void *dv_)
{
    const long rows = (long)p.B * p.H * p.L;
    const int D = p.D, w = p.dv + (p.normalize ? 1 : 0);
    BwdBufs b;
    bwd_floats(rows, D, p.dv, p.normalize, (float *)p.workspace, &b);
    cudaStream_t st = p.stream;
    const unsigned grid = (unsigned)rows;
    bw_phi_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)p.q, b.fq, rows, p.dk, D, p.fm, p.omega, p.m);
    bw_phi_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)p.k, b.fk, rows, p.dk, D, p.fm, p.omega, p.m);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    int rc;
    if (p.normalize) {
        bw_fill_kernel<<<1024, 256, 0, st>>>(b.ones, rows, 1.f);
        if ((rc = pass(p, b.fq, b.fk, b.ones, b.den, D, 1, 0)) != LA_OK) return rc;
    }
    bw_prep_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)dout, (const T *)out, (const T *)p.v, b.den,
                                                 b.dn, b.dw, b.vw, rows, p.dv, p.normalize);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    if ((rc = pass(p, b.dw, b.vw, b.fk, b.dfq, w, D, 0)) != LA_OK) return rc;   // dphi(q)
    if ((rc = pass(p, b.vw, b.dw, b.fq, b.dfk, w, D, 1)) != LA_OK) return rc;   // dphi(k)
    if ((rc = pass(p, b.fk, b.fq, b.dn, b.dvf, D, p.dv, 1)) != LA_OK) return rc;  // dv
    bw_chain_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)p.q, b.dfq, (T *)dq, rows, p.dk, D, p.fm,
                                                  p.omega, p.m);
    bw_chain_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)p.k, b.dfk, (T *)dk_, rows, p.dk, D, p.fm,
                                                  p.omega, p.m);
    bw_cast_kernel<T><<<1024, 256, 0, st>>>(b.dvf, (T *)dv_, rows * p.dv);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace

size_t bwd_workspace_bytes(const Problem &p)
{
    return bwd_floats((long)p.B * p.H * p.L, p.D, p.dv, p.normalize, nullptr, nullptr) * sizeof(float);
}

// D, dk <= 512 and dv < 512 (the generic kernel's shared-memory rows); no level weights
bool bwd_supported(const Problem &p) { return p.D <= 512 && p.dk <= 512 && p.dv < 512 && !p.lam; }

int bwd_launch(const Problem &p, const void *out, const void *dout, void *dq, void *dk, void *dv)
{
    if (!bwd_supported(p)) return LA_ERR_UNSUPPORTED;
    if (!p.workspace || p.workspace_bytes < bwd_workspace_bytes(p)) return LA_ERR_WORKSPACE;
    if (p.dtype == LA_BF16) return bwd_t<__nv_bfloat16>(p, out, dout, dq, dk, dv);
    return bwd_t<float>(p, out, dout, dq, dk, dv);
}

}  // namespace la
