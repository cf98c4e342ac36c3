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
// anti-causal pass is its sweep over the reversed sequence).  With the normaliser the
// forward output is recomputed in fp32 by one more causal pass, causal(q = phi(q), k =
// phi(k), v = v') = [num, den]: dphi(q) is a small difference of two large sums (g_t Z_t
// against sum_s (D_t . v_s) phi(k_s)), and a bf16-stored output's rounding would come back
// amplified about thirtyfold.  Finally dq = dphi(q) through the
// feature map's derivative (elu+1: 1 or e^x; FAVOR+: s sum_l dphi_l phi_l (omega_l - s x)),
// likewise dk, and the gradients are stored in the input dtype.
//
// Workspace (fp32, per (b, h) head, rows of L): phi(q), phi(k) [D]; [num, den] [w];
// D' [w = dv + normalise]; v' [w]; D [dv]; dphi(q), dphi(k) [D]; dv [dv].
//
// Tensor-core route (bf16, identity / elu+1, plain or decayed): the same passes run on the
// tensor-core forward with identity features, the anti-causal ones in its anti-causal mode
// (the causal pass over the mirrored sequence, read and written in place, so no reversed
// copies are made).  The normaliser's extra column becomes two more passes against constant
// rows e = (1, 0, ..., 0), which the kernel keeps in shared memory instead of reading them:
// Z_t = sum_{s<=t} phi(k_s) (so den_t =
// phi(q_t).Z_t and dphi(q)_t -= g_t Z_t) and the suffix sums sum_{t>=s} g_t phi(q_t)
// (subtracted from dphi(k)_s); the forward output is recomputed by one more pass, num =
// causal(phi(q), phi(k), v), over the same bf16 features, so that out = num / den and the
// other sums cancel exactly for those features.  With the normaliser these passes run in
// the kernel's fp32-output mode (bf16 hi / lo state copy and P, fp32 rows out) and the
// last elementwise kernel forms dq, dk; without it every pass writes its gradient rows in
// place, in bf16.
#include <math.h>
#include <stdint.h>
#include <stdio.h>

#include <type_traits>

#include "common.cuh"

namespace la {

int simt_launch(const Problem &p, int n_inter, int log2C);
int simt_inter_levels(int L, int C);
size_t simt_workspace_bytes(int B, int H, int L, int D, int dv, int C, bool loglinear);
size_t ll_anti_state_floats(int L, int C, int Da, int Wc);
int ll_anti_pass(int BH, int L, int C, const float *a, const float *b, const float *c,
                 const float *lam, int nl, float *out, int Da, int Wc, float *W, cudaStream_t st);
bool tc_supported(const Problem &p, int num_sms);
int tc_plan(const Problem &p, int num_sms, la_plan_info *info);
int tc_launch(const Problem &p, int num_sms);

namespace {

constexpr int BW_THREADS = 256;

struct BwdBufs {
    float *fq, *fk, *nd, *dw, *vw, *dn, *dfq, *dfk, *dvf;
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
    take(&t->nd, normalize ? (size_t)rows * w : 0);
    take(&t->dw, (size_t)rows * w);
    take(&t->vw, (size_t)rows * w);
    take(&t->dn, (size_t)rows * dv);
    take(&t->dfq, (size_t)rows * D);
    take(&t->dfk, (size_t)rows * D);
    take(&t->dvf, (size_t)rows * dv);
    return off;
}

// The log-linear mask's passes use chunks of this many rows (the result does not depend on
// it), a level-state buffer for the causal passes and the block states of the anti-causal
// sums (bwd_ll.cu), placed after the per-row buffers.
constexpr int BW_LL_C = 64;

// level states of the causal passes (bytes, rounded to 256)
size_t bwd_ll_level_bytes(const Problem &p)
{
    const int D = p.D, w = p.dv + (p.normalize ? 1 : 0);
    size_t lv = simt_workspace_bytes(p.B, p.H, p.L, w, D, BW_LL_C, true);        // dphi(q)
    if (p.normalize) {
        const size_t l2 = simt_workspace_bytes(p.B, p.H, p.L, D, w, BW_LL_C, true);  // [num, den]
        lv = lv > l2 ? lv : l2;
    }
    return ((lv + 255) / 256) * 256;
}

// Identity features, no normaliser, bf16 storage: the causal gradient pass dphi(q) =
// sum_{s<=t} M_ts (dout_t . v_s) k_s has bf16 inputs exactly (q' = dout, k' = v, v' = k) and
// is dq itself, so it runs on the tensor-core log-linear forward when that covers the
// shape.  Returns false (and leaves *tp alone) otherwise.
bool bwd_ll_tc_dq(const Problem &p, int sms, Problem *tp)
{
    if (!p.lam || p.dtype != LA_BF16 || p.fm != LA_FM_IDENTITY || p.normalize || p.decay) return false;
    if (((uintptr_t)p.lam & 15) != 0) return false;
    Problem t = p;
    t.dk = p.dv; t.dv = p.dk; t.D = p.dv;
    t.C = 64;
    t.rev = 0; t.out_f32 = 0; t.S0 = nullptr; t.z0 = nullptr;
    if (!tc_supported(t, sms)) return false;
    *tp = t;
    return true;
}

size_t bwd_ll_tc_bytes(const Problem &p, int sms)
{
    Problem t;
    if (!bwd_ll_tc_dq(p, sms, &t)) return 0;
    la_plan_info info;
    if (tc_plan(t, sms, &info) != LA_OK) return 0;
    return ((info.workspace_bytes + 255) / 256) * 256;
}

size_t bwd_ll_extra_bytes(const Problem &p)
{
    if (!p.lam) return 0;
    const int w = p.dv + (p.normalize ? 1 : 0);
    const size_t s1 = ll_anti_state_floats(p.L, BW_LL_C, w, p.D), s2 = ll_anti_state_floats(p.L, BW_LL_C, p.D, p.dv);
    return bwd_ll_level_bytes(p) + (size_t)p.B * p.H * (s1 > s2 ? s1 : s2) * sizeof(float);
}

// the part of the workspace after the per-row buffers and the log-linear buffers: the
// tensor-core dq pass's own workspace (segment totals, snapshot stack)
size_t bwd_ll_tail_bytes(const Problem &p, int sms)
{
    const size_t t = p.lam ? bwd_ll_tc_bytes(p, sms) : 0;
    return t ? t + 256 : 0;  // + alignment of its start
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

// v' = [v, 1] (normalised) or v, fp32
template <typename T>
__global__ void bw_vw_kernel(const T *v, float *vw, long rows, int dv, int normalize)
{
    const int w = dv + (normalize ? 1 : 0);
    for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < rows * w; e += (long)gridDim.x * blockDim.x) {
        const long r = e / w;
        const int j = (int)(e - r * w);
        vw[e] = j < dv ? to_f32(v[r * dv + j]) : 1.f;
    }
}

// per row: D = dout (/ den), D' = [D, -D . out] with out = num / den from nd = [num, den]
// (normalised), or D' = D
template <typename T>
__global__ void __launch_bounds__(BW_THREADS) bw_prep_kernel(const T *dout, const float *nd, float *dn,
                                                           float *dw, long rows, int dv, int normalize)
{
    const long r = blockIdx.x;
    if (r >= rows) return;
    const int w = dv + (normalize ? 1 : 0);
    const float inv = normalize ? 1.f / nd[r * w + dv] : 1.f;
    __shared__ float red[BW_THREADS / 32];
    float g = 0.f;
    for (int j = threadIdx.x; j < dv; j += BW_THREADS) {
        const float d = to_f32(dout[r * dv + j]) * inv;
        dn[r * dv + j] = d;
        dw[r * w + j] = d;
        if (normalize) g = fmaf(d, nd[r * w + j] * inv, g);
    }
    if (!normalize) return;
    for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = g;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int wi = 0; wi < BW_THREADS / 32; ++wi) t += red[wi];
        dw[r * w + dv] = -t;
    }
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

// one identity-feature, unnormalised causal pass under the log-linear mask (the caller's
// level weights, query-side as in the forward) on the generic kernel, levels in `lv`
int pass_ll(const Problem &base, const float *q, const float *k, const float *v, float *out, int dk,
            int dv, void *lv)
{
    Problem p = base;
    p.q = q; p.k = k; p.v = v; p.out = out;
    p.dk = dk; p.dv = dv; p.D = dk;
    p.C = BW_LL_C;
    p.fm = LA_FM_IDENTITY; p.m = 0; p.omega = nullptr;
    p.normalize = 0;
    p.dtype = LA_F32;
    p.rev = 0;
    p.workspace = lv;
    p.workspace_bytes = simt_workspace_bytes(p.B, p.H, p.L, dk, dv, BW_LL_C, true);
    return simt_launch(p, simt_inter_levels(p.L, BW_LL_C), ilog2(BW_LL_C));
}

template <typename T>
int bwd_t(const Problem &p, int sms, const void *dout, void *dq, void *dk_, void *dv_)
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
    bw_vw_kernel<T><<<1024, 256, 0, st>>>((const T *)p.v, b.vw, rows, p.dv, p.normalize);
    if (p.lam) {
        // log-linear mask: the causal passes carry the level weights of the query rows; the
        // anti-causal sums weigh each pair by the later row's level weight (bwd_ll.cu)
        uint8_t *extra = (uint8_t *)p.workspace + bwd_floats(rows, D, p.dv, p.normalize, nullptr, nullptr) * sizeof(float);
        void *lv = extra;
        float *W = (float *)(extra + bwd_ll_level_bytes(p));
        const int BH = p.B * p.H;
        if (p.normalize && (rc = pass_ll(p, b.fq, b.fk, b.vw, b.nd, D, w, lv)) != LA_OK) return rc;  // [num, den]
        bw_prep_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)dout, b.nd, b.dn, b.dw, rows, p.dv,
                                                     p.normalize);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
        Problem tq;
        const bool tc_dq = bwd_ll_tc_dq(p, sms, &tq);
        if (tc_dq) {
            // dq = the tensor-core log-linear forward of (q' = dout, k' = v, v' = k)
            tq.q = dout; tq.k = p.v; tq.v = p.k; tq.out = dq;
            tq.workspace = (void *)(((uintptr_t)(extra + bwd_ll_extra_bytes(p)) + 255) & ~(uintptr_t)255);
            tq.workspace_bytes = bwd_ll_tc_bytes(p, sms);
            if ((rc = tc_launch(tq, sms)) != LA_OK) return rc;
        } else if ((rc = pass_ll(p, b.dw, b.vw, b.fk, b.dfq, w, D, lv)) != LA_OK) {
            return rc;  // dphi(q)
        }
        if ((rc = ll_anti_pass(BH, p.L, BW_LL_C, b.vw, b.dw, b.fq, p.lam, p.nl, b.dfk, w, D, W, st)) != LA_OK)
            return rc;  // dphi(k)
        if ((rc = ll_anti_pass(BH, p.L, BW_LL_C, b.fk, b.fq, b.dn, p.lam, p.nl, b.dvf, D, p.dv, W, st)) != LA_OK)
            return rc;  // dv
        if (tc_dq) {
            bw_chain_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)p.k, b.dfk, (T *)dk_, rows, p.dk, D, p.fm,
                                                          p.omega, p.m);
            bw_cast_kernel<T><<<1024, 256, 0, st>>>(b.dvf, (T *)dv_, rows * p.dv);
            return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
        }
    } else {
        if (p.normalize && (rc = pass(p, b.fq, b.fk, b.vw, b.nd, D, w, 0)) != LA_OK) return rc;  // [num, den]
        bw_prep_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)dout, b.nd, b.dn, b.dw, rows, p.dv,
                                                     p.normalize);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
        if ((rc = pass(p, b.dw, b.vw, b.fk, b.dfq, w, D, 0)) != LA_OK) return rc;   // dphi(q)
        if ((rc = pass(p, b.vw, b.dw, b.fq, b.dfk, w, D, 1)) != LA_OK) return rc;   // dphi(k)
        if ((rc = pass(p, b.fk, b.fq, b.dn, b.dvf, D, p.dv, 1)) != LA_OK) return rc;  // dv
    }
    bw_chain_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)p.q, b.dfq, (T *)dq, rows, p.dk, D, p.fm,
                                                  p.omega, p.m);
    bw_chain_kernel<T><<<grid, BW_THREADS, 0, st>>>((const T *)p.k, b.dfk, (T *)dk_, rows, p.dk, D, p.fm,
                                                  p.omega, p.m);
    bw_cast_kernel<T><<<1024, 256, 0, st>>>(b.dvf, (T *)dv_, rows * p.dv);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

// ---------------------------------------------------------------- tensor-core route
typedef __nv_bfloat16 bf16;

struct TcBufs {
    bf16 *fq, *fk, *dn, *gq;            // operands (fq, fk: elu+1 only; dn, gq: normaliser)
    float *zc, *num, *zsu, *dqm, *dkm;  // pass outputs (fp32 rows, normaliser)
    float *g;                           // normaliser: g_t = D_t . out_t
    void *ws;                           // tensor-core pass workspace (segment totals)
    size_t ws_bytes;
};

// one identity-feature, unnormalised pass on the tensor cores (bf16 rows), causal or (rev)
// anti-causal, with the caller's Retention decay if any (gamma^|t-s| is the same mask read
// in either direction)
Problem tc_pass(const Problem &base, const void *q, const void *k, const void *v, void *out, int dk,
                int dv, int rev = 0)
{
    Problem p = base;
    p.q = q; p.k = k; p.v = v; p.out = out;
    p.dk = dk; p.dv = dv; p.D = dk;
    p.C = 64;
    p.fm = LA_FM_IDENTITY; p.m = 0; p.omega = nullptr;
    p.normalize = 0;
    p.lam = nullptr; p.nl = 0;
    p.dtype = LA_BF16;
    p.rev = rev;
    p.out_f32 = 0;
    p.S0 = nullptr; p.z0 = nullptr;
    p.esyn = 0;
    return p;
}

// a pass whose q and k are the constant rows e = (1, 0, ..., 0) (dk = 64): out_t = the sum of
// the rows v_s, s <= t (causal) or s >= t (anti-causal).  The kernel writes e into shared
// memory itself; the tensor maps of q and k only need a valid, aligned address.
Problem e_pass(const Problem &base, const void *v, void *out, int dv, int rev)
{
    Problem p = tc_pass(base, base.v, base.v, v, out, 64, dv, rev);
    p.esyn = 1;
    return p;
}

// The passes of the route, in order.  Without the normaliser dphi(q), dphi(k) and dv go
// straight into dq, dk, dv (bf16; with elu+1 the chain kernel then applies its derivative
// to dq, dk in place).  With it: Z, num and (after the prep kernel) the suffix sums, then
// dphi(q), dphi(k) in fp32, since dphi(q) = pass - g Z and dphi(k) = pass - suffix can
// cancel and so are formed (by the chain kernel) before any rounding to bf16; then dv.
int tc_passes(const Problem &p, const TcBufs &b, const void *dout, void *dq, void *dk, void *dv, Problem *ps)
{
    const int D = p.D, w = p.dv;
    int n = 0;
    if (p.normalize) {
        ps[n++] = e_pass(p, b.fk, b.zc, D, 0);                             // Z
        ps[n++] = tc_pass(p, b.fq, b.fk, p.v, b.num, D, w);                // num
        ps[n++] = e_pass(p, b.gq, b.zsu, D, 1);                            // suffix, anti
        ps[n++] = tc_pass(p, b.dn, p.v, b.fk, b.dqm, w, D);                // dphi(q)
        ps[n++] = tc_pass(p, p.v, b.dn, b.fq, b.dkm, w, D, 1);             // dphi(k), anti
        for (int i = 0; i < n; ++i) ps[i].out_f32 = 1;
    } else {
        ps[n++] = tc_pass(p, dout, p.v, b.fk, dq, w, D);                   // dphi(q)
        ps[n++] = tc_pass(p, p.v, dout, b.fq, dk, w, D, 1);                // dphi(k), anti
    }
    ps[n++] = tc_pass(p, b.fk, b.fq, p.normalize ? (const void *)b.dn : dout, dv, D, w, 1);  // dv, anti
    return n;
}

size_t tc_bufs(const Problem &p, int sms, char *base, TcBufs *b)
{
    const size_t rows = (size_t)p.B * p.H * p.L;
    const int D = p.D, dv = p.dv;
    size_t off = 0;
    TcBufs dummy;
    TcBufs *t = b ? b : &dummy;
    auto take = [&](auto **ptr, size_t bytes) {
        if (b) *ptr = (std::remove_reference_t<decltype(**ptr)> *)(base + off);
        off += (bytes + 1023) / 1024 * 1024;
    };
    const size_t N = p.normalize ? 1 : 0, F = p.fm == LA_FM_IDENTITY ? 0 : 1;
    take(&t->fq, F * rows * D * 2);  // identity features: the passes read q, k themselves
    take(&t->fk, F * rows * D * 2);
    take(&t->dn, N * rows * dv * 2);
    take(&t->gq, N * rows * D * 2);
    take(&t->zc, N * rows * D * 4);
    take(&t->num, N * rows * dv * 4);
    take(&t->zsu, N * rows * D * 4);
    take(&t->dqm, N * rows * D * 4);
    take(&t->dkm, N * rows * D * 4);
    take(&t->g, N * rows * 4);
    // the passes run one after another on the stream and share one workspace
    Problem ps[6];
    TcBufs nb{};
    const int n = tc_passes(p, nb, nullptr, nullptr, nullptr, nullptr, ps);
    size_t wmax = 0;
    for (int i = 0; i < n; ++i) {
        la_plan_info info;
        if (tc_plan(ps[i], sms, &info) == LA_OK && info.workspace_bytes > wmax) wmax = info.workspace_bytes;
    }
    if (b) {
        t->ws = base + off;
        t->ws_bytes = wmax;
    }
    off += (wmax + 1023) / 1024 * 1024;
    return off;
}

// The elementwise kernels of the route: one warp per row, four consecutive elements per
// lane (8-byte bf16 / 16-byte fp32 accesses), reductions by warp shuffles.  D and dv are
// 64 or 128 here.
constexpr int TB_ROWS = 8;  // rows (warps) per block

__device__ __forceinline__ void ld4(const bf16 *p, float (&x)[4])
{
    const uint2 u = *(const uint2 *)p;
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
__device__ __forceinline__ void st4(bf16 *p, const float (&x)[4])
{
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *(const uint32_t *)&a;
    u.y = *(const uint32_t *)&b;
    *(uint2 *)p = u;
}
__device__ __forceinline__ void ld4(const float *p, float (&x)[4])
{
    const float4 f = *(const float4 *)p;
    x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
}
__device__ __forceinline__ float warp_sum(float x)
{
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// phi(q), phi(k) as bf16 rows (elu+1)
__global__ void __launch_bounds__(32 * TB_ROWS) tb_feat_kernel(const bf16 *q, const bf16 *k, TcBufs b,
                                                             long rows, int dk)
{
    const long r = (long)blockIdx.x * TB_ROWS + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    for (int i = 4 * lane; i < dk; i += 128) {
        float xq[4], xk[4];
        ld4(q + r * dk + i, xq);
        ld4(k + r * dk + i, xk);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            xq[e] = phi_elu1(xq[e]);
            xk[e] = phi_elu1(xk[e]);
        }
        st4(b.fq + r * dk + i, xq);
        st4(b.fk + r * dk + i, xk);
    }
}

// With the normaliser: D = dout / den (den = phi(q).Z), g = D . num / den and g phi(q)
__global__ void __launch_bounds__(32 * TB_ROWS) tb_prep_kernel(const bf16 *dout, TcBufs b, long rows, int D,
                                                             int dv)
{
    const long r = (long)blockIdx.x * TB_ROWS + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    float part = 0.f;
    for (int i = 4 * lane; i < D; i += 128) {
        float f[4], z[4];
        ld4(b.fq + r * D + i, f);
        ld4(b.zc + r * D + i, z);
        part += f[0] * z[0] + f[1] * z[1] + f[2] * z[2] + f[3] * z[3];
    }
    const float inv = 1.f / warp_sum(part);
    float gp = 0.f;
    for (int j = 4 * lane; j < dv; j += 128) {
        // g from the same bf16 D the passes read, so dphi(q) = pass - g Z is the exact
        // gradient for that D (its rounding is not amplified by the subtraction)
        float d[4], n[4];
        ld4(dout + r * dv + j, d);
        ld4(b.num + r * dv + j, n);
#pragma unroll
        for (int e = 0; e < 4; ++e) d[e] = __bfloat162float(__float2bfloat16_rn(d[e] * inv));
        st4(b.dn + r * dv + j, d);
#pragma unroll
        for (int e = 0; e < 4; ++e) gp += d[e] * (n[e] * inv);
    }
    const float g = warp_sum(gp);
    if (lane == 0) b.g[r] = g;
    for (int i = 4 * lane; i < D; i += 128) {
        float f[4];
        ld4(b.fq + r * D + i, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] *= g;
        st4(b.gq + r * D + i, f);
    }
}

// dq, dk through the feature map: with the normaliser from the fp32 pass outputs,
// dphi(q) = dqm - g Z and dphi(k) = dkm - suffix; without it (elu+1 only) from the bf16
// dphi rows the passes left in dq, dk, in place
__global__ void __launch_bounds__(32 * TB_ROWS) tb_chain_kernel(const bf16 *q, const bf16 *k, TcBufs b,
                                                              bf16 *dq, bf16 *dk, long rows, int D, int fm,
                                                              int normalize)
{
    const long r = (long)blockIdx.x * TB_ROWS + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float g = normalize ? b.g[r] : 0.f;
    for (int i = 4 * lane; i < D; i += 128) {
        float a[4], c[4];
        if (normalize) {
            float z[4], zs[4];
            ld4(b.dqm + r * D + i, a);
            ld4(b.dkm + r * D + i, c);
            ld4(b.zc + r * D + i, z);
            ld4(b.zsu + r * D + i, zs);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                a[e] -= g * z[e];
                c[e] -= zs[e];
            }
        } else {
            ld4(dq + r * D + i, a);
            ld4(dk + r * D + i, c);
        }
        if (fm == LA_FM_ELU1) {
            float xq[4], xk[4];
            ld4(q + r * D + i, xq);
            ld4(k + r * D + i, xk);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (xq[e] < 0.f) a[e] *= expf(xq[e]);
                if (xk[e] < 0.f) c[e] *= expf(xk[e]);
            }
        }
        st4(dq + r * D + i, a);
        st4(dk + r * D + i, c);
    }
}

int tc_route(const Problem &p, int sms, const void *dout, void *dq, void *dk, void *dv)
{
    TcBufs b;
    tc_bufs(p, sms, (char *)p.workspace, &b);
    if (p.fm == LA_FM_IDENTITY) {
        b.fq = (bf16 *)p.q;  // read only
        b.fk = (bf16 *)p.k;
    }
    const long rows = (long)p.B * p.H * p.L;
    cudaStream_t st = p.stream;
    const unsigned tgrid = (unsigned)((rows + TB_ROWS - 1) / TB_ROWS);
    if (p.fm == LA_FM_ELU1) {
        tb_feat_kernel<<<tgrid, 32 * TB_ROWS, 0, st>>>((const bf16 *)p.q, (const bf16 *)p.k, b, rows, p.dk);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    Problem ps[6];
    const int n = tc_passes(p, b, dout, dq, dk, dv, ps);
    for (int i = 0; i < n; ++i) {
        ps[i].workspace = b.ws;
        ps[i].workspace_bytes = b.ws_bytes;
    }
    int i = 0, rc;
    if (p.normalize) {  // Z, num, then D, g and g phi(q) from them
        for (; i < 2; ++i)
            if ((rc = tc_launch(ps[i], sms)) != LA_OK) return rc;
        tb_prep_kernel<<<tgrid, 32 * TB_ROWS, 0, st>>>((const bf16 *)dout, b, rows, p.D, p.dv);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    for (; i < n; ++i)
        if ((rc = tc_launch(ps[i], sms)) != LA_OK) return rc;
    if (p.fm == LA_FM_IDENTITY && !p.normalize) return LA_OK;  // the passes wrote dq, dk, dv
    tb_chain_kernel<<<tgrid, 32 * TB_ROWS, 0, st>>>((const bf16 *)p.q, (const bf16 *)p.k, b, (bf16 *)dq,
                                                   (bf16 *)dk, rows, p.D, p.fm, p.normalize);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

// ---------------------------------------------------------------- FAVOR+ tensor-core route
// FAVOR+ features ("Linear Attention / Performerの理論と実装", the FAVOR+ section): phi(x)_l =
// exp(w_l . x - |x s|^2 / 2) / sqrt(m) with w_l = s omega_l and s = dk^(-1/4).  The m features
// are cut into NH = m / 128 blocks of 128 columns (bf16 rows, one buffer each), and every
// pass of the identity route runs once per block: the passes whose scores are phi(q).phi(k)
// (num, dv) add their blocks' fp32 outputs, the others (Z, suffix, dphi) give a block of
// their m-wide output each.  All passes store fp32; the last kernel forms dphi, contracts it with
// the features' derivative and sums dv.
struct TfBufs {
    bf16 *fq, *fk;           // [NH][rows][128]
    bf16 *dn, *gq;           // [rows][dv], [NH][rows][128] (normaliser)
    float *zc, *num, *zsu;   // [NH][rows][128], [NH][rows][dv], [NH][rows][128] (normaliser)
    float *dqm, *dkm, *dvp;  // [NH][rows][128], [NH][rows][128], [NH][rows][dv]
    float *g;                // [rows] (normaliser)
    bf16 *omt;               // omega^T as bf16 hi / lo rows: [2][64][m + 8]
    void *ws;
    size_t ws_bytes;
};
constexpr int TF_MAXP = 6 * 4;  // passes: six per feature block, m <= 512
constexpr int TF_DK = 64;        // dk = dv of the route

int tf_passes(const Problem &p, const TfBufs &b, const void *dout, Problem *ps)
{
    const long rows = (long)p.B * p.H * p.L;
    const int NH = p.m / 128, w = p.dv;
    const bool nz = p.normalize != 0;
    const void *dd = nz ? (const void *)b.dn : dout;
    auto fq = [&](int h) { return b.fq ? b.fq + h * rows * 128 : nullptr; };
    auto fk = [&](int h) { return b.fk ? b.fk + h * rows * 128 : nullptr; };
    auto f32 = [&](float *x, int h, int width) { return x ? x + h * rows * width : nullptr; };
    auto b16 = [&](bf16 *x, int h) { return x ? x + h * rows * 128 : nullptr; };
    int n = 0;
    for (int h = 0; h < NH && nz; ++h) ps[n++] = e_pass(p, fk(h), f32(b.zc, h, 128), 128, 0);          // Z
    for (int h = 0; h < NH && nz; ++h) ps[n++] = tc_pass(p, fq(h), fk(h), p.v, f32(b.num, h, w), 128, w);  // num
    for (int h = 0; h < NH && nz; ++h) ps[n++] = e_pass(p, b16(b.gq, h), f32(b.zsu, h, 128), 128, 1);  // suffix
    for (int h = 0; h < NH; ++h) ps[n++] = tc_pass(p, dd, p.v, fk(h), f32(b.dqm, h, 128), w, 128);     // dphi(q)
    for (int h = 0; h < NH; ++h) ps[n++] = tc_pass(p, p.v, dd, fq(h), f32(b.dkm, h, 128), w, 128, 1);  // dphi(k)
    for (int h = 0; h < NH; ++h) ps[n++] = tc_pass(p, fk(h), fq(h), dd, f32(b.dvp, h, w), 128, w, 1);  // dv
    for (int i = 0; i < n; ++i) ps[i].out_f32 = 1;
    return n;
}

size_t tf_bufs(const Problem &p, int sms, char *base, TfBufs *b)
{
    const size_t rows = (size_t)p.B * p.H * p.L, NH = p.m / 128, w = p.dv;
    const size_t N = p.normalize ? 1 : 0;
    size_t off = 0;
    TfBufs dummy;
    TfBufs *t = b ? b : &dummy;
    auto take = [&](auto **ptr, size_t bytes) {
        if (b) *ptr = (std::remove_reference_t<decltype(**ptr)> *)(base + off);
        off += (bytes + 1023) / 1024 * 1024;
    };
    take(&t->fq, NH * rows * 128 * 2);
    take(&t->fk, NH * rows * 128 * 2);
    take(&t->dn, N * rows * w * 2);
    take(&t->gq, N * NH * rows * 128 * 2);
    take(&t->zc, N * NH * rows * 128 * 4);
    take(&t->num, N * NH * rows * w * 4);
    take(&t->zsu, N * NH * rows * 128 * 4);
    take(&t->dqm, NH * rows * 128 * 4);
    take(&t->dkm, NH * rows * 128 * 4);
    take(&t->dvp, NH * rows * w * 4);
    take(&t->g, N * rows * 4);
    take(&t->omt, (size_t)2 * TF_DK * (p.m + 8) * 2);
    Problem ps[TF_MAXP];
    TfBufs nb{};
    const int n = tf_passes(p, nb, nullptr, ps);
    size_t wmax = 0;
    for (int i = 0; i < n; ++i) {
        la_plan_info info;
        if (tc_plan(ps[i], sms, &info) == LA_OK && info.workspace_bytes > wmax) wmax = info.workspace_bytes;
    }
    if (b) {
        t->ws = base + off;
        t->ws_bytes = wmax;
    }
    off += (wmax + 1023) / 1024 * 1024;
    return off;
}

// Normaliser, RW rows per warp (their loads in flight together): den = phi(q).Z over all
// NH feature blocks, D = bf16(dout / den), g = D . num / den (num summed over the blocks),
// g phi(q) by block.  dv = 64: lanes 0-15 hold one group of four columns of D.
template <int NH>
__global__ void __launch_bounds__(32 * TB_ROWS) tf_prep_kernel(const bf16 *dout, TfBufs b, long rows)
{
    constexpr int RW = NH <= 2 ? 2 : 1, DV = 64;
    const long r0 = ((long)blockIdx.x * TB_ROWS + (threadIdx.x >> 5)) * RW;
    const int lane = threadIdx.x & 31, c = 4 * lane;
    const bool dl = c < DV;
    float f[RW][NH][4], z[RW][NH][4], d[RW][4], nm[RW][NH][4];
#pragma unroll
    for (int w = 0; w < RW; ++w) {
        const long r = r0 + w < rows ? r0 + w : rows - 1;  // past the end: a valid row, not stored
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            ld4(b.fq + (h * rows + r) * 128 + c, f[w][h]);
            ld4(b.zc + (h * rows + r) * 128 + c, z[w][h]);
            if (dl) ld4(b.num + (h * rows + r) * DV + c, nm[w][h]);
        }
        if (dl) ld4(dout + r * DV + c, d[w]);
    }
#pragma unroll
    for (int w = 0; w < RW; ++w) {
        const long r = r0 + w;
        float part = 0.f;
#pragma unroll
        for (int h = 0; h < NH; ++h)
            part += f[w][h][0] * z[w][h][0] + f[w][h][1] * z[w][h][1] + f[w][h][2] * z[w][h][2] +
                    f[w][h][3] * z[w][h][3];
        const float inv = 1.f / warp_sum(part);
        float gp = 0.f;
        if (dl) {
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) s4[e] += nm[w][h][e];
#pragma unroll
            for (int e = 0; e < 4; ++e) d[w][e] = __bfloat162float(__float2bfloat16_rn(d[w][e] * inv));
            if (r < rows) st4(b.dn + r * DV + c, d[w]);
#pragma unroll
            for (int e = 0; e < 4; ++e) gp += d[w][e] * (s4[e] * inv);
        }
        const float g = warp_sum(gp);
        if (r >= rows) continue;
        if (lane == 0) b.g[r] = g;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
#pragma unroll
            for (int e = 0; e < 4; ++e) f[w][h][e] *= g;
            st4(b.gq + (h * rows + r) * 128 + c, f[w][h]);
        }
    }
}

// The two contractions with omega (features: x omega^T; chain: u omega) on the warp-level
// tensor-core instruction, m16n8k16 bf16 in, fp32 accumulate.  omega enters as a bf16 hi / lo
// pair (omega = hi + lo to about 2^-16 relative): x is exact in bf16, u is split the same
// way, and the products hi.hi + hi.lo (+ lo.hi) keep the contraction at fp32 accuracy.
// Fragment layout of the instruction (PTX ISA, mma.m16n8k16 with 16-bit operands), with
// g = lane / 4 and t = lane % 4: A holds rows g and g+8 at columns 2t, 2t+1 and 2t+8, 2t+9;
// B holds column g at rows 2t, 2t+1 and 2t+8, 2t+9; the accumulator holds rows g and g+8 at
// columns 2t, 2t+1.  The lower half of each 32-bit register is the lower index.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                 "{%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t bf2(float lo, float hi)
{
    const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *(const uint32_t *)&t;
}
__device__ __forceinline__ float bf_to(bf16 x) { return __bfloat162float(x); }

// Features: persistent blocks of 8 warps, one 16-row tile per warp at a time; W = s omega
// as bf16 hi / lo rows [m][TFM_WS] in shared memory (the padded stride makes the B loads
// conflict-free); 64 features per accumulator pass.
constexpr int TFM_WS = 72;
__global__ void __launch_bounds__(256) tf_feat_mma_kernel(const bf16 *x, const float *omega, bf16 *f, long rows,
                                                          int m, bf16 *omt)
{
    extern __shared__ uint4 tfm_sm[];
    bf16 *const Whi = (bf16 *)tfm_sm, *const Wlo = Whi + m * TFM_WS;
    const float s = rsqrtf(8.f);  // dk^(-1/4), dk = 64
    for (int e = threadIdx.x; e < m * TF_DK; e += blockDim.x) {
        const float w = s * __ldg(omega + e);
        const bf16 h = __float2bfloat16_rn(w);
        Whi[(e >> 6) * TFM_WS + (e & 63)] = h;
        Wlo[(e >> 6) * TFM_WS + (e & 63)] = __float2bfloat16_rn(w - bf_to(h));
        if (omt && blockIdx.x == 0) {
            // omega^T hi / lo rows for the chain kernel (unscaled)
            const float o = __ldg(omega + e);
            const bf16 oh = __float2bfloat16_rn(o);
            omt[(e & 63) * (m + 8) + (e >> 6)] = oh;
            omt[(TF_DK + (e & 63)) * (m + 8) + (e >> 6)] = __float2bfloat16_rn(o - bf_to(oh));
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float inv = rsqrtf((float)m);
    const long ntiles = (rows + 15) / 16;
    for (long tile = (long)blockIdx.x * 8 + warp; tile < ntiles; tile += (long)gridDim.x * 8) {
        const long ra = tile * 16 + g, rb = ra + 8;
        uint32_t a[4][4];
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int c = kk * 16 + 2 * t;
            a[kk][0] = ra < rows ? *(const uint32_t *)(x + ra * TF_DK + c) : 0u;
            a[kk][1] = rb < rows ? *(const uint32_t *)(x + rb * TF_DK + c) : 0u;
            a[kk][2] = ra < rows ? *(const uint32_t *)(x + ra * TF_DK + c + 8) : 0u;
            a[kk][3] = rb < rows ? *(const uint32_t *)(x + rb * TF_DK + c + 8) : 0u;
#pragma unroll
            for (int h = 0; h < 4; h += 2) {
                const float x0 = __uint_as_float(a[kk][h] << 16), x1 = __uint_as_float(a[kk][h] & 0xFFFF0000u);
                const float y0 = __uint_as_float(a[kk][h + 1] << 16), y1 = __uint_as_float(a[kk][h + 1] & 0xFFFF0000u);
                sa += x0 * x0 + x1 * x1;
                sb += y0 * y0 + y1 * y1;
            }
        }
        sa += __shfl_xor_sync(0xffffffffu, sa, 1);
        sa += __shfl_xor_sync(0xffffffffu, sa, 2);
        sb += __shfl_xor_sync(0xffffffffu, sb, 1);
        sb += __shfl_xor_sync(0xffffffffu, sb, 2);
        const float ha = 0.5f * s * s * sa, hb = 0.5f * s * s * sb;
        for (int c0 = 0; c0 < m; c0 += 64) {
            float acc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int at = (c0 + nt * 8 + g) * TFM_WS + kk * 16 + 2 * t;
                    const uint32_t *wh = (const uint32_t *)(Whi + at), *wl = (const uint32_t *)(Wlo + at);
                    mma_bf16(acc[nt], a[kk], wh[0], wh[4]);
                    mma_bf16(acc[nt], a[kk], wl[0], wl[4]);
                }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int col = c0 + nt * 8 + 2 * t;
                bf16 *const fo = f + (size_t)(col >> 7) * rows * 128 + (col & 127);
                if (ra < rows)
                    *(uint32_t *)(fo + ra * 128) = bf2(expf(acc[nt][0] - ha) * inv, expf(acc[nt][1] - ha) * inv);
                if (rb < rows)
                    *(uint32_t *)(fo + rb * 128) = bf2(expf(acc[nt][2] - hb) * inv, expf(acc[nt][3] - hb) * inv);
            }
        }
    }
}

// Chain: persistent blocks of 8 warps over tiles of TFC_RB rows, blockIdx.y = 0 for dq, 1 for
// dk.  The block first forms u = dphi phi (as bf16 hi / lo rows) and sum_l u_l for its rows in
// shared memory; then warp w takes rows 16 (w / 4) .. +15 and output columns 16 (w % 4) .. +15:
// sum_l u_l omega_li with omega^T as bf16 hi / lo rows [64][m + 8], read through the L1 (it is
// the same 2 x 64 x (m + 8) values for every block), which leaves shared memory to u alone
// and so lets four blocks share an SM.  The y = 0 blocks also sum the per-block dv parts of their rows.
constexpr int TFC_RB = 32;
constexpr int TFC_IT = 4;  // staged items in flight per thread
__global__ void __launch_bounds__(256, 4) tf_chain_mma_kernel(const bf16 *q, const bf16 *k, const float *omega,
                                                           TfBufs b, bf16 *dq, bf16 *dk, bf16 *dv, long rows,
                                                           int m, int dvn, int normalize)
{
    extern __shared__ uint4 tfc_sm[];
    const int OS = m + 8;  // bf16 stride of the omega^T and u rows
    const bf16 *const Ohi = b.omt, *const Olo = b.omt + TF_DK * OS;
    bf16 *const Uhi = (bf16 *)tfc_sm, *const Ulo = Uhi + TFC_RB * OS;
    float *const usum = (float *)(Ulo + TFC_RB * OS);
    const bool isq = blockIdx.y == 0;
    const bf16 *const feat = isq ? b.fq : b.fk;
    const float *const dm = isq ? b.dqm : b.dkm;
    const float *const sub = normalize ? (isq ? b.zc : b.zsu) : nullptr;
    const bf16 *const x = isq ? q : k;
    bf16 *const dx = isq ? dq : dk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int NH = m / 128, lm = 31 - __clz(m);  // m: a power of two
    const float s = rsqrtf(8.f);
    const long ntiles = (rows + TFC_RB - 1) / TFC_RB;
    for (long tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const long r0 = tile * TFC_RB;
        __syncthreads();  // the previous tile's u read
        if (threadIdx.x < TFC_RB) usum[threadIdx.x] = 0.f;
        __syncthreads();
        // u rows in groups of four columns: item e = r (m / 4) + l4, TFC_IT per thread with
        // their loads in flight together; a warp's 32 items share one row (m / 4 is a multiple
        // of 32), so each row sum is one shuffle reduction per warp
        const int lg = lm - 2;  // log2(m / 4)
        for (int e0 = 0; e0 < TFC_RB << lg; e0 += TFC_IT * 256) {
            float4 d4[TFC_IT], s4[TFC_IT];
            uint2 f4[TFC_IT];
#pragma unroll
            for (int j = 0; j < TFC_IT; ++j) {
                const int e = e0 + j * 256 + threadIdx.x, r = e >> lg, l = (e & ((1 << lg) - 1)) << 2;
                const long row = r0 + r;
                d4[j] = s4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                f4[j] = make_uint2(0u, 0u);
                if (r < TFC_RB && row < rows) {
                    const size_t at = ((size_t)(l >> 7) * rows + row) * 128 + (l & 127);
                    d4[j] = *(const float4 *)(dm + at);
                    if (sub) {
                        const float c = isq ? b.g[row] : 1.f;
                        const float4 z = *(const float4 *)(sub + at);
                        s4[j] = make_float4(c * z.x, c * z.y, c * z.z, c * z.w);
                    }
                    f4[j] = *(const uint2 *)(feat + at);
                }
            }
#pragma unroll
            for (int j = 0; j < TFC_IT; ++j) {
                const int e = e0 + j * 256 + threadIdx.x, r = e >> lg, l = (e & ((1 << lg) - 1)) << 2;
                const float u0 = (d4[j].x - s4[j].x) * __uint_as_float(f4[j].x << 16);
                const float u1 = (d4[j].y - s4[j].y) * __uint_as_float(f4[j].x & 0xFFFF0000u);
                const float u2 = (d4[j].z - s4[j].z) * __uint_as_float(f4[j].y << 16);
                const float u3 = (d4[j].w - s4[j].w) * __uint_as_float(f4[j].y & 0xFFFF0000u);
                if (r < TFC_RB) {
                    const uint2 h = make_uint2(bf2(u0, u1), bf2(u2, u3));
                    const float h0 = __uint_as_float(h.x << 16), h1 = __uint_as_float(h.x & 0xFFFF0000u);
                    const float h2 = __uint_as_float(h.y << 16), h3 = __uint_as_float(h.y & 0xFFFF0000u);
                    *(uint2 *)(Uhi + r * OS + l) = h;
                    *(uint2 *)(Ulo + r * OS + l) = make_uint2(bf2(u0 - h0, u1 - h1), bf2(u2 - h2, u3 - h3));
                }
                const float part = warp_sum(u0 + u1 + u2 + u3);
                if (lane == 0 && r < TFC_RB) atomicAdd(&usum[r], part);
            }
        }
        __syncthreads();
        const int rt = 16 * (warp >> 2), n0 = 2 * (warp & 3);  // row tile, first of two n-tiles
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int kk = 0; kk < m / 16; ++kk) {
            const int c = kk * 16 + 2 * t;
            const int ua = (rt + g) * OS + c, ub = ua + 8 * OS;
            const uint32_t ah[4] = {*(const uint32_t *)(Uhi + ua), *(const uint32_t *)(Uhi + ub),
                                    *(const uint32_t *)(Uhi + ua + 8), *(const uint32_t *)(Uhi + ub + 8)};
            const uint32_t al[4] = {*(const uint32_t *)(Ulo + ua), *(const uint32_t *)(Ulo + ub),
                                    *(const uint32_t *)(Ulo + ua + 8), *(const uint32_t *)(Ulo + ub + 8)};
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int at = ((n0 + j) * 8 + g) * OS + c;
                const uint32_t *oh = (const uint32_t *)(Ohi + at), *ol = (const uint32_t *)(Olo + at);
                const uint32_t h0 = __ldg(oh), h1 = __ldg(oh + 4), l0 = __ldg(ol), l1 = __ldg(ol + 4);
                mma_bf16(acc[j], ah, h0, h1);
                mma_bf16(acc[j], ah, l0, l1);
                mma_bf16(acc[j], al, h0, h1);
            }
        }
        const long ra = r0 + rt + g, rb = ra + 8;
        const float sa = usum[rt + g], sb = usum[rt + g + 8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = (n0 + j) * 8 + 2 * t;
            if (ra < rows) {
                const uint32_t xv = *(const uint32_t *)(x + ra * TF_DK + i);
                *(uint32_t *)(dx + ra * TF_DK + i) =
                    bf2(s * acc[j][0] - s * s * __uint_as_float(xv << 16) * sa,
                        s * acc[j][1] - s * s * __uint_as_float(xv & 0xFFFF0000u) * sa);
            }
            if (rb < rows) {
                const uint32_t xv = *(const uint32_t *)(x + rb * TF_DK + i);
                *(uint32_t *)(dx + rb * TF_DK + i) =
                    bf2(s * acc[j][2] - s * s * __uint_as_float(xv << 16) * sb,
                        s * acc[j][3] - s * s * __uint_as_float(xv & 0xFFFF0000u) * sb);
            }
        }
        if (isq)
            for (int e = threadIdx.x; e < TFC_RB * dvn; e += blockDim.x) {
                const long row = r0 + e / dvn;
                const int j = e % dvn;
                if (row >= rows) continue;
                float a = 0.f;
                for (int h = 0; h < NH; ++h) a += b.dvp[((size_t)h * rows + row) * dvn + j];
                dv[row * dvn + j] = __float2bfloat16_rn(a);
            }
    }
}

int tf_route(const Problem &p, int sms, const void *dout, void *dq, void *dk, void *dv)
{
    TfBufs b;
    tf_bufs(p, sms, (char *)p.workspace, &b);
    const long rows = (long)p.B * p.H * p.L;
    const int NH = p.m / 128;
    cudaStream_t st = p.stream;
    const size_t fsm = (size_t)2 * p.m * TFM_WS * sizeof(bf16);
    if (cudaFuncSetAttribute(tf_feat_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm) != cudaSuccess)
        return LA_ERR_CUDA;
    const long ftiles = (rows + 127) / 128;
    const unsigned fgrid = (unsigned)(ftiles < 3L * sms ? ftiles : 3L * sms);
    tf_feat_mma_kernel<<<fgrid, 256, fsm, st>>>((const bf16 *)p.q, p.omega, b.fq, rows, p.m, b.omt);
    tf_feat_mma_kernel<<<fgrid, 256, fsm, st>>>((const bf16 *)p.k, p.omega, b.fk, rows, p.m, nullptr);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    Problem ps[TF_MAXP];
    const int n = tf_passes(p, b, dout, ps);
    for (int i = 0; i < n; ++i) {
        ps[i].workspace = b.ws;
        ps[i].workspace_bytes = b.ws_bytes;
    }
    int i = 0, rc;
    if (p.normalize) {  // Z and num of every feature block, then D, g and g phi(q)
        for (; i < 2 * NH; ++i)
            if ((rc = tc_launch(ps[i], sms)) != LA_OK) return rc;
        const long rw = NH <= 2 ? 2 : 1;  // rows per warp of the prep kernel
        const unsigned tgrid = (unsigned)((rows + TB_ROWS * rw - 1) / (TB_ROWS * rw));
        if (NH == 1) tf_prep_kernel<1><<<tgrid, 32 * TB_ROWS, 0, st>>>((const bf16 *)dout, b, rows);
        if (NH == 2) tf_prep_kernel<2><<<tgrid, 32 * TB_ROWS, 0, st>>>((const bf16 *)dout, b, rows);
        if (NH == 4) tf_prep_kernel<4><<<tgrid, 32 * TB_ROWS, 0, st>>>((const bf16 *)dout, b, rows);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    }
    for (; i < n; ++i)
        if ((rc = tc_launch(ps[i], sms)) != LA_OK) return rc;
    const size_t csm = (size_t)2 * TFC_RB * (p.m + 8) * sizeof(bf16) + TFC_RB * sizeof(float);
    if (csm > 48 * 1024 &&
        cudaFuncSetAttribute(tf_chain_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm) != cudaSuccess)
        return LA_ERR_CUDA;
    const long ctiles = (rows + TFC_RB - 1) / TFC_RB;
    const unsigned cgrid = (unsigned)(ctiles < 4L * sms ? ctiles : 4L * sms);
    tf_chain_mma_kernel<<<dim3(cgrid, 2), 256, csm, st>>>((const bf16 *)p.q, (const bf16 *)p.k, p.omega, b,
                                                          (bf16 *)dq, (bf16 *)dk, (bf16 *)dv, rows, p.m, p.dv,
                                                          p.normalize);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

// bf16 FAVOR+ with dk = dv = 64, m = 128, 256 or 512, no decay, every pass on the tensor
// cores
bool tf_supported(const Problem &p, int sms)
{
    if (p.dtype != LA_BF16 || p.fm != LA_FM_FAVOR || p.lam || p.decay || p.L < 128) return false;
    if (p.dk != TF_DK || p.dv != 64 || (p.m != 128 && p.m != 256 && p.m != 512) || !p.omega) return false;
    Problem ps[TF_MAXP];
    TfBufs nb{};
    const int n = tf_passes(p, nb, nullptr, ps);
    for (int i = 0; i < n; ++i)
        if (!tc_supported(ps[i], sms)) return false;
    return true;
}

}  // namespace

// The tensor-core routes: bf16, identity / elu+1 features, plain or decayed, and every pass of
// a shape the tensor-core forward covers (with the decay: gamma >= 0.5); FAVOR+ with dk = dv =
// 64 and m = 128, 256 or 512, without the decay.  The decay with the
// normaliser stays on the generic route: dphi(q) is then the difference of two passes, and the
// decay mode rounds its gamma-scaled key rows to bf16 differently in each, so the sums no
// longer cancel to the bf16 bar (measured relative RMS 5.5e-3 on dq at gamma = 0.95).
bool bwd_tc_supported(const Problem &p, int sms)
{
    if (p.dtype != LA_BF16 || p.lam || p.L < 128) return false;
    if (p.fm == LA_FM_FAVOR) return tf_supported(p, sms);
    if (p.decay && p.normalize) return false;
    if (p.fm != LA_FM_IDENTITY && p.fm != LA_FM_ELU1) return false;
    Problem ps[6];
    TcBufs nb{};
    const int n = tc_passes(p, nb, nullptr, nullptr, nullptr, nullptr, ps);
    for (int i = 0; i < n; ++i)
        if (!tc_supported(ps[i], sms)) return false;
    return true;
}

size_t bwd_workspace_bytes(const Problem &p, int sms)
{
    const size_t simt = bwd_floats((long)p.B * p.H * p.L, p.D, p.dv, p.normalize, nullptr, nullptr) * sizeof(float) +
                        bwd_ll_extra_bytes(p) + bwd_ll_tail_bytes(p, sms);
    const size_t tc = !bwd_tc_supported(p, sms) ? 0
                      : p.fm == LA_FM_FAVOR ? tf_bufs(p, sms, nullptr, nullptr)
                                            : tc_bufs(p, sms, nullptr, nullptr);
    return simt > tc ? simt : tc;
}

// D, dk <= 512 and dv < 512 (the generic kernel's shared-memory rows); with level weights
// no decay, and levels enough for the sequence (the generic route only)
bool bwd_supported(const Problem &p)
{
    if (!(p.D <= 512 && p.dk <= 512 && p.dv < 512)) return false;
    if (p.lam && (p.decay || p.nl < 1 + simt_inter_levels(p.L, 1))) return false;
    return true;
}

int bwd_launch(const Problem &p, int sms, int path, const void *dout, void *dq, void *dk, void *dv)
{
    if (!bwd_supported(p)) return LA_ERR_UNSUPPORTED;
    if (!p.workspace || p.workspace_bytes < bwd_workspace_bytes(p, sms)) return LA_ERR_WORKSPACE;
    // the route's elementwise kernels use 8- and 16-byte accesses on the caller's rows
    const uintptr_t al = (uintptr_t)p.q | (uintptr_t)p.k | (uintptr_t)p.v | (uintptr_t)dout |
                         (uintptr_t)dq | (uintptr_t)dk | (uintptr_t)dv;
    const bool tc = bwd_tc_supported(p, sms) && (al & 15) == 0;
    if (path == LA_PATH_TC && !tc) return LA_ERR_UNSUPPORTED;
    if (path != LA_PATH_SIMT && tc)
        return p.fm == LA_FM_FAVOR ? tf_route(p, sms, dout, dq, dk, dv) : tc_route(p, sms, dout, dq, dk, dv);
    if (p.dtype == LA_BF16) return bwd_t<__nv_bfloat16>(p, sms, dout, dq, dk, dv);
    return bwd_t<float>(p, sms, dout, dq, dk, dv);
}

}  // namespace la
