// noncausal.cu -- bidirectional (non-causal) linear attention, generic CUDA-core path.
//
// "Linear Attention / Performerの理論と実装", the non-causal normalised form (and the
// Performer's bidirectional FAVOR+ attention): every query sees every key, so one global
// state per (b, h) head serves all rows:
//     S = sum_s phi(k_s) v_s^T,  z = sum_s phi(k_s),  out_t = phi(q_t)^T S / phi(q_t)^T z
// ("attention と線形の間" section 1, StateFirst, is the unnormalised case).
//
// Two launches: (1) the state and z of every head into the workspace, one CTA per (head,
// 32-column slice of dv), summing over the tokens in 32-token tiles; (2) the output, one
// CTA per (head, 32-token tile, 32-column slice), with the state slice in shared memory.
// The feature maps are applied to tiles in shared memory (FAVOR+: the projection by omega
// on the CUDA cores).  Any dtype; D (dk, or m for FAVOR+) up to 256.
#include <stdio.h>

#include "common.cuh"

namespace la {

namespace {

constexpr int NC_THREADS = 256;
constexpr int NC_TT = 32;     // tokens per tile
constexpr int NC_COLS = 32;   // dv columns per CTA
constexpr int NC_RG = NC_THREADS / NC_COLS;

struct NcArgs {
    const void *q, *k, *v;
    void *out;
    int L, dk, dv, D, fm, m, normalize;
    const float *omega;
    float *S;  // [BH][D][dv]
    float *z;  // [BH][D]
    int decay;   // final state of a decayed causal pass: token t weighted by gamma^(L-1-t)
    float l2g;   // log2(gamma)
};

// phi of `rows` raw rows x[rows][dk] (shared) into f[rows][D] (shared); FAVOR+ uses omega
__device__ void nc_phi(const NcArgs &a, const float *x, float *f, int rows)
{
    const int tid = threadIdx.x;
    if (a.fm == LA_FM_FAVOR) {
        const float s = rsqrtf(sqrtf((float)a.dk));  // dk^{-1/4}
        const float inv = rsqrtf((float)a.m);
        for (int e = tid; e < rows * a.D; e += NC_THREADS) {
            const int r = e / a.D, l = e % a.D;
            const float *xr = x + (size_t)r * a.dk;
            const float *w = a.omega + (size_t)l * a.dk;
            float p = 0.f, n2 = 0.f;
            for (int i = 0; i < a.dk; ++i) {
                p = fmaf(__ldg(w + i), xr[i], p);
                n2 = fmaf(xr[i], xr[i], n2);
            }
            f[e] = expf(p * s - 0.5f * n2 * s * s) * inv;
        }
    } else {
        for (int e = tid; e < rows * a.D; e += NC_THREADS)
            f[e] = a.fm == LA_FM_ELU1 ? phi_elu1(x[e]) : x[e];
    }
}

template <typename T>
__global__ void __launch_bounds__(NC_THREADS) nc_state_kernel(const NcArgs a)
{
    extern __shared__ float nsm[];
    float *x = nsm;                          // [TT][dk] raw k
    float *f = x + NC_TT * a.dk;             // [TT][D]  phi(k)
    float *vt = f + NC_TT * a.D;             // [TT][COLS]
    const int head = blockIdx.x, jb = blockIdx.y * NC_COLS, tid = threadIdx.x;
    const int j = tid % NC_COLS, rg = tid / NC_COLS;
    const int jj = jb + j;
    const T *k = (const T *)a.k + (size_t)head * a.L * a.dk;
    const T *v = (const T *)a.v + (size_t)head * a.L * a.dv;
    constexpr int MAXR = 256 / NC_RG;  // D <= 256
    float acc[MAXR];
#pragma unroll
    for (int u = 0; u < MAXR; ++u) acc[u] = 0.f;
    float zacc[MAXR];
#pragma unroll
    for (int u = 0; u < MAXR; ++u) zacc[u] = 0.f;
    for (int t0 = 0; t0 < a.L; t0 += NC_TT) {
        const int rows = min(NC_TT, a.L - t0);
        __syncthreads();
        for (int e = tid; e < rows * a.dk; e += NC_THREADS) x[e] = to_f32(k[(size_t)t0 * a.dk + e]);
        for (int e = tid; e < rows * NC_COLS; e += NC_THREADS) {
            const int r = e / NC_COLS, c = jb + e % NC_COLS;
            vt[e] = c < a.dv ? to_f32(v[(size_t)(t0 + r) * a.dv + c]) : 0.f;
        }
        __syncthreads();
        nc_phi(a, x, f, rows);
        __syncthreads();
        if (a.decay) {
            for (int e = tid; e < rows * a.D; e += NC_THREADS) f[e] *= exp2f(a.l2g * (float)(a.L - 1 - t0 - e / a.D));
            __syncthreads();
        }
        for (int r = 0; r < rows; ++r) {
            const float vv = vt[r * NC_COLS + j];
#pragma unroll
            for (int u = 0; u < MAXR; ++u) {
                const int i = rg + u * NC_RG;
                if (i < a.D) {
                    const float fk = f[r * a.D + i];
                    acc[u] = fmaf(fk, vv, acc[u]);
                    zacc[u] += fk;
                }
            }
        }
    }
    float *S = a.S + (size_t)head * a.D * a.dv;
#pragma unroll
    for (int u = 0; u < MAXR; ++u) {
        const int i = rg + u * NC_RG;
        if (i < a.D && jj < a.dv) S[(size_t)i * a.dv + jj] = acc[u];
        if (i < a.D && a.normalize && blockIdx.y == 0 && j == 0) a.z[(size_t)head * a.D + i] = zacc[u];
    }
}

template <typename T>
__global__ void __launch_bounds__(NC_THREADS) nc_out_kernel(const NcArgs a)
{
    extern __shared__ float nsm[];
    float *Ss = nsm;                          // [D][COLS] state slice
    float *zs = Ss + a.D * NC_COLS;           // [D]
    float *x = zs + a.D;                      // [TT][dk] raw q
    float *f = x + NC_TT * a.dk;              // [TT][D]  phi(q)
    const int head = blockIdx.x, t0 = blockIdx.y * NC_TT, jb = blockIdx.z * NC_COLS, tid = threadIdx.x;
    const int rows = min(NC_TT, a.L - t0);
    const T *q = (const T *)a.q + (size_t)head * a.L * a.dk;
    const float *S = a.S + (size_t)head * a.D * a.dv;
    for (int e = tid; e < a.D * NC_COLS; e += NC_THREADS) {
        const int i = e / NC_COLS, c = jb + e % NC_COLS;
        Ss[e] = c < a.dv ? S[(size_t)i * a.dv + c] : 0.f;
    }
    if (a.normalize)
        for (int i = tid; i < a.D; i += NC_THREADS) zs[i] = a.z[(size_t)head * a.D + i];
    for (int e = tid; e < rows * a.dk; e += NC_THREADS) x[e] = to_f32(q[(size_t)t0 * a.dk + e]);
    __syncthreads();
    nc_phi(a, x, f, rows);
    __syncthreads();
    // thread: token t = tid / 8, columns 4 * (tid % 8) .. + 3 of the slice
    const int t = tid / 8, c4 = 4 * (tid % 8);
    if (t >= rows) return;
    const float *fr = f + t * a.D;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f, den = 0.f;
    for (int i = 0; i < a.D; ++i) {
        const float g = fr[i];
        const float *sr = Ss + i * NC_COLS + c4;
        o0 = fmaf(g, sr[0], o0);
        o1 = fmaf(g, sr[1], o1);
        o2 = fmaf(g, sr[2], o2);
        o3 = fmaf(g, sr[3], o3);
        if (a.normalize) den = fmaf(g, zs[i], den);
    }
    const float o[4] = {o0, o1, o2, o3};
    T *out = (T *)a.out + ((size_t)head * a.L + t0 + t) * a.dv;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int c = jb + c4 + u;
        if (c < a.dv) out[c] = from_f32<T>(a.normalize ? o[u] / den : o[u]);
    }
}

}  // namespace

size_t nc_simt_workspace_bytes(int BH, int D, int dv) { return (size_t)BH * ((size_t)D * dv + D) * sizeof(float); }

bool nc_simt_supported(int D, int dk) { return D <= 256 && dk <= 512; }

// S = sum_t w_t phi(k_t) v_t^T and z = sum_t w_t phi(k_t) (w_t = 1, or gamma^(L-1-t)) of
// every head straight into S [BH][D][dv] and z [BH][D] (z may be NULL): the state a causal
// pass ends with.  One launch of the state kernel above.
int nc_state_launch(const Problem &p, float *S, float *z)
{
    if (!nc_simt_supported(p.D, p.dk)) return LA_ERR_UNSUPPORTED;
    NcArgs a;
    a.q = nullptr; a.k = p.k; a.v = p.v; a.out = nullptr;
    a.L = p.L; a.dk = p.dk; a.dv = p.dv; a.D = p.D;
    a.fm = p.fm; a.m = p.m; a.normalize = z ? 1 : 0;
    a.omega = p.omega;
    a.S = S;
    a.z = z;
    a.decay = p.decay;
    a.l2g = p.l2g;
    const size_t sm1 = sizeof(float) * ((size_t)NC_TT * p.dk + NC_TT * p.D + NC_TT * NC_COLS);
    dim3 g1((unsigned)(p.B * p.H), (unsigned)((p.dv + NC_COLS - 1) / NC_COLS));
    auto go = [&](auto k1) -> int {
        if (sm1 > 48 * 1024 &&
            cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1) != cudaSuccess)
            return LA_ERR_CUDA;
        k1<<<g1, NC_THREADS, sm1, p.stream>>>(a);
        return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
    };
    if (p.dtype == LA_BF16) return go(nc_state_kernel<__nv_bfloat16>);
    return go(nc_state_kernel<float>);
}

// state = factor * state + seg (and z alike): one step of an exclusive prefix over segments
__global__ void state_combine_kernel(float *S, float *z, const float *Sg, const float *zg, long nS, long nz,
                                     float factor)
{
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < nS + nz; i += (long)gridDim.x * blockDim.x) {
        if (i < nS)
            S[i] = factor * S[i] + Sg[i];
        else
            z[i - nS] = factor * z[i - nS] + zg[i - nS];
    }
}

int state_combine_launch(float *S, float *z, const float *Sg, const float *zg, long nS, long nz, float factor,
                         cudaStream_t st)
{
    const long n = nS + nz;
    const unsigned blocks = (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    state_combine_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(S, z, Sg, zg, nS, nz, factor);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int nc_simt_launch(const Problem &p)
{
    const int BH = p.B * p.H;
    if (!nc_simt_supported(p.D, p.dk)) return LA_ERR_UNSUPPORTED;
    if (!p.workspace || p.workspace_bytes < nc_simt_workspace_bytes(BH, p.D, p.dv)) return LA_ERR_WORKSPACE;
    NcArgs a;
    a.q = p.q; a.k = p.k; a.v = p.v; a.out = p.out;
    a.L = p.L; a.dk = p.dk; a.dv = p.dv; a.D = p.D;
    a.fm = p.fm; a.m = p.m; a.normalize = p.normalize;
    a.omega = p.omega;
    a.decay = 0;
    a.l2g = 0.f;
    a.S = (float *)p.workspace;
    a.z = a.S + (size_t)BH * p.D * p.dv;
    const size_t sm1 = sizeof(float) * ((size_t)NC_TT * p.dk + NC_TT * p.D + NC_TT * NC_COLS);
    const size_t sm2 = sizeof(float) * ((size_t)p.D * NC_COLS + p.D + NC_TT * p.dk + NC_TT * p.D);
    const unsigned ncb = (unsigned)((p.dv + NC_COLS - 1) / NC_COLS);
    dim3 g1((unsigned)BH, ncb), g2((unsigned)BH, (unsigned)((p.L + NC_TT - 1) / NC_TT), ncb);
    auto go = [&](auto k1, auto k2) -> int {
        if ((sm1 > 48 * 1024 &&
             cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1) != cudaSuccess) ||
            (sm2 > 48 * 1024 &&
             cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2) != cudaSuccess))
            return LA_ERR_CUDA;
        k1<<<g1, NC_THREADS, sm1, p.stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
        k2<<<g2, NC_THREADS, sm2, p.stream>>>(a);
        return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
    };
    if (p.dtype == LA_BF16) return go(nc_state_kernel<__nv_bfloat16>, nc_out_kernel<__nv_bfloat16>);
    return go(nc_state_kernel<float>, nc_out_kernel<float>);
}

}  // namespace la
