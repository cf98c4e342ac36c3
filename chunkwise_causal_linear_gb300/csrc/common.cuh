// common.cuh -- small helpers shared by the kernels of liblachunked (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "la_chunked.h"

namespace la {

// ---- storage <-> fp32 ---------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// ---- feature maps applied to one fp32 value ------------------------------------------
// elu(x) + 1 = x + 1 for x >= 0, e^x below ("Linear Attention / Performerの理論と実装",
// ELU feature map).
__device__ __forceinline__ float phi_elu1(float x) { return x >= 0.f ? x + 1.f : expf(x); }

// ---- Fenwick level of (t, s), s <= t: 0 if equal, else 1 + floor(log2(t ^ s)) ------
__device__ __forceinline__ int fenwick_level(int t, int s)
{
    return (t == s) ? 0 : 1 + (31 - __clz(t ^ s));
}

// ---- device error word ----------------------------------------------------------------
// Kernels receive a pointer to the library's error word and record the first failure.
__device__ __forceinline__ void record_error(int *err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

// Per-problem description handed from the host plan to a kernel launcher.
struct Problem {
    const void *q, *k, *v;
    void *out;
    int B, H, L, dk, dv, C;  // C already clamped to [1, L]
    int D;                   // feature dimension (dk, or m for FAVOR+)
    int fm;                  // enum la_fm_kind
    int m;
    const float *omega;
    int normalize;
    const float *lam;        // NULL or [B, H, L, nl]
    int nl;
    int dtype;               // enum la_dtype
    void *workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
    int *err;                // device error word
    int decay;               // 1: Retention decay S_t = gamma S_{t-1} + phi(k_t) v_t^T
    float gamma;             // decay factor, 0 < gamma <= 1
    float l2g;               // log2(gamma), rounded from the double value
    int rev;                 // 1: anti-causal: row t reads the rows s >= t, computed as the
                             // causal pass over the reversed sequence (generic path; the
                             // tensor-core path for identity features, no normaliser, C = 64)
    int out_f32;             // 1: out is fp32 rows (tensor-core path, identity features, no
                             // normaliser; the backward pass's internal passes)
    const float *S0, *z0;    // NULL, or the state (and normaliser) before row 0: fp32
                             // [B*H][D][dv] and [B*H][D] (the decoding state's layout)
    // The backward pass's internal passes on the tensor-core path (identity features, no
    // normaliser, no decay):
    int esyn;                // 1: q and k are the constant rows e = (1, 0, ..., 0), dk = 64;
                             // q, k are not read
};

// Host-side queries used by the planner.
int required_levels(int L);
bool is_pow2(int x);
int ilog2(int x);

}  // namespace la
