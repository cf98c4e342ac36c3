// tc_common.cuh -- pieces shared by the tensor-core kernels: bounded mbarrier waits with
// an abort flag, bf16 unpacking, and the host-side TMA tensor-map encoding.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace la {
namespace tcc {

using namespace ptx;

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
    for (;;) {
        // sleeps (up to 0.2 ms) until the phase completes; no busy probing
        if (mbar_try_sleep(bar, parity, 200000u)) return true;
        if (*ctl.abort) return false;
        if (globaltimer() - t0 > ctl.timeout_ns) {
            *ctl.abort = 1;
            record_error(ctl.err, LA_ERR_TIMEOUT);
            return false;
        }
    }
}

// Group wait: only the group's leader polls the mbarrier(s); the others park on the
// hardware named barrier, which also hands every thread the same decision.  The leader's
// acquire plus the barrier order the other threads' later reads after the awaited writes.
__device__ __forceinline__ bool group_wait(bool leader, int bar_id, uint64_t *b1, uint32_t p1,
                                           uint64_t *b2, uint32_t p2, bool use2, const Ctl &ctl,
                                           int nthreads = 128)
{
    bool ok = true;
    if (leader) {
        ok = wait_phase(b1, p1, ctl);
        if (ok && use2) ok = wait_phase(b2, p2, ctl);
    }
    return named_bar_and(bar_id, nthreads, ok);
}

// Programmatic dependent launch.  A pass that produces segment totals lets the pass that
// reads them be scheduled early (its CTAs start their set-up on free SMs as soon as every
// producer CTA has signalled); the reader waits for the producer grid to complete, with its
// memory visible, before it touches the totals.  Both are no-ops for a launch without the
// attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// bf16 (raw 16-bit) -> fp32 for the two halves of a 32-bit word
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---- host side ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn()
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
inline bool make_map(CUtensorMap *m, const void *ptr, int BH, int L, int d, int C)
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

// fp32 rows [BH][L][d]: boxes of 32 columns (128 bytes) x C rows, 128-byte swizzle
inline bool make_map_f32(CUtensorMap *m, const void *ptr, int BH, int L, int d, int C)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)L * d * 4};
    cuuint32_t box[3] = {32, (cuuint32_t)C, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches `kern` on `stream` with programmatic stream serialization: it may start while the
// kernel before it in the stream is still running, and must call pdl_wait() before reading
// what that kernel writes.
template <typename Kern, typename Args>
inline cudaError_t launch_dependent(Kern kern, int grid, int block, int smem, cudaStream_t stream,
                                    const Args &args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

// Segments per head for a sequence of `tiles` 64-row tiles: split when the heads alone leave
// most SMs idle, keeping at least `min_tiles` tiles per segment.
inline int split_segments(int BH, int tiles, int num_sms, int min_tiles, int *seg_tiles)
{
    int g = 1;
    if (BH < num_sms / 2) g = max(1, min(num_sms / BH, tiles / min_tiles));
    const int st = (tiles + g - 1) / g;
    if (seg_tiles) *seg_tiles = st;
    return (tiles + st - 1) / st;
}

}  // namespace tcc
}  // namespace la
