// noalloc.cu -- la_chunked_fwd_noalloc: the forward pass for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain device scratch: code that runs inside an allocator or
// a memory-pool callback, plugins whose host application owns every device allocation and
// exposes no allocation hook, or real-time loops where any cudaMalloc / cudaFree (with its
// implicit synchronisation) is forbidden.  The main entry point takes its workspace from
// the caller; this one takes it from a fixed array that lives in the library image, so it
// never allocates.
//
// Every plan with a nonzero la_chunked_workspace_bytes takes its scratch from the array:
//   - the tensor-core paths when they cut a sequence into segments (few heads: any feature
//     map and chunk size), for the fp32 segment totals S and z;
//   - the log-linear mask: the per-level fp32 chunk states of the generic path, and the
//     segment totals and running-state snapshots of the tensor-core path.
// Each call writes every scratch word it later reads (the totals launch writes the totals
// before the main launch reads them; the generic kernel zeroes its level states first), so
// nothing left over from an earlier call is ever read.
#include <mutex>

#include "common.cuh"

namespace {

// Fixed scratch, 8 MiB: enough for, e.g., the log-linear mask over 16 heads at L = 65,536,
// d = 64, C = 64, or the fp32 totals of 127 segments of d = 128 heads (66 KB each).  Every GPU that loads the library holds it until
// the process exits.
constexpr size_t kScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char la_noalloc_scratch[kScratchBytes];

// In host code `la_noalloc_scratch` only names the symbol; its device address is looked up
// once per device (with that device current) and cached here.  cudaDeviceReset destroys the
// context that address belongs to, so calls after a reset of that device are not supported.
std::mutex g_mu;
void *g_scratch[64] = {nullptr};

int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, la_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return LA_OK;
}

}  // namespace

extern "C" int la_chunked_fwd_noalloc(const void *q, const void *k, const void *v, void *out,
                                      int B, int H, int L, int dk, int dv, int C,
                                      const la_feature_map *feature_map, int normalize,
                                      const float *level_weights, int num_levels, int dtype,
                                      void *stream)
{
    if (!q || !k || !v || !out) return LA_ERR_NULL;
    const size_t need = la_chunked_workspace_bytes(B, H, L, dk, dv, C, feature_map, normalize,
                                                   level_weights ? num_levels : 0, dtype);
    if (need > kScratchBytes) return LA_ERR_SCRATCH_LIMIT;
    void *ws = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&ws);
        if (rc != LA_OK) return rc;
    }
    return la_chunked_fwd(q, k, v, out, B, H, L, dk, dv, C, feature_map, normalize,
                          level_weights, num_levels, dtype, ws, need > 0 ? kScratchBytes : 0,
                          stream);
}
