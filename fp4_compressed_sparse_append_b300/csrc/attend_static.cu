// csa_sparse_attend_noalloc: sparse attention whose split partials live in a
// fixed device array that belongs to the library, so the caller supplies no
// workspace and nothing is allocated on any call.
//
// Who needs this: callers whose device memory is owned by someone else - a
// host framework with its own caching allocator or a fixed arena sized at
// start-up, where a raw cudaMalloc would bypass its accounting or simply fail
// once the arena is full - and serving loops that must not pay for an
// allocation (cudaMalloc can synchronise the device) in the middle of a step.
//
// The array below is created when the library is loaded onto a GPU and stays
// there until the process exits, on every GPU that loads the library.
#include <mutex>

#include "common.cuh"
#include "csa_internal.h"

namespace {

constexpr size_t kScratchBytes = CSA_NOALLOC_SCRATCH_BYTES;

// Split partials (O, m, l) of csa_sparse_attend_noalloc.  In host code this
// name is only a stand-in for the device array: the kernels get the device
// address obtained below, never this symbol.
static __device__ __align__(256) uint8_t g_attend_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; looked up once
// per device, with that device current.
void *scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attend_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" csa_status csa_sparse_attend_noalloc(const csa_cache *cache, int32_t P, int32_t H, const uint16_t *q,
                                               float scale, const int32_t *idx, int32_t K, float *out, float *lse,
                                               csa_stream_t stream)
{
    if (!cache || !cache->codes || !cache->scales || !cache->ikeys || !cache->lengths) return CSA_ERR_INVALID_ARG;
    size_t need = 0;
    const csa_status s = csa_attend_workspace_size(cache, P, H, K, &need);
    if (s != CSA_OK) return s;
    if (need > kScratchBytes) return CSA_ERR_WORKSPACE;  // larger than the fixed array: refuse, never allocate
    void *scratch = scratch_address();
    if (!scratch) return CSA_ERR_CUDA;
    // Every slot of the partials that the merge reads is written first by the
    // split kernel, so the array needs no clearing between calls.
    return csa_sparse_attend(cache, P, H, q, scale, idx, K, out, lse, scratch, kScratchBytes, stream);
}
