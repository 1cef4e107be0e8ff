// noalloc.cu -- dsa_sparse_mla_decode_noalloc: sparse-MLA decode for callers
// that cannot allocate device memory.
//
// dsa_sparse_mla_decode needs a caller-provided workspace for the partial
// outputs of its split-K passes.  Some callers have no way to provide one:
// a host framework whose allocator has reserved (nearly) all device memory
// for its own pools and hands out no extra buffers, a plugin that only sees
// the tensors it is given, or a latency-critical loop that must not call
// cudaMalloc (which can block and synchronise the device).  This variant keeps
// that scratch in a fixed-size array in the library's own device memory
// instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds kNoAllocScratchBytes of it until the process exits.  The
// first call on a device looks up the array's device address (with that
// device current) and caches it; make that first call before capturing any
// stream.  The cached address belongs to the device's primary context: a
// cudaDeviceReset voids it, so this entry point must not be called again in a
// process that has reset the device.  All calls share the one array, so calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it; calls ordered on one stream are fine.  Nothing in the scratch needs to start at
// zero: every call overwrites every partial it later reads.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dsa.h"
#include "kernels.h"

namespace dsa {
namespace {

// Sized for DSA_NOALLOC_MAX_ROWS rows of k <= 2048 selected tokens and <= 96 heads (the
// split partial outputs, their maxima and sums, and the rows' prepared queries).
constexpr size_t kNoAllocScratchBytes = mla_workspace_bytes_for(DSA_NOALLOC_MAX_ROWS, 96, 2048);
static_assert(kNoAllocScratchBytes == 13569024, "the size the header documents");

static __device__ __align__(256) unsigned char g_mla_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_mla_scratch on the current device (looked up once per device).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mla_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" int dsa_sparse_mla_decode_noalloc(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                                             const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale,
                                             float *out, float *lse, int32_t *dev_status, void *stream) {
    // the shape checks of dsa_sparse_mla_decode first, so a bad shape gets the same status as there
    if (latent_cache == nullptr || num_rows < 0 || k < 1) return DSA_ERR_INVALID_ARG;
    if (num_heads < 16 || num_heads > 96 || num_heads % 16 != 0) return DSA_ERR_UNSUPPORTED;
    if (dsa::mla_splits(static_cast<size_t>(k)) > static_cast<size_t>(dsa::kMlaMaxSplits)) return DSA_ERR_UNSUPPORTED;
    if (num_rows > DSA_NOALLOC_MAX_ROWS) return DSA_ERR_WORKSPACE;
    const size_t need = dsa::mla_workspace_bytes(num_rows, num_heads, k);
    if (need > dsa::kNoAllocScratchBytes) return DSA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0 && num_rows > 0) {
        const int rc = dsa::scratch_address(&scratch);
        if (rc != DSA_OK) return rc;
    }
    return dsa_sparse_mla_decode(latent_cache, q, num_heads, slots, num_rows, k, sm_scale, out, lse, dev_status,
                                 scratch, need > 0 ? dsa::kNoAllocScratchBytes : 0, stream);
}
