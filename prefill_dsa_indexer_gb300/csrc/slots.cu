// slots.cu -- logical token positions -> physical cache slots.
//
// vLLM blog "Day-0 support for Kimi K3.1 Pro", section "One KV cache, three
// states": before each step the block table and cache slots are translated
// to the kernel's page addresses.  Here: slot = block_table[req][t / 64] * 64
// + t % 64, so the attention kernel addresses a latent row as
// base + slot * row_bytes (pages of one pool are contiguous).
#include "kernels.h"
#include "ptx.cuh"

namespace dsa {

namespace {

__global__ void page_to_slot_kernel(const SlotArgs a) {
    const int64_t total = static_cast<int64_t>(a.num_rows) * a.k;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(e / a.k);
        const int32_t t = a.idx[e];
        int32_t slot = -1;
        if (t >= 0) {
            const int32_t req = a.row_req[r];
            const int32_t ctx = a.row_ctx[r];
            if (req < 0 || req >= a.num_requests || t >= ctx || t >= a.max_ctx) {
                report(a.status, DSA_ERR_BOUNDS);
            } else {
                const int32_t page = a.block_table[static_cast<int64_t>(req) * a.bt_stride + t / DSA_PAGE_SIZE];
                if (page < 0 || page >= a.pool_pages) report(a.status, DSA_ERR_BOUNDS);
                else slot = page * DSA_PAGE_SIZE + t % DSA_PAGE_SIZE;
            }
        }
        a.slots[e] = slot;
    }
}

}  // namespace

cudaError_t launch_page_to_slot(const SlotArgs &a, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(a.num_rows) * a.k;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    page_to_slot_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dsa
