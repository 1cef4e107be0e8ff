// api.cu -- the extern "C" entry points of libdsa declared in include/dsa.h.
//
// Each call validates its arguments on the host, encodes the TMA tensor maps
// it needs, and enqueues its kernels on the caller's stream.  Nothing here
// allocates device memory or synchronises with the device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/dsa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace dsa {

namespace {

static_assert(DSA_HIST_BINS == kHistBins, "the header and the kernels agree on the histogram size");

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D byte tensor [rows, 128 B] with a [box_rows, 128 B] box, 128-byte swizzle.
bool encode_rows128(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
    auto enc = get_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2D tensor of 4-bit values [rows, 128] with 64-byte rows (MXFP4 index keys), a [box_rows, 128]
// box landing in shared memory as 128-byte rows (each 16 values in the low 8 bytes of a 16-byte
// unit, the layout 4-bit tensor-core operands take), 128-byte swizzle.  Base: 32-byte aligned.
bool encode_fp4_rows64(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
    auto enc = get_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {64};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_rows(const dsa_rows *rows) {
    if (rows == nullptr) return DSA_ERR_INVALID_ARG;
    if (rows->num_rows < 0 || rows->max_ctx < 0 || rows->num_requests < 0) return DSA_ERR_INVALID_ARG;
    if (rows->num_rows == 0) return DSA_OK;
    if (!rows->block_table || !rows->row_req || !rows->row_ctx) return DSA_ERR_INVALID_ARG;
    const int64_t need_pages = (static_cast<int64_t>(rows->max_ctx) + DSA_PAGE_SIZE - 1) / DSA_PAGE_SIZE;
    if (rows->bt_stride < need_pages) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

}  // namespace

bool encode_rows128_map(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
    return encode_rows128(map, base, rows, box_rows);
}

int device_sm_count() {
    static int counts[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    if (counts[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        counts[dev] = n;
    }
    return counts[dev];
}

}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_version(void) { return 100; }

const char *dsa_status_string(int status) {
    switch (status) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported configuration";
        case DSA_ERR_CUDA: return "CUDA error";
        case DSA_ERR_WORKSPACE: return "workspace too small";
        case DSA_ERR_TIMEOUT: return "device wait timed out";
        case DSA_ERR_BOUNDS: return "index out of bounds in device data";
        case DSA_ERR_RANGE: return "value out of representable range";
        default: return "unknown status";
    }
}

static int indexer_common(const dsa_cache *index_cache, const dsa_rows *rows, const uint8_t *q_idx,
                          const float *head_w, float *logits, int64_t logits_stride, uint32_t *hist,
                          int32_t *dev_status, void *stream) {
    if (index_cache == nullptr) return DSA_ERR_INVALID_ARG;
    int rc = check_rows(rows);
    if (rc != DSA_OK) return rc;
    if (index_cache->page_size != DSA_PAGE_SIZE) return DSA_ERR_UNSUPPORTED;
    if (index_cache->format != DSA_KEY_FP8 && index_cache->format != DSA_KEY_MXFP4) return DSA_ERR_UNSUPPORTED;
    const bool mx = index_cache->format == DSA_KEY_MXFP4;
    const int G = rows->rows_per_group;
    if (G != 1 && G != 2 && G != 4 && G != 8) return DSA_ERR_UNSUPPORTED;
    if (rows->num_rows % G != 0) return DSA_ERR_INVALID_ARG;
    if (rows->num_rows == 0) return DSA_OK;
    if (!index_cache->base || index_cache->num_pages <= 0 || !q_idx || !head_w || !logits)
        return DSA_ERR_INVALID_ARG;
    if (!aligned(index_cache->base, mx ? 32 : 16) || !aligned(q_idx, 16)) return DSA_ERR_INVALID_ARG;
    if (logits_stride < rows->max_ctx) return DSA_ERR_INVALID_ARG;
    const uint64_t pool_rows = static_cast<uint64_t>(index_cache->num_pages) * (mx ? 68u : 66u);
    if (pool_rows >= (1ull << 31)) return DSA_ERR_UNSUPPORTED;
    const int sms = device_sm_count();
    if (sms <= 0) return DSA_ERR_CUDA;

    CUtensorMap key_map, q_map;
    if (mx ? !encode_fp4_rows64(&key_map, index_cache->base, pool_rows, DSA_PAGE_SIZE)
           : !encode_rows128(&key_map, index_cache->base, pool_rows, DSA_PAGE_SIZE))
        return DSA_ERR_CUDA;
    if (!encode_rows128(&q_map, q_idx, static_cast<uint64_t>(rows->num_rows) * DSA_INDEX_HEADS,
                        static_cast<uint32_t>(G * DSA_INDEX_HEADS)))
        return DSA_ERR_CUDA;
    IndexerArgs a;
    a.pool = static_cast<const uint8_t *>(index_cache->base);
    a.num_pages = index_cache->num_pages;
    a.block_table = rows->block_table;
    a.bt_stride = rows->bt_stride;
    a.num_requests = rows->num_requests;
    a.row_req = rows->row_req;
    a.row_ctx = rows->row_ctx;
    a.max_ctx = rows->max_ctx;
    a.head_w = head_w;
    a.logits = logits;
    a.logits_stride = logits_stride;
    a.status = dev_status;
    a.hist = hist;
    const int num_groups = rows->num_rows / G;
    for (int g0 = 0; g0 < num_groups; g0 += kIndexerMaxGroups) {
        a.group0 = g0;
        a.num_groups = num_groups - g0 < kIndexerMaxGroups ? num_groups - g0 : kIndexerMaxGroups;
        cudaError_t e = launch_indexer(key_map, q_map, a, mx, G, sms, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

int dsa_indexer_logits(const dsa_cache *index_cache, const dsa_rows *rows, const uint8_t *q_idx,
                       const float *head_w, float *logits, int64_t logits_stride, int32_t *dev_status,
                       void *stream) {
    return indexer_common(index_cache, rows, q_idx, head_w, logits, logits_stride, nullptr, dev_status, stream);
}

int dsa_indexer_logits_hist(const dsa_cache *index_cache, const dsa_rows *rows, const uint8_t *q_idx,
                            const float *head_w, float *logits, int64_t logits_stride, uint32_t *hist,
                            int32_t *dev_status, void *stream) {
    if (hist == nullptr && rows != nullptr && rows->num_rows > 0) return DSA_ERR_INVALID_ARG;
    return indexer_common(index_cache, rows, q_idx, head_w, logits, logits_stride, hist, dev_status, stream);
}

static int topk_common(const float *logits, int64_t logits_stride, const int32_t *row_ctx, int32_t num_rows,
                       int32_t max_ctx, int32_t k, uint32_t *hist, bool discard, int32_t *idx_out,
                       int32_t *dev_status, void *stream, const dsa_rows *slot_rows = nullptr,
                       int64_t pool_pages = 0, int32_t *slots_out = nullptr, const uint8_t *warm_pool = nullptr,
                       void *workspace = nullptr, size_t workspace_bytes = 0) {
    if (num_rows < 0 || max_ctx < 0) return DSA_ERR_INVALID_ARG;
    if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
    if (num_rows == 0) return DSA_OK;
    if (!logits || !row_ctx || !idx_out || logits_stride < max_ctx) return DSA_ERR_INVALID_ARG;
    TopkArgs a{logits, logits_stride, row_ctx, num_rows, max_ctx, k, idx_out, dev_status, hist, discard,
               nullptr, nullptr, 0, nullptr, 0, 0};
    if (workspace != nullptr && hist == nullptr) {
        // with a large enough workspace, few long rows take the histogram selection
        const TopkChunkPlan p = topk_chunk_plan(num_rows, max_ctx, k, device_sm_count());
        if (p.bytes > 0) {
            if (workspace_bytes < p.bytes) return DSA_ERR_WORKSPACE;
            if (!aligned(workspace, 256)) return DSA_ERR_INVALID_ARG;
            topk_chunk_bind(a, p, workspace);
        }
    }
    if (slots_out != nullptr) {
        if (slot_rows == nullptr || pool_pages <= 0) return DSA_ERR_INVALID_ARG;
        if (pool_pages * DSA_PAGE_SIZE > INT32_MAX) return DSA_ERR_UNSUPPORTED;
        a.slots_out = slots_out;
        a.block_table = slot_rows->block_table;
        a.bt_stride = slot_rows->bt_stride;
        a.row_req = slot_rows->row_req;
        a.num_requests = slot_rows->num_requests;
        a.pool_pages = pool_pages;
        a.warm_pool = warm_pool;
    }
    return launch_status(launch_topk(a, static_cast<cudaStream_t>(stream)));
}

size_t dsa_topk_workspace_size(int32_t num_rows, int32_t max_ctx, int32_t k) {
    return topk_chunk_plan(num_rows, max_ctx, k, device_sm_count()).bytes;
}

int dsa_topk_slots_warm(const float *logits, int64_t logits_stride, const dsa_rows *rows, const dsa_cache *latent_cache,
                        int32_t k, int32_t *idx_out, int32_t *slots_out, int32_t *dev_status, void *workspace,
                        size_t workspace_bytes, void *stream) {
    int rc = check_rows(rows);
    if (rc != DSA_OK) return rc;
    if (latent_cache == nullptr || latent_cache->page_size != DSA_PAGE_SIZE) return DSA_ERR_INVALID_ARG;
    if (rows->num_rows > 0 && (slots_out == nullptr || latent_cache->base == nullptr)) return DSA_ERR_INVALID_ARG;
    if (!aligned(latent_cache->base, 16)) return DSA_ERR_INVALID_ARG;
    // FP8 rows are one contiguous 576-byte run each; NVFP4 tokens are spread over a page, not warmed
    const uint8_t *warm =
        latent_cache->format == DSA_LATENT_FP8 ? static_cast<const uint8_t *>(latent_cache->base) : nullptr;
    if (latent_cache->format != DSA_LATENT_FP8 && latent_cache->format != DSA_LATENT_NVFP4) return DSA_ERR_UNSUPPORTED;
    return topk_common(logits, logits_stride, rows->row_ctx, rows->num_rows, rows->max_ctx, k, nullptr, false,
                       idx_out, dev_status, stream, rows, latent_cache->num_pages, slots_out, warm, workspace,
                       workspace_bytes);
}

int dsa_topk_slots(const float *logits, int64_t logits_stride, const dsa_rows *rows, int64_t pool_pages, int32_t k,
                   int32_t *idx_out, int32_t *slots_out, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                   void *stream) {
    int rc = check_rows(rows);
    if (rc != DSA_OK) return rc;
    if (rows->num_rows > 0 && slots_out == nullptr) return DSA_ERR_INVALID_ARG;
    return topk_common(logits, logits_stride, rows->row_ctx, rows->num_rows, rows->max_ctx, k, nullptr, false,
                       idx_out, dev_status, stream, rows, pool_pages, slots_out, nullptr, workspace, workspace_bytes);
}

int dsa_topk(const float *logits, int64_t logits_stride, const int32_t *row_ctx, int32_t num_rows,
             int32_t max_ctx, int32_t k, int32_t *idx_out, int32_t *dev_status, void *workspace,
             size_t workspace_bytes, void *stream) {
    return topk_common(logits, logits_stride, row_ctx, num_rows, max_ctx, k, nullptr, false, idx_out, dev_status,
                       stream, nullptr, 0, nullptr, nullptr, workspace, workspace_bytes);
}

int dsa_topk_hist(const float *logits, int64_t logits_stride, const int32_t *row_ctx, int32_t num_rows,
                  int32_t max_ctx, int32_t k, uint32_t *hist, int32_t *idx_out, int32_t *dev_status, void *stream) {
    if (hist == nullptr && num_rows > 0) return DSA_ERR_INVALID_ARG;
    return topk_common(logits, logits_stride, row_ctx, num_rows, max_ctx, k, hist, false, idx_out, dev_status,
                       stream);
}

// Workspace of dsa_indexer_topk: [histogram rows x DSA_HIST_BINS u32][logits rows x stride fp32],
// the logits row stride rounded up to 32 floats (128-byte rows).
static int64_t fused_logits_stride(int32_t max_ctx) { return (static_cast<int64_t>(max_ctx) + 31) / 32 * 32; }

size_t dsa_indexer_topk_workspace_size(int32_t num_rows, int32_t max_ctx) {
    if (num_rows <= 0 || max_ctx <= 0) return 0;
    return align256(static_cast<size_t>(num_rows) * DSA_HIST_BINS * 4) +
           align256(static_cast<size_t>(num_rows) * static_cast<size_t>(fused_logits_stride(max_ctx)) * 4);
}

int dsa_indexer_topk(const dsa_cache *index_cache, const dsa_rows *rows, const uint8_t *q_idx, const float *head_w,
                     int32_t k, int32_t *idx_out, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                     void *stream) {
    int rc = check_rows(rows);
    if (rc != DSA_OK) return rc;
    if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
    if (rows->num_rows == 0) return DSA_OK;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < dsa_indexer_topk_workspace_size(rows->num_rows, rows->max_ctx))
        return DSA_ERR_WORKSPACE;
    uint32_t *hist = static_cast<uint32_t *>(workspace);
    float *logits = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                              align256(static_cast<size_t>(rows->num_rows) * DSA_HIST_BINS * 4));
    const int64_t stride = fused_logits_stride(rows->max_ctx);
    rc = indexer_common(index_cache, rows, q_idx, head_w, logits, stride, hist, dev_status, stream);
    if (rc != DSA_OK) return rc;
    return topk_common(logits, stride, rows->row_ctx, rows->num_rows, rows->max_ctx, k, hist, true, idx_out,
                       dev_status, stream);
}

int dsa_page_to_slot(const dsa_rows *rows, int64_t pool_pages, const int32_t *idx, int32_t k, int32_t *slots,
                     int32_t *dev_status, void *stream) {
    int rc = check_rows(rows);
    if (rc != DSA_OK) return rc;
    if (k < 1) return DSA_ERR_INVALID_ARG;
    if (rows->num_rows == 0) return DSA_OK;
    if (!idx || !slots || pool_pages <= 0) return DSA_ERR_INVALID_ARG;
    if (pool_pages * DSA_PAGE_SIZE > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    SlotArgs a{rows->block_table, rows->bt_stride, rows->num_requests, rows->row_req, rows->row_ctx, rows->num_rows,
               rows->max_ctx, pool_pages, idx, k, slots, dev_status};
    return launch_status(launch_page_to_slot(a, static_cast<cudaStream_t>(stream)));
}

size_t dsa_sparse_mla_workspace_size(int32_t num_rows, int32_t num_heads, int32_t k) {
    if (num_rows <= 0 || num_heads <= 0 || k <= 0) return 0;
    return mla_workspace_bytes(num_rows, num_heads, k);
}


enum class MlaMode { kPrefill, kDecode, kDecodePrepareOnly, kDecodePrepared };

static int sparse_mla_common(const dsa_cache *lat, const uint16_t *q, int32_t num_heads, const int32_t *slots,
                             int32_t num_rows, int32_t k, float sm_scale, float *out, float *lse,
                             int32_t *dev_status, void *ws, size_t ws_bytes, void *stream, MlaMode mode) {
    const bool decode = mode != MlaMode::kPrefill;
    const bool prep_only = mode == MlaMode::kDecodePrepareOnly;
    if (lat == nullptr || num_rows < 0) return DSA_ERR_INVALID_ARG;
    if (lat->page_size != DSA_PAGE_SIZE) return DSA_ERR_UNSUPPORTED;
    if (lat->format != DSA_LATENT_FP8 && lat->format != DSA_LATENT_NVFP4) return DSA_ERR_UNSUPPORTED;
    if (num_heads < 16 || num_heads > 96 || num_heads % 16 != 0) return DSA_ERR_UNSUPPORTED;
    if (k < 1) return DSA_ERR_INVALID_ARG;
    if (num_rows == 0) return DSA_OK;
    if (!lat->base || lat->num_pages <= 0 || !q || (!prep_only && (!slots || !out))) return DSA_ERR_INVALID_ARG;
    if (!aligned(lat->base, 16) || !aligned(q, 16)) return DSA_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale) || !std::isfinite(lat->tensor_scale)) return DSA_ERR_INVALID_ARG;
    MlaArgs a{};
    a.pool = static_cast<const uint8_t *>(lat->base);
    a.format = lat->format;
    a.num_pages = lat->num_pages;
    a.tensor_scale = lat->tensor_scale;
    a.q = q;
    a.num_heads = num_heads;
    a.slots = slots;
    a.num_rows = num_rows;
    a.k = k;
    a.sm_scale = sm_scale;
    a.out = out;
    a.lse = lse;
    a.status = dev_status;
    a.splits = 1;
    if (decode) {
        const size_t splits = mla_splits(static_cast<size_t>(k));
        if (splits > static_cast<size_t>(kMlaMaxSplits)) return DSA_ERR_UNSUPPORTED;
        if (splits > 1) {
            const size_t need = mla_workspace_bytes(num_rows, num_heads, k);
            if (ws == nullptr || ws_bytes < need) return DSA_ERR_WORKSPACE;
            if (!aligned(ws, 256)) return DSA_ERR_INVALID_ARG;
            uint8_t *w = static_cast<uint8_t *>(ws);
            a.part_o = reinterpret_cast<uint16_t *>(w);
            w += mla_part_o_bytes(num_rows, num_heads, splits);
            a.part_ml = reinterpret_cast<float *>(w);
            w += mla_part_ml_bytes(num_rows, num_heads, splits);
            a.qprep = w;
            a.splits = static_cast<int32_t>(splits);
        }
    }
    // split decode over FP8 latents runs on the FP8 tensor cores (mla_fp8.cu); NVFP4 latents,
    // prefill and single-part decode decode the latents to fp16 (mla.cu)
    const bool fp8_decode = decode && a.splits > 1 && lat->format == DSA_LATENT_FP8;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (prep_only) return launch_status(fp8_decode ? launch_mla_qprep_fp8(a, st) : launch_mla_qprep(a, st));
    a.q_prepared = mode == MlaMode::kDecodePrepared;
    return launch_status(fp8_decode ? launch_sparse_mla_fp8_decode(a, st) : launch_sparse_mla(a, st));
}

int dsa_sparse_mla_decode(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                          const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale, float *out,
                          float *lse, int32_t *dev_status, void *workspace, size_t workspace_bytes, void *stream) {
    return sparse_mla_common(latent_cache, q, num_heads, slots, num_rows, k, sm_scale, out, lse, dev_status,
                             workspace, workspace_bytes, stream, MlaMode::kDecode);
}

int dsa_sparse_mla_decode_prepare(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                                  int32_t num_rows, int32_t k, int32_t *dev_status, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    return sparse_mla_common(latent_cache, q, num_heads, nullptr, num_rows, k, 1.0f, nullptr, nullptr, dev_status,
                             workspace, workspace_bytes, stream, MlaMode::kDecodePrepareOnly);
}

int dsa_sparse_mla_decode_prepared(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                                   const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale, float *out,
                                   float *lse, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    return sparse_mla_common(latent_cache, q, num_heads, slots, num_rows, k, sm_scale, out, lse, dev_status,
                             workspace, workspace_bytes, stream, MlaMode::kDecodePrepared);
}

int dsa_sparse_mla_prefill(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                           const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale, float *out,
                           float *lse, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                           void *stream) {
    return sparse_mla_common(latent_cache, q, num_heads, slots, num_rows, k, sm_scale, out, lse, dev_status,
                             workspace, workspace_bytes, stream, MlaMode::kPrefill);
}

int dsa_cache_insert(const dsa_cache *index_cache, const dsa_cache *latent_cache, const int32_t *slots,
                     int32_t num_tokens, const uint16_t *index_keys, const uint16_t *latents, int32_t *dev_status,
                     void *stream) {
    if (index_cache == nullptr || latent_cache == nullptr || num_tokens < 0) return DSA_ERR_INVALID_ARG;
    if (index_cache->page_size != DSA_PAGE_SIZE || latent_cache->page_size != DSA_PAGE_SIZE) return DSA_ERR_UNSUPPORTED;
    if (index_cache->format != DSA_KEY_FP8 && index_cache->format != DSA_KEY_MXFP4) return DSA_ERR_UNSUPPORTED;
    if (latent_cache->format != DSA_LATENT_FP8 && latent_cache->format != DSA_LATENT_NVFP4) return DSA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return DSA_OK;
    if (!index_cache->base || !latent_cache->base || !slots || !index_keys || !latents) return DSA_ERR_INVALID_ARG;
    if (index_cache->num_pages != latent_cache->num_pages || index_cache->num_pages <= 0) return DSA_ERR_INVALID_ARG;
    if (!aligned(index_cache->base, 16) || !aligned(latent_cache->base, 16) || !aligned(index_keys, 16) ||
        !aligned(latents, 16))
        return DSA_ERR_INVALID_ARG;
    if (!std::isfinite(latent_cache->tensor_scale) || !(latent_cache->tensor_scale > 0.f)) return DSA_ERR_INVALID_ARG;
    InsertArgs a;
    a.idx_pool = static_cast<uint8_t *>(const_cast<void *>(index_cache->base));
    a.key_fmt = index_cache->format;
    a.lat_pool = static_cast<uint8_t *>(const_cast<void *>(latent_cache->base));
    a.lat_fmt = latent_cache->format;
    a.tensor_scale = latent_cache->tensor_scale;
    a.num_pages = index_cache->num_pages;
    a.slots = slots;
    a.num_tokens = num_tokens;
    a.keys = index_keys;
    a.latents = latents;
    a.status = dev_status;
    return launch_status(launch_cache_insert(a, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ failure-path self-test

static __global__ void wait_timeout_kernel(int32_t *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);  // one arrival that never comes
        fence_mbar_init();
    }
    __syncthreads();
    // lane 0 of every warp waits: the first to reach the limit reports and raises the abort
    // flag, the others then return at once
    if ((threadIdx.x & 31) == 0) mbar_wait(&bar, 0, &abort_flag, status);
    __syncthreads();
}

int dsa_selftest_wait_timeout(int32_t *dev_status, void *stream) {
    if (dev_status == nullptr) return DSA_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
    return launch_status(cudaGetLastError());
}

// ------------------------------------------------------------------ MSA block-sparse variant

static int msa_check_rows(const dsa_rows *rows) {
    if (rows == nullptr) return DSA_ERR_INVALID_ARG;
    if (rows->num_rows < 0 || rows->max_ctx < 0 || rows->num_requests < 0) return DSA_ERR_INVALID_ARG;
    if (rows->num_rows == 0) return DSA_OK;
    if (!rows->block_table || !rows->row_req || !rows->row_ctx) return DSA_ERR_INVALID_ARG;
    const int64_t need_pages = (static_cast<int64_t>(rows->max_ctx) + DSA_MSA_PAGE - 1) / DSA_MSA_PAGE;
    if (rows->bt_stride < need_pages) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

int dsa_msa_block_scores(const void *index_pool, int64_t num_pages, const dsa_rows *rows, const uint8_t *q_idx,
                         float *scores, int64_t score_stride, int32_t *dev_status, void *stream) {
    int rc = msa_check_rows(rows);
    if (rc != DSA_OK || rows->num_rows == 0) return rc;
    const int G = rows->rows_per_group;
    if (G != 1 && G != 2 && G != 4 && G != 8) return DSA_ERR_UNSUPPORTED;
    if (rows->num_rows % G != 0) return DSA_ERR_INVALID_ARG;
    if (!index_pool || num_pages <= 0 || !q_idx || !scores) return DSA_ERR_INVALID_ARG;
    if (!aligned(index_pool, 16) || !aligned(q_idx, 16)) return DSA_ERR_INVALID_ARG;
    const int64_t max_blocks = (static_cast<int64_t>(rows->max_ctx) + DSA_MSA_PAGE - 1) / DSA_MSA_PAGE;
    if (score_stride < max_blocks) return DSA_ERR_INVALID_ARG;
    const uint64_t pool_rows = static_cast<uint64_t>(num_pages) * DSA_MSA_PAGE;
    if (pool_rows >= (1ull << 31)) return DSA_ERR_UNSUPPORTED;
    const int sms = device_sm_count();
    if (sms <= 0) return DSA_ERR_CUDA;
    CUtensorMap key_map, q_map;
    const uint32_t q_box = static_cast<uint32_t>(G * DSA_MSA_GROUPS < 16 ? 16 : G * DSA_MSA_GROUPS);
    if (!encode_rows128(&key_map, index_pool, pool_rows, DSA_MSA_PAGE)) return DSA_ERR_CUDA;
    if (!encode_rows128(&q_map, q_idx, static_cast<uint64_t>(rows->num_rows) * DSA_MSA_GROUPS, q_box))
        return DSA_ERR_CUDA;
    const int num_groups = rows->num_rows / G;
    // pages per CTA: two CTAs per SM cover the rows' pages in about one wave (4..64 pages each)
    const int64_t total_pages = static_cast<int64_t>(num_groups) * (max_blocks > 0 ? max_blocks : 1);
    int64_t cp = (total_pages + 2 * sms - 1) / (2 * sms);
    cp = cp < 4 ? 4 : (cp > 64 ? 64 : cp);
    MsaScoreArgs a;
    a.num_pages = num_pages;
    a.block_table = rows->block_table;
    a.bt_stride = rows->bt_stride;
    a.num_requests = rows->num_requests;
    a.row_req = rows->row_req;
    a.row_ctx = rows->row_ctx;
    a.max_ctx = rows->max_ctx;
    a.chunk_pages = static_cast<int32_t>(cp);
    a.chunks = static_cast<int32_t>(max_blocks > 0 ? (max_blocks + cp - 1) / cp : 1);
    a.scores = scores;
    a.score_stride = score_stride;
    a.status = dev_status;
    return launch_status(launch_msa_scores(key_map, q_map, a, num_groups, G, static_cast<cudaStream_t>(stream)));
}

int dsa_msa_select(const float *scores, int64_t score_stride, const int32_t *row_ctx, int32_t num_rows,
                   int32_t max_ctx, int32_t *blocks, int32_t *dev_status, void *stream) {
    if (num_rows < 0 || max_ctx < 0) return DSA_ERR_INVALID_ARG;
    if (num_rows == 0) return DSA_OK;
    if (!scores || !row_ctx || !blocks) return DSA_ERR_INVALID_ARG;
    const int64_t max_blocks = (static_cast<int64_t>(max_ctx) + DSA_MSA_PAGE - 1) / DSA_MSA_PAGE;
    if (score_stride < max_blocks) return DSA_ERR_INVALID_ARG;
    if (max_blocks > 16384) return DSA_ERR_UNSUPPORTED;  // candidate keys live in shared memory
    MsaSelectArgs a;
    a.scores = scores;
    a.score_stride = score_stride;
    a.row_ctx = row_ctx;
    a.max_ctx = max_ctx;
    a.blocks = blocks;
    a.status = dev_status;
    return launch_status(launch_msa_select(a, num_rows, static_cast<cudaStream_t>(stream)));
}

size_t dsa_msa_attention_workspace_size(int32_t num_rows, int32_t heads_per_group) {
    if (num_rows <= 0 || heads_per_group <= 0) return 0;
    return msa_attention_workspace_bytes(static_cast<size_t>(num_rows), static_cast<size_t>(heads_per_group));
}

int dsa_msa_attention(const void *kv_pool, int64_t num_pages, float k_scale, float v_scale, const dsa_rows *rows,
                      const uint8_t *q, float q_scale, int32_t heads_per_group, const int32_t *blocks, float sm_scale,
                      float *out, float *lse, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                      void *stream) {
    int rc = msa_check_rows(rows);
    if (rc != DSA_OK || rows->num_rows == 0) return rc;
    const int hpg = heads_per_group;
    if (hpg < 16 || hpg > DSA_MSA_MAX_HPG || hpg % 16 != 0) return DSA_ERR_UNSUPPORTED;
    if (!kv_pool || num_pages <= 0 || !q || !blocks || !out) return DSA_ERR_INVALID_ARG;
    if (!aligned(kv_pool, 16) || !aligned(q, 16)) return DSA_ERR_INVALID_ARG;
    for (float v : {k_scale, v_scale, q_scale, sm_scale})
        if (!std::isfinite(v) || !(v > 0.f)) return DSA_ERR_INVALID_ARG;
    const size_t need = msa_attention_workspace_bytes(static_cast<size_t>(rows->num_rows), static_cast<size_t>(hpg));
    if (workspace == nullptr || workspace_bytes < need) return DSA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return DSA_ERR_INVALID_ARG;
    const uint64_t kv_rows = static_cast<uint64_t>(num_pages) * DSA_MSA_GROUPS * 2 * DSA_MSA_PAGE;
    if (kv_rows >= (1ull << 31)) return DSA_ERR_UNSUPPORTED;
    CUtensorMap kv_map, q_map;
    if (!encode_rows128(&kv_map, kv_pool, kv_rows, DSA_MSA_PAGE)) return DSA_ERR_CUDA;
    if (!encode_rows128(&q_map, q, static_cast<uint64_t>(rows->num_rows) * DSA_MSA_GROUPS * hpg,
                        static_cast<uint32_t>(hpg)))
        return DSA_ERR_CUDA;
    const size_t parts = static_cast<size_t>(rows->num_rows) * DSA_MSA_GROUPS * DSA_MSA_BLOCKS * hpg;
    MsaAttnArgs a;
    a.num_pages = num_pages;
    a.block_table = rows->block_table;
    a.bt_stride = rows->bt_stride;
    a.num_requests = rows->num_requests;
    a.row_req = rows->row_req;
    a.row_ctx = rows->row_ctx;
    a.max_ctx = rows->max_ctx;
    a.heads_per_group = hpg;
    a.blocks = blocks;
    a.s_scale = static_cast<float>(static_cast<double>(sm_scale) * q_scale * k_scale * 1.4426950408889634);
    a.v_scale = v_scale;
    a.part_o = static_cast<float *>(workspace);
    a.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                          (parts * DSA_MSA_DIM * sizeof(float) + 255) / 256 * 256);
    a.out = out;
    a.lse = lse;
    a.status = dev_status;
    return launch_status(launch_msa_attention(kv_map, q_map, a, rows->num_rows, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
