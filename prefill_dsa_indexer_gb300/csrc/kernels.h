// kernels.h -- launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Internal to libdsa.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

// Launch `kern` on `s` with programmatic stream serialization: its CTAs may start while the
// previous kernel of the stream finishes; the kernel does on-chip set-up only, then pdl_wait()
// before touching global memory.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}


struct IndexerArgs {
    const uint8_t *pool;        // index pool base
    int64_t num_pages;
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t num_requests;
    const int32_t *row_req;
    const int32_t *row_ctx;
    int32_t max_ctx;
    int32_t group0;             // first group of this launch
    int32_t num_groups;         // groups in this launch (<= kIndexerMaxGroups)
    const float *head_w;
    float *logits;
    int64_t logits_stride;
    int32_t *status;
    uint32_t *hist;             // optional [rows][kHistBins]: each written logit adds 1 at its key's top 16 bits
};

constexpr int kIndexerMaxGroups = 1024;

// Per-row histogram shared by the scorer and the top-k: 65,536 bins of the top 16 bits of the
// order-preserving key of each logit.
constexpr int kHistBins = 65536;

// Order-preserving map fp32 -> uint32 (a larger float gives a larger key); -0 folds onto +0
// and NaN maps to 0, below every number.  The scorer and the top-k must agree on it exactly.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f != f) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Launch the indexer for groups of `rows_per_group` rows.  key_map: FP8 keys, the pool as a byte
// tensor [pages * 66, 128]; MXFP4 keys, the pool as 4-bit values [pages * 68, 128] (64-byte rows).
cudaError_t launch_indexer(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a,
                           bool mxfp4_keys, int rows_per_group, int num_sms, cudaStream_t s);

struct TopkArgs {
    const float *logits;
    int64_t logits_stride;
    const int32_t *row_ctx;
    int32_t num_rows;
    int32_t max_ctx;
    int32_t k;
    int32_t *idx_out;
    int32_t *status;
    uint32_t *hist;             // optional: the scorer's histogram of exactly these logits (read, left zeroed)
    bool discard_logits;        // the logits are library scratch: drop their L2 lines once read
    // optional page -> slot translation of the selection (slots_out == nullptr: none)
    int32_t *slots_out;         // [num_rows, k]: block_table[row_req[r]][t / 64] * 64 + t % 64, -1 padded
    const int32_t *block_table;
    int64_t bt_stride;
    const int32_t *row_req;
    int32_t num_requests;
    int64_t pool_pages;
    // optional: FP8 latent pool whose selected rows (576 B per slot) are prefetched into L2 as
    // the slots are written, so the attention that follows gathers from L2
    const uint8_t *warm_pool;
    // optional histogram selection (chunks > 0; see topk_chunk_plan and topk_chunk_bind), in a caller
    // workspace
    uint32_t *hs_list;   // [rows][chunks][4096] each chunk's nonzero bins, ascending: bin << 20 | count
    uint32_t *hs_nlist;  // [rows][chunks] their numbers
    uint32_t *hs_key;    // [rows][row_cap] the row's keys in bins >= the threshold bin, position order
    int32_t *hs_pos;     // [rows][row_cap] their positions
    uint32_t *hs_chunk;  // [rows][chunks][2] each chunk's offset and count in hs_key
    uint32_t *hs_row;    // [rows][4] the threshold bin, the keys above it, the keys in it
    int32_t chunks, chunk_len, row_cap;
};

cudaError_t launch_topk(const TopkArgs &a, cudaStream_t s);

// Histogram selection of few long rows: limits, the plan for a batch (bytes == 0: not used) and the
// binding of a workspace of plan.bytes to the arguments.  Its three launches of independent CTAs
// beat the cluster selection once rows are longer than a cluster keeps in shared memory; measured
// on a GB300 per step: 256K keys 90.0 vs 102.1 us, 1M keys 76.6 vs 93.5 us; at 128K keys the two are
// even (61.2-61.4 us each, measured back to back on one GPU), and the cluster path needs no workspace.
constexpr int kChunkedMaxRows = 64;
constexpr int kChunkedMinCtx = 131072;
constexpr int kChunkMinKeys = 2048;
constexpr int kChunkedMaxChunks = 96;
constexpr int kChunkMaxKeys = 16384;
constexpr int kHsInCap = 12288;  // keys of a row's threshold bin the select kernel holds
struct TopkChunkPlan {
    int32_t chunks, chunk_len, row_cap;
    size_t bytes;
};
TopkChunkPlan topk_chunk_plan(int32_t num_rows, int32_t max_ctx, int32_t k, int sms);
void topk_chunk_bind(TopkArgs &a, const TopkChunkPlan &p, void *workspace);

struct SlotArgs {
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t num_requests;
    const int32_t *row_req;
    const int32_t *row_ctx;
    int32_t num_rows;
    int32_t max_ctx;
    int64_t pool_pages;
    const int32_t *idx;
    int32_t k;
    int32_t *slots;
    int32_t *status;
};

cudaError_t launch_page_to_slot(const SlotArgs &a, cudaStream_t s);

struct MlaArgs {
    const uint8_t *pool;
    int32_t format;
    int64_t num_pages;
    float tensor_scale;
    const uint16_t *q;
    int32_t num_heads;
    const int32_t *slots;
    int32_t num_rows;
    int32_t k;
    float sm_scale;
    float *out;
    float *lse;
    int32_t *status;
    uint16_t *part_o;   // decode: [R, splits, H, 512] fp16 partial outputs (normalised by their own sum)
    float *part_ml;     // decode: [R, splits, H, 2] running max (log2 units) and sum
    uint8_t *qprep;     // decode: per row (mla_qprep_row_bytes(H) apart) the query image laid out as the
                        // kernel's operand: fp16 [9 x H x 128 B] (NVFP4 latents), or e4m3 hi x 4, lo x 4,
                        // RoPE hi|lo blocks [9 x H x 128 B] then H fp32 factors 2^-e_h (FP8 latents)
    int32_t splits;     // 1 = write the final output directly
    bool q_prepared;    // decode: the query images are already in qprep (no prep launch)
};

// ---- MSA block-sparse variant (msa.cu)
struct MsaScoreArgs {
    int64_t num_pages;
    const int32_t *block_table;  // 128-token pages
    int64_t bt_stride;
    int32_t num_requests;
    const int32_t *row_req;
    const int32_t *row_ctx;
    int32_t max_ctx;
    int32_t chunks;       // CTAs per row group
    int32_t chunk_pages;  // pages per CTA
    float *scores;        // [R, 4, score_stride]
    int64_t score_stride;
    int32_t *status;
};

struct MsaSelectArgs {
    const float *scores;
    int64_t score_stride;
    const int32_t *row_ctx;
    int32_t max_ctx;
    int32_t *blocks;  // [R, 4, 16]
    int32_t *status;
};

struct MsaAttnArgs {
    int64_t num_pages;
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t num_requests;
    const int32_t *row_req;
    const int32_t *row_ctx;
    int32_t max_ctx;
    int32_t heads_per_group;
    const int32_t *blocks;
    float s_scale;   // sm_scale * q_scale * k_scale * log2(e)
    float v_scale;
    float *part_o;   // [R, 4, 16, hpg, 128] normalised block parts
    float *part_ml;  // [R, 4, 16, hpg, 2] (max in log2 units, sum)
    float *out;
    float *lse;
    int32_t *status;
};

cudaError_t launch_msa_scores(const CUtensorMap &key_map, const CUtensorMap &q_map, const MsaScoreArgs &a,
                              int num_groups, int rows_per_group, cudaStream_t s);
cudaError_t launch_msa_select(const MsaSelectArgs &a, int num_rows, cudaStream_t s);
cudaError_t launch_msa_attention(const CUtensorMap &kv_map, const CUtensorMap &q_map, const MsaAttnArgs &a,
                                 int num_rows, cudaStream_t s);
size_t msa_attention_workspace_bytes(size_t num_rows, size_t heads_per_group);

// 2D byte tensor [rows, 128 B] with a [box_rows, 128 B] box, 128-byte swizzle (api.cu).
bool encode_rows128_map(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows);

// Decode query preparation alone (bf16 query -> the fp16 operand images in a.qprep).
cudaError_t launch_mla_qprep(const MlaArgs &a, cudaStream_t s);

// Merge of a decode's split partials (a.part_o, a.part_ml) into a.out / a.lse.
cudaError_t launch_mla_combine(const MlaArgs &a, cudaStream_t s);

// FP8-latent decode on FP8 tensor cores (mla_fp8.cu): query preparation alone, and the whole call
// (preparation unless a.q_prepared, one CTA per 128-token part, merge).  Needs a.splits >= 2.
cudaError_t launch_mla_qprep_fp8(const MlaArgs &a, cudaStream_t s);
cudaError_t launch_sparse_mla_fp8_decode(const MlaArgs &a, cudaStream_t s);

// Decode splits every row's selected tokens into parts of this many tokens (fixed, so a row's
// result does not depend on the batch), merged by log-sum-exp.
constexpr int kMlaTokensPerSplit = 128;
constexpr int kMlaMaxSplits = 16;

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t mla_part_o_bytes(size_t R, size_t H, size_t S) { return align256(R * S * H * 512 * 2); }
constexpr size_t mla_part_ml_bytes(size_t R, size_t H, size_t S) { return align256(R * S * H * 2 * 4); }
__host__ __device__ constexpr size_t mla_qprep_row_bytes(size_t H) { return 9 * H * 128 + 4 * H; }
constexpr size_t mla_qprep_bytes(size_t R, size_t H) { return align256(R * mla_qprep_row_bytes(H)); }
constexpr size_t mla_splits(size_t k) { return (k + kMlaTokensPerSplit - 1) / kMlaTokensPerSplit; }
constexpr size_t mla_workspace_bytes_for(size_t R, size_t H, size_t k) {
    return mla_splits(k) <= 1 ? 0
                               : mla_part_o_bytes(R, H, mla_splits(k)) + mla_part_ml_bytes(R, H, mla_splits(k)) +
                                     mla_qprep_bytes(R, H);
}

cudaError_t launch_sparse_mla(const MlaArgs &a, cudaStream_t s);

size_t mla_workspace_bytes(int32_t num_rows, int32_t num_heads, int32_t k);

struct InsertArgs {
    uint8_t *idx_pool;
    int32_t key_fmt;
    uint8_t *lat_pool;
    int32_t lat_fmt;
    float tensor_scale;
    int64_t num_pages;
    const int32_t *slots;
    int32_t num_tokens;
    const uint16_t *keys;     // [n, 128] bf16 bits
    const uint16_t *latents;  // [n, 576] bf16 bits
    int32_t *status;
};

cudaError_t launch_cache_insert(const InsertArgs &a, cudaStream_t s);

int device_sm_count();

}  // namespace dsa
