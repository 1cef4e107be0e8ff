/*
 * dsa.h -- C ABI of libdsa, a single-GPU (sm_103a) implementation of the
 * DeepSeek-style sparse attention (DSA) layer as used in Kimi K3.1 Pro.
 *
 * The layer (vLLM blog "Day-0 support for Kimi K3.1 Pro", section "Sparse
 * attention in K3.1 Pro", Fig. 1): for every query row a small indexer with
 * 32 FP8 heads scores every earlier token against that token's FP8 index key
 * (132 B with its scale); a top-k step keeps the 2,048 best tokens; exact
 * absorbed-MLA attention of 96 query heads then runs over only those tokens'
 * 576-byte latents (512 latent + 64 RoPE dims).  Both caches are paged and
 * are read through a block table that is translated to physical slots
 * before the attention step (section "One KV cache, three states"; in the
 * fused decode path the scorer and the top-k hand attention the physical
 * cache rows to read, section "Low-latency decode: fused DSA decode path").
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     its comment says "host".  Struct arguments themselves are host memory
 *     and are read only during the call.  The library allocates no device
 *     memory and keeps no state between calls (per-device tensor-map encoder
 *     lookup aside).
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Every call only enqueues work and returns; nothing
 *     synchronises with the host.
 *   - The int return value is a host-side status: arguments are checked
 *     before anything is launched, and a launch error is reported as
 *     DSA_ERR_CUDA.  No exceptions cross the boundary.
 *   - Errors the kernels find in device data (a page id outside the pool, a
 *     context longer than max_ctx, a timed-out wait) are written to the
 *     optional `dev_status` word (int32, device memory): the first error
 *     code is kept (compare-and-swap from 0), later ones are dropped.  The
 *     caller zeroes it before the calls and reads it after synchronising.
 *     Outputs of a call that reported a device error are unspecified.
 *   - Results are deterministic, and a row's results do not depend on the
 *     other rows of the batch (batch invariance).
 *
 * Cache page layouts (page_size 64; the per-token widths are the blog's,
 * "One KV cache, three states": index key 132 B FP8 / 68 B MXFP4, latent
 * 576 B FP8 / 352 B NVFP4; the arrangement within a page is this library's):
 *   DSA_KEY_FP8      [64 x 128 B e4m3 key][64 x fp32 per-token scale]   8448 B
 *   DSA_KEY_MXFP4    [64 x 64 B e2m1 pairs][64 x 4 B e8m0, one per 32]  4352 B
 *   DSA_LATENT_FP8   [64 x 576 B e4m3], scale = dsa_cache.tensor_scale 36864 B
 *   DSA_LATENT_NVFP4 [64 x 256 B e2m1 pairs][64 x 32 B e4m3 scale, one per 16]
 *                    [64 x 64 B e4m3 RoPE dims, scale = tensor_scale]   22528 B
 * e2m1 pairs hold element 2j in the low nibble.  Token t of a request lives
 * in page block_table[req][t / 64], row t % 64; its physical slot is
 * page * 64 + t % 64, the same slot id in the index and the latent pool.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes */
#define DSA_OK 0
#define DSA_ERR_INVALID_ARG (-1)  /* host: null pointer, bad size or stride */
#define DSA_ERR_UNSUPPORTED (-2)  /* host: format, page size, head count or k not supported */
#define DSA_ERR_CUDA (-3)         /* host: a CUDA call or launch failed */
#define DSA_ERR_WORKSPACE (-4)    /* host: workspace smaller than dsa_*_workspace_size() */
#define DSA_ERR_TIMEOUT (-5)      /* device: a bounded wait inside a kernel gave up */
#define DSA_ERR_BOUNDS (-6)       /* device: page id, slot or context outside its range */
#define DSA_ERR_RANGE (-7)        /* device: a value the kernel cannot represent (e.g. |q| > 65504) */

/* ---- cache formats */
#define DSA_KEY_FP8 1
#define DSA_KEY_MXFP4 2
#define DSA_LATENT_FP8 3
#define DSA_LATENT_NVFP4 4

/* ---- fixed dimensions of the layer */
#define DSA_PAGE_SIZE 64
#define DSA_INDEX_HEADS 32
#define DSA_INDEX_DIM 128
#define DSA_LATENT_DIM 576 /* 512 latent + 64 RoPE dims */
#define DSA_VALUE_DIM 512
#define DSA_MAX_HEADS 128  /* MLA query heads per row, multiple of 16 */
#define DSA_MAX_TOPK 2048

/* One paged cache pool (index keys or latents). */
typedef struct dsa_cache {
    const void *base;     /* device, num_pages * page bytes, 16-byte aligned (DSA_KEY_MXFP4: 32-byte
                             aligned, the rule of the 4-bit tensor copies; else DSA_ERR_INVALID_ARG) */
    int32_t format;       /* DSA_KEY_* for an index pool, DSA_LATENT_* for a latent pool */
    int32_t page_size;    /* must be DSA_PAGE_SIZE */
    int64_t num_pages;
    float tensor_scale;   /* latent pools: per-tensor scale of the e4m3 codes; ignored for index pools */
} dsa_cache;

/* Query rows and their addressing. */
typedef struct dsa_rows {
    const int32_t *block_table; /* device [num_requests, bt_stride] physical page ids */
    int64_t bt_stride;          /* entries per request, >= ceil(max_ctx / 64) */
    int32_t num_requests;       /* rows of block_table; row_req outside [0, num_requests) is DSA_ERR_BOUNDS */
    const int32_t *row_req;     /* device [num_rows] request of each row */
    const int32_t *row_ctx;     /* device [num_rows] visible tokens L_r (positions 0..L_r-1, incl. itself) */
    int32_t num_rows;
    int32_t max_ctx;            /* host bound on every row_ctx; larger values are DSA_ERR_BOUNDS */
    int32_t rows_per_group;     /* 1, 2, 4 or 8: consecutive rows of one request that the indexer
                                   scores against one read of the keys (speculative-verify rows,
                                   prefill query blocks); num_rows must be a multiple of it */
} dsa_rows;

/*
 * Indexer logits (blog section "Sparse attention in K3.1 Pro"; the weighted,
 * fp32-accumulated reduction across heads is the AMD section "Quantization:
 * native MXFP4 indexer"; the query carries no scale because the head
 * weights are folded into its quantisation, section "Low-latency decode:
 * fused DSA decode path"):
 *
 *   logits[r * logits_stride + t] = sum_{h<32} head_w[r,h] * max(0, s_t * <q_idx[r,h,:], k_t>)
 *   for 0 <= t < row_ctx[r]
 *
 * k_t is token t's decoded key (e4m3 codes with s_t its fp32 scale, or
 * MXFP4 e2m1 * 2^(e8m0-127) with s_t = 1).  q_idx: [num_rows, 32, 128] e4m3
 * codes (16-byte aligned); head_w: [num_rows, 32] fp32; logits: fp32 with
 * row stride logits_stride >= max_ctx.  Entries at t >= row_ctx[r] are not
 * written.  Products are exact and accumulate in fp32 on the tensor cores,
 * so a logit differs from an exact evaluation by accumulation rounding only.
 * MXFP4 keys multiply their e2m1 codes by the block scales inside the MMA
 * (block-scaled e2m1 x e4m3); a visible key with the e8m0 NaN code 0xff is
 * DSA_ERR_RANGE (its logits are then unspecified).
 */
int dsa_indexer_logits(const dsa_cache *index_cache, const dsa_rows *rows, const uint8_t *q_idx,
                       const float *head_w, float *logits, int64_t logits_stride, int32_t *dev_status,
                       void *stream);

/*
 * Top-k (blog section "Sparse attention in K3.1 Pro": only the 2,048 best
 * scored tokens are kept; the fused path's selection is exact, section
 * "Low-latency decode"):
 *
 *   idx_out[r, 0..k) = the min(k, row_ctx[r]) positions t < row_ctx[r] with
 *   the largest logits[r * logits_stride + t], ties broken toward the lower t,
 *   written in ascending order of t and padded with -1.
 *
 * Logits compare as floats (-0 == +0); they must be finite.  k in
 * [1, DSA_MAX_TOPK].  Exact and deterministic: given identical logits the
 * result is bit-identical.
 *
 * workspace (device, 256-byte aligned, no initial contents) may be NULL.
 * With workspace_bytes >= dsa_topk_workspace_size(num_rows, max_ctx, k) > 0
 * (at most 64 rows, max_ctx above 131,072), the selection runs as three launches of
 * independent CTAs over chunks of each row: every chunk counts its keys in
 * 4096 bins (the top 12 bits of the order-preserving key: one bin per 1/8
 * binade); every chunk sums its row's counts, finds the bin holding the k-th
 * largest key and passes on its keys at or above that bin, in position order;
 * every chunk then finds the exact threshold among the row's keys in that bin
 * and writes its share of the selection.  A row whose threshold bin holds more
 * than 12,288 keys (heavy ties, or scores within 1/8 binade of each other) is
 * selected from its whole logits by one CTA instead (slower).  Without it
 * (NULL, or a size of 0 for this shape), one thread-block cluster per row
 * selects.  A workspace smaller than the size is DSA_ERR_WORKSPACE.  The
 * result is the same either way.
 */
int dsa_topk(const float *logits, int64_t logits_stride, const int32_t *row_ctx, int32_t num_rows,
             int32_t max_ctx, int32_t k, int32_t *idx_out, int32_t *dev_status, void *workspace,
             size_t workspace_bytes, void *stream);

/* Workspace bytes of the histogram top-k for this batch on the current device; 0 when the shape
 * (more than 64 rows, or rows of at most 131,072 keys) takes the cluster selection, which needs none. */
size_t dsa_topk_workspace_size(int32_t num_rows, int32_t max_ctx, int32_t k);

/*
 * Top-k and page -> slot in one call (the two steps below, dsa_topk then
 * dsa_page_to_slot, with the translation done where the selection is
 * written): idx_out as dsa_topk over rows->row_ctx / rows->max_ctx, and
 * slots_out[r, i] = block_table[row_req[r]][t / 64] * 64 + t % 64 for each
 * selected t = idx_out[r, i] (-1 where idx_out is -1).  A page id outside
 * [0, pool_pages) or a bad row_req is DSA_ERR_BOUNDS with slot -1.  workspace
 * as for dsa_topk.
 */
int dsa_topk_slots(const float *logits, int64_t logits_stride, const dsa_rows *rows, int64_t pool_pages, int32_t k,
                   int32_t *idx_out, int32_t *slots_out, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * dsa_topk_slots whose output pass also warms L2 with the selected tokens'
 * latents, so that the sparse attention launched next gathers them from L2
 * instead of HBM (the fused decode path of blog section "Low-latency decode"
 * hands attention the physical rows to read as soon as they are chosen).
 * latent_cache: the latent pool the slots index (its num_pages bounds the
 * slots).  FP8 latents (576 contiguous bytes per slot) are prefetched; an
 * NVFP4 pool gets the plain dsa_topk_slots result.  Outputs are identical to
 * dsa_topk_slots.  workspace as for dsa_topk.
 */
int dsa_topk_slots_warm(const float *logits, int64_t logits_stride, const dsa_rows *rows, const dsa_cache *latent_cache,
                        int32_t k, int32_t *idx_out, int32_t *slots_out, int32_t *dev_status, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Single-pass scorer + top-k (blog section "Low-latency decode: fused DSA
 * decode path": the scorer feeds a batch-invariant exact top-k; here the
 * scorer's epilogue also builds the histogram the selection starts from).
 *
 * DSA_HIST_BINS bins per row of the top 16 bits of each logit's
 * order-preserving 32-bit key (larger float, larger key; -0 folds onto +0).
 *
 * dsa_indexer_logits_hist: dsa_indexer_logits, and for every logit it writes
 *   hist[r * DSA_HIST_BINS + (key(logit) >> 16)] += 1.
 *   hist: [num_rows, DSA_HIST_BINS] uint32, device, all zero on entry.
 *
 * dsa_topk_hist: dsa_topk (same arguments and result), starting from that
 *   histogram: the bin holding the k-th key is read off it, one pass over the
 *   logits collects that bin's keys, and the selection finishes on those.
 *   hist must be the histogram dsa_indexer_logits_hist produced for exactly
 *   these logits and row_ctx (otherwise the result is undefined); the call
 *   leaves it all zero, ready for the next scorer call.  A bin holding more
 *   keys than the candidate list falls back to refinement rounds.
 *
 * dsa_indexer_topk: both calls in one, with the logits and the histogram in
 *   a workspace of dsa_indexer_topk_workspace_size() bytes (device, 256-byte
 *   aligned) that must be all zero before the first call; every call leaves
 *   its histogram part zero again, and the logits part holds no defined
 *   contents afterwards (their L2 lines are dropped once read, so they cost no
 *   HBM write-back).
 */
#define DSA_HIST_BINS 65536
int dsa_indexer_logits_hist(const dsa_cache *index_cache, const dsa_rows *rows, const uint8_t *q_idx,
                            const float *head_w, float *logits, int64_t logits_stride, uint32_t *hist,
                            int32_t *dev_status, void *stream);
int dsa_topk_hist(const float *logits, int64_t logits_stride, const int32_t *row_ctx, int32_t num_rows,
                  int32_t max_ctx, int32_t k, uint32_t *hist, int32_t *idx_out, int32_t *dev_status, void *stream);
int dsa_indexer_topk(const dsa_cache *index_cache, const dsa_rows *rows, const uint8_t *q_idx, const float *head_w,
                     int32_t k, int32_t *idx_out, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                     void *stream);
size_t dsa_indexer_topk_workspace_size(int32_t num_rows, int32_t max_ctx);

/*
 * Page -> slot translation (blog section "One KV cache, three states": the
 * block table and cache slots are translated to kernel page addresses
 * before each step):
 *
 *   slots[r, i] = block_table[row_req[r]][t / 64] * 64 + t % 64 for t = idx[r, i] >= 0,
 *   slots[r, i] = -1 for t = -1.
 *
 * idx and slots are [num_rows, k] int32.  A position t >= row_ctx[r], or a
 * page id outside [0, pool_pages) (the page count of the pools the slots
 * will address), is DSA_ERR_BOUNDS and yields slot -1.
 */
int dsa_page_to_slot(const dsa_rows *rows, int64_t pool_pages, const int32_t *idx, int32_t k, int32_t *slots,
                     int32_t *dev_status, void *stream);

/*
 * Sparse absorbed MLA (blog section "Sparse attention in K3.1 Pro": MLA
 * attention runs exactly, but only over the selected tokens; the latent is
 * both key and value, section "Low-latency decode": absorbed key
 * projection):
 *
 *   S[h, t] = sm_scale * <q[r,h,:], kv_t>                     (576 dims)
 *   out[r,h,:] = sum_t softmax_t(S[h, .]) * kv_t[0:512]      over t in slots[r, :] with slot >= 0
 *   lse[r,h] = ln sum_t exp(S[h,t])
 *
 * kv_t is the decoded latent of slot t (FP8: e4m3 * tensor_scale; NVFP4:
 * e2m1 * per-16 e4m3 scale for dims 0..511 and e4m3 * tensor_scale for the
 * RoPE dims).  q: [num_rows, num_heads, 576] bf16 bits, num_heads a multiple
 * of 16 and <= 96; slots: [num_rows, k] int32, -1 = unused; out:
 * [num_rows, num_heads, 512] fp32; lse: [num_rows, num_heads] fp32 or NULL.
 * A row with no valid slot gets out = 0 and lse = -inf.  Precision:
 *   - _decode over FP8 latents (k > 128) contracts e4m3 x e4m3 -> fp32 on the
 *     latents as stored.  Each head's query is scaled by a power of two and
 *     written as the sum of two e4m3 terms (exact for bf16 values within
 *     about 2^10 of the head's largest |q|; smaller ones keep an absolute
 *     error of at most 2^-17 of that largest), and the softmax weights likewise
 *     (about 8 significant bits).  A non-finite q is DSA_ERR_RANGE.
 *   - NVFP4 latents, _prefill, and decode with k <= 128 contract
 *     fp16 x fp16 -> fp32: latents decode to fp16 exactly, q rounds from bf16
 *     to fp16 (|q| > 65504 is DSA_ERR_RANGE), weights are fp16.
 *
 * _decode splits each row's k tokens into parts of 128 (k <= 2048, else
 * DSA_ERR_UNSUPPORTED), one CTA per part, keeps each part's normalised
 * output in fp16 and merges the parts by log-sum-exp; it needs a workspace
 * of dsa_sparse_mla_workspace_size() bytes (device, 256-byte aligned, no
 * initial contents; it also holds the rows' queries converted once to the
 * kernel's fp16 layout).  _prefill runs one CTA per row, needs no workspace
 * (pass NULL, 0) and suits many rows.  The split is fixed, so both are
 * batch-invariant; their results differ from each other by rounding.
 */
int dsa_sparse_mla_decode(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                          const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale, float *out,
                          float *lse, int32_t *dev_status, void *workspace, size_t workspace_bytes, void *stream);

int dsa_sparse_mla_prefill(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                           const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale, float *out,
                           float *lse, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * dsa_sparse_mla_decode in two parts, so the query conversion can run ahead
 * of (or beside) the scorer and the top-k, which it does not depend on:
 * _prepare writes each row's query, converted once to the attention
 * kernel's fp16 operand layout, into the workspace (nothing when k <= 128,
 * where decode uses no workspace); _prepared then runs the attention on it.
 * Both take the arguments of dsa_sparse_mla_decode (_prepare ignores the
 * slots, outputs and sm_scale) and the same workspace; _prepared must be
 * ordered after _prepare with the same q, num_heads, num_rows and k.  The
 * result equals dsa_sparse_mla_decode's bit for bit.
 */
int dsa_sparse_mla_decode_prepare(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                                  int32_t num_rows, int32_t k, int32_t *dev_status, void *workspace,
                                  size_t workspace_bytes, void *stream);
int dsa_sparse_mla_decode_prepared(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                                   const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale, float *out,
                                   float *lse, int32_t *dev_status, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * dsa_sparse_mla_decode without a caller workspace.  The paper has no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory: a host framework whose allocator has reserved the device's
 * memory for its own pools and hands out no extra buffers, a plugin that
 * only sees the tensors it is given, or a latency-critical loop that must not
 * call cudaMalloc (it can block and synchronise the device).
 *
 * Same arguments, semantics and results as dsa_sparse_mla_decode, minus the
 * workspace.  The split-K partial outputs live in a fixed array in the
 * library's own device memory, sized for DSA_NOALLOC_MAX_ROWS rows of
 * k <= 2048 tokens and num_heads <= 96 (13,569,024 bytes, held by every GPU
 * that loads the library until the process exits).  Larger calls return
 * DSA_ERR_WORKSPACE without launching.  The first call on a device looks up
 * the array's address with that device current; make it before capturing
 * any stream.  That address belongs to the device's primary context: after a
 * cudaDeviceReset of the device this call must not be used again in the
 * process.  Shape errors return the statuses dsa_sparse_mla_decode returns.  All calls share the array: calls whose kernels may overlap on
 * the GPU (unordered streams) race on it; calls ordered on one stream do not.
 * No part of the array needs to start zeroed.
 */
#define DSA_NOALLOC_MAX_ROWS 8
int dsa_sparse_mla_decode_noalloc(const dsa_cache *latent_cache, const uint16_t *q, int32_t num_heads,
                                  const int32_t *slots, int32_t num_rows, int32_t k, float sm_scale, float *out,
                                  float *lse, int32_t *dev_status, void *stream);

/*
 * Quantise new tokens and write them into the caches (blog section
 * "Low-latency decode: fused DSA decode path": the front end quantises the
 * new token's index key, FP8 or MXFP4, and the new latent is written into
 * the cache before the indexer scores).  For each i with slots[i] >= 0 the
 * token's index key index_keys[i, 0:128] (bf16 bits) and latent
 * latents[i, 0:576] (bf16 bits) are written at that physical slot of the two
 * pools (the pools' base pointers are written through):
 *   DSA_KEY_FP8:      s = amax / 448 (1 if amax = 0), code = e4m3(x / s), s stored as fp32
 *   DSA_KEY_MXFP4:    per 32 values E = floor(log2 amax) - 2 + 127 clamped to [0, 254]
 *                     (0 for an all-zero block), code = e2m1(x * 2^(127 - E))
 *   DSA_LATENT_FP8:   code = e4m3(x / tensor_scale)
 *   DSA_LATENT_NVFP4: per 16 values scale code = e4m3(amax / 6), code = e2m1(x / scale)
 *                     (0 when the scale is 0); RoPE dims e4m3(x / tensor_scale)
 * Scales and quotients are IEEE fp32 operations; codes are round-to-nearest-
 * even with saturation (e4m3 to +-448, e2m1 to +-6), so the bytes are exact.
 * Both pools must have the same num_pages; tensor_scale > 0 comes from the
 * latent pool.  A slot outside the pools is DSA_ERR_BOUNDS (not written).
 */
int dsa_cache_insert(const dsa_cache *index_cache, const dsa_cache *latent_cache, const int32_t *slots,
                     int32_t num_tokens, const uint16_t *index_keys, const uint16_t *latents, int32_t *dev_status,
                     void *stream);

/* Workspace bytes dsa_sparse_mla_decode needs for num_rows rows of k slots. */
size_t dsa_sparse_mla_workspace_size(int32_t num_rows, int32_t num_heads, int32_t k);

/*
 * ---- MSA, the block-sparse variant (vLLM blog "Day-0 support for
 * MiniMax-M3.1-Flash", section "MSA primer" and its Fig. 1; FP8 queries over an
 * FP8 K/V cache, section "Blackwell-optimised MSA kernels").  The cache is cut
 * into 128-token blocks, which are also its pages; one index query per GQA
 * group (4 groups = 4 KV heads) scores every visible token against the one
 * 128-B index key all groups share, the scores are max-pooled per block, each
 * group keeps its most recent block and the 15 best others, and the group's
 * query heads attend exactly to the tokens of those blocks.
 *
 * Page layouts (128 tokens; the widths are the blog's, the arrangement inside
 * a page is this library's):
 *   index  [128 x 128 B e4m3]                                          16384 B
 *   kv     [4 KV heads] x ([K: 128 x 128 B e4m3] [V: 128 x 128 B e4m3]) 131072 B
 * For these calls dsa_rows.block_table holds 128-token page ids (bt_stride >=
 * ceil(max_ctx / 128)); token t of a request is row t % 128 of page
 * block_table[req][t / 128].  Pools and queries are 16-byte aligned.
 */
#define DSA_MSA_PAGE 128
#define DSA_MSA_DIM 128
#define DSA_MSA_GROUPS 4
#define DSA_MSA_BLOCKS 16   /* blocks kept per (row, group): the most recent + the 15 best others */
#define DSA_MSA_MAX_HPG 64  /* query heads per group: a multiple of 16, at most this */

/*
 * Block scores: scores[(r * 4 + g) * score_stride + b] = max over tokens t of
 * block b with t < row_ctx[r] of <q_idx[r, g, :], k_t> (e4m3 codes; the index
 * key has no scale), for b < ceil(row_ctx[r] / 128); other entries are not
 * written.  q_idx: [num_rows, 4, 128] e4m3.  rows->rows_per_group (1, 2, 4 or
 * 8) consecutive rows of one request share each read of the keys.  Products
 * are exact and accumulate in fp32 on the tensor cores.  score_stride >=
 * ceil(max_ctx / 128).  A page id outside [0, num_pages) or a bad row is
 * DSA_ERR_BOUNDS on dev_status.
 */
int dsa_msa_block_scores(const void *index_pool, int64_t num_pages, const dsa_rows *rows, const uint8_t *q_idx,
                         float *scores, int64_t score_stride, int32_t *dev_status, void *stream);

/*
 * Block selection, per (row r, group g), nb = ceil(row_ctx[r] / 128): nb <= 16
 * keeps every block; otherwise block nb - 1 and the 15 highest scores among
 * blocks 0 .. nb - 2, ties to the lower block, a NaN score counting as -inf.
 * blocks[(r * 4 + g) * 16 + i] lists them ascending, -1 padded.  row_ctx
 * outside [0, max_ctx] is DSA_ERR_BOUNDS (clamped).
 */
int dsa_msa_select(const float *scores, int64_t score_stride, const int32_t *row_ctx, int32_t num_rows,
                   int32_t max_ctx, int32_t *blocks, int32_t *dev_status, void *stream);

/*
 * Block-sparse GQA attention: head h of row r belongs to group g = h / hpg
 * (hpg = heads_per_group) and attends to the visible tokens (t < row_ctx[r])
 * of its group's selected blocks:
 *   out[r, h, :] = sum_t softmax_t(sm_scale * <q_scale q[r,h,:], k_scale K_g,t>) v_scale V_g,t
 *   lse[r, h]    = natural log of the softmax denominator's sum, with the max folded in
 * q: [num_rows, 4 * hpg, 128] e4m3 codes; out: fp32 [num_rows, 4 * hpg, 128];
 * lse: fp32 [num_rows, 4 * hpg] or NULL.  A head with no visible selected
 * token gets out = 0 and lse = -inf.  S = Q K^T runs on FP8 tensor cores
 * (exact products, fp32 accumulation); P is fp16 and V is decoded exactly to
 * fp16 for P V.  The workspace (dsa_msa_attention_workspace_size bytes,
 * 256-byte aligned) holds one normalised part per selected block, merged by
 * log-sum-exp.  A selected block at or past ceil(row_ctx / 128) or a page id
 * outside the pool is DSA_ERR_BOUNDS.
 */
int dsa_msa_attention(const void *kv_pool, int64_t num_pages, float k_scale, float v_scale, const dsa_rows *rows,
                      const uint8_t *q, float q_scale, int32_t heads_per_group, const int32_t *blocks, float sm_scale,
                      float *out, float *lse, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                      void *stream);

/* Workspace bytes dsa_msa_attention needs for num_rows rows. */
size_t dsa_msa_attention_workspace_size(int32_t num_rows, int32_t heads_per_group);

/*
 * Failure-path self-test (no counterpart on the pages): one CTA whose
 * threads wait on a barrier that nothing ever arrives on.  The wait is the
 * bounded wait every kernel of the library uses; it gives up after the
 * library's wait limit (4e9 SM cycles, about two seconds), writes
 * DSA_ERR_TIMEOUT to dev_status (required), and every other waiter of the CTA
 * then leaves at once.  The kernel exits normally: nothing faults or hangs,
 * and the context stays usable.  Returns DSA_OK once launched.
 */
int dsa_selftest_wait_timeout(int32_t *dev_status, void *stream);

/* Human-readable text of a status code (static storage). */
const char *dsa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
