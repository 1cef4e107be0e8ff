// msa.cu -- the block-sparse MSA variant on the sm_103a tensor cores.
//
// What it computes (vLLM blog "Day-0 support for MiniMax-M3.1-Flash", section
// "MSA primer" and its Fig. 1): the cache is cut into 128-token blocks, which
// are also the pages; one FP8 index query per GQA group scores every visible
// token against the single 128-B index key all groups share, and the scores
// are max-pooled to one score per block; each group keeps its most recent
// block plus the 15 best others (ties to the lower block); the group's query
// heads then attend exactly to the tokens of those blocks only, with FP8
// queries and an FP8 K/V cache (section "Blackwell-optimised MSA kernels").
//
//   block score  S[r,g,b] = max_{t in block b, t < L_r} <qi[r,g,:], ki_t>
//   selection    b = nb - 1 and the 15 best of 0 .. nb - 2 (all blocks when nb <= 16)
//   attention    O[r,h,:] = sum_t softmax_t(sm_scale <q[r,h,:], K_g,t>) V_g,t
//
// Design (GB300):
//   * scores: the scan of all index keys is HBM-bound (128 B per token per
//     row group).  One CTA per (row group, chunk of pages), two per SM; a TMA
//     producer brings one 128-token page per stage (one 16 KB, 128-byte
//     swizzled box = the K-major A operand), one thread issues
//     tcgen05.mma kind::f8f6f4 with the page's keys on M = 128 and the group's
//     rows x 4 index queries on N, and four epilogue warps take the block max
//     over TMEM lanes with warp shuffles; the MMA's commit releases the stage.
//   * selection: one CTA per (row, group); the candidates' 64-bit keys
//     (order-preserving score bits, then the inverted block id) stay in shared
//     memory; each warp takes the 15 best of its slice by warp argmax rounds,
//     and one warp takes the 15 best of those.
//   * attention: one CTA per (row, group, selected block).  TMA brings the
//     group's FP8 queries and the block's FP8 K and V (16 KB each); S = Q K^T
//     runs on kind::f8f6f4 (queries on M, padded to 128 rows, tokens on N =
//     128); one softmax thread per head reduces its row exactly (a block is
//     one tile, so no online rescale); V is decoded exactly to fp16 in the
//     MN-major image that O^T = V^T P^T (kind::f16, dims on M, heads on N)
//     reads with fp16 P; each block's normalised part and its (max, sum) go
//     to the workspace and a combine kernel merges the 16 parts by
//     log-sum-exp.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kMsaPage = DSA_MSA_PAGE;     // tokens per block and page
constexpr int kMsaDim = DSA_MSA_DIM;       // index key, query, K and V dims (bytes in FP8)
constexpr int kMsaGroups = DSA_MSA_GROUPS; // GQA groups = KV heads
constexpr int kMsaBlocks = DSA_MSA_BLOCKS; // blocks kept per (row, group)
constexpr int kMsaKvPageRows = kMsaGroups * 2 * kMsaPage;  // 128-byte rows of one K/V page

__device__ __forceinline__ uint32_t msa_sw128(int row, int u) {
    return static_cast<uint32_t>(row * 128 + ((u ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two_bytes)));
    return r;
}

__device__ __forceinline__ float msa_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld_n<16>(uint32_t taddr, uint32_t (&r)[16]) {
    tmem_ld16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_n<32>(uint32_t taddr, uint32_t (&r)[32]) {
    tmem_ld32(taddr, r);
}

// ================================================================== block scores

template <int G>
struct ScoreCfg {
    static constexpr int kCols = kMsaGroups * G;          // real accumulator columns: (row, group)
    static constexpr int N = kCols < 16 ? 16 : kCols;     // MMA N (>= 16; extra columns unread)
    static constexpr int kAcc = 4;                        // TMEM accumulators in flight
    static constexpr uint32_t kTmemCols = static_cast<uint32_t>(kAcc * N) < 32u ? 32u : kAcc * N;
    static constexpr int kStages = 6;                     // 16 KB key pages in flight
    static constexpr int kThreads = 256;                  // 0 TMA, 1 MMA, 4-7 epilogue
    static constexpr int OFF_KEYS = 0;
    static constexpr int OFF_Q = OFF_KEYS + kStages * kMsaPage * 128;
    static constexpr int OFF_RED = OFF_Q + ((N * 128 + 1023) / 1024) * 1024;
    static constexpr int OFF_BARS = OFF_RED + 2 * 4 * 32 * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kAcc + 2;
    static constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
    static constexpr int kSmemBytes = OFF_MISC + 64 + 1024;
    static_assert(kCols <= 32, "at most 8 rows per group");
    static_assert(kSmemBytes <= 228 * 1024 / 2 - 1024, "two CTAs per SM");
};

template <int G>
__global__ void __launch_bounds__(256, 2)
    msa_scores_kernel(const __grid_constant__ CUtensorMap key_map, const __grid_constant__ CUtensorMap q_map,
                      const MsaScoreArgs a) {
    using C = ScoreCfg<G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *keys = smem + C::OFF_KEYS;
    uint8_t *qbuf = smem + C::OFF_Q;
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);  // [2][4 quadrants][32 columns]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BARS);
    uint64_t *full = bars;                    // [kStages] TMA -> MMA
    uint64_t *empty = bars + C::kStages;      // [kStages] MMA commit -> TMA
    uint64_t *tfull = empty + C::kStages;     // [kAcc] MMA commit -> epilogue
    uint64_t *tempty = tfull + C::kAcc;       // [kAcc] epilogue warps -> MMA
    uint64_t *qfull = tempty + C::kAcc;       // [1] query -> MMA
    uint64_t *mma_done = qfull + 1;           // [1] every MMA (and its commits) retired
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    volatile int *epi_ok = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = blockIdx.x / a.chunks, chunk = blockIdx.x % a.chunks;
    const int row0 = grp * G;

    // the group's request and longest visible context (rows of a group share a request)
    const int req = a.row_req[row0];
    int gmax = 0;
    bool bad = req < 0 || req >= a.num_requests;
    for (int j = 0; j < G; ++j) {
        const int c = a.row_ctx[row0 + j];
        if (a.row_req[row0 + j] != req || c < 0 || c > a.max_ctx) bad = true;
        gmax = max(gmax, min(max(c, 0), a.max_ctx));
    }
    if (bad) {
        if (tid == 0) report(a.status, DSA_ERR_BOUNDS);
        return;
    }
    const int np = (gmax + kMsaPage - 1) / kMsaPage;
    const int p_begin = chunk * a.chunk_pages;
    const int p_end = min(np, p_begin + a.chunk_pages);
    if (p_begin >= p_end) return;
    const int n_pages = p_end - p_begin;

    if (tid == 0) {
        *abort = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < C::kAcc; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);
        }
        mbar_init(qfull, 1);
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // lane j looks up the page id of page base + j; lane 0 issues the copies
        const int32_t *bt = a.block_table + static_cast<int64_t>(req) * a.bt_stride;
        if (lane == 0) {
            prefetch_tensormap(&key_map);
            mbar_arrive_expect_tx(qfull, C::N * 128);
            tma_load_2d(qbuf, &q_map, qfull, 0, row0 * kMsaGroups);
        }
        const uint64_t policy = l2_evict_first_policy();
        bool ok = true;
        for (int base = 0; ok && base < n_pages; base += 32) {
            int32_t pg = 0;
            if (base + lane < n_pages) {
                pg = bt[p_begin + base + lane];
                if (pg < 0 || pg >= a.num_pages) {
                    report(a.status, DSA_ERR_BOUNDS);
                    pg = 0;
                }
            }
            const int cnt = min(32, n_pages - base);
            for (int j = 0; j < cnt; ++j) {
                const int i = base + j, s = i % C::kStages;
                const int32_t pj = __shfl_sync(0xffffffffu, pg, j);
                int got = 0;
                if (lane == 0) got = mbar_wait(&empty[s], ((i / C::kStages) & 1) ^ 1, abort, a.status);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], kMsaPage * 128);
                    tma_load_2d_hint(keys + s * (kMsaPage * 128), &key_map, &full[s], 0, pj * kMsaPage, policy);
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = make_idesc(128, C::N, 0, 0, false, false);
            const uint64_t qdesc = sdesc_sw128(smem_u32(qbuf), 16, 1024);
            bool ok = mbar_wait(qfull, 0, abort, a.status);
            for (int i = 0; ok && i < n_pages; ++i) {
                const int s = i % C::kStages, b = i % C::kAcc;
                if (!mbar_wait(&tempty[b], ((i / C::kAcc) & 1) ^ 1, abort, a.status)) break;
                if (!mbar_wait(&full[s], (i / C::kStages) & 1, abort, a.status)) break;
                tc_fence_after();
                const uint64_t kdesc = sdesc_sw128(smem_u32(keys + s * (kMsaPage * 128)), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kMsaDim / 32; ++kk)
                    mma_f8(tmem_base + b * C::N, kdesc + kk * 2, qdesc + kk * 2, idesc, kk > 0 ? 1u : 0u);
                mma_commit(&empty[s]);  // the keys are consumed once the products are done
                mma_commit(&tfull[b]);
            }
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, abort, a.status);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue: block max
        const int quad = warp & 3;  // TMEM lane quadrant: keys 32 quad .. 32 quad + 31 of the page
        int ctx[G];
#pragma unroll
        for (int j = 0; j < G; ++j) ctx[j] = min(a.row_ctx[row0 + j], a.max_ctx);
        for (int i = 0; i < n_pages; ++i) {
            const int b = i % C::kAcc, p = p_begin + i;
            // one thread waits; the named barrier passes the result on, so the four warps
            // always leave the loop together
            if (quad == 0 && lane == 0) *epi_ok = mbar_wait(&tfull[b], (i / C::kAcc) & 1, abort, a.status) ? 1 : 0;
            named_bar_sync(1, 128);
            if (!*epi_ok) break;
            tc_fence_after();
            uint32_t acc[C::N];
            tmem_ld_n<C::N>(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + b * C::N, acc);
            tmem_ld_wait();
            reg_fence(acc);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
            const int t = p * kMsaPage + quad * 32 + lane;
            float *rd = red + (i & 1) * (4 * 32);
#pragma unroll
            for (int c = 0; c < C::kCols; ++c) {
                // fmaxf drops a NaN, so a NaN score never wins and an all-NaN block stays -inf
                float v = t < ctx[c / kMsaGroups] ? __uint_as_float(acc[c]) : -INFINITY;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                if (lane == 0) rd[quad * 32 + c] = v;
            }
            named_bar_sync(1, 128);
            if (quad == 0 && lane < C::kCols) {
                const float m = fmaxf(fmaxf(rd[lane], rd[32 + lane]), fmaxf(rd[64 + lane], rd[96 + lane]));
                const int j = lane / kMsaGroups, g = lane % kMsaGroups;
                if (p * kMsaPage < ctx[j])  // a row's blocks past its context are not written
                    a.scores[(static_cast<int64_t>(row0 + j) * kMsaGroups + g) * a.score_stride + p] = m;
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// ================================================================== block selection

// Larger key = better block: higher score (NaN counts as -inf, -0 as +0), then lower block id.
__device__ __forceinline__ unsigned long long msa_select_key(float s, int b) {
    if (s != s) s = -INFINITY;
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(b));
}

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

// One warp's argmax over keys[lo, hi) (shared memory), 15 times: the winners' keys go to
// top[0..14] in decreasing order (0 once the range is exhausted) and are zeroed in keys.
// Candidate keys are > 0 and distinct (the block id is in the low bits), so each round's
// winner sits at exactly one position, which the lane that saw it clears.
__device__ __forceinline__ void warp_top15(unsigned long long *keys, int lo, int hi, unsigned long long *top,
                                           int lane) {
    for (int round = 0; round < kMsaBlocks - 1; ++round) {
        unsigned long long mine = 0ull;
        int at = -1;
        for (int b = lo + lane; b < hi; b += 32) {
            const unsigned long long k = keys[b];
            if (k > mine) {
                mine = k;
                at = b;
            }
        }
        // 64-bit warp max as two 32-bit reductions: the score half, then the block half among
        // the lanes holding that score
        const uint32_t hi = static_cast<uint32_t>(mine >> 32), lo = static_cast<uint32_t>(mine);
        const uint32_t bh = __reduce_max_sync(0xffffffffu, hi);
        const uint32_t bl = __reduce_max_sync(0xffffffffu, hi == bh ? lo : 0u);
        const unsigned long long best = (static_cast<unsigned long long>(bh) << 32) | bl;
        if (lane == 0) top[round] = best;
        if (best != 0ull && mine == best) keys[at] = 0ull;
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kSelThreads) msa_select_kernel(const MsaSelectArgs a) {
    extern __shared__ unsigned long long cand[];  // [nb - 1] keys; a taken key becomes 0
    __shared__ unsigned long long wtop[kSelWarps * (kMsaBlocks - 1)];
    __shared__ int32_t won[kMsaBlocks];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x / kMsaGroups;
    int L = a.row_ctx[r];
    if (L < 0 || L > a.max_ctx) {
        if (tid == 0) report(a.status, DSA_ERR_BOUNDS);
        L = min(max(L, 0), a.max_ctx);
    }
    const int nb = (L + kMsaPage - 1) / kMsaPage;
    int32_t *out = a.blocks + static_cast<int64_t>(blockIdx.x) * kMsaBlocks;
    if (nb <= kMsaBlocks) {
        if (tid < kMsaBlocks) out[tid] = tid < nb ? tid : -1;
        return;
    }
    const float *sc = a.scores + static_cast<int64_t>(blockIdx.x) * a.score_stride;
    const int m = nb - 1;  // candidates: every block but the most recent one
    for (int b = tid; b < m; b += kSelThreads) cand[b] = msa_select_key(sc[b], b);
    __syncthreads();
    // each warp takes the 15 best of its slice; the 15 best of those 8 x 15 are the row's 15 best
    const int per = (m + kSelWarps - 1) / kSelWarps;
    warp_top15(cand, min(m, warp * per), min(m, (warp + 1) * per), wtop + warp * (kMsaBlocks - 1), lane);
    __syncthreads();
    if (warp == 0) {
        unsigned long long top[kMsaBlocks - 1];
        warp_top15(wtop, 0, kSelWarps * (kMsaBlocks - 1), top, lane);
        if (lane == 0) {
            for (int i = 0; i < kMsaBlocks - 1; ++i)
                won[i] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(top[i] & 0xFFFFFFFFull));
            won[kMsaBlocks - 1] = nb - 1;
            // ascending block order (insertion sort of 16 ids)
            for (int i = 1; i < kMsaBlocks; ++i) {
                const int v = won[i];
                int j = i - 1;
                while (j >= 0 && won[j] > v) {
                    won[j + 1] = won[j];
                    --j;
                }
                won[j + 1] = v;
            }
        }
    }
    __syncthreads();
    if (tid < kMsaBlocks) out[tid] = won[tid];
}

// ================================================================== attention

constexpr int kAttThreads = 256;  // warp 0: TMA + MMA issue; warps 4-7: V decode, softmax, epilogue
constexpr int kAttTmemCols = 256; // S at columns 0..127 (heads on lanes), O^T at 128.. (dims on lanes)
constexpr int kAttOFF_Q = 0;                         // FP8 queries, 128 rows x 128 B (rows >= hpg unused)
constexpr int kAttOFF_K = kAttOFF_Q + 128 * 128;     // FP8 K of the block, 128 tokens x 128 B
constexpr int kAttOFF_V8 = kAttOFF_K + 128 * 128;    // FP8 V of the block
constexpr int kAttOFF_V16 = kAttOFF_V8 + 128 * 128;  // fp16 V image: [2 x 64 dims][128 tokens][128 B]
constexpr int kAttOFF_P = kAttOFF_V16 + 2 * 128 * 128;  // fp16 P: [2 x 64 tokens][hpg heads][128 B]
constexpr int kAttOFF_L = kAttOFF_P + 2 * DSA_MSA_MAX_HPG * 128;  // per-head row sum
constexpr int kAttOFF_BARS = kAttOFF_L + DSA_MSA_MAX_HPG * 4;
constexpr int kAttOFF_MISC = kAttOFF_BARS + 8 * 8;
constexpr int kAttSmemBytes = kAttOFF_MISC + 64 + 1024;
static_assert(kAttSmemBytes <= 228 * 1024 / 2 - 1024, "two CTAs per SM");

__global__ void __launch_bounds__(kAttThreads, 2)
    msa_attention_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                         const MsaAttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem + kAttOFF_Q;
    uint8_t *ks = smem + kAttOFF_K;
    uint8_t *v8 = smem + kAttOFF_V8;
    uint8_t *v16 = smem + kAttOFF_V16;
    uint8_t *ps = smem + kAttOFF_P;
    float *lsum = reinterpret_cast<float *>(smem + kAttOFF_L);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kAttOFF_BARS);
    uint64_t *in_full = bars + 0;   // Q, K, V landed (tx bytes)
    uint64_t *s_full = bars + 1;    // S = Q K^T done (commit)
    uint64_t *v_ready = bars + 2;   // fp16 V image written (4 warps)
    uint64_t *p_full = bars + 3;    // P written (4 warps)
    uint64_t *o_full = bars + 4;    // O^T done (commit)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kAttOFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kAttOFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hpg = a.heads_per_group, H = kMsaGroups * hpg;
    const int slot = blockIdx.x % kMsaBlocks;
    const int rg = blockIdx.x / kMsaBlocks;  // row * 4 + group
    const int r = rg / kMsaGroups, g = rg % kMsaGroups;
    float *part_o = a.part_o + static_cast<int64_t>(blockIdx.x) * hpg * kMsaDim;
    float *part_ml = a.part_ml + static_cast<int64_t>(blockIdx.x) * hpg * 2;

    // the block this CTA attends to, and its page; an unused slot or an empty block is a
    // part with no weight
    const int req = a.row_req[r];
    const int L = a.row_ctx[r];
    const int b = a.blocks[static_cast<int64_t>(rg) * kMsaBlocks + slot];
    const int nb = (max(L, 0) + kMsaPage - 1) / kMsaPage;
    bool valid = b >= 0;
    int32_t page = 0;
    if (valid) {
        const bool ok_rq = req >= 0 && req < a.num_requests && L >= 0 && L <= a.max_ctx && b < nb;
        if (ok_rq) page = a.block_table[static_cast<int64_t>(req) * a.bt_stride + b];
        if (!ok_rq || page < 0 || page >= a.num_pages) {
            if (tid == 0) report(a.status, DSA_ERR_BOUNDS);
            valid = false;
        }
    }
    if (!valid) {
        for (int h = tid; h < hpg; h += kAttThreads) {
            part_ml[2 * h] = -INFINITY;
            part_ml[2 * h + 1] = 0.f;
        }
        return;
    }
    const int n_valid = min(kMsaPage, L - b * kMsaPage);  // tokens of the block inside the context

    if (tid == 0) {
        *abort = 0;
        mbar_init(in_full, 1);
        mbar_init(s_full, 1);
        mbar_init(v_ready, 4);
        mbar_init(p_full, 4);
        mbar_init(o_full, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kAttTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 128;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ loads and MMAs
            prefetch_tensormap(&kv_map);
            prefetch_tensormap(&q_map);
            const int kv_row = page * kMsaKvPageRows + g * 2 * kMsaPage;
            mbar_arrive_expect_tx(in_full, static_cast<uint32_t>(hpg * 128 + 2 * kMsaPage * 128));
            tma_load_2d(qs, &q_map, in_full, 0, r * H + g * hpg);
            tma_load_2d(ks, &kv_map, in_full, 0, kv_row);
            tma_load_2d(v8, &kv_map, in_full, 0, kv_row + kMsaPage);
            bool ok = mbar_wait(in_full, 0, abort, a.status);
            if (ok) {
                // S[heads, tokens] = Q . K^T, FP8, M = 128 (rows >= hpg unused), N = 128 tokens
                tc_fence_after();
                constexpr uint32_t idesc_s = make_idesc(128, kMsaPage, 0, 0, false, false);
                const uint64_t qd = sdesc_sw128(smem_u32(qs), 16, 1024);
                const uint64_t kd = sdesc_sw128(smem_u32(ks), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kMsaDim / 32; ++kk) mma_f8(tmem, qd + kk * 2, kd + kk * 2, idesc_s, kk > 0 ? 1u : 0u);
                mma_commit(s_full);
                ok = mbar_wait(v_ready, 0, abort, a.status) && mbar_wait(p_full, 0, abort, a.status);
            }
            if (ok) {
                // O^T[dims, heads] = V^T . P^T, fp16: A = the V image (MN-major: 64-dim blocks
                // 16 KB apart, 8-token groups 1 KB apart), B = P (K-major), K = 128 tokens
                tc_fence_after();
                const uint32_t idesc_o = make_idesc(128, hpg, 0, 0, true, false);
                const uint64_t vd = sdesc_sw128(smem_u32(v16), kMsaPage * 128, 1024);
                const uint64_t pd = sdesc_sw128(smem_u32(ps), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kMsaPage / 16; ++kk) {
                    const uint64_t off_v = static_cast<uint64_t>(kk * 2048) >> 4;
                    const uint64_t off_p = static_cast<uint64_t>((kk >> 2) * hpg * 128 + (kk & 3) * 32) >> 4;
                    mma_f16(tmem_o, vd + off_v, pd + off_p, idesc_o, kk > 0 ? 1u : 0u);
                }
            }
            mma_commit(o_full);  // also retires S if the wait above gave up
        }
    } else if (warp >= 4) {
        const int quad = warp & 3;
        const int t = quad * 32 + lane;  // this thread's token (V decode) or TMEM lane (S row, O^T dim)
        bool ok = mbar_wait_warp(in_full, 0, abort, a.status);
        if (ok) {
            // ---- V: FP8 (TMA 128-byte swizzle) -> fp16 image, exact; token t's 16-dim unit c
            // becomes two 8-dim units of its 64-dim block c / 4; tokens past the context are 0
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int4 w = *reinterpret_cast<const int4 *>(v8 + msa_sw128(t, c));
                const uint32_t x[4] = {static_cast<uint32_t>(w.x), static_cast<uint32_t>(w.y),
                                       static_cast<uint32_t>(w.z), static_cast<uint32_t>(w.w)};
                int4 o0, o1;
                o0.x = e4m3x2_to_f16x2(x[0] & 0xffffu);
                o0.y = e4m3x2_to_f16x2(x[0] >> 16);
                o0.z = e4m3x2_to_f16x2(x[1] & 0xffffu);
                o0.w = e4m3x2_to_f16x2(x[1] >> 16);
                o1.x = e4m3x2_to_f16x2(x[2] & 0xffffu);
                o1.y = e4m3x2_to_f16x2(x[2] >> 16);
                o1.z = e4m3x2_to_f16x2(x[3] & 0xffffu);
                o1.w = e4m3x2_to_f16x2(x[3] >> 16);
                if (t >= n_valid) o0 = o1 = make_int4(0, 0, 0, 0);  // P is 0 there; V may hold NaN codes
                uint8_t *blk = v16 + (c >> 2) * (kMsaPage * 128);
                *reinterpret_cast<int4 *>(blk + msa_sw128(t, 2 * (c & 3))) = o0;
                *reinterpret_cast<int4 *>(blk + msa_sw128(t, 2 * (c & 3) + 1)) = o1;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(v_ready);
            // ---- softmax of row h = t over the block's tokens (log2 units; masked tokens -inf)
            ok = mbar_wait_warp(s_full, 0, abort, a.status);
        }
        if (ok) {
            tc_fence_after();
            if (quad * 32 < hpg) {
                const uint32_t srow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
                const float sc = a.s_scale;
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(srow + c * 32, v);
                    tmem_ld_wait();
                    reg_fence(v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c * 32 + j < n_valid) mx = fmaxf(mx, __uint_as_float(v[j]) * sc);
                }
                float l = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(srow + c * 32, v);
                    tmem_ld_wait();
                    reg_fence(v);
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float p0 = (c * 32 + j < n_valid) ? msa_exp2(__uint_as_float(v[j]) * sc - mx) : 0.f;
                        const float p1 = (c * 32 + j + 1 < n_valid) ? msa_exp2(__uint_as_float(v[j + 1]) * sc - mx) : 0.f;
                        l += p0 + p1;
                        __half2 hh = __floats2half2_rn(p0, p1);
                        pk[j / 2] = *reinterpret_cast<uint32_t *>(&hh);
                    }
                    if (t < hpg) {
                        // tokens 32c .. 32c + 31: 64-token block c / 2, 8-token units 4 (c & 1) .. + 3
                        uint8_t *prow = ps + (c >> 1) * (hpg * 128);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            *reinterpret_cast<int4 *>(prow + msa_sw128(t, 4 * (c & 1) + u)) =
                                make_int4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                    }
                }
                if (t < hpg) {
                    lsum[t] = l;
                    part_ml[2 * t] = mx;
                    part_ml[2 * t + 1] = l;
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            ok = mbar_wait_warp(o_full, 0, abort, a.status);
        }
        named_bar_sync(1, 128);  // lsum is complete
        if (ok) {
            // ---- O^T lane t = dim t: part O[h, t] = v_scale * acc / l_h
            tc_fence_after();
            const uint32_t orow = tmem_o + (static_cast<uint32_t>(quad * 32) << 16);
            for (int h0 = 0; h0 < hpg; h0 += 16) {
                uint32_t v[16];
                tmem_ld16(orow + h0, v);
                tmem_ld_wait();
                reg_fence(v);
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float l = lsum[h0 + x];
                    part_o[static_cast<int64_t>(h0 + x) * kMsaDim + t] =
                        l > 0.f ? __uint_as_float(v[x]) * (a.v_scale / l) : 0.f;
                }
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kAttTmemCols);
    }
}

// Merge the 16 block parts of one (row, head): O = sum_i w_i O_i / sum_i w_i with
// w_i = l_i 2^(m_i - M), M = max_i m_i (log2 units); lse in natural log.  One thread per
// output dim; every part's load is issued before any is used, and a part with no weight
// (unused slot, never written) enters through a select, so its bytes never reach the sum.
__global__ void __launch_bounds__(kMsaDim) msa_combine_kernel(const MsaAttnArgs a) {
    const int hpg = a.heads_per_group, H = kMsaGroups * hpg;
    const int r = blockIdx.x / H, h = blockIdx.x % H;
    const int g = h / hpg, hh = h % hpg;
    const int d = threadIdx.x;
    const int64_t base = (static_cast<int64_t>(r) * kMsaGroups + g) * kMsaBlocks;  // part of slot 0
    float mi[kMsaBlocks], li[kMsaBlocks], x[kMsaBlocks];
#pragma unroll
    for (int i = 0; i < kMsaBlocks; ++i) {
        mi[i] = a.part_ml[((base + i) * hpg + hh) * 2];
        li[i] = a.part_ml[((base + i) * hpg + hh) * 2 + 1];
        x[i] = a.part_o[((base + i) * hpg + hh) * kMsaDim + d];
    }
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMsaBlocks; ++i) M = fmaxf(M, mi[i]);
    float ws = 0.f, o = 0.f;
#pragma unroll
    for (int i = 0; i < kMsaBlocks; ++i) {
        const bool on = M > -INFINITY && li[i] > 0.f;
        const float w = on ? li[i] * msa_exp2(mi[i] - M) : 0.f;
        ws += w;
        o += on ? w * x[i] : 0.f;
    }
    a.out[(static_cast<int64_t>(r) * H + h) * kMsaDim + d] = ws > 0.f ? o / ws : 0.f;
    if (d == 0 && a.lse != nullptr)
        a.lse[static_cast<int64_t>(r) * H + h] = ws > 0.f ? (M + log2f(ws)) * 0.6931471805599453f : -INFINITY;
}

template <int G>
cudaError_t launch_scores_g(const CUtensorMap &key_map, const CUtensorMap &q_map, const MsaScoreArgs &a,
                            int num_groups, cudaStream_t s) {
    using C = ScoreCfg<G>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(msa_scores_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int64_t grid = static_cast<int64_t>(num_groups) * a.chunks;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    msa_scores_kernel<G><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, s>>>(key_map, q_map, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_msa_scores(const CUtensorMap &key_map, const CUtensorMap &q_map, const MsaScoreArgs &a,
                              int num_groups, int rows_per_group, cudaStream_t s) {
    switch (rows_per_group) {
        case 1: return launch_scores_g<1>(key_map, q_map, a, num_groups, s);
        case 2: return launch_scores_g<2>(key_map, q_map, a, num_groups, s);
        case 4: return launch_scores_g<4>(key_map, q_map, a, num_groups, s);
        case 8: return launch_scores_g<8>(key_map, q_map, a, num_groups, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_msa_select(const MsaSelectArgs &a, int num_rows, cudaStream_t s) {
    if (num_rows == 0) return cudaSuccess;
    const int max_nb = (a.max_ctx + kMsaPage - 1) / kMsaPage;
    const size_t smem = static_cast<size_t>(max_nb > 1 ? max_nb : 1) * sizeof(unsigned long long);
    static int configured_device = -1;
    static size_t configured_smem = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev || smem > configured_smem) {
        cudaError_t e = cudaFuncSetAttribute(msa_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured_device = dev;
        configured_smem = smem;
    }
    msa_select_kernel<<<num_rows * kMsaGroups, kSelThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_msa_attention(const CUtensorMap &kv_map, const CUtensorMap &q_map, const MsaAttnArgs &a,
                                 int num_rows, cudaStream_t s) {
    if (num_rows == 0) return cudaSuccess;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(msa_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kAttSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    msa_attention_kernel<<<num_rows * kMsaGroups * kMsaBlocks, kAttThreads, kAttSmemBytes, s>>>(kv_map, q_map, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    msa_combine_kernel<<<num_rows * kMsaGroups * a.heads_per_group, kMsaDim, 0, s>>>(a);
    return cudaGetLastError();
}

size_t msa_attention_workspace_bytes(size_t num_rows, size_t heads_per_group) {
    const size_t parts = num_rows * kMsaGroups * kMsaBlocks * heads_per_group;
    return (parts * kMsaDim * sizeof(float) + 255) / 256 * 256 + (parts * 2 * sizeof(float) + 255) / 256 * 256;
}

}  // namespace dsa
