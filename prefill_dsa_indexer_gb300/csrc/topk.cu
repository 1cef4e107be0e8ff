// topk.cu -- exact top-k of every row's indexer logits.
//
// Semantics (vLLM blog "Day-0 support for Kimi K3.1 Pro": the indexer keeps
// the 2,048 best-scoring tokens, section "Sparse attention in K3.1 Pro"; the
// selection is exact, section "Low-latency decode"; batch-invariant top-k,
// section "Day-0 zero-mismatch RL"): the k largest logits of [0, L_r), ties
// to the lower position, reported in ascending position order, -1 padded.
//
// Method: radix selection on order-preserving 32-bit keys, one thread-block
// cluster of CL = 1..16 CTAs per row (CL chosen on the host so that a batch
// of rows covers the SMs).  The row is cut into one contiguous chunk per CTA;
// the first kCacheElems keys of a chunk are read from memory once and kept in
// shared memory for every later pass.
//   1. The cluster agrees on the row's key range [min, max].
//   2. Cluster rounds: every CTA histograms its chunk into 2048 bins spanning
//      the current interval (power-of-two bin width); the histograms are summed
//      by a reduce-scatter over distributed shared memory (CTA r adds up bin
//      slice r of every CTA and writes the sums back to all of them), so every
//      CTA reaches the same decision: the bin holding the k-th key becomes the
//      next interval.  Each CTA also tracks how many of its own keys lie above
//      the interval.
//   3. Once the interval holds at most kCandCap keys, every CTA publishes its
//      keys inside it (its candidates) and its count above it; every CTA then
//      gathers all of them in rank order and refines alone (identically) down
//      to the exact threshold key T and the number of keys equal to T to take:
//      by ranking when there are at most kRankMax candidates (each counts the
//      candidates above and at it), else by further histogram rounds.  The
//      gathered candidates also give every CTA the number of selected keys in
//      the lower-ranked chunks, so no further cluster barrier is needed.
//   4. The selection is written in position order.  A chunk's selections fill
//      one contiguous range of the output; each warp stages its segment's keys
//      >= T in order (one pass when the chunk is in shared memory, else a
//      counting pass and a placing pass), and all threads then write the
//      range.  Output order and values never depend on timing.
//
// A few rows longer than 128K keys, with a caller workspace, take the histogram selection at the end
// of this file instead: three launches of independent CTAs over chunks of each row (bin counts, the
// threshold bin's candidates, the exact threshold and the output), no clusters.
#include <cooperative_groups.h>

#include "kernels.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kCacheElems = 40960;
constexpr int kCandCap = 4096;
constexpr int kRankMax = 256;  // up to this many gathered candidates, the threshold is found by ranking
static_assert(DSA_MAX_TOPK <= kCandCap, "a chunk's selections are staged in cand_all");
constexpr int kMaxCluster = 16;
constexpr int kMinChunk = 4096;  // a row is not cut into chunks shorter than this
constexpr int kBtCache = 1026;   // block-table entries of a chunk kept in shared memory (64K keys)

struct TopkSmem {
    uint32_t cache[kCacheElems];
    uint32_t hist[kBins];         // this CTA's histogram (read by the cluster's reduce-scatter)
    uint32_t hsum[kBins];         // the cluster's histogram (written by the cluster)
    uint32_t cand[kCandCap];      // this CTA's keys inside the interval (read by the cluster)
    uint32_t cand_all[kCandCap];  // every CTA's candidates, in rank order
    unsigned long long wsum[kWarps];
    uint32_t wgt[kWarps], weq[kWarps];
    uint32_t red[2 * kWarps];
    uint32_t roff[kMaxCluster + 1];  // rank r's candidates start at cand_all[roff[r]]
    uint32_t mm[2];      // this CTA's chunk key range (read by the cluster)
    uint32_t pub[3];     // published: candidates, keys above the interval, keys == T (read by the cluster)
    uint32_t sel[5];     // selected bin, cluster keys above / in it, local keys above / in it
    uint32_t ncand;
    uint32_t range[2];
    uint32_t before[2];  // selected keys > T and == T in the lower-ranked chunks
    int32_t bt_cache[kBtCache];  // page ids of this chunk's pages, when slots are written
    uint32_t hpub;       // histogram path: this CTA's slice total (read by the cluster)
    uint32_t hsel[2];    // histogram path: owner rank, the cluster's keys above its slice
    uint32_t hres[3];    // histogram path, owner: the bin, the cluster's keys above it / in it
    uint32_t rank_t[2];  // ranking: the threshold key and the candidates above it ([1] = ~0: none)
    int32_t bad;
};

// Order-preserving map float -> uint32 (larger float -> larger key);
// -0 folds onto +0; NaN maps below every number and is reported.
__device__ __forceinline__ uint32_t f2key(float f, bool &nan) {
    uint32_t u = __float_as_uint(f);
    if (f != f) {
        nan = true;
        return 0u;
    }
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

__device__ __forceinline__ uint32_t warp_incl_scan32(uint32_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// 32-bit shared::cluster address of `p` in the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
    uint32_t a;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}
__device__ __forceinline__ uint32_t ld_peer(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_peer(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// The chunk's keys [0, n): the first kCacheElems from shared memory, the rest from global memory.
struct Chunk {
    const float *src;
    int n, ncache;
    bool vec;  // src is 16-byte aligned
    __device__ __forceinline__ uint32_t key(const TopkSmem &s, int i) const {
        bool nan = false;
        return i < ncache ? s.cache[i] : f2key(src[i], nan);
    }
};

// Keys i .. i+3 of the chunk (i a multiple of 4), in two steps so that a loop can start the next
// step's loads before it uses the current keys: keys4_load issues the reads (shared memory, or
// the raw fp32 logits of the part of a long chunk beyond the shared-memory copy: `raw`), and
// keys4_finish turns raw logits into keys.  Positions >= lim read as key 0.
__device__ __forceinline__ void keys4_load(const TopkSmem &s, const Chunk &c, int i, int lim, uint32_t (&k)[4],
                                           bool &raw) {
    raw = false;
    if (i + 3 < c.ncache && i + 3 < lim) {
        const uint4 v = *reinterpret_cast<const uint4 *>(&s.cache[i]);
        k[0] = v.x;
        k[1] = v.y;
        k[2] = v.z;
        k[3] = v.w;
    } else if (i >= c.ncache) {
        raw = true;
        if (c.vec && i + 3 < lim) {
            const int4 v = ldg_nc_v4(c.src + i);
            k[0] = static_cast<uint32_t>(v.x);
            k[1] = static_cast<uint32_t>(v.y);
            k[2] = static_cast<uint32_t>(v.z);
            k[3] = static_cast<uint32_t>(v.w);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) k[q] = (i + q < lim) ? __float_as_uint(__ldg(c.src + i + q)) : 0u;
        }
    } else {  // straddles the end of the shared-memory copy
#pragma unroll
        for (int q = 0; q < 4; ++q) k[q] = (i + q < lim) ? c.key(s, i + q) : 0u;
    }
}

__device__ __forceinline__ void keys4_finish(uint32_t (&k)[4], bool raw, int i, int lim) {
    if (!raw) return;
    bool nan = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) k[q] = (i + q < lim) ? f2key(__uint_as_float(k[q]), nan) : 0u;
}

__device__ __forceinline__ void keys4(const TopkSmem &s, const Chunk &c, int i, int lim, uint32_t (&k)[4]) {
    bool raw;
    keys4_load(s, c, i, lim, k, raw);
    keys4_finish(k, raw, i, lim);
}

// First pass: reads every key of the chunk (16-byte loads, four per thread in
// flight), fills the shared-memory copy and calls f(key).
template <typename F>
__device__ __forceinline__ void first_pass(TopkSmem &s, const Chunk &c, bool &nan, F &&f) {
    const bool vec = (reinterpret_cast<uintptr_t>(c.src) & 15) == 0;
    int i0 = 0;
    if (vec) {
        const int n16 = c.n & ~(16 * kThreads - 1);
        for (; i0 < n16; i0 += 16 * kThreads) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = reinterpret_cast<const float4 *>(c.src + i0)[u * kThreads + threadIdx.x];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + 4 * (u * kThreads + threadIdx.x);
                const uint32_t k4[4] = {f2key(v[u].x, nan), f2key(v[u].y, nan), f2key(v[u].z, nan),
                                        f2key(v[u].w, nan)};
                if (i + 3 < c.ncache) {
                    *reinterpret_cast<uint4 *>(&s.cache[i]) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (i + q < c.ncache) s.cache[i + q] = k4[q];
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) f(k4[q]);
            }
        }
    }
    for (int i = i0 + threadIdx.x; i < c.n; i += kThreads) {
        const uint32_t key = f2key(c.src[i], nan);
        if (i < c.ncache) s.cache[i] = key;
        f(key);
    }
}

// Calls f(key) for every key of the chunk (order irrelevant).
template <typename F>
__device__ __forceinline__ void each_key(const TopkSmem &s, const Chunk &c, F &&f) {
    const int nc4 = c.ncache & ~3;
    for (int i = 4 * threadIdx.x; i < nc4; i += 4 * kThreads) {
        const uint4 k4 = *reinterpret_cast<const uint4 *>(&s.cache[i]);
        f(k4.x);
        f(k4.y);
        f(k4.z);
        f(k4.w);
    }
    // the part beyond the shared-memory copy: eight loads per thread in flight before any use
    for (int i0 = nc4; i0 < c.n; i0 += 8 * kThreads) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * kThreads + threadIdx.x;
            v[u] = i < c.n ? (i < c.ncache ? 0.f : __ldg(c.src + i)) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * kThreads + threadIdx.x;
            if (i < c.n) {
                bool nan = false;
                f(i < c.ncache ? s.cache[i] : f2key(v[u], nan));
            }
        }
    }
}

// Finds the bin holding the need-th largest key, scanning bins from the top.
// cl: the counts deciding the selection; s.hist: this CTA's own counts (the
// same array when the CTA decides alone), left zeroed for the next round.
// Result in s.sel.
__device__ void select_bin(TopkSmem &s, const uint32_t *cl, uint32_t need) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b1 = kBins - 1 - 2 * tid, b0 = b1 - 1;
    const uint32_t c1 = cl[b1], c0 = cl[b0], l1 = s.hist[b1], l0 = s.hist[b0];
    const unsigned long long v = (static_cast<unsigned long long>(l1 + l0) << 32) | (c1 + c0);
    const unsigned long long incl = warp_incl_scan(v, lane);
    if (lane == 31) s.wsum[warp] = incl;
    __syncthreads();
    s.hist[b1] = 0;  // every thread has read its bins
    s.hist[b0] = 0;
    const unsigned long long wincl = warp_incl_scan(s.wsum[lane], lane);
    const unsigned long long wex = warp == 0 ? 0ull : __shfl_sync(0xffffffffu, wincl, (warp + 31) & 31);
    const unsigned long long above = wex + incl - v;
    const uint32_t ca = static_cast<uint32_t>(above), la = static_cast<uint32_t>(above >> 32);
    if (ca < need && need <= ca + c1) {
        s.sel[0] = b1;
        s.sel[1] = ca;
        s.sel[2] = c1;
        s.sel[3] = la;
        s.sel[4] = l1;
    } else if (ca + c1 < need && need <= ca + c1 + c0) {
        s.sel[0] = b0;
        s.sel[1] = ca + c1;
        s.sel[2] = c0;
        s.sel[3] = la + l1;
        s.sel[4] = l0;
    }
    __syncthreads();
}

// Physical slot of position t of a request's block-table row (-1 and a status report when the
// page id is outside the pool), the translation of slots.cu done where the selection is written.
// Pages [pg0, pg0 + npg) come from the shared-memory copy of the chunk's entries.
__device__ __forceinline__ int32_t slot_of(const TopkArgs &a, const int32_t *bt_row, const int32_t *bt_cache,
                                           int pg0, int npg, int32_t t) {
    if (bt_row == nullptr) {
        report(a.status, DSA_ERR_BOUNDS);
        return -1;
    }
    const int pi = t / DSA_PAGE_SIZE;
    const int32_t page = (pi - pg0 >= 0 && pi - pg0 < npg) ? bt_cache[pi - pg0] : bt_row[pi];
    if (page < 0 || page >= a.pool_pages) {
        report(a.status, DSA_ERR_BOUNDS);
        return -1;
    }
    return page * DSA_PAGE_SIZE + t % DSA_PAGE_SIZE;
}

// kHist: start from the scorer's histogram (a.hist); kSlots: also write the slots (a.slots_out).
template <bool kHist, bool kSlots>
__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const TopkArgs a) {
    extern __shared__ uint8_t smem_raw[];
    TopkSmem &s = *reinterpret_cast<TopkSmem *>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int CL = static_cast<int>(cluster.num_blocks());
    const int crank = static_cast<int>(cluster.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x / CL;
    const int k = a.k;
    // nothing to set up on chip: global memory from here on, once the previous kernel has finished
    pdl_launch_dependents();
    pdl_wait();
    int32_t *out = a.idx_out + static_cast<int64_t>(row) * k;
    int32_t *sout = kSlots ? a.slots_out + static_cast<int64_t>(row) * k : nullptr;
    const int32_t *bt_row = nullptr;  // this row's block-table row, when slots are wanted
    if constexpr (kSlots) {
        const int32_t req = a.row_req[row];
        if (req >= 0 && req < a.num_requests) bt_row = a.block_table + static_cast<int64_t>(req) * a.bt_stride;
    }
    int n = a.row_ctx[row];
    if (n < 0 || n > a.max_ctx) {
        if (tid == 0 && crank == 0) report(a.status, DSA_ERR_BOUNDS);
        n = min(max(n, 0), a.max_ctx);
    }
    const int hspan = kHistBins / CL;  // histogram path: this CTA's slice of the row's bins
    uint32_t *hrow = kHist ? a.hist + static_cast<int64_t>(row) * kHistBins : nullptr;
    if (n <= k) {  // the same branch for every CTA of the cluster: no cluster barrier below
        if (crank == 0)
            for (int i = tid; i < k; i += kThreads) {
                out[i] = i < n ? i : -1;
                if constexpr (kSlots) {
                    const int32_t sl = i < n ? slot_of(a, bt_row, nullptr, 0, 0, i) : -1;
                    sout[i] = sl;
                    if (a.warm_pool != nullptr && sl >= 0)
                        bulk_prefetch_l2(a.warm_pool + static_cast<int64_t>(sl) * DSA_LATENT_DIM, DSA_LATENT_DIM);
                }
            }
        if constexpr (kHist)  // leave the scorer's histogram zeroed for the next call
            for (int b = tid; b < hspan; b += kThreads) hrow[crank * hspan + b] = 0u;
        return;
    }
    // this CTA's chunk [c0, c0 + nloc) of the row; chunk starts are multiples of 4 elements
    const int ch = ((n + CL - 1) / CL + 3) & ~3;
    const int c0 = min(n, crank * ch);
    const int nloc = min(n, c0 + ch) - c0;
    const float *csrc = a.logits + static_cast<int64_t>(row) * a.logits_stride + c0;
    Chunk chunk{csrc, nloc, min(nloc, kCacheElems), (reinterpret_cast<uintptr_t>(csrc) & 15) == 0};
    if (tid == 0) {
        s.bad = 0;
        s.ncand = 0;
        s.rank_t[1] = 0xffffffffu;
    }
    for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
    // the chunk's block-table entries, so that writing slots at the end stays local: loaded into
    // registers now, stored after the first pass (the loads overlap it)
    const int pg0 = c0 / DSA_PAGE_SIZE;
    const int npg = (bt_row != nullptr && nloc > 0)
                        ? min(kBtCache, (c0 + nloc - 1) / DSA_PAGE_SIZE - pg0 + 1)
                        : 0;
    static_assert(kBtCache <= 2 * kThreads, "two block-table entries per thread");
    int32_t btr[2] = {0, 0};
#pragma unroll
    for (int q = 0; q < 2; ++q)
        if (tid + q * kThreads < npg) btr[q] = bt_row[pg0 + tid + q * kThreads];
    __syncthreads();

    uint32_t base = 0, top = 0;
    uint32_t need = static_cast<uint32_t>(k);
    uint32_t my_above = 0;                         // this chunk's keys above [base, top]
    uint32_t my_in = static_cast<uint32_t>(nloc);  // this chunk's keys inside it
    uint32_t hist_sc = 0xffffffffu;                // histogram path: the cluster's keys in [base, top]
    bool nan = false;
    if constexpr (kHist) {
        // ---- 1h. the scorer's histogram of this row fixes the 16-bit bin of the k-th key.
        // CTA r scans bin slice r (its threads take `per` consecutive bins each, thread 0 the
        // slice's top ones), the cluster combines the slice totals from the highest slice
        // down, and the owning CTA finds the bin.
        const int per = hspan / kThreads;  // >= 4
        const int hb0 = crank * hspan + hspan - (tid + 1) * per;
        uint32_t tsum = 0;
        for (int q = 0; q < per; ++q) tsum += hrow[hb0 + q];
        const uint32_t tincl = warp_incl_scan32(tsum, lane);
        if (lane == 31) s.red[warp] = tincl;
        __syncthreads();
        const uint32_t wincl = warp_incl_scan32(s.red[lane], lane);
        const uint32_t wex = warp == 0 ? 0u : __shfl_sync(0xffffffffu, wincl, (warp + 31) & 31);
        const uint32_t t_above = wex + tincl - tsum;  // this slice's keys above my bins
        const uint32_t slice_total = __shfl_sync(0xffffffffu, wincl, 31);  // every lane takes part
        if (tid == 0) s.hpub = slice_total;
        cluster.sync();
        if (warp == 0) {
            uint32_t tot = 0;
            if (lane < CL) tot = ld_peer(peer_addr(&s.hpub, lane));
            // slices from the highest rank down: keys above slice r = totals of the ranks > r
            // (an exclusive suffix sum over the lanes)
            uint32_t suf = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t2 = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += t2;
            }
            const uint32_t above_r = suf - tot;
            const bool mine = lane < CL && above_r < need && need <= above_r + tot;
            const unsigned m = __ballot_sync(0xffffffffu, mine);
            const int owner = m ? __ffs(m) - 1 : 0;
            if (lane == owner) {
                s.hsel[0] = static_cast<uint32_t>(owner);
                s.hsel[1] = above_r;
            }
            if (lane == 0) s.hres[0] = 0xffffffffu;  // "not found" unless the owner finds the bin
        }
        __syncthreads();
        const int owner = static_cast<int>(s.hsel[0]);
        if (crank == owner) {
            const uint32_t need_s = need - s.hsel[1];  // rank of the k-th key inside this slice
            if (t_above < need_s && need_s <= t_above + tsum) {
                uint32_t acc = t_above;
                for (int q = per - 1; q >= 0; --q) {
                    const uint32_t c = hrow[hb0 + q];
                    if (acc < need_s && need_s <= acc + c) {
                        s.hres[0] = static_cast<uint32_t>(hb0 + q);  // the bin
                        s.hres[1] = acc + (need - need_s);           // the cluster's keys above it
                        s.hres[2] = c;                               // the cluster's keys in it
                        break;
                    }
                    acc += c;
                }
            }
        }
        cluster.sync();
        if (tid == 0) {
            const uint32_t *hs = cluster.map_shared_rank(s.hres, owner);
            s.range[0] = hs[0];
            s.range[1] = hs[1];
            s.mm[0] = hs[2];
        }
        for (int q = 0; q < per; ++q) hrow[hb0 + q] = 0u;  // left zeroed for the next call
        __syncthreads();
        if (s.range[0] == 0xffffffffu) {
            // the histogram does not describe these logits: report it and search the whole range
            if (tid == 0 && crank == 0) report(a.status, DSA_ERR_RANGE);
            base = 0u;
            top = 0xffffffffu;
        } else {
            need -= s.range[1];
            hist_sc = s.mm[0];
            base = s.range[0] << 16;
            top = base | 0xffffu;
        }
        // one pass over the chunk: shared-memory copy, this chunk's keys above / inside the bin,
        // and its candidates when the cluster's bin fits the candidate list
        const bool collect = hist_sc <= static_cast<uint32_t>(kCandCap);
        uint32_t na = 0, ni = 0;
        first_pass(s, chunk, nan, [&](uint32_t key) {
            if (key > top) {
                ++na;
            } else if (key >= base) {
                ++ni;
                if (collect) {
                    const uint32_t at = atomicAdd(&s.ncand, 1u);
                    if (at < static_cast<uint32_t>(kCandCap)) s.cand[at] = key;
                }
            }
        });
        if (nan) s.bad = 1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            na += __shfl_xor_sync(0xffffffffu, na, o);
            ni += __shfl_xor_sync(0xffffffffu, ni, o);
        }
        __syncthreads();  // s.red is reused
        if (lane == 0) {
            s.red[warp] = na;
            s.red[kWarps + warp] = ni;
        }
        __syncthreads();
        na = s.red[lane];
        ni = s.red[kWarps + lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            na += __shfl_xor_sync(0xffffffffu, na, o);
            ni += __shfl_xor_sync(0xffffffffu, ni, o);
        }
        my_above = na;
        my_in = ni;
        if (tid == 0 && s.bad) report(a.status, DSA_ERR_RANGE);
    } else {
        // ---- 1. key range of the chunk (and its shared-memory copy), then of the row
        uint32_t lo = 0xffffffffu, hi = 0u;
        first_pass(s, chunk, nan, [&](uint32_t key) {
            lo = min(lo, key);
            hi = max(hi, key);
        });
        if (nan) s.bad = 1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) {
            s.red[warp] = lo;
            s.red[kWarps + warp] = hi;
        }
        __syncthreads();
        if (warp == 0) {
            lo = s.red[lane];
            hi = s.red[kWarps + lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            }
            if (lane == 0) {
                s.mm[0] = lo;
                s.mm[1] = hi;
            }
        }
        if (tid == 0 && s.bad) report(a.status, DSA_ERR_RANGE);
        cluster.sync();
        if (warp == 0) {
            lo = 0xffffffffu;
            hi = 0u;
            if (lane < CL) {
                const uint32_t *mm = cluster.map_shared_rank(s.mm, lane);
                lo = mm[0];
                hi = mm[1];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            }
            if (lane == 0) {
                s.range[0] = lo;
                s.range[1] = hi;
            }
        }
        __syncthreads();
            base = s.range[0];
            top = s.range[1];
    }
#pragma unroll
    for (int q = 0; q < 2; ++q)
        if (tid + q * kThreads < npg) s.bt_cache[tid + q * kThreads] = btr[q];
    if (a.discard_logits && chunk.ncache == nloc) {
        // the chunk now lives in shared memory and the logits are scratch: drop the L2 lines
        // that lie wholly inside this chunk, unwritten
        __syncthreads();
        const uintptr_t p0 = (reinterpret_cast<uintptr_t>(chunk.src) + 127) & ~uintptr_t(127);
        const uintptr_t p1 = (reinterpret_cast<uintptr_t>(chunk.src + nloc)) & ~uintptr_t(127);
        for (uintptr_t p = p0 + 128 * static_cast<uintptr_t>(tid); p < p1; p += 128 * kThreads)
            l2_discard_line(reinterpret_cast<const void *>(p));
    }

    // Publish this chunk's candidates and its count above the interval, gather every CTA's
    // candidates in rank order, and arrive on the closing cluster barrier.
    auto publish_and_gather = [&]() {
        if (tid == 0) s.pub[1] = my_above;
        __syncthreads();
        if (tid == 0) s.pub[0] = min(s.ncand, static_cast<uint32_t>(kCandCap));
        cluster.sync();
        if (warp == 0) {
            uint32_t nr = 0, ar = 0;
            if (lane < CL) {
                const uint32_t *pub = cluster.map_shared_rank(s.pub, lane);
                nr = pub[0];
                ar = pub[1];
            }
            const uint32_t incl = warp_incl_scan32(nr, lane);
            if (lane < CL) s.roff[lane] = incl - nr;
            if (lane == CL - 1) s.roff[CL] = incl;
            // selected keys above the interval in the lower-ranked chunks
            const uint32_t ab = warp_incl_scan32(lane < crank ? ar : 0u, lane);
            if (lane == 31) s.before[0] = ab;
        }
        __syncthreads();
        const uint32_t total = s.roff[CL];
        constexpr int kPer = kCandCap / kThreads;
        uint32_t v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {  // all peer loads in flight before any store
            const uint32_t j = tid + u * kThreads;
            if (j < total) {
                int r = 0;
                while (r + 1 < CL && s.roff[r + 1] <= j) ++r;
                v[u] = ld_peer(peer_addr(&s.cand[j - s.roff[r]], r));
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            if (tid + u * kThreads < total) s.cand_all[tid + u * kThreads] = v[u];
        cluster_arrive();  // this CTA reads no peer memory after this point
        __syncthreads();
    };

    bool gathered = false;
    if (kHist && hist_sc <= static_cast<uint32_t>(kCandCap) && top > base) {
        publish_and_gather();  // the bin's candidates were collected in the first pass
        gathered = true;
    }

    // ---- 2. cluster rounds, until the interval is one key or few enough keys to gather
    while (!gathered && top > base) {
        const uint32_t span = top - base;
        const int bits = 32 - __clz(span);            // span < 2^bits
        const int shift = bits > 11 ? bits - 11 : 0;  // (span >> shift) < 2048
        each_key(s, chunk, [&](uint32_t key) {
            if (key >= base && key <= top) atomicAdd(&s.hist[(key - base) >> shift], 1u);
        });
        const uint32_t *cl_counts = s.hist;
        if (CL > 1) {
            cluster.sync();  // every chunk's histogram is complete
            // reduce-scatter: this CTA sums bin slice `crank` over the cluster, writes it to all
            const int slice = (kBins + CL - 1) / CL;
            if (tid < slice && crank * slice + tid < kBins) {
                const int b = crank * slice + tid;
                uint32_t v[kMaxCluster];
#pragma unroll
                for (int r = 0; r < kMaxCluster; ++r)
                    if (r < CL) v[r] = ld_peer(peer_addr(&s.hist[b], r));
                uint32_t sum = 0;
#pragma unroll
                for (int r = 0; r < kMaxCluster; ++r)
                    if (r < CL) sum += v[r];
#pragma unroll
                for (int r = 0; r < kMaxCluster; ++r)
                    if (r < CL) st_peer(peer_addr(&s.hsum[b], r), sum);
            }
            cluster.sync();  // every CTA holds the cluster histogram
            cl_counts = s.hsum;
        } else {
            __syncthreads();
        }
        select_bin(s, cl_counts, need);
        const uint32_t sb = s.sel[0], sa = s.sel[1], sc = s.sel[2];
        my_above += s.sel[3];
        my_in = s.sel[4];
        need -= sa;
        const uint32_t nbase = base + (sb << shift);
        const unsigned long long bin_top = static_cast<unsigned long long>(nbase) + (1ull << shift) - 1ull;
        base = nbase;
        top = static_cast<uint32_t>(min(static_cast<unsigned long long>(top), bin_top));
        if (top > base && sc <= static_cast<uint32_t>(kCandCap)) {
            // publish this chunk's keys inside [base, top] (one shared atomic per warp) and its
            // count above, then gather every CTA's share in rank order
            uint32_t nk[4];
            bool nraw;
            keys4_load(s, chunk, 4 * tid, nloc, nk, nraw);
            for (int i0 = 0; i0 < nloc; i0 += 4 * kThreads) {
                const int i = i0 + 4 * tid;
                uint32_t kq[4] = {nk[0], nk[1], nk[2], nk[3]};
                const bool raw = nraw;
                if (i0 + 4 * kThreads < nloc) keys4_load(s, chunk, i + 4 * kThreads, nloc, nk, nraw);
                keys4_finish(kq, raw, i, nloc);
                uint32_t c = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) c += (i + q < nloc && kq[q] >= base && kq[q] <= top) ? 1u : 0u;
                const uint32_t incl = warp_incl_scan32(c, lane);
                const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
                uint32_t wbase = 0;
                if (lane == 0 && wtot) wbase = atomicAdd(&s.ncand, wtot);
                uint32_t at = __shfl_sync(0xffffffffu, wbase, 0) + incl - c;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (i + q < nloc && kq[q] >= base && kq[q] <= top) s.cand[at++] = kq[q];
            }
            publish_and_gather();
            gathered = true;
            break;
        }
    }

    // ---- 3. refine alone on the gathered candidates
    uint32_t gt_before = 0, eq_before = 0;
    if (gathered) {
        const int nc = static_cast<int>(min(s.roff[CL], static_cast<uint32_t>(kCandCap)));
        if (top > base && nc <= kRankMax) {
            // Few candidates (all inside [base, top]): the threshold is the candidate with fewer
            // than `need` candidates above it and at least `need` at or above it.  Every thread
            // holding that key writes the same two values.
            if (tid < nc) {
                const uint32_t key = s.cand_all[tid];
                uint32_t gt = 0, ge = 0;
                const int nc4 = nc & ~3;
                for (int j = 0; j < nc4; j += 4) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(&s.cand_all[j]);
                    gt += (v.x > key ? 1u : 0u) + (v.y > key ? 1u : 0u) + (v.z > key ? 1u : 0u) + (v.w > key ? 1u : 0u);
                    ge += (v.x >= key ? 1u : 0u) + (v.y >= key ? 1u : 0u) + (v.z >= key ? 1u : 0u) +
                          (v.w >= key ? 1u : 0u);
                }
                for (int j = nc4; j < nc; ++j) {
                    const uint32_t v = s.cand_all[j];
                    gt += v > key ? 1u : 0u;
                    ge += v >= key ? 1u : 0u;
                }
                if (gt < need && need <= ge) {
                    s.rank_t[0] = key;
                    s.rank_t[1] = gt;
                }
            }
            __syncthreads();
            if (s.rank_t[1] != 0xffffffffu) {  // else (inconsistent counts) the rounds below decide
                base = top = s.rank_t[0];
                need -= s.rank_t[1];
            }
        }
        while (top > base) {
            const uint32_t span = top - base;
            const int bits = 32 - __clz(span);
            const int shift = bits > 11 ? bits - 11 : 0;
            for (int i = tid; i < nc; i += kThreads) {
                const uint32_t key = s.cand_all[i];
                if (key >= base && key <= top) atomicAdd(&s.hist[(key - base) >> shift], 1u);
            }
            __syncthreads();
            select_bin(s, s.hist, need);
            need -= s.sel[1];
            const uint32_t nbase = base + (s.sel[0] << shift);
            const unsigned long long bin_top = static_cast<unsigned long long>(nbase) + (1ull << shift) - 1ull;
            base = nbase;
            top = static_cast<uint32_t>(min(static_cast<unsigned long long>(top), bin_top));
        }
        // the lower-ranked chunks' candidates above / equal to T
        const uint32_t T = base;
        const int lower = static_cast<int>(min(s.roff[crank], static_cast<uint32_t>(kCandCap)));
        uint32_t g = 0, e = 0;
        if (lower <= kThreads) {  // one candidate per thread: the barrier counts them
            const uint32_t key = tid < lower ? s.cand_all[tid] : 0u;
            g = static_cast<uint32_t>(__syncthreads_count(tid < lower && key > T));
            e = static_cast<uint32_t>(__syncthreads_count(tid < lower && key == T));
        } else {
            for (int i = tid; i < lower; i += kThreads) {
                const uint32_t key = s.cand_all[i];
                g += key > T;
                e += key == T;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o);
                e += __shfl_xor_sync(0xffffffffu, e, o);
            }
            if (lane == 0) {
                s.red[warp] = g;
                s.red[kWarps + warp] = e;
            }
            __syncthreads();
            g = s.red[lane];
            e = s.red[kWarps + lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o);
                e += __shfl_xor_sync(0xffffffffu, e, o);
            }
        }
        gt_before = s.before[0] + g;
        eq_before = e;
    } else {
        // the cluster rounds reached one key: publish this chunk's counts, read the lower ranks'
        if (tid == 0) {
            s.pub[1] = my_above;
            s.pub[2] = my_in;
        }
        cluster.sync();
        uint32_t g = 0, e = 0;
        if (lane < crank) {
            const uint32_t *pub = cluster.map_shared_rank(s.pub, lane);
            g = pub[1];
            e = pub[2];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        gt_before = g;
        eq_before = e;
        cluster_arrive();
    }
    const uint32_t T = base;  // exact threshold key; `need` keys equal to T are taken (lowest positions)

    // ---- 4. ordered compaction.  Warp w owns a contiguous segment of the chunk and walks it
    // 128 keys at a time, four consecutive keys per lane (lane order = position order).  A
    // selection's output index is its rank among the row's selections in position order, so
    // this chunk's selections fill one contiguous range [p0, p1); they are staged in shared
    // memory (cand_all, free by now) and all threads then write the outputs (and slots) of
    // that range together.
    const int seg = ((nloc + kWarps - 1) / kWarps + 127) & ~127;
    const int w0 = min(nloc, warp * seg), w1 = min(nloc, w0 + seg);
    uint32_t p0, p1;
    if (chunk.ncache == nloc) {
        // One pass: each warp stages the positions of its keys >= T (bit 31 marks == T) in
        // order at the start of its own segment of the shared-memory copy, overwriting keys
        // it has already read (a step's writes end before the step's last key, and every lane
        // has read its keys before the scan that places the writes).  Then each warp walks
        // its short list and keeps the keys > T and the first `need` keys == T of the row.
        uint32_t ns = 0, ngt = 0, neq = 0;
        uint32_t nk[4];
        bool nraw;
        keys4_load(s, chunk, w0 + 4 * lane, w1, nk, nraw);
        for (int i0 = w0; i0 < w1; i0 += 128) {
            const int i = i0 + 4 * lane;
            uint32_t kq[4] = {nk[0], nk[1], nk[2], nk[3]};
            const bool raw = nraw;
            if (i0 + 128 < w1) keys4_load(s, chunk, i + 128, w1, nk, nraw);
            keys4_finish(kq, raw, i, w1);
            uint32_t g = 0, e = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                g += (i + q < w1 && kq[q] > T) ? 1u : 0u;
                e += (i + q < w1 && kq[q] == T) ? 1u : 0u;
            }
            const uint32_t packed = g | (e << 16);  // at most 128 each per warp step
            const uint32_t incl = warp_incl_scan32(packed, lane);
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t ex = incl - packed;
            uint32_t at = static_cast<uint32_t>(w0) + ns + (ex & 0xffffu) + (ex >> 16);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (i + q < w1 && kq[q] >= T)
                    s.cache[at++] = static_cast<uint32_t>(c0 + i + q) | (kq[q] == T ? 0x80000000u : 0u);
            ngt += tot & 0xffffu;
            neq += tot >> 16;
            ns += (tot & 0xffffu) + (tot >> 16);
        }
        if (lane == 0) {
            s.wgt[warp] = ngt;
            s.weq[warp] = neq;
        }
        __syncthreads();
        {
            const uint32_t vg = s.wgt[lane], ve = s.weq[lane];
            const uint32_t ig = warp_incl_scan32(vg, lane), ie = warp_incl_scan32(ve, lane);
            const uint32_t tg = __shfl_sync(0xffffffffu, ig, 31), te = __shfl_sync(0xffffffffu, ie, 31);
            p0 = gt_before + min(eq_before, need);            // selections in the lower chunks
            p1 = gt_before + tg + min(eq_before + te, need);  // ... and in this one
            gt_before += __shfl_sync(0xffffffffu, ig - vg, warp);
            eq_before += __shfl_sync(0xffffffffu, ie - ve, warp);
        }
        const unsigned lt = (1u << lane) - 1u;
        for (uint32_t j0 = 0; j0 < ns; j0 += 32) {
            const uint32_t j = j0 + lane;
            const uint32_t v = j < ns ? s.cache[w0 + j] : 0u;
            const bool is_eq = j < ns && (v >> 31) != 0u, is_gt = j < ns && (v >> 31) == 0u;
            const unsigned bg = __ballot_sync(0xffffffffu, is_gt), be = __ballot_sync(0xffffffffu, is_eq);
            const uint32_t gb = gt_before + __popc(bg & lt), eb = eq_before + __popc(be & lt);
            if (is_gt || (is_eq && eb < need)) {
                const uint32_t pos = gb + min(eb, need);
                if (pos >= p0 && pos < p1 && pos < static_cast<uint32_t>(k))
                    s.cand_all[pos - p0] = v & 0x7fffffffu;
                else
                    report(a.status, DSA_ERR_BOUNDS);  // inconsistent counts: never expected
            }
            gt_before += __popc(bg);
            eq_before += __popc(be);
        }
    } else {
        // Chunk larger than the shared-memory copy: pass 1 counts keys > T and == T per warp,
        // pass 2 places each selected position after the lower warps' and chunks' selections.
        uint32_t ngt = 0, neq = 0;
        uint32_t nk[4];
        bool nraw;
        keys4_load(s, chunk, w0 + 4 * lane, w1, nk, nraw);
        for (int i0 = w0; i0 < w1; i0 += 128) {
            const int i = i0 + 4 * lane;
            uint32_t kq[4] = {nk[0], nk[1], nk[2], nk[3]};
            const bool raw = nraw;
            if (i0 + 128 < w1) keys4_load(s, chunk, i + 128, w1, nk, nraw);
            keys4_finish(kq, raw, i, w1);
            uint32_t g = 0, e = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                g += (i + q < w1 && kq[q] > T) ? 1u : 0u;
                e += (i + q < w1 && kq[q] == T) ? 1u : 0u;
            }
            ngt += __reduce_add_sync(0xffffffffu, g);
            neq += __reduce_add_sync(0xffffffffu, e);
        }
        if (lane == 0) {
            s.wgt[warp] = ngt;
            s.weq[warp] = neq;
        }
        __syncthreads();
        {
            const uint32_t vg = s.wgt[lane], ve = s.weq[lane];
            const uint32_t ig = warp_incl_scan32(vg, lane), ie = warp_incl_scan32(ve, lane);
            const uint32_t tg = __shfl_sync(0xffffffffu, ig, 31), te = __shfl_sync(0xffffffffu, ie, 31);
            p0 = gt_before + min(eq_before, need);            // selections in the lower chunks
            p1 = gt_before + tg + min(eq_before + te, need);  // ... and in this one
            gt_before += __shfl_sync(0xffffffffu, ig - vg, warp);
            eq_before += __shfl_sync(0xffffffffu, ie - ve, warp);
        }
        keys4_load(s, chunk, w0 + 4 * lane, w1, nk, nraw);
        for (int i0 = w0; i0 < w1; i0 += 128) {
            const int i = i0 + 4 * lane;
            uint32_t kq[4] = {nk[0], nk[1], nk[2], nk[3]};
            const bool raw = nraw;
            if (i0 + 128 < w1) keys4_load(s, chunk, i + 128, w1, nk, nraw);
            keys4_finish(kq, raw, i, w1);
            uint32_t g = 0, e = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                g += (i + q < w1 && kq[q] > T) ? 1u : 0u;
                e += (i + q < w1 && kq[q] == T) ? 1u : 0u;
            }
            // counts of >T and ==T packed in one word: at most 128 each per warp step
            const uint32_t packed = g | (e << 16);
            const uint32_t incl = warp_incl_scan32(packed, lane);
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            uint32_t gb = gt_before + ((incl - packed) & 0xffffu), eb = eq_before + ((incl - packed) >> 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool in = i + q < w1;
                const bool gt = in && kq[q] > T, eq = in && kq[q] == T;
                if (gt || (eq && eb < need)) {
                    const uint32_t pos = gb + min(eb, need);
                    if (pos >= p0 && pos < p1 && pos < static_cast<uint32_t>(k))
                        s.cand_all[pos - p0] = static_cast<uint32_t>(c0 + i + q);
                    else
                        report(a.status, DSA_ERR_BOUNDS);  // inconsistent counts: never expected
                }
                gb += gt ? 1u : 0u;
                eb += eq ? 1u : 0u;
            }
            gt_before += tot & 0xffffu;
            eq_before += tot >> 16;
        }
    }
    __syncthreads();
    const uint32_t pe = min(p1, static_cast<uint32_t>(k));  // p1 - p0 <= k <= kCandCap
    for (uint32_t j = p0 + tid; j < pe; j += kThreads) {
        const int32_t t = static_cast<int32_t>(s.cand_all[j - p0]);
        out[j] = t;
        if constexpr (kSlots) {
            const int32_t sl = slot_of(a, bt_row, s.bt_cache, pg0, npg, t);
            sout[j] = sl;
            if (a.warm_pool != nullptr && sl >= 0)
                bulk_prefetch_l2(a.warm_pool + static_cast<int64_t>(sl) * DSA_LATENT_DIM, DSA_LATENT_DIM);
        }
    }
    cluster_wait();  // no CTA leaves while a peer may still read its shared memory
}

struct ClusterLimits {
    int device = -1;
    int max_clusters[kMaxCluster + 1] = {0};  // co-resident clusters of each size (0: not launchable)
};

// CTAs per row: at least enough that a chunk fits the shared-memory copy, as many as keep the
// batch within the SMs (chunks not shorter than kMinChunk), and no more than the GPU holds
// `num_rows` co-resident clusters of (a second wave would double the time).  The histogram-seeded
// variant splits the 65,536 scorer bins evenly over the cluster: powers of two only.
int cluster_size_for(const TopkArgs &a, int sms, const ClusterLimits &lim, bool pow2_only) {
    int fit = 1;
    while (fit < kMaxCluster && (a.max_ctx + fit - 1) / fit > kCacheElems) fit = pow2_only ? 2 * fit : fit + 1;
    int par = 1;
    while (true) {
        const int nxt = pow2_only ? 2 * par : par + 1;
        if (nxt > kMaxCluster || nxt * a.num_rows > sms || a.max_ctx / nxt < kMinChunk) break;
        par = nxt;
    }
    int cl = fit > par ? fit : par;
    while (cl > 1 && lim.max_clusters[cl] < a.num_rows) cl = pow2_only ? cl / 2 : cl - 1;
    return cl;
}

template <bool kHist, bool kSlots>
cudaError_t launch_variant(const TopkArgs &a, cudaStream_t s) {
    static ClusterLimits lim;
    auto kern = topk_kernel<kHist, kSlots>;
    int dev = 0;
    cudaGetDevice(&dev);
    if (lim.device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(TopkSmem));
        if (e != cudaSuccess) return e;
        const bool nonportable = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                                 cudaSuccess;
        for (int c = 1; c <= kMaxCluster; ++c) {
            lim.max_clusters[c] = 0;
            if (c > 8 && !nonportable) continue;
            cudaLaunchConfig_t probe = {};
            probe.gridDim = dim3(c);
            probe.blockDim = dim3(kThreads);
            probe.dynamicSmemBytes = sizeof(TopkSmem);
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = c;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            probe.attrs = at;
            probe.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &probe) == cudaSuccess) lim.max_clusters[c] = n;
        }
        cudaGetLastError();  // a refused cluster size only disables it
        lim.device = dev;
    }
    const int cl = cluster_size_for(a, device_sm_count(), lim, kHist);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.num_rows * cl));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(TopkSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// ---------------------------------------------------------------- histogram selection
//
// For a few long rows, with a caller workspace.  Each row is cut into chunks that independent CTAs
// (no clusters, two per SM) handle in three launches:
//   count:   each chunk counts its keys' top 12 bits (sign, exponent and 3 mantissa bits of the
//            logit: one bin per 1/8 binade) and writes its nonzero bins as a short list;
//   collect: each chunk adds its row's lists into the row's histogram, finds the bin B that holds
//            the row's k-th largest key, and writes its own keys in bins >= B, in position order,
//            to the row's candidate array (at the offset the lists give for the chunks before it);
//   select:  each chunk finds the exact threshold T among the row's candidates in bin B and writes
//            its share of the selection (its keys above T, and keys equal to T while the row's
//            ties last) at the offset that the candidates of the chunks before it give, with the
//            slots and the latent prefetches.
// By construction that is the whole row's selection by (key desc, position asc).  A row whose bin B
// holds more than kHsInCap keys (ties, or scores within 1/8 binade) is selected from its whole
// logits by one CTA instead: slower, exact.

constexpr int kHsThreads = 512;
constexpr int kHsWarps = kHsThreads / 32;
constexpr int kHsBins = 4096;
constexpr int kHsShift = 20;  // bin of a key: key >> kHsShift
constexpr uint32_t kHsCountMask = (1u << kHsShift) - 1u;
static_assert(kChunkMaxKeys <= static_cast<int>(kHsCountMask), "a list entry holds a chunk's count");
constexpr int kHsCacheChunks = 96;  // the collect kernel keeps the first kHsCacheLen entries of
constexpr int kHsCacheLen = 64;     // the lists of this many chunks in shared memory
constexpr int kHsMaxChunks = 1024;

// Block-wide: the bin holding the need-th largest key of `hist` (NB counts, scanned from the
// top): res[0] = bin, res[1] = keys above it, res[2] = keys in it.
template <int NT, int NB = kBins>
__device__ void find_bin(const uint32_t *hist, uint32_t need, uint32_t *wred, uint32_t *res) {
    constexpr int per = NB / NT;
    static_assert(per >= 1 && NB % NT == 0, "whole bins per thread");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b_hi = NB - 1 - per * tid;  // this thread: bins b_hi, b_hi - 1, ..., b_hi - per + 1
    uint32_t c[per], tsum = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) {
        c[q] = hist[b_hi - q];
        tsum += c[q];
    }
    const uint32_t incl = warp_incl_scan32(tsum, lane);
    if (lane == 31) wred[warp] = incl;
    __syncthreads();
    const uint32_t wincl = warp_incl_scan32(lane < NT / 32 ? wred[lane] : 0u, lane);
    const uint32_t wex = warp == 0 ? 0u : __shfl_sync(0xffffffffu, wincl, (warp + 31) & 31);
    const uint32_t above = wex + incl - tsum;
    if (above < need && need <= above + tsum) {
        uint32_t acc = above;
#pragma unroll
        for (int q = 0; q < per; ++q) {
            if (acc < need && need <= acc + c[q]) {
                res[0] = static_cast<uint32_t>(b_hi - q);
                res[1] = acc;
                res[2] = c[q];
            }
            acc += c[q];
        }
    }
    __syncthreads();
}

// The need-th largest of items 0 .. n-1 (their keys from key_at, all within [lo, hi]), exactly:
// T and need_eq = how many items with key T the selection takes (it takes every key above T).
template <int NT, typename KeyAt>
__device__ void find_threshold(int n, KeyAt key_at, uint32_t lo, uint32_t hi, uint32_t need, uint32_t *hist,
                               uint32_t *wred, uint32_t *res, uint32_t &T, uint32_t &need_eq) {
    uint32_t base = lo, top = hi;
    while (top > base) {
        const uint32_t span = top - base;
        const int bits = 32 - __clz(span);
        const int shift = bits > 11 ? bits - 11 : 0;  // (span >> shift) < 2048 bins
        for (int b = threadIdx.x; b < kBins; b += NT) hist[b] = 0u;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += NT) {
            const uint32_t key = key_at(i);
            if (key >= base && key <= top) atomicAdd(&hist[(key - base) >> shift], 1u);
        }
        __syncthreads();
        find_bin<NT>(hist, need, wred, res);
        need -= res[1];
        const uint32_t nbase = base + (res[0] << shift);
        const unsigned long long bin_top = static_cast<unsigned long long>(nbase) + (1ull << shift) - 1ull;
        base = nbase;
        top = static_cast<uint32_t>(min(static_cast<unsigned long long>(top), bin_top));
        __syncthreads();  // res is rewritten by the next round
    }
    T = base;
    need_eq = need;
}

// Calls emit(j, i), in item order, for every item whose key is above T and for the first need_eq
// items whose key equals T; j is the item's rank among the emitted ones (its output index).
// Warps own contiguous item segments: one pass counts, the second places.
template <int NT, typename KeyAt, typename Emit>
__device__ void emit_ordered(int n, KeyAt key_at, uint32_t T, uint32_t need_eq, uint32_t *wgt, uint32_t *weq,
                             Emit emit) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = (((n + NW - 1) / NW) + 31) & ~31;
    const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
    uint32_t g = 0, e = 0;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t key = i < w1 ? key_at(i) : 0u;
        g += __popc(__ballot_sync(0xffffffffu, i < w1 && key > T));
        e += __popc(__ballot_sync(0xffffffffu, i < w1 && key == T));
    }
    if (lane == 0) {
        wgt[warp] = g;
        weq[warp] = e;
    }
    __syncthreads();
    uint32_t gb = 0, eb = 0;  // the lower warps' counts
    for (int w = 0; w < warp; ++w) {
        gb += wgt[w];
        eb += weq[w];
    }
    const unsigned lt = (1u << lane) - 1u;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t key = i < w1 ? key_at(i) : 0u;
        const bool is_gt = i < w1 && key > T, is_eq = i < w1 && key == T;
        const unsigned bg = __ballot_sync(0xffffffffu, is_gt), be = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t eq_rank = eb + __popc(be & lt);
        if (is_gt || (is_eq && eq_rank < need_eq)) emit(gb + __popc(bg & lt) + min(eq_rank, need_eq), i);
        gb += __popc(bg);
        eb += __popc(be);
    }
    __syncthreads();
}

// Block-wide min and max of (lo, hi) over the threads, into res[0], res[1].
template <int NT>
__device__ void block_minmax(uint32_t lo, uint32_t hi, uint32_t *wred, uint32_t *res) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
        wred[warp] = lo;
        wred[32 + warp] = hi;
    }
    __syncthreads();
    if (warp == 0) {
        lo = lane < NT / 32 ? wred[lane] : 0xffffffffu;
        hi = lane < NT / 32 ? wred[32 + lane] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) {
            res[0] = lo;
            res[1] = hi;
        }
    }
    __syncthreads();
}


// Warp-wide sums of two counters.
__device__ __forceinline__ void warp_sum2(uint32_t &x, uint32_t &y) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        x += __shfl_xor_sync(0xffffffffu, x, o);
        y += __shfl_xor_sync(0xffffffffu, y, o);
    }
}

// Logits i .. i+3 of a chunk (i a multiple of 4), 0 at or past lim: one 16-byte load when all four
// are below lim and the chunk start is 16-byte aligned (vec), else one load per logit.
__device__ __forceinline__ float4 ld4(const float *src, int i, int lim, bool vec) {
    if (vec && i + 3 < lim) return __ldg(reinterpret_cast<const float4 *>(src + i));
    float4 v;
    v.x = i < lim ? __ldg(src + i) : 0.f;
    v.y = i + 1 < lim ? __ldg(src + i + 1) : 0.f;
    v.z = i + 2 < lim ? __ldg(src + i + 2) : 0.f;
    v.w = i + 3 < lim ? __ldg(src + i + 3) : 0.f;
    return v;
}

constexpr int kHsUnroll = 8;  // 16-byte loads per thread in flight

// Asynchronous global -> shared copies (cp.async) of 16 bytes (both addresses 16-byte aligned) or
// 4 bytes, committed as a group and waited for all together.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_groups() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Count: CTA (row, c) writes chunk c's nonzero bins, ascending, as bin << kHsShift | count.
__global__ void __launch_bounds__(kHsThreads, 2) topk_hs_count_kernel(const TopkArgs a) {
    __shared__ uint32_t hist[kHsBins];
    __shared__ uint32_t wsum[kHsWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < kHsBins; b += kHsThreads) hist[b] = 0u;
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x / a.chunks, c = blockIdx.x % a.chunks;
    const int L = min(max(a.row_ctx[row], 0), a.max_ctx);
    if (L <= a.k) return;  // the select kernel writes such rows whole
    const int c0 = c * a.chunk_len;
    const int n = max(0, min(L, c0 + a.chunk_len) - c0);
    const int64_t slot = static_cast<int64_t>(row) * a.chunks + c;
    const float *src = a.logits + static_cast<int64_t>(row) * a.logits_stride + c0;
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0u;
    __syncthreads();  // hist is zeroed
    bool nan = false;
    for (int i0 = 0; i0 < n; i0 += kHsUnroll * 4 * kHsThreads) {
        float4 v[kHsUnroll];
#pragma unroll
        for (int u = 0; u < kHsUnroll; ++u) v[u] = ld4(src, i0 + (u * kHsThreads + tid) * 4, n, vec);
#pragma unroll
        for (int u = 0; u < kHsUnroll; ++u) {
            const int i = i0 + (u * kHsThreads + tid) * 4;
            const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (i + q < n) atomicAdd(&hist[f2key(x[q], nan) >> kHsShift], 1u);
        }
    }
    if (nan) report(a.status, DSA_ERR_RANGE);
    __syncthreads();
    constexpr int per = kHsBins / kHsThreads;  // thread t: bins per * t .. per * t + per - 1
    uint32_t cnt[per], nz = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) {
        cnt[q] = hist[per * tid + q];
        nz += cnt[q] != 0u ? 1u : 0u;
    }
    const uint32_t incl = warp_incl_scan32(nz, lane);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    uint32_t at = incl - nz;
    for (int w = 0; w < warp; ++w) at += wsum[w];
    uint32_t *list = a.hs_list + slot * kHsBins;
#pragma unroll
    for (int q = 0; q < per; ++q)
        if (cnt[q] != 0u) list[at++] = static_cast<uint32_t>(per * tid + q) << kHsShift | cnt[q];
    if (tid == kHsThreads - 1) a.hs_nlist[slot] = at;
}

// Collect: CTA (row, c) sums the row's lists, finds the threshold bin B (the row's meta is written
// by chunk 0), and writes chunk c's keys in bins >= B with their positions, in position order, at
// the row's candidates before which the chunks 0 .. c-1 put theirs.
__global__ void __launch_bounds__(kHsThreads, 2) topk_hs_collect_kernel(const TopkArgs a) {
    extern __shared__ __align__(16) uint32_t hc_smem[];
    uint32_t *hist = hc_smem;                   // [kHsBins]
    uint32_t *keys = hist + kHsBins;            // [chunk_len] the chunk's keys
    uint32_t *lcache = keys + a.chunk_len;      // [kHsCacheChunks][kHsCacheLen] the lists' first entries
    uint32_t *nl = lcache + kHsCacheChunks * kHsCacheLen;  // [chunks] the lists' lengths
    __shared__ uint32_t wred[64], res[8], wcnt[kHsWarps], before;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < kHsBins; b += kHsThreads) hist[b] = 0u;
    if (tid == 0) before = 0u;
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x / a.chunks, c = blockIdx.x % a.chunks;
    const int L = min(max(a.row_ctx[row], 0), a.max_ctx);
    if (L <= a.k) return;
    const int nch = (L + a.chunk_len - 1) / a.chunk_len;
    if (c >= nch) return;
    const int64_t rslot = static_cast<int64_t>(row) * a.chunks;
    const uint32_t *lists = a.hs_list + rslot * kHsBins;
    // the chunk's logits into shared memory (as raw floats), copied while the lists are read
    const int c0 = c * a.chunk_len;
    const int n = min(L, c0 + a.chunk_len) - c0;
    {
        const float *src = a.logits + static_cast<int64_t>(row) * a.logits_stride + c0;
        int i = tid;
        if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0u) {
            const int n4 = n >> 2;
            for (; i < n4; i += kHsThreads) cp_async_16(keys + 4 * i, src + 4 * i);
            i = 4 * n4 + tid;
        }
        for (; i < n; i += kHsThreads) cp_async_4(keys + i, src + i);
        cp_async_commit_group();
    }
    __syncthreads();  // hist and before are zeroed
    // the row's histogram from the chunks' lists: warp w takes chunks w, w + kHsWarps, ...; a lane
    // loads a list's length with its entries lane and lane + 32 in one round, four lists at a time
    // (entries past the length are not used), and the rest of longer lists after
    for (int cc0 = warp; cc0 < nch; cc0 += 4 * kHsWarps) {
        uint32_t m[4], e0[4], e1[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int cc = cc0 + q * kHsWarps;
            m[q] = e0[q] = e1[q] = 0u;
            if (cc < nch) {
                const uint32_t *l = lists + static_cast<int64_t>(cc) * kHsBins;
                m[q] = __ldg(a.hs_nlist + rslot + cc);
                e0[q] = __ldg(l + lane);
                e1[q] = __ldg(l + lane + 32);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int cc = cc0 + q * kHsWarps;
            if (cc >= nch) continue;
            const int mm = static_cast<int>(min(m[q], static_cast<uint32_t>(kHsBins)));
            const bool keep = cc < kHsCacheChunks;
            if (lane == 0) nl[cc] = static_cast<uint32_t>(mm);
            if (lane < mm) {
                atomicAdd(&hist[e0[q] >> kHsShift], e0[q] & kHsCountMask);
                if (keep) lcache[cc * kHsCacheLen + lane] = e0[q];
            }
            if (lane + 32 < mm) {
                atomicAdd(&hist[e1[q] >> kHsShift], e1[q] & kHsCountMask);
                if (keep) lcache[cc * kHsCacheLen + lane + 32] = e1[q];
            }
            for (int j = kHsCacheLen + lane; j < mm; j += 32) {
                const uint32_t e = __ldg(lists + static_cast<int64_t>(cc) * kHsBins + j);
                atomicAdd(&hist[e >> kHsShift], e & kHsCountMask);
            }
        }
    }
    __syncthreads();
    find_bin<kHsThreads, kHsBins>(hist, static_cast<uint32_t>(a.k), wred, res);
    const uint32_t B = res[0], inb = res[2];
    if (c == 0 && tid == 0) {
        uint32_t *rm = a.hs_row + static_cast<int64_t>(row) * 4;
        rm[0] = B;
        rm[1] = res[1];
        rm[2] = inb;
    }
    if (inb > static_cast<uint32_t>(kHsInCap)) {  // the select kernel takes the row from its logits
        cp_async_wait_all();
        return;
    }
    // the candidates of chunks 0 .. c-1: their lists' counts in bins >= B
    uint32_t part = 0;
    for (int cc = warp; cc < c; cc += kHsWarps) {
        const int mm = static_cast<int>(nl[cc]);
        for (int j = lane; j < mm; j += 32) {
            const uint32_t e = (j < kHsCacheLen && cc < kHsCacheChunks)
                                   ? lcache[cc * kHsCacheLen + j]
                                   : __ldg(lists + static_cast<int64_t>(cc) * kHsBins + j);
            if ((e >> kHsShift) >= B) part += e & kHsCountMask;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0 && part != 0u) atomicAdd(&before, part);
    // this chunk's keys in bins >= B: warps own contiguous segments (multiples of 128 keys); one
    // pass turns the copied logits into keys and counts, the second places
    const uint32_t thr = B << kHsShift;
    const int seg = (((n + kHsWarps - 1) / kHsWarps) + 127) & ~127;
    const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
    bool nan = false;  // reported by the count kernel
    uint32_t g = 0;
    cp_async_wait_all();
    __syncthreads();  // every thread's copies have landed
    for (int i = w0 + 4 * lane; i < w1; i += 128) {
        if (i + 3 < w1) {
            const uint4 f = *reinterpret_cast<const uint4 *>(keys + i);
            const uint4 k4 = make_uint4(f2key(__uint_as_float(f.x), nan), f2key(__uint_as_float(f.y), nan),
                                        f2key(__uint_as_float(f.z), nan), f2key(__uint_as_float(f.w), nan));
            *reinterpret_cast<uint4 *>(keys + i) = k4;
            g += (k4.x >= thr ? 1u : 0u) + (k4.y >= thr ? 1u : 0u) + (k4.z >= thr ? 1u : 0u) + (k4.w >= thr ? 1u : 0u);
        } else {
            for (int q = i; q < w1; ++q) {
                const uint32_t key = f2key(__uint_as_float(keys[q]), nan);
                keys[q] = key;
                g += key >= thr ? 1u : 0u;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
    if (lane == 0) wcnt[warp] = g;
    __syncthreads();
    const uint32_t off = before;
    uint32_t base = off, total = 0;
    for (int w = 0; w < kHsWarps; ++w) {
        base += w < warp ? wcnt[w] : 0u;
        total += wcnt[w];
    }
    const int64_t rbase = static_cast<int64_t>(row) * a.row_cap;
    const unsigned lt = (1u << lane) - 1u;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t key = i < w1 ? keys[i] : 0u;
        const bool take = i < w1 && key >= thr;
        const unsigned m = __ballot_sync(0xffffffffu, take);
        const uint32_t at = base + __popc(m & lt);
        if (take && at < static_cast<uint32_t>(a.row_cap)) {
            a.hs_key[rbase + at] = key;
            a.hs_pos[rbase + at] = c0 + i;
        }
        base += __popc(m);
    }
    if (tid == 0) {
        a.hs_chunk[(rslot + c) * 2] = off;
        a.hs_chunk[(rslot + c) * 2 + 1] = total;
    }
}

constexpr int kHsBtCache = kChunkMaxKeys / DSA_PAGE_SIZE;  // block-table entries of a chunk
constexpr int kHsSpecKeys = 4096;  // candidates the select kernel copies before their number is known
constexpr int kHsRankMax = 64;     // a threshold sub-bin of up to this many keys is resolved by ranking

// The need-th largest key among those of ckey[0 .. M) that lie in bin B (1 <= need <= their number),
// exactly: T, and need_eq = how many keys equal to T the selection takes.  One round counts 2048
// sub-bins of 512 keys each; the keys of the chosen sub-bin are then ranked against each other
// when they are few, else counted in a second round of 512 bins.  Block-wide; the caller has
// zeroed hist[0 .. kBins) and res[4], with a barrier since.
__device__ void threshold_in_bin(const uint32_t *ckey, int M, uint32_t B, uint32_t need, uint32_t *hist,
                                 uint32_t *wred, uint32_t *res, uint32_t &T, uint32_t &need_eq) {
    const int tid = threadIdx.x, lane = tid & 31;
    for (int j = tid; j < M; j += kHsThreads) {
        const uint32_t key = ckey[j];
        if ((key >> kHsShift) == B) atomicAdd(&hist[(key >> 9) & (kBins - 1)], 1u);
    }
    __syncthreads();
    find_bin<kHsThreads>(hist, need, wred, res);
    const uint32_t sub = ((B << kHsShift) | (res[0] << 9)) >> 9;  // the sub-bin: keys >> 9 == sub
    const uint32_t n_in = res[2];
    need -= res[1];
    if (n_in <= static_cast<uint32_t>(kHsRankMax)) {
        uint32_t *cand = hist;  // the sub-bin's keys, in any order
        const unsigned lt = (1u << lane) - 1u;
        for (int j0 = 0; j0 < M; j0 += kHsThreads) {
            const int j = j0 + tid;
            const uint32_t key = j < M ? ckey[j] : 0u;
            const bool in = j < M && (key >> 9) == sub;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            uint32_t p = 0;
            if (lane == 0 && m != 0u) p = atomicAdd(&res[4], static_cast<uint32_t>(__popc(m)));
            p = __shfl_sync(0xffffffffu, p, 0) + __popc(m & lt);
            if (in && p < static_cast<uint32_t>(kHsRankMax)) cand[p] = key;
        }
        __syncthreads();
        if (tid < static_cast<int>(n_in)) {
            const uint32_t x = cand[tid];
            uint32_t gt = 0, eq = 0;
            for (int i = 0; i < static_cast<int>(n_in); ++i) {
                gt += cand[i] > x ? 1u : 0u;
                eq += cand[i] == x ? 1u : 0u;
            }
            if (gt < need && need <= gt + eq) {  // every key equal to x writes the same values
                res[5] = x;
                res[6] = need - gt;
            }
        }
        __syncthreads();
        T = res[5];
        need_eq = res[6];
    } else {
        for (int b = tid; b < 512; b += kHsThreads) hist[b] = 0u;
        __syncthreads();
        for (int j = tid; j < M; j += kHsThreads) {
            const uint32_t key = ckey[j];
            if ((key >> 9) == sub) atomicAdd(&hist[key & 511u], 1u);
        }
        __syncthreads();
        find_bin<kHsThreads, 512>(hist, need, wred, res);
        T = (sub << 9) | res[0];
        need_eq = need - res[1];
    }
    __syncthreads();  // res and hist are reused
}

// Select: CTA (row, c) writes chunk c's share of the row's selection (ascending positions), its
// slots and the latent prefetches; CTA (row, 0) writes rows of at most k keys, and rows whose
// threshold bin overflowed, whole.
template <bool kSlots>
__global__ void __launch_bounds__(kHsThreads, 2) topk_hs_select_kernel(const TopkArgs a) {
    extern __shared__ __align__(16) uint32_t hsel_smem[];
    uint32_t *ckey = hsel_smem;                                // [row_cap] the row's candidates' keys
    uint32_t *hist = ckey + a.row_cap;                         // [kBins]
    int32_t *sel = reinterpret_cast<int32_t *>(hist + kBins);  // [k] the chunk's first candidate positions
    int32_t *btc = sel + a.k;                                  // [kHsBtCache] the chunk's page ids
    __shared__ uint32_t wred[64], res[8], wgt[32], weq[32], cnt[2];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int b = tid; b < kBins; b += kHsThreads) hist[b] = 0u;  // for threshold_in_bin
    if (tid == 0) res[4] = 0u;
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x / a.chunks, c = blockIdx.x % a.chunks, k = a.k;
    const int64_t rbase = static_cast<int64_t>(row) * a.row_cap;
    const uint32_t *rk = a.hs_key + rbase;
    const int32_t *rp = a.hs_pos + rbase;
    // the row's first candidates are copied before their number is known (most rows have fewer;
    // the rest follow), and what the CTA reads next is loaded meanwhile (the meta of rows and
    // chunks without candidates is not used)
    const int spec = min(kHsSpecKeys, a.row_cap);
    for (int j = tid; 4 * j < spec; j += kHsThreads) cp_async_16(ckey + 4 * j, rk + 4 * j);
    cp_async_commit_group();
    int n = a.row_ctx[row];
    const uint32_t *rm = a.hs_row + static_cast<int64_t>(row) * 4;
    const uint32_t *cm = a.hs_chunk + (static_cast<int64_t>(row) * a.chunks + c) * 2;
    const uint32_t B = rm[0], above = rm[1], inb = rm[2];
    const uint32_t off_raw = cm[0], own_raw = cm[1];
    int32_t *out = a.idx_out + static_cast<int64_t>(row) * k;
    int32_t *sout = kSlots ? a.slots_out + static_cast<int64_t>(row) * k : nullptr;
    const int32_t *bt_row = nullptr;
    if constexpr (kSlots) {
        const int32_t req = a.row_req[row];
        if (req >= 0 && req < a.num_requests) bt_row = a.block_table + static_cast<int64_t>(req) * a.bt_stride;
    }
    int pg0 = 0, npg = 0;  // pages of the block-table cache
    auto put_out = [&](int j, int32_t t) {  // output j of the row: token t (-1: none)
        out[j] = t;
        if constexpr (kSlots) {
            const int32_t sl = t >= 0 ? slot_of(a, bt_row, btc, pg0, npg, t) : -1;
            sout[j] = sl;
            if (a.warm_pool != nullptr && sl >= 0)
                bulk_prefetch_l2(a.warm_pool + static_cast<int64_t>(sl) * DSA_LATENT_DIM, DSA_LATENT_DIM);
        }
    };
    if (n < 0 || n > a.max_ctx) {
        if (c == 0 && tid == 0) report(a.status, DSA_ERR_BOUNDS);
        n = min(max(n, 0), a.max_ctx);
    }
    if (n <= k) {
        if (c == 0)
            for (int j = tid; j < k; j += kHsThreads) put_out(j, j < n ? j : -1);
        cp_async_wait_all();
        return;
    }
    const int nch = (n + a.chunk_len - 1) / a.chunk_len;
    if (c >= nch || (inb > static_cast<uint32_t>(kHsInCap) && c != 0)) {
        cp_async_wait_all();
        return;
    }
    if (inb > static_cast<uint32_t>(kHsInCap)) {
        // the row's whole logits (the candidates were not written)
        const float *src = a.logits + static_cast<int64_t>(row) * a.logits_stride;
        auto gkey = [&](int i) {
            bool nan = false;
            return f2key(__ldg(src + i), nan);
        };
        uint32_t lo = 0xffffffffu, hi = 0u;
        for (int i = tid; i < n; i += kHsThreads) {
            const uint32_t key = gkey(i);
            lo = min(lo, key);
            hi = max(hi, key);
        }
        block_minmax<kHsThreads>(lo, hi, wred, res);
        lo = res[0];
        hi = res[1];
        __syncthreads();
        uint32_t T, need_eq;
        find_threshold<kHsThreads>(n, gkey, lo, hi, static_cast<uint32_t>(k), hist, wred, res, T, need_eq);
        emit_ordered<kHsThreads>(n, gkey, T, need_eq, wgt, weq, [&](uint32_t j, int i) {
            if (j < static_cast<uint32_t>(k)) sel[j] = i;
        });
        for (int j = tid; j < k; j += kHsThreads) put_out(j, sel[j]);
        cp_async_wait_all();
        return;
    }
    const int M = min(static_cast<int>(above + inb), a.row_cap);
    const int off = min(static_cast<int>(off_raw), M), own = min(static_cast<int>(own_raw), M - off);
    if (tid < 2) cnt[tid] = 0u;
    // the rest of the candidates; then the chunk's first k candidate positions and its block-table
    // entries, needed only once the threshold is known
    for (int j = spec + tid; j < M; j += kHsThreads) cp_async_4(ckey + j, rk + j);
    cp_async_commit_group();
    const int ocache = min(own, k);
    for (int i = tid; i < ocache; i += kHsThreads) cp_async_4(sel + i, rp + off + i);
    if constexpr (kSlots) {
        const int c0 = c * a.chunk_len;
        pg0 = c0 / DSA_PAGE_SIZE;
        npg = min((min(n, c0 + a.chunk_len) - c0 + DSA_PAGE_SIZE - 1) / DSA_PAGE_SIZE, kHsBtCache);
        if (bt_row != nullptr)
            for (int i = tid; i < npg; i += kHsThreads) cp_async_4(btc + i, bt_row + pg0 + i);
        else
            npg = 0;
    }
    cp_async_commit_group();
    cp_async_wait_groups<1>();
    __syncthreads();  // the candidates have landed
    // the exact threshold among the candidates in bin B
    uint32_t T, need_eq;
    threshold_in_bin(ckey, M, B, static_cast<uint32_t>(k) - above, hist, wred, res, T, need_eq);
    // keys above T and equal to T among the candidates of the chunks before this one
    uint32_t g = 0, e = 0;
    for (int j = tid; j < off; j += kHsThreads) {
        const uint32_t key = ckey[j];
        g += key > T ? 1u : 0u;
        e += key == T ? 1u : 0u;
    }
    warp_sum2(g, e);
    if (lane == 0 && (g | e) != 0u) {
        atomicAdd(&cnt[0], g);
        atomicAdd(&cnt[1], e);
    }
    cp_async_wait_all();
    __syncthreads();  // the counts, the positions and the block-table entries
    const uint32_t gb = cnt[0], eb = cnt[1];
    const uint32_t eq_left = need_eq > eb ? need_eq - eb : 0u;
    const uint32_t obase = gb + min(eb, need_eq);
    emit_ordered<kHsThreads>(own, [&](int i) { return ckey[off + i]; }, T, eq_left, wgt, weq,
                             [&](uint32_t j, int i) {
                                 const uint32_t o = obase + j;
                                 if (o < static_cast<uint32_t>(k))
                                     put_out(static_cast<int>(o), i < ocache ? sel[i] : __ldg(rp + off + i));
                             });
}

}  // namespace

TopkChunkPlan topk_chunk_plan(int32_t num_rows, int32_t max_ctx, int32_t k, int sms) {
    TopkChunkPlan p{};
    if (num_rows <= 0 || num_rows > kChunkedMaxRows || max_ctx <= kChunkedMinCtx || k < 1 || k > DSA_MAX_TOPK ||
        sms <= 0)
        return p;
    // chunks per row: about two CTAs per SM over the batch, chunks of at most kChunkMaxKeys keys
    int C = (2 * sms + num_rows - 1) / num_rows;
    C = C < kChunkedMaxChunks ? C : kChunkedMaxChunks;  // each collect CTA adds up its row's lists
    const int by_len = (max_ctx + kChunkMaxKeys - 1) / kChunkMaxKeys;
    C = C > by_len ? C : by_len;
    int Lc = ((max_ctx + C - 1) / C + 63) / 64 * 64;
    if (Lc < kChunkMinKeys) Lc = kChunkMinKeys;
    C = (max_ctx + Lc - 1) / Lc;
    if (C > kHsMaxChunks) return p;  // rows of more than 16M keys: the cluster selection
    p.chunks = C;
    p.chunk_len = Lc;
    // a row's candidates: fewer than k above the threshold bin, and the bin's keys (16-byte rows)
    p.row_cap = (k + kHsInCap + 3) / 4 * 4;
    const size_t rc = static_cast<size_t>(num_rows) * C;
    p.bytes = align256(rc * kHsBins * 4) + align256(rc * 4) + 2 * align256(static_cast<size_t>(num_rows) * p.row_cap * 4) +
              align256(rc * 8) + align256(static_cast<size_t>(num_rows) * 16);
    return p;
}

void topk_chunk_bind(TopkArgs &a, const TopkChunkPlan &p, void *workspace) {
    const size_t rc = static_cast<size_t>(a.num_rows) * p.chunks;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    a.hs_list = reinterpret_cast<uint32_t *>(w);
    w += align256(rc * kHsBins * 4);
    a.hs_nlist = reinterpret_cast<uint32_t *>(w);
    w += align256(rc * 4);
    a.hs_key = reinterpret_cast<uint32_t *>(w);
    w += align256(static_cast<size_t>(a.num_rows) * p.row_cap * 4);
    a.hs_pos = reinterpret_cast<int32_t *>(w);
    w += align256(static_cast<size_t>(a.num_rows) * p.row_cap * 4);
    a.hs_chunk = reinterpret_cast<uint32_t *>(w);
    w += align256(rc * 8);
    a.hs_row = reinterpret_cast<uint32_t *>(w);
    a.chunks = p.chunks;
    a.chunk_len = p.chunk_len;
    a.row_cap = p.row_cap;
}

namespace {

template <bool kSlots>
cudaError_t launch_hist_select(const TopkArgs &a, cudaStream_t s) {
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem_collect_max = (static_cast<size_t>(kHsBins) + kChunkMaxKeys + kHsCacheChunks * kHsCacheLen + kHsMaxChunks) *
                                     4;
    const size_t smem_select_max = (static_cast<size_t>(DSA_MAX_TOPK) + kHsInCap + kBins + DSA_MAX_TOPK + kHsBtCache) * 4;
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(topk_hs_collect_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem_collect_max));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(topk_hs_select_kernel<kSlots>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_select_max));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const dim3 grid(static_cast<unsigned>(a.num_rows * a.chunks));
    cudaError_t e = launch_pdl(topk_hs_count_kernel, grid, dim3(kHsThreads), 0, s, a);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_hs_collect_kernel, grid, dim3(kHsThreads),
                   (static_cast<size_t>(kHsBins) + a.chunk_len + kHsCacheChunks * kHsCacheLen + a.chunks) * 4, s, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_hs_select_kernel<kSlots>, grid, dim3(kHsThreads),
                      (static_cast<size_t>(a.row_cap) + kBins + a.k + kHsBtCache) * 4, s, a);
}

}  // namespace

cudaError_t launch_topk(const TopkArgs &a, cudaStream_t s) {
    if (a.num_rows == 0) return cudaSuccess;
    if (a.chunks > 0 && a.hist == nullptr)  // the caller planned the histogram selection
        return a.slots_out != nullptr ? launch_hist_select<true>(a, s) : launch_hist_select<false>(a, s);
    const bool h = a.hist != nullptr, sl = a.slots_out != nullptr;
    if (h && sl) return launch_variant<true, true>(a, s);
    if (h) return launch_variant<true, false>(a, s);
    if (sl) return launch_variant<false, true>(a, s);
    return launch_variant<false, false>(a, s);
}

}  // namespace dsa
