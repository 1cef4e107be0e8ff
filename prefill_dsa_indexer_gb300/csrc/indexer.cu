// indexer.cu -- DSA indexer logits on the sm_103a tensor cores.
//
// What it computes (vLLM blog "Day-0 support for Kimi K3.1 Pro", section
// "Sparse attention in K3.1 Pro"; weighted fp32 reduction across heads from
// the AMD section "Quantization: native MXFP4 indexer"):
//     logit[r, t] = sum_h w[r, h] * max(0, s_t * <q[r, h, :], k_t>)
// for every cached token t < L_r of the row's request.
//
// Design (GB300): the scan over all cached index keys is the dominant HBM
// stream of the layer (132 B per token per row group), so the kernel is a
// persistent, key-balanced pipeline:
//   * work = (row group g, key tile of 256 keys, 128 for prefill); the tiles
//     of all groups form one list that is split evenly over the CTAs (the
//     blog's scorer is "key-balanced" too, section "Low-latency decode").
//     Decode runs two CTAs per SM: one CTA's bulk-copy stream alone stays
//     below the SM's share of HBM bandwidth;
//   * warp 0 streams key tiles with TMA (one 64-row, 128-byte-swizzled box
//     per 64-token page) plus the pages' fp32 scales into a ring of
//     shared-memory stages;
//   * warp 1 issues tcgen05.mma kind::f8f6f4 (e4m3 x e4m3 -> fp32) with the
//     KEYS on M = 128 and the group's G rows x 32 heads on N, K = 128, into a
//     ring of TMEM accumulators, so the MMA runs ahead of the read-out; a
//     group's G rows (speculative-verify rows or a prefill query block) share
//     every key read;
//   * 4, 8 or 16 epilogue warps read one key lane each from TMEM, two
//     32-column items per warp and tile; each warp waits for its tile, reads
//     both items, releases the stage and the accumulator at once, and only
//     then reduces sum_h w_h * relu(acc_h) in registers (packed fp32x2 FMAs),
//     scales by s_t (s_t > 0 commutes with the relu), masks t >= L_r and
//     writes coalesced fp32 logits.
#include "indexer_common.cuh"

namespace dsa {

namespace {

constexpr int kIdxPageBytes = DSA_PAGE_SIZE * (DSA_INDEX_DIM + 4);  // 8448
constexpr int kIdxPageRows = kIdxPageBytes / 128;                    // 66 rows of 128 B

template <int G>
struct IdxCfg {
    static constexpr int N = 32 * G;
    // Decode (G <= 2) streams every key from HBM with a light epilogue: two CTAs share each SM,
    // because one CTA's bulk-copy stream tops out below the SM's share of HBM bandwidth however
    // many stages it keeps in flight.  Each CTA then gets half of the TMEM and of the shared
    // memory.  Verify (G = 4) and prefill (G = 8) need more epilogue warps, registers and TMEM
    // per key: one CTA per SM.
    static constexpr int kCtasPerSm = G <= 2 ? 2 : 1;
    static constexpr int kMaxGroups = kCtasPerSm == 2 ? 256 : kIndexerMaxGroups;  // groups per launch
    static constexpr int kSmemBudget = kCtasPerSm == 2 ? 228 * 1024 / 2 - 1024 : 227 * 1024;
    // keys per tile: 256 (four pages, two M = 128 products) halves every per-tile cost of the
    // pipeline for decode and verify; prefill's N = 256 accumulators keep 128-key tiles
    static constexpr int kTileKeys = G >= 8 ? 128 : 256;
    static constexpr int kPagesPerTile = kTileKeys / DSA_PAGE_SIZE;
    static constexpr int kHalves = kTileKeys / 128;
    // query buffers: two, so the next group's query loads during this group's last tiles, except
    // where a second one would cost a key stage (G = 4 at two CTAs per SM; few groups per CTA)
    static constexpr int kQBufs = (G == 4 && kCtasPerSm == 2) ? 1 : 2;
    // Epilogue: kEpiSplit warps per TMEM lane quadrant split the group's rows, so that every
    // warp reads exactly two 32-column items of a tile (two rows, or one row over two 128-key
    // halves).  Each warp waits for a tile by itself, reads both items, releases the accumulator
    // and the stage at once (so the MMA can run ahead) and only then reduces the heads.
    static constexpr int kEpiSplit = G * (kTileKeys / 128) / 2;
    static constexpr int kEpiWarps = 4 * kEpiSplit;
    static constexpr int kRowsPerEpiWarp = G / kEpiSplit;
    static constexpr int kThreads = 128 + 32 * kEpiWarps;
    // arrivals that release a stage or an accumulator: one per epilogue warp
    static constexpr uint32_t kRelease = kEpiWarps;
    // head weights in shared memory, per warp: its own rows
    static constexpr int kWFloats = kEpiWarps * kRowsPerEpiWarp * 32;
    // TMEM accumulators (kHalves x N columns each): enough that the MMA runs several tiles ahead
    static constexpr int kAccCols = kHalves * N;
    static constexpr int kTmemBudget = 512 / kCtasPerSm;
    static constexpr int kAcc = (kTmemBudget / kAccCols) < 8 ? (kTmemBudget / kAccCols) : 8;
    static constexpr uint32_t kTmemCols = static_cast<uint32_t>(kAcc * kAccCols);
    static constexpr int kKeyBytes = kTileKeys * 128;
    static constexpr int kQBytes = N * 128;
    static constexpr int kNumBarsFor(int st) { return 2 * st + 2 * kAcc + 5; }
    // shared memory for `st` key stages (layout below)
    static constexpr int smem_for(int st) {
        return st * kKeyBytes + kQBufs * kQBytes + st * kTileKeys * 4 + kWFloats * 4 + (kMaxGroups + 4) * 4 +
               2 * kMaxGroups * 4 + kNumBarsFor(st) * 8 + 64 + 1024;
    }
    // as many key stages as fit (up to 12 x 128 keys)
    static constexpr int pick_stages() {
        int st = 12 / kHalves;
        while (smem_for(st) > kSmemBudget) --st;
        return st;
    }
    static constexpr int kStages = pick_stages();
    static constexpr int OFF_KEYS = 0;
    static constexpr int OFF_Q = OFF_KEYS + kStages * kKeyBytes;
    static constexpr int OFF_SCALES = OFF_Q + kQBufs * kQBytes;
    static constexpr int OFF_W = OFF_SCALES + kStages * kTileKeys * 4;
    static constexpr int OFF_PREFIX = OFF_W + kWFloats * 4;
    static constexpr int OFF_GREQ = OFF_PREFIX + (kMaxGroups + 4) * 4;
    static constexpr int OFF_GMAX = OFF_GREQ + kMaxGroups * 4;
    static constexpr int OFF_BARS = OFF_GMAX + kMaxGroups * 4;
    static constexpr int kNumBars = kNumBarsFor(kStages);
    static constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
    static constexpr int kSmemBytes = OFF_MISC + 64 + 1024;  // + slack for 1024-byte alignment
    static_assert(kTmemCols == 32 || kTmemCols == 64 || kTmemCols == 128 || kTmemCols == 256 ||
                      kTmemCols == 512,
                  "TMEM allocation must be a power of two >= 32");
    static_assert(kHalves * kRowsPerEpiWarp == 2, "two TMEM items per epilogue warp and tile");
    static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
    static_assert(kTmemCols <= static_cast<uint32_t>(kTmemBudget), "TMEM budget of a CTA");
    static_assert(kSmemBytes == smem_for(kStages), "stage sizing matches the layout");
};

template <int G, bool kHist>
__global__ void __launch_bounds__(IdxCfg<G>::kThreads, IdxCfg<G>::kCtasPerSm)
    indexer_fp8_kernel(const __grid_constant__ CUtensorMap key_map, const __grid_constant__ CUtensorMap q_map,
                       const IndexerArgs a) {
    using C = IdxCfg<G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *keys = smem + C::OFF_KEYS;
    uint8_t *qbuf = smem + C::OFF_Q;
    float *scales = reinterpret_cast<float *>(smem + C::OFF_SCALES);
    float *wbuf = reinterpret_cast<float *>(smem + C::OFF_W);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + C::OFF_PREFIX);
    int32_t *greq = reinterpret_cast<int32_t *>(smem + C::OFF_GREQ);
    int32_t *gmax = reinterpret_cast<int32_t *>(smem + C::OFF_GMAX);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BARS);
    uint64_t *full = bars;                       // [kStages] TMA -> MMA, epilogue
    uint64_t *empty = bars + C::kStages;         // [kStages] epilogue -> TMA
    uint64_t *tfull = bars + 2 * C::kStages;     // [kAcc] MMA -> epilogue
    uint64_t *tempty = tfull + C::kAcc;          // [kAcc] epilogue -> MMA
    uint64_t *qfull = tempty + C::kAcc;          // [2] TMA -> MMA (query of a group)
    uint64_t *qempty = qfull + 2;                // [2] MMA -> TMA
    uint64_t *mma_done = qempty + 2;             // [1] all MMAs retired
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ng = a.num_groups;

    plan_groups<G, C::kTileKeys>(a, prefix, greq, gmax);
    if (tid == 0) {
        *abort = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            // the epilogue set (or each of its warps) that read a tile releases its stage: it
            // saw the MMA's completion (so the keys are consumed) and has read the scales
            mbar_init(&empty[s], C::kRelease);
        }
        for (int i = 0; i < C::kAcc; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], C::kRelease);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    if (warp == 0) plan_scan(prefix, ng, lane);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int32_t w_begin, w_end;
    plan_share(prefix[ng], w_begin, w_end);

    constexpr uint32_t kIdesc = make_idesc(128, C::N, 0, 0, false, false);

    if (w_begin < w_end) {
        if (warp == 0) {
            // ------------------------------------------------ TMA producer (whole warp)
            // Lane j looks up the page ids of tile base + j ahead of time (one coalesced
            // batch of block-table reads per 32 tiles); lane 0 issues the copies.
            if (lane == 0) {
                prefetch_tensormap(&key_map);
                prefetch_tensormap(&q_map);
            }
            const uint64_t stream_policy = l2_evict_first_policy();
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1, gc = -1;
            int32_t it = 0;
            bool ok = true;
            // page ids of tile `base + lane`; the next batch is in flight while this one is issued
            constexpr int PPT = C::kPagesPerTile;
            auto fetch = [&](int32_t base, int32_t (&pg)[PPT]) {
#pragma unroll
                for (int p = 0; p < PPT; ++p) pg[p] = 0;
                if (base + lane < w_end) {
                    TileWalker mine{prefix, 0};
                    mine.seek(base + lane, ng);
                    const int g = mine.g, kt = base + lane - prefix[g];
                    const int nkeys = min(C::kTileKeys, gmax[g] - kt * C::kTileKeys);
                    const int32_t *bt = a.block_table + static_cast<int64_t>(greq[g]) * a.bt_stride;
#pragma unroll
                    for (int p = 0; p < PPT; ++p)
                        if (p * DSA_PAGE_SIZE < nkeys) pg[p] = bt[kt * PPT + p];
                }
            };
            int32_t nx[PPT];
            fetch(w_begin, nx);
            for (int32_t base = w_begin; ok && base < w_end; base += 32) {
                int32_t pg[PPT];
                bool bad = false;
#pragma unroll
                for (int p = 0; p < PPT; ++p) {
                    pg[p] = nx[p];
                    if (pg[p] < 0 || pg[p] >= a.num_pages) {
                        bad = true;
                        pg[p] = 0;
                    }
                }
                if (bad) report(a.status, DSA_ERR_BOUNDS);
                if (base + 32 < w_end) fetch(base + 32, nx);
                const int cnt = min(32, w_end - base);
                for (int j = 0; j < cnt; ++j, ++it) {
                    const int32_t w = base + j;
                    int32_t pj[PPT];
#pragma unroll
                    for (int p = 0; p < PPT; ++p) pj[p] = __shfl_sync(0xffffffffu, pg[p], j);
                    wk.advance(w);
                    const int g = wk.g;
                    if (g != cur) {
                        ++gc;
                        cur = g;
                        const int qb = gc % C::kQBufs;
                        int got = 0;
                        if (lane == 0)
                            got = mbar_wait(&qempty[qb], ((gc / C::kQBufs) & 1) ^ 1, abort, a.status);
                        if (!__shfl_sync(0xffffffffu, got, 0)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            mbar_arrive_expect_tx(&qfull[qb], C::kQBytes);
                            tma_load_2d(qbuf + qb * C::kQBytes, &q_map, &qfull[qb], 0,
                                        (a.group0 + g) * G * DSA_INDEX_HEADS);
                        }
                    }
                    const int stage = it % C::kStages;
                    int got = 0;
                    if (lane == 0) got = mbar_wait(&empty[stage], ((it / C::kStages) & 1) ^ 1, abort, a.status);
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const int kt = w - prefix[g];
                        const int nkeys = min(C::kTileKeys, gmax[g] - kt * C::kTileKeys);
                        const int npages = (nkeys + DSA_PAGE_SIZE - 1) / DSA_PAGE_SIZE;
                        mbar_arrive_expect_tx(&full[stage], npages * (DSA_PAGE_SIZE * 128 + DSA_PAGE_SIZE * 4));
#pragma unroll
                        for (int p = 0; p < PPT; ++p) {
                            if (p >= npages) break;
                            // keys are read once per launch: evict them first, keep the rest of L2
                            tma_load_2d_hint(keys + stage * C::kKeyBytes + p * (DSA_PAGE_SIZE * 128), &key_map,
                                             &full[stage], 0, pj[p] * kIdxPageRows, stream_policy);
                            bulk_load_hint(scales + stage * C::kTileKeys + p * DSA_PAGE_SIZE,
                                           a.pool + static_cast<int64_t>(pj[p]) * kIdxPageBytes + DSA_PAGE_SIZE * 128,
                                           DSA_PAGE_SIZE * 4, &full[stage], stream_policy);
                        }
                    }
                    __syncwarp();
                }
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------ MMA issuer
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1, gc = -1;
            int32_t it = 0;
            for (int32_t w = w_begin; w < w_end; ++w, ++it) {
                wk.advance(w);
                const int g = wk.g;
                if (g != cur) {
                    ++gc;
                    cur = g;
                    if (!mbar_wait(&qfull[gc % C::kQBufs], (gc / C::kQBufs) & 1, abort, a.status)) break;
                }
                const int qb = gc % C::kQBufs;
                const int stage = it % C::kStages, b = it % C::kAcc;
                if (!mbar_wait(&tempty[b], ((it / C::kAcc) & 1) ^ 1, abort, a.status)) break;
                if (!mbar_wait(&full[stage], (it / C::kStages) & 1, abort, a.status)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(keys + stage * C::kKeyBytes);
                const uint32_t b_addr = smem_u32(qbuf + qb * C::kQBytes);
                const int kt = w - prefix[g];
                const int nkeys = min(C::kTileKeys, gmax[g] - kt * C::kTileKeys);
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    if (hf * 128 >= nkeys) break;  // a half past the context's end is not loaded
#pragma unroll
                    for (int kk = 0; kk < DSA_INDEX_DIM / 32; ++kk) {
                        mma_f8(tmem_base + b * C::kAccCols + hf * C::N,
                               sdesc_sw128(a_addr + hf * (128 * 128) + kk * 32, 16, 1024),
                               sdesc_sw128(b_addr + kk * 32, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&tfull[b]);
                const bool last_of_group = (w + 1 == w_end) || (prefix[g + 1] <= w + 1);
                if (last_of_group) mma_commit(&qempty[qb]);
            }
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, abort, a.status);
        } else if (warp >= 4) {
            // ------------------------------------------------ epilogue: two TMEM items per warp and tile
            constexpr int R = C::kRowsPerEpiWarp;
            const int e = warp - 4;
            const int quad = warp & 3;  // TMEM lane quadrant this warp may read
            const int rbeg = (e >> 2) * R;
            const int key_lane = quad * 32 + lane;
            float *wp = wbuf + e * (R * 32);  // this warp's rows' head weights
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1;
            int ctx[R];
            int64_t row_off[R];
            int hrow[R];  // global row of each of this warp's rows
            int32_t it = 0;
            for (int32_t w = w_begin; w < w_end; ++w, ++it) {
                wk.advance(w);
                const int g = wk.g;
                if (g != cur) {
                    cur = g;
                    const int row0 = (a.group0 + g) * G + rbeg;
                    __syncwarp();  // every lane is done with the previous group's weights
#pragma unroll
                    for (int j = 0; j < R; ++j) {
                        wp[j * 32 + lane] = a.head_w[static_cast<int64_t>(row0 + j) * DSA_INDEX_HEADS + lane];
                        ctx[j] = min(a.row_ctx[row0 + j], a.max_ctx);
                        row_off[j] = static_cast<int64_t>(row0 + j) * a.logits_stride;
                        hrow[j] = row0 + j;
                    }
                    __syncwarp();
                }
                const int stage = it % C::kStages, b = it % C::kAcc;
                // lane 0 waits for the accumulator and for the stage (its bulk-copied scales); the
                // stage cannot be re-armed before every warp of the tile has released it
                int ok = 1;
                if (lane == 0)
                    ok = mbar_wait(&tfull[b], (it / C::kAcc) & 1, abort, a.status) &&
                         mbar_wait(&full[stage], (it / C::kStages) & 1, abort, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                __syncwarp();
                if (!ok) break;
                tc_fence_after();
                // item k: half k / R of the tile, row k % R of this warp.  A half past the
                // context's end was neither loaded nor computed; its lanes are never stored.
                uint32_t acc[2][32];
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    tmem_ld32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + b * C::kAccCols + (k / R) * C::N +
                                  (rbeg + k % R) * 32,
                              acc[k]);
                tmem_ld_wait();
                reg_fence(acc[0]);
                reg_fence(acc[1]);
                float s_t[C::kHalves];
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf) s_t[hf] = scales[stage * C::kTileKeys + hf * 128 + key_lane];
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&empty[stage]);
                    mbar_arrive(&tempty[b]);
                }
                const int t0 = (w - prefix[g]) * C::kTileKeys + key_lane;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int j = k % R, hf = k / R;
                    const float v = head_relu_sum(acc[k], wp + j * 32) * s_t[hf];
                    const int t = t0 + hf * 128;
                    if (t < ctx[j]) {
                        a.logits[row_off[j] + t] = v;
                        if constexpr (kHist)
                            atomicAdd(a.hist + static_cast<int64_t>(hrow[j]) * kHistBins + (order_key(v) >> 16), 1u);
                    }
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int G, bool kHist>
cudaError_t launch_gh(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a, int num_sms,
                      cudaStream_t s) {
    using C = IdxCfg<G>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(indexer_fp8_kernel<G, kHist>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    // the caller's range of groups, in launches of at most kMaxGroups (the planning arrays)
    IndexerArgs b = a;
    for (int done = 0; done < a.num_groups; done += C::kMaxGroups) {
        b.group0 = a.group0 + done;
        b.num_groups = a.num_groups - done < C::kMaxGroups ? a.num_groups - done : C::kMaxGroups;
        indexer_fp8_kernel<G, kHist><<<num_sms * C::kCtasPerSm, C::kThreads, C::kSmemBytes, s>>>(key_map, q_map, b);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int G>
cudaError_t launch_g(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a, int num_sms,
                     cudaStream_t s) {
    return a.hist ? launch_gh<G, true>(key_map, q_map, a, num_sms, s) : launch_gh<G, false>(key_map, q_map, a, num_sms, s);
}

}  // namespace

cudaError_t launch_indexer_fp8(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a,
                               int rows_per_group, int num_sms, cudaStream_t s) {
    switch (rows_per_group) {
        case 1: return launch_g<1>(key_map, q_map, a, num_sms, s);
        case 2: return launch_g<2>(key_map, q_map, a, num_sms, s);
        case 4: return launch_g<4>(key_map, q_map, a, num_sms, s);
        case 8: return launch_g<8>(key_map, q_map, a, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dsa
