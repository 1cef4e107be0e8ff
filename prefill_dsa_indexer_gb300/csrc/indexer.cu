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
//
// MXFP4 keys (blog "KV cache footprint" and "One KV cache, three states";
// AMD section "Quantization: native MXFP4 indexer": 128 e2m1 values plus one
// e8m0 scale per 32 values, 68 B per token) run the same pipeline at half the
// bytes, with no dequantisation step: the TMA unpacks each 64-byte key row
// into the 128-byte-per-row operand layout 4-bit MMA inputs use, the MMA is
// the block-scaled kind::mxf8f6f4 (e2m1 keys x e4m3 queries, K = 32 per
// instruction, one ue8m0 scale per key and 32 values), and the keys' four
// scale bytes reach TMEM by tcgen05.cp after the MMA warp has regrouped them
// into the 32-lane x 16-byte layout that copy takes.  Each 32-value block's
// partial dot product is scaled by its own 2^(E - 127) inside the MMA, so a
// key is exact over the whole E8M0 range, whatever the spread of its block
// exponents; there is no per-token scale (s_t = 1).
#include "indexer_common.cuh"

namespace dsa {

namespace {

constexpr int kIdxPageBytes = DSA_PAGE_SIZE * (DSA_INDEX_DIM + 4);  // 8448
constexpr int kIdxPageRows = kIdxPageBytes / 128;                    // 66 rows of 128 B
constexpr int kMxPageBytes = DSA_PAGE_SIZE * (DSA_INDEX_DIM / 2 + DSA_INDEX_DIM / 32);  // 4352
constexpr int kMxPageRows = kMxPageBytes / 64;                                        // 68 rows of 64 B

template <int G, bool kMx>
struct IdxCfg {
    static constexpr int N = 32 * G;
    // Decode and verify (G <= 4) stream every key from HBM with a light epilogue: two CTAs share
    // each SM, because one CTA's bulk-copy stream tops out below the SM's share of HBM bandwidth
    // however many stages it keeps in flight.  Each CTA then gets half of the TMEM and of the
    // shared memory.  Prefill (G = 8) needs more epilogue warps, registers and TMEM per key: one
    // CTA per SM.
    // (MXFP4 keys: two CTAs only for G = 1, whose accumulators leave room for the scale factors.)
    static constexpr int kCtasPerSm = kMx ? (G == 1 ? 2 : 1) : (G <= 4 ? 2 : 1);
    static constexpr int kMaxGroups = kCtasPerSm == 2 ? 256 : kIndexerMaxGroups;  // groups per launch
    static constexpr int kSmemBudget = kCtasPerSm == 2 ? 228 * 1024 / 2 - 1024 : 227 * 1024;
    // keys per tile: 256 (four pages, two M = 128 products) halves every per-tile cost of the
    // pipeline for decode; from G = 4 on (N >= 128) 128-key tiles leave TMEM room for two or more
    // accumulators in half of an SM's TMEM (verify) and for prefill's N = 256 ring
    static constexpr int kTileKeys = G >= 4 ? 128 : 256;
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
    // warp 0 producer, warp 1 MMA, then the epilogue warps (warp w reads TMEM lane quadrant w % 4;
    // any four consecutive epilogue warps cover the four quadrants).  They start at warp 2, so that
    // two CTAs of 4 or 8 epilogue warps hold 20 warps per SM and 96 registers a thread; prefill's
    // 16 epilogue warps start at warp 4 (18 or 20 warps give the same registers; 20 spill less).
    static constexpr int kEpiWarp0 = G >= 8 ? 4 : 2;
    static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
    // arrivals that release a stage or an accumulator: one per epilogue warp
    static constexpr uint32_t kRelease = kEpiWarps;
    // head weights in shared memory, per warp: its own rows
    static constexpr int kWFloats = kEpiWarps * kRowsPerEpiWarp * 32;
    // TMEM accumulators (kHalves x N columns each): enough that the MMA runs several tiles ahead.
    // MXFP4 keys add, per accumulator, 4 scale-factor columns per 128-key half (the keys' ue8m0
    // scales), and 8 columns of unit scale factors for the queries.
    static constexpr int kAccCols = kHalves * N;
    static constexpr int kSfaCols = kMx ? 4 * kHalves : 0;
    static constexpr int kSfbCols = kMx ? 8 : 0;
    static constexpr int kTmemBudget = 512 / kCtasPerSm;
    static constexpr int kAccFit = (kTmemBudget - kSfbCols) / (kAccCols + kSfaCols);
    static constexpr int kAcc = kAccFit < 8 ? kAccFit : 8;
    static constexpr int kTmemUsed = kAcc * (kAccCols + kSfaCols) + kSfbCols;
    static constexpr uint32_t kTmemCols = kTmemUsed <= 32    ? 32u
                                          : kTmemUsed <= 64  ? 64u
                                          : kTmemUsed <= 128 ? 128u
                                          : kTmemUsed <= 256 ? 256u
                                                             : 512u;
    static constexpr uint32_t kSfbCol = static_cast<uint32_t>(kAcc * kAccCols);   // unit query scales
    static constexpr uint32_t kSfaCol0 = kSfbCol + kSfbCols;                      // key scales of accumulator 0
    static constexpr int kKeyBytes = kTileKeys * 128;  // shared-memory bytes of a tile's keys (both formats)
    // global bytes a 64-token page brings: keys + 256 B of per-token scales
    static constexpr uint32_t kPageTx = kMx ? DSA_PAGE_SIZE * 64 + 256 : DSA_PAGE_SIZE * 128 + 256;
    static constexpr int kQBytes = N * 128;
    static constexpr int kUnitSfBytes = kMx ? 512 : 0;  // source of the queries' unit scale factors
    static constexpr int kNumBarsFor(int st) { return 2 * st + 2 * kAcc + 5; }
    // shared memory for `st` key stages (layout below)
    static constexpr int smem_for(int st) {
        return st * kKeyBytes + kQBufs * kQBytes + st * kTileKeys * 4 + kUnitSfBytes + kWFloats * 4 +
               (kMaxGroups + 4) * 4 + 2 * kMaxGroups * 4 + kNumBarsFor(st) * 8 + 64 + 1024;
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
    static constexpr int OFF_UNITSF = OFF_SCALES + kStages * kTileKeys * 4;
    static constexpr int OFF_W = OFF_UNITSF + kUnitSfBytes;
    static constexpr int OFF_PREFIX = OFF_W + kWFloats * 4;
    static constexpr int OFF_GREQ = OFF_PREFIX + (kMaxGroups + 4) * 4;
    static constexpr int OFF_GMAX = OFF_GREQ + kMaxGroups * 4;
    static constexpr int OFF_BARS = OFF_GMAX + kMaxGroups * 4;
    static constexpr int kNumBars = kNumBarsFor(kStages);
    static constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
    static constexpr int kSmemBytes = OFF_MISC + 64 + 1024;  // + slack for 1024-byte alignment
    static_assert(kAcc >= 1 && kTmemUsed <= static_cast<int>(kTmemCols), "TMEM plan");
    static_assert(kSfbCol % 4 == 0 && kSfaCol0 % 4 == 0, "scale-factor columns in groups of four");
    static_assert(kHalves * kRowsPerEpiWarp == 2, "two TMEM items per epilogue warp and tile");
    static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
    static_assert(kTmemCols <= static_cast<uint32_t>(kTmemBudget), "TMEM budget of a CTA");
    static_assert(kSmemBytes == smem_for(kStages), "stage sizing matches the layout");
    static_assert(OFF_SCALES % 512 == 0 && OFF_UNITSF % 16 == 0, "scale-factor copy sources are aligned");
};

template <int G, bool kHist, bool kMx>
__global__ void __launch_bounds__(IdxCfg<G, kMx>::kThreads, IdxCfg<G, kMx>::kCtasPerSm)
    indexer_kernel(const __grid_constant__ CUtensorMap key_map, const __grid_constant__ CUtensorMap q_map,
                   const IndexerArgs a) {
    using C = IdxCfg<G, kMx>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *keys = smem + C::OFF_KEYS;
    uint8_t *qbuf = smem + C::OFF_Q;
    float *scales = reinterpret_cast<float *>(smem + C::OFF_SCALES);  // FP8: fp32 s_t; MXFP4: 4 x e8m0 per key
    uint32_t *unit_sf = reinterpret_cast<uint32_t *>(smem + C::OFF_UNITSF);
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

    if constexpr (kMx) {
        // the queries carry no scale: their scale factors are all 2^0 (ue8m0 code 127)
        for (int i = tid; i < C::kUnitSfBytes / 4; i += blockDim.x) unit_sf[i] = 0x7f7f7f7fu;
        fence_async_smem();
    }
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
    // on-chip set-up above; global memory from here on, once the previous kernel has finished
    pdl_launch_dependents();
    pdl_wait();
    plan_groups<G, C::kTileKeys>(a, prefix, greq, gmax);
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
                        mbar_arrive_expect_tx(&full[stage], npages * C::kPageTx);
#pragma unroll
                        for (int p = 0; p < PPT; ++p) {
                            if (p >= npages) break;
                            // keys are read once per launch: evict them first, keep the rest of L2.
                            // MXFP4: the 64-row box of 64-byte rows lands unpacked as 128-byte rows.
                            const int64_t page = pj[p];
                            tma_load_2d_hint(keys + stage * C::kKeyBytes + p * (DSA_PAGE_SIZE * 128), &key_map,
                                             &full[stage], 0,
                                             static_cast<int32_t>(page * (kMx ? kMxPageRows : kIdxPageRows)),
                                             stream_policy);
                            const uint8_t *sc_src = kMx ? a.pool + page * kMxPageBytes + DSA_PAGE_SIZE * 64
                                                        : a.pool + page * kIdxPageBytes + DSA_PAGE_SIZE * 128;
                            bulk_load_hint(scales + stage * C::kTileKeys + p * DSA_PAGE_SIZE, sc_src,
                                           DSA_PAGE_SIZE * 4, &full[stage], stream_policy);
                        }
                    }
                    __syncwarp();
                }
            }
        } else if (warp == 1 && (kMx || lane == 0)) {
            // ------------------------------------------------ MMA issuer (lane 0; MXFP4: the whole
            // warp regroups each tile's key scale factors first)
            uint32_t sfb = 0;
            if constexpr (kMx) {
                sfb = tmem_base + C::kSfbCol;
                if (lane == 0) {
                    tc_fence_after();
                    tmem_cp_32x128b_x4(sfb, sdesc_plain(smem_u32(unit_sf), 128));
                    tmem_cp_32x128b_x4(sfb + 4, sdesc_plain(smem_u32(unit_sf), 128));
                }
            }
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1, gc = -1;
            int32_t it = 0;
            for (int32_t w = w_begin; w < w_end; ++w, ++it) {
                wk.advance(w);
                const int g = wk.g;
                const int qb_next = (g != cur) ? (gc + 1) % C::kQBufs : gc % C::kQBufs;
                const int stage = it % C::kStages, b = it % C::kAcc;
                int ok = 1;
                if (lane == 0) {
                    if (g != cur) ok = mbar_wait(&qfull[qb_next], ((gc + 1) / C::kQBufs) & 1, abort, a.status);
                    ok = ok && mbar_wait(&tempty[b], ((it / C::kAcc) & 1) ^ 1, abort, a.status) &&
                         mbar_wait(&full[stage], (it / C::kStages) & 1, abort, a.status);
                }
                if constexpr (kMx) {
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    __syncwarp();
                }
                if (!ok) break;
                if (g != cur) {
                    ++gc;
                    cur = g;
                }
                const int qb = gc % C::kQBufs;
                const int kt = w - prefix[g];
                const int nkeys = min(C::kTileKeys, gmax[g] - kt * C::kTileKeys);
                if constexpr (kMx) {
                    // Regroup each 128-key half's scales (4 bytes per key, in key order) in place into
                    // the layout the 32x128b copy takes: key m's word at word 4 (m % 32) + m / 32.
                    // A visible key with an e8m0 NaN code (0xff) is DSA_ERR_RANGE.
                    uint32_t *sw = reinterpret_cast<uint32_t *>(scales + stage * C::kTileKeys);
                    uint32_t v[C::kHalves][4];
                    bool nan_code = false;
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            v[hf][i] = sw[hf * 128 + 32 * i + lane];
                            if (hf * 128 + 32 * i + lane < nkeys && __vcmpeq4(v[hf][i], 0xffffffffu) != 0)
                                nan_code = true;
                        }
                    __syncwarp();
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        *reinterpret_cast<uint4 *>(sw + hf * 128 + 4 * lane) =
                            make_uint4(v[hf][0], v[hf][1], v[hf][2], v[hf][3]);
                    if (nan_code) report(a.status, DSA_ERR_RANGE);
                    fence_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(keys + stage * C::kKeyBytes);
                    const uint32_t b_addr = smem_u32(qbuf + qb * C::kQBytes);
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf) {
                        if (hf * 128 >= nkeys) break;  // a half past the context's end is not loaded
                        const uint32_t d = tmem_base + b * C::kAccCols + hf * C::N;
                        if constexpr (kMx) {
                            const uint32_t sfa = tmem_base + C::kSfaCol0 + b * C::kSfaCols + hf * 4;
                            tmem_cp_32x128b_x4(sfa, sdesc_plain(smem_u32(scales + stage * C::kTileKeys + hf * 128), 128));
#pragma unroll
                            for (int kk = 0; kk < DSA_INDEX_DIM / 32; ++kk)
                                mma_mx(d, sdesc_sw128(a_addr + hf * (128 * 128) + kk * 32, 16, 1024),
                                       sdesc_sw128(b_addr + kk * 32, 16, 1024),
                                       make_idesc_bs(128, C::N, 5, 0, static_cast<uint32_t>(kk),
                                                     static_cast<uint32_t>(kk)),
                                       sfa, sfb, kk > 0 ? 1u : 0u);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < DSA_INDEX_DIM / 32; ++kk)
                                mma_f8(d, sdesc_sw128(a_addr + hf * (128 * 128) + kk * 32, 16, 1024),
                                       sdesc_sw128(b_addr + kk * 32, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&tfull[b]);
                    const bool last_of_group = (w + 1 == w_end) || (prefix[g + 1] <= w + 1);
                    if (last_of_group) mma_commit(&qempty[qb]);
                }
                if constexpr (kMx) __syncwarp();
            }
            if (lane == 0) {
                mma_commit(mma_done);
                mbar_wait(mma_done, 0, abort, a.status);
            }
        } else if (warp >= C::kEpiWarp0) {
            // ------------------------------------------------ epilogue: two TMEM items per warp and tile
            constexpr int R = C::kRowsPerEpiWarp;
            const int e = warp - C::kEpiWarp0;
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
                // lane 0 waits for the accumulator and (FP8) for the stage's bulk-copied scales; the
                // stage cannot be re-armed before every warp of the tile has released it
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(&tfull[b], (it / C::kAcc) & 1, abort, a.status);
                    if constexpr (!kMx) ok = ok && mbar_wait(&full[stage], (it / C::kStages) & 1, abort, a.status);
                }
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
                for (int hf = 0; hf < C::kHalves; ++hf)
                    s_t[hf] = kMx ? 1.0f : scales[stage * C::kTileKeys + hf * 128 + key_lane];
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
                    float v = head_relu_sum(acc[k], wp + j * 32);
                    if constexpr (!kMx) v *= s_t[hf];
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

template <int G, bool kHist, bool kMx>
cudaError_t launch_gh(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a, int num_sms,
                      cudaStream_t s) {
    using C = IdxCfg<G, kMx>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(indexer_kernel<G, kHist, kMx>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    // the caller's range of groups, in launches of at most kMaxGroups (the planning arrays)
    IndexerArgs b = a;
    for (int done = 0; done < a.num_groups; done += C::kMaxGroups) {
        b.group0 = a.group0 + done;
        b.num_groups = a.num_groups - done < C::kMaxGroups ? a.num_groups - done : C::kMaxGroups;
        cudaError_t e = launch_pdl(indexer_kernel<G, kHist, kMx>, dim3(num_sms * C::kCtasPerSm), dim3(C::kThreads),
                                   C::kSmemBytes, s, key_map, q_map, b);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int G, bool kMx>
cudaError_t launch_g(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a, int num_sms,
                     cudaStream_t s) {
    return a.hist ? launch_gh<G, true, kMx>(key_map, q_map, a, num_sms, s)
                  : launch_gh<G, false, kMx>(key_map, q_map, a, num_sms, s);
}

template <bool kMx>
cudaError_t launch_fmt(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a,
                       int rows_per_group, int num_sms, cudaStream_t s) {
    switch (rows_per_group) {
        case 1: return launch_g<1, kMx>(key_map, q_map, a, num_sms, s);
        case 2: return launch_g<2, kMx>(key_map, q_map, a, num_sms, s);
        case 4: return launch_g<4, kMx>(key_map, q_map, a, num_sms, s);
        case 8: return launch_g<8, kMx>(key_map, q_map, a, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_indexer(const CUtensorMap &key_map, const CUtensorMap &q_map, const IndexerArgs &a,
                           bool mxfp4_keys, int rows_per_group, int num_sms, cudaStream_t s) {
    return mxfp4_keys ? launch_fmt<true>(key_map, q_map, a, rows_per_group, num_sms, s)
                      : launch_fmt<false>(key_map, q_map, a, rows_per_group, num_sms, s);
}

}  // namespace dsa
