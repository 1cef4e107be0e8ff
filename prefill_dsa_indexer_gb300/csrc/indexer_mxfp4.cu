// indexer_mxfp4.cu -- DSA indexer logits over MXFP4 index keys.
//
// Key format (vLLM blog "Day-0 support for Kimi K3.1 Pro", "KV cache
// footprint" and "One KV cache, three states"; AMD section "Quantization:
// native MXFP4 indexer"): 128 e2m1 values (64 B) plus one e8m0 scale per 32
// values (4 B), 68 B per token.  k_t[i] = e2m1[i] * 2^(E_b - 127), b = i / 32.
//
// The key stream is half the bytes of the FP8 keys, so the kernel stays
// HBM-bound as long as the dequantisation keeps up.  Raw pages arrive by plain
// bulk copies; eight converter warps (four lanes per key, one 32-value block
// each, so every shared-memory read is a contiguous 512 bytes per warp)
// rewrite each key exactly as e4m3 codes times a per-token power of two:
//     e2m1 * 2^(E_b-127) = [e2m1 * 2^(6 - (E_max - E_b))] * 2^(E_max - 133)
// where the bracket is an e4m3 value (exact while E_max - E_b <= 14) looked up
// for eight nibbles per two byte-permutes from a per-shift table, and the
// power of two becomes the per-token scale s_t that the FP8 epilogue already
// applies.  Tiles (256 keys for decode and verify), the MMA (kind::f8f6f4, keys
// on M), the TMEM accumulator ring and the head-reduction epilogue sets are
// those of the FP8 kernel.
#include <cuda_fp8.h>

#include "indexer_common.cuh"

namespace dsa {

namespace {

constexpr int kMxPageBytes = DSA_PAGE_SIZE * (DSA_INDEX_DIM / 2 + DSA_INDEX_DIM / 32);  // 4352
constexpr int kLutMinShift = -12;
constexpr int kLutEntries = 6 - kLutMinShift + 1;  // shifts -12..6

template <int G>
struct MxCfg {
    static constexpr int N = 32 * G;
    // tiles, accumulator ring and epilogue sets as in the FP8 kernel
    static constexpr int kTileKeys = G >= 8 ? 128 : 256;
    static constexpr int kPagesPerTile = kTileKeys / DSA_PAGE_SIZE;
    static constexpr int kHalves = kTileKeys / 128;
    static constexpr int kEpiSplit = G >= 8 ? 2 : 1;
    static constexpr int kEpiGroups = G >= 8 ? 1 : 2;
    static constexpr int kWarpsPerTile = 4 * kEpiSplit;
    static constexpr int kEpiWarps = kWarpsPerTile * kEpiGroups;
    static constexpr int kRowsPerEpiWarp = G / kEpiSplit;
    static constexpr int kConvWarps = 8;  // converting is the busiest role: two warps per SM quarter
    static constexpr int kConvWarp0 = 4 + kEpiWarps;
    static constexpr int kThreads = 32 * (kConvWarp0 + kConvWarps);
    static constexpr int kAccCols = kHalves * N;
    static constexpr int kAcc = (512 / kAccCols) < 8 ? (512 / kAccCols) : 8;
    static constexpr uint32_t kTmemCols = static_cast<uint32_t>(kAcc * kAccCols);
    static constexpr int kOpBytes = kTileKeys * 128;
    static constexpr int kQBytes = N * 128;
    static constexpr int kRawBytes = kPagesPerTile * kMxPageBytes;
    static constexpr int kOps = 3;
    static constexpr int kNumBarsFor(int raw) { return 2 * raw + 2 * kOps + 3 * kAcc + 5; }
    static constexpr int smem_for(int raw) {
        return kOps * kOpBytes + 2 * kQBytes + raw * kRawBytes + kAcc * kTileKeys * 4 + kEpiGroups * 2 * N * 4 +
               (kIndexerMaxGroups + 4) * 4 + 2 * kIndexerMaxGroups * 4 + kLutEntries * 8 + kNumBarsFor(raw) * 8 +
               64 + 1024;
    }
    // as many raw (in-flight) stages as fit, up to 12 x 128 keys
    static constexpr int pick_raw() {
        int r = 12 / kHalves;
        while (smem_for(r) > 227 * 1024) --r;
        return r;
    }
    static constexpr int kRaw = pick_raw();
    static constexpr int OFF_OPS = 0;
    static constexpr int OFF_Q = OFF_OPS + kOps * kOpBytes;
    static constexpr int OFF_RAW = OFF_Q + 2 * kQBytes;
    static constexpr int OFF_OPSC = OFF_RAW + kRaw * kRawBytes;
    static constexpr int OFF_W = OFF_OPSC + kAcc * kTileKeys * 4;
    static constexpr int OFF_PREFIX = OFF_W + kEpiGroups * 2 * N * 4;
    static constexpr int OFF_GREQ = OFF_PREFIX + (kIndexerMaxGroups + 4) * 4;
    static constexpr int OFF_GMAX = OFF_GREQ + kIndexerMaxGroups * 4;
    static constexpr int OFF_LUT = OFF_GMAX + kIndexerMaxGroups * 4;
    static constexpr int OFF_BARS = OFF_LUT + kLutEntries * 8;
    static constexpr int kNumBars = kNumBarsFor(kRaw);
    static constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
    static constexpr int kSmemBytes = OFF_MISC + 64 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kSmemBytes == smem_for(kRaw), "stage sizing matches the layout");
    static_assert(kRaw >= 2, "at least double-buffered raw pages");
    static_assert(OFF_BARS % 8 == 0 && OFF_RAW % 16 == 0 && kMxPageBytes % 16 == 0, "alignment");
    static_assert(kAcc % kEpiGroups == 0, "an accumulator always belongs to the same epilogue set");
};

// 8 e2m1 nibbles (one 32-bit word) -> 8 e4m3 bytes through the table of one shift.
__device__ __forceinline__ void nib8_to_e4m3(uint32_t w, uint2 lut, uint32_t &lo, uint32_t &hi) {
    const uint32_t mlo = __byte_perm(lut.x, lut.y, w & 0x7777u);
    const uint32_t mhi = __byte_perm(lut.x, lut.y, (w >> 16) & 0x7777u);
    const uint32_t xl = __byte_perm(w, 0u, 0x1100u);  // [b0, b0, b1, b1]
    const uint32_t xh = __byte_perm(w, 0u, 0x3322u);  // [b2, b2, b3, b3]
    lo = mlo | ((xl << 4) & 0x00800080u) | (xl & 0x80008000u);
    hi = mhi | ((xh << 4) & 0x00800080u) | (xh & 0x80008000u);
}

template <int G>
__global__ void __launch_bounds__(MxCfg<G>::kThreads, 1)
    indexer_mxfp4_kernel(const __grid_constant__ CUtensorMap q_map, const IndexerArgs a) {
    using C = MxCfg<G>;
    constexpr int TK = C::kTileKeys, PPT = C::kPagesPerTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ops = smem + C::OFF_OPS;
    uint8_t *qbuf = smem + C::OFF_Q;
    uint8_t *raw = smem + C::OFF_RAW;
    float *opsc = reinterpret_cast<float *>(smem + C::OFF_OPSC);  // [kAcc][TK] per-token scales, by accumulator
    float *wbuf = reinterpret_cast<float *>(smem + C::OFF_W);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + C::OFF_PREFIX);
    int32_t *greq = reinterpret_cast<int32_t *>(smem + C::OFF_GREQ);
    int32_t *gmax = reinterpret_cast<int32_t *>(smem + C::OFF_GMAX);
    uint2 *lut = reinterpret_cast<uint2 *>(smem + C::OFF_LUT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BARS);
    uint64_t *raw_full = bars;                       // [kRaw] bulk copies -> converter
    uint64_t *raw_empty = raw_full + C::kRaw;        // [kRaw] converter -> producer
    uint64_t *op_full = raw_empty + C::kRaw;         // [kOps] converter -> MMA
    uint64_t *op_empty = op_full + C::kOps;          // [kOps] MMA (commit) -> converter
    uint64_t *tfull = op_empty + C::kOps;            // [kAcc] MMA -> epilogue
    uint64_t *tempty = tfull + C::kAcc;              // [kAcc] epilogue -> MMA, converter (scales)
    uint64_t *sfull = tempty + C::kAcc;              // [kAcc] converter -> epilogue (scales)
    uint64_t *qfull = sfull + C::kAcc;               // [2]
    uint64_t *qempty = qfull + 2;                    // [2]
    uint64_t *mma_done = qempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    volatile int *epi_ok = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);  // [2]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ng = a.num_groups;
    plan_groups<G, TK>(a, prefix, greq, gmax);
    if (tid < kLutEntries * 8) {
        // table entry (shift s, code m): e4m3 RNE of |e2m1 code m| * 2^s
        const int sh = tid / 8 + kLutMinShift, m = tid % 8;
        const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
        reinterpret_cast<uint8_t *>(lut)[tid] = static_cast<uint8_t>(
            __nv_cvt_float_to_fp8(ldexpf(mag[m], sh), __NV_SATFINITE, __NV_E4M3));
    }
    if (tid == 0) {
        *abort = 0;
        for (int i = 0; i < C::kRaw; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], C::kConvWarps);
        }
        for (int i = 0; i < C::kOps; ++i) {
            mbar_init(&op_full[i], C::kConvWarps);
            mbar_init(&op_empty[i], 1);  // the MMA's commit: the operand has been read
        }
        for (int i = 0; i < C::kAcc; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 1);
            mbar_init(&sfull[i], C::kConvWarps);
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
            // ------------------------------------------------ bulk-copy producer (whole warp)
            // Lane j looks up the page ids of tile base + j one 32-tile batch ahead; lane 0 issues.
            if (lane == 0) prefetch_tensormap(&q_map);
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1, gc = -1;
            int32_t it = 0;
            bool ok = true;
            auto fetch = [&](int32_t base, int32_t(&pg)[PPT]) {
#pragma unroll
                for (int p = 0; p < PPT; ++p) pg[p] = 0;
                if (base + lane < w_end) {
                    TileWalker mine{prefix, 0};
                    mine.seek(base + lane, ng);
                    const int g = mine.g, kt = base + lane - prefix[g];
                    const int nkeys = min(TK, gmax[g] - kt * TK);
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
                        const int qb = gc & 1;
                        int got = 0;
                        if (lane == 0) got = mbar_wait(&qempty[qb], ((gc >> 1) & 1) ^ 1, abort, a.status);
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
                    const int rs = it % C::kRaw;
                    int got = 0;
                    if (lane == 0) got = mbar_wait(&raw_empty[rs], ((it / C::kRaw) & 1) ^ 1, abort, a.status);
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const int kt = w - prefix[g];
                        const int nkeys = min(TK, gmax[g] - kt * TK);
                        const int npages = (nkeys + DSA_PAGE_SIZE - 1) / DSA_PAGE_SIZE;
                        mbar_arrive_expect_tx(&raw_full[rs], npages * kMxPageBytes);
#pragma unroll
                        for (int p = 0; p < PPT; ++p) {
                            if (p >= npages) break;
                            bulk_load(raw + rs * C::kRawBytes + p * kMxPageBytes,
                                      a.pool + static_cast<int64_t>(pj[p]) * kMxPageBytes, kMxPageBytes,
                                      &raw_full[rs]);
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
                    if (!mbar_wait(&qfull[gc & 1], (gc >> 1) & 1, abort, a.status)) break;
                }
                const int qb = gc & 1;
                const int os = it % C::kOps, b = it % C::kAcc;
                if (!mbar_wait(&tempty[b], ((it / C::kAcc) & 1) ^ 1, abort, a.status)) break;
                if (!mbar_wait(&op_full[os], (it / C::kOps) & 1, abort, a.status)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(ops + os * C::kOpBytes);
                const uint32_t b_addr = smem_u32(qbuf + qb * C::kQBytes);
                const int kt = w - prefix[g];
                const int nkeys = min(TK, gmax[g] - kt * TK);
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    if (hf * 128 >= nkeys) break;
#pragma unroll
                    for (int kk = 0; kk < DSA_INDEX_DIM / 32; ++kk) {
                        mma_f8(tmem_base + b * C::kAccCols + hf * C::N,
                               sdesc_sw128(a_addr + hf * (128 * 128) + kk * 32, 16, 1024),
                               sdesc_sw128(b_addr + kk * 32, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&op_empty[os]);
                mma_commit(&tfull[b]);
                const bool last_of_group = (w + 1 == w_end) || (prefix[g + 1] <= w + 1);
                if (last_of_group) mma_commit(&qempty[qb]);
            }
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, abort, a.status);
        } else if (warp >= C::kConvWarp0) {
            // ------------------------------------------------ MXFP4 -> e4m3 converter
            // Four lanes per key, one 16-byte chunk (32 codes, one e8m0 block) each, so a warp
            // reads eight keys' 512 contiguous code bytes per load.
            static_assert((TK * 4) % (32 * C::kConvWarps) == 0, "whole keys per converter lane");
            const int ct = tid - 32 * C::kConvWarp0;  // 0 .. 32 kConvWarps - 1
            const int cb = ct & 3;                    // this lane's block / chunk
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int32_t it = 0;
            for (int32_t w = w_begin; w < w_end; ++w, ++it) {
                wk.advance(w);
                const int g = wk.g;
                const int rs = it % C::kRaw, os = it % C::kOps, b = it % C::kAcc;
                if (!mbar_wait_warp(&raw_full[rs], (it / C::kRaw) & 1, abort, a.status)) break;
                if (!mbar_wait_warp(&op_empty[os], ((it / C::kOps) & 1) ^ 1, abort, a.status)) break;
                // the scales go with the accumulator: free once the epilogue has read tile it - kAcc
                if (!mbar_wait_warp(&tempty[b], ((it / C::kAcc) & 1) ^ 1, abort, a.status)) break;
                const int kt = w - prefix[g];
                const int nkeys = min(TK, gmax[g] - kt * TK);
                uint8_t *obase = ops + os * C::kOpBytes;
                // every load of the tile's keys first: the operand stores below go through
                // generic pointers the compiler cannot tell apart from the raw pages, so loads
                // issued after a store would wait for it
                constexpr int KPL = TK * 4 / (32 * C::kConvWarps);  // keys per lane
                constexpr int KSTEP = 8 * C::kConvWarps;              // keys per converter pass
                uint32_t ew[KPL];
                uint4 cv[KPL];
#pragma unroll
                for (int i = 0; i < KPL; ++i) {
                    const int key = (ct >> 2) + KSTEP * i;
                    const int p = key / DSA_PAGE_SIZE, j = key % DSA_PAGE_SIZE;
                    const uint8_t *pg = raw + rs * C::kRawBytes + p * kMxPageBytes;
                    ew[i] = *reinterpret_cast<const uint32_t *>(pg + DSA_PAGE_SIZE * 64 + j * 4);
                    cv[i] = *reinterpret_cast<const uint4 *>(pg + j * 64 + cb * 16);
                }
                uint2 lt[KPL];
                int emax[KPL];
#pragma unroll
                for (int i = 0; i < KPL; ++i) {
                    const uint32_t e = ew[i];
                    emax[i] = max(max(static_cast<int>(e & 0xff), static_cast<int>((e >> 8) & 0xff)),
                                  max(static_cast<int>((e >> 16) & 0xff), static_cast<int>(e >> 24)));
                    const int sh = 6 - (emax[i] - static_cast<int>((e >> (8 * cb)) & 0xff));
                    lt[i] = (sh >= kLutMinShift) ? lut[sh - kLutMinShift] : make_uint2(0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < KPL; ++i) {
                    const int key = (ct >> 2) + KSTEP * i;  // key of the tile
                    if (key >= nkeys) continue;          // never stored: the epilogue masks it
                    uint32_t o[8];
                    nib8_to_e4m3(cv[i].x, lt[i], o[0], o[1]);
                    nib8_to_e4m3(cv[i].y, lt[i], o[2], o[3]);
                    nib8_to_e4m3(cv[i].z, lt[i], o[4], o[5]);
                    nib8_to_e4m3(cv[i].w, lt[i], o[6], o[7]);
                    // elements 32cb..32cb+31 -> 16-byte units 2cb, 2cb+1 of the key's row (half
                    // key / 128, row key % 128 of that half's 128-row operand)
                    uint8_t *orow = obase + (key >> 7) * (128 * 128) + (key & 127) * 128;
                    const int r7 = key & 7;
                    *reinterpret_cast<uint4 *>(orow + (((2 * cb) ^ r7) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(orow + (((2 * cb + 1) ^ r7) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                    if (cb == 0) {
                        // 2^(emax - 133) built from its bits (a subnormal below emax = 7)
                        const int em = emax[i];
                        opsc[b * TK + key] = (em == 0xff) ? __int_as_float(0x7fc00000)
                                             : (em >= 7)  ? __int_as_float((em - 6) << 23)
                                                          : __int_as_float(1 << (em + 16));
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&op_full[os]);
                    mbar_arrive(&raw_empty[rs]);
                    mbar_arrive(&sfull[b]);
                }
            }
        } else if (warp >= 4) {
            // ------------------------------------------------ epilogue (as in the FP8 kernel)
            const int e = warp - 4;
            const int grp = e / C::kWarpsPerTile;
            const int sub = e % C::kWarpsPerTile;
            const int quad = warp & 3;
            const int rbeg = (sub >> 2) * C::kRowsPerEpiWarp;
            const int key_lane = quad * 32 + lane;
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1, gc = -1;
            int ctx[C::kRowsPerEpiWarp];
            int64_t row_off[C::kRowsPerEpiWarp];
            int hrow[C::kRowsPerEpiWarp];  // global row of each of this warp's rows
            for (int32_t it = grp, w = w_begin + grp; w < w_end; it += C::kEpiGroups, w += C::kEpiGroups) {
                wk.advance(w);
                const int g = wk.g;
                if (g != cur) {
                    ++gc;
                    cur = g;
                    float *wb = wbuf + (grp * 2 + (gc & 1)) * C::N;
                    const int row0 = (a.group0 + g) * G;
                    for (int i = sub * 32 + lane; i < C::N; i += 32 * C::kWarpsPerTile)
                        wb[i] = a.head_w[static_cast<int64_t>(row0) * DSA_INDEX_HEADS + i];
                    named_bar_sync(1 + grp, 32 * C::kWarpsPerTile);
#pragma unroll
                    for (int jj = 0; jj < C::kRowsPerEpiWarp; ++jj) {
                        ctx[jj] = min(a.row_ctx[row0 + rbeg + jj], a.max_ctx);
                        row_off[jj] = static_cast<int64_t>(row0 + rbeg + jj) * a.logits_stride;
                        hrow[jj] = row0 + rbeg + jj;
                    }
                }
                const float *wb = wbuf + (grp * 2 + (gc & 1)) * C::N;
                const int b = it % C::kAcc;
                // one thread of the set waits for the accumulator and its scales; the set's named
                // barrier passes the acquire on
                if (sub == 0 && lane == 0) {
                    const bool ok = mbar_wait(&tfull[b], (it / C::kAcc) & 1, abort, a.status) &&
                                    mbar_wait(&sfull[b], (it / C::kAcc) & 1, abort, a.status);
                    epi_ok[grp] = ok ? 1 : 0;
                }
                named_bar_sync(1 + grp, 32 * C::kWarpsPerTile);
                if (!epi_ok[grp]) break;
                tc_fence_after();
                const int t0 = (w - prefix[g]) * TK;
                const int nkeys = min(TK, gmax[g] - t0);
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    if (hf * 128 >= nkeys) break;
                    const float s_t = opsc[b * TK + hf * 128 + key_lane];
                    const int t = t0 + hf * 128 + key_lane;
#pragma unroll
                    for (int jj = 0; jj < C::kRowsPerEpiWarp; ++jj) {
                        uint32_t acc[32];
                        tmem_ld32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + b * C::kAccCols + hf * C::N +
                                      (rbeg + jj) * 32,
                                  acc);
                        tmem_ld_wait();
                        const float sum = head_relu_sum(acc, wb + (rbeg + jj) * 32);
                        if (t < ctx[jj]) {
                            const float v = sum * s_t;
                            a.logits[row_off[jj] + t] = v;
                            if (a.hist)
                                atomicAdd(a.hist + static_cast<int64_t>(hrow[jj]) * kHistBins + (order_key(v) >> 16), 1u);
                        }
                    }
                }
                tc_fence_before();
                named_bar_sync(1 + grp, 32 * C::kWarpsPerTile);
                if (sub == 0 && lane == 0) mbar_arrive(&tempty[b]);
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int G>
cudaError_t launch_mx(const CUtensorMap &q_map, const IndexerArgs &a, int num_sms, cudaStream_t s) {
    using C = MxCfg<G>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(indexer_mxfp4_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    indexer_mxfp4_kernel<G><<<num_sms, C::kThreads, C::kSmemBytes, s>>>(q_map, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_mxfp4(const CUtensorMap &q_map, const IndexerArgs &a, int rows_per_group, int num_sms,
                                 cudaStream_t s) {
    switch (rows_per_group) {
        case 1: return launch_mx<1>(q_map, a, num_sms, s);
        case 2: return launch_mx<2>(q_map, a, num_sms, s);
        case 4: return launch_mx<4>(q_map, a, num_sms, s);
        case 8: return launch_mx<8>(q_map, a, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dsa
