// indexer_mxfp4.cu -- DSA indexer logits over MXFP4 index keys.
//
// Key format (vLLM blog "Day-0 support for Kimi K3.1 Pro", "KV cache
// footprint" and "One KV cache, three states"; AMD section "Quantization:
// native MXFP4 indexer"): 128 e2m1 values (64 B) plus one e8m0 scale per 32
// values (4 B), 68 B per token.  k_t[i] = e2m1[i] * 2^(E_b - 127), b = i / 32.
//
// The key stream is half the bytes of the FP8 keys, so the kernel stays
// HBM-bound as long as the dequantisation keeps up.  Raw pages arrive by plain
// bulk copies; four converter warps (one thread per key of a 128-key tile)
// rewrite each key exactly as e4m3 codes times a per-token power of two:
//     e2m1 * 2^(E_b-127) = [e2m1 * 2^(6 - (E_max - E_b))] * 2^(E_max - 133)
// where the bracket is an e4m3 value (exact while E_max - E_b <= 14) looked up
// for eight nibbles per two byte-permutes from a per-shift table, and the
// power of two becomes the per-token scale s_t that the FP8 epilogue already
// applies.  The MMA (kind::f8f6f4, keys on M) and the head-reduction epilogue
// are those of the FP8 kernel.
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
    static constexpr int kRaw = 6;
    static constexpr int kOps = 3;
    static constexpr int kEpiSplit = G >= 8 ? 2 : 1;
    static constexpr int kEpiWarps = 4 * kEpiSplit;
    static constexpr int kRowsPerEpiWarp = G / kEpiSplit;
    static constexpr int kConvWarp0 = 4 + kEpiWarps;
    static constexpr int kThreads = 32 * (kConvWarp0 + 4);
    static constexpr uint32_t kTmemCols = (2 * N < 32) ? 32u : static_cast<uint32_t>(2 * N);
    static constexpr int kOpBytes = kIdxTileKeys * 128;
    static constexpr int kQBytes = N * 128;
    static constexpr int kRawBytes = 2 * kMxPageBytes;  // 8704
    static constexpr int OFF_OPS = 0;
    static constexpr int OFF_Q = OFF_OPS + kOps * kOpBytes;
    static constexpr int OFF_RAW = OFF_Q + 2 * kQBytes;
    static constexpr int OFF_OPSC = OFF_RAW + kRaw * kRawBytes;
    static constexpr int OFF_W = OFF_OPSC + kOps * kIdxTileKeys * 4;
    static constexpr int OFF_PREFIX = OFF_W + 2 * N * 4;
    static constexpr int OFF_GREQ = OFF_PREFIX + (kIndexerMaxGroups + 4) * 4;
    static constexpr int OFF_GMAX = OFF_GREQ + kIndexerMaxGroups * 4;
    static constexpr int OFF_LUT = OFF_GMAX + kIndexerMaxGroups * 4;
    static constexpr int OFF_BARS = OFF_LUT + kLutEntries * 8;
    static constexpr int kNumBars = 2 * kRaw + 2 * kOps + 9;
    static constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
    static constexpr int kSmemBytes = OFF_MISC + 64 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(OFF_BARS % 8 == 0 && OFF_RAW % 16 == 0, "alignment");
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
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ops = smem + C::OFF_OPS;
    uint8_t *qbuf = smem + C::OFF_Q;
    uint8_t *raw = smem + C::OFF_RAW;
    float *opsc = reinterpret_cast<float *>(smem + C::OFF_OPSC);
    float *wbuf = reinterpret_cast<float *>(smem + C::OFF_W);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + C::OFF_PREFIX);
    int32_t *greq = reinterpret_cast<int32_t *>(smem + C::OFF_GREQ);
    int32_t *gmax = reinterpret_cast<int32_t *>(smem + C::OFF_GMAX);
    uint2 *lut = reinterpret_cast<uint2 *>(smem + C::OFF_LUT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BARS);
    uint64_t *raw_full = bars;                       // [kRaw] TMA -> converter
    uint64_t *raw_empty = raw_full + C::kRaw;        // [kRaw] converter -> TMA
    uint64_t *op_full = raw_empty + C::kRaw;         // [kOps] converter -> MMA, epilogue
    uint64_t *op_empty = op_full + C::kOps;          // [kOps] MMA + epilogue -> converter
    uint64_t *tfull = op_empty + C::kOps;            // [2]
    uint64_t *tempty = tfull + 2;                    // [2]
    uint64_t *qfull = tfull + 4;                     // [2]
    uint64_t *qempty = tfull + 6;                    // [2]
    uint64_t *mma_done = tfull + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ng = a.num_groups;
    plan_groups<G>(a, prefix, greq, gmax);
    if (tid < kLutEntries * 8) {
        // table entry (shift s, code m): e4m3 RNE of |e2m1 code m| * 2^s
        const int s = tid / 8 + kLutMinShift, m = tid % 8;
        const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
        reinterpret_cast<uint8_t *>(lut)[tid] = static_cast<uint8_t>(
            __nv_cvt_float_to_fp8(ldexpf(mag[m], s), __NV_SATFINITE, __NV_E4M3));
    }
    if (tid == 0) {
        *abort = 0;
        for (int i = 0; i < C::kRaw; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 4);
        }
        for (int i = 0; i < C::kOps; ++i) {
            mbar_init(&op_full[i], 4);
            mbar_init(&op_empty[i], 1 + C::kEpiWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], C::kEpiWarps);
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
            // Lane j looks up the page ids of tile base + j ahead of time; lane 0 issues.
            if (lane == 0) prefetch_tensormap(&q_map);
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1, gc = -1;
            int32_t it = 0;
            bool ok = true;
            for (int32_t base = w_begin; ok && base < w_end; base += 32) {
                int32_t pg0 = 0, pg1 = 0;
                if (base + lane < w_end) {
                    TileWalker mine{prefix, 0};
                    mine.seek(base + lane, ng);
                    const int g = mine.g, kt = base + lane - prefix[g];
                    const int nkeys = min(kIdxTileKeys, gmax[g] - kt * kIdxTileKeys);
                    const int32_t *bt = a.block_table + static_cast<int64_t>(greq[g]) * a.bt_stride;
                    pg0 = bt[kt * 2];
                    pg1 = nkeys > DSA_PAGE_SIZE ? bt[kt * 2 + 1] : 0;
                    if (pg0 < 0 || pg0 >= a.num_pages || pg1 < 0 || pg1 >= a.num_pages) {
                        report(a.status, DSA_ERR_BOUNDS);
                        pg0 = (pg0 < 0 || pg0 >= a.num_pages) ? 0 : pg0;
                        pg1 = (pg1 < 0 || pg1 >= a.num_pages) ? 0 : pg1;
                    }
                }
                const int cnt = min(32, w_end - base);
                for (int j = 0; j < cnt; ++j, ++it) {
                    const int32_t w = base + j;
                    const int32_t p0 = __shfl_sync(0xffffffffu, pg0, j), p1 = __shfl_sync(0xffffffffu, pg1, j);
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
                        const int nkeys = min(kIdxTileKeys, gmax[g] - kt * kIdxTileKeys);
                        const int npages = (nkeys + DSA_PAGE_SIZE - 1) / DSA_PAGE_SIZE;
                        mbar_arrive_expect_tx(&raw_full[rs], npages * kMxPageBytes);
                        for (int p = 0; p < npages; ++p)
                            bulk_load(raw + rs * C::kRawBytes + p * kMxPageBytes,
                                      a.pool + static_cast<int64_t>(p == 0 ? p0 : p1) * kMxPageBytes, kMxPageBytes,
                                      &raw_full[rs]);
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
                const int os = it % C::kOps, as = it & 1;
                if (!mbar_wait(&tempty[as], ((it >> 1) & 1) ^ 1, abort, a.status)) break;
                if (!mbar_wait(&op_full[os], (it / C::kOps) & 1, abort, a.status)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(ops + os * C::kOpBytes);
                const uint32_t b_addr = smem_u32(qbuf + qb * C::kQBytes);
#pragma unroll
                for (int kk = 0; kk < DSA_INDEX_DIM / 32; ++kk) {
                    mma_f8(tmem_base + as * C::N, sdesc_sw128(a_addr + kk * 32, 16, 1024),
                           sdesc_sw128(b_addr + kk * 32, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&op_empty[os]);
                mma_commit(&tfull[as]);
                const bool last_of_group = (w + 1 == w_end) || (prefix[g + 1] <= w + 1);
                if (last_of_group) mma_commit(&qempty[qb]);
            }
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, abort, a.status);
        } else if (warp >= C::kConvWarp0) {
            // ------------------------------------------------ MXFP4 -> e4m3 converter
            const int t = tid - 32 * C::kConvWarp0;  // key lane of the tile
            const int p = t / DSA_PAGE_SIZE, j = t % DSA_PAGE_SIZE;
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int32_t it = 0;
            for (int32_t w = w_begin; w < w_end; ++w, ++it) {
                wk.advance(w);
                const int g = wk.g;
                const int rs = it % C::kRaw, os = it % C::kOps;
                if (!mbar_wait_warp(&raw_full[rs], (it / C::kRaw) & 1, abort, a.status)) break;
                if (!mbar_wait_warp(&op_empty[os], ((it / C::kOps) & 1) ^ 1, abort, a.status)) break;
                const int kt = w - prefix[g];
                const int nkeys = min(kIdxTileKeys, gmax[g] - kt * kIdxTileKeys);
                float s_t = 0.f;
                if (p * DSA_PAGE_SIZE < nkeys) {
                    const uint8_t *pg = raw + rs * C::kRawBytes + p * kMxPageBytes;
                    const uint32_t ew = *reinterpret_cast<const uint32_t *>(pg + DSA_PAGE_SIZE * 64 + j * 4);
                    const uint4 *cw = reinterpret_cast<const uint4 *>(pg + j * 64);
                    const int e0 = ew & 0xff, e1 = (ew >> 8) & 0xff, e2 = (ew >> 16) & 0xff, e3 = ew >> 24;
                    const int emax = max(max(e0, e1), max(e2, e3));
                    s_t = (emax == 0xff) ? __int_as_float(0x7fc00000) : ldexpf(1.f, emax - 133);
                    uint8_t *orow = ops + os * C::kOpBytes;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int eb = (ew >> (8 * b)) & 0xff;
                        const int sh = 6 - (emax - eb);
                        const uint2 lt = (sh >= kLutMinShift) ? lut[sh - kLutMinShift] : make_uint2(0u, 0u);
                        const uint4 v = cw[b];
                        uint32_t o[8];
                        nib8_to_e4m3(v.x, lt, o[0], o[1]);
                        nib8_to_e4m3(v.y, lt, o[2], o[3]);
                        nib8_to_e4m3(v.z, lt, o[4], o[5]);
                        nib8_to_e4m3(v.w, lt, o[6], o[7]);
                        // elements 32b..32b+31 -> 16-byte units 2b, 2b+1 of this key's row
                        *reinterpret_cast<uint4 *>(orow + t * 128 + (((2 * b) ^ (t & 7)) << 4)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4 *>(orow + t * 128 + (((2 * b + 1) ^ (t & 7)) << 4)) =
                            make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                opsc[os * kIdxTileKeys + t] = s_t;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&op_full[os]);
                    mbar_arrive(&raw_empty[rs]);
                }
            }
        } else if (warp >= 4) {
            // ------------------------------------------------ epilogue (as in the FP8 kernel)
            const int e = warp - 4;
            const int quad = warp & 3;
            const int rbeg = (e >> 2) * C::kRowsPerEpiWarp;
            const int key_lane = quad * 32 + lane;
            TileWalker wk{prefix, 0};
            wk.seek(w_begin, ng);
            int cur = -1, gc = -1;
            int ctx[C::kRowsPerEpiWarp];
            int64_t row_off[C::kRowsPerEpiWarp];
            int32_t it = 0;
            for (int32_t w = w_begin; w < w_end; ++w, ++it) {
                wk.advance(w);
                const int g = wk.g;
                if (g != cur) {
                    ++gc;
                    cur = g;
                    float *wb = wbuf + (gc & 1) * C::N;
                    const int row0 = (a.group0 + g) * G;
                    for (int i = tid - 128; i < C::N; i += 32 * C::kEpiWarps)
                        wb[i] = a.head_w[static_cast<int64_t>(row0) * DSA_INDEX_HEADS + i];
                    named_bar_sync(1, 32 * C::kEpiWarps);
#pragma unroll
                    for (int jj = 0; jj < C::kRowsPerEpiWarp; ++jj) {
                        ctx[jj] = min(a.row_ctx[row0 + rbeg + jj], a.max_ctx);
                        row_off[jj] = static_cast<int64_t>(row0 + rbeg + jj) * a.logits_stride;
                    }
                }
                const float *wb = wbuf + (gc & 1) * C::N;
                const int os = it % C::kOps, as = it & 1;
                if (!mbar_wait_warp(&tfull[as], (it >> 1) & 1, abort, a.status)) break;
                if (!mbar_wait_warp(&op_full[os], (it / C::kOps) & 1, abort, a.status)) break;
                tc_fence_after();
                const float s_t = opsc[os * kIdxTileKeys + key_lane];
                __syncwarp();
                if (lane == 0) mbar_arrive(&op_empty[os]);
                const int t = (w - prefix[g]) * kIdxTileKeys + key_lane;
#pragma unroll
                for (int jj = 0; jj < C::kRowsPerEpiWarp; ++jj) {
                    uint32_t acc[32];
                    tmem_ld32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + as * C::N + (rbeg + jj) * 32,
                              acc);
                    tmem_ld_wait();
                    const float *wr = wb + (rbeg + jj) * 32;
                    float sum = 0.f;
#pragma unroll
                    for (int h = 0; h < 32; ++h) sum = fmaf(wr[h], fmaxf(__uint_as_float(acc[h]), 0.f), sum);
                    if (t < ctx[jj]) a.logits[row_off[jj] + t] = sum * s_t;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[as]);
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
