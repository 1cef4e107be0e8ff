// mla.cu -- sparse absorbed-MLA attention over the selected tokens.
//
// What it computes (vLLM blog "Day-0 support for Kimi K3.1 Pro", section
// "Sparse attention in K3.1 Pro": exact MLA attention, only over the 2,048
// selected tokens, 576-byte FP8 latents of 512 latent + 64 RoPE dims; the
// latent is the value because the key projection is absorbed, section
// "Low-latency decode: fused DSA decode path"):
//     S[h, t] = sm_scale * <q[h, :576], kv_t>,   O[h] = sum_t softmax_t(S[h, .]) kv_t[:512]
//
// Design (GB300):
//   * one CTA per (row, split of the row's selected tokens); 64-token tiles;
//   * four gather warps load the tile's latent rows (FP8: one token's 512
//     latent bytes per warp load instruction, so a load touches four
//     128-byte lines; NVFP4: two lanes per token), decode them exactly into fp16
//     (cvt e4m3x2 -> f16x2; NVFP4 e2m1 * e4m3 scale is exact in fp16 too) and
//     store them 128-byte swizzled, so one shared-memory image serves as the
//     K-major B operand of S and the MN-major A operand of PV;
//   * one thread issues tcgen05.mma kind::f16:
//       S  [heads (M=128) x 64 tokens]    = Q[128 x 576] . KV^T   (36 MMAs)
//       O^T[dims (4 x M=128) x heads (N=H)] += KV^T . P^T         (16 MMAs)
//     S keeps heads on TMEM lanes, so each softmax thread owns one head row
//     and reduces over tokens in registers; O is kept transposed so that
//     S (2 x 64 columns) and O^T (4 x 96 columns) fit the 512 TMEM columns
//     without padding the 96 heads to 128 in the PV product;
//   * four softmax warps run an online softmax in log2 units with a lazy
//     rescale of O^T (only when a head's running max grows by more than
//     2^8), write P in fp16 and keep the row sums;
//   * Q's rows beyond the real heads only feed S rows nobody reads, so Q's
//     128-row operand is packed at a stride of H rows per 64-dim block and
//     the unused rows alias the next block.
// Decode converts each row's query once into the kernel's fp16 operand image
// (a small prep kernel), splits a row's tokens over several CTAs (fixed split
// size, so the result does not depend on the batch), keeps each part's
// normalised output in fp16 and merges the parts by log-sum-exp in a third
// kernel; prefill converts Q in the kernel and writes the output directly.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kTok = 64;                  // tokens per tile
constexpr int kChunks = DSA_LATENT_DIM / 64;  // 9 blocks of 64 dims
constexpr int kMaxH = 96;
constexpr int kThreads = 384;             // warp 0 MMA, 4-7 softmax, 8-11 gather/epilogue
constexpr float kLazyRescaleLog2 = 8.0f;  // rescale O only when a max grows by > 2^8

constexpr int kKvBytes = kChunks * kTok * 128;  // 73,728: fp16 tile, [chunk][token][64 dims]
constexpr int kPBytes = kMaxH * 128;            // 12,288: fp16 P, [head][64 tokens]
constexpr int OFF_Q = 0;
constexpr int kQBytesMax = kChunks * kMaxH * 128 + (128 - 16) * 128;  // room for the aliased tail rows
constexpr int OFF_KV = (OFF_Q + kQBytesMax + 1023) / 1024 * 1024;
constexpr int OFF_P = OFF_KV + kKvBytes;
constexpr int OFF_ALPHA = OFF_P + kPBytes;
constexpr int OFF_INVL = OFF_ALPHA + 128 * 4;
constexpr int OFF_MASK = OFF_INVL + 128 * 4;
constexpr int OFF_FLAG = OFF_MASK + 16;
constexpr int OFF_BARS = OFF_FLAG + 16;
constexpr int kNumBars = 8;
constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
constexpr int kSmemBytes = OFF_MISC + 32 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 2 * kTok;  // O^T starts after the two S accumulators

__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two_bytes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two_bytes)));
    return r;
}

__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

// 2^x by the hardware approximation (relative error ~2^-22); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// Byte offset of 16-byte unit `u` (0..7) of row `row` in a 128-byte-swizzled
// tile whose 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint32_t sw128(int row, int u) {
    return static_cast<uint32_t>(row * 128 + ((u ^ (row & 7)) << 4));
}

// Eight bf16 query values -> fp16 (times `sc`), flagging values outside fp16's finite range.
__device__ __forceinline__ int4 q_unit_to_f16(int4 v, float sc, bool &range_err) {
    const uint32_t w[4] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y), static_cast<uint32_t>(v.z),
                           static_cast<uint32_t>(v.w)};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16) * sc, hi = __uint_as_float(w[j] & 0xffff0000u) * sc;
        if (!(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f)) range_err = true;
        __half2 hh = __floats2half2_rn(lo, hi);
        o[j] = *reinterpret_cast<uint32_t *>(&hh);
    }
    return make_int4(o[0], o[1], o[2], o[3]);
}

struct GatherRegs {
    int4 v[18];
    int32_t slot;
};

// FP8 latents, gather warp gw (0..3) loads tokens [16 gw, 16 gw + 16) of the tile: each
// token's 512 latent bytes are one 32-lane x 16-byte row load (four 128-byte lines per
// instruction), and the 64 RoPE bytes of eight tokens one more.  Lanes 0..15 hold the slots;
// an unused or rejected slot loads zeros, which decode to a zero row.
__device__ __forceinline__ void gather_load_fp8(const MlaArgs &a, const int32_t *row_slots, int t0, int n_tok,
                                                int gw, int lane, GatherRegs &g) {
    int32_t slot = -1;
    if (lane < 16) {
        const int t = t0 + 16 * gw + lane;
        slot = t < n_tok ? row_slots[t] : -1;
        if (slot >= 0 && static_cast<int64_t>(slot) >= a.num_pages * DSA_PAGE_SIZE) {
            report(a.status, DSA_ERR_BOUNDS);
            slot = -1;
        }
    }
    g.slot = slot;
    // Predicated loads into zeroed registers: nothing consumes a result before the store pass,
    // so all 18 loads are in flight together (a select on each result would wait for it).
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int32_t sj = __shfl_sync(0xffffffffu, slot, j);
        g.v[j] = make_int4(0, 0, 0, 0);
        ldg_nc_v4_if(a.pool + static_cast<int64_t>(max(sj, 0)) * DSA_LATENT_DIM + lane * 16, sj >= 0, g.v[j]);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int32_t sj = __shfl_sync(0xffffffffu, slot, 8 * b + (lane >> 2));
        g.v[16 + b] = make_int4(0, 0, 0, 0);
        ldg_nc_v4_if(a.pool + static_cast<int64_t>(max(sj, 0)) * DSA_LATENT_DIM + DSA_VALUE_DIM + (lane & 3) * 16,
                     sj >= 0, g.v[16 + b]);
    }
}

__device__ __forceinline__ void e4m3x16_to_f16(const int4 v, int4 &o0, int4 &o1) {
    const uint32_t w[4] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y), static_cast<uint32_t>(v.z),
                           static_cast<uint32_t>(v.w)};
    o0.x = cvt_e4m3x2_f16x2(w[0] & 0xffffu);
    o0.y = cvt_e4m3x2_f16x2(w[0] >> 16);
    o0.z = cvt_e4m3x2_f16x2(w[1] & 0xffffu);
    o0.w = cvt_e4m3x2_f16x2(w[1] >> 16);
    o1.x = cvt_e4m3x2_f16x2(w[2] & 0xffffu);
    o1.y = cvt_e4m3x2_f16x2(w[2] >> 16);
    o1.z = cvt_e4m3x2_f16x2(w[3] & 0xffffu);
    o1.w = cvt_e4m3x2_f16x2(w[3] >> 16);
}

// Lane l's 16 latent dims [16 l, 16 l + 16) of token j go to 64-dim block l / 4, 16-byte units
// 2 (l % 4) and 2 (l % 4) + 1 of the token's 128-byte row; RoPE lanes fill block 8.
__device__ __forceinline__ void gather_store_fp8(uint8_t *kv, int gw, int lane, const GatherRegs &g) {
    const int c = lane >> 2, u = 2 * (lane & 3);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int t = 16 * gw + j;
        int4 o0, o1;
        e4m3x16_to_f16(g.v[j], o0, o1);
        uint8_t *base = kv + c * (kTok * 128);
        *reinterpret_cast<int4 *>(base + sw128(t, u)) = o0;
        *reinterpret_cast<int4 *>(base + sw128(t, u + 1)) = o1;
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int t = 16 * gw + 8 * b + (lane >> 2);
        int4 o0, o1;
        e4m3x16_to_f16(g.v[16 + b], o0, o1);
        uint8_t *base = kv + 8 * (kTok * 128);
        *reinterpret_cast<int4 *>(base + sw128(t, u)) = o0;
        *reinterpret_cast<int4 *>(base + sw128(t, u + 1)) = o1;
    }
}

// NVFP4 latents: two lanes per token (lanes 2t, 2t+1 of the gather warps hold token t).
template <int FMT>
__device__ __forceinline__ void gather_load(const MlaArgs &a, const int32_t *row_slots, int t0, int n_tok,
                                            int gtid, GatherRegs &g) {
    const int t = gtid >> 1, half = gtid & 1;
    int32_t slot = (t0 + t < n_tok) ? row_slots[t0 + t] : -1;
    if (slot >= 0 && static_cast<int64_t>(slot) >= a.num_pages * DSA_PAGE_SIZE) {
        report(a.status, DSA_ERR_BOUNDS);
        slot = -1;
    }
    g.slot = slot;
    if (slot < 0) return;
    if (FMT == DSA_LATENT_FP8) {
        const uint8_t *src = a.pool + static_cast<int64_t>(slot) * DSA_LATENT_DIM;
#pragma unroll
        for (int i = 0; i < 18; ++i) g.v[i] = ldg_nc_v4(src + (half + 2 * i) * 16);
    } else {
        // NVFP4 page: [64 x 256 B e2m1][64 x 32 B e4m3 scales][64 x 64 B e4m3 RoPE]
        const int64_t page = slot / DSA_PAGE_SIZE, j = slot % DSA_PAGE_SIZE;
        const uint8_t *pg = a.pool + page * (DSA_PAGE_SIZE * 352);
        const uint8_t *codes = pg + j * 256;
        const uint8_t *sc = pg + DSA_PAGE_SIZE * 256 + j * 32;
        const uint8_t *rope = pg + DSA_PAGE_SIZE * 288 + j * 64;
        // this thread: code units half, half+2, ..., both 16-byte scale units, RoPE units half, half+2
#pragma unroll
        for (int i = 0; i < 8; ++i) g.v[i] = ldg_nc_v4(codes + (half + 2 * i) * 16);
        g.v[8] = ldg_nc_v4(sc);
        g.v[9] = ldg_nc_v4(sc + 16);
        g.v[10] = ldg_nc_v4(rope + half * 16);
        g.v[11] = ldg_nc_v4(rope + (half + 2) * 16);
    }
}

template <int FMT>
__device__ __forceinline__ void gather_store(uint8_t *kv, int gtid, const GatherRegs &g) {
    const int t = gtid >> 1, half = gtid & 1;
    if (g.slot < 0) {
        const int4 z = make_int4(0, 0, 0, 0);
        // zero this thread's share of the token row (all 9 chunks, 8 units each)
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
            for (int u = half * 4; u < half * 4 + 4; ++u)
                *reinterpret_cast<int4 *>(kv + c * (kTok * 128) + sw128(t, u)) = z;
        return;
    }
    if (FMT == DSA_LATENT_FP8) {
#pragma unroll
        for (int i = 0; i < 18; ++i) {
            const int u = half + 2 * i;  // 16-dim unit of the 576-dim row
            const int c = u >> 2, gq = u & 3;
            const uint32_t w[4] = {static_cast<uint32_t>(g.v[i].x), static_cast<uint32_t>(g.v[i].y),
                                   static_cast<uint32_t>(g.v[i].z), static_cast<uint32_t>(g.v[i].w)};
            int4 o0, o1;
            o0.x = cvt_e4m3x2_f16x2(w[0] & 0xffffu);
            o0.y = cvt_e4m3x2_f16x2(w[0] >> 16);
            o0.z = cvt_e4m3x2_f16x2(w[1] & 0xffffu);
            o0.w = cvt_e4m3x2_f16x2(w[1] >> 16);
            o1.x = cvt_e4m3x2_f16x2(w[2] & 0xffffu);
            o1.y = cvt_e4m3x2_f16x2(w[2] >> 16);
            o1.z = cvt_e4m3x2_f16x2(w[3] & 0xffffu);
            o1.w = cvt_e4m3x2_f16x2(w[3] >> 16);
            uint8_t *base = kv + c * (kTok * 128);
            *reinterpret_cast<int4 *>(base + sw128(t, 2 * gq)) = o0;
            *reinterpret_cast<int4 *>(base + sw128(t, 2 * gq + 1)) = o1;
        }
    } else {
        // 32 e4m3 scales, one per 16 latent dims
        const uint32_t scw[8] = {static_cast<uint32_t>(g.v[8].x), static_cast<uint32_t>(g.v[8].y),
                                 static_cast<uint32_t>(g.v[8].z), static_cast<uint32_t>(g.v[8].w),
                                 static_cast<uint32_t>(g.v[9].x), static_cast<uint32_t>(g.v[9].y),
                                 static_cast<uint32_t>(g.v[9].z), static_cast<uint32_t>(g.v[9].w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int cu = half + 2 * i;  // code unit: dims [32 cu, 32 cu + 32)
            const uint32_t w[4] = {static_cast<uint32_t>(g.v[i].x), static_cast<uint32_t>(g.v[i].y),
                                   static_cast<uint32_t>(g.v[i].z), static_cast<uint32_t>(g.v[i].w)};
            uint32_t o[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int sidx = 2 * cu + (q >> 1);  // word q holds dims 32cu + 8q .. +8
                const uint32_t sbyte = (scw[sidx >> 2] >> (8 * (sidx & 3))) & 0xffu;
                const uint32_t sh2 = cvt_e4m3x2_f16x2(sbyte | (sbyte << 8));
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    o[4 * q + b] = hmul2_u32(cvt_e2m1x2_f16x2((w[q] >> (8 * b)) & 0xffu), sh2);
            }
            // 32 dims = 64 B of fp16 = 4 swizzle units of chunk cu / 2
            const int c = cu >> 1, u0 = (cu & 1) * 4;
            uint8_t *base = kv + c * (kTok * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<int4 *>(base + sw128(t, u0 + q)) =
                    make_int4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
        // RoPE dims 512..575 (chunk 8): 64 e4m3 bytes; this thread holds units half and half+2
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int u = half + 2 * i;  // 16-dim unit of the RoPE block
            const int4 v = g.v[10 + i];
            const uint32_t w[4] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y),
                                   static_cast<uint32_t>(v.z), static_cast<uint32_t>(v.w)};
            int4 o0, o1;
            o0.x = cvt_e4m3x2_f16x2(w[0] & 0xffffu);
            o0.y = cvt_e4m3x2_f16x2(w[0] >> 16);
            o0.z = cvt_e4m3x2_f16x2(w[1] & 0xffffu);
            o0.w = cvt_e4m3x2_f16x2(w[1] >> 16);
            o1.x = cvt_e4m3x2_f16x2(w[2] & 0xffffu);
            o1.y = cvt_e4m3x2_f16x2(w[2] >> 16);
            o1.z = cvt_e4m3x2_f16x2(w[3] & 0xffffu);
            o1.w = cvt_e4m3x2_f16x2(w[3] >> 16);
            uint8_t *base = kv + 8 * (kTok * 128);
            *reinterpret_cast<int4 *>(base + sw128(t, 2 * u)) = o0;
            *reinterpret_cast<int4 *>(base + sw128(t, 2 * u + 1)) = o1;
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem + OFF_Q;
    uint8_t *kv = smem + OFF_KV;
    uint8_t *ps = smem + OFF_P;
    float *alpha = reinterpret_cast<float *>(smem + OFF_ALPHA);
    float *inv_l = reinterpret_cast<float *>(smem + OFF_INVL);  // o_scale / l per head
    unsigned long long *mask = reinterpret_cast<unsigned long long *>(smem + OFF_MASK);
    int *flag = reinterpret_cast<int *>(smem + OFF_FLAG);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *kv_full = bars + 0;   // gather -> MMA, softmax          (count 4)
    uint64_t *s_full = bars + 1;    // MMA -> softmax                   (commit)
    uint64_t *q_full = bars + 2;    // bulk copy of the prepared Q -> MMA (tx bytes)
    uint64_t *s_free = bars + 3;    // softmax -> MMA                   (count 4)
    uint64_t *p_full = bars + 5;    // softmax -> MMA                   (count 4)
    uint64_t *pv_done = bars + 6;   // MMA -> gather, softmax           (commit)
    uint64_t *stats = bars + 7;     // softmax -> epilogue              (count 4)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.num_heads;
    const int row = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
    const int tps = (a.k + a.splits - 1) / a.splits;
    const int t_begin = split * tps, t_end = min(a.k, t_begin + tps);
    const int n_tok = t_end - t_begin;
    const int n_tiles = (n_tok + kTok - 1) / kTok;
    const int32_t *row_slots = a.slots + static_cast<int64_t>(row) * a.k + t_begin;
    const float ts = a.tensor_scale;
    // FP8 latents stay as raw e4m3 values in fp16; their per-tensor scale is applied to S and O.
    const float s_scale = (FMT == DSA_LATENT_FP8 ? ts : 1.0f) * a.sm_scale * 1.4426950408889634f;
    const float o_scale = (FMT == DSA_LATENT_FP8 ? ts : 1.0f);
    const float q_rope_scale = (FMT == DSA_LATENT_FP8 ? 1.0f : ts);

    if (tid == 0) {
        *abort = 0;
        flag[0] = flag[1] = 0;
        mbar_init(kv_full, 4);
        mbar_init(s_full, 1);
        mbar_init(q_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(stats, 4);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // ---- gather warps start tile 0's latent loads; the other warps convert Q meanwhile
    GatherRegs g;
    const int gtid = tid - 256;  // 0..127 in the gather warps
    if (warp >= 8 && n_tiles > 0) {
        if (FMT == DSA_LATENT_FP8) gather_load_fp8(a, row_slots, 0, n_tok, warp - 8, lane, g);
        else gather_load<FMT>(a, row_slots, 0, n_tok, gtid, g);
    }
    // ---- Q: fp16, 128-byte swizzled K-major, block c (64 dims) at c * H * 128.  Decode
    // copies the image the prep kernel made for this row; prefill converts from bf16 here,
    // issuing all loads of a batch before any conversion.
    if (a.qprep != nullptr) {
        if (tid == 0 && n_tiles > 0) {
            const uint32_t blk = static_cast<uint32_t>(H) * 128;
            const uint8_t *src = a.qprep + static_cast<int64_t>(row) * mla_qprep_row_bytes(H);
            mbar_arrive_expect_tx(q_full, kChunks * blk);
            for (int c = 0; c < kChunks; ++c) bulk_load(qs + c * blk, src + c * blk, blk, q_full);
        }
    } else if (warp < 8) {
        constexpr int kUnits = DSA_LATENT_DIM / 8;  // 8-dim units per head
        constexpr int kBatch = 9;
        const uint16_t *qg = a.q + static_cast<int64_t>(row) * H * DSA_LATENT_DIM;
        const int total = H * kUnits;
        bool range_err = false;
        for (int e0 = tid; e0 < total; e0 += 256 * kBatch) {
            int4 v[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int e = e0 + i * 256;
                if (e < total) v[i] = *reinterpret_cast<const int4 *>(qg + static_cast<int64_t>(e) * 8);
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int e = e0 + i * 256;
                if (e >= total) break;
                const int h = e / kUnits, u = e % kUnits;
                const float sc = (u >= DSA_VALUE_DIM / 8) ? q_rope_scale : 1.0f;
                const int c = u >> 3, uu = u & 7;
                *reinterpret_cast<int4 *>(qs + c * H * 128 + sw128(h, uu)) = q_unit_to_f16(v[i], sc, range_err);
            }
        }
        if (range_err) report(a.status, DSA_ERR_RANGE);
    }
    fence_async_smem();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0 && n_tiles > 0) {
            // ------------------------------------------------------------ MMA issuer
            // S = Q . KV^T accumulates into two TMEM accumulators (even / odd 64-dim blocks)
            // issued alternately, and PV issues its four independent output blocks
            // round-robin, so consecutive MMAs never wait on each other's accumulator.
            // Descriptors are built once and advanced by their 16-byte address field.
            const uint32_t idesc_s = make_idesc(128, kTok, 0, 0, false, false);
            const uint32_t idesc_pv = make_idesc(128, H, 0, 0, true, false);
            const uint64_t q_desc = sdesc_sw128(smem_u32(qs), 16, 1024);
            const uint64_t kv_desc = sdesc_sw128(smem_u32(kv), 16, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(kv), kTok * 128, 1024);
            const uint64_t p_desc = sdesc_sw128(smem_u32(ps), 16, 1024);
            const uint32_t q_blk = (H * 128) >> 4, kv_blk = (kTok * 128) >> 4;  // 16-byte units
            // the copied Q must land before the first S product (and before this CTA can exit)
            const bool q_ok = a.qprep == nullptr || mbar_wait(q_full, 0, abort, a.status);
            for (int i = 0; q_ok && i < n_tiles; ++i) {
                if (!mbar_wait(kv_full, i & 1, abort, a.status)) break;
                if (!mbar_wait(s_free, (i & 1) ^ 1, abort, a.status)) break;
                tc_fence_after();
                for (int c0 = 0; c0 < kChunks; c0 += 2) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int c = c0 + e;
                            if (c < kChunks) {
                                const uint64_t off_q = c * q_blk + kk * 2, off_kv = c * kv_blk + kk * 2;
                                mma_f16(tmem + e * kTok, q_desc + off_q, kv_desc + off_kv, idesc_s,
                                        (c0 | kk) ? 1u : 0u);
                            }
                        }
                    }
                }
                mma_commit(s_full);
                if (!mbar_wait(p_full, i & 1, abort, a.status)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kTok / 16; ++ks) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // A = V^T block j: dims [128j, 128j+128) x 16 tokens, MN-major:
                        // 64-dim blocks 8 KB apart (LBO), 8-token groups 1 KB apart (SBO)
                        const uint64_t off_v = (2 * j) * kv_blk + ks * (2048 >> 4), off_p = ks * 2;
                        mma_f16(tmem + kTmemO + j * H, v_desc + off_v, p_desc + off_p, idesc_pv, (i | ks) ? 1u : 0u);
                    }
                }
                mma_commit(pv_done);
            }
        }
    } else if (warp >= 4) {
        const bool is_softmax = warp < 8;
        const int quad = warp & 3;
        bool ok = true;
        if (is_softmax) {
            // ------------------------------------------------------------ softmax
            const int h = quad * 32 + lane;
            float m = -INFINITY, l = 0.f;
            for (int i = 0; i < n_tiles; ++i) {
                if (!mbar_wait_warp(s_full, i & 1, abort, a.status) || !mbar_wait_warp(kv_full, i & 1, abort, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[64], s2[64];
                const uint32_t srow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
                tmem_ld32(srow, *reinterpret_cast<uint32_t(*)[32]>(sr));
                tmem_ld32(srow + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
                tmem_ld32(srow + kTok, *reinterpret_cast<uint32_t(*)[32]>(s2));
                tmem_ld32(srow + kTok + 32, *reinterpret_cast<uint32_t(*)[32]>(s2 + 32));
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);
                const unsigned long long msk = *mask;
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (msk == ~0ull) {
#pragma unroll
                    for (int j = 0; j < kTok; ++j) {
                        const float sv = (__uint_as_float(sr[j]) + __uint_as_float(s2[j])) * s_scale;
                        sr[j] = __float_as_uint(sv);
                        mx[j & 3] = fmaxf(mx[j & 3], sv);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kTok; ++j) {
                        const float sv = ((msk >> j) & 1ull)
                                             ? (__uint_as_float(sr[j]) + __uint_as_float(s2[j])) * s_scale
                                             : -INFINITY;
                        sr[j] = __float_as_uint(sv);
                        mx[j & 3] = fmaxf(mx[j & 3], sv);
                    }
                }
                const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                float al = 1.f;
                bool resc = false;
                if (mt > m + kLazyRescaleLog2 || (m == -INFINITY && mt > -INFINITY)) {
                    if (m > -INFINITY) {
                        al = exp2f(m - mt);
                        resc = true;
                    }
                    l *= al;
                    m = mt;
                }
                alpha[h] = al;
                if (__any_sync(0xffffffffu, resc && h < H) && lane == 0) atomicOr(&flag[i & 1], 1);
                named_bar_sync(1, 128);
                const bool do_resc = flag[i & 1] != 0;
                if (quad == 0 && lane == 0) flag[(i + 1) & 1] = 0;
                // P's buffer is free (and O^T stable) once the previous PV product is done
                if (i > 0 && !mbar_wait_warp(pv_done, (i - 1) & 1, abort, a.status)) {
                    ok = false;
                    break;
                }
                if (do_resc) {
                    // rescale O^T columns by alpha[head]: this warp owns TMEM lanes (dims) 32q..32q+31
                    tc_fence_after();
                    for (int j = 0; j < 4; ++j) {
                        for (int c = 0; c < H / 16; ++c) {
                            const uint32_t ta =
                                tmem + (static_cast<uint32_t>(quad * 32) << 16) + kTmemO + j * H + c * 16;
                            uint32_t v[16];
                            tmem_ld16(ta, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int x = 0; x < 16; ++x)
                                v[x] = __float_as_uint(__uint_as_float(v[x]) * alpha[c * 16 + x]);
                            tmem_st16(ta, v);
                        }
                    }
                    tmem_st_wait();
                }
                // P = 2^(s - m) in fp16, row h of the [head][64 tokens] swizzled operand.
                // Masked scores are -inf and give 0; m = -inf means this tile is all masked.
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[32];
                const float msub = (m == -INFINITY) ? 0.f : m;
#pragma unroll
                for (int j = 0; j < kTok; j += 2) {
                    const float p0 = fast_exp2(__uint_as_float(sr[j]) - msub);
                    const float p1 = fast_exp2(__uint_as_float(sr[j + 1]) - msub);
                    __half2 hh = __floats2half2_rn(p0, p1);
                    ls[(j >> 1) & 3] += p0 + p1;
                    pk[j / 2] = *reinterpret_cast<uint32_t *>(&hh);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                if (h < H) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<int4 *>(ps + sw128(h, u)) =
                            make_int4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
            // final statistics of this head
            // a split's part stays in decoded-latent units (|value| <= 2688, safe in fp16);
            // the merge applies the tensor scale
            inv_l[h] = (l > 0.f) ? (a.splits == 1 ? o_scale : 1.0f) / l : 0.f;
            if (h < H) {
                const float lse2 = (l > 0.f) ? m + log2f(l) : -INFINITY;
                if (a.splits == 1) {
                    if (a.lse) a.lse[static_cast<int64_t>(row) * H + h] = lse2 * 0.6931471805599453f;
                } else {
                    float *ml = a.part_ml + (static_cast<int64_t>(row) * a.splits + split) * H * 2;
                    ml[2 * h] = (l > 0.f) ? m : -INFINITY;
                    ml[2 * h + 1] = l;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(stats);
        } else {
            // ------------------------------------------------------------ gather
            for (int i = 0; i < n_tiles; ++i) {
                if (i > 0 && !mbar_wait_warp(pv_done, (i - 1) & 1, abort, a.status)) {
                    ok = false;
                    break;
                }
                unsigned long long tok = 0;
                const unsigned long long vm = __ballot_sync(0xffffffffu, g.slot >= 0);
                if (FMT == DSA_LATENT_FP8) {
                    gather_store_fp8(kv, quad, lane, g);
                    tok = vm & 0xffffull;  // lanes 0..15 hold this warp's 16 tokens
                } else {
                    gather_store<FMT>(kv, gtid, g);
                    // lanes 2t, 2t+1 hold token t of this warp's 16 tokens: keep even lanes' bits
#pragma unroll
                    for (int b = 0; b < 16; ++b) tok |= ((vm >> (2 * b)) & 1ull) << b;
                }
                if (lane == 0) reinterpret_cast<unsigned short *>(mask)[quad] = static_cast<unsigned short>(tok);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(kv_full);
                if (i + 1 < n_tiles) {
                    if (FMT == DSA_LATENT_FP8) gather_load_fp8(a, row_slots, (i + 1) * kTok, n_tok, quad, lane, g);
                    else gather_load<FMT>(a, row_slots, (i + 1) * kTok, n_tok, gtid, g);
                }
            }
        }
        // ---------------------------------------------------------------- epilogue, 8 warps:
        // softmax warps store dim blocks 0 and 1 of O, gather warps blocks 2 and 3;
        // lane = dim, one store instruction writes 32 consecutive dims of one head
        if (ok && n_tiles > 0) ok = mbar_wait_warp(pv_done, (n_tiles - 1) & 1, abort, a.status);
        if (ok) ok = mbar_wait_warp(stats, 0, abort, a.status);
        // A split's part is written as fp16: neighbouring lanes (dims d, d + 1) swap one value
        // so that each lane stores a 4-byte pair of dims of one head (two heads per step).
        // The direct output is written as fp32 rows.
        if (ok) {
            tc_fence_after();
            const bool to_part = a.splits > 1;
            float *dst = a.out + static_cast<int64_t>(row) * H * DSA_VALUE_DIM;
            __half *dst_h = reinterpret_cast<__half *>(a.part_o) +
                            (static_cast<int64_t>(row) * a.splits + split) * H * DSA_VALUE_DIM;
            const bool odd = (lane & 1) != 0;
            const int j0 = is_softmax ? 0 : 2;
            for (int j = j0; j < j0 + 2; ++j) {
                const int d = 128 * j + 32 * quad + lane;
                const uint32_t tb = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kTmemO + j * H;
                for (int c = 0; c < H; c += 32) {
                    uint32_t v[32];
                    const bool full32 = c + 32 <= H;
                    if (n_tiles > 0) {
                        if (full32) tmem_ld32(tb + c, v);
                        else tmem_ld16(tb + c, *reinterpret_cast<uint32_t(*)[16]>(v));
                        tmem_ld_wait();
                    }
                    // the 32 heads' factors into registers first: the stores below may alias
                    // inv_l as far as the compiler knows, which would serialise every element
                    float il[32];
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        const float4 f = (x < 16 || full32) ? *reinterpret_cast<const float4 *>(inv_l + c + x)
                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                        il[x] = f.x;
                        il[x + 1] = f.y;
                        il[x + 2] = f.z;
                        il[x + 3] = f.w;
                    }
                    if (to_part) {
#pragma unroll
                        for (int x = 0; x < 32; x += 2) {
                            if (x >= 16 && !full32) break;
                            const float o0 = (n_tiles > 0) ? __uint_as_float(v[x]) * il[x] : 0.f;
                            const float o1 = (n_tiles > 0) ? __uint_as_float(v[x + 1]) * il[x + 1] : 0.f;
                            const float got = __shfl_xor_sync(0xffffffffu, odd ? o0 : o1, 1);
                            // even lane: head c+x, dims (d, d+1); odd lane: head c+x+1, dims (d-1, d)
                            const __half2 hh = odd ? __floats2half2_rn(got, o1) : __floats2half2_rn(o0, got);
                            const int at = (c + x + (odd ? 1 : 0)) * DSA_VALUE_DIM + (d & ~1);
                            *reinterpret_cast<__half2 *>(dst_h + at) = hh;
                        }
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            if (x >= 16 && !full32) break;
                            const float o = (n_tiles > 0) ? __uint_as_float(v[x]) * il[x] : 0.f;
                            dst[(c + x) * DSA_VALUE_DIM + d] = o;
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge the splits of each (row, head): O = o_scale * sum_s w_s O_s / sum_s w_s with
// w_s = l_s 2^(m_s - M), M = max_s m_s (log2 units), O_s the split's normalised fp16 output.
// One CTA per (row, head): warp 0 turns the splits' (max, sum) into the normalised weights once,
// every thread then sums four output dims over the splits (its partial loads issued first).
__global__ void __launch_bounds__(128) mla_combine_kernel(const MlaArgs a) {
    __shared__ float wn[kMlaMaxSplits];
    pdl_launch_dependents();
    pdl_wait();
    const int H = a.num_heads, S = a.splits;
    const int row = blockIdx.x / H, h = blockIdx.x % H;
    const int tid = threadIdx.x;
    // all partial loads in flight at once
    uint2 o[kMlaMaxSplits];
#pragma unroll
    for (int s = 0; s < kMlaMaxSplits; ++s)
        if (s < S)
            o[s] = reinterpret_cast<const uint2 *>(
                a.part_o + ((static_cast<int64_t>(row) * S + s) * H + h) * DSA_VALUE_DIM)[tid];
    if (tid < 32) {
        const float *ml = a.part_ml + static_cast<int64_t>(row) * S * H * 2;
        const float m = tid < S ? ml[(tid * H + h) * 2] : -INFINITY;
        const float l = tid < S ? ml[(tid * H + h) * 2 + 1] : 0.f;
        float M = m;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float w = (m == -INFINITY) ? 0.f : l * exp2f(m - M);
        float W = w;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
        const float o_scale = a.format == DSA_LATENT_FP8 ? a.tensor_scale : 1.0f;
        if (tid < S) wn[tid] = W > 0.f ? w * (o_scale / W) : 0.f;
        if (tid == 0 && a.lse)
            a.lse[static_cast<int64_t>(row) * H + h] = W > 0.f ? (M + log2f(W)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kMlaMaxSplits; ++s) {
        if (s >= S) continue;
        const float w = wn[s];
        const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&o[s].x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&o[s].y));
        acc.x = fmaf(w, lo.x, acc.x);
        acc.y = fmaf(w, lo.y, acc.y);
        acc.z = fmaf(w, hi.x, acc.z);
        acc.w = fmaf(w, hi.y, acc.w);
    }
    reinterpret_cast<float4 *>(a.out + (static_cast<int64_t>(row) * H + h) * DSA_VALUE_DIM)[tid] = acc;
    // The partials are workspace scratch, dead once read: drop their L2 lines unwritten
    // (S x 8 lines of 128 B for this head) so they cost no HBM write-back.
    __syncthreads();
    if (tid < S * 8)
        l2_discard_line(a.part_o + ((static_cast<int64_t>(row) * S + (tid >> 3)) * H + h) * DSA_VALUE_DIM +
                        (tid & 7) * 64);
}

// Decode query preparation: each row's bf16 query becomes, once, the exact fp16 shared-memory
// image the attention kernel's Q operand needs (RoPE dims of NVFP4 latents times the tensor
// scale), so every split of the row starts with one bulk copy instead of its own conversion.
__global__ void __launch_bounds__(256) mla_qprep_kernel(const MlaArgs a) {
    constexpr int kUnits = DSA_LATENT_DIM / 8;  // 8-dim units per head
    const int H = a.num_heads;
    const int64_t total = static_cast<int64_t>(a.num_rows) * H * kUnits;
    const float q_rope_scale = (a.format == DSA_LATENT_FP8) ? 1.0f : a.tensor_scale;
    bool range_err = false;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * 256) {
        const int64_t rh = e / kUnits;
        const int u = static_cast<int>(e % kUnits);
        const int64_t row = rh / H;
        const int h = static_cast<int>(rh % H);
        const int4 v = *reinterpret_cast<const int4 *>(a.q + e * 8);
        const float sc = (u >= DSA_VALUE_DIM / 8) ? q_rope_scale : 1.0f;
        const int c = u >> 3, uu = u & 7;
        uint8_t *dst = a.qprep + row * static_cast<int64_t>(mla_qprep_row_bytes(H)) + c * H * 128 + sw128(h, uu);
        *reinterpret_cast<int4 *>(dst) = q_unit_to_f16(v, sc, range_err);
    }
    if (range_err) report(a.status, DSA_ERR_RANGE);
}

template <int FMT>
cudaError_t launch_fmt(const MlaArgs &a, cudaStream_t s) {
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e =
            cudaFuncSetAttribute(sparse_mla_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    if (a.qprep != nullptr && !a.q_prepared) {
        cudaError_t e = launch_mla_qprep(a, s);
        if (e != cudaSuccess) return e;
    }
    sparse_mla_kernel<FMT><<<a.num_rows * a.splits, kThreads, kSmemBytes, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.splits == 1) return e;
    return launch_mla_combine(a, s);
}

}  // namespace

cudaError_t launch_mla_qprep(const MlaArgs &a, cudaStream_t s) {
    if (a.num_rows == 0 || a.qprep == nullptr) return cudaSuccess;
    const int64_t units = static_cast<int64_t>(a.num_rows) * a.num_heads * (DSA_LATENT_DIM / 8);
    const int blocks = static_cast<int>(units / 256 < 4096 ? (units + 255) / 256 : 4096);
    mla_qprep_kernel<<<blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_mla_combine(const MlaArgs &a, cudaStream_t s) {
    if (a.num_rows == 0 || a.splits < 2) return cudaSuccess;
    return launch_pdl(mla_combine_kernel, dim3(a.num_rows * a.num_heads), dim3(DSA_VALUE_DIM / 4), 0, s, a);
}

size_t mla_workspace_bytes(int32_t num_rows, int32_t num_heads, int32_t k) {
    return mla_workspace_bytes_for(static_cast<size_t>(num_rows), static_cast<size_t>(num_heads),
                                   static_cast<size_t>(k));
}

cudaError_t launch_sparse_mla(const MlaArgs &a, cudaStream_t s) {
    if (a.num_rows == 0) return cudaSuccess;
    if (a.num_heads < 16 || a.num_heads > kMaxH || a.num_heads % 16 != 0) return cudaErrorInvalidValue;
    if (a.format == DSA_LATENT_FP8) return launch_fmt<DSA_LATENT_FP8>(a, s);
    if (a.format == DSA_LATENT_NVFP4) return launch_fmt<DSA_LATENT_NVFP4>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace dsa
