// mla_fp8_common.cuh -- the FP8-latent attention's query image and operand helpers (mla_fp8.cu).
//
// The split decode kernel runs S = Q . KV^T and O^T += V^T . P^T as e4m3 x e4m3 -> fp32 MMAs on the latents exactly as
// stored (vLLM blog "Day-0 support for Kimi K3.1 Pro", section "One KV cache, three states": the
// 576-byte FP8 latent).  An e4m3 value has 4 significant bits, a bf16 query 8, so each query head
// is written as the sum of two e4m3 terms at a power of two per head, and the softmax weights P
// likewise; the products stay exact and accumulate in fp32.
#pragma once

#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {
namespace fp8mla {

// Byte offset of 16-byte unit u of row `row` in a 128-byte-swizzled operand block.
__device__ __forceinline__ uint32_t sw128(int row, int u) {
    return static_cast<uint32_t>(row * 128 + ((u ^ (row & 7)) << 4));
}

// Two fp32 -> two e4m3 (round to nearest even, saturating): lo value in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The two e4m3 values of the low 16 bits back to fp32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(v)));
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// x = hi + lo with hi = e4m3(x) and lo = e4m3(x - hi), for a pair: returns (hi pair, lo pair).
__device__ __forceinline__ uint2 split_pair(float x0, float x1) {
    const uint32_t hi = e4m3x2(x0, x1);
    const float2 d = e4m3x2_to_f2(hi);
    return make_uint2(hi, e4m3x2(x0 - d.x, x1 - d.y));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A softmax weight p (0 <= p <= 448) as hi + lo e4m3 codes: hi = p rounded to 3 mantissa bits
// (exact in e4m3 for normal values), lo = the rest (exact in fp32) rounded to e4m3.
__device__ __forceinline__ void p_split4(const float (&p)[4], uint32_t &hw, uint32_t &lw) {
    float hi[4], lo[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        hi[x] = __uint_as_float((__float_as_uint(p[x]) + 0x80000u) & 0xfff00000u);
        lo[x] = p[x] - hi[x];
    }
    hw = e4m3x2(hi[0], hi[1]) | (e4m3x2(hi[2], hi[3]) << 16);
    lw = e4m3x2(lo[0], lo[1]) | (e4m3x2(lo[2], lo[3]) << 16);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A query head's 576 bf16 values as lane `lane` holds them for convert_q_head: 16-value units lane
// and lane + 32 (units 32..35 are the RoPE dims), two 16-byte loads each.  Issuing the loads of
// several heads before converting any keeps them in flight together.
__device__ __forceinline__ void load_q_head(const uint16_t *q_head, int lane, int4 (&x)[4]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int unit = lane + 32 * k;
        if (unit < DSA_LATENT_DIM / 16) {
            x[2 * k] = *reinterpret_cast<const int4 *>(q_head + unit * 16);
            x[2 * k + 1] = *reinterpret_cast<const int4 *>(q_head + unit * 16 + 8);
        } else {
            x[2 * k] = x[2 * k + 1] = make_int4(0, 0, 0, 0);
        }
    }
}

// One query head (its values loaded by load_q_head) as the K-major operand image the kernels' S
// product reads: blocks 0-3 the hi terms of dims 0..511 (128 per block), blocks 4-7 the lo terms,
// block 8 the RoPE dims as [hi 64 B | lo 64 B]; block c of the image starts at img + c * H * 128
// and holds head h at row h, 128-byte swizzled.  The head is scaled by 2^e with its largest
// |q| * 2^e in (224, 448]; *inv_scale receives 2^-e.  A NaN or an infinity is DSA_ERR_RANGE.
// Warp-collective.
__device__ __forceinline__ void convert_q_head(const int4 (&x)[4], int h, int H, uint8_t *img, float *inv_scale,
                                               int32_t *status, int lane) {
    float v[2][16];
    float amax = 0.f;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t wd[8] = {static_cast<uint32_t>(x[2 * k].x),     static_cast<uint32_t>(x[2 * k].y),
                                static_cast<uint32_t>(x[2 * k].z),     static_cast<uint32_t>(x[2 * k].w),
                                static_cast<uint32_t>(x[2 * k + 1].x), static_cast<uint32_t>(x[2 * k + 1].y),
                                static_cast<uint32_t>(x[2 * k + 1].z), static_cast<uint32_t>(x[2 * k + 1].w)};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[k][2 * j] = __uint_as_float(wd[j] << 16);
            v[k][2 * j + 1] = __uint_as_float(wd[j] & 0xffff0000u);
            amax = fmaxf(amax, fmaxf(fabsf(v[k][2 * j]), fabsf(v[k][2 * j + 1])));
            bad |= !(fabsf(v[k][2 * j]) <= 3.4e38f) || !(fabsf(v[k][2 * j + 1]) <= 3.4e38f);
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) report(status, DSA_ERR_RANGE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = 0;
    if (amax > 0.f && amax <= 3.4e38f) {
        int xp;
        const float f = frexpf(amax, &xp);  // amax = f 2^xp, f in [0.5, 1)
        e = (f <= 0.875f ? 9 : 8) - xp;
        e = max(-120, min(120, e));
    }
    const float sc = ldexpf(1.0f, e);
    const int H128 = H * 128;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int unit = lane + 32 * k;
        if (unit >= DSA_LATENT_DIM / 16) continue;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint2 p0 = split_pair(v[k][4 * j] * sc, v[k][4 * j + 1] * sc);
            const uint2 p1 = split_pair(v[k][4 * j + 2] * sc, v[k][4 * j + 3] * sc);
            hi[j] = p0.x | (p1.x << 16);
            lo[j] = p0.y | (p1.y << 16);
        }
        uint8_t *dh, *dl;
        if (unit < 32) {  // latent dims: chunk unit / 8, 16-byte unit unit % 8 of the head's row
            const int c = unit >> 3, u = unit & 7;
            dh = img + c * H128 + sw128(h, u);
            dl = img + (4 + c) * H128 + sw128(h, u);
        } else {  // RoPE dims: units 0..3 (hi) and 4..7 (lo) of the head's row of the last block
            const int r = unit - 32;
            dh = img + 8 * H128 + sw128(h, r);
            dl = img + 8 * H128 + sw128(h, 4 + r);
        }
        *reinterpret_cast<uint4 *>(dh) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(dl) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (lane == 0) *inv_scale = ldexpf(1.0f, -e);
}

}  // namespace fp8mla
}  // namespace dsa
