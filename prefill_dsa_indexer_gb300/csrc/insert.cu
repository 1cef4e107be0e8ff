// insert.cu -- quantise new tokens and write them into the paged caches.
//
// vLLM blog "Day-0 support for Kimi K3.1 Pro", section "Low-latency decode:
// fused DSA decode path": the front end quantises the new token's index key
// (FP8 or MXFP4) and the new latent is written into the cache before the
// indexer scores.  Formats ("One KV cache, three states"):
//   index FP8:   code = e4m3(x / s), s = amax/448 (1 if amax = 0), fp32 scale stored
//   index MXFP4: per 32 values E = floor(log2 amax) - 2 + 127 in [0, 254]
//                (0 for an all-zero block), code = e2m1(x * 2^(127 - E))
//   latent FP8:  code = e4m3(x / tensor_scale)
//   latent NVFP4: per 16 values scale code = e4m3(amax / 6), code = e2m1(x / scale)
//                (0 when the scale is 0); RoPE dims e4m3(x / tensor_scale)
// Every scale and quotient is an IEEE fp32 operation and every code a
// round-to-nearest-even conversion with saturation, so the bytes are exactly
// defined.  One warp per token; loads and stores are coalesced per token.
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {

namespace {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ uint8_t e4m3_rne(float x) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// Two e2m1 codes in one byte: lo in bits 0-3, hi in bits 4-7 (RNE, saturating).
__device__ __forceinline__ uint32_t e2m1x2_rne(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float e4m3_value(uint8_t code) {
    __nv_fp8_e4m3 v;
    v.__x = code;
    return static_cast<float>(v);
}

__device__ __forceinline__ float warp_max(float v, int width) {
    for (int o = width / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__global__ void __launch_bounds__(256) cache_insert_kernel(const InsertArgs a) {
    const int lane = threadIdx.x & 31;
    const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (tok >= a.num_tokens) return;
    const int32_t slot = a.slots[tok];
    if (slot < 0) return;
    if (static_cast<int64_t>(slot) >= a.num_pages * DSA_PAGE_SIZE) {
        if (lane == 0) report(a.status, DSA_ERR_BOUNDS);
        return;
    }
    const int64_t page = slot / DSA_PAGE_SIZE;
    const int j = slot % DSA_PAGE_SIZE;

    // ---- index key: lane l holds dims 4l .. 4l+3
    {
        const uint2 raw = reinterpret_cast<const uint2 *>(a.keys + static_cast<int64_t>(tok) * DSA_INDEX_DIM)[lane];
        const float x[4] = {bf16_bits_to_f32(raw.x & 0xffffu), bf16_bits_to_f32(raw.x >> 16),
                            bf16_bits_to_f32(raw.y & 0xffffu), bf16_bits_to_f32(raw.y >> 16)};
        float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
        if (a.key_fmt == DSA_KEY_FP8) {
            uint8_t *pg = a.idx_pool + page * (DSA_PAGE_SIZE * (DSA_INDEX_DIM + 4));
            am = warp_max(am, 32);
            const float s = am > 0.f ? am / 448.0f : 1.0f;
            const uint32_t c = e4m3_rne(x[0] / s) | (e4m3_rne(x[1] / s) << 8) | (e4m3_rne(x[2] / s) << 16) |
                               (static_cast<uint32_t>(e4m3_rne(x[3] / s)) << 24);
            reinterpret_cast<uint32_t *>(pg + j * DSA_INDEX_DIM)[lane] = c;
            if (lane == 0) reinterpret_cast<float *>(pg + DSA_PAGE_SIZE * DSA_INDEX_DIM)[j] = s;
        } else {
            uint8_t *pg = a.idx_pool + page * (DSA_PAGE_SIZE * (DSA_INDEX_DIM / 2 + DSA_INDEX_DIM / 32));
            am = warp_max(am, 8);  // the 8 lanes of this lane's 32-value block
            int E = 0;
            if (am > 0.f) {
                const int ex = (__float_as_uint(am) >> 23) & 0xff;  // biased exponent: floor(log2) + 127
                E = min(max(ex - 2, 0), 254);                        // subnormal amax clamps to 0 as well
            }
            const float up = ldexpf(1.0f, 127 - E);
            const uint32_t c = e2m1x2_rne(x[0] * up, x[1] * up) | (e2m1x2_rne(x[2] * up, x[3] * up) << 8);
            reinterpret_cast<uint16_t *>(pg + j * (DSA_INDEX_DIM / 2))[lane] = static_cast<uint16_t>(c);
            if ((lane & 7) == 0) pg[DSA_PAGE_SIZE * (DSA_INDEX_DIM / 2) + j * 4 + (lane >> 3)] = static_cast<uint8_t>(E);
        }
    }

    // ---- latent
    const uint16_t *xl = a.latents + static_cast<int64_t>(tok) * DSA_LATENT_DIM;
    const float inv_ts_div = a.tensor_scale;  // divided by, not multiplied by its reciprocal
    if (a.lat_fmt == DSA_LATENT_FP8) {
        uint8_t *row = a.lat_pool + page * (DSA_PAGE_SIZE * DSA_LATENT_DIM) + j * DSA_LATENT_DIM;
        for (int u = lane; u < DSA_LATENT_DIM / 16; u += 32) {  // 36 units of 16 dims
            const uint4 r0 = reinterpret_cast<const uint4 *>(xl)[2 * u];
            const uint4 r1 = reinterpret_cast<const uint4 *>(xl)[2 * u + 1];
            const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t w0 = w[2 * q], w1 = w[2 * q + 1];
                o[q] = e4m3_rne(bf16_bits_to_f32(w0 & 0xffffu) / inv_ts_div) |
                       (e4m3_rne(bf16_bits_to_f32(w0 >> 16) / inv_ts_div) << 8) |
                       (e4m3_rne(bf16_bits_to_f32(w1 & 0xffffu) / inv_ts_div) << 16) |
                       (static_cast<uint32_t>(e4m3_rne(bf16_bits_to_f32(w1 >> 16) / inv_ts_div)) << 24);
            }
            reinterpret_cast<uint4 *>(row)[u] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    } else {
        uint8_t *pg = a.lat_pool + page * (DSA_PAGE_SIZE * 352);
        // lane l owns the 16-value block l of the 512 latent dims
        const uint4 r0 = reinterpret_cast<const uint4 *>(xl)[2 * lane];
        const uint4 r1 = reinterpret_cast<const uint4 *>(xl)[2 * lane + 1];
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float v[16];
        float am = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            v[2 * q] = bf16_bits_to_f32(w[q] & 0xffffu);
            v[2 * q + 1] = bf16_bits_to_f32(w[q] >> 16);
            am = fmaxf(am, fmaxf(fabsf(v[2 * q]), fabsf(v[2 * q + 1])));
        }
        const uint8_t scode = e4m3_rne(am / 6.0f);
        const float sc = e4m3_value(scode);
        uint32_t o[2] = {0u, 0u};
        if (sc > 0.f) {
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q >> 2] |= e2m1x2_rne(v[2 * q] / sc, v[2 * q + 1] / sc) << (8 * (q & 3));
        }
        reinterpret_cast<uint2 *>(pg + j * (DSA_VALUE_DIM / 2))[lane] = make_uint2(o[0], o[1]);
        pg[DSA_PAGE_SIZE * (DSA_VALUE_DIM / 2) + j * (DSA_VALUE_DIM / 16) + lane] = scode;
        // RoPE dims: lane l owns dims 512 + 2l, 513 + 2l
        const uint32_t wr = reinterpret_cast<const uint32_t *>(xl + DSA_VALUE_DIM)[lane];
        const uint32_t rc = e4m3_rne(bf16_bits_to_f32(wr & 0xffffu) / inv_ts_div) |
                            (e4m3_rne(bf16_bits_to_f32(wr >> 16) / inv_ts_div) << 8);
        reinterpret_cast<uint16_t *>(pg + DSA_PAGE_SIZE * (DSA_VALUE_DIM / 2 + DSA_VALUE_DIM / 16) +
                                     j * (DSA_LATENT_DIM - DSA_VALUE_DIM))[lane] = static_cast<uint16_t>(rc);
    }
}

}  // namespace

cudaError_t launch_cache_insert(const InsertArgs &a, cudaStream_t s) {
    if (a.num_tokens == 0) return cudaSuccess;
    cache_insert_kernel<<<(a.num_tokens + 7) / 8, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dsa
