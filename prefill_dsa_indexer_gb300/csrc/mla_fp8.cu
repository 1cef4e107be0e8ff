// mla_fp8.cu -- split-K sparse absorbed-MLA decode over FP8 latents, on FP8 tensor cores.
//
// What it computes is that of mla.cu (vLLM blog "Day-0 support for Kimi K3.1
// Pro", section "Sparse attention in K3.1 Pro": exact MLA over the 2,048
// selected tokens' 576-byte FP8 latents; the latent is also the value,
// section "Low-latency decode: fused DSA decode path"):
//     S[h, t] = sm_scale * <q[h, :576], kv_t>,   O[h] = sum_t softmax_t(S[h, .]) kv_t[:512]
// for one 128-token part of a row's selection per CTA; mla_combine_kernel
// merges the parts by log-sum-exp.
//
// Design (GB300): both products run as e4m3 x e4m3 -> fp32 MMAs on the
// latents exactly as stored, so a part is ONE 128-token tile with no decode
// step and no serial chain of tiles:
//   * the query is written (once per row, by mla_qprep_fp8_kernel) as the sum
//     of two e4m3 terms, q * 2^e_h = hi + lo, with a power of two e_h per head
//     that puts the head's largest |q| in (224, 448].  A bf16 value has 8
//     significant bits and each e4m3 term carries 4, so hi + lo equals
//     q * 2^e_h exactly for every |q * 2^e_h| >= 1/4 (all but values some 2^-10
//     below the head's largest), and S = KV . hi + KV . lo is the fp32 sum of
//     exact products: 18 K-steps x 2 MMAs of M = 128 (heads) x N = 128 tokens;
//     the RoPE dims take 4 of them, the hi and lo halves of a 128-byte row
//     against a row that holds the token's 64 RoPE bytes twice;
//   * P = 2^(s - m + 8) <= 256 (m the part's own max, so no rescaling) is also
//     written as hi + lo e4m3 (hi: P rounded to 3 mantissa bits; lo: the rest,
//     rounded; about 8 significant bits, the precision of bf16), and O^T[dims x heads] += V^T . P^T runs as 2 x 16 MMAs with the
//     latents read MN-major from the same shared-memory tile (M = 128 dims,
//     N = H heads, K = 32 tokens);
//   * 8 gather warps fill the tile's four latent chunks (128-byte columns) with 16-byte cp.async
//     copies, one mbarrier per chunk, so the S MMAs of a chunk start as soon as it has landed;
//     three more warps fetch the RoPE chunk (each token's 64 RoPE bytes written twice across its
//     row) at the same time; unused slots (-1) are zero-filled and masked;
//   * the softmax runs on the 8 gather warps, two per TMEM lane quadrant, each
//     thread one head over 64 tokens; the two halves of a head swap their max and
//     sum through shared memory;
//   * S (128 TMEM columns) and O^T (4 x H columns) share the 512 columns;
//     the part's output is normalised by its own sum, stored in fp16 with its
//     (max, sum), and merged by mla_combine_kernel as in mla.cu.
#include "mla_fp8_common.cuh"

namespace dsa {

namespace {

using namespace fp8mla;

constexpr int kTok = kMlaTokensPerSplit;  // 128 tokens: the whole part
constexpr int kMaxH = 96;
constexpr int kThreads = 384;  // warp 0 MMA + TMEM; warps 4-11 gather, softmax and epilogue
constexpr int kChunk = kTok * 128;          // 16 KB: 128 token rows x 128 B
constexpr int kQBytesMax = 9 * kMaxH * 128;  // hi x 4, lo x 4, RoPE hi|lo
constexpr int OFF_Q = 0;
constexpr int OFF_KV = kQBytesMax;  // directly after Q: rows >= H of the last Q block alias into it
constexpr int OFF_P = OFF_KV + 5 * kChunk;
constexpr int kPBytes = 2 * kMaxH * 128;  // P hi, P lo: [H heads][128 tokens] e4m3
constexpr int OFF_INVL = OFF_P + kPBytes;
constexpr int OFF_RED = OFF_INVL + 128 * 4;    // [4][128] partial max / sum exchange of the softmax
constexpr int OFF_MASK = OFF_RED + 4 * 128 * 4;
constexpr int OFF_BARS = OFF_MASK + 16;
constexpr int kNumBars = 10;
constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
constexpr int kSmemBytes = OFF_MISC + 32 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0, "operand blocks at 1024-byte boundaries");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = kTok;  // O^T after the S accumulator

// ---------------------------------------------------------------- query preparation
// One warp per (row, head): the head's 576 bf16 values become hi + lo e4m3 at 2^e_h, written as
// the kernel's 128-byte-swizzled K-major operand blocks, plus 2^-e_h after the image.  A warp
// takes kQprepHeads heads (more heads per warp occupy fewer SMs but take proportionally longer).
constexpr int kQprepHeads = 1;
__device__ __forceinline__ void qprep_head(const MlaArgs &a, int64_t w, int lane);
__global__ void __launch_bounds__(256) mla_qprep_fp8_kernel(const MlaArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kQprepHeads;
#pragma unroll
    for (int i = 0; i < kQprepHeads; ++i)
        if (w0 + i < static_cast<int64_t>(a.num_rows) * a.num_heads) qprep_head(a, w0 + i, threadIdx.x & 31);
}

__device__ __forceinline__ void qprep_head(const MlaArgs &a, int64_t w, int lane) {
    const int H = a.num_heads;
    const int64_t row = w / H;
    const int h = static_cast<int>(w % H);
    uint8_t *img = a.qprep + row * mla_qprep_row_bytes(H);
    int4 x[4];
    load_q_head(a.q + w * DSA_LATENT_DIM, lane, x);
    convert_q_head(x, h, H, img, reinterpret_cast<float *>(img + 9 * H * 128) + h, a.status, lane);
}

// ---------------------------------------------------------------- attention over one part
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_fp8_kernel(const MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem + OFF_Q;
    uint8_t *kv = smem + OFF_KV;
    uint8_t *ph = smem + OFF_P;
    float *inv_l = reinterpret_cast<float *>(smem + OFF_INVL);
    float *red = reinterpret_cast<float *>(smem + OFF_RED);
    uint32_t *mask = reinterpret_cast<uint32_t *>(smem + OFF_MASK);  // [4] valid-token bits
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *kv_full = bars;       // [5] gather chunk c -> MMA (latent chunks: 8 warps; RoPE: 3)
    uint64_t *q_full = bars + 5;    // bulk copy of the prepared Q -> MMA
    uint64_t *s_full = bars + 6;    // MMA -> softmax (commit)
    uint64_t *p_full = bars + 7;    // softmax -> MMA (count 8)
    uint64_t *pv_done = bars + 8;   // MMA -> epilogue (commit)
    uint64_t *stats = bars + 9;     // softmax -> epilogue (count 4)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.num_heads;
    const int row = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
    const int t_begin = split * kTok, n_tok = min(kTok, a.k - t_begin);
    const int32_t *row_slots = a.slots + static_cast<int64_t>(row) * a.k + t_begin;
    const uint8_t *qimg = a.qprep + static_cast<int64_t>(row) * mla_qprep_row_bytes(H);

    if (tid == 0) {
        *abort = 0;
        for (int c = 0; c < 4; ++c) mbar_init(&kv_full[c], 8);  // latent chunks: warps 4-11
        mbar_init(&kv_full[4], 3);                                // RoPE chunk: warps 1-3
        mbar_init(q_full, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, 8);
        mbar_init(pv_done, 1);
        mbar_init(stats, 4);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid < 4) mask[tid] = 0u;
    // on-chip set-up above; global memory from here on, once the previous kernel has finished
    pdl_launch_dependents();
    pdl_wait();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ Q copy + MMA issuer
            const uint32_t blk = static_cast<uint32_t>(H) * 128;
            mbar_arrive_expect_tx(q_full, 9 * blk);
            for (int c = 0; c < 9; ++c) bulk_load(qs + c * blk, qimg + c * blk, blk, q_full);
            const uint32_t idesc_s = make_idesc(128, kTok, 0, 0, false, false);
            const uint32_t idesc_pv = make_idesc(128, H, 0, 0, true, false);
            const uint32_t qa = smem_u32(qs), kva = smem_u32(kv), pa = smem_u32(ph);
            bool ok = mbar_wait(q_full, 0, abort, a.status);
            // S = (hi + lo) . KV^T over the four latent chunks, then the RoPE chunk
            for (int c = 0; ok && c < 5; ++c) {
                ok = mbar_wait(&kv_full[c], 0, abort, a.status);
                if (!ok) break;
                tc_fence_after();
                if (c < 4) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                        for (int part = 0; part < 2; ++part)
                            mma_f8(tmem, sdesc_sw128(qa + (part * 4 + c) * blk + ks * 32, 16, 1024),
                                   sdesc_sw128(kva + c * kChunk + ks * 32, 16, 1024), idesc_s,
                                   (c | ks | part) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f8(tmem, sdesc_sw128(qa + 8 * blk + ks * 32, 16, 1024),
                               sdesc_sw128(kva + 4 * kChunk + ks * 32, 16, 1024), idesc_s, 1u);
                }
            }
            if (ok) mma_commit(s_full);
            // O^T[dims x heads] = V^T . (P_hi + P_lo)^T: V^T read MN-major from the latent chunks
            if (ok) ok = mbar_wait(p_full, 0, abort, a.status);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                        for (int part = 0; part < 2; ++part)
                            mma_f8(tmem + kTmemO + j * H, sdesc_sw128(kva + j * kChunk + ks * 4096, 16, 1024),
                                   sdesc_sw128(pa + part * H * 128 + ks * 32, 16, 1024), idesc_pv,
                                   (ks | part) ? 1u : 0u);
                mma_commit(pv_done);
            }
        }
    } else if (warp < 4) {
        // ---------------------------------------------------------------- gather of the RoPE chunk
        // (warps 1-3): each token's 64 RoPE bytes, written twice across its 128-byte row
        const uint32_t kvb = smem_u32(kv) + 4 * kChunk;
        for (int e = tid - 32; e < kTok * 8; e += 96) {
            const int t = e >> 3, u = e & 7;
            int32_t s = t < n_tok ? row_slots[t] : -1;
            if (s >= 0 && static_cast<int64_t>(s) >= a.num_pages * DSA_PAGE_SIZE) s = -1;  // reported by warps 4-11
            const uint8_t *src = a.pool + static_cast<int64_t>(max(s, 0)) * DSA_LATENT_DIM + DSA_VALUE_DIM + (u & 3) * 16;
            cp_async16(kvb + sw128(t, u), src, s >= 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_full[4]);
    } else if (warp >= 4) {
        const int gtid = tid - 128;      // 0..255
        const int quad = warp & 3;
        const bool lower = warp < 8;  // warps 4-7: dim blocks 0, 1 of the output; warps 8-11: 2, 3
        bool ok = true;
        // ---------------------------------------------------------------- gather
        // Thread gtid copies 16-byte unit u = gtid % 8 of tokens gtid / 8 + 32 i (i < 4) in every
        // chunk; a warp's copies of one chunk are four full 128-byte rows.
        {
            const int u = gtid & 7, t0 = gtid >> 3;
            int32_t slot[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = t0 + 32 * i;
                int32_t s = t < n_tok ? row_slots[t] : -1;
                if (s >= 0 && static_cast<int64_t>(s) >= a.num_pages * DSA_PAGE_SIZE) {
                    report(a.status, DSA_ERR_BOUNDS);
                    s = -1;
                }
                slot[i] = s;
                if (u == 0 && s >= 0) atomicOr(&mask[t >> 5], 1u << (t & 31));
            }
            const uint32_t kvb = smem_u32(kv);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t0 + 32 * i;
                    const uint8_t *src = a.pool + static_cast<int64_t>(max(slot[i], 0)) * DSA_LATENT_DIM + c * 128 + u * 16;
                    cp_async16(kvb + c * kChunk + sw128(t, u), src, slot[i] >= 0);
                }
                cp_async_commit();
            }
            // chunk c is complete once all but the 3 - c later groups have landed (the valid-token
            // mask above is complete once chunk 3 is)
            auto done = [&](int c) {
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kv_full[c]);
            };
            cp_async_wait<3>();
            done(0);
            cp_async_wait<2>();
            done(1);
            cp_async_wait<1>();
            done(2);
            cp_async_wait<0>();
            done(3);
        }
        {
            // ------------------------------------------------------------ softmax, 8 warps: thread
            // (half, h) takes head h = 32 quad + lane over tokens [64 half, 64 half + 64)
            const int h = quad * 32 + lane, half = (warp - 4) >> 2;
            ok = mbar_wait_warp(s_full, 0, abort, a.status) && mbar_wait_warp(&kv_full[3], 0, abort, a.status);
            float m = -INFINITY, l = 0.f, lp = 0.f;
            const float hs = h < H ? reinterpret_cast<const float *>(qimg + 9 * H * 128)[h] : 0.f;
            const float s_scale = a.tensor_scale * a.sm_scale * 1.4426950408889634f * hs;
            const uint32_t srow = tmem + (static_cast<uint32_t>(quad * 32) << 16) + 64 * half;
            const uint32_t mk[2] = {mask[2 * half], mask[2 * half + 1]};
            float mp = -INFINITY;
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t sr[32];
                    tmem_ld32(srow + 32 * c, sr);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if ((mk[c] >> j) & 1u) mp = fmaxf(mp, __uint_as_float(sr[j]) * s_scale);
                }
            }
            red[half * 128 + h] = mp;
            named_bar_sync(1, 256);
            m = fmaxf(red[h], red[128 + h]);
            if (ok) {
                // P = 2^(s - m + 8) <= 256 as hi + lo: hi = P rounded to 3 mantissa bits (exact in
                // e4m3), lo = P - hi (exact in fp32) rounded to e4m3
                const float msub = (m == -INFINITY) ? 0.f : m - 8.0f;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t sr[32];
                    tmem_ld32(srow + 32 * c, sr);
                    tmem_ld_wait();
                    uint32_t hw[8], lw[8];
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        float p[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            p[x] = ((mk[c] >> (j + x)) & 1u)
                                       ? fast_exp2(__uint_as_float(sr[j + x]) * s_scale - msub)
                                       : 0.f;
                            ls[x] += p[x];
                        }
                        p_split4(p, hw[j / 4], lw[j / 4]);
                    }
                    if (h < H) {
                        const int u = 4 * half + 2 * c;
                        *reinterpret_cast<uint4 *>(ph + sw128(h, u)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4 *>(ph + sw128(h, u + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                        uint8_t *pl = ph + H * 128;
                        *reinterpret_cast<uint4 *>(pl + sw128(h, u)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        *reinterpret_cast<uint4 *>(pl + sw128(h, u + 1)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
                    }
                }
                lp = (ls[0] + ls[1]) + (ls[2] + ls[3]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            red[256 + half * 128 + h] = lp;
            named_bar_sync(1, 256);
            l = red[256 + h] + red[384 + h];
            // the part's statistics (log2 units): max m - 8 of the P written, and its sum
            if (half == 0) {
                inv_l[h] = (l > 0.f) ? 1.0f / l : 0.f;
                if (h < H) {
                    float *ml = a.part_ml + (static_cast<int64_t>(row) * a.splits + split) * H * 2;
                    ml[2 * h] = (l > 0.f) ? m - 8.0f : -INFINITY;
                    ml[2 * h + 1] = l;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(stats);
            }
        }
        // ---------------------------------------------------------------- epilogue, 8 warps:
        // warps 4-7 store dim blocks 0 and 1 of O, warps 8-11 blocks 2 and 3; lane = dim.  The part
        // is written in fp16 (decoded-latent units, |value| <= 448); neighbouring lanes (dims d,
        // d + 1) swap one value so each lane stores a 4-byte pair of dims of one head.
        if (ok) ok = mbar_wait_warp(pv_done, 0, abort, a.status);
        if (ok) ok = mbar_wait_warp(stats, 0, abort, a.status);
        if (ok) {
            tc_fence_after();
            __half *dst_h = reinterpret_cast<__half *>(a.part_o) +
                            (static_cast<int64_t>(row) * a.splits + split) * H * DSA_VALUE_DIM;
            const bool odd = (lane & 1) != 0;
            const int j0 = lower ? 0 : 2;
            for (int j = j0; j < j0 + 2; ++j) {
                const int d = 128 * j + 32 * quad + lane;
                const uint32_t tb = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kTmemO + j * H;
                for (int c = 0; c < H; c += 32) {
                    uint32_t v[32];
                    const bool full32 = c + 32 <= H;
                    if (full32) tmem_ld32(tb + c, v);
                    else tmem_ld16(tb + c, *reinterpret_cast<uint32_t(*)[16]>(v));
                    tmem_ld_wait();
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
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        if (x >= 16 && !full32) break;
                        const float o0 = __uint_as_float(v[x]) * il[x];
                        const float o1 = __uint_as_float(v[x + 1]) * il[x + 1];
                        const float got = __shfl_xor_sync(0xffffffffu, odd ? o0 : o1, 1);
                        const __half2 hh = odd ? __floats2half2_rn(got, o1) : __floats2half2_rn(o0, got);
                        const int at = (c + x + (odd ? 1 : 0)) * DSA_VALUE_DIM + (d & ~1);
                        *reinterpret_cast<__half2 *>(dst_h + at) = hh;
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

}  // namespace

cudaError_t launch_mla_qprep_fp8(const MlaArgs &a, cudaStream_t s) {
    if (a.num_rows == 0 || a.qprep == nullptr) return cudaSuccess;
    const int64_t warps = (static_cast<int64_t>(a.num_rows) * a.num_heads + kQprepHeads - 1) / kQprepHeads;
    return launch_pdl(mla_qprep_fp8_kernel, dim3(static_cast<unsigned>((warps + 7) / 8)), dim3(256), 0, s, a);
}

cudaError_t launch_sparse_mla_fp8_decode(const MlaArgs &a, cudaStream_t s) {
    if (a.num_rows == 0) return cudaSuccess;
    if (a.num_heads < 16 || a.num_heads > kMaxH || a.num_heads % 16 != 0 || a.splits < 2 || a.qprep == nullptr)
        return cudaErrorInvalidValue;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(sparse_mla_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    if (!a.q_prepared) {
        cudaError_t e = launch_mla_qprep_fp8(a, s);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_pdl(sparse_mla_fp8_kernel, dim3(a.num_rows * a.splits), dim3(kThreads), kSmemBytes, s, a);
    if (e != cudaSuccess) return e;
    return launch_mla_combine(a, s);
}

}  // namespace dsa
