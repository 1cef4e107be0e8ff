// mla_fp8_prefill.cu -- sparse absorbed-MLA over FP8 latents, one CTA per query row, on FP8 tensor
// cores.  Serves prefill rows and decode rows whose selection fits one 128-token part.
//
// What it computes is that of mla.cu (vLLM blog "Day-0 support for Kimi K3.1 Pro", section "Sparse
// attention in K3.1 Pro": exact MLA over the selected tokens' 576-byte FP8 latents; the latent is
// also the value, section "Low-latency decode: fused DSA decode path"; prefill rows, section
// "Prefill: shard attention by token"):
//     S[h, t] = sm_scale * <q[h, :576], kv_t>,   O[h] = sum_t softmax_t(S[h, .]) kv_t[:512]
// with the row's log-sum-exp.
//
// Design (GB300): the row's tokens stream through 64-token tiles with two shared-memory buffers, so
// that the gather of tile i + 1 runs while tile i is multiplied:
//   * the query is converted once per row into the hi + lo e4m3 operand image (mla_fp8_common.cuh)
//     by eight warps while the first tiles' gathers are in flight;
//   * four gather warps copy a tile's 64 latents with 16-byte cp.async in five 128-byte column
//     chunks (four latent chunks, then the RoPE bytes written twice across the row), one mbarrier
//     per chunk, so the S MMAs of a chunk start as soon as it has landed; -1 slots are zero-filled
//     and masked;
//   * S = Q . KV^T runs as 36 e4m3 MMAs (M = 128 heads x N = 64 tokens, K = 32) in two independent
//     accumulation chains, the query's hi terms and its lo terms (consecutive MMAs into one
//     accumulator wait for each other: two chains of 18 take half the time of one of 36); the
//     softmax sums them and frees S as soon as it has read it, so S of tile i + 1 overlaps the
//     softmax of tile i.  The MMA thread issues in readiness order (a tile's PV as soon as its
//     weights exist, else the next landed S chunk);
//   * the softmax (four warps, one thread per head) keeps a reference max m per head and writes
//     P = 2^(s - m + 4) as hi + lo e4m3 (about 8 significant bits); while the tile's max stays
//     within 4.75 of m, P <= 2^8.75 < 448 needs no rescaling.  When it grows further, m moves up
//     to the tile's max and the same warps rescale the accumulated O^T column of that head in
//     TMEM (after the previous PV has completed) before this tile's PV is released;
//   * O^T[dims x heads] += V^T . (P_hi + P_lo)^T runs as 16 MMAs with the latents read MN-major
//     from the same tile (M = 128 dims, N = H heads, K = 32 tokens), the four dim blocks' chains
//     interleaved; P of consecutive tiles alternates between the two 64-byte halves of each
//     head's 128-byte operand row;
//   * at the end eight warps write O = O^T * tensor_scale / sum and the log-sum-exp.
// TMEM: S_hi, S_lo (64 columns each) and O^T (4 x H columns) fill the 512 columns.
#include "mla_fp8_common.cuh"

namespace dsa {

namespace {

using namespace fp8mla;

constexpr int kTile = 64;  // tokens per tile
constexpr int kMaxH = 96;
constexpr int kThreads = 384;  // warp 0 MMA + TMEM; warps 4-7 softmax; warps 8-11 gather; 4-11 query + epilogue
constexpr int kChunk = kTile * 128;  // 8 KB: 64 token rows x 128 B
constexpr int kKvBuf = 5 * kChunk;   // one tile: four latent chunks + the RoPE chunk
constexpr int kQBytesMax = 9 * kMaxH * 128;
constexpr int OFF_Q = 0;
constexpr int OFF_KV = kQBytesMax;  // two tile buffers; Q rows >= H of the last block alias into them
constexpr int OFF_P = OFF_KV + 2 * kKvBuf;
constexpr int kPBytes = 2 * kMaxH * 128;  // P hi, P lo: [H heads][128 B]; tile parity b uses bytes 64b..64b+63
constexpr int OFF_QS = OFF_P + kPBytes;   // [128] fp32 2^-e_h of the query image
constexpr int OFF_ALPHA = OFF_QS + 128 * 4;  // [128] fp32 rescale factor of each head's O^T column
constexpr int OFF_OSC = OFF_ALPHA + 128 * 4;  // [128] fp32 output factor tensor_scale / sum
constexpr int OFF_VALID = OFF_OSC + 128 * 4;  // [2][64] bytes: tile token has a slot
constexpr int OFF_RMASK = OFF_VALID + 2 * kTile;  // [4] heads of each lane quadrant to rescale
constexpr int OFF_BARS = OFF_RMASK + 16;
// kv_full[2][5] (gather -> MMA, softmax), q_ready (query image -> MMA), s_full (MMA -> softmax),
// s_free (softmax -> MMA), p_full[2] (softmax -> MMA), pv_done[2] (MMA -> gather, softmax,
// epilogue), mma_idle (all MMAs retired)
constexpr int kNumBars = 10 + 1 + 1 + 1 + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BARS + kNumBars * 8;
constexpr int kSmemBytes = OFF_MISC + 32 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0 && kKvBuf % 1024 == 0, "operand blocks at 1024-byte boundaries");
static_assert(OFF_BARS % 8 == 0, "mbarrier alignment");
constexpr uint32_t kTmemCols = 512;
// S = Q_hi . KV^T + Q_lo . KV^T as two independent accumulation chains (18 MMAs each instead of
// one chain of 36: consecutive MMAs into one accumulator wait for each other), summed by the softmax
constexpr uint32_t kTmemSHi = 0, kTmemSLo = kTile;
constexpr uint32_t kTmemO = 2 * kTile;  // O^T after S
constexpr int kGatherThreads = 128;
constexpr int kSoftmaxThreads = 128;
// P = 2^(s - m + kPExp) <= 448 (the e4m3 maximum) while s <= m + kHeadroom: a tile's max may exceed
// the reference max m by kHeadroom log2 units before the head is rescaled.  Weights down to 2^-6
// (10 binades below the reference token) keep all 8 significant bits of their hi + lo terms.
constexpr float kPExp = 4.0f;
constexpr float kHeadroom = 4.75f;
constexpr int kBarSoftmax = 1;      // named barrier of the four softmax warps
constexpr int kBarEpilogue = 2;     // named barrier of warps 4-11

// OR of `pred` over the `n` threads at named barrier `id` (all of them wait).
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "barrier.cta.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// One 32-bit TMEM column of the warp's 32 lanes (lane i: TMEM lane taddr.lane + i).
__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t &r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r) : "memory");
}

// Bounded wait that ignores the abort flag: used once, for the MMAs still in flight, before the
// CTA frees its TMEM.
__device__ __forceinline__ void wait_retired(uint64_t *bar, int32_t *status) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, 0)) {
        if (clock64() - t0 > kWaitTimeoutCycles) {
            report(status, DSA_ERR_TIMEOUT);
            return;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_fp8_row_kernel(const MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem + OFF_Q;
    uint8_t *kv = smem + OFF_KV;
    uint8_t *pb = smem + OFF_P;
    float *qscale = reinterpret_cast<float *>(smem + OFF_QS);
    float *alpha = reinterpret_cast<float *>(smem + OFF_ALPHA);
    float *osc = reinterpret_cast<float *>(smem + OFF_OSC);
    uint8_t *valid = smem + OFF_VALID;
    uint32_t *rmask = reinterpret_cast<uint32_t *>(smem + OFF_RMASK);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *kv_full = bars;       // [2][5] gather chunk c of buffer b -> MMA, softmax (count 4 warps)
    uint64_t *q_ready = bars + 10;  // query image -> MMA
    uint64_t *s_full = bars + 11;   // MMA -> softmax (commit)
    uint64_t *s_free = bars + 12;   // softmax -> MMA (count 4 warps): S read, the next tile's S may start
    uint64_t *p_full = bars + 13;   // [2] softmax -> MMA (count 4 warps)
    uint64_t *pv_done = bars + 15;  // [2] MMA -> gather, softmax, epilogue (commit)
    uint64_t *mma_idle = bars + 17;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.num_heads;
    const int row = blockIdx.x;
    const int ntiles = (a.k + kTile - 1) / kTile;
    const int32_t *row_slots = a.slots + static_cast<int64_t>(row) * a.k;

    if (tid == 0) {
        *abort = 0;
        for (int i = 0; i < 10; ++i) mbar_init(&kv_full[i], kGatherThreads / 32);
        mbar_init(q_ready, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, kSoftmaxThreads / 32);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&p_full[b], kSoftmaxThreads / 32);
            mbar_init(&pv_done[b], 1);
        }
        mbar_init(mma_idle, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // on-chip set-up above; global memory from here on, once the previous kernel has finished
    pdl_launch_dependents();
    pdl_wait();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer: S(i), then PV(i - 1)
            const uint32_t blk = static_cast<uint32_t>(H) * 128;
            const uint32_t idesc_s = make_idesc(128, kTile, 0, 0, false, false);
            const uint32_t idesc_pv = make_idesc(128, H, 0, 0, true, false);
            const uint32_t qa = smem_u32(qs), kva = smem_u32(kv), pa = smem_u32(pb);
            bool ok = mbar_wait(q_ready, 0, abort, a.status);
            // Issue in readiness order: PV(np) as soon as its weights are written (its completion
            // frees the tile buffer the gather of tile np + 2 waits for), else the next chunk of
            // S(ns) once it has landed and the softmax has read S(ns - 1).
            int ns = 0, nc = 0, np = 0;
            long long t_last = clock64();
            while (ok && np < ntiles) {
                bool progressed = false;
                if (np < ns && mbar_test_wait(&p_full[np & 1], (np >> 1) & 1)) {
                    tc_fence_after();
                    const int b = np & 1;
                    const uint32_t kb = kva + b * kKvBuf;
                    // four independent accumulation chains (the dim blocks), interleaved
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                        for (int part = 0; part < 2; ++part)
#pragma unroll
                            for (int dblk = 0; dblk < 4; ++dblk)
                                mma_f8(tmem + kTmemO + dblk * H, sdesc_sw128(kb + dblk * kChunk + ks * 4096, 16, 1024),
                                       sdesc_sw128(pa + part * blk + b * 64 + ks * 32, 16, 1024), idesc_pv,
                                       (np > 0 || ks > 0 || part > 0) ? 1u : 0u);
                    mma_commit(&pv_done[b]);
                    ++np;
                    progressed = true;
                } else if (ns < ntiles) {
                    const int b = ns & 1;
                    const uint32_t ph = (ns >> 1) & 1;
                    if ((nc > 0 || ns == 0 || mbar_test_wait(s_free, (ns - 1) & 1)) &&
                        mbar_test_wait(&kv_full[b * 5 + nc], ph)) {
                        tc_fence_after();
                        const uint32_t kb = kva + b * kKvBuf + nc * kChunk;
                        if (nc < 4) {  // latent dims 128 nc ..: Q_hi -> S_hi, Q_lo -> S_lo, alternating
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                                for (int part = 0; part < 2; ++part)
                                    mma_f8(tmem + (part ? kTmemSLo : kTmemSHi),
                                           sdesc_sw128(qa + (part * 4 + nc) * blk + ks * 32, 16, 1024),
                                           sdesc_sw128(kb + ks * 32, 16, 1024), idesc_s, (nc | ks) ? 1u : 0u);
                        } else {  // RoPE dims: [Q_hi | Q_lo] against [kv | kv]
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                mma_f8(tmem + (ks < 2 ? kTmemSHi : kTmemSLo), sdesc_sw128(qa + 8 * blk + ks * 32, 16, 1024),
                                       sdesc_sw128(kb + ks * 32, 16, 1024), idesc_s, 1u);
                        }
                        if (++nc == 5) {
                            mma_commit(s_full);
                            nc = 0;
                            ++ns;
                        }
                        progressed = true;
                    }
                }
                if (progressed) {
                    t_last = clock64();
                } else if (*abort) {
                    ok = false;
                } else if (clock64() - t_last > kWaitTimeoutCycles) {
                    *abort = 1;
                    report(a.status, DSA_ERR_TIMEOUT);
                    ok = false;
                } else {
                    __nanosleep(20);
                }
            }
            // every MMA issued has retired before the CTA frees its TMEM (after an abort too)
            mma_commit(mma_idle);
            wait_retired(mma_idle, a.status);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- query image (warps 4-11)
        auto convert_q = [&]() {
            // warp w converts heads w - 4 + 8 j; the loads of four heads are in flight together
            const uint16_t *qrow = a.q + static_cast<int64_t>(row) * H * DSA_LATENT_DIM;
            for (int h0 = warp - 4; h0 < H; h0 += 32) {
                int4 x[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (h0 + 8 * j < H) load_q_head(qrow + (h0 + 8 * j) * DSA_LATENT_DIM, lane, x[j]);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (h0 + 8 * j < H) convert_q_head(x[j], h0 + 8 * j, H, qs, qscale + h0 + 8 * j, a.status, lane);
            }
            fence_async_smem();
            named_bar_sync(kBarEpilogue, 256);
            if (tid == 128) mbar_arrive(q_ready);
        };
        bool ok = true;
        if (warp >= 8) {
            // ------------------------------------------------------------ gather (warps 8-11)
            // Thread g copies 16-byte unit u = g % 8 of tokens g / 8 + 16 m (m < 4) in every chunk; a
            // warp's copies of one chunk are four full 128-byte rows.
            const int g = tid - 256;
            const int u = g & 7, t0 = g >> 3;
            const uint32_t kvb = smem_u32(kv);
            auto issue = [&](int i) {
                const int b = i & 1;
                int32_t slot[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = t0 + 16 * m, tg = i * kTile + t;
                    int32_t s = tg < a.k ? row_slots[tg] : -1;
                    if (s >= 0 && static_cast<int64_t>(s) >= a.num_pages * DSA_PAGE_SIZE) {
                        report(a.status, DSA_ERR_BOUNDS);
                        s = -1;
                    }
                    slot[m] = s;
                    if (u == 0) valid[b * kTile + t] = s >= 0 ? 1 : 0;
                }
#pragma unroll
                for (int c = 0; c < 5; ++c) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int t = t0 + 16 * m;
                        const int src_off = c < 4 ? c * 128 + u * 16 : DSA_VALUE_DIM + (u & 3) * 16;
                        const uint8_t *src = a.pool + static_cast<int64_t>(max(slot[m], 0)) * DSA_LATENT_DIM + src_off;
                        cp_async16(kvb + b * kKvBuf + c * kChunk + sw128(t, u), src, slot[m] >= 0);
                    }
                    cp_async_commit();
                }
            };
            auto done = [&](int b, int c) {  // chunk c of buffer b has landed for this thread
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kv_full[b * 5 + c]);
            };
            // the first two tiles' copies are in flight while the query is converted
            issue(0);
            if (ntiles > 1) issue(1);
            convert_q();
            if (ntiles > 1) {
                cp_async_wait<9>();
                done(0, 0);
                cp_async_wait<8>();
                done(0, 1);
                cp_async_wait<7>();
                done(0, 2);
                cp_async_wait<6>();
                done(0, 3);
                cp_async_wait<5>();
                done(0, 4);
            }
            for (int i = ntiles > 1 ? 1 : 0; i < ntiles; ++i) {
                const int b = i & 1;
                if (i >= 2) {
                    // buffer b is free once PV(i - 2) has read it
                    ok = mbar_wait_warp(&pv_done[b], ((i >> 1) & 1) ^ 1, abort, a.status);
                    if (!ok) break;
                    issue(i);
                }
                cp_async_wait<4>();
                done(b, 0);
                cp_async_wait<3>();
                done(b, 1);
                cp_async_wait<2>();
                done(b, 2);
                cp_async_wait<1>();
                done(b, 3);
                cp_async_wait<0>();
                done(b, 4);
            }
            cp_async_wait<0>();  // nothing of this thread's is in flight past this point
        } else {
            // ------------------------------------------------------------ softmax (warps 4-7): thread
            // h = 32 quad + lane takes head h over each tile's 64 tokens
            convert_q();
        }
        const int quad = warp & 3;
        const int h = quad * 32 + lane;
        const bool live = h < H;
        float m_ref = -INFINITY, l = 0.f;
        if (warp < 8) {
            const float s_scale = live ? a.tensor_scale * a.sm_scale * 1.4426950408889634f * qscale[h] : 0.f;
            const uint32_t srow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            for (int i = 0; i < ntiles; ++i) {
                const int b = i & 1;
                const uint32_t ph = (i >> 1) & 1;
                if (ok) ok = mbar_wait_warp(s_full, i & 1, abort, a.status) &&
                             mbar_wait_warp(&kv_full[b * 5 + 4], ph, abort, a.status);
                uint32_t sr[2][32];
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t lo[32];
                        tmem_ld32(srow + kTmemSHi + 32 * c, sr[c]);
                        tmem_ld32(srow + kTmemSLo + 32 * c, lo);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            sr[c][j] = __float_as_uint(__uint_as_float(sr[c][j]) + __uint_as_float(lo[j]));
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(s_free);  // S may take the next tile's products
                }
                uint32_t vw[16];  // valid bytes of the tile's 64 tokens
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v4 = reinterpret_cast<const uint4 *>(valid + b * kTile)[q];
                    vw[4 * q] = v4.x;
                    vw[4 * q + 1] = v4.y;
                    vw[4 * q + 2] = v4.z;
                    vw[4 * q + 3] = v4.w;
                }
                auto is_valid = [&](int t) { return ((vw[t >> 2] >> (8 * (t & 3))) & 0xffu) != 0u; };
                float mt = -INFINITY;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (is_valid(32 * c + j)) mt = fmaxf(mt, __uint_as_float(sr[c][j]) * s_scale);
                // reference max: set by the first tile with a valid token, moved up (with a rescale of
                // the head's sum and O^T column) when a tile's max exceeds it by more than the headroom
                bool resc = false;
                float al = 1.0f;
                if (ok && live && mt > -INFINITY) {
                    if (m_ref == -INFINITY) {
                        m_ref = mt;
                    } else if (mt > m_ref + kHeadroom) {
                        al = fast_exp2(m_ref - mt);
                        m_ref = mt;
                        l *= al;
                        resc = true;
                    }
                }
                const float msub = (m_ref == -INFINITY) ? 0.f : m_ref - kPExp;
                // P half b is free once PV(i - 2) has read it
                if (ok && i >= 2) ok = mbar_wait_warp(&pv_done[b], ph ^ 1, abort, a.status);
                if (ok) {
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t hw[8], lw[8];
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            float p[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                p[x] = is_valid(32 * c + j + x)
                                           ? fast_exp2(__uint_as_float(sr[c][j + x]) * s_scale - msub)
                                           : 0.f;
                                ls[x] += p[x];
                            }
                            p_split4(p, hw[j / 4], lw[j / 4]);
                        }
                        if (live) {
                            const int u = 4 * b + 2 * c;  // tokens 32c .. 32c + 31 of half b
                            *reinterpret_cast<uint4 *>(pb + sw128(h, u)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                            *reinterpret_cast<uint4 *>(pb + sw128(h, u + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                            uint8_t *pl = pb + H * 128;
                            *reinterpret_cast<uint4 *>(pl + sw128(h, u)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                            *reinterpret_cast<uint4 *>(pl + sw128(h, u + 1)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
                        }
                    }
                    if (live) l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                }
                fence_async_smem();
                // rescale the O^T columns of heads whose reference max moved, once PV(i - 1) has
                // completed and before PV(i) is released: each warp its 32 lanes (dims) of the
                // four column blocks of every such head
                alpha[h] = al;
                const uint32_t bal = __ballot_sync(0xffffffffu, resc);
                if (lane == 0) rmask[quad] = bal;
                if (named_bar_or(kBarSoftmax, kSoftmaxThreads, resc)) {
                    if (ok && i >= 1) ok = mbar_wait_warp(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, abort, a.status);
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int q = 0; q < 4; ++q) {
                            uint32_t m = rmask[q];
                            while (m != 0u) {
                                const int hh = 32 * q + __ffs(m) - 1;
                                m &= m - 1u;
                                const float f = alpha[hh];
                                uint32_t v[4];
#pragma unroll
                                for (int dblk = 0; dblk < 4; ++dblk) tmem_ld1(srow + kTmemO + dblk * H + hh, v[dblk]);
                                tmem_ld_wait();
#pragma unroll
                                for (int dblk = 0; dblk < 4; ++dblk) {
                                    v[dblk] = __float_as_uint(__uint_as_float(v[dblk]) * f);
                                    tmem_st1(srow + kTmemO + dblk * H + hh, v[dblk]);
                                }
                            }
                        }
                        tmem_st_wait();
                    }
                    named_bar_sync(kBarSoftmax, kSoftmaxThreads);  // alpha and rmask are rewritten by the next tile
                }
                tc_fence_before();
                __syncwarp();
                if (ok && lane == 0) mbar_arrive(&p_full[b]);
            }
            // the row's output factor and log-sum-exp (natural log)
            osc[h] = (l > 0.f) ? a.tensor_scale / l : 0.f;
            if (live && a.lse != nullptr)
                a.lse[static_cast<int64_t>(row) * H + h] =
                    (l > 0.f) ? (m_ref - kPExp + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        // ---------------------------------------------------------------- epilogue (warps 4-11): warps
        // 4-7 store dim blocks 0 and 1 of O, warps 8-11 blocks 2 and 3; lane = dim
        named_bar_sync(kBarEpilogue, 256);
        const int last = ntiles - 1;
        if (ok && !*abort) ok = mbar_wait_warp(&pv_done[last & 1], (last >> 1) & 1, abort, a.status);
        if (ok && !*abort) {
            tc_fence_after();
            const int j0 = warp < 8 ? 0 : 2;
            float *orow = a.out + static_cast<int64_t>(row) * H * DSA_VALUE_DIM;
            for (int j = j0; j < j0 + 2; ++j) {
                const int d = 128 * j + 32 * quad + lane;
                const uint32_t tb = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kTmemO + j * H;
#pragma unroll 1
                for (int c = 0; c < H; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tb + c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 16; ++x)
                        orow[static_cast<int64_t>(c + x) * DSA_VALUE_DIM + d] = __uint_as_float(v[x]) * osc[c + x];
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

cudaError_t launch_sparse_mla_fp8_rows(const MlaArgs &a, cudaStream_t s) {
    if (a.num_rows == 0) return cudaSuccess;
    if (a.num_heads < 16 || a.num_heads > kMaxH || a.num_heads % 16 != 0 || a.k < 1) return cudaErrorInvalidValue;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(sparse_mla_fp8_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    return launch_pdl(sparse_mla_fp8_row_kernel, dim3(static_cast<unsigned>(a.num_rows)), dim3(kThreads), kSmemBytes, s,
                      a);
}

}  // namespace dsa
