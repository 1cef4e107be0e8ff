/*
 * dsa_oracle.c -- plain, slow CPU oracle for the DSA layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this code:
 * only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no code, header, table or constant generator
 * with the CUDA library; the two meet only at the byte layouts of their
 * inputs and outputs.
 *
 * What it computes (source: vLLM blog "Day-0 support for Kimi K3.1 Pro",
 * section "Sparse attention in K3.1 Pro" (Fig. 1), "One KV cache, three
 * states", "Low-latency decode: fused DSA decode path", and the AMD section
 * "Quantization: native MXFP4 indexer"):
 *
 *   indexer   logit[r,t] = sum_h w[r,h] * max(0, s_t * <q[r,h,:], k_t>)
 *             for every earlier token t < L_r (L_r counts the query itself)
 *   top-k     the k = 2048 highest logits of [0, L_r); ties go to the lower
 *             token index; fewer than k visible tokens -> all of them
 *   slots     physical slot = block_table[req][t / 64] * 64 + t % 64
 *   sparse    exact attention of each of the 96 query heads over only the
 *   MLA       selected tokens' 576-dim latents (512 latent + 64 RoPE dims);
 *             the latent itself is the value (absorbed MLA), so
 *             O[h] = sum_t softmax_t(S[h,t]) * kv[t, 0:512],
 *             S[h,t] = sm_scale * <q[h,:], kv[t,:]>.
 *
 * Every floating-point sum runs in double, in index order.  Cache entries are
 * decoded exactly from their stored bytes; the codec definitions are written
 * from the OCP 8-bit floating point spec (E4M3, "FN" variant: no infinities,
 * S.1111.111 is NaN) and the OCP Microscaling v1.0 spec (E2M1 elements, E8M0
 * scales with 0xFF = NaN, as the SM120 MXFP4 experiment log restates in its
 * "NaN/Inf decision record").
 *
 * Byte layouts of one 64-token page (the pages fix the per-token widths:
 * FP8 index key 132 B, MXFP4 index key 68 B, FP8 latent 576 B, NVFP4 latent
 * 352 B; the arrangement inside a page is this library's reading):
 *   index FP8   [64 x 128 B e4m3 codes][64 x fp32 scale]            8448 B
 *   index MXFP4 [64 x 64 B e2m1 pairs][64 x 4 B e8m0 (one per 32)]  4352 B
 *   latent FP8  [64 x 576 B e4m3], one per-tensor fp32 scale       36864 B
 *   latent NVFP4 [64 x 256 B e2m1 pairs][64 x 32 B e4m3 scale (one per 16)]
 *                [64 x 64 B e4m3 RoPE dims, per-tensor scale]       22528 B
 * Packed e2m1 pairs hold element 2j in the low nibble, 2j+1 in the high one.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>

/* tokens per indexer work item (a row is cut into such chunks for the threads) */
#define OR_CHUNK 4096
#endif

#define OR_OK 0
#define OR_ERR_ARG -1
#define OR_ERR_BOUNDS -6

#define OR_KEY_FP8 1
#define OR_KEY_MXFP4 2
#define OR_LATENT_FP8 3
#define OR_LATENT_NVFP4 4

#define OR_PAGE 64
#define OR_IDX_DIM 128
#define OR_IDX_HEADS 32
#define OR_LAT_DIM 576
#define OR_V_DIM 512

/* ---------------------------------------------------------------- codecs */

/* E4M3 (OCP FP8, "FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (m/8 * 2^-6); 0x7F / 0xFF are NaN. */
double oracle_e4m3_decode(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* E2M1 (OCP MX FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; no
 * specials.  Exponent 0 is subnormal: m * 0.5. */
double oracle_e2m1_decode(uint8_t nib) {
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* E8M0 (OCP MX shared scale): 2^(e-127); 0xFF is NaN. */
double oracle_e8m0_decode(uint8_t b) {
    if (b == 0xFF) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* bf16: the upper half of an IEEE binary32. */
double oracle_bf16_decode(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double rd_f32(const uint8_t *p) {
    float f;
    memcpy(&f, p, 4);
    return (double)f;
}

/* ------------------------------------------------------- cache addressing */

int64_t oracle_index_page_bytes(int fmt) {
    if (fmt == OR_KEY_FP8) return OR_PAGE * (OR_IDX_DIM + 4);
    if (fmt == OR_KEY_MXFP4) return OR_PAGE * (OR_IDX_DIM / 2 + OR_IDX_DIM / 32);
    return -1;
}

int64_t oracle_latent_page_bytes(int fmt) {
    if (fmt == OR_LATENT_FP8) return OR_PAGE * OR_LAT_DIM;
    if (fmt == OR_LATENT_NVFP4) return OR_PAGE * (OR_V_DIM / 2 + OR_V_DIM / 16 + (OR_LAT_DIM - OR_V_DIM));
    return -1;
}

/* Decode the index key of slot (page, j) into k[128] and its per-token scale.
 * FP8: k = e4m3 code values, scale = the stored fp32.
 * MXFP4: k = e2m1 * 2^(E-127) per 32-element block, scale = 1. */
static void decode_index_key(const uint8_t *pool, int fmt, int64_t page, int j, double *k, double *scale) {
    const uint8_t *pg = pool + page * oracle_index_page_bytes(fmt);
    if (fmt == OR_KEY_FP8) {
        const uint8_t *codes = pg + (int64_t)j * OR_IDX_DIM;
        for (int i = 0; i < OR_IDX_DIM; ++i) k[i] = oracle_e4m3_decode(codes[i]);
        *scale = rd_f32(pg + OR_PAGE * OR_IDX_DIM + 4 * j);
    } else {
        const uint8_t *pairs = pg + (int64_t)j * (OR_IDX_DIM / 2);
        const uint8_t *sc = pg + OR_PAGE * (OR_IDX_DIM / 2) + (int64_t)j * (OR_IDX_DIM / 32);
        for (int i = 0; i < OR_IDX_DIM; ++i) {
            uint8_t byte = pairs[i / 2];
            uint8_t nib = (i & 1) ? (byte >> 4) : (byte & 15);
            k[i] = oracle_e2m1_decode(nib) * oracle_e8m0_decode(sc[i / 32]);
        }
        *scale = 1.0;
    }
}

/* Decode the latent of a physical slot into kv[576] (exact, in double).
 * FP8: e4m3 * tensor_scale for all 576 dims.
 * NVFP4: dims 0..511 are e2m1 * (e4m3 scale of their 16-block); the 64 RoPE
 * dims are e4m3 * tensor_scale. */
static void decode_latent(const uint8_t *pool, int fmt, int64_t slot, double tensor_scale, double *kv) {
    int64_t page = slot / OR_PAGE;
    int j = (int)(slot % OR_PAGE);
    const uint8_t *pg = pool + page * oracle_latent_page_bytes(fmt);
    if (fmt == OR_LATENT_FP8) {
        const uint8_t *codes = pg + (int64_t)j * OR_LAT_DIM;
        for (int i = 0; i < OR_LAT_DIM; ++i) kv[i] = oracle_e4m3_decode(codes[i]) * tensor_scale;
    } else {
        const uint8_t *pairs = pg + (int64_t)j * (OR_V_DIM / 2);
        const uint8_t *sc = pg + OR_PAGE * (OR_V_DIM / 2) + (int64_t)j * (OR_V_DIM / 16);
        const uint8_t *rope = pg + OR_PAGE * (OR_V_DIM / 2 + OR_V_DIM / 16) + (int64_t)j * (OR_LAT_DIM - OR_V_DIM);
        for (int i = 0; i < OR_V_DIM; ++i) {
            uint8_t byte = pairs[i / 2];
            uint8_t nib = (i & 1) ? (byte >> 4) : (byte & 15);
            kv[i] = oracle_e2m1_decode(nib) * oracle_e4m3_decode(sc[i / 16]);
        }
        for (int i = OR_V_DIM; i < OR_LAT_DIM; ++i) kv[i] = oracle_e4m3_decode(rope[i - OR_V_DIM]) * tensor_scale;
    }
}

/* ---------------------------------------------------------------- indexer */

/* logits[r * stride + t] for t < row_ctx[r]; entries at t >= row_ctx[r] are
 * left untouched.  q_idx is [R, 32, 128] e4m3 (no query scale: the head
 * weights carry it), w is [R, 32] fp32.  Returns OR_ERR_BOUNDS if a block
 * table entry a row needs is outside [0, num_pages). */
int oracle_indexer_logits(const uint8_t *pool, int fmt, int64_t num_pages,
                          const int32_t *block_table, int64_t bt_stride,
                          const int32_t *row_req, const int32_t *row_ctx, int num_rows,
                          const uint8_t *q_idx, const float *w,
                          double *logits, int64_t stride) {
    if (oracle_index_page_bytes(fmt) < 0) return OR_ERR_ARG;
    int err = OR_OK;
    /* work items: (row, chunk of OR_CHUNK tokens); each logit is computed alone, in the same
     * order whatever the thread count */
    int max_ctx = 0;
    for (int r = 0; r < num_rows; ++r) max_ctx = row_ctx[r] > max_ctx ? row_ctx[r] : max_ctx;
    const int chunks = (max_ctx + OR_CHUNK - 1) / OR_CHUNK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < (int64_t)num_rows * chunks; ++item) {
        const int r = (int)(item / chunks), c = (int)(item % chunks);
        const int t0 = c * OR_CHUNK, t1 = row_ctx[r] < t0 + OR_CHUNK ? row_ctx[r] : t0 + OR_CHUNK;
        if (t0 >= t1) continue;
        double q[OR_IDX_HEADS][OR_IDX_DIM], k[OR_IDX_DIM], s;
        for (int h = 0; h < OR_IDX_HEADS; ++h)
            for (int i = 0; i < OR_IDX_DIM; ++i)
                q[h][i] = oracle_e4m3_decode(q_idx[((int64_t)r * OR_IDX_HEADS + h) * OR_IDX_DIM + i]);
        const int32_t *bt = block_table + (int64_t)row_req[r] * bt_stride;
        for (int t = t0; t < t1; ++t) {
            int64_t page = bt[t / OR_PAGE];
            if (page < 0 || page >= num_pages) {
#pragma omp atomic write
                err = OR_ERR_BOUNDS;
                continue;
            }
            decode_index_key(pool, fmt, page, t % OR_PAGE, k, &s);
            double logit = 0.0;
            for (int h = 0; h < OR_IDX_HEADS; ++h) {
                double dot = 0.0;
                for (int i = 0; i < OR_IDX_DIM; ++i) dot += q[h][i] * k[i];
                double a = s * dot;
                logit += (double)w[(int64_t)r * OR_IDX_HEADS + h] * (a > 0.0 ? a : 0.0);
            }
            logits[(int64_t)r * stride + t] = logit;
        }
    }
    return err;
}

/* ------------------------------------------------------------------ top-k */

typedef struct {
    double v;
    int32_t t;
} scored;

/* descending value, ascending index: the selection order the method uses */
static int cmp_scored(const void *a, const void *b) {
    const scored *x = (const scored *)a, *y = (const scored *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->t > y->t) - (x->t < y->t);
}

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* One row: select the first min(k, n) of (value desc, index asc), then
 * report them sorted by token index, padded with -1 up to k.  Signed zero
 * compares equal (the C comparison already does so). */
static void topk_row(const double *vals, int n, int k, int32_t *out) {
    scored *buf = (scored *)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    for (int t = 0; t < n; ++t) {
        buf[t].v = vals[t];
        buf[t].t = t;
    }
    qsort(buf, (size_t)n, sizeof(scored), cmp_scored);
    int m = n < k ? n : k;
    for (int i = 0; i < m; ++i) out[i] = buf[i].t;
    qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);
    for (int i = m; i < k; ++i) out[i] = -1;
    free(buf);
}

/* top-k over fp32 logits (the decision is taken in the precision the
 * logits are stored in). */
int oracle_topk_f32(const float *logits, int64_t stride, const int32_t *row_ctx, int num_rows, int k, int32_t *out) {
    if (k <= 0) return OR_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < num_rows; ++r) {
        int n = row_ctx[r];
        double *v = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        for (int t = 0; t < n; ++t) v[t] = (double)logits[(int64_t)r * stride + t];
        topk_row(v, n, k, out + (int64_t)r * k);
        free(v);
    }
    return OR_OK;
}

/* top-k over double logits (end-to-end oracle path). */
int oracle_topk_f64(const double *logits, int64_t stride, const int32_t *row_ctx, int num_rows, int k, int32_t *out) {
    if (k <= 0) return OR_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < num_rows; ++r)
        topk_row(logits + (int64_t)r * stride, row_ctx[r], k, out + (int64_t)r * k);
    return OR_OK;
}

/* ------------------------------------------------------------------ slots */

/* slot = block_table[req][t / 64] * 64 + t % 64; -1 stays -1. */
int oracle_page_to_slot(const int32_t *block_table, int64_t bt_stride, const int32_t *row_req, int num_rows,
                        const int32_t *idx, int k, int32_t *slots) {
    for (int r = 0; r < num_rows; ++r) {
        const int32_t *bt = block_table + (int64_t)row_req[r] * bt_stride;
        for (int i = 0; i < k; ++i) {
            int32_t t = idx[(int64_t)r * k + i];
            slots[(int64_t)r * k + i] = t < 0 ? -1 : bt[t / OR_PAGE] * OR_PAGE + t % OR_PAGE;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------- sparse MLA */

/* q is [R, H, 576] bf16 bits; slots is [R, k] physical slots, -1 = unused.
 * out is [R, H, 512], lse is [R, H] (natural log).  An empty selection gives
 * out = 0 and lse = -inf. */
int oracle_sparse_mla(const uint8_t *pool, int fmt, int64_t num_pages, double tensor_scale,
                      const uint16_t *q, int num_heads, const int32_t *slots, int num_rows, int k,
                      double sm_scale, double *out, double *lse) {
    if (oracle_latent_page_bytes(fmt) < 0 || num_heads <= 0) return OR_ERR_ARG;
    int err = OR_OK;
    /* first every row's selected latents, decoded (rows in parallel); then every (row, head)
     * alone, in the same order whatever the thread count */
    double **kvs = (double **)calloc((size_t)(num_rows > 0 ? num_rows : 1), sizeof(double *));
    int *ns = (int *)calloc((size_t)(num_rows > 0 ? num_rows : 1), sizeof(int));
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < num_rows; ++r) {
        const int32_t *sl = slots + (int64_t)r * k;
        int n = 0;
        for (int i = 0; i < k; ++i) n += sl[i] >= 0;
        double *kv = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * OR_LAT_DIM);
        int j = 0;
        for (int i = 0; i < k; ++i) {
            if (sl[i] < 0) continue;
            if ((int64_t)sl[i] >= num_pages * OR_PAGE) {
#pragma omp atomic write
                err = OR_ERR_BOUNDS;
                continue;
            }
            decode_latent(pool, fmt, sl[i], tensor_scale, kv + (int64_t)j * OR_LAT_DIM);
            ++j;
        }
        kvs[r] = kv;
        ns[r] = j;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t item = 0; item < (int64_t)num_rows * num_heads; ++item) {
        const int r = (int)(item / num_heads), h = (int)(item % num_heads);
        const int n = ns[r];
        const double *kv = kvs[r];
        double *sc = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        {
            double qh[OR_LAT_DIM];
            const uint16_t *qp = q + ((int64_t)r * num_heads + h) * OR_LAT_DIM;
            for (int i = 0; i < OR_LAT_DIM; ++i) qh[i] = oracle_bf16_decode(qp[i]);
            double *o = out + ((int64_t)r * num_heads + h) * OR_V_DIM;
            for (int d = 0; d < OR_V_DIM; ++d) o[d] = 0.0;
            if (n == 0) {
                if (lse) lse[(int64_t)r * num_heads + h] = -INFINITY;
                free(sc);
                continue;
            }
            double m = -INFINITY;
            for (int t = 0; t < n; ++t) {
                double s = 0.0;
                for (int i = 0; i < OR_LAT_DIM; ++i) s += qh[i] * kv[(int64_t)t * OR_LAT_DIM + i];
                sc[t] = sm_scale * s;
                if (sc[t] > m) m = sc[t];
            }
            double l = 0.0;
            for (int t = 0; t < n; ++t) {
                double p = exp(sc[t] - m);
                l += p;
                for (int d = 0; d < OR_V_DIM; ++d) o[d] += p * kv[(int64_t)t * OR_LAT_DIM + d];
            }
            for (int d = 0; d < OR_V_DIM; ++d) o[d] /= l;
            if (lse) lse[(int64_t)r * num_heads + h] = m + log(l);
        }
        free(sc);
    }
    for (int r = 0; r < num_rows; ++r) free(kvs[r]);
    free(kvs);
    free(ns);
    return err;
}

/* ---------------------------------------------------------------- encoders
 *
 * Quantisation of a new token before it is written into the caches (the
 * fused decode front end quantises the index key and writes the new token's
 * key and latent, vLLM blog "Day-0 support for Kimi K3.1 Pro", section
 * "Low-latency decode: fused DSA decode path").  Inputs are bf16; every
 * scale and quotient is computed in fp32 in the order written here, and the
 * rounding to a code is round-to-nearest-even from that fp32 value, so an
 * implementation that follows the same order reproduces the bytes exactly.
 */

/* fp32 -> e4m3 code, round to nearest even, saturating to +-448; NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(float xf) {
    double x = xf;
    if (x != x) return 0x7F;
    int s = signbit(x) ? 1 : 0;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)((s << 7) | 0x7E);
    if (a == 0.0) return (uint8_t)(s << 7);
    int e;
    frexp(a, &e);           /* a in [2^(e-1), 2^e) */
    int ue = e - 1;
    if (ue < -6) ue = -6;   /* below the normal range the quantum stays 2^-9 */
    double q = ldexp(1.0, ue - 3);
    double r = nearbyint(a / q) * q;
    if (r == 0.0) return (uint8_t)(s << 7);
    if (r > 448.0) r = 448.0;
    frexp(r, &e);
    ue = e - 1;
    uint8_t code;
    if (ue < -6) code = (uint8_t)nearbyint(r / ldexp(1.0, -9));              /* subnormal: m * 2^-9 */
    else code = (uint8_t)(((ue + 7) << 3) | (int)nearbyint((r / ldexp(1.0, ue) - 1.0) * 8.0));
    return (uint8_t)((s << 7) | code);
}

/* fp32 -> e2m1 nibble, round to nearest even, saturating to +-6. */
uint8_t oracle_e2m1_encode(float xf) {
    double x = xf;
    int s = signbit(x) ? 1 : 0;
    double a = fabs(x);
    if (a != a) a = 0.0;
    double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double r = nearbyint(a / q) * q;
    if (r > 6.0) r = 6.0;
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t code = 0;
    for (uint8_t c = 0; c < 8; ++c)
        if (mag[c] == r) code = c;
    return (uint8_t)((s << 3) | code);
}

static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Write n new tokens into the caches at physical slots[i] (-1: skipped).
 * keys: [n, 128] bf16; latents: [n, 576] bf16.
 *   FP8 key:     s = amax/448 (1 if amax = 0), code = e4m3(x / s), scale stored fp32
 *   MXFP4 key:   per 32 values E = floor(log2 amax) - 2 + 127 clamped to [0, 254]
 *                (E = 0 for an all-zero block), code = e2m1(x * 2^(127 - E))
 *   FP8 latent:  code = e4m3(x / tensor_scale)
 *   NVFP4 latent: per 16 values scale code = e4m3(amax / 6), code = e2m1(x / scale)
 *                (all codes 0 when the scale is 0); RoPE dims e4m3(x / tensor_scale). */
int oracle_cache_insert(uint8_t *idx_pool, int key_fmt, uint8_t *lat_pool, int lat_fmt, float tensor_scale,
                        int64_t num_pages, const int32_t *slots, int n, const uint16_t *keys,
                        const uint16_t *latents) {
    if (oracle_index_page_bytes(key_fmt) < 0 || oracle_latent_page_bytes(lat_fmt) < 0) return OR_ERR_ARG;
    int err = OR_OK;
    for (int i = 0; i < n; ++i) {
        int32_t slot = slots[i];
        if (slot < 0) continue;
        if ((int64_t)slot >= num_pages * OR_PAGE) {
            err = OR_ERR_BOUNDS;
            continue;
        }
        int64_t page = slot / OR_PAGE;
        int j = slot % OR_PAGE;
        const uint16_t *k = keys + (int64_t)i * OR_IDX_DIM;
        uint8_t *ip = idx_pool + page * oracle_index_page_bytes(key_fmt);
        if (key_fmt == OR_KEY_FP8) {
            float amax = 0.0f;
            for (int d = 0; d < OR_IDX_DIM; ++d) amax = fmaxf(amax, fabsf(bf16_to_f32(k[d])));
            float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            for (int d = 0; d < OR_IDX_DIM; ++d) ip[(int64_t)j * OR_IDX_DIM + d] = oracle_e4m3_encode(bf16_to_f32(k[d]) / sc);
            memcpy(ip + OR_PAGE * OR_IDX_DIM + 4 * j, &sc, 4);
        } else {
            uint8_t *codes = ip + (int64_t)j * (OR_IDX_DIM / 2);
            uint8_t *es = ip + OR_PAGE * (OR_IDX_DIM / 2) + (int64_t)j * (OR_IDX_DIM / 32);
            for (int b = 0; b < OR_IDX_DIM / 32; ++b) {
                float amax = 0.0f;
                for (int d = 0; d < 32; ++d) amax = fmaxf(amax, fabsf(bf16_to_f32(k[32 * b + d])));
                int E = 0;
                if (amax > 0.0f) {
                    int e;
                    frexpf(amax, &e);
                    E = (e - 1) - 2 + 127;
                    if (E < 0) E = 0;
                    if (E > 254) E = 254;
                }
                es[b] = (uint8_t)E;
                for (int d = 0; d < 32; d += 2) {
                    uint8_t lo = oracle_e2m1_encode(ldexpf(bf16_to_f32(k[32 * b + d]), 127 - E));
                    uint8_t hi = oracle_e2m1_encode(ldexpf(bf16_to_f32(k[32 * b + d + 1]), 127 - E));
                    codes[(32 * b + d) / 2] = (uint8_t)(lo | (hi << 4));
                }
            }
        }
        const uint16_t *x = latents + (int64_t)i * OR_LAT_DIM;
        uint8_t *lp = lat_pool + page * oracle_latent_page_bytes(lat_fmt);
        if (lat_fmt == OR_LATENT_FP8) {
            for (int d = 0; d < OR_LAT_DIM; ++d)
                lp[(int64_t)j * OR_LAT_DIM + d] = oracle_e4m3_encode(bf16_to_f32(x[d]) / tensor_scale);
        } else {
            uint8_t *codes = lp + (int64_t)j * (OR_V_DIM / 2);
            uint8_t *scs = lp + OR_PAGE * (OR_V_DIM / 2) + (int64_t)j * (OR_V_DIM / 16);
            uint8_t *rope = lp + OR_PAGE * (OR_V_DIM / 2 + OR_V_DIM / 16) + (int64_t)j * (OR_LAT_DIM - OR_V_DIM);
            for (int b = 0; b < OR_V_DIM / 16; ++b) {
                float amax = 0.0f;
                for (int d = 0; d < 16; ++d) amax = fmaxf(amax, fabsf(bf16_to_f32(x[16 * b + d])));
                uint8_t scode = oracle_e4m3_encode(amax / 6.0f);
                float sc = (float)oracle_e4m3_decode(scode);
                scs[b] = scode;
                for (int d = 0; d < 16; d += 2) {
                    uint8_t lo = sc > 0.0f ? oracle_e2m1_encode(bf16_to_f32(x[16 * b + d]) / sc) : 0;
                    uint8_t hi = sc > 0.0f ? oracle_e2m1_encode(bf16_to_f32(x[16 * b + d + 1]) / sc) : 0;
                    codes[(16 * b + d) / 2] = (uint8_t)(lo | (hi << 4));
                }
            }
            for (int d = 0; d < OR_LAT_DIM - OR_V_DIM; ++d)
                rope[d] = oracle_e4m3_encode(bf16_to_f32(x[OR_V_DIM + d]) / tensor_scale);
        }
    }
    return err;
}

/* ------------------------------------------------- MSA (block-sparse variant)
 *
 * MiniMax sparse attention (vLLM blog "Day-0 support for MiniMax-M3.1-Flash",
 * section "MSA primer", and its Fig. 1): the cache is cut into 128-token
 * blocks; one index query per GQA group scores every visible key against the
 * one index-key head all groups share; the scores are max-pooled to one score
 * per block; each group's query heads then attend, exactly, to that group's
 * selected blocks only: the most recent block always, plus the best of the
 * others, at most 2,048 keys (16 blocks) in all.
 *
 *   score      s[r,g,t] = <qi[r,g,:], ki_t>                          t < L_r
 *   block      S[r,g,b] = max of s[r,g,t] over t in [128b, 128b + 128), t < L_r
 *              (a NaN score never wins; a block of NaNs scores -inf)
 *   select     nb = ceil(L_r / 128).  nb <= 16: every block.  Otherwise block
 *              nb - 1 and the 15 highest S among blocks 0 .. nb - 2, ties to
 *              the lower block.  Listed ascending, -1 padded to 16.
 *   attention  O[r,h,:] = sum_t softmax_t(sm_scale * <q[r,h,:], K_g,t>) V_g,t
 *              over t < L_r in the selected blocks of group g = h / (H / 4);
 *              the query stays in FP8 (section "Blackwell-optimised MSA
 *              kernels"): e4m3 codes times one per-tensor fp32 scale
 *
 * Byte layouts of one 128-token MSA page (the block is the page; the index
 * key is 128 B/token and K/V are 4 KV heads x 128 dims in FP8, 1,024 B/token,
 * as the page states; the arrangement inside a page is this library's reading):
 *   index  [128 x 128 B e4m3]                                          16384 B
 *   kv     [4 heads] x ([K: 128 x 128 B e4m3] [V: 128 x 128 B e4m3])  131072 B
 * K and V codes are scaled by one per-tensor fp32 factor each (k_scale,
 * v_scale); the index key has no scale (a positive factor would not change
 * the selection).
 */
#define OR_MSA_PAGE 128
#define OR_MSA_DIM 128
#define OR_MSA_GROUPS 4
#define OR_MSA_BLOCKS 16

int64_t oracle_msa_index_page_bytes(void) { return (int64_t)OR_MSA_PAGE * OR_MSA_DIM; }

int64_t oracle_msa_kv_page_bytes(void) { return (int64_t)OR_MSA_GROUPS * 2 * OR_MSA_PAGE * OR_MSA_DIM; }

static int msa_num_blocks(int L) { return L > 0 ? (L + OR_MSA_PAGE - 1) / OR_MSA_PAGE : 0; }

/* scores[(r * 4 + g) * stride + b] for b < ceil(L_r / 128); q_idx is
 * [R, 4, 128] e4m3.  Returns OR_ERR_BOUNDS for a page id outside the pool. */
int oracle_msa_block_scores(const uint8_t *idx_pool, int64_t num_pages, const int32_t *block_table,
                            int64_t bt_stride, const int32_t *row_req, const int32_t *row_ctx, int num_rows,
                            const uint8_t *q_idx, double *scores, int64_t stride) {
    int err = OR_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < num_rows; ++r) {
        double q[OR_MSA_GROUPS][OR_MSA_DIM];
        for (int g = 0; g < OR_MSA_GROUPS; ++g)
            for (int i = 0; i < OR_MSA_DIM; ++i)
                q[g][i] = oracle_e4m3_decode(q_idx[((int64_t)r * OR_MSA_GROUPS + g) * OR_MSA_DIM + i]);
        const int32_t *bt = block_table + (int64_t)row_req[r] * bt_stride;
        const int L = row_ctx[r];
        for (int b = 0; b < msa_num_blocks(L); ++b) {
            double best[OR_MSA_GROUPS];
            for (int g = 0; g < OR_MSA_GROUPS; ++g) best[g] = -INFINITY;
            const int64_t page = bt[b];
            if (page < 0 || page >= num_pages) {
#pragma omp atomic write
                err = OR_ERR_BOUNDS;
            } else {
                for (int t = b * OR_MSA_PAGE; t < L && t < (b + 1) * OR_MSA_PAGE; ++t) {
                    const uint8_t *key = idx_pool + page * oracle_msa_index_page_bytes() +
                                         (int64_t)(t % OR_MSA_PAGE) * OR_MSA_DIM;
                    for (int g = 0; g < OR_MSA_GROUPS; ++g) {
                        double dot = 0.0;
                        for (int i = 0; i < OR_MSA_DIM; ++i) dot += q[g][i] * oracle_e4m3_decode(key[i]);
                        if (dot > best[g]) best[g] = dot;
                    }
                }
            }
            for (int g = 0; g < OR_MSA_GROUPS; ++g) scores[((int64_t)r * OR_MSA_GROUPS + g) * stride + b] = best[g];
        }
    }
    return err;
}

/* One (row, group): choose the blocks as the header states. */
static void msa_select_one(const double *S, int nb, int32_t *out) {
    int m = 0;
    if (nb <= OR_MSA_BLOCKS) {
        for (int b = 0; b < nb; ++b) out[m++] = b;
    } else {
        scored *buf = (scored *)malloc(sizeof(scored) * (size_t)(nb - 1));
        for (int b = 0; b < nb - 1; ++b) {
            buf[b].v = S[b] != S[b] ? -INFINITY : S[b];
            buf[b].t = b;
        }
        qsort(buf, (size_t)(nb - 1), sizeof(scored), cmp_scored);
        for (int i = 0; i < OR_MSA_BLOCKS - 1; ++i) out[m++] = buf[i].t;
        out[m++] = nb - 1;
        free(buf);
        qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);
    }
    for (int i = m; i < OR_MSA_BLOCKS; ++i) out[i] = -1;
}

/* blocks[(r * 4 + g) * 16 + i] from double block scores (end-to-end path). */
int oracle_msa_select_f64(const double *scores, int64_t stride, const int32_t *row_ctx, int num_rows,
                          int32_t *blocks) {
    for (int r = 0; r < num_rows; ++r)
        for (int g = 0; g < OR_MSA_GROUPS; ++g)
            msa_select_one(scores + ((int64_t)r * OR_MSA_GROUPS + g) * stride, msa_num_blocks(row_ctx[r]),
                           blocks + ((int64_t)r * OR_MSA_GROUPS + g) * OR_MSA_BLOCKS);
    return OR_OK;
}

/* The same decision over fp32 block scores (the precision they are stored in). */
int oracle_msa_select_f32(const float *scores, int64_t stride, const int32_t *row_ctx, int num_rows,
                          int32_t *blocks) {
    for (int r = 0; r < num_rows; ++r) {
        const int nb = msa_num_blocks(row_ctx[r]);
        double *S = (double *)malloc(sizeof(double) * (size_t)(nb > 0 ? nb : 1));
        for (int g = 0; g < OR_MSA_GROUPS; ++g) {
            for (int b = 0; b < nb; ++b) S[b] = (double)scores[((int64_t)r * OR_MSA_GROUPS + g) * stride + b];
            msa_select_one(S, nb, blocks + ((int64_t)r * OR_MSA_GROUPS + g) * OR_MSA_BLOCKS);
        }
        free(S);
    }
    return OR_OK;
}

/* q: [R, 4 * hpg, 128] e4m3 codes (times q_scale); blocks: [R, 4, 16] logical block ids (-1
 * unused).  out: [R, 4 * hpg, 128], lse: [R, 4 * hpg] (natural log).  A head
 * with no visible selected token gets out = 0, lse = -inf.  A block id at or
 * past ceil(L_r / 128), or a page id outside the pool, is OR_ERR_BOUNDS. */
int oracle_msa_attention(const uint8_t *kv_pool, int64_t num_pages, double k_scale, double v_scale,
                         const int32_t *block_table, int64_t bt_stride, const int32_t *row_req,
                         const int32_t *row_ctx, int num_rows, const uint8_t *q, double q_scale, int heads_per_group,
                         const int32_t *blocks, double sm_scale, double *out, double *lse) {
    if (heads_per_group <= 0) return OR_ERR_ARG;
    const int H = OR_MSA_GROUPS * heads_per_group;
    const int64_t head_bytes = 2 * OR_MSA_PAGE * OR_MSA_DIM;
    int err = OR_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < num_rows; ++r) {
        const int32_t *bt = block_table + (int64_t)row_req[r] * bt_stride;
        const int L = row_ctx[r];
        double *K = (double *)malloc(sizeof(double) * OR_MSA_BLOCKS * OR_MSA_PAGE * OR_MSA_DIM);
        double *V = (double *)malloc(sizeof(double) * OR_MSA_BLOCKS * OR_MSA_PAGE * OR_MSA_DIM);
        double *sc = (double *)malloc(sizeof(double) * OR_MSA_BLOCKS * OR_MSA_PAGE);
        for (int g = 0; g < OR_MSA_GROUPS; ++g) {
            const int32_t *bl = blocks + ((int64_t)r * OR_MSA_GROUPS + g) * OR_MSA_BLOCKS;
            int n = 0;  /* gather the group's visible tokens, decoded */
            for (int i = 0; i < OR_MSA_BLOCKS; ++i) {
                const int b = bl[i];
                if (b < 0) continue;
                if (b >= msa_num_blocks(L) || bt[b] < 0 || bt[b] >= num_pages) {
#pragma omp atomic write
                    err = OR_ERR_BOUNDS;
                    continue;
                }
                const uint8_t *kp = kv_pool + (int64_t)bt[b] * oracle_msa_kv_page_bytes() + g * head_bytes;
                const uint8_t *vp = kp + OR_MSA_PAGE * OR_MSA_DIM;
                for (int t = b * OR_MSA_PAGE; t < L && t < (b + 1) * OR_MSA_PAGE; ++t, ++n) {
                    const int j = t % OR_MSA_PAGE;
                    for (int d = 0; d < OR_MSA_DIM; ++d) {
                        K[(int64_t)n * OR_MSA_DIM + d] = oracle_e4m3_decode(kp[j * OR_MSA_DIM + d]) * k_scale;
                        V[(int64_t)n * OR_MSA_DIM + d] = oracle_e4m3_decode(vp[j * OR_MSA_DIM + d]) * v_scale;
                    }
                }
            }
            for (int hh = 0; hh < heads_per_group; ++hh) {
                const int h = g * heads_per_group + hh;
                double qh[OR_MSA_DIM];
                for (int d = 0; d < OR_MSA_DIM; ++d) qh[d] = oracle_e4m3_decode(q[((int64_t)r * H + h) * OR_MSA_DIM + d]) * q_scale;
                double *o = out + ((int64_t)r * H + h) * OR_MSA_DIM;
                for (int d = 0; d < OR_MSA_DIM; ++d) o[d] = 0.0;
                if (n == 0) {
                    lse[(int64_t)r * H + h] = -INFINITY;
                    continue;
                }
                double m = -INFINITY;
                for (int t = 0; t < n; ++t) {
                    double s = 0.0;
                    for (int d = 0; d < OR_MSA_DIM; ++d) s += qh[d] * K[(int64_t)t * OR_MSA_DIM + d];
                    sc[t] = s * sm_scale;
                    if (sc[t] > m) m = sc[t];
                }
                double l = 0.0;
                for (int t = 0; t < n; ++t) {
                    const double p = exp(sc[t] - m);
                    l += p;
                    for (int d = 0; d < OR_MSA_DIM; ++d) o[d] += p * V[(int64_t)t * OR_MSA_DIM + d];
                }
                for (int d = 0; d < OR_MSA_DIM; ++d) o[d] = o[d] / l;
                lse[(int64_t)r * H + h] = m + log(l);
            }
        }
        free(K);
        free(V);
        free(sc);
    }
    return err;
}

/* ------------------------------------------------------------------- misc */

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
