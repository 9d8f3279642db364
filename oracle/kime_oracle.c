/*
 * kime_oracle.c -- plain FP64 CPU oracle for packed variable-length attention
 * with RoPE applied to q and k, the in-place KV-cache append, single-token
 * decode and chunked prefill against the cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header, table generator or constant with the CUDA library: every
 * line below is written from the definitions on the source pages.
 *
 * Sources (docs.rs pages):
 *   [kime-cpu]   kime-cpu 0.0.17, src/kime_cpu/plan.rs
 *                  - Step::Rope: positions are token row minus the start of
 *                    its sequence; q then k heads of a fused qkv row rotate.
 *                  - Step::Attention: one task per (sequence, query block,
 *                    head) over rows cu[s]..cu[s+1].
 *   [kime-cuda]  kime-cuda 0.0.3, src/plan.rs
 *                  - fn rope_tables: cos/sin tables [len, 32] for heads of 64.
 *                  - Op::Attention lowering: window None is encoded as -1;
 *                    qkv width is 3*heads*64 for multi-head attention.
 *   [argus]      ffai-argus 0.7.3, src/text.rs
 *                  - CausalSoftmax: row i sees keys 0..=i+offset; the tail is
 *                    exactly zero; decode is offset = k_len-1.
 *                  - module doc, "Why deleting the mask is BIT-IDENTICAL":
 *                    skipping a masked column gives the same floats as
 *                    writing -inf and running softmax.
 *                  - Block::q doc: the 1/8 scale fold is exact.
 *                  - TextTower::block, GQA fold: q head h uses kv head
 *                    h / (heads/kv_heads).
 *                  - KvAppend: write rows at pos, checking pos+seq <= cap
 *                    before anything is written.
 *                  - TextTower::block, KV cache: a block of seq new tokens at
 *                    index_pos is written into the preallocated cache, then
 *                    attends cache rows 0..index_pos+seq with CausalSoftmax
 *                    offset index_pos (chunked prefill; decode is seq = 1).
 *
 * Everything is computed in double precision.  Inputs are widened exactly
 * (float64, float32, or bfloat16 bit patterns).  The one place the oracle
 * does not compute in double is the KV append, whose output is a bfloat16
 * code: there the rotation is evaluated in float32 with one rounding per
 * operation (no fused multiply-add; build with -ffp-contract=off) and then
 * rounded to bfloat16 to nearest-even, the precision the kernel takes that
 * decision in.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define HEAD 64
#define HALF 32

enum { DT_F64 = 0, DT_F32 = 1, DT_BF16 = 2 };

/* ---- element access ---------------------------------------------------- */

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double load_elem(const void *base, int dtype, size_t idx) {
    switch (dtype) {
    case DT_F64: return ((const double *)base)[idx];
    case DT_F32: return (double)((const float *)base)[idx];
    default: return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    }
}

/* float32 -> bfloat16 bit pattern, round to nearest, ties to even.  NaN stays
 * a (quiet) NaN. */
uint16_t kime_oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ---- RoPE tables ([kime-cuda] fn rope_tables) ---------------------------- */

/* The tables both kime backends use: inverse frequency inv_i, for i < 32, is
 * the float32 reciprocal of theta^(2i/64) where the exponent 2i/64 is a float32
 * quotient and the power is taken in double then narrowed to float32.  The
 * angle at position p is the float32 product (float)p * inv_i; its cosine and
 * sine are taken in double and narrowed to float32. */
void kime_oracle_rope_tables_f32(double theta, int len, float *cos_out, float *sin_out) {
    float inv[HALF];
    for (int i = 0; i < HALF; i++) {
        float e = (float)(2 * i) / (float)HEAD;
        float pw = (float)pow(theta, (double)e);
        inv[i] = 1.0f / pw;
    }
    for (int p = 0; p < len; p++) {
        for (int i = 0; i < HALF; i++) {
            float a32 = (float)p * inv[i];
            double a = (double)a32;
            cos_out[(size_t)p * HALF + i] = (float)cos(a);
            sin_out[(size_t)p * HALF + i] = (float)sin(a);
        }
    }
}

/* Exact-angle tables in double: angle p * theta^(-2i/64), no float32 steps.
 * Used by the RoPE invariants (norm preservation, relative position). */
void kime_oracle_rope_tables_f64(double theta, int len, double *cos_out, double *sin_out) {
    for (int p = 0; p < len; p++) {
        for (int i = 0; i < HALF; i++) {
            double a = (double)p * pow(theta, -(double)(2 * i) / (double)HEAD);
            cos_out[(size_t)p * HALF + i] = cos(a);
            sin_out[(size_t)p * HALF + i] = sin(a);
        }
    }
}

/* Rotate-half RoPE of one 64-wide head at table row (c, s): element t pairs
 * with t+32.  y[t] = x[t] c_t - x[t+32] s_t ; y[t+32] = x[t+32] c_t + x[t] s_t.
 * (candle's non-interleaved rope, which ffai-argus TextTower::rope calls; the
 * kime Rope::apply body is not on the pages.) */
void kime_oracle_rope(const double *x, const double *c, const double *s, double *y) {
    for (int t = 0; t < HALF; t++) {
        double a = x[t], b = x[t + HALF];
        y[t] = a * c[t] - b * s[t];
        y[t + HALF] = b * c[t] + a * s[t];
    }
}

/* ---- attention over a packed batch ------------------------------------- */

typedef struct {
    const void *qkv;
    int dtype;
    const int32_t *cu;
    int n_seqs, heads, kv_heads, window, causal;
    double scale;
    const double *cos, *sin;
    int rope_len;
} varlen_args;

/* Is key j visible from query i of a length-L sequence?  Causal: j <= i
 * ([argus] CausalSoftmax with offset 0).  Window w >= 0: |i - j| <= w
 * (window -1 means none, [kime-cuda] Op::Attention).  Both: the intersection. */
static int allowed(int i, int j, int L, int causal, int window) {
    if (j < 0 || j >= L) return 0;
    if (causal && j > i) return 0;
    if (window >= 0) {
        int d = i > j ? i - j : j - i;
        if (d > window) return 0;
    }
    return 1;
}

/* The sequence owning token row r: the largest s < n_seqs with cu[s] <= r.
 * Maximality gives cu[s+1] > r, so empty sequences are stepped over. */
static int seq_of_row(const int32_t *cu, int n_seqs, int r) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static void load_head(const varlen_args *a, int row, int col0, double *x) {
    size_t W = (size_t)HEAD * (a->heads + 2 * a->kv_heads);
    for (int t = 0; t < HEAD; t++) x[t] = load_elem(a->qkv, a->dtype, (size_t)row * W + col0 + t);
}

/* One query: output row (r, h).  mode 0 visits only the allowed keys; mode 1
 * materialises the full length-L score row with -inf at masked keys and runs
 * softmax over all of it (the form the skip is claimed to equal bit for bit).
 * If probs is non-null it receives the L probabilities (masked ones 0). */
static void one_query(const varlen_args *a, int r, int h, int mode, double *out, double *probs) {
    int s = seq_of_row(a->cu, a->n_seqs, r);
    int start = a->cu[s], L = a->cu[s + 1] - start, i = r - start;
    int G = a->heads / a->kv_heads, g = h / G;
    int kcol = (a->heads + g) * HEAD, vcol = (a->heads + a->kv_heads + g) * HEAD;
    double xq[HEAD], yq[HEAD], xk[HEAD], yk[HEAD], xv[HEAD];
    load_head(a, r, h * HEAD, xq);
    kime_oracle_rope(xq, a->cos + (size_t)i * HALF, a->sin + (size_t)i * HALF, yq);

    double *sc = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double m = -INFINITY;
    for (int j = 0; j < L; j++) {
        int ok = allowed(i, j, L, a->causal, a->window);
        if (!ok) {
            sc[j] = -INFINITY;
            continue;
        }
        load_head(a, start + j, kcol, xk);
        kime_oracle_rope(xk, a->cos + (size_t)j * HALF, a->sin + (size_t)j * HALF, yk);
        double d = 0.0;
        for (int t = 0; t < HEAD; t++) d += yq[t] * yk[t];
        sc[j] = a->scale * d;
    }
    for (int j = 0; j < L; j++) {
        if (mode == 0 && !allowed(i, j, L, a->causal, a->window)) continue;
        if (sc[j] > m) m = sc[j];
    }
    double den = 0.0, num[HEAD];
    for (int t = 0; t < HEAD; t++) num[t] = 0.0;
    for (int j = 0; j < L; j++) {
        int ok = allowed(i, j, L, a->causal, a->window);
        if (mode == 0 && !ok) {
            if (probs) probs[j] = 0.0;
            continue;
        }
        double p = exp(sc[j] - m); /* exp(-inf) = 0 for masked keys in mode 1 */
        den += p;
        load_head(a, start + j, vcol, xv);
        for (int t = 0; t < HEAD; t++) num[t] += p * xv[t];
        if (probs) probs[j] = p;
    }
    if (probs)
        for (int j = 0; j < L; j++) probs[j] /= den;
    for (int t = 0; t < HEAD; t++) out[t] = num[t] / den;
    free(sc);
}

typedef struct {
    const varlen_args *a;
    const int32_t *rows, *row_heads;
    long n_items;
    int mode, tid, nthreads;
    double *out;
} varlen_job;

static void *varlen_worker(void *p) {
    varlen_job *job = (varlen_job *)p;
    const varlen_args *a = job->a;
    for (long k = job->tid; k < job->n_items; k += job->nthreads) {
        int r, h;
        if (job->rows) {
            r = job->rows[k];
            h = job->row_heads[k];
        } else {
            r = (int)(k / a->heads);
            h = (int)(k % a->heads);
        }
        one_query(a, r, h, job->mode, job->out + (size_t)k * HEAD, NULL);
    }
    return NULL;
}

static int check_varlen(const varlen_args *a) {
    if (a->n_seqs < 0 || a->heads <= 0 || a->kv_heads <= 0 || a->heads % a->kv_heads) return -1;
    if (a->window < -1) return -1;
    if (a->n_seqs > 0 && a->cu[0] != 0) return -2;
    for (int s = 0; s < a->n_seqs; s++) {
        if (a->cu[s + 1] < a->cu[s]) return -2;
        if (a->cu[s + 1] - a->cu[s] > a->rope_len) return -2;
    }
    return 0;
}

/* Attention outputs for n_items (token row, head) pairs, or for every row and
 * head when rows is NULL (then out is [T, heads*64]).  Item k is written at
 * out + 64k.  qkv is [T, 64*(heads+2*kv_heads)] in dtype; tables are [>=maxL,
 * 32].  Returns 0, or a negative code for malformed arguments. */
int kime_oracle_attn_varlen(const void *qkv, int dtype, const int32_t *cu, int n_seqs, int heads,
                            int kv_heads, int window, int causal, double scale, const double *cos_t,
                            const double *sin_t, int rope_len, const int32_t *rows,
                            const int32_t *row_heads, long n_items, double *out, int mode,
                            int nthreads) {
    varlen_args a = {qkv, dtype, cu, n_seqs, heads, kv_heads, window, causal, scale, cos_t, sin_t, rope_len};
    int rc = check_varlen(&a);
    if (rc) return rc;
    if (n_seqs == 0) return 0;
    if (!rows) n_items = (long)cu[n_seqs] * heads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    varlen_job jobs[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (varlen_job){&a, rows, row_heads, n_items, mode, t, nthreads, out};
        if (nthreads == 1) varlen_worker(&jobs[t]);
        else pthread_create(&th[t], NULL, varlen_worker, &jobs[t]);
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
    return 0;
}

/* The probability row of query (r, h): probs[j] for j in [0, L) of r's
 * sequence, exactly 0 where key j is masked. */
int kime_oracle_attn_probs(const void *qkv, int dtype, const int32_t *cu, int n_seqs, int heads,
                           int kv_heads, int window, int causal, double scale, const double *cos_t,
                           const double *sin_t, int rope_len, int r, int h, double *probs, int mode) {
    varlen_args a = {qkv, dtype, cu, n_seqs, heads, kv_heads, window, causal, scale, cos_t, sin_t, rope_len};
    int rc = check_varlen(&a);
    if (rc) return rc;
    double out[HEAD];
    one_query(&a, r, h, mode, out, probs);
    return 0;
}

/* ---- KV cache append ([argus] KvAppend) --------------------------------- */

/* For each sequence s, writes the new token's k heads, rotated at position
 * pos[s], and its v heads into row pos[s] of caches laid out
 * [n_seqs, kv_heads, cap, 64] (bfloat16 bit patterns).  qkv_new is
 * [n_seqs, 64*(heads+2*kv_heads)] bfloat16 bits.  The rotation runs in float32
 * with one rounding per multiply and per add, then rounds to bfloat16.  A
 * sequence whose pos is outside [0, min(cap, rope_len)) is not written; the
 * return value counts those. */
int kime_oracle_kv_append(const uint16_t *qkv_new, const int32_t *pos, int n_seqs, int heads,
                          int kv_heads, int cap, const float *cos_t, const float *sin_t,
                          int rope_len, uint16_t *k_cache, uint16_t *v_cache) {
    size_t W = (size_t)HEAD * (heads + 2 * kv_heads);
    int bad = 0;
    for (int s = 0; s < n_seqs; s++) {
        int P = pos[s];
        if (P < 0 || P >= cap || P >= rope_len) {
            bad++;
            continue;
        }
        const float *c = cos_t + (size_t)P * HALF, *sn = sin_t + (size_t)P * HALF;
        for (int g = 0; g < kv_heads; g++) {
            const uint16_t *xk = qkv_new + (size_t)s * W + (size_t)(heads + g) * HEAD;
            const uint16_t *xv = qkv_new + (size_t)s * W + (size_t)(heads + kv_heads + g) * HEAD;
            size_t dst = (((size_t)s * kv_heads + g) * cap + P) * HEAD;
            for (int t = 0; t < HALF; t++) {
                float a = (float)bf16_bits_to_double(xk[t]);
                float b = (float)bf16_bits_to_double(xk[t + HALF]);
                float ac = a * c[t], bs = b * sn[t], bc = b * c[t], as = a * sn[t];
                float y0 = ac - bs, y1 = bc + as;
                k_cache[dst + t] = kime_oracle_f32_to_bf16(y0);
                k_cache[dst + t + HALF] = kime_oracle_f32_to_bf16(y1);
            }
            for (int t = 0; t < HEAD; t++) v_cache[dst + t] = xv[t];
        }
    }
    return bad;
}

/* ---- single-token decode ------------------------------------------------ */

typedef struct {
    const uint16_t *qkv_new;
    const int32_t *pos;
    int n_seqs, heads, kv_heads, cap;
    double scale;
    const double *cos, *sin;
    int rope_len;
    const uint16_t *k_cache, *v_cache;
    const int32_t *items;
    long n_items;
    double *out;
    int tid, nthreads;
} decode_job;

/* Query of sequence s, head h: the new row's q head rotated at P = pos[s]
 * attends to cache rows 0..=P of kv head h/(heads/kv_heads) (row P being the
 * appended token): CausalSoftmax with q_len 1 and offset k_len-1. */
static void decode_one(const decode_job *d, int s, int h, double *out) {
    int P = d->pos[s];
    int G = d->heads / d->kv_heads, g = h / G;
    size_t W = (size_t)HEAD * (d->heads + 2 * d->kv_heads);
    double xq[HEAD], yq[HEAD];
    for (int t = 0; t < HEAD; t++) xq[t] = bf16_bits_to_double(d->qkv_new[(size_t)s * W + (size_t)h * HEAD + t]);
    kime_oracle_rope(xq, d->cos + (size_t)P * HALF, d->sin + (size_t)P * HALF, yq);
    const uint16_t *K = d->k_cache + ((size_t)s * d->kv_heads + g) * d->cap * HEAD;
    const uint16_t *V = d->v_cache + ((size_t)s * d->kv_heads + g) * d->cap * HEAD;
    int n = P + 1;
    double *sc = (double *)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; j++) {
        double dot = 0.0;
        for (int t = 0; t < HEAD; t++) dot += yq[t] * bf16_bits_to_double(K[(size_t)j * HEAD + t]);
        sc[j] = d->scale * dot;
        if (sc[j] > m) m = sc[j];
    }
    double den = 0.0, num[HEAD];
    for (int t = 0; t < HEAD; t++) num[t] = 0.0;
    for (int j = 0; j < n; j++) {
        double p = exp(sc[j] - m);
        den += p;
        for (int t = 0; t < HEAD; t++) num[t] += p * bf16_bits_to_double(V[(size_t)j * HEAD + t]);
    }
    for (int t = 0; t < HEAD; t++) out[t] = num[t] / den;
    free(sc);
}

static void *decode_worker(void *p) {
    decode_job *d = (decode_job *)p;
    for (long k = d->tid; k < d->n_items; k += d->nthreads) {
        long it = d->items ? d->items[k] : k;
        int s = (int)(it / d->heads), h = (int)(it % d->heads);
        decode_one(d, s, h, d->out + (size_t)k * HEAD);
    }
    return NULL;
}

/* Decode outputs for n_items items (item = s*heads + h), or all n_seqs*heads
 * when items is NULL (then out is [n_seqs, heads*64]).  Caches must already
 * hold the appended row at pos[s].  Returns 0 or a negative code. */
int kime_oracle_attn_decode(const uint16_t *qkv_new, const int32_t *pos, int n_seqs, int heads,
                            int kv_heads, int cap, double scale, const double *cos_t,
                            const double *sin_t, int rope_len, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *items, long n_items,
                            double *out, int nthreads) {
    if (heads <= 0 || kv_heads <= 0 || heads % kv_heads || n_seqs < 0) return -1;
    for (int s = 0; s < n_seqs; s++)
        if (pos[s] < 0 || pos[s] >= cap || pos[s] >= rope_len) return -2;
    if (!items) n_items = (long)n_seqs * heads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    decode_job jobs[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (decode_job){qkv_new, pos, n_seqs, heads, kv_heads, cap, scale, cos_t, sin_t, rope_len,
                               k_cache, v_cache, items, n_items, out, t, nthreads};
        if (nthreads == 1) decode_worker(&jobs[t]);
        else pthread_create(&th[t], NULL, decode_worker, &jobs[t]);
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
    return 0;
}

/* ---- chunked prefill against the cache ([argus] TextTower::block) -------- */

/* Multi-token append: sequence s owns rows cu[s]..cu[s+1]-1 of qkv
 * [T, 64*(heads+2*kv_heads)] (bfloat16 bits); its row i is the token at
 * position pos[s] + i, whose k heads (rotated there) and v heads go to cache
 * row pos[s] + i.  [argus] KvAppend refuses a block with pos + seq > cap before
 * writing anything: a sequence with pos[s] < 0 or pos[s] + L above cap or
 * rope_len is not written at all, and the return value counts those.  The
 * rotation and rounding are the single-token append's. */
int kime_oracle_kv_append_varlen(const uint16_t *qkv, const int32_t *cu, const int32_t *pos, int n_seqs,
                                 int heads, int kv_heads, int cap, const float *cos_t, const float *sin_t,
                                 int rope_len, uint16_t *k_cache, uint16_t *v_cache) {
    size_t W = (size_t)HEAD * (heads + 2 * kv_heads);
    int bad = 0;
    for (int s = 0; s < n_seqs; s++) {
        int L = cu[s + 1] - cu[s], P0 = pos[s];
        if (P0 < 0 || (long)P0 + L > cap || (long)P0 + L > rope_len) {
            bad++;
            continue;
        }
        for (int i = 0; i < L; i++) {
            int P = P0 + i;
            const uint16_t *row = qkv + (size_t)(cu[s] + i) * W;
            const float *c = cos_t + (size_t)P * HALF, *sn = sin_t + (size_t)P * HALF;
            for (int g = 0; g < kv_heads; g++) {
                const uint16_t *xk = row + (size_t)(heads + g) * HEAD;
                const uint16_t *xv = row + (size_t)(heads + kv_heads + g) * HEAD;
                size_t dst = (((size_t)s * kv_heads + g) * cap + P) * HEAD;
                for (int t = 0; t < HALF; t++) {
                    float a = (float)bf16_bits_to_double(xk[t]);
                    float b = (float)bf16_bits_to_double(xk[t + HALF]);
                    float ac = a * c[t], bs = b * sn[t], bc = b * c[t], as = a * sn[t];
                    k_cache[dst + t] = kime_oracle_f32_to_bf16(ac - bs);
                    k_cache[dst + t + HALF] = kime_oracle_f32_to_bf16(bc + as);
                }
                for (int t = 0; t < HEAD; t++) v_cache[dst + t] = xv[t];
            }
        }
    }
    return bad;
}

typedef struct {
    const uint16_t *qkv;
    const int32_t *cu, *pos;
    int n_seqs, heads, kv_heads, cap;
    double scale;
    const double *cos, *sin;
    const uint16_t *k_cache, *v_cache;
    const int32_t *rows, *row_heads;
    long n_items;
    double *out;
    int tid, nthreads;
} chunk_job;

/* Query row r (row i of its sequence s), head h: q is rotated at position
 * P = pos[s] + i and attends cache rows 0..=P of kv head h/(heads/kv_heads),
 * the cache already holding the chunk's own keys ([argus] CausalSoftmax: row i
 * of a block at offset index_pos sees keys 0..=i+offset).  Only visible keys
 * are visited. */
static void chunk_one(const chunk_job *d, int r, int h, double *out) {
    int s = seq_of_row(d->cu, d->n_seqs, r);
    int P = d->pos[s] + (r - d->cu[s]);
    int g = h / (d->heads / d->kv_heads);
    size_t W = (size_t)HEAD * (d->heads + 2 * d->kv_heads);
    double xq[HEAD], yq[HEAD];
    for (int t = 0; t < HEAD; t++) xq[t] = bf16_bits_to_double(d->qkv[(size_t)r * W + (size_t)h * HEAD + t]);
    kime_oracle_rope(xq, d->cos + (size_t)P * HALF, d->sin + (size_t)P * HALF, yq);
    const uint16_t *K = d->k_cache + ((size_t)s * d->kv_heads + g) * d->cap * HEAD;
    const uint16_t *V = d->v_cache + ((size_t)s * d->kv_heads + g) * d->cap * HEAD;
    double *sc = (double *)malloc(sizeof(double) * (size_t)(P + 1));
    double m = -INFINITY;
    for (int j = 0; j <= P; j++) {
        double dot = 0.0;
        for (int t = 0; t < HEAD; t++) dot += yq[t] * bf16_bits_to_double(K[(size_t)j * HEAD + t]);
        sc[j] = d->scale * dot;
        if (sc[j] > m) m = sc[j];
    }
    double den = 0.0, num[HEAD];
    for (int t = 0; t < HEAD; t++) num[t] = 0.0;
    for (int j = 0; j <= P; j++) {
        double p = exp(sc[j] - m);
        den += p;
        for (int t = 0; t < HEAD; t++) num[t] += p * bf16_bits_to_double(V[(size_t)j * HEAD + t]);
    }
    for (int t = 0; t < HEAD; t++) out[t] = num[t] / den;
    free(sc);
}

static void *chunk_worker(void *p) {
    chunk_job *d = (chunk_job *)p;
    for (long k = d->tid; k < d->n_items; k += d->nthreads) {
        int r, h;
        if (d->rows) {
            r = d->rows[k];
            h = d->row_heads[k];
        } else {
            r = (int)(k / d->heads);
            h = (int)(k % d->heads);
        }
        chunk_one(d, r, h, d->out + (size_t)k * HEAD);
    }
    return NULL;
}

/* Chunked-prefill attention outputs for n_items (token row, head) pairs, or
 * for every row and head when rows is NULL (then out is [T, heads*64]).  The
 * caches must already hold every sequence's chunk (kime_oracle_kv_append_varlen).
 * Returns 0, or a negative code when an argument is malformed or a sequence's
 * positions leave [0, min(cap, rope_len)). */
int kime_oracle_attn_chunk(const uint16_t *qkv, const int32_t *cu, const int32_t *pos, int n_seqs, int heads,
                           int kv_heads, int cap, double scale, const double *cos_t, const double *sin_t,
                           int rope_len, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *rows, const int32_t *row_heads, long n_items, double *out,
                           int nthreads) {
    if (heads <= 0 || kv_heads <= 0 || heads % kv_heads || n_seqs < 0) return -1;
    if (n_seqs > 0 && cu[0] != 0) return -1;
    for (int s = 0; s < n_seqs; s++) {
        if (cu[s + 1] < cu[s]) return -1;
        if (pos[s] < 0 || (long)pos[s] + (cu[s + 1] - cu[s]) > cap ||
            (long)pos[s] + (cu[s + 1] - cu[s]) > rope_len)
            return -2;
    }
    if (n_seqs == 0) return 0;
    if (!rows) n_items = (long)cu[n_seqs] * heads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    chunk_job jobs[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (chunk_job){qkv, cu, pos, n_seqs, heads, kv_heads, cap, scale, cos_t, sin_t,
                              k_cache, v_cache, rows, row_heads, n_items, out, t, nthreads};
        if (nthreads == 1) chunk_worker(&jobs[t]);
        else pthread_create(&th[t], NULL, chunk_worker, &jobs[t]);
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
    return 0;
}

/* ---- QKV projection (the step before attention) ------------------------
 *
 * qkv[t, o] = sum_k x[t, k] * w[o, k] for every token row t of the packed
 * batch and every output column o (o in [0, 64*(heads + 2*kv_heads))): the
 * weight is stored [out width, in width], as kime-cuda 0.0.3 src/plan.rs lays
 * out the weight of Op::Gemm (shape [out.width, a.width]), and q, k and v are
 * the one fused [960, 576] weight ffai-argus 0.7.3 src/text.rs describes
 * under Block::q (q rows first, then k, then v; argus keeps them as three
 * matrices, which is the same product column block by column block).  x and w
 * are bfloat16 bit patterns, widened exactly; every product and sum is in
 * double, k in increasing order.  No bias, no activation (the attention
 * projection of both towers has neither). */
typedef struct {
    const uint16_t *x, *w;
    int rows, in_w, out_w;
    double *out;
    int t0, t1;
} proj_job;

static void *proj_worker(void *p) {
    const proj_job *j = (const proj_job *)p;
    for (int t = j->t0; t < j->t1; ++t)
        for (int o = 0; o < j->out_w; ++o) {
            double acc = 0.0;
            for (int k = 0; k < j->in_w; ++k)
                acc += bf16_bits_to_double(j->x[(size_t)t * j->in_w + k]) *
                       bf16_bits_to_double(j->w[(size_t)o * j->in_w + k]);
            j->out[(size_t)t * j->out_w + o] = acc;
        }
    return NULL;
}

int kime_oracle_qkv_proj(const uint16_t *x, const uint16_t *w, int rows, int in_w, int out_w, double *out,
                         int nthreads) {
    if (rows < 0 || in_w <= 0 || out_w <= 0) return -1;
    if (rows == 0) return 0;
    if (!x || !w || !out) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > rows) nthreads = rows;
    proj_job jobs[256];
    pthread_t th[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (proj_job){x, w, rows, in_w, out_w, out, (int)((long)rows * i / nthreads),
                             (int)((long)rows * (i + 1) / nthreads)};
        pthread_create(&th[i], NULL, proj_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    return 0;
}
