/*
 * Float64 CPU oracle for tree-masked verification attention and for attention
 * over an affine-quantized K/V cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the CPU baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * Everything here is the plain definition: full logits, an explicit softmax
 * with max-subtraction, no split, no online rescaling, no blocking.  Inputs are
 * widened exactly from their stored type (binary32, binary16, bfloat16) to
 * binary64 by decoders written from the IEEE 754 / bfloat16 bit layouts.
 *
 * Sources (mlx-native 0.9.x, metaltile-std 0.1.0):
 *  - tree_attention.metal, header comment and the QK / online-softmax / PV
 *    sections of tree_attention_impl: logit = qk * scale + mask, GQA head
 *    kv_head = h / (n_heads / n_kv_heads), mask cells >= kv_seq_len ignored,
 *    a 32-key chunk whose cells are all <= -65504 contributes nothing, a row
 *    that never accumulates (S == 0) yields 0.
 *  - tree_attention.rs, `tree_attention` buffer docs: Q [n_heads, q_l, D],
 *    K/V [n_kv_heads, kv_capacity, D], mask [q_l, mask_stride],
 *    output [q_l, n_heads, D] (query-outer, head-inner).
 *  - the implicit causal mask of the parent kernel (tree_attention.metal header
 *    comment): row i attends keys [window_start, kv_seq_len - q_l + i].
 *  - flash_quantized_sdpa.rs, module doc "Layout" and the kernel body: pack-
 *    strided codes (element d at bit (d % pf) * bits of word d / pf,
 *    pf = 32 / bits), value = scale[g] * code + bias[g] with g = d / group_size,
 *    query pre-multiplied by the attention scale, sink = virtual key with logit
 *    sinks[q_idx % num_q_heads] (unscaled) and value 0, sliding window keeps t
 *    with t + window > tokens - 1, bool mask 0 drops a token, float mask is
 *    added to the logit, out = o / l when l > 0 else o.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

#define ORC_MASKED (-65504.0)

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double orc_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24);                /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        mag = (f == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp((double)(1024 + f), e - 25);    /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of a binary32. */
static double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double orc_load(const void *base, int dtype, size_t idx) {
    if (dtype == ORC_F32) return (double)((const float *)base)[idx];
    if (dtype == ORC_F16) return orc_half_to_double(((const uint16_t *)base)[idx]);
    return orc_bf16_to_double(((const uint16_t *)base)[idx]);
}

/* Decode n elements of the given type to binary64 (exposed for the pins). */
void oracle_decode(int dtype, int64_t n, const void *src, double *dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_load(src, dtype, (size_t)i);
}

/* ---------------------------------------------------------- worker pool */

typedef void (*orc_row_fn)(void *ctx, int64_t row);
typedef struct {
    orc_row_fn fn;
    void *ctx;
    int64_t n;
    int tid, nthreads;
} orc_job;

static void *orc_worker(void *arg) {
    orc_job *j = (orc_job *)arg;
    for (int64_t r = j->tid; r < j->n; r += j->nthreads) j->fn(j->ctx, r);
    return NULL;
}

static void orc_parallel_rows(orc_row_fn fn, void *ctx, int64_t n, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    orc_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].n = n;
        jobs[t].tid = t; jobs[t].nthreads = nthreads;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
    orc_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* --------------------------------------------------------- tree attention */

typedef struct {
    int H, Hk, D, N, C, L, stride, window_start, kv_dtype;
    double scale;
    const float *q;
    const void *k, *v;
    const float *mask;      /* NULL: implicit causal mask */
    const int32_t *sel;     /* rows as h * L + i, or NULL for all rows */
    double *out;
} orc_tree_ctx;

static double orc_tree_mask_value(const orc_tree_ctx *c, int i, int j) {
    if (c->mask) return (double)c->mask[(size_t)i * c->stride + j];
    /* implicit causal / sliding window: attend [window_start, N - L + i] */
    return (j >= c->window_start && j <= c->N - c->L + i) ? 0.0 : ORC_MASKED;
}

static void orc_tree_row(void *vctx, int64_t s) {
    const orc_tree_ctx *c = (const orc_tree_ctx *)vctx;
    int64_t rid = c->sel ? c->sel[s] : s;          /* all rows: rid = h * L + i */
    int h = (int)(rid / c->L), i = (int)(rid % c->L);
    int g = c->H / c->Hk;
    int kh = h / g;                                /* GQA: query head -> KV head */
    double *o = c->sel ? c->out + (size_t)s * c->D
                       : c->out + ((size_t)i * c->H + h) * c->D;   /* [L, H, D] */
    const float *qrow = c->q + ((size_t)h * c->L + i) * c->D;
    size_t kbase = (size_t)kh * c->C * c->D;

    double *logit = (double *)malloc(sizeof(double) * (size_t)(c->N > 0 ? c->N : 1));
    unsigned char *att = (unsigned char *)malloc((size_t)(c->N > 0 ? c->N : 1));
    double mx = -INFINITY;
    int any = 0;
    for (int j = 0; j < c->N; ++j) {
        double mv = orc_tree_mask_value(c, i, j);
        att[j] = mv > ORC_MASKED;                  /* -65504 (or below) = masked */
        if (!att[j]) continue;
        double dot = 0.0;
        for (int d = 0; d < c->D; ++d)
            dot += (double)qrow[d] * orc_load(c->k, c->kv_dtype, kbase + (size_t)j * c->D + d);
        logit[j] = dot * c->scale + mv;
        if (logit[j] > mx) mx = logit[j];
        any = 1;
    }
    for (int d = 0; d < c->D; ++d) o[d] = 0.0;
    if (any) {
        double z = 0.0;
        for (int j = 0; j < c->N; ++j) {
            if (!att[j]) continue;
            double w = exp(logit[j] - mx);
            z += w;
            for (int d = 0; d < c->D; ++d)
                o[d] += w * orc_load(c->v, c->kv_dtype, kbase + (size_t)j * c->D + d);
        }
        for (int d = 0; d < c->D; ++d) o[d] /= z;
    }
    free(logit);
    free(att);
}

/*
 * out: if sel == NULL, [L, H, D] in the pages' output layout; else [n_sel, D]
 * with row s for query row sel[s] = h * L + i.  Returns 0, or -1 on bad shapes.
 */
int oracle_tree_attention(int H, int Hk, int D, int N, int C, double scale, int L, int stride,
                          const float *q, const void *k, const void *v, int kv_dtype,
                          const float *mask, int window_start,
                          int n_sel, const int32_t *sel, double *out, int nthreads) {
    if (H <= 0 || Hk <= 0 || H % Hk || D <= 0 || N < 0 || C < N || L <= 0) return -1;
    if (mask && stride < N) return -1;
    orc_tree_ctx c = {H, Hk, D, N, C, L, stride, window_start, kv_dtype, scale,
                      q, k, v, mask, sel, out};
    int64_t n = sel ? n_sel : (int64_t)H * L;
    orc_parallel_rows(orc_tree_row, &c, n, nthreads);
    return 0;
}

/* ------------------------------------------------- quantized-KV attention */

typedef struct {
    int B, nQ, nKV, dim, N, bits, G, has_sinks, window, t_dtype;
    double scale;
    const void *queries;
    const uint32_t *kp, *vp;
    const void *ks, *kb, *vs, *vb;
    const float *sinks;
    const uint32_t *mask_bool;   /* nullable */
    const void *mask_float;      /* nullable, type T */
    const int32_t *sel;
    double *out;
} orc_quant_ctx;

/* value of element d of token t of KV row kv: scale * code + bias */
static double orc_dequant(const orc_quant_ctx *c, const uint32_t *packed, const void *sc,
                          const void *bi, int kv, int t, int d) {
    int pf = 32 / c->bits;
    int words = c->dim / pf;
    int groups = c->dim / c->G;
    size_t tok = (size_t)kv * c->N + t;
    uint32_t w = packed[tok * words + d / pf];
    uint32_t code = (w >> ((d % pf) * c->bits)) & ((1u << c->bits) - 1u);
    int g = d / c->G;
    return orc_load(sc, c->t_dtype, tok * groups + g) * (double)code +
           orc_load(bi, c->t_dtype, tok * groups + g);
}

static void orc_quant_row(void *vctx, int64_t s) {
    const orc_quant_ctx *c = (const orc_quant_ctx *)vctx;
    int64_t r = c->sel ? c->sel[s] : s;            /* query row q_idx in [0, B*nQ) */
    int rep = c->nQ / c->nKV;
    int kv = (int)(r / rep);
    double *o = c->out + (size_t)s * c->dim;
    double *qs = (double *)malloc(sizeof(double) * c->dim);
    double *logit = (double *)malloc(sizeof(double) * (size_t)c->N);
    unsigned char *use = (unsigned char *)malloc((size_t)c->N);
    for (int d = 0; d < c->dim; ++d)
        qs[d] = c->scale * orc_load(c->queries, c->t_dtype, (size_t)r * c->dim + d);

    double mx = -INFINITY;
    double sink = c->has_sinks ? (double)c->sinks[r % c->nQ] : 0.0;
    if (c->has_sinks) mx = sink;
    for (int t = 0; t < c->N; ++t) {
        int in_window = (c->window == 0) || ((int64_t)t + c->window > (int64_t)c->N - 1);
        int visible = !c->mask_bool || c->mask_bool[(size_t)r * c->N + t] != 0u;
        use[t] = in_window && visible;
        if (!use[t]) continue;
        double dot = 0.0;
        for (int d = 0; d < c->dim; ++d)
            dot += qs[d] * orc_dequant(c, c->kp, c->ks, c->kb, kv, t, d);
        if (c->mask_float) dot += orc_load(c->mask_float, c->t_dtype, (size_t)r * c->N + t);
        if (dot == -INFINITY) { use[t] = 0; continue; }
        logit[t] = dot;
        if (dot > mx) mx = dot;
    }
    for (int d = 0; d < c->dim; ++d) o[d] = 0.0;
    double z = c->has_sinks ? exp(sink - mx) : 0.0;   /* sink: value 0, counted once */
    for (int t = 0; t < c->N; ++t) {
        if (!use[t]) continue;
        double w = exp(logit[t] - mx);
        z += w;
        for (int d = 0; d < c->dim; ++d) o[d] += w * orc_dequant(c, c->vp, c->vs, c->vb, kv, t, d);
    }
    if (z > 0.0)
        for (int d = 0; d < c->dim; ++d) o[d] /= z;
    free(qs);
    free(logit);
    free(use);
}

/* out: [n_sel, dim] for rows sel[s], or [B*nQ, dim] when sel == NULL. */
int oracle_quant_sdpa(int B, int nQ, int nKV, int dim, int N, int bits, int G, int has_sinks,
                      int window, double scale, int t_dtype, const void *queries,
                      const uint32_t *k_packed, const void *k_scales, const void *k_biases,
                      const uint32_t *v_packed, const void *v_scales, const void *v_biases,
                      const float *sinks, const uint32_t *mask_bool, const void *mask_float,
                      int n_sel, const int32_t *sel, double *out, int nthreads) {
    if (B <= 0 || nQ <= 0 || nKV <= 0 || nQ % nKV || (bits != 4 && bits != 8)) return -1;
    if (dim <= 0 || dim % (32 / bits) || G <= 0 || dim % G || N <= 0) return -1;
    orc_quant_ctx c = {B, nQ, nKV, dim, N, bits, G, has_sinks, window, t_dtype, scale,
                       queries, k_packed, v_packed, k_scales, k_biases, v_scales, v_biases,
                       sinks, mask_bool, mask_float, sel, out};
    int64_t n = sel ? n_sel : (int64_t)B * nQ;
    orc_parallel_rows(orc_quant_row, &c, n, nthreads);
    return 0;
}

/* Dequantized values of one token: out[d] for d < dim (exposed for the pins). */
int oracle_dequant_token(int dim, int N, int bits, int G, int t_dtype, const uint32_t *packed,
                         const void *scales, const void *biases, int kv, int t, double *out) {
    orc_quant_ctx c;
    memset(&c, 0, sizeof c);
    c.dim = dim; c.N = N; c.bits = bits; c.G = G; c.t_dtype = t_dtype;
    for (int d = 0; d < dim; ++d) out[d] = orc_dequant(&c, packed, scales, biases, kv, t, d);
    return 0;
}

/*
 * Tree mask from a parent array (the step before the verify pass): the draft
 * tree's node i sits at KV position kv_seq_len - q_l + i and attends the
 * prefix [0, kv_seq_len - q_l), its ancestors and itself (tree_attention.metal
 * header comment and the tree_attention.rs tests: 0 = attend, -65504 =
 * masked).  Node a is an ancestor of i when the chain i, parents[i],
 * parents[parents[i]], ... reaches a; the chain ends at a value outside
 * [0, current node) (-1 for the root).  Cells at positions >= kv_seq_len, up
 * to mask_stride, are -65504.  out is [q_l, mask_stride] binary32.
 */
int oracle_tree_mask(const int32_t *parents, int q_l, int kv_seq_len, int mask_stride, float *out) {
    if (q_l < 1 || kv_seq_len < q_l || mask_stride < kv_seq_len) return 1;
    const int prefix = kv_seq_len - q_l;
    unsigned char *anc = (unsigned char *)malloc((size_t)q_l);
    if (anc == NULL) return 2;
    for (int i = 0; i < q_l; ++i) {
        for (int a = 0; a < q_l; ++a) anc[a] = 0;
        int node = i;
        anc[node] = 1;
        for (;;) {
            const int up = parents[node];
            if (up < 0 || up >= node) break;
            anc[up] = 1;
            node = up;
        }
        float *row = out + (size_t)i * mask_stride;
        for (int j = 0; j < mask_stride; ++j) {
            int attend = 0;
            if (j < prefix) attend = 1;
            else if (j < kv_seq_len) attend = anc[j - prefix];
            row[j] = attend ? 0.0f : -65504.0f;
        }
    }
    free(anc);
    return 0;
}
