/*
 * moe_oracle.c -- plain fp64 CPU oracle for the forward pass of one sparse
 * Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the GPU library is
 * measured against.  It shares no code, header, table or helper with the CUDA
 * library; only tests, the package's smoke check and the benchmark's CPU
 * baseline load it.  Nothing here is tuned: every loop is the definition
 * written out, accumulated in double precision on the exact values of the
 * stored inputs (bf16 or fp32), with no intermediate rounding.
 *
 * The layer (sources, by page title and section):
 *   - "Sparse MoE inference kernels: expert parallelism, dynamic routing gates
 *     and all-to-all overlap" (blog.llmgo.top), section 1.1: a shared expert
 *     that every token passes through plus K routed experts picked by the gate
 *     network W_g; each expert is a gated FFN with W_gate, W_up, W_down
 *     (section 1.2).
 *   - adg.csdn.net sparse-MoE explainer ("1.8T parameters, 2% active"),
 *     section 2.2: scoring s = Router(h), selection of the K best scores,
 *     softmax over only the K selected scores, output = sum_i w_i*Expert_i(h).
 *   - Same llmgo page, section 4.3: flatten the [T,K] expert ids, order the
 *     slots by expert id, gather the rows, per-expert counts and offsets for a
 *     grouped GEMM.  (The page's code uses an unstable argsort and an
 *     inclusive cumsum; this oracle uses the stable order by flat slot and an
 *     exclusive scan with E+1 entries.)
 *   - "Computation and Data Movement for Inference", section 4: expert outputs
 *     go back to token order, are weighted and summed.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): ties in top-K go to the lower expert index; the K selected experts
 * of a token are ordered by descending score, which defines slot j; the
 * expert FFN is SwiGLU, h = SiLU(W_gate x) * (W_up x), y = W_down h, with
 * SiLU(z) = z / (1 + exp(-z)); the optional per-expert bias b is added to the
 * logits before both selection and softmax; the combine adds the shared
 * expert first, then slots j = 0..K-1 in order.
 *
 * Storage: row-major; weights are stored [out][in] like nn.Linear:
 *   x [T][d], w_g [E][d], w_gate/w_up [E][I][d], w_down [E][d][I],
 *   shared ws_gate/ws_up [Is][d], ws_down [d][Is].
 * dtype 0 = fp32 (float), 1 = bf16 (uint16_t bit patterns).
 *
 * 8-bit expert weights ("LLM from scratch, ch. 6", section "second route:
 * make every byte cheaper": x_q = round(x / s) + z, x_hat = (x_q - z) s, with
 * the scale per tensor, per channel or per group): codes are OCP E4M3 floats
 * (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; largest finite
 * magnitude 448; S.1111.111 is NaN; no infinities), zero point 0, one fp32
 * scale per weight row (output channel).  The dequantised weight is
 * w_hat[r][c] = value(code[r][c]) * scale[r]; the fp8 layer is the layer
 * above with every expert matrix replaced by w_hat (router weights stay in
 * the activation dtype).  Readings: "round" is round-to-nearest, ties to an
 * even mantissa, onto the E4M3 grid, clamped to +-448; the row scale maps the
 * row's largest magnitude to 448 (scale = amax / 448 in fp32, 1 for a row of
 * zeros).
 *
 * 8-bit activations (W8A8, the *_w8a8 entry points at the end): the same
 * per-row quantisation applied to x and to the expert's hidden row h, which
 * is first rounded to fp32 and then to bf16; these roundings are part of
 * that method's definition and the only intermediate roundings in the file.
 * The *_a2 entry points carry x and h as two E4M3 planes each (a code and
 * the code of its remainder, one scale per row): the library's form of the
 * 8-bit-weight layer on its 8-bit-by-8-bit tensor-core path.
 *
 * Block-scaled weights (the *_blocks entry points; the section's "per
 * group" granularity, in the square 128 x 128 blocks of DeepSeek-V3's 8-bit
 * checkpoints): one fp32 scale per block of 128 rows x 128 columns of the
 * stacked weight matrix, w_hat[r][c] = value(code[r][c]) *
 * scale[r / 128][c / 128], each block quantised by the row rule above
 * applied to its elements.
 *
 * Every entry point returns 0 on success and a negative number on a bad
 * argument; nothing is allocated that is not freed before return.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_E4M3 2 /* weight codes only: 8-bit E4M3 float times a per-row (or per-block) scale */
#define ORC_FP8_BLOCK 128 /* side of a square weight-scale block */

/* ------------------------------------------------------------------------ */
/* element access: the exact stored value, widened to double                */
/* ------------------------------------------------------------------------ */

static double bf16_bits_to_double(uint16_t b)
{
    /* a bf16 value is the upper half of an IEEE binary32 */
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int dtype, int64_t i)
{
    if (dtype == ORC_BF16)
        return bf16_bits_to_double(((const uint16_t *)base)[i]);
    return (double)((const float *)base)[i];
}

static size_t elem_size(int dtype) { return dtype == ORC_BF16 ? 2u : 4u; }

/* ------------------------------------------------------------------------ */
/* E4M3 codes                                                               */
/* ------------------------------------------------------------------------ */

/* The value of an E4M3 code: exponent field E (bias 7), mantissa M (3 bits);
 * E = 0 is the subnormal range M/8 * 2^-6; S.1111.111 is NaN. */
static double e4m3_value(uint8_t c)
{
    const int sgn = c >> 7, E = (c >> 3) & 15, M = c & 7;
    double v;
    if (E == 15 && M == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)M, -9);
    else
        v = ldexp(8.0 + M, E - 10); /* (1 + M/8) * 2^(E-7) */
    return sgn ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid; magnitudes above 448 (and
 * infinities) clamp to 448, NaN gives S.1111.111.  The grid spacing is 2^-9
 * below 2^-6 (subnormals) and 2^(e-3) in the binade [2^e, 2^(e+1)). */
static uint8_t e4m3_code(float f)
{
    const uint8_t sgn = signbit(f) ? 0x80 : 0x00;
    if (isnan(f))
        return sgn | 0x7F;
    const double a = fabs((double)f);
    if (a >= 448.0)
        return sgn | 0x7E;
    double unit;
    if (a < ldexp(1.0, -6)) {
        unit = ldexp(1.0, -9);
    } else {
        int ex;
        frexp(a, &ex); /* a = m 2^ex, 0.5 <= m < 1: the binade is [2^(ex-1), 2^ex) */
        unit = ldexp(1.0, ex - 1 - 3);
    }
    const double v = nearbyint(a / unit) * unit; /* ties to even (default mode) */
    if (v < ldexp(1.0, -6))
        return sgn | (uint8_t)(v * 512.0); /* zero or subnormal: M = v / 2^-9 */
    int ex;
    const double m = frexp(v, &ex);
    return sgn | (uint8_t)(((ex - 1 + 7) << 3) | (int)(m * 16.0 - 8.0));
}

/* A weight matrix as the FFN reads it: fp32 / bf16 elements, or E4M3 codes
 * with one scale per row of row_len elements, or (block > 0) one scale per
 * block of block x block elements (row-major over the blocks of the row-major
 * matrix: scale[(r / block) * (row_len / block) + c / block]). */
typedef struct {
    const void *base;
    int fmt; /* ORC_F32, ORC_BF16 or ORC_E4M3 */
    const float *scale;
    int64_t row_len;
    int64_t block; /* 0: a scale per row */
} orc_weight;

static orc_weight plain_weight(const void *base, int dtype)
{
    orc_weight w = {base, dtype, NULL, 1, 0};
    return w;
}

static orc_weight fp8_weight(const void *codes, const float *scale, int64_t row_len)
{
    orc_weight w = {codes, ORC_E4M3, scale, row_len, 0};
    return w;
}

static orc_weight fp8_block_weight(const void *codes, const float *scale, int64_t row_len)
{
    orc_weight w = {codes, ORC_E4M3, scale, row_len, ORC_FP8_BLOCK};
    return w;
}

/* E4M3 codes with row scales (blocks = 0) or 128 x 128 block scales */
static orc_weight fp8w(const void *codes, const float *scale, int64_t row_len, int blocks)
{
    return blocks ? fp8_block_weight(codes, scale, row_len) : fp8_weight(codes, scale, row_len);
}

/* w_hat[i] = value(code[i]) * its scale (the row's or the block's), or the
 * stored element */
static double load_weight(const orc_weight *w, int64_t i)
{
    if (w->fmt == ORC_E4M3) {
        const int64_t r = i / w->row_len;
        double sc;
        if (w->block > 0) {
            const int64_t c = i % w->row_len;
            const int64_t nbc = (w->row_len + w->block - 1) / w->block;
            sc = (double)w->scale[(r / w->block) * nbc + c / w->block];
        } else {
            sc = (double)w->scale[r];
        }
        return e4m3_value(((const uint8_t *)w->base)[i]) * sc;
    }
    return load_elem(w->base, w->fmt, i);
}

/* ------------------------------------------------------------------------ */
/* a plain parallel-for over independent rows (tokens or permuted rows)     */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(void *ctx, int64_t row);

typedef struct {
    row_fn fn;
    void *ctx;
    int64_t begin, end;
} par_slice;

static void *par_worker(void *arg)
{
    par_slice *s = (par_slice *)arg;
    for (int64_t r = s->begin; r < s->end; ++r)
        s->fn(s->ctx, r);
    return NULL;
}

int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void par_for(int64_t n, int nthreads, row_fn fn, void *ctx)
{
    if (nthreads <= 0)
        nthreads = oracle_default_threads();
    if (nthreads > n)
        nthreads = (int)(n > 0 ? n : 1);
    if (nthreads <= 1) {
        for (int64_t r = 0; r < n; ++r)
            fn(ctx, r);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    par_slice *sl = (par_slice *)malloc(sizeof(par_slice) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        sl[i].fn = fn;
        sl[i].ctx = ctx;
        sl[i].begin = n * i / nthreads;
        sl[i].end = n * (i + 1) / nthreads;
        if (pthread_create(&th[i], NULL, par_worker, &sl[i]) != 0) {
            /* could not start a thread: run this slice here */
            par_worker(&sl[i]);
            th[i] = 0;
        } else {
            ++started;
        }
    }
    for (int i = 0; i < nthreads; ++i)
        if (th[i])
            pthread_join(th[i], NULL);
    (void)started;
    free(th);
    free(sl);
}

/* ------------------------------------------------------------------------ */
/* stage 1: router scores, top-K, softmax over the K selected               */
/* ------------------------------------------------------------------------ */

#define ORC_ROUTER_SOFTMAX 0
#define ORC_ROUTER_SIGMOID 1

/* s_e = sum_k x[k] * w_g[e][k], the raw router score.  The gate network is a
 * linear map with one score per expert (explainer section 2.2, step 1; llmgo
 * page section 2.1). */
static void router_scores(int64_t d, int64_t E, int dtype, const void *x,
                          int64_t t, const void *w_g, double *s)
{
    for (int64_t e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int64_t k = 0; k < d; ++k)
            acc += load_elem(x, dtype, t * d + k) * load_elem(w_g, dtype, e * d + k);
        s[e] = acc;
    }
}

/* Selection keys, then the K picks and their weights.
 *
 * Softmax router (explainer section 2.2, steps 2-3): key_e = s_e + b_e;
 * w_j = exp(key_{i_j} - key_{i_0}) / sum_j' exp(key_{i_j'} - key_{i_0}), the
 * softmax over only the K selected keys.
 *
 * Sigmoid router (DeepSeek-V3 auxiliary-loss-free routing, llmgo page section
 * 2.2 and the dispatcher code of section 4.3): affinity a_e = 1/(1+exp(-s_e));
 * key_e = a_e + b_e, the bias steering the selection only; the weights use
 * the affinities alone, w_j = a_{i_j} / (sum_j' a_{i_j'} + 1e-6) (the code's
 * form; the section's formula omits the 1e-6 guard).
 *
 * Picks: the K largest keys one at a time; a strictly larger key replaces the
 * current best while scanning e upward, so among equal keys the lower index is
 * kept.  Slot j holds the j-th pick (descending key). */
static void select_and_weigh(int mode, int64_t E, int64_t K, const double *s,
                             const double *bias, double *key, double *aff,
                             unsigned char *taken, int32_t *idx, double *w)
{
    for (int64_t e = 0; e < E; ++e) {
        const double b = bias ? bias[e] : 0.0;
        if (mode == ORC_ROUTER_SIGMOID) {
            aff[e] = 1.0 / (1.0 + exp(-s[e]));
            key[e] = aff[e] + b;
        } else {
            key[e] = s[e] + b;
        }
    }
    memset(taken, 0, (size_t)E);
    for (int64_t j = 0; j < K; ++j) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || key[e] > key[best])
                best = e;
        }
        taken[best] = 1;
        idx[j] = (int32_t)best;
    }
    double denom = 0.0;
    if (mode == ORC_ROUTER_SIGMOID) {
        for (int64_t j = 0; j < K; ++j)
            denom += aff[idx[j]];
        for (int64_t j = 0; j < K; ++j)
            w[j] = aff[idx[j]] / (denom + 1e-6);
        return;
    }
    const double kmax = key[idx[0]];
    for (int64_t j = 0; j < K; ++j) {
        w[j] = exp(key[idx[j]] - kmax);
        denom += w[j];
    }
    for (int64_t j = 0; j < K; ++j)
        w[j] /= denom;
}

typedef struct {
    int64_t d, E, K;
    int dtype, mode;
    const void *x, *w_g;
    const double *bias;
    const float *logits_in;
    double *logits_out;
    int32_t *topk_idx;
    double *topk_w;
} route_ctx;

static void route_row(void *vctx, int64_t t)
{
    route_ctx *c = (route_ctx *)vctx;
    double *s = (double *)malloc(sizeof(double) * (size_t)c->E * 3);
    double *key = s + c->E, *aff = s + 2 * c->E;
    unsigned char *taken = (unsigned char *)malloc((size_t)c->E);
    if (c->logits_in) {
        for (int64_t e = 0; e < c->E; ++e)
            s[e] = (double)c->logits_in[t * c->E + e];
    } else {
        router_scores(c->d, c->E, c->dtype, c->x, t, c->w_g, s);
    }
    select_and_weigh(c->mode, c->E, c->K, s, c->bias, key, aff, taken,
                     c->topk_idx + t * c->K, c->topk_w + t * c->K);
    if (c->logits_out)
        memcpy(c->logits_out + t * c->E, key, sizeof(double) * (size_t)c->E);
    free(s);
    free(taken);
}

/*
 * oracle_route: scores, top-K and weights for T tokens; mode 0 = softmax
 * router, 1 = sigmoid router (see select_and_weigh).  Raw scores are
 * x . w_g^T in fp64, or the fp32 values of logits_in when it is non-NULL
 * (x and w_g are then ignored); bias (may be NULL) enters the keys either way.
 * logits_out [T][E] (optional) receives the selection keys.
 */
int oracle_route(int64_t T, int64_t d, int64_t E, int64_t K, int dtype,
                 int mode, const void *x, const void *w_g, const double *bias,
                 const float *logits_in, double *logits_out,
                 int32_t *topk_idx, double *topk_w, int nthreads)
{
    if (T < 0 || E < 1 || K < 1 || K > E || !topk_idx || !topk_w)
        return -1;
    if (mode != ORC_ROUTER_SOFTMAX && mode != ORC_ROUTER_SIGMOID)
        return -1;
    if (!logits_in && (!x || !w_g || d < 1))
        return -1;
    route_ctx c = {d, E, K, dtype, mode, x, w_g, bias, logits_in, logits_out, topk_idx, topk_w};
    par_for(T, nthreads, route_row, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* stage 2: counts, exclusive offsets, stable permutation                   */
/* ------------------------------------------------------------------------ */

/*
 * Flat slot f = t*K + j.  counts[e] = #{f : idx[f] == e}; offsets is the
 * exclusive scan (offsets[0] = 0, offsets[E] = T*K); perm lists the slots of
 * expert 0 in increasing f, then expert 1, ... (a counting sort, stable by
 * construction); inv_perm[perm[p]] = p.  llmgo page section 4.3 (flatten,
 * order by expert id, bincount, offsets); "Computation and Data Movement for
 * Inference" section 15 (sort the routing records by expert).
 */
int oracle_permute(int64_t T, int64_t E, int64_t K, const int32_t *topk_idx,
                   int32_t *counts, int32_t *offsets, int32_t *perm,
                   int32_t *inv_perm)
{
    if (T < 0 || E < 1 || K < 1 || !counts || !offsets)
        return -1;
    const int64_t n = T * K;
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t f = 0; f < n; ++f) {
        int32_t e = topk_idx[f];
        if (e < 0 || e >= E)
            return -2;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    for (int64_t e = 0; e < E; ++e)
        cursor[e] = offsets[e];
    for (int64_t f = 0; f < n; ++f) {
        int32_t p = cursor[topk_idx[f]]++;
        if (perm)
            perm[p] = (int32_t)f;
        if (inv_perm)
            inv_perm[f] = p;
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* stage 3: SwiGLU expert FFN over expert-contiguous rows                   */
/* ------------------------------------------------------------------------ */

/* y = W_down . (SiLU(W_gate . x) * (W_up . x)) for one row x of length d,
 * expert matrices given by their base element offsets.  The gated FFN with
 * W_gate, W_up, W_down is the expert of the llmgo page (section 1.2) and the
 * gated MLP "up, gate, down" of "LLM from scratch, ch. 6" (MLP roofline). */
static void swiglu_row(int64_t d, int64_t I, int dtype, const void *xrow_base,
                       int64_t xrow_off, const orc_weight *w_gate, const orc_weight *w_up,
                       const orc_weight *w_down, int64_t wg_off, int64_t wu_off,
                       int64_t wd_off, double *h, double *y)
{
    for (int64_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int64_t k = 0; k < d; ++k) {
            double xv = load_elem(xrow_base, dtype, xrow_off + k);
            g += load_weight(w_gate, wg_off + i * d + k) * xv;
            u += load_weight(w_up, wu_off + i * d + k) * xv;
        }
        double silu = g / (1.0 + exp(-g));
        h[i] = silu * u;
    }
    for (int64_t j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i)
            acc += load_weight(w_down, wd_off + j * I + i) * h[i];
        y[j] = acc;
    }
}

typedef struct {
    int64_t d, E, I;
    int dtype;
    const void *x_perm;
    const int32_t *offsets;
    orc_weight w_gate, w_up, w_down;
    double *y_perm;
} ffn_ctx;

static int64_t expert_of_row(const int32_t *offsets, int64_t E, int64_t p)
{
    /* the expert e with offsets[e] <= p < offsets[e+1] (empty experts have
     * offsets[e] == offsets[e+1] and never match) */
    for (int64_t e = 0; e < E; ++e)
        if (p >= offsets[e] && p < offsets[e + 1])
            return e;
    return -1;
}

static void ffn_row(void *vctx, int64_t p)
{
    ffn_ctx *c = (ffn_ctx *)vctx;
    int64_t e = expert_of_row(c->offsets, c->E, p);
    double *h = (double *)malloc(sizeof(double) * (size_t)c->I);
    const int64_t wgu = e * c->I * c->d, wd = e * c->d * c->I;
    swiglu_row(c->d, c->I, c->dtype, c->x_perm, p * c->d, &c->w_gate, &c->w_up,
               &c->w_down, wgu, wgu, wd, h, c->y_perm + p * c->d);
    free(h);
}

/*
 * oracle_expert_ffn: rows [0, offsets[E]) of x_perm belong to experts by the
 * offsets array (grouped-GEMM form, llmgo page section 4.2); y_perm [rows][d]
 * in fp64.  Experts with zero rows contribute nothing and read nothing
 * (llmgo page, FAQ Q1).
 */
static int expert_ffn(int64_t d, int64_t E, int64_t I, int dtype, const void *x_perm,
                      const int32_t *offsets, orc_weight w_gate, orc_weight w_up,
                      orc_weight w_down, double *y_perm, int nthreads)
{
    if (d < 1 || E < 1 || I < 1 || !offsets || !y_perm)
        return -1;
    if (offsets[0] != 0)
        return -1;
    for (int64_t e = 0; e < E; ++e)
        if (offsets[e + 1] < offsets[e])
            return -1;
    ffn_ctx c = {d, E, I, dtype, x_perm, offsets, w_gate, w_up, w_down, y_perm};
    par_for(offsets[E], nthreads, ffn_row, &c);
    return 0;
}

int oracle_expert_ffn(int64_t d, int64_t E, int64_t I, int dtype,
                      const void *x_perm, const int32_t *offsets,
                      const void *w_gate, const void *w_up, const void *w_down,
                      double *y_perm, int nthreads)
{
    return expert_ffn(d, E, I, dtype, x_perm, offsets, plain_weight(w_gate, dtype),
                      plain_weight(w_up, dtype), plain_weight(w_down, dtype), y_perm, nthreads);
}

/* The same with E4M3 expert weights: codes w_gate/w_up [E][I][d] with scales
 * s_gate/s_up [E][I], w_down [E][d][I] with s_down [E][d] (one scale per
 * weight row); x_perm in dtype. */
int oracle_expert_ffn_fp8(int64_t d, int64_t E, int64_t I, int dtype,
                          const void *x_perm, const int32_t *offsets,
                          const uint8_t *w_gate, const uint8_t *w_up,
                          const uint8_t *w_down, const float *s_gate,
                          const float *s_up, const float *s_down,
                          double *y_perm, int nthreads)
{
    if (!w_gate || !w_up || !w_down || !s_gate || !s_up || !s_down)
        return -1;
    return expert_ffn(d, E, I, dtype, x_perm, offsets, fp8_weight(w_gate, s_gate, d),
                      fp8_weight(w_up, s_up, d), fp8_weight(w_down, s_down, I), y_perm,
                      nthreads);
}

/* The same with 128 x 128 block scales (oracle_quantize_fp8_blocks of the
 * stacked matrices): s_gate/s_up [ceil(E*I/128)][ceil(d/128)], s_down
 * [ceil(E*d/128)][ceil(I/128)]. */
int oracle_expert_ffn_fp8_blocks(int64_t d, int64_t E, int64_t I, int dtype,
                                 const void *x_perm, const int32_t *offsets,
                                 const uint8_t *w_gate, const uint8_t *w_up,
                                 const uint8_t *w_down, const float *s_gate,
                                 const float *s_up, const float *s_down,
                                 double *y_perm, int nthreads)
{
    if (!w_gate || !w_up || !w_down || !s_gate || !s_up || !s_down)
        return -1;
    return expert_ffn(d, E, I, dtype, x_perm, offsets, fp8_block_weight(w_gate, s_gate, d),
                      fp8_block_weight(w_up, s_up, d), fp8_block_weight(w_down, s_down, I),
                      y_perm, nthreads);
}

/* ------------------------------------------------------------------------ */
/* stage 4: combine                                                         */
/* ------------------------------------------------------------------------ */

/*
 * y[t] = y_shared[t] + sum_{j=0..K-1} w[t][j] * y_perm[inv_perm[t*K+j]],
 * the shared term first, then j ascending.  Explainer section 2.2 step 4
 * (weighted sum of the selected experts); llmgo page section 1.1 (shared
 * expert output added to the routed sum); "Computation and Data Movement for
 * Inference" section 4 (back to token order, weighted, merged).
 */
int oracle_combine(int64_t T, int64_t d, int64_t K, const double *y_perm,
                   const int32_t *inv_perm, const double *topk_w,
                   const double *y_shared, double *y)
{
    if (T < 0 || d < 1 || K < 1 || !y)
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < d; ++c) {
            double acc = y_shared ? y_shared[t * d + c] : 0.0;
            for (int64_t j = 0; j < K; ++j) {
                int64_t p = inv_perm[t * K + j];
                acc += topk_w[t * K + j] * y_perm[p * d + c];
            }
            y[t * d + c] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* the shared expert                                                         */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t d, Is;
    int dtype;
    const void *x;
    orc_weight ws_gate, ws_up, ws_down;
    const int32_t *tokens;
    double *y_s;
} shared_ctx;

static void shared_row(void *vctx, int64_t r)
{
    shared_ctx *c = (shared_ctx *)vctx;
    int64_t t = c->tokens ? c->tokens[r] : r;
    double *h = (double *)malloc(sizeof(double) * (size_t)c->Is);
    swiglu_row(c->d, c->Is, c->dtype, c->x, t * c->d, &c->ws_gate, &c->ws_up,
               &c->ws_down, 0, 0, 0, h, c->y_s + r * c->d);
    free(h);
}

/* y_s[t] = SwiGLU_shared(x[t]) for every token (weight 1, no routing):
 * the always-active shared expert of the llmgo page, section 1.1. */
int oracle_shared_ffn(int64_t T, int64_t d, int64_t Is, int dtype,
                      const void *x, const void *ws_gate, const void *ws_up,
                      const void *ws_down, double *y_s, int nthreads)
{
    if (T < 0 || d < 1 || Is < 1 || !y_s)
        return -1;
    shared_ctx c = {d, Is, dtype, x, plain_weight(ws_gate, dtype), plain_weight(ws_up, dtype),
                    plain_weight(ws_down, dtype), NULL, y_s};
    par_for(T, nthreads, shared_row, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* the whole layer, four stages                                             */
/* ------------------------------------------------------------------------ */

/*
 * oracle_forward: route -> permute (+ gather x rows into expert order) ->
 * expert FFN -> shared expert -> combine, for all T tokens.  Outputs in fp64:
 * y [T][d]; optional topk_idx [T][K], topk_w [T][K], counts [E],
 * offsets [E+1], perm / inv_perm [T*K].  Is == 0 means no shared expert;
 * mode selects the router (0 softmax, 1 sigmoid; see select_and_weigh).
 */
int oracle_forward(int64_t T, int64_t d, int64_t E, int64_t K, int64_t I,
                   int64_t Is, int dtype, int mode, const void *x, const void *w_g,
                   const double *bias, const void *w_gate, const void *w_up,
                   const void *w_down, const void *ws_gate, const void *ws_up,
                   const void *ws_down, double *y, int32_t *topk_idx_out,
                   double *topk_w_out, int32_t *counts_out,
                   int32_t *offsets_out, int32_t *perm_out,
                   int32_t *inv_perm_out, int nthreads)
{
    if (T < 0 || d < 1 || E < 1 || K < 1 || K > E || I < 1 || Is < 0 || !y)
        return -1;
    const int64_t n = T * K;
    const size_t es = elem_size(dtype);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)(n ? n : 1));
    int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
    int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
    unsigned char *x_perm = (unsigned char *)malloc(es * (size_t)(n ? n : 1) * (size_t)d);
    double *y_perm = (double *)malloc(sizeof(double) * (size_t)(n ? n : 1) * (size_t)d);
    double *y_s = Is ? (double *)malloc(sizeof(double) * (size_t)(T ? T : 1) * (size_t)d) : NULL;
    int rc = oracle_route(T, d, E, K, dtype, mode, x, w_g, bias, NULL, NULL, idx, w, nthreads);
    if (rc == 0)
        rc = oracle_permute(T, E, K, idx, counts, offsets, perm, inv);
    if (rc == 0) {
        /* gather: row p of x_perm is the token row perm[p] / K (an exact copy) */
        for (int64_t p = 0; p < n; ++p)
            memcpy(x_perm + (size_t)p * (size_t)d * es,
                   (const unsigned char *)x + (size_t)(perm[p] / K) * (size_t)d * es,
                   (size_t)d * es);
        rc = oracle_expert_ffn(d, E, I, dtype, x_perm, offsets, w_gate, w_up,
                               w_down, y_perm, nthreads);
    }
    if (rc == 0 && Is)
        rc = oracle_shared_ffn(T, d, Is, dtype, x, ws_gate, ws_up, ws_down, y_s, nthreads);
    if (rc == 0)
        rc = oracle_combine(T, d, K, y_perm, inv, w, y_s, y);
    if (rc == 0) {
        if (topk_idx_out) memcpy(topk_idx_out, idx, sizeof(int32_t) * (size_t)n);
        if (topk_w_out) memcpy(topk_w_out, w, sizeof(double) * (size_t)n);
        if (counts_out) memcpy(counts_out, counts, sizeof(int32_t) * (size_t)E);
        if (offsets_out) memcpy(offsets_out, offsets, sizeof(int32_t) * (size_t)(E + 1));
        if (perm_out) memcpy(perm_out, perm, sizeof(int32_t) * (size_t)n);
        if (inv_perm_out) memcpy(inv_perm_out, inv, sizeof(int32_t) * (size_t)n);
    }
    free(idx); free(w); free(counts); free(offsets); free(perm); free(inv);
    free(x_perm); free(y_perm); free(y_s);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* the layer for a sample of tokens, straight from the definition           */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t d, E, K, I, Is;
    int dtype, mode;
    const void *x, *w_g;
    const double *bias;
    orc_weight w_gate, w_up, w_down, ws_gate, ws_up, ws_down;
    const int32_t *tokens;
    double *y, *logits;
    int32_t *idx;
    double *w;
    int planes;  /* 8-bit-activation experts: 1 or 2 E4M3 planes per row */
} tok_ctx;

static void token_row(void *vctx, int64_t r)
{
    tok_ctx *c = (tok_ctx *)vctx;
    const int64_t t = c->tokens[r];
    const int64_t d = c->d;
    int64_t hmax = c->I > c->Is ? c->I : c->Is;
    double *s = (double *)malloc(sizeof(double) * (size_t)c->E * 3);
    double *key = s + c->E, *aff = s + 2 * c->E;
    unsigned char *taken = (unsigned char *)malloc((size_t)c->E);
    double *h = (double *)malloc(sizeof(double) * (size_t)hmax);
    double *ye = (double *)malloc(sizeof(double) * (size_t)d);
    int32_t *idx = c->idx + r * c->K;
    double *w = c->w + r * c->K;
    double *y = c->y + r * d;

    router_scores(d, c->E, c->dtype, c->x, t, c->w_g, s);
    select_and_weigh(c->mode, c->E, c->K, s, c->bias, key, aff, taken, idx, w);
    if (c->logits)
        memcpy(c->logits + r * c->E, key, sizeof(double) * (size_t)c->E);

    /* y = SharedExpert(x_t) + sum_j w_j * Expert_{i_j}(x_t) */
    if (c->Is) {
        swiglu_row(d, c->Is, c->dtype, c->x, t * d, &c->ws_gate, &c->ws_up,
                   &c->ws_down, 0, 0, 0, h, y);
    } else {
        for (int64_t k = 0; k < d; ++k)
            y[k] = 0.0;
    }
    for (int64_t j = 0; j < c->K; ++j) {
        const int64_t e = idx[j];
        const int64_t wgu = e * c->I * d, wd = e * d * c->I;
        swiglu_row(d, c->I, c->dtype, c->x, t * d, &c->w_gate, &c->w_up,
                   &c->w_down, wgu, wgu, wd, h, ye);
        for (int64_t k = 0; k < d; ++k)
            y[k] += w[j] * ye[k];
    }
    free(s); free(taken); free(h); free(ye);
}

/*
 * oracle_forward_tokens: the layer output for the listed tokens only,
 * y_r = SharedExpert(x_t) + sum_{j} w_j Expert_{i_j}(x_t) with t = tokens[r].
 * Each token's output depends on its own row only (routing and the expert
 * weights do not depend on the other tokens; "Computation and Data Movement
 * for Inference", sections 5 and 16), so a sample of rows is checked
 * exactly as in the full layer.  Outputs: y [n][d], topk_idx [n][K],
 * topk_w [n][K], logits [n][E] (optional: the selection keys); mode selects
 * the router (0 softmax, 1 sigmoid).
 */
static int forward_tokens(int64_t n, const int32_t *tokens, int64_t T, int64_t d,
                          int64_t E, int64_t K, int64_t I, int64_t Is, int dtype,
                          int mode, const void *x, const void *w_g,
                          const double *bias, const orc_weight w[6], double *y,
                          int32_t *topk_idx, double *topk_w, double *logits,
                          int nthreads)
{
    if (n < 0 || d < 1 || E < 1 || K < 1 || K > E || I < 1 || Is < 0 || !y ||
        !topk_idx || !topk_w || (n > 0 && !tokens) ||
        (mode != ORC_ROUTER_SOFTMAX && mode != ORC_ROUTER_SIGMOID))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        if (tokens[r] < 0 || tokens[r] >= T)
            return -1;
    tok_ctx c = {d, E, K, I, Is, dtype, mode, x, w_g, bias, w[0], w[1], w[2],
                 w[3], w[4], w[5], tokens, y, logits, topk_idx, topk_w, 0};
    par_for(n, nthreads, token_row, &c);
    return 0;
}

int oracle_forward_tokens(int64_t n, const int32_t *tokens, int64_t T,
                          int64_t d, int64_t E, int64_t K, int64_t I,
                          int64_t Is, int dtype, int mode, const void *x,
                          const void *w_g, const double *bias,
                          const void *w_gate, const void *w_up,
                          const void *w_down, const void *ws_gate,
                          const void *ws_up, const void *ws_down, double *y,
                          int32_t *topk_idx, double *topk_w, double *logits,
                          int nthreads)
{
    const orc_weight w[6] = {plain_weight(w_gate, dtype), plain_weight(w_up, dtype),
                             plain_weight(w_down, dtype), plain_weight(ws_gate, dtype),
                             plain_weight(ws_up, dtype), plain_weight(ws_down, dtype)};
    return forward_tokens(n, tokens, T, d, E, K, I, Is, dtype, mode, x, w_g, bias, w, y,
                          topk_idx, topk_w, logits, nthreads);
}

/*
 * oracle_forward_tokens_fp8: oracle_forward_tokens with E4M3 expert weights
 * (routed and shared), one fp32 scale per weight row: s_gate/s_up [E][I],
 * s_down [E][d], ss_gate/ss_up [Is], ss_down [d].  x and w_g are in dtype.
 */
int oracle_forward_tokens_fp8(int64_t n, const int32_t *tokens, int64_t T,
                              int64_t d, int64_t E, int64_t K, int64_t I,
                              int64_t Is, int dtype, int mode, const void *x,
                              const void *w_g, const double *bias,
                              const uint8_t *w_gate, const uint8_t *w_up,
                              const uint8_t *w_down, const float *s_gate,
                              const float *s_up, const float *s_down,
                              const uint8_t *ws_gate, const uint8_t *ws_up,
                              const uint8_t *ws_down, const float *ss_gate,
                              const float *ss_up, const float *ss_down,
                              double *y, int32_t *topk_idx, double *topk_w,
                              double *logits, int nthreads)
{
    if (!w_gate || !w_up || !w_down || !s_gate || !s_up || !s_down)
        return -1;
    if (Is > 0 && (!ws_gate || !ws_up || !ws_down || !ss_gate || !ss_up || !ss_down))
        return -1;
    const orc_weight w[6] = {fp8_weight(w_gate, s_gate, d), fp8_weight(w_up, s_up, d),
                             fp8_weight(w_down, s_down, I), fp8_weight(ws_gate, ss_gate, d),
                             fp8_weight(ws_up, ss_up, d), fp8_weight(ws_down, ss_down, Is)};
    return forward_tokens(n, tokens, T, d, E, K, I, Is, dtype, mode, x, w_g, bias, w, y,
                          topk_idx, topk_w, logits, nthreads);
}

/*
 * oracle_forward_tokens_fp8_blocks: oracle_forward_tokens_fp8 with 128 x 128
 * block scales: s_gate/s_up [ceil(E*I/128)][ceil(d/128)], s_down
 * [ceil(E*d/128)][ceil(I/128)], ss_gate/ss_up [ceil(Is/128)][ceil(d/128)],
 * ss_down [ceil(d/128)][ceil(Is/128)].
 */
int oracle_forward_tokens_fp8_blocks(int64_t n, const int32_t *tokens, int64_t T,
                                     int64_t d, int64_t E, int64_t K, int64_t I,
                                     int64_t Is, int dtype, int mode, const void *x,
                                     const void *w_g, const double *bias,
                                     const uint8_t *w_gate, const uint8_t *w_up,
                                     const uint8_t *w_down, const float *s_gate,
                                     const float *s_up, const float *s_down,
                                     const uint8_t *ws_gate, const uint8_t *ws_up,
                                     const uint8_t *ws_down, const float *ss_gate,
                                     const float *ss_up, const float *ss_down,
                                     double *y, int32_t *topk_idx, double *topk_w,
                                     double *logits, int nthreads)
{
    if (!w_gate || !w_up || !w_down || !s_gate || !s_up || !s_down)
        return -1;
    if (Is > 0 && (!ws_gate || !ws_up || !ws_down || !ss_gate || !ss_up || !ss_down))
        return -1;
    const orc_weight w[6] = {fp8_block_weight(w_gate, s_gate, d),
                             fp8_block_weight(w_up, s_up, d),
                             fp8_block_weight(w_down, s_down, I),
                             fp8_block_weight(ws_gate, ss_gate, d),
                             fp8_block_weight(ws_up, ss_up, d),
                             fp8_block_weight(ws_down, ss_down, Is)};
    return forward_tokens(n, tokens, T, d, E, K, I, Is, dtype, mode, x, w_g, bias, w, y,
                          topk_idx, topk_w, logits, nthreads);
}

/* ------------------------------------------------------------------------ */
/* E4M3 codes and row quantisation                                          */
/* ------------------------------------------------------------------------ */

/* out[i] = value(codes[i]) (NaN for the NaN codes) */
int oracle_e4m3_decode(int64_t n, const uint8_t *codes, double *out)
{
    if (n < 0 || (n > 0 && (!codes || !out)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_value(codes[i]);
    return 0;
}

/* codes[i] = the E4M3 code nearest to v[i] (ties to even, clamped to +-448) */
int oracle_e4m3_encode(int64_t n, const float *v, uint8_t *codes)
{
    if (n < 0 || (n > 0 && (!v || !codes)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        codes[i] = e4m3_code(v[i]);
    return 0;
}

/* One scale for n fp32 values (amax / 448 in fp32, 1 when all are zero) and
 * the code of each value / scale (fp32 division); returns the scale. */
static float quantize_vec(const float *v, int64_t n, uint8_t *codes)
{
    float amax = 0.0f;
    for (int64_t c = 0; c < n; ++c) {
        const float a = fabsf(v[c]);
        if (a > amax)
            amax = a;
    }
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int64_t c = 0; c < n; ++c)
        codes[c] = e4m3_code(v[c] / s);
    return s;
}

/*
 * oracle_quantize_fp8_rows: per-channel quantisation of a row-major
 * [rows][cols] weight matrix (fp32 or bf16) to E4M3 codes with one fp32
 * scale per row (the x_q = round(x / s) + z form of the "make every byte cheaper" section
 * with z = 0): scale[r] = amax_r / 448 (1 when the row is all zeros), computed
 * in fp32; code = nearest E4M3 to (w / scale[r]) computed as an fp32 division.
 */
int oracle_quantize_fp8_rows(int64_t rows, int64_t cols, int dtype, const void *w,
                             uint8_t *codes, float *scale)
{
    if (rows < 0 || cols < 1 || (rows > 0 && (!w || !codes || !scale)))
        return -1;
    float *row = (float *)malloc(sizeof(float) * (size_t)cols);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c)
            row[c] = (float)load_elem(w, dtype, r * cols + c);
        scale[r] = quantize_vec(row, cols, codes + r * cols);
    }
    free(row);
    return 0;
}

/*
 * oracle_quantize_fp8_blocks: per-group quantisation ("per tensor, per
 * channel or per group" in the "make every byte cheaper" section) of a
 * row-major [rows][cols] matrix with one fp32 scale per square block of 128
 * rows x 128 columns (the last block row / column may be shorter):
 * scale[(r / 128) * ceil(cols / 128) + c / 128] = amax over the block / 448
 * (1 for a block of zeros), computed in fp32; code = nearest E4M3 to
 * (w / scale) computed as an fp32 division -- the row rule of
 * oracle_quantize_fp8_rows applied to each block's elements.
 */
int oracle_quantize_fp8_blocks(int64_t rows, int64_t cols, int dtype, const void *w,
                               uint8_t *codes, float *scale)
{
    if (rows < 0 || cols < 1 || (rows > 0 && (!w || !codes || !scale)))
        return -1;
    const int64_t B = ORC_FP8_BLOCK;
    const int64_t nbr = (rows + B - 1) / B, nbc = (cols + B - 1) / B;
    float *blk = (float *)malloc(sizeof(float) * (size_t)(B * B));
    uint8_t *cb = (uint8_t *)malloc((size_t)(B * B));
    for (int64_t br = 0; br < nbr; ++br) {
        for (int64_t bc = 0; bc < nbc; ++bc) {
            const int64_t r0 = br * B, c0 = bc * B;
            const int64_t nr = rows - r0 < B ? rows - r0 : B;
            const int64_t nc = cols - c0 < B ? cols - c0 : B;
            for (int64_t i = 0; i < nr; ++i)
                for (int64_t j = 0; j < nc; ++j)
                    blk[i * nc + j] = (float)load_elem(w, dtype, (r0 + i) * cols + c0 + j);
            scale[br * nbc + bc] = quantize_vec(blk, nr * nc, cb);
            for (int64_t i = 0; i < nr; ++i)
                for (int64_t j = 0; j < nc; ++j)
                    codes[(r0 + i) * cols + c0 + j] = cb[i * nc + j];
        }
    }
    free(blk);
    free(cb);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 8-bit activations (W8A8)                                                 */
/* ------------------------------------------------------------------------ */

/*
 * The same x_q = round(x / s) + z rule ("LLM from scratch, ch. 6", section
 * "second route: make every byte cheaper"; the section notes that a method
 * may quantise weights, activations or the KV cache) applied to the two
 * activations that enter an expert's matrix products, each with one scale
 * per row, exactly as a weight row is quantised:
 *   x_hat = value(quant(x)) * s_x         (the token's row, bf16 input)
 *   h     = SiLU(W_gate x_hat) * (W_up x_hat)
 *   h_b   = bf16(fp32(h))                  (h held in fp32, stored in bf16,
 *                                           the layer's activation type)
 *   h_hat = value(quant(h_b)) * s_h
 *   y     = W_down h_hat
 * with the E4M3 expert weights above.  Reading: the pages name activation
 * quantisation without fixing its granularity or where h is rounded; one
 * scale per row (per token for x, per routed row for h) and a bf16 h are
 * taken here.
 */

/* fp32 -> bf16, round to nearest even (NaN stays NaN, overflow gives inf) */
static float round_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {
        u = (u & 0xffff0000u) | ((u & 0x007fffffu) ? 0x00400000u : 0u);
    } else {
        u += 0x7fffu + ((u >> 16) & 1u);
        u &= 0xffff0000u;
    }
    float r;
    memcpy(&r, &u, sizeof r);
    return r;
}

/* out[i] = round_bf16(v[i]) (exposed for its pin) */
int oracle_round_bf16(int64_t n, const float *v, float *out)
{
    if (n < 0 || (n > 0 && (!v || !out)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = round_bf16(v[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* activations as two E4M3 planes                                           */
/* ------------------------------------------------------------------------ */

/*
 * A bf16 activation row carried by two E4M3 codes per element and one fp32
 * scale per row (the same "make every byte cheaper" rule, x_q = round(x / s),
 * applied twice): s = amax / 448 as for one plane, q = v / s (fp32 division),
 * hi = round(q) onto the E4M3 grid, r = q - value(hi) (an fp32 subtraction,
 * exact: r is a multiple of q's unit in the last place and smaller than half
 * of hi's grid step), lo = round(r).  The row is then read as
 *   x_tilde = s * (value(hi) + value(lo)),
 * within 2^-8 of |x| relative plus 2^-10 s absolute (lo's subnormal step),
 * and exactly x when s is a power of two and |x| >= s / 4 (a bf16 value has
 * 8 significant bits; hi keeps the top 4 after rounding, r needs at most 3
 * more, none finer than the 2^-9 step).  Reading:
 * the page names 8-bit activations without a second plane; this split is
 * how the library feeds bf16 activations to an 8-bit-by-8-bit tensor-core
 * product, an approximation of the exact W8A16 layer defined here so that it
 * can be checked on its own.
 */
static float split_vec(const float *v, int64_t n, uint8_t *hi, uint8_t *lo)
{
    float amax = 0.0f;
    for (int64_t c = 0; c < n; ++c) {
        const float a = fabsf(v[c]);
        if (a > amax)
            amax = a;
    }
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int64_t c = 0; c < n; ++c) {
        const float q = v[c] / s;
        hi[c] = e4m3_code(q);
        const float r = q - (float)e4m3_value(hi[c]);
        lo[c] = e4m3_code(r);
    }
    return s;
}

/*
 * oracle_split_e4m3_rows: the two-plane codes of a row-major [rows][cols]
 * matrix (fp32 or bf16): hi[r][c], lo[r][c] and scale[r] as in split_vec.
 */
int oracle_split_e4m3_rows(int64_t rows, int64_t cols, int dtype, const void *x, uint8_t *hi,
                           uint8_t *lo, float *scale)
{
    if (rows < 0 || cols < 1 || (rows > 0 && (!x || !hi || !lo || !scale)))
        return -1;
    float *row = (float *)malloc(sizeof(float) * (size_t)cols);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c)
            row[c] = (float)load_elem(x, dtype, r * cols + c);
        scale[r] = split_vec(row, cols, hi + r * cols, lo + r * cols);
    }
    free(row);
    return 0;
}

/* Scratch of one W8A8 expert row: n = max(d, I). */
typedef struct {
    float *f;    /* [n] fp32 row being quantised  */
    uint8_t *c;  /* [n] its codes (hi plane)      */
    uint8_t *c2; /* [n] lo plane (two planes)     */
    double *xh;  /* [d] x_hat                     */
    double *h;   /* [I] h, then h_hat             */
} a8_scratch;

static int a8_alloc(a8_scratch *s, int64_t d, int64_t I)
{
    const int64_t n = d > I ? d : I;
    s->f = (float *)malloc(sizeof(float) * (size_t)n);
    s->c = (uint8_t *)malloc((size_t)n);
    s->c2 = (uint8_t *)malloc((size_t)n);
    s->xh = (double *)malloc(sizeof(double) * (size_t)d);
    s->h = (double *)malloc(sizeof(double) * (size_t)I);
    return s->f && s->c && s->c2 && s->xh && s->h;
}

static void a8_free(a8_scratch *s)
{
    free(s->f); free(s->c); free(s->c2); free(s->xh); free(s->h);
}

/* The row s->f[0..n) as the expert reads it: one plane (planes = 1:
 * value(code) * s) or two (planes = 2: (value(hi) + value(lo)) * s). */
static void act_hat(a8_scratch *s, int64_t n, int planes, double *out)
{
    if (planes == 2) {
        const float sc = split_vec(s->f, n, s->c, s->c2);
        for (int64_t k = 0; k < n; ++k)
            out[k] = (e4m3_value(s->c[k]) + e4m3_value(s->c2[k])) * (double)sc;
    } else {
        const float sc = quantize_vec(s->f, n, s->c);
        for (int64_t k = 0; k < n; ++k)
            out[k] = e4m3_value(s->c[k]) * (double)sc;
    }
}

/* One row through a W8A8 expert (see above); planes = 2: x and h each as two
 * E4M3 planes (split_vec) instead of one.  h_pre (optional, [I]) gets h
 * before rounding, h_hat_out (optional, [I]) gets h_hat. */
static void swiglu_row_a8(int64_t d, int64_t I, int dtype, const void *xrow_base,
                          int64_t xrow_off, const orc_weight *w_gate, const orc_weight *w_up,
                          const orc_weight *w_down, int64_t wg_off, int64_t wu_off,
                          int64_t wd_off, a8_scratch *s, double *y, double *h_pre,
                          double *h_hat_out, int planes)
{
    for (int64_t k = 0; k < d; ++k)
        s->f[k] = (float)load_elem(xrow_base, dtype, xrow_off + k);
    act_hat(s, d, planes, s->xh);
    for (int64_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int64_t k = 0; k < d; ++k) {
            g += load_weight(w_gate, wg_off + i * d + k) * s->xh[k];
            u += load_weight(w_up, wu_off + i * d + k) * s->xh[k];
        }
        s->h[i] = g / (1.0 + exp(-g)) * u;
    }
    if (h_pre)
        memcpy(h_pre, s->h, sizeof(double) * (size_t)I);
    for (int64_t i = 0; i < I; ++i)
        s->f[i] = round_bf16((float)s->h[i]);
    act_hat(s, I, planes, s->h);
    if (h_hat_out)
        memcpy(h_hat_out, s->h, sizeof(double) * (size_t)I);
    for (int64_t j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i)
            acc += load_weight(w_down, wd_off + j * I + i) * s->h[i];
        y[j] = acc;
    }
}

typedef struct {
    int64_t d, E, I;
    int dtype;
    const void *x_perm;
    const int32_t *offsets;
    orc_weight w_gate, w_up, w_down;
    double *y_perm, *h_pre, *h_hat;
    int planes;
} ffn_a8_ctx;

static void ffn_row_a8(void *vctx, int64_t p)
{
    ffn_a8_ctx *c = (ffn_a8_ctx *)vctx;
    const int64_t e = expert_of_row(c->offsets, c->E, p);
    const int64_t wgu = e * c->I * c->d, wd = e * c->d * c->I;
    a8_scratch s;
    if (a8_alloc(&s, c->d, c->I))
        swiglu_row_a8(c->d, c->I, c->dtype, c->x_perm, p * c->d, &c->w_gate, &c->w_up,
                      &c->w_down, wgu, wgu, wd, &s, c->y_perm + p * c->d,
                      c->h_pre ? c->h_pre + p * c->I : NULL,
                      c->h_hat ? c->h_hat + p * c->I : NULL, c->planes);
    a8_free(&s);
}

/*
 * oracle_expert_ffn_w8a8: oracle_expert_ffn_fp8 with 8-bit activations: each
 * row of x_perm (dtype) is quantised per row, h per row after its bf16
 * rounding.  Optional taps [rows][I] (fp64): h_pre = h before rounding,
 * h_hat = the dequantised quantised h.
 */
static int expert_ffn_a8(int64_t d, int64_t E, int64_t I, int dtype, const void *x_perm,
                         const int32_t *offsets, const uint8_t *w_gate, const uint8_t *w_up,
                         const uint8_t *w_down, const float *s_gate, const float *s_up,
                         const float *s_down, double *y_perm, double *h_pre, double *h_hat,
                         int nthreads, int planes, int blocks);

int oracle_expert_ffn_w8a8(int64_t d, int64_t E, int64_t I, int dtype,
                           const void *x_perm, const int32_t *offsets,
                           const uint8_t *w_gate, const uint8_t *w_up,
                           const uint8_t *w_down, const float *s_gate,
                           const float *s_up, const float *s_down, double *y_perm,
                           double *h_pre, double *h_hat, int nthreads)
{
    return expert_ffn_a8(d, E, I, dtype, x_perm, offsets, w_gate, w_up, w_down, s_gate, s_up,
                         s_down, y_perm, h_pre, h_hat, nthreads, 1, 0);
}

/*
 * oracle_expert_ffn_a2: oracle_expert_ffn_fp8 with each row of x_perm and
 * each hidden row h (after its bf16 rounding) carried as two E4M3 planes
 * (split_vec).  Same arguments and taps as oracle_expert_ffn_w8a8.
 */
int oracle_expert_ffn_a2(int64_t d, int64_t E, int64_t I, int dtype, const void *x_perm,
                         const int32_t *offsets, const uint8_t *w_gate, const uint8_t *w_up,
                         const uint8_t *w_down, const float *s_gate, const float *s_up,
                         const float *s_down, double *y_perm, double *h_pre, double *h_hat,
                         int nthreads)
{
    return expert_ffn_a8(d, E, I, dtype, x_perm, offsets, w_gate, w_up, w_down, s_gate, s_up,
                         s_down, y_perm, h_pre, h_hat, nthreads, 2, 0);
}

/* oracle_expert_ffn_w8a8 with the 128 x 128 block scales of
 * oracle_expert_ffn_fp8_blocks (x and h still quantised per row). */
int oracle_expert_ffn_w8a8_blocks(int64_t d, int64_t E, int64_t I, int dtype,
                                  const void *x_perm, const int32_t *offsets,
                                  const uint8_t *w_gate, const uint8_t *w_up,
                                  const uint8_t *w_down, const float *s_gate,
                                  const float *s_up, const float *s_down, double *y_perm,
                                  double *h_pre, double *h_hat, int nthreads)
{
    return expert_ffn_a8(d, E, I, dtype, x_perm, offsets, w_gate, w_up, w_down, s_gate, s_up,
                         s_down, y_perm, h_pre, h_hat, nthreads, 1, 1);
}

/* oracle_expert_ffn_a2 with the 128 x 128 block scales of
 * oracle_expert_ffn_fp8_blocks. */
int oracle_expert_ffn_a2_blocks(int64_t d, int64_t E, int64_t I, int dtype,
                                const void *x_perm, const int32_t *offsets,
                                const uint8_t *w_gate, const uint8_t *w_up,
                                const uint8_t *w_down, const float *s_gate,
                                const float *s_up, const float *s_down, double *y_perm,
                                double *h_pre, double *h_hat, int nthreads)
{
    return expert_ffn_a8(d, E, I, dtype, x_perm, offsets, w_gate, w_up, w_down, s_gate, s_up,
                         s_down, y_perm, h_pre, h_hat, nthreads, 2, 1);
}

static int expert_ffn_a8(int64_t d, int64_t E, int64_t I, int dtype, const void *x_perm,
                         const int32_t *offsets, const uint8_t *w_gate, const uint8_t *w_up,
                         const uint8_t *w_down, const float *s_gate, const float *s_up,
                         const float *s_down, double *y_perm, double *h_pre, double *h_hat,
                         int nthreads, int planes, int blocks)
{
    if (d < 1 || E < 1 || I < 1 || !offsets || !y_perm || !w_gate || !w_up || !w_down ||
        !s_gate || !s_up || !s_down || offsets[0] != 0)
        return -1;
    for (int64_t e = 0; e < E; ++e)
        if (offsets[e + 1] < offsets[e])
            return -1;
    ffn_a8_ctx c = {d, E, I, dtype, x_perm, offsets, fp8w(w_gate, s_gate, d, blocks),
                    fp8w(w_up, s_up, d, blocks), fp8w(w_down, s_down, I, blocks), y_perm,
                    h_pre, h_hat, planes};
    par_for(offsets[E], nthreads, ffn_row_a8, &c);
    return 0;
}

static void token_row_a8(void *vctx, int64_t r)
{
    tok_ctx *c = (tok_ctx *)vctx;
    const int64_t t = c->tokens[r];
    const int64_t d = c->d;
    const int64_t hmax = c->I > c->Is ? c->I : c->Is;
    double *sc = (double *)malloc(sizeof(double) * (size_t)c->E * 3);
    double *key = sc + c->E, *aff = sc + 2 * c->E;
    unsigned char *taken = (unsigned char *)malloc((size_t)c->E);
    double *ye = (double *)malloc(sizeof(double) * (size_t)d);
    int32_t *idx = c->idx + r * c->K;
    double *w = c->w + r * c->K;
    double *y = c->y + r * d;
    a8_scratch s;
    a8_alloc(&s, d, hmax);

    router_scores(d, c->E, c->dtype, c->x, t, c->w_g, sc);
    select_and_weigh(c->mode, c->E, c->K, sc, c->bias, key, aff, taken, idx, w);
    if (c->logits)
        memcpy(c->logits + r * c->E, key, sizeof(double) * (size_t)c->E);

    /* y = SharedExpert(x_t) + sum_j w_j * Expert_{i_j}(x_t), every expert W8A8 */
    if (c->Is) {
        swiglu_row_a8(d, c->Is, c->dtype, c->x, t * d, &c->ws_gate, &c->ws_up, &c->ws_down,
                      0, 0, 0, &s, y, NULL, NULL, c->planes);
    } else {
        for (int64_t k = 0; k < d; ++k)
            y[k] = 0.0;
    }
    for (int64_t j = 0; j < c->K; ++j) {
        const int64_t e = idx[j];
        const int64_t wgu = e * c->I * d, wd = e * d * c->I;
        swiglu_row_a8(d, c->I, c->dtype, c->x, t * d, &c->w_gate, &c->w_up, &c->w_down, wgu,
                      wgu, wd, &s, ye, NULL, NULL, c->planes);
        for (int64_t k = 0; k < d; ++k)
            y[k] += w[j] * ye[k];
    }
    free(sc); free(taken); free(ye);
    a8_free(&s);
}

static int forward_tokens_a8(int64_t n, const int32_t *tokens, int64_t T, int64_t d, int64_t E,
                             int64_t K, int64_t I, int64_t Is, int dtype, int mode,
                             const void *x, const void *w_g, const double *bias,
                             const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down,
                             const float *s_gate, const float *s_up, const float *s_down,
                             const uint8_t *ws_gate, const uint8_t *ws_up,
                             const uint8_t *ws_down, const float *ss_gate, const float *ss_up,
                             const float *ss_down, double *y, int32_t *topk_idx,
                             double *topk_w, double *logits, int nthreads, int planes,
                             int blocks);

/*
 * oracle_forward_tokens_w8a8: oracle_forward_tokens_fp8 with every expert
 * (routed and shared) run W8A8 as above; the router still reads the
 * unquantised x.  Same arguments and outputs as oracle_forward_tokens_fp8.
 */
int oracle_forward_tokens_w8a8(int64_t n, const int32_t *tokens, int64_t T,
                               int64_t d, int64_t E, int64_t K, int64_t I,
                               int64_t Is, int dtype, int mode, const void *x,
                               const void *w_g, const double *bias,
                               const uint8_t *w_gate, const uint8_t *w_up,
                               const uint8_t *w_down, const float *s_gate,
                               const float *s_up, const float *s_down,
                               const uint8_t *ws_gate, const uint8_t *ws_up,
                               const uint8_t *ws_down, const float *ss_gate,
                               const float *ss_up, const float *ss_down,
                               double *y, int32_t *topk_idx, double *topk_w,
                               double *logits, int nthreads)
{
    return forward_tokens_a8(n, tokens, T, d, E, K, I, Is, dtype, mode, x, w_g, bias, w_gate,
                             w_up, w_down, s_gate, s_up, s_down, ws_gate, ws_up, ws_down,
                             ss_gate, ss_up, ss_down, y, topk_idx, topk_w, logits, nthreads, 1,
                             0);
}

/*
 * oracle_forward_tokens_a2: oracle_forward_tokens_fp8 with every expert's
 * input row and hidden row carried as two E4M3 planes (split_vec): the
 * library's form of the 8-bit-weight layer for expert groups on its
 * 8-bit-by-8-bit tensor-core path.  Same arguments and outputs.
 */
int oracle_forward_tokens_a2(int64_t n, const int32_t *tokens, int64_t T,
                             int64_t d, int64_t E, int64_t K, int64_t I,
                             int64_t Is, int dtype, int mode, const void *x,
                             const void *w_g, const double *bias,
                             const uint8_t *w_gate, const uint8_t *w_up,
                             const uint8_t *w_down, const float *s_gate,
                             const float *s_up, const float *s_down,
                             const uint8_t *ws_gate, const uint8_t *ws_up,
                             const uint8_t *ws_down, const float *ss_gate,
                             const float *ss_up, const float *ss_down,
                             double *y, int32_t *topk_idx, double *topk_w,
                             double *logits, int nthreads)
{
    return forward_tokens_a8(n, tokens, T, d, E, K, I, Is, dtype, mode, x, w_g, bias, w_gate,
                             w_up, w_down, s_gate, s_up, s_down, ws_gate, ws_up, ws_down,
                             ss_gate, ss_up, ss_down, y, topk_idx, topk_w, logits, nthreads, 2,
                             0);
}

/* oracle_forward_tokens_w8a8 with the 128 x 128 block scales of
 * oracle_forward_tokens_fp8_blocks (x and h still quantised per row). */
int oracle_forward_tokens_w8a8_blocks(int64_t n, const int32_t *tokens, int64_t T,
                                      int64_t d, int64_t E, int64_t K, int64_t I,
                                      int64_t Is, int dtype, int mode, const void *x,
                                      const void *w_g, const double *bias,
                                      const uint8_t *w_gate, const uint8_t *w_up,
                                      const uint8_t *w_down, const float *s_gate,
                                      const float *s_up, const float *s_down,
                                      const uint8_t *ws_gate, const uint8_t *ws_up,
                                      const uint8_t *ws_down, const float *ss_gate,
                                      const float *ss_up, const float *ss_down,
                                      double *y, int32_t *topk_idx, double *topk_w,
                                      double *logits, int nthreads)
{
    return forward_tokens_a8(n, tokens, T, d, E, K, I, Is, dtype, mode, x, w_g, bias, w_gate,
                             w_up, w_down, s_gate, s_up, s_down, ws_gate, ws_up, ws_down,
                             ss_gate, ss_up, ss_down, y, topk_idx, topk_w, logits, nthreads, 1,
                             1);
}

/* oracle_forward_tokens_a2 with the 128 x 128 block scales of
 * oracle_forward_tokens_fp8_blocks. */
int oracle_forward_tokens_a2_blocks(int64_t n, const int32_t *tokens, int64_t T,
                                    int64_t d, int64_t E, int64_t K, int64_t I,
                                    int64_t Is, int dtype, int mode, const void *x,
                                    const void *w_g, const double *bias,
                                    const uint8_t *w_gate, const uint8_t *w_up,
                                    const uint8_t *w_down, const float *s_gate,
                                    const float *s_up, const float *s_down,
                                    const uint8_t *ws_gate, const uint8_t *ws_up,
                                    const uint8_t *ws_down, const float *ss_gate,
                                    const float *ss_up, const float *ss_down,
                                    double *y, int32_t *topk_idx, double *topk_w,
                                    double *logits, int nthreads)
{
    return forward_tokens_a8(n, tokens, T, d, E, K, I, Is, dtype, mode, x, w_g, bias, w_gate,
                             w_up, w_down, s_gate, s_up, s_down, ws_gate, ws_up, ws_down,
                             ss_gate, ss_up, ss_down, y, topk_idx, topk_w, logits, nthreads, 2,
                             1);
}

static int forward_tokens_a8(int64_t n, const int32_t *tokens, int64_t T,
                               int64_t d, int64_t E, int64_t K, int64_t I,
                               int64_t Is, int dtype, int mode, const void *x,
                               const void *w_g, const double *bias,
                               const uint8_t *w_gate, const uint8_t *w_up,
                               const uint8_t *w_down, const float *s_gate,
                               const float *s_up, const float *s_down,
                               const uint8_t *ws_gate, const uint8_t *ws_up,
                               const uint8_t *ws_down, const float *ss_gate,
                               const float *ss_up, const float *ss_down,
                               double *y, int32_t *topk_idx, double *topk_w,
                               double *logits, int nthreads, int planes, int blocks)
{
    if (!w_gate || !w_up || !w_down || !s_gate || !s_up || !s_down)
        return -1;
    if (Is > 0 && (!ws_gate || !ws_up || !ws_down || !ss_gate || !ss_up || !ss_down))
        return -1;
    if (n < 0 || d < 1 || E < 1 || K < 1 || K > E || I < 1 || Is < 0 || !y ||
        !topk_idx || !topk_w || (n > 0 && !tokens) ||
        (mode != ORC_ROUTER_SOFTMAX && mode != ORC_ROUTER_SIGMOID))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        if (tokens[r] < 0 || tokens[r] >= T)
            return -1;
    tok_ctx c = {d, E, K, I, Is, dtype, mode, x, w_g, bias,
                 fp8w(w_gate, s_gate, d, blocks), fp8w(w_up, s_up, d, blocks),
                 fp8w(w_down, s_down, I, blocks),
                 fp8w(ws_gate, ss_gate, d, blocks), fp8w(ws_up, ss_up, d, blocks),
                 fp8w(ws_down, ss_down, Is, blocks),
                 tokens, y, logits, topk_idx, topk_w, planes};
    par_for(n, nthreads, token_row_a8, &c);
    return 0;
}
