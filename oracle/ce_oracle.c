/*
 * ce_oracle.c -- CPU oracle for the fused vocabulary cross-entropy pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, double-precision
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check in __graft_entry__ and the CPU-baseline leg of bench.py load it.  The
 * GPU library never links, includes or calls anything in this directory, and
 * this file shares no code, header or constant with the GPU library.
 *
 * Sources (web pages; cited by title and section):
 *   [TENPU-29]  Ascend/TransformerEngineNPU issue #29, "Parallel Cross Entropy
 *               (Triton)": section 1 "Interface" (argument list and the
 *               precision contract: FP32 accumulation, FP32 loss, gradient
 *               written back in the input dtype), section 6 "Memory" (gradient
 *               staged in place in the input buffer), section 7 "Known
 *               limitations" (n_non_ignore).
 *   [HYPER-269] mindspore/hyper-parallel issue #269, section 3.1 "What Hyper
 *               already has" (vocab-sharded CE: MAX all-reduce, SUM all-reduce,
 *               target-logit gather; uneven ceil(V/tp) split; ignore_index
 *               -100).
 *   [OPSNN-CE]  CSDN, "Ascend CANN ops-nn cross-entropy fusion: from three
 *               kernel launches to one": section "Fusion scheme: log_softmax +
 *               NLL" (loss = logsumexp(x) - x[target]), section "Backward"
 *               (d logits = softmax - onehot), pitfall 1 (max-stabilised
 *               logsumexp), pitfall 3 (label-smoothing gradient).
 *
 * Readings taken where the pages are silent or disagree (each is listed in
 * the design notes with its reason):
 *   - label smoothing follows PyTorch: the smoothing mass a is spread over
 *     all V classes, the target included, so the smoothed loss is
 *     (1-a)*nll + a*mean_j(-log_softmax_j) and the gradient subtracts a/V
 *     from every class.  The ops-nn page divides by V-1 and skips the target;
 *     that variant is not what the TENPU interface (aligned with NVTE and
 *     checked against torch F.cross_entropy) computes.
 *   - a row whose target equals ignore_idx has loss 0 and gradient 0 and is
 *     left out of n (the ignore test is made before the range test).
 *   - a row whose target is outside [0, V) and not ignore_idx is an error:
 *     the error word gets ORACLE_ERR_TARGET_RANGE, its loss is NaN, its
 *     gradient row is 0, and it still counts in n.
 *   - reduce_loss: dloss is the upstream gradient of the mean (one scalar),
 *     so each kept row is scaled by dloss/n; n == 0 gives a NaN mean and an
 *     all-zero gradient, as torch F.cross_entropy does.
 *   - class weights (optional) follow torch F.cross_entropy(weight=...): each
 *     class's term of the smoothed target is weighted, and the mean divides by
 *     the summed weight of the kept rows' targets.
 *   - without reduce_loss, dloss holds one scale per row (NULL means 1).
 *   - rows are visited in the flattened (dim0, dim1) order r = i*dim1 + j for
 *     both layouts (B,SQ,V) and (SQ,B,V); targets use the same (dim0, dim1).
 *
 * Parity pins live in tests/test_oracle_pins.py (closed forms, brute force,
 * finite differences, torch float64 F.cross_entropy, split == unsplit,
 * exhaustive rounding checks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F16 2

#define ORACLE_ERR_TARGET_RANGE 1u

/* ---------------------------------------------------------------------------
 * Storage formats.  Decoding is exact; encoding rounds once from double to the
 * nearest value of the format, ties to even (IEEE 754 roundTiesToEven).
 * ------------------------------------------------------------------------- */

static double f16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_decode(const void* base, int dtype, int64_t idx) {
    if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
    if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    return f16_bits_to_double(((const uint16_t*)base)[idx]);
}

/* Round v to a binary format with `p` significand bits (implicit bit
 * included), minimum normal exponent `emin` and largest finite `maxf`. */
static double round_to_format(double v, int p, int emin, double maxf) {
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int e;
    frexp(fabs(v), &e);           /* |v| = f * 2^e, f in [0.5, 1) */
    int lead = e - 1;             /* exponent of the leading bit  */
    if (lead < emin) lead = emin; /* subnormal range: fixed spacing */
    double q = ldexp(1.0, lead - (p - 1)); /* spacing of the format at |v| */
    double r = nearbyint(v / q) * q;       /* v/q is exact; nearbyint ties to even */
    if (fabs(r) > maxf) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

double oracle_round(double v, int dtype) {
    if (dtype == ORACLE_F32) return round_to_format(v, 24, -126, 3.4028234663852886e38);
    if (dtype == ORACLE_BF16) return round_to_format(v, 8, -126, 3.3895313892515355e38);
    return round_to_format(v, 11, -14, 65504.0);
}

/* Bits of oracle_round(v, dtype) in the storage format (fp32 bits for F32). */
uint32_t oracle_encode(double v, int dtype) {
    double r = oracle_round(v, dtype);
    if (dtype == ORACLE_F32 || dtype == ORACLE_BF16) {
        float f = (float)r; /* exact: r is an fp32 (and bf16) value */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        if (dtype == ORACLE_BF16) {
            if (isnan(r)) return 0x7fc0u;
            return u >> 16;
        }
        return u;
    }
    /* fp16 */
    uint32_t sign = signbit(r) ? 0x8000u : 0u;
    if (isnan(r)) return 0x7e00u;
    double a = fabs(r);
    if (isinf(a)) return sign | 0x7c00u;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14)) return sign | (uint32_t)(a / ldexp(1.0, -24)); /* subnormal */
    int e;
    frexp(a, &e);
    int lead = e - 1;
    uint32_t mant = (uint32_t)(a / ldexp(1.0, lead - 10)) - 1024u;
    return sign | ((uint32_t)(lead + 15) << 10) | mant;
}

/* oracle_round over an array (out may alias in). */
void oracle_round_array(const double* in, int64_t n, int dtype, double* out) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_round(in[k], dtype);
}

/* ---------------------------------------------------------------------------
 * One token row, from the definitions.
 *   lse    = m + log(sum_j exp(x_j - m)),  m = max_j x_j   [OPSNN-CE pitfall 1]
 *   nll    = lse - x_y                                      [OPSNN-CE fusion scheme]
 *   smooth = lse - (1/V) sum_j x_j = mean_j(-log_softmax_j)
 *   loss   = (1-a) nll + a smooth                           (PyTorch reading)
 *   grad_j = g (exp(x_j - lse) - (1-a)[j==y] - a/V)         [OPSNN-CE backward,
 *                                                            pitfall 3, V reading]
 * x holds the row in double; grad may be NULL (forward only).
 * ------------------------------------------------------------------------- */
static void row_reference(const double* x, int64_t V, int64_t y, double a, double g,
                          double* loss, double* lse_out, double* grad) {
    double m = -INFINITY;
    for (int64_t j = 0; j < V; ++j)
        if (x[j] > m) m = x[j];
    double d = 0.0, S = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        d += exp(x[j] - m);
        S += x[j];
    }
    double lse = m + log(d);
    double nll = lse - x[y];
    double smooth = lse - S / (double)V;
    *loss = (1.0 - a) * nll + a * smooth;
    if (lse_out) *lse_out = lse;
    if (grad) {
        for (int64_t j = 0; j < V; ++j) {
            double q = (j == y ? 1.0 - a : 0.0) + a / (double)V; /* smoothed target */
            grad[j] = g * (exp(x[j] - lse) - q);
        }
    }
}

/* The same row with per-class weights w (the weighted cross-entropy of torch
 * F.cross_entropy(weight=w), which hyper-parallel #269's comparison table lists
 * as supported by PyTorch and Hyper): the smoothed target q_j is weighted by
 * w_j,
 *   loss = -sum_j q_j w_j log softmax_j
 *        = (1-a) w_y (lse - x_y) + (a/V) sum_j w_j (lse - x_j),
 *   grad_j = g (softmax_j ((1-a) w_y + (a/V) sum_k w_k) - q_j w_j). */
static void row_reference_weighted(const double* x, const double* w, int64_t V, int64_t y,
                                   double a, double g, double* loss, double* lse_out,
                                   double* grad) {
    double m = -INFINITY;
    for (int64_t j = 0; j < V; ++j)
        if (x[j] > m) m = x[j];
    double d = 0.0, Sw = 0.0, W = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        d += exp(x[j] - m);
        Sw += w[j] * x[j];
        W += w[j];
    }
    double lse = m + log(d);
    *loss = (1.0 - a) * w[y] * (lse - x[y]) + (a / (double)V) * (W * lse - Sw);
    if (lse_out) *lse_out = lse;
    if (grad) {
        double c = (1.0 - a) * w[y] + (a / (double)V) * W;
        for (int64_t j = 0; j < V; ++j) {
            double q = (j == y ? 1.0 - a : 0.0) + a / (double)V;
            grad[j] = g * (exp(x[j] - lse) * c - q * w[j]);
        }
    }
}

/* ---------------------------------------------------------------------------
 * Vocabulary-split statistics and their combine, the exchange the pages run
 * across vocabulary-parallel ranks [HYPER-269 section 3.1; TENPU-29 section 6,
 * the m_d_Xy gather].  The main oracle path does not use these: they exist so
 * the tests can show that combining the partials of any split reproduces the
 * unsplit row, the invariant a split-vocabulary kernel relies on.
 *   part = {m_k, d_k, S_k, x_y (0 if absent), has_y}
 * ------------------------------------------------------------------------- */
void oracle_chunk_partials(const double* x, int64_t k0, int64_t k1, int64_t y, double* part) {
    double m = -INFINITY;
    for (int64_t j = k0; j < k1; ++j)
        if (x[j] > m) m = x[j];
    double d = 0.0, S = 0.0;
    for (int64_t j = k0; j < k1; ++j) {
        d += exp(x[j] - m);
        S += x[j];
    }
    if (k1 <= k0) d = 0.0; /* empty chunk: m = -inf, d = 0 */
    part[0] = m;
    part[1] = d;
    part[2] = S;
    part[3] = (y >= k0 && y < k1) ? x[y] : 0.0;
    part[4] = (y >= k0 && y < k1) ? 1.0 : 0.0;
}

/* MAX over chunks, then SUM of each d_k rescaled to the global max, then the
 * target logit from whichever chunk holds it. out = {lse, x_y, S}. */
void oracle_combine(const double* parts, int K, double* out) {
    double m = -INFINITY;
    for (int k = 0; k < K; ++k)
        if (parts[5 * k] > m) m = parts[5 * k];
    double d = 0.0, S = 0.0, xy = 0.0;
    for (int k = 0; k < K; ++k) {
        const double* p = parts + 5 * k;
        if (p[1] > 0.0) d += p[1] * exp(p[0] - m);
        S += p[2];
        if (p[4] != 0.0) xy = p[3];
    }
    out[0] = m + log(d);
    out[1] = xy;
    out[2] = S;
}

/* ---------------------------------------------------------------------------
 * The whole pass over a (dim0, dim1, V) logits tensor.
 *
 *   logits      storage of the logits; element (i, j, v) at i*s0 + j*s1 + v
 *   dtype       ORACLE_F32 / ORACLE_BF16 / ORACLE_F16
 *   targets     int64; target of row (i, j) at i*ts0 + j*ts1
 *   a           label smoothing in [0, 1]
 *   reduce      0: loss_out[r] per row;  1: loss_out[0] = mean over kept rows
 *   dloss       reduce: one scalar (upstream gradient of the mean);
 *               otherwise one scale per row; NULL means 1
 *   class_weights  double[V] per-class weights, or NULL (all ones)
 *   loss_out    double[N] or double[1]
 *   lse_out     double[N] or NULL (NaN for rows that are ignored or in error)
 *   grad_out    double[N*V] in flattened row order (r*V + v), or NULL; the
 *               exact gradient before rounding to the storage format
 *   n_out       number of rows whose target is not ignore_idx
 *   err_out     OR of ORACLE_ERR_* bits
 * Returns 0, or -1 when host memory runs out.
 * ------------------------------------------------------------------------- */
int oracle_ce(const void* logits, int dtype, int64_t dim0, int64_t dim1, int64_t V,
              int64_t s0, int64_t s1, const int64_t* targets, int64_t ts0, int64_t ts1,
              double a, int64_t ignore_idx, int reduce, const double* dloss,
              const double* class_weights, double* loss_out, double* lse_out, double* grad_out,
              int64_t* n_out, uint32_t* err_out) {
    const int64_t N = dim0 * dim1;

    /* Ignore mask, count and range check [TENPU-29 section 1, ignore_idx;
     * section 7, n_non_ignore].  With class weights the mean divides by the
     * summed weight of the kept rows' targets instead of their count. */
    int64_t n = 0;
    double wsum = 0.0;
    uint32_t err = 0;
    for (int64_t r = 0; r < N; ++r) {
        int64_t i = r / dim1, j = r % dim1;
        int64_t y = targets[i * ts0 + j * ts1];
        if (y == ignore_idx) continue;
        ++n;
        if (y < 0 || y >= V) err |= ORACLE_ERR_TARGET_RANGE;
        else if (class_weights) wsum += class_weights[y];
    }
    const double denom = class_weights ? wsum : (double)n;

    /* Per-row losses, kept in row order so the mean is summed sequentially. */
    double* row_loss = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!row_loss) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < N; ++r) {
        int64_t i = r / dim1, j = r % dim1;
        int64_t y = targets[i * ts0 + j * ts1];
        double* grow = grad_out ? grad_out + r * V : NULL;
        double loss, lse = NAN;
        if (y == ignore_idx || y < 0 || y >= V) {
            loss = (y == ignore_idx) ? 0.0 : NAN;
            if (grow)
                for (int64_t v = 0; v < V; ++v) grow[v] = 0.0;
        } else {
            /* per-row scale of the gradient */
            double g;
            if (reduce)
                g = (dloss ? dloss[0] : 1.0) / denom;
            else
                g = dloss ? dloss[r] : 1.0;
            double* row = (double*)malloc((size_t)V * sizeof(double));
            for (int64_t v = 0; v < V; ++v)
                row[v] = oracle_decode(logits, dtype, i * s0 + j * s1 + v);
            if (class_weights)
                row_reference_weighted(row, class_weights, V, y, a, g, &loss, &lse, grow);
            else
                row_reference(row, V, y, a, g, &loss, &lse, grow);
            free(row);
        }
        if (lse_out) lse_out[r] = lse;
        row_loss[r] = loss;
    }
    double sum_loss = 0.0;
    for (int64_t r = 0; r < N; ++r) {
        if (!reduce) loss_out[r] = row_loss[r];
        sum_loss += row_loss[r];
    }
    free(row_loss);
    if (reduce) loss_out[0] = sum_loss / denom; /* 0/0 = NaN when all rows are ignored */
    if (n_out) *n_out = n;
    if (err_out) *err_out = err;
    return 0;
}

/* ---------------------------------------------------------------------------
 * lm_head + cross-entropy, the chunked-loss pipeline of the TorchTitan
 * ChunkedLossWrapper that hyper-parallel #269 describes (background: a
 * sequence-chunked lm_head + CE to bound the O(B*L*V) logits memory), in the
 * dataflow of a training step where hidden states, weights, logits and the
 * logits gradient are tensors of the storage dtype:
 *   logits = round_T(hidden . weight^T)          (double sum, one rounding)
 *   loss, dlogits_exact = the cross-entropy pass of oracle_ce on those logits
 *   dlogits = round_T(dlogits_exact)             (the pass writes dtype T)
 *   grad_hidden = dlogits . weight               (double, not rounded)
 *   grad_weight = dlogits^T . hidden             (double, not rounded)
 *   hidden [N][H], weight [V][H] row-major storage of `dtype`; targets [N].
 *   loss_out: N values or 1 (reduce); grad_hidden [N][H], grad_weight [V][H]
 *   doubles, either may be NULL; dlogits_out [N][V] (the rounded logits
 *   gradient) or NULL.
 * Returns 0, or -1 when host memory runs out.
 * ------------------------------------------------------------------------- */
int oracle_linear_ce(const void* hidden, const void* weight, int dtype, int64_t N, int64_t H,
                     int64_t V, const int64_t* targets, double a, int64_t ignore_idx, int reduce,
                     const double* dloss, double* loss_out, double* grad_hidden,
                     double* grad_weight, double* dlogits_out, int64_t* n_out, uint32_t* err_out) {
    /* logits rounded to the storage dtype, stored as that dtype's bits so the
     * pass below reads them exactly as a GPU tensor of that dtype */
    const size_t es = dtype == ORACLE_F32 ? 4 : 2;
    unsigned char* lg = (unsigned char*)malloc((size_t)(N > 0 ? N : 1) * (size_t)V * es);
    double* dl = (double*)malloc((size_t)(N > 0 ? N : 1) * (size_t)V * sizeof(double));
    if (!lg || !dl) {
        free(lg);
        free(dl);
        return -1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        for (int64_t v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h)
                acc += oracle_decode(hidden, dtype, r * H + h) * oracle_decode(weight, dtype, v * H + h);
            uint32_t bits = oracle_encode(acc, dtype);
            if (es == 4)
                memcpy(lg + ((size_t)r * V + v) * 4, &bits, 4);
            else {
                uint16_t b16 = (uint16_t)bits;
                memcpy(lg + ((size_t)r * V + v) * 2, &b16, 2);
            }
        }
    }
    int rc = oracle_ce(lg, dtype, 1, N, V, N * V, V, targets, N, 1, a, ignore_idx, reduce, dloss,
                       NULL, loss_out, NULL, dl, n_out, err_out);
    free(lg);
    if (rc != 0) {
        free(dl);
        return rc;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N * V; ++i) dl[i] = oracle_round(dl[i], dtype);
    if (dlogits_out) memcpy(dlogits_out, dl, (size_t)N * (size_t)V * sizeof(double));
    if (grad_hidden) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < N; ++r)
            for (int64_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int64_t v = 0; v < V; ++v)
                    acc += dl[r * V + v] * oracle_decode(weight, dtype, v * H + h);
                grad_hidden[r * H + h] = acc;
            }
    }
    if (grad_weight) {
#pragma omp parallel for schedule(static)
        for (int64_t v = 0; v < V; ++v)
            for (int64_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int64_t r = 0; r < N; ++r)
                    acc += dl[r * V + v] * oracle_decode(hidden, dtype, r * H + h);
                grad_weight[v * H + h] = acc;
            }
    }
    free(dl);
    return 0;
}

/* Number of OpenMP threads the oracle runs on (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
