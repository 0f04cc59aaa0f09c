/*
 * moe_oracle.c -- plain, slow CPU oracle for the routed MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code with the CUDA path.
 *
 * Sources (page title, section):
 *   [HP41]  "HyperParallel加速DeepSeek-V4.1多模态1M长序列训练",
 *           §2.3 MegaKernel -- MegaGate bullet (score, bias ranking, top-k,
 *           score extraction, normalisation and scaling; separate text and
 *           vision routing bias; fused backward of the normalisation chain;
 *           the projection matmul stays a library GEMM) and MegaMoE bullet
 *           (token dispatch, two expert matmuls, SwiGLU with clamp, result
 *           return); §01 item 5 (native multimodal MoE, separate text/vision
 *           load balance).
 *   [HPF]   "MindSpore HyperParallel一键开箱DeepSeek-V4.1-Flash", §01
 *           (1 shared + 384 routed experts per MoE layer, 6 active).
 *   [TW]    "Twinkle x 昇腾，率先实现Deepseek-V4系列模型高效训练",
 *           "FSDP2-4D并行引擎适配" (TopKRouter returns router logits, routing
 *           weights and selected experts; HashRouter takes ids from
 *           tid2eid[input_ids] and still weights them with the gate logits;
 *           dispatch, local expert compute, return and combine by routing
 *           weight).
 *
 * The pages print no formulas, so every function below is the plain
 * definition of the step they name, in fp64, one token at a time.  Numeric
 * choices the pages leave open (sigmoid scoring, clamp value, routed scaling,
 * the rounding points of the interface) are parameters or are stated at the
 * function.  Parity pins: every function is pinned by the CPU tests against
 * brute force, closed forms, invariants, library routines and finite
 * differences; none is pinned by a number the pages print (they print none).
 *
 * Float tensors (x, W_g, W13, W2, dY) are passed as `const void*` plus one
 * flag `bf`: bf=1 means raw bfloat16 bit patterns (uint16), bf=0 means
 * double.  The conversion of bf16 to double is exact.
 *
 * `exact`=1 turns off every interface rounding (fp32 logits, scores, keys and
 * weights; bf16 intermediate h) so that the chain is a smooth fp64 function
 * for finite-difference checks.  `exact`=0 rounds at the interface points:
 * z, s, key and w to fp32, h to bf16.
 *
 * Weight layouts (row-major):
 *   W_g  [E, d]
 *   W13  [E+1, 2I, d]  rows 0..I-1 = gate projection, I..2I-1 = up projection;
 *                      group E is the shared expert
 *   W2   [E+1, d, I]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ scalars */

static double bf16_to_f64(uint16_t v)
{
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double ld(const void *p, size_t i, int bf)
{
    return bf ? bf16_to_f64(((const uint16_t *)p)[i]) : ((const double *)p)[i];
}

static double dot(const void *a, size_t ia, const void *b, size_t ib, int n, int bf)
{
    double s = 0.0;
    if (bf) {
        const uint16_t *pa = (const uint16_t *)a + ia, *pb = (const uint16_t *)b + ib;
        for (int i = 0; i < n; ++i) s += bf16_to_f64(pa[i]) * bf16_to_f64(pb[i]);
    } else {
        const double *pa = (const double *)a + ia, *pb = (const double *)b + ib;
        for (int i = 0; i < n; ++i) s += pa[i] * pb[i];
    }
    return s;
}

/* Round to the nearest fp32 (ties to even, the C default rounding mode). */
static double r32(double v) { return (double)(float)v; }

/* Round to the nearest bfloat16 value (8 significant bits, ties to even),
 * written from the format's definition: scale so that one unit in the last
 * place is 1, round to the nearest integer, scale back. */
static double rbf16(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    int ex;
    frexp(v, &ex);               /* v = m * 2^ex, 0.5 <= |m| < 1 */
    if (ex < -125) ex = -125;    /* subnormal range keeps the fixed quantum */
    double quantum = ldexp(1.0, ex - 8);
    return nearbyint(v / quantum) * quantum;
}

/* Logistic sigmoid, the score function of the routing step. */
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* silu(a) = a * sigmoid(a) */
static double silu(double a) { return a * sigmoid(a); }

/* d silu / d a = s + a s (1 - s), s = sigmoid(a) */
static double dsilu(double a)
{
    double s = sigmoid(a);
    return s + a * s * (1.0 - s);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------ gate (F1) */

/* z[t,e] = sum_i x[t,i] W_g[e,i] + offset[e]           ([HP41] §2.3 MegaGate:
 * the projection is an ordinary matmul ahead of the routing pipeline).
 * `offset` (nullable) is a per-expert logit shift used by workloads with a
 * prescribed expert-load skew; it has no gradient.  tok (nullable) lists the
 * token rows of x to use; z has one row per listed token. */
void orc_gate_logits(const void *x, const void *Wg, int bf, const float *offset,
                     int n, const int64_t *tok, int d, int E, int exact, double *z)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < n; ++r) {
        int64_t t = tok ? tok[r] : r;
        for (int e = 0; e < E; ++e) {
            double v = dot(x, (size_t)t * d, Wg, (size_t)e * d, d, bf);
            if (offset) v += (double)offset[e];
            z[(size_t)r * E + e] = exact ? v : r32(v);
        }
    }
}

/* ------------------------------------------------------------ route (F2) */

/* Routing of one token ([HP41] §2.3 MegaGate; [TW] FSDP2-4D section).
 *   s_e   = sigmoid(z_e)                                  (score)
 *   key_e = s_e + b[m, e], m = 1 for a vision token else 0 (bias ranking,
 *                                                         per-modality bias)
 *   ids   = the k experts with the largest key, in descending key order,
 *           equal keys ordered by the lower expert id     (top-k)
 *   hash mode: ids = tid2eid[input_id], bias unused       ([TW] HashRouter)
 *   s_j   = s at ids_j (unbiased)                         (score extraction)
 *   w_j   = rho * s_j / sum_i s_i                         (normalise, scale)
 * `margin` = the smallest difference between consecutive keys among the
 * k+1 largest (top-k mode; +inf in hash mode or when k == E): a selection
 * whose margin is tiny can legitimately flip under a last-bit change of z. */
static void route_token(const double *zt, const float *bias, int vis, int mode,
                        const int32_t *table_row, int E, int k, double rho, int exact,
                        int32_t *ids, double *w, double *ssel, double *margin,
                        char *taken)
{
    if (mode == 0) {
        memset(taken, 0, (size_t)E);
        double prev = 0.0;
        *margin = INFINITY;
        int rounds = k < E ? k + 1 : k;
        for (int j = 0; j < rounds; ++j) {
            int best = -1;
            double bk = -INFINITY;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                double s = sigmoid(zt[e]);
                if (!exact) s = r32(s);
                float b = bias[(size_t)vis * E + e];
                /* one fp32 round-to-nearest add of the fp32 score and bias */
                double key = exact ? s + (double)b : (double)((float)s + b);
                if (best < 0 || key > bk) { best = e; bk = key; }  /* strict: lowest id wins ties */
            }
            if (j > 0 && prev - bk < *margin) *margin = prev - bk;
            prev = bk;
            if (j < k) { ids[j] = best; taken[best] = 1; }
        }
    } else {
        for (int j = 0; j < k; ++j) ids[j] = table_row[j];
        *margin = INFINITY;
    }
    double S = 0.0;
    for (int j = 0; j < k; ++j) {
        double s = sigmoid(zt[ids[j]]);
        if (!exact) s = r32(s);
        ssel[j] = s;
        S += s;
    }
    for (int j = 0; j < k; ++j) {
        double v = S > 0.0 ? rho * ssel[j] / S : 0.0;
        w[j] = exact ? v : r32(v);
    }
}

/* Route n tokens given their logits z[n,E].  mode 0 = top-k, 1 = hash.
 * is_vision (nullable = all text) and input_ids are indexed by the token
 * numbers in tok (nullable = 0..n-1).  tid2eid is [vocab, k]. */
void orc_route(const double *z, const float *bias, const uint8_t *is_vision, int mode,
               const int32_t *input_ids, const int32_t *tid2eid, int vocab,
               int n, const int64_t *tok, int E, int k, double rho, int exact,
               int32_t *ids, double *w, double *ssel, double *margin)
{
#pragma omp parallel
    {
        char *taken = (char *)malloc((size_t)E);
#pragma omp for schedule(static)
        for (int r = 0; r < n; ++r) {
            int64_t t = tok ? tok[r] : r;
            int vis = is_vision ? (is_vision[t] != 0) : 0;
            const int32_t *row = NULL;
            if (mode == 1) {
                int32_t id = input_ids[t];
                if (id < 0 || id >= vocab) id = 0;  /* callers validate; keep in bounds */
                row = tid2eid + (size_t)id * k;
            }
            route_token(z + (size_t)r * E, bias, vis, mode, row, E, k, rho, exact,
                        ids + (size_t)r * k, w + (size_t)r * k, ssel + (size_t)r * k,
                        margin + r, taken);
        }
        free(taken);
    }
}

/* --------------------------------------------------------- permute (F3) */

/* Expert-contiguous permutation of the T*k routed slots ([HP41] §2.3 MegaMoE
 * "token dispatch"; [TW] FSDP2-4D: selected experts become global expert ids
 * of one unified dispatch).  Rows are ordered by expert, then token, then slot
 * position -- the plain stable order, built by the plain triple loop.
 *   counts[e]           = number of slots routed to e
 *   offsets[e]          = first row of expert e (offsets[E] = T*k)
 *   row_token[row]      = token of that row
 *   slot_row[t*k + j]   = row that holds slot j of token t */
void orc_permute(const int32_t *ids, int T, int E, int k, int32_t *counts,
                 int32_t *offsets, int32_t *row_token, int32_t *slot_row)
{
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long s = 0; s < (long)T * k; ++s) counts[ids[s]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t row = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (ids[(size_t)t * k + j] == e) {
                    row_token[row] = t;
                    slot_row[(size_t)t * k + j] = row;
                    ++row;
                }
}

/* Expert load per modality ([HP41] §01 item 5, native multimodal MoE: the
 * text and the vision load of the experts are balanced separately).
 *   counts[m*E + e] = number of slots (t, j) with ids[t*k + j] = e whose token
 *                     has modality m = is_vision[t] (0 text, 1 vision;
 *                     is_vision NULL = all text) */
void orc_modality_counts(const int32_t *ids, const uint8_t *is_vision, int T, int E, int k,
                         int32_t *counts)
{
    for (int i = 0; i < 2 * E; ++i) counts[i] = 0;
    for (int t = 0; t < T; ++t) {
        const int m = (is_vision && is_vision[t]) ? 1 : 0;
        for (int j = 0; j < k; ++j) counts[m * E + ids[(size_t)t * k + j]]++;
    }
}

/* ------------------------------------------------------ expert FFN (F4/F5) */

/* One expert on one input row ([HP41] §2.3 MegaMoE: two expert matmuls around
 * SwiGLU with the clamp V4.1 needs):
 *   g = W13[e, 0:I] x,   u = W13[e, I:2I] x
 *   h = silu(min(g, c)) * clamp(u, -c, c)      (h rounded to bf16 unless exact)
 *   o = W2[e] h                                 (length d)
 * Optional outputs g, u, h (length I) and o (length d). */
static void ffn_row(const void *x, size_t xoff, const void *W13, const void *W2, int bf,
                    int e, int d, int I, double c, int exact,
                    double *g, double *u, double *h, double *o)
{
    size_t w13 = (size_t)e * 2 * I * d, w2 = (size_t)e * d * I;
    for (int i = 0; i < I; ++i) {
        double gi = dot(x, xoff, W13, w13 + (size_t)i * d, d, bf);
        double ui = dot(x, xoff, W13, w13 + (size_t)(I + i) * d, d, bf);
        double a = gi < c ? gi : c;
        double b = ui < -c ? -c : (ui > c ? c : ui);
        double hi = silu(a) * b;
        g[i] = gi;
        u[i] = ui;
        h[i] = exact ? hi : rbf16(hi);
    }
    if (o)
        for (int n = 0; n < d; ++n) {
            double acc = 0.0;
            for (int i = 0; i < I; ++i) acc += h[i] * ld(W2, w2 + (size_t)n * I + i, bf);
            o[n] = acc;
        }
}

/* Expert FFN over a list of rows with per-row expert and weight:
 *   y[r] = row_w[r] * W2[e_r] h(x[row_tok[r]])
 * h[r] (length I) is returned as well.  This is the per-expert computation of
 * the dispatched rows, without any layer around it. */
void orc_expert_rows(const void *x, const void *W13, const void *W2, int bf,
                     int n, const int64_t *row_tok, const int32_t *row_exp,
                     const double *row_w, int d, int I, double c, int exact,
                     double *h, double *y)
{
#pragma omp parallel
    {
        double *g = (double *)malloc(sizeof(double) * (size_t)I * 2);
        double *u = g + I;
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r) {
            ffn_row(x, (size_t)row_tok[r] * d, W13, W2, bf, row_exp[r], d, I, c, exact,
                    g, u, h + (size_t)r * I, o);
            double wr = row_w ? row_w[r] : 1.0;
            for (int m = 0; m < d; ++m) y[(size_t)r * d + m] = wr * o[m];
        }
        free(g);
        free(o);
    }
}

/* ------------------------------------------------------- layer forward */

/* Forward of the whole layer for the listed tokens (F1, F2, F4-F6):
 *   y_t = shared(x_t) + sum_j w_j expert_{ids_j}(x_t)
 * ([HPF] §01: one always-on shared expert plus k routed experts; [TW] FSDP2-4D:
 * the expert results come back and are combined by routing weight).  The
 * dispatch permutation (F3) does not change the value of y_t, so it is
 * checked on its own by orc_permute.  Outputs: z[n,E], ids/w/ssel[n,k],
 * margin[n], y[n,d]. */
void orc_layer_forward(const void *x, const void *Wg, const void *W13, const void *W2, int bf,
                       const float *offset, const float *bias, const uint8_t *is_vision,
                       int mode, const int32_t *input_ids, const int32_t *tid2eid, int vocab,
                       int n, const int64_t *tok, int d, int E, int k, int I,
                       double rho, double c, int exact,
                       double *z, int32_t *ids, double *w, double *ssel, double *margin,
                       double *y)
{
    orc_gate_logits(x, Wg, bf, offset, n, tok, d, E, exact, z);
    orc_route(z, bias, is_vision, mode, input_ids, tid2eid, vocab, n, tok, E, k, rho, exact,
              ids, w, ssel, margin);
#pragma omp parallel
    {
        double *g = (double *)malloc(sizeof(double) * (size_t)I * 3);
        double *u = g + I, *h = g + 2 * I;
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r) {
            int64_t t = tok ? tok[r] : r;
            double *yt = y + (size_t)r * d;
            ffn_row(x, (size_t)t * d, W13, W2, bf, E, d, I, c, exact, g, u, h, o);
            for (int m = 0; m < d; ++m) yt[m] = o[m];
            for (int j = 0; j < k; ++j) {
                ffn_row(x, (size_t)t * d, W13, W2, bf, ids[(size_t)r * k + j], d, I, c, exact,
                        g, u, h, o);
                double wj = w[(size_t)r * k + j];
                for (int m = 0; m < d; ++m) yt[m] += wj * o[m];
            }
        }
        free(g);
        free(o);
    }
}

/* ------------------------------------------------------- layer backward */

/* Backward of one expert on one row, for upstream gradient dy (length d) and
 * routing weight wr.  Chain rule of ffn_row, with the clamp gradients passing
 * where the argument equals the bound (torch.clamp convention):
 *   dA = W2[e]^T dy                       (length I)
 *   dw = <h, dA>                          (gradient of the routing weight)
 *   dH = wr dA
 *   dg = dH * clamp(u) * silu'(min(g,c)) * [g <= c]
 *   du = dH * silu(min(g,c)) * [-c <= u <= c]
 *   dx = W13[e, 0:I]^T dg + W13[e, I:2I]^T du   (accumulated into dx)
 * dgu (length 2I, nullable) receives [dg | du]. */
static double ffn_row_backward(const void *x, size_t xoff, const void *dY, size_t dyoff,
                               const void *W13, const void *W2, int bf, int e, int d, int I,
                               double c, int exact, double wr, double *g, double *u,
                               double *h, double *dA, double *dgu, double *dx)
{
    ffn_row(x, xoff, W13, W2, bf, e, d, I, c, exact, g, u, h, NULL);
    size_t w13 = (size_t)e * 2 * I * d, w2 = (size_t)e * d * I;
    for (int i = 0; i < I; ++i) dA[i] = 0.0;
    for (int m = 0; m < d; ++m) {
        double dym = ld(dY, dyoff + m, bf);
        if (dym == 0.0) continue;
        for (int i = 0; i < I; ++i) dA[i] += dym * ld(W2, w2 + (size_t)m * I + i, bf);
    }
    double dw = 0.0;
    for (int i = 0; i < I; ++i) dw += h[i] * dA[i];
    for (int i = 0; i < I; ++i) {
        double dH = wr * dA[i];
        double a = g[i] < c ? g[i] : c;
        double b = u[i] < -c ? -c : (u[i] > c ? c : u[i]);
        double dg = g[i] <= c ? dH * b * dsilu(a) : 0.0;
        double du = (u[i] >= -c && u[i] <= c) ? dH * silu(a) : 0.0;
        if (dgu) { dgu[i] = dg; dgu[I + i] = du; }
        if (dx)
            for (int m = 0; m < d; ++m)
                dx[m] += dg * ld(W13, w13 + (size_t)i * d + m, bf) +
                         du * ld(W13, w13 + (size_t)(I + i) * d + m, bf);
    }
    return dw;
}

/* Backward of the routing weights (the normalisation chain fused by MegaGate,
 * [HP41] §2.3).  With w_j = rho s_j / S, S = sum_i s_i, the Jacobian is
 *   dw_j/ds_m = rho (delta_jm / S - s_j / S^2),
 * so ds_m = sum_j dw_j dw_j/ds_m, and through the sigmoid
 *   dz_m = ds_m s_m (1 - s_m).
 * The bias only ranks, so it receives no gradient; unselected experts get
 * dz = 0.  (s here is the unrounded sigmoid of z.) */
static void route_backward(const double *zt, const int32_t *ids, const double *dw, int k,
                           double rho, double *dz_sel)
{
    double s[64], S = 0.0;
    for (int j = 0; j < k; ++j) { s[j] = sigmoid(zt[ids[j]]); S += s[j]; }
    for (int m = 0; m < k; ++m) {
        double ds = 0.0;
        for (int j = 0; j < k; ++j) {
            double jac = rho * ((j == m ? 1.0 / S : 0.0) - s[j] / (S * S));
            ds += dw[j] * jac;
        }
        dz_sel[m] = ds * s[m] * (1.0 - s[m]);
    }
}

/* Token-local backward of the layer for the listed tokens, given upstream
 * dY[n_tok rows of the full dY, indexed by token].  Outputs per listed token:
 *   dX[n,d]  (through the shared expert, the k routed experts and the gate)
 *   dz[n,E]  (logit gradient; zero off the selection)
 *   dw[n,k]  (routing-weight gradient)
 * Routing (ids, w) is recomputed here from x exactly as the forward does. */
void orc_layer_backward(const void *x, const void *Wg, const void *W13, const void *W2,
                        const void *dY, int bf, const float *offset, const float *bias,
                        const uint8_t *is_vision, int mode, const int32_t *input_ids,
                        const int32_t *tid2eid, int vocab, int n, const int64_t *tok,
                        int d, int E, int k, int I, double rho, double c, int exact,
                        double *dX, double *dz, double *dw)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)n * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)n * k);
    double *w = (double *)malloc(sizeof(double) * (size_t)n * k);
    double *ssel = (double *)malloc(sizeof(double) * (size_t)n * k);
    double *margin = (double *)malloc(sizeof(double) * (size_t)n);
    orc_gate_logits(x, Wg, bf, offset, n, tok, d, E, exact, z);
    orc_route(z, bias, is_vision, mode, input_ids, tid2eid, vocab, n, tok, E, k, rho, exact,
              ids, w, ssel, margin);
#pragma omp parallel
    {
        double *buf = (double *)malloc(sizeof(double) * (size_t)I * 4);
        double *g = buf, *u = buf + I, *h = buf + 2 * I, *dA = buf + 3 * I;
        double dzs[64];
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r) {
            int64_t t = tok ? tok[r] : r;
            double *dxt = dX + (size_t)r * d;
            for (int m = 0; m < d; ++m) dxt[m] = 0.0;
            ffn_row_backward(x, (size_t)t * d, dY, (size_t)t * d, W13, W2, bf, E, d, I, c,
                             exact, 1.0, g, u, h, dA, NULL, dxt);
            for (int j = 0; j < k; ++j)
                dw[(size_t)r * k + j] = ffn_row_backward(
                    x, (size_t)t * d, dY, (size_t)t * d, W13, W2, bf, ids[(size_t)r * k + j],
                    d, I, c, exact, w[(size_t)r * k + j], g, u, h, dA, NULL, dxt);
            route_backward(z + (size_t)r * E, ids + (size_t)r * k, dw + (size_t)r * k, k, rho,
                           dzs);
            double *dzt = dz + (size_t)r * E;
            for (int e = 0; e < E; ++e) dzt[e] = 0.0;
            for (int j = 0; j < k; ++j) dzt[ids[(size_t)r * k + j]] += dzs[j];
            for (int e = 0; e < E; ++e) {
                if (dzt[e] == 0.0) continue;
                for (int m = 0; m < d; ++m) dxt[m] += dzt[e] * ld(Wg, (size_t)e * d + m, bf);
            }
        }
        free(buf);
    }
    free(z); free(ids); free(w); free(ssel); free(margin);
}

/* Rows of the gate weight gradient.  The gate projection z = x W_g^T (+ a
 * constant offset) is an ordinary matmul ([HP41] §2.3 MegaGate), so by the
 * chain rule
 *   dW_g[e, i] = sum_t dz[t, e] x[t, i]
 * over every token t.  Here for the experts rows[0..n_rows) and the n listed
 * tokens (x row tok[r], NULL = tokens 0..n-1), with dz[n, E] given.  One
 * fp64 sum per entry, tokens in order. */
void orc_gate_wgrad_rows(const void *x, int bf, const double *dz, int n, const int64_t *tok,
                         int d, int E, int n_rows, const int32_t *rows, double *out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int j = 0; j < n_rows; ++j)
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int r = 0; r < n; ++r) {
                size_t t = tok ? (size_t)tok[r] : (size_t)r;
                acc += dz[(size_t)r * E + rows[j]] * ld(x, t * d + i, bf);
            }
            out[(size_t)j * d + i] = acc;
        }
}

/* Gradient reaching the SwiGLU output of one expert row, before the routing
 * weight (the first product of the expert backward):
 *   dA[r, i] = sum_m dY[t_r, m] W2[e_r][m, i]          (length I per row)
 * for rows with token row_tok[r] and expert row_exp[r]. */
void orc_rows_dA(const void *dY, const void *W2, int bf, int n, const int64_t *row_tok,
                 const int32_t *row_exp, int d, int I, double *dA)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
        double *out = dA + (size_t)r * I;
        for (int i = 0; i < I; ++i) out[i] = 0.0;
        size_t w2 = (size_t)row_exp[r] * d * I;
        for (int m = 0; m < d; ++m) {
            double y = ld(dY, (size_t)row_tok[r] * d + m, bf);
            if (y == 0.0) continue;
            for (int i = 0; i < I; ++i) out[i] += y * ld(W2, w2 + (size_t)m * I + i, bf);
        }
    }
}

/* Entries of the down-projection weight gradient of one expert from given
 * intermediate rows h (the plain sum, for checking the matmul alone):
 *   out[q] = sum_r dY[t_r, qa[q]] * w_r h[r, qb[q]]
 * with w_r h rounded to bf16 when store_bf16 (h is [n_rows, I]). */
void orc_wgrad2_entries_given_h(const void *dY, const void *h, int bf, int n_rows,
                                const int64_t *row_tok, const double *row_w, int d, int I,
                                int store_bf16, int nq, const int32_t *qa, const int32_t *qb,
                                double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < nq; ++q) {
        double acc = 0.0;
        for (int r = 0; r < n_rows; ++r) {
            double hw = row_w[r] * ld(h, (size_t)r * I + qb[q], bf);
            if (store_bf16) hw = rbf16(hw);
            acc += ld(dY, (size_t)row_tok[r] * d + qa[q], bf) * hw;
        }
        out[q] = acc;
    }
}

/* Weight gradients of one expert e from the rows routed to it:
 *   dW2[e]  = sum_r dy_r (w_r h_r)^T           [d, I]
 *   dW13[e] = sum_r [dg_r | du_r] x_r^T        [2I, d]
 * rows: n_rows rows with token row_tok[r] and weight row_w[r] (the shared
 * expert uses every token with weight 1).  Either output may be NULL.  Full
 * matrices: for experts with few rows only.
 * store_bf16 = 1 rounds the two per-row factors that a bf16 training step
 * stores between its backward matmuls -- [dg | du] and w h -- to bf16 before
 * the sums (the sums themselves stay fp64).  Over thousands of rows these
 * roundings do not average away against a max-abs criterion, so a check of
 * a bf16 implementation compares like with like. */
void orc_expert_wgrad(const void *x, const void *W13, const void *W2, const void *dY, int bf,
                      int e, int n_rows, const int64_t *row_tok, const double *row_w,
                      int d, int I, double c, int exact, int store_bf16, double *dW13,
                      double *dW2)
{
    double *G = (double *)malloc(sizeof(double) * (size_t)n_rows * 2 * I);  /* dgu rows */
    double *H = (double *)malloc(sizeof(double) * (size_t)n_rows * I);      /* w h rows */
#pragma omp parallel
    {
        double *buf = (double *)malloc(sizeof(double) * (size_t)I * 4);
        double *g = buf, *u = buf + I, *h = buf + 2 * I, *dA = buf + 3 * I;
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_rows; ++r) {
            size_t t = (size_t)row_tok[r];
            double *Gr = G + (size_t)r * 2 * I;
            ffn_row_backward(x, t * d, dY, t * d, W13, W2, bf, e, d, I, c, exact, row_w[r],
                             g, u, h, dA, Gr, NULL);
            for (int i = 0; i < I; ++i) {
                double v = row_w[r] * h[i];
                H[(size_t)r * I + i] = store_bf16 ? rbf16(v) : v;
            }
            if (store_bf16)
                for (int i = 0; i < 2 * I; ++i) Gr[i] = rbf16(Gr[i]);
        }
        free(buf);
    }
    if (dW2) {
#pragma omp parallel for schedule(static)
        for (int m = 0; m < d; ++m)
            for (int i = 0; i < I; ++i) {
                double acc = 0.0;
                for (int r = 0; r < n_rows; ++r)
                    acc += ld(dY, (size_t)row_tok[r] * d + m, bf) * H[(size_t)r * I + i];
                dW2[(size_t)m * I + i] = acc;
            }
    }
    if (dW13) {
#pragma omp parallel for schedule(static)
        for (int j = 0; j < 2 * I; ++j)
            for (int m = 0; m < d; ++m) {
                double acc = 0.0;
                for (int r = 0; r < n_rows; ++r)
                    acc += G[(size_t)r * 2 * I + j] * ld(x, (size_t)row_tok[r] * d + m, bf);
                dW13[(size_t)j * d + m] = acc;
            }
    }
    free(G);
    free(H);
}

/* Sampled entries of the same weight gradients (store_bf16 as above), each
 * computed on its own from every row of expert e (for experts with many rows):
 *   dW2[e][n][i]  = sum_r dy_r[n] w_r h_r[i]
 *   dW13[e][j][m] = sum_r dgu_r[j] x_r[m]
 * kind[q] = 0 for a dW2 entry (a = n, b = i), 1 for a dW13 entry (a = j, b = m). */
void orc_expert_wgrad_entries(const void *x, const void *W13, const void *W2, const void *dY,
                              int bf, int e, int n_rows, const int64_t *row_tok,
                              const double *row_w, int d, int I, double c, int exact,
                              int store_bf16, int nq, const int32_t *kind, const int32_t *qa,
                              const int32_t *qb, double *out)
{
    size_t w13 = (size_t)e * 2 * I * d, w2 = (size_t)e * d * I;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < nq; ++q) {
        int i = kind[q] == 0 ? qb[q] : (qa[q] % I);
        double acc = 0.0;
        for (int r = 0; r < n_rows; ++r) {
            size_t t = (size_t)row_tok[r];
            double gi = dot(x, t * d, W13, w13 + (size_t)i * d, d, bf);
            double ui = dot(x, t * d, W13, w13 + (size_t)(I + i) * d, d, bf);
            double a = gi < c ? gi : c;
            double b = ui < -c ? -c : (ui > c ? c : ui);
            double hi = silu(a) * b;
            if (!exact) hi = rbf16(hi);
            if (kind[q] == 0) {
                double hw = row_w[r] * hi;
                if (store_bf16) hw = rbf16(hw);
                acc += ld(dY, t * d + qa[q], bf) * hw;
            } else {
                double dAi = 0.0;
                for (int m = 0; m < d; ++m) dAi += ld(dY, t * d + m, bf) * ld(W2, w2 + (size_t)m * I + i, bf);
                double dH = row_w[r] * dAi;
                double gr = qa[q] < I ? (gi <= c ? dH * b * dsilu(a) : 0.0)
                                      : ((ui >= -c && ui <= c) ? dH * silu(a) : 0.0);
                if (store_bf16) gr = rbf16(gr);
                acc += gr * ld(x, t * d + qb[q], bf);
            }
        }
        out[q] = acc;
    }
}

/* ------------------------------------------------------------- MXFP8 */
/*
 * MXFP8 expert matmuls, the low-precision variant.  The page "DeepSeek-V4昇腾
 * 训练支持：基于 CANN 平台的TorchTitan-NPU + AutoFuse 极简训练优化实践",
 * 性能结果与未来展望 (outlook), names FP8 training on MxFP8 compute as the
 * next step and defines no format, so the format is the published OCP
 * Microscaling Formats (MX) specification v1.0:
 *   - a block is 32 consecutive elements along the contraction dimension;
 *   - the block's shared scale is E8M0: code c stands for 2^(c - 127);
 *   - elements are OCP FP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa
 *     bits, no infinities; largest finite 448 = 1.75 * 2^8, smallest normal
 *     2^-6, subnormal quantum 2^-9; code 0x7F / 0xFF is NaN.
 * Quantisation of one block (the spec's conversion section):
 *   e  = floor(log2(max_i |v_i|)),
 *   X  = 2^(e - 8)       (8 = exponent of E4M3's largest normal), with the
 *                         exponent clamped to the E8M0 range [-127, 127],
 *   p_i = v_i / X rounded to the nearest E4M3 value (ties to even), a
 *         magnitude above 448 saturated to 448; the sign of p_i is that of
 *         v_i (a negative value that rounds to zero gives -0).
 * A block of zeros gets scale code 0 and zero elements.  Readings: the
 * scale is taken from the block's own values (no global amax), elements
 * saturate rather than becoming NaN, and in the expert FFN the intermediate
 * h goes from the SwiGLU straight to MXFP8 (no bf16 step in between).
 *
 * Layouts: a quantised [rows, K] matrix is q [rows, K] (one E4M3 code per
 * byte, row-major) plus sf [rows, sf_pitch] (E8M0 code of block b of row r
 * at sf[r * sf_pitch + b]; sf_pitch >= K / 32).
 */

/* Value of an E4M3 code, from the format's definition. */
static double e4m3_value(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 15, m = c & 7;
    double v;
    if (E == 15 && m == 7) return NAN;
    if (E == 0) v = ldexp((double)m, -9);                   /* m/8 * 2^-6 */
    else v = ldexp(1.0 + m / 8.0, E - 7);
    return s ? -v : v;
}

/* Nearest E4M3 code of y (ties to even), magnitude saturated at 448. */
static uint8_t e4m3_code(double y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    if (a == 0.0) return sign;
    /* spacing of the E4M3 values around a: 2^-9 below the smallest normal,
     * else 2^(exponent - 3) (3 mantissa bits) */
    int ex;
    frexp(a, &ex);                      /* a = f * 2^ex, 0.5 <= f < 1 */
    int e = ex - 1;                     /* floor(log2 a) */
    double quantum = e < -6 ? ldexp(1.0, -9) : ldexp(1.0, e - 3);
    double r = nearbyint(a / quantum) * quantum;   /* ties to even */
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6)) return sign | (uint8_t)(r / ldexp(1.0, -9));
    frexp(r, &ex);
    e = ex - 1;
    int mant = (int)((r / ldexp(1.0, e) - 1.0) * 8.0);
    return sign | (uint8_t)(((e + 7) << 3) | mant);
}

/* E8M0 code of the shared scale of a block of n values. */
static uint8_t e8m0_block_code(const double *v, int n)
{
    double amax = 0.0;
    for (int i = 0; i < n; ++i)
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    if (amax == 0.0) return 0;
    int ex;
    frexp(amax, &ex);
    int se = (ex - 1) - 8;
    if (se < -127) se = -127;
    if (se > 127) se = 127;
    return (uint8_t)(se + 127);
}

static double e8m0_value(uint8_t c) { return ldexp(1.0, (int)c - 127); }

/* Quantise one row of K values (K % 32 == 0) into codes q[K] and scale codes
 * sf[K/32]; dq (nullable) receives the dequantised values. */
static void mx_quantize_row(const double *v, int K, uint8_t *q, uint8_t *sf, double *dq)
{
    for (int b = 0; b < K / 32; ++b) {
        const double *vb = v + 32 * b;
        uint8_t c = e8m0_block_code(vb, 32);
        double X = e8m0_value(c);
        sf[b] = c;
        for (int i = 0; i < 32; ++i) {
            uint8_t p = e4m3_code(vb[i] / X);
            q[32 * b + i] = p;
            if (dq) dq[32 * b + i] = e4m3_value(p) * X;
        }
    }
}

/* MX quantisation of a [rows, K] matrix (bf16 bit patterns when bf = 1, else
 * doubles) into q [rows, K] and sf [rows, sf_pitch]; padding bytes of sf are
 * left untouched. */
void orc_mx_quantize(const void *src, int bf, int rows, int K, int sf_pitch, uint8_t *q,
                     uint8_t *sf)
{
#pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int r = 0; r < rows; ++r) {
            for (int i = 0; i < K; ++i) row[i] = ld(src, (size_t)r * K + i, bf);
            mx_quantize_row(row, K, q + (size_t)r * K, sf + (size_t)r * sf_pitch, NULL);
        }
        free(row);
    }
}

/* Values of a quantised [rows, K] matrix. */
void orc_mx_dequantize(const uint8_t *q, const uint8_t *sf, int rows, int K, int sf_pitch,
                       double *out)
{
    for (int r = 0; r < rows; ++r)
        for (int i = 0; i < K; ++i)
            out[(size_t)r * K + i] =
                e4m3_value(q[(size_t)r * K + i]) * e8m0_value(sf[(size_t)r * sf_pitch + i / 32]);
}

/* Value tables for the pins: E4M3 code -> value (256 entries) and the code
 * of each y[i]. */
void orc_e4m3_decode_all(double *out)
{
    for (int c = 0; c < 256; ++c) out[c] = e4m3_value((uint8_t)c);
}

void orc_e4m3_encode(const double *y, int n, uint8_t *out)
{
    for (int i = 0; i < n; ++i) out[i] = e4m3_code(y[i]);
}

/* MXFP8 expert FFN over a list of rows (the MX form of orc_expert_rows):
 *   x~ = MX(x[row_tok[r]]) along d,  W13~[e] and W2~[e] = MX of each weight
 *   row along its contraction (d for W13, I for W2),
 *   g = W13~[e, 0:I] x~,  u = W13~[e, I:2I] x~   (fp64 sums of exact products)
 *   h = MX(silu(min(g, c)) * clamp(u, -c, c))     along I
 *   y[r] = row_w[r] * W2~[e] h
 * h[r] (length I) returns the dequantised MX h; x and the weights are bf16
 * bit patterns.  Each weight row is quantised on the fly, so the cost is
 * that of the plain FFN plus one quantisation pass per weight row used. */
void orc_expert_rows_mx(const uint16_t *x, const uint16_t *W13, const uint16_t *W2, int n,
                        const int64_t *row_tok, const int32_t *row_exp, const double *row_w,
                        int d, int I, double c, double *h, double *y)
{
#pragma omp parallel
    {
        double *xr = (double *)malloc(sizeof(double) * (size_t)d);
        double *xq = (double *)malloc(sizeof(double) * (size_t)d);
        double *wr = (double *)malloc(sizeof(double) * (size_t)(d > I ? d : I));
        double *wq = (double *)malloc(sizeof(double) * (size_t)(d > I ? d : I));
        double *hv = (double *)malloc(sizeof(double) * (size_t)I);
        uint8_t *qb = (uint8_t *)malloc((size_t)(d > I ? d : I));
        uint8_t *sb = (uint8_t *)malloc((size_t)(d > I ? d : I) / 32);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r) {
            const int e = row_exp[r];
            for (int i = 0; i < d; ++i) xr[i] = bf16_to_f64(x[(size_t)row_tok[r] * d + i]);
            mx_quantize_row(xr, d, qb, sb, xq);
            for (int i = 0; i < I; ++i) {
                double gu[2];
                for (int half = 0; half < 2; ++half) {
                    const uint16_t *w = W13 + ((size_t)e * 2 * I + (size_t)half * I + i) * d;
                    for (int k = 0; k < d; ++k) wr[k] = bf16_to_f64(w[k]);
                    mx_quantize_row(wr, d, qb, sb, wq);
                    double s = 0.0;
                    for (int k = 0; k < d; ++k) s += xq[k] * wq[k];
                    gu[half] = s;
                }
                double a = gu[0] < c ? gu[0] : c;
                double b = gu[1] < -c ? -c : (gu[1] > c ? c : gu[1]);
                hv[i] = silu(a) * b;
            }
            double *hq = h + (size_t)r * I;
            mx_quantize_row(hv, I, qb, sb, hq);
            const double w = row_w ? row_w[r] : 1.0;
            for (int m = 0; m < d; ++m) {
                const uint16_t *w2 = W2 + ((size_t)e * d + m) * I;
                for (int i = 0; i < I; ++i) wr[i] = bf16_to_f64(w2[i]);
                mx_quantize_row(wr, I, qb, sb, wq);
                double s = 0.0;
                for (int i = 0; i < I; ++i) s += hq[i] * wq[i];
                y[(size_t)r * d + m] = w * s;
            }
        }
        free(xr); free(xq); free(wr); free(wq); free(hv); free(qb); free(sb);
    }
}

/* Backward of the MXFP8 expert FFN over a list of rows, in the training form
 * where every matmul takes MXFP8 operands quantised along its own contraction
 * (the forward quantises x and W13 along d and h and W2 along I; the
 * backward's two data-gradient matmuls contract over d and over 2I):
 *   forward, as orc_expert_rows_mx:  g, u from x~ and W13~;  h~ = MX_I(h)
 *   dY~  = MX_d(dY[row_tok[r]])
 *   W2^  = W2[e] quantised along d (each of its I columns as a row of d)
 *   dA   = W2^ dY~                                  (length I)
 *   dw   = <h~, dA>                                 (routing-weight gradient)
 *   dH   = w dA;  dg = dH clamp(u) silu'(min(g,c)) [g <= c];
 *                 du = dH silu(min(g,c)) [-c <= u <= c]
 *   dGU~ = MX_2I([dg | du])
 *   W13^ = W13[e] quantised along 2I (each of its d columns as a row of 2I)
 *   dX   = W13^ dGU~                                (length d)
 * Outputs per row: dw[r], dgu[r] (the [dg | du] before quantisation, length
 * 2I), hq[r] (h~, length I) and dx[r] (length d), all fp64.  The rows are
 * taken expert by expert so that each expert's transposed weights are
 * quantised once.  x, dY and the weights are bf16 bit patterns. */
void orc_expert_rows_mx_backward(const uint16_t *x, const uint16_t *W13, const uint16_t *W2,
                                 const uint16_t *dY, int n, const int64_t *row_tok,
                                 const int32_t *row_exp, const double *row_w, int d, int I,
                                 double c, double *dw, double *dgu, double *hq, double *dx)
{
    int emax = -1;
    for (int r = 0; r < n; ++r) if (row_exp[r] > emax) emax = row_exp[r];
    const int K2 = 2 * I;
    double *w2t = (double *)malloc(sizeof(double) * (size_t)I * d);    /* [I][d] */
    double *w13t = (double *)malloc(sizeof(double) * (size_t)d * K2);  /* [d][2I] */
    for (int e = 0; e <= emax; ++e) {
        int any = 0;
        for (int r = 0; r < n && !any; ++r) any = row_exp[r] == e;
        if (!any) continue;
#pragma omp parallel
        {
            double *col = (double *)malloc(sizeof(double) * (size_t)(d > K2 ? d : K2));
            uint8_t *qb = (uint8_t *)malloc((size_t)(d > K2 ? d : K2));
            uint8_t *sb = (uint8_t *)malloc((size_t)(d > K2 ? d : K2) / 32);
#pragma omp for schedule(static)
            for (int i = 0; i < I; ++i) {
                for (int m = 0; m < d; ++m)
                    col[m] = bf16_to_f64(W2[((size_t)e * d + m) * I + i]);
                mx_quantize_row(col, d, qb, sb, w2t + (size_t)i * d);
            }
#pragma omp for schedule(static)
            for (int m = 0; m < d; ++m) {
                for (int j = 0; j < K2; ++j)
                    col[j] = bf16_to_f64(W13[((size_t)e * K2 + j) * d + m]);
                mx_quantize_row(col, K2, qb, sb, w13t + (size_t)m * K2);
            }
            free(col); free(qb); free(sb);
        }
#pragma omp parallel
        {
            double *xr = (double *)malloc(sizeof(double) * (size_t)d);
            double *xq = (double *)malloc(sizeof(double) * (size_t)d);
            double *wr = (double *)malloc(sizeof(double) * (size_t)d);
            double *wq = (double *)malloc(sizeof(double) * (size_t)d);
            double *g = (double *)malloc(sizeof(double) * (size_t)I);
            double *u = (double *)malloc(sizeof(double) * (size_t)I);
            double *hv = (double *)malloc(sizeof(double) * (size_t)I);
            double *dA = (double *)malloc(sizeof(double) * (size_t)I);
            double *dyq = (double *)malloc(sizeof(double) * (size_t)d);
            double *gq = (double *)malloc(sizeof(double) * (size_t)K2);
            uint8_t *qb = (uint8_t *)malloc((size_t)(d > K2 ? d : K2));
            uint8_t *sb = (uint8_t *)malloc((size_t)(d > K2 ? d : K2) / 32);
#pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < n; ++r) {
                if (row_exp[r] != e) continue;
                const size_t t = (size_t)row_tok[r];
                const double w = row_w ? row_w[r] : 1.0;
                /* forward: g, u from the MX operands, h~ */
                for (int k = 0; k < d; ++k) xr[k] = bf16_to_f64(x[t * d + k]);
                mx_quantize_row(xr, d, qb, sb, xq);
                for (int i = 0; i < I; ++i) {
                    for (int half = 0; half < 2; ++half) {
                        const uint16_t *wrow = W13 + ((size_t)e * K2 + (size_t)half * I + i) * d;
                        for (int k = 0; k < d; ++k) wr[k] = bf16_to_f64(wrow[k]);
                        mx_quantize_row(wr, d, qb, sb, wq);
                        double s = 0.0;
                        for (int k = 0; k < d; ++k) s += xq[k] * wq[k];
                        if (half == 0) g[i] = s; else u[i] = s;
                    }
                    double a = g[i] < c ? g[i] : c;
                    double b = u[i] < -c ? -c : (u[i] > c ? c : u[i]);
                    hv[i] = silu(a) * b;
                }
                double *hr = hq + (size_t)r * I;
                mx_quantize_row(hv, I, qb, sb, hr);
                /* dA = W2^ dY~ */
                for (int k = 0; k < d; ++k) xr[k] = bf16_to_f64(dY[t * d + k]);
                mx_quantize_row(xr, d, qb, sb, dyq);
                for (int i = 0; i < I; ++i) {
                    double s = 0.0;
                    for (int k = 0; k < d; ++k) s += w2t[(size_t)i * d + k] * dyq[k];
                    dA[i] = s;
                }
                double acc = 0.0;
                for (int i = 0; i < I; ++i) acc += hr[i] * dA[i];
                dw[r] = acc;
                /* SwiGLU-clamp backward, then dX = W13^ dGU~ */
                double *gr = dgu + (size_t)r * K2;
                for (int i = 0; i < I; ++i) {
                    const double dH = w * dA[i];
                    const double a = g[i] < c ? g[i] : c;
                    const double b = u[i] < -c ? -c : (u[i] > c ? c : u[i]);
                    gr[i] = g[i] <= c ? dH * b * dsilu(a) : 0.0;
                    gr[I + i] = (u[i] >= -c && u[i] <= c) ? dH * silu(a) : 0.0;
                }
                mx_quantize_row(gr, K2, qb, sb, gq);
                double *xo = dx + (size_t)r * d;
                for (int m = 0; m < d; ++m) {
                    double s = 0.0;
                    for (int j = 0; j < K2; ++j) s += w13t[(size_t)m * K2 + j] * gq[j];
                    xo[m] = s;
                }
            }
            free(xr); free(xq); free(wr); free(wq); free(g); free(u); free(hv); free(dA);
            free(dyq); free(gq); free(qb); free(sb);
        }
    }
    free(w2t);
    free(w13t);
}

/* Token-local backward of the layer with the MXFP8 expert matmuls, for the
 * listed tokens: the routing and its backward chain are those of
 * orc_layer_backward (interface rounding on, exact = 0), the expert rows those
 * of orc_expert_rows_mx_backward.  Per listed token t with routed experts
 * ids_j and weights w_j:
 *   rows    (t, shared expert, 1) and (t, ids_j, w_j)
 *   dw[j]   = the row (t, ids_j)'s <h~, dA>
 *   dz      = route_backward(dw)            (zero off the selection)
 *   dX[t]   = sum over the token's k + 1 rows of their dx + sum_e dz_e W_g[e]
 * bf16 inputs only (uint16 bit patterns). */
void orc_layer_backward_mx(const uint16_t *x, const uint16_t *Wg, const uint16_t *W13,
                           const uint16_t *W2, const uint16_t *dY, const float *offset,
                           const float *bias, const uint8_t *is_vision, int mode,
                           const int32_t *input_ids, const int32_t *tid2eid, int vocab, int n,
                           const int64_t *tok, int d, int E, int k, int I, double rho, double c,
                           double *dX, double *dz, double *dw)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)n * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)n * k);
    double *w = (double *)malloc(sizeof(double) * (size_t)n * k);
    double *ssel = (double *)malloc(sizeof(double) * (size_t)n * k);
    double *margin = (double *)malloc(sizeof(double) * (size_t)n);
    orc_gate_logits(x, Wg, 1, offset, n, tok, d, E, 0, z);
    orc_route(z, bias, is_vision, mode, input_ids, tid2eid, vocab, n, tok, E, k, rho, 0, ids, w,
              ssel, margin);
    /* the token's rows: slot 0 the shared expert, slots 1..k the routed ones */
    const int nr = n * (k + 1);
    int64_t *rt = (int64_t *)malloc(sizeof(int64_t) * (size_t)nr);
    int32_t *re = (int32_t *)malloc(sizeof(int32_t) * (size_t)nr);
    double *rw = (double *)malloc(sizeof(double) * (size_t)nr);
    for (int r = 0; r < n; ++r) {
        const int64_t t = tok ? tok[r] : r;
        for (int j = 0; j <= k; ++j) {
            const size_t i = (size_t)r * (k + 1) + j;
            rt[i] = t;
            re[i] = j == 0 ? E : ids[(size_t)r * k + j - 1];
            rw[i] = j == 0 ? 1.0 : w[(size_t)r * k + j - 1];
        }
    }
    double *dwr = (double *)malloc(sizeof(double) * (size_t)nr);
    double *dgu = (double *)malloc(sizeof(double) * (size_t)nr * 2 * I);
    double *hq = (double *)malloc(sizeof(double) * (size_t)nr * I);
    double *dxr = (double *)malloc(sizeof(double) * (size_t)nr * d);
    orc_expert_rows_mx_backward(x, W13, W2, dY, nr, rt, re, rw, d, I, c, dwr, dgu, hq, dxr);
    for (int r = 0; r < n; ++r) {
        double *dxt = dX + (size_t)r * d;
        for (int m = 0; m < d; ++m) dxt[m] = 0.0;
        for (int j = 0; j <= k; ++j) {
            const double *src = dxr + ((size_t)r * (k + 1) + j) * d;
            for (int m = 0; m < d; ++m) dxt[m] += src[m];
        }
        for (int j = 0; j < k; ++j) dw[(size_t)r * k + j] = dwr[(size_t)r * (k + 1) + j + 1];
        double dzs[64];
        route_backward(z + (size_t)r * E, ids + (size_t)r * k, dw + (size_t)r * k, k, rho, dzs);
        double *dzt = dz + (size_t)r * E;
        for (int e = 0; e < E; ++e) dzt[e] = 0.0;
        for (int j = 0; j < k; ++j) dzt[ids[(size_t)r * k + j]] += dzs[j];
        for (int e = 0; e < E; ++e) {
            if (dzt[e] == 0.0) continue;
            for (int m = 0; m < d; ++m) dxt[m] += dzt[e] * bf16_to_f64(Wg[(size_t)e * d + m]);
        }
    }
    free(z); free(ids); free(w); free(ssel); free(margin);
    free(rt); free(re); free(rw); free(dwr); free(dgu); free(hq); free(dxr);
}

/* A^T B with both operands MX-quantised along their rows (the contraction):
 * A [K, M] and B [K, N] (doubles, row-major); rows are taken in blocks of 32
 * from row 0, the last block zero-padded; every column of a block is one MX
 * block (one scale), in A and in B alike.  out [M, N] = sum over blocks of
 * q(A_block)^T q(B_block), accumulated in fp64.  This is the weight-gradient
 * matmul of the MX training form, where the contraction runs over an
 * expert's token rows. */
void orc_mx_rows_matmul(const double *A, const double *B, int K, int M, int N, double *out)
{
    for (size_t i = 0; i < (size_t)M * N; ++i) out[i] = 0.0;
    const int nb = (K + 31) / 32;
    double *qa = (double *)malloc(sizeof(double) * (size_t)32 * M);
    double *qb = (double *)malloc(sizeof(double) * (size_t)32 * N);
    for (int b = 0; b < nb; ++b) {
#pragma omp parallel
        {
            double col[32], dq[32];
            uint8_t q[32], sf[1];
#pragma omp for schedule(static)
            for (int m = 0; m < M; ++m) {
                for (int j = 0; j < 32; ++j) {
                    const int r = 32 * b + j;
                    col[j] = r < K ? A[(size_t)r * M + m] : 0.0;
                }
                mx_quantize_row(col, 32, q, sf, dq);
                for (int j = 0; j < 32; ++j) qa[(size_t)j * M + m] = dq[j];
            }
#pragma omp for schedule(static)
            for (int n = 0; n < N; ++n) {
                for (int j = 0; j < 32; ++j) {
                    const int r = 32 * b + j;
                    col[j] = r < K ? B[(size_t)r * N + n] : 0.0;
                }
                mx_quantize_row(col, 32, q, sf, dq);
                for (int j = 0; j < 32; ++j) qb[(size_t)j * N + n] = dq[j];
            }
#pragma omp for schedule(static)
            for (int m = 0; m < M; ++m) {
                double *o = out + (size_t)m * N;
                for (int j = 0; j < 32; ++j) {
                    const double a = qa[(size_t)j * M + m];
                    if (a == 0.0) continue;
                    const double *bq = qb + (size_t)j * N;
                    for (int n = 0; n < N; ++n) o[n] += a * bq[n];
                }
            }
        }
    }
    free(qa);
    free(qb);
}

/* Weight gradients of one expert in the MX training form, over its rows in
 * the given order (the permuted order of its group): with h~, [dg|du] and
 * the routing weights w of orc_expert_rows_mx_backward,
 *   dW2  [d, I]  = mx_rows_matmul(dY rows, bf16(w h~))
 *   dW13 [2I, d] = mx_rows_matmul(bf16([dg|du]), x rows)
 * w h~ and [dg|du] are stored in bf16 before their quantisation, the
 * interface rounding point of the layer's weight-gradient operands (as in
 * orc_expert_wgrad's store_bf16 mode).  W13 [2I, d] and W2 [d, I] are the
 * expert's weights (bf16). */
void orc_expert_wgrad_mx(const uint16_t *x, const uint16_t *W13, const uint16_t *W2,
                         const uint16_t *dY, int n, const int64_t *row_tok, const double *row_w,
                         int d, int I, double c, double *dW13, double *dW2)
{
    const int K2 = 2 * I;
    int32_t *re = (int32_t *)calloc((size_t)(n > 0 ? n : 1), sizeof(int32_t));
    double *dw = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *dgu = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * K2);
    double *h = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * I);
    double *dx = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    double *xr = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    double *dyr = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    if (n > 0)
        orc_expert_rows_mx_backward(x, W13, W2, dY, n, row_tok, re, row_w, d, I, c, dw, dgu, h,
                                    dx);
    for (int r = 0; r < n; ++r) {
        const double w = row_w ? row_w[r] : 1.0;
        for (int i = 0; i < I; ++i) h[(size_t)r * I + i] = rbf16(w * h[(size_t)r * I + i]);
        for (int j = 0; j < K2; ++j) dgu[(size_t)r * K2 + j] = rbf16(dgu[(size_t)r * K2 + j]);
        for (int m = 0; m < d; ++m) {
            xr[(size_t)r * d + m] = bf16_to_f64(x[(size_t)row_tok[r] * d + m]);
            dyr[(size_t)r * d + m] = bf16_to_f64(dY[(size_t)row_tok[r] * d + m]);
        }
    }
    orc_mx_rows_matmul(dyr, h, n, d, I, dW2);
    orc_mx_rows_matmul(dgu, xr, n, K2, d, dW13);
    free(re); free(dw); free(dgu); free(h); free(dx); free(xr); free(dyr);
}
