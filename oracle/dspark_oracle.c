/*
 * CPU oracle for the DSpark per-step hot path.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the benchmark's
 * CPU-baseline / reference leg load this library.  The CUDA path never calls it and
 * shares no source, header, table or helper with it.
 *
 * It is the plain, slow, obviously correct statement of what one speculative step
 * computes, in fp64 from the fp32 / bf16 inputs, following the pages in their order:
 *
 *   draft       billytse.dev DSpark page, section 3.2 ("Sequential head": the
 *               semi-autoregressive block distribution p_k = softmax(U_k + B_k)) and
 *               section 3.3 ("Markov head": B(x_{k-1}, .) = W1[x_{k-1}] W2, the
 *               left-to-right loop prev = anchor; bias; softmax; sample; prev = token).
 *               Sampling is Gumbel-max.
 *   confidence  weigao.cc DSpark-vs-MTP page, "3. confidence head" (c_k is one linear
 *               layer on [h_k ; markov_embedding(prev)] followed by a sigmoid) and
 *               billytse.dev section 5 (a_j = prod_{i<=j} c_i).
 *   schedule    billytse.dev section 6 (B = sum_r (1 + l_r), tau = sum_r (1 + sum_{j<=l_r}
 *               a_{r,j}), maximise Theta = tau * SPS(B) by adding positions in descending
 *               order of expected return and stopping as soon as Theta stops rising) and
 *               section 7 (early stopping keeps the rule non-anticipating).
 *   verify      billytse.dev section 1 (accept x_k with probability min(1, p/q), stop at
 *               the first reject and draw the correction from the residual) and the
 *               xhh.club DSpark page, Q&A on the acceptance rule (residual norm(max(0,
 *               p - q))).
 *   variants    greedy drafting (billytse.dev section 11, the serving example's draft
 *               sampling method) with its point-mass proposal in verification; the
 *               asynchronous two-step capacity scheduler (weigao.cc "4. hardware-aware
 *               prefix scheduler"; billytse.dev section 7); fixed confidence-threshold
 *               truncation (billytse.dev section 8; xhh.club page on load-dependent
 *               thresholds); the RNN head (weigao.cc "2. Markov head and RNN head").
 *
 * Readings where the pages are silent (the same list is kept with the design notes):
 *   - Random numbers: Philox4x32 with 7 rounds (Salmon, Moraes, Dror, Shaw, "Parallel
 *     Random Numbers: As Easy as 1, 2, 3", SC'11: the Philox4x32 round function; 7 is the
 *     fewest rounds that paper reports passing TestU01 BigCrush, its default being 10),
 *     key = (seed low 32 bits, seed high 32 bits),
 *     counter = (floor(v/4), k, b, stream), the draw is output word v mod 4.  Positions k
 *     are 1-based, requests b 0-based.  Streams: 0 draft Gumbel, 1 verify uniform (v = 0),
 *     2 residual Gumbel, 3 bonus Gumbel.
 *   - U01(x) = ((x >> 9) + 1/2) * 2^-23, exactly representable, strictly inside (0, 1).
 *     w = 1 - U01(x) is formed exactly from the complemented bits and the Gumbel value is
 *     g = -log(-log1p(-w)).
 *   - Gumbel-max: x = argmax_v (z_v + g_v); ties go to the smallest v.
 *   - Scheduler: a is clamped to [0, 1] (NaN -> 0) and taken in fixed point
 *     A = floor(a * 2^32 + 1/2); items are sorted by (A desc, r asc, j asc); sums are
 *     exact integers; Theta_n = double(R * 2^32 + S_n) * double(sps[R + n]) is compared
 *     with Theta_{n-1} as a plain double product; the first non-rise stops.
 *   - Verify: the bonus row is target row l + 1; the residual draw is Gumbel-max over
 *     log(P - Q) restricted to P > Q; if that set is empty, Gumbel-max over log P with
 *     the same stream (counted as a fallback).
 *   - Greedy draft: x_k = argmax z_k, ties to the smallest v; the proposal is the point
 *     mass at x_k (q = 1), so verification accepts with probability p(x_k) and the
 *     residual is p without x_k.
 *   - Two-step scheduler: K for step t is the early-stop count of step t - 2; the steps
 *     without such history use their own count; the K admitted items are the first K in
 *     the scheduler's order (a desc, r asc, j asc).
 *   - Threshold truncation: l_r is the leading run of positions with a[r, j] > threshold
 *     (strict, like the marginal rule of the adaptive scheduler).
 *   - RNN head: state of r entries, token embedding = W1 row, gate = sigmoid, candidate =
 *     tanh, s_0 = 0, one linear layer W_rnn [2r + H, 3r] (+ b_rnn) on [s; W1[prev]; h_k]
 *     with column blocks (gate, candidate, output), E_k = tanh(output) unrounded.
 *
 * Parity pins live in tests/test_oracle_*.py.  Every function here is pinned there.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define DSO_OK 0
#define DSO_ERR_ARG 1
#define DSO_ERR_NOMEM 2
#define DSO_PHILOX_ROUNDS 7   /* rounds of the generator every draw uses */

/* ------------------------------------------------------------------------------------ */
/* Counter-based random numbers                                                          */
/* ------------------------------------------------------------------------------------ */

/* Philox4x32 with R rounds: each round multiplies counter words 0 and 2 by the two
 * round constants, swaps and mixes the high halves with the other counter words and the
 * key; the key is advanced by the two Weyl constants between rounds. */
void dso_philox4x32(const uint32_t ctr[4], uint64_t seed, int rounds, uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFu), k1 = (uint32_t)(seed >> 32);
    for (int round = 0; round < rounds; ++round) {
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(prod1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)prod1;
        uint32_t n2 = (uint32_t)(prod0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)prod0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit draw for vocabulary index v of (request b, position k, stream). */
uint32_t dso_draw(uint64_t seed, int b, int k, int v, int stream)
{
    uint32_t ctr[4] = {(uint32_t)v / 4u, (uint32_t)k, (uint32_t)b, (uint32_t)stream};
    uint32_t out[4];
    dso_philox4x32(ctr, seed, DSO_PHILOX_ROUNDS, out);
    return out[(uint32_t)v % 4u];
}

double dso_u01(uint32_t x)
{
    return ((double)(x >> 9) + 0.5) * (1.0 / 8388608.0);
}

/* 1 - U01(x), formed exactly from the complemented top 23 bits. */
double dso_one_minus_u01(uint32_t x)
{
    return ((double)((~x) >> 9 & 0x7FFFFFu) + 0.5) * (1.0 / 8388608.0);
}

/* Standard Gumbel variate g = -log(E) with E = -log(u) an Exp(1) variate. */
double dso_gumbel(uint32_t x)
{
    double w = dso_one_minus_u01(x);
    double E = -log1p(-w);
    return -log(E);
}

static double bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------------------ */
/* Draft: Markov bias, softmax, Gumbel-max                                               */
/* ------------------------------------------------------------------------------------ */

/* z_v = U[k][v] + sum_i e[i] * W2[i][v], all in double; e is the head's output row
 * (W1[prev] for the Markov head, tanh(output) for the RNN head). */
static void draft_logits(const float *U_row, const double *erow, const uint16_t *W2,
                         int V, int r, double *z)
{
    for (int v = 0; v < V; ++v) z[v] = 0.0;
    for (int i = 0; i < r; ++i) {
        double e = erow[i];
        const uint16_t *w2 = W2 + (size_t)i * V;
        for (int v = 0; v < V; ++v) z[v] += e * bf16_to_double(w2[v]);
    }
    for (int v = 0; v < V; ++v) z[v] += (double)U_row[v];
}

/* the bf16 row W1[prev] in double */
static void markov_row(const uint16_t *W1, int prev, int r, double *e)
{
    for (int i = 0; i < r; ++i) e[i] = bf16_to_double(W1[(size_t)prev * r + i]);
}

static void softmax_stats(const double *z, int V, double *m_out, double *s_out)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) if (z[v] > m) m = z[v];
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp(z[v] - m);
    *m_out = m;
    *s_out = s;
}

/* argmax_v (score_v + g_v) over the v with mask[v] != 0 (mask NULL: all v); ties to the
 * smallest v.  Returns -1 when no v is eligible.  *gap = best - second best score. */
static int gumbel_argmax(const double *score, const unsigned char *mask, int V,
                         uint64_t seed, int b, int k, int stream, double *gap)
{
    int best = -1;
    double b1 = -INFINITY, b2 = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (mask && !mask[v]) continue;
        double s = score[v] + dso_gumbel(dso_draw(seed, b, k, v, stream));
        if (best < 0 || s > b1) {
            b2 = b1;
            b1 = s;
            best = v;
        } else if (s > b2) {
            b2 = s;
        }
    }
    *gap = b1 - b2;
    return best;
}

/*
 * U       [n_req, gamma, V]  base logits of the requests in req_ids
 * W1      [V, r] bf16, W2 [r, V] bf16
 * anchor  [n_req]            last committed token
 * req_ids [n_req]            request index b used by the random counter
 * outputs [n_req, gamma]:    tokens, q_tok = q_k(x_k), row_max, row_sumexp, gap (top-two
 *                            Gumbel score gap of the draw, for the tie band)
 */
int dso_draft(const float *U, const uint16_t *W1, const uint16_t *W2, const int32_t *anchor,
              const int32_t *req_ids, int n_req, int gamma, int V, int r, uint64_t seed,
              int32_t *tokens, double *q_tok, double *row_max, double *row_sumexp,
              double *gap, int nthreads)
{
    if (n_req < 0 || gamma < 1 || V < 1 || r < 1) return DSO_ERR_ARG;
    int err = DSO_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int i = 0; i < n_req; ++i) {
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
        double *e = (double *)malloc(sizeof(double) * (size_t)r);
        if (!z || !e) { free(z); free(e); err = DSO_ERR_NOMEM; continue; }
        int b = req_ids[i];
        int prev = anchor[i];
        for (int k = 1; k <= gamma; ++k) {
            size_t o = (size_t)i * gamma + (k - 1);
            if (prev < 0 || prev >= V) { err = DSO_ERR_ARG; break; }
            markov_row(W1, prev, r, e);
            draft_logits(U + o * V, e, W2, V, r, z);
            double m, s;
            softmax_stats(z, V, &m, &s);
            double g;
            int x = gumbel_argmax(z, NULL, V, seed, b, k, 0, &g);
            tokens[o] = x;
            q_tok[o] = exp(z[x] - m) / s;
            row_max[o] = m;
            row_sumexp[o] = s;
            gap[o] = g;
            prev = x;
        }
        free(z);
        free(e);
    }
    return err;
}

/*
 * Greedy draft (billytse.dev DSpark page, section 11: the serving example selects the
 * greedy draft sampling method): the same loop as dso_draft with x_k = argmax_v z_v, ties
 * to the smallest v.  The proposal is then the point mass at x_k, so q_tok = 1; row_max
 * and row_sumexp are still the softmax statistics of z, and gap is the top-two logit gap
 * (the tie band of this draw).  No random numbers are used.
 */
int dso_draft_greedy(const float *U, const uint16_t *W1, const uint16_t *W2,
                     const int32_t *anchor, int n_req, int gamma, int V, int r, int32_t *tokens,
                     double *q_tok, double *row_max, double *row_sumexp, double *gap,
                     int nthreads)
{
    if (n_req < 0 || gamma < 1 || V < 1 || r < 1) return DSO_ERR_ARG;
    int err = DSO_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int i = 0; i < n_req; ++i) {
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
        double *e = (double *)malloc(sizeof(double) * (size_t)r);
        if (!z || !e) { free(z); free(e); err = DSO_ERR_NOMEM; continue; }
        int prev = anchor[i];
        for (int k = 1; k <= gamma; ++k) {
            size_t o = (size_t)i * gamma + (k - 1);
            if (prev < 0 || prev >= V) { err = DSO_ERR_ARG; break; }
            markov_row(W1, prev, r, e);
            draft_logits(U + o * V, e, W2, V, r, z);
            double m, s;
            softmax_stats(z, V, &m, &s);
            int x = 0;
            double second = -INFINITY;
            for (int v = 1; v < V; ++v) {
                if (z[v] > z[x]) {
                    second = z[x];
                    x = v;
                } else if (z[v] > second) {
                    second = z[v];
                }
            }
            tokens[o] = x;
            q_tok[o] = 1.0;
            row_max[o] = m;
            row_sumexp[o] = s;
            gap[o] = z[x] - second;
            prev = x;
        }
        free(z);
        free(e);
    }
    return err;
}

/* Markov bias alone: out[i][v] = sum_k W1[prev_i][k] * W2[k][v] in double
 * (prev_i = -1 gives a zero row). */
int dso_markov_bias(const uint16_t *W1, const uint16_t *W2, const int32_t *prev, int n, int V,
                    int r, double *out)
{
    for (int i = 0; i < n; ++i) {
        double *o = out + (size_t)i * V;
        for (int v = 0; v < V; ++v) o[v] = 0.0;
        if (prev[i] == -1) continue;
        if (prev[i] < 0 || prev[i] >= V) return DSO_ERR_ARG;
        for (int k = 0; k < r; ++k) {
            double e = bf16_to_double(W1[(size_t)prev[i] * r + k]);
            for (int v = 0; v < V; ++v) o[v] += e * bf16_to_double(W2[(size_t)k * V + v]);
        }
    }
    return DSO_OK;
}

/* ------------------------------------------------------------------------------------ */
/* RNN head                                                                              */
/* ------------------------------------------------------------------------------------ */

/*
 * The hidden-state block of the RNN head's linear layer (weigao.cc DSpark-vs-MTP page,
 * "2. Markov head and RNN head": one linear layer on [state; previous-token embedding;
 * hidden state]; this block does not depend on the drafted tokens):
 *   hp[i][c] = b_rnn[c] + sum_j h[i][j] * W_rnn[2r + j][c],   c < 3r
 * h [n, H] fp32, W_rnn [2r + H, 3r] bf16, b_rnn [3r] fp32 -> hp [n, 3r] double.
 */
int dso_rnn_project(const float *h, const uint16_t *W_rnn, const float *b_rnn, int n, int H,
                    int r, double *hp)
{
    if (n < 0 || H < 0 || r < 1) return DSO_ERR_ARG;
    const int C = 3 * r;
    for (int i = 0; i < n; ++i) {
        double *o = hp + (size_t)i * C;
        for (int c = 0; c < C; ++c) o[c] = (double)b_rnn[c];
        for (int j = 0; j < H; ++j) {
            double hv = (double)h[(size_t)i * H + j];
            const uint16_t *w = W_rnn + (size_t)(2 * r + j) * C;
            for (int c = 0; c < C; ++c) o[c] += hv * bf16_to_double(w[c]);
        }
    }
    return DSO_OK;
}

/*
 * Draft with the RNN head (weigao.cc page, "2. Markov head and RNN head"; billytse.dev
 * section 3.3 names it as the head that remembers the whole block prefix).  For k = 1..gamma:
 *   y = [s_{k-1}; W1[x_{k-1}]; h_k] W_rnn + b_rnn          (3r values; x_0 = the anchor)
 *   gate = sigmoid(y[0:r]), cand = tanh(y[r:2r]), out = y[2r:3r]
 *   s_k = gate * s_{k-1} + (1 - gate) * cand,  s_0 = 0
 *   E_k = tanh(out),  z = U_k + E_k W2,  x_k drawn from softmax(z) as in dso_draft
 *   (greedy = 1: x_k = argmax z as in dso_draft_greedy, q_tok = 1).
 * Readings: the state has r entries (W2 [r, V] projects tanh(output)); the token embedding
 * is the head's W1 row; gate = sigmoid and candidate = tanh of their blocks; s_0 = 0; the
 * head computes in the precision of the rest of the path (no rounding of E).
 * Outputs as dso_draft / dso_draft_greedy, plus E [n, gamma, r] (the projected rows) and
 * state [n, r] (s_gamma).
 */
int dso_draft_rnn(const float *U, const float *h, const uint16_t *W1, const uint16_t *W2,
                  const uint16_t *W_rnn, const float *b_rnn, const int32_t *anchor,
                  const int32_t *req_ids, int n_req, int gamma, int V, int r, int H,
                  uint64_t seed, int greedy, int32_t *tokens, double *q_tok, double *row_max,
                  double *row_sumexp, double *gap, double *E, double *state, int nthreads)
{
    if (n_req < 0 || gamma < 1 || V < 1 || r < 1 || H < 0) return DSO_ERR_ARG;
    const int C = 3 * r;
    int err = DSO_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int i = 0; i < n_req; ++i) {
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
        double *y = (double *)malloc(sizeof(double) * (size_t)C);
        double *st = (double *)calloc((size_t)r, sizeof(double));
        if (!z || !y || !st) { free(z); free(y); free(st); err = DSO_ERR_NOMEM; continue; }
        int b = req_ids[i];
        int prev = anchor[i];
        for (int k = 1; k <= gamma; ++k) {
            size_t o = (size_t)i * gamma + (k - 1);
            if (prev < 0 || prev >= V) { err = DSO_ERR_ARG; break; }
            /* the linear layer on [s_{k-1}; W1[prev]; h_k] */
            dso_rnn_project(h + o * H, W_rnn, b_rnn, 1, H, r, y);
            for (int j = 0; j < r; ++j) {
                const uint16_t *ws = W_rnn + (size_t)j * C;
                const uint16_t *we = W_rnn + (size_t)(r + j) * C;
                double sv = st[j];
                double ev = bf16_to_double(W1[(size_t)prev * r + j]);
                for (int c = 0; c < C; ++c)
                    y[c] += sv * bf16_to_double(ws[c]) + ev * bf16_to_double(we[c]);
            }
            double *Erow = E + o * (size_t)r;
            for (int j = 0; j < r; ++j) {
                double gate = 1.0 / (1.0 + exp(-y[j]));
                double cand = tanh(y[r + j]);
                st[j] = gate * st[j] + (1.0 - gate) * cand;
                Erow[j] = tanh(y[2 * r + j]);
            }
            draft_logits(U + o * V, Erow, W2, V, r, z);
            double m, s;
            softmax_stats(z, V, &m, &s);
            int x;
            double g;
            if (greedy) {
                x = 0;
                double second = -INFINITY;
                for (int v = 1; v < V; ++v) {
                    if (z[v] > z[x]) { second = z[x]; x = v; }
                    else if (z[v] > second) second = z[v];
                }
                g = z[x] - second;
                q_tok[o] = 1.0;
            } else {
                x = gumbel_argmax(z, NULL, V, seed, b, k, 0, &g);
                q_tok[o] = exp(z[x] - m) / s;
            }
            tokens[o] = x;
            row_max[o] = m;
            row_sumexp[o] = s;
            gap[o] = g;
            prev = x;
        }
        for (int j = 0; j < r; ++j) state[(size_t)i * r + j] = st[j];
        free(z); free(y); free(st);
    }
    return err;
}

/* ------------------------------------------------------------------------------------ */
/* Confidence head and survival                                                          */
/* ------------------------------------------------------------------------------------ */

/*
 * c[b,k] = sigmoid( sum_j w_c[j] h[b,k,j] + sum_i w_c[H+i] W1[prev,i] + b_c ),
 * prev = anchor[b] for k = 1, tokens[b,k-1] otherwise;  a[b,k] = prod_{i<=k} c[b,i].
 */
int dso_confidence(const float *h, const int32_t *anchor, const int32_t *tokens,
                   const uint16_t *W1, const float *w_c, float b_c, int n_req, int gamma,
                   int H, int r, int V, double *c, double *a)
{
    if (n_req < 0 || gamma < 1 || H < 0 || r < 1) return DSO_ERR_ARG;
    for (int i = 0; i < n_req; ++i) {
        double surv = 1.0;
        for (int k = 1; k <= gamma; ++k) {
            size_t o = (size_t)i * gamma + (k - 1);
            int prev = (k == 1) ? anchor[i] : tokens[o - 1];
            if (prev < 0 || prev >= V) return DSO_ERR_ARG;
            double acc = (double)b_c;
            for (int j = 0; j < H; ++j) acc += (double)w_c[j] * (double)h[o * H + j];
            for (int j = 0; j < r; ++j)
                acc += (double)w_c[H + j] * bf16_to_double(W1[(size_t)prev * r + j]);
            double ck = 1.0 / (1.0 + exp(-acc));
            surv *= ck;
            c[o] = ck;
            a[o] = surv;
        }
    }
    return DSO_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Hardware-aware prefix scheduler                                                       */
/* ------------------------------------------------------------------------------------ */

typedef struct { int64_t A; int r; int j; } sched_item;

static int item_before(const sched_item *x, const sched_item *y)
{
    if (x->A != y->A) return x->A > y->A;
    if (x->r != y->r) return x->r < y->r;
    return x->j < y->j;
}

static int64_t fixed_point_a(float a)
{
    double x = (double)a;
    if (!(x > 0.0)) return 0;          /* also NaN */
    if (x > 1.0) x = 1.0;
    return (int64_t)floor(x * 4294967296.0 + 0.5);
}

/* The R * gamma items (A, r, j) sorted by (A desc, r asc, j asc); NULL if out of memory. */
static sched_item *sorted_items(const float *a, int R, int gamma)
{
    int N = R * gamma;
    sched_item *it = (sched_item *)malloc(sizeof(sched_item) * (size_t)N);
    sched_item *tmp = (sched_item *)malloc(sizeof(sched_item) * (size_t)N);
    if (!it || !tmp) { free(it); free(tmp); return NULL; }
    for (int r = 0; r < R; ++r)
        for (int j = 1; j <= gamma; ++j) {
            sched_item s = {fixed_point_a(a[(size_t)r * gamma + (j - 1)]), r, j};
            it[(size_t)r * gamma + (j - 1)] = s;
        }
    /* bottom-up merge sort */
    for (int width = 1; width < N; width *= 2) {
        for (int lo = 0; lo < N; lo += 2 * width) {
            int mid = lo + width < N ? lo + width : N;
            int hi = lo + 2 * width < N ? lo + 2 * width : N;
            int p = lo, q = mid, o = lo;
            while (p < mid && q < hi) tmp[o++] = item_before(&it[q], &it[p]) ? it[q++] : it[p++];
            while (p < mid) tmp[o++] = it[p++];
            while (q < hi) tmp[o++] = it[q++];
        }
        sched_item *sw = it; it = tmp; tmp = sw;
    }
    free(tmp);
    return it;
}

/* theta[0] = Theta at the returned stop; ell [R]; *B_total = R + admitted. */
int dso_schedule(const float *a, int R, int gamma, const float *sps, int sps_len,
                 int32_t *ell, int32_t *B_total, double *theta)
{
    if (R < 1 || gamma < 1 || sps_len < R * (gamma + 1) + 1) return DSO_ERR_ARG;
    int N = R * gamma;
    sched_item *it = sorted_items(a, R, gamma);
    if (!it) return DSO_ERR_NOMEM;
    for (int r = 0; r < R; ++r) ell[r] = 0;
    const double scale = 4294967296.0;
    int64_t S = 0;
    double theta_prev = (double)((int64_t)R * (int64_t)4294967296LL) * (double)sps[R];
    int admitted = 0;
    for (int n = 1; n <= N; ++n) {
        int64_t S_n = S + it[n - 1].A;
        double th = (double)((int64_t)R * (int64_t)4294967296LL + S_n) * (double)sps[R + n];
        if (!(th > theta_prev)) break;
        S = S_n;
        theta_prev = th;
        admitted = n;
        ell[it[n - 1].r] += 1;
    }
    *B_total = R + admitted;
    *theta = theta_prev / scale;
    free(it);
    return DSO_OK;
}

/*
 * Asynchronous two-step capacity scheduler (weigao.cc DSpark-vs-MTP page, "4. hardware-
 * aware prefix scheduler", last paragraph; billytse.dev DSpark page, section 7): the number
 * of positions the target verifies at step t, K, is fixed from the survival probabilities
 * of step t - 2, so that the batch size is known ahead of the step; the K positions
 * themselves are the first K in the order of the current survival probabilities.
 *
 * K_in >= 0: the capacity decided two steps earlier (clamped to [0, R gamma]).
 * K_in < 0:  no earlier decision (the first steps of a sequence): K is this step's own
 *            early-stop count, which makes the call equal to dso_schedule.
 * Outputs: ell [R] (request r's count among the first K items), B_total = R + K,
 * theta = (R + S_K) SPS(R + K) with the same fixed-point sum as dso_schedule, and K_out =
 * the early-stop count n* of this step's a (dso_schedule's B_total - R): the capacity
 * for step t + 2.
 */
int dso_schedule_async(const float *a, int R, int gamma, const float *sps, int sps_len,
                       int K_in, int32_t *ell, int32_t *B_total, double *theta, int32_t *K_out)
{
    if (R < 1 || gamma < 1 || sps_len < R * (gamma + 1) + 1) return DSO_ERR_ARG;
    int N = R * gamma;
    int32_t *ell_now = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    if (!ell_now) return DSO_ERR_NOMEM;
    int32_t Bt_now;
    double th_now;
    int rc = dso_schedule(a, R, gamma, sps, sps_len, ell_now, &Bt_now, &th_now);
    free(ell_now);
    if (rc != DSO_OK) return rc;
    int n_star = Bt_now - R;
    int K = K_in < 0 ? n_star : (K_in > N ? N : K_in);
    sched_item *it = sorted_items(a, R, gamma);
    if (!it) return DSO_ERR_NOMEM;
    for (int r = 0; r < R; ++r) ell[r] = 0;
    int64_t S = 0;
    for (int n = 1; n <= K; ++n) {
        S += it[n - 1].A;
        ell[it[n - 1].r] += 1;
    }
    *B_total = R + K;
    *theta = (double)((int64_t)R * (int64_t)4294967296LL + S) * (double)sps[R + K] / 4294967296.0;
    *K_out = n_star;
    free(it);
    return DSO_OK;
}

/*
 * Fixed confidence-threshold truncation (billytse.dev DSpark page, section 8: the
 * confidence-threshold sweep under fixed-length verification; xhh.club DSpark page, on why
 * the scheduler's threshold must move with the load: a fixed threshold on the survival
 * probability is the load-blind baseline).  Request r keeps its draft positions 1..l_r
 * where l_r is the last j of the leading run with a[r, j] > threshold (the scan stops at
 * the first j that fails, so admission looks only at positions up to j).  B_total =
 * sum_r (1 + l_r).  threshold < 0 verifies every position (fixed-length verification).
 */
int dso_schedule_threshold(const float *a, int R, int gamma, float threshold, int32_t *ell,
                           int32_t *B_total)
{
    if (R < 1 || gamma < 1) return DSO_ERR_ARG;
    int64_t total = 0;
    for (int r = 0; r < R; ++r) {
        int l = 0;
        for (int j = 1; j <= gamma; ++j) {
            if (!((double)a[(size_t)r * gamma + (j - 1)] > (double)threshold)) break;
            l = j;
        }
        ell[r] = l;
        total += 1 + l;
    }
    *B_total = (int32_t)total;
    return DSO_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Lossless verification                                                                 */
/* ------------------------------------------------------------------------------------ */

/*
 * T [n_req, gamma+1, V] target logits; U [n_req, gamma, V]; tokens [n_req, gamma];
 * ell [n_req] verified lengths.  Outputs: accept_len [n_req], out_tokens [n_req, gamma+1]
 * (-1 padded), n_out [n_req], band [n_req, gamma] (|u - p/q| of every accept test, NaN
 * where no test ran), gap [n_req] (top-two score gap of the correction / bonus draw),
 * fallback [n_req] (1 when the residual was empty and P itself was sampled).
 *
 * point_mass = 0: the proposal of position k is Q_k = softmax(U[k] + W1[prev] W2), the
 * distribution the tokens were sampled from; with E_rows ([n_req, gamma, r], the RNN
 * head's output rows tanh(output) of the draft) it is softmax(U[k] + E_rows[k] W2).  point_mass = 1: the tokens were drafted
 * greedily, so the proposal is the point mass at x_k (Q_k(v) = 1 if v = x_k, else 0) and
 * U, W1, W2 are not read.  The acceptance test and the residual are the same formulas
 * with that Q.
 */
static int verify_impl(const float *T, const float *U, const uint16_t *W1, const uint16_t *W2,
                       const double *E_rows, const int32_t *anchor, const int32_t *tokens,
                       const int32_t *ell, const int32_t *req_ids, int n_req, int gamma, int V,
                       int r, uint64_t seed, int point_mass, int32_t *accept_len,
                       int32_t *out_tokens, int32_t *n_out, double *band, double *gap,
                       int32_t *fallback, int nthreads)
{
    if (n_req < 0 || gamma < 1 || V < 1 || (!point_mass && r < 1)) return DSO_ERR_ARG;
    int err = DSO_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int i = 0; i < n_req; ++i) {
        int b = req_ids[i];
        int L = ell[i];
        for (int k = 0; k < gamma; ++k) band[(size_t)i * gamma + k] = NAN;
        for (int k = 0; k <= gamma; ++k) out_tokens[(size_t)i * (gamma + 1) + k] = -1;
        fallback[i] = 0;
        if (L < 0 || L > gamma) { err = DSO_ERR_ARG; continue; }
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
        double *P = (double *)malloc(sizeof(double) * (size_t)V);
        double *Q = (double *)malloc(sizeof(double) * (size_t)V);
        double *score = (double *)malloc(sizeof(double) * (size_t)V);
        unsigned char *mask = (unsigned char *)malloc((size_t)V);
        double *erow_m = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
        if (!z || !P || !Q || !score || !mask || !erow_m) {
            free(z); free(P); free(Q); free(score); free(mask); free(erow_m);
            err = DSO_ERR_NOMEM;
            continue;
        }
        int reject_at = 0;   /* 1-based position of the first reject, 0: none */
        int prev = anchor ? anchor[i] : -1;
        for (int k = 1; k <= L; ++k) {
            size_t o = (size_t)i * gamma + (k - 1);
            int x = tokens[o];
            if (x < 0 || x >= V) { err = DSO_ERR_ARG; break; }
            /* target p_k = softmax(T[k]) */
            const float *Trow = T + ((size_t)i * (gamma + 1) + (k - 1)) * V;
            double M = -INFINITY, Ssum = 0.0;
            for (int v = 0; v < V; ++v) if ((double)Trow[v] > M) M = (double)Trow[v];
            for (int v = 0; v < V; ++v) Ssum += exp((double)Trow[v] - M);
            double p = exp((double)Trow[x] - M) / Ssum;
            /* the proposal Q_k the token was drawn from */
            if (point_mass) {
                for (int v = 0; v < V; ++v) Q[v] = (v == x) ? 1.0 : 0.0;
            } else {
                const double *erow = erow_m;
                if (E_rows)
                    erow = E_rows + o * (size_t)r;
                else
                    markov_row(W1, prev, r, erow_m);
                draft_logits(U + o * V, erow, W2, V, r, z);
                double m, s;
                softmax_stats(z, V, &m, &s);
                for (int v = 0; v < V; ++v) Q[v] = exp(z[v] - m) / s;
            }
            double q = Q[x];
            double u = dso_u01(dso_draw(seed, b, k, 0, 1));
            double ratio = p / q;
            band[o] = fabs(u - ratio);
            if (u < ratio) {          /* accept with probability min(1, p/q) */
                prev = x;
                continue;
            }
            reject_at = k;
            /* residual norm(max(0, P - Q)) by Gumbel-max over log(P - Q), P > Q */
            int any = 0;
            for (int v = 0; v < V; ++v) {
                double Pv = exp((double)Trow[v] - M) / Ssum;
                double Qv = Q[v];
                P[v] = Pv;
                mask[v] = Pv > Qv;
                score[v] = mask[v] ? log(Pv - Qv) : -INFINITY;
                any |= mask[v];
            }
            double gp;
            int y;
            if (any) {
                y = gumbel_argmax(score, mask, V, seed, b, k, 2, &gp);
            } else {
                for (int v = 0; v < V; ++v) score[v] = log(P[v]);
                y = gumbel_argmax(score, NULL, V, seed, b, k, 2, &gp);
                fallback[i] = 1;
            }
            gap[i] = gp;
            for (int j = 1; j < k; ++j)
                out_tokens[(size_t)i * (gamma + 1) + (j - 1)] = tokens[(size_t)i * gamma + (j - 1)];
            out_tokens[(size_t)i * (gamma + 1) + (k - 1)] = y;
            accept_len[i] = k - 1;
            n_out[i] = k;
            break;
        }
        if (!reject_at) {
            /* every verified position accepted: the target's bonus token from row L+1 */
            const float *Trow = T + ((size_t)i * (gamma + 1) + L) * V;
            for (int v = 0; v < V; ++v) score[v] = (double)Trow[v];
            double gp;
            int y = gumbel_argmax(score, NULL, V, seed, b, L + 1, 3, &gp);
            gap[i] = gp;
            for (int j = 1; j <= L; ++j)
                out_tokens[(size_t)i * (gamma + 1) + (j - 1)] = tokens[(size_t)i * gamma + (j - 1)];
            out_tokens[(size_t)i * (gamma + 1) + L] = y;
            accept_len[i] = L;
            n_out[i] = L + 1;
        }
        free(z); free(P); free(Q); free(score); free(mask); free(erow_m);
    }
    return err;
}

int dso_verify(const float *T, const float *U, const uint16_t *W1, const uint16_t *W2,
               const int32_t *anchor, const int32_t *tokens, const int32_t *ell,
               const int32_t *req_ids, int n_req, int gamma, int V, int r, uint64_t seed,
               int32_t *accept_len, int32_t *out_tokens, int32_t *n_out, double *band,
               double *gap, int32_t *fallback, int nthreads)
{
    return verify_impl(T, U, W1, W2, NULL, anchor, tokens, ell, req_ids, n_req, gamma, V, r, seed,
                       0, accept_len, out_tokens, n_out, band, gap, fallback, nthreads);
}

/* Verification of greedily drafted tokens (proposal = point mass at each token). */
int dso_verify_greedy(const float *T, const int32_t *tokens, const int32_t *ell,
                      const int32_t *req_ids, int n_req, int gamma, int V, uint64_t seed,
                      int32_t *accept_len, int32_t *out_tokens, int32_t *n_out, double *band,
                      double *gap, int32_t *fallback, int nthreads)
{
    return verify_impl(T, NULL, NULL, NULL, NULL, NULL, tokens, ell, req_ids, n_req, gamma, V, 0,
                       seed, 1, accept_len, out_tokens, n_out, band, gap, fallback, nthreads);
}

/* Verification of an RNN-head draft: Q_k = softmax(U[k] + E[k] W2), E from dso_draft_rnn. */
int dso_verify_rnn(const float *T, const float *U, const double *E, const uint16_t *W2,
                   const int32_t *tokens, const int32_t *ell, const int32_t *req_ids, int n_req,
                   int gamma, int V, int r, uint64_t seed, int32_t *accept_len,
                   int32_t *out_tokens, int32_t *n_out, double *band, double *gap,
                   int32_t *fallback, int nthreads)
{
    if (!E) return DSO_ERR_ARG;
    return verify_impl(T, U, NULL, W2, E, NULL, tokens, ell, req_ids, n_req, gamma, V, r, seed, 0,
                       accept_len, out_tokens, n_out, band, gap, fallback, nthreads);
}
