/*
 * dspark_oracle.c -- plain float64 CPU oracle of the DSpark draft + verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark load it.  It shares no header, helper, table or constant
 * with the CUDA sources: each side implements the published Philox generator
 * on its own.
 *
 * Sources (page title, then section):
 *   [P2] "DSpark：半自回归生成与置信度调度的投机解码" (pinghaoyang.com.cn/aigc/posts/dspark/)
 *   [P3] "拒绝盲猜与算力空转：深度拆解 DeepSeek 开源投机采样方案 DeepSpec & DSpark"
 *        (val213.github.io/2026/06/28/DSpark&DSpec/)
 *   [P4] "DeepSeek-AI与北京大学联手破局：AI聊天机器人"慢速打字"的终极解决方案"
 *        (techwalker.com/2026/0716/3193540.shtml)
 *   [Philox] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *        1, 2, 3", SC'11, section 3 (Philox4x32, 10 rounds).
 *
 * Every function computes its definition directly: exact matrix products in
 * double, two-pass log-sum-exp, Gumbel-max over all V entries, a sort followed
 * by a linear scan, and a literal accept / reject loop.  Nothing is blocked,
 * fused or reordered beyond the definition.  Requests are independent in the
 * draft and verify steps, so those loops may run in parallel over requests
 * (OpenMP); each request's arithmetic is sequential and identical either way.
 *
 * Random numbers.  The pages say only that drafts are sampled; the draw is a
 * Gumbel-max over the draft logits, driven by Philox4x32-10 with
 *   key     = (seed mod 2^32, seed div 2^32)
 *   counter = (col div 4, req*(gamma+1) + row, step mod 2^32,
 *              domain + 4*(step div 2^32))            (all mod 2^32)
 *   word    = col mod 4 of the four outputs
 * and the uniform u = (2*(x div 2^9) + 1) * 2^-24 in (0, 1), exact in binary32
 * and binary64.  Domains: 0 draft Gumbel, 1 acceptance uniform (col 0),
 * 2 residual Gumbel, 3 bonus Gumbel.  "row" is the 0-based position row:
 * draft position k uses row k-1; target row i (the distribution p_{i+1}) uses
 * row i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 [Philox, section 3]: multipliers and Weyl key increments.    */
/* ------------------------------------------------------------------------ */
static const uint32_t PHILOX_M0 = 0xD2511F53u, PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W0 = 0x9E3779B9u, PHILOX_W1 = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += PHILOX_W0; k1 += PHILOX_W1; }
        uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* One 32-bit word of the stream described in the file header. */
uint32_t oracle_random_word(uint64_t seed, uint64_t step, uint32_t domain,
                            uint32_t row, uint32_t col)
{
    uint32_t ctr[4] = { col >> 2, row, (uint32_t)step,
                        domain + 4u * (uint32_t)(step >> 32) };
    uint32_t key[2] = { (uint32_t)seed, (uint32_t)(seed >> 32) };
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[col & 3u];
}

/* u = (2*(x >> 9) + 1) / 2^24: 2^23 equally spaced points, symmetric about 1/2. */
double oracle_uniform(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, uint32_t col)
{
    uint32_t x = oracle_random_word(seed, step, domain, row, col);
    return (double)(2u * (x >> 9) + 1u) * (1.0 / 16777216.0);
}

/* Standard Gumbel variate G = -log(-log u). */
double oracle_gumbel(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, uint32_t col)
{
    double u = oracle_uniform(seed, step, domain, row, col);
    return -log(-log(u));
}

/* G for columns col0 .. col0+n-1 of one stream (the definition above,
 * column by column; the vocabulary-split checks draw on slices of a row). */
void oracle_gumbel_span(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, uint32_t col0, int n,
                        double* out)
{
    for (int i = 0; i < n; ++i) out[i] = oracle_gumbel(seed, step, domain, row, col0 + (uint32_t)i);
}

/* Two-pass log-sum-exp of x[0..n). */
static double logsumexp(const double* x, int n)
{
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (x[i] > m) m = x[i];
    if (m == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += exp(x[i] - m);
    return m + log(s);
}

/* Gumbel-max: argmax_v (score[v] + G_v) over entries with finite score; the
 * lowest index wins an exact tie.  Returns the index (or -1 if no entry is
 * finite) and, through gap, the distance between the best and the runner-up
 * perturbed score (+inf when only one entry competes). */
static int gumbel_argmax(const double* score, int n, uint64_t seed, uint64_t step,
                         uint32_t domain, uint32_t row, double* gap)
{
    int best = -1;
    double b1 = -INFINITY, b2 = -INFINITY;
    for (int v = 0; v < n; ++v) {
        if (!(score[v] > -INFINITY)) continue;
        double s = score[v] + oracle_gumbel(seed, step, domain, row, (uint32_t)v);
        if (best < 0 || s > b1) { b2 = b1; b1 = s; best = v; }
        else if (s > b2) { b2 = s; }
    }
    if (gap) *gap = (b2 == -INFINITY) ? INFINITY : b1 - b2;
    return best;
}

/* Transition bias [P2 §Markov Head：一阶转移偏置], [P3 §DSpark 的解法 ...
 * 低秩马尔可夫头]: B(v) = h . W2[:, v] for every vocabulary entry v, from a
 * rank-r row h: the Markov head's h = W1[x~_{k-1}], the RNN head's state.
 * Accumulated row by row of W2, i.e. in increasing rho for every v. */
static void bias_of_row(const double* h, const double* W2, int V, int r, double* bias)
{
    for (int v = 0; v < V; ++v) bias[v] = 0.0;
    for (int rho = 0; rho < r; ++rho) {
        const double hr = h[rho];
        const double* w = W2 + (size_t)rho * V;
        for (int v = 0; v < V; ++v) bias[v] += hr * w[v];
    }
}

/* Draft logits of one position: z = (U_k + B_k) / tau, B_k from the row h
 * [P2 §整体架构: the draft distribution is built from U_k plus B_k]. */
static void draft_logits(const double* U_row, const double* h, const double* W2, int V, int r,
                         double tau, double* z)
{
    bias_of_row(h, W2, V, r, z);
    for (int v = 0; v < V; ++v) z[v] = (U_row[v] + z[v]) / tau;
}

/* ------------------------------------------------------------------------ */
/* Steps a1-a3: the semi-autoregressive draft loop [P2 §整体架构, §Markov Head]. */
/* For k = 1..gamma: x_prev = x~_{k-1} (the anchor for k = 1), q_k =          */
/* softmax((U_k + B_k(x_prev))/tau), x~_k ~ q_k by Gumbel-max.                */
/* ------------------------------------------------------------------------ */
int oracle_draft_markov(const double* U, const double* W1, const double* W2,
                        const int32_t* anchor, const int32_t* req,
                        int nb, int gamma, int V, int r, double tau,
                        uint64_t seed, uint64_t step,
                        int32_t* draft_tok, double* lse_q, double* z_tok, double* gap,
                        double* logits)
{
    if (nb < 0 || gamma < 1 || V < 1 || r < 1 || !(tau > 0.0)) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < nb; ++b) {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        if (!z) { bad = 1; continue; }
        int x_prev = anchor[b];
        for (int k = 1; k <= gamma; ++k) {
            if (x_prev < 0 || x_prev >= V) { bad = 1; break; }
            const size_t row = (size_t)b * gamma + (size_t)(k - 1);
            draft_logits(U + row * V, W1 + (size_t)x_prev * r, W2, V, r, tau, z);
            if (logits) memcpy(logits + row * V, z, sizeof(double) * (size_t)V);
            double g;
            const uint32_t prow = (uint32_t)req[b] * (uint32_t)(gamma + 1) + (uint32_t)(k - 1);
            int x = gumbel_argmax(z, V, seed, step, 0u, prow, &g);
            draft_tok[row] = x;
            lse_q[row] = logsumexp(z, V);
            z_tok[row] = z[x];
            if (gap) gap[row] = g;
            x_prev = x;
        }
        free(z);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Step a4: confidence head, sequential temperature scaling and prefix       */
/* survival [P2 §置信度头, §校准问题], [P4 §四].                              */
/*   c_k   = sigmoid(w . [h_k ; emb(x~_{k-1})] + b)                           */
/*   c~_k  = sigmoid(logit(c_k) / T_k)                                        */
/*   log a_k = sum_{i<=k} log c~_i                                            */
/* ------------------------------------------------------------------------ */
void oracle_confidence_sts(const double* h, int d, const double* emb, int e,
                           const int32_t* anchor, const int32_t* draft_tok,
                           const double* w_c, double b_c, const double* T,
                           int nb, int gamma,
                           double* conf_raw, double* conf_cal, double* log_surv)
{
    for (int b = 0; b < nb; ++b) {
        double acc_log = 0.0;
        for (int k = 1; k <= gamma; ++k) {
            const size_t row = (size_t)b * gamma + (size_t)(k - 1);
            const int x_prev = (k == 1) ? anchor[b] : draft_tok[row - 1];
            const double* hk = h + row * (size_t)d;
            const double* ek = emb + (size_t)x_prev * (size_t)e;
            double s = b_c;
            for (int i = 0; i < d; ++i) s += w_c[i] * hk[i];
            for (int i = 0; i < e; ++i) s += w_c[d + i] * ek[i];
            const double c = 1.0 / (1.0 + exp(-s));
            const double logit_c = log(c) - log1p(-c);
            const double c_cal = 1.0 / (1.0 + exp(-logit_c / T[k - 1]));
            acc_log += log(c_cal);
            conf_raw[row] = c;
            conf_cal[row] = c_cal;
            log_surv[row] = acc_log;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Step a5: hardware-aware greedy prefix scheduler [P2 §硬件感知前缀调度器],   */
/* [P4 §四, §五].                                                             */
/* Candidates (b, j), j = 1..gamma, with survival a_{b,j}; sorted by a         */
/* descending, ties by b then j.  R = B tokens are always emitted.            */
/*   Theta(n) = (R + sum of the first n survivals) * SPS(R + n),              */
/* SPS(m) = sps[m - 1].  mode 0: every request verifies its whole block.      */
/* mode 1 (synchronous): admit candidates in order while Theta strictly       */
/* rises; stop at the first candidate that does not raise it.                 */
/* mode 2 (asynchronous): capacity n* = argmax_n Theta_hist(n) over the list  */
/* built from survivals two steps old (no early stop, smallest n on ties);    */
/* then admit the n* best candidates of the current list.                     */
/* ------------------------------------------------------------------------ */
typedef struct { double la; int b; int j; } cand_t;

static int cand_cmp(const void* pa, const void* pb)
{
    const cand_t* a = (const cand_t*)pa;
    const cand_t* c = (const cand_t*)pb;
    if (a->la > c->la) return -1;
    if (a->la < c->la) return 1;
    if (a->b != c->b) return a->b < c->b ? -1 : 1;
    if (a->j != c->j) return a->j < c->j ? -1 : 1;
    return 0;
}

static cand_t* sorted_candidates(const double* log_surv, int B, int gamma)
{
    const int n = B * gamma;
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
    if (!c) return NULL;
    for (int b = 0; b < B; ++b)
        for (int j = 1; j <= gamma; ++j) {
            cand_t* t = &c[b * gamma + (j - 1)];
            t->la = log_surv[(size_t)b * gamma + (j - 1)];
            t->b = b; t->j = j;
        }
    qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
    return c;
}

/* Theta(n) for n = 0..B*gamma along a sorted list. */
static void theta_curve(const cand_t* c, int B, int gamma, const double* sps, double* theta)
{
    const int n = B * gamma;
    double tau = (double)B;
    theta[0] = tau * sps[B - 1];
    for (int i = 0; i < n; ++i) {
        tau += exp(c[i].la);
        theta[i + 1] = tau * sps[B + i];
    }
}

int oracle_schedule(const double* log_surv, const double* log_surv_hist,
                    const double* sps, int sps_len, int B, int gamma, int mode,
                    int32_t* K, int32_t* n_total, double* theta_out,
                    int32_t* order_out, double* curve_out)
{
    const int n = B * gamma;
    if (B < 1 || gamma < 1 || sps_len < B + n || mode < 0 || mode > 2) return -1;
    for (int b = 0; b < B; ++b) K[b] = 0;
    if (mode == 0) {
        for (int b = 0; b < B; ++b) K[b] = gamma;
        *n_total = n;
        *theta_out = 0.0;
        return 0;
    }
    cand_t* cur = sorted_candidates(log_surv, B, gamma);
    double* curve = (double*)malloc(sizeof(double) * (size_t)(n + 1));
    if (!cur || !curve) { free(cur); free(curve); return -1; }
    theta_curve(cur, B, gamma, sps, curve);
    int admit = 0;
    double theta = curve[0];
    if (mode == 1) {
        while (admit < n && curve[admit + 1] > curve[admit]) ++admit;
        theta = curve[admit];
    } else {
        cand_t* old = log_surv_hist ? sorted_candidates(log_surv_hist, B, gamma) : NULL;
        double* hcurve = (double*)malloc(sizeof(double) * (size_t)(n + 1));
        if ((log_surv_hist && !old) || !hcurve) { free(cur); free(curve); free(old); free(hcurve); return -1; }
        if (old) theta_curve(old, B, gamma, sps, hcurve);
        else memcpy(hcurve, curve, sizeof(double) * (size_t)(n + 1));
        double best = hcurve[0];
        for (int m = 1; m <= n; ++m) if (hcurve[m] > best) { best = hcurve[m]; admit = m; }
        theta = curve[admit];
        free(old); free(hcurve);
    }
    for (int i = 0; i < admit; ++i) K[cur[i].b] += 1;
    *n_total = admit;
    *theta_out = theta;
    if (order_out) for (int i = 0; i < n; ++i) order_out[i] = cur[i].b * gamma + (cur[i].j - 1);
    if (curve_out) memcpy(curve_out, curve, sizeof(double) * (size_t)(n + 1));
    free(cur); free(curve);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* RNN head [P2 §RNN Head：长程依赖], [P4 §三].  The pages name a GRU-style    */
/* recurrent state started from a learned vector and mapped to the           */
/* vocabulary like the Markov head's row; the cell's formula is not printed. */
/* Taken here: the standard GRU cell (Cho et al. 2014, in the form with the  */
/* reset gate applied to the hidden projection, as PyTorch's GRUCell),       */
/*   r  = sigma(W_ir x + b_ir + W_hr h + b_hr)                               */
/*   z  = sigma(W_iz x + b_iz + W_hz h + b_hz)                               */
/*   n  = tanh(W_in x + b_in + r * (W_hn h + b_hn))                          */
/*   h' = (1 - z) * n + z * h,                                               */
/* gate rows stacked (r, z, n) in W_ih [3r][r_in], W_hh [3r][r], b_ih, b_hh. */
/* For k = 1..gamma: s_k = GRU(s_{k-1}, E[x~_{k-1}]) with s_0 the learned     */
/* vector and x~_0 the anchor; B_k is formed from s_k rounded to bfloat16,   */
/* the dtype of W2 (and of the Markov head's W1 rows).                      */
/* ------------------------------------------------------------------------ */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

void oracle_gru_cell(const double* x, const double* h, const double* W_ih, const double* W_hh,
                     const double* b_ih, const double* b_hh, int r_in, int r, double* h_out)
{
    for (int j = 0; j < r; ++j) {
        double gi[3], gh[3];
        for (int g = 0; g < 3; ++g) {
            const double* wi = W_ih + ((size_t)g * r + j) * r_in;
            const double* wh = W_hh + ((size_t)g * r + j) * r;
            double si = b_ih[g * r + j], sh = b_hh[g * r + j];
            for (int i = 0; i < r_in; ++i) si += wi[i] * x[i];
            for (int i = 0; i < r; ++i) sh += wh[i] * h[i];
            gi[g] = si;
            gh[g] = sh;
        }
        const double rg = sigmoid(gi[0] + gh[0]);
        const double zg = sigmoid(gi[1] + gh[1]);
        const double ng = tanh(gi[2] + rg * gh[2]);
        h_out[j] = (1.0 - zg) * ng + zg * h[j];
    }
}

/* Nearest bfloat16 value (8 significant bits, ties to even). */
double oracle_bf16_round(double x)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);                       /* |x| = f 2^e, f in [1/2, 1) */
    const double q = ldexp(1.0, e - 8);  /* spacing of 8-bit significands at |x| */
    return rint(x / q) * q;
}

/* The RNN head's states along given tokens (the drafts of another run):
 * states[b][k-1] = s_k = GRU(s_{k-1}, E[tok_{k-1}]) with tok_0 = anchor[b],
 * arows = the states rounded to bfloat16.  Returns -1 on a token outside [0, V). */
int oracle_rnn_states(const double* E, const double* W_ih, const double* W_hh, const double* b_ih,
                      const double* b_hh, const double* s0, const int32_t* anchor, const int32_t* tok,
                      int nb, int gamma, int V, int r, double* states, double* arows)
{
    double* h = (double*)malloc(sizeof(double) * (size_t)r);
    double* hn = (double*)malloc(sizeof(double) * (size_t)r);
    int bad = (!h || !hn);
    for (int b = 0; b < nb && !bad; ++b) {
        memcpy(h, s0, sizeof(double) * (size_t)r);
        for (int k = 1; k <= gamma; ++k) {
            const size_t row = (size_t)b * gamma + (size_t)(k - 1);
            const int x = (k == 1) ? anchor[b] : tok[row - 1];
            if (x < 0 || x >= V) { bad = 1; break; }
            oracle_gru_cell(E + (size_t)x * r, h, W_ih, W_hh, b_ih, b_hh, r, r, hn);
            memcpy(h, hn, sizeof(double) * (size_t)r);
            for (int i = 0; i < r; ++i) {
                states[row * r + i] = h[i];
                arows[row * r + i] = oracle_bf16_round(h[i]);
            }
        }
    }
    free(h); free(hn);
    return bad ? -1 : 0;
}

int oracle_draft_rnn(const double* U, const double* E, const double* W_ih, const double* W_hh,
                     const double* b_ih, const double* b_hh, const double* s0, const double* W2,
                     const int32_t* anchor, const int32_t* req,
                     int nb, int gamma, int V, int r, double tau,
                     uint64_t seed, uint64_t step,
                     int32_t* draft_tok, double* lse_q, double* z_tok, double* gap,
                     double* states, double* arows)
{
    if (nb < 0 || gamma < 1 || V < 1 || r < 1 || !(tau > 0.0)) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < nb; ++b) {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* h = (double*)malloc(sizeof(double) * (size_t)r);
        double* hn = (double*)malloc(sizeof(double) * (size_t)r);
        double* hq = (double*)malloc(sizeof(double) * (size_t)r);
        if (!z || !h || !hn || !hq) { bad = 1; free(z); free(h); free(hn); free(hq); continue; }
        memcpy(h, s0, sizeof(double) * (size_t)r);
        int x_prev = anchor[b];
        for (int k = 1; k <= gamma; ++k) {
            if (x_prev < 0 || x_prev >= V) { bad = 1; break; }
            const size_t row = (size_t)b * gamma + (size_t)(k - 1);
            oracle_gru_cell(E + (size_t)x_prev * r, h, W_ih, W_hh, b_ih, b_hh, r, r, hn);
            memcpy(h, hn, sizeof(double) * (size_t)r);
            for (int i = 0; i < r; ++i) hq[i] = oracle_bf16_round(h[i]);
            if (states) memcpy(states + row * r, h, sizeof(double) * (size_t)r);
            if (arows) memcpy(arows + row * r, hq, sizeof(double) * (size_t)r);
            draft_logits(U + row * V, hq, W2, V, r, tau, z);
            double g;
            const uint32_t prow = (uint32_t)req[b] * (uint32_t)(gamma + 1) + (uint32_t)(k - 1);
            const int x = gumbel_argmax(z, V, seed, step, 0u, prow, &g);
            draft_tok[row] = x;
            lse_q[row] = logsumexp(z, V);
            z_tok[row] = z[x];
            if (gap) gap[row] = g;
            x_prev = x;
        }
        free(z); free(h); free(hn); free(hq);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Steps a6-a8: lossless verification and ragged output [P2 §形式化定义],      */
/* [P4 §四, §五].  For request b with verify length K_b:                       */
/*   p_i = softmax(target[b, i] / tau) for rows i = 0..K_b (p_{i+1});         */
/*   q_k = softmax(z_k) with z_k the draft logits of position k;              */
/*   walk k = 1..K_b: accept x~_k iff u_k < min(1, p_k(x~_k) / q_k(x~_k));    */
/*   at the first rejection j draw from norm(max(0, p_j - q_j)) (from p_j if   */
/*   that residual is identically zero); if all K_b are accepted draw the      */
/*   bonus token from p_{K_b + 1}.                                            */
/* q_k is rebuilt from the same bias row as the draft: W1[x~_{k-1}], or, when  */
/* arows [nb][gamma][r] is given (the RNN head), arows[b][k-1].              */
/* Outputs are laid out flat: offsets = exclusive scan of (A_b + 1).          */
/* diag[b*6 + .] = { min |u_k - min(1, p/q)| over the walk, gap of the final   */
/*   draw, residual mass sum max(0, p - q) (0 if none), final-draw row,         */
/*   final-draw kind (0 residual, 1 bonus, 2 residual fell back to p),         */
/*   accepted count }.                                                          */
/* ------------------------------------------------------------------------ */
int oracle_verify(const double* target, const double* U, const double* W1, const double* W2,
                  const double* arows,
                  const int32_t* anchor, const int32_t* draft_tok, const int32_t* K,
                  const int32_t* req, int nb, int gamma, int V, int r, double tau,
                  uint64_t seed, uint64_t step,
                  int32_t* accepted, int32_t* final_tok, double* p_tok, double* q_tok,
                  double* diag)
{
    if (nb < 0 || gamma < 1 || V < 1 || r < 1 || !(tau > 0.0) || (!W1 && !arows)) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int b = 0; b < nb; ++b) {
        const int Kb = K[b];
        double* t = (double*)malloc(sizeof(double) * (size_t)V);
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* s = (double*)malloc(sizeof(double) * (size_t)V);
        if (!t || !z || !s || Kb < 0 || Kb > gamma) { bad = 1; free(t); free(z); free(s); continue; }
        const uint32_t row0 = (uint32_t)req[b] * (uint32_t)(gamma + 1);
        double min_margin = INFINITY;
        int A = Kb, rej = 0;
        for (int k = 1; k <= Kb; ++k) {
            const size_t drow = (size_t)b * gamma + (size_t)(k - 1);
            const int x = draft_tok[drow];
            const int x_prev = (k == 1) ? anchor[b] : draft_tok[drow - 1];
            const double* trow = target + ((size_t)b * (gamma + 1) + (size_t)(k - 1)) * V;
            for (int v = 0; v < V; ++v) t[v] = trow[v] / tau;
            const double lse_p = logsumexp(t, V);
            const double* hrow = arows ? arows + drow * (size_t)r : W1 + (size_t)x_prev * r;
            draft_logits(U + drow * V, hrow, W2, V, r, tau, z);
            const double lse_q = logsumexp(z, V);
            const double p = exp(t[x] - lse_p);
            const double q = exp(z[x] - lse_q);
            const double u = oracle_uniform(seed, step, 1u, row0 + (uint32_t)(k - 1), 0u);
            const double thr = fmin(1.0, p / q);
            p_tok[drow] = p;
            q_tok[drow] = q;
            const double margin = fabs(u - thr);
            if (margin < min_margin) min_margin = margin;
            if (!(u < thr)) { A = k - 1; rej = k; break; }
        }
        double gap = INFINITY, mass = 0.0;
        int kind, frow, tok;
        if (rej > 0) {
            /* t and z still hold row rej-1's target and draft logits. */
            const double lse_p = logsumexp(t, V);
            const double lse_q = logsumexp(z, V);
            for (int v = 0; v < V; ++v) {
                const double rv = exp(t[v] - lse_p) - exp(z[v] - lse_q);
                if (rv > 0.0) { s[v] = log(rv); mass += rv; }
                else s[v] = -INFINITY;
            }
            frow = rej - 1;
            if (mass > 0.0) {
                kind = 0;
                tok = gumbel_argmax(s, V, seed, step, 2u, row0 + (uint32_t)frow, &gap);
            } else {
                kind = 2;
                tok = gumbel_argmax(t, V, seed, step, 2u, row0 + (uint32_t)frow, &gap);
            }
        } else {
            frow = Kb;
            kind = 1;
            const double* trow = target + ((size_t)b * (gamma + 1) + (size_t)Kb) * V;
            for (int v = 0; v < V; ++v) t[v] = trow[v] / tau;
            tok = gumbel_argmax(t, V, seed, step, 3u, row0 + (uint32_t)frow, &gap);
        }
        accepted[b] = A;
        final_tok[b] = tok;
        if (diag) {
            double* dg = diag + (size_t)b * 6;
            dg[0] = min_margin; dg[1] = gap; dg[2] = mass;
            dg[3] = frow; dg[4] = kind; dg[5] = A;
        }
        free(t); free(z); free(s);
    }
    return bad ? -1 : 0;
}

/* Ragged compaction [P4 §五: all requests' tokens flattened, with a marker
 * tensor recording request and position].  offsets[b] = sum_{c<b} (A_c + 1);
 * the A_b accepted drafts are followed by the final (correction or bonus)
 * token; next_anchor[b] is the last emitted token. */
void oracle_compact(const int32_t* draft_tok, const int32_t* accepted, const int32_t* final_tok,
                    int nb, int gamma, int32_t* out_tok, int32_t* out_req, int32_t* out_pos,
                    int32_t* out_off, int32_t* next_anchor)
{
    int32_t off = 0;
    for (int b = 0; b < nb; ++b) {
        out_off[b] = off;
        for (int i = 0; i < accepted[b]; ++i) {
            out_tok[off] = draft_tok[(size_t)b * gamma + i];
            out_req[off] = b; out_pos[off] = i; ++off;
        }
        out_tok[off] = final_tok[b];
        out_req[off] = b; out_pos[off] = accepted[b]; ++off;
        next_anchor[b] = final_tok[b];
    }
    out_off[nb] = off;
}

/* ------------------------------------------------------------------------ */
/* STS fitting [P2 §校准问题：原始置信度不可靠], [P4 §四].                      */
/* A validation set of N drafted blocks: score[n][i] = logit(c_i) of the      */
/* confidence head (its pre-sigmoid score), acc_len[n] = the number of drafts */
/* the target accepted.  The label of prefix j is acc_len >= j.  Positions    */
/* are fitted left to right; at position k the earlier temperatures stay as   */
/* chosen, and the survival of prefix k under candidate temperature T is      */
/*   a_n(T) = prod_{i<k} sigma(score[n][i] / T_i) * sigma(score[n][k] / T),   */
/* multiplied in order of i.  Its expected calibration error over M equal-    */
/* width bins on [0, 1] (bin m holds m/M <= a < (m+1)/M, a = 1 in bin M-1) is */
/*   ECE = sum_m |B_m|/N * |mean label - mean a over B_m|                    */
/*       = (1/N) sum_m | sum_{n in B_m} (label_n - a_n) |.                   */
/* T_k is the grid value with the smallest ECE (the lowest grid index among  */
/* equal values).                                                            */
/* ------------------------------------------------------------------------ */
/* Survival of prefix k (1-based) for every sample and every grid value:
 * out[n][g] = a_n(grid[g]) with the earlier temperatures T_prev[0..k-2]. */
void oracle_sts_survival(const double* score, int N, int gamma, const double* T_prev, int k,
                         const double* grid, int G, double* out)
{
    for (int n = 0; n < N; ++n) {
        const double* s = score + (size_t)n * gamma;
        double prefix = 1.0;
        for (int i = 1; i < k; ++i) prefix *= sigmoid(s[i - 1] / T_prev[i - 1]);
        for (int g = 0; g < G; ++g) out[(size_t)n * G + g] = prefix * sigmoid(s[k - 1] / grid[g]);
    }
}

/* ECE of predictions a[n] against labels y[n] in {0, 1} over M bins. */
static double ece_of(const double* a, const int* y, int N, int M, double* sums)
{
    for (int m = 0; m < M; ++m) sums[m] = 0.0;
    for (int n = 0; n < N; ++n) {
        int m = (int)floor(a[n] * M);
        if (m > M - 1) m = M - 1;
        if (m < 0) m = 0;
        sums[m] += (double)y[n] - a[n];
    }
    double e = 0.0;
    for (int m = 0; m < M; ++m) e += fabs(sums[m]);
    return e / N;
}

/* The left-to-right fit.  ece[k-1][g] = ECE of prefix k under grid[g];
 * idx[k-1] and T_out[k-1] the chosen grid entry.  T_fixed, when non-NULL,
 * replaces the chosen temperatures as the earlier positions' T_i (the
 * choices are still reported), so that another fit's choices can be
 * re-evaluated.  Returns 0, or -1 for bad sizes / out-of-memory. */
int oracle_sts_fit(const double* score, const int32_t* acc_len, int N, int gamma,
                   const double* grid, int G, int M, const double* T_fixed,
                   double* ece, int32_t* idx, double* T_out)
{
    if (N < 1 || gamma < 1 || G < 1 || M < 1) return -1;
    double* a = (double*)malloc(sizeof(double) * (size_t)N * G);
    double* col = (double*)malloc(sizeof(double) * (size_t)N);
    double* sums = (double*)malloc(sizeof(double) * (size_t)M);
    double* T_prev = (double*)malloc(sizeof(double) * (size_t)gamma);
    int* y = (int*)malloc(sizeof(int) * (size_t)N);
    if (!a || !col || !sums || !T_prev || !y) { free(a); free(col); free(sums); free(T_prev); free(y); return -1; }
    for (int k = 1; k <= gamma; ++k) {
        oracle_sts_survival(score, N, gamma, T_prev, k, grid, G, a);
        for (int n = 0; n < N; ++n) y[n] = acc_len[n] >= k;
        int best = 0;
        for (int g = 0; g < G; ++g) {
            for (int n = 0; n < N; ++n) col[n] = a[(size_t)n * G + g];
            const double e = ece_of(col, y, N, M, sums);
            ece[(size_t)(k - 1) * G + g] = e;
            if (e < ece[(size_t)(k - 1) * G + best]) best = g;
        }
        idx[k - 1] = best;
        T_out[k - 1] = grid[best];
        T_prev[k - 1] = T_fixed ? T_fixed[k - 1] : grid[best];
    }
    free(a); free(col); free(sums); free(T_prev); free(y);
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
