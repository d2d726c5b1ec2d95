/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the confidence-driven
 * variable-length verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library; it is written from the method's
 * description, not from the kernels.
 *
 * Sources (cited by page title and section):
 *   [DS]  "DFlash to DSpark in SGLang: 4.3x faster decode, and DeepSeek-V4
 *          support" -- sections "Background", "DSpark: a sequential head and a
 *          verify budget", "The confidence scheduler and verify modes",
 *          "Ragged verify under full CUDA graphs", "Zero-overhead scheduling
 *          and kernels", "Serving DeepSeek-V4 with SGLang".
 *   [KC]  "SGLang Integrates DSpark: How Confidence-Driven Speculative
 *          Decoding Cracks the High-Concurrency Failure Problem" -- section
 *          "The Old Problem with Speculative Decoding: It Breaks Down at
 *          Scale", which names the speculative-sampling method of Chen et al.
 *          2023, "Accelerating Large Language Model Decoding with Speculative
 *          Sampling" (accept with min(1, p/q), else resample from the
 *          normalised positive part of p - q).
 *   [SC11] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *          1, 2, 3", SC'11 -- the Philox4x64-10 counter-based generator.
 *
 * Every floating-point quantity is computed in double precision.  Logits and
 * hidden states arrive as fp32 (dtype 0) or bf16 bit patterns (dtype 1) and
 * are widened exactly.
 *
 * Each decision that floating point takes (S >= c, the cap threshold, u < r,
 * the inverse-CDF crossing) also reports a "near tie" when the fp64 margin is
 * smaller than the caller's eps; a reduced-precision implementation may
 * legitimately decide such a case the other way.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Philox4x64-10 [SC11]: a 4x64-bit counter and a 2x64-bit key; ten rounds,  */
/* each two 64x64->128 multiplies and a word permutation, the key bumped by  */
/* two Weyl constants between rounds.                                        */
/* ------------------------------------------------------------------------ */
static void mul_hi_lo_64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo)
{
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(p >> 64);
    *lo = (uint64_t)p;
}

void orc_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2], uint64_t out[4])
{
    /* Multipliers and Weyl increments as published for Philox4x64 [SC11]. */
    const uint64_t mult0 = 0xD2E7470EE14C6C93ULL;
    const uint64_t mult1 = 0xCA5A826395121157ULL;
    const uint64_t weyl0 = 0x9E3779B97F4A7C15ULL; /* golden ratio */
    const uint64_t weyl1 = 0xBB67AE8584CAA73BULL; /* sqrt(3) - 1 */
    uint64_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += weyl0;
            k1 += weyl1;
        }
        uint64_t hi0, lo0, hi1, lo1;
        mul_hi_lo_64(mult0, x0, &hi0, &lo0);
        mul_hi_lo_64(mult1, x2, &hi1, &lo1);
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* A uniform in [0,1) from the top 24 bits of a 64-bit word (exact in fp32). */
double orc_uniform24(uint64_t word)
{
    return (double)(word >> 40) * (1.0 / 16777216.0);
}

/* The uniforms of draft position k of request b: counter (b, k, 0, 0), key
 * (seed, 0); word 0 is the accept uniform u, word 1 the block uniform u' and
 * word 2 the in-block uniform u'' of a draw at that position. */
void orc_uniforms(uint64_t seed, int64_t b, int64_t k, double *u, double *u2, double *u3)
{
    uint64_t ctr[4] = {(uint64_t)b, (uint64_t)k, 0, 0};
    uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    orc_philox4x64_10(ctr, key, out);
    *u = orc_uniform24(out[0]);
    *u2 = orc_uniform24(out[1]);
    *u3 = orc_uniform24(out[2]);
}

/* ------------------------------------------------------------------------ */
/* Element access: dtype 0 = IEEE fp32, dtype 1 = bfloat16 bit pattern.      */
/* ------------------------------------------------------------------------ */
static double elem(const void *base, int dtype, int64_t i)
{
    if (dtype == 0) {
        return (double)((const float *)base)[i];
    }
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* a1 + a2, entropy-confidence variant.                                     */
/*   [KC] "DSpark's Core Idea: Only Verify the Parts You're Confident        */
/*   About": the lower the entropy of the drafter's output distribution at  */
/*   a position, the more certain the drafter and the likelier the draft is */
/*   accepted; verification goes to low-entropy positions.  Reading taken:   */
/*   q = softmax(z_q / theta) over the vocabulary, H = -sum_y q(y) ln q(y)    */
/*   (nats), conf = exp(-H) -- the q-weighted geometric mean of q, in        */
/*   (1/V, 1], 1 for a one-hot q and 1/V for a uniform one.  The survival    */
/*   curve and the budget then follow orc_score's definitions.               */
/* H is taken from its definition with a shifted exponent: with m the row   */
/* maximum of x = z / theta, e_y = exp(x_y - m), s = sum e_y,                */
/*   H = ln s - sum_y (e_y / s) (x_y - m).                                   */
/* Inputs: draft_logits [B, gamma, V] (dtype 0 fp32 / 1 bf16), theta > 0.    */
/* Outputs as orc_score.                                                     */
/* ------------------------------------------------------------------------ */
int orc_score_entropy(int B, int gamma, int V, int dtype, const void *draft_logits,
                      double theta, double c, double eps, double *conf, double *surv,
                      int32_t *L0, int32_t *tie)
{
    if (B < 0 || gamma < 1 || V < 1 || !(theta > 0.0)) return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)V);
    if (!x) return -2;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < gamma; ++i) {
            const int64_t row = ((int64_t)b * gamma + i) * V;
            double m = -INFINITY;
            for (int y = 0; y < V; ++y) {
                x[y] = elem(draft_logits, dtype, row + y) / theta;
                if (x[y] > m) m = x[y];
            }
            double s = 0.0;
            for (int y = 0; y < V; ++y) s += exp(x[y] - m);
            double mean = 0.0; /* sum_y q(y) (x_y - m) */
            for (int y = 0; y < V; ++y) {
                const double e = exp(x[y] - m);
                if (e > 0.0) mean += (e / s) * (x[y] - m);
            }
            const double H = log(s) - mean;
            conf[b * gamma + i] = exp(-H);
        }
        double S = 1.0; /* S_0 */
        int32_t L = (1.0 >= c) ? 0 : -1;
        int32_t ties = 0;
        for (int k = 1; k <= gamma; ++k) {
            S = S * conf[b * gamma + (k - 1)];
            surv[b * gamma + (k - 1)] = S;
            if (S >= c) L = k;
            if (fabs(S - c) < eps) ties++;
        }
        if (fabs(1.0 - c) < eps) ties++;
        L0[b] = (L < 0) ? 0 : L;
        tie[b] = ties;
    }
    free(x);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* STS temperature fitting (offline calibration of a1).                      */
/*   [DS] "DSpark: a sequential head and a verify budget": Sequential        */
/*   Temperature Scaling calibrates the head's survival product to match     */
/*   true acceptance rates.  Reading taken: the temperature tau_i of         */
/*   position i in conf = sigmoid(x / tau_i) is the maximum-likelihood fit   */
/*   to logged accept outcomes.  A logged request-step n (verify length L_n, */
/*   accepted drafts a_n) observes position i when i < L_n and i <= a_n      */
/*   (verified, every earlier draft accepted); the outcome is accept         */
/*   (i < a_n) or reject (i = a_n).  Positions past the first rejection are  */
/*   not observed.  The head logit is recovered from the logged confidence   */
/*   and the temperature that produced it: x = tau_used_i * logit(conf),     */
/*   conf clamped to [2^-126, 1 - 2^-24] (the fp32 confidences' range).       */
/*   With beta = 1 / tau,                                                    */
/*     NLL_i(beta) = sum_obs [ log(1 + e^{beta x}) - y beta x ],             */
/*   convex in beta; minimised over [1/tau_max, 1/tau_min] by golden-section */
/*   search in fp64.  No observation: tau_out = tau_used, nll = 0.           */
/* ------------------------------------------------------------------------ */
static double softplus(double z)
{
    return z > 0.0 ? z + log1p(exp(-z)) : log1p(exp(z));
}

static double sts_nll(const double *x, const int32_t *y, int n, double beta)
{
    double s = 0.0;
    for (int j = 0; j < n; ++j) s += softplus(beta * x[j]) - (y[j] ? beta * x[j] : 0.0);
    return s;
}

int orc_fit_sts_tau(int N, int gamma, const float *conf, const float *tau_used,
                    const int32_t *L, const int32_t *accept_len, double tau_min,
                    double tau_max, double *tau_out, double *nll_out, int32_t *n_obs)
{
    if (N < 0 || gamma < 1 || !(tau_min > 0.0) || !(tau_max >= tau_min)) return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    int32_t *y = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    if (!x || !y) { free(x); free(y); return -2; }
    const double cmin = ldexp(1.0, -126), cmax = 1.0 - ldexp(1.0, -24);
    for (int i = 0; i < gamma; ++i) {
        int n = 0;
        for (int b = 0; b < N; ++b) {
            if (!(i < L[b] && i <= accept_len[b])) continue;
            double c = (double)conf[(int64_t)b * gamma + i];
            if (c < cmin) c = cmin;
            if (c > cmax) c = cmax;
            x[n] = (double)tau_used[i] * (log(c) - log1p(-c));
            y[n] = i < accept_len[b];
            ++n;
        }
        n_obs[i] = n;
        if (n == 0) {
            tau_out[i] = (double)tau_used[i];
            nll_out[i] = 0.0;
            continue;
        }
        const double g = (sqrt(5.0) - 1.0) / 2.0;
        double lo = 1.0 / tau_max, hi = 1.0 / tau_min;
        double c1 = hi - g * (hi - lo), c2 = lo + g * (hi - lo);
        double f1 = sts_nll(x, y, n, c1), f2 = sts_nll(x, y, n, c2);
        for (int it = 0; it < 300 && hi - lo > 1e-15 * hi; ++it) {
            if (f1 <= f2) {
                hi = c2; c2 = c1; f2 = f1;
                c1 = hi - g * (hi - lo); f1 = sts_nll(x, y, n, c1);
            } else {
                lo = c1; c1 = c2; f1 = f2;
                c2 = lo + g * (hi - lo); f2 = sts_nll(x, y, n, c2);
            }
        }
        /* the interval's ends are candidates too (a minimum on a bound) */
        double best = 0.5 * (lo + hi), fb = sts_nll(x, y, n, best);
        const double ends[2] = {1.0 / tau_max, 1.0 / tau_min};
        for (int e = 0; e < 2; ++e) {
            const double fe = sts_nll(x, y, n, ends[e]);
            if (fe < fb) { fb = fe; best = ends[e]; }
        }
        tau_out[i] = 1.0 / best;
        nll_out[i] = fb;
    }
    free(x);
    free(y);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* a1 + a2.  Confidence head with Sequential Temperature Scaling, survival,  */
/* pre-cap verify length.                                                    */
/*   [DS] "DSpark: a sequential head and a verify budget": the head is a     */
/*   linear projection plus a sigmoid on the drafter hidden state; the       */
/*   product of scores across the block is the survival probability; STS    */
/*   calibrates it.  Reading taken: x = (w.h + bias_b) / tau_i,              */
/*   conf = sigmoid(x), S_0 = 1, S_{k+1} = S_k * conf_k.                      */
/*   [DS] same section and "The confidence scheduler and verify modes":      */
/*   walk down the survival curve and stop where the gain no longer covers   */
/*   the marginal cost c.  Reading taken: L0 = max{k in 0..gamma : S_k >= c}, */
/*   with max of the empty set = 0.                                          */
/* Outputs: conf[b*gamma+i], surv[b*gamma+k-1] = S_{b,k} (k = 1..gamma),     */
/* L0[b], and tie[b] = number of k in 1..gamma with |S_{b,k} - c| < eps.     */
/* ------------------------------------------------------------------------ */
int orc_score(int B, int gamma, int d, int hidden_dtype, const void *hidden,
              const float *w, const float *bias, const float *tau, double c,
              double eps, double *conf, double *surv, int32_t *L0, int32_t *tie)
{
    if (B < 0 || gamma < 1 || d < 1) return -1;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < gamma; ++i) {
            const int64_t row = ((int64_t)b * gamma + i) * d;
            double dot = 0.0;
            for (int j = 0; j < d; ++j) {
                dot += (double)w[j] * elem(hidden, hidden_dtype, row + j);
            }
            double x = (dot + (double)bias[b]) / (double)tau[i];
            conf[b * gamma + i] = 1.0 / (1.0 + exp(-x));
        }
        double S = 1.0; /* S_0 */
        int32_t L = (1.0 >= c) ? 0 : -1;
        int32_t ties = 0;
        for (int k = 1; k <= gamma; ++k) {
            S = S * conf[b * gamma + (k - 1)];
            surv[b * gamma + (k - 1)] = S;
            if (S >= c) L = k; /* the largest qualifying k wins */
            if (fabs(S - c) < eps) ties++;
        }
        if (fabs(1.0 - c) < eps) ties++;
        L0[b] = (L < 0) ? 0 : L;
        tie[b] = ties;
    }
    return 0;
}

/* Fixed-budget mode ([DS] "The confidence scheduler and verify modes",      */
/* the static no-trim arm): every request verifies min(F, gamma) drafts.     */
int orc_fixed_budget(int B, int gamma, int F, int32_t *L)
{
    if (B < 0 || gamma < 1 || F < 0) return -1;
    for (int b = 0; b < B; ++b) L[b] = F < gamma ? F : gamma;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* a3.  Batch-wide token cap: keep the T largest marginal gains.             */
/*   [DS] "Zero-overhead scheduling and kernels" names a verify-length top-k */
/*   schedule.  Reading taken: the candidates are (S_{b,k}, b, k) for        */
/*   1 <= k <= L0_b; if their number exceeds T, keep the first T in the      */
/*   order (S descending, b ascending, k ascending); L_b = number kept in b. */
/*   T < 0 means no cap.                                                     */
/* *tie is set to 1 when the T-th and (T+1)-th kept gains differ by < eps.   */
/* ------------------------------------------------------------------------ */
typedef struct {
    double S;
    int32_t b, k;
} orc_cand;

static int cand_order(const void *pa, const void *pb)
{
    const orc_cand *a = (const orc_cand *)pa, *o = (const orc_cand *)pb;
    if (a->S > o->S) return -1;
    if (a->S < o->S) return 1;
    if (a->b != o->b) return a->b < o->b ? -1 : 1;
    if (a->k != o->k) return a->k < o->k ? -1 : 1;
    return 0;
}

int orc_cap(int B, int gamma, const double *surv, const int32_t *L0, int T,
            double eps, int32_t *L, int32_t *tie)
{
    if (B < 0 || gamma < 1) return -1;
    *tie = 0;
    int64_t n = 0;
    for (int b = 0; b < B; ++b) n += L0[b];
    if (T < 0 || n <= T) {
        for (int b = 0; b < B; ++b) L[b] = L0[b];
        return 0;
    }
    orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(n > 0 ? n : 1));
    if (!cand) return -2;
    int64_t m = 0;
    for (int b = 0; b < B; ++b) {
        for (int k = 1; k <= L0[b]; ++k) {
            cand[m].S = surv[b * gamma + (k - 1)];
            cand[m].b = b;
            cand[m].k = k;
            m++;
        }
    }
    qsort(cand, (size_t)n, sizeof(orc_cand), cand_order);
    for (int b = 0; b < B; ++b) L[b] = 0;
    for (int64_t t = 0; t < T; ++t) L[cand[t].b] += 1;
    if (T > 0 && cand[T - 1].S - cand[T].S < eps) *tie = 1;
    free(cand);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* a4.  Ragged packing by exclusive scan.                                    */
/*   [DS] "Ragged verify under full CUDA graphs": the scheduled verify       */
/*   tokens are front-packed into one buffer and a cu_seqlens-style offset   */
/*   array marks where each request's segment starts.  Reading taken: each   */
/*   request contributes the rows [root, d_1 .. d_L]; draft_off is the       */
/*   exclusive scan of L, row_off the exclusive scan of L + 1; a row's       */
/*   position is seq_len_b + j.  Rows past the packed total (capacity        */
/*   B*(gamma+1)) are padding: id -1, position 0, request -1, index -1.      */
/* ------------------------------------------------------------------------ */
int orc_compact(int B, int gamma, const int32_t *L, const int32_t *draft_tokens,
                const int32_t *last_tokens, const int32_t *seq_lens,
                int32_t *draft_off, int32_t *row_off, int32_t *packed_ids,
                int32_t *packed_pos, int32_t *row_req, int32_t *row_k)
{
    if (B < 0 || gamma < 1) return -1;
    draft_off[0] = 0;
    row_off[0] = 0;
    for (int b = 0; b < B; ++b) {
        draft_off[b + 1] = draft_off[b] + L[b];
        row_off[b + 1] = row_off[b] + L[b] + 1;
    }
    const int64_t cap = (int64_t)B * (gamma + 1);
    for (int64_t r = 0; r < cap; ++r) {
        packed_ids[r] = -1;
        packed_pos[r] = 0;
        row_req[r] = -1;
        row_k[r] = -1;
    }
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j <= L[b]; ++j) {
            const int64_t r = row_off[b] + j;
            int32_t id;
            if (j == 0) id = last_tokens ? last_tokens[b] : -1;
            else id = draft_tokens[(int64_t)b * gamma + (j - 1)];
            packed_ids[r] = id;
            packed_pos[r] = (seq_lens ? seq_lens[b] : 0) + j;
            row_req[r] = b;
            row_k[r] = j;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* a5 + a6.  Verify one request.                                             */
/*   [DS] "Background": the target checks all drafts in one forward, the     */
/*   accepted prefix is committed and one bonus token is emitted.            */
/*   [KC] "The Old Problem with Speculative Decoding" (speculative sampling, */
/*   Chen et al. 2023) and [DS] "Serving DeepSeek-V4 with SGLang" (the       */
/*   output distribution is unchanged): accept draft k with probability     */
/*   r = min(1, p(d)/q(d)); on the first rejection sample from               */
/*   norm(max(0, p - q)); if every kept draft is accepted, sample the bonus  */
/*   from p at row L.                                                        */
/* Readings taken: p = softmax(z_target / Tm), q = softmax(z_draft / Tm);    */
/* q(d) = 0 gives r = 1; a draft id outside [0, V) is rejected (r = 0);      */
/* sampling is the inverse CDF over ascending token index: the smallest x    */
/* with C(x) > u' * Z, C the running sum of the weights and Z their total;   */
/* Z = 0 falls back to p; if rounding leaves no such x, the last x with a    */
/* positive weight.  Tm = 0 is greedy: accept iff d == argmax z_target       */
/* (lowest index on ties) and the emitted token is that argmax.             */
/*                                                                           */
/* tgt: L+1 contiguous rows of V logits; dft: L contiguous rows (unused when */
/* Tm == 0).  u[k], u2[k], u3[k] (u, u', u'') for k = 0..L.  Returns the    */
/* accepted count in *a,                                                     */
/* the correction/bonus token in *tok, p(d_k), q(d_k) for k < L, and in      */
/* *tie the number of near-tie decisions that the outcome depends on.        */
/* ------------------------------------------------------------------------ */
static int64_t argmax_row(const void *row, int dtype, int V)
{
    int64_t best = 0;
    double bv = elem(row, dtype, 0);
    for (int64_t y = 1; y < V; ++y) {
        double v = elem(row, dtype, y);
        if (v > bv) { bv = v; best = y; }
    }
    return best;
}

/* prob[y] = softmax(row / Tm)[y] */
static void softmax_row(const void *row, int dtype, int V, double Tm, double *prob)
{
    double mx = -INFINITY;
    for (int64_t y = 0; y < V; ++y) {
        double v = elem(row, dtype, y);
        if (v > mx) mx = v;
    }
    double s = 0.0;
    for (int64_t y = 0; y < V; ++y) {
        prob[y] = exp((elem(row, dtype, y) - mx) / Tm);
        s += prob[y];
    }
    for (int64_t y = 0; y < V; ++y) prob[y] /= s;
}

/* Tokens per sampling block of the two-level draw (reading, see below). */
#define ORC_SAMPLE_BLOCK 4096

/* Two-level inverse-CDF draw from nonnegative weights wt[0..V-1].
 * Reading taken (the pages do not fix how a token is drawn): ids are split
 * into consecutive blocks of ORC_SAMPLE_BLOCK; the block is the smallest j
 * whose running block mass exceeds u_blk * Z (Z the total), and the token is
 * the smallest x of that block whose running in-block weight exceeds
 * u_tok * (the block's mass).  By the chain rule this draws x with
 * probability wt[x] / Z.  When rounding leaves no crossing, the last block or
 * token with positive weight is taken.  *tie counts draws whose margin to a
 * crossing is below eps_blk * Z (block level) or eps_tok * mass (token level).
 * Returns -1 when every weight is zero. */
static int32_t draw_two_level(const double *wt, int V, double u_blk, double u_tok,
                              double eps_blk, double eps_tok, int32_t *tie)
{
    const int nb = (V + ORC_SAMPLE_BLOCK - 1) / ORC_SAMPLE_BLOCK;
    double *mass = (double *)malloc(sizeof(double) * (size_t)nb);
    if (!mass) return -2;
    double Z = 0.0;
    for (int j = 0; j < nb; ++j) {
        mass[j] = 0.0;
        const int64_t y1 = (int64_t)(j + 1) * ORC_SAMPLE_BLOCK < V ? (int64_t)(j + 1) * ORC_SAMPLE_BLOCK : V;
        for (int64_t y = (int64_t)j * ORC_SAMPLE_BLOCK; y < y1; ++y) mass[j] += wt[y];
        Z += mass[j];
    }
    if (!(Z > 0.0)) { free(mass); return -1; }
    const double t = u_blk * Z;
    int jsel = -1;
    double before = 0.0;
    for (int j = 0; j < nb; ++j) {
        const double after = before + mass[j];
        if (after > t) {
            if (t - before < eps_blk * Z || after - t < eps_blk * Z) (*tie)++;
            jsel = j;
            break;
        }
        before = after;
    }
    if (jsel < 0) {
        (*tie)++;
        for (int j = nb - 1; j >= 0; --j)
            if (mass[j] > 0.0) { jsel = j; break; }
    }
    const double m = mass[jsel];
    free(mass);
    const int64_t y0 = (int64_t)jsel * ORC_SAMPLE_BLOCK;
    const int64_t y1 = y0 + ORC_SAMPLE_BLOCK < V ? y0 + ORC_SAMPLE_BLOCK : V;
    const double t2 = u_tok * m;
    double cum = 0.0;
    for (int64_t x = y0; x < y1; ++x) {
        const double after = cum + wt[x];
        if (after > t2) {
            if (t2 - cum < eps_tok * m || after - t2 < eps_tok * m) (*tie)++;
            return (int32_t)x;
        }
        cum = after;
    }
    (*tie)++;
    for (int64_t x = y1 - 1; x >= y0; --x)
        if (wt[x] > 0.0) return (int32_t)x;
    return (int32_t)y0;
}

int orc_verify_request(int L, int V, int dtype, const int32_t *drafts,
                       const void *tgt, const void *dft, double Tm,
                       const double *u, const double *u2, const double *u3,
                       double eps, double eps_blk, double eps_tok,
                       int32_t *a_out, int32_t *tok_out, double *p_out,
                       double *q_out, int32_t *tie)
{
    if (L < 0 || V < 1 || Tm < 0.0) return -1;
    const size_t es = dtype == 0 ? 4 : 2;
    const char *tbase = (const char *)tgt;
    const char *dbase = (const char *)dft;
    *tie = 0;

    if (Tm == 0.0) {
        int32_t a = L;
        for (int k = 0; k < L; ++k) {
            int64_t g = argmax_row(tbase + (size_t)k * V * es, dtype, V);
            p_out[k] = 0.0;
            q_out[k] = 0.0;
            if (a == L && drafts[k] != g) a = k;
        }
        *a_out = a;
        *tok_out = (int32_t)argmax_row(tbase + (size_t)a * V * es, dtype, V);
        return 0;
    }

    double *P = (double *)malloc(sizeof(double) * (size_t)V);
    double *Q = (double *)malloc(sizeof(double) * (size_t)V);
    double *W = (double *)malloc(sizeof(double) * (size_t)V);
    if (!P || !Q || !W) { free(P); free(Q); free(W); return -2; }

    int32_t a = L;
    for (int k = 0; k < L; ++k) {
        softmax_row(tbase + (size_t)k * V * es, dtype, V, Tm, P);
        softmax_row(dbase + (size_t)k * V * es, dtype, V, Tm, Q);
        const int32_t d = drafts[k];
        double r;
        if (d < 0 || d >= V) {
            p_out[k] = 0.0;
            q_out[k] = 0.0;
            r = 0.0;
        } else {
            p_out[k] = P[d];
            q_out[k] = Q[d];
            r = Q[d] > 0.0 ? fmin(1.0, P[d] / Q[d]) : 1.0;
        }
        if (a == L) {
            if (fabs(u[k] - r) < eps) (*tie)++;
            if (!(u[k] < r)) a = k;
        }
    }

    int32_t tok;
    if (a < L) {
        softmax_row(tbase + (size_t)a * V * es, dtype, V, Tm, P);
        softmax_row(dbase + (size_t)a * V * es, dtype, V, Tm, Q);
        double Z = 0.0;
        for (int64_t y = 0; y < V; ++y) {
            W[y] = fmax(0.0, P[y] - Q[y]);
            Z += W[y];
        }
        if (Z < eps) (*tie)++;
        tok = draw_two_level(W, V, u2[a], u3[a], eps_blk, eps_tok, tie);
        if (tok == -1) tok = draw_two_level(P, V, u2[a], u3[a], eps_blk, eps_tok, tie);
    } else {
        softmax_row(tbase + (size_t)L * V * es, dtype, V, Tm, P);
        tok = draw_two_level(P, V, u2[L], u3[L], eps_blk, eps_tok, tie);
    }
    if (tok < 0) { free(P); free(Q); free(W); return -2; }
    *a_out = a;
    *tok_out = tok;
    free(P); free(Q); free(W);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The outcomes a request admits once every decision inside its tolerance    */
/* window may go either way.  A reduced-precision verify agrees with the     */
/* fp64 definition above except where a decision's fp64 margin is below the  */
/* error it is held to; there either side is a correct outcome.  Reading     */
/* taken for the comparison (the pages fix no precision): an accept test is  */
/* open when |u - r| < eps; a draw may land on any token whose interval of   */
/* the running mass meets the window [t - e, t + e] around its target t,     */
/* e = eps_blk * Z at the block level and eps_tok * (block mass) inside the  */
/* block; a residual mass Z < eps leaves the residual draw and the fallback  */
/* draw from p both open.  Everything else must be met exactly.              */
/* ------------------------------------------------------------------------ */

/* Whether token x is an outcome of the two-level draw from weights wt with */
/* targets (u_blk, u_tok) and windows (eps_blk, eps_tok), as above. */
static int draw_admits(const double *wt, int V, double u_blk, double u_tok, double eps_blk,
                       double eps_tok, int64_t x)
{
    if (x < 0 || x >= V || !(wt[x] > 0.0)) return 0;
    const int nb = (V + ORC_SAMPLE_BLOCK - 1) / ORC_SAMPLE_BLOCK;
    const int jx = (int)(x / ORC_SAMPLE_BLOCK);
    double Z = 0.0, before_x = 0.0, mass_x = 0.0;
    int last_pos = -1;
    for (int j = 0; j < nb; ++j) {
        double m = 0.0;
        const int64_t y1 = (int64_t)(j + 1) * ORC_SAMPLE_BLOCK < V ? (int64_t)(j + 1) * ORC_SAMPLE_BLOCK : V;
        for (int64_t y = (int64_t)j * ORC_SAMPLE_BLOCK; y < y1; ++y) m += wt[y];
        if (j == jx) { before_x = Z; mass_x = m; }
        if (m > 0.0) last_pos = j;
        Z += m;
    }
    const double t = u_blk * Z, e = eps_blk * Z;
    /* block jx: its interval [before, before + mass) meets the window, or it
     * is the fallback (the last block with mass) when no block crosses t */
    const int blk_ok = (before_x <= t + e && before_x + mass_x > t - e) ||
                       (jx == last_pos && t + e >= Z);
    if (!blk_ok) return 0;
    const int64_t y0 = (int64_t)jx * ORC_SAMPLE_BLOCK;
    const int64_t y1 = y0 + ORC_SAMPLE_BLOCK < V ? y0 + ORC_SAMPLE_BLOCK : V;
    const double t2 = u_tok * mass_x, e2 = eps_tok * mass_x;
    double cum = 0.0, cum_x = 0.0;
    int64_t last_tok = -1;
    for (int64_t y = y0; y < y1; ++y) {
        if (y == x) cum_x = cum;
        if (wt[y] > 0.0) last_tok = y;
        cum += wt[y];
    }
    return (cum_x <= t2 + e2 && cum_x + wt[x] > t2 - e2) || (x == last_tok && t2 + e2 >= cum);
}

/* Check a computed outcome (a_g accepted drafts, token tok_g) of one request
 * (arguments as orc_verify_request) against the outcomes it admits.
 * *verdict: 0 admitted; 1 a_g outside [0, L]; 2 a test before a_g rejects
 * outside its window; 3 the test at a_g accepts outside its window; 4 the
 * token is not an outcome of the draw at row a_g; 5 greedy: a_g or the
 * token differs from the argmax rule.  tok_g < 0 checks the accept length
 * alone (a verify whose token is not emitted).  kinds[0..2] count the open decisions
 * on the path the outcome takes: accept tests, residual masses Z < eps, and
 * draws with a block-level or in-block near tie (as draw_two_level counts). */
int orc_check_request(int L, int V, int dtype, const int32_t *drafts,
                      const void *tgt, const void *dft, double Tm,
                      const double *u, const double *u2, const double *u3,
                      double eps, double eps_blk, double eps_tok,
                      int32_t a_g, int32_t tok_g, int32_t *kinds, int32_t *verdict)
{
    if (L < 0 || V < 1 || Tm < 0.0) return -1;
    for (int i = 0; i < 3; ++i) kinds[i] = 0;
    *verdict = 0;
    if (a_g < 0 || a_g > L) { *verdict = 1; return 0; }
    const size_t es = dtype == 0 ? 4 : 2;
    const char *tbase = (const char *)tgt;
    const char *dbase = (const char *)dft;
    if (Tm == 0.0) {
        int32_t a = L;
        for (int k = 0; k < L && a == L; ++k)
            if (drafts[k] != argmax_row(tbase + (size_t)k * V * es, dtype, V)) a = k;
        if (a_g != a || (tok_g >= 0 && tok_g != argmax_row(tbase + (size_t)a * V * es, dtype, V)))
            *verdict = 5;
        return 0;
    }
    double *P = (double *)malloc(sizeof(double) * (size_t)V);
    double *Q = (double *)malloc(sizeof(double) * (size_t)V);
    double *W = (double *)malloc(sizeof(double) * (size_t)V);
    if (!P || !Q || !W) { free(P); free(Q); free(W); return -2; }
    const int last_test = a_g < L ? a_g : L - 1;
    for (int k = 0; k <= last_test; ++k) {
        softmax_row(tbase + (size_t)k * V * es, dtype, V, Tm, P);
        softmax_row(dbase + (size_t)k * V * es, dtype, V, Tm, Q);
        const int32_t d = drafts[k];
        double r = 0.0;
        if (d >= 0 && d < V) r = Q[d] > 0.0 ? fmin(1.0, P[d] / Q[d]) : 1.0;
        const int open = fabs(u[k] - r) < eps;
        kinds[0] += open;
        const int accepts = u[k] < r;
        if (*verdict == 0 && k < a_g && !accepts && !open) *verdict = 2;
        if (*verdict == 0 && k == a_g && accepts && !open) *verdict = 3;
    }
    if (*verdict == 0 && tok_g >= 0) {
        int32_t tie = 0, own;
        softmax_row(tbase + (size_t)a_g * V * es, dtype, V, Tm, P);
        if (a_g < L) {
            softmax_row(dbase + (size_t)a_g * V * es, dtype, V, Tm, Q);
            double Z = 0.0;
            for (int64_t y = 0; y < V; ++y) {
                W[y] = fmax(0.0, P[y] - Q[y]);
                Z += W[y];
            }
            const int zopen = Z < eps;
            kinds[1] += zopen;
            int ok = 0;
            if (Z > 0.0) {
                own = draw_two_level(W, V, u2[a_g], u3[a_g], eps_blk, eps_tok, &tie);
                ok = draw_admits(W, V, u2[a_g], u3[a_g], eps_blk, eps_tok, tok_g);
            }
            if (!(Z > 0.0) || zopen) {
                own = draw_two_level(P, V, u2[a_g], u3[a_g], eps_blk, eps_tok, &tie);
                ok = ok || draw_admits(P, V, u2[a_g], u3[a_g], eps_blk, eps_tok, tok_g);
            }
            if (!ok) *verdict = 4;
        } else {
            own = draw_two_level(P, V, u2[L], u3[L], eps_blk, eps_tok, &tie);
            if (!draw_admits(P, V, u2[L], u3[L], eps_blk, eps_tok, tok_g)) *verdict = 4;
        }
        (void)own;
        kinds[2] += tie;
    }
    free(P); free(Q); free(W);
    return 0;
}

/* The whole batch: request b reads target rows row_off[b] .. row_off[b]+L_b */
/* of the ragged target array and draft rows b*gamma .. b*gamma+L_b-1;       */
/* uniforms come from Philox keyed by (seed, b, k).  Outputs: accept_len,    */
/* num_emitted = a+1, out_tokens[b][0..gamma] = d_0..d_{a-1}, token, -1 pad; */
/* p_tok/q_tok at draft_off[b] + k; seq_lens (if not NULL) += a+1;           */
/* tie[b] as in orc_verify_request.                                          */
/* Request b of the batch (its uniforms u, u2, u3 are scratch of gamma+1). */
static int verify_one(int b, int gamma, int V, int dtype, const int32_t *draft_tokens,
                      const void *draft_logits, const void *target_logits,
                      const int32_t *L, const int32_t *row_off, const int32_t *draft_off,
                      double Tm, uint64_t seed, double eps, double eps_blk, double eps_tok,
                      int32_t *accept_len, int32_t *num_emitted, int32_t *out_tokens,
                      double *p_tok, double *q_tok, int32_t *seq_lens, int32_t *tie,
                      double *u, double *u2, double *u3)
{
    const size_t es = dtype == 0 ? 4 : 2;
    const int Lb = L[b];
    for (int k = 0; k <= Lb; ++k) orc_uniforms(seed, b, k, &u[k], &u2[k], &u3[k]);
    const void *tgt = (const char *)target_logits + (size_t)row_off[b] * V * es;
    const void *dft = (const char *)draft_logits + (size_t)b * gamma * V * es;
    int32_t a, tok;
    const int rc = orc_verify_request(Lb, V, dtype, draft_tokens + (size_t)b * gamma, tgt, dft,
                                      Tm, u, u2, u3, eps, eps_blk, eps_tok, &a, &tok,
                                      p_tok + draft_off[b], q_tok + draft_off[b], &tie[b]);
    if (rc) return rc;
    accept_len[b] = a;
    num_emitted[b] = a + 1;
    for (int j = 0; j <= gamma; ++j) {
        int32_t v = -1;
        if (j < a) v = draft_tokens[(size_t)b * gamma + j];
        else if (j == a) v = tok;
        out_tokens[(size_t)b * (gamma + 1) + j] = v;
    }
    if (seq_lens) seq_lens[b] += a + 1;
    return 0;
}

int orc_verify(int B, int gamma, int V, int dtype, const int32_t *draft_tokens,
               const void *draft_logits, const void *target_logits,
               const int32_t *L, const int32_t *row_off, const int32_t *draft_off,
               double Tm, uint64_t seed, double eps, double eps_blk, double eps_tok,
               int32_t *accept_len, int32_t *num_emitted, int32_t *out_tokens,
               double *p_tok, double *q_tok, int32_t *seq_lens, int32_t *tie)
{
    if (B < 0 || gamma < 1 || V < 1) return -1;
    double *u = (double *)malloc(sizeof(double) * (size_t)(gamma + 1));
    double *u2 = (double *)malloc(sizeof(double) * (size_t)(gamma + 1));
    double *u3 = (double *)malloc(sizeof(double) * (size_t)(gamma + 1));
    if (!u || !u2 || !u3) { free(u); free(u2); free(u3); return -2; }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b)
        rc = verify_one(b, gamma, V, dtype, draft_tokens, draft_logits, target_logits, L,
                        row_off, draft_off, Tm, seed, eps, eps_blk, eps_tok, accept_len,
                        num_emitted, out_tokens, p_tok, q_tok, seq_lens, tie, u, u2, u3);
    free(u);
    free(u2);
    free(u3);
    return rc;
}

#ifdef ORC_OMP
/* The batch verify with the requests spread over the host's threads
 * (OpenMP), for the benchmark's multi-core CPU baseline only.  It is built
 * separately (liboracle_omp.so, -fopenmp -DORC_OMP); the plain library above
 * stays single-threaded.  Requests are independent, so the results are those
 * of orc_verify. */
#include <omp.h>

int orc_omp_threads(int n)
{
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
}

int orc_verify_omp(int B, int gamma, int V, int dtype, const int32_t *draft_tokens,
                   const void *draft_logits, const void *target_logits,
                   const int32_t *L, const int32_t *row_off, const int32_t *draft_off,
                   double Tm, uint64_t seed, double eps, double eps_blk, double eps_tok,
                   int32_t *accept_len, int32_t *num_emitted, int32_t *out_tokens,
                   double *p_tok, double *q_tok, int32_t *seq_lens, int32_t *tie)
{
    if (B < 0 || gamma < 1 || V < 1) return -1;
    int rc = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : rc)
    for (int b = 0; b < B; ++b) {
        double *u = (double *)malloc(sizeof(double) * (size_t)(gamma + 1) * 3);
        if (!u) {
            rc |= 2;
            continue;
        }
        rc |= verify_one(b, gamma, V, dtype, draft_tokens, draft_logits, target_logits, L,
                         row_off, draft_off, Tm, seed, eps, eps_blk, eps_tok, accept_len,
                         num_emitted, out_tokens, p_tok, q_tok, seq_lens, tie, u,
                         u + gamma + 1, u + 2 * (gamma + 1)) != 0;
        free(u);
    }
    return rc ? -2 : 0;
}
#endif
