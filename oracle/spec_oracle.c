/*
 * spec_oracle.c -- CPU oracle for the target-side verification step of speculative decoding.
 *
 * TEST INFRASTRUCTURE.  This file is the plain, slow, scalar reference that the CUDA library is
 * checked against.  Only the test suite, the package's smoke check and the benchmark's CPU
 * baseline leg load it; the product path never does.  It shares no code with the CUDA library.
 *
 * Arithmetic: IEEE double throughout (inputs are widened exactly from fp32 / bf16 / fp16),
 * scalar loops in index order, no blocking, no reordering.  Compile with -ffp-contract=off.
 *
 * Source of the method -- "Speculative Decoding in Production: From Draft Models to EAGLE-3
 * Dynamic Trees for 3x-5x Lossless Acceleration" (blog.llmgo.top), section I.1 "Verification
 * via Modified Rejection Sampling":
 *   step 1  acceptance probability  alpha = min(1, p(x_k) / q(x_k))
 *   step 2  r ~ Uniform(0,1); accept x_k iff r <= alpha, otherwise reject and stop verifying
 *           the later draft tokens
 *   step 3  after a rejection at position k, resample from
 *           max(0, p(x) - q(x)) / sum_x max(0, p(x) - q(x))
 *   the "Invariance Theorem" paragraph below it: the emitted tokens follow p exactly, for
 *   greedy decoding as well as temperature sampling.
 * Tree verification -- same page, section III.2 "The Tree Attention Verification Mechanism"
 * (the branch whose tokens match is accepted, a rejected sibling branch is skipped), and
 * "Speculative Decoding with Medusa, EAGLE and vLLM" (vikram-blog.pages.dev), "System Topology
 * & Data Flow" diagram (branch A accepted, branch B rejected).
 *
 * Readings where the pages are silent (each one also listed in the design notes):
 *   R1  p = softmax(logits / T) with the row maximum subtracted; T = 0 means greedy.
 *   R2  alpha = 1 when q(x_k) == 0 (p/0 taken as +inf) or p(x_k) >= q(x_k).
 *   R3  r in (0, 1]; u in [0, 1); one u per request serves both the residual and the bonus draw.
 *   R4  inverse-CDF sampling: the smallest i with C_i = sum_{t<=i} w_t > u * S (strict), so a
 *       zero-weight token is never drawn; if rounding leaves no such i, the largest i with w_i > 0.
 *   R5  if the residual mass S is not positive, draw from p at that position instead (flagged).
 *   R6  all K drafts accepted: a bonus token is drawn from p at row K (the (K+1)-th target row).
 *   R7  greedy: argmax over the raw logits, lowest index on ties; accept x_k iff it equals the
 *       target argmax; the emitted token after the accepted prefix is the argmax of that row.
 *   R8  n-gram prompt lookup: q is one-hot at the draft token.
 *   R9  tree: from the root, move to the child whose token equals the argmax of the current
 *       node's row (lowest node index if several), until no child matches; the final token is
 *       the argmax of the last node's row.
 *   R10 flagged ties, in two tiers.  Strict (tol = 1e-6, the stated band): |r_k - alpha_k| <= tol
 *       at an evaluated position, or u within tol of C_{i*-1}/S or C_{i*}/S at the drawn index
 *       i*.  Widened (reported apart): for the draft-model residual max(0, p - q), whose total
 *       S < 1 comes from cancelling p against q, its normalised CDF is resolved in fp32 only to
 *       about tol / S, so a crossing within tol / S of u that is not within tol is flagged in a
 *       second tier.  A flagged draw admits every positive-weight token whose CDF interval comes
 *       within the band of u; oracle_chain_draw_rows gives the weights and the normalised CDF for
 *       that check.  In the widened tier a token whose residual weight is 0 only by a margin below
 *       that resolution (p_t - q_t > -(tol / 2)(p_t + q_t), the per-token precision the band tol / S
 *       stands for) is admissible too; the draw rows give that bound as wmax.  A flagged accept
 *       test admits either decision; for the tree walk oracle_tree_sample_alt gives the outcome of
 *       the opposite decision.
 *   R11 invalid input: a draft token outside [0, V), a logits row holding NaN (or, when a softmax
 *       is taken, +inf, or only -inf), or a malformed parent array sets an error bit (every bit
 *       that applies, all rows checked); the request then accepts nothing and emits no token (-1).
 *   R12 tree layout: node 0 is the root, parents[0] = -1, 0 <= parents[i] < i; row n of the
 *       logits scores the children of node n.
 *   R13-R15 the stochastic tree walk: see the section "stochastic tree verification" below.
 *   R18 per-request temperature (the x078.com page's production section sets the temperature per
 *       request): with a temperatures array, request b uses temps[b] (0 = greedy for that
 *       request); NaN, a negative value or infinity fails that request (ORE_BAD_TEMP alone).  On
 *       the chain, the n-gram chain and the tree walk.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

/* per-request / per-position tie flags (R10, R5): strict tier, zero residual, widened tier */
enum { ORF_ACCEPT_TIE = 1, ORF_CDF_TIE = 2, ORF_ZERO_RESIDUAL = 4, ORF_CDF_TIE_WIDE = 8,
       ORF_ACCEPT_TIE_WIDE = 16 };
/* per-request error bits (R11) */
enum { ORE_BAD_TOKEN = 1, ORE_NONFINITE = 2, ORE_BAD_TREE = 8, ORE_BAD_TEMP = 16 };

/* ---------------------------------------------------------------- exact input widening ---- */
static double half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + man), ex - 25);
    return sign ? -v : v;
}

double oracle_load(const void *base, int dtype, size_t i)
{
    if (dtype == OR_F32)
        return (double)((const float *)base)[i];
    if (dtype == OR_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return half_to_double(((const uint16_t *)base)[i]);
}

static void load_row(const void *base, int dtype, size_t row, int V, double *out)
{
    for (int i = 0; i < V; i++)
        out[i] = oracle_load(base, dtype, row * (size_t)V + (size_t)i);
}

/* ------------------------------------------------------------------- temperature softmax ---- */
/* R1: p_i = exp((l_i - m) / T) / sum_j exp((l_j - m) / T), m = max_j l_j.
 * Returns ORE_NONFINITE (and leaves p unspecified) for NaN, +inf, or an all -inf row. */
int oracle_softmax(const double *l, int V, double T, double *p)
{
    double m = -INFINITY;
    for (int i = 0; i < V; i++) {
        if (isnan(l[i]) || l[i] == INFINITY)
            return ORE_NONFINITE;
        if (l[i] > m)
            m = l[i];
    }
    if (m == -INFINITY)
        return ORE_NONFINITE;
    double Z = 0.0;
    for (int i = 0; i < V; i++) {
        p[i] = exp((l[i] - m) / T);
        Z += p[i];
    }
    for (int i = 0; i < V; i++)
        p[i] = p[i] / Z;
    return 0;
}

/* R7: first index of the maximum (strict > keeps the lowest index on ties). */
int oracle_argmax(const double *l, int V)
{
    int a = 0;
    for (int i = 1; i < V; i++)
        if (l[i] > l[a])
            a = i;
    return a;
}

static int row_has_nan(const double *l, int V)
{
    for (int i = 0; i < V; i++)
        if (isnan(l[i]))
            return 1;
    return 0;
}

/* ------------------------------------------------------------------- inverse-CDF sampling ---- */
/* R4: smallest i with C_i > u * S; S = sum of w.  Returns -1 when S is not positive.
 * *flag is set when u lies within tol of C_{i-1}/S or C_i/S (R10). */
int oracle_inverse_cdf(const double *w, int V, double u, double tol, double *S_out, int *flag)
{
    double S = 0.0;
    for (int i = 0; i < V; i++)
        S += w[i];
    *S_out = S;
    *flag = 0;
    if (!(S > 0.0))
        return -1;
    double target = u * S, C = 0.0, Cprev = 0.0;
    int pick = -1;
    for (int i = 0; i < V; i++) {
        Cprev = C;
        C += w[i];
        if (C > target) {
            pick = i;
            break;
        }
    }
    if (pick < 0) { /* rounding left u*S at or above the total: the last positive weight */
        for (int i = V - 1; i >= 0; i--)
            if (w[i] > 0.0) {
                pick = i;
                break;
            }
        *flag = 1;
        return pick;
    }
    if (fabs(Cprev / S - u) <= tol || fabs(C / S - u) <= tol)
        *flag = 1;
    return pick;
}

/* ------------------------------------------------------ chain verification on probabilities ---- */
/*
 * p: [K+1][V] target probabilities (row K = bonus row), q: [K][V] draft probabilities,
 * x: [K] draft tokens (must lie in [0, V)), r: [K], u: scalar.
 * Outputs (all per request):
 *   n_acc, out_tokens[K+1] (accepted prefix, then the drawn token, then -1),
 *   alpha[K] (step 1 at every position), cand[K+1] (the token step 3 would draw at position k,
 *   and the bonus draw at K), mass[K+1] (the residual mass S at k; sum of p at K),
 *   pos_flag[K+1] (CDF tie / zero-residual at k), req_flag (flags of the evaluated positions).
 */
/* The weights of the draw at position k (p: [K+1][V], q: [K][V]): the step-3 residual
 * max(0, p_k - q_k) at a draft position, p_K itself at the bonus row (R6). */
static void draw_weights(int K, int V, const double *p, const double *q, int k, double *w)
{
    const double *pk = p + (size_t)k * V;
    if (k < K) {
        const double *qk = q + (size_t)k * V;
        for (int i = 0; i < V; i++) { /* step 3 residual */
            double d = pk[i] - qk[i];
            w[i] = d > 0.0 ? d : 0.0;
        }
    } else {
        for (int i = 0; i < V; i++) /* R6 bonus: draw from p */
            w[i] = pk[i];
    }
}

static void verify_probs_impl(int K, int V, const double *p, const double *q, const int *x,
                              const float *r, float u, double tol, int scale_band, int *n_acc,
                              int *out_tokens, double *alpha, int *cand, double *mass,
                              int *pos_flag, int *req_flag)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    *req_flag = 0;
    for (int k = 0; k <= K; k++) {
        const double *pk = p + (size_t)k * V;
        int f = 0;
        if (k < K) {
            double px = pk[x[k]], qx = q[(size_t)k * V + x[k]];
            alpha[k] = (qx == 0.0 || px >= qx) ? 1.0 : px / qx; /* step 1, R2 */
        }
        draw_weights(K, V, p, q, k, w);
        double S;
        int fl, flw = 0;
        int c = oracle_inverse_cdf(w, V, (double)u, tol, &S, &fl);
        mass[k] = S;
        if (c < 0) { /* R5: no residual mass left, draw from p instead */
            double S2;
            c = oracle_inverse_cdf(pk, V, (double)u, tol, &S2, &fl);
            f |= ORF_ZERO_RESIDUAL;
        } else if (scale_band && k < K && S < 1.0 && !fl) {
            /* R10, widened tier: the residual max(0, p - q) cancels where p and q overlap; its
             * normalised CDF is resolved only to about tol / S */
            double S3;
            oracle_inverse_cdf(w, V, (double)u, tol / S, &S3, &flw);
        }
        if (fl)
            f |= ORF_CDF_TIE;
        if (flw)
            f |= ORF_CDF_TIE_WIDE;
        cand[k] = c;
        pos_flag[k] = f;
    }
    /* step 2: accept while r_k <= alpha_k, stop at the first rejection */
    int n = 0;
    while (n < K) {
        if (fabs((double)r[n] - alpha[n]) <= tol)
            *req_flag |= ORF_ACCEPT_TIE;
        if ((double)r[n] <= alpha[n])
            n++;
        else
            break;
    }
    *req_flag |= pos_flag[n];
    *n_acc = n;
    for (int i = 0; i <= K; i++)
        out_tokens[i] = i < n ? x[i] : (i == n ? cand[n] : -1);
    free(w);
}

/* Draft-model chain on probabilities (the residual tie band scales with 1 / S, reading R10). */
void oracle_verify_probs(int K, int V, const double *p, const double *q, const int *x,
                         const float *r, float u, double tol, int *n_acc, int *out_tokens,
                         double *alpha, int *cand, double *mass, int *pos_flag, int *req_flag)
{
    verify_probs_impl(K, V, p, q, x, r, u, tol, 1, n_acc, out_tokens, alpha, cand, mass, pos_flag,
                      req_flag);
}

static void fail_request(int K, int *n_acc, int *out_tokens, double *alpha, int *cand,
                         double *mass)
{
    *n_acc = 0;
    for (int i = 0; i <= K; i++) {
        out_tokens[i] = -1;
        cand[i] = -1;
        mass[i] = 0.0;
        if (i < K)
            alpha[i] = 0.0;
    }
}

/* R7, greedy chain on logits rows lt: [K+1][V]. */
static int greedy_chain(int K, int V, const double *lt, const int *x, int *n_acc,
                        int *out_tokens, double *alpha, int *cand, double *mass)
{
    for (int k = 0; k <= K; k++) {
        if (row_has_nan(lt + (size_t)k * V, V))
            return ORE_NONFINITE;
        cand[k] = oracle_argmax(lt + (size_t)k * V, V);
        mass[k] = 1.0; /* one-hot p minus one-hot q leaves mass 1 (or p itself at the bonus) */
        if (k < K)
            alpha[k] = (x[k] == cand[k]) ? 1.0 : 0.0;
    }
    int n = 0;
    while (n < K && x[n] == cand[n])
        n++;
    *n_acc = n;
    for (int i = 0; i <= K; i++)
        out_tokens[i] = i < n ? x[i] : (i == n ? cand[n] : -1);
    return 0;
}

/* R18 per-request temperature: request b's temperature (temps[b] when given, else T), and
 * whether it is valid (not NaN, negative or infinite). */
static int request_temperature(float T, const float *temps, int b, float *Tb)
{
    *Tb = temps ? temps[b] : T;
    return (*Tb >= 0.0f) && !isinf(*Tb);
}

/*
 * Chain verification on logits (draft model / EAGLE head: the draft side is logits).
 * target: [B][K+1][V], draft: [B][K][V] (ignored when T == 0), dtype OR_*.
 * temps: NULL, or [B] per-request temperatures used instead of T (R18: 0 = greedy for that
 * request; NaN, negative or infinite fails the request with ORE_BAD_TEMP alone).
 * Per request b the outputs are laid out as in oracle_verify_probs:
 *   n_acc[B], out_tokens[B][K+1], alpha[B][K], cand[B][K+1], mass[B][K+1],
 *   pos_flag[B][K+1], req_flag[B], err[B].
 * Requests [b0, b1) only are processed (lets a caller split the batch across threads).
 */
void oracle_verify_chain(int dtype, const void *target, const void *draft, int B, int K, int V,
                         float T, const float *temps, const int *x, const float *r,
                         const float *u, double tol,
                         int b0, int b1, int *n_acc, int *out_tokens, double *alpha, int *cand,
                         double *mass, int *pos_flag, int *req_flag, int *err)
{
    size_t rowsT = (size_t)(K + 1) * V, rowsD = (size_t)K * V;
    double *lt = (double *)malloc(sizeof(double) * (rowsT ? rowsT : 1));
    double *ld = (double *)malloc(sizeof(double) * (rowsD ? rowsD : 1));
    double *p = (double *)malloc(sizeof(double) * (rowsT ? rowsT : 1));
    double *q = (double *)malloc(sizeof(double) * (rowsD ? rowsD : 1));
    (void)B;
    for (int b = b0; b < b1; b++) {
        const int *xb = x + (size_t)b * K;
        int *o_n = n_acc + b, *o_tok = out_tokens + (size_t)b * (K + 1);
        double *o_al = alpha + (size_t)b * K, *o_ms = mass + (size_t)b * (K + 1);
        int *o_cd = cand + (size_t)b * (K + 1), *o_pf = pos_flag + (size_t)b * (K + 1);
        int e = 0;
        req_flag[b] = 0;
        for (int k = 0; k < K + 1; k++)
            o_pf[k] = 0;
        for (int k = 0; k < K; k++)
            if (xb[k] < 0 || xb[k] >= V)
                e |= ORE_BAD_TOKEN;
        float Tb;
        if (!request_temperature(T, temps, b, &Tb)) {
            e = ORE_BAD_TEMP;
        } else if (Tb == 0.0f) {
            for (int k = 0; k <= K; k++)
                load_row(target, dtype, (size_t)b * (K + 1) + k, V, lt + (size_t)k * V);
            e |= greedy_chain(K, V, lt, xb, o_n, o_tok, o_al, o_cd, o_ms);
        } else {
            for (int k = 0; k <= K; k++)
                load_row(target, dtype, (size_t)b * (K + 1) + k, V, lt + (size_t)k * V);
            for (int k = 0; k < K; k++)
                load_row(draft, dtype, (size_t)b * K + k, V, ld + (size_t)k * V);
            for (int k = 0; k <= K; k++)
                e |= oracle_softmax(lt + (size_t)k * V, V, (double)Tb, p + (size_t)k * V);
            for (int k = 0; k < K; k++)
                e |= oracle_softmax(ld + (size_t)k * V, V, (double)Tb, q + (size_t)k * V);
            if (!e)
                oracle_verify_probs(K, V, p, q, xb, r + (size_t)b * K, u[b], tol, o_n, o_tok, o_al,
                                    o_cd, o_ms, o_pf, req_flag + b);
        }
        if (e) {
            fail_request(K, o_n, o_tok, o_al, o_cd, o_ms);
            req_flag[b] = 0;
        }
        err[b] = e;
    }
    free(lt);
    free(ld);
    free(p);
    free(q);
}

/*
 * n-gram (prompt lookup) verification, R8: q_k is one-hot at x_k.  This is the general path of
 * oracle_verify_probs with explicit one-hot q rows.  Same layout (and temps) as
 * oracle_verify_chain.
 */
void oracle_verify_ngram(int dtype, const void *target, int B, int K, int V, float T,
                         const float *temps, const int *x, const float *r, const float *u,
                         double tol, int b0, int b1,
                         int *n_acc, int *out_tokens, double *alpha, int *cand, double *mass,
                         int *pos_flag, int *req_flag, int *err)
{
    size_t rowsT = (size_t)(K + 1) * V, rowsD = (size_t)K * V;
    double *lt = (double *)malloc(sizeof(double) * (rowsT ? rowsT : 1));
    double *p = (double *)malloc(sizeof(double) * (rowsT ? rowsT : 1));
    double *q = (double *)malloc(sizeof(double) * (rowsD ? rowsD : 1));
    (void)B;
    for (int b = b0; b < b1; b++) {
        const int *xb = x + (size_t)b * K;
        int *o_n = n_acc + b, *o_tok = out_tokens + (size_t)b * (K + 1);
        double *o_al = alpha + (size_t)b * K, *o_ms = mass + (size_t)b * (K + 1);
        int *o_cd = cand + (size_t)b * (K + 1), *o_pf = pos_flag + (size_t)b * (K + 1);
        int e = 0;
        req_flag[b] = 0;
        for (int k = 0; k < K + 1; k++)
            o_pf[k] = 0;
        for (int k = 0; k < K; k++)
            if (xb[k] < 0 || xb[k] >= V)
                e |= ORE_BAD_TOKEN;
        float Tb;
        if (!request_temperature(T, temps, b, &Tb)) {
            e = ORE_BAD_TEMP;
        } else if (Tb == 0.0f) {
            for (int k = 0; k <= K; k++)
                load_row(target, dtype, (size_t)b * (K + 1) + k, V, lt + (size_t)k * V);
            e |= greedy_chain(K, V, lt, xb, o_n, o_tok, o_al, o_cd, o_ms);
        } else {
            for (int k = 0; k <= K; k++)
                load_row(target, dtype, (size_t)b * (K + 1) + k, V, lt + (size_t)k * V);
            for (int k = 0; k <= K; k++)
                e |= oracle_softmax(lt + (size_t)k * V, V, (double)Tb, p + (size_t)k * V);
            for (size_t i = 0; i < rowsD; i++)
                q[i] = 0.0;
            for (int k = 0; k < K && !e; k++)
                q[(size_t)k * V + xb[k]] = 1.0;
            if (!e)
                verify_probs_impl(K, V, p, q, xb, r + (size_t)b * K, u[b], tol, 0, o_n, o_tok,
                                  o_al, o_cd, o_ms, o_pf, req_flag + b);
        }
        if (e) {
            fail_request(K, o_n, o_tok, o_al, o_cd, o_ms);
            req_flag[b] = 0;
        }
        err[b] = e;
    }
    free(lt);
    free(p);
    free(q);
}

/*
 * n-gram shortcut on probabilities, written directly from R8: with q one-hot at x_k,
 * alpha_k = min(1, p_k(x_k)) and the residual is p_k with x_k's entry zeroed; the bonus draws
 * from p_K.  Used by the tests to pin the general path; same outputs as oracle_verify_probs.
 */
void oracle_verify_ngram_direct(int K, int V, const double *p, const int *x, const float *r,
                                float u, double tol, int *n_acc, int *out_tokens, double *alpha,
                                int *cand, double *mass, int *pos_flag, int *req_flag)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    *req_flag = 0;
    for (int k = 0; k <= K; k++) {
        const double *pk = p + (size_t)k * V;
        int f = 0;
        for (int i = 0; i < V; i++)
            w[i] = pk[i];
        if (k < K) {
            alpha[k] = pk[x[k]] >= 1.0 ? 1.0 : pk[x[k]];
            w[x[k]] = 0.0;
        }
        double S;
        int fl;
        int c = oracle_inverse_cdf(w, V, (double)u, tol, &S, &fl);
        mass[k] = S;
        if (c < 0) {
            double S2;
            c = oracle_inverse_cdf(pk, V, (double)u, tol, &S2, &fl);
            f |= ORF_ZERO_RESIDUAL;
        }
        if (fl)
            f |= ORF_CDF_TIE;
        cand[k] = c;
        pos_flag[k] = f;
    }
    int n = 0;
    while (n < K) {
        if (fabs((double)r[n] - alpha[n]) <= tol)
            *req_flag |= ORF_ACCEPT_TIE;
        if ((double)r[n] <= alpha[n])
            n++;
        else
            break;
    }
    *req_flag |= pos_flag[n];
    *n_acc = n;
    for (int i = 0; i <= K; i++)
        out_tokens[i] = i < n ? x[i] : (i == n ? cand[n] : -1);
    free(w);
}

/* Cumulative sums of w in index order (as oracle_inverse_cdf sums them) divided by their total:
 * cdf[i] = (w[0] + ... + w[i]) / S.  Returns S. */
static double normalised_cdf(const double *w, int V, double *cdf)
{
    double S = 0.0, C = 0.0;
    for (int i = 0; i < V; i++)
        S += w[i];
    for (int i = 0; i < V; i++) {
        C += w[i];
        cdf[i] = S > 0.0 ? C / S : 0.0;
    }
    return S;
}

/* The largest weight of each token of the residual max(0, p - q) when p and q are each known to a
 * relative tol / 2 (the widened tier of R10): max(0, p_i - q_i + (tol / 2)(p_i + q_i)). */
static void residual_wmax(const double *p, const double *q, int V, double tol, double *wmax)
{
    for (int i = 0; i < V; i++) {
        double d = p[i] - q[i] + 0.5 * tol * (p[i] + q[i]);
        wmax[i] = d > 0.0 ? d : 0.0;
    }
}

/*
 * The draws of request b, for checking a flagged tie (R10): for every position k = 0..K, the
 * weights the draw at k uses, w[k][i] (the step-3 residual at a draft position, p_K at the bonus
 * row, p_k itself when the residual is empty, R5), and cdf[k][i], their normalised cumulative
 * sums.  Token t is drawn at k exactly when u lies in [cdf[k][t-1], cdf[k][t]) (cdf[k][-1] = 0).
 * wmax[k][i]: the largest weight of token i within the widened tier's precision (residual_wmax) at
 * a draft-model residual position, w[k][i] elsewhere (no cancellation there).
 * ngram != 0 takes q one-hot at the draft tokens (R8; draft unused).  T > 0.  Layout of the
 * inputs as oracle_verify_chain; w, cdf and wmax are [K+1][V].  Returns the request's error bits
 * (the outputs are unspecified when they are not 0).
 */
int oracle_chain_draw_rows(int dtype, const void *target, const void *draft, int ngram, int K,
                           int V, float T, const int *x, int b, double tol, double *w_out,
                           double *cdf_out, double *wmax_out)
{
    size_t rowsT = (size_t)(K + 1) * V, rowsD = (size_t)K * V;
    double *l = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    double *p = (double *)malloc(sizeof(double) * (rowsT ? rowsT : 1));
    double *q = (double *)malloc(sizeof(double) * (rowsD ? rowsD : 1));
    const int *xb = x + (size_t)b * K;
    int e = 0;
    for (int k = 0; k < K; k++)
        if (xb[k] < 0 || xb[k] >= V)
            e |= ORE_BAD_TOKEN;
    for (int k = 0; k <= K; k++) {
        load_row(target, dtype, (size_t)b * (K + 1) + k, V, l);
        e |= oracle_softmax(l, V, (double)T, p + (size_t)k * V);
    }
    for (size_t i = 0; i < rowsD; i++)
        q[i] = 0.0;
    for (int k = 0; k < K && !e; k++) {
        if (ngram) {
            q[(size_t)k * V + xb[k]] = 1.0;
        } else {
            load_row(draft, dtype, (size_t)b * K + k, V, l);
            e |= oracle_softmax(l, V, (double)T, q + (size_t)k * V);
        }
    }
    for (int k = 0; k <= K && !e; k++) {
        double *w = w_out + (size_t)k * V, *wm = wmax_out + (size_t)k * V;
        draw_weights(K, V, p, q, k, w);
        double S = 0.0;
        for (int i = 0; i < V; i++)
            S += w[i];
        if (!(S > 0.0)) /* R5 */
            for (int i = 0; i < V; i++)
                w[i] = p[(size_t)k * V + i];
        normalised_cdf(w, V, cdf_out + (size_t)k * V);
        if (!ngram && k < K && S > 0.0)
            residual_wmax(p + (size_t)k * V, q + (size_t)k * V, V, tol, wm);
        else
            for (int i = 0; i < V; i++)
                wm[i] = w[i];
    }
    free(l);
    free(p);
    free(q);
    return e;
}

/* ---------------------------------------------------------------------- greedy tree walk ---- */
/* Parent array check: parents[0] == -1, 0 <= parents[i] < i; node tokens in [0, V) (root
 * excluded). */
int oracle_tree_check(int N1, int V, const int *parents, const int *tokens)
{
    if (N1 < 1 || parents[0] != -1)
        return ORE_BAD_TREE;
    for (int i = 1; i < N1; i++) {
        if (parents[i] < 0 || parents[i] >= i)
            return ORE_BAD_TREE;
        if (tokens[i] < 0 || tokens[i] >= V)
            return ORE_BAD_TOKEN;
    }
    return 0;
}

/* R9: walk from the root along children whose token equals the argmax of the current node's
 * row.  amax[n] = argmax of row n.  Outputs: *accept_len, path[N1] (root first, -1 padded),
 * out_tokens[N1] (accepted tokens then the final argmax token, -1 padded). */
void oracle_tree_walk(int N1, const int *parents, const int *tokens, const int *amax,
                      int *accept_len, int *path, int *out_tokens)
{
    int cur = 0, len = 0;
    for (int i = 0; i < N1; i++) {
        path[i] = -1;
        out_tokens[i] = -1;
    }
    path[0] = 0;
    for (int step = 0; step < N1; step++) {
        int a = amax[cur], next = -1;
        for (int c = cur + 1; c < N1; c++)
            if (parents[c] == cur && tokens[c] == a) {
                next = c;
                break;
            }
        if (next < 0)
            break;
        out_tokens[len] = tokens[next];
        len++;
        path[len] = next;
        cur = next;
    }
    out_tokens[len] = amax[cur];
    *accept_len = len;
}

/* Brute force over every node v: v is reachable when every edge u->w on the root-to-v path has
 * tokens[w] == amax[u].  Returns the deepest reachable node (lowest index among the deepest)
 * and its depth in *depth.  Independent of the walk; used to pin it. */
int oracle_tree_bruteforce(int N1, const int *parents, const int *tokens, const int *amax,
                           int *depth)
{
    int best = 0, best_d = 0;
    for (int v = 1; v < N1; v++) {
        int ok = 1, d = 0;
        for (int w = v; w != 0; w = parents[w]) {
            if (tokens[w] != amax[parents[w]]) {
                ok = 0;
                break;
            }
            d++;
        }
        if (ok && d > best_d) {
            best = v;
            best_d = d;
        }
    }
    *depth = best_d;
    return best;
}

/* Greedy tree verification on logits: target [B][N+1][V]; node_tokens, parents [B][N+1].
 * Outputs: accept_len[B], path[B][N+1], out_tokens[B][N+1], amax[B][N+1], err[B]. */
void oracle_verify_tree_greedy(int dtype, const void *target, int B, int N, int V,
                               const int *node_tokens, const int *parents, int b0, int b1,
                               int *accept_len, int *path, int *out_tokens, int *amax, int *err)
{
    int N1 = N + 1;
    double *row = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    (void)B;
    for (int b = b0; b < b1; b++) {
        const int *pb = parents + (size_t)b * N1, *tb = node_tokens + (size_t)b * N1;
        int *ab = amax + (size_t)b * N1;
        int e = oracle_tree_check(N1, V, pb, tb);
        for (int n = 0; n < N1; n++) {
            load_row(target, dtype, (size_t)b * N1 + n, V, row);
            if (row_has_nan(row, V))
                e |= ORE_NONFINITE;
            ab[n] = oracle_argmax(row, V);
        }
        if (e) {
            accept_len[b] = 0;
            for (int i = 0; i < N1; i++) {
                path[(size_t)b * N1 + i] = -1;
                out_tokens[(size_t)b * N1 + i] = -1;
            }
        } else {
            oracle_tree_walk(N1, pb, tb, ab, accept_len + b, path + (size_t)b * N1,
                             out_tokens + (size_t)b * N1);
        }
        err[b] = e;
    }
    free(row);
}

/* ------------------------------------------------------------ stochastic tree verification ---- */
/*
 * R13 (tree, T > 0): the step of section I.1 applied to every sibling in turn.  At a node, p is
 * the target distribution of the node's row and q the draft distribution of the node's draft row
 * (the distribution its children were drawn from; siblings are read as independent draws from
 * the same q).  Children are tested in ascending node index.  Child c with token x is accepted
 * when r[c] <= alpha = min(1, p(x) / q(x)) (R2 when q(x) == 0 or p(x) >= q(x)), and the walk
 * moves to c.  A rejected child replaces the target by its residual,
 *     p <- max(0, p - q) / sum_i max(0, p_i - q_i),
 * and the next sibling is tested against the new p and the same q.  When no child is accepted,
 * or the node has none, the final token is drawn from the current p with the request's u (R4).
 * A chain (one child per node) is exactly the chain verification above.
 * R14: the mass R reported for a request is the product of the residual sums met at its final
 * node (1 when nothing was rejected there).  An accept test, and the final draw, is flagged in
 * the strict tier within tol, and in the widened tier within tol / R (the resolution of the
 * residual in fp32, as in R10) but not tol.  A residual sum that is not positive stops the
 * sibling tests; the draw is then taken from the node's own p (R5, flagged).
 * R15: the walk reads only the rows of the nodes it visits (a node's draft row only when it has
 * children); a non-finite value in another row is not seen.  T == 0 is the greedy walk of R9,
 * with alpha = 1 for the matching child and 0 for the siblings tested before it.
 */

/* Supplies the probability rows of one node: p always, q when need_q.  Returns error bits. */
typedef int (*tree_rows_fn)(void *ctx, int node, int need_q, double *p, double *q);

static void tree_fail(int N1, int *accept_len, int *path, int *out_tokens, double *alpha,
                      double *mass)
{
    *accept_len = 0;
    *mass = 0.0;
    for (int i = 0; i < N1; i++) {
        path[i] = -1;
        out_tokens[i] = -1;
        alpha[i] = -1.0;
    }
}

/* One request.  parents / tokens: [N1]; r: [N1] (r[c] is used when child c is tested; r[0] is
 * unused); outputs as oracle_verify_tree_sample.  flip != 0 decides the first flagged accept test
 * (either tier) the opposite way.  draw_w / draw_cdf (NULL to skip): [V], the final draw's weights
 * and their normalised cumulative sums.  Returns error bits (outputs failed when set). */
static int tree_sample_walk(int N1, int V, tree_rows_fn rows, void *ctx, const int *parents,
                            const int *tokens, const float *r, float u, double tol, int flip,
                            int *accept_len, int *path, int *out_tokens, double *alpha,
                            double *mass, int *req_flag, double *draw_w, double *draw_cdf,
                            double *draw_wmax)
{
    size_t n = (size_t)(V > 0 ? V : 1);
    double *p0 = (double *)malloc(sizeof(double) * n), *p = (double *)malloc(sizeof(double) * n);
    double *q = (double *)malloc(sizeof(double) * n), *w = (double *)malloc(sizeof(double) * n);
    double *pprev = (double *)malloc(sizeof(double) * n); /* the target before the last rejection */
    double Slast = 1.0;
    int e = 0, cur = 0, len = 0;
    *req_flag = 0;
    for (int i = 0; i < N1; i++) {
        path[i] = -1;
        out_tokens[i] = -1;
        alpha[i] = -1.0;
    }
    path[0] = 0;
    for (int depth = 0; depth < N1; depth++) {
        int has_kids = 0;
        for (int c = cur + 1; c < N1; c++)
            if (parents[c] == cur)
                has_kids = 1;
        e = rows(ctx, cur, has_kids, p0, q);
        if (e)
            break;
        for (int i = 0; i < V; i++)
            p[i] = p0[i];
        double R = 1.0;
        int next = -1, empty = 0;
        for (int c = cur + 1; c < N1 && next < 0 && !empty; c++) {
            if (parents[c] != cur)
                continue;
            int x = tokens[c];
            double a = (q[x] == 0.0 || p[x] >= q[x]) ? 1.0 : p[x] / q[x]; /* step 1, R2 */
            alpha[c] = a;
            if (fabs((double)r[c] - a) <= tol)
                *req_flag |= ORF_ACCEPT_TIE;
            else if (fabs((double)r[c] - a) <= tol / R)
                *req_flag |= ORF_ACCEPT_TIE_WIDE;
            int acc = (double)r[c] <= a; /* step 2: accepted */
            if (flip && fabs((double)r[c] - a) <= tol / R) { /* the other decision of a flagged test */
                acc = !acc;
                flip = 0;
            }
            if (acc) {
                next = c;
                break;
            }
            double S = 0.0; /* step 3: the residual becomes the target of the next sibling */
            for (int i = 0; i < V; i++) {
                double d = p[i] - q[i];
                w[i] = d > 0.0 ? d : 0.0;
                S += w[i];
            }
            R *= S;
            if (!(S > 0.0)) {
                empty = 1;
                break;
            }
            for (int i = 0; i < V; i++) {
                pprev[i] = p[i];
                p[i] = w[i] / S;
            }
            Slast = S;
        }
        if (next >= 0) {
            out_tokens[len] = tokens[next];
            len++;
            path[len] = next;
            cur = next;
            continue;
        }
        double S2;
        int fl, flw = 0, tok;
        const double *wd = p;
        if (empty) { /* R14 / R5: nothing left of the residual, draw from the node's own p */
            wd = p0;
            tok = oracle_inverse_cdf(p0, V, (double)u, tol, &S2, &fl);
            *req_flag |= ORF_ZERO_RESIDUAL;
        } else {
            tok = oracle_inverse_cdf(p, V, (double)u, tol, &S2, &fl);
            if (!fl && R < 1.0) /* R14, widened tier */
                oracle_inverse_cdf(p, V, (double)u, tol / R, &S2, &flw);
        }
        if (fl)
            *req_flag |= ORF_CDF_TIE;
        if (flw)
            *req_flag |= ORF_CDF_TIE_WIDE;
        if (draw_w) {
            for (int i = 0; i < V; i++)
                draw_w[i] = wd[i];
            normalised_cdf(draw_w, V, draw_cdf);
            /* the widened tier's largest weights: the last residual with p and q each known to a
             * relative tol / 2 (no rejection at the node: p itself) */
            if (!empty && R < 1.0) {
                residual_wmax(pprev, q, V, tol, draw_wmax);
                for (int i = 0; i < V; i++)
                    draw_wmax[i] /= Slast;
            } else {
                for (int i = 0; i < V; i++)
                    draw_wmax[i] = wd[i];
            }
        }
        out_tokens[len] = tok;
        *mass = R;
        break;
    }
    *accept_len = len;
    free(p0);
    free(p);
    free(q);
    free(w);
    free(pprev);
    return e;
}

struct probs_ctx {
    int V;
    const double *p, *q;
};

static int probs_rows(void *ctx, int node, int need_q, double *p, double *q)
{
    struct probs_ctx *c = (struct probs_ctx *)ctx;
    for (int i = 0; i < c->V; i++) {
        p[i] = c->p[(size_t)node * c->V + i];
        if (need_q)
            q[i] = c->q[(size_t)node * c->V + i];
    }
    return 0;
}

/* Stochastic tree verification on probability rows p, q: [N1][V] (row n of q = the draft
 * distribution of node n's children).  Outputs: *accept_len, path[N1], out_tokens[N1],
 * alpha[N1] (alpha of each tested child, -1 elsewhere), *mass (R14), *req_flag.  flip and
 * draw_w / draw_cdf / draw_wmax as oracle_tree_sample_alt (0 and NULL for the walk itself). */
void oracle_tree_sample_probs(int N1, int V, const double *p, const double *q,
                              const int *parents, const int *tokens, const float *r, float u,
                              double tol, int flip, int *accept_len, int *path, int *out_tokens,
                              double *alpha, double *mass, int *req_flag, double *draw_w,
                              double *draw_cdf, double *draw_wmax)
{
    struct probs_ctx c = {V, p, q};
    *mass = 0.0;
    tree_sample_walk(N1, V, probs_rows, &c, parents, tokens, r, u, tol, flip, accept_len, path,
                     out_tokens, alpha, mass, req_flag, draw_w, draw_cdf, draw_wmax);
}

struct logits_ctx {
    int dtype, V;
    double T;
    const void *target, *draft;
    size_t row0;
    double *l;
};

static int logits_rows(void *ctx, int node, int need_q, double *p, double *q)
{
    struct logits_ctx *c = (struct logits_ctx *)ctx;
    load_row(c->target, c->dtype, c->row0 + (size_t)node, c->V, c->l);
    int e = oracle_softmax(c->l, c->V, c->T, p);
    if (need_q) {
        load_row(c->draft, c->dtype, c->row0 + (size_t)node, c->V, c->l);
        e |= oracle_softmax(c->l, c->V, c->T, q);
    }
    return e;
}

/* R15, T == 0: the greedy walk on the rows of the visited nodes only. */
static int tree_greedy_visited(int dtype, const void *target, size_t row0, int N1, int V,
                               const int *parents, const int *tokens, int *accept_len, int *path,
                               int *out_tokens, double *alpha)
{
    double *l = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    int cur = 0, len = 0, e = 0;
    for (int i = 0; i < N1; i++) {
        path[i] = -1;
        out_tokens[i] = -1;
        alpha[i] = -1.0;
    }
    path[0] = 0;
    for (int depth = 0; depth < N1; depth++) {
        load_row(target, dtype, row0 + (size_t)cur, V, l);
        if (row_has_nan(l, V)) {
            e = ORE_NONFINITE;
            break;
        }
        int a = oracle_argmax(l, V), next = -1;
        for (int c = cur + 1; c < N1; c++) {
            if (parents[c] != cur)
                continue;
            alpha[c] = tokens[c] == a ? 1.0 : 0.0;
            if (tokens[c] == a) {
                next = c;
                break;
            }
        }
        if (next < 0) {
            out_tokens[len] = a;
            break;
        }
        out_tokens[len] = tokens[next];
        len++;
        path[len] = next;
        cur = next;
    }
    *accept_len = len;
    free(l);
    return e;
}

/* Request b of the walk (outputs for that request alone: path / out_tokens / alpha [N+1]; draw_w /
 * draw_cdf [V] or NULL).  Returns the request's error bits. */
static int tree_sample_request(int dtype, const void *target, const void *draft, int N, int V,
                               float T, const float *temps, const int *node_tokens,
                               const int *parents, const float *r, const float *u, double tol,
                               int b, int flip, double *l, int *accept_len, int *o_path,
                               int *o_tok, double *o_al, double *mass, int *req_flag,
                               double *draw_w, double *draw_cdf, double *draw_wmax)
{
    int N1 = N + 1;
    const int *pb = parents + (size_t)b * N1, *tb = node_tokens + (size_t)b * N1;
    int e = oracle_tree_check(N1, V, pb, tb);
    float Tb = temps ? temps[b] : T;
    *req_flag = 0;
    *mass = 0.0;
    if (!(Tb >= 0.0f) || isinf(Tb))
        e = ORE_BAD_TEMP;
    if (!e) {
        if (Tb == 0.0f) {
            e = tree_greedy_visited(dtype, target, (size_t)b * N1, N1, V, pb, tb, accept_len, o_path,
                                    o_tok, o_al);
            *mass = 1.0;
        } else {
            struct logits_ctx c = {dtype, V, (double)Tb, target, draft, (size_t)b * N1, l};
            e = tree_sample_walk(N1, V, logits_rows, &c, pb, tb, r + (size_t)b * N1, u[b], tol, flip,
                                 accept_len, o_path, o_tok, o_al, mass, req_flag, draw_w, draw_cdf,
                                 draw_wmax);
        }
    }
    if (e) {
        tree_fail(N1, accept_len, o_path, o_tok, o_al, mass);
        *req_flag = 0;
    }
    return e;
}

/*
 * Tree verification by walking (R13-R15).  target, draft: [B][N+1][V] (draft ignored when
 * T == 0); node_tokens, parents: [B][N+1]; r: [B][N+1]; u: [B].
 * R18 per-request temperature (the x078.com page's production section sets the temperature per
 * request): when temps is not NULL, request b uses temps[b] instead of T (0 = greedy); a value
 * that is NaN, negative or infinite fails the request with ORE_BAD_TEMP.
 * Outputs: accept_len[B], path[B][N+1], out_tokens[B][N+1], alpha[B][N+1], mass[B],
 * req_flag[B], err[B].  Requests [b0, b1) only are processed.
 */
void oracle_verify_tree_sample(int dtype, const void *target, const void *draft, int B, int N,
                               int V, float T, const float *temps, const int *node_tokens,
                               const int *parents, const float *r, const float *u, double tol,
                               int b0, int b1, int *accept_len, int *path, int *out_tokens,
                               double *alpha, double *mass, int *req_flag, int *err)
{
    int N1 = N + 1;
    double *l = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    (void)B;
    for (int b = b0; b < b1; b++)
        err[b] = tree_sample_request(dtype, target, draft, N, V, T, temps, node_tokens, parents, r,
                                     u, tol, b, 0, l, accept_len + b, path + (size_t)b * N1,
                                     out_tokens + (size_t)b * N1, alpha + (size_t)b * N1, mass + b,
                                     req_flag + b, NULL, NULL, NULL);
    free(l);
}

/*
 * Request b of oracle_verify_tree_sample (same inputs; outputs for that request alone), for
 * checking a flagged tie (R10, R14): with flip != 0 the first flagged accept test is decided the
 * opposite way (the walk's other admissible outcome), and draw_w / draw_cdf / draw_wmax ([V], or
 * NULL) receive the final draw's weights, their normalised cumulative sums and the widened tier's
 * largest weights (residual_wmax of the last residual) when the request ends in a draw (T > 0, no
 * error).  Returns the request's error bits.
 */
int oracle_tree_sample_alt(int dtype, const void *target, const void *draft, int N, int V,
                           float T, const float *temps, const int *node_tokens,
                           const int *parents, const float *r, const float *u, double tol, int b,
                           int flip, int *accept_len, int *path, int *out_tokens, double *alpha,
                           double *mass, int *req_flag, double *draw_w, double *draw_cdf,
                           double *draw_wmax)
{
    double *l = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    int e = tree_sample_request(dtype, target, draft, N, V, T, temps, node_tokens, parents, r, u,
                                tol, b, flip, l, accept_len, path, out_tokens, alpha, mass,
                                req_flag, draw_w, draw_cdf, draw_wmax);
    free(l);
    return e;
}

/* ------------------------------------------------------------- prompt n-gram lookup draft ---- */
/*
 * Prompt lookup drafting: "Accelerating Autoregressive LLM Inference 3x with Lossless
 * Speculative Decoding and EAGLE Heads" (x078.com), opening section (a zero-VRAM prompt n-gram
 * lookup proposes K = 5 candidate tokens) and its serving example (--num-speculative-tokens 5
 * --ngram-prompt-lookup-max 4).
 * R16: for n = n_max down to n_min, take the context's last n tokens; find their most recent
 * earlier occurrence, i.e. the largest start i with i + n <= L - 1 and ctx[i + j] == ctx[L - n + j]
 * for j < n (it may overlap the suffix itself); the first n that has one wins, and the draft is
 * the tokens that follow it, ctx[i + n .. min(i + n + K, L)) (at least one, at most K).  No
 * match for any n: an empty draft.  n_min = 1 (the pages give only the maximum).
 * Outputs: draft[K] (then -1), *draft_len, *match_n (0 when empty), *match_end (i + n, or -1).
 */
void oracle_ngram_draft(const int *ctx, int L, int n_max, int n_min, int K, int *draft,
                        int *draft_len, int *match_n, int *match_end)
{
    for (int k = 0; k < K; k++)
        draft[k] = -1;
    *draft_len = 0;
    *match_n = 0;
    *match_end = -1;
    for (int n = n_max; n >= n_min && n >= 1; n--) {
        for (int i = L - n - 1; i >= 0; i--) {
            int same = 1;
            for (int j = 0; j < n && same; j++)
                if (ctx[i + j] != ctx[L - n + j])
                    same = 0;
            if (!same)
                continue;
            int e = i + n, m = 0;
            for (int k = 0; k < K && e + k < L; k++) {
                draft[k] = ctx[e + k];
                m++;
            }
            *draft_len = m;
            *match_n = n;
            *match_end = e;
            return;
        }
    }
}

/* Batched: ctx [B][Lmax] with lengths ctx_len[B] (a length outside [0, Lmax] gives an empty
 * draft and err[b] = ORE_BAD_TOKEN); outputs draft [B][K], draft_len / match_n / match_end /
 * err [B].  Requests [b0, b1). */
void oracle_ngram_draft_batch(const int *ctx, const int *ctx_len, int B, int Lmax, int n_max,
                              int n_min, int K, int b0, int b1, int *draft, int *draft_len,
                              int *match_n, int *match_end, int *err)
{
    (void)B;
    for (int b = b0; b < b1; b++) {
        int L = ctx_len[b];
        err[b] = 0;
        if (L < 0 || L > Lmax) {
            err[b] = ORE_BAD_TOKEN;
            L = 0;
        }
        oracle_ngram_draft(ctx + (size_t)b * Lmax, L, n_max, n_min, K, draft + (size_t)b * K,
                           draft_len + b, match_n + b, match_end + b);
    }
}

/* ------------------------------------------------------------- accepted-path KV compaction ---- */
/*
 * "Speculative Decoding with Medusa, EAGLE and vLLM" (vikram-blog.pages.dev), "System Topology &
 * Data Flow" diagram: after the tree is verified, the accepted branch's tokens are committed to
 * the KV cache.
 * R17: the target's forward pass wrote the KV row of tree node n into slot slots[n] of a cache of
 * rows (row_bytes each).  With the accepted path p_0 = 0, p_1, ..., p_L (path[0..L]), the row of
 * p_j moves to the slot of position j: new[slots[j]] = old[slots[p_j]] for j = 1..L; every other
 * slot keeps its row.  (Position j's slot is that of node j in the tree's numbering, so the
 * accepted tokens end up in the first L + 1 slots, in order.)
 */
void oracle_kv_compact(unsigned char *cache, int row_bytes, const int *slots, int L,
                       const int *path)
{
    if (L <= 0)
        return;
    unsigned char *tmp = (unsigned char *)malloc((size_t)L * (size_t)row_bytes);
    for (int j = 1; j <= L; j++) /* read every accepted row before any slot is written */
        memcpy(tmp + (size_t)(j - 1) * row_bytes, cache + (size_t)slots[path[j]] * row_bytes,
               (size_t)row_bytes);
    for (int j = 1; j <= L; j++)
        memcpy(cache + (size_t)slots[j] * row_bytes, tmp + (size_t)(j - 1) * row_bytes,
               (size_t)row_bytes);
    free(tmp);
}

/* Batched over requests and caches: caches [C][num_slots][row_bytes] (C caches, e.g. the K and V
 * tensors of every layer), slots [B][N1], accept_len [B], path [B][N1].  A request whose path is
 * not a valid accepted path (L outside [0, N1), path[0] != 0, a node not a child of the previous
 * one, a slot outside [0, num_slots)) is left untouched and err[b] = ORE_BAD_TREE. */
void oracle_kv_compact_batch(unsigned char *caches, int C, long long num_slots, int row_bytes,
                             int B, int N1, const int *slots, const int *parents,
                             const int *accept_len, const int *path, int *err)
{
    for (int b = 0; b < B; b++) {
        const int *sl = slots + (size_t)b * N1, *pa = parents + (size_t)b * N1;
        const int *pt = path + (size_t)b * N1;
        int L = accept_len[b], ok = L >= 0 && L < N1 && pt[0] == 0;
        for (int j = 1; ok && j <= L; j++)
            ok = pt[j] > 0 && pt[j] < N1 && pa[pt[j]] == pt[j - 1];
        for (int n = 0; ok && n < N1; n++)
            ok = sl[n] >= 0 && sl[n] < num_slots;
        err[b] = ok ? 0 : ORE_BAD_TREE;
        if (!ok)
            continue;
        for (int c = 0; c < C; c++)
            oracle_kv_compact(caches + (size_t)c * (size_t)num_slots * (size_t)row_bytes, row_bytes,
                              sl, L, pt);
    }
}
