/*
 * spec_oracle.c -- plain, slow, fp64 CPU oracle for speculative-decoding
 * verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, constant or helper with the CUDA
 * library: the two meet only at the seeded inputs.
 *
 * Every function takes the same bits the GPU path reads (bf16 or fp32 logits,
 * fp32 uniforms) and widens them exactly to double before doing anything.
 * All arithmetic after that is fp64, written in the order the pages state it:
 *
 *   softmax        p = softmax(logits / T)   ("投机解码:为什么一个字都不改",
 *                  section "一轮能出几个 token", the P = softmax(f(x)/T) box)
 *   greedy verify  accept draft i while it equals the target's own choice,
 *                  stop at the first mismatch, then append the target's own
 *                  token at that point ("第 13 篇：推理引擎一次猜几个字",
 *                  section ③ 伪代码 and 逐行要点; "Speculative decoding
 *                  explained", the four-case table)
 *   sample verify  accept x ~ q with probability min(1, p(x)/q(x)); on the
 *                  first rejection draw from norm(max(0, p - q)) and drop the
 *                  rest; if all are accepted draw one more token from p
 *                  ("投机解码:为什么一个字都不改", section "改进方案" and the
 *                  replay section: every round emits accepted + 1 tokens)
 *   tree verify    apply the sampling rule recursively at each node, testing
 *                  the children in turn and replacing p by the normalised
 *                  residual after every rejected child ("Speculative Decoding
 *                  II", EAGLE section, the paragraph on verifying the draft
 *                  tree with tree attention, "consistent with SpecInfer");
 *                  variant 2, for siblings drawn from q WITHOUT replacement,
 *                  also removes each rejected sibling's token from q and
 *                  renormalises it, since the next sibling was drawn from
 *                  that distribution (a reading; the pages name SpecInfer
 *                  only)
 *   n-gram draft   take the last `window` tokens, find the same segment
 *                  earlier in the history, propose what followed it
 *                  ("第 13 篇", 逐行要点, the 草稿器.猜 line)
 *   tree rerank    EAGLE-2's post-processing of a candidate tree: value =
 *                  product of the draft confidences along the path, keep
 *                  the m best (ties: shallower first), flatten by depth,
 *                  each node attending to its ancestors ("Speculative
 *                  Decoding II", section "Context-Aware Dynamic Draft Tree"
 *                  and its worked example)
 *
 * Readings where the pages are silent:
 *   - the uniform u_i tests draft position i; u_k (the last one) drives the
 *     final draw, whether it is a residual draw or the bonus draw;
 *   - "accept with probability min(1, p/q)" is realised as accept iff
 *     u < min(1, p(x)/q(x)), with u in [0,1); q(x) = 0 accepts iff p(x) > 0;
 *   - an inverse-CDF draw returns the smallest v whose inclusive prefix sum
 *     of the (normalised) distribution exceeds u; if rounding leaves no such
 *     v, the last v with positive mass;
 *   - argmax ties go to the lowest index;
 *   - n-gram: the rightmost earlier occurrence wins, the continuation is cut
 *     at the end of the history, no match gives an empty draft;
 *   - a residual with zero mass (impossible in exact arithmetic after a
 *     rejection) falls back to p and is counted.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_ENOMEM -2

/* per-request status codes, the same meanings the library documents */
#define ST_OK 0
#define ST_TOKEN_RANGE 1
#define ST_BAD_TREE 2
#define ST_BAD_LENGTH 3

/* ---------------------------------------------------------------- inputs */

/* Widen one logit to double.  dtype 0 = fp32, 1 = bf16 (the top 16 bits of
 * an IEEE binary32), so both conversions are exact. */
static double logit_at(const void *base, int dtype, int64_t off)
{
    if (dtype == 0)
        return (double)((const float *)base)[off];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[off] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* --------------------------------------------------------- distributions */

/* p = softmax(x / T) over one row of V logits, in fp64. */
static void softmax_row(const void *row, int dtype, int V, double T, double *p)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        p[v] = logit_at(row, dtype, v) / T;
        if (p[v] > m)
            m = p[v];
    }
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp(p[v] - m);
        S += p[v];
    }
    for (int v = 0; v < V; ++v)
        p[v] /= S;
}

/* ------------------------------------------------- top-k / top-p filtering
 *
 * A sampling variant the pages defer to another lesson ("投机解码", the
 * section that sets temperature, top-k and top-p aside): verification stays
 * lossless against the FILTERED target when both p and q are filtered the
 * same way and the drafter drew from the filtered q.  The plainest reading,
 * applied in this order:
 *   1. p = softmax(x / T);
 *   2. top-k (0 < top_k < V): theta_k = the top_k-th largest logit (counting
 *      repeats); keep every v with x_v >= theta_k (ties at the cut stay);
 *   3. top-p (top_p < 1): over the kept tokens in descending logit order,
 *      with p renormalised to them, the smallest prefix whose mass reaches
 *      top_p; theta_p = the logit of its last token; keep every kept v with
 *      x_v >= theta_p;
 *   4. p' = p renormalised over the kept tokens, 0 elsewhere.
 * theta = the smallest kept logit.  top_k <= 0 or >= V, and top_p >= 1,
 * switch their filter off. */

typedef struct {
    double x;
    int v;
} orc_keyed;

static int keyed_desc(const void *pa, const void *pb)
{
    const orc_keyed *a = pa, *b = pb;
    if (a->x != b->x)
        return a->x > b->x ? -1 : 1;
    return a->v < b->v ? -1 : (a->v > b->v);
}

/* p' of one row (written to p), the threshold logit and the kept count. */
static int filter_row(const void *row, int dtype, int V, double T, int top_k, double top_p,
                      double *p, double *theta_out, int *kept_out)
{
    softmax_row(row, dtype, V, T, p);
    double theta = -INFINITY;
    int use_k = top_k > 0 && top_k < V, use_p = top_p < 1.0;
    if (use_k || use_p) {
        orc_keyed *ord = malloc(sizeof(orc_keyed) * (size_t)V);
        if (!ord)
            return ORC_ENOMEM;
        for (int v = 0; v < V; ++v) {
            ord[v].x = logit_at(row, dtype, v);
            ord[v].v = v;
        }
        qsort(ord, (size_t)V, sizeof *ord, keyed_desc);
        int n = V; /* kept tokens form the prefix ord[0..n) */
        if (use_k) {
            theta = ord[top_k - 1].x;
            n = top_k;
            while (n < V && ord[n].x >= theta)
                ++n;
        }
        if (use_p) {
            double SK = 0.0, cum = 0.0;
            for (int j = 0; j < n; ++j)
                SK += p[ord[j].v];
            int j = 0;
            for (; j < n; ++j) {
                cum += p[ord[j].v] / SK;
                if (cum >= top_p)
                    break;
            }
            if (j == n) /* rounding: the mass never reached top_p, keep all */
                j = n - 1;
            if (ord[j].x > theta)
                theta = ord[j].x;
        }
        free(ord);
    }
    double S = 0.0;
    int kept = 0;
    for (int v = 0; v < V; ++v) {
        if (logit_at(row, dtype, v) >= theta) {
            S += p[v];
            ++kept;
        } else {
            p[v] = 0.0;
        }
    }
    for (int v = 0; v < V; ++v)
        p[v] /= S;
    if (theta == -INFINITY) {
        theta = INFINITY; /* no filter: the smallest logit */
        for (int v = 0; v < V; ++v) {
            double x = logit_at(row, dtype, v);
            if (x < theta)
                theta = x;
        }
    }
    if (theta_out)
        *theta_out = theta;
    if (kept_out)
        *kept_out = kept;
    return ORC_OK;
}

/* Index of the largest logit; ties go to the lowest index. */
static int argmax_row(const void *row, int dtype, int V)
{
    int best = 0;
    double bv = logit_at(row, dtype, 0);
    for (int v = 1; v < V; ++v) {
        double x = logit_at(row, dtype, v);
        if (x > bv) {
            bv = x;
            best = v;
        }
    }
    return best;
}

/* Inverse CDF of a normalised distribution d[0..V): the smallest v with
 * d[0] + ... + d[v] > u.  If rounding leaves the total at or below u, the
 * last v with d[v] > 0.  Returns -1 only for an all-zero distribution. */
static int inverse_cdf(const double *d, int V, double u)
{
    double cum = 0.0;
    int last_pos = -1;
    for (int v = 0; v < V; ++v) {
        cum += d[v];
        if (d[v] > 0.0)
            last_pos = v;
        if (cum > u)
            return v;
    }
    return last_pos;
}

/* r = norm(max(0, p - q)); returns the mass sum(max(0, p - q)) before the
 * normalisation.  When that mass is zero r is left all zero. */
static double residual(const double *p, const double *q, int V, double *r)
{
    double R = 0.0;
    for (int v = 0; v < V; ++v) {
        r[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;
        R += r[v];
    }
    if (R > 0.0)
        for (int v = 0; v < V; ++v)
            r[v] /= R;
    return R;
}

/* The acceptance rule: accept with probability min(1, p/q), realised with
 * one uniform u in [0,1) as u < min(1, p/q).  A draft token the draft model
 * gives zero probability is accepted whenever the target gives it any. */
static int accept_test(double u, double px, double qx)
{
    if (qx <= 0.0)
        return px > 0.0;
    double ratio = px / qx;
    return u < (ratio < 1.0 ? ratio : 1.0);
}

/* ------------------------------------------------------------ exported API */

int orc_softmax(const void *row, int dtype, int V, double T, double *p)
{
    if (!row || !p || V <= 0 || !(T > 0.0) || (dtype != 0 && dtype != 1))
        return ORC_EINVAL;
    softmax_row(row, dtype, V, T, p);
    return ORC_OK;
}

int orc_argmax(const void *row, int dtype, int V)
{
    if (!row || V <= 0 || (dtype != 0 && dtype != 1))
        return ORC_EINVAL;
    return argmax_row(row, dtype, V);
}

int orc_inverse_cdf(const double *d, int V, double u) { return inverse_cdf(d, V, u); }

double orc_residual(const double *p, const double *q, int V, double *r)
{
    return residual(p, q, V, r);
}

/* n-gram history lookup ("第 13 篇", 逐行要点: use the last few tokens of the
 * context as a window, find an identical earlier segment in the history,
 * propose the tokens that followed it).
 *
 * history: [B, hist_stride] int32, request b holds hist_len[b] tokens.
 * The window is h[n-w .. n).  An earlier occurrence starts at i < n - w.
 * The rightmost such i wins; the draft is h[i+w .. min(i+w+k, n)).
 * draft: [B, k], padded with -1; draft_len: [B]; status: [B]. */
int orc_ngram_draft(const int32_t *history, const int32_t *hist_len, int B,
                    int hist_stride, int window, int k, int32_t *draft,
                    int32_t *draft_len, int32_t *status)
{
    if (B < 0 || window <= 0 || k < 0 || hist_stride < 0)
        return ORC_EINVAL;
    for (int b = 0; b < B; ++b) {
        const int32_t *h = history + (int64_t)b * hist_stride;
        int n = hist_len[b];
        for (int j = 0; j < k; ++j)
            draft[(int64_t)b * k + j] = -1;
        draft_len[b] = 0;
        status[b] = ST_OK;
        if (n < 0 || n > hist_stride) {
            status[b] = ST_BAD_LENGTH;
            continue;
        }
        int found = -1;
        for (int i = 0; i + window < n; ++i) { /* i < n - w */
            int same = 1;
            for (int j = 0; j < window; ++j)
                if (h[i + j] != h[n - window + j]) {
                    same = 0;
                    break;
                }
            if (same)
                found = i; /* keep scanning: the rightmost match wins */
        }
        if (found < 0)
            continue;
        int len = 0;
        for (int j = found + window; j < n && len < k; ++j)
            draft[(int64_t)b * k + len++] = h[j];
        draft_len[b] = len;
    }
    return ORC_OK;
}

/* Greedy chain verification.
 * target: logits of request b, position i at target + b*t_req + i*row,
 *         positions 0..k (k+1 rows).
 * draft: [B, k] tokens; draft_len: [B] or NULL (= k); max_emit: [B] or NULL.
 * Outputs accepted[B], out_tokens[B, k+1] (pad -1), n_emit[B], status[B]. */
int orc_verify_greedy(const void *target, int dtype, int B, int k, int V,
                      int64_t t_req, int64_t row, const int32_t *draft,
                      const int32_t *draft_len, const int32_t *max_emit,
                      int32_t *accepted, int32_t *out_tokens, int32_t *n_emit,
                      int32_t *status)
{
    if (!target || B < 0 || k < 0 || V <= 0 || (dtype != 0 && dtype != 1))
        return ORC_EINVAL;
    const size_t es = dtype == 0 ? 4 : 2;
    for (int b = 0; b < B; ++b) {
        int32_t *out = out_tokens + (int64_t)b * (k + 1);
        for (int j = 0; j <= k; ++j)
            out[j] = -1;
        accepted[b] = 0;
        n_emit[b] = 0;
        status[b] = ST_OK;
        int L = draft_len ? draft_len[b] : k;
        if (L < 0 || L > k) {
            status[b] = ST_BAD_LENGTH;
            continue;
        }
        const int32_t *x = draft + (int64_t)b * k;
        int bad = 0;
        for (int i = 0; i < L; ++i)
            if (x[i] < 0 || x[i] >= V)
                bad = 1;
        if (bad) {
            status[b] = ST_TOKEN_RANGE;
            continue;
        }
        /* walk the draft left to right; stop at the first mismatch */
        int m = 0;
        while (m < L) {
            const char *r = (const char *)target + ((int64_t)b * t_req + (int64_t)m * row) * es;
            if (argmax_row(r, dtype, V) != x[m])
                break;
            ++m;
        }
        const char *rm = (const char *)target + ((int64_t)b * t_req + (int64_t)m * row) * es;
        int final_tok = argmax_row(rm, dtype, V);
        int cap = max_emit ? max_emit[b] : k + 1;
        int ne = m + 1 < cap ? m + 1 : cap;
        if (ne < 0)
            ne = 0;
        for (int j = 0; j < m && j < ne; ++j)
            out[j] = x[j];
        if (m < ne)
            out[m] = final_tok;
        accepted[b] = m;
        n_emit[b] = ne;
    }
    return ORC_OK;
}

/* Sampling chain verification.
 *
 * variant 0: the lossless rule (min(1,p/q) acceptance, residual resampling).
 * variant 1: negative control from the pages -- after a rejection draw from
 *            p instead of the residual (counts the shared mass twice).
 * variant 2: negative control from the pages -- the target samples its own
 *            token with u_i, the draft token is kept only if they are equal,
 *            otherwise the target's sample is emitted.
 *
 * uniforms: [B, k+1]; u[b][i] tests position i, u[b][k] drives the final draw.
 * Optional outputs (may be NULL): p_tok/q_tok [B,k] = p_i(x_i), q_i(x_i) for
 * i < draft_len (else -1); resid_mass [B] = sum max(0, p_m - q_m) at the
 * rejected position (0 when every draft token was accepted).
 * degenerate (may be NULL): incremented once per zero-mass residual.
 * top_p_rows (may be NULL): one top_p per row, [B][2k+1] in the order target
 * rows 0..k then draft rows 0..k-1, in place of top_p (the same filter, each
 * row with its own mass). */
int orc_filter_row(const void *row, int dtype, int V, double T, int top_k, double top_p,
                   double *p, double *theta, int32_t *kept)
{
    if (!row || !p || V <= 0 || !(T > 0.0) || (dtype != 0 && dtype != 1) || !(top_p > 0.0))
        return ORC_EINVAL;
    int n = 0;
    int rc = filter_row(row, dtype, V, T, top_k, top_p, p, theta, &n);
    if (kept)
        *kept = n;
    return rc;
}

int orc_verify_sample(const void *target, int64_t t_req, const void *draft_logits,
                      int64_t d_req, int64_t row, int dtype, int B, int k, int V,
                      double T, int top_k, double top_p, const int32_t *draft, const int32_t *draft_len,
                      const int32_t *max_emit, const float *uniforms,
                      int32_t *accepted, int32_t *out_tokens, int32_t *n_emit,
                      double *p_tok, double *q_tok, double *resid_mass,
                      int32_t *status, int variant, int threads,
                      int64_t *degenerate, const double *top_p_rows)
{
    if (!target || !draft_logits || B < 0 || k < 0 || V <= 0 || !(T > 0.0) ||
        (dtype != 0 && dtype != 1) || variant < 0 || variant > 2 || !(top_p > 0.0))
        return ORC_EINVAL;
    const size_t es = dtype == 0 ? 4 : 2;
    int64_t degen = 0;
    int fail = 0;
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads) reduction(+ : degen) reduction(| : fail)
    for (int b = 0; b < B; ++b) {
        double *p = malloc(sizeof(double) * (size_t)V);
        double *q = malloc(sizeof(double) * (size_t)V);
        double *r = malloc(sizeof(double) * (size_t)V);
        if (!p || !q || !r) {
            fail = 1;
            free(p), free(q), free(r);
            continue;
        }
        int32_t *out = out_tokens + (int64_t)b * (k + 1);
        const int32_t *x = draft + (int64_t)b * k;
        const float *u = uniforms + (int64_t)b * (k + 1);
        for (int j = 0; j <= k; ++j)
            out[j] = -1;
        for (int j = 0; j < k; ++j) {
            if (p_tok)
                p_tok[(int64_t)b * k + j] = -1.0;
            if (q_tok)
                q_tok[(int64_t)b * k + j] = -1.0;
        }
        if (resid_mass)
            resid_mass[b] = 0.0;
        accepted[b] = 0;
        n_emit[b] = 0;
        status[b] = ST_OK;
        int L = draft_len ? draft_len[b] : k;
        int ok = 1;
        if (L < 0 || L > k) {
            status[b] = ST_BAD_LENGTH;
            ok = 0;
        }
        for (int i = 0; ok && i < L; ++i)
            if (x[i] < 0 || x[i] >= V) {
                status[b] = ST_TOKEN_RANGE;
                ok = 0;
            }
        if (!ok) {
            free(p), free(q), free(r);
            continue;
        }
        const char *tb = (const char *)target + (int64_t)b * t_req * es;
        const char *db = (const char *)draft_logits + (int64_t)b * d_req * es;
        /* the top_p of target row i and of draft row i */
        const double *tpr = top_p_rows ? top_p_rows + (int64_t)b * (2 * k + 1) : NULL;
#define TP_T(i) (tpr ? tpr[(i)] : top_p)
#define TP_D(i) (tpr ? tpr[k + 1 + (i)] : top_p)

        /* the per-position probabilities of the drafted tokens */
        for (int i = 0; i < L; ++i) {
            fail |= filter_row(tb + (int64_t)i * row * es, dtype, V, T, top_k, TP_T(i), p, NULL, NULL);
            fail |= filter_row(db + (int64_t)i * row * es, dtype, V, T, top_k, TP_D(i), q, NULL, NULL);
            if (p_tok)
                p_tok[(int64_t)b * k + i] = p[x[i]];
            if (q_tok)
                q_tok[(int64_t)b * k + i] = q[x[i]];
        }

        /* left to right: accept, or stop at the first rejection */
        int m = 0, final_tok = -1;
        for (; m < L; ++m) {
            fail |= filter_row(tb + (int64_t)m * row * es, dtype, V, T, top_k, TP_T(m), p, NULL, NULL);
            int acc;
            if (variant == 2) {
                acc = inverse_cdf(p, V, (double)u[m]) == x[m];
            } else {
                fail |= filter_row(db + (int64_t)m * row * es, dtype, V, T, top_k, TP_D(m), q, NULL, NULL);
                acc = accept_test((double)u[m], p[x[m]], q[x[m]]);
            }
            if (!acc)
                break;
        }
        if (m < L) {
            /* rejected at position m: p already holds p_m */
            if (variant == 0) {
                double R = residual(p, q, V, r);
                if (resid_mass)
                    resid_mass[b] = R;
                if (R > 0.0) {
                    final_tok = inverse_cdf(r, V, (double)u[k]);
                } else {
                    degen += 1;
                    final_tok = inverse_cdf(p, V, (double)u[k]);
                }
            } else if (variant == 1) {
                final_tok = inverse_cdf(p, V, (double)u[k]);
            } else {
                final_tok = inverse_cdf(p, V, (double)u[m]);
            }
        } else {
            /* all L accepted: the bonus token comes from p_L */
            fail |= filter_row(tb + (int64_t)L * row * es, dtype, V, T, top_k, TP_T(L), p, NULL, NULL);
            final_tok = inverse_cdf(p, V, (double)u[k]);
        }
#undef TP_T
#undef TP_D
        int cap = max_emit ? max_emit[b] : k + 1;
        int ne = m + 1 < cap ? m + 1 : cap;
        if (ne < 0)
            ne = 0;
        for (int j = 0; j < m && j < ne; ++j)
            out[j] = x[j];
        if (m < ne)
            out[m] = final_tok;
        accepted[b] = m;
        n_emit[b] = ne;
        free(p), free(q), free(r);
    }
    if (degenerate)
        *degenerate += degen;
    return fail ? ORC_ENOMEM : ORC_OK;
}

/* Tree verification ("Speculative Decoding II", EAGLE: one target forward
 * with tree attention scores every node; the sampling rule is applied
 * recursively at each node, as in SpecInfer).
 *
 * Node 0 is the root (the last committed token, parents[0] = -1); every other
 * node i has 0 <= parents[i] < i and carries the drafted token node_tok[i].
 * target/draft rows of node u: the target's and the draft's distribution of
 * the token after u.  uniforms: [B, N+1]; u[c] tests child c, u[N] drives the
 * final draw.  T > 0 samples; T <= 0 is the greedy tree walk (follow the first
 * child, in id order, whose token is the target's argmax).
 *
 * Sampling at node u, children c_1 < c_2 < ... in id order:
 *   p <- softmax(t_u / T), q <- softmax(d_u / T)
 *   for each child c: accept with probability min(1, p(x_c)/q(x_c));
 *     accepted -> emit x_c, descend to c;
 *     rejected -> p <- norm(max(0, p - q)), try the next child.
 *   no child accepted (or u is a leaf) -> draw the final token from p.
 *
 * Outputs: accepted_len[B] (tree nodes accepted), path_nodes[B, max_depth+1]
 * (node ids from the root, pad -1), out_tokens[B, max_depth+1] (emitted
 * tokens, pad -1), n_emit[B] = accepted_len + 1, status[B].
 *
 * variant 0 is the rule above; variant 1 is a negative control that keeps p
 * unchanged after a rejected child (it over-weights the shared mass). */
int orc_verify_tree(const void *target, int64_t t_req, const void *draft_logits,
                    int64_t d_req, int64_t row, int dtype, int B, int N, int V,
                    double T, const int32_t *parents, const int32_t *node_tok,
                    const float *uniforms, int max_depth, int32_t *accepted_len,
                    int32_t *path_nodes, int32_t *out_tokens, int32_t *n_emit,
                    int32_t *status, int variant, int threads, int64_t *degenerate)
{
    if (!target || B < 0 || N < 1 || V <= 0 || max_depth < 0 ||
        (dtype != 0 && dtype != 1) || variant < 0 || variant > 2)
        return ORC_EINVAL;
    const int greedy = !(T > 0.0);
    if (!greedy && !draft_logits)
        return ORC_EINVAL;
    const size_t es = dtype == 0 ? 4 : 2;
    const int W = max_depth + 1;
    int64_t degen = 0;
    int fail = 0;
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads) reduction(+ : degen) reduction(| : fail)
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parents + (int64_t)b * N;
        const int32_t *tok = node_tok + (int64_t)b * N;
        const float *u = uniforms + (int64_t)b * (N + 1);
        int32_t *pn = path_nodes + (int64_t)b * W;
        int32_t *out = out_tokens + (int64_t)b * W;
        for (int j = 0; j < W; ++j)
            pn[j] = out[j] = -1;
        accepted_len[b] = 0;
        n_emit[b] = 0;
        status[b] = ST_OK;

        /* the tree must be well formed and no deeper than max_depth */
        int *depth = malloc(sizeof(int) * (size_t)N);
        double *p = malloc(sizeof(double) * (size_t)V);
        double *q = malloc(sizeof(double) * (size_t)V);
        double *r = malloc(sizeof(double) * (size_t)V);
        if (!depth || !p || !q || !r) {
            fail = 1;
            free(depth), free(p), free(q), free(r);
            continue;
        }
        int ok = par[0] == -1;
        depth[0] = 0;
        for (int i = 1; ok && i < N; ++i) {
            if (par[i] < 0 || par[i] >= i) {
                ok = 0;
                break;
            }
            depth[i] = depth[par[i]] + 1;
            if (depth[i] > max_depth)
                ok = 0;
        }
        if (!ok) {
            status[b] = ST_BAD_TREE;
            free(depth), free(p), free(q), free(r);
            continue;
        }
        for (int i = 1; i < N; ++i)
            if (tok[i] < 0 || tok[i] >= V)
                ok = 0;
        if (!ok) {
            status[b] = ST_TOKEN_RANGE;
            free(depth), free(p), free(q), free(r);
            continue;
        }

        const char *tb = (const char *)target + (int64_t)b * t_req * es;
        const char *db = greedy ? NULL : (const char *)draft_logits + (int64_t)b * d_req * es;
        int node = 0, nacc = 0, final_tok = -1;
        pn[0] = 0;
        for (;;) {
            const char *trow = tb + (int64_t)node * row * es;
            int next = -1;
            if (greedy) {
                int a = argmax_row(trow, dtype, V);
                for (int c = node + 1; c < N; ++c)
                    if (par[c] == node && tok[c] == a) {
                        next = c;
                        break;
                    }
                if (next < 0)
                    final_tok = a;
            } else {
                softmax_row(trow, dtype, V, T, p);
                int has_child = 0;
                for (int c = node + 1; c < N; ++c)
                    if (par[c] == node)
                        has_child = 1;
                if (has_child)
                    softmax_row(db + (int64_t)node * row * es, dtype, V, T, q);
                for (int c = node + 1; c < N && next < 0; ++c) {
                    if (par[c] != node)
                        continue;
                    if (accept_test((double)u[c], p[tok[c]], q[tok[c]])) {
                        next = c;
                    } else if (variant == 0 || variant == 2) {
                        double R = residual(p, q, V, r);
                        if (R > 0.0) {
                            memcpy(p, r, sizeof(double) * (size_t)V);
                            if (variant == 2) {
                                /* siblings drawn without replacement: the next
                                 * one came from q with this token removed */
                                double Q = 0.0;
                                q[tok[c]] = 0.0;
                                for (int v = 0; v < V; ++v)
                                    Q += q[v];
                                for (int v = 0; v < V; ++v)
                                    q[v] = Q > 0.0 ? q[v] / Q : 0.0;
                            }
                        } else {
                            degen += 1; /* keep p (and q): see the header */
                        }
                    }
                }
                if (next < 0)
                    final_tok = inverse_cdf(p, V, (double)u[N]);
            }
            if (next < 0)
                break;
            out[nacc] = tok[next];
            ++nacc;
            pn[nacc] = next;
            node = next;
        }
        out[nacc] = final_tok;
        accepted_len[b] = nacc;
        n_emit[b] = nacc + 1;
        free(depth), free(p), free(q), free(r);
    }
    if (degenerate)
        *degenerate += degen;
    return fail ? ORC_ENOMEM : ORC_OK;
}

/* ----------------------------------------------------------- tree rerank */

/* One candidate node: its value, depth and id. */
typedef struct {
    float v;
    int depth, id;
} rr_node;

/* Rerank order: larger value first; equal values, the shallower node
 * ("Speculative Decoding II", Context-Aware Dynamic Draft Tree: nodes of
 * equal value are taken shallower first, so the kept nodes form a tree);
 * equal value and depth, the lower id. */
static int rr_rank_cmp(const void *pa, const void *pb)
{
    const rr_node *a = (const rr_node *)pa, *b = (const rr_node *)pb;
    if (a->v != b->v)
        return a->v > b->v ? -1 : 1;
    if (a->depth != b->depth)
        return a->depth < b->depth ? -1 : 1;
    return a->id < b->id ? -1 : (a->id > b->id);
}

/* Flattened order: by depth, then id (the page's [I, do, make, it, this, a,
 * now, plan] with relative positions [0, 1, 1, 2, 2, 2, 3, 3]). */
static int rr_flat_cmp(const void *pa, const void *pb)
{
    const rr_node *a = (const rr_node *)pa, *b = (const rr_node *)pb;
    if (a->depth != b->depth)
        return a->depth < b->depth ? -1 : 1;
    return a->id < b->id ? -1 : (a->id > b->id);
}

/*
 * EAGLE-2 post-processing of a candidate draft tree ("Speculative Decoding
 * II", section "Context-Aware Dynamic Draft Tree" and its worked example).
 *   value    V(root) = 1, V(i) = V(parent(i)) * c_i: the product of the draft
 *            confidences along the path, multiplied from the root down as the
 *            page does (V = 0.60 x 0.80 = 0.48).  It is computed in binary32,
 *            the library's precision, because it decides the ranking below
 *            (an integer result) and both sides must decide alike;
 *   rerank   keep the m nodes of largest V (rr_rank_cmp);
 *   flatten  the kept nodes in rr_flat_cmp order; relative position = depth;
 *            the mask row of a node marks itself and its ancestors.
 * parents [B, N]: parents[0] = -1, 0 <= parents[i] < i; conf [B, N]: c_i in
 * [0, 1] (conf[0] is not read); node_tok [B, N] or NULL.  Outputs, n_sel =
 * min(m, N) entries per request then padding (-1; values -1; mask 0):
 * sel_nodes, sel_parents (flattened index of the parent, -1 for the root),
 * sel_depth, sel_value, sel_tok (when node_tok is given), mask [B, m, m]
 * (NULL to skip), n_sel, status (ST_BAD_TREE for a malformed parent array, a
 * depth beyond max_depth, or a confidence outside [0, 1]; such a request
 * keeps nothing).
 */
int orc_tree_rerank(const int32_t *parents, const float *conf, const int32_t *node_tok, int B, int N,
                    int m, int max_depth, int32_t *sel_nodes, int32_t *sel_parents, int32_t *sel_depth,
                    float *sel_value, int32_t *sel_tok, uint8_t *mask, int32_t *n_sel, int32_t *status)
{
    if (B < 0 || N < 1 || m < 1 || max_depth < 0 || !parents || !conf || !sel_nodes || !sel_parents ||
        !sel_depth || !n_sel || !status)
        return ORC_EINVAL;
    rr_node *nodes = (rr_node *)malloc(sizeof(rr_node) * (size_t)N);
    int *depth = (int *)malloc(sizeof(int) * (size_t)N), *pos = (int *)malloc(sizeof(int) * (size_t)N);
    float *val = (float *)malloc(sizeof(float) * (size_t)N);
    if (!nodes || !depth || !pos || !val) {
        free(nodes), free(depth), free(pos), free(val);
        return ORC_ENOMEM;
    }
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parents + (int64_t)b * N;
        const float *c = conf + (int64_t)b * N;
        int32_t *o_node = sel_nodes + (int64_t)b * m, *o_par = sel_parents + (int64_t)b * m;
        int32_t *o_dep = sel_depth + (int64_t)b * m;
        for (int j = 0; j < m; ++j) {
            o_node[j] = o_par[j] = o_dep[j] = -1;
            if (sel_value) sel_value[(int64_t)b * m + j] = -1.0f;
            if (sel_tok) sel_tok[(int64_t)b * m + j] = -1;
        }
        if (mask) memset(mask + (int64_t)b * m * m, 0, (size_t)m * (size_t)m);
        n_sel[b] = 0;
        /* the tree, its depths and values, from the root down (parents[i] < i) */
        int bad = par[0] != -1;
        depth[0] = 0;
        val[0] = 1.0f;
        for (int i = 1; i < N && !bad; ++i) {
            if (par[i] < 0 || par[i] >= i || !(c[i] >= 0.0f && c[i] <= 1.0f)) {
                bad = 1;
                break;
            }
            depth[i] = depth[par[i]] + 1;
            if (depth[i] > max_depth) bad = 1;
            val[i] = val[par[i]] * c[i];
        }
        if (bad) {
            status[b] = ST_BAD_TREE;
            continue;
        }
        for (int i = 0; i < N; ++i) {
            nodes[i].v = val[i];
            nodes[i].depth = depth[i];
            nodes[i].id = i;
        }
        qsort(nodes, (size_t)N, sizeof(rr_node), rr_rank_cmp);
        const int n = m < N ? m : N;
        qsort(nodes, (size_t)n, sizeof(rr_node), rr_flat_cmp);
        for (int i = 0; i < N; ++i) pos[i] = -1;
        for (int j = 0; j < n; ++j) pos[nodes[j].id] = j;
        for (int j = 0; j < n; ++j) {
            const int u = nodes[j].id;
            o_node[j] = u;
            o_par[j] = u == 0 ? -1 : pos[par[u]];
            o_dep[j] = nodes[j].depth;
            if (sel_value) sel_value[(int64_t)b * m + j] = nodes[j].v;
            if (sel_tok) sel_tok[(int64_t)b * m + j] = node_tok ? node_tok[(int64_t)b * N + u] : -1;
            if (mask) {
                uint8_t *row = mask + ((int64_t)b * m + j) * m;
                for (int a = u; a >= 0; a = a == 0 ? -1 : par[a])
                    if (pos[a] >= 0) row[pos[a]] = 1;
            }
        }
        n_sel[b] = n;
        status[b] = ST_OK;
    }
    free(nodes), free(depth), free(pos), free(val);
    return ORC_OK;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
