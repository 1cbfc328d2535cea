/*
 * spec_oracle.c -- plain, slow, fp64 CPU oracle for the target-side
 * verify-and-resample step of speculative decoding, and for the draft-side
 * softmax + multinomial.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the CUDA path; the two meet only in the seeded inputs.
 *
 * Sources (three web pages on the method; cited by title and section):
 *   [P1] "【大模型】- 推测解码" (sxl-space.tk), sections 基础推测解码器
 *        (SpeculativeDecoder.draft_generate / target_verify) and 批量推测解码
 *        (BatchSpeculativeDecoder.verify_single).
 *   [P2] "投机解码" (docs.ifdog.com), sections 投机解码的三步流程 (the 3-step
 *        procedure), 无损保证：数学推导 (losslessness proof), 动手实践
 *        (speculative_decode, greedy and sampling branches).
 *   [P3] "大模型推理无损加速:投机采样(Speculative Decoding)数学原理与工业级落地实践"
 *        (bbs.huaweicloud.com), sections 二.1 (acceptance probability
 *        alpha = min(1, p/q)), 二.2 (residual distribution p'), 三
 *        (speculative_sampling_step).
 *
 * Readings taken where the pages are silent or disagree:
 *   - accept iff u < alpha, u in [0,1)    ([P1]/[P2] use '<', [P3] '<=')
 *   - no epsilon guards; the ratio p/q is formed as exp(log p - log q).
 *     q(x) = 0 (draft logit -inf) gives alpha = 1 when p(x) > 0 and
 *     alpha = 0 when p(x) = 0.
 *   - the same temperature T_b scales every target and draft row of
 *     sequence b ([P2] divides the draft logits and the bonus logits by T).
 *   - the residual subtracts the full draft distribution of the rejected
 *     position ([P2] step 3 and [P3] 二.2; [P1] subtracts a gathered scalar).
 *   - multinomial sampling = inverse CDF in ascending vocabulary order:
 *     the smallest v with C_v > u * (sum of weights).
 *   - if every draft token is accepted, a bonus token is drawn from the
 *     target distribution at position k ([P2] step 3, [P3] 三 step 4).
 *   - greedy (T = 0): accept while x_i == argmax p_i (lowest index on ties);
 *     the first mismatch emits argmax p_i; full acceptance emits argmax p_k.
 *   - uniforms: u_accept[k_offsets[b] + i] for the test at position i,
 *     u_resample[k_offsets[b] + b + j] for the resample / bonus at position j.
 *   - a row holding NaN or +inf, a row that is entirely -inf, a draft token
 *     outside [0, V), or an invalid temperature makes the whole sequence a
 *     data error: num_accepted = -1 and all its token slots -1.
 *   - if the residual mass Z rounds to 0, sample p with the same uniform and
 *     report a zero decision margin.
 *
 * Decision margins (for boundary flagging in parity tests): for every
 * accept test evaluated, |u - alpha|; for the inverse CDF that chose token v,
 * min(u*Z - C_{v-1}, C_v - u*Z) / Z.  The smallest over one sequence is
 * reported.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_MAX_K 32

/* Convert one logit row to double (bf16: the 16 stored bits are the high
 * half of an fp32 pattern, so the conversion is exact). */
static void load_row(const void *base, int dtype, int64_t row, int V, double *dst)
{
    if (dtype == ORACLE_F32) {
        const float *p = (const float *)base + row * (int64_t)V;
        for (int v = 0; v < V; ++v) dst[v] = (double)p[v];
    } else {
        const uint16_t *p = (const uint16_t *)base + row * (int64_t)V;
        for (int v = 0; v < V; ++v) {
            uint32_t bits = (uint32_t)p[v] << 16;
            float f;
            memcpy(&f, &bits, sizeof f);
            dst[v] = (double)f;
        }
    }
}

static double logit_at(const void *base, int dtype, int64_t row, int V, int v)
{
    double d;
    if (dtype == ORACLE_F32) {
        d = (double)((const float *)base)[row * (int64_t)V + v];
    } else {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[row * (int64_t)V + v] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        d = (double)f;
    }
    return d;
}

/* log-sum-exp of z/T, two passes: M = max z/T, lse = M + log sum exp(z/T - M).
 * Returns -1 for a row that has no valid distribution. */
static int row_lse(const double *z, int V, double T, double *lse)
{
    double M = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double y = z[v] / T;
        if (isnan(y)) return -1;
        if (y > M) M = y;
    }
    if (!isfinite(M)) return -1; /* +inf present, or every entry -inf */
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp(z[v] / T - M);
    *lse = M + log(s);
    return 0;
}

/* argmax over raw logits, lowest index on ties; -1 if any NaN. */
static int row_argmax(const double *z, int V, int *arg)
{
    int best = 0;
    double bv = z[0];
    if (isnan(bv)) return -1;
    for (int v = 1; v < V; ++v) {
        if (isnan(z[v])) return -1;
        if (z[v] > bv) {
            bv = z[v];
            best = v;
        }
    }
    *arg = best;
    return 0;
}

/* Multinomial draw from non-negative weights w by inverse CDF: the smallest
 * v whose ascending cumulative sum exceeds u * sum(w).  If rounding leaves no
 * such v, the largest v with w_v > 0 (margin 0). */
static int inverse_cdf(const double *w, int V, double u, double *margin)
{
    double Z = 0.0;
    for (int v = 0; v < V; ++v) Z += w[v];
    double t = u * Z;
    double C = 0.0, Cprev = 0.0;
    for (int v = 0; v < V; ++v) {
        Cprev = C;
        C += w[v];
        if (C > t) {
            double a = (t - Cprev) / Z, b = (C - t) / Z;
            *margin = a < b ? a : b;
            return v;
        }
    }
    *margin = 0.0;
    for (int v = V - 1; v >= 0; --v)
        if (w[v] > 0.0) return v;
    return 0;
}

static int valid_temperature(float T)
{
    return T >= 0.0f && isfinite(T);
}

/* k_offsets must start at 0 and give 0 <= k_b <= ORACLE_MAX_K. */
static int valid_offsets(const int32_t *k_offsets, int B)
{
    if (k_offsets[0] != 0) return 0;
    for (int b = 0; b < B; ++b) {
        int32_t k = k_offsets[b + 1] - k_offsets[b];
        if (k < 0 || k > ORACLE_MAX_K) return 0;
    }
    return 1;
}

typedef struct {
    const void *target, *draft;
    int dtype, V;
    const int32_t *tokens;
    const float *u_accept, *u_resample, *temperature;
    const int32_t *k_offsets;
    int32_t *out_tokens, *out_num;
    double *accept_prob, *residual_mass, *lse_t, *lse_d, *margin;
} verify_args;

/* One sequence of the verify step ([P2] 三步流程 step 3; [P3] 三). */
static void verify_one(const verify_args *a, int b, double *rt, double *rd, double *w)
{
    const int V = a->V;
    const int32_t k = a->k_offsets[b + 1] - a->k_offsets[b];
    const int64_t ot = (int64_t)a->k_offsets[b] + b; /* first target row / output slot */
    const int64_t od = a->k_offsets[b];              /* first draft row */
    int32_t x[ORACLE_MAX_K];
    double lt[ORACLE_MAX_K + 1], ld[ORACLE_MAX_K], alpha[ORACLE_MAX_K];

    for (int i = 0; i <= k; ++i) a->out_tokens[ot + i] = -1;
    a->out_num[b] = -1;
    if (a->accept_prob)
        for (int i = 0; i < k; ++i) a->accept_prob[od + i] = NAN;
    if (a->lse_t)
        for (int i = 0; i <= k; ++i) a->lse_t[ot + i] = NAN;
    if (a->lse_d)
        for (int i = 0; i < k; ++i) a->lse_d[od + i] = NAN;
    if (a->residual_mass) a->residual_mass[b] = NAN;
    if (a->margin) a->margin[b] = INFINITY;

    const float Tf = a->temperature[b];
    if (!valid_temperature(Tf)) return;
    const double T = (double)Tf;
    for (int i = 0; i < k; ++i) {
        x[i] = a->tokens[od + i];
        if (x[i] < 0 || x[i] >= V) return;
    }

    if (T == 0.0) {
        /* Greedy ([P2] 动手实践, temperature == 0 branch): accept while the
         * draft token equals argmax of the target row. */
        int am[ORACLE_MAX_K + 1];
        for (int i = 0; i <= k; ++i) {
            load_row(a->target, a->dtype, ot + i, V, rt);
            if (row_argmax(rt, V, &am[i]) != 0) return;
        }
        int n = k;
        for (int i = 0; i < k; ++i) {
            if (x[i] != am[i]) {
                n = i;
                break;
            }
        }
        for (int i = 0; i < n; ++i) a->out_tokens[ot + i] = x[i];
        a->out_tokens[ot + n] = am[n];
        a->out_num[b] = n;
        return;
    }

    /* (a) temperature-scaled log-sum-exp of every row of the sequence. */
    for (int i = 0; i <= k; ++i) {
        load_row(a->target, a->dtype, ot + i, V, rt);
        if (row_lse(rt, V, T, &lt[i]) != 0) return;
    }
    for (int i = 0; i < k; ++i) {
        load_row(a->draft, a->dtype, od + i, V, rd);
        if (row_lse(rd, V, T, &ld[i]) != 0) return;
    }

    /* (b) alpha_i = min(1, p_i(x_i) / q_i(x_i)) ([P3] 二.1), ratio in the
     * log domain. */
    for (int i = 0; i < k; ++i) {
        double zt = logit_at(a->target, a->dtype, ot + i, V, x[i]);
        double zd = logit_at(a->draft, a->dtype, od + i, V, x[i]);
        if (zt == -INFINITY) {
            alpha[i] = 0.0;
        } else if (zd == -INFINITY) {
            alpha[i] = 1.0;
        } else {
            double lp = zt / T - lt[i];
            double lq = zd / T - ld[i];
            double r = exp(lp - lq);
            alpha[i] = r < 1.0 ? r : 1.0;
        }
    }

    /* Left-to-right accept test, stopping at the first rejection. */
    double mg = INFINITY;
    int j = k;
    for (int i = 0; i < k; ++i) {
        double u = (double)a->u_accept[od + i];
        double d = fabs(u - alpha[i]);
        if (d < mg) mg = d;
        if (u < alpha[i]) continue;
        j = i;
        break;
    }

    int32_t token;
    double cdf_margin;
    const double ur = (double)a->u_resample[ot + j];
    if (j < k) {
        /* (c) residual norm(max(0, p - q)) at the rejected position
         * ([P2] step 3; [P3] 二.2), sampled by inverse CDF. */
        load_row(a->target, a->dtype, ot + j, V, rt);
        load_row(a->draft, a->dtype, od + j, V, rd);
        double Z = 0.0;
        for (int v = 0; v < V; ++v) {
            double p = exp(rt[v] / T - lt[j]);
            double q = exp(rd[v] / T - ld[j]);
            double d = p - q;
            w[v] = d > 0.0 ? d : 0.0;
            Z += w[v];
        }
        if (a->residual_mass) a->residual_mass[b] = Z;
        if (Z > 0.0) {
            token = inverse_cdf(w, V, ur, &cdf_margin);
        } else {
            for (int v = 0; v < V; ++v) w[v] = exp(rt[v] / T - lt[j]);
            token = inverse_cdf(w, V, ur, &cdf_margin);
            cdf_margin = 0.0;
        }
    } else {
        /* Bonus token from the target distribution at position k
         * ([P2] step 3, last bullet; [P3] 三 step 4). */
        load_row(a->target, a->dtype, ot + k, V, rt);
        for (int v = 0; v < V; ++v) w[v] = exp(rt[v] / T - lt[k]);
        token = inverse_cdf(w, V, ur, &cdf_margin);
    }
    if (cdf_margin < mg) mg = cdf_margin;

    for (int i = 0; i < j; ++i) a->out_tokens[ot + i] = x[i];
    a->out_tokens[ot + j] = token;
    a->out_num[b] = j;
    if (a->margin) a->margin[b] = mg;
    if (a->accept_prob)
        for (int i = 0; i < k; ++i) a->accept_prob[od + i] = alpha[i];
    if (a->lse_t)
        for (int i = 0; i <= k; ++i) a->lse_t[ot + i] = lt[i];
    if (a->lse_d)
        for (int i = 0; i < k; ++i) a->lse_d[od + i] = ld[i];
}

/*
 * Verify B sequences (or only those listed in seq_list, if it is non-NULL).
 * Layout: target rows k_offsets[b]+b .. k_offsets[b+1]+b, draft rows
 * k_offsets[b] .. k_offsets[b+1]-1, both [rows, V] row-major.
 * out_tokens [k_offsets[B]+B]: accepted prefix, then the resampled or bonus
 * token, then -1.  out_num_accepted [B].  Aux arrays may be NULL.
 * Returns 0, or -1 if k_offsets is invalid (then every out_num_accepted = -1).
 */
int oracle_verify(const void *target_logits, const void *draft_logits, int dtype,
                  const int32_t *draft_tokens, const float *u_accept,
                  const float *u_resample, const float *temperature, int B,
                  const int32_t *k_offsets, int V, int32_t *out_tokens,
                  int32_t *out_num_accepted, double *accept_prob,
                  double *residual_mass, double *lse_target, double *lse_draft,
                  double *margin, const int32_t *seq_list, int n_list, int nthreads)
{
    if (B < 0 || V <= 0 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -2;
    if (B == 0) return 0;
    if (!valid_offsets(k_offsets, B)) {
        for (int b = 0; b < B; ++b) out_num_accepted[b] = -1;
        return -1;
    }
    verify_args a = {target_logits, draft_logits, dtype, V, draft_tokens, u_accept,
                     u_resample, temperature, k_offsets, out_tokens, out_num_accepted,
                     accept_prob, residual_mass, lse_target, lse_draft, margin};
    const int n = seq_list ? n_list : B;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *rt = (double *)malloc(sizeof(double) * (size_t)V);
        double *rd = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < n; ++t) {
            int b = seq_list ? seq_list[t] : t;
            if (b >= 0 && b < B) verify_one(&a, b, rt, rd, w);
        }
        free(rt);
        free(rd);
        free(w);
    }
    return 0;
}

/*
 * Draft-side sampling ([P2] 动手实践 drafting loop; [P1] draft_generate;
 * [P3] 三 step 1): for every draft row of sequence b, x = argmax if
 * T_b = 0, else the inverse-CDF draw from softmax(z / T_b) with u_draft[row].
 * Invalid rows (NaN / +inf / all -inf, or a bad temperature) give -1.
 */
int oracle_draft_sample(const void *draft_logits, int dtype, const float *temperature,
                        const float *u_draft, int B, const int32_t *k_offsets, int V,
                        int32_t *out_draft_tokens, double *margin, double *lse,
                        int nthreads)
{
    if (B < 0 || V <= 0 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -2;
    if (B == 0) return 0;
    if (!valid_offsets(k_offsets, B)) return -1;
    const int R = k_offsets[B];
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
        int b = 0;
#pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < R; ++r) {
            /* sequence owning row r */
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                int mid = (lo + hi + 1) / 2;
                if (k_offsets[mid] <= r) lo = mid; else hi = mid - 1;
            }
            b = lo;
            out_draft_tokens[r] = -1;
            if (margin) margin[r] = INFINITY;
            if (lse) lse[r] = NAN;
            const float Tf = temperature[b];
            if (!valid_temperature(Tf)) continue;
            load_row(draft_logits, dtype, r, V, z);
            if (Tf == 0.0f) {
                int am;
                if (row_argmax(z, V, &am) == 0) out_draft_tokens[r] = am;
                continue;
            }
            const double T = (double)Tf;
            double L;
            if (row_lse(z, V, T, &L) != 0) continue;
            for (int v = 0; v < V; ++v) w[v] = exp(z[v] / T - L);
            double m;
            out_draft_tokens[r] = inverse_cdf(w, V, (double)u_draft[r], &m);
            if (margin) margin[r] = m;
            if (lse) lse[r] = L;
        }
        (void)b;
        free(z);
        free(w);
    }
    return 0;
}

/* softmax(z / T) of one row, with its log-sum-exp.  Returns -1 for an
 * invalid row.  Used by the oracle's own tests. */
int oracle_softmax_row(const void *logits, int dtype, int V, double T, double *p_out,
                       double *lse_out)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    load_row(logits, dtype, 0, V, z);
    double L;
    int rc = row_lse(z, V, T, &L);
    if (rc == 0) {
        for (int v = 0; v < V; ++v) p_out[v] = exp(z[v] / T - L);
        *lse_out = L;
    }
    free(z);
    return rc;
}

/* ------------------------------------------------------------------------
 * Tree (multi-candidate) verify.
 *
 * The pages show draft trees (docs.ifdog.com "投机解码", 进阶方案: Medusa and
 * EAGLE verify a tree of candidates in one target forward) but give no
 * acceptance rule for them.  Reading taken: the plainest lossless extension
 * of the single-candidate rule of 三步流程 step 3 / [P3] 二.1-二.2 to several
 * candidates drawn i.i.d. from the same draft distribution.  At node u with
 * target distribution p (the target row of u) and draft distribution q (the
 * draft row of u), u's children c_1 < c_2 < ... (ascending node index) are
 * tried in order:
 *   - child c_j is accepted iff u_accept[c_j] < min(1, p^(j-1)(x) / q(x)),
 *     x its token, p^(0) = p;
 *   - on its rejection p^(j) = norm(max(0, p^(j-1) - q));
 *   - an accepted child becomes u, with p and q of its own rows;
 *   - when every child of u is rejected, one token is drawn from the last
 *     residual with u_resample[u] by inverse CDF (ascending vocabulary, on
 *     the unnormalised weights max(0, p^(m-1) - q), as the single-candidate
 *     residual draw); a node without children (a leaf, or the root of a
 *     one-node tree) draws the bonus token from its p.
 * Greedy (T = 0): the first child whose token equals argmax p (lowest index
 * on ties) is accepted; if none, argmax p is emitted.
 * Degenerate: if a residual mass rounds to 0, p^(j) = p^(j-1) (margin 0).
 * Every convention of the chain verify above (temperature, strict test,
 * q(x) = 0, data errors) carries over.
 * ---------------------------------------------------------------------- */
#define ORACLE_MAX_TREE 64

typedef struct {
    const void *target, *draft;
    int dtype, V;
    const int32_t *node_offsets, *parent, *tokens;
    const float *u_accept, *u_resample, *temperature;
    int32_t *out_tokens, *out_num, *out_last;
    double *margin;
} tree_args;

/* Nodes of sequence b are valid: 1..ORACLE_MAX_TREE of them, the first is
 * the root (parent -1), every other node's parent is an earlier node of the
 * same sequence. */
static int valid_tree(const tree_args *a, int b)
{
    const int32_t g0 = a->node_offsets[b], n = a->node_offsets[b + 1] - g0;
    if (n < 1 || n > ORACLE_MAX_TREE) return 0;
    if (a->parent[g0] != -1) return 0;
    for (int i = 1; i < n; ++i) {
        int32_t pa = a->parent[g0 + i];
        if (pa < g0 || pa >= g0 + i) return 0;
    }
    return 1;
}

/* One sequence of the tree verify.  p, q, w: scratch rows of V doubles. */
static void tree_verify_one(const tree_args *a, int b, double *rt, double *rd, double *p, double *q,
                            double *w)
{
    const int V = a->V;
    const int32_t g0 = a->node_offsets[b], n = a->node_offsets[b + 1] - g0;
    for (int i = 0; i < n; ++i) a->out_tokens[g0 + i] = -1;
    a->out_num[b] = -1;
    if (a->out_last) a->out_last[b] = -1;
    if (a->margin) a->margin[b] = INFINITY;
    if (!valid_tree(a, b)) return;
    const float Tf = a->temperature[b];
    if (!valid_temperature(Tf)) return;
    for (int i = 1; i < n; ++i)
        if (a->tokens[g0 + i] < 0 || a->tokens[g0 + i] >= V) return;
    const double T = (double)Tf;

    int32_t path[ORACLE_MAX_TREE];
    int nacc = 0;
    int32_t u = g0, token = -1;
    double mg = INFINITY;
    for (;;) {
        if (T == 0.0) {
            /* greedy: the first child whose token is argmax p */
            int am;
            load_row(a->target, a->dtype, u, V, rt);
            if (row_argmax(rt, V, &am) != 0) return;
            int32_t next = -1;
            for (int32_t c = u + 1; c < g0 + n && next < 0; ++c)
                if (a->parent[c] == u && a->tokens[c] == am) next = c;
            if (next < 0) {
                token = am;
                break;
            }
            path[nacc++] = a->tokens[next];
            u = next;
            continue;
        }
        double Lt, Ld = 0.0;
        load_row(a->target, a->dtype, u, V, rt);
        if (row_lse(rt, V, T, &Lt) != 0) return;
        for (int v = 0; v < V; ++v) p[v] = exp(rt[v] / T - Lt);
        int has_child = 0;
        for (int32_t c = u + 1; c < g0 + n; ++c) has_child |= a->parent[c] == u;
        if (!has_child) {
            /* a leaf: the bonus token from p */
            double m;
            token = inverse_cdf(p, V, (double)a->u_resample[u], &m);
            if (m < mg) mg = m;
            break;
        }
        load_row(a->draft, a->dtype, u, V, rd);
        if (row_lse(rd, V, T, &Ld) != 0) return;
        for (int v = 0; v < V; ++v) q[v] = exp(rd[v] / T - Ld);
        int32_t next = -1, j = 0;
        for (int32_t c = u + 1; c < g0 + n; ++c) {
            if (a->parent[c] != u) continue;
            const int32_t x = a->tokens[c];
            double alpha;
            if (rd[x] == -INFINITY) {
                alpha = p[x] > 0.0 ? 1.0 : 0.0;
            } else if (j == 0) {
                /* first candidate: the ratio in the log domain, as the chain */
                double r = rt[x] == -INFINITY ? 0.0 : exp((rt[x] / T - Lt) - (rd[x] / T - Ld));
                alpha = r < 1.0 ? r : 1.0;
            } else {
                double r = p[x] / q[x];
                alpha = r < 1.0 ? r : 1.0;
            }
            const double uc = (double)a->u_accept[c];
            const double d = fabs(uc - alpha);
            if (d < mg) mg = d;
            if (uc < alpha) {
                next = c;
                break;
            }
            /* rejected: p <- norm(max(0, p - q)) */
            double Z = 0.0;
            for (int v = 0; v < V; ++v) {
                double e = p[v] - q[v];
                w[v] = e > 0.0 ? e : 0.0;
                Z += w[v];
            }
            if (Z > 0.0) {
                for (int v = 0; v < V; ++v) p[v] = w[v] / Z;
            } else {
                mg = 0.0;
                for (int v = 0; v < V; ++v) w[v] = p[v];
            }
            ++j;
        }
        if (next >= 0) {
            path[nacc++] = a->tokens[next];
            u = next;
            continue;
        }
        /* every child rejected: draw from the last residual weights */
        double m;
        token = inverse_cdf(w, V, (double)a->u_resample[u], &m);
        if (m < mg) mg = m;
        break;
    }
    for (int i = 0; i < nacc; ++i) a->out_tokens[g0 + i] = path[i];
    a->out_tokens[g0 + nacc] = token;
    a->out_num[b] = nacc;
    if (a->out_last) a->out_last[b] = u;
    if (a->margin) a->margin[b] = mg;
}

/*
 * Tree verify of B sequences.  Sequence b owns nodes node_offsets[b] ..
 * node_offsets[b+1]-1 (the first is its root); parent [N] (-1 for a root),
 * tokens [N] (a root's is ignored), target and draft logits [N, V] (row g:
 * the distributions after the path to node g; draft rows of leaves are not
 * read), u_accept [N] (the test of node g), u_resample [N] (the draw at node
 * g), temperature [B].  Outputs: out_tokens [N] (the accepted path's tokens,
 * then the drawn token, then -1, from slot node_offsets[b]),
 * out_num_accepted [B], out_last_node [B] and margin [B] (may be NULL).
 * Returns 0, or -1 if node_offsets is invalid (node_offsets[0] != 0 or a
 * sequence without 1..64 nodes; then every out_num_accepted = -1).
 */
int oracle_tree_verify(const void *target_logits, const void *draft_logits, int dtype,
                       const int32_t *node_offsets, const int32_t *parent, const int32_t *tokens,
                       const float *u_accept, const float *u_resample, const float *temperature,
                       int B, int V, int32_t *out_tokens, int32_t *out_num_accepted,
                       int32_t *out_last_node, double *margin, int nthreads)
{
    if (B < 0 || V <= 0 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -2;
    if (B == 0) return 0;
    int ok = node_offsets[0] == 0;
    for (int b = 0; b < B && ok; ++b) {
        int32_t n = node_offsets[b + 1] - node_offsets[b];
        ok = n >= 1 && n <= ORACLE_MAX_TREE;
    }
    if (!ok) {
        for (int b = 0; b < B; ++b) out_num_accepted[b] = -1;
        return -1;
    }
    tree_args a = {target_logits, draft_logits, dtype, V, node_offsets, parent, tokens, u_accept,
                   u_resample, temperature, out_tokens, out_num_accepted, out_last_node, margin};
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *buf = (double *)malloc(sizeof(double) * (size_t)V * 5);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b)
            tree_verify_one(&a, b, buf, buf + V, buf + 2 * (size_t)V, buf + 3 * (size_t)V, buf + 4 * (size_t)V);
        free(buf);
    }
    return 0;
}

/*
 * Tree drafting: every non-root node g takes its token from the draft
 * distribution of its parent, x_g = argmax z (T_b = 0) or the inverse-CDF
 * draw from softmax(z / T_b) at u_draft[g], z the draft row of parent(g):
 * siblings are independent draws from one distribution, as the tree verify
 * above requires.  Roots and invalid rows give -1; margin [N] as for the
 * chain draft sample.
 */
int oracle_tree_draft_sample(const void *draft_logits, int dtype, const int32_t *node_offsets,
                             const int32_t *parent, const float *temperature, const float *u_draft,
                             int B, int V, int32_t *out_tokens, double *margin, int nthreads)
{
    if (B < 0 || V <= 0 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -2;
    if (B == 0) return 0;
    const int N = node_offsets[B];
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 4)
        for (int g = 0; g < N; ++g) {
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                int mid = (lo + hi + 1) / 2;
                if (node_offsets[mid] <= g) lo = mid; else hi = mid - 1;
            }
            const int b = lo;
            out_tokens[g] = -1;
            if (margin) margin[g] = INFINITY;
            const int32_t pa = parent[g];
            if (pa < node_offsets[b] || pa >= g) continue;
            const float Tf = temperature[b];
            if (!valid_temperature(Tf)) continue;
            load_row(draft_logits, dtype, pa, V, z);
            if (Tf == 0.0f) {
                int am;
                if (row_argmax(z, V, &am) == 0) out_tokens[g] = am;
                continue;
            }
            const double T = (double)Tf;
            double L;
            if (row_lse(z, V, T, &L) != 0) continue;
            for (int v = 0; v < V; ++v) w[v] = exp(z[v] / T - L);
            double m;
            out_tokens[g] = inverse_cdf(w, V, (double)u_draft[g], &m);
            if (margin) margin[g] = m;
        }
        free(z);
        free(w);
    }
    return 0;
}
