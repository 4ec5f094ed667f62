/*
 * oracle.c -- plain fp64 CPU oracle for batched draft-token verification by
 * modified rejection sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg load this library; the GPU library
 * never links, includes or calls it, and the two share no code, header,
 * table or helper.  The product path must never route through this file.
 *
 * What it follows (page title, then the section):
 *  [P1] tech-tldr.com "投機的デコーディングとドラフトモデル",
 *       section 受理判定の数理：修正版棄却サンプリング: a proposal x_i is kept when
 *       a uniform r in [0,1) satisfies r < min(1, p(x_i)/q(x_i)); at the first
 *       failure the round stops and one token is drawn from the normalised
 *       positive part of p - q.
 *  [P2] r-jc.jp "LLM推論の高速化｜KVキャッシュと投機的デコーディングを自作で実測",
 *       section 投機的デコーディングとは（speculative decoding の仕組み): the
 *       verification loop -- p = probs(logits_i, temp) per position, tests in
 *       order, break at the first rejection, then row nacc supplies either the
 *       residual (some proposal rejected) or the target distribution itself
 *       (all accepted, the bonus token), and one token is drawn from it.
 *       Section 投機的デコーディングを実装して受理率と速度を実測: at temperature 0
 *       the test becomes "the target argmax equals the proposal".
 *  [P3] issoh.co.jp "Speculative Decoding（投機的デコーディング）とは？仕組みと速くなる条件…",
 *       section 受理・棄却の規則と出力分布が変わらない理由, steps 1-5.
 *
 * Readings where the pages leave a step open:
 *  R1 probs(l, T) is softmax(l / T); the pages use it without printing it.
 *  R2 the test is strict, r < min(1, p/q), with r in [0, 1).  When q(x) = 0
 *     the ratio is undefined; the token is then kept iff p(x) > 0.
 *  R3 uniforms sit in fixed slots: slot i < K_b is the test of position i,
 *     slot K_b the final draw (resample or bonus).
 *  R4 the draw normalises r and takes the smallest j with u < C_j, C_j the
 *     running sum in index order; if rounding leaves no such j, the largest j
 *     with r_j > 0.
 *  R5 if the positive part of p - q sums to 0 at a rejected row, the draw
 *     uses p of that row (counted and returned).
 *  R6 greedy (T = 0): g_i is the argmax, lowest index on ties; keep iff
 *     x_i == g_i; the final token is g_nacc.  Uniforms are not used.
 *  R7 a row is unusable if it holds a NaN or +inf or has no finite entry; a
 *     temperature is usable if it is 0 or a normal, finite, positive float; a
 *     token must lie in [0, V); a uniform in [0, 1).  Any unusable input that
 *     the loop reaches makes that sequence's outputs -1.
 *
 * Layout (row-major, contiguous): target [B][Kmax+1][V], draft [B][Kmax][V],
 * tokens [B][Kmax], uniforms [B][Kmax+1], temperature [B], K [B];
 * outputs out_tokens [B][Kmax+1] (unused slots -1), out_nacc [B].
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_TIE_BAND 1e-6

/* Exact conversion of one stored logit to double. */
static double logit_at(const void* base, int dtype, size_t idx)
{
    if (dtype == ORC_F32)
        return (double)((const float*)base)[idx];
    uint32_t w = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* R7: the row's maximum, or 0 if the row is unusable. */
static int row_max(const void* base, int dtype, size_t off, int V, double* m_out)
{
    double m = -INFINITY;
    for (int j = 0; j < V; ++j) {
        double x = logit_at(base, dtype, off + (size_t)j);
        if (isnan(x) || x == INFINITY)
            return 0;
        if (x > m)
            m = x;
    }
    if (m == -INFINITY)
        return 0;
    *m_out = m;
    return 1;
}

/* R1: out[j] = exp((l_j - m)/T) / sum_k exp((l_k - m)/T). */
static int probs(const void* base, int dtype, size_t off, int V, double T, double* out)
{
    double m;
    if (!row_max(base, dtype, off, V, &m))
        return 0;
    double S = 0.0;
    for (int j = 0; j < V; ++j) {
        out[j] = exp((logit_at(base, dtype, off + (size_t)j) - m) / T);
        S += out[j];
    }
    for (int j = 0; j < V; ++j)
        out[j] /= S;
    return 1;
}

/* R6: lowest index holding the row maximum. */
static int argmax_row(const void* base, int dtype, size_t off, int V, int* g)
{
    double m;
    if (!row_max(base, dtype, off, V, &m))
        return 0;
    for (int j = 0; j < V; ++j)
        if (logit_at(base, dtype, off + (size_t)j) == m) {
            *g = j;
            return 1;
        }
    return 0;
}

/* R2: keep x when u < min(1, p(x)/q(x)). */
static int keep(double u, double px, double qx)
{
    if (qx > 0.0)
        return u < fmin(1.0, px / qx);
    return px > 0.0;
}

/* [P1][P2]: r = max(0, p - q) normalised; R5 fallback to p.  Returns 1 when
 * the fallback was taken. */
static int residual(const double* p, const double* q, int V, double* r)
{
    double S = 0.0;
    for (int j = 0; j < V; ++j) {
        r[j] = fmax(p[j] - q[j], 0.0);
        S += r[j];
    }
    if (!(S > 0.0)) {
        memcpy(r, p, (size_t)V * sizeof *r);
        return 1;
    }
    for (int j = 0; j < V; ++j)
        r[j] /= S;
    return 0;
}

/* R4: inverse-CDF draw from a normalised r.  *tie is set when u lies within
 * ORC_TIE_BAND of either boundary of the chosen token's interval. */
static int draw(const double* r, int V, double u, int* tie)
{
    double C = 0.0, Cprev = 0.0;
    int tok = -1;
    for (int j = 0; j < V; ++j) {
        Cprev = C;
        C += r[j];
        if (u < C) {
            tok = j;
            break;
        }
    }
    if (tok < 0) {
        for (int j = V - 1; j >= 0; --j)
            if (r[j] > 0.0) {
                tok = j;
                break;
            }
        C = 0.0;
        for (int j = 0; j <= tok; ++j) {
            Cprev = C;
            C += r[j];
        }
    }
    if (fabs(u - Cprev) < ORC_TIE_BAND || fabs(u - C) < ORC_TIE_BAND)
        *tie = 1;
    return tok;
}

static int temperature_usable(float T)
{
    return T == 0.0f || (isfinite(T) && T >= FLT_MIN);
}

static int uniform_usable(float u)
{
    return u >= 0.0f && u < 1.0f;
}

/*
 * Verify B sequences.  Returns the number of R5 fallbacks taken, or -1 on a
 * bad argument.  tie (nullable, [B]) flags sequences with a decision within
 * ORC_TIE_BAND of its threshold; final_row (nullable, [B]) receives nacc.
 */
int oracle_verify(const void* target, const void* draft, int dtype,
                  const int32_t* tokens, const float* uniforms, const float* temperature,
                  int32_t B, const int32_t* K, int32_t Kmax, int32_t V,
                  int32_t* out_tokens, int32_t* out_nacc,
                  uint8_t* tie, int32_t* final_row)
{
    if (B < 0 || V < 1 || Kmax < 0 || (dtype != ORC_F32 && dtype != ORC_BF16))
        return -1;
    if (B == 0)
        return 0;
    if (!target || !uniforms || !temperature || !K || !out_tokens || !out_nacc)
        return -1;
    if (Kmax > 0 && !tokens)
        return -1;
    double* p = (double*)malloc((size_t)V * sizeof(double));
    double* q = (double*)malloc((size_t)V * sizeof(double));
    double* r = (double*)malloc((size_t)V * sizeof(double));
    if (!p || !q || !r) {
        free(p); free(q); free(r);
        return -1;
    }
    int fallbacks = 0;
    for (int b = 0; b < B; ++b) {
        const int Kb = K[b];
        const float T = temperature[b];
        int32_t* orow = out_tokens + (size_t)b * (Kmax + 1);
        for (int j = 0; j <= Kmax; ++j)
            orow[j] = -1;
        out_nacc[b] = -1;
        if (tie)
            tie[b] = 0;
        if (final_row)
            final_row[b] = -1;
        if (Kb < 0 || Kb > Kmax || !temperature_usable(T))
            continue;
        const int greedy = (T == 0.0f);
        int nacc = 0, rejected = 0, ok = 1, t = 0, g = -1;
        for (int i = 0; i < Kb; ++i) {
            const int x = tokens[(size_t)b * Kmax + i];
            const size_t toff = ((size_t)b * (Kmax + 1) + i) * (size_t)V;
            const size_t doff = ((size_t)b * Kmax + i) * (size_t)V;
            if (x < 0 || x >= V) { ok = 0; break; }
            if (greedy) {
                if (!argmax_row(target, dtype, toff, V, &g)) { ok = 0; break; }
                if (x != g) { rejected = 1; break; }
            } else {
                const float u = uniforms[(size_t)b * (Kmax + 1) + i];
                if (!uniform_usable(u) || !draft) { ok = 0; break; }
                if (!probs(target, dtype, toff, V, (double)T, p) ||
                    !probs(draft, dtype, doff, V, (double)T, q)) { ok = 0; break; }
                if (q[x] > 0.0 && fabs((double)u - p[x] / q[x]) < ORC_TIE_BAND)
                    t = 1;
                if (!keep((double)u, p[x], q[x])) { rejected = 1; break; }
            }
            ++nacc;
        }
        if (!ok)
            continue;
        int token;
        const size_t foff = ((size_t)b * (Kmax + 1) + nacc) * (size_t)V;
        if (greedy) {
            if (!rejected && !argmax_row(target, dtype, foff, V, &g))
                continue;
            token = g;
        } else {
            const float u = uniforms[(size_t)b * (Kmax + 1) + Kb];
            if (!uniform_usable(u))
                continue;
            if (rejected) {
                fallbacks += residual(p, q, V, r);
            } else {
                if (!probs(target, dtype, foff, V, (double)T, p))
                    continue;
                memcpy(r, p, (size_t)V * sizeof *r);
            }
            token = draw(r, V, (double)u, &t);
        }
        for (int j = 0; j < nacc; ++j)
            orow[j] = tokens[(size_t)b * Kmax + j];
        orow[nacc] = token;
        out_nacc[b] = nacc;
        if (tie)
            tie[b] = (uint8_t)t;
        if (final_row)
            final_row[b] = nacc;
    }
    free(p); free(q); free(r);
    return fallbacks;
}

/*
 * Per-position quantities at every draft position i < K_b of a sampling
 * sequence (not only the tested ones): p_i(x_i), q_i(x_i) and the residual
 * mass sum_j max(0, p_i(j) - q_i(j)) = 1 - alpha_i.  Entries that do not
 * apply (greedy sequence, i >= K_b, unusable input) are NaN.  Outputs are
 * [B][Kmax].  Returns 0, or -1 on a bad argument.
 */
int oracle_position_probs(const void* target, const void* draft, int dtype,
                          const int32_t* tokens, const float* temperature,
                          int32_t B, const int32_t* K, int32_t Kmax, int32_t V,
                          double* p_x, double* q_x, double* resid_mass)
{
    if (B < 0 || V < 1 || Kmax < 0 || (dtype != ORC_F32 && dtype != ORC_BF16))
        return -1;
    if (B == 0 || Kmax == 0)
        return 0;
    if (!target || !tokens || !temperature || !K || !p_x || !q_x || !resid_mass)
        return -1;
    double* p = (double*)malloc((size_t)V * sizeof(double));
    double* q = (double*)malloc((size_t)V * sizeof(double));
    if (!p || !q) {
        free(p); free(q);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const float T = temperature[b];
        for (int i = 0; i < Kmax; ++i) {
            const size_t o = (size_t)b * Kmax + i;
            p_x[o] = q_x[o] = resid_mass[o] = NAN;
            if (i >= K[b] || T == 0.0f || !temperature_usable(T) || !draft)
                continue;
            const int x = tokens[o];
            if (x < 0 || x >= V)
                continue;
            const size_t toff = ((size_t)b * (Kmax + 1) + i) * (size_t)V;
            const size_t doff = ((size_t)b * Kmax + i) * (size_t)V;
            if (!probs(target, dtype, toff, V, (double)T, p) ||
                !probs(draft, dtype, doff, V, (double)T, q))
                continue;
            double S = 0.0;
            for (int j = 0; j < V; ++j)
                S += fmax(p[j] - q[j], 0.0);
            p_x[o] = p[x];
            q_x[o] = q[x];
            resid_mass[o] = S;
        }
    }
    free(p); free(q);
    return 0;
}

/*
 * The distribution the final draw uses for one row: the normalised residual
 * max(0, p - q) when a draft row is given (R5 fallback to p), else p itself.
 * Returns 1 (residual or p), 2 (R5 fallback taken) or 0 (unusable input).
 */
int oracle_final_distribution(const void* target_row, const void* draft_row, int dtype,
                              int32_t V, float T, double* r_out)
{
    if (V < 1 || !target_row || !r_out || !(isfinite(T) && T >= FLT_MIN))
        return 0;
    double* p = (double*)malloc((size_t)V * sizeof(double));
    double* q = (double*)malloc((size_t)V * sizeof(double));
    int rc = 0;
    if (p && q && probs(target_row, dtype, 0, V, (double)T, p)) {
        if (draft_row) {
            if (probs(draft_row, dtype, 0, V, (double)T, q))
                rc = residual(p, q, V, r_out) ? 2 : 1;
        } else {
            memcpy(r_out, p, (size_t)V * sizeof *r_out);
            rc = 1;
        }
    }
    free(p); free(q);
    return rc;
}

/*
 * Token-tree verification: the pages' accept rule applied at every node of a
 * tree of proposals.  A chain (one child per node) is exactly oracle_verify.
 *
 * Per sequence b, nodes 0 .. n_nodes[b] - 1, node 0 the root; parent[b][n] < n
 * for n >= 1.  The candidates at node v are its children (the nodes whose
 * parent is v) in increasing index.  Target row n: the target's logits after
 * node n; draft row n: the draft's logits after node n, the distribution the
 * children of n were drawn from.  uniforms[b][n] (n >= 1) is the test of node
 * n; uniforms[b][0] is the final draw.  Layouts: logits [B][Nmax][V], tokens,
 * parent, uniforms [B][Nmax].
 *
 * Walk from the root.  At node v, with P = softmax(target_v / T),
 * Q = softmax(draft_v / T) and R = P, the children are tested in order: child
 * c (token x) is kept iff u_c < min(1, R(x) / Q(x)) ([P1][P2][P3], with R in
 * the place of p); a kept child becomes the node walked next.  After a
 * rejection R becomes normalize(max(0, R - Q)), the distribution [P1] draws
 * from after a rejection, against which the next child is tested (R is left
 * unchanged if that has no mass, as R5 does for a chain).  With no child
 * kept, the token is drawn from R by inverse CDF with uniforms[b][0]; at a
 * leaf R = P, the bonus token.  At T = 0 the first child equal to
 * argmax target_v is kept, and the token is argmax target_v.
 *
 * Outputs ([B][Nmax]): out_path[b][0 .. len-1] the kept nodes,
 * out_tokens[b][0 .. len-1] their tokens and out_tokens[b][len] the drawn
 * token, -1 after; out_len[b] = len.  Unusable input on the walk (bad tree,
 * temperature, token, uniform or row) gives len -1 and -1 everywhere.  tie
 * (nullable) flags a decision within ORC_TIE_BAND of its threshold.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_tree_verify(const void* target, const void* draft, int dtype, const int32_t* tokens,
                       const int32_t* parent, const float* uniforms, const float* temperature,
                       int32_t B, const int32_t* n_nodes, int32_t Nmax, int32_t V,
                       int32_t* out_tokens, int32_t* out_path, int32_t* out_len, uint8_t* tie)
{
    if (B < 0 || V < 1 || Nmax < 1 || (dtype != ORC_F32 && dtype != ORC_BF16))
        return -1;
    if (B == 0)
        return 0;
    if (!target || !tokens || !parent || !uniforms || !temperature || !n_nodes || !out_tokens ||
        !out_path || !out_len)
        return -1;
    double* p = (double*)malloc((size_t)V * sizeof(double));
    double* q = (double*)malloc((size_t)V * sizeof(double));
    double* r = (double*)malloc((size_t)V * sizeof(double));
    int32_t* path = (int32_t*)malloc((size_t)Nmax * sizeof(int32_t));
    if (!p || !q || !r || !path) {
        free(p); free(q); free(r); free(path);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const size_t row0 = (size_t)b * Nmax;
        for (int j = 0; j < Nmax; ++j) {
            out_tokens[row0 + j] = -1;
            out_path[row0 + j] = -1;
        }
        out_len[b] = -1;
        if (tie)
            tie[b] = 0;
        const int N = n_nodes[b];
        const float T = temperature[b];
        if (N < 1 || N > Nmax || !temperature_usable(T))
            continue;
        int ok = 1;
        for (int n = 1; n < N; ++n)
            if (parent[row0 + n] < 0 || parent[row0 + n] >= n)
                ok = 0;
        if (!ok)
            continue;
        const int greedy = (T == 0.0f);
        int v = 0, len = 0, t = 0, token = -1;
        for (;;) {
            const size_t off = (row0 + v) * (size_t)V;
            int moved = 0;
            if (greedy) {
                int g = -1;
                if (!argmax_row(target, dtype, off, V, &g)) { ok = 0; break; }
                for (int c = v + 1; c < N && ok && !moved; ++c) {
                    if (parent[row0 + c] != v)
                        continue;
                    const int x = tokens[row0 + c];
                    if (x < 0 || x >= V) { ok = 0; break; }
                    if (x == g) {
                        path[len++] = c;
                        v = c;
                        moved = 1;
                    }
                }
                if (!ok)
                    break;
                if (moved)
                    continue;
                token = g;
                break;
            }
            if (!probs(target, dtype, off, V, (double)T, p)) { ok = 0; break; }
            memcpy(r, p, (size_t)V * sizeof *r);
            int have_q = 0;
            for (int c = v + 1; c < N && ok && !moved; ++c) {
                if (parent[row0 + c] != v)
                    continue;
                const int x = tokens[row0 + c];
                const float u = uniforms[row0 + c];
                if (x < 0 || x >= V || !uniform_usable(u)) { ok = 0; break; }
                if (!have_q) {
                    if (!draft || !probs(draft, dtype, off, V, (double)T, q)) { ok = 0; break; }
                    have_q = 1;
                }
                if (q[x] > 0.0 && fabs((double)u - r[x] / q[x]) < ORC_TIE_BAND)
                    t = 1;
                if (keep((double)u, r[x], q[x])) {
                    path[len++] = c;
                    v = c;
                    moved = 1;
                    break;
                }
                double S = 0.0;   // the next residual: normalize(max(0, r - q))
                for (int j = 0; j < V; ++j)
                    S += fmax(r[j] - q[j], 0.0);
                if (S > 0.0)
                    for (int j = 0; j < V; ++j)
                        r[j] = fmax(r[j] - q[j], 0.0) / S;
            }
            if (!ok)
                break;
            if (moved)
                continue;
            const float u0 = uniforms[row0];
            if (!uniform_usable(u0)) { ok = 0; break; }
            token = draw(r, V, (double)u0, &t);
            break;
        }
        if (!ok)
            continue;
        for (int j = 0; j < len; ++j) {
            out_path[row0 + j] = path[j];
            out_tokens[row0 + j] = tokens[row0 + path[j]];
        }
        out_tokens[row0 + len] = token;
        out_len[b] = len;
        if (tie)
            tie[b] = (uint8_t)t;
    }
    free(p); free(q); free(r); free(path);
    return 0;
}

int oracle_abi_version(void)
{
    return 1;
}
