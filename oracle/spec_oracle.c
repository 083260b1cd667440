/*
 * spec_oracle.c -- plain, slow, float64 CPU oracle for batched speculative
 * sampling verification, greedy verification, DDTree building and walking,
 * and DSpark adaptive verify length.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may call this code.  It shares nothing with the CUDA
 * library: no header, helper, table or constant.
 *
 * Source page (cited by section below):
 *   [SD-survey] "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
 *               (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash,
 *               DDTree and DSpark), chzhyang.github.io.
 *
 * Every step is a scalar loop in double precision, in the order the page
 * states it.  Library primitives used as steps: qsort (ordering a row),
 * exp (libm).  Compile with -ffp-contract=off so that no multiply-add is
 * fused: the results then do not depend on the host architecture.
 *
 * Readings of points the page leaves open (each one is also listed in the
 * design notes):
 *   - temperature and top-k fold into p: S = {x : l_x >= tau} with tau the
 *     top_k-th largest raw logit (ties at tau kept), p = softmax(l/T) on S,
 *     0 elsewhere.  q is used exactly as given (not truncated, not rescaled).
 *   - accept position i iff u_i < p_i(y_i)/q_i(y_i); with u_i uniform on
 *     [0,1) this happens with probability min(1, p/q).
 *   - uniforms u[b, 0..K]: u[b, i] decides position i, u[b, k] drives the one
 *     inverse-CDF sample (correction or bonus).
 *   - inverse CDF: ascending token id; the smallest x with C(x) > u * W.
 *   - q(y) == 0: ratio +inf if p(y) > 0 else 0 (status bit 2).
 *   - residual mass <= 0 after a rejection: sample from p instead (bit 4).
 *   - an invalid logits row (NaN, +Inf, or all -Inf) stops the walk with the
 *     drafts accepted so far and no correction token (bit 1).
 */
#include "spec_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* element access                                                       */
/* ------------------------------------------------------------------ */

static double logit_at(const void* base, int ldt, int64_t off)
{
    if (ldt == 0) return (double)((const float*)base)[off];
    /* bf16: the 16 stored bits are the top half of an IEEE binary32 */
    uint16_t h = ((const uint16_t*)base)[off];
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void load_row(const void* base, int ldt, int64_t start, int V, double* out)
{
    for (int x = 0; x < V; ++x) out[x] = logit_at(base, ldt, start + x);
}

/* NaN, +Inf, or no entry above -Inf */
static int row_valid(const double* l, int V)
{
    int any = 0;
    for (int x = 0; x < V; ++x) {
        if (isnan(l[x]) || l[x] == INFINITY) return 0;
        if (l[x] > -INFINITY) any = 1;
    }
    return any;
}

static int cmp_double_desc(const void* a, const void* b)
{
    double x = *(const double*)a, y = *(const double*)b;
    return (x < y) - (x > y);
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §1: temperature and truncation are part of p             */
/* ------------------------------------------------------------------ */

/* p(x) = exp((l_x - m)/T) / Z on S = {x : l_x >= tau}, 0 elsewhere.
 * m = max l, tau = top_k-th largest l (ties kept) or -inf without top-k.
 * Writes p (normalised) and returns Z = sum over S of exp((l_x - m)/T). */
static double form_p(const double* l, int V, double T, int top_k,
                     double* p, double* scratch)
{
    double m = -INFINITY;
    for (int x = 0; x < V; ++x)
        if (l[x] > m) m = l[x];
    double tau = -INFINITY;
    if (top_k > 0 && top_k < V) {
        memcpy(scratch, l, (size_t)V * sizeof(double));
        qsort(scratch, (size_t)V, sizeof(double), cmp_double_desc);
        tau = scratch[top_k - 1];
    }
    double Z = 0.0;
    for (int x = 0; x < V; ++x) {
        double w = (l[x] >= tau) ? exp((l[x] - m) / T) : 0.0;
        p[x] = w;
        Z += w;
    }
    for (int x = 0; x < V; ++x) p[x] = p[x] / Z;
    return Z;
}

/* Inverse CDF over weights w in ascending id: the smallest x with
 * C(x) = w_0 + ... + w_x > u * W, W = C(V-1).  *near is set when u*W lies
 * within 1e-6*W of C(x-1) or C(x). */
static int sample_icdf(const double* w, int V, double u, int* near, double* W_out)
{
    double W = 0.0;
    for (int x = 0; x < V; ++x) W += w[x];
    double t = u * W;
    double C = 0.0, Cprev = 0.0;
    int pick = -1;
    for (int x = 0; x < V; ++x) {
        Cprev = C;
        C += w[x];
        if (C > t) { pick = x; break; }
    }
    if (pick < 0) {
        /* unreachable for 0 <= u < 1 and W > 0; keep the last positive weight */
        for (int x = V - 1; x >= 0; --x)
            if (w[x] > 0.0) { pick = x; break; }
        *near = 1;
    } else {
        *near = (t - Cprev <= ORC_NEAR_TIE * W) || (C - t <= ORC_NEAR_TIE * W);
    }
    if (W_out) *W_out = W;
    return pick;
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §1: chain speculative sampling                            */
/* ------------------------------------------------------------------ */

void oracle_verify_chain(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const float* q, int64_t q_bstride, int64_t q_rstride,
    const int32_t* draft, const float* uniforms,
    int B, int K, int V, float temperature, int top_k,
    const int32_t* k_per_req, const int32_t* l_row_off, const int32_t* q_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    double* diag, int32_t* near_tie, int32_t* rows_read)
{
    double* l = (double*)malloc((size_t)V * sizeof(double));
    double* p = (double*)malloc((size_t)V * sizeof(double));
    double* r = (double*)malloc((size_t)V * sizeof(double));
    double* scratch = (double*)malloc((size_t)V * sizeof(double));
    const double T = (double)temperature;

    for (int b = 0; b < B; ++b) {
        int32_t* tok = out_tokens + (int64_t)b * (K + 1);
        for (int i = 0; i <= K; ++i) tok[i] = -1;
        int st = 0, nt = 0, nread = 0, n = 0;

        int k = K;
        if (k_per_req) {
            k = k_per_req[b];
            if (k < 0 || k > K) {
                num_accepted[b] = 0; status[b] = ORC_ST_BAD_K;
                if (near_tie) near_tie[b] = 0;
                if (rows_read) rows_read[b] = 0;
                continue;
            }
        }
        const float* u = uniforms + (int64_t)b * (K + 1);
        const double u_sample = (double)u[k];

        int finished = 0;
        for (int i = 0; i < k && !finished; ++i) {
            int64_t lrow = l_row_off ? ((int64_t)l_row_off[b] + i) * l_rstride
                                     : (int64_t)b * l_bstride + (int64_t)i * l_rstride;
            int64_t qrow = q_row_off ? ((int64_t)q_row_off[b] + i) * q_rstride
                                     : (int64_t)b * q_bstride + (int64_t)i * q_rstride;
            load_row(logits, ldt, lrow, V, l);
            nread++;
            if (!row_valid(l, V)) { st |= ORC_ST_BAD_ROW; n = i; finished = 1; break; }
            double Z = form_p(l, V, T, top_k, p, scratch);

            /* [SD-survey] §1 eq. alpha: accept with probability min(1, p/q) */
            int y = draft[(int64_t)b * K + i];
            double py = 0.0, qy = 0.0, ratio = 0.0;
            if (y < 0 || y >= V) {
                st |= ORC_ST_BAD_TOKEN;
                ratio = 0.0;
            } else {
                py = p[y];
                qy = (double)q[qrow + y];
                if (qy == 0.0) {
                    st |= ORC_ST_Q_ZERO;
                    ratio = (py > 0.0) ? INFINITY : 0.0;
                } else {
                    ratio = py / qy;
                }
            }
            double ui = (double)u[i];
            if (i < 31 && fabs(ui - ratio) <= ORC_NEAR_TIE) nt |= (1 << i);
            if (diag) {
                double* dg = diag + ((int64_t)b * (K + 1) + i) * 4;
                dg[0] = py; dg[1] = qy; dg[2] = Z; dg[3] = 0.0;
            }
            if (ui < ratio) {
                tok[i] = y;
                continue;
            }
            /* [SD-survey] §1: at the first rejection, sample the correction
             * token from the normalised positive residual [p - q]_+ */
            for (int x = 0; x < V; ++x) {
                double d = p[x] - (double)q[qrow + x];
                r[x] = d > 0.0 ? d : 0.0;
            }
            double R = 0.0;
            for (int x = 0; x < V; ++x) R += r[x];
            if (diag) diag[((int64_t)b * (K + 1) + i) * 4 + 3] = R;
            int near = 0, x;
            if (R > 0.0) {
                x = sample_icdf(r, V, u_sample, &near, NULL);
            } else {
                st |= ORC_ST_R_ZERO;
                x = sample_icdf(p, V, u_sample, &near, NULL);
            }
            if (near) nt |= (int)(1u << 31);
            tok[i] = x;
            n = i;
            finished = 1;
        }

        if (!finished) {
            /* [SD-survey] §1: every draft passed, sample one more token from
             * the target distribution of the next position */
            int64_t lrow = l_row_off ? ((int64_t)l_row_off[b] + k) * l_rstride
                                     : (int64_t)b * l_bstride + (int64_t)k * l_rstride;
            load_row(logits, ldt, lrow, V, l);
            nread++;
            n = k;
            if (!row_valid(l, V)) {
                st |= ORC_ST_BAD_ROW;
            } else {
                double Z = form_p(l, V, T, top_k, p, scratch);
                int near = 0;
                int x = sample_icdf(p, V, u_sample, &near, NULL);
                if (near) nt |= (int)(1u << 31);
                tok[k] = x;
                if (diag) {
                    double* dg = diag + ((int64_t)b * (K + 1) + k) * 4;
                    dg[0] = p[x]; dg[1] = 0.0; dg[2] = Z; dg[3] = 0.0;
                }
            }
        }
        num_accepted[b] = n;
        status[b] = st;
        if (near_tie) near_tie[b] = nt;
        if (rows_read) rows_read[b] = nread;
    }
    free(l); free(p); free(r); free(scratch);
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §1: greedy consistency -- accept while the draft equals   */
/* the target argmax; the first mismatch commits the argmax              */
/* ------------------------------------------------------------------ */

/* lowest index among the maximal values */
static int argmax_row(const double* l, int V)
{
    int best = 0;
    for (int x = 1; x < V; ++x)
        if (l[x] > l[best]) best = x;
    return best;
}

void oracle_verify_greedy(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const int32_t* draft, int B, int K, int V,
    const int32_t* k_per_req, const int32_t* l_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    int32_t* rows_read)
{
    double* l = (double*)malloc((size_t)V * sizeof(double));
    for (int b = 0; b < B; ++b) {
        int32_t* tok = out_tokens + (int64_t)b * (K + 1);
        for (int i = 0; i <= K; ++i) tok[i] = -1;
        int st = 0, nread = 0, n = 0;
        int k = K;
        if (k_per_req) {
            k = k_per_req[b];
            if (k < 0 || k > K) {
                num_accepted[b] = 0; status[b] = ORC_ST_BAD_K;
                if (rows_read) rows_read[b] = 0;
                continue;
            }
        }
        for (int i = 0; i <= k; ++i) {
            int64_t lrow = l_row_off ? ((int64_t)l_row_off[b] + i) * l_rstride
                                     : (int64_t)b * l_bstride + (int64_t)i * l_rstride;
            load_row(logits, ldt, lrow, V, l);
            nread++;
            n = i;
            if (!row_valid(l, V)) { st |= ORC_ST_BAD_ROW; break; }
            int t = argmax_row(l, V);
            if (i == k) { tok[i] = t; break; }      /* bonus token */
            int y = draft[(int64_t)b * K + i];
            if (y < 0 || y >= V) st |= ORC_ST_BAD_TOKEN;
            tok[i] = t;
            if (y != t) break;                      /* correction token */
        }
        num_accepted[b] = n;
        status[b] = st;
        if (rows_read) rows_read[b] = nread;
    }
    free(l);
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §5 "DDTree": Q(u) = prod_i q_i(u_i), best-first heap      */
/* under a node budget, positions by depth, ancestor-only visibility     */
/* ------------------------------------------------------------------ */

typedef struct { double v; int32_t id; } vid_t;

/* descending value, ascending id */
static int cmp_vid(const void* a, const void* b)
{
    const vid_t* x = (const vid_t*)a;
    const vid_t* y = (const vid_t*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* Candidate list of one depth: the M most probable tokens of q_d, by
 * probability descending, ties to the lower id.  Returns its length, or -1
 * when the row holds a NaN or +Inf. */
static int depth_list(const float* row, int V, int M, vid_t* all, vid_t* out)
{
    for (int x = 0; x < V; ++x) {
        double v = (double)row[x];
        if (isnan(v) || v == INFINITY) return -1;
        all[x].v = v;
        all[x].id = x;
    }
    qsort(all, (size_t)V, sizeof(vid_t), cmp_vid);
    int n = M < V ? M : V;
    for (int i = 0; i < n; ++i) out[i] = all[i];
    return n;
}

#define ORC_MAX_L 64

typedef struct {
    double Q;
    int depth;
    int parent;            /* node id of the parent */
    int rank;              /* rank of the token in its depth's list */
    uint8_t path[ORC_MAX_L];
} orc_cand;

/* order of the best-first pops: higher Q first, then smaller depth, then the
 * lexicographically smaller rank path */
static int cand_before(const orc_cand* a, const orc_cand* b)
{
    if (a->Q != b->Q) return a->Q > b->Q;
    if (a->depth != b->depth) return a->depth < b->depth;
    for (int i = 0; i < a->depth; ++i)
        if (a->path[i] != b->path[i]) return a->path[i] < b->path[i];
    return 0;
}

static void write_masks(const int32_t* par, int count, int N, uint64_t* mask)
{
    int W = (N + 63) / 64;
    memset(mask, 0, (size_t)N * W * sizeof(uint64_t));
    for (int n = 0; n < count; ++n) {
        uint64_t* mn = mask + (int64_t)n * W;
        if (par[n] >= 0) {
            const uint64_t* mp = mask + (int64_t)par[n] * W;
            for (int w = 0; w < W; ++w) mn[w] = mp[w];
        }
        mn[n / 64] |= (uint64_t)1 << (n % 64);
    }
}

void oracle_tree_build(
    const float* q, int64_t q_bstride, int64_t q_rstride,
    int B, int L, int V, int budget,
    int32_t* token, int32_t* parent, int32_t* depth, double* score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status,
    int32_t* rows_needed)
{
    const int N = budget;
    const int M = N - 1;
    const int W = (N + 63) / 64;
    vid_t* all = (vid_t*)malloc((size_t)V * sizeof(vid_t));
    vid_t* lists = (vid_t*)malloc((size_t)(L + 1) * (M > 0 ? M : 1) * sizeof(vid_t));
    int* list_len = (int*)malloc((size_t)(L + 1) * sizeof(int));
    orc_cand* pend = (orc_cand*)malloc((size_t)(2 * N + 2) * sizeof(orc_cand));
    orc_cand* node = (orc_cand*)malloc((size_t)(N + 1) * sizeof(orc_cand));

    for (int b = 0; b < B; ++b) {
        int32_t* tk = token + (int64_t)b * N;
        int32_t* pr = parent + (int64_t)b * N;
        int32_t* dp = depth + (int64_t)b * N;
        double* sc = score + (int64_t)b * N;
        for (int n = 0; n < N; ++n) { tk[n] = -1; pr[n] = -1; dp[n] = -1; sc[n] = 0.0; }
        for (int d = 0; d <= L; ++d) list_len[d] = -2;   /* -2: not read yet */
        int st = 0, need = 0, npend = 0, count = 0;

        /* the root: the empty prefix, Q = 1, depth 0 */
        memset(&node[0], 0, sizeof(orc_cand));
        node[0].Q = 1.0; node[0].depth = 0; node[0].parent = -1; node[0].rank = -1;
        tk[0] = -1; pr[0] = -1; dp[0] = 0; sc[0] = 1.0;
        count = 1;
        int want_child = 0;   /* node whose first child must enter the frontier */

        while (count < N) {
            if (want_child >= 0) {
                int d = node[want_child].depth + 1;
                if (d <= L) {
                    if (list_len[d] == -2) {
                        const float* row = q + (int64_t)b * q_bstride + (int64_t)(d - 1) * q_rstride;
                        list_len[d] = depth_list(row, V, M, all, lists + (int64_t)d * M);
                        if (list_len[d] < 0) { st |= ORC_ST_BAD_ROW; list_len[d] = 0; }
                        if (d > need) need = d;
                    }
                    if (list_len[d] > 0) {
                        orc_cand* c = &pend[npend++];
                        *c = node[want_child];
                        c->depth = d;
                        c->parent = want_child;
                        c->rank = 0;
                        c->path[d - 1] = 0;
                        c->Q = node[want_child].Q * lists[(int64_t)d * M + 0].v;
                    }
                }
                want_child = -1;
            }
            if (npend == 0) break;
            int best = 0;
            for (int j = 1; j < npend; ++j)
                if (cand_before(&pend[j], &pend[best])) best = j;
            orc_cand c = pend[best];
            pend[best] = pend[--npend];

            int n = count++;
            node[n] = c;
            tk[n] = lists[(int64_t)c.depth * M + c.rank].id;
            pr[n] = c.parent;
            dp[n] = c.depth;
            sc[n] = c.Q;
            /* next sibling: same parent, next rank of the same depth list */
            if (c.rank + 1 < list_len[c.depth]) {
                orc_cand* s = &pend[npend++];
                *s = c;
                s->rank = c.rank + 1;
                s->path[c.depth - 1] = (uint8_t)(c.rank + 1);
                s->Q = node[c.parent].Q * lists[(int64_t)c.depth * M + c.rank + 1].v;
            }
            want_child = n;
        }
        num_nodes[b] = count;
        status[b] = st;
        if (rows_needed) rows_needed[b] = need;
        write_masks(pr, count, N, anc_mask + (int64_t)b * N * W);
    }
    free(all); free(lists); free(list_len); free(pend); free(node);
}


/* Rank of token x in row q_d: how many tokens come before it in the order
 * "probability descending, then id ascending".  Counted pairwise, so that the
 * brute force shares no ordering code with the heap's candidate lists. */
static int rank_by_count(const float* row, int V, int x)
{
    int r = 0;
    for (int z = 0; z < V; ++z) {
        if (z == x) continue;
        if (row[z] > row[x] || (row[z] == row[x] && z < x)) r++;
    }
    return r;
}

int oracle_tree_build_bruteforce(
    const float* q, int64_t q_bstride, int64_t q_rstride,
    int B, int L, int V, int budget, int64_t max_prefixes,
    int32_t* token, int32_t* parent, int32_t* depth, double* score,
    uint64_t* anc_mask, int32_t* num_nodes)
{
    const int N = budget;
    const int W = (N + 63) / 64;
    if (L > ORC_MAX_L || V > 255) return -1;
    int* rank = (int*)malloc((size_t)(L + 1) * V * sizeof(int));
    int rc = 0;

    for (int b = 0; b < B && rc == 0; ++b) {
        /* every token of every depth: V + V^2 + ... + V^L prefixes */
        int64_t total = 1, level = 1;
        for (int d = 1; d <= L; ++d) {
            const float* row = q + (int64_t)b * q_bstride + (int64_t)(d - 1) * q_rstride;
            for (int x = 0; x < V; ++x) {
                if (isnan(row[x]) || row[x] == INFINITY) { rc = -1; break; }
                rank[(int64_t)d * V + x] = rank_by_count(row, V, x);
            }
            if (rc) break;
            level *= V;
            total += level;
            if (total > max_prefixes) { rc = -1; break; }
        }
        if (rc) break;
        orc_cand* pre = (orc_cand*)calloc((size_t)total, sizeof(orc_cand));
        int32_t* tok_of = (int32_t*)calloc((size_t)total, sizeof(int32_t));
        int64_t cnt = 0;
        pre[cnt].Q = 1.0; pre[cnt].depth = 0; tok_of[cnt] = -1; cnt++;
        /* each prefix of length d extends one of length d - 1 by any token x;
         * Q multiplies q_d(x), and the tie order uses x's rank in row d */
        int64_t lo = 0, hi = 1;
        for (int d = 1; d <= L; ++d) {
            const float* row = q + (int64_t)b * q_bstride + (int64_t)(d - 1) * q_rstride;
            for (int64_t j = lo; j < hi; ++j) {
                for (int x = 0; x < V; ++x) {
                    orc_cand c = pre[j];
                    c.depth = d;
                    c.rank = rank[(int64_t)d * V + x];
                    c.path[d - 1] = (uint8_t)c.rank;
                    c.Q = pre[j].Q * (double)row[x];
                    tok_of[cnt] = x;
                    pre[cnt++] = c;
                }
            }
            lo = hi; hi = cnt;
        }
        /* sort indices (not the records) so that each keeps its token */
        int64_t* ord = (int64_t*)malloc((size_t)cnt * sizeof(int64_t));
        for (int64_t i = 0; i < cnt; ++i) ord[i] = i;
        /* insertion sort by the pop order: tiny inputs only */
        for (int64_t i = 1; i < cnt; ++i) {
            int64_t v = ord[i], j = i - 1;
            while (j >= 0 && cand_before(&pre[v], &pre[ord[j]])) { ord[j + 1] = ord[j]; --j; }
            ord[j + 1] = v;
        }
        int take = (int)(cnt < N ? cnt : N);
        int32_t* tk = token + (int64_t)b * N;
        int32_t* pr = parent + (int64_t)b * N;
        int32_t* dp = depth + (int64_t)b * N;
        double* sc = score + (int64_t)b * N;
        for (int n = 0; n < N; ++n) { tk[n] = -1; pr[n] = -1; dp[n] = -1; sc[n] = 0.0; }
        for (int n = 0; n < take; ++n) {
            const orc_cand* c = &pre[ord[n]];
            dp[n] = c->depth;
            sc[n] = c->Q;
            tk[n] = tok_of[ord[n]];
            pr[n] = -1;
            if (n > 0) {
                /* parent: the kept prefix one token shorter (must precede n) */
                for (int m = 0; m < n; ++m) {
                    const orc_cand* a = &pre[ord[m]];
                    if (a->depth != c->depth - 1) continue;
                    if (memcmp(a->path, c->path, (size_t)a->depth) == 0) { pr[n] = m; break; }
                }
                if (pr[n] < 0) rc = -2;   /* the kept set is not prefix-closed */
            }
        }
        num_nodes[b] = take;
        write_masks(pr, take, N, anc_mask + (int64_t)b * N * W);
        free(pre); free(tok_of); free(ord);
    }
    free(rank);
    return rc;
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §5 "DDTree": follow the target-selected token down the    */
/* tree; when no child carries it, it becomes the bonus token            */
/* ------------------------------------------------------------------ */

void oracle_verify_tree(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes,
    int B, int N, int V, int max_depth,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted,
    int32_t* status)
{
    double* l = (double*)malloc((size_t)V * sizeof(double));
    for (int b = 0; b < B; ++b) {
        int32_t* pn = path_nodes + (int64_t)b * (max_depth + 1);
        int32_t* ot = out_tokens + (int64_t)b * (max_depth + 1);
        for (int i = 0; i <= max_depth; ++i) { pn[i] = -1; ot[i] = -1; }
        int st = 0, acc = 0, cur = 0;
        int nn = num_nodes[b];
        pn[0] = 0;
        for (;;) {
            load_row(logits, ldt, (int64_t)b * l_bstride + (int64_t)cur * l_rstride, V, l);
            if (!row_valid(l, V)) { st |= ORC_ST_BAD_ROW; break; }
            int t = argmax_row(l, V);
            int child = -1;
            for (int c = 0; c < nn && c < N; ++c)
                if (parent[(int64_t)b * N + c] == cur && token[(int64_t)b * N + c] == t) { child = c; break; }
            ot[acc] = t;
            if (child < 0 || acc >= max_depth) break;
            acc++;
            pn[acc] = child;
            cur = child;
        }
        num_accepted[b] = acc;
        status[b] = st;
    }
    free(l);
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §1 (the chain rule is not a tree sampler: a tree needs a   */
/* sampling rule of its own) and §5 "DDTree" (follow the target-selected  */
/* token): at every walked node the target token is drawn from that      */
/* node's p (temperature and top-k folded in) with the depth's uniform;   */
/* a child carrying it is accepted and the walk continues there,          */
/* otherwise the drawn token is the bonus.  Every committed token is a    */
/* draw from the target, so the committed sequence follows the target.   */
/* ------------------------------------------------------------------ */

void oracle_verify_tree_sample(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes,
    const float* uniforms, int B, int N, int V, int max_depth,
    float temperature, int top_k,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted,
    int32_t* status, int32_t* near_tie)
{
    double* l = (double*)malloc((size_t)V * sizeof(double));
    double* p = (double*)malloc((size_t)V * sizeof(double));
    double* scratch = (double*)malloc((size_t)V * sizeof(double));
    const double T = (double)temperature;
    for (int b = 0; b < B; ++b) {
        int32_t* pn = path_nodes + (int64_t)b * (max_depth + 1);
        int32_t* ot = out_tokens + (int64_t)b * (max_depth + 1);
        const float* u = uniforms + (int64_t)b * (max_depth + 1);
        for (int i = 0; i <= max_depth; ++i) { pn[i] = -1; ot[i] = -1; }
        int st = 0, acc = 0, cur = 0, nt = 0;
        int nn = num_nodes[b];
        pn[0] = 0;
        for (;;) {
            load_row(logits, ldt, (int64_t)b * l_bstride + (int64_t)cur * l_rstride, V, l);
            if (!row_valid(l, V)) { st |= ORC_ST_BAD_ROW; break; }
            form_p(l, V, T, top_k, p, scratch);
            int near = 0;
            int t = sample_icdf(p, V, (double)u[acc], &near, NULL);
            if (near && acc < 31) nt |= 1 << acc;
            int child = -1;
            for (int c = 0; c < nn && c < N; ++c)
                if (parent[(int64_t)b * N + c] == cur && token[(int64_t)b * N + c] == t) { child = c; break; }
            ot[acc] = t;
            if (child < 0 || acc >= max_depth) break;
            acc++;
            pn[acc] = child;
            cur = child;
        }
        num_accepted[b] = acc;
        status[b] = st;
        if (near_tie) near_tie[b] = nt;
    }
    free(l); free(p); free(scratch);
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §5 "DDTree": the KV cache keeps the accepted path only.   */
/* Request b's accepted path is path_nodes[b, 0..n_b] (the root, then    */
/* the accepted nodes by depth); its rows move, in that order, to        */
/* destination rows dst_pos[b] + 0 .. dst_pos[b] + n_b of every plane    */
/* (a layer's keys or values).  Other destination rows are not written.  */
/* ------------------------------------------------------------------ */

void oracle_kv_compact(
    const unsigned char* src, int64_t s_plane, int64_t s_batch, int64_t s_row,
    unsigned char* dst, int64_t d_plane, int64_t d_batch, int64_t d_row,
    int P, int B, int N, int64_t row_bytes,
    const int32_t* path_nodes, int W, const int32_t* num_accepted, const int32_t* dst_pos)
{
    for (int p = 0; p < P; ++p)
        for (int b = 0; b < B; ++b) {
            const int n = num_accepted[b];
            const int base = dst_pos ? dst_pos[b] : 0;
            for (int j = 0; j <= n && j < W; ++j) {
                const int node = path_nodes[(int64_t)b * W + j];
                if (node < 0 || node >= N) continue;
                const unsigned char* from = src + p * s_plane + b * s_batch + node * s_row;
                unsigned char* to = dst + p * d_plane + b * d_batch + (int64_t)(base + j) * d_row;
                for (int64_t x = 0; x < row_bytes; ++x) to[x] = from[x];
            }
        }
}

/* ------------------------------------------------------------------ */
/* [SD-survey] §5 "DSpark": s_j = prod_{i<=j} c_i, expected advance      */
/* 1 + sum_{j<=k} s_j; the verify length maximises advance per cost      */
/* a + b*k (ties to the smaller k)                                        */
/* ------------------------------------------------------------------ */

void oracle_adaptive_len(
    const float* conf, int B, int Kmax, float a, float b, const double* cost,
    int32_t* k_out, double* surv, double* exp_adv,
    int32_t* l_row_off, int32_t* q_row_off, int32_t* near_tie)
{
    const double A = (double)a, Bc = (double)b;
    int32_t lo = 0, qo = 0;
    for (int r = 0; r < B; ++r) {
        double s = 1.0, E = 1.0;
        double best = 1.0 / (cost ? cost[0] : A + Bc * 0.0);
        double second = -INFINITY;
        double best_E = 1.0;
        int best_k = 0;
        for (int j = 1; j <= Kmax; ++j) {
            s = s * (double)conf[(int64_t)r * Kmax + (j - 1)];
            if (surv) surv[(int64_t)r * Kmax + (j - 1)] = s;
            E = E + s;
            /* [SD-survey] §9: with a profiled cost table the cost of verifying
             * j positions is its entry j, otherwise a + b*j */
            double ratio = E / (cost ? cost[j] : A + Bc * (double)j);
            if (ratio > best) { second = best; best = ratio; best_k = j; best_E = E; }
            else if (ratio > second) { second = ratio; }
        }
        k_out[r] = best_k;
        if (exp_adv) exp_adv[r] = best_E;
        if (near_tie) near_tie[r] = (best - second) <= ORC_NEAR_TIE * fabs(best);
        if (l_row_off) l_row_off[r] = lo;
        if (q_row_off) q_row_off[r] = qo;
        lo += best_k + 1;
        qo += best_k;
    }
    if (l_row_off) l_row_off[B] = lo;
    if (q_row_off) q_row_off[B] = qo;
}

/* ---------------------------------------------------------------------------
 * EAGLE-2 dynamic draft tree ([SD-survey] §4 "EAGLE-2")
 * ------------------------------------------------------------------------- */

void oracle_eagle_expand(
    const float* q, int64_t q_bstride, int64_t q_rstride,
    int B, int F, int V, int K2, int Fn, int G,
    int32_t* token, int32_t* parent, int32_t* depth, double* score, int32_t* num_gen,
    const int32_t* front_in, const int32_t* num_front_in,
    int32_t* front_out, int32_t* num_front_out, int32_t* status)
{
    vid_t* all = (vid_t*)malloc((size_t)(V > 0 ? V : 1) * sizeof(vid_t));
    vid_t* kids = (vid_t*)malloc((size_t)(K2 > 0 ? K2 : 1) * sizeof(vid_t));
    char* taken = (char*)malloc((size_t)(G > 0 ? G : 1));
    for (int b = 0; b < B; ++b) {
        int32_t* tk = token + (int64_t)b * G;
        int32_t* pr = parent + (int64_t)b * G;
        int32_t* dp = depth + (int64_t)b * G;
        double* sc = score + (int64_t)b * G;
        int st = 0;
        int g0 = num_gen[b];
        if (g0 < 1 || g0 > G) { st |= ORC_ST_BAD_NODE; g0 = g0 < 1 ? 0 : G; }
        int g = g0;
        int nf = num_front_in[b];
        if (nf < 0) nf = 0;
        if (nf > F) nf = F;
        /* children of every frontier row, in slot order, ranks in order */
        for (int f = 0; f < nf; ++f) {
            const int u = front_in[(int64_t)b * F + f];
            if (u < 0 || u >= g0) { st |= ORC_ST_BAD_NODE; continue; }
            const float* row = q + (int64_t)b * q_bstride + (int64_t)f * q_rstride;
            const int n = depth_list(row, V, K2, all, kids);
            if (n < 0) { st |= ORC_ST_BAD_ROW; continue; }
            for (int r = 0; r < n; ++r) {
                if (g >= G) { st |= ORC_ST_TREE_FULL; break; }
                tk[g] = kids[r].id;
                pr[g] = u;
                dp[g] = dp[u] + 1;
                sc[g] = sc[u] * kids[r].v;
                g++;
            }
        }
        num_gen[b] = g;
        /* the next frontier: repeatedly the best child not yet chosen */
        const int nc = g - g0;
        const int nn = Fn < nc ? Fn : nc;
        memset(taken, 0, (size_t)(G > 0 ? G : 1));
        for (int j = 0; j < Fn; ++j) front_out[(int64_t)b * Fn + j] = -1;
        for (int j = 0; j < nn; ++j) {
            int best = -1;
            for (int c = g0; c < g; ++c) {
                if (taken[c]) continue;
                if (best < 0 || sc[c] > sc[best]) best = c;   /* strict: the earlier wins a tie */
            }
            taken[best] = 1;
            front_out[(int64_t)b * Fn + j] = best;
        }
        num_front_out[b] = nn;
        status[b] = st;
    }
    free(all); free(kids); free(taken);
}

typedef struct { double s; int32_t d; int32_t i; } rerank_t;

/* rerank order: score descending, then depth ascending, then generated first */
static int cmp_rerank(const void* a, const void* b)
{
    const rerank_t* x = (const rerank_t*)a;
    const rerank_t* y = (const rerank_t*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    if (x->d != y->d) return x->d < y->d ? -1 : 1;
    return (x->i > y->i) - (x->i < y->i);
}

void oracle_eagle_rerank(
    const int32_t* token, const int32_t* parent, const int32_t* depth, const double* score,
    const int32_t* num_gen, int B, int G, int budget,
    int32_t* out_token, int32_t* out_parent, int32_t* out_depth, double* out_score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status)
{
    const int N = budget;
    const int W = (N + 63) / 64;
    rerank_t* cand = (rerank_t*)malloc((size_t)(G > 0 ? G : 1) * sizeof(rerank_t));
    int32_t* newid = (int32_t*)malloc((size_t)(G > 0 ? G : 1) * sizeof(int32_t));
    for (int b = 0; b < B; ++b) {
        const int32_t* tk = token + (int64_t)b * G;
        const int32_t* pr = parent + (int64_t)b * G;
        const int32_t* dp = depth + (int64_t)b * G;
        const double* sc = score + (int64_t)b * G;
        int32_t* ot = out_token + (int64_t)b * N;
        int32_t* op = out_parent + (int64_t)b * N;
        int32_t* od = out_depth + (int64_t)b * N;
        double* os = out_score + (int64_t)b * N;
        int st = 0;
        int g = num_gen[b];
        if (g < 1 || g > G) { st |= ORC_ST_BAD_NODE; g = g < 1 ? 1 : G; }
        for (int n = 0; n < N; ++n) { ot[n] = -1; op[n] = -1; od[n] = -1; os[n] = 0.0; }
        for (int i = 0; i < G; ++i) newid[i] = -1;
        /* the root, then the generated nodes in rerank order */
        ot[0] = -1; op[0] = -1; od[0] = 0; os[0] = 1.0;
        newid[0] = 0;
        int count = N > 0 ? 1 : 0;
        int nc = 0;
        for (int i = 1; i < g; ++i) {
            cand[nc].s = sc[i]; cand[nc].d = dp[i]; cand[nc].i = i;
            nc++;
        }
        qsort(cand, (size_t)nc, sizeof(rerank_t), cmp_rerank);
        for (int c = 0; c < nc && count < N; ++c) {
            const int i = cand[c].i;
            const int p = pr[i];
            if (p < 0 || p >= g || newid[p] < 0) { st |= ORC_ST_BAD_NODE; continue; }
            newid[i] = count;
            ot[count] = tk[i];
            op[count] = newid[p];
            od[count] = dp[i];
            os[count] = sc[i];
            count++;
        }
        num_nodes[b] = count;
        status[b] = st;
        write_masks(op, count, N, anc_mask + (int64_t)b * N * W);
    }
    free(cand); free(newid);
}
