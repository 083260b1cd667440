/*
 * spec_oracle.h -- float64 CPU oracle for batched speculative-sampling
 * verification.  TEST INFRASTRUCTURE: only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may call it.  It shares no code, header, table
 * or helper with the CUDA library.
 *
 * Source pages (cited by name below):
 *   [SD-survey]  "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
 *                (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash,
 *                DDTree and DSpark), chzhyang.github.io.
 *
 * Conventions shared by every function here:
 *   - logits rows are fp32 (ldt = 0) or bf16 given as raw uint16 bits (ldt = 1);
 *     every value is converted exactly to double before any arithmetic.
 *   - dense addressing: row (b, i) starts at b*batch_stride + i*row_stride
 *     elements; ragged addressing (k_per_req != NULL): row (b, i) starts at
 *     (row_off[b] + i) * row_stride.
 *   - "row invalid": the row holds a NaN or +Inf, or every entry is -Inf.
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status bits written per request */
#define ORC_ST_BAD_ROW      1   /* a read row was invalid: walk stopped          */
#define ORC_ST_Q_ZERO       2   /* q(y) == 0 for a drafted token                  */
#define ORC_ST_R_ZERO       4   /* residual mass <= 0: sampled from p instead     */
#define ORC_ST_BAD_TOKEN    8   /* drafted token id outside [0, V)                */
#define ORC_ST_BAD_K       16   /* per-request draft length outside [0, K]        */

#define ORC_ST_TREE_FULL   32   /* EAGLE-2: the node arrays' capacity was reached */
#define ORC_ST_BAD_NODE    64   /* EAGLE-2: a frontier or parent id out of range   */

/* near-tie window (absolute on the ratio, relative to the mass on the CDF) */
#define ORC_NEAR_TIE 1e-6

/* Chain speculative sampling ([SD-survey] §1).  With k_per_req and no row
 * offsets the rows keep the dense layout and request b verifies only its
 * first k_b positions ([SD-survey] §9 "cap-accept": the full window is
 * computed, the commit is capped).  near_tie[b]: bit i set when
 * |u_i - p_i(y_i)/q_i(y_i)| <= 1e-6 at an examined position i (i < 31);
 * bit 31 set when the final sample's target lies within 1e-6 (normalised) of
 * either boundary of the chosen token's CDF interval.  rows_read[b] = number
 * of logits rows examined.  diag[b, i, 0..3] = p_i(y_i), q_i(y_i), Z_i, R_i
 * for examined draft rows; for the bonus row p_k(x*), 0, Z_k, 0. */
void oracle_verify_chain(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const float* q, int64_t q_bstride, int64_t q_rstride,
    const int32_t* draft, const float* uniforms,
    int B, int K, int V, float temperature, int top_k,
    const int32_t* k_per_req, const int32_t* l_row_off, const int32_t* q_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    double* diag, int32_t* near_tie, int32_t* rows_read);

/* Greedy argmax-match verification ([SD-survey] §1, greedy consistency). */
void oracle_verify_greedy(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const int32_t* draft, int B, int K, int V,
    const int32_t* k_per_req, const int32_t* l_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    int32_t* rows_read);

/* DDTree best-first tree ([SD-survey] §5 "DDTree", Q(u) equation).
 * q: [B, L, V] probabilities, row (b, d-1) is the marginal of depth d.
 * budget N includes the root.  anc_mask has W = ceil(N/64) words per node.
 * rows_needed[b] = deepest per-depth list the best-first order consulted. */
void oracle_tree_build(
    const float* q, int64_t q_bstride, int64_t q_rstride,
    int B, int L, int V, int budget,
    int32_t* token, int32_t* parent, int32_t* depth, double* score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status,
    int32_t* rows_needed);

/* Brute force for tiny V (<= 255) and L: every prefix of length <= L over
 * ALL V tokens of every depth (no candidate list, no sort of the rows: each
 * token's rank is counted pairwise), sorted by (Q desc, depth asc, rank path
 * asc), first N kept.  Same outputs as oracle_tree_build.  Returns -1 when
 * the prefix count exceeds max_prefixes. */
int oracle_tree_build_bruteforce(
    const float* q, int64_t q_bstride, int64_t q_rstride,
    int B, int L, int V, int budget, int64_t max_prefixes,
    int32_t* token, int32_t* parent, int32_t* depth, double* score,
    uint64_t* anc_mask, int32_t* num_nodes);

/* Tree-walk verification ([SD-survey] §5 "DDTree", verification walk). */
void oracle_verify_tree(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes,
    int B, int N, int V, int max_depth,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted,
    int32_t* status);

/* Stochastic tree-walk verification ([SD-survey] §1, a tree needs its own
 * sampling rule; §5 "DDTree", follow the target-selected token).  At depth d
 * the current node's target token is the inverse-CDF draw from its p
 * (temperature, top-k, ties kept) with uniforms[b, d]; a child carrying it is
 * accepted, otherwise it is the bonus token.  uniforms [B, max_depth+1].
 * near_tie[b] bit d: the draw at depth d lay within 1e-6 (normalised) of a
 * CDF boundary. */
void oracle_verify_tree_sample(
    const void* logits, int ldt, int64_t l_bstride, int64_t l_rstride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes,
    const float* uniforms, int B, int N, int V, int max_depth,
    float temperature, int top_k,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted,
    int32_t* status, int32_t* near_tie);

/* Accepted-path KV compaction ([SD-survey] §5 "DDTree": only the accepted
 * path's KV is kept).  For every plane p and request b, destination row
 * dst_pos[b] + j (dst_pos NULL: j) receives source row path_nodes[b, j],
 * j = 0..num_accepted[b] (node ids outside [0, N) are skipped).  Strides in
 * bytes; W = path width (max depth + 1). */
void oracle_kv_compact(
    const unsigned char* src, int64_t s_plane, int64_t s_batch, int64_t s_row,
    unsigned char* dst, int64_t d_plane, int64_t d_batch, int64_t d_row,
    int P, int B, int N, int64_t row_bytes,
    const int32_t* path_nodes, int W, const int32_t* num_accepted, const int32_t* dst_pos);

/* DSpark prefix survival and adaptive verify length ([SD-survey] §5
 * "DSpark", s_j equation and expected advance).  The cost of verifying k
 * positions is a + b*k, or cost[k] when a table (Kmax+1 entries, [SD-survey]
 * §9's profiled per-deployment table) is given.  near_tie[b] = 1 when the
 * best and second-best E(k)/cost(k) differ by <= 1e-6 relative. */
void oracle_adaptive_len(
    const float* conf, int B, int Kmax, float a, float b, const double* cost,
    int32_t* k_out, double* surv, double* exp_adv,
    int32_t* l_row_off, int32_t* q_row_off, int32_t* near_tie);

/* EAGLE-2 dynamic draft tree, one expansion step ([SD-survey] §4
 * "EAGLE-2": the branches of highest cumulative path confidence are
 * expanded; depth and width follow the context).  Per request b the
 * generated nodes so far are node arrays of capacity G (token, parent,
 * depth, score = product of the draft probabilities along the path; node 0
 * is the root: token -1, parent -1, depth 0, score 1), num_gen[b] of them.
 * front_in[b, 0..num_front_in[b]) are node ids whose conditional draft rows
 * q[b, f, 0..V) are given.  For each frontier slot f in order, the K2 most
 * probable tokens of its row (probability descending, lower id first)
 * become children, appended in (f, rank) order with score = score(parent) *
 * q(token).  The next frontier is the Fn children of this step with the
 * highest score (ties: appended earlier first), in that order, into
 * front_out[b, 0..Fn), padded with -1; num_front_out[b] of them. */
void oracle_eagle_expand(
    const float* q, int64_t q_bstride, int64_t q_rstride,
    int B, int F, int V, int K2, int Fn, int G,
    int32_t* token, int32_t* parent, int32_t* depth, double* score, int32_t* num_gen,
    const int32_t* front_in, const int32_t* num_front_in,
    int32_t* front_out, int32_t* num_front_out, int32_t* status);

/* EAGLE-2 rerank ([SD-survey] §4 "EAGLE-2": every candidate is reranked and
 * the best form the verification tree).  The tree is the root and the
 * budget - 1 generated nodes of highest score (ties: smaller depth, then
 * generated earlier), emitted in that order -- a parent always precedes its
 * children -- with parent ids renumbered.  Outputs as oracle_tree_build. */
void oracle_eagle_rerank(
    const int32_t* token, const int32_t* parent, const int32_t* depth, const double* score,
    const int32_t* num_gen, int B, int G, int budget,
    int32_t* out_token, int32_t* out_parent, int32_t* out_depth, double* out_score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status);

#ifdef __cplusplus
}
#endif
#endif
