/*
 * spec_verify.h -- C ABI of libspecverify, batched verification of
 * speculative-decoding drafts on one NVIDIA GB300 (sm_103a).
 *
 * Source page for every operation below:
 *   [SD-survey] "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
 *               (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash,
 *               DDTree and DSpark), chzhyang.github.io.
 *
 * Conventions for every call
 *   - Array pointers are owned by the caller and point to device memory or
 *     to PINNED host memory (page-locked: cudaHostAlloc, cudaMallocHost or
 *     cudaHostRegister).  Pinned host arrays are read and written in place
 *     through their mapping into the device's address space -- on a Grace
 *     host over the NVLink-C2C link -- so a call on host-resident inputs
 *     moves only the bytes it reads (rows past a rejection never cross the
 *     link).  Pageable host memory cannot be reached by the kernels and is
 *     refused with SPEC_INVALID_ARG before anything is enqueued.
 *   - The library never allocates device memory; scratch space comes from
 *     the caller's `ws` buffer (device memory), sized by the matching
 *     *_workspace_size() query.  The workspace must not be shared by two
 *     calls in flight at once.
 *     One exception: spec_verify_greedy_static takes no `ws` and uses a
 *     fixed array the library reserves in device memory (described there).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work and return without synchronising; they are
 *     free of host-device synchronisation and of allocation.
 *   - The return value reports only synchronous problems: argument checks
 *     (SPEC_INVALID_ARG), unsupported shapes (SPEC_UNSUPPORTED) and launch
 *     errors (SPEC_CUDA_ERROR).  spec_last_error() returns a thread-local
 *     description of the last non-OK status.
 *   - Problems found on the device are reported per request in `status`
 *     (bits SPEC_ST_*), and device-wide ones (a bounded wait that gave up)
 *     in the workspace error word, read with spec_workspace_error().
 *   - Row strides are in elements.  Rows whose start address is 16-byte
 *     aligned are streamed by the Tensor Memory Accelerator; other layouts
 *     are accepted and read with plain loads (slower).
 *   - Token ids are int32 in [0, V).  Output token rows are padded with -1.
 *   - Shape limits (SPEC_UNSUPPORTED beyond them): K <= 4096 draft
 *     positions; N <= 8192 tree nodes; tree build L <= 16, budget <= 256.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_INVALID_ARG = 1,
    SPEC_UNSUPPORTED = 2,
    SPEC_CUDA_ERROR = 3
} spec_status;

typedef enum {
    SPEC_F32 = 0,   /* IEEE binary32 */
    SPEC_BF16 = 1   /* bfloat16 */
} spec_dtype;

/* per-request status bits */
#define SPEC_ST_BAD_ROW   1   /* a read logits row held NaN/+Inf or only -Inf: the walk
                                 stopped there, no correction/bonus token */
#define SPEC_ST_Q_ZERO    2   /* q(y) == 0 for a drafted token: ratio taken as +inf
                                 when p(y) > 0, else 0 */
#define SPEC_ST_R_ZERO    4   /* residual mass <= 0 after a rejection: the correction
                                 token was sampled from p instead */
#define SPEC_ST_BAD_TOKEN 8   /* a drafted or tree token id outside [0, V) */
#define SPEC_ST_BAD_K    16   /* per-request draft length outside [0, K] */
#define SPEC_ST_TREE_FULL 32  /* EAGLE-2: the node arrays' capacity G was reached */
#define SPEC_ST_BAD_NODE  64  /* EAGLE-2: a frontier or parent id (or num_gen) out of range */

/* workspace error bits */
#define SPEC_WS_ERR_WAIT     1u   /* a bounded device wait gave up; outputs invalid */
#define SPEC_WS_ERR_QUEUE    2u   /* the device task queue overflowed; outputs invalid */

const char* spec_last_error(void);
int spec_version(void);

/*
 * Optional tuning, for benchmarking sweeps.  The kernels run on thread-block
 * clusters: every CTA of a cluster takes one slice of every vocabulary row
 * the cluster reads.  slices_per_row: CTAs per cluster, 1..16 (0 =
 * automatic: a power of two up to 8, each slice at least 2048 elements).
 * slots_per_cta: requests each CTA's cluster keeps in flight per CTA, 1..4
 * (0 = automatic, 2).  Affects later calls of this process.
 */
spec_status spec_set_tuning(int slices_per_row, int slots_per_cta);

/*
 * Reads the device error word of a workspace after the stream is drained
 * (synchronises `stream`).  For diagnostics and tests; not for hot loops.
 */
spec_status spec_workspace_error(const void* ws, void* stream, uint32_t* err_out);

/* ------------------------------------------------------------------------
 * spec_verify_chain -- batched chain speculative sampling
 * [SD-survey] §1 "what speculative decoding guarantees": acceptance
 * alpha_i(y_i) = min(1, p_i(y_i)/q_i(y_i)); at the first rejection the
 * correction token is drawn from the normalised residual [p_i - q_i]_+;
 * if every draft passes, a bonus token is drawn from p_{K+1}.  Temperature
 * and top-k truncation are folded into p (same section).
 *
 *   logits   target logits, dtype `ldt`.  Dense layout (no row offsets):
 *            row (b, i), i = 0..K, starts at b*l_batch_stride + i*l_row_stride.
 *            Packed layout: row (b, i), i = 0..k_b, starts at
 *            (l_row_off[b] + i) * l_row_stride; l_batch_stride is ignored.
 *   q        draft proposal probabilities, fp32, used as given (not
 *            truncated or renormalised).  Row (b, i), i = 0..k-1, addressed
 *            like logits with q_batch_stride / q_row_stride / q_row_off.
 *   draft    [B, K] int32 drafted tokens (ragged: the first k_b of each row).
 *   uniforms [B, K+1] fp32 in [0, 1): u[b, i] decides position i (accept iff
 *            u < p/q), u[b, k] drives the single inverse-CDF sample (ascending
 *            token id, smallest x with C(x) > u * total).
 *   temperature > 0.  top_k <= 0 or >= V disables truncation; otherwise
 *            S = {x : l_x >= tau}, tau = top_k-th largest raw logit, ties kept.
 *   k_per_req, l_row_off, q_row_off  Ragged verify ([SD-survey] §9): NULL,
 *            NULL, NULL = "static" (every request verifies all K rows);
 *            k_per_req [B] with row offsets [B+1], [B+1] = "compact" (packed
 *            rows, request b verifies k_b positions); k_per_req alone =
 *            "cap-accept" (the dense rows of the full window, request b
 *            verifies and commits only its first k_b positions).
 * Outputs:
 *   out_tokens   [B, K+1]: accepted drafts, then the correction or bonus token, then -1.
 *   num_accepted [B]: accepted draft tokens (excludes the correction/bonus token).
 *   status       [B]: SPEC_ST_* bits.
 *   diag         NULL or [B, K+1, 4] fp32: for each examined draft row
 *                {p(y), q(y), Z, R} (R = residual mass at the rejection row,
 *                else 0); for the bonus row {p(x), 0, Z, 0}.  Z is
 *                sum over S of exp((l_x - max l)/T).  Rows not examined are
 *                left untouched.
 * Rows past the first rejection are never read.
 * ---------------------------------------------------------------------- */
size_t spec_verify_chain_workspace_size(int B, int K, int V, int top_k);
spec_status spec_verify_chain(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    const int32_t* draft, const float* uniforms,
    int B, int K, int V, float temperature, int top_k,
    const int32_t* k_per_req, const int32_t* l_row_off, const int32_t* q_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status, float* diag,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spec_verify_greedy -- greedy argmax-match verification
 * [SD-survey] §1, "greedy-consistent" results: accept while the drafted
 * token equals the target argmax (raw logits, lowest id on ties); the first
 * mismatch commits the argmax; if all K match, the bonus is the argmax of
 * row K.  Layout of logits, draft, k_per_req, l_row_off and the outputs as in
 * spec_verify_chain; no q, no uniforms.
 * ---------------------------------------------------------------------- */
size_t spec_verify_greedy_workspace_size(int B, int K, int V);
spec_status spec_verify_greedy(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* draft, int B, int K, int V,
    const int32_t* k_per_req, const int32_t* l_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spec_verify_greedy_static -- spec_verify_greedy without a caller workspace
 * No counterpart on the source pages: this is a library convenience.
 *
 * For callers that cannot allocate device memory when they verify (code in
 * host callbacks or allocator-free runtimes, plugins handed raw buffers by an
 * engine that owns every allocation, loops that forbid allocation after
 * start-up).  Same arguments and results as spec_verify_greedy, minus `ws`
 * and `ws_bytes`: the scratch space is a 64 KiB array in device memory that
 * the library reserves on every GPU it is loaded on, until the process exits.
 * Batches whose spec_verify_greedy_workspace_size() exceeds 64 KiB are
 * rejected with SPEC_INVALID_ARG (greedy verification needs a fixed 256 bytes
 * whatever the batch, so every shape within the other limits fits).  Nothing
 * is allocated.
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  The address is kept per device together with the context
 * it belongs to; a call that finds another context current (after a device
 * reset) looks it up again, so make the first call after a reset outside
 * capture too.  Every call on a device shares the array: calls whose GPU
 * work overlaps (different streams or host threads) race and must be
 * serialised by the caller.
 * ---------------------------------------------------------------------- */
spec_status spec_verify_greedy_static(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* draft, int B, int K, int V,
    const int32_t* k_per_req, const int32_t* l_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * spec_tree_build -- DDTree best-first draft tree
 * [SD-survey] §5 "DDTree": prefixes u scored by the factorised proxy
 * Q(u) = prod_{i=1}^{|u|} q_i(u_i) over the block drafter's per-position
 * marginals; a best-first heap picks prefixes under a node budget; nodes take
 * position id = depth and see only themselves and their ancestors.
 *
 *   q        [B, L, V] fp32 marginals: row (b, d-1) at b*q_batch_stride +
 *            (d-1)*q_row_stride is depth d's distribution.  Depth d uses its
 *            budget-1 most probable tokens (ties to the lower id).
 *   budget   N nodes including the root (node 0, depth 0, Q = 1, token -1),
 *            1 <= N <= 256; L <= 16.
 * Outputs ([B, N], node order = pop order, so parents precede children;
 * slots >= num_nodes[b] hold -1 / 0):
 *   token, parent (-1 for the root), depth (position id), score (Q, fp64),
 *   anc_mask [B, N, ceil(N/64)] uint64: bit m of node n set iff m is n or an
 *   ancestor of n; num_nodes [B]; status [B].
 * Pop order: higher Q, then smaller depth, then lexicographically smaller
 * path of per-depth ranks.  Depth rows are read in order and reading stops as
 * soon as the best-first order no longer needs a deeper row.
 * ---------------------------------------------------------------------- */
size_t spec_tree_build_workspace_size(int B, int L, int V, int budget);
spec_status spec_tree_build(
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    int B, int L, int V, int budget,
    int32_t* token, int32_t* parent, int32_t* depth, double* score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spec_eagle_expand -- one expansion step of an EAGLE-2 dynamic draft tree
 * [SD-survey] §4 "EAGLE-2": candidates grow along the branches of highest
 * cumulative path confidence; the tree's depth and width follow the context.
 *
 * Node arrays of capacity G per request (caller-owned, in/out):
 *   token, parent, depth [B, G] int32; score [B, G] fp64 = the product of
 *   the draft probabilities along the node's path; num_gen [B] = nodes so
 *   far.  Node 0 is the root (token -1, parent -1, depth 0, score 1,
 *   num_gen 1) -- the caller initialises it.
 *   q        [B, F, V] fp32: row (b, f) at b*q_batch_stride + f*q_row_stride
 *            is the draft's conditional distribution after the path of node
 *            front_in[b, f], f < num_front_in[b] (other rows are not read).
 *   K2       children per expanded node: its row's K2 most probable tokens
 *            (probability descending, lower id first), 1 <= K2 <= 255.
 *   Fn       next frontier width, 0 <= Fn <= 64; F <= 64; F * K2 <= 2048;
 *            G <= 8192.
 * The children are appended in (slot, rank) order with depth = parent's + 1
 * and score = parent's score * q; when G is reached the rest are dropped
 * (SPEC_ST_TREE_FULL).  front_out [B, Fn] receives the Fn appended children
 * of highest score (ties: appended first), padded with -1; num_front_out [B]
 * their count.  A row holding NaN/+Inf adds no children (SPEC_ST_BAD_ROW);
 * a frontier id outside [0, num_gen) is skipped (SPEC_ST_BAD_NODE).
 * status [B] is written, not accumulated.  front_in and front_out must not
 * overlap; ws as sized below, 16-byte aligned.
 * ---------------------------------------------------------------------- */
size_t spec_eagle_expand_workspace_size(int B, int F, int K2);
spec_status spec_eagle_expand(
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    int B, int F, int V, int K2, int Fn, int G,
    int32_t* token, int32_t* parent, int32_t* depth, double* score, int32_t* num_gen,
    const int32_t* front_in, const int32_t* num_front_in,
    int32_t* front_out, int32_t* num_front_out, int32_t* status,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spec_eagle_rerank -- the EAGLE-2 verification tree
 * [SD-survey] §4 "EAGLE-2": every generated candidate is reranked and the
 * best form the tree the target verifies.
 *
 * The tree is the root and the budget-1 generated nodes of highest score
 * (ties: smaller depth, then lower index), emitted in that order -- a
 * parent always precedes its children -- with parents renumbered.  Outputs
 * exactly as spec_tree_build (token, parent, depth, score, anc_mask
 * [B, budget, ceil(budget/64)], num_nodes, status), so the tree feeds
 * spec_verify_tree, spec_verify_tree_sample and spec_kv_compact.
 * 1 <= budget <= 1024, G <= 8192.  A generated node whose parent is out of
 * range or not emitted before it is skipped (SPEC_ST_BAD_NODE).
 * ---------------------------------------------------------------------- */
spec_status spec_eagle_rerank(
    const int32_t* token, const int32_t* parent, const int32_t* depth, const double* score,
    const int32_t* num_gen, int B, int G, int budget,
    int32_t* out_token, int32_t* out_parent, int32_t* out_depth, double* out_score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * spec_verify_tree -- greedy tree-walk verification
 * [SD-survey] §5 "DDTree": verification walks the target-selected token;
 * when no child of the current node carries it, that token becomes the
 * bonus token; only the accepted path is kept.
 *
 *   logits   [B, N, V]: row (b, n) at b*l_batch_stride + n*l_row_stride is
 *            the target's distribution after node n.
 *   token, parent, num_nodes   the tree (as produced by spec_tree_build).
 *   max_depth  the tree's depth limit L (output width L+1).
 * Outputs: path_nodes [B, L+1] (root 0, then accepted nodes, then -1),
 *   out_tokens [B, L+1] (accepted tokens, then the bonus, then -1),
 *   num_accepted [B], status [B].  Only rows on the walked path are read.
 * ---------------------------------------------------------------------- */
size_t spec_verify_tree_workspace_size(int B, int N, int V);
spec_status spec_verify_tree(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes,
    int B, int N, int V, int max_depth,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spec_verify_tree_sample -- stochastic tree-walk verification
 * [SD-survey] §1: the chain acceptance rule is not a sampler for a tree of
 * drafts, a tree needs its own rule; §5 "DDTree": verification follows the
 * target-selected token, and a token no child carries becomes the bonus.
 * At depth d the current node's target token is drawn from its p
 * (temperature and top-k folded in exactly as in spec_verify_chain: ascending
 * token id, the smallest x with C(x) > u[b, d] * total); a child carrying it
 * is accepted and the walk continues there, otherwise the drawn token is the
 * bonus.  Every committed token is a draw from the target, so the committed
 * sequence follows the target distribution.
 *
 *   logits   [B, N, V] target rows of the tree's nodes (as spec_verify_tree).
 *   token, parent, num_nodes   the tree (as produced by spec_tree_build).
 *   uniforms [B, max_depth+1] fp32 in [0, 1): u[b, d] draws at depth d.
 * Outputs as spec_verify_tree: path_nodes [B, L+1], out_tokens [B, L+1],
 *   num_accepted [B], status [B].  Only rows on the walked path are read.
 * ---------------------------------------------------------------------- */
size_t spec_verify_tree_sample_workspace_size(int B, int N, int V);
spec_status spec_verify_tree_sample(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes, const float* uniforms,
    int B, int N, int V, int max_depth, float temperature, int top_k,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spec_kv_compact -- keep the accepted path's KV rows
 * [SD-survey] §5 "DDTree": after the tree walk only the accepted path's KV
 * is kept.  The tree's forward pass wrote one KV row per tree node; for
 * every plane p (a layer's keys or values) and request b, the rows of the
 * root and the accepted nodes, path_nodes[b, 0..num_accepted[b]], move in
 * that order to destination rows dst_pos[b] + 0 .. dst_pos[b] +
 * num_accepted[b] (dst_pos NULL: rows 0 ..).  No other destination row is
 * written.  A gather bound by HBM bandwidth.
 *
 *   src      row (p, b, n) at src + p*src_plane_stride +
 *            b*src_batch_stride + n*src_row_stride (strides in BYTES), n < N.
 *   dst      row (p, b, m) at dst + p*dst_plane_stride +
 *            b*dst_batch_stride + m*dst_row_stride (bytes).  The rows written
 *            must not overlap the rows read (copy from the tree's own buffer
 *            into the cache, not within one buffer).
 *   row_bytes  bytes of one row (a 16-byte-aligned layout moves 16 bytes a
 *            load; others 4 or 1).
 *   path_nodes [B, path_width], num_accepted [B] (spec_verify_tree or
 *            spec_verify_tree_sample outputs); node ids outside [0, N) are
 *            skipped.  dst_pos NULL or [B] int32.
 * ---------------------------------------------------------------------- */
spec_status spec_kv_compact(
    const void* src, int64_t src_plane_stride, int64_t src_batch_stride, int64_t src_row_stride,
    void* dst, int64_t dst_plane_stride, int64_t dst_batch_stride, int64_t dst_row_stride,
    int P, int B, int N, int64_t row_bytes,
    const int32_t* path_nodes, int path_width, const int32_t* num_accepted, const int32_t* dst_pos,
    void* stream);

/* ------------------------------------------------------------------------
 * spec_adaptive_len -- DSpark verify length
 * [SD-survey] §5 "DSpark": prefix survival s_j = prod_{i<=j} c_i, expected
 * advance 1 + sum_{j<=k} s_j; each request verifies the k in [0, Kmax] that
 * maximises (1 + sum_{j<=k} s_j) / (a + b*k), ties to the smaller k.
 * Computed in fp64 without fused multiply-add.
 *
 *   conf   [B, Kmax] fp32 conditional confidences c_i.   a > 0, b >= 0.
 * Outputs: k_out [B]; surv NULL or [B, Kmax] fp64; exp_adv NULL or [B] fp64
 *   (the advance at the chosen k); l_row_off [B+1] = exclusive scan of
 *   k_b + 1; q_row_off [B+1] = exclusive scan of k_b (the ragged layout of
 *   spec_verify_chain, SGLang's "compact" mode, [SD-survey] §9).
 * ---------------------------------------------------------------------- */
spec_status spec_adaptive_len(
    const float* conf, int B, int Kmax, float a, float b,
    int32_t* k_out, double* surv, double* exp_adv,
    int32_t* l_row_off, int32_t* q_row_off, void* stream);

/* ------------------------------------------------------------------------
 * spec_adaptive_len_table -- DSpark verify length with a profiled cost table
 * [SD-survey] §9 (DSpark in SGLang): the cost of verifying k positions comes
 * from a table profiled for the deployment rather than a formula.  As
 * spec_adaptive_len with the cost a + b*k replaced by cost[k]:
 *   cost   [Kmax+1] fp64, every entry finite and > 0 (the
 *          caller's responsibility: the kernel divides by it).
 * Outputs as spec_adaptive_len.
 * ---------------------------------------------------------------------- */
spec_status spec_adaptive_len_table(
    const float* conf, int B, int Kmax, const double* cost,
    int32_t* k_out, double* surv, double* exp_adv,
    int32_t* l_row_off, int32_t* q_row_off, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
