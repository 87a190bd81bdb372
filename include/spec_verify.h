/*
 * spec_verify.h -- C ABI of libspecverify.so, the GB300 (sm_103a) library for
 * the verify-and-accept step of speculative decoding.
 *
 * The step runs after the target model's one forward over k drafted tokens
 * (or over a flattened draft tree).  It reads the V-wide logit rows that
 * forward produced, decides how much of the draft to keep, and supplies the
 * one token the target adds at the break point ("accepted + 1").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is CALLER-OWNED DEVICE MEMORY unless stated.  The
 *    library allocates nothing and frees nothing.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream).  Nothing is synchronised inside.
 *  - The return value is a status.  SPEC_OK means the work was enqueued.  A
 *    negative value means the arguments were rejected on the host and NOTHING
 *    was launched (SPEC_ECUDA: a launch failed; spec_last_error() has the CUDA
 *    message).  The library never traps, asserts or exits on the device.
 *  - Problems found on the device in one request's data (a draft token
 *    outside [0, V), a malformed tree, a bad length) are written to that
 *    request's `status[b]` (SPEC_STATUS_*); such a request emits nothing
 *    (n_emit = 0, outputs -1) and the other requests are unaffected.
 *  - Logits: dtype SPEC_DTYPE_F32 or SPEC_DTYPE_BF16.  Each row holds V
 *    contiguous values.  Row i of request b starts at element
 *        b * req_stride + i * row_stride
 *    of its buffer.  Strides are in elements and may be 0 (broadcast).  The
 *    fast path wants every row start 16-byte aligned; other layouts are
 *    served by a scalar path with the same results.  NaN logits are not
 *    supported; -inf is (a masked token).
 *  - Uniforms are fp32 in [0, 1), drawn by the caller.
 *  - Argmax ties resolve to the lowest index.
 *  - Workspace: `workspace` must hold spec_workspace_size(...) bytes and be
 *    256-byte aligned.  It needs no initialisation: every call first writes
 *    whatever it later reads.  A workspace may be reused by any later call
 *    of any shape; calls that may overlap on the GPU (other streams) must
 *    not share one.
 *  - p = softmax(target_logits / T), q = softmax(draft_logits / T), the
 *    target's and the draft's next-token distributions at a position
 *    ("投机解码:为什么一个字都不改", section "一轮能出几个 token", the box
 *    P = softmax(f([x1 ... xk]) / T)).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes (host side) */
#define SPEC_OK 0
#define SPEC_EINVAL (-1)     /* bad pointer, size, stride or scalar argument */
#define SPEC_EDTYPE (-2)     /* dtype is neither SPEC_DTYPE_F32 nor SPEC_DTYPE_BF16 */
#define SPEC_EWORKSPACE (-3) /* workspace missing, misaligned or too small */
#define SPEC_ECUDA (-4)      /* a CUDA call failed; see spec_last_error() */

/* per-request status codes (device side, in status[b]) */
#define SPEC_STATUS_OK 0
#define SPEC_STATUS_TOKEN_RANGE 1 /* a draft/node token is outside [0, V) */
#define SPEC_STATUS_BAD_TREE 2    /* parents[] is not a tree rooted at 0, or too deep */
#define SPEC_STATUS_BAD_LENGTH 3  /* draft_len or hist_len outside its range */

#define SPEC_DTYPE_F32 0
#define SPEC_DTYPE_BF16 1

/* `op` argument of spec_workspace_size */
#define SPEC_OP_NGRAM 0
#define SPEC_OP_GREEDY 1
#define SPEC_OP_SAMPLE 2
#define SPEC_OP_TREE 3
#define SPEC_OP_DRAW 4
#define SPEC_OP_FILTER 5 /* spec_filter_rows: B = rows */

/* Limits checked on the host. */
#define SPEC_MAX_K 64        /* draft length of a chain */
#define SPEC_MAX_WINDOW 64   /* n-gram window */
#define SPEC_MAX_NODES 4096  /* nodes of a draft tree, root included */
#define SPEC_MAX_DEPTH 64    /* depth of a draft tree */

/*
 * spec_ngram_draft -- the history-lookup drafter.
 * ("第 13 篇：推理引擎一次猜几个字", 逐行要点, the 草稿器.猜 line: take the
 * last few tokens of the context as a window, find the identical segment
 * earlier in the history, and propose the tokens that followed it; no
 * parameters, and a miss costs nothing.)
 *
 *   history    int32 [B, hist_stride]; request b holds hist_len[b] tokens.
 *   hist_len   int32 [B], each in [0, hist_stride] (else SPEC_STATUS_BAD_LENGTH).
 *   window     w in [1, SPEC_MAX_WINDOW]: the last w tokens h[n-w .. n).
 *   k          draft length in [0, SPEC_MAX_K].
 *   draft      out int32 [B, k]: h[i+w .. min(i+w+k, n)) for the RIGHTMOST
 *              start i < n - w with h[i .. i+w) == h[n-w .. n); padded -1.
 *   draft_len  out int32 [B]: number of proposed tokens (0 when no match).
 *   status     out int32 [B].
 */
int spec_ngram_draft(const int32_t *history, const int32_t *hist_len, int B, int hist_stride,
                     int window, int k, int32_t *draft, int32_t *draft_len, int32_t *status,
                     void *stream);

/*
 * spec_verify_greedy -- greedy (argmax) prefix verification.
 * ("第 13 篇", section ③ 伪代码 and 逐行要点: compare draft token i with the
 * token the model would choose at that position, stop at the first
 * difference, keep the accepted prefix and append the model's own token at
 * the break point; "Speculative decoding explained", the four-case table.)
 *
 *   target        logits of positions 0..k: request b, position i at
 *                 b*target_req_stride + i*row_stride (k+1 rows of V).
 *   draft         int32 [B, k] drafted tokens.
 *   draft_len     int32 [B] or NULL (= k): positions >= draft_len[b] are
 *                 ignored and the final token comes from row draft_len[b].
 *   max_emit      int32 [B] or NULL (= k+1): cap on emitted tokens, for a
 *                 draft that reaches the end of the sequence (no extra token).
 *   accepted      out int32 [B]: m = length of the accepted prefix.
 *   out_tokens    out int32 [B, k+1]: draft[0..m) then argmax(row m), cut to
 *                 n_emit tokens, padded -1.
 *   n_emit        out int32 [B] = min(m + 1, max_emit[b]).
 *   status        out int32 [B].
 *   workspace     see the conventions; size from spec_workspace_size(
 *                 SPEC_OP_GREEDY, B, k, V, dtype).
 */
int spec_verify_greedy(const void *target, int64_t target_req_stride, int64_t row_stride,
                       int dtype, int B, int k, int V, const int32_t *draft,
                       const int32_t *draft_len, const int32_t *max_emit, int32_t *accepted,
                       int32_t *out_tokens, int32_t *n_emit, int32_t *status, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * spec_verify_sample -- lossless sampling verification of a chain.
 * ("投机解码:为什么一个字都不改", section 改进方案: accept the draft token x
 * for sure when p(x) >= q(x), else with probability p(x)/q(x); on a
 * rejection resample from norm(max(0, p - q)) and drop the rest of the
 * draft; replay section: each round emits accepted + 1 tokens, the last one
 * drawn from p when all k were accepted.)
 *
 *   target          [B, k+1, V] logits (strides as above).
 *   draft_logits    [B, k, V] logits of the draft model, same dtype and
 *                   row_stride, request stride draft_req_stride.
 *   temperature     T > 0, applied to both: p = softmax(t/T), q = softmax(d/T).
 *   draft           int32 [B, k]: x_i, drawn by the drafter from q_i.
 *   draft_len, max_emit   as in spec_verify_greedy.
 *   uniforms        fp32 [B, k+1]: u[b][i] tests position i (accept iff
 *                   u_i * q_i(x_i) < p_i(x_i), i.e. u_i < min(1, p/q));
 *                   u[b][k] drives the final draw: the smallest v whose
 *                   prefix sum of the residual (or, after a full accept, of
 *                   p_L) exceeds u times its total.
 *   accepted, out_tokens, n_emit, status   as in spec_verify_greedy.
 *   p_tok, q_tok    out fp32 [B, k] or NULL: p_i(x_i), q_i(x_i) for every
 *                   i < draft_len (whether or not the test reached it); -1
 *                   beyond draft_len.
 *   resid_mass      out fp32 [B] or NULL: sum max(0, p_m - q_m) = 1 - alpha_m
 *                   at the rejected position, 0 when everything was accepted.
 *   workspace       size from spec_workspace_size(SPEC_OP_SAMPLE, B, k, V, dtype).
 */
int spec_verify_sample(const void *target, int64_t target_req_stride, const void *draft_logits,
                       int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int k,
                       int V, float temperature, const int32_t *draft, const int32_t *draft_len,
                       const int32_t *max_emit, const float *uniforms, int32_t *accepted,
                       int32_t *out_tokens, int32_t *n_emit, float *p_tok, float *q_tok,
                       float *resid_mass, int32_t *status, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * spec_verify_tree -- verification of a draft tree, one target forward over
 * all nodes with tree attention.
 * ("Speculative Decoding II", EAGLE section: the sampling rule is applied
 * recursively at each node of the draft tree, as in SpecInfer, so the output
 * keeps the target's distribution.)
 *
 *   Node 0 is the root (the last committed token); parents int32 [B, N] with
 *   parents[b][0] = -1 and 0 <= parents[b][i] < i; node_tok int32 [B, N] the
 *   drafted token of each node (node_tok[b][0] is not read).  Depth of the
 *   tree <= max_depth <= SPEC_MAX_DEPTH, N <= SPEC_MAX_NODES.
 *   target, draft_logits   [B, N, V]: row u is the target's / the draft's
 *                   next-token logits after node u.  Draft rows of leaves
 *                   are never read; draft_logits may be NULL when T <= 0.
 *   temperature     T > 0: sampling walk.  At node u, p = softmax(t_u/T),
 *                   q = softmax(d_u/T); children are tested in increasing id
 *                   order, child c accepted iff u[b][c] * q(x_c) < p(x_c);
 *                   after a rejected child p <- norm(max(0, p - q)) (q kept);
 *                   an accepted child is descended into; when no child is
 *                   accepted, or u is a leaf, the final token is drawn from
 *                   the current p with u[b][N].
 *                   T <= 0: greedy walk, descend into the first child (id
 *                   order) whose token is argmax(t_u); else emit argmax(t_u).
 *   uniforms        fp32 [B, N+1].
 *   accepted_len    out int32 [B]: number of tree nodes accepted.
 *   path_nodes      out int32 [B, max_depth+1]: node ids from the root, pad -1.
 *   out_tokens      out int32 [B, max_depth+1]: emitted tokens, pad -1.
 *   n_emit          out int32 [B] = accepted_len + 1 (0 on a bad request).
 *   status          out int32 [B].
 *   workspace       size from spec_workspace_size(SPEC_OP_TREE, B, N, V, dtype)
 *                   (may be 0; then workspace may be NULL).
 */
int spec_verify_tree(const void *target, int64_t target_req_stride, const void *draft_logits,
                     int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int N,
                     int V, float temperature, const int32_t *parents, const int32_t *node_tok,
                     const float *uniforms, int max_depth, int32_t *accepted_len,
                     int32_t *path_nodes, int32_t *out_tokens, int32_t *n_emit,
                     int32_t *status, void *workspace, size_t workspace_bytes, void *stream);

/* Flags of spec_verify_tree_ex. */
#define SPEC_TREE_SIBLINGS_WITHOUT_REPLACEMENT 1

/*
 * spec_verify_tree_ex -- spec_verify_tree with flags (bitwise OR; 0 gives
 * spec_verify_tree exactly; an unknown bit is SPEC_EINVAL).
 *
 *   SPEC_TREE_SIBLINGS_WITHOUT_REPLACEMENT: the drafter drew the children of
 *   a node from q one after another WITHOUT replacement, each from q with the
 *   earlier children's tokens removed and q renormalised.  Then after a
 *   rejected child x, besides p <- norm(max(0, p - q)), q <- q with x zeroed,
 *   renormalised (a rejected child's q(x) = 0 from then on, and a child whose
 *   q(x) = 0 is accepted iff p(x) > 0).  With this reading the walk keeps the
 *   target's distribution for such drafts, where the default rule assumes
 *   the children were drawn independently from q ("Speculative Decoding II",
 *   EAGLE section, the tree verified as in SpecInfer; the without-replacement
 *   variant is a reading of that rule for drafts drawn so).  Ignored when
 *   T <= 0.
 */
int spec_verify_tree_ex(const void *target, int64_t target_req_stride, const void *draft_logits,
                        int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int N,
                        int V, float temperature, const int32_t *parents, const int32_t *node_tok,
                        const float *uniforms, int max_depth, int flags, int32_t *accepted_len,
                        int32_t *path_nodes, int32_t *out_tokens, int32_t *n_emit,
                        int32_t *status, void *workspace, size_t workspace_bytes, void *stream);

/* Size of the scratch array behind spec_verify_sample_noalloc (4 MiB). */
#define SPEC_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/*
 * spec_verify_sample_noalloc -- spec_verify_sample for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry
 * point; it exists for the library's users.
 *
 * Some callers cannot supply a workspace: a serving loop that divides its
 * whole device-memory budget up at start-up and forbids allocations while it
 * serves, or code that must not stall on a cudaMalloc (which can synchronise
 * the device).  This entry point takes the same arguments as
 * spec_verify_sample minus the workspace, and uses instead a fixed scratch
 * array of SPEC_NOALLOC_SCRATCH_BYTES compiled into the library.  It calls no
 * allocator.
 *
 *  - Every GPU on which the library is loaded holds that array in device
 *    memory until the process exits.
 *  - The first call on a device looks up the array's device address on the
 *    current device (cudaGetSymbolAddress) and caches it; make that first
 *    call before any stream capture.  `stream` must belong to the current
 *    device.
 *  - A problem whose scratch (spec_workspace_size(SPEC_OP_SAMPLE, B, k, V,
 *    dtype)) exceeds the array is refused with SPEC_EWORKSPACE and a message
 *    in spec_last_error(); use spec_verify_sample then.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it has to start at zero (each call's first kernel clears
 *    what it counts with), but calls that may overlap on the GPU (different
 *    streams, or different host threads without ordering) race on it.
 */
int spec_verify_sample_noalloc(const void *target, int64_t target_req_stride,
                               const void *draft_logits, int64_t draft_req_stride,
                               int64_t row_stride, int dtype, int B, int k, int V,
                               float temperature, const int32_t *draft, const int32_t *draft_len,
                               const int32_t *max_emit, const float *uniforms, int32_t *accepted,
                               int32_t *out_tokens, int32_t *n_emit, float *p_tok, float *q_tok,
                               float *resid_mass, int32_t *status, void *stream);

/*
 * spec_sample -- draw one token from each row's softmax: the drafter's side
 * of speculative sampling, x ~ q.  ("投机解码:为什么一个字都不改", 改进方案:
 * the draft model proposes x by sampling its own distribution
 * q = softmax(draft logits / T), and verification later needs q(x); the
 * draw is the one the verify step uses for its final token.)
 *
 *   logits       request b's row starts at element b*req_stride (V logits,
 *                contiguous); dtype SPEC_DTYPE_F32 or SPEC_DTYPE_BF16.
 *   temperature  T > 0 (finite).
 *   uniforms     fp32 [B] in [0, 1).
 *   tokens       out int32 [B]: the smallest v whose inclusive prefix sum of
 *                softmax(row / T) exceeds u_b (if rounding leaves none, the
 *                last v with positive probability).
 *   probs        out fp32 [B] or NULL: the probability of tokens[b].
 *   status       out int32 [B] or NULL.
 *   workspace    size from spec_workspace_size(SPEC_OP_DRAW, B, 0, V, dtype);
 *                needs no initialisation.
 */
int spec_sample(const void *logits, int64_t req_stride, int dtype, int B, int V, float temperature,
                const float *uniforms, int32_t *tokens, float *probs, int32_t *status, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * Top-k / top-p filtered sampling.  The pages leave temperature, top-k and
 * top-p to another lesson ("投机解码:为什么一个字都不改", the section that sets
 * them aside); verification stays lossless against the FILTERED target when
 * the target's and the draft's distributions are filtered alike and the
 * drafter drew from the filtered q.  The filter of one row, in this order:
 *   p = softmax(x / T);
 *   top_k (0 < top_k < V): keep every v whose logit is >= the top_k-th
 *     largest logit (repeats counted; ties at the cut are all kept);
 *   top_p (top_p < 1): over the kept logits in descending order, with p
 *     renormalised to them, keep the smallest prefix whose mass reaches
 *     top_p, and every logit equal to its last one;
 *   p' = p renormalised over the kept logits, 0 elsewhere.
 * top_k = 0 (or >= V) and top_p = 1 switch a filter off; top_k < 0, or
 * top_p outside (0, 1], is SPEC_EINVAL.  A kept set is always {v : x_v >=
 * theta} for one threshold theta, the smallest kept logit.  Rows of more
 * than 16 x 96 KB of logits (V > 786,432 bf16 or 393,216 fp32) are
 * SPEC_EINVAL.  The top-p cut adds masses in 2^-44 fixed point, so it is
 * the same on every run; against exact arithmetic it can differ only where
 * the mass at the cut is within about 1e-7 of top_p.
 *
 * spec_verify_sample_topkp -- spec_verify_sample with p and q filtered: the
 *   acceptance test, p_tok / q_tok, the residual and the bonus draw all use
 *   p' and q'.  A drafted token that q' excludes has q'(x) = 0 and is
 *   accepted iff p'(x) > 0.  Same arguments and workspace
 *   (SPEC_OP_SAMPLE) as spec_verify_sample, plus top_k and top_p.  With
 *   both filters off it is spec_verify_sample.
 * spec_sample_topkp -- spec_sample from the filtered rows (the drafter's
 *   draw from q'); probs gets q'(x).  Workspace as spec_sample.
 * spec_filter_rows -- the filter alone, for R rows of V logits (row r at
 *   r * row_stride): theta fp32 [R] (the smallest kept logit; with both
 *   filters off, the smallest logit) and kept int32 [R] or NULL (the kept
 *   count).  workspace: spec_workspace_size(SPEC_OP_FILTER, R, 0, V, dtype)
 *   bytes.
 */
int spec_verify_sample_topkp(const void *target, int64_t target_req_stride, const void *draft_logits,
                             int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int k, int V,
                             float temperature, int top_k, float top_p, const int32_t *draft,
                             const int32_t *draft_len, const int32_t *max_emit, const float *uniforms,
                             int32_t *accepted, int32_t *out_tokens, int32_t *n_emit, float *p_tok, float *q_tok,
                             float *resid_mass, int32_t *status, void *workspace, size_t workspace_bytes,
                             void *stream);
int spec_sample_topkp(const void *logits, int64_t req_stride, int dtype, int B, int V, float temperature,
                      int top_k, float top_p, const float *uniforms, int32_t *tokens, float *probs,
                      int32_t *status, void *workspace, size_t workspace_bytes, void *stream);
int spec_filter_rows(const void *logits, int64_t row_stride, int dtype, int R, int V, float temperature, int top_k,
                     float top_p, float *theta, int32_t *kept, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * spec_tree_rerank -- EAGLE-2 post-processing of candidate draft trees.
 * ("Speculative Decoding II", section "Context-Aware Dynamic Draft Tree"
 * and its worked example: a node's value is the product of the draft
 * model's confidences along its path from the root; the m most valuable
 * nodes are kept, equal values going to the shallower node, which keeps the
 * kept nodes a tree rooted at the root; they are flattened for the target's
 * forward, each node attending only to itself and its ancestors.)
 *
 *   parents      int32 [B, N]: parents[0] = -1, 0 <= parents[i] < i.
 *   conf         fp32 [B, N]: c_i in [0, 1], the draft model's probability
 *                of node i's token given its parent (conf[b][0] is not read;
 *                the root's value is 1).
 *   node_tok     int32 [B, N], or NULL when sel_tok is NULL.
 *   N            in [1, SPEC_MAX_NODES]; m in [1, SPEC_MAX_NODES]: nodes to
 *                keep (all N when m >= N).
 *   max_depth    in [0, SPEC_MAX_DEPTH]: a deeper tree is malformed.
 *   sel_nodes    out int32 [B, m]: the kept nodes' ids, flattened (by depth,
 *                then id).
 *   sel_parents  out int32 [B, m]: each kept node's parent as an index into
 *                the flattened order, -1 for the root.
 *   sel_depth    out int32 [B, m]: depths (the relative positions).
 *   sel_value    out fp32 [B, m] or NULL: values, computed from the root down
 *                in fp32 (V(i) = V(parent) * c_i).
 *   sel_tok      out int32 [B, m] or NULL: node_tok in the flattened order.
 *   mask         out uint8 [B, m, m] or NULL: mask[b][i][j] = 1 iff
 *                flattened node j is node i or one of its ancestors.
 *   n_sel        out int32 [B]: min(m, N), or 0 for a malformed tree.
 *   status       out int32 [B] or NULL: SPEC_STATUS_BAD_TREE for a malformed
 *                parent array, a depth beyond max_depth, or a confidence
 *                outside [0, 1] (NaN included).
 * Entries from n_sel on are -1 (values -1.0, mask rows and columns 0).
 * Ties in value go to the shallower node, then to the lower id.  sel_parents
 * and sel_tok describe a tree that spec_verify_tree accepts (node 0 the
 * root, every parent before its child).  No workspace.
 */
int spec_tree_rerank(const int32_t *parents, const float *conf, const int32_t *node_tok, int B, int N,
                     int m, int max_depth, int32_t *sel_nodes, int32_t *sel_parents, int32_t *sel_depth,
                     float *sel_value, int32_t *sel_tok, uint8_t *mask, int32_t *n_sel, int32_t *status,
                     void *stream);

/*
 * spec_workspace_size -- bytes of workspace a call needs.
 *   op = SPEC_OP_*; rows_per_req = k for chains, N for trees.
 *   Returns 0 for invalid arguments and for ops that need none.
 */
size_t spec_workspace_size(int op, int B, int rows_per_req, int V, int dtype);

/* Static text for a SPEC_* return code or a SPEC_STATUS_* value (pass
 * status codes as 100 + status). */
const char *spec_status_string(int code);

/* Message of the last CUDA failure seen by this thread ("" if none). */
const char *spec_last_error(void);

/*
 * Tracing.  With tracing on, every kernel the library launches is bracketed
 * by a pair of CUDA events recorded on the launching stream.
 * spec_trace_collect() waits for the recorded events, adds each launch's
 * elapsed time to its kernel's total, writes up to `cap` entries (kernel
 * name, total milliseconds, launch count) and clears the record.  It
 * returns the number of distinct kernels, or a negative SPEC_* code.
 * Tracing is process-wide.  Calls made while their stream is being captured
 * into a CUDA graph put the events into the graph as event-record nodes:
 * each replay of the graph stamps them again, so collect after the replay
 * to be timed (the record keeps one pair per captured launch, whatever the
 * number of replays).  Dependent launches are not chained while tracing is
 * on, so each bracket holds one kernel.
 * spec_trace_repeat(reps), reps in [1, 1024] (default 1, else SPEC_EINVAL):
 * while tracing, each kernel is launched reps times back to back inside its
 * event pair, so the bracket divided by reps approaches the kernel's own
 * duration (one launch's set-up no longer in it).  Every kernel of the
 * library gives the same outputs when launched again on its own inputs, so
 * the results do not change; the launch count grows by the repeats.
 */
int spec_trace_enable(int on);
int spec_trace_repeat(int reps);
int spec_trace_collect(const char **names, double *total_ms, int64_t *launches, int cap);

/* Number of kernels this process has launched through the library. */
int64_t spec_launch_count(void);

/*
 * Chain verification paths.  spec_verify_greedy and spec_verify_sample give
 * the same results on either path; the paths differ in speed:
 *   SPEC_CHAIN_TWO_PASS  a streaming pass over every row on all SMs, then the
 *                        cluster accept kernel: one thread-block cluster
 *                        per request forms the final draw (the chunked one
 *                        below when the clusters cannot all be resident);
 *   SPEC_CHAIN_CHUNKED   the streaming pass, then the chunked accept kernel:
 *                        CTAs over chunks of every request's draw row, the
 *                        last of a request's CTAs to finish draws;
 *   SPEC_CHAIN_FUSED     one thread-block cluster per request does the whole
 *                        call in one launch and uses no workspace (suits
 *                        small problems: latency-bound); when the requests'
 *                        clusters cannot all be resident at once the call
 *                        runs on the two-pass path instead;
 *   SPEC_CHAIN_AUTO      the library picks per call (the default).
 * spec_set_chain_path sets the path for calls made after it, process-wide;
 * it returns SPEC_OK, or SPEC_EINVAL for an unknown value.  The workspace
 * requirements of the entry points do not change with the path.  This
 * switch has no counterpart in the method; it exists for tuning and so that
 * every path can be tested on any shape.
 */
#define SPEC_CHAIN_AUTO 0
#define SPEC_CHAIN_TWO_PASS 1
#define SPEC_CHAIN_FUSED 2
#define SPEC_CHAIN_CHUNKED 3
int spec_set_chain_path(int path);

/*
 * Host analysis helpers, for choosing the draft length k from measured
 * acceptance ("投机解码:为什么一个字都不改", the bookkeeping section: with
 * every position accepted independently with probability alpha a round
 * yields (1 - alpha^(k+1)) / (1 - alpha) tokens; its experiments weigh the
 * draft's cost c against k, and it points to Leviathan et al., appendix A.1
 * and theorem 3.8, for the best k under that cost).  These run on the host:
 * their pointers are HOST memory, they launch nothing and return SPEC_OK or
 * SPEC_EINVAL (alpha outside [0, 1], k < 0, c < 0 or not finite, a null
 * output).
 *
 *   spec_expected_tokens  *out = 1 + alpha + ... + alpha^k, the expected
 *                         tokens per round (k + 1 at alpha = 1).
 *   spec_speedup          *out = expected tokens / (k c + 1): a round costs
 *                         k draft forwards of c target forwards each plus
 *                         one target forward (the verify step's own time is
 *                         not counted).
 *   spec_best_k           the k in [0, k_max] with the largest speedup
 *                         (k = 0: plain decoding, speedup 1; ties keep the
 *                         smaller k), and that speedup (speedup_out may be
 *                         NULL).
 *   spec_alpha_estimate   alpha from n observed rounds: accepted[r] (the m a
 *                         verify call returned) and draft_len[r] (NULL: all
 *                         k).  A round tested m + 1 positions when m < L and
 *                         m when m = L, m of them accepted; the estimate is
 *                         sum(m) / sum(tested), NaN when nothing was tested.
 *                         *tests_out (may be NULL) = sum(tested).
 *                         SPEC_EINVAL also when some m > L or L < 0.
 */
int spec_expected_tokens(double alpha, int k, double *out);
int spec_speedup(double alpha, int k, double draft_cost, double *out);
int spec_best_k(double alpha, double draft_cost, int k_max, int *k_out, double *speedup_out);
int spec_alpha_estimate(const int32_t *accepted, const int32_t *draft_len, int n, int k, double *alpha_out,
                        int64_t *tests_out);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
