/*
 * treeverify.h -- C ABI of libtreeverify: verification of a whole draft tree
 * through a gated linear-recurrence layer, greedy acceptance, and commit of the
 * accepted path's state, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (Bole summary page, "Core techniques" §1):
 *   the layer's recurrence h_{t+1} = S_t h_t + u_t, specialised to
 *   S_i = diag(exp g_i) and u_i = k_i v_i^T, with read-out o_i = H_i^T q_i.
 *   On a draft tree every node continues its parent's state:
 *     H_i = diag(exp g_i) H_parent(i) + k_i v_i^T,    H_parent = H0 at the context.
 *   The library never forms H_i.  It evaluates the tree closed form
 *     o_i = H0^T (e^{G_i} * q_i) + sum_{j in anc*(i)} (sum_c q_ic k_jc e^{G_ic - G_jc}) v_j
 *   with anc*(i) the root path of node i including i and G_i = sum_{j in anc*(i)} g_j,
 *   so all nodes are verified in parallel and only the per-token factors
 *   (g_i, k_i, v_i) are kept (§2, "token-level factor encoding").
 *
 * Conventions shared by every call
 *   - All array pointers are DEVICE memory owned by the caller.  The library
 *     allocates nothing, keeps no state between calls and is thread-safe.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream) and returns after the launch.
 *   - Array pointers must be 16-byte aligned (TV_ERR_ALIGN otherwise).
 *   - Host-checkable errors are returned synchronously and launch nothing.
 *   - Errors only the device can see (a malformed tree, offsets or path) are
 *     written into *dev_status (int32, device memory, zeroed by the caller) with
 *     an atomic compare-and-swap, so the first error wins; the kernels never
 *     trap.  The affected request's outputs are then defined per call below.
 *   - Packed ragged layout: the B requests' trees are concatenated, T nodes in
 *     all; node_offsets[b] .. node_offsets[b+1]-1 are request b's nodes.  Per
 *     node t and head h, rows are contiguous:
 *       q, k  [T][H][dk]   (bf16 or fp32, per tv_problem.qkv_dtype)
 *       v     [T][H][dv]
 *       g     [T][H]       (scalar decay)  or  [T][H][dk]  (per-channel decay), fp32,
 *                          natural-log decay: the state is scaled by exp(g) (g <= 0
 *                          gives a contraction; any finite g is accepted)
 *       out   [T][H][dv]   fp32
 *       H0, H_new [B][H][dk][dv] fp32 (row = key channel, dv contiguous)
 *     Several layers of one request fold into H (they share the request's tree).
 */
#ifndef TREEVERIFY_H
#define TREEVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TV_VERSION 1

/* Limits of the library. */
#define TV_MAX_NODES 256  /* nodes per request tree */
#define TV_MAX_DEPTH 32   /* depth of any node (1 = child of the context) */
#define TV_MAX_DIM   256  /* dk and dv */

typedef enum tv_status {
    TV_OK = 0,
    TV_ERR_NULL = 1,        /* a required pointer is NULL */
    TV_ERR_SHAPE = 2,       /* B, H, dk, dv, T, max_nodes or max_depth out of range */
    TV_ERR_DTYPE = 3,       /* unknown decay kind or element type */
    TV_ERR_ALIGN = 4,       /* an array pointer is not 16-byte aligned */
    TV_ERR_UNSUPPORTED = 5, /* a limit of the library is exceeded, or a forced variant
                               cannot run this shape */
    TV_ERR_TREE = 6,        /* device-detected: bad node_offsets, parent, depth or path */
    TV_ERR_CUDA = 7,        /* a CUDA runtime call failed (launch error) */
    TV_ERR_TIMEOUT = 8      /* device-detected: a bounded wait inside a kernel expired */
} tv_status;

typedef enum tv_decay {
    TV_DECAY_SCALAR = 0,    /* g[T][H]: one decay per node and head */
    TV_DECAY_DIAG = 1       /* g[T][H][dk]: one decay per node, head and key channel */
} tv_decay;

typedef enum tv_dtype {
    TV_BF16 = 0,            /* q, k, v are bfloat16 */
    TV_F32 = 1              /* q, k, v are float32 */
} tv_dtype;

/* Kernel choice for tv_verify_ex (tv_verify uses TV_VARIANT_AUTO). */
typedef enum tv_variant {
    TV_VARIANT_AUTO = 0,    /* tensor-core kernel where it applies, else SIMT */
    TV_VARIANT_SIMT = 1,    /* CUDA-core kernel, every supported shape */
    TV_VARIANT_TC = 2,      /* tcgen05 tensor-core kernel, one (request, head) per CTA:
                               bf16 q/k/v, dk in {64,128}, dv in {64,128};
                               TV_ERR_UNSUPPORTED otherwise */
    TV_VARIANT_TC_FUSED = 3, /* tcgen05 kernels with the decay folded into the factors,
                               one kernel for a unit's whole path, bf16 q/k/v: scalar
                               decay with dk and dv in {64,128} and max_nodes <= 32 (the
                               context term, the pair scores and the tree term all on
                               tensor cores); per-channel decay with dk in {64,128} and
                               dv = 128: max_nodes <= 64 with all three on tensor cores,
                               or max_nodes <= 256 and max_depth <= 16 with the context
                               term on tensor cores and the pair weights and tree term
                               by fp32 walks up the root paths (the pair decays summed
                               along the walk).  The 64-node kernel's factors are e^{G} q
                               and e^{-G} k where every path sum |G| <= 69; a unit
                               outside that range takes its pair weights from a walk
                               with the decays as running products.
                               TV_ERR_UNSUPPORTED otherwise.  What TV_VARIANT_AUTO picks
                               where it applies */
    TV_VARIANT_TC_TILED = 4  /* tcgen05 kernels for large trees, one (request, head) per
                               CTA: bf16 q/k/v, dk = dv = 128, trees up to TV_MAX_NODES.
                               Where a request's k, decay and v rows fit shared memory
                               (depth up to 21 at 256 nodes) they are loaded once and
                               both terms run on the tensor cores; deeper trees walk
                               their ancestors through the caches in node tiles of 64;
                               TV_ERR_UNSUPPORTED otherwise */
} tv_variant;

/*
 * Test hook, OR-ed into tv_verify_ex's `variant` together with TV_VARIANT_TC_FUSED
 * (TV_ERR_UNSUPPORTED with any other variant): the kernel treats its first wait for
 * an input copy (a state chunk, or the large-tree kernel's first group of rows) as
 * expired, so the call takes the library's timeout path -- it
 * writes TV_ERR_TIMEOUT to dev_status, waits for its copies and products in flight,
 * frees its tensor memory and returns.  The outputs are then undefined.  For tests
 * of that failure path; never needed otherwise.
 */
#define TV_VARIANT_TEST_EXPIRE_WAIT 0x100

/*
 * Shape and tree of one batch.  The three tree arrays are device memory.
 *   B            number of requests (>= 0)
 *   H            heads per request, layers folded in (>= 1)
 *   dk, dv       key and value widths: multiples of 8 in [8, 256]
 *   total_nodes  T = node_offsets[B] (host copy, used for bounds)
 *   max_nodes    bound on any request's node count, 1..256
 *   max_depth    bound on any node's depth, 1..32; also the row length of `path`
 *   decay        tv_decay
 *   qkv_dtype    tv_dtype
 *   node_offsets [B+1] int32, non-decreasing, node_offsets[0] = 0, node_offsets[B] = T
 *   parent       [T] int32, local index within the request: -1 (child of the
 *                committed context) or an earlier node of the same request
 *   depth        [T] int32: 1 for a child of the context, else depth(parent)+1;
 *                redundant with parent and validated, never trusted
 */
typedef struct tv_problem {
    int32_t B, H, dk, dv;
    int32_t total_nodes;
    int32_t max_nodes;
    int32_t max_depth;
    int32_t decay;
    int32_t qkv_dtype;
    const int32_t *node_offsets;
    const int32_t *parent;
    const int32_t *depth;
} tv_problem;

/*
 * tv_verify -- outputs of every draft node through the recurrence layer.
 * Bole summary page, "Core techniques" §1 (tree closed form, all nodes in
 * parallel) and §2 (per-token factors instead of per-node states).
 *
 *   H0    [B][H][dk][dv] fp32   state of the committed context (read only)
 *   q, k  [T][H][dk]            bf16 or fp32
 *   v     [T][H][dv]            bf16 or fp32
 *   g     [T][H] or [T][H][dk]  fp32 log-decay
 *   out   [T][H][dv] fp32       o_i = H_i^T q_i for every node i and head
 *   dev_status  int32 (device)  see conventions
 * Device-detected errors: a request whose offsets, parent or depth entries are
 * malformed gets status TV_ERR_TREE and its out rows are written as zeros
 * (rows of requests whose offsets themselves are unusable are left untouched).
 * Transient memory: shared memory only; nothing is allocated.
 */
tv_status tv_verify(const tv_problem *p, const float *H0, const void *q, const void *k,
                    const void *v, const float *g, float *out, int32_t *dev_status,
                    void *stream);

/*
 * tv_verify_serial -- the same outputs as tv_verify, computed the naive way that
 * the tree closed form replaces (Bole summary page, "Core techniques" §1-§2 and
 * the serial baseline it is compared with): inside each (request, head) the nodes
 * are processed one after another, S_i = diag(exp g_i) S_parent(i) + k_i v_i^T is
 * formed and stored for every node, and o_i = S_i^T q_i.  A measurement baseline
 * (speed-up of the closed form over serial verification) and a second evaluator
 * of the same function; not the fast path.
 *
 *   p, H0, q, k, v, g, out, dev_status   as in tv_verify
 *   workspace        device memory of at least tv_verify_serial_workspace_bytes(p)
 *                    bytes, 16-byte aligned, owned by the caller; it receives the
 *                    per-node states [B*H][max_nodes][dk][dv] fp32 (contents are
 *                    scratch for the caller)
 *   workspace_bytes  its size
 * Host errors as tv_verify, plus TV_ERR_NULL for a NULL workspace and TV_ERR_SHAPE
 * for one that is too small.  Device-detected errors as tv_verify.
 */
size_t tv_verify_serial_workspace_bytes(const tv_problem *p);
tv_status tv_verify_serial(const tv_problem *p, const float *H0, const void *q, const void *k,
                           const void *v, const float *g, float *out, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * tv_accept_stochastic -- stochastic acceptance of every request's draft tree.
 * LLM Primer VI ch. 9 §9.1: a draft token x drawn from the draft distribution q
 * is accepted with probability min(1, p(x)/q(x)), p the target's distribution;
 * after a rejection the emitted token comes from the normalized residual
 * (p - q)_+, so the output follows the target's distribution.  On a tree: the
 * children of the current node are tried in index order against the current
 * residual (each rejection replaces p by (p - q)_+ / sum, unchanged if that sum is
 * 0); the first accepted child becomes the current node, with its own p and q;
 * when none is accepted the bonus token is drawn from the current residual: the
 * first index whose running sum exceeds u_bonus * (sum of the row).
 *
 *   vocab              V >= 1
 *   root_p, root_q     [B][V] fp32: target / draft probabilities at the context
 *   node_p, node_q     [T][V] fp32: target / draft probabilities after each node
 *                      (q of a node is the distribution its children were drawn from)
 *   u_accept           [T] fp64 uniforms in [0,1): child c is accepted when
 *                      u_accept[c] * q(x_c) < p(x_c) (p the current residual)
 *   u_bonus            [B] fp64 uniforms in [0,1) for the bonus draw
 *   other arguments as in tv_accept_greedy (draft tokens must lie in [0, V))
 * Arithmetic that decides a token is fp64.  Device-detected errors (bad offsets or
 * parents, a draft token outside the vocabulary, a path longer than max_depth):
 * TV_ERR_TREE with accept_len 0, path -1, bonus -1 for that request.
 */
tv_status tv_accept_stochastic(int32_t B, int32_t total_nodes, int32_t max_nodes,
                               int32_t max_depth, int32_t vocab, const int32_t *node_offsets,
                               const int32_t *parent, const int32_t *draft_tokens,
                               const float *root_p, const float *node_p, const float *root_q,
                               const float *node_q, const double *u_accept,
                               const double *u_bonus, int32_t *accept_len, int32_t *path,
                               int32_t *bonus, int32_t *dev_status, void *stream);

/*
 * tv_build_tree -- draft trees by best-first expansion of path scores.
 * BASTION page, Method §1-§3: for every position k the drafter gives a
 * distribution q_k over C candidates; a node at depth d holding candidates
 * x_1..x_d has path score rho = prod_k q_k(x_k).  Starting from the C children of
 * the context, the frontier node with the largest rho joins the tree next, and its
 * C children join the frontier (in candidate order) unless it is at depth_cap;
 * among equal scores the node that joined the frontier first wins.  With a cost
 * table the growth stops before the node that would lower sum(rho) / cost[N].
 * Node index = order of addition: parents precede children, ready for tv_verify.
 *
 *   B            requests (>= 0)
 *   C            candidates per position, 1..32
 *   depth_cap    deepest allowed node, 1..32
 *   n            node budget per request, 1..256
 *   marginals    [B][depth_cap][C] fp64, finite and >= 0 (q_k of request b at row k-1)
 *   cost         [n+1] fp64 > 0, cost[N] = the step cost with N nodes (index 0
 *                unused); NULL for a fixed budget of n nodes
 *   parent, token [B][n] int32 out: local parent (-1 = child of the context) and
 *                candidate of each node; slots past count[b] hold -1
 *   rho          [B][n] fp64 out: path scores (0 past count[b])
 *   count        [B] int32 out: nodes built (fewer than n when the frontier empties
 *                or the cost stop applies)
 * One warp per request; the choices are made on fp64 products, so equal inputs give
 * equal trees on every run.
 */
tv_status tv_build_tree(int32_t B, int32_t C, int32_t depth_cap, int32_t n,
                        const double *marginals, const double *cost, int32_t *parent,
                        int32_t *token, double *rho, int32_t *count, void *stream);

/* Size of the scratch array built into the library for tv_verify_serial_static. */
#define TV_SERIAL_STATIC_BYTES (16u << 20)

/*
 * tv_verify_serial_static -- tv_verify_serial for callers that cannot allocate
 * device memory.  The pages have no counterpart; this entry point exists for the
 * library's users.  A process whose allocator has already reserved the device
 * memory for its own pool, or a loop with a fixed memory budget where an
 * allocation could fail or stall, cannot hand tv_verify_serial a workspace.  This
 * call needs none: the per-node states go to a scratch array of
 * TV_SERIAL_STATIC_BYTES (16 MiB) compiled into the library, which every GPU that
 * loads the library holds until the process exits.
 *
 *   arguments, results and errors as tv_verify_serial, without the workspace
 *   Problems whose states need more than TV_SERIAL_STATIC_BYTES
 *   (tv_verify_serial_workspace_bytes(p)) are rejected with TV_ERR_UNSUPPORTED
 *   before anything is launched.
 * Set-up: every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress).  The array's 16 MiB are taken when the CUDA runtime
 * loads the library's serial-verification code on a device: with lazy module
 * loading (the CUDA default) that is the first call of tv_verify_serial or
 * tv_verify_serial_static on that device.  So make that first call before the
 * process reserves the rest of the device memory for its own pool (else it can
 * fail with TV_ERR_CUDA, out of memory) and before any stream capture; later calls
 * take no device memory.  Every call on a device shares the one array, and it
 * keeps the last call's contents; the kernel writes every state before it reads
 * it, so nothing has to be cleared between calls.  Calls that overlap on the same
 * GPU (for instance on two streams) race on the array and give wrong results:
 * serialize them.  No device memory is allocated or freed by the call itself.
 */
tv_status tv_verify_serial_static(const tv_problem *p, const float *H0, const void *q,
                                  const void *k, const void *v, const float *g, float *out,
                                  int32_t *dev_status, void *stream);

/*
 * tv_workspace_bytes -- device workspace tv_verify needs for problem p: always 0.
 * Every kernel behind tv_verify keeps its transient data (root paths, decay
 * sums, weights, operand tiles, accumulators) in shared and tensor memory, so
 * there is no workspace argument.  Kept so that callers written against a
 * workspace-sizing interface can ask and get the answer.  Returns 0 also for an
 * invalid problem (tv_verify reports that one).
 */
size_t tv_workspace_bytes(const tv_problem *p);

/* tv_verify with an explicit kernel choice (tv_variant). */
tv_status tv_verify_ex(const tv_problem *p, const float *H0, const void *q, const void *k,
                       const void *v, const float *g, float *out, int32_t *dev_status,
                       void *stream, int32_t variant);

/*
 * tv_accept_greedy -- greedy acceptance walk of every request's tree.
 * LLM Primer VI ch. 9 §9.1: the longest draft prefix that matches the target is
 * accepted, and at the first mismatch the target's own token is kept.  On a tree:
 * start at the context with t = root_argmax[b]; repeatedly move to the
 * lowest-index child whose draft token equals t and set t = target_argmax of
 * that child; stop when no child matches.  bonus[b] = t.
 *
 *   node_offsets [B+1], parent [T]       as in tv_problem (total_nodes = T)
 *   draft_tokens [T]   token each node proposes
 *   target_argmax[T]   the target model's argmax after each node
 *   root_argmax  [B]   the target model's argmax at the committed context
 *   accept_len   [B]   out: accepted node count L (0..max_depth)
 *   path         [B][max_depth]  out: accepted local node indices, root first,
 *                      -1 after the first L entries
 *   bonus        [B]   out: the target's token after the accepted prefix
 * Device-detected errors (bad offsets, a parent outside [-1, i), or an accepted
 * path longer than max_depth): TV_ERR_TREE, accept_len = 0, path = -1, bonus = -1
 * for that request.  Integer-only; results are exact.
 */
tv_status tv_accept_greedy(int32_t B, int32_t total_nodes, int32_t max_nodes, int32_t max_depth,
                           const int32_t *node_offsets, const int32_t *parent,
                           const int32_t *draft_tokens, const int32_t *target_argmax,
                           const int32_t *root_argmax, int32_t *accept_len, int32_t *path,
                           int32_t *bonus, int32_t *dev_status, void *stream);

/*
 * tv_accept_greedy_logits -- tv_accept_greedy with the target's choices taken
 * from its logits: the target argmax at the committed context and after every
 * draft node (LLM Primer VI ch. 9 §9.1: the target model's own most likely
 * token decides).  Two kernels on `stream`: the argmax of every row, then the walk.
 *
 *   vocab        V >= 1, the row length of the logits
 *   root_logits  [B][V] bf16   the target's logits at the committed context
 *   node_logits  [T][V] bf16   the target's logits after each draft node
 *   root_argmax  [B] out: argmax of each root row
 *   target_argmax [T] out: argmax of each node row (the walk reads both)
 *   other arguments as in tv_accept_greedy (the walk uses the computed argmaxes)
 * Argmax: the first index of the largest value; a NaN counts as larger than any
 * number, -0 equals +0.  Rows are read with 16-byte loads when V is a multiple
 * of 8 (logit pointers must be 16-byte aligned in any case).  Device-detected
 * errors and outputs of a malformed request as in tv_accept_greedy.  Results are
 * exact.
 */
tv_status tv_accept_greedy_logits(int32_t B, int32_t total_nodes, int32_t max_nodes,
                                  int32_t max_depth, int32_t vocab, const int32_t *node_offsets,
                                  const int32_t *parent, const int32_t *draft_tokens,
                                  const void *root_logits, const void *node_logits,
                                  int32_t *root_argmax, int32_t *target_argmax,
                                  int32_t *accept_len, int32_t *path, int32_t *bonus,
                                  int32_t *dev_status, void *stream);

/*
 * tv_commit -- state after the accepted path, rebuilt from the factors.
 * Bole summary page, "Core techniques" §2: only the accepted path's state is
 * restored, h_k = Chain(S_k..S_1) h_0 + accumulated updates; here
 *   H_new = diag(e^{G_L}) H0 + sum_{m=1..L} diag(e^{G_L - G_{p_m}}) k_{p_m} v_{p_m}^T
 * with p_1..p_L = path[b][0..L), L = accept_len[b] and G the running sum of g
 * along the path.  L = 0 gives H_new = H0.
 *
 *   p          shape and tree (tv_problem; node_offsets and parent are read)
 *   H0         [B][H][dk][dv] fp32
 *   g, k, v    as in tv_verify
 *   path, accept_len   as written by tv_accept_greedy (path rows of max_depth)
 *   H_new      [B][H][dk][dv] fp32; may equal H0 (in place), must not overlap it
 *              otherwise
 * Device-detected errors (L outside [0, max_depth], a path entry outside the
 * request, or a path that is not a root path of the tree): TV_ERR_TREE and that
 * request's H_new is left untouched.
 */
tv_status tv_commit(const tv_problem *p, const float *H0, const float *g, const void *k,
                    const void *v, const int32_t *path, const int32_t *accept_len,
                    float *H_new, int32_t *dev_status, void *stream);

/*
 * tv_accept_commit -- tv_accept_greedy and tv_commit in one launch.
 * Same results as tv_accept_greedy followed by tv_commit with the path it found:
 * every commit block re-runs its request's greedy walk (LLM Primer VI ch. 9
 * §9.1) on shared memory and restores the accepted path's state from the
 * factors (Bole summary page, "Core techniques" §2), so the state update does
 * not wait for a separate acceptance launch.
 *
 *   p, H0, g, k, v, H_new          as in tv_commit (H_new may equal H0)
 *   draft_tokens, target_argmax, root_argmax, accept_len, path, bonus
 *                                  as in tv_accept_greedy
 * Device-detected errors (bad offsets, a parent outside [-1, i), a walk longer
 * than max_depth): TV_ERR_TREE; that request gets accept_len = 0, path = -1,
 * bonus = -1 and its H_new is left untouched.
 */
tv_status tv_accept_commit(const tv_problem *p, const float *H0, const float *g, const void *k,
                           const void *v, const int32_t *draft_tokens,
                           const int32_t *target_argmax, const int32_t *root_argmax,
                           int32_t *accept_len, int32_t *path, int32_t *bonus, float *H_new,
                           int32_t *dev_status, void *stream);

/*
 * tv_pending -- a commit that has not been applied yet: the accepted paths of
 * the previous step and that step's tree and factors.  B, H, dk, dv, decay and
 * qkv_dtype are those of the tv_problem it is passed with; the other sizes and
 * all arrays are the previous step's (they may be the current step's buffers).
 *
 *   total_nodes, max_nodes, max_depth   sizes of the previous step's batch
 *   node_offsets [B+1], parent [T']     its packed tree (local parents)
 *   g, k, v      its factors, layouts as in tv_verify
 *   path [B][max_depth], accept_len [B] its accepted paths (tv_accept_greedy)
 */
typedef struct tv_pending {
    int32_t total_nodes;
    int32_t max_nodes;
    int32_t max_depth;
    const int32_t *node_offsets;
    const int32_t *parent;
    const float *g;
    const void *k;
    const void *v;
    const int32_t *path;
    const int32_t *accept_len;
} tv_pending;

/*
 * tv_commit_verify -- apply the pending commit to the state in place, then
 * verify the current tree against the updated state.
 * Same results as tv_commit(pending's problem, H, ..., H_new = H) followed by
 * tv_verify(p, H, ...): the commit is the restore of the accepted path's state
 * from its factors (Bole summary page, "Core techniques" §2) and the
 * verification is the tree closed form (§1).  The state is the only operand
 * both steps stream, so for scalar decay with bf16 q/k/v and dk, dv in
 * {64, 128} one kernel reads H once, writes the updated rows back and feeds
 * them to the context term; other shapes run the two kernels in sequence.
 *
 *   p, q, k, v, g, out   the current step, as in tv_verify
 *   pend       the previous step's accepted paths and factors; NULL for none
 *              (then this is tv_verify with H0 = H)
 *   H          [B][H][dk][dv] fp32, read and written (the committed state)
 * Device-detected errors: a malformed pending path (as in tv_commit) gives
 * TV_ERR_TREE and leaves that request's state untouched, and its outputs are
 * computed from the untouched state; a malformed current tree is handled as in
 * tv_verify.  Requests without current nodes still get their pending commit.
 */
tv_status tv_commit_verify(const tv_problem *p, const tv_pending *pend, float *H, const void *q,
                           const void *k, const void *v, const float *g, float *out,
                           int32_t *dev_status, void *stream);

/*
 * tv_accept_commit_verify -- one step of the loop in one launch: the greedy walk of
 * the previous step's tree (LLM Primer VI ch. 9 §9.1), the commit of the path it
 * finds (Bole summary page, "Core techniques" §2) and the verification of the
 * current tree against the committed state (§1).
 * Same results as tv_accept_greedy on the previous tree followed by
 * tv_commit_verify with the paths it wrote.  For tv_commit_verify's one-kernel shapes
 * every block of a request runs the walk itself on shared memory (the head-0 block
 * writes its results), so the commit does not wait for a separate acceptance launch;
 * other shapes run the walk and then tv_commit_verify.
 *
 *   p, H, q, k, v, g, out   the current step, as in tv_commit_verify
 *   prev         the previous step's tree and factors, as in tv_pending; its path and
 *                accept_len fields are not read
 *   draft_tokens, target_argmax [T'], root_argmax [B]   the previous tree's tokens,
 *                as in tv_accept_greedy
 *   accept_len [B], path [B][prev->max_depth], bonus [B]   outputs, as written by
 *                tv_accept_greedy
 * Device-detected errors: those of tv_accept_greedy on the previous tree (that
 * request then commits nothing) and of tv_verify on the current one.
 */
tv_status tv_accept_commit_verify(const tv_problem *p, const tv_pending *prev,
                                  const int32_t *draft_tokens, const int32_t *target_argmax,
                                  const int32_t *root_argmax, int32_t *accept_len, int32_t *path,
                                  int32_t *bonus, float *H, const void *q, const void *k,
                                  const void *v, const float *g, float *out, int32_t *dev_status,
                                  void *stream);

/*
 * tv_tree_attention -- softmax attention of one attention layer over every
 * request's draft tree, the attention layers' share of the verification pass of a
 * hybrid model.  LLM Primer VI ch. 9: the target runs one forward pass over the
 * prefix followed by the candidates (§9.1) and checks a candidate tree in one
 * attention pass with a custom mask (§9.2); Bole summary page ("Why existing tree
 * speculation fails on hybrid models"): all branches share the prefix's KV and each
 * adds only its own.  Query row (node i of request b, head h) sees the first
 * ctx_len[b] cached positions of KV head h / (H / Hkv) and the tree nodes on i's
 * root path, i included:
 *     out[i][h] = sum_j softmax_j(scale * q[i][h] . k_j) v_j.
 *
 *   B, total_nodes (T), max_nodes   as in tv_problem (max_nodes <= TV_MAX_NODES)
 *   H, Hkv     query heads and KV heads; H / Hkv a power of two <= 128
 *   d          head dimension, 64 or 128
 *   P          positions per (request, KV head) in the cache (capacity), >= 1
 *   node_offsets [B+1], parent [T]   the trees, as in tv_verify (parents precede
 *              children; depth is not needed)
 *   ctx_len    [B] int32 (device): valid cached positions of each request, <= P
 *   q          [T][H][d] bf16
 *   k_cache, v_cache  [B][Hkv][P][d] bf16; positions >= ctx_len[b] are never read
 *              into the result (they may hold anything, NaN included)
 *   k_tree, v_tree    [T][Hkv][d] bf16: the tree nodes' own keys and values
 *   scale      softmax scale, positive and finite; usually 1/sqrt(d)
 *   out        [T][H][d] fp32
 *   workspace  optional device memory (16-byte aligned, caller-owned scratch) for
 *              partial results when the context is split over several CTAs, which
 *              the library does when B * Hkv * ceil(max_nodes * H / Hkv / 128) is
 *              below half the SM count.  tv_tree_attention_workspace_bytes gives
 *              the size that allows the library's preferred split; with less (or
 *              NULL, 0) it splits less (not at all with NULL).  Results do not
 *              depend on the split beyond fp32 rounding.
 *   dev_status, stream   see conventions
 * Arithmetic: bf16 inputs, fp32 scores and accumulation on tensor cores; the
 * softmax weights enter the weighted sum of values as bf16 (relative rounding
 * 2^-9), so outputs carry a relative error of order 2^-9.
 * Host errors: TV_ERR_NULL, TV_ERR_ALIGN as usual; TV_ERR_SHAPE for sizes out of
 * range (H not a multiple of Hkv, T > B * max_nodes, P < 1, scale not positive and
 * finite);
 * TV_ERR_UNSUPPORTED for d not in {64, 128}, H / Hkv not a power of two <= 128 or
 * max_nodes > TV_MAX_NODES.  Device-detected errors: bad offsets or parents give
 * TV_ERR_TREE (rows of a request with a bad tree are written as zeros; requests
 * whose offsets are unusable are left untouched); ctx_len[b] outside [0, P] gives
 * TV_ERR_SHAPE and zero rows for that request.
 */
size_t tv_tree_attention_workspace_bytes(int32_t B, int32_t total_nodes, int32_t max_nodes,
                                         int32_t H, int32_t Hkv, int32_t d, int32_t P);
tv_status tv_tree_attention(int32_t B, int32_t total_nodes, int32_t max_nodes, int32_t H,
                            int32_t Hkv, int32_t d, int32_t P, const int32_t *node_offsets,
                            const int32_t *parent, const int32_t *ctx_len, const void *q,
                            const void *k_cache, const void *v_cache, const void *k_tree,
                            const void *v_tree, float scale, float *out, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * tv_verify_variant -- the kernel tv_verify (TV_VARIANT_AUTO) would launch for
 * this problem: TV_VARIANT_TC_STREAM, TV_VARIANT_TC, TV_VARIANT_TC_TILED (trees too
 * large for TV_VARIANT_TC's shared-memory plan, and per-channel decay trees of 64
 * or more nodes, where its staged kernel is the faster) or TV_VARIANT_SIMT.  Reads
 * only the sizes and kinds in *p (no device memory; the current device's SM count
 * and shared memory); returns the negative tv_status of an invalid problem (e.g.
 * -TV_ERR_SHAPE).  The tensor-core kernels take bf16 q/k/v with dk, dv in
 * {64, 128} when their shared-memory plan for max_nodes fits one CTA.
 */
int32_t tv_verify_variant(const tv_problem *p);

/*
 * tv_verify_supports -- 1 when tv_verify_ex would take `variant` for this problem
 * (TV_VARIANT_AUTO and TV_VARIANT_SIMT: any valid problem; the tensor-core
 * variants: the shapes their kernels take), 0 when it would return
 * TV_ERR_UNSUPPORTED, and the negative tv_status of an invalid problem or variant.
 * Reads only the sizes and kinds in *p, like tv_verify_variant.
 */
int32_t tv_verify_supports(const tv_problem *p, int32_t variant);

/* Human-readable name of a status code (static string). */
const char *tv_status_string(int32_t status);

/* TV_VERSION of the loaded library. */
int32_t tv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H */
