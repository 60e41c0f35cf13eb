/*
 * spec_verify.h -- C ABI of a GB300 (sm_103a) library for the target-side verification step of
 * lossless speculative decoding.
 *
 * The method: "Speculative Decoding in Production: From Draft Models to EAGLE-3 Dynamic Trees
 * for 3x-5x Lossless Acceleration" (blog.llmgo.top), section I.1 "Verification via Modified
 * Rejection Sampling": for each draft token x_k, alpha = min(1, p(x_k)/q(x_k)); draw r ~ U(0,1);
 * accept iff r <= alpha, and stop at the first rejection; after a rejection, resample from the
 * normalised positive residual max(0, p - q) / sum max(0, p - q).  The "Invariance Theorem"
 * paragraph that follows states that the emitted tokens then follow p exactly, for greedy
 * decoding and for temperature sampling.  Tree verification: same page, section III.2 "The Tree
 * Attention Verification Mechanism" (a rejected branch is skipped, the matching sibling branch
 * is accepted).  Draft mechanisms (draft model, EAGLE head, prompt n-gram lookup): "Accelerating
 * Autoregressive LLM Inference 3x with Lossless Speculative Decoding and EAGLE Heads"
 * (x078.com), opening section.
 *
 * Conventions common to every call
 *  - Every pointer argument is a DEVICE pointer (cudaMalloc / torch CUDA tensor) unless stated;
 *    the caller owns every buffer; the library allocates nothing.
 *  - Layouts are row-major and contiguous with the vocabulary innermost.  Logits pointers must
 *    be aligned to their element size (16-byte alignment is fastest).
 *  - Calls are asynchronous on `stream` and never synchronise the host.  A status other than
 *    SPEC_OK means nothing was launched (argument errors) or a launch failed (SPEC_ERR_CUDA).
 *  - Per-request problems found on the device (a draft token outside [0, V), a logits row with
 *    NaN, or with +inf / only -inf where a softmax is taken, a malformed parent array, a device
 *    wait that timed out) set bits in err_flags[b]; that request then accepts nothing and emits
 *    no token (num_accepted = 0 / accept_len = 0, every output token -1).  Nothing traps.
 *  - Temperature: p = softmax(logits / T) for T > 0.  T == 0 selects greedy verification: the
 *    target distribution is one-hot at the row argmax (lowest index on ties) and draft logits
 *    are not read.
 *  - Uniforms: r[b][k] in (0, 1] for the acceptance test; u[b] in [0, 1) for the draw after the
 *    accepted prefix (residual resample or bonus token).  Draws use the inverse CDF: the smallest
 *    token i whose cumulative weight exceeds u * (total weight); zero-weight tokens are never
 *    drawn.
 *  - Workspace: `workspace` (device memory, 256-byte aligned) must hold
 *    spec_verify_workspace_bytes(...) bytes; its contents need no initialisation.  The first
 *    call on a workspace (and the first after a change of B, rows or V) clears it with one
 *    cudaMemsetAsync on `stream`; every call leaves it ready for the next (its counters zero,
 *    its epoch advanced), so later calls of the same shape, graph replays included, skip the
 *    clearing.  Between
 *    calls the workspace belongs to the library: when anything else may have written to it (the
 *    memory was freed and allocated again, say), call spec_verify_workspace_reset first.  A
 *    workspace must not be shared by calls that may run concurrently.
 *  - Reads: every logits row is read from HBM once; a draft-model chain call that rejects at
 *    position n reads the target and draft rows at n a second time (the residual max(0, p - q)
 *    needs both rows' normalisers first).  A call is one kernel launch (two when probability
 *    rows are requested), after the clearing above when there is one.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *spec_stream_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* bad shape, NULL required pointer, bad temperature, ... */
    SPEC_ERR_CUDA = 2,        /* a CUDA runtime call or a kernel launch failed */
    SPEC_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than required */
    SPEC_ERR_UNSUPPORTED = 4  /* a size beyond the supported maximum */
} spec_status_t;

typedef enum { SPEC_DTYPE_F32 = 0, SPEC_DTYPE_BF16 = 1, SPEC_DTYPE_F16 = 2 } spec_dtype_t;

/* Bits of err_flags[b]. */
#define SPEC_ERRF_BAD_TOKEN 1 /* a draft / node token outside [0, V) */
#define SPEC_ERRF_NONFINITE 2 /* NaN logits, or +inf / all -inf where a softmax is taken */
#define SPEC_ERRF_TIMEOUT 4   /* a bounded device wait gave up (should never happen) */
#define SPEC_ERRF_BAD_TREE 8  /* parents[0] != -1 or parents[i] not in [0, i) */
#define SPEC_ERRF_BAD_TEMPERATURE 16 /* a per-request temperature that is NaN, negative or infinite */

/* Largest supported sizes. */
#define SPEC_MAX_K 256           /* draft tokens per request (chain / n-gram) */
#define SPEC_MAX_TREE_NODES 4096 /* N + 1 for spec_verify_tree_greedy */
#define SPEC_MAX_WALK_NODES 1024 /* N + 1 for spec_verify_tree_walk */
#define SPEC_MAX_WALK_VOCAB 262144 /* V for spec_verify_tree_walk */
#define SPEC_MAX_NGRAM 32          /* n_max for spec_ngram_draft */
#define SPEC_MAX_KV_CACHES 1024    /* caches (layers x K/V) per spec_kv_compact call */

/* Bytes of workspace for a call on B requests with vocabulary V of `dtype`, where
 * rows_per_request is the number of logits rows the call reads per request:
 *   spec_verify_chain with T > 0: 2K + 1;  spec_verify_chain with T == 0 and spec_verify_ngram:
 *   K + 1;  spec_verify_tree_greedy: N + 1.
 * A workspace sized for more rows (or a larger B) also serves a smaller call.  Returns 0 for
 * invalid sizes. */
size_t spec_verify_workspace_bytes(int B, int rows_per_request, int V, spec_dtype_t dtype);

/* Marks `workspace` (the pointer a call was given) as holding contents the library did not leave
 * there, so that its next call clears it first.  Host-side only; touches no memory and never
 * fails.  Needed only when something other than these calls wrote to it. */
void spec_verify_workspace_reset(const void *workspace);

/*
 * Chain verification with a draft model or an EAGLE head (the draft side is logits).
 *
 * target_logits  [B][K+1][V] dtype; row k scores draft position k given the accepted prefix,
 *                row K scores the bonus position.
 * draft_logits   [B][K][V] dtype; the draft distribution at each draft position.  Not read
 *                (may be NULL) when temperature == 0 and temperatures is NULL.
 * temperatures   [B] float or NULL: each request's own temperature, used instead of
 *                `temperature` (the x078.com page's production section sets the temperature per
 *                request).  0 verifies that request greedily (its draft rows are not read); NaN, a
 *                negative value or infinity fails the request with SPEC_ERRF_BAD_TEMPERATURE alone.
 *                When given, draft_logits (K > 0), r and u are required and the workspace is sized
 *                for 2K + 1 rows.
 * draft_tokens   [B][K] int32, the drafted tokens x_k.
 * r              [B][K] float, acceptance uniforms in (0, 1].  Not read when temperature == 0.
 * u              [B] float, uniforms in [0, 1) for the residual / bonus draw.  Not read when
 *                temperature == 0.
 * Outputs:
 * num_accepted   [B] int32, n in [0, K]: the length of the accepted prefix.
 * out_tokens     [B][K+1] int32: x_1..x_n, then the drawn token (residual resample at position
 *                n if n < K, bonus token from row K if n == K), then -1.
 * residual_mass  [B] float or NULL: the total weight the draw used, i.e. sum max(0, p - q) at
 *                the rejected position (the total-variation distance of p and q there), 1 for a
 *                bonus draw, 1 in greedy mode.
 * err_flags      [B] int32 or NULL: SPEC_ERRF_* bits, 0 when the request verified normally.
 * Optional per-position diagnostics (NULL to skip):
 * accept_prob    [B][K] float: alpha_k = min(1, p_k(x_k)/q_k(x_k)) at every position (greedy:
 *                1 if x_k equals the target argmax, else 0).
 * cand_tokens    [B][K+1] int32: the token the draw would emit at position k (residual at
 *                k < K, bonus at K; greedy: the argmax of row k).
 * pos_mass       [B][K+1] float: the residual mass at each position (bonus row: 1).
 * target_probs   [B][K+1][V] float: p rows (T > 0 only; an extra launch, for testing; with
 *                per-request temperatures, the rows of greedy requests are left untouched).
 * draft_probs    [B][K][V] float: q rows (T > 0 only).
 * Requesting cand_tokens or pos_mass makes the call draw at every position, which re-reads the
 * pair (draft-model chain) or one chunk per row (n-gram); leave them NULL on the hot path.
 */
spec_status_t spec_verify_chain(const void *target_logits, const void *draft_logits,
                                spec_dtype_t dtype, int B, int K, int V, float temperature,
                                const float *temperatures, const int32_t *draft_tokens,
                                const float *r, const float *u,
                                int32_t *num_accepted, int32_t *out_tokens, float *residual_mass,
                                int32_t *err_flags, float *accept_prob, int32_t *cand_tokens,
                                float *pos_mass, float *target_probs, float *draft_probs,
                                void *workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * Chain verification with a prompt n-gram lookup draft: q_k is one-hot at x_k, so
 * alpha_k = p_k(x_k) and the residual at a rejected position is p_k with x_k removed.  No draft
 * logits exist.  Arguments and outputs as spec_verify_chain (target_probs and temperatures
 * likewise optional; the workspace takes K + 1 rows either way); temperature == 0 gives the
 * greedy chain.
 */
spec_status_t spec_verify_ngram(const void *target_logits, spec_dtype_t dtype, int B, int K,
                                int V, float temperature, const float *temperatures,
                                const int32_t *draft_tokens,
                                const float *r, const float *u, int32_t *num_accepted,
                                int32_t *out_tokens, float *residual_mass, int32_t *err_flags,
                                float *accept_prob, int32_t *cand_tokens, float *pos_mass,
                                float *target_probs, void *workspace, size_t workspace_bytes,
                                spec_stream_t stream);

/*
 * Greedy verification of a draft tree (EAGLE-2 style).  Node 0 is the root (the last accepted
 * token); nodes 1..N are draft tokens, each with a parent of smaller index.
 *
 * target_logits  [B][N+1][V] dtype; row n is the target's prediction after node n.
 * node_tokens    [B][N+1] int32; entry 0 is ignored.
 * parents        [B][N+1] int32; parents[0] = -1 and 0 <= parents[i] < i.
 * The walk starts at the root and repeatedly moves to the child whose token equals the argmax
 * of the current node's row (the lowest node index if several do), until no child matches.
 * Outputs:
 * accept_len     [B] int32: accepted draft tokens on the path (0..depth).
 * path_nodes     [B][N+1] int32: node ids on the accepted path, root first, then -1.
 * out_tokens     [B][N+1] int32: the accepted tokens, then the argmax of the last node's row
 *                (the correction or bonus token), then -1.
 * err_flags      [B] int32 or NULL.
 * node_argmax    [B][N+1] int32 or NULL: the argmax of every row.
 */
spec_status_t spec_verify_tree_greedy(const void *target_logits, spec_dtype_t dtype, int B,
                                      int N, int V, const int32_t *node_tokens,
                                      const int32_t *parents, int32_t *accept_len,
                                      int32_t *path_nodes, int32_t *out_tokens,
                                      int32_t *err_flags, int32_t *node_argmax, void *workspace,
                                      size_t workspace_bytes, spec_stream_t stream);

/*
 * Verification of a draft tree by walking it from the root, stochastic (T > 0) or greedy
 * (T == 0).  Reads only the rows of the nodes the walk visits.
 *
 * Stochastic walk: section I.1 of the page named at the top, applied to the children of each
 * visited node in turn.  With p = softmax(target row / T) and q = softmax(draft row / T) of the
 * visited node, its children are tested in ascending node index: child c with token x is accepted
 * when r[b][c] <= alpha = min(1, p'(x) / q(x)), where p' is the current target (p at first); the
 * walk then moves to c.  A rejected child replaces the target by its residual
 * max(0, p' - q) / sum max(0, p' - q) before the next sibling is tested (same q).  When no child
 * is accepted, or the node has none, the token is drawn from the current target by the inverse
 * CDF with u[b].  Lossless when the children of a node are independent draws from its q.  A
 * chain (one child per node) is exactly spec_verify_chain.  Greedy walk (T == 0): the child whose
 * token equals the argmax of the node's target row (the lowest node index if several), as in
 * spec_verify_tree_greedy, but reading only the visited rows.
 *
 * target_logits  [B][N+1][V] dtype; row n is the target's prediction after node n.
 * draft_logits   [B][N+1][V] dtype; row n is the draft distribution the children of node n were
 *                drawn from.  Rows of nodes without children are never read; not read at all
 *                (may be NULL) when temperature == 0 and temperatures is NULL.
 * temperatures   [B] float or NULL: each request's own temperature, used instead of
 *                `temperature` (the x078.com page's production section sets it per request).  0
 *                walks that request greedily; NaN, a negative value or infinity fails the request
 *                with SPEC_ERRF_BAD_TEMPERATURE.  When given, draft_logits, r and u are required.
 * node_tokens    [B][N+1] int32 (entry 0 ignored); parents [B][N+1] int32, parents[0] = -1 and
 *                0 <= parents[i] < i.
 * r              [B][N+1] float in (0, 1]: r[b][c] is the uniform of child c's test (entry 0
 *                unused).  u [B] float in [0, 1).  Neither is read when temperature == 0.
 * Outputs:
 * accept_len     [B] int32: accepted draft tokens on the path.
 * path_nodes     [B][N+1] int32: the accepted path, root first, then -1.
 * out_tokens     [B][N+1] int32: the accepted tokens, then the drawn (greedy: argmax) token,
 *                then -1.
 * residual_mass  [B] float or NULL: the total weight of the draw's residual when siblings were
 *                rejected at the last node; 1 when none was (and in greedy mode); 0 when the
 *                residual vanished in rounding and the draw fell back to p.
 * err_flags      [B] int32 or NULL: SPEC_ERRF_* bits.  A malformed tree or a node token outside
 *                [0, V) (the lowest offending node decides), or a non-finite visited row, fails
 *                the request: accept_len 0, path and tokens -1.  Rows the walk does not visit are
 *                not checked.
 * accept_prob    [B][N+1] float or NULL: alpha of every child tested (greedy: 1 for the matching
 *                child, 0 for the siblings tested before it), -1 for the others.
 * Limits: N + 1 <= SPEC_MAX_WALK_NODES, V <= SPEC_MAX_WALK_VOCAB (SPEC_ERR_UNSUPPORTED beyond).
 * One kernel launch; no workspace.  A request occupies a cluster of up to 16 CTAs (V / 16384
 * rounded up to a power of two; one CTA for V <= 4096); as many clusters as fit run at once.
 */
spec_status_t spec_verify_tree_walk(const void *target_logits, const void *draft_logits,
                                    spec_dtype_t dtype, int B, int N, int V, float temperature,
                                    const float *temperatures, const int32_t *node_tokens, const int32_t *parents,
                                    const float *r, const float *u, int32_t *accept_len,
                                    int32_t *path_nodes, int32_t *out_tokens,
                                    float *residual_mass, int32_t *err_flags,
                                    float *accept_prob, spec_stream_t stream);

/*
 * Prompt n-gram lookup drafting: the draft side of spec_verify_ngram, computed on the GPU.
 * "Accelerating Autoregressive LLM Inference 3x with Lossless Speculative Decoding and EAGLE
 * Heads" (x078.com), opening section: a zero-VRAM prompt n-gram lookup proposes K candidate
 * tokens (its serving example uses K = 5 and --ngram-prompt-lookup-max 4).
 *
 * For n = n_max down to n_min, the last n tokens of the context are looked up in the context;
 * their most recent earlier occurrence (the largest start i with i + n <= L - 1 whose n tokens
 * equal them; it may overlap them) wins, and the draft is the tokens that follow it,
 * context[i + n .. min(i + n + K, L)).  No match for any n gives an empty draft.
 *
 * context        [B][Lmax] int32 token ids (any values; only equality is used).
 * context_len    [B] int32, L in [0, Lmax]; another value gives an empty draft and sets
 *                SPEC_ERRF_BAD_TOKEN in err_flags.
 * n_max, n_min   1 <= n_min <= n_max <= SPEC_MAX_NGRAM;  K in [1, SPEC_MAX_K].
 * Outputs:
 * draft_tokens   [B][K] int32: the draft, then -1.
 * draft_len      [B] int32: its length (0..K).
 * match_n        [B] int32 or NULL: the n that matched (0 for none).
 * match_end      [B] int32 or NULL: i + n, where the draft starts in the context (-1 for none).
 * err_flags      [B] int32 or NULL.
 * One kernel launch (one CTA per context); the context is read once.  No workspace.
 */
spec_status_t spec_ngram_draft(const int32_t *context, const int32_t *context_len, int B,
                               int Lmax, int n_max, int n_min, int K, int32_t *draft_tokens,
                               int32_t *draft_len, int32_t *match_n, int32_t *match_end,
                               int32_t *err_flags, spec_stream_t stream);

/*
 * Accepted-path KV-cache compaction after tree verification: "Speculative Decoding with Medusa,
 * EAGLE and vLLM" (vikram-blog.pages.dev), "System Topology & Data Flow" diagram (the accepted
 * branch's tokens are committed to the KV cache).
 *
 * The target's forward pass over the flattened tree wrote the KV row of node n of request b into
 * slot slots[b][n] of every cache.  With the accepted path p_0 = 0, p_1, ..., p_L (as written by
 * spec_verify_tree_greedy / spec_verify_tree_walk), the row of p_j moves to slot slots[b][j] for
 * j = 1..L, so the accepted tokens occupy the request's first L + 1 slots in order; every other
 * slot keeps its contents.  Moves happen in place.
 *
 * caches         HOST array of num_caches DEVICE pointers (16-byte aligned), each a cache of
 *                num_slots rows of row_bytes bytes (a layer's K or V tensor, any element type).
 * row_bytes      a multiple of 16.
 * slots          [B][N+1] int32: the slot of each tree node; distinct within a request, and the
 *                requests' slots disjoint.
 * parents        [B][N+1] int32 (the tree), accept_len [B], path_nodes [B][N+1] int32.
 * err_flags      [B] int32 or NULL: SPEC_ERRF_BAD_TREE when accept_len is outside [0, N], the
 *                path is not a chain of parent links from the root, or a slot is outside
 *                [0, num_slots); that request's rows are left untouched.
 * Limits: num_caches <= SPEC_MAX_KV_CACHES, N + 1 <= SPEC_MAX_WALK_NODES, B <= 65535.
 * One kernel launch; reads and writes each moved row once.  No workspace.  The launch allows
 * programmatic stream serialisation: its blocks may start while the previous kernel in the stream
 * drains, but they wait for that kernel to complete before reading or writing anything, so the
 * call keeps stream order.
 */
spec_status_t spec_kv_compact(void *const *caches, int num_caches, long long num_slots,
                              int row_bytes, int B, int N, const int32_t *slots,
                              const int32_t *parents, const int32_t *accept_len,
                              const int32_t *path_nodes, int32_t *err_flags,
                              spec_stream_t stream);

/*
 * spec_verify_chain without a workspace argument, for callers that cannot allocate device memory
 * (a plugin inside an engine that has reserved all GPU memory for its own pool, a hook that must
 * not call cudaMalloc because it can synchronise the device, a binding with no CUDA allocator).
 * The pages have no counterpart of this entry point; it is an interface convenience.
 *
 * Scratch lives in one device array of SPEC_STATIC_WORKSPACE_BYTES inside the library, which every
 * GPU that loads the library holds until the process exits.  Calls whose scratch would not fit
 * (spec_verify_workspace_bytes(B, 2K + 1, V, dtype) above the limit, K + 1 rows for T == 0) return
 * SPEC_ERR_UNSUPPORTED.  The first call on a device looks up that device's copy of the array
 * (cudaGetSymbolAddress, with the device current); make that first call before any stream
 * capture.  Every call on a device shares the same array and leaves its contents behind: the first
 * call of a shape (B, rows, V) clears it, and every later call of that shape relies on the previous
 * call having left its counters at zero, which every call does, one whose device wait timed out
 * included.  Calls that may overlap on the GPU (other streams, other host threads) race on the
 * array and must be serialised by the caller.  K > SPEC_MAX_K returns SPEC_ERR_UNSUPPORTED, as
 * spec_verify_chain does.  The call allocates nothing.
 * Arguments and outputs as spec_verify_chain, without the optional per-position outputs.
 */
#define SPEC_STATIC_WORKSPACE_BYTES (4u << 20)
spec_status_t spec_verify_chain_static(const void *target_logits, const void *draft_logits,
                                       spec_dtype_t dtype, int B, int K, int V, float temperature,
                                       const int32_t *draft_tokens, const float *r, const float *u,
                                       int32_t *num_accepted, int32_t *out_tokens,
                                       float *residual_mass, int32_t *err_flags,
                                       spec_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *spec_status_string(spec_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
