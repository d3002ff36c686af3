/*
 * dartree.h — C ABI of the DARTree draft-tree build and verify step on sm_103a.
 *
 * Method: DARTree: Speculative Diffusion Decoding with Autoregressive Draft Trees,
 * as described on the marsggbo.github.io blog post (section 3.1 "Basic flow",
 * section 3.2) and the ainews.surl.tw article "DARTree Builds Trees in Batches
 * Before Pruning". One speculative round is:
 *   S1  top-K candidates of every block position's base logits        (3.1, candidate generation)
 *   S2  root state h = E[anchor], score 0
 *   S3-S7 for d = 1..L: correction head on all parents of depth d-1 in one
 *       batch, s = s_parent + log q + beta, keep the top-W children      (3.1, depth-wise expansion,
 *       (the kept nodes of all depths form the supertree)                   scoring function, per-depth pruning)
 *   S8  deferred pruning: global top-B of the supertree                (3.1, deferred pruning, Lemma 1)
 *   S9  tree-attention mask and position ids                           (3.2)
 *   S10 greedy longest accepted prefix against the target's logits     (3.2)
 *
 * The pages do not define the correction head; this library implements the
 * stand-in head  u_p = W_q h_p,  z[p,c] = L^base[d-1,c] + <u_p, E[c]>/sqrt(H),
 * q = softmax over the K candidates of position d-1,
 * h_child = RMSNorm(h_p + E[tok] + H_d[d-1]) (eps 1e-6, unit weight), stored in
 * the input storage type.
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller, row-major and
 *    contiguous. The library allocates no memory: scratch lives in a caller
 *    allocated workspace of dartree_workspace_bytes() bytes (device memory,
 *    256-byte aligned).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All work is enqueued asynchronously on it; outputs are valid after the
 *    caller synchronises the stream. No call synchronises, except
 *    dartree_read_status.
 *  - Argument errors are detected on the host before anything is enqueued and
 *    returned as a negative dartree_status; nothing is written then. Launch
 *    failures return DARTREE_ECUDA. Errors detected on the device (a bounded
 *    wait that ran out, a buffer overflow) are recorded in a status word at the
 *    start of the workspace (first error wins) and read with
 *    dartree_read_status.
 *  - Floating point inputs are finite. Equal values are ordered as stated per
 *    step; -0.0 and +0.0 compare equal.
 *  - Calls that share a workspace must not overlap on the device.
 *  - Process-wide state (no device memory): forks inside a call (the second half
 *    of a batch of 32 or more requests in S2-S7, the target-row maxima of
 *    dartree_round) run on library-owned side streams, one pair per (device,
 *    caller stream), created with their events on the first call that needs them
 *    on that stream; make that call before capturing the stream into a CUDA graph.
 *    Callers on different streams use different side streams and do not wait for
 *    each other; a host mutex is held while a call enqueues its forks. Besides
 *    these: the device address of the array of dartree_verify_static, and the
 *    records of dartree_timing.
 */
#ifndef DARTREE_H
#define DARTREE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DARTREE_API __attribute__((visibility("default")))
#else
#define DARTREE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DARTREE_OK = 0,
    DARTREE_EINVAL = -1,       /* bad size, null pointer or beta > 0 */
    DARTREE_EDTYPE = -2,       /* unknown dtype or row mode */
    DARTREE_EWORKSPACE = -3,   /* workspace null, misaligned or too small */
    DARTREE_ECUDA = -4,        /* a CUDA runtime call or launch failed */
    DARTREE_ETIMEOUT = -5,     /* device: a bounded wait ran out */
    DARTREE_EINTERNAL = -6,    /* device: an internal consistency check failed */
    DARTREE_EUNSUPPORTED = -7  /* sizes beyond the limits below */
} dartree_status;

typedef enum { DARTREE_F32 = 0, DARTREE_BF16 = 1 } dartree_dtype;

/* Layout of the target logits handed to dartree_verify. */
typedef enum {
    DARTREE_ROWS_PER_POSITION = 0, /* [C, L, V]: the slot at depth delta is checked with row delta */
    DARTREE_ROWS_PER_NODE = 1      /* [C, B+1, V]: slot j is checked with row j (row 0 = root) */
} dartree_rows;

/* Limits (DARTREE_EUNSUPPORTED beyond them). */
#define DARTREE_MAX_K 1024
#define DARTREE_MAX_W 256
#define DARTREE_MAX_L 64
#define DARTREE_MAX_SLOTS 1024   /* B + 1 */
#define DARTREE_MAX_CHILDREN 8192 /* W * K children scored per depth and request */

/* Stand-in correction head (shared model weights). */
typedef struct {
    const void* E;   /* [V, H] token embeddings, dtype */
    const void* Wq;  /* [H, H] projection, row-major, u = Wq h */
    int V;
    int H;           /* multiple of 8 */
    int dtype;       /* dartree_dtype of E, Wq, base logits and block hidden states */
    const void* WqT; /* [H, H] W_q transposed, filled by dartree_head_prepare; NULL until then */
} dartree_head;

/* Shape of one round. */
typedef struct {
    int C;       /* requests in the batch */
    int L;       /* block length = maximum depth, 1..DARTREE_MAX_L */
    int K;       /* candidates per position, 1..min(V, DARTREE_MAX_K) */
    int W;       /* nodes kept per depth, 1..DARTREE_MAX_W, W*K <= DARTREE_MAX_CHILDREN */
    int B;       /* node budget (root excluded), 1..min(L*W, DARTREE_MAX_SLOTS-1) */
    float beta;  /* depth term, <= 0 (Lemma 1 needs beta <= 0) */
} dartree_params;

/* Candidate table of S1: per (request, position) the K best tokens ordered by
 * (logit desc, token id asc), and their logits as float. */
typedef struct {
    int32_t* tok;   /* [C, L, K] */
    float* logit;   /* [C, L, K] */
} dartree_candidates;

/* Supertree of S7: the kept nodes of every depth d (index d-1), in rank order
 * (score desc, flat index p*K+c asc). par is the parent's rank at depth d-1
 * (0 = the root for d = 1). Unused entries: tok = par = -1, score = 0. */
typedef struct {
    int32_t* tok;   /* [C, L, W] */
    int32_t* par;   /* [C, L, W] */
    float* score;   /* [C, L, W] s_beta of the node */
    int32_t* n;     /* [C, L] kept nodes per depth: min(W, n_{d-1} * K), n_0 = 1 */
} dartree_supertree;

/* Verification tree of S8/S9, B+1 slots per request. Slot 0 is the root
 * (tok = anchor, par = -1, depth 0, score 0). Slots 1..n_nodes-1 hold the
 * chosen nodes depth-major, by rank within a depth; par holds slot ids
 * (par < own slot). Unused slots: tok = par = depth = pos = -1, score = 0,
 * mask row and column 0. n_nodes = 1 + min(B, supertree size). */
typedef struct {
    int32_t* tok;      /* [C, B+1] */
    int32_t* par;      /* [C, B+1] */
    int32_t* depth;    /* [C, B+1] */
    float* score;      /* [C, B+1] */
    int32_t* n_nodes;  /* [C] */
    uint8_t* mask;     /* [C, B+1, B+1] mask[i][j] = 1 iff slot j is an ancestor of slot i or i itself */
    int32_t* pos;      /* [C, B+1] position id = depth */
} dartree_tree;

/* Checks and stores the head description. E and Wq must stay valid while the
 * head is used. Returns DARTREE_OK or a negative status. */
DARTREE_API int dartree_head_init(dartree_head* head, const void* E, const void* Wq, int V, int H, int dtype);

/* Derived per-model data for the small-batch path: writes W_q^T into `wqt`
 * (caller-owned device memory of H*H elements of the head's dtype, valid while the
 * head is used) on `stream` and records it in head->WqT. Call once after
 * dartree_head_init and again whenever W_q changes. Without it, every batch takes
 * the per-depth projection path. bf16 heads only (DARTREE_EUNSUPPORTED otherwise). */
DARTREE_API int dartree_head_prepare(dartree_head* head, void* wqt, void* stream);

/* Workspace bytes needed by every call below for this shape (0 on bad arguments). */
DARTREE_API size_t dartree_workspace_bytes(const dartree_params* p, int V, int H, int dtype);

/* S1 alone: top-K of `rows` rows of `V` logits (dtype), written to tok/val
 * [rows, K] ordered by (logit desc, token id asc). Uses only the workspace's
 * status word (ws_bytes >= 256). */
DARTREE_API int dartree_topk(const void* logits, int rows, int V, int K, int dtype,
                 int32_t* tok, float* val, void* ws, size_t ws_bytes, void* stream);

/* S2-S7: expand all depths from a given candidate table.
 *   base_logits  unused (the candidate table carries the logits); may be NULL
 *   block_hidden [C, L, H] dtype, H_d of the block drafter
 *   anchor       [C] int32 anchor tokens
 *   cand         candidate table of S1
 *   st           supertree output */
DARTREE_API int dartree_expand(const dartree_head* head, const dartree_params* p, const void* block_hidden,
                   const int32_t* anchor, const dartree_candidates* cand, dartree_supertree* st,
                   void* ws, size_t ws_bytes, void* stream);

/* S8: deferred pruning of a supertree into tree.tok/par/depth/score/n_nodes.
 * Global order: score desc, depth asc, rank asc. tree.mask and tree.pos are not touched. */
DARTREE_API int dartree_prune(const dartree_params* p, const dartree_supertree* st, const int32_t* anchor,
                  dartree_tree* tree, void* stream);

/* S9: tree.mask and tree.pos from tree.par, tree.depth and tree.n_nodes. */
DARTREE_API int dartree_tree_mask(const dartree_params* p, dartree_tree* tree, void* stream);

/* S1-S9: one full tree build.
 *   base_logits  [C, L, V] dtype, L^base of the block drafter
 *   block_hidden [C, L, H] dtype
 *   anchor       [C] int32
 *   tree         output (mask and pos are built when non-NULL)
 *   st, cand     optional outputs (NULL: kept in the workspace) */
DARTREE_API int dartree_build_tree(const dartree_head* head, const dartree_params* p, const void* base_logits,
                       const void* block_hidden, const int32_t* anchor, dartree_tree* tree,
                       dartree_supertree* st, dartree_candidates* cand,
                       void* ws, size_t ws_bytes, void* stream);

/* S10: greedy longest accepted prefix. From the root, t = argmax of the current
 * slot's target row (lowest token id among equal maxima); move to the child
 * carrying t while one exists.
 *   target        [C, L, V] (rows = DARTREE_ROWS_PER_POSITION) or [C, B+1, V]
 *                 (DARTREE_ROWS_PER_NODE), dtype
 *   accepted_len  [C] accepted drafted tokens, 0..L
 *   path          [C, L] slot ids of the accepted nodes in depth order, -1 padded
 *   bonus         [C] the target's token after the accepted prefix (argmax of the
 *                 last accepted slot's row), -1 when that row does not exist
 *                 (per-position rows and a fully accepted block)
 * A tree whose walk would take more than L steps (a parent that is not one depth
 * above its child) is malformed: the walk stops and DARTREE_EINTERNAL is recorded
 * in the status word of ws. */
DARTREE_API int dartree_verify(const dartree_params* p, const dartree_tree* tree, const void* target,
                   int rows, int V, int dtype, int32_t* accepted_len, int32_t* path,
                   int32_t* bonus, void* ws, size_t ws_bytes, void* stream);

/* S10 when the target samples at a temperature T > 0 (DARTree blog post, section 4
 * and Table 1: results at temperatures 0 and 1, speed-ups called lossless; the pages
 * print no acceptance rule for T > 0). The same walk as dartree_verify, on a drawn
 * token instead of the row's maximum: t = argmax_v (x_v / T + G_v), lowest token id
 * among equal values, G_v = -log(-log U_v), a Gumbel-max draw from softmax(row / T).
 * Every emitted token (accepted drafts and the bonus) is a draw of the target at T,
 * so the output distribution is the target's own. U_v comes from Philox4x32-10
 * (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC
 * 2011) with key (seed & 0xffffffff, seed >> 32), counter (v / 4, row, request, 0)
 * and output word v % 4, U_v = (2 (word >> 9) + 1) 2^-24; row is the slot's depth
 * for per-position rows and the slot index for per-node rows. x_v / T, the sum and
 * the logarithms are float32.
 *   temperature  T, positive and finite (DARTREE_EINVAL otherwise)
 *   seed         64-bit generator key; equal seeds give equal draws
 *   other arguments, outputs, workspace and errors as for dartree_verify. */
DARTREE_API int dartree_verify_sample(const dartree_params* p, const dartree_tree* tree, const void* target,
                                      int rows, int V, int dtype, float temperature, uint64_t seed,
                                      int32_t* accepted_len, int32_t* path, int32_t* bonus, void* ws,
                                      size_t ws_bytes, void* stream);

/* The block drafter's LM head fused with S1 (DARTree blog post, "3.1 Basic flow",
 * candidate generation: the top-K tokens of every block position's base logits).
 * The base logits L[r, v] = <hidden[r], W_lm[v]> (a linear head without bias; the
 * pages do not print the drafter's head) are accumulated in fp32 on the tensor
 * cores and reduced to candidates on chip: they are never written to memory.
 *   hidden    [R, H] bf16, one row per (request, block position): R = C * L
 *   W_lm      [V, H] bf16, one row per vocabulary token (row-major)
 *   K         candidates per row, 1..128, K <= V
 *   tok, val  [R, K] outputs: tokens ordered by (logit desc, token id asc) and
 *             their fp32 logits; the same layout as dartree_candidates, so the
 *             result can be handed to dartree_expand
 * H must be a multiple of 64; hidden and W_lm start on 16-byte boundaries. Rows
 * are processed 64 at a time (each group of 64 rows streams W_lm once). fp32
 * operands: DARTREE_EUNSUPPORTED. Workspace: dartree_lm_head_workspace_bytes
 * (status word + one K-key list per row and SM). */
DARTREE_API size_t dartree_lm_head_workspace_bytes(int R, int V, int H, int K);
DARTREE_API int dartree_lm_head_topk(const void* hidden, const void* W_lm, int R, int V, int H, int K,
                                     int dtype, int32_t* tok, float* val, void* ws, size_t ws_bytes,
                                     void* stream);

/* One attention layer of the target's verification pass over the pruned tree
 * (DARTree blog post, "3.2": all drafted tokens are checked in one target pass with
 * a tree-attention mask). Slot j of request c, query head h, attends to the c-th
 * request's n_ctx[c] cached keys and to the tree slots tree->mask[c, j, :] marks
 * (ancestor-or-self, S9), with rotary embedding at position n_ctx[c] + tree->pos[c, j]
 * (pos = depth, S9) applied to the tree's queries and keys:
 *   x'_i = x_i cos a_i - x_(i+D/2) sin a_i,  x'_(i+D/2) = x_(i+D/2) cos a_i + x_i sin a_i,
 *   a_i = position * theta^(-2i/D), i < D/2;
 * query head h reads key/value head h / (Hq / Hkv); scores are scaled by 1/sqrt(D).
 * All tensors bf16, row-major, 16-byte aligned:
 *   q         [C, S, Hq, D]    the tree's queries (unrotated)
 *   k_tree    [C, S, Hkv, D]   the tree's keys (unrotated)
 *   v_tree    [C, S, Hkv, D]   the tree's values
 *   k_cache   [C, Hkv, N, D]   cached keys (already rotated), position = row
 *   vt_cache  [C, Hkv, D, N]   cached values stored transposed (one head's keys
 *                              contiguous per dimension: the operand layout of P V)
 *   n_ctx     [C] int32        cached length of each request, 0..N (clamped to it);
 *                              cache entries past it are not used but must be finite
 *   tree      S9 output: mask [C, S, S], pos [C, S], n_nodes [C] are read
 *   out       [C, S, Hq, D]    output rows (zero for slots j >= n_nodes[c])
 * Scores and sums in fp32; probabilities are rounded to bf16 for the P V product.
 * Limits (DARTREE_EUNSUPPORTED): D = 128, S <= 128, Hq a multiple of Hkv,
 * (Hq / Hkv) * S <= 384, N a multiple of 8, theta > 0. Workspace:
 * dartree_tree_attention_workspace_bytes (rotated tree operands and, for small
 * batches, the partial results of the key-block chunks run in parallel). */
typedef struct {
    int C;        /* requests */
    int S;        /* tree slots per request (B + 1) */
    int Hq, Hkv;  /* query heads, key/value heads */
    int D;        /* head dimension */
    int N;        /* cache capacity per request and head */
    float theta;  /* rotary base */
} dartree_attn_params;

DARTREE_API size_t dartree_tree_attention_workspace_bytes(const dartree_attn_params* p);
DARTREE_API int dartree_tree_attention(const dartree_attn_params* p, const void* q, const void* k_tree,
                                       const void* v_tree, const void* k_cache, const void* vt_cache,
                                       const int32_t* n_ctx, const dartree_tree* tree, void* out, void* ws,
                                       size_t ws_bytes, void* stream);

/* Node budget and width for a batch of C concurrent requests (DARTree blog post,
 * section 4.4: at concurrency 4 the budget B shrinks from 64 to 32 and the width W
 * from 12 to 3; at concurrency 1 and 2 the defaults run). Reading: the reduced pair
 * applies from C = DARTREE_REDUCED_BUDGET_FROM_C on. Host only, no GPU work.
 *   C     requests in the batch, >= 1 (DARTREE_EINVAL otherwise)
 *   B, W  outputs: (64, 12) below the threshold, (32, 3) from it */
#define DARTREE_REDUCED_BUDGET_FROM_C 4
DARTREE_API int dartree_adaptive_budget(int C, int* B, int* W);

/* S1-S10 in one call: dartree_build_tree (no supertree or candidate outputs)
 * followed by dartree_verify, with the same results as those two calls.
 * target, rows: as for dartree_verify, with V and dtype of the head. With
 * per-position rows the target-row maxima do not depend on the tree: when S1 runs
 * as one cluster per row (few rows) and the target and logit rows start on 16-byte
 * boundaries, the S1 launch computes them too; otherwise they are computed on a
 * library-owned side stream of `stream` (see the conventions above) forked after
 * S1 and joined before the walk; the fork is captured with the rest when `stream`
 * is being captured into a CUDA graph. The row
 * maxima go to a workspace region of their own (the workspace of
 * dartree_workspace_bytes suffices). Later kernels of the call may be launched as
 * programmatic dependents of the one before (each waits for it on the device
 * before reading its results), so their set-up overlaps its tail; the results and
 * stream order seen by the caller are those of plain launches. Errors as for the
 * two calls. */
DARTREE_API int dartree_round(const dartree_head* head, const dartree_params* p, const void* base_logits,
                              const void* block_hidden, const int32_t* anchor, const void* target, int rows,
                              dartree_tree* tree, int32_t* accepted_len, int32_t* path, int32_t* bonus,
                              void* ws, size_t ws_bytes, void* stream);

/* Rounds fed from host memory (the serving loop's view of dartree_round): a
 * caller-owned session holds two device sets of a round's inputs, the device
 * tree, results and workspace (one device allocation made at creation; nothing is
 * allocated per round) and a copy stream of its own. Round i runs from input set
 * i % 2, so the caller stages round i + 1's inputs while round i runs:
 *   dartree_host_stage(s, in_0); for i: [dartree_host_stage(s, in_i+1);]
 *   dartree_host_round(s, out_i, stream)
 * dartree_host_stage enqueues the host -> device copies of one round's inputs on
 * the session's copy stream, into the set no unfinished round reads (the copy
 * waits on the device for the round that last read that set). At most two staged
 * sets may be waiting: a third stage before a round returns DARTREE_EINVAL.
 * dartree_host_round makes `stream` wait for the oldest staged set, enqueues
 * dartree_round on it (same results and errors) and then the device -> host copies
 * of accepted_len, path and bonus into `out`; they are valid once `stream` has been
 * synchronised. Host buffers: pinned memory for copies that overlap the rounds
 * (pageable memory works, with synchronous copies). A session is used by one host
 * thread at a time; it keeps the head's pointers (E, Wq, WqT), which must stay
 * valid. dartree_host_session_destroy waits for the session's copies and rounds
 * (and their result copies) before freeing its memory. Errors: DARTREE_EINVAL (null pointers, C < 1, a shape dartree_round
 * rejects), DARTREE_EDTYPE (dtype or row mode), DARTREE_ECUDA (allocation, stream,
 * event or copy failures).
 *   head, p, rows  as for dartree_round; the inputs of every round have its shapes:
 *   base_logits [C, L, V] and block_hidden [C, L, H] in the head's dtype, anchor
 *   [C] int32, target [C, L, V] or [C, B+1, V] (rows) in the head's dtype. */
typedef struct dartree_host_session dartree_host_session;
typedef struct {
    const void* base_logits;
    const void* block_hidden;
    const int32_t* anchor;
    const void* target;
} dartree_host_inputs;
typedef struct {
    int32_t* accepted_len; /* [C] */
    int32_t* path;         /* [C, L] */
    int32_t* bonus;        /* [C] */
} dartree_host_outputs;
DARTREE_API int dartree_host_session_create(const dartree_head* head, const dartree_params* p, int rows,
                                            dartree_host_session** out);
DARTREE_API void dartree_host_session_destroy(dartree_host_session* s);
DARTREE_API int dartree_host_stage(dartree_host_session* s, const dartree_host_inputs* in);
DARTREE_API int dartree_host_round(dartree_host_session* s, const dartree_host_outputs* out, void* stream);
/* Bytes of one staged input (which: 0 base_logits, 1 block_hidden, 2 anchor,
 * 3 target); 0 for a null session or another index. */
DARTREE_API size_t dartree_host_input_bytes(const dartree_host_session* s, int which);

/* Baseline of the deferred search: node-by-node best-first drafting with one
 * correction-head evaluation per popped node ("heap pop -> correction"; DARTree
 * blog post, section 2, latency breakdown, and section 4.3, Table 2). After S1 and
 * the candidate-side projection (the same launches as dartree_build_tree), one CTA
 * per request pops B nodes one at a time from all children pushed so far, largest
 * score first (ties: shallower depth, then earlier push; a node's K children are
 * pushed in candidate order when it is popped), computes the popped node's state
 * and, below depth L, its K children's scores with the stand-in head. The root is
 * expanded first and is not counted. With W >= B the deferred tree holds the same
 * nodes (its per-depth top-W never drops a node the heap pops).
 *   p            C, L, K (<= 64), B (<= 256) and beta; W is not used
 *   head         bf16, prepared with dartree_head_prepare (W_q^T), H a multiple of
 *                128 and at most 6144
 *   tok, parent, depth, score  [C, B] in pop order: token, pop index of the parent
 *                (-1 = the root), depth (1..L), score s_beta
 *   ws           dartree_heap_workspace_bytes() bytes, 256-byte aligned
 * Returns DARTREE_EUNSUPPORTED outside these limits (nothing enqueued). */
DARTREE_API size_t dartree_heap_workspace_bytes(const dartree_params* p, int V, int H, int dtype);
DARTREE_API int dartree_heap_build(const dartree_head* head, const dartree_params* p, const void* base_logits,
                                   const void* block_hidden, const int32_t* anchor, int32_t* tok, int32_t* parent,
                                   int32_t* depth, float* score, void* ws, size_t ws_bytes, void* stream);

/* S10 without a workspace, for callers that cannot allocate device memory where
 * they verify (for example a serving loop whose caching allocator holds all free
 * HBM, or a plugin behind a plain C interface with no allocator handle). The
 * paper has no counterpart: this is a deployment variant of dartree_verify with
 * the same arguments, minus the workspace, and the same results.
 * Scratch is one file-scope device array of DARTREE_STATIC_VERIFY_BYTES bytes
 * (a 256-byte header + 8 bytes per target row key), kept by every GPU that loads the
 * library until the process exits. Limit: 256 + 8*C*max(L, B+1) bytes must fit,
 * else DARTREE_EUNSUPPORTED (before anything is enqueued). The first call on a
 * device looks up the array's device address with that device current (a
 * cudaGetSymbolAddress, no allocation); make that first call before any stream
 * capture. All calls share the one array and each starts by clearing what must
 * start at zero: calls that overlap on the GPU (other streams, other threads)
 * race on it and must be serialised by the caller. There is no status word the
 * caller can read, so a malformed tree (DARTREE_EINTERNAL for dartree_verify)
 * is not reported by this variant. Allocates nothing: no cudaMalloc, cudaFree
 * or allocating library call. */
#define DARTREE_STATIC_VERIFY_BYTES (256u * 1024u)
DARTREE_API int dartree_verify_static(const dartree_params* p, const dartree_tree* tree, const void* target,
                                      int rows, int V, int dtype, int32_t* accepted_len, int32_t* path,
                                      int32_t* bonus, void* stream);

/* Self-test of the bounded device-side waits (failure detection without a GPU
 * fault). The library's own wait helpers wait for something that is never
 * signalled: which = 0, an mbarrier phase that nothing completes; which = 1, a
 * grid barrier whose target counts one CTA more than the launch has. The wait
 * gives up after limit_us microseconds (1..1000000), records DARTREE_ETIMEOUT in
 * the status word at the start of ws (read it with dartree_read_status) and the
 * kernel returns; the context stays usable. ws: >= 512 bytes, 256-byte aligned
 * (its second 256-byte block holds the barrier counter). Returns DARTREE_OK once
 * enqueued, DARTREE_EINVAL for a bad `which` or limit. */
DARTREE_API int dartree_selftest_wait(void* ws, size_t ws_bytes, int which, unsigned limit_us, void* stream);

/* Per-kernel launch timing (profiling). dartree_timing(1) clears the records and
 * starts bracketing every library kernel launch with two CUDA events on the
 * launch's stream; dartree_timing(0) stops. dartree_timing_read synchronises the
 * recorded events of one kernel family and returns its launch count and summed
 * device time. Kernel ids 0..DARTREE_NUM_KERNEL_IDS-1, named by
 * dartree_kernel_name. Not for launches captured into a CUDA graph; adds two
 * event records per launch while on. */
#define DARTREE_NUM_KERNEL_IDS 15
DARTREE_API int dartree_timing(int enable);
DARTREE_API int dartree_timing_read(int kernel_id, int* launches, double* total_ms);
DARTREE_API const char* dartree_kernel_name(int kernel_id);

/* Building block exposed for testing: the tcgen05 GEMM used for the per-depth
 * parent projection. D[M,N] = A[M,K] . B[N,K]^T with A, B bf16 row-major (K
 * contiguous, 16-byte aligned, K a multiple of 8), D fp32 row-major; N must be a
 * multiple of 128 (else DARTREE_EUNSUPPORTED). `status` (device int, may be NULL)
 * receives DARTREE_ETIMEOUT if a bounded wait runs out. */
DARTREE_API int dartree_gemm_bf16(const void* A, const void* B, float* D, int M, int N, int K, int32_t* status,
                                  void* stream);

/* Copies the device status word of `ws` to *status (synchronises `stream`). */
DARTREE_API int dartree_read_status(const void* ws, int32_t* status, void* stream);

/* Resets the device status word of `ws` to DARTREE_OK (enqueued on `stream`). */
DARTREE_API int dartree_clear_status(void* ws, void* stream);

/* Static text for a status code. */
DARTREE_API const char* dartree_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* DARTREE_H */
