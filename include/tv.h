/*
 * tv.h: C ABI of the GB300 tree-verify library (one shared object,
 * libtreeverify.so).  One call per step of a speculative-decoding verify
 * round of a hybrid Gated DeltaNet + attention mixer stack, never one per
 * operator; activations stay on the device.
 *
 * Sources (page title, section):
 *  [TOUR]  "One request, end to end", 2.6 "The decode loop": the target
 *          verifies the whole draft tree in one forward pass through every
 *          layer, walks it with its own tokens, keeps the longest agreeing
 *          path plus one token of its own, and commits that path's KV rows
 *          and recurrent state.
 *  [LEAF]  "How ignis serves a request", "The shape of the process": the
 *          kernel leaf sits behind a flat C ABI named after its step
 *          granularity; nothing it computes crosses the ABI as a host pointer.
 *  [MODEL] "Adding a model", step 4 (hot verbs forward_tree, commit_tree,
 *          rollback_to): every verified row must equal the decode step's row
 *          bit for bit; "What is still specific to Qwen3.8": Gated DeltaNet
 *          heads of 128 by 128 and attention layers.
 *  [STATE] "Adding a model", "The model layer": per-sequence cache state is
 *          the recurrent state (copied whole) plus K and V views with a token
 *          axis sliced by length.
 *  [PAR]   "Parallel requests", "Joint verify": several sequences' trees in
 *          one pass, the mixers running per sequence.
 *  [POOL]  "Parallel requests", "The shared KV pool": whole windows reserved
 *          as address space, 2 MiB pages committed as rows are written.
 *
 * Conventions shared by every call
 *  - Ownership: the caller allocates and owns every buffer (device memory
 *    unless marked host).  The library allocates nothing in these calls and
 *    keeps no pointer after a call returns (the tv_kvpool_* calls, below, are
 *    the exception: an allocator the caller may use for its caches).  Verify inputs (k_t, v_t, k, v,
 *    alpha, beta) must stay alive until tv_commit_path has run on the stream.
 *  - Streams: every call only enqueues work on `stream` (a cudaStream_t; NULL
 *    is the legacy default stream) and never synchronises, so a whole round
 *    can be captured in a CUDA graph.
 *  - Errors: argument errors that the host can see return a tv_status
 *    immediately and enqueue nothing.  Errors only the device can see (a
 *    malformed tree, a cache that would overflow, a bounded wait that
 *    expired) write their tv_status code into the caller's device status word
 *    (first error wins) and make every later call that is given the same
 *    word a no-op.  The word belongs to a launch, not to one sequence: an
 *    error in any sequence of a joint launch stops the round for all of its
 *    sequences (a caller that wants the others to go on gives them their own
 *    tree descriptors and words, at the cost of one launch each).  Calls
 *    already running when the word is set may still finish their work.
 *    Nothing traps.
 *  - Node-indexed arrays concatenate the sequences' trees: sequence s owns
 *    global nodes node_off[s] .. node_off[s+1]-1, whose local index 0 is the
 *    root.  The root is the last committed token: it is not yet in the cache
 *    or in the state, and it is always accepted.
 *  - Rows: a tree node at depth d (root depth 0) sees the L committed cache
 *    rows plus its ancestors-or-self at logical positions L .. L+d, exactly
 *    where decoding them one by one would have put them.
 *  - Alignment: every device pointer 16-byte aligned.
 */
#ifndef TV_H
#define TV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tv_stream; /* same type as cudaStream_t */

#define TV_MAX_SEQ 8    /* sequences in one launch */
#define TV_MAX_NODES 64 /* nodes in one sequence's tree */
#define TV_MAX_PATH 16  /* nodes on a root path, root included */

typedef enum {
  TV_OK = 0,
  TV_ERR_ARG = 1,       /* null pointer, bad count or length bound */
  TV_ERR_SHAPE = 2,     /* unsupported head count / head dim combination */
  TV_ERR_DTYPE = 3,     /* unsupported element type */
  TV_ERR_ALIGN = 4,     /* pointer not 16-byte aligned */
  TV_ERR_TREE = 5,      /* device: malformed parent array or node offsets */
  TV_ERR_CAPACITY = 6,  /* device: a write past a cache's `cap` rows */
  TV_ERR_CUDA = 7,      /* a CUDA runtime call failed (launch, attribute) */
  TV_ERR_WORKSPACE = 8, /* workspace smaller than the *_workspace_bytes bound */
  TV_ERR_TIMEOUT = 9,   /* device: a bounded wait inside a kernel expired */
  TV_ERR_LEN = 10,      /* device: a sequence length above the host bound max_len */
  TV_ERR_SCRATCH = 11   /* host: request larger than the fixed scratch of tv_attn_tree_verify_static */
} tv_status;

typedef enum { TV_F32 = 0, TV_BF16 = 1 } tv_dtype;

/* Human-readable name of a status code (static string). */
const char* tv_status_string(tv_status s);
/* Library version string (static). */
const char* tv_version(void);

/* ------------------------------------------------------------------------
 * Draft trees
 * ------------------------------------------------------------------------
 * [TOUR] (the block drafter's chain merged with the lookup drafter's
 * branches into one tree).  A tree is a parent-index array in topological
 * order: parent[0] = -1 and 0 <= parent[i] < i (sequence-local indices),
 * 1..TV_MAX_NODES nodes, at most TV_MAX_PATH nodes on any root path.
 */
typedef struct {
  int32_t n_seq;           /* sequences, 1..TV_MAX_SEQ (host) */
  int32_t n_total;         /* nodes over all sequences (host) */
  int32_t n_max;           /* host bound on any one tree's size, 1..TV_MAX_NODES */
  const int32_t* node_off; /* device [n_seq+1], node_off[0] = 0, node_off[n_seq] = n_total */
  const int32_t* parent;   /* device [n_total], sequence-local parent, -1 at the root */
  void* meta;              /* device, tv_tree_meta_bytes() bytes: derived tables (private layout) */
  int32_t* status;         /* device [1] error word, 0 = ok; shared by the calls of a round */
  int32_t flags;           /* TV_TREE_* bits (host), 0 by default */
} tv_tree;

/* TV_TREE_OVERLAP: the calls that take this tree launch their kernels with
 * programmatic dependent launch, so that a kernel can start (shared- and
 * tensor-memory setup, loads of the recurrent state, work that needs nothing
 * from its predecessor) while the kernel before it on the stream finishes.
 * A kernel lets the next one in right after its own wait for its
 * predecessor has returned (the attention split and tail kernels, GDN
 * verify), or at exit, so everything older than the predecessor has
 * completed.  Before
 * waiting, a kernel reads only the recurrent states (GDN verify, which also
 * reads its sequence's node range from the tree tables to prefetch its node
 * inputs into L2, a cache hint clamped to the buffers; the fused GDN verify
 * copies its convolution weights; GDN commit, whose predecessor is always a
 * kernel of the same commit call, and which prefetches every node's key and
 * value rows into L2 from the tree tables' node range), the lengths
 * and node_off (attention; the split kernel also prefetches K/V tiles and
 * its first query rows into L2, which is only a cache hint), and the tree tables, the query rows, the
 * tree's K/V rows and the cache rows of its own segment (the attention tail,
 * whose predecessor is always its own split kernel, and which computes the
 * node's own segment before waiting); no kernel of a verify round (prepare,
 * per-layer verify, accept, commit, in that order on one stream) writes
 * these directly before such a read.  The caller must not enqueue its own
 * kernel that writes them directly before a call with this flag. */
#define TV_TREE_OVERLAP 1
/* Every call that takes a tv_tree returns TV_ERR_ARG, enqueueing nothing, when
 * the descriptor is ill formed on the host: NULL, counts out of range, or a
 * NULL or non-16-byte-aligned pointer field. */

/* Bytes of the `meta` buffer for a launch of n_total nodes. */
size_t tv_tree_meta_bytes(int32_t n_seq, int32_t n_total);

/* Validate the trees and derive, into tree->meta, each node's depth,
 * ancestor-or-self bitmask, ancestor at every depth, and the traversal order
 * the recurrent layers use.  Must run (stream-ordered) before any call that
 * takes the tree.  A malformed tree sets TV_ERR_TREE in *tree->status. */
tv_status tv_tree_prepare(const tv_tree* tree, tv_stream stream);

/* ------------------------------------------------------------------------
 * Attention: tree-masked grouped-query attention over the KV cache
 * ------------------------------------------------------------------------
 * [TOUR], [MODEL].  For every node i and query head h (KV head
 * g = h / (Hq/Hkv)):
 *     out[i,h] = sum_p softmax_p(scale * q[i,h] . key_p) value_p
 * over the L context rows of the cache and the ancestors-or-self of i.
 */
typedef struct {
  tv_dtype dtype; /* element type of cache, q, k_t, v_t and out: TV_BF16 (tensor-core
                     path, D in {64,128,256}) or TV_F32 (CUDA-core path, D in {64,128,256}) */
  int32_t Hq, Hkv, D; /* Hq % Hkv == 0, Hq/Hkv <= 128 */
  int32_t cap;        /* rows per KV head of every cache */
  void* const* K;     /* host array [n_seq] of device pointers, each [Hkv][cap][D] */
  void* const* V;     /* same layout as K */
} tv_attn_layer;

/* Fixed per model and shared by verify and decode: the positions of one KV
 * split (a multiple of 64).  The split structure is part of the row function,
 * so verify rows equal decode rows bit for bit only under the same plan. */
typedef struct {
  int32_t split;
} tv_plan;

/* Device scratch bytes needed by tv_attn_tree_verify / tv_decode_step for
 * this layer shape, n_seq sequences of at most n_max nodes and contexts of at
 * most max_len rows.  0 for the TV_F32 path. */
size_t tv_attn_workspace_bytes(const tv_plan* plan, const tv_attn_layer* layer, int32_t n_seq,
                               int32_t n_max, int32_t max_len);

/* Verify every tree node of every sequence for one attention layer.
 *  len       device [n_seq]: committed rows L_s (read only)
 *  max_len   host bound, >= every L_s (sizes the launch; a larger L_s sets TV_ERR_LEN)
 *  q         [n_total][Hq][D]; k_t, v_t [n_total][Hkv][D]: the nodes' own rows
 *  out       [n_total][Hq][D]
 *  scale     score scale (D^-1/2 for standard attention)
 *  workspace device scratch of at least tv_attn_workspace_bytes() bytes
 * The cache is read only; the tree rows enter it only through tv_commit_path,
 * so rolling back a rejected tree costs nothing. */
tv_status tv_attn_tree_verify(const tv_plan* plan, const tv_attn_layer* layer, const tv_tree* tree,
                              const int32_t* len, int32_t max_len, const void* q, const void* k_t,
                              const void* v_t, void* out, float scale, void* workspace,
                              size_t workspace_bytes, tv_stream stream);

/* Size of the fixed device scratch array behind tv_attn_tree_verify_static. */
#define TV_STATIC_SCRATCH_BYTES ((size_t)48 << 20)
size_t tv_attn_static_scratch_bytes(void);

/* tv_attn_tree_verify without a workspace argument: the per-split partial
 * states go to a fixed 48 MiB array of device memory inside the library (one
 * per device), so the call allocates nothing and needs no scratch from the
 * caller.  The pages have no counterpart; it serves callers that cannot hand
 * over device scratch: a C or foreign-language host that links only this
 * library and has no device allocator of its own, and a caller whose memory
 * plan is fixed before the round starts and must not take a cudaMalloc in the
 * middle of it (cudaMalloc can synchronise the device and stall other
 * streams).
 *  Arguments, layout and results: exactly those of tv_attn_tree_verify.
 *  Limit: requests whose tv_attn_workspace_bytes(plan, layer, tree->n_seq,
 *    tree->n_max, max_len) exceeds TV_STATIC_SCRATCH_BYTES return
 *    TV_ERR_SCRATCH before anything is enqueued.
 *  Errors: TV_ERR_ARG for a NULL or ill-formed tree descriptor or a negative
 *    max_len (checked before the size), then everything tv_attn_tree_verify
 *    returns.
 *  Setup: the first call on each device looks up the array's device address
 *    (this loads the module); make that first call before any stream capture.
 *    The address is cached per device and looked up again when the device's
 *    context changes (after cudaDeviceReset), so the first call after a reset
 *    must also come before any capture.
 *  Start values: none needed; every scratch record a call reads was written
 *    earlier in the same call.
 *  Concurrency: all calls on one device share the one array, so two calls
 *    whose work can overlap (different streams, or different host threads
 *    without ordering) race on it and give wrong results.  Calls ordered on
 *    one stream are safe. */
tv_status tv_attn_tree_verify_static(const tv_plan* plan, const tv_attn_layer* layer, const tv_tree* tree,
                                     const int32_t* len, int32_t max_len, const void* q, const void* k_t,
                                     const void* v_t, void* out, float scale, tv_stream stream);

/* ------------------------------------------------------------------------
 * Attention front end: partial rotary embedding and the gated output
 * ------------------------------------------------------------------------
 * "Adding a model", "What is still specific to Qwen3.8": the model's
 * attention has a gated output and partial rotary.  The pages give neither
 * formula; the library takes the plainest reading:
 *   rotary: the first rot_dims dimensions of every query and key head turn
 *     as rot_dims/2 planes, plane j pairing dimension j with j + rot_dims/2
 *     and turning by pos * theta^(-2j/rot_dims); the rest pass through;
 *   position: a tree node at depth d sits at L + d, where decoding its root
 *     path would put it (a decode token at L), so the key rows a commit
 *     copies into the cache are rotated at their final positions;
 *   gate: out = attention * sigmoid(gate), elementwise over [Hq][D].
 * A row's bits depend only on its own inputs and position, so verified rows
 * still equal decoded rows bit for bit. */

/* Rotate the rows of one attention layer's queries and keys.
 *  tree      verify: every node of the tree, at len[s] + depth(i); the
 *            tree's status word receives device errors (n_seq, status unused)
 *            or NULL: decode, one token per sequence at len[s] (n_seq tokens,
 *            errors to *status)
 *  len       device [n_seq] committed rows; max_len host bound (a larger
 *            length sets TV_ERR_LEN and leaves the row unwritten)
 *  q_raw     [rows][Hq][D], k_raw [rows][Hkv][D] in the layer's dtype;
 *  q, k      outputs of the same shapes (may alias q_raw, k_raw)
 *  rot_dims  even, 0 <= rot_dims <= D; theta > 1 finite
 * Values need no rotation: pass the projection's values as v_t.
 * Host-checkable errors return without enqueueing anything. */
tv_status tv_attn_rope(const tv_attn_layer* layer, const tv_tree* tree, int32_t n_seq, const int32_t* len,
                       int32_t max_len, int32_t rot_dims, float theta, const void* q_raw, const void* k_raw,
                       void* q, void* k, int32_t* status, tv_stream stream);

/* tv_attn_tree_verify with the output gate applied in the same kernel:
 * out[i,h,:] = attention row * sigmoid(gate[i,h,:]); gate [n_total][Hq][D]
 * in the layer's dtype, 16-byte aligned.  Other arguments as there. */
tv_status tv_attn_tree_verify_gated(const tv_plan* plan, const tv_attn_layer* layer, const tv_tree* tree,
                                    const int32_t* len, int32_t max_len, const void* q, const void* k_t,
                                    const void* v_t, const void* gate, void* out, float scale, void* workspace,
                                    size_t workspace_bytes, tv_stream stream);

/* The attention half of tv_decode_step with the output gate applied in the
 * same kernel (gate [n_seq][Hq][D]); appends each token's k, v at row len[s]. */
tv_status tv_attn_decode_gated(const tv_plan* plan, const tv_attn_layer* attn, int32_t n_seq, const int32_t* len,
                               int32_t max_len, const void* q, const void* k, const void* v, const void* gate,
                               void* out, float scale, void* workspace, size_t workspace_bytes, int32_t* status,
                               tv_stream stream);

/* ------------------------------------------------------------------------
 * Gated DeltaNet: the gated delta rule along every node's ancestor path
 * ------------------------------------------------------------------------
 * [MODEL].  For value head h (key head g = h / (Hv/Hk)) and node i, with
 * S_{par(root)} = S (the committed state):
 *     S_i = alpha_i S_{par(i)} (I - beta_i k_i k_i^T) + beta_i v_i k_i^T
 *     out[i,h] = scale * S_i q_i
 * No per-node state is written to memory.
 */
typedef struct {
  tv_dtype dtype;         /* element type of q, k, v and out (TV_BF16 or TV_F32) */
  int32_t Hk, Hv, dk, dv; /* Hv % Hk == 0, dk in {64,128}, dv <= 256 */
  float* const* S;        /* host array [n_seq] of device pointers, each fp32 [Hv][dv][dk] */
} tv_gdn_layer;

/*  q, k  [n_total][Hk][dk]; v [n_total][Hv][dv]; alpha, beta fp32 [n_total][Hv]
 *  out   [n_total][Hv][dv]
 *  scale output scale (dk^-1/2 by default).  The state is read only. */
tv_status tv_gdn_tree_verify(const tv_gdn_layer* layer, const tv_tree* tree, const void* q,
                             const void* k, const void* v, const float* alpha, const float* beta,
                             void* out, float scale, tv_stream stream);

/* ------------------------------------------------------------------------
 * Gated DeltaNet front end and gated output norm
 * ------------------------------------------------------------------------
 * "Adding a model", "What is still specific to Qwen3.8": the Gated DeltaNet
 * layer with its gated norm; "The model layer": the per-sequence state
 * includes the convolution tails.  The pages give no formula; the library
 * takes the plainest reading:
 *   channels: the raw query, key and value projections side by side,
 *     C = 2 Hk dk + Hv dv per token;
 *   short convolution: depthwise and causal, width W; a token's output at
 *     channel c is sum_j wconv[c][j] x[t - (W-1) + j][c] over its root path,
 *     continuing past the root into the committed tail; then SiLU;
 *   q, k: divided per head by sqrt(sum of squares + 1e-6);
 *   gates: beta = sigmoid(b_raw), alpha = exp(-softplus(a_raw));
 *   output: o / sqrt(mean(o^2) + 1e-6) * w_norm * SiLU(z).
 * Values are formed in fp32 in a fixed order, so verified rows equal decoded
 * rows bit for bit. */
typedef struct {
  tv_dtype dtype;      /* x, tails, q/k/v, o, z, out: TV_BF16 or TV_F32 */
  int32_t Hk, Hv, dk, dv; /* dk = dv in {64, 128} */
  int32_t width;       /* convolution width W, 1..8 */
  const float* wconv;  /* device [C][W] fp32 */
  void* const* tail;   /* host array [n_seq] of device pointers, each [W-1][C]: the
                          last W-1 committed raw inputs, oldest first (unused if W = 1) */
} tv_gdn_front_layer;

/* Convolution, SiLU, q/k norm and gates for every tree node (tree) or one
 * decode token per sequence (tree NULL: n_seq tokens, errors to *status).
 *  x      [rows][C] raw projections (layer dtype)
 *  a_raw, b_raw [rows][Hv] fp32
 *  q, k   [rows][Hk][dk]; v [rows][Hv][dv] (layer dtype); alpha, beta [rows][Hv] fp32:
 *         the inputs of tv_gdn_tree_verify / tv_decode_step.
 * The tails are read only. */
tv_status tv_gdn_front(const tv_gdn_front_layer* layer, const tv_tree* tree, int32_t n_seq, const void* x,
                       const float* a_raw, const float* b_raw, void* q, void* k, void* v, float* alpha,
                       float* beta, int32_t* status, tv_stream stream);

/* Gated RMS norm of rows outputs [rows][Hv][dv]: out = o / rms(o) * w_norm * SiLU(z);
 * o, z, out in the layer dtype (out may alias o); w_norm [dv] fp32. */
tv_status tv_gdn_out_norm(const tv_gdn_front_layer* layer, int32_t rows, const void* o, const void* z,
                          const float* w_norm, void* out, tv_stream stream);

/* tv_gdn_front, tv_gdn_tree_verify and tv_gdn_out_norm in one launch: the
 * verify kernel forms each node's query, key, value and gates from the raw
 * projections inside its staging (no q, k, v, alpha or beta in memory), runs
 * the recurrence and applies the gated norm to its outputs.  The CTAs that
 * share a key head run as one thread-block cluster: they split the key head's
 * queries and keys by node and exchange them, and gather each (node, value
 * head)'s dv outputs for the norm, through distributed shared memory.  Where
 * no such cluster fits (more than 16 CTAs to a key head, or the shared memory
 * of the gather) the norm runs as a second kernel over out.  The result
 * equals the three calls bit for bit.
 *  layer  tv_gdn_tree_verify's layer (states read only, as there)
 *  front  the front-end layer: same dtype, Hk, Hv, dk, dv; wconv and each
 *         tail 16-byte aligned
 *  x [n_total][C], a_raw, b_raw [n_total][Hv], z [n_total][Hv][dv], w_norm [dv]
 *         (x, z, w_norm 16-byte aligned)
 *  out    [n_total][Hv][dv], 16-byte aligned
 * Errors as tv_gdn_tree_verify's and tv_gdn_front's; TV_ERR_SHAPE when the two
 * layers disagree, TV_ERR_ALIGN for a misaligned buffer.  The tails are read
 * only. */
tv_status tv_gdn_tree_verify_fused(const tv_gdn_layer* layer, const tv_gdn_front_layer* front, const tv_tree* tree,
                                   const void* x, const float* a_raw, const float* b_raw, const void* z,
                                   const float* w_norm, void* out, float scale, tv_stream stream);

/* The decode counterpart of tv_gdn_tree_verify_fused: tv_gdn_front (one token
 * a sequence), the GDN half of tv_decode_step and tv_gdn_out_norm in one
 * launch, one CTA per (value head, sequence).  The states advance in place
 * as tv_decode_step advances them; the result and the states equal the three
 * calls' bit for bit, so a row verified by tv_gdn_tree_verify_fused equals
 * the same token decoded here.
 *  x [n_seq][C], a_raw, b_raw [n_seq][Hv], z [n_seq][Hv][dv], w_norm [dv];
 *  out [n_seq][Hv][dv]; errors go to *status (16-byte aligned), and a call
 *  given a status word that holds an error does nothing.
 * The tails are read only: run tv_gdn_conv_commit (tree NULL) afterwards. */
tv_status tv_gdn_decode_fused(const tv_gdn_layer* layer, const tv_gdn_front_layer* front, int32_t n_seq,
                              const void* x, const float* a_raw, const float* b_raw, const void* z,
                              const float* w_norm, void* out, float scale, int32_t* status, tv_stream stream);

/* Commit of the convolution tails: each sequence's tail becomes the last W-1
 * of (tail, x[path[0..a-1]]) for the accepted path of tv_accept_path (tree),
 * or of (tail, x[s]) for a decoded token (tree NULL, n_seq tokens).  Run it
 * after every call that reads the tails for this round. */
tv_status tv_gdn_conv_commit(const tv_gdn_front_layer* layer, const tv_tree* tree, int32_t n_seq, const void* x,
                             const int32_t* path, const int32_t* acc_len, int32_t* status, tv_stream stream);

/* ------------------------------------------------------------------------
 * Accept walk: longest agreeing path plus one token
 * ------------------------------------------------------------------------
 * [TOUR].  A node agrees when every node on its root path below the root
 * carries the token the target chose greedily at that node's parent.  The
 * accepted path is the root path of the deepest agreeing node (lowest local
 * index among equally deep ones); the bonus token is the target's greedy
 * token at the path's last node (it becomes the next round's root).
 *  tok, greedy device [n_total] int32: each node's draft token / the target's argmax after it
 *  path        device [n_seq][TV_MAX_PATH] out: local node indices, root first, -1 padded
 *  acc_len     device [n_seq] out: accepted path length a (1..TV_MAX_PATH, root included)
 *  bonus       device [n_seq] out */
tv_status tv_accept_path(const tv_tree* tree, const int32_t* tok, const int32_t* greedy,
                         int32_t* path, int32_t* acc_len, int32_t* bonus, tv_stream stream);

/* ------------------------------------------------------------------------
 * Commit the accepted path into every layer's cache state
 * ------------------------------------------------------------------------
 * [TOUR], [MODEL] commit_tree, [STATE].  For every sequence s with
 * a = acc_len[s] and L = len[s]:
 *   attention layer l: rows L..L+a-1 of K_l[s], V_l[s] <- k_t[l], v_t[l] rows of
 *     the path's nodes (bit copies);
 *   GDN layer l: S_l[s] <- S_l[s] advanced along the path with the same step
 *     function tv_gdn_tree_verify and tv_decode_step use;
 *   then len[s] += a.
 * k_t, v_t, k, v, alpha, beta are host arrays (one device pointer per layer)
 * of the same buffers that layer's verify call read.  A sequence with
 * L + a > cap sets TV_ERR_CAPACITY and commits nothing. */
tv_status tv_commit_path(const tv_tree* tree, const int32_t* path, const int32_t* acc_len,
                         int32_t n_attn, const tv_attn_layer* attn, const void* const* k_t,
                         const void* const* v_t, int32_t n_gdn, const tv_gdn_layer* gdn,
                         const void* const* k, const void* const* v, const float* const* alpha,
                         const float* const* beta, int32_t* len, tv_stream stream);

/* ------------------------------------------------------------------------
 * Single-token decode (the row every verified row must equal)
 * ------------------------------------------------------------------------
 * [MODEL] step 4 and its load-time self-check.  One token per sequence for
 * exactly one layer (attn XOR gdn non-NULL), run through the same tiles,
 * splits and step function as verify:
 *   attention: writes the token's k, v at row len[s] of the cache and attends
 *     over rows 0..len[s]; q [n_seq][Hq][D], k, v [n_seq][Hkv][D];
 *     workspace as for tv_attn_tree_verify with n_max = 1.
 *   GDN: S <- step(S) in place and out = scale * S q; q, k [n_seq][Hk][dk],
 *     v [n_seq][Hv][dv], alpha, beta [n_seq][Hv].
 * len is not advanced here: after the last layer of a token call
 * tv_len_advance.  status: device error word (as in tv_tree). */
tv_status tv_decode_step(const tv_plan* plan, const tv_attn_layer* attn, const tv_gdn_layer* gdn,
                         int32_t n_seq, const int32_t* len, int32_t max_len, const void* q,
                         const void* k, const void* v, const float* alpha, const float* beta,
                         void* out, float scale, void* workspace, size_t workspace_bytes,
                         int32_t* status, tv_stream stream);

/* len[s] += by[s] (device [n_seq]) if `by` is non-NULL, else len[s] += inc. */
tv_status tv_len_advance(int32_t* len, const int32_t* by, int32_t inc, int32_t n_seq,
                         tv_stream stream);

/* ------------------------------------------------------------------------
 * KV pool: address space reserved for a whole window, pages committed as
 * rows are written
 * ------------------------------------------------------------------------
 * [POOL] "Parallel requests", "The shared KV pool": each KV tensor's full
 * size is reserved as virtual addresses and physical pages are mapped only
 * for the rows a sequence writes; the tensor keeps the static buffer's shape,
 * dtype and strides, so every call above, every view and every captured CUDA
 * graph is unchanged and the results are the same bits by construction.
 * Commit rows (plus a margin) before a round writes them; a fresh page is
 * zeroed; pages wholly past the rows a sequence still holds can be given back.
 *
 * These are the library's only allocating calls.  They are host calls made
 * between rounds (mapping is not a stream operation and cannot be captured);
 * a pool is internally locked, so threads may share one.  The caller must
 * not release or destroy pages that queued work still reads or writes.
 *
 * A tensor laid out as n_heads blocks of `head_stride` bytes, each holding
 * rows of `row_bytes` (a cache [Hkv][cap][D] has head_stride = cap * D * esize
 * and row_bytes = D * esize), is reserved as one range of
 * n_heads * head_stride bytes rounded up to whole pages. */
typedef struct tv_kv_pool tv_kv_pool; /* opaque */

/* Physical page size the pool would use on `device` for a request of
 * page_bytes (0: 2 MiB), rounded up to the device's allocation granularity;
 * 0 when the device does not support virtual memory management. */
size_t tv_kvpool_page_bytes(int32_t device, size_t page_bytes);

/* New pool for `device` (host call, no stream work).  *pool receives the
 * handle.  TV_ERR_ARG for a NULL out pointer, TV_ERR_CUDA when the device
 * or driver lacks virtual memory management. */
tv_status tv_kvpool_create(int32_t device, size_t page_bytes, tv_kv_pool** pool);

/* Reserve address space for one tensor of `bytes` (rounded up to pages) and
 * return its base in *base (aligned to a page).  Nothing is mapped yet: the
 * device must not touch a row before it is committed. */
tv_status tv_kvpool_reserve(tv_kv_pool* pool, size_t bytes, void** base);

/* Map and zero (on `stream`, ordered before later work on it) the pages that
 * hold rows [0, rows) of every head of the tensor reserved at `base`; pages
 * already mapped are left as they are.  TV_ERR_ARG for an unknown base or a
 * row range outside the reservation, TV_ERR_CAPACITY when the device is out
 * of memory (the pages mapped so far stay mapped). */
tv_status tv_kvpool_commit_rows(tv_kv_pool* pool, void* base, int32_t n_heads, size_t head_stride,
                                size_t row_bytes, int64_t rows, tv_stream stream);

/* Give back the pages of the tensor at `base` that hold no row below
 * `keep_rows` of any head. */
tv_status tv_kvpool_release_rows(tv_kv_pool* pool, void* base, int32_t n_heads, size_t head_stride,
                                 size_t row_bytes, int64_t keep_rows);

/* Bytes of physical pages mapped, and of address space reserved, by the pool. */
size_t tv_kvpool_committed_bytes(const tv_kv_pool* pool);
size_t tv_kvpool_reserved_bytes(const tv_kv_pool* pool);

/* Unmap and free every page and reservation of the pool, then the pool. */
tv_status tv_kvpool_destroy(tv_kv_pool* pool);

/* ------------------------------------------------------------------------
 * Diagnostics
 * ------------------------------------------------------------------------
 * Every wait inside the pipelined kernel (the attention split kernel) is
 * bounded: after a limit it raises a give-up flag the other
 * roles see, lets its own copies land, and the kernel writes TV_ERR_TIMEOUT
 * into the status word instead of hanging.  This call runs those same wait
 * routines against barriers that nothing arrives at, with a caller-chosen
 * limit, so that the give-up path can be checked on a device without
 * faulting or hanging it.  One CTA; the pages have no counterpart (the
 * load-time self-check of "Adding a model", step 4, is the nearest).
 *  status  device [1] word: TV_ERR_TIMEOUT is written when a wait gave up
 *  result  device int32 [4]: 1 = the wait succeeded, 0 = it gave up, for
 *          [0] a barrier that has completed (expect 1), [1] the warp-wide
 *          wait, [2] the single-thread wait, [3] the plain wait on barriers
 *          that never complete (expect 0 each)
 *  limit_cycles  1 .. 2^31 SM clocks per wait (the kernels use 2^31) */
tv_status tv_wait_selftest(int32_t* status, int32_t* result, int64_t limit_cycles, tv_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TV_H */
