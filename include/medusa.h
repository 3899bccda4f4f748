/*
 * medusa.h -- C ABI of the Medusa draft-and-verify decode step on one GPU (sm_103a).
 *
 * One call of medusa_step() performs a full decode step for B independent sequences:
 *   (1) the K residual SiLU heads and the LM head on the last hidden state h_t, with a
 *       top-s_k per head and the greedy root token,
 *   (2) the packed candidate tree (tokens, depth position ids, ancestor bitmask, paths),
 *   (3) tree attention of every node over the KV prefix plus its own ancestors, through
 *       one synthetic attention layer standing in for the backbone,
 *   (4) verification logits, greedy or typical acceptance, longest accepted path,
 *   (5) KV-cache compaction to the accepted path, and the carried state for the next step.
 * Sources (cited below by tag):
 *   [MEDUSA]  "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
 *             Heads" (structured summary of arXiv 2401.10774), Section 3.
 *   [NOTES]   "Accelerating LLM Inference with Speculative Decoding: Notes on Medusa".
 *   [READING] "MEDUSA 精读", sections 3, 4 and 6.
 *
 * Conventions (every entry point):
 *   - Pointers marked "device" are CUDA device pointers owned by the caller; "host" are
 *     host pointers owned by the caller.  The library allocates no device memory per call:
 *     scratch comes from the caller's workspace (medusa_workspace_size()).  Only
 *     medusa_plan_create() allocates (the uploaded tree spec and a status word) and
 *     medusa_plan_destroy() frees it.
 *   - Matrices are row-major [out][in]: a projection R^in -> R^out is stored out rows of
 *     in contiguous elements.  "dtype" elements are float (MEDUSA_F32) or bfloat16
 *     (MEDUSA_BF16) as the plan says; hidden states and every float output are float32.
 *   - `stream` is a cudaStream_t passed as void*.  Calls only enqueue work on it: they do
 *     not synchronise and may return before the GPU has finished.
 *   - Argument, shape and alignment errors are detected on the host before anything is
 *     launched and return MEDUSA_ERR_INVALID / MEDUSA_ERR_UNSUPPORTED.  Anomalies only the
 *     GPU can see (a KV length past capacity, a page id out of range, non-finite logits)
 *     set bits of the plan's device status word (MEDUSA_FLAG_*) and never trap; read them
 *     with medusa_get_status().  Launch failures return MEDUSA_ERR_CUDA.
 *   - Calls on one plan may run on different streams only if the caller orders them;
 *     concurrent calls must use distinct workspaces.
 */
#ifndef MEDUSA_H_
#define MEDUSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MEDUSA_MAX_HEADS 8     /* K <= 8 Medusa heads ([MEDUSA] §3.4: five suffice) */
#define MEDUSA_MAX_TOPS 16     /* s_k <= 16 candidates per head */
#define MEDUSA_MAX_NODES 256   /* N + 1 <= 256 packed tree nodes (root included) */
#define MEDUSA_MAX_LAYERS 1024 /* backbone layers of medusa_step_layers */

typedef enum {
  MEDUSA_OK = 0,
  MEDUSA_ERR_INVALID = -1,      /* bad argument, shape, tree spec or pointer alignment */
  MEDUSA_ERR_UNSUPPORTED = -2,  /* valid but outside the built kernels' limits */
  MEDUSA_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
  MEDUSA_ERR_DEVICE = -4,       /* medusa_get_status(): the device status word is set */
  MEDUSA_ERR_WORKSPACE = -6     /* workspace NULL or smaller than medusa_workspace_size */
} medusa_status;

enum { MEDUSA_F32 = 0, MEDUSA_BF16 = 1 };
enum { MEDUSA_GREEDY = 0, MEDUSA_TYPICAL = 1, MEDUSA_REJECT = 2 };

/* device status word bits */
#define MEDUSA_FLAG_TOKEN_RANGE 0x1u  /* a selected token id fell outside [0, V) */
#define MEDUSA_FLAG_KV_CAPACITY 0x2u  /* len + tree/path length would exceed capacity */
#define MEDUSA_FLAG_PAGE_RANGE  0x4u  /* a page-table entry fell outside [0, num_pages) */
#define MEDUSA_FLAG_NONFINITE   0x8u  /* a logit or softmax statistic was NaN or Inf */
#define MEDUSA_FLAG_TIMEOUT     0x10u /* a bounded wait in a pipelined kernel expired */

typedef struct medusa_plan medusa_plan;   /* opaque */

/* Model and batch sizes. */
typedef struct {
  int B;            /* sequences */
  int d;            /* hidden size */
  int V;            /* vocabulary */
  int K;            /* Medusa heads, 1..MEDUSA_MAX_HEADS */
  int Hq, Hkv, dh;  /* query heads, key/value heads (Hq % Hkv == 0), head dim */
  int dtype;        /* MEDUSA_F32 or MEDUSA_BF16: weights, embedding and KV cache */
  float rope_base;  /* rotary base (10000 for Llama) */
  int capacity;     /* KV slots per sequence */
  int page_size;    /* 0: contiguous cache; > 0: tokens per page */
  int num_pages;    /* paged cache: pages in the pool (bounds for page-table entries) */
} medusa_dims;

/* Packed candidate tree ([MEDUSA] §3.4 Tree Attention, Steps 1-2; [READING] section 6).
 * Node 0 is the root (the LM head's greedy token).  Node n >= 1 takes the rank[n]-th
 * best token of head depth(n); parent[n] < n.  depth(n) = depth(parent[n]) + 1 <= K. */
typedef struct {
  int K;                           /* heads the tree draws on */
  int s[MEDUSA_MAX_HEADS];         /* top-s_k per head, 1..MEDUSA_MAX_TOPS */
  int N;                           /* candidate nodes, root excluded */
  const int32_t* parent;           /* host [N+1], parent[0] = -1 */
  const int32_t* rank;             /* host [N+1], rank[0] = 0, rank[n] < s[depth(n)-1] */
} medusa_tree_spec;

/* Weights (device, dtype elements, row-major [out][in]). */
typedef struct {
  const void* w1;   /* [K][d][d]   head k's first projection ([MEDUSA] §3.4 head eq.) */
  const void* w2;   /* [K][V][d]   head k's vocabulary projection */
  const void* lm;   /* [V][d]      LM head */
  const void* emb;  /* [V][d]      token embedding of the synthetic layer */
  const void* wq;   /* [Hq*dh][d]  query projection */
  const void* wk;   /* [Hkv*dh][d] key projection */
  const void* wv;   /* [Hkv*dh][d] value projection */
  const void* wo;   /* [d][Hq*dh]  output projection */
} medusa_weights;

/* KV cache (device).  Contiguous: k, v each [B][capacity][Hkv][dh].  Paged: k, v each
 * [num_pages][page_size][Hkv][dh] and page_table [B][capacity/page_size]; slot t of
 * sequence b is row t % page_size of page page_table[b][t / page_size].  Keys are stored
 * after RoPE. */
typedef struct {
  void* k;
  void* v;
  const int32_t* page_table;  /* device, NULL for a contiguous cache */
  const int32_t* len;         /* device [B] prefix lengths at the start of the step */
  int32_t* len_out;           /* device [B] lengths after compaction (may alias len) */
} medusa_kv;

/* Acceptance rule ([MEDUSA] §3.4 Typical Acceptance Scheme and the speculative-decoding
 * rejection rule it replaces).
 *   MEDUSA_GREEDY   a candidate is kept iff it is its parent's greedy token.
 *   MEDUSA_TYPICAL  kept iff p(x) > min(eps, delta * exp(-H(p))), p = softmax(z / T).
 *   MEDUSA_REJECT   rejection sampling with the heads' top-s tokens as point-mass drafts:
 *                   from the root, the current node's children are tried in rank order,
 *                   child x kept iff u < p(x) / R (R = probability mass not yet rejected
 *                   at this node, 1 at first), else R -= p(x); the first kept child becomes
 *                   the current node.  Where no child is kept, the next step's root is
 *                   drawn from p at the current node without the rejected tokens (the
 *                   smallest token whose cumulative weight exceeds u_final times the
 *                   remaining total).  The emitted tokens are then distributed as p.
 *                   uniforms: device [B][1 + 16 K] floats in [0, 1): [b][0] = u_final,
 *                   [b][1 + 16 (d - 1) + j] = u of the j-th child tried at depth d.  A new
 *                   set is needed for every step, so the decode loop rejects this mode.
 * Temperature 0 is greedy in every mode. */
typedef struct {
  int mode;           /* MEDUSA_GREEDY, MEDUSA_TYPICAL or MEDUSA_REJECT */
  float temperature;  /* typical / reject: softmax temperature; 0 means greedy */
  float eps;          /* typical: hard threshold epsilon */
  float delta;        /* typical: entropy-threshold multiplier delta */
  const float* uniforms;  /* reject: see above; unused (may be NULL) otherwise */
} medusa_accept;

/* Step outputs (device). */
typedef struct {
  int32_t* out_tok;     /* [B][K+1] root then accepted tokens, -1 past n_acc */
  int32_t* n_acc;       /* [B] kept tokens = 1 + accepted candidates */
  int32_t* path_nodes;  /* [B][K+1] packed indices of the kept nodes, -1 padded */
  float* h_next;        /* [B][d] hidden state at the last kept node (next h_t) */
  int32_t* root_next;   /* [B] greedy token at the last kept node (next root) */
} medusa_outputs;

/* ------------------------------------------------------------------ plan */
/* Validates dims and the tree spec, uploads the spec and allocates the status word.
 * Returns MEDUSA_ERR_INVALID for inconsistent sizes or a malformed tree (parent >= own
 * index, depth > K, rank >= s), MEDUSA_ERR_UNSUPPORTED past the kernels' limits
 * (N+1 > 256, s_k > 16, K > 8, dh not in {32, 64, 128}, d or Hq*dh not a multiple
 * of 64 for bf16). */
medusa_status medusa_plan_create(const medusa_dims* dims, const medusa_tree_spec* tree,
                                 medusa_plan** out);
void medusa_plan_destroy(medusa_plan* plan);
/* Bytes of device workspace one medusa_step (or any stage call) needs. */
size_t medusa_workspace_size(const medusa_plan* plan);
/* Synchronises `stream`, returns the device status word in *flags and clears it.
 * MEDUSA_ERR_DEVICE when a flag was set, MEDUSA_OK otherwise. */
medusa_status medusa_get_status(const medusa_plan* plan, void* stream, uint32_t* flags);
/* Failure-path testing (the pages have no counterpart): the next verification-logit GEMM
 * this plan launches (in medusa_step, medusa_step_layers, medusa_verify_logits or a
 * decode loop captured after this call) has its MMA thread first wait, for at most `ns`
 * nanoseconds, on a barrier that nothing arrives on.  The wait runs out and the kernel
 * takes the path of a wait on a copy that never landed: it sets MEDUSA_FLAG_TIMEOUT,
 * lets its other waits run to their own ~1 s limits, drains its copies in flight, frees
 * its tensor memory and returns, so the call's outputs are meaningless but the CUDA
 * context stays usable.  One-shot: the setting is cleared when that GEMM is launched.
 * MEDUSA_ERR_INVALID for ns = 0 or above 10 s; MEDUSA_ERR_UNSUPPORTED for plans without
 * the tensor-core projections (fp32). */
medusa_status medusa_plan_expire_wait_once(medusa_plan* plan, unsigned long long ns);

/* ------------------------------------------------------------------ full step */
/* One decode step ([MEDUSA] §3.2 information flow, steps (2)-(6); [READING] section 3).
 * h: device [B][d] last hidden state.  root_in: device [B] first token carried from the
 * previous step's root_next, or NULL to take the LM head's greedy token on h.  With
 * root_in given the LM head is not applied to h (it would only yield the root), so a
 * step of the steady-state decode loop reads the LM head once, for verification.
 * out->h_next may alias h and out->root_next may alias root_in: both inputs are read
 * before the step writes its outputs. */
medusa_status medusa_step(const medusa_plan* plan, const float* h, const int32_t* root_in,
                          const medusa_weights* w, const medusa_kv* kv, medusa_accept acc,
                          const medusa_outputs* out, void* workspace, size_t ws_bytes,
                          void* stream);

/* ---- multi-layer backbone
 * The tree nodes pass through n synthetic layers instead of one, the way a real
 * backbone's per-layer calls would ([MEDUSA] §3.4 Tree Attention: every layer attends
 * over its own cache plus the tree under the same mask and position ids):
 *   x_0 = E[tok];  layer l: q, k, v = Wq_l x_l, Wk_l x_l, Wv_l x_l (RoPE at the node
 *   position), o_l = tree attention over layer l's prefix and the tree's layer-l keys,
 *   x_{l+1} = x_l + Wo_l o_l;  h' = x_n  (verification, acceptance and h_next as in
 *   medusa_step).  After acceptance the kept nodes' keys/values are appended to every
 *   layer's cache.
 * One medusa_layer per layer: its projections ([out][in] row-major, the plan's dtype,
 * 16-byte aligned; shapes as in medusa_weights) and its KV cache (the layout medusa_kv
 * describes; every layer shares the page table and the lengths). */
typedef struct {
  const void* wq;   /* [Hq*dh][d]  */
  const void* wk;   /* [Hkv*dh][d] */
  const void* wv;   /* [Hkv*dh][d] */
  const void* wo;   /* [d][Hq*dh]  */
  void* k;          /* this layer's cached keys   (device, caller-owned, updated) */
  void* v;          /* this layer's cached values (device, caller-owned, updated) */
} medusa_layer;

/* Bytes of workspace medusa_step_layers needs for n_layers layers (the single-layer size
 * plus each further layer's tree keys/values); 0 for n_layers outside 1..MEDUSA_MAX_LAYERS. */
size_t medusa_workspace_size_layers(const medusa_plan* plan, int n_layers);

/* One decode step through an n_layers-layer backbone.  h, root_in, acc, out, stream as
 * in medusa_step; w supplies the heads, the LM head and the embedding (its wq..wo are not
 * read); layers: host array of n_layers entries (read during the call only); kv supplies
 * the page table, len and len_out (its k, v are not read; len_out may alias len).
 * Errors: MEDUSA_ERR_INVALID for n_layers outside 1..MEDUSA_MAX_LAYERS, a NULL layer
 * pointer or misaligned weights, plus medusa_step's conditions.  With n_layers = 1 the
 * result equals medusa_step's with that layer's weights and cache. */
medusa_status medusa_step_layers(const medusa_plan* plan, const float* h, const int32_t* root_in,
                                 const medusa_weights* w, const medusa_layer* layers, int n_layers,
                                 const medusa_kv* kv, medusa_accept acc, const medusa_outputs* out,
                                 void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ stages */
/* (a) Heads ([MEDUSA] §3.4 MEDUSA Heads eq.; Tree Attention Step 1).  Writes the
 * logits [B][K+1][V] (row 0: LM head, row k: head k) to `logits` (device, may be NULL to
 * keep them in the workspace; row 0 is left unwritten when root_in is given, as the LM
 * head pass is then skipped), topk_tok/topk_val [B][K][16] (ranks past s_k unspecified)
 * and root [B] (root_in's value when given, else the LM head's greedy token; ties to the
 * lowest token id). */
medusa_status medusa_heads(const medusa_plan* plan, const float* h, const int32_t* root_in,
                           const medusa_weights* w, float* logits, int32_t* topk_tok,
                           float* topk_val, int32_t* root, void* workspace, size_t ws_bytes,
                           void* stream);
/* (a') Heads stage without a workspace.  The paper has no counterpart to this: it is a
 * deployment aid for callers that cannot allocate device memory when they run the heads
 * (an engine that plans every buffer up front and forbids allocation while decoding, a
 * plug-in confined to another framework's memory pool, code that may run while the
 * stream is being captured into a CUDA graph).  It computes exactly what medusa_heads()
 * computes and writes the same topk_tok / topk_val / root outputs (the logits are not
 * returned).  Its scratch lives in one library-owned device array of
 * MEDUSA_NOALLOC_SCRATCH_BYTES, present on every GPU that loads the library until the
 * process exits; no cudaMalloc, cudaFree or other allocating call is made.
 *   - Like the step, it keeps no logits: the vocab projections keep each CTA's best
 *     candidates and a selection merges them.  Plans whose heads scratch exceeds the array
 *     (about B*(K+1)*slots*128 bytes of candidate lists, slots = V/128 from batch 2 and a
 *     few hundred at batch 1, plus B*K*d*8 bytes of head activations) get
 *     MEDUSA_ERR_UNSUPPORTED and nothing is launched.
 *   - The first call on a device looks up the array's address with that device current;
 *     make that first call before any stream capture begins.  The address is kept per
 *     device and context; the first call after a cudaDeviceReset looks it up again and
 *     must likewise come before any capture.
 *   - All calls share the array and it keeps the last call's contents (nothing in it
 *     needs to start at zero).  Calls whose GPU work overlaps race on it: order them on
 *     one stream. */
#define MEDUSA_NOALLOC_SCRATCH_BYTES (4u << 20)
medusa_status medusa_heads_noalloc(const medusa_plan* plan, const float* h, const int32_t* root_in,
                                   const medusa_weights* w, int32_t* topk_tok, float* topk_val,
                                   int32_t* root, void* stream);
/* (b) Tree build ([MEDUSA] §3.4 Tree Attention Steps 2-4; [READING] section 6).
 * tok [B][N+1] node tokens, pos [B][N+1] = len + depth, mask [N+1][8] uint32 ancestor
 * bitmask (bit j of word j/32 set iff node j is on the root->n path), retrieve [N+1][K+1]
 * packed root->leaf paths (leaves in packed order, -1 padded; rows past the path count
 * are -1).  topk_tok as written by medusa_heads. */
medusa_status medusa_tree_build(const medusa_plan* plan, const int32_t* topk_tok,
                                const int32_t* root, const int32_t* len, int32_t* tok,
                                int32_t* pos, uint32_t* mask, int32_t* retrieve, void* stream);
/* (c) Synthetic layer projections: x = E[tok]; q = Wq x, k = Wk x, v = Wv x per head;
 * rotate-half RoPE of q and k at pos ([MEDUSA] §3.4 Step 4).  q: [B][N+1][Hq][dh] float;
 * tree_k, tree_v: [B][N+1][Hkv][dh] dtype. */
medusa_status medusa_layer_qkv(const medusa_plan* plan, const medusa_weights* w,
                               const int32_t* tok, const int32_t* pos, float* q, void* tree_k,
                               void* tree_v, void* workspace, size_t ws_bytes, void* stream);
/* (d) Tree attention ([MEDUSA] §3.4 Tree Attention Steps 3 and 5): node n, query head h
 * attends to the prefix slots [0, len) of key/value head h/(Hq/Hkv) and to the tree keys
 * of its ancestors (mask).  o: [B][N+1][Hq][dh] float. */
medusa_status medusa_tree_attention(const medusa_plan* plan, const float* q,
                                    const medusa_kv* kv, const void* tree_k,
                                    const void* tree_v, const uint32_t* mask, float* o,
                                    void* workspace, size_t ws_bytes, void* stream);
/* (e) Synthetic layer output h' = E[tok] + Wo o.  hprime: [B][N+1][d] float. */
medusa_status medusa_layer_out(const medusa_plan* plan, const medusa_weights* w,
                               const int32_t* tok, const float* o, float* hprime,
                               void* workspace, size_t ws_bytes, void* stream);
/* (f) Verification logits z_n = LM h'_n ([MEDUSA] §3.4 Tree Attention Step 6) and, per
 * node row, the statistics acceptance needs: am [B][N+1] greedy token (lowest id on ties);
 * stats [B][N+1][4] = {max_v z/T, log sum_v exp(z/T - max), entropy H (nats), z_parent at
 * this node's token / T} (T = 1 when greedy; entry 3 of the root is 0).  logits: device
 * [B][N+1][V] or NULL to keep them in the workspace. */
medusa_status medusa_verify_logits(const medusa_plan* plan, const medusa_weights* w,
                                   const float* hprime, const int32_t* tok, medusa_accept acc,
                                   float* logits, int32_t* am, float* stats, void* workspace,
                                   size_t ws_bytes, void* stream);
/* (g) Acceptance ([MEDUSA] §3.4 Typical Acceptance Scheme, whole-candidate and first-token
 * handling): the root is kept; candidate c is accepted iff tok[c] == am[parent[c]]
 * (greedy, or typical at T = 0) or log p_parent(tok[c]) > min(log eps, log delta - H)
 * (typical).  The longest run of accepted nodes along a root->leaf path wins, ties to the
 * lowest path index.  MEDUSA_REJECT walks the tree instead (see medusa_accept) and draws
 * root_next from `logits` ([B][N+1][V], as written by medusa_verify_logits; required in that
 * mode, unused and may be NULL otherwise).  Writes every medusa_outputs field; h_next is
 * hprime at the last kept node and root_next its greedy token (or the draw). */
medusa_status medusa_verify(const medusa_plan* plan, const int32_t* tok, const int32_t* am,
                            const float* stats, const float* logits, const int32_t* retrieve,
                            const float* hprime, medusa_accept acc, const medusa_outputs* out,
                            void* stream);
/* (h) KV compaction ([READING] section 3: only the accepted path stays in the cache):
 * slots len .. len+n_acc-1 receive the tree keys/values of path_nodes; len_out = len +
 * n_acc.  Slots past capacity are not written and set MEDUSA_FLAG_KV_CAPACITY. */
medusa_status medusa_kv_compact(const medusa_plan* plan, const medusa_kv* kv,
                                const void* tree_k, const void* tree_v,
                                const int32_t* path_nodes, const int32_t* n_acc, void* stream);

/* ------------------------------------------------------------------ decode loop */
/* The steady-state decode loop ([MEDUSA] §3.2: every step's first token is the previous
 * step's greedy token at the last accepted node, and decoding continues from the hidden
 * state there).  medusa_loop_create() captures, once, one medusa_step whose state is
 * carried in place (root_in = root_next = root, h = h_next = h, kv->len_out == kv->len:
 * the cache grows by each step's kept tokens) followed by the bookkeeping that appends the
 * step's out_tok [B][K+1] and n_acc [B] to the caller's rings tokens [max_steps][B][K+1] and
 * n_acc [max_steps][B] (position: steps appended so far, modulo max_steps) as a CUDA graph;
 * medusa_loop_run() replays it n_steps times on `stream` (asynchronous).
 *   - h: device [B][d], root: device [B] (e.g. a first medusa_step's h_next and root_next);
 *     both hold the latest state after every step.
 *   - Every pointer given here (weights, cache, lengths, state, rings, workspace) is used by
 *     every replay: keep them allocated, and the plan alive, until medusa_loop_destroy().
 *   - The cache must have room for the steps to be run (len + K + 1 <= capacity at every
 *     step); past that MEDUSA_FLAG_KV_CAPACITY is set, as in medusa_step.
 *   - Creation allocates the loop's small device state (B*(K+2) ints and a counter) and
 *     captures on a private stream; it launches nothing.
 * medusa_loop_steps() synchronises `stream` and returns the number of steps appended. */
typedef struct medusa_loop medusa_loop;
medusa_status medusa_loop_create(const medusa_plan* plan, const medusa_weights* w,
                                 const medusa_kv* kv, medusa_accept acc, float* h, int32_t* root,
                                 int32_t* tokens, int32_t* n_acc, int max_steps, void* workspace,
                                 size_t ws_bytes, medusa_loop** out);
medusa_status medusa_loop_run(medusa_loop* loop, int n_steps, void* stream);
medusa_status medusa_loop_steps(const medusa_loop* loop, void* stream, long long* steps);
void medusa_loop_destroy(medusa_loop* loop);

/* ------------------------------------------------------------------ tracing */
/* Per-stage timing (CUDA events recorded on the launching stream around every stage the
 * following calls on this plan run; a stage is one kernel, or a projection and its split-K
 * summation pass).  medusa_profile_start() creates the events for up to max_launches stages
 * (host-side resource, no device memory); stages past that are not timed.
 * medusa_profile_stop() synchronises `stream`, aggregates by stage name into out (up to
 * max_kernels entries, in first-launch order), writes the entry count to *n and the number
 * of kernels the calling thread launched meanwhile (split-K passes included) to
 * *launches, and ends profiling.  Each call also appears as an NVTX range named after it. */
typedef struct {
  char name[32];
  int launches;
  double total_ms;
} medusa_kernel_time;
medusa_status medusa_profile_start(medusa_plan* plan, int max_launches);
medusa_status medusa_profile_stop(medusa_plan* plan, void* stream, medusa_kernel_time* out,
                                  int max_kernels, int* n, int* launches);

/* ------------------------------------------------------------------ host tree builders */
/* Cartesian tree of the per-head top-s_k ([MEDUSA] §3.4 Tree Attention Step 2) in
 * canonical packing (by depth, then rank path).  parent/rank: host arrays of at least
 * max_nodes entries.  Returns N+1 (nodes incl. the root) or a negative medusa_status. */
int medusa_tree_cartesian(int K, const int* s, int max_nodes, int32_t* parent, int32_t* rank);
/* Optimized tree ([MEDUSA] §3.4 Optimized Tree Construction; [NOTES] section 4): from
 * the root, repeatedly add the frontier node with the largest product of marginal
 * accuracies a[k*smax + i] along its path (ties to the smaller rank path) until N nodes;
 * canonical packing.  Returns N+1 or a negative medusa_status. */
int medusa_tree_greedy(int K, const int* s, int smax, const double* a, int N, int32_t* parent,
                       int32_t* rank);

/* ---- optimized tree on the device, and the tree size
 * The same construction as medusa_tree_greedy, on the GPU from a device table: one CTA
 * repeatedly takes the frontier node with the largest path product (formed root to leaf in
 * double precision, as the host builder forms it; ties to the smaller rank path) and adds
 * its children to the frontier, then packs the N chosen nodes canonically.
 *   a:        device [K][smax] doubles, a[k*smax + i] = head k+1's marginal accuracy at
 *             rank i (values in [0, 1]); s: host [K], 1 <= s[k] <= smax <= MEDUSA_MAX_TOPS
 *   N:        candidates, 1 <= N <= MEDUSA_MAX_NODES - 1 and at most the Cartesian tree's size
 *   parent, rank: device [N+1] outputs in canonical packing (parent[0] = -1, rank[0] = 0)
 *   expected: device [N+1] output or NULL: expected[n] = the expected number of accepted
 *             candidates of the tree of the first n nodes added (sum of their path
 *             products), so one call gives the curve for every size up to N
 * Asynchronous on `stream`.  MEDUSA_ERR_INVALID on a bad size or NULL pointer. */
medusa_status medusa_tree_greedy_device(int K, const int* s, int smax, const double* a, int N,
                                        int32_t* parent, int32_t* rank, double* expected,
                                        void* stream);
/* Tree size for the current batch and context ([MEDUSA] §6 Limitations and Trade-offs: the
 * best tree size depends on the context length; "Follow-Up Research": dynamic candidate
 * counts for batched inference): among n candidate sizes with measured (or modelled) step
 * times step_ms[i], the index maximising the expected tokens per unit time
 * (1 + expected[sizes[i]]) / step_ms[i], ties to the smaller size.  expected: host
 * [max_n + 1] as from medusa_tree_greedy_device.  Returns the index or a negative status. */
int medusa_tree_size_choose(const double* expected, int max_n, const int* sizes,
                            const double* step_ms, int n);

#ifdef __cplusplus
}
#endif
#endif /* MEDUSA_H_ */
