// C ABI of the Medusa decode step: validation, plan, workspace layout and the launch
// sequences of the stages and of the whole step.  Every stage runs in this library's
// kernels on the caller's stream; nothing here computes on the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <queue>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <set>
#include <utility>
#include <vector>

#include "../../include/medusa.h"
#include "kernels.h"
#include "launch.cuh"

using namespace medusa;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Tracing: CUDA events around every kernel launch (enabled by medusa_profile_start).
enum KernelName {
  KN_H_SPLIT, KN_H_W1, KN_H_VOCAB, KN_TOPK_PARTIAL, KN_TOPK_MERGE, KN_TREE_BUILD, KN_GATHER,
  KN_QKV, KN_ROPE, KN_ATTN, KN_COMBINE, KN_O_SPLIT, KN_OUT, KN_HP_SPLIT, KN_VLOGITS, KN_VSTATS,
  KN_ACCEPT, KN_COMPACT, KN_QCAST, KN_SELECT, KN_COMMIT, KN_COUNT
};
static const char* const kKernelNames[KN_COUNT] = {
  "split_h", "heads_w1", "heads_vocab", "topk_partial", "topk_merge", "tree_build",
  "embed_gather", "layer_qkv", "rope_split", "tree_attention", "attn_combine", "split_o",
  "layer_out", "split_hprime", "verify_logits", "verify_stats", "verify_accept", "kv_compact",
  "cast_q", "heads_select", "verify_commit"};

struct Profiler {
  bool on = false;
  int used = 0;
  std::vector<cudaEvent_t> ev;      // two per timed launch
  std::vector<int> name;
  long kernels0 = 0;                // kernel-launch count when profiling started
  void release() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
    name.clear();
    used = 0;
    on = false;
  }
};

struct medusa_plan {
  mutable Profiler prof;
  medusa_dims d;
  int K, N, n1, P, smax;
  int s[MEDUSA_MAX_HEADS];
  int need[MEDUSA_MAX_HEADS + 1];   // ranks the tree uses per head (LM head: the root only)
  std::vector<int32_t> parent, rank, depth;
  int32_t* d_spec = nullptr;        // device [3][n1]: parent, depth, rank
  uint32_t* d_status = nullptr;
  float* d_rope = nullptr;          // device [rope_rows][dh]: cos | sin of p * theta_i
  int rope_rows = 0;
  size_t o_kpart = 0, kpart_bytes = 0;   // split-K partials of the node projections
  size_t o_cnt = 0;                      // completion counters of the fused kernels
  size_t o_vparts = 0;                   // per-row partial statistics of the fused commit
  uint32_t* d_mask = nullptr;            // device [n1][8] ancestor bitmask of the tree
  int32_t* d_retr = nullptr;             // device [n1][K+1] root->leaf paths
  int device = 0, num_sms = 148;
  // failure-path tests: one-shot wait limit for the next verification-logit GEMM
  mutable std::atomic<unsigned long long> test_wait_ns{0};
  bool tc_heads = false, tc_nodes = false;   // tensor-core projections
  bool tc_attn = false;                      // tensor-core tree attention
  int M;                                     // node rows B * n1
  int topk_splits, topk_chunk;
  int cand_ld = 1;                           // fused top-k: slots per (sequence, head)
  int nsplit, chunk, rpw, rows_per_block, nrb;
  // workspace layout (byte offsets)
  size_t o_logits, o_u, o_uhi, o_ulo, o_hhi, o_hlo, o_cv, o_ci, o_ttok, o_tval, o_root;
  size_t o_tok, o_pos, o_mask, o_retr, o_x, o_qkv, o_q, o_tk, o_tv, o_po, o_pml;
  size_t o_o, o_ohi, o_olo, o_hp, o_hphi, o_hplo, o_vlog, o_am, o_stats, o_path, o_nacc;
  size_t o_otok, o_hnext, o_rnext, o_qb;
  size_t o_fcv, o_fci, o_finv, o_fini;       // fused top-k: slot lists, per-head final lists
  size_t ws_bytes;

  const int32_t* dparent() const { return d_spec; }
  const int32_t* ddepth() const { return d_spec + n1; }
  const int32_t* drank() const { return d_spec + 2 * n1; }
  size_t esize() const { return d.dtype == MEDUSA_F32 ? 4 : 2; }
};

namespace {

template <typename T> T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

medusa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MEDUSA_OK : MEDUSA_ERR_CUDA; }
#define MEDUSA_TRY(x)                                  \
  do {                                                 \
    cudaError_t e_ = (x);                              \
    if (e_ != cudaSuccess) return MEDUSA_ERR_CUDA;     \
  } while (0)

template <typename F>
cudaError_t timed(const medusa_plan* p, int name, cudaStream_t st, F&& launch) {
  Profiler& pr = p->prof;
  if (!pr.on || pr.used >= (int)pr.name.size()) return launch();
  const int i = pr.used++;
  cudaEventRecord(pr.ev[2 * i], st);
  cudaError_t e = launch();
  cudaEventRecord(pr.ev[2 * i + 1], st);
  pr.name[i] = name;
  return e;
}
#define LAUNCH(p, kn, st, expr) MEDUSA_TRY(timed(p, kn, st, [&]() { return (expr); }))

medusa_status check_dims(const medusa_dims* d) {
  if (!d) return MEDUSA_ERR_INVALID;
  if (d->B < 1 || d->d < 1 || d->V < 1 || d->K < 1 || d->Hq < 1 || d->Hkv < 1 || d->dh < 1)
    return MEDUSA_ERR_INVALID;
  if (d->Hq % d->Hkv != 0) return MEDUSA_ERR_INVALID;
  if (d->dtype != MEDUSA_F32 && d->dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID;
  if (d->capacity < 1 || d->page_size < 0 || !(d->rope_base > 0.f)) return MEDUSA_ERR_INVALID;
  if (d->page_size > 0 && (d->capacity % d->page_size != 0 || d->num_pages < 1))
    return MEDUSA_ERR_INVALID;
  if (d->K > MEDUSA_MAX_HEADS) return MEDUSA_ERR_UNSUPPORTED;
  if (d->dh != 32 && d->dh != 64 && d->dh != 128) return MEDUSA_ERR_UNSUPPORTED;
  const int vec = d->dtype == MEDUSA_F32 ? 4 : 8;        // elements per 16-byte load
  if (d->d % vec != 0) return MEDUSA_ERR_UNSUPPORTED;
  return MEDUSA_OK;
}

medusa_status check_tree(const medusa_dims* d, const medusa_tree_spec* t, std::vector<int32_t>& depth) {
  if (!t || !t->parent || !t->rank) return MEDUSA_ERR_INVALID;
  if (t->K != d->K) return MEDUSA_ERR_INVALID;
  if (t->N < 0) return MEDUSA_ERR_INVALID;
  if (t->N + 1 > MEDUSA_MAX_NODES) return MEDUSA_ERR_UNSUPPORTED;
  for (int k = 0; k < t->K; ++k) {
    if (t->s[k] < 1 || t->s[k] > d->V) return MEDUSA_ERR_INVALID;
    if (t->s[k] > MEDUSA_MAX_TOPS) return MEDUSA_ERR_UNSUPPORTED;
  }
  const int n1 = t->N + 1;
  if (t->parent[0] != -1 || t->rank[0] != 0) return MEDUSA_ERR_INVALID;
  depth.assign(n1, 0);
  std::set<std::pair<int, int>> seen;
  for (int n = 1; n < n1; ++n) {
    const int p = t->parent[n];
    if (p < 0 || p >= n) return MEDUSA_ERR_INVALID;
    depth[n] = depth[p] + 1;
    if (depth[n] > t->K) return MEDUSA_ERR_INVALID;
    if (t->rank[n] < 0 || t->rank[n] >= t->s[depth[n] - 1]) return MEDUSA_ERR_INVALID;
    if (!seen.insert({p, t->rank[n]}).second) return MEDUSA_ERR_INVALID;   // duplicate child
  }
  return MEDUSA_OK;
}

void layout(medusa_plan* p) {
  const medusa_dims& d = p->d;
  const size_t B = d.B, K = p->K, V = d.V, D = d.d, n1 = p->n1, M = p->M;
  const size_t qd = (size_t)d.Hq * d.dh, kd = (size_t)d.Hkv * d.dh;
  const size_t R = n1 * (d.Hq / d.Hkv);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + std::max<size_t>(bytes, 1)); return o; };
  p->o_logits = take(B * (K + 1) * V * 4);
  p->o_u = take(B * K * D * 4);
  p->o_uhi = take(p->tc_heads ? B * K * D * 2 : 0);
  p->o_ulo = take(p->tc_heads ? B * K * D * 2 : 0);
  p->o_hhi = take(p->tc_heads ? B * D * 2 : 0);
  p->o_hlo = take(p->tc_heads ? B * D * 2 : 0);
  p->o_cv = take(B * (K + 1) * p->topk_splits * kTops * 4);
  p->o_ci = take(B * (K + 1) * p->topk_splits * kTops * 4);
  p->o_fcv = take(B * (K + 1) * p->cand_ld * kTops * 4);
  p->o_fci = take(B * (K + 1) * p->cand_ld * kTops * 4);
  p->o_finv = take(B * (K + 1) * kTops * 4);
  p->o_fini = take(B * (K + 1) * kTops * 4);
  p->o_ttok = take(B * K * kTops * 4);
  p->o_tval = take(B * K * kTops * 4);
  p->o_root = take(B * 4);
  p->o_tok = take(B * n1 * 4);
  p->o_pos = take(B * n1 * 4);
  p->o_mask = take(n1 * kMaskWords * 4);
  p->o_retr = take(n1 * (K + 1) * 4);
  p->o_x = take(M * D * 4);
  p->o_qkv = take(M * (qd + 2 * kd) * 4);
  p->o_q = take(M * qd * 4);
  p->o_tk = take(M * kd * p->esize());
  p->o_tv = take(M * kd * p->esize());
  p->o_po = take(B * d.Hkv * (p->nsplit + 1) * R * d.dh * 4);
  p->o_pml = take(B * d.Hkv * (p->nsplit + 1) * R * 2 * 4);
  p->o_o = take(M * qd * 4);
  p->o_ohi = take(p->tc_nodes ? M * qd * 2 : 0);
  p->o_olo = take(p->tc_nodes ? M * qd * 2 : 0);
  p->o_hp = take(M * D * 4);
  p->o_hphi = take(p->tc_nodes ? M * D * 2 : 0);
  p->o_hplo = take(p->tc_nodes ? M * D * 2 : 0);
  p->o_vlog = take(M * V * 4);
  p->o_am = take(M * 4);
  p->o_stats = take(M * 4 * 4);
  p->o_path = take(B * (K + 1) * 4);
  p->o_nacc = take(B * 4);
  p->o_otok = take(B * (K + 1) * 4);
  p->o_hnext = take(B * D * 4);
  p->o_rnext = take(B * 4);
  p->o_qb = take(p->tc_attn ? M * qd * 2 : 0);
  const size_t widest = std::max(std::max(D, qd), std::min<size_t>(V, 128 * 148));
  p->kpart_bytes = p->tc_nodes ? std::min<size_t>(8 * M * widest * 4, (size_t)64 << 20) : 0;
  p->o_kpart = take(p->kpart_bytes);
  // counters: [0,B) selection, [B,2B) commit per sequence, one per node row, then [B]
  // for the multi-layer compaction
  p->o_cnt = take((3 * B + M) * 4);
  p->o_vparts = take(M * kVerifySlicesMax * 6 * 4);
  p->ws_bytes = off;
}

medusa_status check_ws(const medusa_plan* p, void* ws, size_t bytes) {
  if (!ws || bytes < p->ws_bytes || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
    return MEDUSA_ERR_WORKSPACE;
  return MEDUSA_OK;
}

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// ------------------------------------------------------------------ stage bodies
// Upper bound of the fused top-k's slots over the heads launches a step makes: with the
// row-dot the LM head (when computed) joins the first launch after the K blocks of d rows
// and the second launch has the K heads' blocks of V rows.
int plan_cand_ld(const medusa_plan* p) {
  const medusa_dims& d = p->d;
  if (p->tc_heads) return (d.V + kCandTileRows - 1) / kCandTileRows;
  int most = 1;
  for (int first = 0; first < 2; ++first) {
    MatArgs a{};
    a.M = d.B;
    a.k = d.d;
    a.nseg = first ? p->K + 1 : p->K;
    for (int i = 0; i < a.nseg; ++i) {
      a.seg[i].rows = first && i < p->K ? d.d : d.V;
      a.seg[i].cand = !first || i == p->K;           // flagged as heads_impl flags them
    }
    for (int i = first ? p->K : 0; i < a.nseg; ++i) {
      int n = 0, c0 = 0;
      if (cand_geometry(a, i, false, d.dtype, &n, &c0)) most = std::max(most, n);
    }
  }
  return most;
}

// The heads' projections.  cand_count null: the logits of the computed heads go to
// `logits` ([B][K+1][V]).  Otherwise the vocab projections keep the fused top-k instead
// (slot lists in the workspace, per head the need[k] best) and cand_count[k] receives the
// slots of head k.
medusa_status heads_impl(const medusa_plan* p, const float* h, const int32_t* root_in,
                         const medusa_weights* w, float* logits, int32_t* ttok, float* tval,
                         int32_t* root, void* ws, cudaStream_t st, int* cand_count = nullptr) {
  const medusa_dims& d = p->d;
  const int B = d.B, K = p->K, D = d.d, V = d.V;
  const size_t es = p->esize();
  float* u = at<float>(ws, p->o_u);
  MatArgs a{};
  // u_k = SiLU(W1_k h) + h, k = 1..K
  a.nseg = K;
  a.M = B;
  a.k = D;
  a.out = u;
  a.ldo = (long)K * D;
  a.epi = EPI_SILU_RES;
  a.res_f32 = h;
  a.ldr = D;
  bf16* hhi = nullptr; bf16* hlo = nullptr;
  if (p->tc_heads) {
    hhi = at<bf16>(ws, p->o_hhi);
    hlo = at<bf16>(ws, p->o_hlo);
    LAUNCH(p, KN_H_SPLIT, st, launch_split(h, hhi, hlo, (long)B * D, st));
    a.out_hi = at<bf16>(ws, p->o_uhi);
    a.out_lo = at<bf16>(ws, p->o_ulo);
  }
  for (int k = 0; k < K; ++k) {
    MatSeg& s = a.seg[k];
    s.w = static_cast<const char*>(w->w1) + (size_t)k * D * D * es;
    s.x = h; s.a_hi = hhi; s.a_lo = hlo; s.ldx = D;
    s.rows = D;
    s.out_off = k * D;
  }
  // z_0 = LM h (only when the root is not given) reads h, not u: on the CUDA-core path it
  // joins this launch, whose few rows per warp otherwise leave the warps unevenly loaded
  const bool lm_first = !p->tc_heads && !root_in;
  if (lm_first) {
    MatSeg& s = a.seg[K];
    s.w = w->lm;
    s.x = h; s.ldx = D;
    s.rows = V;
    s.out_off = 0;
    a.nseg = K + 1;
    a.alt_from = K;
    a.out_alt = logits;
    a.ldo_alt = (long)(K + 1) * V;
  }
  // fused top-k: flag the candidate segments of a launch (head of segment i: head0 + i),
  // then take their slot counts from that launch's own geometry
  auto want_cand = [&](MatArgs& x, int i0, int head0) -> bool {
    x.cand_val = at<float>(ws, p->o_fcv);
    x.cand_idx = at<int32_t>(ws, p->o_fci);
    x.cand_nh = K + 1;
    x.cand_ld = p->cand_ld;
    for (int i = i0; i < x.nseg; ++i) {
      x.seg[i].cand = 1;
      x.seg[i].head = head0 + i;
      x.seg[i].rounds = p->need[head0 + i];
    }
    for (int i = i0; i < x.nseg; ++i) {
      int n = 0, c0 = 0;
      if (!cand_geometry(x, i, p->tc_heads, d.dtype, &n, &c0) || n < 1 || n > p->cand_ld) return false;
      cand_count[head0 + i] = n;
      x.seg[i].slot0 = c0;
    }
    return true;
  };
  if (cand_count && lm_first && !want_cand(a, K, -K)) return MEDUSA_ERR_CUDA;
  LAUNCH(p, KN_H_W1, st, p->tc_heads ? launch_umma_gemm(a, p->d_status, st) : launch_rowdot(a, d.dtype, st));
  // z_k = W2_k u_k (and z_0 here when it did not join the first launch)
  const int k0 = root_in || lm_first ? 1 : 0;
  MatArgs b{};
  b.nseg = K + 1 - k0;
  b.M = B;
  b.k = D;
  b.out = logits;
  b.ldo = (long)(K + 1) * V;
  b.epi = EPI_STORE;
  if (k0 == 0) {
    b.seg[0].w = w->lm;
    b.seg[0].x = h; b.seg[0].a_hi = hhi; b.seg[0].a_lo = hlo; b.seg[0].ldx = D;
    b.seg[0].rows = V;
    b.seg[0].out_off = 0;
  }
  for (int k = 1; k <= K; ++k) {
    MatSeg& s = b.seg[k - k0];
    s.w = static_cast<const char*>(w->w2) + (size_t)(k - 1) * V * D * es;
    s.x = u + (size_t)(k - 1) * D;
    s.a_hi = p->tc_heads ? at<bf16>(ws, p->o_uhi) + (size_t)(k - 1) * D : nullptr;
    s.a_lo = p->tc_heads ? at<bf16>(ws, p->o_ulo) + (size_t)(k - 1) * D : nullptr;
    s.ldx = (long)K * D;
    s.rows = V;
    s.out_off = k * V;
  }
  if (cand_count && !want_cand(b, 0, k0)) return MEDUSA_ERR_CUDA;
  LAUNCH(p, KN_H_VOCAB, st, p->tc_heads ? launch_umma_gemm(b, p->d_status, st) : launch_rowdot(b, d.dtype, st));
  (void)root_in; (void)ttok; (void)tval; (void)root;
  return MEDUSA_OK;
}

// Head 0 (the LM head) is selected only when the root is not given.
TopkArgs topk_args(const medusa_plan* p, const float* logits, const int32_t* root_in, void* ws) {
  TopkArgs t{logits, p->d.B, p->K + 1, p->d.V, p->topk_splits, p->topk_chunk,
             at<float>(ws, p->o_cv), at<int32_t>(ws, p->o_ci)};
  t.k0 = root_in ? 1 : 0;
  return t;
}
MergeArgs merge_args(const medusa_plan* p, const int32_t* root_in, int32_t* ttok, float* tval,
                     int32_t* root, void* ws) {
  MergeArgs m{at<float>(ws, p->o_cv), at<int32_t>(ws, p->o_ci), p->d.B, p->K, p->d.V,
              p->topk_splits, root_in, ttok, tval, root, p->d_status};
  m.k0 = root_in ? 1 : 0;
  return m;
}

// per-head top-16 and root from the head logits (the heads stage's selection)
medusa_status heads_topk(const medusa_plan* p, const float* logits, const int32_t* root_in,
                         int32_t* ttok, float* tval, int32_t* root, void* ws, cudaStream_t st) {
  const TopkArgs t = topk_args(p, logits, root_in, ws);
  LAUNCH(p, KN_TOPK_PARTIAL, st, launch_topk_partial(t, st));
  const MergeArgs mg = merge_args(p, root_in, ttok, tval, root, ws);
  LAUNCH(p, KN_TOPK_MERGE, st, launch_topk_merge(mg, st));
  return MEDUSA_OK;
}

medusa_status tree_impl(const medusa_plan* p, const int32_t* ttok, const int32_t* root,
                        const int32_t* len, int32_t* tok, int32_t* pos, uint32_t* mask,
                        int32_t* retr, cudaStream_t st) {
  TreeArgs a{ttok, root, len, p->d.B, p->K, p->d.V, p->n1, p->dparent(), p->ddepth(), p->drank(),
             tok, pos, mask, retr, p->d_status};
  LAUNCH(p, KN_TREE_BUILD, st, launch_tree_build(a, st));
  return MEDUSA_OK;
}

// x = E[tok] into the workspace (fp32 for the CUDA-core path, bf16 for tensor cores)
medusa_status gather_impl(const medusa_plan* p, const medusa_weights* w, const int32_t* tok,
                          void* ws, cudaStream_t st) {
  const medusa_dims& d = p->d;
  float* xf = p->tc_nodes ? nullptr : at<float>(ws, p->o_x);
  bf16* xb = p->tc_nodes ? at<bf16>(ws, p->o_x) : nullptr;
  LAUNCH(p, KN_GATHER, st, launch_gather(w->emb, d.dtype, tok, p->M, d.d, d.V, xf, xb, st));
  return MEDUSA_OK;
}

// q (fp32) may be null when only the bf16 copy for tensor-core attention is needed.
// x_in: the previous layer's h' (fp32; its bf16 hi/lo halves in the workspace) for backbone
// layers past the first; null for the first layer, which reads x = E[tok].
medusa_status qkv_impl(const medusa_plan* p, const medusa_weights* w, const int32_t* pos, float* q,
                       void* tk, void* tv, void* ws, cudaStream_t st, const float* x_in = nullptr) {
  const medusa_dims& d = p->d;
  const int qd = d.Hq * d.dh, kd = d.Hkv * d.dh;
  float* qkv = at<float>(ws, p->o_qkv);
  MatArgs a{};
  a.nseg = 3;
  a.M = p->M;
  a.k = d.d;
  a.out = qkv;
  a.ldo = qd + 2 * kd;
  a.epi = EPI_STORE;
  a.kpart = p->kpart_bytes ? at<float>(ws, p->o_kpart) : nullptr;
  a.kpart_bytes = p->kpart_bytes;
  const void* ws_[3] = {w->wq, w->wk, w->wv};
  const int rows[3] = {qd, kd, kd}, offs[3] = {0, qd, qd + kd};
  for (int i = 0; i < 3; ++i) {
    MatSeg& s = a.seg[i];
    s.w = ws_[i];
    if (x_in) {                               // h' of the previous layer
      s.x = p->tc_nodes ? nullptr : x_in;
      s.a_hi = p->tc_nodes ? at<bf16>(ws, p->o_hphi) : nullptr;
      s.a_lo = p->tc_nodes ? at<bf16>(ws, p->o_hplo) : nullptr;
    } else {
      s.x = p->tc_nodes ? nullptr : at<float>(ws, p->o_x);
      s.a_hi = p->tc_nodes ? at<bf16>(ws, p->o_x) : nullptr;
      s.a_lo = nullptr;                       // embedding rows are exact in bf16
    }
    s.ldx = d.d;
    s.rows = rows[i];
    s.out_off = offs[i];
  }
  if (p->tc_nodes) {
    // rotary embedding and the q / k / v outputs in the projection's own epilogue
    a.epi = EPI_ROPE;
    a.rope_pos = pos;
    a.rope_table = p->d_rope;
    a.rope_rows = p->rope_rows;
    a.rope_dh = d.dh;
    a.rope_qcols = qd;
    a.rope_kcols = kd;
    a.rq = q;
    a.rqb = p->tc_attn ? at<bf16>(ws, p->o_qb) : nullptr;
    a.rk = tk;
    a.rv = tv;
    a.rkv_bf16 = d.dtype == MEDUSA_BF16;
    a.rope_status = p->d_status;
    LAUNCH(p, KN_QKV, st, launch_umma_gemm(a, p->d_status, st));
    return MEDUSA_OK;
  }
  if (!q) return MEDUSA_ERR_INVALID;
  LAUNCH(p, KN_QKV, st, launch_rowdot(a, d.dtype, st));
  LAUNCH(p, KN_ROPE, st, launch_rope_split(qkv, pos, p->M, d.Hq, d.Hkv, d.dh, p->d_rope, p->rope_rows,
                                           p->d_status, d.dtype, q,
                                           p->tc_attn ? at<bf16>(ws, p->o_qb) : nullptr, tk, tv, st));
  return MEDUSA_OK;
}

medusa_status attn_impl(const medusa_plan* p, const float* q, const medusa_kv* kv, const void* tk,
                        const void* tv, const uint32_t* mask, float* o, bool split_out, bool q_ready, void* ws,
                        cudaStream_t st) {
  const medusa_dims& d = p->d;
  AttnArgs a{};
  a.q = q;
  a.kc = kv->k;
  a.vc = kv->v;
  a.page_table = d.page_size > 0 ? kv->page_table : nullptr;
  a.page_size = d.page_size > 0 ? d.page_size : 1;
  a.pages_per_seq = d.page_size > 0 ? d.capacity / d.page_size : 0;
  a.num_pages = d.num_pages;
  a.len = kv->len;
  a.capacity = d.capacity;
  a.tk = tk;
  a.tv = tv;
  a.mask = mask;
  a.B = d.B;
  a.n1 = p->n1;
  a.Hq = d.Hq;
  a.Hkv = d.Hkv;
  a.G = d.Hq / d.Hkv;
  a.dh = d.dh;
  a.nsplit = p->nsplit;
  a.chunk = p->chunk;
  a.rows_per_block = p->rows_per_block;
  a.nrb = p->nrb;
  a.rpw = p->rpw;
  a.part_o = at<float>(ws, p->o_po);
  a.part_ml = at<float>(ws, p->o_pml);
  // the step's tensor-core out projection reads only the bf16 halves: no fp32 copy then
  a.o = split_out && p->tc_nodes ? nullptr : o;
  a.o_hi = split_out && p->tc_nodes ? at<bf16>(ws, p->o_ohi) : nullptr;
  a.o_lo = split_out && p->tc_nodes ? at<bf16>(ws, p->o_olo) : nullptr;
  a.status = p->d_status;
  a.scale = 1.0f / std::sqrt((float)d.dh);
  if (p->tc_attn) {
    bf16* qb = at<bf16>(ws, p->o_qb);
    if (!q_ready) LAUNCH(p, KN_QCAST, st, launch_to_bf16(q, qb, (long)p->M * d.Hq * d.dh, st));
    LAUNCH(p, KN_ATTN, st, launch_tree_attention_pp(a, qb, p->num_sms, st));
  } else {
    LAUNCH(p, KN_ATTN, st, launch_tree_attention(a, d.dtype, st));
  }
  LAUNCH(p, KN_COMBINE, st, launch_attn_combine(a, st));
  return MEDUSA_OK;
}

// h' = x + Wo o ; x gathered by gather_impl (res_in null), or the previous layer's h'
// (res_in, fp32, may be hp itself: each element is read and then written by one thread);
// o split to bf16 hi/lo when split_ready
medusa_status out_impl(const medusa_plan* p, const medusa_weights* w, const float* o, bool split_ready,
                       float* hp, bool want_split, void* ws, cudaStream_t st, const float* res_in = nullptr) {
  const medusa_dims& d = p->d;
  const int qd = d.Hq * d.dh;
  MatArgs a{};
  a.nseg = 1;
  a.M = p->M;
  a.k = qd;
  a.out = hp;
  a.ldo = d.d;
  a.epi = EPI_RES_ADD;
  a.ldr = d.d;
  a.kpart = p->kpart_bytes ? at<float>(ws, p->o_kpart) : nullptr;
  a.kpart_bytes = p->kpart_bytes;
  if (p->tc_nodes) {
    if (!split_ready)
      LAUNCH(p, KN_O_SPLIT, st, launch_split(o, at<bf16>(ws, p->o_ohi), at<bf16>(ws, p->o_olo), (long)p->M * qd, st));
    if (res_in) a.res_f32 = res_in;
    else a.res_w = at<bf16>(ws, p->o_x);
    if (want_split) {
      a.out_hi = at<bf16>(ws, p->o_hphi);
      a.out_lo = at<bf16>(ws, p->o_hplo);
    }
  } else {
    a.res_f32 = res_in ? res_in : at<float>(ws, p->o_x);
  }
  MatSeg& s = a.seg[0];
  s.w = w->wo;
  s.x = o;
  s.a_hi = p->tc_nodes ? at<bf16>(ws, p->o_ohi) : nullptr;
  s.a_lo = p->tc_nodes ? at<bf16>(ws, p->o_olo) : nullptr;
  s.ldx = qd;
  s.rows = d.d;
  s.out_off = 0;
  LAUNCH(p, KN_OUT, st, p->tc_nodes ? launch_umma_gemm(a, p->d_status, st) : launch_rowdot(a, d.dtype, st));
  return MEDUSA_OK;
}

VerifyArgs verify_args(const medusa_plan* p, const int32_t* tok, medusa_accept acc) {
  VerifyArgs v{};
  v.tok = tok;
  v.parent = p->dparent();
  v.depth = p->ddepth();
  v.B = p->d.B;
  v.n1 = p->n1;
  v.V = p->d.V;
  v.K = p->K;
  v.P = p->P;
  v.d = p->d.d;
  // rejection sampling needs the same per-row softmax statistics as typical acceptance
  v.reject = acc.mode == MEDUSA_REJECT && acc.temperature > 0.f;
  v.typical = (acc.mode == MEDUSA_TYPICAL && acc.temperature > 0.f) || v.reject;
  v.temperature = v.typical ? acc.temperature : 1.f;
  v.uniforms = v.reject ? acc.uniforms : nullptr;
  v.eps = acc.eps;
  v.delta = acc.delta;
  v.status = p->d_status;
  return v;
}

medusa_status vlogits_impl(const medusa_plan* p, const medusa_weights* w, const float* hp,
                           bool split_ready, const int32_t* tok, medusa_accept acc, float* logits,
                           int32_t* am, float* stats, void* ws, cudaStream_t st,
                           bool with_stats = true) {
  const medusa_dims& d = p->d;
  MatArgs a{};
  a.nseg = 1;
  a.M = p->M;
  a.k = d.d;
  a.out = logits;
  a.ldo = d.V;
  a.epi = EPI_STORE;
  a.kpart = p->kpart_bytes ? at<float>(ws, p->o_kpart) : nullptr;
  a.kpart_bytes = p->kpart_bytes;
  if (p->tc_nodes && !split_ready)
    LAUNCH(p, KN_HP_SPLIT, st, launch_split(hp, at<bf16>(ws, p->o_hphi), at<bf16>(ws, p->o_hplo), (long)p->M * d.d, st));
  MatSeg& s = a.seg[0];
  s.w = w->lm;
  s.x = hp;
  s.a_hi = p->tc_nodes ? at<bf16>(ws, p->o_hphi) : nullptr;
  s.a_lo = p->tc_nodes ? at<bf16>(ws, p->o_hplo) : nullptr;
  s.ldx = d.d;
  s.rows = d.V;
  s.out_off = 0;
  if (p->tc_nodes) a.test_wait_ns = p->test_wait_ns.exchange(0);
  LAUNCH(p, KN_VLOGITS, st, p->tc_nodes ? launch_umma_gemm(a, p->d_status, st) : launch_rowdot(a, d.dtype, st));
  if (!with_stats) return MEDUSA_OK;
  VerifyArgs v = verify_args(p, tok, acc);
  v.logits = logits;
  v.am = am;
  v.stats = stats;
  LAUNCH(p, KN_VSTATS, st, launch_verify_stats(v, st));
  return MEDUSA_OK;
}

medusa_status accept_impl(const medusa_plan* p, const int32_t* tok, const int32_t* am,
                          const float* stats, const float* logits, const int32_t* retr,
                          const float* hp, medusa_accept acc, int32_t* out_tok, int32_t* n_acc,
                          int32_t* path, float* h_next, int32_t* root_next, cudaStream_t st) {
  VerifyArgs v = verify_args(p, tok, acc);
  v.logits = logits;                           // rejection sampling draws from these
  v.am = const_cast<int32_t*>(am);
  v.stats = const_cast<float*>(stats);
  v.retrieve = retr;
  v.hprime = hp;
  v.out_tok = out_tok;
  v.n_acc = n_acc;
  v.path_nodes = path;
  v.h_next = h_next;
  v.root_next = root_next;
  LAUNCH(p, KN_ACCEPT, st, launch_verify_accept(v, st));
  return MEDUSA_OK;
}

CompactArgs compact_args(const medusa_plan* p, const medusa_kv* kv, const void* tk, const void* tv,
                         const int32_t* path, const int32_t* n_acc) {
  const medusa_dims& d = p->d;
  CompactArgs c{};
  c.kc = kv->k;
  c.vc = kv->v;
  c.page_table = d.page_size > 0 ? kv->page_table : nullptr;
  c.page_size = d.page_size > 0 ? d.page_size : 1;
  c.pages_per_seq = d.page_size > 0 ? d.capacity / d.page_size : 0;
  c.num_pages = d.num_pages;
  c.len = kv->len;
  c.len_out = kv->len_out;
  c.capacity = d.capacity;
  c.tk = tk;
  c.tv = tv;
  c.path_nodes = path;
  c.n_acc = n_acc;
  c.B = d.B;
  c.n1 = p->n1;
  c.Hkv = d.Hkv;
  c.dh = d.dh;
  c.K = p->K;
  c.dtype = d.dtype;
  c.status = p->d_status;
  return c;
}

medusa_status compact_impl(const medusa_plan* p, const medusa_kv* kv, const void* tk, const void* tv,
                           const int32_t* path, const int32_t* n_acc, cudaStream_t st) {
  const CompactArgs c = compact_args(p, kv, tk, tv, path, n_acc);
  LAUNCH(p, KN_COMPACT, st, launch_kv_compact(c, st));
  return MEDUSA_OK;
}

medusa_status check_weights(const medusa_plan* p, const medusa_weights* w, bool heads, bool layer, bool lm) {
  if (!w) return MEDUSA_ERR_INVALID;
  if (heads && (!aligned16(w->w1) || !aligned16(w->w2))) return MEDUSA_ERR_INVALID;
  if (lm && !aligned16(w->lm)) return MEDUSA_ERR_INVALID;
  if (layer && (!aligned16(w->emb) || !aligned16(w->wq) || !aligned16(w->wk) || !aligned16(w->wv) ||
                !aligned16(w->wo)))
    return MEDUSA_ERR_INVALID;
  (void)p;
  return MEDUSA_OK;
}

medusa_status check_kv(const medusa_plan* p, const medusa_kv* kv, bool compact) {
  if (!kv || !kv->k || !kv->v || !kv->len) return MEDUSA_ERR_INVALID;
  if (p->d.page_size > 0 && !kv->page_table) return MEDUSA_ERR_INVALID;
  if (compact && !kv->len_out) return MEDUSA_ERR_INVALID;
  return MEDUSA_OK;
}

medusa_status check_accept(medusa_accept a) {
  if (a.mode != MEDUSA_GREEDY && a.mode != MEDUSA_TYPICAL && a.mode != MEDUSA_REJECT)
    return MEDUSA_ERR_INVALID;
  if (a.mode != MEDUSA_GREEDY && (!(a.temperature >= 0.f) || !std::isfinite(a.temperature)))
    return MEDUSA_ERR_INVALID;
  if (a.mode == MEDUSA_TYPICAL && a.temperature > 0.f && (!(a.eps > 0.f) || !(a.delta > 0.f)))
    return MEDUSA_ERR_INVALID;
  if (a.mode == MEDUSA_REJECT && a.temperature > 0.f && !a.uniforms) return MEDUSA_ERR_INVALID;
  return MEDUSA_OK;
}

}  // namespace

// Read-only view of the plan fields the workspace-free heads entry point needs.
bool medusa::heads_plan_view(const medusa_plan* p, HeadsPlanView* v) {
  if (!p || !v) return false;
  v->dims = p->d;
  v->K = p->K;
  v->tc_heads = p->tc_heads;
  v->topk_splits = p->topk_splits;
  v->topk_chunk = p->topk_chunk;
  v->status = p->d_status;
  return true;
}

// ===================================================================== exported API
namespace medusa {
namespace {
thread_local long t_kernels = 0;             // kernels launched by this host thread
thread_local bool t_pdl_armed = false;       // a library kernel was the last launch ...
thread_local cudaStream_t t_pdl_stream = nullptr;   // ... on this stream
bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("MEDUSA_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}
}  // namespace
long kernels_launched() { return t_kernels; }
bool pdl_take(cudaStream_t st) {
  ++t_kernels;                                // every kernel launch passes through here
  const bool ok = t_pdl_armed && t_pdl_stream == st && pdl_enabled();
  t_pdl_armed = true;
  t_pdl_stream = st;
  return ok;
}
void pdl_reset() { t_pdl_armed = false; }
}  // namespace medusa

extern "C" {

medusa_status medusa_plan_create(const medusa_dims* dims, const medusa_tree_spec* tree,
                                 medusa_plan** out) {
  if (!out) return MEDUSA_ERR_INVALID;
  *out = nullptr;
  medusa_status s = check_dims(dims);
  if (s != MEDUSA_OK) return s;
  std::vector<int32_t> depth;
  s = check_tree(dims, tree, depth);
  if (s != MEDUSA_OK) return s;
  medusa_plan* p = new (std::nothrow) medusa_plan();
  if (!p) return MEDUSA_ERR_CUDA;
  p->d = *dims;
  p->K = dims->K;
  p->N = tree->N;
  p->n1 = tree->N + 1;
  for (int k = 0; k < MEDUSA_MAX_HEADS; ++k) p->s[k] = k < p->K ? tree->s[k] : 0;
  p->smax = *std::max_element(p->s, p->s + p->K);
  p->parent.assign(tree->parent, tree->parent + p->n1);
  p->rank.assign(tree->rank, tree->rank + p->n1);
  p->depth = depth;
  std::vector<int> haschild(p->n1, 0);
  for (int n = 1; n < p->n1; ++n) haschild[p->parent[n]] = 1;
  p->P = (int)std::count(haschild.begin(), haschild.end(), 0);
  p->M = dims->B * p->n1;
  // Row-dot re-reads the staged activations from shared memory once per batch row for
  // every 16 bytes of weights; from two rows on, the tensor-core path streams faster.
  p->tc_heads = dims->dtype == MEDUSA_BF16 && dims->B >= 2;
  p->tc_nodes = dims->dtype == MEDUSA_BF16;

  cudaGetDevice(&p->device);
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) == cudaSuccess && sms > 0)
    p->num_sms = sms;
  // vocab slices for the top-k pass: as many as one resident wave of the selection's
  // 256-thread CTAs holds, but no fewer than one per 4096 logits (at most 16 per thread)
  // and no more than one per 1024 logits or 32 per head; slices start on 16-byte
  // boundaries when V allows (the selection then loads float4)
  {
    const long pairs = (long)dims->B * (p->K + 1);
    const long wave = (long)std::max(1, topk_partial_ctas_per_sm()) * p->num_sms;
    const long lo = (dims->V + 4095) / 4096, hi = std::max(1, std::min(32, (dims->V + 1023) / 1024));
    const long sp = std::min<long>(32, std::max(lo, std::min(hi, wave / pairs)));
    p->topk_splits = (int)std::max(1L, sp);
  }
  p->topk_chunk = (dims->V + p->topk_splits - 1) / p->topk_splits;
  if (dims->V % 4 == 0) p->topk_chunk = (p->topk_chunk + 3) / 4 * 4;
  // attention: query-row blocks and prefix splits so the grid covers the SMs ~2x
  const int G = dims->Hq / dims->Hkv;
  const int R = p->n1 * G;
  p->tc_attn = tree_attention_pp_supported(dims->dtype, dims->dh, G, dims->page_size);
  p->rpw = R <= 32 ? 4 : (R <= 72 ? 9 : 12);
  p->rows_per_block = p->tc_attn ? (R > 128 ? 256 : 128) : 8 * p->rpw;
  p->nrb = (R + p->rows_per_block - 1) / p->rows_per_block;
  const int base = dims->B * dims->Hkv * p->nrb;
  const int want = std::max(1, (2 * p->num_sms + base - 1) / base);
  const int gran = p->tc_attn ? 128 : 32;             // keys per chunk of the kernel
  const int max_splits = std::max(1, (dims->capacity + gran - 1) / gran);
  p->nsplit = std::min(want, max_splits);
  if (p->tc_attn) {
    // One persistent CTA per SM, CTA c taking units c, c + grid, ... (units split-major, the
    // tree units last).  Cost in key loads of one SM: the busiest CTA's chunks (a unit also
    // pays about four chunks' time for its query tile, the pipeline refill and its partial:
    // measured at the 13B, Zephyr and 7B shapes), plus the partials that the splits write
    // and the combine reads back, in the same units.
    const double key_bytes = 2.0 * dims->dh * 2;                 // one key's K and V
    const double part_bytes = 2.0 * dims->B * dims->Hq * p->n1 * (dims->dh * 4 + 8);
    const long tree_chunks = (p->n1 + gran - 1) / gran;
    double best = -1;
    std::vector<long> load;
    for (int ns = 1; ns <= std::min(max_splits, 64); ++ns) {
      const long chunk = ((dims->capacity + ns - 1) / ns + gran - 1) / gran * gran;
      const long nsp = (dims->capacity + chunk - 1) / chunk;      // splits that exist
      if (nsp != ns) continue;
      const long units = (long)base * (ns + 1);
      const long grid = std::min<long>(units, p->num_sms);
      load.assign(grid, 0);
      for (long u = 0; u < units; ++u) {
        const bool tree = u / base == ns;
        load[u % grid] += (tree ? tree_chunks : chunk / gran) + 4;
      }
      const double busiest = (double)*std::max_element(load.begin(), load.end()) * gran;
      const double cost = busiest + (ns + 1) * part_bytes / (p->num_sms * key_bytes);
      if (best < 0 || cost < best) { best = cost; p->nsplit = ns; }
    }
  }
  p->chunk = ((dims->capacity + p->nsplit - 1) / p->nsplit + gran - 1) / gran * gran;
  p->nsplit = (dims->capacity + p->chunk - 1) / p->chunk;
  p->cand_ld = plan_cand_ld(p);
  layout(p);

  for (int k = 0; k <= MEDUSA_MAX_HEADS; ++k) p->need[k] = 1;
  for (int n = 1; n < p->n1; ++n) p->need[p->depth[n]] = std::max(p->need[p->depth[n]], p->rank[n] + 1);
  std::vector<int32_t> spec(3 * p->n1);
  for (int n = 0; n < p->n1; ++n) {
    spec[n] = p->parent[n];
    spec[p->n1 + n] = p->depth[n];
    spec[2 * p->n1 + n] = p->rank[n];
  }
  // static tree tables: ancestor bitmask and root->leaf paths (leaves in packed order)
  std::vector<uint32_t> tmask((size_t)p->n1 * kMaskWords, 0u);
  std::vector<int32_t> tretr((size_t)p->n1 * (p->K + 1), -1);
  {
    std::vector<int> haschild(p->n1, 0);
    for (int n = 1; n < p->n1; ++n) haschild[p->parent[n]] = 1;
    int leaf = 0;
    for (int n = 0; n < p->n1; ++n) {
      for (int j = n; j >= 0; j = p->parent[j]) tmask[(size_t)n * kMaskWords + j / 32] |= 1u << (j % 32);
      if (haschild[n]) continue;
      for (int j = n; j >= 0; j = p->parent[j]) tretr[(size_t)leaf * (p->K + 1) + p->depth[j]] = j;
      ++leaf;
    }
  }
  // rotary table for every position a step can produce: len + depth <= capacity + K
  p->rope_rows = dims->capacity + p->K + 1;
  std::vector<float> rope((size_t)p->rope_rows * dims->dh);
  rope_table(dims->rope_base, dims->dh, p->rope_rows, rope.data());
  if (cudaMalloc(&p->d_spec, spec.size() * sizeof(int32_t)) != cudaSuccess ||
      cudaMalloc(&p->d_status, sizeof(uint32_t)) != cudaSuccess ||
      cudaMalloc(&p->d_rope, rope.size() * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&p->d_mask, tmask.size() * sizeof(uint32_t)) != cudaSuccess ||
      cudaMalloc(&p->d_retr, tretr.size() * sizeof(int32_t)) != cudaSuccess ||
      cudaMemcpy(p->d_mask, tmask.data(), tmask.size() * sizeof(uint32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(p->d_retr, tretr.data(), tretr.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(p->d_spec, spec.data(), spec.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(p->d_rope, rope.data(), rope.size() * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(p->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
    medusa_plan_destroy(p);
    return MEDUSA_ERR_CUDA;
  }
  *out = p;
  return MEDUSA_OK;
}

void medusa_plan_destroy(medusa_plan* p) {
  if (!p) return;
  p->prof.release();
  if (p->d_rope) cudaFree(p->d_rope);
  if (p->d_mask) cudaFree(p->d_mask);
  if (p->d_retr) cudaFree(p->d_retr);
  if (p->d_spec) cudaFree(p->d_spec);
  if (p->d_status) cudaFree(p->d_status);
  delete p;
}

size_t medusa_workspace_size(const medusa_plan* p) { return p ? p->ws_bytes : 0; }

medusa_status medusa_profile_start(medusa_plan* p, int max_launches) {
  if (!p || max_launches < 1) return MEDUSA_ERR_INVALID;
  p->prof.release();
  p->prof.ev.resize(2 * (size_t)max_launches);
  p->prof.name.assign(max_launches, -1);
  for (auto& e : p->prof.ev)
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      p->prof.release();
      return MEDUSA_ERR_CUDA;
    }
  p->prof.on = true;
  p->prof.kernels0 = kernels_launched();
  return MEDUSA_OK;
}

medusa_status medusa_profile_stop(medusa_plan* p, void* stream, medusa_kernel_time* out,
                                  int max_kernels, int* n, int* launches) {
  if (!p || !n || !launches || (max_kernels > 0 && !out)) return MEDUSA_ERR_INVALID;
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MEDUSA_ERR_CUDA;
  std::vector<int> order, count(KN_COUNT, 0);
  std::vector<double> ms(KN_COUNT, 0.0);
  for (int i = 0; i < p->prof.used; ++i) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, p->prof.ev[2 * i], p->prof.ev[2 * i + 1]) != cudaSuccess) {
      p->prof.release();
      return MEDUSA_ERR_CUDA;
    }
    const int k = p->prof.name[i];
    if (count[k]++ == 0) order.push_back(k);
    ms[k] += t;
  }
  *launches = (int)(kernels_launched() - p->prof.kernels0);   // kernels, incl. split-K passes
  int m = 0;
  for (int k : order) {
    if (m >= max_kernels) break;
    std::memset(out[m].name, 0, sizeof(out[m].name));
    std::strncpy(out[m].name, kKernelNames[k], sizeof(out[m].name) - 1);
    out[m].launches = count[k];
    out[m].total_ms = ms[k];
    ++m;
  }
  *n = m;
  p->prof.release();
  return MEDUSA_OK;
}

medusa_status medusa_plan_expire_wait_once(medusa_plan* p, unsigned long long ns) {
  if (!p || ns == 0 || ns > 10000000000ull) return MEDUSA_ERR_INVALID;
  if (!p->tc_nodes) return MEDUSA_ERR_UNSUPPORTED;
  p->test_wait_ns.store(ns);
  return MEDUSA_OK;
}

medusa_status medusa_get_status(const medusa_plan* p, void* stream, uint32_t* flags) {
  if (!p || !flags) return MEDUSA_ERR_INVALID;
  uint32_t v = 0;
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaMemcpy(&v, p->d_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaMemset(p->d_status, 0, sizeof(v)) != cudaSuccess) return MEDUSA_ERR_CUDA;
  *flags = v;
  return v ? MEDUSA_ERR_DEVICE : MEDUSA_OK;
}

medusa_status medusa_heads(const medusa_plan* p, const float* h, const int32_t* root_in,
                           const medusa_weights* w, float* logits, int32_t* topk_tok,
                           float* topk_val, int32_t* root, void* ws, size_t ws_bytes, void* stream) {
  EntryScope scope("medusa_heads");
  if (!p || !h || !topk_tok || !topk_val || !root) return MEDUSA_ERR_INVALID;
  medusa_status s = check_weights(p, w, true, false, true);
  if (s != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  if (!logits) logits = at<float>(ws, p->o_logits);
  medusa_status s2 = heads_impl(p, h, root_in, w, logits, topk_tok, topk_val, root, ws, S(stream));
  if (s2 != MEDUSA_OK) return s2;
  return heads_topk(p, logits, root_in, topk_tok, topk_val, root, ws, S(stream));
}

medusa_status medusa_tree_build(const medusa_plan* p, const int32_t* topk_tok, const int32_t* root,
                                const int32_t* len, int32_t* tok, int32_t* pos, uint32_t* mask,
                                int32_t* retrieve, void* stream) {
  EntryScope scope("medusa_tree_build");
  if (!p || !topk_tok || !root || !len || !tok || !pos || !mask || !retrieve) return MEDUSA_ERR_INVALID;
  return tree_impl(p, topk_tok, root, len, tok, pos, mask, retrieve, S(stream));
}

medusa_status medusa_layer_qkv(const medusa_plan* p, const medusa_weights* w, const int32_t* tok,
                               const int32_t* pos, float* q, void* tk, void* tv, void* ws,
                               size_t ws_bytes, void* stream) {
  EntryScope scope("medusa_layer_qkv");
  if (!p || !tok || !pos || !q || !tk || !tv) return MEDUSA_ERR_INVALID;
  medusa_status s = check_weights(p, w, false, true, false);
  if (s != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  if ((s = gather_impl(p, w, tok, ws, S(stream))) != MEDUSA_OK) return s;
  return qkv_impl(p, w, pos, q, tk, tv, ws, S(stream));
}

medusa_status medusa_tree_attention(const medusa_plan* p, const float* q, const medusa_kv* kv,
                                    const void* tk, const void* tv, const uint32_t* mask, float* o,
                                    void* ws, size_t ws_bytes, void* stream) {
  EntryScope scope("medusa_tree_attention");
  if (!p || !q || !tk || !tv || !mask || !o) return MEDUSA_ERR_INVALID;
  medusa_status s = check_kv(p, kv, false);
  if (s != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  return attn_impl(p, q, kv, tk, tv, mask, o, false, false, ws, S(stream));
}

medusa_status medusa_layer_out(const medusa_plan* p, const medusa_weights* w, const int32_t* tok,
                               const float* o, float* hprime, void* ws, size_t ws_bytes, void* stream) {
  EntryScope scope("medusa_layer_out");
  if (!p || !tok || !o || !hprime) return MEDUSA_ERR_INVALID;
  medusa_status s = check_weights(p, w, false, true, false);
  if (s != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  if ((s = gather_impl(p, w, tok, ws, S(stream))) != MEDUSA_OK) return s;
  return out_impl(p, w, o, false, hprime, false, ws, S(stream));
}

medusa_status medusa_verify_logits(const medusa_plan* p, const medusa_weights* w, const float* hprime,
                                   const int32_t* tok, medusa_accept acc, float* logits, int32_t* am,
                                   float* stats, void* ws, size_t ws_bytes, void* stream) {
  EntryScope scope("medusa_verify_logits");
  if (!p || !hprime || !tok || !am || !stats) return MEDUSA_ERR_INVALID;
  medusa_status s = check_weights(p, w, false, false, true);
  if (s != MEDUSA_OK) return s;
  if ((s = check_accept(acc)) != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  if (!logits) logits = at<float>(ws, p->o_vlog);
  return vlogits_impl(p, w, hprime, false, tok, acc, logits, am, stats, ws, S(stream));
}

medusa_status medusa_verify(const medusa_plan* p, const int32_t* tok, const int32_t* am,
                            const float* stats, const float* logits, const int32_t* retrieve,
                            const float* hprime, medusa_accept acc, const medusa_outputs* out,
                            void* stream) {
  EntryScope scope("medusa_verify");
  if (!p || !tok || !am || !stats || !retrieve || !hprime || !out) return MEDUSA_ERR_INVALID;
  if (!out->out_tok || !out->n_acc || !out->h_next || !out->root_next) return MEDUSA_ERR_INVALID;
  medusa_status s = check_accept(acc);
  if (s != MEDUSA_OK) return s;
  if (acc.mode == MEDUSA_REJECT && acc.temperature > 0.f && !logits) return MEDUSA_ERR_INVALID;
  return accept_impl(p, tok, am, stats, logits, retrieve, hprime, acc, out->out_tok, out->n_acc,
                     out->path_nodes, out->h_next, out->root_next, S(stream));
}

medusa_status medusa_kv_compact(const medusa_plan* p, const medusa_kv* kv, const void* tk,
                                const void* tv, const int32_t* path_nodes, const int32_t* n_acc,
                                void* stream) {
  EntryScope scope("medusa_kv_compact");
  if (!p || !tk || !tv || !path_nodes || !n_acc) return MEDUSA_ERR_INVALID;
  medusa_status s = check_kv(p, kv, true);
  if (s != MEDUSA_OK) return s;
  return compact_impl(p, kv, tk, tv, path_nodes, n_acc, S(stream));
}

namespace {

// Tree keys/values of backbone layer l >= 1 live past the single-layer workspace.
size_t layer_kv_bytes(const medusa_plan* p) {
  return align_up((size_t)p->M * p->d.Hkv * p->d.dh * p->esize());
}
size_t layers_ws_bytes(const medusa_plan* p, int n_layers) {
  return p->ws_bytes + (size_t)(n_layers - 1) * 2 * layer_kv_bytes(p);
}

// The decode step through nl backbone layers (nl = 1: medusa_step).  With one layer the
// fused commit also compacts the cache; with more, it only accepts and kv_compact_layers
// then appends the kept nodes to every layer's cache.
medusa_status step_core(const medusa_plan* p, const float* h, const int32_t* root_in,
                        const medusa_weights* w, const medusa_layer* layers, int nl, const medusa_kv* kv,
                        medusa_accept acc, const medusa_outputs* out, void* ws, cudaStream_t st) {
  medusa_status s = MEDUSA_OK;
  int32_t* ttok = at<int32_t>(ws, p->o_ttok);
  int32_t* root = at<int32_t>(ws, p->o_root);
  int32_t* tok = at<int32_t>(ws, p->o_tok);
  int32_t* pos = at<int32_t>(ws, p->o_pos);
  float* q = at<float>(ws, p->o_q);
  float* o = at<float>(ws, p->o_o);
  float* hp = at<float>(ws, p->o_hp);
  int32_t* am = at<int32_t>(ws, p->o_am);
  float* stats = at<float>(ws, p->o_stats);
  int32_t* path = out->path_nodes ? out->path_nodes : at<int32_t>(ws, p->o_path);
  float* logits = at<float>(ws, p->o_logits);
  int32_t* cnt = at<int32_t>(ws, p->o_cnt);
  const int B = p->d.B;
  MEDUSA_TRY(cudaMemsetAsync(cnt, 0, sizeof(int32_t) * (3 * B + p->M), st));
  int ccount[MEDUSA_MAX_HEADS + 1] = {0};
  if ((s = heads_impl(p, h, root_in, w, logits, ttok, at<float>(ws, p->o_tval), root, ws, st, ccount)) !=
      MEDUSA_OK)
    return s;
  {   // fused top-k lists -> per-head top lists, head merge and node tokens / positions
    CandArgs c{at<float>(ws, p->o_fcv), at<int32_t>(ws, p->o_fci), B, p->K + 1, p->cand_ld,
               root_in ? 1 : 0};
    for (int k = 0; k <= p->K; ++k) { c.count[k] = ccount[k]; c.rounds[k] = p->need[k]; }
    c.fin_val = at<float>(ws, p->o_finv);
    c.fin_idx = at<int32_t>(ws, p->o_fini);
    MergeArgs mg = merge_args(p, root_in, ttok, at<float>(ws, p->o_tval), root, ws);
    mg.cand_val = c.fin_val;
    mg.cand_idx = c.fin_idx;
    mg.splits = 1;
    for (int k = 0; k <= p->K; ++k) mg.rounds[k] = p->need[k];
    TreeArgs tr{ttok, root, kv->len, p->d.B, p->K, p->d.V, p->n1, p->dparent(), p->ddepth(), p->drank(),
                tok, pos, nullptr, nullptr, p->d_status};
    LAUNCH(p, KN_SELECT, st, launch_cand_select(c, mg, tr, cnt, st));
  }
  if ((s = gather_impl(p, w, tok, ws, st)) != MEDUSA_OK) return s;
  auto tk_of = [&](int l) -> void* {
    return l == 0 ? at<char>(ws, p->o_tk) : at<char>(ws, p->ws_bytes + (size_t)(l - 1) * 2 * layer_kv_bytes(p));
  };
  auto tv_of = [&](int l) -> void* {
    return l == 0 ? at<char>(ws, p->o_tv)
                  : at<char>(ws, p->ws_bytes + (size_t)(l - 1) * 2 * layer_kv_bytes(p) + layer_kv_bytes(p));
  };
  for (int l = 0; l < nl; ++l) {
    medusa_weights wl = *w;
    wl.wq = layers[l].wq;
    wl.wk = layers[l].wk;
    wl.wv = layers[l].wv;
    wl.wo = layers[l].wo;
    medusa_kv kl = *kv;
    kl.k = layers[l].k;
    kl.v = layers[l].v;
    // tensor-core attention reads the bf16 copy of q only
    if ((s = qkv_impl(p, &wl, pos, p->tc_attn && p->tc_nodes ? nullptr : q, tk_of(l), tv_of(l), ws, st,
                      l == 0 ? nullptr : hp)) != MEDUSA_OK)
      return s;
    if ((s = attn_impl(p, q, &kl, tk_of(l), tv_of(l), p->d_mask, o, true, true, ws, st)) != MEDUSA_OK) return s;
    if ((s = out_impl(p, &wl, o, true, hp, true, ws, st, l == 0 ? nullptr : hp)) != MEDUSA_OK) return s;
  }
  float* vlog = at<float>(ws, p->o_vlog);
  if ((s = vlogits_impl(p, w, hp, true, tok, acc, vlog, am, stats, ws, st, false)) != MEDUSA_OK) return s;
  medusa_kv k0 = *kv;
  k0.k = layers[0].k;
  k0.v = layers[0].v;
  CompactArgs c = compact_args(p, &k0, tk_of(0), tv_of(0), path, out->n_acc);
  c.no_copy = nl > 1;
  {   // fused: per-row statistics, acceptance and (one layer) KV compaction
    VerifyArgs v = verify_args(p, tok, acc);
    v.logits = vlog;
    v.am = am;
    v.stats = stats;
    v.retrieve = p->d_retr;
    v.hprime = hp;
    v.out_tok = out->out_tok;
    v.n_acc = out->n_acc;
    v.path_nodes = path;
    v.h_next = out->h_next;
    v.root_next = out->root_next;
    LAUNCH(p, KN_COMMIT, st,
           launch_verify_commit(v, c, cnt + 2 * B, cnt + B, at<float>(ws, p->o_vparts), st));
  }
  for (int l0 = 0; nl > 1 && l0 < nl; l0 += kLayersPerLaunch) {
    CompactLayersArgs g{};
    g.base = c;
    g.base.no_copy = 0;
    g.nl = std::min(kLayersPerLaunch, nl - l0);
    g.write_len = l0 + g.nl == nl;              // the last launch sets len_out
    g.cnt = cnt + 2 * B + p->M;
    for (int i = 0; i < g.nl; ++i) {
      g.kc[i] = layers[l0 + i].k;
      g.vc[i] = layers[l0 + i].v;
      g.tk[i] = tk_of(l0 + i);
      g.tv[i] = tv_of(l0 + i);
    }
    LAUNCH(p, KN_COMPACT, st, launch_kv_compact_layers(g, st));
  }
  return MEDUSA_OK;
}

}  // namespace

medusa_status medusa_step(const medusa_plan* p, const float* h, const int32_t* root_in,
                          const medusa_weights* w, const medusa_kv* kv, medusa_accept acc,
                          const medusa_outputs* out, void* ws, size_t ws_bytes, void* stream) {
  EntryScope scope("medusa_step");
  if (!p || !h || !out) return MEDUSA_ERR_INVALID;
  if (!out->out_tok || !out->n_acc || !out->h_next || !out->root_next) return MEDUSA_ERR_INVALID;
  medusa_status s = check_weights(p, w, true, true, true);
  if (s != MEDUSA_OK) return s;
  if ((s = check_kv(p, kv, true)) != MEDUSA_OK) return s;
  if ((s = check_accept(acc)) != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  const medusa_layer one{w->wq, w->wk, w->wv, w->wo, kv->k, kv->v};
  return step_core(p, h, root_in, w, &one, 1, kv, acc, out, ws, S(stream));
}

size_t medusa_workspace_size_layers(const medusa_plan* p, int n_layers) {
  if (!p || n_layers < 1 || n_layers > MEDUSA_MAX_LAYERS) return 0;
  return layers_ws_bytes(p, n_layers);
}

medusa_status medusa_step_layers(const medusa_plan* p, const float* h, const int32_t* root_in,
                                 const medusa_weights* w, const medusa_layer* layers, int n_layers,
                                 const medusa_kv* kv, medusa_accept acc, const medusa_outputs* out,
                                 void* ws, size_t ws_bytes, void* stream) {
  EntryScope scope("medusa_step_layers");
  if (!p || !h || !out || !layers || n_layers < 1 || n_layers > MEDUSA_MAX_LAYERS) return MEDUSA_ERR_INVALID;
  if (!out->out_tok || !out->n_acc || !out->h_next || !out->root_next) return MEDUSA_ERR_INVALID;
  medusa_status s = check_weights(p, w, true, false, true);
  if (s != MEDUSA_OK) return s;
  if (!w->emb || !aligned16(w->emb)) return MEDUSA_ERR_INVALID;
  for (int l = 0; l < n_layers; ++l) {
    const medusa_layer& L = layers[l];
    if (!L.wq || !L.wk || !L.wv || !L.wo || !L.k || !L.v) return MEDUSA_ERR_INVALID;
    if (!aligned16(L.wq) || !aligned16(L.wk) || !aligned16(L.wv) || !aligned16(L.wo)) return MEDUSA_ERR_INVALID;
  }
  if (!kv || !kv->len || !kv->len_out) return MEDUSA_ERR_INVALID;
  if (p->d.page_size > 0 && !kv->page_table) return MEDUSA_ERR_INVALID;
  if ((s = check_accept(acc)) != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  if (ws_bytes < layers_ws_bytes(p, n_layers)) return MEDUSA_ERR_WORKSPACE;
  return step_core(p, h, root_in, w, layers, n_layers, kv, acc, out, ws, S(stream));
}

// ------------------------------------------------------------------ decode loop
struct medusa_loop {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int32_t* d_tok = nullptr;      // [B][K+1] tokens of the step in flight
  int32_t* d_nacc = nullptr;     // [B]
  long long* d_count = nullptr;  // steps appended so far
};

void medusa_loop_destroy(medusa_loop* L) {
  if (!L) return;
  if (L->exec) cudaGraphExecDestroy(L->exec);
  if (L->graph) cudaGraphDestroy(L->graph);
  if (L->d_tok) cudaFree(L->d_tok);
  if (L->d_nacc) cudaFree(L->d_nacc);
  if (L->d_count) cudaFree(L->d_count);
  delete L;
}

medusa_status medusa_loop_create(const medusa_plan* p, const medusa_weights* w, const medusa_kv* kv,
                                 medusa_accept acc, float* h, int32_t* root, int32_t* tokens,
                                 int32_t* n_acc, int max_steps, void* ws, size_t ws_bytes,
                                 medusa_loop** out) {
  if (!p || !kv || !h || !root || !tokens || !n_acc || !out || max_steps < 1) return MEDUSA_ERR_INVALID;
  if (!kv->len_out || (const int32_t*)kv->len_out != kv->len) return MEDUSA_ERR_INVALID;
  *out = nullptr;
  if (acc.mode == MEDUSA_REJECT && acc.temperature > 0.f) return MEDUSA_ERR_UNSUPPORTED;   // fixed uniforms
  medusa_status s = check_weights(p, w, true, true, true);
  if (s != MEDUSA_OK) return s;
  if ((s = check_kv(p, kv, true)) != MEDUSA_OK) return s;
  if ((s = check_accept(acc)) != MEDUSA_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MEDUSA_OK) return s;
  medusa_loop* L = new (std::nothrow) medusa_loop();
  if (!L) return MEDUSA_ERR_CUDA;
  const int B = p->d.B, W = p->K + 1;
  if (cudaMalloc(&L->d_tok, sizeof(int32_t) * B * W) != cudaSuccess ||
      cudaMalloc(&L->d_nacc, sizeof(int32_t) * B) != cudaSuccess ||
      cudaMalloc(&L->d_count, sizeof(long long)) != cudaSuccess ||
      cudaMemset(L->d_count, 0, sizeof(long long)) != cudaSuccess) {
    medusa_loop_destroy(L);
    return MEDUSA_ERR_CUDA;
  }
  // One step with its state updated in place (h_next = h, root_next = root, len_out = len),
  // then the append, captured on a private stream (the legacy default stream cannot
  // capture).  Per-launch profiling is suspended during the capture.
  cudaStream_t cap = nullptr;
  if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) {
    medusa_loop_destroy(L);
    return MEDUSA_ERR_CUDA;
  }
  const bool prof = p->prof.on;
  p->prof.on = false;
  medusa_outputs o{L->d_tok, L->d_nacc, nullptr, h, root};
  cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    s = medusa_step(p, h, root, w, kv, acc, &o, ws, ws_bytes, cap);
    if (s == MEDUSA_OK && launch_loop_append(L->d_tok, L->d_nacc, B, W, max_steps, L->d_count, tokens,
                                             n_acc, cap) != cudaSuccess)
      s = MEDUSA_ERR_CUDA;
    const cudaError_t e2 = cudaStreamEndCapture(cap, &L->graph);
    if (s == MEDUSA_OK && e2 != cudaSuccess) s = MEDUSA_ERR_CUDA;
  } else {
    s = MEDUSA_ERR_CUDA;
  }
  p->prof.on = prof;
  if (s == MEDUSA_OK && cudaGraphInstantiate(&L->exec, L->graph, 0) != cudaSuccess) s = MEDUSA_ERR_CUDA;
  cudaStreamDestroy(cap);
  if (s != MEDUSA_OK) {
    medusa_loop_destroy(L);
    return s;
  }
  *out = L;
  return MEDUSA_OK;
}

medusa_status medusa_loop_run(medusa_loop* L, int n_steps, void* stream) {
  if (!L || n_steps < 0) return MEDUSA_ERR_INVALID;
  for (int i = 0; i < n_steps; ++i)
    if (cudaGraphLaunch(L->exec, S(stream)) != cudaSuccess) return MEDUSA_ERR_CUDA;
  return MEDUSA_OK;
}

medusa_status medusa_loop_steps(const medusa_loop* L, void* stream, long long* steps) {
  if (!L || !steps) return MEDUSA_ERR_INVALID;
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaMemcpy(steps, L->d_count, sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  return MEDUSA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ optimized tree on the device
extern "C" medusa_status medusa_tree_greedy_device(int K, const int* s, int smax, const double* a, int N,
                                                   int32_t* parent, int32_t* rank, double* expected,
                                                   void* stream) {
  EntryScope scope("medusa_tree_greedy_device");
  if (K < 1 || K > MEDUSA_MAX_HEADS || !s || !a || !parent || !rank) return MEDUSA_ERR_INVALID;
  if (smax < 1 || smax > MEDUSA_MAX_TOPS || N < 1 || N > MEDUSA_MAX_NODES - 1) return MEDUSA_ERR_INVALID;
  long cart = 0, level = 1;                      // nodes of the Cartesian tree (root excluded)
  for (int k = 0; k < K; ++k) {
    if (s[k] < 1 || s[k] > smax) return MEDUSA_ERR_INVALID;
    level = std::min<long>(level * s[k], 1L << 20);
    cart += level;
  }
  if (cart < N) return MEDUSA_ERR_INVALID;
  medusa::TreeGreedyArgs g{};
  g.acc = a;
  g.K = K;
  g.smax = smax;
  g.N = N;
  g.fmax = N * smax + smax;
  for (int k = 0; k < K; ++k) g.s[k] = s[k];
  g.parent = parent;
  g.rank = rank;
  g.expected = expected;
  if (medusa::launch_tree_greedy(g, S(stream)) != cudaSuccess) return MEDUSA_ERR_CUDA;
  return MEDUSA_OK;
}
