// Workspace-free variant of the heads stage: medusa_heads_noalloc().
//
// Some callers cannot allocate device memory when they want to run the heads: a serving
// engine that sizes every buffer up front and forbids allocation on its decode path, a
// plug-in that lives inside another framework's memory pool and may not call cudaMalloc
// behind its back, or code that must not allocate because the stream may be in the
// middle of being captured into a CUDA graph.  This entry point needs no workspace from
// them: its scratch (the head activations and the fused top-k's candidate lists) lives in
// one fixed array in device global memory that belongs to this library.
//
// Limits and behaviour:
//   * The array holds MEDUSA_NOALLOC_SCRATCH_BYTES (4 MiB) on every GPU that loads the
//     library, for as long as the process lives.  Plans whose heads scratch needs more
//     (the candidate lists, B * (K+1) * slots * 128 bytes with slots = V/128 at batch >= 2
//     and up to a few hundred at batch 1, plus B * K * d * 8 bytes of head activations) are
//     rejected with MEDUSA_ERR_UNSUPPORTED before anything is launched.
//   * The first call on a device looks up the array's device address (a CUDA runtime
//     symbol lookup, no allocation) with that device current; make that first call
//     before starting any stream capture.  The address is kept per device and CUDA
//     context: after cudaDeviceReset the next call looks it up again, so that call too
//     should come before any capture.
//   * Every call shares the one array and leaves its last contents there; nothing in it
//     has to start at zero (each call clears its completion counts with a memset and
//     overwrites everything else it reads).  Calls whose
//     GPU work overlaps (different streams, or different plans at the same time) race on
//     the array: order them on one stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/medusa.h"
#include "kernels.h"
#include "launch.cuh"

using namespace medusa;

// The scratch array itself (file scope, one copy per GPU that loads the library).
static __device__ __align__(256) unsigned char g_heads_scratch[MEDUSA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
  CUcontext ctx;      // the context the address was looked up in
  void* ptr;          // device address of g_heads_scratch in that context
};
ScratchAddr g_scratch[kMaxDevices] = {};

// The calling thread's current CUDA context (null before the runtime has made one
// current), through the driver entry point the runtime hands out.
CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Host code must not use g_heads_scratch's name as an address: it is only a host-side
// stand-in for the device symbol.  The real address is looked up once per device and
// context, and again when the current context is not the one it was found in (after a
// cudaDeviceReset the runtime loads the module into a new primary context).
medusa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MEDUSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchAddr& e = g_scratch[dev];
  const CUcontext ctx = current_context();
  if (!e.ptr || !ctx || ctx != e.ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_heads_scratch) != cudaSuccess || !p) return MEDUSA_ERR_CUDA;
    e.ptr = p;
    e.ctx = current_context();          // current now: the lookup made it so
  }
  *out = e.ptr;
  return MEDUSA_OK;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct Layout {
  size_t u, uhi, ulo, hhi, hlo, cv, ci, fv, fi, cnt, total;
};

Layout layout_of(const HeadsPlanView& v, int ld) {
  const size_t B = v.dims.B, K = v.K, D = v.dims.d;
  const size_t tc = v.tc_heads ? 1 : 0;
  Layout l{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = up256(off + bytes); return o; };
  l.u = take(B * K * D * 4);
  l.uhi = take(tc * B * K * D * 2);
  l.ulo = take(tc * B * K * D * 2);
  l.hhi = take(tc * B * D * 2);
  l.hlo = take(tc * B * D * 2);
  l.cv = take(B * (K + 1) * (size_t)ld * kTops * 4);
  l.ci = take(B * (K + 1) * (size_t)ld * kTops * 4);
  l.fv = take(B * (K + 1) * kTops * 4);
  l.fi = take(B * (K + 1) * kTops * 4);
  l.cnt = take(B * 4);
  l.total = off;
  return l;
}

bool ok16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// The heads' projections with the fused top-k (each CTA keeps its rows' best candidates;
// no logits) and the candidate selection, as the step runs them, but with all 16 ranks of
// every head kept, as medusa_heads() returns them.
extern "C" medusa_status medusa_heads_noalloc(const medusa_plan* plan, const float* h,
                                              const int32_t* root_in, const medusa_weights* w,
                                              int32_t* topk_tok, float* topk_val, int32_t* root,
                                              void* stream) {
  EntryScope scope("medusa_heads_noalloc");
  HeadsPlanView v;
  if (!heads_plan_view(plan, &v)) return MEDUSA_ERR_INVALID;
  const int B = v.dims.B, K = v.K, D = v.dims.d, V = v.dims.V;
  const size_t es = v.dims.dtype == MEDUSA_F32 ? 4 : 2;
  const bool tc = v.tc_heads;

  // u_k = SiLU(W1_k h) + h; on the row-dot path z_0 = LM h joins this launch when the root
  // is not given
  MatArgs a{};
  a.nseg = K;
  a.M = B;
  a.k = D;
  a.ldo = (long)K * D;
  a.epi = EPI_SILU_RES;
  a.res_f32 = h;
  a.ldr = D;
  for (int k = 0; k < K; ++k) {
    a.seg[k].rows = D;
    a.seg[k].out_off = k * D;
  }
  const bool lm_first = !tc && !root_in;
  if (lm_first) {
    a.seg[K].rows = V;
    a.seg[K].cand = 1;
    a.seg[K].head = 0;
    a.seg[K].rounds = kTops;
    a.nseg = K + 1;
  }
  // z_k = W2_k u_k (and z_0 here when it did not join the first launch)
  const int k0 = root_in || lm_first ? 1 : 0;
  MatArgs b{};
  b.nseg = K + 1 - k0;
  b.M = B;
  b.k = D;
  b.epi = EPI_STORE;
  for (int i = 0; i < b.nseg; ++i) {
    b.seg[i].rows = V;
    b.seg[i].cand = 1;
    b.seg[i].head = i + k0;
    b.seg[i].rounds = kTops;
  }
  // candidate slots of both launches, then the scratch they need
  int count[MEDUSA_MAX_HEADS + 1] = {0};
  int ld = 1;
  auto geometry = [&](MatArgs& x, int i0) -> bool {
    for (int i = i0; i < x.nseg; ++i) {
      int n = 0, c0 = 0;
      if (!cand_geometry(x, i, tc, v.dims.dtype, &n, &c0) || n < 1) return false;
      x.seg[i].slot0 = c0;
      count[x.seg[i].head] = n;
      ld = n > ld ? n : ld;
    }
    return true;
  };
  if ((lm_first && !geometry(a, K)) || !geometry(b, 0)) return MEDUSA_ERR_CUDA;
  const Layout l = layout_of(v, ld);
  if (l.total > (size_t)MEDUSA_NOALLOC_SCRATCH_BYTES) return MEDUSA_ERR_UNSUPPORTED;
  if (!h || !w || !topk_tok || !topk_val || !root) return MEDUSA_ERR_INVALID;
  if (!ok16(w->w1) || !ok16(w->w2) || (!root_in && !ok16(w->lm))) return MEDUSA_ERR_INVALID;
  void* base = nullptr;
  medusa_status s = scratch_address(&base);
  if (s != MEDUSA_OK) return s;
  char* sc = static_cast<char*>(base);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* u = reinterpret_cast<float*>(sc + l.u);
  bf16* uhi = tc ? reinterpret_cast<bf16*>(sc + l.uhi) : nullptr;
  bf16* ulo = tc ? reinterpret_cast<bf16*>(sc + l.ulo) : nullptr;
  bf16* hhi = tc ? reinterpret_cast<bf16*>(sc + l.hhi) : nullptr;
  bf16* hlo = tc ? reinterpret_cast<bf16*>(sc + l.hlo) : nullptr;
  float* cv = reinterpret_cast<float*>(sc + l.cv);
  int32_t* ci = reinterpret_cast<int32_t*>(sc + l.ci);
  float* fv = reinterpret_cast<float*>(sc + l.fv);
  int32_t* fi = reinterpret_cast<int32_t*>(sc + l.fi);
  int32_t* cnt = reinterpret_cast<int32_t*>(sc + l.cnt);
  // the selection's completion counts start at zero (a memset, not an allocation)
  if (cudaMemsetAsync(cnt, 0, sizeof(int32_t) * B, st) != cudaSuccess) return MEDUSA_ERR_CUDA;

  a.out = u;
  a.out_hi = uhi;
  a.out_lo = ulo;
  for (int k = 0; k < K; ++k) {
    MatSeg& g = a.seg[k];
    g.w = static_cast<const char*>(w->w1) + (size_t)k * D * D * es;
    g.x = h; g.a_hi = hhi; g.a_lo = hlo; g.ldx = D;
  }
  if (lm_first) {
    a.seg[K].w = w->lm;
    a.seg[K].x = h;
    a.seg[K].ldx = D;
  }
  for (MatArgs* x : {&a, &b}) {
    x->cand_val = cv;
    x->cand_idx = ci;
    x->cand_nh = K + 1;
    x->cand_ld = ld;
  }
  if (tc && launch_split(h, hhi, hlo, (long)B * D, st) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if ((tc ? launch_umma_gemm(a, v.status, st) : launch_rowdot(a, v.dims.dtype, st)) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  for (int i = 0; i < b.nseg; ++i) {
    MatSeg& g = b.seg[i];
    const int k = i + k0;                                  // 0: the LM head
    if (k == 0) {
      g.w = w->lm;
      g.x = h; g.a_hi = hhi; g.a_lo = hlo; g.ldx = D;
    } else {
      g.w = static_cast<const char*>(w->w2) + (size_t)(k - 1) * V * D * es;
      g.x = u + (size_t)(k - 1) * D;
      g.a_hi = uhi ? uhi + (size_t)(k - 1) * D : nullptr;
      g.a_lo = ulo ? ulo + (size_t)(k - 1) * D : nullptr;
      g.ldx = (long)K * D;
    }
  }
  if ((tc ? launch_umma_gemm(b, v.status, st) : launch_rowdot(b, v.dims.dtype, st)) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  CandArgs c{cv, ci, B, K + 1, ld, root_in ? 1 : 0};
  for (int k = 0; k <= K; ++k) { c.count[k] = count[k]; c.rounds[k] = kTops; }
  c.fin_val = fv;
  c.fin_idx = fi;
  MergeArgs mg{fv, fi, B, K, V, 1, root_in, topk_tok, topk_val, root, v.status};
  mg.k0 = c.k0;
  TreeArgs tr{};                                           // no tree: selection only
  tr.n1 = 0;
  if (launch_cand_select(c, mg, tr, cnt, st) != cudaSuccess) return MEDUSA_ERR_CUDA;
  return MEDUSA_OK;
}
