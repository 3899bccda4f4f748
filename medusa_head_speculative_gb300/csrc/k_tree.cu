// Candidate selection and tree construction of the Medusa step.
//   cand_select   the step's selection: per head the merge of the candidate lists that the
//                 vocab projections wrote (fused top-k), then per sequence the root, the
//                 heads' top-s_k and the node tokens and depth position ids
//   topk_partial  (per-stage entry point, from stored logits) per (sequence, head, vocab
//   topk_merge    slice) the 16 best (logit, token) pairs, then their merge
//   tree_build    node tokens and depth position ids; ancestor bitmask and root->leaf paths
//   rope_split    q/k/v of the tree nodes with rotary embedding at the node positions
// Sources: "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads" §3.4 Tree Attention, Steps 1-4; "MEDUSA 精读" section 6 (tree mask, tree position
// ids, flatten/restore indices).  Order of candidates: larger logit first, lower token id
// on equal logits.
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "topk.cuh"

namespace medusa {

// The 16 best (logit, token) pairs of one vocab slice of one head, by a 256-thread CTA.
// When the slice starts on a 16-byte boundary each thread loads F float4 of it (4F <= 16
// logits, all loads issued first), sorts them with a network and the warp merges the 32
// sorted lists; otherwise per-thread lists are filled by insertion.  The 8 warps' lists
// (one run of up to 16 per warp) are then spread 4 entries per lane over warp 0 and merged
// the same way.  NaN logits never enter a list.
__device__ void slice_topk(const TopkArgs& a, int sp, int k, int b) {
  __shared__ float sv[8][kTops];
  __shared__ int si[8][kTops];
  const float* z = a.logits + ((long)b * a.nh + k) * a.V;
  const int lo = sp * a.chunk, hi = min(a.V, lo + a.chunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto local = [&](auto L) {                            // N logits per thread, loads first
    constexpr int N = sizeof(L.v) / sizeof(float);
    L.init();
    float x[N];
#pragma unroll
    for (int u = 0; u < N; ++u) {
      const int v = lo + threadIdx.x + u * blockDim.x;
      x[u] = v < hi ? z[v] : NEG_INF;
    }
#pragma unroll
    for (int u = 0; u < N; ++u) {
      const int v = lo + threadIdx.x + u * blockDim.x;
      if (v < hi) L.insert(x[u], v);
    }
    warp_merge(L, sv[warp], si[warp], a.rounds[k]);
  };
  // F float4 per thread (loads first), sorted into a list of NP = 4, 8 or 16 entries
  auto local_vec = [&](auto L, auto f) {
    constexpr int NP = sizeof(L.v) / sizeof(float);
    constexpr int F = decltype(f)::value;
    const float4* z4 = reinterpret_cast<const float4*>(z);
    const int q0 = lo >> 2, q1 = hi >> 2;
    float4 x[F];
#pragma unroll
    for (int u = 0; u < F; ++u) {
      const int q = q0 + threadIdx.x + u * blockDim.x;
      x[u] = q < q1 ? z4[q] : make_float4(NEG_INF, NEG_INF, NEG_INF, NEG_INF);
    }
#pragma unroll
    for (int u = 0; u < F; ++u) {
      const int q = q0 + threadIdx.x + u * blockDim.x;
      const float e[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const bool ok = q < q1 && !(e[c] != e[c]);
        L.v[4 * u + c] = ok ? e[c] : NEG_INF;
        L.i[4 * u + c] = ok ? 4 * q + c : NO_IDX;
      }
    }
#pragma unroll
    for (int t = 4 * F; t < NP; ++t) { L.v[t] = NEG_INF; L.i[t] = NO_IDX; }
    bitonic_sort_desc(L.v, L.i);
    warp_merge(L, sv[warp], si[warp], a.rounds[k]);
  };
  const int bd = (int)blockDim.x;
  const bool vec = (a.V & 3) == 0 && (a.chunk & 3) == 0;   // slices start on 16 bytes
  const int n4 = (hi - lo + 3) >> 2;
  if (vec && n4 <= bd) {
    local_vec(TopListN<4>{}, std::integral_constant<int, 1>{});
  } else if (vec && n4 <= 2 * bd) {
    local_vec(TopListN<8>{}, std::integral_constant<int, 2>{});
  } else if (vec && n4 <= 3 * bd) {
    local_vec(TopListN<16>{}, std::integral_constant<int, 3>{});
  } else if (vec && n4 <= 4 * bd) {
    local_vec(TopListN<16>{}, std::integral_constant<int, 4>{});
  } else if (hi - lo <= 4 * bd) {
    local(TopListN<4>{});
  } else if (hi - lo <= 8 * (int)blockDim.x) {
    local(TopListN<8>{});
  } else if (hi - lo <= 12 * (int)blockDim.x) {
    local(TopListN<12>{});
  } else {
    TopList L;
    L.init();
    for (int v = lo + threadIdx.x; v < hi; v += blockDim.x) L.insert(z[v], v);
    warp_merge(L, sv[warp], si[warp], a.rounds[k]);
  }
  __syncthreads();
  if (warp == 0) {
    TopListN<4> L;                                  // lane l: entries 4(l/8).. of warp l%8
#pragma unroll
    for (int t = 0; t < 4; ++t) { L.v[t] = sv[lane & 7][4 * (lane >> 3) + t]; L.i[t] = si[lane & 7][4 * (lane >> 3) + t]; }
    const long o = (((long)b * a.nh + k) * a.splits + sp) * kTops;
    warp_merge(L, a.cand_val + o, a.cand_idx + o, a.rounds[k]);
  }
}

__global__ void __launch_bounds__(256) topk_partial_kernel(TopkArgs a) {
  pdl_trigger();
  pdl_wait();
  slice_topk(a, blockIdx.x, blockIdx.y + a.k0, blockIdx.z);
}

cudaError_t launch_topk_partial(const TopkArgs& a, cudaStream_t st) {
  dim3 grid(a.splits, a.nh - a.k0, a.B);
  return launch_kernel(topk_partial_kernel, grid, dim3(256), 0, st, 1, a);
}

// Merge of sequence b's vocab slices: warp w merges heads w, w+8 (head 0 is the LM head,
// heads 1..K the Medusa heads) into their final top-16; writes the root and the heads'
// lists.  Candidates are read through L2 (they may come from other CTAs of this launch).
__device__ void merge_heads(const MergeArgs& a, int b, float (*tv)[kTops], int (*ti)[kTops],
                            int* s_root) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int nh = a.K + 1;
  for (int k = warp + a.k0; k < nh; k += nw) {
    if (a.splits == 1) {           // one list per head: it is the head's final list
      const long o = ((long)b * nh + k) * kTops;
      const int r = a.rounds[k] < 1 || a.rounds[k] > kTops ? kTops : a.rounds[k];
      if (lane < kTops) {
        tv[k][lane] = lane < r ? __ldcg(a.cand_val + o + lane) : NEG_INF;
        ti[k][lane] = lane < r ? __ldcg(a.cand_idx + o + lane) : NO_IDX;
      }
      continue;
    }
    TopList L;
    L.init();
    if (lane < a.splits) {
      const long o = (((long)b * nh + k) * a.splits + lane) * kTops;
#pragma unroll
      for (int t = 0; t < kTops; ++t) { L.v[t] = __ldcg(a.cand_val + o + t); L.i[t] = __ldcg(a.cand_idx + o + t); }
    }
    warp_merge(L, tv[k], ti[k], a.rounds[k]);
  }
  __syncthreads();
  if (tid == 0) {
    int r = a.root_in ? a.root_in[b] : (a.k0 == 0 ? ti[0][0] : -1);
    if (r < 0 || r >= a.V) { set_flag(a.status, MEDUSA_FLAG_TOKEN_RANGE); r = 0; }
    a.root_out[b] = r;
    *s_root = r;
  }
  for (int e = tid; e < a.K * kTops; e += blockDim.x) {
    const int k = e / kTops, t = e - k * kTops;
    a.topk_tok[(long)b * a.K * kTops + e] = ti[k + 1][t];
    a.topk_val[(long)b * a.K * kTops + e] = tv[k + 1][t];
  }
  __syncthreads();
}

// Node tokens and position ids of sequence b, from the merged lists in shared memory.
__device__ void node_tokens(const TreeArgs& a, int b, const int (*ti)[kTops], int root) {
  if (a.n1 <= 0) return;                     // selection only (no tree)
  int L = a.len[b];
  if (L < 0) L = 0;
  for (int n = threadIdx.x; n < a.n1; n += blockDim.x) {
    int t = root;
    if (n > 0) t = ti[a.depth[n]][a.rank[n]];
    if (t < 0 || t >= a.V) { set_flag(a.status, MEDUSA_FLAG_TOKEN_RANGE); t = 0; }
    a.tok[(long)b * a.n1 + n] = t;
    a.pos[(long)b * a.n1 + n] = L + a.depth[n];
  }
}

__global__ void __launch_bounds__(256) topk_merge_kernel(MergeArgs a) {
  __shared__ float tv[MEDUSA_MAX_HEADS + 1][kTops];
  __shared__ int ti[MEDUSA_MAX_HEADS + 1][kTops];
  __shared__ int s_root;
  pdl_trigger();
  pdl_wait();
  merge_heads(a, blockIdx.x, tv, ti, &s_root);
}

cudaError_t launch_topk_merge(const MergeArgs& a, cudaStream_t st) {
  return launch_kernel(topk_merge_kernel, dim3(a.B), dim3(256), 0, st, 1, a);
}

int topk_partial_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, topk_partial_kernel, 256, 0) != cudaSuccess) n = 0;
  return n;
}

// Selection from the fused top-k candidates: CTA (head k, sequence b) reads the head's
// slot lists (each sorted, written by the projection's CTAs), thread t merging slots t,
// t + 256, ... by insertion until an entry no longer enters; the warps' lists and then the
// 8 warp lists are merged into the head's final list.  The last CTA of a sequence takes the
// heads' final lists, picks the root and writes the node tokens and positions.
__global__ void __launch_bounds__(256) cand_select_kernel(CandArgs c, MergeArgs m, TreeArgs tr,
                                                          int32_t* counter) {
  __shared__ float sv[8][kTops];
  __shared__ int si[8][kTops];
  __shared__ float tv[MEDUSA_MAX_HEADS + 1][kTops];
  __shared__ int ti[MEDUSA_MAX_HEADS + 1][kTops];
  __shared__ int s_root, s_last;
  pdl_trigger();
  pdl_wait();
  const int k = blockIdx.x + c.k0, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, n = c.count[k];
  const long base = ((long)b * c.nh + k) * c.ld;
  TopList L;
  L.init();
  auto load = [&](int slot, float (&v)[kTops], int (&ix)[kTops]) {
    const float4* pv = reinterpret_cast<const float4*>(c.cand_val + (base + slot) * kTops);
    const int4* pi = reinterpret_cast<const int4*>(c.cand_idx + (base + slot) * kTops);
#pragma unroll
    for (int q = 0; q < kTops / 4; ++q) {
      const float4 x = __ldcg(pv + q);
      const int4 y = __ldcg(pi + q);
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
      ix[4 * q] = y.x; ix[4 * q + 1] = y.y; ix[4 * q + 2] = y.z; ix[4 * q + 3] = y.w;
    }
  };
  if ((int)threadIdx.x < n) load(threadIdx.x, L.v, L.i);     // a sorted list as it stands
  for (int slot = threadIdx.x + blockDim.x; slot < n; slot += blockDim.x) {
    float v[kTops];
    int ix[kTops];
    load(slot, v, ix);
#pragma unroll
    for (int t = 0; t < kTops; ++t) {
      if (!better(v[t], ix[t], L.v[kTops - 1], L.i[kTops - 1])) break;
      L.insert(v[t], ix[t]);
    }
  }
  warp_merge(L, sv[warp], si[warp], c.rounds[k]);
  __syncthreads();
  {
    const long o = ((long)b * c.nh + k) * kTops;
    rank_merge(sv, si, 8, c.rounds[k], c.fin_val + o, c.fin_idx + o, threadIdx.x, blockDim.x);
  }
  __threadfence();                 // the head's final list, before the count below
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(counter + b, 1) == c.nh - c.k0 - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  merge_heads(m, b, tv, ti, &s_root);
  node_tokens(tr, b, ti, s_root);
  if (threadIdx.x == 0) counter[b] = 0;
}

cudaError_t launch_cand_select(const CandArgs& c, const MergeArgs& m, const TreeArgs& tr,
                               int32_t* counter, cudaStream_t st) {
  if (m.splits != 1 || m.cand_val != c.fin_val || m.cand_idx != c.fin_idx) return cudaErrorInvalidValue;
  dim3 grid(c.nh - c.k0, c.B);
  return launch_kernel(cand_select_kernel, grid, dim3(256), 0, st, 1, c, m, tr, counter);
}

// One CTA per sequence: node tokens and position ids.  Block 0 also writes the per-tree
// tables (ancestor bitmask, root->leaf paths), which are the same for every sequence.
__global__ void __launch_bounds__(256) tree_build_kernel(TreeArgs a) {
  __shared__ int haschild[MEDUSA_MAX_NODES];
  __shared__ int leafidx[MEDUSA_MAX_NODES];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  int L = a.len[b];
  if (L < 0) L = 0;
  for (int n = tid; n < a.n1; n += blockDim.x) {
    int t = a.root[b];
    if (n > 0) t = a.topk_tok[((long)b * a.K + a.depth[n] - 1) * kTops + a.rank[n]];
    if (t < 0 || t >= a.V) { set_flag(a.status, MEDUSA_FLAG_TOKEN_RANGE); t = 0; }
    a.tok[(long)b * a.n1 + n] = t;
    a.pos[(long)b * a.n1 + n] = L + a.depth[n];
  }
  if (b != 0) return;
  for (int n = tid; n < MEDUSA_MAX_NODES; n += blockDim.x) haschild[n] = 0;
  __syncthreads();
  for (int n = tid; n < a.n1; n += blockDim.x) {
    uint32_t wmask[kMaskWords];
#pragma unroll
    for (int q = 0; q < kMaskWords; ++q) wmask[q] = 0u;
    for (int j = n, guard = 0; j >= 0 && guard <= MEDUSA_MAX_HEADS + 1; j = a.parent[j], ++guard)
      wmask[j >> 5] |= 1u << (j & 31);
#pragma unroll
    for (int q = 0; q < kMaskWords; ++q) a.mask[(long)n * kMaskWords + q] = wmask[q];
    if (n > 0) haschild[a.parent[n]] = 1;
  }
  __syncthreads();
  if (tid == 0) {
    int c = 0;
    for (int n = 0; n < a.n1; ++n) leafidx[n] = haschild[n] ? -1 : c++;
  }
  const int W = a.K + 1;
  for (int e = tid; e < a.n1 * W; e += blockDim.x) a.retrieve[e] = -1;
  __syncthreads();
  for (int n = tid; n < a.n1; n += blockDim.x) {
    const int p = leafidx[n];
    if (p < 0) continue;
    for (int j = n; j >= 0; j = a.parent[j]) a.retrieve[(long)p * W + a.depth[j]] = j;
  }
}

cudaError_t launch_tree_build(const TreeArgs& a, cudaStream_t st) {
  return launch_kernel(tree_build_kernel, dim3(a.B), dim3(256), 0, st, 1, a);
}

// One CTA per node row.  cos/sin of pos * theta_i come from the plan's table (computed on
// the host in double precision, rounded to float) and are applied to every query and key
// head (rotate-half convention).  Positions past the table are clamped and flagged.
template <typename T>
__global__ void __launch_bounds__(1024) rope_split_kernel(
    const float* __restrict__ qkv, const int32_t* __restrict__ pos, int Hq, int Hkv, int dh,
    const float* __restrict__ table, int rows, uint32_t* status, float* __restrict__ q,
    bf16* __restrict__ qb, T* __restrict__ tk, T* __restrict__ tv) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float cs[];                      // [dh/2] cos, [dh/2] sin
  const int m = blockIdx.x, half = dh / 2;
  int p = pos[m];
  if (p < 0 || p >= rows) {
    if (threadIdx.x == 0) set_flag(status, MEDUSA_FLAG_KV_CAPACITY);
    p = p < 0 ? 0 : rows - 1;
  }
  for (int i = threadIdx.x; i < dh; i += blockDim.x) cs[i] = table[(long)p * dh + i];
  __syncthreads();
  const int W = (Hq + 2 * Hkv) * dh;
  const float* row = qkv + (long)m * W;
  // Every load of a batch goes out before its first store (one round trip per batch).
  constexpr int NB = 4;
  const int npair = (Hq + Hkv) * half, step = blockDim.x;
  for (int e0 = threadIdx.x; e0 < npair; e0 += NB * step) {
    float a[NB], bb[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int e = e0 + u * step;
      if (e < npair) {
        const int h = e / half, i = e - h * half;
        a[u] = row[h * dh + i];
        bb[u] = row[h * dh + i + half];
      }
    }
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int e = e0 + u * step;
      if (e >= npair) continue;
      const int h = e / half, i = e - h * half;
      const float c = cs[i], s = cs[half + i];
      const float y0 = a[u] * c - bb[u] * s;
      const float y1 = bb[u] * c + a[u] * s;
      if (h < Hq) {
        const long o = ((long)m * Hq + h) * dh;
        q[o + i] = y0;
        q[o + i + half] = y1;
        if (qb) {
          qb[o + i] = __float2bfloat16_rn(y0);
          qb[o + i + half] = __float2bfloat16_rn(y1);
        }
      } else {
        T* ko = tk + ((long)m * Hkv + (h - Hq)) * dh;
        ko[i] = from_f32<T>(y0);
        ko[i + half] = from_f32<T>(y1);
      }
    }
  }
  const float* vr = row + (Hq + Hkv) * dh;
  const int nv = Hkv * dh;
  for (int e0 = threadIdx.x; e0 < nv; e0 += NB * step) {
    float x[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u)
      if (e0 + u * step < nv) x[u] = vr[e0 + u * step];
#pragma unroll
    for (int u = 0; u < NB; ++u)
      if (e0 + u * step < nv) tv[(long)m * nv + e0 + u * step] = from_f32<T>(x[u]);
  }
}

cudaError_t launch_rope_split(const float* qkv, const int32_t* pos, int M, int Hq, int Hkv, int dh,
                              const float* table, int rows, uint32_t* status, int dtype, float* q,
                              bf16* qb, void* tk, void* tv, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const size_t smem = dh * sizeof(float);
  if (dtype == 0)
    return launch_kernel(rope_split_kernel<float>, dim3(M), dim3(1024), smem, st, 1, qkv, pos, Hq, Hkv,
                         dh, table, rows, status, q, qb, reinterpret_cast<float*>(tk),
                         reinterpret_cast<float*>(tv));
  return launch_kernel(rope_split_kernel<bf16>, dim3(M), dim3(1024), smem, st, 1, qkv, pos, Hq, Hkv, dh,
                       table, rows, status, q, qb, reinterpret_cast<bf16*>(tk),
                       reinterpret_cast<bf16*>(tv));
}

void rope_table(float base, int dh, int rows, float* out) {
  for (int p = 0; p < rows; ++p)
    for (int i = 0; i < dh / 2; ++i) {
      const double theta = std::pow((double)base, -2.0 * i / dh);
      out[(long)p * dh + i] = (float)std::cos(p * theta);
      out[(long)p * dh + dh / 2 + i] = (float)std::sin(p * theta);
    }
}

}  // namespace medusa
