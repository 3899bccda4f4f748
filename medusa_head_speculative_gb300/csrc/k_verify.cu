// Verification and commit of the Medusa step.
//   verify_stats   per node row of the verification logits: greedy token (lowest id on
//                  ties) and, for typical acceptance, max z/T, log-sum-exp and entropy, in
//                  one pass (running max with rescaled sums)
//   verify_accept  accept flags, longest accepted root->leaf path, step outputs
//   kv_compact     copies the kept nodes' keys/values into the cache after the prefix
// Sources: "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads" §3.4 Tree Attention Step 6 and Typical Acceptance Scheme (criterion
// p(x) > min(eps, delta exp(-H)), first token greedy and always kept, longest accepted
// prefix); "MEDUSA 精读" section 3 (only the accepted path stays in the KV cache).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace medusa {

__device__ __forceinline__ void block_argmax(float& v, int& i, float* sv, int* si) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  warp_argmax(v, i);
  __syncthreads();
  if (lane == 0) { sv[warp] = v; si[warp] = i; }
  __syncthreads();
  if (warp == 0) {
    v = lane < nw ? sv[lane] : -INFINITY;
    i = lane < nw ? si[lane] : 0x7fffffff;
    warp_argmax(v, i);
    if (lane == 0) { sv[0] = v; si[0] = i; }
  }
  __syncthreads();
  v = sv[0];
  i = si[0];
}

// Softmax statistics relative to a running max m: S = sum e^(y-m), U = sum (y-m) e^(y-m).
struct SoftStat {
  float m, S, U;
};
__device__ __forceinline__ SoftStat stat_merge(SoftStat a, SoftStat b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return a;
  SoftStat r{M, 0.f, 0.f};
  if (a.m != -INFINITY) {
    const float e = __expf(a.m - M);
    r.S += e * a.S;
    r.U += e * (a.U + (a.m - M) * a.S);
  }
  if (b.m != -INFINITY) {
    const float e = __expf(b.m - M);
    r.S += e * b.S;
    r.U += e * (b.U + (b.m - M) * b.S);
  }
  return r;
}
__device__ __forceinline__ void stat_add(SoftStat& s, float y) {
  if (y > s.m) {
    if (s.m != -INFINITY) {
      const float e = __expf(s.m - y);
      s.U = e * (s.U + (s.m - y) * s.S);
      s.S *= e;
    }
    s.m = y;
  }
  const float e = __expf(y - s.m);
  s.S += e;
  s.U += (y - s.m) * e;
}

// Partial statistics of logits [v0, v1) of one node row: max/argmax and, for typical
// acceptance, the running-max softmax sums of z/T.  Result valid in thread 0.
struct RowPart {
  float bv;
  int bi;
  SoftStat st;
  bool nonfinite;
};
// Each thread visits its logits in increasing index order, so a strict ">" keeps the
// lowest index among equal maxima (the merge across threads breaks ties by index).  The
// softmax sums move their reference maximum once per batch of 32 logits.  A non-finite
// logit makes the running sum of the logits non-finite.
__device__ RowPart row_part(const VerifyArgs& a, int row, int v0, int v1) {
  __shared__ float sv[32], sS[32], sU[32];
  __shared__ int si[32];
  constexpr int NB = 4;                                // float4 loads in flight per thread
  const float* z = a.logits + (long)row * a.V;
  const bool typ = a.typical != 0;
  const float invT = typ ? 1.f / a.temperature : 0.f;
  RowPart r{-INFINITY, 0x7fffffff, SoftStat{-INFINITY, 0.f, 0.f}, false};
  float sx = 0.f;
  auto raise_to = [&](float bm) {                      // move the reference maximum up to bm
    if (bm > r.st.m) {
      if (r.st.m != -INFINITY) {
        const float f = __expf(r.st.m - bm);
        r.st.U = f * (r.st.U + (r.st.m - bm) * r.st.S);
        r.st.S *= f;
      }
      r.st.m = bm;
    }
  };
  const bool vec = (a.V & 3) == 0 && (v0 & 3) == 0;
  const int q0 = vec ? v0 / 4 : 0, q1 = vec ? v1 / 4 : 0;
  for (int qb = q0 + threadIdx.x; qb < q1; qb += NB * blockDim.x) {
    float4 x[NB];
    bool ok[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int q = qb + u * blockDim.x;
      ok[u] = q < q1;
      x[u] = ok[u] ? reinterpret_cast<const float4*>(z)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      if (!ok[u]) continue;
      const int q = qb + u * blockDim.x;
      const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sx += xs[e];
        if (xs[e] > r.bv) { r.bv = xs[e]; r.bi = 4 * q + e; }
        bm = fmaxf(bm, xs[e]);
      }
    }
    if (typ) {
      raise_to(bm * invT);
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        if (!ok[u]) continue;
        const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float d = xs[e] * invT - r.st.m;
          const float w = __expf(d);
          r.st.S += w;
          r.st.U += d * w;
        }
      }
    }
  }
  for (int v = (vec ? 4 * q1 : v0) + threadIdx.x; v < v1; v += blockDim.x) {   // ragged tail
    const float x = z[v];
    sx += x;
    if (x > r.bv) { r.bv = x; r.bi = v; }
    if (typ) {
      raise_to(x * invT);
      const float d = x * invT - r.st.m;
      const float w = __expf(d);
      r.st.S += w;
      r.st.U += d * w;
    }
  }
  r.nonfinite = __syncthreads_or(!isfinite(sx)) != 0;   // any thread's logits
  if (typ) {                                   // merge the statistics across the CTA
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      SoftStat other{__shfl_xor_sync(0xffffffffu, r.st.m, o), __shfl_xor_sync(0xffffffffu, r.st.S, o),
                     __shfl_xor_sync(0xffffffffu, r.st.U, o)};
      r.st = stat_merge(r.st, other);
    }
    __syncthreads();
    if (lane == 0) { sv[warp] = r.st.m; sS[warp] = r.st.S; sU[warp] = r.st.U; }
    __syncthreads();
    if (warp == 0) {
      r.st = lane < nw ? SoftStat{sv[lane], sS[lane], sU[lane]} : SoftStat{-INFINITY, 0.f, 0.f};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        SoftStat other{__shfl_xor_sync(0xffffffffu, r.st.m, o), __shfl_xor_sync(0xffffffffu, r.st.S, o),
                       __shfl_xor_sync(0xffffffffu, r.st.U, o)};
        r.st = stat_merge(r.st, other);
      }
    }
    __syncthreads();
  }
  block_argmax(r.bv, r.bi, sv, si);
  return r;
}

// Thread 0: final am / stats of a row from its (merged) partial.
__device__ void row_finish(const VerifyArgs& a, int row, RowPart r) {
  const int b = row / a.n1, n = row - b * a.n1;
  if (r.nonfinite) set_flag(a.status, MEDUSA_FLAG_NONFINITE);
  if (r.bi < 0 || r.bi >= a.V) { set_flag(a.status, MEDUSA_FLAG_TOKEN_RANGE); r.bi = 0; }
  float out[4] = {r.bv, 0.f, 0.f, 0.f};
  if (a.typical) {
    const float logS = logf(r.st.S);
    out[0] = r.st.m;
    out[1] = logS;
    out[2] = logS - r.st.U / r.st.S;           // H = log S - sum(y e^y) / S
    if (n > 0) {
      const int p = a.parent[n];
      const int t = a.tok[(long)b * a.n1 + n];
      out[3] = a.logits[((long)b * a.n1 + p) * a.V + t] / a.temperature;
    }
    if (!isfinite(out[1]) || !isfinite(out[2])) set_flag(a.status, MEDUSA_FLAG_NONFINITE);
  }
  a.am[row] = r.bi;
#pragma unroll
  for (int q = 0; q < 4; ++q) a.stats[(long)row * 4 + q] = out[q];
}

// Statistics of one node row (b, n) by one CTA.
__device__ void row_stats(const VerifyArgs& a, int row) {
  RowPart r = row_part(a, row, 0, a.V);
  if (threadIdx.x == 0) row_finish(a, row, r);
}

__global__ void __launch_bounds__(1024) verify_stats_kernel(VerifyArgs a) {
  pdl_trigger();
  pdl_wait();
  row_stats(a, blockIdx.x);
}

cudaError_t launch_verify_stats(const VerifyArgs& a, cudaStream_t st) {
  return launch_kernel(verify_stats_kernel, dim3(a.B * a.n1), dim3(1024), 0, st, 1, a);
}

// Acceptance of sequence b by one CTA; thread c decides candidate c, thread p walks path
// p.  Statistics are read through L2 (other CTAs of the same launch may have written them).
// Rejection-sampling verification of sequence b (whole CTA).  Thread 0 walks the tree from
// the root: the current node's children, in packed (rank) order, are tested with their own
// uniforms against the mass R not yet rejected at that node (child x kept iff u R < p(x),
// else R -= p(x) and x leaves the distribution); the first kept child becomes the current
// node.  The CTA then draws the next root from the current node's remaining distribution
// by inverse CDF in token order: per-thread contiguous token ranges, their sums scanned in
// thread order, and the thread whose range holds u_final times the total walks it.
__device__ void reject_seq(const VerifyArgs& a, int b) {
  __shared__ int s_path[MEDUSA_MAX_HEADS + 1];
  __shared__ int s_excl[kTops];
  __shared__ int s_m, s_nex, s_v;
  __shared__ float s_sum[1024];
  const int tid = threadIdx.x;
  const long rb = (long)b * a.n1;
  const int W = a.K + 1, ustride = 1 + 16 * a.K;
  const float* uni = a.uniforms + (long)b * ustride;
  if (tid == 0) {
    int u = 0, m = 0, nex = 0;
    s_path[0] = 0;
    for (;;) {
      const float* su = a.stats + (rb + u) * 4;
      const float mu = __ldcg(su), lsu = __ldcg(su + 1);   // max z/T, log sum e^(z/T - max)
      float R = 1.f;
      int j = 0, next = -1;
      nex = 0;
      for (int c = u + 1; c < a.n1 && next < 0; ++c) {
        if (a.parent[c] != u) continue;
        const float px = __expf(__ldcg(a.stats + (rb + c) * 4 + 3) - mu - lsu);   // p_u(tok_c)
        const float uu = __ldg(uni + 1 + 16 * m + j);
        if (uu * R < px) {
          next = c;
        } else {
          R -= px;
          if (nex < kTops) s_excl[nex++] = a.tok[rb + c];
          ++j;
        }
      }
      if (next < 0 || m + 1 >= W) break;
      s_path[++m] = next;
      u = next;
    }
    s_m = m;
    s_nex = nex;
    s_v = -1;
  }
  __syncthreads();
  const int m = s_m, nex = s_nex, last = s_path[m];
  if (!a.logits) {                                       // checked on the host; never read null
    if (tid == 0) set_flag(a.status, MEDUSA_FLAG_TOKEN_RANGE);
    return;
  }
  const float* z = a.logits + (rb + last) * a.V;
  const float mu = __ldcg(a.stats + (rb + last) * 4), invT = 1.f / a.temperature;
  auto weight = [&](int v) {
    for (int e = 0; e < nex; ++e)
      if (s_excl[e] == v) return 0.f;
    return __expf(__ldcg(z + v) * invT - mu);
  };
  const int chunk = (a.V + blockDim.x - 1) / blockDim.x;
  const int v0 = min(a.V, tid * chunk), v1 = min(a.V, v0 + chunk);
  float own = 0.f;
  for (int v = v0; v < v1; ++v) own += weight(v);
  s_sum[tid] = own;
  __syncthreads();
  if (tid == 0) {                                        // exclusive scan in thread order
    float c = 0.f;
    for (int t = 0; t < (int)blockDim.x; ++t) {
      const float x = s_sum[t];
      s_sum[t] = c;
      c += x;
    }
    s_sum[blockDim.x] = c;                               // blockDim.x < 1024
  }
  __syncthreads();
  const float total = s_sum[blockDim.x], thr = __ldg(uni) * total;
  const float before = s_sum[tid];
  if (own > 0.f && before <= thr && thr < before + own) {
    float c = before;
    for (int v = v0; v < v1; ++v) {
      const float w = weight(v);
      if (w > 0.f && c + w > thr) { s_v = v; break; }
      c += w;
    }
  }
  __syncthreads();
  if (tid == 0 && s_v < 0) {                             // thr at the very top (rounding)
    for (int v = a.V - 1; v >= 0; --v)
      if (weight(v) > 0.f) { s_v = v; break; }
  }
  __syncthreads();
  if (tid < W) {
    const int node = tid <= m ? s_path[tid] : -1;
    if (a.path_nodes) a.path_nodes[(long)b * W + tid] = node;
    a.out_tok[(long)b * W + tid] = node >= 0 ? a.tok[rb + node] : -1;
    if (tid == 0) {
      a.n_acc[b] = m + 1;
      int v = s_v;
      if (v < 0 || v >= a.V) { set_flag(a.status, MEDUSA_FLAG_TOKEN_RANGE); v = 0; }
      a.root_next[b] = v;
    }
  }
  const float4* __restrict__ src = reinterpret_cast<const float4*>(a.hprime + (rb + last) * a.d);
  float4* __restrict__ dst = reinterpret_cast<float4*>(a.h_next + (long)b * a.d);
  for (int j = tid; j < a.d / 4; j += blockDim.x) dst[j] = src[j];
  __syncthreads();
}

__device__ void accept_seq(const VerifyArgs& a, int b) {
  if (a.reject) {
    reject_seq(a, b);
    return;
  }
  __shared__ int acc[MEDUSA_MAX_NODES];
  __shared__ int sret[MEDUSA_MAX_NODES * (MEDUSA_MAX_HEADS + 1)];
  __shared__ float sv[32];
  __shared__ int si[32];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const long rb = (long)b * a.n1;
  const int W = a.K + 1;
  for (int e = tid; e < a.P * W; e += blockDim.x) sret[e] = a.retrieve[e];
  const float log_eps = logf(a.eps), log_delta = logf(a.delta);
  for (int c = tid; c < a.n1; c += blockDim.x) {
    int ok = 1;                                     // the root is always kept
    if (c > 0) {
      const int p = a.parent[c];
      if (a.typical) {
        const float* sp = a.stats + (rb + p) * 4;
        const float lp = __ldcg(a.stats + (rb + c) * 4 + 3) - __ldcg(sp) - __ldcg(sp + 1);
        ok = lp > fminf(log_eps, log_delta - __ldcg(sp + 2));         // log p_parent(tok_c)
      } else {
        ok = a.tok[rb + c] == __ldcg(a.am + rb + p);
      }
    }
    acc[c] = ok;
  }
  __syncthreads();
  // longest run of accepted nodes after the root, per path; best = max, lowest index
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int p = tid; p < a.P; p += blockDim.x) {
    int m = 0;
    while (m + 1 < W) {
      const int node = sret[p * W + m + 1];
      if (node < 0 || !acc[node]) break;
      ++m;
    }
    if (better((float)m, p, bv, bi)) { bv = (float)m; bi = p; }
  }
  block_argmax(bv, bi, sv, si);
  if (tid < W) {
    const int m = (int)bv, best = bi, l = tid;
    const int node = l <= m ? sret[best * W + l] : -1;
    if (a.path_nodes) a.path_nodes[(long)b * W + l] = node;
    a.out_tok[(long)b * W + l] = node >= 0 ? a.tok[rb + node] : -1;
    if (l == m) {
      a.n_acc[b] = m + 1;
      a.root_next[b] = __ldcg(a.am + rb + node);
      s_last = node;
    }
  }
  __syncthreads();
  const float4* __restrict__ src = reinterpret_cast<const float4*>(a.hprime + (rb + s_last) * a.d);
  float4* __restrict__ dst = reinterpret_cast<float4*>(a.h_next + (long)b * a.d);
  const int nv = a.d / 4;
  for (int j0 = tid; j0 < nv; j0 += blockDim.x * 4) {   // four loads in flight per thread
    float4 t[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j0 + u * (int)blockDim.x < nv) t[u] = src[j0 + u * blockDim.x];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j0 + u * (int)blockDim.x < nv) dst[j0 + u * blockDim.x] = t[u];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256) verify_accept_kernel(VerifyArgs a) {
  pdl_trigger();
  pdl_wait();
  accept_seq(a, blockIdx.x);
}

cudaError_t launch_verify_accept(const VerifyArgs& a, cudaStream_t st) {
  return launch_kernel(verify_accept_kernel, dim3(a.B), dim3(256), 0, st, 1, a);
}

// One CTA per sequence: slot len + l <- tree node path_nodes[l], l < n_acc, in 16-byte
// pieces spread over all threads, for the cache (kc, vc) and tree K/V (tk, tv) given.
// Returns the new length in thread 0 (len_out is written by the caller).
template <typename T>
__device__ int compact_copy(const CompactArgs& a, int b, void* kcache, void* vcache, const void* tkeys,
                            const void* tvals) {
  __shared__ int s_len, s_n;
  __shared__ long s_dst[MEDUSA_MAX_HEADS + 1], s_src[MEDUSA_MAX_HEADS + 1];
  const long row = (long)a.Hkv * a.dh;                // elements per cached token
  if (threadIdx.x == 0) {
    int L = a.len[b];
    L = L < 0 ? 0 : L;
    int n = a.n_acc[b];
    n = n < 0 ? 0 : (n > a.K + 1 ? a.K + 1 : n);
    if (L + n > a.capacity) {
      set_flag(a.status, MEDUSA_FLAG_KV_CAPACITY);
      n = a.capacity > L ? a.capacity - L : 0;
    }
    s_len = L;
    s_n = n;
  }
  __syncthreads();
  if (threadIdx.x < s_n) {                            // one thread per kept token
    const int l = threadIdx.x;
    const int node = a.path_nodes[(long)b * (a.K + 1) + l];
    const int t = s_len + l;
    long slot = -1;
    if (node >= 0 && node < a.n1) {
      if (a.page_table) {
        const int page = a.page_table[(long)b * a.pages_per_seq + t / a.page_size];
        if (page < 0 || page >= a.num_pages)
          set_flag(a.status, MEDUSA_FLAG_PAGE_RANGE);
        else
          slot = (long)page * a.page_size + t % a.page_size;
      } else {
        slot = (long)b * a.capacity + t;
      }
    }
    s_dst[l] = slot * row;
    s_src[l] = ((long)b * a.n1 + (node < 0 ? 0 : node)) * row;
  }
  __syncthreads();
  const int n = s_n;
  const int per = (int)(row * sizeof(T) / 16);         // 16-byte pieces per token row
  uint4* kc = reinterpret_cast<uint4*>(kcache);
  uint4* vc = reinterpret_cast<uint4*>(vcache);
  const uint4* tk = reinterpret_cast<const uint4*>(tkeys);
  const uint4* tv = reinterpret_cast<const uint4*>(tvals);
  constexpr int EPV = 16 / sizeof(T);                   // elements per piece
  constexpr int BATCH = 4;                              // loads in flight before the stores
  const int total = n * per, step = blockDim.x;
  for (int e0 = threadIdx.x; e0 < total; e0 += step * BATCH) {
    uint4 kb[BATCH], vb[BATCH];
    long dst[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int e = e0 + u * step;
      dst[u] = -1;
      if (e < total) {
        const int l = e / per, c = e - l * per;
        if (s_dst[l] >= 0) {
          const long s = s_src[l] / EPV + c;
          kb[u] = tk[s];
          vb[u] = tv[s];
          dst[u] = s_dst[l] / EPV + c;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u)
      if (dst[u] >= 0) {
        kc[dst[u]] = kb[u];
        vc[dst[u]] = vb[u];
      }
  }
  __syncthreads();
  return s_len + n;
}

template <typename T>
__device__ void compact_seq(const CompactArgs& a, int b) {
  if (a.no_copy) return;
  const int len = compact_copy<T>(a, b, a.kc, a.vc, a.tk, a.tv);
  if (threadIdx.x == 0) a.len_out[b] = len;
}

// Multi-layer compaction: block (b, l) handles layer l of sequence b; the lengths before
// the step are read by every block before the last one of the sequence (atomic counter)
// writes len_out, so len_out may alias len.
template <typename T>
__global__ void __launch_bounds__(256) kv_compact_layers_kernel(const __grid_constant__ CompactLayersArgs a) {
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, l = blockIdx.y;
  const int len = compact_copy<T>(a.base, b, a.kc[l], a.vc[l], a.tk[l], a.tv[l]);
  if (!a.write_len) return;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.cnt + b, 1) == a.nl - 1;
    if (s_last) {
      a.base.len_out[b] = len;
      a.cnt[b] = 0;
    }
  }
}

cudaError_t launch_kv_compact_layers(const CompactLayersArgs& a, cudaStream_t st) {
  if (a.nl < 1 || a.nl > kLayersPerLaunch) return cudaErrorInvalidValue;
  const dim3 grid(a.base.B, a.nl);
  if (a.base.dtype == 0) return launch_kernel(kv_compact_layers_kernel<float>, grid, dim3(256), 0, st, 1, a);
  return launch_kernel(kv_compact_layers_kernel<bf16>, grid, dim3(256), 0, st, 1, a);
}

template <typename T>
__global__ void __launch_bounds__(256) kv_compact_kernel(CompactArgs a) {
  pdl_trigger();
  pdl_wait();
  compact_seq<T>(a, blockIdx.x);
}

// Fused verification for the whole step.  Each node row's vocabulary is split over
// `slices` CTAs (gridDim.y: about one resident wave of CTAs in all, 1..4);
// the last slice CTA of a row (per-row counter) merges the partials and finishes the row;
// the last row of a sequence (per-sequence counter) runs that sequence's acceptance and KV
// compaction.  Nothing waits; every counter is reset after use.
template <typename T>
__global__ void __launch_bounds__(256, 4) verify_commit_kernel(VerifyArgs v, CompactArgs c, int32_t* row_cnt,
                                                            int32_t* seq_cnt, float* parts) {
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x, sl = blockIdx.y, b = row / v.n1, slices = gridDim.y;
  const int per = ((v.V + slices - 1) / slices + 3) / 4 * 4;
  const int v0 = min(v.V, sl * per), v1 = min(v.V, v0 + per);
  RowPart r = row_part(v, row, v0, v1);
  float* pp = parts + ((long)row * kVerifySlicesMax + sl) * 6;
  if (threadIdx.x == 0) {
    pp[0] = r.bv;
    pp[1] = __int_as_float(r.bi);
    pp[2] = r.st.m;
    pp[3] = r.st.S;
    pp[4] = r.st.U;
    pp[5] = r.nonfinite ? 1.f : 0.f;
    __threadfence();
    s_last = atomicAdd(row_cnt + row, 1) == slices - 1;
  }
  __syncthreads();
  if (!s_last) return;
  if (threadIdx.x == 0) {                         // merge the row's slices
    __threadfence();
    RowPart m{-INFINITY, 0x7fffffff, SoftStat{-INFINITY, 0.f, 0.f}, false};
    for (int q = 0; q < slices; ++q) {
      const float* x = parts + ((long)row * kVerifySlicesMax + q) * 6;
      const float bv = __ldcg(x), m0 = __ldcg(x + 2), S = __ldcg(x + 3), U = __ldcg(x + 4);
      const int bi = __float_as_int(__ldcg(x + 1));
      if (better(bv, bi, m.bv, m.bi)) { m.bv = bv; m.bi = bi; }
      m.st = stat_merge(m.st, SoftStat{m0, S, U});
      m.nonfinite |= __ldcg(x + 5) != 0.f;
    }
    row_finish(v, row, m);
    row_cnt[row] = 0;
    __threadfence();
    s_last = atomicAdd(seq_cnt + b, 1) == v.n1 - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  accept_seq(v, b);
  compact_seq<T>(c, b);
  if (threadIdx.x == 0) seq_cnt[b] = 0;
}

cudaError_t launch_verify_commit(const VerifyArgs& v, const CompactArgs& c, int32_t* row_cnt,
                                 int32_t* seq_cnt, float* parts, cudaStream_t st) {
  static int num_sms = 0;
  if (!num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      num_sms = 148;
  }
  const int rows = v.B * v.n1;
  // about one resident wave (4 CTAs per SM), at most 4 slices: more made the per-row merge
  // cost more than the shorter slices saved
  const int slices = std::max(1, std::min(4, 4 * num_sms / rows));
  dim3 grid(rows, slices);
  if (c.dtype == 0)
    return launch_kernel(verify_commit_kernel<float>, grid, dim3(256), 0, st, 1, v, c, row_cnt, seq_cnt, parts);
  return launch_kernel(verify_commit_kernel<bf16>, grid, dim3(256), 0, st, 1, v, c, row_cnt, seq_cnt, parts);
}

cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t st) {
  if (a.dtype == 0) return launch_kernel(kv_compact_kernel<float>, dim3(a.B), dim3(256), 0, st, 1, a);
  return launch_kernel(kv_compact_kernel<bf16>, dim3(a.B), dim3(256), 0, st, 1, a);
}

}  // namespace medusa
