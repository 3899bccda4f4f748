// Verification and commit of the Medusa step.
//   verify_stats   per node row of the verification logits: greedy token (lowest id on
//                  ties) and, for typical acceptance, max z/T, log-sum-exp and entropy
//   verify_accept  accept flags, longest accepted root->leaf path, step outputs
//   kv_compact     copies the kept nodes' keys/values into the cache after the prefix
// Sources: "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads" §3.4 Tree Attention Step 6 and Typical Acceptance Scheme (criterion
// p(x) > min(eps, delta exp(-H)), first token greedy and always kept, longest accepted
// prefix); "MEDUSA 精读" section 3 (only the accepted path stays in the KV cache).
#include "common.cuh"
#include "kernels.h"

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

__device__ __forceinline__ float block_sum(float v, float* sv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) sv[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < nw ? sv[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) sv[0] = v;
  }
  __syncthreads();
  return sv[0];
}

// One CTA per node row (b, n).
__global__ void __launch_bounds__(256) verify_stats_kernel(VerifyArgs a) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const int row = blockIdx.x;
  const int b = row / a.n1, n = row - b * a.n1;
  const float* z = a.logits + (long)row * a.V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool nonfinite = false;
  for (int v = threadIdx.x; v < a.V; v += blockDim.x) {
    const float x = z[v];
    nonfinite |= !isfinite(x);
    if (better(x, v, bv, bi)) { bv = x; bi = v; }
  }
  if (nonfinite) set_flag(a.status, MEDUSA_FLAG_NONFINITE);
  block_argmax(bv, bi, sv, si);
  if (bi < 0 || bi >= a.V) { set_flag(a.status, MEDUSA_FLAG_TOKEN_RANGE); bi = 0; }
  float st[4] = {bv, 0.f, 0.f, 0.f};
  if (a.typical) {
    const float T = a.temperature;
    const float ymax = bv / T;
    float S = 0.f, U = 0.f;
    for (int v = threadIdx.x; v < a.V; v += blockDim.x) {
      const float y = z[v] / T - ymax;
      const float e = __expf(y);
      S += e;
      U += y * e;
    }
    S = block_sum(S, sv);
    U = block_sum(U, sv);
    const float logS = logf(S);
    st[0] = ymax;
    st[1] = logS;
    st[2] = logS - U / S;                         // H = log S - sum(y e^y) / S
    if (n > 0) {
      const int p = a.parent[n];
      const int t = a.tok[(long)b * a.n1 + n];
      st[3] = a.logits[((long)b * a.n1 + p) * a.V + t] / T;
    }
    if (!isfinite(st[1]) || !isfinite(st[2])) set_flag(a.status, MEDUSA_FLAG_NONFINITE);
  }
  if (threadIdx.x == 0) {
    a.am[row] = bi;
#pragma unroll
    for (int q = 0; q < 4; ++q) a.stats[(long)row * 4 + q] = st[q];
  }
}

cudaError_t launch_verify_stats(const VerifyArgs& a, cudaStream_t st) {
  verify_stats_kernel<<<a.B * a.n1, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// One CTA per sequence; thread c decides candidate c, thread p walks path p.
__global__ void __launch_bounds__(256) verify_accept_kernel(VerifyArgs a) {
  __shared__ int acc[MEDUSA_MAX_NODES];
  __shared__ float sv[32];
  __shared__ int si[32];
  __shared__ int s_last;
  const int b = blockIdx.x, tid = threadIdx.x;
  const long rb = (long)b * a.n1;
  const float log_eps = logf(a.eps), log_delta = logf(a.delta);
  for (int c = tid; c < a.n1; c += blockDim.x) {
    int ok = 1;                                     // the root is always kept
    if (c > 0) {
      const int p = a.parent[c];
      if (a.typical) {
        const float* sp = a.stats + (rb + p) * 4;
        const float lp = a.stats[(rb + c) * 4 + 3] - sp[0] - sp[1];   // log p_parent(tok_c)
        ok = lp > fminf(log_eps, log_delta - sp[2]);
      } else {
        ok = a.tok[rb + c] == a.am[rb + p];
      }
    }
    acc[c] = ok;
  }
  __syncthreads();
  // longest run of accepted nodes after the root, per path; best = max, lowest index
  const int W = a.K + 1;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int p = tid; p < a.P; p += blockDim.x) {
    int m = 0;
    while (m + 1 < W) {
      const int node = a.retrieve[(long)p * W + m + 1];
      if (node < 0 || !acc[node]) break;
      ++m;
    }
    if (better((float)m, p, bv, bi)) { bv = (float)m; bi = p; }
  }
  block_argmax(bv, bi, sv, si);
  if (tid == 0) {
    const int m = (int)bv, best = bi;
    int last = 0;
    for (int l = 0; l < W; ++l) {
      const int node = l <= m ? a.retrieve[(long)best * W + l] : -1;
      if (node >= 0) last = node;
      if (a.path_nodes) a.path_nodes[(long)b * W + l] = node;
      a.out_tok[(long)b * W + l] = node >= 0 ? a.tok[rb + node] : -1;
    }
    a.n_acc[b] = m + 1;
    a.root_next[b] = a.am[rb + last];
    s_last = last;
  }
  __syncthreads();
  const float* src = a.hprime + (rb + s_last) * a.d;
  for (int j = tid; j < a.d; j += blockDim.x) a.h_next[(long)b * a.d + j] = src[j];
}

cudaError_t launch_verify_accept(const VerifyArgs& a, cudaStream_t st) {
  verify_accept_kernel<<<a.B, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// One CTA per sequence: slot len + l <- tree node path_nodes[l], l < n_acc.
template <typename T>
__global__ void __launch_bounds__(256) kv_compact_kernel(CompactArgs a) {
  __shared__ int s_len, s_n;
  const int b = blockIdx.x;
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
  const int L = s_len, n = s_n;
  const int row = a.Hkv * a.dh;
  T* kc = reinterpret_cast<T*>(a.kc);
  T* vc = reinterpret_cast<T*>(a.vc);
  const T* tk = reinterpret_cast<const T*>(a.tk);
  const T* tv = reinterpret_cast<const T*>(a.tv);
  for (int l = 0; l < n; ++l) {
    const int node = a.path_nodes[(long)b * (a.K + 1) + l];
    if (node < 0 || node >= a.n1) continue;
    const int t = L + l;
    long slot;
    if (a.page_table) {
      const int page = a.page_table[(long)b * a.pages_per_seq + t / a.page_size];
      if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0) set_flag(a.status, MEDUSA_FLAG_PAGE_RANGE);
        continue;
      }
      slot = (long)page * a.page_size + t % a.page_size;
    } else {
      slot = (long)b * a.capacity + t;
    }
    const long src = ((long)b * a.n1 + node) * row, dst = slot * row;
    for (int e = threadIdx.x; e < row; e += blockDim.x) {
      kc[dst + e] = tk[src + e];
      vc[dst + e] = tv[src + e];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) a.len_out[b] = L + n;
}

cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t st) {
  if (a.dtype == 0)
    kv_compact_kernel<float><<<a.B, 256, 0, st>>>(a);
  else
    kv_compact_kernel<bf16><<<a.B, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace medusa
