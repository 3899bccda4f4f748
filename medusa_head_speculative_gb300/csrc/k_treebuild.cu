// On-device construction of the optimized (greedy) candidate tree from a table of per-head
// marginal accuracies ("Medusa: Simple LLM Inference Acceleration Framework with Multiple
// Decoding Heads" §3.4 Optimized Tree Construction; "Accelerating LLM Inference with
// Speculative Decoding: Notes on Medusa" section 4): from the root, repeatedly add the
// frontier node (a child of a chosen node) with the largest product of accuracies along its
// path, ties to the lexicographically smaller rank path, until N nodes; then pack the tree
// canonically (root, then by depth, then by rank path).  The expected accepted length of the
// first n nodes added (the sum of their path products) comes out alongside, so a caller can
// pick the tree size.
//
// One CTA.  A path (r_1, ..., r_d) is encoded with field j (5 bits) = r_j + 1, left-aligned
// in 40 bits, so integer order is the tuple order (a prefix sorts first).  Path products are
// formed root to leaf in double precision, as the host builder and the oracle form them.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace medusa {

constexpr int TB_THREADS = 256;
constexpr int TB_FIELD = 5;
constexpr int TB_DEPTH = 8;                          // MEDUSA_MAX_HEADS fields

__device__ __forceinline__ int path_depth(uint64_t c) {
  int d = 0;
  for (int j = 0; j < TB_DEPTH; ++j)
    if ((c >> (TB_FIELD * (TB_DEPTH - 1 - j))) & 31u) d = j + 1;
  return d;
}
// (score, code) a better than b: larger score, then smaller code
__device__ __forceinline__ bool tb_better(double sa, uint64_t ca, double sb, uint64_t cb) {
  return sa > sb || (sa == sb && ca < cb);
}

__global__ void __launch_bounds__(TB_THREADS) tree_greedy_kernel(const TreeGreedyArgs a) {
  extern __shared__ uint8_t smem[];
  double* fs = reinterpret_cast<double*>(smem);                    // frontier scores
  uint64_t* fc = reinterpret_cast<uint64_t*>(fs + a.fmax);         // frontier codes
  uint64_t* cc = fc + a.fmax;                                      // chosen codes (insertion order)
  double* cs = reinterpret_cast<double*>(cc + a.N);                // chosen scores
  __shared__ double ws[TB_THREADS / 32];
  __shared__ uint64_t wc[TB_THREADS / 32];
  __shared__ int wi[TB_THREADS / 32];
  __shared__ int s_nf, s_win;
  __shared__ double s_score;
  __shared__ uint64_t s_code;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();
  if (tid < a.s[0]) {
    fs[tid] = a.acc[tid];                               // depth 1: a[0][i]
    fc[tid] = (uint64_t)(tid + 1) << (TB_FIELD * (TB_DEPTH - 1));
  }
  if (tid == 0) s_nf = a.s[0];
  __syncthreads();
  for (int n = 0; n < a.N; ++n) {
    const int nf = s_nf;
    double bs = -INFINITY;
    uint64_t bc = ~0ull;
    int bi = -1;
    for (int j = tid; j < nf; j += TB_THREADS)
      if (fc[j] != ~0ull && tb_better(fs[j], fc[j], bs, bc)) { bs = fs[j]; bc = fc[j]; bi = j; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double os = __shfl_xor_sync(0xffffffffu, bs, o);
      const uint64_t oc = __shfl_xor_sync(0xffffffffu, bc, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi >= 0 && (bi < 0 || tb_better(os, oc, bs, bc))) { bs = os; bc = oc; bi = oi; }
    }
    if (lane == 0) { ws[warp] = bs; wc[warp] = bc; wi[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
      double s2 = -INFINITY;
      uint64_t c2 = ~0ull;
      int i2 = -1;
      for (int w = 0; w < TB_THREADS / 32; ++w)
        if (wi[w] >= 0 && (i2 < 0 || tb_better(ws[w], wc[w], s2, c2))) { s2 = ws[w]; c2 = wc[w]; i2 = wi[w]; }
      s_win = i2;
      if (i2 >= 0) {
        s_score = s2;
        s_code = c2;
        cc[n] = c2;
        cs[n] = s2;
        fc[i2] = ~0ull;                                  // taken off the frontier
      }
    }
    __syncthreads();
    if (s_win < 0) return;                               // the host checks the tree has N nodes
    const int d = path_depth(s_code);
    if (d < a.K && tid < a.s[d]) {                       // its children join the frontier
      const int j = nf + tid;
      if (j < a.fmax) {
        fs[j] = s_score * a.acc[d * a.smax + tid];
        fc[j] = s_code | ((uint64_t)(tid + 1) << (TB_FIELD * (TB_DEPTH - 1 - d)));
      }
    }
    __syncthreads();
    if (tid == 0 && d < a.K) s_nf = min(a.fmax, nf + a.s[d]);
    __syncthreads();
  }
  // canonical packing: key = depth, then path; node 0 is the root (code 0)
  for (int j = tid; j < a.N; j += TB_THREADS) {
    const uint64_t c = cc[j];
    const int d = path_depth(c);
    const uint64_t key = ((uint64_t)d << 40) | c;
    int pos = 1;
    for (int m = 0; m < a.N; ++m) pos += (((uint64_t)path_depth(cc[m]) << 40) | cc[m]) < key;
    const uint64_t pc = c & ~((uint64_t)31u << (TB_FIELD * (TB_DEPTH - d)));   // drop the last field
    int ppos = 0;
    if (pc != 0) {
      const int pd = d - 1;
      const uint64_t pkey = ((uint64_t)pd << 40) | pc;
      ppos = 1;
      for (int m = 0; m < a.N; ++m) ppos += (((uint64_t)path_depth(cc[m]) << 40) | cc[m]) < pkey;
    }
    a.parent[pos] = ppos;
    a.rank[pos] = (int)((c >> (TB_FIELD * (TB_DEPTH - d))) & 31u) - 1;
  }
  if (tid == 0) {
    a.parent[0] = -1;
    a.rank[0] = 0;
    if (a.expected) {
      double e = 0.0;
      a.expected[0] = 0.0;
      for (int j = 0; j < a.N; ++j) {
        e += cs[j];
        a.expected[j + 1] = e;
      }
    }
  }
}

size_t tree_greedy_smem(int N, int smax) {
  const size_t fmax = (size_t)N * smax + smax;
  return fmax * (sizeof(double) + sizeof(uint64_t)) + (size_t)N * (sizeof(uint64_t) + sizeof(double));
}

cudaError_t launch_tree_greedy(const TreeGreedyArgs& a, cudaStream_t st) {
  const size_t smem = tree_greedy_smem(a.N, a.smax);
  cudaError_t e = cudaFuncSetAttribute(tree_greedy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(tree_greedy_kernel, dim3(1), dim3(TB_THREADS), smem, st, 1, a);
}

}  // namespace medusa
