// Top-k building blocks of the candidate selection ("Medusa: Simple LLM Inference
// Acceleration Framework with Multiple Decoding Heads", §3.4 Tree Attention, Step 1: the
// top-s_k predictions of each head).  Order of candidates everywhere: larger logit first,
// lower token id on equal logits; NaN never enters a list.
#pragma once
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace medusa {

#define NEG_INF (-INFINITY)
constexpr int NO_IDX = 0x7fffffff;

// Sorted (descending) per-thread candidate list of depth N kept in registers.
template <int N>
struct TopListN {
  float v[N];
  int i[N];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int t = 0; t < N; ++t) { v[t] = NEG_INF; i[t] = NO_IDX; }
  }
  __device__ __forceinline__ void insert(float x, int idx) {
    if (!better(x, idx, v[N - 1], i[N - 1])) return;
    v[N - 1] = x;
    i[N - 1] = idx;
#pragma unroll
    for (int t = N - 1; t > 0; --t) {
      if (better(v[t], i[t], v[t - 1], i[t - 1])) {
        float tv = v[t]; v[t] = v[t - 1]; v[t - 1] = tv;
        int ti = i[t]; i[t] = i[t - 1]; i[t - 1] = ti;
      }
    }
  }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int t = 0; t < N - 1; ++t) { v[t] = v[t + 1]; i[t] = i[t + 1]; }
    v[N - 1] = NEG_INF;
    i[N - 1] = NO_IDX;
  }
};
using TopList = TopListN<kTops>;

// Order-preserving 32-bit key of a float (larger float -> larger key; -0 as +0; NaN lowest).
__device__ __forceinline__ uint32_t float_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  if (v != v) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Merge the 32 lanes' sorted lists into the first `rounds` ranks of ov/oi (kTops entries;
// ranks past `rounds` are written as sentinels): each round is a warp reduction over the
// list heads (max of the value keys, then min of the token ids among the lanes holding
// that value) and the winning lane pops.  Token ids are distinct across lanes (sentinels
// aside).
template <int N>
__device__ __forceinline__ void warp_merge(TopListN<N>& L, float* ov, int* oi, int rounds = kTops) {
  const int lane = threadIdx.x & 31;
  rounds = rounds < 1 || rounds > kTops ? kTops : rounds;
  if (lane == 0)                                   // ranks past `rounds` are not needed
    for (int t = rounds; t < kTops; ++t) { ov[t] = NEG_INF; oi[t] = NO_IDX; }
#pragma unroll 1
  for (int t = 0; t < rounds; ++t) {
    const uint32_t key = float_key(L.v[0]);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const uint32_t imin = __reduce_min_sync(0xffffffffu, key == kmax ? (uint32_t)L.i[0] : 0x7fffffffu);
    if (key == kmax && (uint32_t)L.i[0] == imin) L.pop();
    if (lane == 0) {
      ov[t] = kmax != 0u ? key_float(kmax) : NEG_INF;
      oi[t] = (int)imin;
    }
  }
}

// Sorts N (value, token) pairs into descending `better` order with a bitonic sorting
// network (N a power of two); every comparator index is a compile-time constant, so the
// pairs stay in registers.
template <int N>
__device__ __forceinline__ void bitonic_sort_desc(float (&v)[N], int (&ix)[N]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int x = 0; x < N; ++x) {
        const int y = x ^ j;
        if (y <= x) continue;
        // blocks of k with bit k clear end descending, the others ascending: each pair of
        // neighbouring blocks is then a bitonic sequence for the next merge
        const bool sw = (x & k) == 0 ? better(v[y], ix[y], v[x], ix[x]) : better(v[x], ix[x], v[y], ix[y]);
        if (sw) {
          const float tv = v[x]; v[x] = v[y]; v[y] = tv;
          const int ti = ix[x]; ix[x] = ix[y]; ix[y] = ti;
        }
      }
}

// ---------------------------------------------------------------- fused producers
// Batch update of a warp's running list (sorted, kTops entries in shared memory, the best
// `rounds` exact): lane l < n offers (xs[l], idx0 + step * l), xs in shared memory.  The offers that beat the list's last kept
// rank are inserted one at a time (lanes 0..15 shift the list), the others cost one
// comparison.  Whole warp; the list is the warp's own.
__device__ __forceinline__ void warp_list_update(float* lv, int* li, const float* xs, int idx0, int step,
                                                 int n, int rounds) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31, l16 = lane & 15;
  __syncwarp();
  const float x = lane < n ? xs[lane] : 0.f;
  const int idx = idx0 + step * lane;
  unsigned bal = __ballot_sync(full, lane < n && better(x, idx, lv[rounds - 1], li[rounds - 1]));
  while (bal) {
    const int src = __ffs(bal) - 1;
    bal &= bal - 1;
    const float xv = __shfl_sync(full, x, src);
    const int xi = __shfl_sync(full, idx, src);
    const float v = lv[l16];
    const int i = li[l16];
    if (!better(xv, xi, lv[rounds - 1], li[rounds - 1])) continue;   // the list has moved on
    const int pos = __popc(__ballot_sync(full, better(v, i, xv, xi)) & 0xffffu);
    const float uv = __shfl_up_sync(full, v, 1, 16);
    const int ui = __shfl_up_sync(full, i, 1, 16);
    __syncwarp();
    if (lane < 16 && lane > pos) { lv[lane] = uv; li[lane] = ui; }
    if (lane == pos) { lv[lane] = xv; li[lane] = xi; }
    __syncwarp();
  }
}

// One offer (x, idx), known to every lane, to a warp's running list in shared memory (as
// warp_list_update): a comparison with the last kept rank, and the insertion when it beats
// it.  Whole warp.
__device__ __forceinline__ void warp_list_offer(float* lv, int* li, float x, int idx, int rounds) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31, l16 = lane & 15;
  if (!better(x, idx, lv[rounds - 1], li[rounds - 1])) return;      // warp-uniform
  const float v = lv[l16];
  const int i = li[l16];
  const int pos = __popc(__ballot_sync(full, better(v, i, x, idx)) & 0xffffu);
  const float uv = __shfl_up_sync(full, v, 1, 16);
  const int ui = __shfl_up_sync(full, i, 1, 16);
  __syncwarp();
  if (lane < 16 && lane > pos) { lv[lane] = uv; li[lane] = ui; }
  if (lane == pos) { lv[lane] = x; li[lane] = idx; }
  __syncwarp();
}

// Merge of nl sorted lists (shared memory, kTops entries each, the first `rounds` used)
// into out[0 .. kTops): the best `rounds` entries in order, then sentinels.  Each entry's
// rank is its position in its own list plus, per other list, a binary search for the
// entries ahead of it (equal entries, i.e. sentinels, are ordered by list), so every rank
// is written by exactly one thread with no sequential rounds.  Threads tid = 0 .. nt-1 of
// the caller take part; the caller synchronises before and after.
__device__ __forceinline__ void rank_merge(const float (*lv)[kTops], const int (*li)[kTops], int nl,
                                           int rounds, float* ov, int* oi, int tid, int nt) {
  for (int e = tid; e < nl * rounds; e += nt) {
    const int w = e / rounds, t = e - w * rounds;
    const float v = lv[w][t];
    const int ix = li[w][t];
    int rank = t;
    for (int j = 0; j < nl; ++j) {
      if (j == w) continue;
      int lo = 0, hi = rounds;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const bool ahead = j < w ? !better(v, ix, lv[j][mid], li[j][mid]) : better(lv[j][mid], li[j][mid], v, ix);
        if (ahead) lo = mid + 1; else hi = mid;
      }
      rank += lo;
    }
    if (rank < rounds) { ov[rank] = v; oi[rank] = ix; }
  }
  for (int t = rounds + tid; t < kTops; t += nt) { ov[t] = NEG_INF; oi[t] = NO_IDX; }
}

// The best `rounds` (logit, token) pairs of 128 values held 4 per lane (tokens tok0 + 4 *
// lane + e for e < 4; entries with tok >= tok_end are absent), written sorted to ov / oi
// (kTops entries, the ranks past `rounds` as sentinels).  Whole warp.
__device__ __forceinline__ void warp_top_of_128(float4 x, int tok0, int tok_end, int rounds,
                                                float* ov, int* oi) {
  const int lane = threadIdx.x & 31;
  TopListN<4> L;
  const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int t = tok0 + 4 * lane + c;
    const bool ok = t < tok_end && !(e[c] != e[c]);
    L.v[c] = ok ? e[c] : NEG_INF;
    L.i[c] = ok ? t : NO_IDX;
  }
  bitonic_sort_desc(L.v, L.i);
  warp_merge(L, ov, oi, rounds);
}

}  // namespace medusa
