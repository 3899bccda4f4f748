// Tree attention of the Medusa step ("Medusa: Simple LLM Inference Acceleration Framework
// with Multiple Decoding Heads" §3.4 Tree Attention, Steps 3 and 5): every packed node
// attends to the whole KV prefix and to its own ancestors in the tree.
//
// Split-KV: CTA (split, kv head g, sequence b, query-row block).  Splits 0..nsplit-1 each
// cover one chunk of the prefix; split `nsplit` covers the tree keys, masked by the
// ancestor bitmask.  Query rows are (node, query head of group g) pairs, so the key/value
// tiles of head g are read once for all G = Hq/Hkv query heads that share them (GQA).
// Each CTA writes an unnormalised partial (o, running max, running sum); a second kernel
// merges the partials by log-sum-exp.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace medusa {

constexpr int TK = 32;   // keys per shared-memory tile (one per lane)

template <typename T>
__device__ __forceinline__ long kv_offset(const AttnArgs& a, int b, int t, int g, bool& ok) {
  long slot;
  ok = true;
  if (a.page_table) {
    const int page = a.page_table[(long)b * a.pages_per_seq + t / a.page_size];
    if (page < 0 || page >= a.num_pages) { ok = false; return 0; }
    slot = (long)page * a.page_size + t % a.page_size;
  } else {
    slot = (long)b * a.capacity + t;
  }
  return (slot * a.Hkv + g) * (long)a.dh;
}

template <typename T, int DH, int RPW>
__global__ void __launch_bounds__(256) tree_attn_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  pdl_trigger();
  pdl_wait();
  constexpr int C = DH / 32;
  float* Qs = sm;                                   // [rows_per_block][DH]
  float* Ks = Qs + a.rows_per_block * DH;           // [TK][DH + 1]
  float* Vs = Ks + TK * (DH + 1);                   // [TK][DH]
  const int split = blockIdx.x, g = blockIdx.y;
  const int b = blockIdx.z / a.nrb, rb = blockIdx.z % a.nrb;
  const int R = a.n1 * a.G;
  const int row0 = rb * a.rows_per_block;
  const int nrows = min(a.rows_per_block, R - row0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool tree = split == a.nsplit;
  int L = a.len[b];
  L = L < 0 ? 0 : (L > a.capacity ? a.capacity : L);
  const int kbeg = tree ? 0 : split * a.chunk;
  const int kend = tree ? a.n1 : min(L, kbeg + a.chunk);

  // stage the block's queries: row r -> node r / G, query head g*G + r % G
  for (int e = tid; e < nrows * DH; e += blockDim.x) {
    const int r = e / DH, i = e - r * DH;
    const int gr = row0 + r, n = gr / a.G, hq = g * a.G + gr % a.G;
    Qs[e] = a.q[(((long)b * a.n1 + n) * a.Hq + hq) * DH + i];
  }

  float o[RPW][C], mrow[RPW], lrow[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    mrow[i] = -INFINITY;
    lrow[i] = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) o[i][c] = 0.f;
  }

  const T* kc = reinterpret_cast<const T*>(a.kc);
  const T* vc = reinterpret_cast<const T*>(a.vc);
  const T* tk = reinterpret_cast<const T*>(a.tk);
  const T* tv = reinterpret_cast<const T*>(a.tv);
  for (int t0 = kbeg; t0 < kend; t0 += TK) {
    __syncthreads();
    // load a tile of TK keys/values (fp32 in shared memory; zero past kend)
    for (int e = tid; e < TK * DH; e += blockDim.x) {
      const int j = e / DH, i = e - j * DH, t = t0 + j;
      float kv = 0.f, vv = 0.f;
      if (t < kend) {
        if (tree) {
          const long off = (((long)b * a.n1 + t) * a.Hkv + g) * DH + i;
          kv = to_f32(tk[off]);
          vv = to_f32(tv[off]);
        } else {
          bool ok;
          const long off = kv_offset<T>(a, b, t, g, ok);
          if (ok) {
            kv = to_f32(kc[off + i]);
            vv = to_f32(vc[off + i]);
          } else if (i == 0) {
            set_flag(a.status, MEDUSA_FLAG_PAGE_RANGE);
          }
        }
      }
      Ks[j * (DH + 1) + i] = kv;
      Vs[j * DH + i] = vv;
    }
    __syncthreads();
    const int t = t0 + lane;
#pragma unroll
    for (int ri = 0; ri < RPW; ++ri) {
      const int r = warp * RPW + ri;
      if (r >= nrows) break;
      bool valid = t < kend;
      if (tree && valid) {
        const int n = (row0 + r) / a.G;
        valid = (a.mask[(long)n * kMaskWords + (t >> 5)] >> (t & 31)) & 1u;
      }
      float s = -INFINITY;
      if (valid) {
        const float* qr = Qs + r * DH;
        const float* kr = Ks + lane * (DH + 1);
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < DH; ++i) acc = fmaf(qr[i], kr[i], acc);
        s = acc * a.scale;
      }
      const float mt = warp_max(s);
      const float mnew = fmaxf(mrow[ri], mt);
      if (mnew == -INFINITY) continue;
      const float p = valid ? __expf(s - mnew) : 0.f;
      const float alpha = __expf(mrow[ri] - mnew);
      lrow[ri] = lrow[ri] * alpha + warp_sum(p);
      mrow[ri] = mnew;
#pragma unroll
      for (int c = 0; c < C; ++c) o[ri][c] *= alpha;
#pragma unroll 4
      for (int j = 0; j < TK; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int c = 0; c < C; ++c) o[ri][c] = fmaf(pj, Vs[j * DH + lane + 32 * c], o[ri][c]);
      }
    }
  }
  // partials: [b][g][split][R][DH] and [b][g][split][R][2]
  const long pbase = (((long)b * a.Hkv + g) * (a.nsplit + 1) + split) * R;
#pragma unroll
  for (int ri = 0; ri < RPW; ++ri) {
    const int r = warp * RPW + ri;
    if (r >= nrows) break;
    const long pr = pbase + row0 + r;
#pragma unroll
    for (int c = 0; c < C; ++c) a.part_o[pr * DH + lane + 32 * c] = o[ri][c];
    if (lane == 0) {
      a.part_ml[pr * 2] = mrow[ri];
      a.part_ml[pr * 2 + 1] = lrow[ri];
    }
  }
}

// One warp per (sequence, kv head, query row): o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s
// over the prefix splits and the tree split, M = max_s m_s.  Lane j holds the VPL
// consecutive columns [j*VPL, (j+1)*VPL) of the head (dh = 32 * VPL).  Splits go in batches
// of 8: every lane loads the batch's (m, l) pairs (the same addresses across the warp) and
// its columns of the batch's outputs in one round trip, and the running maximum moves
// once per batch (the sums are rescaled when it rises).
template <int VPL>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
  constexpr int SB = 8;
  pdl_trigger();
  pdl_wait();
  const int R = a.n1 * a.G, S = a.nsplit + 1;
  const long wg = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wg >= (long)a.B * a.Hkv * R) return;
  const int lane = threadIdx.x & 31;
  const int r = (int)(wg % R);
  const long bg = wg / R;                            // b * Hkv + g
  const int g = (int)(bg % a.Hkv), b = (int)(bg / a.Hkv);
  const long base = bg * S * R + r;                  // partial row of split s: base + s * R
  float M = -INFINITY, Lsum = 0.f;
  float acc[VPL];
#pragma unroll
  for (int c = 0; c < VPL; ++c) acc[c] = 0.f;
  for (int s0 = 0; s0 < S; s0 += SB) {
    float m[SB], l[SB], v[SB][VPL];
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      m[u] = -INFINITY;
      l[u] = 0.f;
#pragma unroll
      for (int c = 0; c < VPL; ++c) v[u][c] = 0.f;
      if (s0 + u < S) {
        const long pr = base + (long)(s0 + u) * R;
        const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + pr * 2);
        m[u] = ml.x;
        l[u] = ml.y;
        const float* src = a.part_o + pr * a.dh + lane * VPL;
        if (VPL == 4) {
          const float4 t = *reinterpret_cast<const float4*>(src);
          v[u][0] = t.x; v[u][VPL > 1 ? 1 : 0] = t.y; v[u][VPL > 2 ? 2 : 0] = t.z; v[u][VPL > 3 ? 3 : 0] = t.w;
        } else if (VPL == 2) {
          const float2 t = *reinterpret_cast<const float2*>(src);
          v[u][0] = t.x; v[u][VPL > 1 ? 1 : 0] = t.y;
        } else {
          v[u][0] = src[0];
        }
      }
    }
    float mb = M;
#pragma unroll
    for (int u = 0; u < SB; ++u) mb = fmaxf(mb, m[u]);
    if (mb == -INFINITY) continue;                   // no keys in any split so far
    const float scale = M == -INFINITY ? 0.f : __expf(M - mb);
    Lsum *= scale;
#pragma unroll
    for (int c = 0; c < VPL; ++c) acc[c] *= scale;
    M = mb;
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      const float w = m[u] == -INFINITY ? 0.f : __expf(m[u] - M);
      Lsum += w * l[u];
#pragma unroll
      for (int c = 0; c < VPL; ++c) acc[c] += w * v[u][c];
    }
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  const int n = r / a.G, hq = g * a.G + r % a.G;
  const long o0 = (((long)b * a.n1 + n) * a.Hq + hq) * a.dh + lane * VPL;
  float y[VPL];
#pragma unroll
  for (int c = 0; c < VPL; ++c) y[c] = Lsum > 0.f ? acc[c] * inv : 0.f;
  if (a.o) {
    if (VPL == 4) {
      *reinterpret_cast<float4*>(a.o + o0) = make_float4(y[0], y[VPL > 1 ? 1 : 0], y[VPL > 2 ? 2 : 0], y[VPL > 3 ? 3 : 0]);
    } else {
#pragma unroll
      for (int c = 0; c < VPL; ++c) a.o[o0 + c] = y[c];
    }
  }
  if (a.o_hi) {
    bf16 hi[VPL], lo[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) split_hi_lo(y[c], hi[c], lo[c]);
    if (VPL == 4) {                                  // 8-byte stores of four halves
      *reinterpret_cast<uint2*>(a.o_hi + o0) = *reinterpret_cast<const uint2*>(hi);
      *reinterpret_cast<uint2*>(a.o_lo + o0) = *reinterpret_cast<const uint2*>(lo);
    } else {
#pragma unroll
      for (int c = 0; c < VPL; ++c) { a.o_hi[o0 + c] = hi[c]; a.o_lo[o0 + c] = lo[c]; }
    }
  }
}

template <typename T, int DH, int RPW>
static cudaError_t attn_go(const AttnArgs& a, cudaStream_t st) {
  const size_t smem = ((size_t)a.rows_per_block * DH + TK * (DH + 1) + TK * DH) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel<T, DH, RPW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nsplit + 1, a.Hkv, a.B * a.nrb);
  return launch_kernel(tree_attn_kernel<T, DH, RPW>, grid, dim3(256), smem, st, 1, a);
}

cudaError_t launch_attn_combine(const AttnArgs& a, cudaStream_t st) {
  const long rows = (long)a.B * a.Hkv * a.n1 * a.G;
  const int blocks = (int)((rows + 7) / 8);           // 8 warps per CTA, one row each
  switch (a.dh) {
    case 32: return launch_kernel(attn_combine_kernel<1>, dim3(blocks), dim3(256), 0, st, 1, a);
    case 64: return launch_kernel(attn_combine_kernel<2>, dim3(blocks), dim3(256), 0, st, 1, a);
    default: return launch_kernel(attn_combine_kernel<4>, dim3(blocks), dim3(256), 0, st, 1, a);
  }
}

template <typename T, int DH>
static cudaError_t attn_rpw(const AttnArgs& a, cudaStream_t st) {
  switch (a.rpw) {
    case 4: return attn_go<T, DH, 4>(a, st);
    case 9: return attn_go<T, DH, 9>(a, st);
    default: return attn_go<T, DH, 12>(a, st);
  }
}

cudaError_t launch_tree_attention(const AttnArgs& a, int dtype, cudaStream_t st) {
  if (dtype == 0) {
    switch (a.dh) {
      case 32: return attn_rpw<float, 32>(a, st);
      case 64: return attn_rpw<float, 64>(a, st);
      default: return attn_rpw<float, 128>(a, st);
    }
  }
  switch (a.dh) {
    case 32: return attn_rpw<bf16, 32>(a, st);
    case 64: return attn_rpw<bf16, 64>(a, st);
    default: return attn_rpw<bf16, 128>(a, st);
  }
}

}  // namespace medusa
