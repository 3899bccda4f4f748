// Projections of the Medusa step: Y[m][r] = sum_k X[m][k] W[r][k] over stacked weight
// blocks (segments), with the epilogues the step needs:
//   EPI_STORE     logits / q,k,v       y = acc
//   EPI_SILU_RES  Medusa head W1       y = SiLU(acc) + h    ("Medusa: Simple LLM Inference
//                 Acceleration Framework with Multiple Decoding Heads", §3.4 head equation)
//   EPI_RES_ADD   synthetic layer out  y = acc + x
// Two kernels: a CUDA-core streaming row-dot for few activation rows (decode at small
// batch is a pure HBM stream of the weights), and a tensor-core GEMM for tens to
// thousands of rows, where the fp32 activations enter as bf16 hi + lo halves so the
// products keep ~fp32 accuracy.
#include "common.cuh"
#include "kernels.h"

namespace medusa {

__device__ __forceinline__ void epilogue_store(const MatArgs& a, const MatSeg& s, int m, int r,
                                               float acc) {
  float y = acc;
  if (a.epi == EPI_SILU_RES) {
    y = silu(acc) + a.res_f32[(long)m * a.ldr + r];
  } else if (a.epi == EPI_RES_ADD) {
    float res = a.res_f32 ? a.res_f32[(long)m * a.ldr + r]
                          : to_f32(reinterpret_cast<const bf16*>(a.res_w)[(long)m * a.ldr + r]);
    y = acc + res;
  }
  const long o = (long)m * a.ldo + s.out_off + r;
  a.out[o] = y;
  if (a.out_hi) {
    bf16 hi, lo;
    split_hi_lo(y, hi, lo);
    a.out_hi[o] = hi;
    a.out_lo[o] = lo;
  }
}

// =========================================================== CUDA-core row-dot
// One CTA = one chunk of rows of one segment; its activations (MT rows x k fp32) are
// staged in shared memory; each warp streams whole weight rows with 16-byte loads, U
// loads in flight per lane, and reduces across the warp.
template <typename W, int MT>
__global__ void __launch_bounds__(256) rowdot_kernel(MatArgs a, int rows_per_cta) {
  extern __shared__ float xs[];                       // [MT][k]
  constexpr int VEC = 16 / sizeof(W);
  constexpr int U = 8;
  const MatSeg& s = a.seg[blockIdx.y];
  const int r0 = blockIdx.x * rows_per_cta;
  if (r0 >= s.rows) return;
  const int r1 = min(s.rows, r0 + rows_per_cta);
  const int k = a.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const W* w = reinterpret_cast<const W*>(s.w);

  for (int m0 = 0; m0 < a.M; m0 += MT) {
    const int mt = min(MT, a.M - m0);
    __syncthreads();
    for (int i = threadIdx.x; i < MT * k; i += blockDim.x) {
      const int mm = i / k, kk = i - mm * k;
      xs[i] = mm < mt ? s.x[(long)(m0 + mm) * s.ldx + kk] : 0.f;
    }
    __syncthreads();
    for (int r = r0 + warp; r < r1; r += 8) {
      const W* wr = w + (long)r * k;
      float acc[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = 0.f;
      for (int kb = lane * VEC; kb < k; kb += 32 * VEC * U) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int kk = kb + u * 32 * VEC;
          if (kk < k) buf[u] = ld_stream16(wr + kk);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int kk = kb + u * 32 * VEC;
          if (kk < k) {
            float f[VEC];
            unpack16(buf[u], f);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const float4* xv = reinterpret_cast<const float4*>(xs + m * k + kk);
#pragma unroll
              for (int e4 = 0; e4 < VEC / 4; ++e4) {
                const float4 x4 = xv[e4];
                acc[m] = fmaf(f[4 * e4 + 0], x4.x, acc[m]);
                acc[m] = fmaf(f[4 * e4 + 1], x4.y, acc[m]);
                acc[m] = fmaf(f[4 * e4 + 2], x4.z, acc[m]);
                acc[m] = fmaf(f[4 * e4 + 3], x4.w, acc[m]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = warp_sum(acc[m]);
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (lane == m && m < mt) epilogue_store(a, s, m0 + m, r, acc[m]);
    }
  }
}

template <typename W, int MT>
static cudaError_t rowdot_go(const MatArgs& a, cudaStream_t st) {
  int maxrows = 0;
  for (int i = 0; i < a.nseg; ++i) maxrows = maxrows > a.seg[i].rows ? maxrows : a.seg[i].rows;
  const int rows_per_cta = 64;
  dim3 grid((maxrows + rows_per_cta - 1) / rows_per_cta, a.nseg);
  const size_t smem = (size_t)MT * a.k * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(rowdot_kernel<W, MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  rowdot_kernel<W, MT><<<grid, 256, smem, st>>>(a, rows_per_cta);
  return cudaGetLastError();
}

cudaError_t launch_rowdot(const MatArgs& a, int dtype, cudaStream_t st) {
  const int mt = a.M >= 4 ? 4 : a.M;
  if (dtype == 0) {
    switch (mt) {
      case 1: return rowdot_go<float, 1>(a, st);
      case 2: return rowdot_go<float, 2>(a, st);
      case 3: return rowdot_go<float, 3>(a, st);
      default: return rowdot_go<float, 4>(a, st);
    }
  }
  switch (mt) {
    case 1: return rowdot_go<bf16, 1>(a, st);
    case 2: return rowdot_go<bf16, 2>(a, st);
    case 3: return rowdot_go<bf16, 3>(a, st);
    default: return rowdot_go<bf16, 4>(a, st);
  }
}

// =========================================================== tensor-core GEMM (mma.sync)
// CTA = 128 weight rows x (MT*8) activation rows; 8 warps each own 16 weight rows.  The
// weights are the MMA's A operand (16x16 row fragments), the activations its B operand,
// so small activation counts waste no MMA work.  K is streamed in 64-wide tiles through a
// 3-stage cp.async ring with a 16-byte-chunk XOR swizzle for conflict-free ldmatrix.
constexpr int GB_R = 128, GB_K = 64, G_STAGES = 3;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {   // byte offset in a tile
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int MT>
__global__ void __launch_bounds__(256) mma_gemm_kernel(MatArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int AR = MT * 8;                               // activation rows per CTA
  constexpr int W_BYTES = GB_R * 128, A_BYTES = AR * 128;
  constexpr int STAGE = W_BYTES + 2 * A_BYTES;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // segment and tile of this CTA
  int si = 0;
  while (si + 1 < a.nseg && (int)blockIdx.y >= a.tile_off[si + 1]) ++si;
  const MatSeg& s = a.seg[si];
  const int rbase = ((int)blockIdx.y - a.tile_off[si]) * GB_R;
  const int m0 = blockIdx.x * AR;
  const bool has_lo = s.a_lo != nullptr;
  const int k = a.k, nk = (k + GB_K - 1) / GB_K;
  const bf16* w = reinterpret_cast<const bf16*>(s.w);
  const uint32_t sbase = smem_u32(smem);

  auto load_stage = [&](int st, int kt) {
    const uint32_t ws = sbase + st * STAGE, as = ws + W_BYTES, ls = as + A_BYTES;
    const int k0 = kt * GB_K;
    for (int c = tid; c < GB_R * 8; c += 256) {
      const int row = c >> 3, ch = c & 7;
      const int gr = rbase + row, kk = k0 + ch * 8;
      const bool ok = gr < s.rows && kk < k;
      const bf16* src = w + (ok ? (long)gr * k + kk : 0);
      cp_async16(ws + swz(row, ch), src, ok ? 16 : 0);
    }
    for (int c = tid; c < AR * 8; c += 256) {
      const int row = c >> 3, ch = c & 7;
      const int gm = m0 + row, kk = k0 + ch * 8;
      const bool ok = gm < a.M && kk < k;
      const long off = ok ? (long)gm * s.ldx + kk : 0;
      cp_async16(as + swz(row, ch), s.a_hi + off, ok ? 16 : 0);
      if (has_lo) cp_async16(ls + swz(row, ch), s.a_lo + off, ok ? 16 : 0);
    }
  };

  float acc[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;

#pragma unroll
  for (int st = 0; st < G_STAGES - 1; ++st) {
    if (st < nk) load_stage(st, st);
    cp_async_commit();
  }
  const int wrow = warp * 16;
  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<G_STAGES - 2>();
    __syncthreads();
    const int nxt = kt + G_STAGES - 1;
    if (nxt < nk) load_stage(nxt % G_STAGES, nxt);
    cp_async_commit();
    const uint32_t ws = sbase + (kt % G_STAGES) * STAGE, as = ws + W_BYTES, ls = as + A_BYTES;
#pragma unroll
    for (int ks = 0; ks < GB_K / 16; ++ks) {
      uint32_t af[4];
      {
        const int row = wrow + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = ks * 2 + (lane >> 4);
        ldsm_x4(ws + swz(row, ch), af[0], af[1], af[2], af[3]);
      }
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const int row = j * 8 + (lane & 7);
        const int ch = ks * 2 + ((lane >> 3) & 1);
        if (has_lo) {
          uint32_t b0, b1, c0, c1;
          const uint32_t base = (lane < 16) ? as : ls;
          ldsm_x4(base + swz(row, ch), b0, b1, c0, c1);
          mma_bf16_16816(acc[j], af, b0, b1);
          mma_bf16_16816(acc[j], af, c0, c1);
        } else {
          uint32_t b0, b1;
          ldsm_x2(as + swz(row, ch), b0, b1);
          mma_bf16_16816(acc[j], af, b0, b1);
        }
      }
    }
  }
  cp_async_wait<0>();

  // C fragment: rows (weights) wrow + lane/4 (+8), columns (activations) 2*(lane%4) (+1)
#pragma unroll
  for (int j = 0; j < MT; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = rbase + wrow + (lane >> 2) + (e >> 1) * 8;
      const int m = m0 + j * 8 + (lane & 3) * 2 + (e & 1);
      if (r < s.rows && m < a.M) epilogue_store(a, s, m, r, acc[j][e]);
    }
  }
}

template <int MT>
static cudaError_t mma_go(MatArgs& a, cudaStream_t st) {
  constexpr int AR = MT * 8;
  const size_t smem = (size_t)G_STAGES * (GB_R * 128 + 2 * AR * 128);
  cudaError_t e = cudaFuncSetAttribute(mma_gemm_kernel<MT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.M + AR - 1) / AR, a.tile_off[a.nseg]);
  mma_gemm_kernel<MT><<<grid, 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_mma_gemm(MatArgs a, cudaStream_t st) {
  a.tile_off[0] = 0;
  for (int i = 0; i < a.nseg; ++i)
    a.tile_off[i + 1] = a.tile_off[i] + (a.seg[i].rows + GB_R - 1) / GB_R;
  const int tiles8 = (a.M + 7) / 8;
  if (tiles8 <= 1) return mma_go<1>(a, st);
  if (tiles8 <= 2) return mma_go<2>(a, st);
  if (tiles8 <= 4) return mma_go<4>(a, st);
  if (tiles8 <= 6) return mma_go<6>(a, st);
  if (tiles8 <= 9) return mma_go<9>(a, st);
  if (tiles8 <= 12) return mma_go<12>(a, st);
  return mma_go<16>(a, st);
}

// =========================================================== small helpers
__global__ void split_kernel(const float* x, bf16* hi, bf16* lo, long n) {
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
    split_hi_lo(x[i], hi[i], lo[i]);
}

cudaError_t launch_split(const float* x, bf16* hi, bf16* lo, long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long blocks = (n + 255) / 256;
  split_kernel<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(x, hi, lo, n);
  return cudaGetLastError();
}

template <typename W>
__global__ void gather_kernel(const W* emb, const int32_t* tok, int d, int V, float* xf, bf16* xb) {
  const int m = blockIdx.x;
  int t = tok[m];
  t = (t < 0 || t >= V) ? 0 : t;                    // ids were range-checked upstream
  const W* src = emb + (long)t * d;
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    const float v = to_f32(src[j]);
    if (xf) xf[(long)m * d + j] = v;
    if (xb) xb[(long)m * d + j] = from_f32<bf16>(v);
  }
}

cudaError_t launch_gather(const void* emb, int dtype, const int32_t* tok, int M, int d, int V,
                          float* xf, bf16* xb, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (dtype == 0)
    gather_kernel<float><<<M, 256, 0, st>>>(reinterpret_cast<const float*>(emb), tok, d, V, xf, xb);
  else
    gather_kernel<bf16><<<M, 256, 0, st>>>(reinterpret_cast<const bf16*>(emb), tok, d, V, xf, xb);
  return cudaGetLastError();
}

}  // namespace medusa
