// Projections of the Medusa step: Y[m][r] = sum_k X[m][k] W[r][k] over stacked weight
// blocks (segments), with the epilogues the step needs:
//   EPI_STORE     logits / q,k,v       y = acc
//   EPI_SILU_RES  Medusa head W1       y = SiLU(acc) + h    ("Medusa: Simple LLM Inference
//                 Acceleration Framework with Multiple Decoding Heads", §3.4 head equation)
//   EPI_RES_ADD   synthetic layer out  y = acc + x
// This file holds the CUDA-core streaming row-dot for few activation rows (decode at
// small batch is a pure HBM stream of the weights); the tensor-core path for tens to
// thousands of rows is in k_umma.cu.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace medusa {

__device__ __forceinline__ void epilogue_store(const MatArgs& a, const MatSeg& s, int si, int m, int r,
                                               float acc) {
  if (a.out_alt && si >= a.alt_from) {
    a.out_alt[(long)m * a.ldo_alt + s.out_off + r] = acc;
    return;
  }
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
// One round of CTAs (as many as fit on the GPU at once): CTA c owns a contiguous, balanced
// range of the rows of all segments taken in order.  For each segment it meets, it stages
// that segment's activations (MT rows x k fp32) in shared memory; each warp then streams
// whole weight rows with 16-byte loads, U loads in flight per lane, and reduces across the
// warp.  A single round avoids the tail of a partly filled last wave.
template <typename W, int MT>
__global__ void __launch_bounds__(256) rowdot_kernel(MatArgs a, long total_rows) {
  extern __shared__ float xs[];                       // [MT][k]
  constexpr int VEC = 16 / sizeof(W);
  constexpr int U = 8;
  const long g0 = total_rows * blockIdx.x / gridDim.x;
  const long g1 = total_rows * (blockIdx.x + 1) / gridDim.x;
  const int k = a.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_trigger();
  long seg_start = 0;
  for (int si = 0; si < a.nseg; ++si) {
    const MatSeg& s = a.seg[si];
    const long lo = g0 > seg_start ? g0 : seg_start;
    const long hi = g1 < seg_start + s.rows ? g1 : seg_start + s.rows;
    if (lo < hi) {
      const int r0 = (int)(lo - seg_start), r1 = (int)(hi - seg_start);
      const W* w = reinterpret_cast<const W*>(s.w);
      for (int m0 = 0; m0 < a.M; m0 += MT) {
        const int mt = min(MT, a.M - m0);
        // The warp's first U weight loads go out before the activations are staged, so
        // the staging round trip overlaps the first HBM one.
        uint4 buf[U];
        const int rf = r0 + warp;
        if (rf < r1) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int kk = lane * VEC + u * 32 * VEC;
            if (kk < k) buf[u] = ld_stream16(w + (long)rf * k + kk);
          }
        }
        pdl_wait();                                    // activations come from earlier kernels
        __syncthreads();
        if ((k & 3) == 0 && (s.ldx & 3) == 0 && (reinterpret_cast<uintptr_t>(s.x) & 15) == 0) {
          const uint32_t xs0 = (uint32_t)__cvta_generic_to_shared(xs);
          for (int i = threadIdx.x * 4; i < MT * k; i += blockDim.x * 4) {
            const int mm = i / k, kk = i - mm * k;
            const bool ok = mm < mt;
            cp_async16(xs0 + 4u * (uint32_t)i, ok ? s.x + (long)(m0 + mm) * s.ldx + kk : s.x, ok ? 16 : 0);
          }
          cp_async_commit();
          cp_async_wait<0>();
        } else {
          for (int i = threadIdx.x; i < MT * k; i += blockDim.x) {
            const int mm = i / k, kk = i - mm * k;
            xs[i] = mm < mt ? s.x[(long)(m0 + mm) * s.ldx + kk] : 0.f;
          }
        }
        __syncthreads();
        bool have = rf < r1;                           // buf holds the loads of (rf, lane*VEC)
        for (int r = rf; r < r1; r += 8) {
          const W* wr = w + (long)r * k;
          float acc[MT];
#pragma unroll
          for (int m = 0; m < MT; ++m) acc[m] = 0.f;
          for (int kb = lane * VEC; kb < k; kb += 32 * VEC * U) {
            if (!have) {
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const int kk = kb + u * 32 * VEC;
                if (kk < k) buf[u] = ld_stream16(wr + kk);
              }
            }
            have = false;
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
            if (lane == m && m < mt) epilogue_store(a, s, si, m0 + m, r, acc[m]);
        }
      }
    }
    seg_start += s.rows;
  }
}

template <typename W, int MT>
static cudaError_t rowdot_go(const MatArgs& a, cudaStream_t st) {
  static int num_sms = 0;
  if (!num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      num_sms = 148;
  }
  long total = 0;
  for (int i = 0; i < a.nseg; ++i) total += a.seg[i].rows;
  const size_t smem = (size_t)MT * a.k * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(rowdot_kernel<W, MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rowdot_kernel<W, MT>, 256, smem) !=
          cudaSuccess || per_sm < 1)
    per_sm = 1;
  long grid = (long)per_sm * num_sms;
  const long by_rows = (total + 7) / 8;               // at least one row per warp
  grid = grid < by_rows ? grid : by_rows;
  return launch_kernel(rowdot_kernel<W, MT>, dim3((unsigned)grid), dim3(256), smem, st, 1, a, total);
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

// =========================================================== small helpers
__global__ void split_kernel(const float* x, bf16* hi, bf16* lo, long n) {
  pdl_trigger();
  pdl_wait();
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
    split_hi_lo(x[i], hi[i], lo[i]);
}

cudaError_t launch_split(const float* x, bf16* hi, bf16* lo, long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long blocks = (n + 255) / 256;
  return launch_kernel(split_kernel, dim3((unsigned)(blocks < 4096 ? blocks : 4096)), dim3(256), 0, st, 1,
                       x, hi, lo, n);
}

__global__ void to_bf16_kernel(const float* x, bf16* y, long n) {
  pdl_trigger();
  pdl_wait();
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
    y[i] = __float2bfloat16_rn(x[i]);
}

cudaError_t launch_to_bf16(const float* x, bf16* y, long n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long blocks = (n + 255) / 256;
  return launch_kernel(to_bf16_kernel, dim3((unsigned)(blocks < 4096 ? blocks : 4096)), dim3(256), 0, st, 1,
                       x, y, n);
}

template <typename W>
__global__ void gather_kernel(const W* emb, const int32_t* tok, int d, int V, float* xf, bf16* xb) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  int t = tok[m];
  t = (t < 0 || t >= V) ? 0 : t;                    // ids were range-checked upstream
  const W* src = emb + (long)t * d;
  if (sizeof(W) == 2 && xb && !xf && d % 8 == 0) {        // bf16 -> bf16: 16-byte copies
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(xb + (long)m * d);
    for (int j = threadIdx.x; j < d / 8; j += blockDim.x) d4[j] = s4[j];
    return;
  }
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
    return launch_kernel(gather_kernel<float>, dim3(M), dim3(256), 0, st, 1,
                         reinterpret_cast<const float*>(emb), tok, d, V, xf, xb);
  return launch_kernel(gather_kernel<bf16>, dim3(M), dim3(256), 0, st, 1,
                       reinterpret_cast<const bf16*>(emb), tok, d, V, xf, xb);
}

}  // namespace medusa
