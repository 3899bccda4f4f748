// Projections of the Medusa step: Y[m][r] = sum_k X[m][k] W[r][k] over stacked weight
// blocks (segments), with the epilogues the step needs:
//   EPI_STORE     logits / q,k,v       y = acc
//   EPI_SILU_RES  Medusa head W1       y = SiLU(acc) + h    ("Medusa: Simple LLM Inference
//                 Acceleration Framework with Multiple Decoding Heads", §3.4 head equation)
//   EPI_RES_ADD   synthetic layer out  y = acc + x
// This file holds the CUDA-core streaming row-dot for few activation rows (decode at
// small batch is a pure HBM stream of the weights); the tensor-core path for tens to
// thousands of rows is in k_umma.cu.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "topk.cuh"

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
// Segments with fused top-k (MatSeg::cand) store nothing per row: each warp offers its row
// sums to its running list of the best rows (per activation row, in shared memory), and at
// the end of the CTA's range the 8 warps' lists are merged into the CTA's candidate slot.
// CM: 0 = no segment has fused top-k, 1 = every segment has, 2 = some have (the kernel is
// instantiated per case so the plain and the candidate paths do not share registers; the
// mixed single-row case is held to 64 registers, 4 CTAs per SM, as the others reach alone).
template <typename W, int MT, int CM>
__global__ void __launch_bounds__(256, MT == 1 ? 4 : 3) rowdot_kernel(MatArgs a, long total_rows) {
  extern __shared__ float xs[];                       // [MT][k]
  __shared__ float s_cv[MT][8][kTops];                // per-warp running candidate lists
  __shared__ int s_ci[MT][8][kTops];
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
    const bool cand = CM == 1 || (CM == 2 && s.cand);
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
        if (cand && lane < kTops) {
#pragma unroll
          for (int m = 0; m < MT; ++m) { s_cv[m][warp][lane] = NEG_INF; s_ci[m][warp][lane] = NO_IDX; }
        }
        // Rolling stream over the warp's rows rf, rf + 8, ... in groups of U 16-byte chunks
        // per lane: as each chunk of the current group is unpacked, the same chunk of the next
        // group (the next row's first group after a row's last) is requested, so U loads stay
        // in flight through the FMAs, the row's reduction and its epilogue.
        constexpr int GK = 32 * VEC * U;               // K covered by one group
        const int G = (k + GK - 1) / GK;               // groups per row (the last may be partial)
        const int nrow = rf < r1 ? (r1 - rf + 7) / 8 : 0;
        const W* wc = w + (long)rf * k + lane * VEC;   // group in buf (loaded above)
        const long to_next_row = 8L * k - (long)(G - 1) * GK;   // last group -> next row's first
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        int g = 0, r = rf;
        for (int left = nrow * G; left > 0; --left) {
          const W* wnx = wc + (g + 1 < G ? (long)GK : to_next_row);
          const int kb = lane * VEC + g * GK;
          const int kbn = g + 1 < G ? kb + GK : lane * VEC;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int kk = kb + u * 32 * VEC;
            const bool cur = kk < k;                   // a row's last group may be partial
            float f[VEC];
            if (cur) unpack16(buf[u], f);
            if (left > 1 && kbn + u * 32 * VEC < k) buf[u] = ld_stream16(wnx + u * 32 * VEC);
            if (!cur) continue;
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
          wc = wnx;
          if (++g == G) {                              // row r complete
            g = 0;
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] = warp_sum(acc[m]);
            if (cand) {
#pragma unroll
              for (int m = 0; m < MT; ++m)
                if (m < mt) warp_list_offer(s_cv[m][warp], s_ci[m][warp], acc[m], r, s.rounds);
            } else {
#pragma unroll
              for (int m = 0; m < MT; ++m)
                if (lane == m && m < mt) epilogue_store(a, s, si, m0 + m, r, acc[m]);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] = 0.f;
            r += 8;
          }
        }
        if (cand) {                                    // CTA-uniform
          __syncthreads();
          const int slot = (int)blockIdx.x - s.slot0;
          for (int m = 0; m < mt; ++m) {
            const long o = (((long)(m0 + m) * a.cand_nh + s.head) * a.cand_ld + slot) * kTops;
            rank_merge(s_cv[m], s_ci[m], 8, s.rounds, a.cand_val + o, a.cand_idx + o, threadIdx.x, blockDim.x);
          }
          __syncthreads();                             // the lists are refilled next
        }
      }
    }
    seg_start += s.rows;
  }
}

// Grid of one launch (or -1): one round of resident CTAs, at least one row per warp.  The
// fused top-k's slot counts come from the same number.
template <typename W, int MT, int CM>
static long rowdot_grid_t(const MatArgs& a, size_t smem) {
  static int num_sms = 0;
  if (!num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      num_sms = 148;
  }
  long total = 0;
  for (int i = 0; i < a.nseg; ++i) total += a.seg[i].rows;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(rowdot_kernel<W, MT, CM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return -1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rowdot_kernel<W, MT, CM>, 256, smem) !=
          cudaSuccess || per_sm < 1)
    per_sm = 1;
  long grid = (long)per_sm * num_sms;
  const long by_rows = (total + 7) / 8;
  grid = grid < by_rows ? grid : by_rows;
  return grid < 1 ? 1 : grid;
}

template <typename W, int MT, int CM>
static cudaError_t rowdot_go(const MatArgs& a, cudaStream_t st) {
  long total = 0;
  for (int i = 0; i < a.nseg; ++i) total += a.seg[i].rows;
  const size_t smem = (size_t)MT * a.k * sizeof(float);
  const long grid = rowdot_grid_t<W, MT, CM>(a, smem);
  if (grid < 0) return cudaErrorInvalidValue;
  return launch_kernel(rowdot_kernel<W, MT, CM>, dim3((unsigned)grid), dim3(256), smem, st, 1, a, total);
}

// Dispatch on the weight type, the activation rows per pass (MT = min(M, 4)) and which
// segments keep fused top-k (CM).
template <int CM, typename F>
static auto rowdot_dispatch_cm(const MatArgs& a, int dtype, F&& f) {
  const int mt = a.M >= 4 ? 4 : a.M;
  using C = std::integral_constant<int, CM>;
  if (dtype == 0) {
    switch (mt) {
      case 1: return f(std::integral_constant<int, 1>{}, float{}, C{});
      case 2: return f(std::integral_constant<int, 2>{}, float{}, C{});
      case 3: return f(std::integral_constant<int, 3>{}, float{}, C{});
      default: return f(std::integral_constant<int, 4>{}, float{}, C{});
    }
  }
  switch (mt) {
    case 1: return f(std::integral_constant<int, 1>{}, bf16{}, C{});
    case 2: return f(std::integral_constant<int, 2>{}, bf16{}, C{});
    case 3: return f(std::integral_constant<int, 3>{}, bf16{}, C{});
    default: return f(std::integral_constant<int, 4>{}, bf16{}, C{});
  }
}
template <typename F>
static auto rowdot_dispatch(const MatArgs& a, int dtype, F&& f) {
  int nc = 0;
  for (int i = 0; i < a.nseg; ++i) nc += a.seg[i].cand ? 1 : 0;
  if (nc == 0) return rowdot_dispatch_cm<0>(a, dtype, f);
  if (nc == a.nseg) return rowdot_dispatch_cm<1>(a, dtype, f);
  return rowdot_dispatch_cm<2>(a, dtype, f);
}

cudaError_t launch_rowdot(const MatArgs& a, int dtype, cudaStream_t st) {
  return rowdot_dispatch(a, dtype, [&](auto mt, auto w, auto cm) {
    return rowdot_go<decltype(w), decltype(mt)::value, decltype(cm)::value>(a, st);
  });
}

bool cand_geometry(const MatArgs& a, int si, bool tensor_cores, int dtype, int* count, int* first) {
  if (tensor_cores) {
    *count = (a.seg[si].rows + kCandTileRows - 1) / kCandTileRows;
    *first = 0;
    return true;
  }
  const long grid = rowdot_grid(a, dtype);
  if (grid < 1) return false;
  long total = 0, s0 = 0;
  for (int i = 0; i < a.nseg; ++i) {
    if (i < si) s0 += a.seg[i].rows;
    total += a.seg[i].rows;
  }
  const long c0 = rowdot_cta_of(s0, total, grid), c1 = rowdot_cta_of(s0 + a.seg[si].rows - 1, total, grid);
  *count = (int)(c1 - c0 + 1);
  *first = (int)c0;
  return true;
}

int rowdot_grid(const MatArgs& a, int dtype) {
  return (int)rowdot_dispatch(a, dtype, [&](auto mt, auto w, auto cm) {
    return rowdot_grid_t<decltype(w), decltype(mt)::value, decltype(cm)::value>(
        a, (size_t)decltype(mt)::value * a.k * sizeof(float));
  });
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
