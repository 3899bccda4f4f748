// Tensor-core (tcgen05) weight-streaming projection for sm_103a:
//   Y[m][r] = sum_k X[m][k] W[r][k]   (+ the step's epilogues, see MatArgs)
// for tens to hundreds of activation rows X against a weight matrix W that is read once.
//
// One CTA owns 128 weight rows and `nbox` activation rows.  The weights are the MMA's A
// operand (M = 128), the activations its B operand (N = nbox), both K-major bf16 tiles of
// 64 columns with the 128-byte swizzle, staged by TMA through an mbarrier ring.  fp32
// activations arrive as bf16 hi + lo halves; both MMAs accumulate into one fp32 TMEM
// accumulator, so the products keep ~fp32 accuracy at no extra TMEM.  Warp 0 lane 0
// issues the TMA loads, warp 1 lane 0 the MMAs; then all four warps read their 32 TMEM
// lanes, transpose through the idle stage ring and run the epilogue on whole rows.
//
// Every wait is bounded (~1 s of GPU time): on expiry the CTA sets MEDUSA_FLAG_TIMEOUT,
// drains (again bounded) the copies it issued, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace medusa {

constexpr int UM_R = 128;           // weight rows per CTA (MMA M)
constexpr int UM_K = 64;            // K per stage (one 128-byte swizzle row)
constexpr uint32_t UM_W_BYTES = UM_R * 128;
static_assert(UM_R == kCandTileRows, "fused top-k slots are the 128-row tiles");

struct UmmaArgs {
  CUtensorMap tw[kMaxSeg];   // weights of each segment: dims {k, rows}, box {64, 128}
  CUtensorMap ta[kMaxSeg];   // activations (hi): dims {k, M}, box {64, nbox}
  CUtensorMap tl[kMaxSeg];   // activations (lo)
  MatArgs m;
  int nbox;                  // activation rows per CTA = MMA N (multiple of 16, <= 256)
  int stages;
  int ksplit;                // K ranges (blockIdx.z); > 1 writes raw partials to kpart
  float* kpart;
  uint32_t tmem_cols;
  uint32_t* status;
};

__device__ __forceinline__ bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }
__device__ __forceinline__ bool aligned8(const void* p) { return ((uintptr_t)p & 7) == 0; }

// Residual of outputs r..r+3 of activation row m for EPI_SILU_RES / EPI_RES_ADD (n of them
// exist): 16-byte (fp32) or 8-byte (bf16) loads where all four exist and the address allows.
__device__ __forceinline__ float4 load_res4(const MatArgs& a, int m, int r, int n) {
  const long ro = (long)m * a.ldr + r;
  float res[4] = {0.f, 0.f, 0.f, 0.f};
  if (a.res_f32) {
    const float* rp = a.res_f32 + ro;
    if (n == 4 && aligned16(rp)) return *reinterpret_cast<const float4*>(rp);
    for (int e = 0; e < n; ++e) res[e] = rp[e];
  } else {
    const bf16* rw = reinterpret_cast<const bf16*>(a.res_w) + ro;
    if (n == 4 && aligned8(rw)) {
      const uint2 q = *reinterpret_cast<const uint2*>(rw);
      const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&q.x);
      const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&q.y);
      return make_float4(__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1));
    }
    for (int e = 0; e < n; ++e) res[e] = to_f32(rw[e]);
  }
  return make_float4(res[0], res[1], res[2], res[3]);
}

// Outputs r..r+3 (weight rows of segment s) of activation row m from the sums v and the
// residual (ignored for EPI_STORE): the activation, the fp32 store and the optional bf16
// hi/lo copies, vectorised where all four exist and the addresses allow it.
__device__ __forceinline__ void finish4(const MatArgs& a, const MatSeg& s, int m, int r, float4 v,
                                        float4 rv, int n) {
  float y[4] = {v.x, v.y, v.z, v.w};
  if (a.epi != EPI_STORE) {
    const float res[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = (a.epi == EPI_SILU_RES ? silu(y[e]) : y[e]) + res[e];
  }
  const long o = (long)m * a.ldo + s.out_off + r;
  float* op = a.out + o;
  if (n == 4 && aligned16(op)) *reinterpret_cast<float4*>(op) = make_float4(y[0], y[1], y[2], y[3]);
  else for (int e = 0; e < n; ++e) op[e] = y[e];
  if (a.out_hi) {
    bf16 hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_hi_lo(y[e], hi[e], lo[e]);
    bf16* hp = a.out_hi + o;
    bf16* lp = a.out_lo + o;
    if (n == 4 && aligned8(hp) && aligned8(lp)) {
      __nv_bfloat162 t[4] = {__halves2bfloat162(hi[0], hi[1]), __halves2bfloat162(hi[2], hi[3]),
                             __halves2bfloat162(lo[0], lo[1]), __halves2bfloat162(lo[2], lo[3])};
      *reinterpret_cast<uint2*>(hp) = *reinterpret_cast<const uint2*>(&t[0]);
      *reinterpret_cast<uint2*>(lp) = *reinterpret_cast<const uint2*>(&t[2]);
    } else {
      for (int e = 0; e < n; ++e) {
        hp[e] = hi[e];
        lp[e] = lo[e];
      }
    }
  }
}

// Outputs r..r+3 (weight rows of segment s) of activation row m: the epilogue, or the raw
// partial sum of a K range into kpart_row.
__device__ __forceinline__ void epilogue4(const MatArgs& a, const MatSeg& s, int m, int r, float4 v,
                                          float* kpart_row) {
  const int n = min(4, s.rows - r);
  if (kpart_row) {                                      // raw partial sum of a K range
    float* kp = kpart_row + s.out_off + r - a.kp_c0;
    const float y[4] = {v.x, v.y, v.z, v.w};
    if (n == 4 && aligned16(kp)) *reinterpret_cast<float4*>(kp) = v;
    else for (int e = 0; e < n; ++e) kp[e] = y[e];
    return;
  }
  const float4 rv = a.epi != EPI_STORE ? load_res4(a, m, r, n) : make_float4(0.f, 0.f, 0.f, 0.f);
  finish4(a, s, m, r, v, rv, n);
}

__device__ __forceinline__ void store4(float* p, const float (&y)[4]) {
  if (aligned16(p)) *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
  else for (int e = 0; e < 4; ++e) p[e] = y[e];
}
__device__ __forceinline__ void store4(bf16* p, const float (&y)[4]) {
  if (aligned8(p)) {
    __nv_bfloat162 t[2] = {__floats2bfloat162_rn(y[0], y[1]), __floats2bfloat162_rn(y[2], y[3])};
    *reinterpret_cast<uint2*>(p) = *reinterpret_cast<const uint2*>(t);
  } else {
    for (int e = 0; e < 4; ++e) p[e] = __float2bfloat16_rn(y[e]);
  }
}

// EPI_ROPE: outputs c0..c0+3 (x0) and c0+half..c0+half+3 (x1) of node row m, columns of
// the stacked q | k | v projection with c0 % dh < dh / 2.  q and k are rotated in pairs
// (i, i + dh/2) at the node's position (rotate-half form, cos | sin rows of the table):
//   y_i = x_i cos - x_{i+dh/2} sin,   y_{i+dh/2} = x_{i+dh/2} cos + x_i sin;
// v is passed through.  (Rotary position embedding as used by Llama, cited by "Medusa:
// Simple LLM Inference Acceleration Framework with Multiple Decoding Heads" for the
// position ids of the tree nodes.)
__device__ void rope4(const MatArgs& a, int m, int c0, float4 v0, float4 v1) {
  const int dh = a.rope_dh, half = dh / 2, qc = a.rope_qcols, kc = a.rope_kcols;
  float x0[4] = {v0.x, v0.y, v0.z, v0.w}, x1[4] = {v1.x, v1.y, v1.z, v1.w};
  if (c0 >= qc + kc) {                                  // v
    const long o = (long)m * kc + (c0 - qc - kc);
    if (a.rkv_bf16) {
      store4(reinterpret_cast<bf16*>(a.rv) + o, x0);
      store4(reinterpret_cast<bf16*>(a.rv) + o + half, x1);
    } else {
      store4(reinterpret_cast<float*>(a.rv) + o, x0);
      store4(reinterpret_cast<float*>(a.rv) + o + half, x1);
    }
    return;
  }
  int p = a.rope_pos[m];
  if (p < 0 || p >= a.rope_rows) {
    set_flag(a.rope_status, MEDUSA_FLAG_KV_CAPACITY);
    p = p < 0 ? 0 : a.rope_rows - 1;
  }
  const int i0 = c0 % dh;
  const float* cs = a.rope_table + (long)p * dh;
  float y0[4], y1[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float c = cs[i0 + e], sn = cs[half + i0 + e];
    y0[e] = x0[e] * c - x1[e] * sn;
    y1[e] = x1[e] * c + x0[e] * sn;
  }
  if (c0 < qc) {                                        // q
    const long o = (long)m * qc + c0;
    if (a.rq) {
      store4(a.rq + o, y0);
      store4(a.rq + o + half, y1);
    }
    if (a.rqb) {
      store4(a.rqb + o, y0);
      store4(a.rqb + o + half, y1);
    }
  } else {                                              // k
    const long o = (long)m * kc + (c0 - qc);
    if (a.rkv_bf16) {
      store4(reinterpret_cast<bf16*>(a.rk) + o, y0);
      store4(reinterpret_cast<bf16*>(a.rk) + o + half, y1);
    } else {
      store4(reinterpret_cast<float*>(a.rk) + o, y0);
      store4(reinterpret_cast<float*>(a.rk) + o + half, y1);
    }
  }
}

// Epilogue of a CTA's accumulators through shared memory.  Thread = TMEM lane = weight
// row, so reading TMEM gives each thread one output column for many activation rows;
// written out directly, a warp's store covers only 128 bytes of 16 different rows.
// Instead each chunk of 32 activation rows goes to `stage` ([32][rt] fp32, rt = 128 per
// accumulator) and comes back row-major: every thread then handles 4 consecutive
// outputs of one row (16-byte loads of the residual and stores of the result).  All 128
// threads must call this together.
__device__ void staged_epilogue(const MatArgs& a, const MatSeg& s, int rbase, int nacc, int m0,
                                int nbox, uint32_t tmem, uint32_t acc_stride, float* stage,
                                float* kpart /* split-K partials for blockIdx.z, or null */) {
  constexpr int CM = 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rt = 128 * nacc, q4 = rt / 4;
  for (int c0 = 0; c0 < nbox; c0 += CM) {
    const int cm = min(CM, nbox - c0);                  // 32, or a 16-column tail
    for (int t = 0; t < nacc; ++t) {
      for (int cc = 0; cc < cm; cc += 16) {
        float v[16];
        tmem_ld16(tmem + t * acc_stride + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c0 + cc), v);
#pragma unroll
        for (int j = 0; j < 16; ++j) stage[(cc + j) * rt + t * 128 + warp * 32 + lane] = v[j];
      }
    }
    __syncthreads();
    if (s.cand && !kpart) {
      // fused top-k: per activation row, the best of each 128 weight rows -> its slot
      for (int ml = warp; ml < cm; ml += 4) {
        const int m = m0 + c0 + ml;
        if (m >= a.M) break;
        for (int t = 0; t < nacc; ++t) {
          const float4 v = *reinterpret_cast<const float4*>(stage + ml * rt + t * 128 + 4 * lane);
          const int r0 = rbase + t * 128;
          const long o = (((long)m * a.cand_nh + s.head) * a.cand_ld + r0 / kCandTileRows) * kTops;
          warp_top_of_128(v, r0, s.rows, s.rounds, a.cand_val + o, a.cand_idx + o);
        }
      }
    } else if (a.epi == EPI_ROPE && !kpart) {
      // weight tiles start on head boundaries: both halves of every head are in the stage
      const int dh = a.rope_dh, half = dh / 2, gh = half / 4, heads = rt / dh;
      for (int i = tid; i < cm * heads * gh; i += 128) {
        const int ml = i / (heads * gh), rem = i - ml * heads * gh;
        const int hh = rem / gh, rl = hh * dh + 4 * (rem - hh * gh);
        const int m = m0 + c0 + ml, r = rbase + rl;
        if (m < a.M && r < s.rows) {
          const float4 v0 = *reinterpret_cast<const float4*>(stage + ml * rt + rl);
          const float4 v1 = *reinterpret_cast<const float4*>(stage + ml * rt + rl + half);
          rope4(a, m, s.out_off + r, v0, v1);
        }
      }
    } else {
      for (int i = tid; i < cm * q4; i += 128) {
        const int ml = i / q4, q = i - ml * q4;
        const int m = m0 + c0 + ml, r = rbase + 4 * q;
        if (m < a.M && r < s.rows) {
          const float4 v = *reinterpret_cast<const float4*>(stage + ml * rt + 4 * q);
          epilogue4(a, s, m, r, v, kpart ? kpart + ((long)blockIdx.z * a.M + m) * a.kp_ld : nullptr);
        }
      }
    }
    __syncthreads();
  }
}

template <bool HAS_LO>
__global__ void __launch_bounds__(128, 2) umma_gemm_kernel(const __grid_constant__ UmmaArgs g) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[2 * 8 + 2];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_issued, s_consumed, s_bad;
  const MatArgs& a = g.m;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int si = 0;
  while (si + 1 < a.nseg && (int)blockIdx.y >= a.tile_off[si + 1]) ++si;
  const MatSeg& s = a.seg[si];
  const int rbase = ((int)blockIdx.y - a.tile_off[si]) * UM_R;
  const int m0 = (int)blockIdx.x * g.nbox;
  const int nk = (a.k + UM_K - 1) / UM_K;
  const int kt0 = (int)((long)blockIdx.z * nk / g.ksplit);      // this CTA's K range
  const int nkl = (int)((long)(blockIdx.z + 1) * nk / g.ksplit) - kt0;
  const int S = g.stages;
  const uint32_t A_BYTES = (uint32_t)g.nbox * 128;
  const uint32_t STAGE = UM_W_BYTES + A_BYTES * (HAS_LO ? 2 : 1);
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (8 + i); };
  const uint32_t accb = bar0 + 8u * 16;
  const uint32_t never = bar0 + 8u * 17;               // nothing arrives on it (test hook)

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    mbar_init(accb, 1);
    mbar_init(never, 1);
    s_issued = 0;
    s_consumed = 0;
    s_bad = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), g.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Dependents may launch only once every CTA holds its TMEM: a later kernel's CTA can
  // then never take the columns an earlier kernel's CTA is still waiting for.
  pdl_trigger();
  const uint32_t tmem = tmem_slot;
  bool timed_out = false;

  if (warp == 0 && lane == 0) {                         // ---- TMA producer
    const uint64_t pw = policy_evict_first(), pa = policy_evict_last();
    // The weights of the first S stages go out before the wait for earlier kernels (no
    // kernel writes them); the activations after it.
    const int pre = nkl < S ? nkl : S;
    for (int j = 0; j < pre; ++j) {
      mbar_expect_tx(full(j), STAGE);
      tma_load_2d(base + j * STAGE, &g.tw[si], (kt0 + j) * UM_K, rbase, full(j), pw);
    }
    pdl_wait();
    const CUtensorMap* tw = &g.tw[si];
    const CUtensorMap* ta = &g.ta[si];
    const CUtensorMap* tl = &g.tl[si];
    int j = 0, st = 0;
    uint32_t ph = 0;                                    // phase of the ring's current pass
    for (; j < nkl; ++j) {
      const int kx = (kt0 + j) * UM_K;
      const uint32_t ws = base + st * STAGE;
      if (j >= pre) {
        if (!mbar_wait(empty(st), ph ^ 1, TC_TIMEOUT_NS)) { timed_out = true; break; }
        mbar_expect_tx(full(st), STAGE);
        tma_load_2d(ws, tw, kx, rbase, full(st), pw);
      }
      tma_load_2d(ws + UM_W_BYTES, ta, kx, m0, full(st), pa);
      if (HAS_LO) tma_load_2d(ws + UM_W_BYTES + A_BYTES, tl, kx, m0, full(st), pa);
      if (++st == S) { st = 0; ph ^= 1; }
    }
    s_issued = j;
    if (timed_out) s_bad = 1;
  } else if (warp == 1 && lane == 0) {                  // ---- MMA issuer
    const uint32_t idesc = idesc_bf16(UM_R, g.nbox);
    // descriptors of stage 0; stage st adds st * STAGE bytes to the start address field
    const uint64_t ad0 = sw128_desc(base), bd0 = sw128_desc(base + UM_W_BYTES);
    const uint64_t ld0 = sw128_desc(base + UM_W_BYTES + A_BYTES);
    const uint64_t dstep = STAGE >> 4;
    int j = 0, st = 0;
    uint32_t ph = 0;
    uint64_t off = 0;
    // failure-path test hook: a wait that runs out, as one on a copy that never lands
    if (a.test_wait_ns && !mbar_wait(never, 0, a.test_wait_ns)) timed_out = true;
    for (; j < nkl && !timed_out; ++j) {
      if (!mbar_wait(full(st), ph, TC_TIMEOUT_NS)) { timed_out = true; break; }
      tc_fence_after();
      const uint64_t ad = ad0 + off, bd = bd0 + off, ld = ld0 + off;
#pragma unroll
      for (int ks = 0; ks < UM_K / 16; ++ks) {          // +32 bytes along K per step
        umma_bf16(tmem, ad + 2 * ks, bd + 2 * ks, idesc, (j | ks) != 0);
        if (HAS_LO) umma_bf16(tmem, ad + 2 * ks, ld + 2 * ks, idesc, 1);
      }
      umma_commit(empty(st));                           // frees the stage when read
      if (++st == S) { st = 0; ph ^= 1; off = 0; } else { off += dstep; }
    }
    s_consumed = j;
    if (timed_out) s_bad = 1;
    umma_commit(accb);                                  // accumulator complete
  }
  __syncwarp();
  pdl_wait();                                           // the epilogue reads and writes globals
  // ---- epilogue, staged through the (now idle) ring
  const bool acc_ok = mbar_wait(accb, 0, TC_TIMEOUT_NS);
  tc_fence_after();
  // every MMA has read its stage and every copy has landed unless a wait expired
  const bool run = __syncthreads_and(acc_ok) && !s_bad && nkl > 0;
  if (run) {
    float* stage = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)));
    staged_epilogue(a, s, rbase, 1, m0, g.nbox, tmem, 0, stage, g.ksplit > 1 ? g.kpart : nullptr);
  }
  if (timed_out || !acc_ok) set_flag(g.status, MEDUSA_FLAG_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {                                       // drain copies issued but not consumed
    for (int j = s_consumed; j < s_issued; ++j)
      mbar_wait(full(j % S), (j / S) & 1, TC_TIMEOUT_NS / 16);
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, g.tmem_cols);
}

// ------------------------------------------------------------------ wide variant
// For hundreds to thousands of activation rows (the node projections at batch > 1) the
// 128 x nbox tiles above re-read their operands from L2 faster than the tensor cores use
// them.  Here a CTA owns 256 weight rows (two 128-row accumulators in TMEM) against up to
// 256 activation rows, for twice the MMA work of a 128-row tile per operand byte.  With
// fp32 activations (bf16 hi + lo tiles) a stage is 32 columns of K with the 64-byte
// swizzle, so the ring holds 4-5 stages instead of 2 and the tensor cores do not wait on
// L2; with bf16 activations it stays at 64 columns with the 128-byte swizzle (3-4 stages,
// and half as many ring hand-offs per MMA).  CTAs of neighbouring weight tiles read the
// same activation tiles, which L2 serves after the first read.
constexpr int UW_R = 256;                    // weight rows per CTA

struct UmmaWideArgs {
  CUtensorMap tw[kMaxSeg];   // weights of each segment: dims {k, rows}, box {64, 256}
  CUtensorMap ta, tl;        // activations (hi, lo), shared by all segments: box {64, nbox}
  MatArgs m;                 // tile_off counts 256-row tiles
  int wtiles;                // weight tiles of the launch (grid.y), from tile wt0 on
  int wt0;
  int nbox, stages, ksplit;
  float* kpart;
  uint32_t tmem_cols, acc_stride;
  uint32_t* status;
};

template <bool HAS_LO, int UW_K>
__global__ void __launch_bounds__(128, 1) umma_wide_kernel(const __grid_constant__ UmmaWideArgs g) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[2 * 8 + 2];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_issued, s_consumed, s_bad;
  constexpr uint32_t UW_W_BYTES = UW_R * UW_K * 2;    // one stage of weights
  const MatArgs& a = g.m;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wtile = (int)blockIdx.y + g.wt0;
  int si = 0;
  while (si + 1 < a.nseg && wtile >= a.tile_off[si + 1]) ++si;
  const MatSeg& s = a.seg[si];
  const int rbase = (wtile - a.tile_off[si]) * UW_R;
  const int rows_here = min(UW_R, s.rows - rbase);
  const int nacc = rows_here > 128 ? 2 : 1;
  const int m0 = (int)blockIdx.x * g.nbox;
  const int nk = (a.k + UW_K - 1) / UW_K;
  const int kt0 = (int)((long)blockIdx.z * nk / g.ksplit);
  const int nkl = (int)((long)(blockIdx.z + 1) * nk / g.ksplit) - kt0;
  const int S = g.stages;
  const uint32_t A_BYTES = (uint32_t)g.nbox * UW_K * 2;
  const uint32_t STAGE = UW_W_BYTES + A_BYTES * (HAS_LO ? 2 : 1);
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (8 + i); };
  const uint32_t accb = bar0 + 8u * 16;
  const uint32_t never = bar0 + 8u * 17;               // nothing arrives on it (test hook)

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    mbar_init(accb, 1);
    mbar_init(never, 1);
    s_issued = 0;
    s_consumed = 0;
    s_bad = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), g.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();                        // after the TMEM allocation, as above
  const uint32_t tmem = tmem_slot;
  bool timed_out = false;

  if (warp == 0 && lane == 0) {                         // ---- TMA producer
    const uint64_t pw = policy_evict_first(), pa = policy_evict_last();
    const uint32_t stage_tx = STAGE;
    // weights of the first S stages before the wait for earlier kernels, as above
    const int pre = nkl < S ? nkl : S;
    for (int j = 0; j < pre; ++j) {
      mbar_expect_tx(full(j), stage_tx);
      tma_load_2d(base + j * STAGE, &g.tw[si], (kt0 + j) * UW_K, rbase, full(j), pw);
    }
    pdl_wait();
    const CUtensorMap* tw = &g.tw[si];
    int j = 0, st = 0;
    uint32_t ph = 0;                                    // phase of the ring's current pass
    for (; j < nkl; ++j) {
      const int kx = (kt0 + j) * UW_K;
      const uint32_t ws = base + st * STAGE;
      if (j >= pre) {
        if (!mbar_wait(empty(st), ph ^ 1, TC_TIMEOUT_NS)) { timed_out = true; break; }
        mbar_expect_tx(full(st), stage_tx);
        tma_load_2d(ws, tw, kx, rbase, full(st), pw);
      }
      tma_load_2d(ws + UW_W_BYTES, &g.ta, kx, m0, full(st), pa);
      if (HAS_LO) tma_load_2d(ws + UW_W_BYTES + A_BYTES, &g.tl, kx, m0, full(st), pa);
      if (++st == S) { st = 0; ph ^= 1; }
    }
    s_issued = j;
    if (timed_out) s_bad = 1;
  } else if (warp == 1 && lane == 0) {                  // ---- MMA issuer
    const uint32_t idesc = idesc_bf16(128, g.nbox);
    // descriptors of stage 0; stage st adds st * STAGE bytes to the start address field
    auto desc = [](uint32_t at) { return UW_K == 32 ? sw64_desc(at) : sw128_desc(at); };
    const uint64_t a0 = desc(base), a1 = desc(base + UW_W_BYTES / 2);
    const uint64_t b0 = desc(base + UW_W_BYTES), l0 = desc(base + UW_W_BYTES + A_BYTES);
    const uint64_t dstep = STAGE >> 4;
    const uint32_t d1 = tmem + g.acc_stride;
    int j = 0, st = 0;
    uint32_t ph = 0;
    uint64_t off = 0;
    // failure-path test hook: a wait that runs out, as one on a copy that never lands
    if (a.test_wait_ns && !mbar_wait(never, 0, a.test_wait_ns)) timed_out = true;
    for (; j < nkl && !timed_out; ++j) {
      if (!mbar_wait(full(st), ph, TC_TIMEOUT_NS)) { timed_out = true; break; }
      tc_fence_after();
      const uint64_t bd = b0 + off, ld = l0 + off;
      {
        const uint64_t ad = a0 + off;
#pragma unroll
        for (int ks = 0; ks < UW_K / 16; ++ks) {
          umma_bf16(tmem, ad + 2 * ks, bd + 2 * ks, idesc, (j | ks) != 0);
          if (HAS_LO) umma_bf16(tmem, ad + 2 * ks, ld + 2 * ks, idesc, 1);
        }
      }
      if (nacc > 1) {
        const uint64_t ad = a1 + off;
#pragma unroll
        for (int ks = 0; ks < UW_K / 16; ++ks) {
          umma_bf16(d1, ad + 2 * ks, bd + 2 * ks, idesc, (j | ks) != 0);
          if (HAS_LO) umma_bf16(d1, ad + 2 * ks, ld + 2 * ks, idesc, 1);
        }
      }
      umma_commit(empty(st));                           // frees the stage
      if (++st == S) { st = 0; ph ^= 1; off = 0; } else { off += dstep; }
    }
    s_consumed = j;
    if (timed_out) s_bad = 1;
    umma_commit(accb);
  }
  __syncwarp();
  pdl_wait();
  const bool acc_ok = mbar_wait(accb, 0, TC_TIMEOUT_NS);
  tc_fence_after();
  // every MMA has read its stage and every copy has landed unless a wait expired: the
  // ring is free for staging
  const bool run = __syncthreads_and(acc_ok) && !s_bad && nkl > 0;
  if (run) {
    float* stage = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)));
    staged_epilogue(a, s, rbase, nacc, m0, g.nbox, tmem, g.acc_stride, stage,
                    g.ksplit > 1 ? g.kpart : nullptr);
  }
  if (timed_out || !acc_ok) set_flag(g.status, MEDUSA_FLAG_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {                                       // drain copies issued but not consumed
    for (int j = s_consumed; j < s_issued; ++j)
      mbar_wait(full(j % S), (j / S) & 1, TC_TIMEOUT_NS / 16);
  }
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, g.tmem_cols);
}

// Sum of the K-range partials (in K order) for 4 consecutive output columns per item, then
// the epilogue (single-segment launches) or a plain store (multi-segment EPI_STORE
// launches).  A thread takes IPT items a grid stride apart and issues all their loads (the
// partials and the residual) before the first sum, so each pass is one round trip.
// cols % 4 == 0.
template <int KS>
constexpr int reduce_ipt() { return KS <= 2 ? 4 : (KS <= 4 ? 2 : 1); }

template <int KS>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const MatArgs a, const float* __restrict__ kpart,
                                                            int cols) {
  constexpr int IPT = reduce_ipt<KS>();
  pdl_trigger();
  pdl_wait();
  const long kld = a.kp_ld;
  const long stride = (long)gridDim.x * blockDim.x;
  if (a.epi == EPI_ROPE) {
    // one item = 4 columns of the first half of a head and their partners dh/2 further on
    const int dh = a.rope_dh, half = dh / 2, gh = half / 4;
    const int per_row = (cols / dh) * gh;
    const long n = (long)a.M * per_row;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += stride) {
      const int m = (int)(i / per_row), rem = (int)(i - (long)m * per_row), hg = rem / gh;
      const int c0 = hg * dh + 4 * (rem - hg * gh);           // column within the partials
      float4 v0[KS], v1[KS];
#pragma unroll
      for (int z = 0; z < KS; ++z) {
        const float* row = kpart + ((long)z * a.M + m) * kld;
        v0[z] = __ldcg(reinterpret_cast<const float4*>(row + c0));
        v1[z] = __ldcg(reinterpret_cast<const float4*>(row + c0 + half));
      }
      float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
#pragma unroll
      for (int z = 0; z < KS; ++z) {
        s0.x += v0[z].x; s0.y += v0[z].y; s0.z += v0[z].z; s0.w += v0[z].w;
        s1.x += v1[z].x; s1.y += v1[z].y; s1.z += v1[z].z; s1.w += v1[z].w;
      }
      rope4(a, m, a.kp_c0 + c0, s0, s1);
    }
    return;
  }
  const int c4 = cols / 4;
  const long n = (long)a.M * c4;
  const bool res = a.nseg == 1 && a.epi != EPI_STORE;
  for (long i0 = blockIdx.x * (long)blockDim.x + threadIdx.x; i0 < n; i0 += stride * IPT) {
    float4 v[IPT][KS], rv[IPT];
#pragma unroll
    for (int t = 0; t < IPT; ++t) {
      const long i = i0 + t * stride;
      rv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < n) {
        const int m = (int)(i / c4), c = (int)(i - (long)m * c4) * 4;
#pragma unroll
        for (int z = 0; z < KS; ++z)
          v[t][z] = __ldcg(reinterpret_cast<const float4*>(kpart + ((long)z * a.M + m) * kld + c));
        if (res) rv[t] = load_res4(a, m, a.kp_c0 + c, 4);
      }
    }
#pragma unroll
    for (int t = 0; t < IPT; ++t) {
      const long i = i0 + t * stride;
      if (i >= n) break;
      const int m = (int)(i / c4), c = (int)(i - (long)m * c4) * 4;
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int z = 0; z < KS; ++z) {
        y.x += v[t][z].x; y.y += v[t][z].y; y.z += v[t][z].z; y.w += v[t][z].w;
      }
      if (a.nseg == 1) {
        finish4(a, a.seg[0], m, a.kp_c0 + c, y, rv[t], 4);
      } else {
        float* op = a.out + (long)m * a.ldo + a.kp_c0 + c;
        if (aligned16(op)) *reinterpret_cast<float4*>(op) = y;
        else { op[0] = y.x; op[1] = y.y; op[2] = y.z; op[3] = y.w; }
      }
    }
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map: `rows` rows of `cols` elements at `ld` elements apart; box
// {64, box_rows} with the 128-byte swizzle (box_cols 64) or {32, box_rows} with the
// 64-byte swizzle (box_cols 32), zero fill out of bounds.
static bool make_map(CUtensorMap* map, const void* ptr, long cols, long rows, long ld, int box_rows,
                     int box_cols = UM_K) {
  auto fn = encode_fn();
  if (!fn || !ptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Sums the partials of output columns kp_c0 .. kp_c0 + ncols - 1 and applies the epilogue.
template <int KS>
static cudaError_t reduce_go(const MatArgs& a, cudaStream_t st, int ncols) {
  static long wave = 0;                               // resident CTAs of this kernel
  if (!wave) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 148;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, splitk_reduce_kernel<KS>, 256, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    wave = (long)sms * per_sm;
  }
  const long n4 = (long)a.M * (ncols / 4);
  long blocks = (n4 + 256L * reduce_ipt<KS>() - 1) / (256L * reduce_ipt<KS>());
  if (blocks > wave) blocks = wave;
  if (blocks < 1) blocks = 1;
  return launch_kernel(splitk_reduce_kernel<KS>, dim3((unsigned)blocks), dim3(256), 0, st, 1, a, a.kpart, ncols);
}

static cudaError_t launch_splitk_reduce(const MatArgs& a, int ksplit, cudaStream_t st, int ncols = -1) {
  if (ncols < 0) ncols = a.nseg == 1 ? a.seg[0].rows : (int)a.ldo;
  switch (ksplit) {
    case 2: return reduce_go<2>(a, st, ncols);
    case 3: return reduce_go<3>(a, st, ncols);
    case 4: return reduce_go<4>(a, st, ncols);
    case 5: return reduce_go<5>(a, st, ncols);
    case 6: return reduce_go<6>(a, st, ncols);
    case 7: return reduce_go<7>(a, st, ncols);
    case 8: return reduce_go<8>(a, st, ncols);
    default: return cudaErrorInvalidValue;
  }
}

// K ranges for a launch of `ctas` CTAs that leaves SMs idle (single-segment launches, or
// plain stores): about per_sm resident CTAs per SM (two for the narrow kernel, one for the
// wide one: a second wave of split CTAs costs more than the idle SMs it would fill), at
// least 4 K blocks each, partials within kpart.
static int choose_ksplit(const MatArgs& a, long ctas, int nk, int num_sms, int per_sm) {
  const bool splittable = a.nseg == 1 || (a.epi == EPI_STORE && !a.out_hi) || a.epi == EPI_ROPE;
  if (!splittable || !a.kpart || ctas >= num_sms || (a.nseg == 1 ? a.seg[0].rows : a.ldo) % 4 != 0)
    return 1;
  int ksplit = (int)((long)per_sm * num_sms / ctas);
  ksplit = ksplit > 8 ? 8 : ksplit;
  ksplit = ksplit > nk / 4 ? nk / 4 : ksplit;
  while (ksplit > 1 && (size_t)ksplit * a.M * a.ldo * sizeof(float) > a.kpart_bytes) --ksplit;
  return ksplit < 1 ? 1 : ksplit;
}

static cudaError_t launch_umma_wide(const MatArgs& m, uint32_t* status, int num_sms, cudaStream_t st) {
  static UmmaWideArgs g;
  std::memset(&g, 0, sizeof(g));
  g.m = m;
  MatArgs& a = g.m;
  a.kp_ld = a.ldo;                                    // a split of the whole output
  a.kp_c0 = 0;
  a.tile_off[0] = 0;
  for (int i = 0; i < a.nseg; ++i) a.tile_off[i + 1] = a.tile_off[i] + (a.seg[i].rows + UW_R - 1) / UW_R;
  g.wtiles = a.tile_off[a.nseg];
  const bool has_lo = a.seg[0].a_lo != nullptr;
  const int UW_K = has_lo ? 32 : 64;                  // K per stage, see the kernel
  // activation tiles of <= 256 rows, as even as the count allows (multiple of 16)
  const int nct = (a.M + 255) / 256;
  g.nbox = ((a.M + nct - 1) / nct + 15) / 16 * 16;
  g.acc_stride = g.nbox > 128 ? 256 : 128;            // two accumulators of nbox columns
  g.tmem_cols = 2 * g.acc_stride;
  const uint32_t stage = (uint32_t)(UW_R + g.nbox * (has_lo ? 2 : 1)) * UW_K * 2;
  int stages = (int)((220u * 1024u) / stage);
  g.stages = stages > 8 ? 8 : stages;
  if (g.stages < 2) return cudaErrorInvalidValue;
  g.status = status;
  const int nk = (a.k + UW_K - 1) / UW_K;
  g.ksplit = choose_ksplit(a, (long)nct * g.wtiles, nk, num_sms, 1);
  g.kpart = a.kpart;
  for (int i = 0; i < a.nseg; ++i)
    if (!make_map(&g.tw[i], a.seg[i].w, a.k, a.seg[i].rows, a.k, UW_R, UW_K)) return cudaErrorInvalidValue;
  if (!make_map(&g.ta, a.seg[0].a_hi, a.k, a.M, a.seg[0].ldx, g.nbox, UW_K)) return cudaErrorInvalidValue;
  if (has_lo && !make_map(&g.tl, a.seg[0].a_lo, a.k, a.M, a.seg[0].ldx, g.nbox, UW_K)) return cudaErrorInvalidValue;
  // at least 116 KB of shared memory keeps one CTA per SM, so the 512-column TMEM
  // allocations of co-resident CTAs never wait on each other
  size_t smem = (size_t)g.stages * stage + 1024;
  if (smem < 116u * 1024u) smem = 116u * 1024u;
  auto kern = has_lo ? umma_wide_kernel<true, 32> : umma_wide_kernel<false, 64>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // A grid of more than one but not a whole number of waves (one CTA per SM) leaves the
  // last wave partly empty.  Then the weight tiles of the whole waves run as they are, and
  // the remaining ones split K so that their CTAs fill one more wave: their partials (for
  // their own output columns only) are summed by the reduce, which applies the epilogue.
  const long tiles = (long)nct * g.wtiles;
  const bool splittable = a.nseg == 1 || (a.epi == EPI_STORE && !a.out_hi) || a.epi == EPI_ROPE;
  if (g.ksplit == 1 && splittable && a.kpart && tiles > num_sms && tiles % num_sms != 0) {
    const int w1 = (int)((tiles / num_sms) * num_sms / nct);     // weight tiles of the whole waves
    const int tail = g.wtiles - w1;
    int si = 0;
    while (si + 1 < a.nseg && w1 >= a.tile_off[si + 1]) ++si;
    const int c0 = a.seg[si].out_off + (w1 - a.tile_off[si]) * UW_R;   // first output column of the tail
    const int c1 = a.nseg == 1 ? a.seg[0].rows : (int)a.ldo;
    int ks = (int)(num_sms / ((long)tail * nct));
    ks = ks > 8 ? 8 : ks;
    ks = ks > nk / 4 ? nk / 4 : ks;
    while (ks > 1 && (size_t)ks * a.M * (c1 - c0) * sizeof(float) > a.kpart_bytes) --ks;
    if (w1 > 0 && tail > 0 && ks >= 2 && (c1 - c0) % 4 == 0) {
      UmmaWideArgs gm = g;
      gm.wtiles = w1;
      gm.wt0 = 0;
      e = launch_kernel(kern, dim3(nct, w1, 1), dim3(128), smem, st, 1, gm);
      if (e != cudaSuccess) return e;
      g.wtiles = tail;
      g.wt0 = w1;
      g.ksplit = ks;
      a.kp_c0 = c0;
      a.kp_ld = c1 - c0;
      e = launch_kernel(kern, dim3(nct, tail, ks), dim3(128), smem, st, 1, g);
      if (e != cudaSuccess) return e;
      return launch_splitk_reduce(a, ks, st, c1 - c0);
    }
  }
  e = launch_kernel(kern, dim3(nct, g.wtiles, g.ksplit), dim3(128), smem, st, 1, g);
  if (e != cudaSuccess || g.ksplit == 1) return e;
  return launch_splitk_reduce(a, g.ksplit, st);
}

static bool any_cand(const MatArgs& a) {
  for (int i = 0; i < a.nseg; ++i)
    if (a.seg[i].cand) return true;
  return false;
}

// The wide variant needs every segment to read the same activations (one shared tile).
static bool shared_activations(const MatArgs& a) {
  for (int i = 1; i < a.nseg; ++i)
    if (a.seg[i].a_hi != a.seg[0].a_hi || a.seg[i].a_lo != a.seg[0].a_lo || a.seg[i].ldx != a.seg[0].ldx)
      return false;
  return true;
}

cudaError_t launch_umma_gemm(const MatArgs& m, uint32_t* status, cudaStream_t st) {
  static UmmaArgs g;                      // ~4.5 KB: keep it off the host stack
  static std::mutex mu;
  static int num_sms = 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      num_sms = 148;
  }
  {
    bool lo_ok = true;
    for (int i = 1; i < m.nseg; ++i)
      if ((m.seg[i].a_lo != nullptr) != (m.seg[0].a_lo != nullptr)) lo_ok = false;
    if (!lo_ok) return cudaErrorInvalidValue;
    if (m.M > 128 && shared_activations(m) && !any_cand(m)) return launch_umma_wide(m, status, num_sms, st);
  }
  std::memset(&g, 0, sizeof(g));
  g.m = m;
  MatArgs& a = g.m;
  a.kp_ld = a.ldo;                                    // a split of the whole output
  a.kp_c0 = 0;
  a.tile_off[0] = 0;
  for (int i = 0; i < a.nseg; ++i) a.tile_off[i + 1] = a.tile_off[i] + (a.seg[i].rows + UM_R - 1) / UM_R;
  const bool has_lo = a.seg[0].a_lo != nullptr;
  int nbox = (a.M + 15) / 16 * 16;
  const int cap = has_lo ? 128 : 256;
  nbox = nbox > cap ? cap : nbox;
  g.nbox = nbox;
  uint32_t cols = 32;
  while (cols < (uint32_t)nbox) cols <<= 1;
  g.tmem_cols = cols;
  // ring depth: two CTAs per SM when that leaves >= 3 stages, else one CTA with a deep ring
  const uint32_t stage = UM_W_BYTES + (uint32_t)nbox * 128 * (has_lo ? 2 : 1);
  int stages = (int)((110u * 1024u) / stage);
  if (stages < 3) stages = (int)((200u * 1024u) / stage);
  g.stages = stages > 8 ? 8 : stages;
  if (g.stages < 2) return cudaErrorInvalidValue;
  g.status = status;
  // split K when the tiles alone cannot cover the SMs
  const int nk = (a.k + UM_K - 1) / UM_K;
  const int mchunks = (a.M + nbox - 1) / nbox;
  // (the fused top-k needs whole sums in the epilogue: no K split)
  const int ksplit = any_cand(a) ? 1 : choose_ksplit(a, (long)mchunks * a.tile_off[a.nseg], nk, num_sms, 2);
  g.ksplit = ksplit;
  g.kpart = a.kpart;
  for (int i = 0; i < a.nseg; ++i) {
    const MatSeg& s = a.seg[i];
    if (!make_map(&g.tw[i], s.w, a.k, s.rows, a.k, UM_R)) return cudaErrorInvalidValue;
    if (!make_map(&g.ta[i], s.a_hi, a.k, a.M, s.ldx, nbox)) return cudaErrorInvalidValue;
    if (has_lo && !make_map(&g.tl[i], s.a_lo, a.k, a.M, s.ldx, nbox)) return cudaErrorInvalidValue;
  }
  const size_t smem = (size_t)g.stages * stage + 1024;
  auto kern = has_lo ? umma_gemm_kernel<true> : umma_gemm_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_kernel(kern, dim3(mchunks, a.tile_off[a.nseg], ksplit), dim3(128), smem, st, 1, g);
  if (e != cudaSuccess || ksplit == 1) return e;
  return launch_splitk_reduce(a, ksplit, st);
}

}  // namespace medusa
