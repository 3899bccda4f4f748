// Tensor-core (tcgen05) tree attention for sm_103a, bf16 caches with dh = 64 or 128.
//
// Same split-KV decomposition and partial format as the CUDA-core kernel in k_attn.cu
// ("Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding Heads"
// §3.4 Tree Attention, Steps 3 and 5): CTA (split, kv head g, sequence b, row block) covers
// one chunk of the prefix, or (split == nsplit) the tree keys under the ancestor bitmask,
// for up to two 128-row query tiles (row = node x query head of the group) that share every
// K/V tile, so up to 256 rows read the prefix once.  Inside the CTA the keys are walked in
// chunks of 128 keys (one query tile) or 64 (two tiles, whose S buffers fill the TMEM):
//   warp 8 (one lane)  TMA: Q once, then K and V chunks through a 2- to 4-stage mbarrier ring
//                      (paged caches: one box per page)
//   warp 9 (one lane)  MMAs: S = Q K^T into one of two TMEM buffers per tile (issued one
//                      chunk ahead), then O += P V into the tile's TMEM accumulator, V as
//                      an MN-major operand
//   warps 0-7          one query row per thread (warps 4t..4t+3 for tile t): masked online
//                      softmax of S in base 2, P written as bf16 into one of two swizzled
//                      shared-memory buffers
// The running maximum is raised lazily: only when a row's new maximum exceeds the one its
// P values are taken against by more than 2^8 does the warp wait for the previous P V and
// rescale O in TMEM; otherwise P is formed against the old maximum (values <= 256) and O
// keeps accumulating in the tensor cores.  Each CTA writes one unnormalised partial
// (o, max, sum) per row, merged by attn_combine_kernel.  Every wait is bounded; on expiry
// MEDUSA_FLAG_TIMEOUT is set.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace medusa {

constexpr int AT_ROWS = 128;      // query rows per tile (MMA M, TMEM lanes)
constexpr int AT_TILES = 2;       // query tiles per CTA at most
constexpr int AT_KEYS = 64;       // keys per chunk with two query tiles (S columns, PV reduction)
constexpr int AT_KEYS1 = 128;     // keys per chunk with one query tile
constexpr int AT_STAGES = 4;      // K/V ring depth at most (3 when two query tiles)
constexpr int AT_WARPS = 4 * AT_TILES + 2;
constexpr float AT_LAZY = 8.f;           // log2 headroom before O is rescaled

struct AttnTcArgs {
  CUtensorMap tq;        // q bf16:    dims {dh, Hq, B*n1},   box {64, G, 128/G}
  CUtensorMap tk, tv;    // cache:     dims {dh, Hkv, slots}, box {64, 1, kbox}
  CUtensorMap ttk, ttv;  // tree K/V:  dims {dh, Hkv, B*n1},  box {64, 1, keys per chunk}
  AttnArgs a;
  int kbox;              // cache rows per TMA box: keys per chunk (contiguous) or the page size
  int nt;                // query tiles per CTA: rows_per_block / 128
  int stages;            // K/V ring depth (<= AT_STAGES)
};

// Barriers: Q loaded; K/V stage full / empty; per tile and buffer: S written (BSF), P V
// done (BOF), P written (BPR).  One P-written barrier per P buffer: the softmax warps can
// finish chunk i + 1 before the MMA thread has waited for chunk i, but never chunk i + 2
// (that needs the P V of chunk i), so no barrier runs two phases ahead of its waiter.
// With 128-key chunks (one tile) each row's keys are split over two softmax warps; BMX
// (two, by chunk parity) collects the 256 half-row maxima before either half forms P.
enum {
  BQ = 0, BKVF = 1, BKVE = BKVF + AT_STAGES, BSF = BKVE + AT_STAGES,
  BOF = BSF + 2 * AT_TILES, BPR = BOF + 2 * AT_TILES, BMX = BPR + 2 * AT_TILES, BCOUNT = BMX + 2
};

// A bounded wait whose outcome is the same in every lane (the TMEM accesses that follow
// are warp-collective).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, TC_TIMEOUT_NS));
}

// KEYS keys per chunk: 64 (up to two query tiles) or 128 (one tile).  TMEM per tile:
// S0 [0, KEYS), S1 [KEYS, 2 KEYS), O [2 KEYS, 2 KEYS + DH).
template <int DH, int KEYS>
__global__ void __launch_bounds__(AT_WARPS * 32, 1)
tree_attn_tc_kernel(const __grid_constant__ AttnTcArgs g) {
  constexpr int H = DH / 64;                        // 64-column halves of a head
  constexpr uint32_t QH = AT_ROWS * 128;            // one half of a Q tile: 16 KB
  constexpr uint32_t KVH = KEYS * 128;              // one half of a K or V chunk
  constexpr uint32_t KV_STAGE = 2 * H * KVH;
  constexpr uint32_t PA = AT_ROWS * 128;            // one 64-key swizzle atom of P: 16 KB
  constexpr uint32_t PT = PA * (KEYS / 64);         // one P buffer: 128 rows x KEYS keys bf16
  constexpr uint32_t TILE_COLS = KEYS == 64 ? 256 : 512;
  constexpr uint32_t OCOL = 2 * KEYS;               // O's first TMEM column
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[BCOUNT];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_issued, s_waited, s_qok;
  const AttnArgs& a = g.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, gk = blockIdx.y;
  const int b = blockIdx.z / a.nrb, rb = blockIdx.z % a.nrb;
  const int G = a.G, R = a.n1 * G, nt = g.nt, ST = g.stages;
  const int row0 = rb * AT_ROWS * nt;
  const int nta = min(nt, (R - row0 + AT_ROWS - 1) / AT_ROWS);   // tiles with rows
  const bool tree = split == a.nsplit;
  int L = a.len[b];
  L = L < 0 ? 0 : (L > a.capacity ? a.capacity : L);
  const int kbeg = tree ? 0 : split * a.chunk;
  const int kend = tree ? a.n1 : min(L, kbeg + a.chunk);
  const int nch = kend > kbeg ? (kend - kbeg + KEYS - 1) / KEYS : 0;
  const uint32_t sraw = smem_u32(smem_raw);
  const uint32_t base = (sraw + 1023u) & ~1023u;
  const uint32_t qs = base, kv0 = base + nt * H * QH, ps = kv0 + ST * KV_STAGE;
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t tmem_cols = TILE_COLS * nt;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  if (tid == 0) {
    mbar_init(bar(BQ), 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(bar(BKVF + i), 1);
      mbar_init(bar(BKVE + i), 1);
    }
    for (int i = 0; i < 2 * AT_TILES; ++i) {
      mbar_init(bar(BSF + i), 1);
      mbar_init(bar(BOF + i), 1);
      mbar_init(bar(BPR + i), KEYS == 128 ? 2 * AT_ROWS : AT_ROWS);   // every softmax thread
    }
    mbar_init(bar(BMX), 2 * AT_ROWS);
    mbar_init(bar(BMX + 1), 2 * AT_ROWS);
    s_issued = 0;
    s_waited = 0;
    s_qok = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 9) tmem_alloc(smem_u32(&tmem_slot), tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();                         // only once this CTA holds its TMEM
  const uint32_t tmem = tmem_slot;
  bool timed_out = false;
  if (warp != 8) pdl_wait();             // q, tree K/V and the outputs belong to this call

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 issues the copies.  For a paged cache the whole warp first reads the page ids
    // of the next 32 pages (lane l: page l), so a chunk's boxes never wait on a
    // dependent page-table load.
    // The cached prefix is written by no kernel of this call: the first ring of its K/V
    // chunks is requested before the wait for earlier kernels, Q and the tree keys after.
    if (nch > 0) {
      const uint64_t pol_kv = policy_evict_first(), pol_q = policy_evict_last();
      auto load_q = [&]() {
        pdl_wait();
        if (lane == 0) {
          mbar_expect_tx(bar(BQ), nta * H * QH);
          for (int t = 0; t < nta; ++t) {
            const int node0 = (row0 + t * AT_ROWS) / G;
#pragma unroll
            for (int h = 0; h < H; ++h)
              tma_load_3d(qs + (t * H + h) * QH, &g.tq, h * 64, gk * G, b * a.n1 + node0, bar(BQ), pol_q);
          }
        }
      };
      const int pre = tree ? 0 : (nch < ST ? nch : ST);
      const bool paged = !tree && a.page_table;
      int pref0 = -1 << 30, my_page = 0;               // first key covered by the page ids held
      int i = 0;
      for (; i < nch; ++i) {
        if (i == pre) load_q();
        const int st = i % ST;
        const int t0 = kbeg + i * KEYS;
        if (paged && (t0 < pref0 || t0 + KEYS > pref0 + 32 * a.page_size)) {
          pref0 = t0 - t0 % a.page_size;
          const int t = pref0 + lane * a.page_size;
          my_page = 0;
          if (t < a.capacity) {
            my_page = a.page_table[(long)b * a.pages_per_seq + t / a.page_size];
            if (my_page < 0 || my_page >= a.num_pages) {
              set_flag(a.status, MEDUSA_FLAG_PAGE_RANGE);
              my_page = 0;
            }
          }
        }
        int pages[KEYS / 8];                             // one per box of this chunk
        if (paged) {
          for (int j = 0, q = 0; j < KEYS; j += g.kbox, ++q)
            pages[q] = __shfl_sync(0xffffffffu, my_page, (t0 + j - pref0) / a.page_size);
        }
        bool ok = true;
        if (lane == 0) ok = mbar_wait(bar(BKVE + st), ((i / ST) & 1) ^ 1, TC_TIMEOUT_NS);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          timed_out = lane == 0;
          break;
        }
        if (lane != 0) continue;
        mbar_expect_tx(bar(BKVF + st), KV_STAGE);
        const uint32_t ks = kv0 + st * KV_STAGE, vs = ks + H * KVH;
        if (tree) {
#pragma unroll
          for (int h = 0; h < H; ++h) {
            tma_load_3d(ks + h * KVH, &g.ttk, h * 64, gk, b * a.n1 + t0, bar(BKVF + st), pol_kv);
            tma_load_3d(vs + h * KVH, &g.ttv, h * 64, gk, b * a.n1 + t0, bar(BKVF + st), pol_kv);
          }
        } else if (paged) {
          for (int j = 0, q = 0; j < KEYS; j += g.kbox, ++q) {
            const int row = pages[q] * a.page_size;
#pragma unroll
            for (int h = 0; h < H; ++h) {
              tma_load_3d(ks + h * KVH + j * 128, &g.tk, h * 64, gk, row, bar(BKVF + st), pol_kv);
              tma_load_3d(vs + h * KVH + j * 128, &g.tv, h * 64, gk, row, bar(BKVF + st), pol_kv);
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < H; ++h) {
            tma_load_3d(ks + h * KVH, &g.tk, h * 64, gk, b * a.capacity + t0, bar(BKVF + st), pol_kv);
            tma_load_3d(vs + h * KVH, &g.tv, h * 64, gk, b * a.capacity + t0, bar(BKVF + st), pol_kv);
          }
        }
      }
      if (i == nch && pre == nch) load_q();            // every chunk went out early
      if (lane == 0) s_issued = i;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // Per chunk i: S = Q K^T of chunk i + 1 goes first when its K/V stage has already
    // landed (the softmax can then move on as soon as it is done with chunk i); otherwise
    // O += P V of chunk i is not held back by that load, and S of chunk i + 1 follows it.
    // Waits block (no polling loop), so the softmax warps keep their issue slots.
    if (lane == 0 && nch > 0) {
      int waited = 0;
      if (!mbar_wait(bar(BQ), 0, TC_TIMEOUT_NS)) {
        timed_out = true;
      } else {
        s_qok = 1;
        const uint32_t id_qk = idesc_bf16(AT_ROWS, KEYS);
        const uint32_t id_pv = idesc_bf16(AT_ROWS, DH) | IDESC_B_MN_MAJOR;
        auto issue_qk = [&](int j) {
          waited = j + 1;
          tc_fence_after();
          const uint32_t ks = kv0 + (j % ST) * KV_STAGE;
          for (int t = 0; t < nta; ++t) {
            const uint32_t d = tmem + t * TILE_COLS + (uint32_t)(j & 1) * KEYS;
#pragma unroll
            for (int h = 0; h < H; ++h)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16(d, sw128_desc(qs + (t * H + h) * QH) + 2 * kk,
                          sw128_desc(ks + h * KVH) + 2 * kk, id_qk, (h | kk) != 0);
            umma_commit(bar(BSF + 2 * t + (j & 1)));
          }
        };
        if (mbar_wait(bar(BKVF), 0, TC_TIMEOUT_NS)) issue_qk(0);
        else timed_out = true;
        for (int i = 0; i < nch && !timed_out; ++i) {
          const int j = i + 1;
          bool qk_pending = j < nch;
          if (qk_pending && mbar_test(bar(BKVF + j % ST), (j / ST) & 1)) {
            issue_qk(j);
            qk_pending = false;
          }
          const uint32_t vs = kv0 + (i % ST) * KV_STAGE + H * KVH;
          for (int t = 0; t < nta && !timed_out; ++t) {
            if (!mbar_wait(bar(BPR + 2 * t + (i & 1)), (i >> 1) & 1, TC_TIMEOUT_NS)) { timed_out = true; break; }
            tc_fence_after();
            const uint32_t pt = ps + (uint32_t)(2 * t + (i & 1)) * PT;
#pragma unroll
            for (int kk = 0; kk < KEYS / 16; ++kk)           // 16 keys per MMA; P atom kk / 4
              umma_bf16(tmem + t * TILE_COLS + OCOL, sw128_desc(pt + (kk >> 2) * PA) + 2 * (kk & 3),
                        sw128_desc_mn(vs + kk * 2048, KVH), id_pv, (i | kk) != 0);
            umma_commit(bar(BOF + 2 * t + (i & 1)));
          }
          if (timed_out) break;
          umma_commit(bar(BKVE + i % ST));               // stage i read by every MMA
          if (qk_pending) {
            if (!mbar_wait(bar(BKVF + j % ST), (j / ST) & 1, TC_TIMEOUT_NS)) { timed_out = true; break; }
            issue_qk(j);
          }
        }
      }
      s_waited = waited;
    }
  } else if (KEYS == 128 && warp < 8) {
    // ------------------------------------------------------------ softmax, split rows
    // One tile: warps q and q + 4 share TMEM lanes 32q.. (row r); warp hf = warp / 4 takes
    // keys [64 hf, 64 hf + 64) of every chunk, writes that 64-key atom of P, rescales and
    // reads back O's columns [hf DH/2, (hf + 1) DH/2).  Per chunk the two halves swap their
    // maxima through spare TMEM columns of their row's lane (BMX orders the store before the
    // partner's load), so both form P against the same m_use.
    const int q = warp & 3, hf = warp >> 2;
    const int r = q * 32 + lane;
    const int gr = row0 + r;
    const int node = gr / G;
    const bool row_ok = gr < R;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t xcol = lane_base + OCOL + DH;    // [parity][half] maxima, then the sum
    uint8_t* pgen = smem_raw + (ps - sraw) + (size_t)hf * PA;
    const float sl2 = a.scale * 1.4426950408889634f;
    float m_use = -INFINITY, l_acc = 0.f;
    const bool live = row0 + q * 32 < R;
    for (int i = 0; i < nch; ++i) {
      const int bm = BMX + (i & 1);
      const uint32_t pmx = (uint32_t)(i >> 1) & 1u;
      if (!live) {                                  // keep pace and keep every barrier's count
        if (i >= 2 && !warp_wait(bar(BOF + (i & 1)), ((i - 2) >> 1) & 1)) { timed_out = true; break; }
        tc_fence_before();
        mbar_arrive(bar(bm));
        if (!warp_wait(bar(bm), pmx)) { timed_out = true; break; }
        mbar_arrive(bar(BPR + (i & 1)));
        continue;
      }
      if (!warp_wait(bar(BSF + (i & 1)), (i >> 1) & 1)) { timed_out = true; break; }
      tc_fence_after();
      float s[64];
      tmem_ld64(lane_base + (uint32_t)(i & 1) * KEYS + 64 * hf, s);
      const int t0 = kbeg + i * KEYS + 64 * hf;     // this half's first key
      const bool full = !tree && t0 + 64 <= kend;
      float mx;
      if (full) {
        float q0 = s[0], q1 = s[1], q2 = s[2], q3 = s[3];
#pragma unroll
        for (int j = 4; j < 64; j += 4) {
          q0 = fmaxf(q0, s[j]);
          q1 = fmaxf(q1, s[j + 1]);
          q2 = fmaxf(q2, s[j + 2]);
          q3 = fmaxf(q3, s[j + 3]);
        }
        mx = fmaxf(fmaxf(q0, q1), fmaxf(q2, q3)) * sl2;
      } else {
        uint32_t w[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int wi = (t0 >> 5) + u;
          w[u] = !tree ? 0xffffffffu
                       : (row_ok && wi < kMaskWords ? a.mask[(long)node * kMaskWords + wi] : 0u);
        }
        mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const bool bit = (w[j >> 5] >> (j & 31)) & 1u;
          const bool valid = (t0 + j < kend) && bit;
          s[j] = valid ? s[j] * sl2 : -INFINITY;
          mx = fmaxf(mx, s[j]);
        }
      }
      tmem_st1(xcol + 2 * (i & 1) + hf, mx);       // swap half-row maxima
      tc_fence_before();
      mbar_arrive(bar(bm));
      if (!warp_wait(bar(bm), pmx)) { timed_out = true; break; }
      tc_fence_after();
      mx = fmaxf(mx, tmem_ld1(xcol + 2 * (i & 1) + (hf ^ 1)));
      // this chunk's P buffer was last read by the P V of chunk i - 2
      if (i >= 2 && !warp_wait(bar(BOF + (i & 1)), ((i - 2) >> 1) & 1)) { timed_out = true; break; }
      const bool raise = m_use != -INFINITY && mx > m_use + AT_LAZY;
      if (__any_sync(0xffffffffu, raise)) {
        if (!warp_wait(bar(BOF + ((i - 1) & 1)), ((i - 1) >> 1) & 1)) { timed_out = true; break; }
        tc_fence_after();
        const float f = raise ? ex2_approx(m_use - mx) : 1.f;
#pragma unroll
        for (int c = 0; c < DH / 2; c += 16) {
          float v[16];
          tmem_ld16(lane_base + OCOL + hf * (DH / 2) + c, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= f;
          tmem_st16(lane_base + OCOL + hf * (DH / 2) + c, v);
        }
        if (raise) {
          l_acc *= f;
          m_use = mx;
        }
      }
      if (m_use == -INFINITY) m_use = mx;
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
      if (full) {
        const float nm = -m_use;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          s[j] = ex2_approx(fmaf(s[j], sl2, nm));
          s[j + 1] = ex2_approx(fmaf(s[j + 1], sl2, nm));
          s[j + 2] = ex2_approx(fmaf(s[j + 2], sl2, nm));
          s[j + 3] = ex2_approx(fmaf(s[j + 3], sl2, nm));
          l0 += s[j];
          l1 += s[j + 1];
          l2 += s[j + 2];
          l3 += s[j + 3];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            s[j + e] = s[j + e] == -INFINITY ? 0.f : ex2_approx(s[j + e] - m_use);
          l0 += s[j];
          l1 += s[j + 1];
          l2 += s[j + 2];
          l3 += s[j + 3];
        }
      }
      l_acc += (l0 + l1) + (l2 + l3);
      uint8_t* prow = pgen + (size_t)(i & 1) * PT + r * 128;   // this half's 64-key atom
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 u;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(s[8 * c + 0], s[8 * c + 1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(s[8 * c + 2], s[8 * c + 3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(s[8 * c + 4], s[8 * c + 5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(s[8 * c + 6], s[8 * c + 7]);
        u.x = *reinterpret_cast<uint32_t*>(&p0);
        u.y = *reinterpret_cast<uint32_t*>(&p1);
        u.z = *reinterpret_cast<uint32_t*>(&p2);
        u.w = *reinterpret_cast<uint32_t*>(&p3);
        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = u;
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bar(BPR + (i & 1)));
    }
    // the row's sum is the two halves' sums (the same m_use), exchanged through BMX once more
    const int bm = BMX + (nch & 1);
    float l_other = 0.f;
    if (!timed_out) {
      if (hf == 1) tmem_st1(xcol + 4, l_acc);
      tc_fence_before();
      mbar_arrive(bar(bm));
      if (!warp_wait(bar(bm), (uint32_t)(nch >> 1) & 1u)) timed_out = true;
      tc_fence_after();
      if (!timed_out && hf == 0) l_other = tmem_ld1(xcol + 4);
    }
    float o[DH / 2];
#pragma unroll
    for (int c = 0; c < DH / 2; ++c) o[c] = 0.f;
    if (!timed_out && nch > 0 && live) {
      if (!warp_wait(bar(BOF + ((nch - 1) & 1)), ((nch - 1) >> 1) & 1)) {
        timed_out = true;
      } else {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DH / 2; c += 16) {
          float v[16];
          tmem_ld16(lane_base + OCOL + hf * (DH / 2) + c, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[c + e] = v[e];
        }
      }
    }
    if (row_ok && !timed_out) {
      const long pr = (((long)b * a.Hkv + gk) * (a.nsplit + 1) + split) * R + gr;
      float4* dst = reinterpret_cast<float4*>(a.part_o + pr * DH + hf * (DH / 2));
#pragma unroll
      for (int c = 0; c < DH / 2; c += 4) dst[c / 4] = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
      if (hf == 0) {
        a.part_ml[pr * 2] = m_use * 0.6931471805599453f;     // back to natural-log units
        a.part_ml[pr * 2 + 1] = l_acc + l_other;
      }
    }
  } else if (KEYS == 64 && warp < 4 * nta) {
    // ------------------------------------------------------------ softmax rows
    const int t = warp >> 2, wl = warp & 3;
    const int r = wl * 32 + lane;                   // row within the tile = TMEM lane
    const int gr = row0 + t * AT_ROWS + r;
    const int node = gr / G;
    const bool row_ok = gr < R;
    const uint32_t lane_base = tmem + t * TILE_COLS + ((uint32_t)(wl * 32) << 16);
    uint8_t* pgen = smem_raw + (ps - sraw) + (size_t)(2 * t) * PT;
    const float sl2 = a.scale * 1.4426950408889634f;      // scores in base-2 units
    float m_use = -INFINITY, l_acc = 0.f;
    // A warp whose 32 rows all lie past the block's rows only keeps pace: its arrivals
    // for chunk i wait, as the others' do, until the P V of chunk i - 2 is done (its P
    // rows are left as they are; their products land in O rows nobody reads).
    const bool live = row0 + t * AT_ROWS + wl * 32 < R;
    for (int i = 0; i < nch && !live; ++i) {
      if (i >= 2 && !warp_wait(bar(BOF + 2 * t + (i & 1)), ((i - 2) >> 1) & 1)) { timed_out = true; break; }
      mbar_arrive(bar(BPR + 2 * t + (i & 1)));
    }

    for (int i = 0; i < nch && live; ++i) {
      if (!warp_wait(bar(BSF + 2 * t + (i & 1)), (i >> 1) & 1)) { timed_out = true; break; }
      tc_fence_after();
      float s[KEYS];
#pragma unroll
      for (int h = 0; h < KEYS / 64; ++h)
        tmem_ld64(lane_base + (uint32_t)(i & 1) * KEYS + 64 * h, *reinterpret_cast<float(*)[64]>(s + 64 * h));
      const int t0 = kbeg + i * KEYS;
      // A whole chunk of prefix keys needs no mask: the maximum is taken over the raw
      // scores and the scale is folded into the exponent's FMA below.
      const bool full = !tree && t0 + KEYS <= kend;
      float mx;
      if (full) {
        float q0 = s[0], q1 = s[1], q2 = s[2], q3 = s[3];
#pragma unroll
        for (int j = 4; j < KEYS; j += 4) {
          q0 = fmaxf(q0, s[j]);
          q1 = fmaxf(q1, s[j + 1]);
          q2 = fmaxf(q2, s[j + 2]);
          q3 = fmaxf(q3, s[j + 3]);
        }
        mx = fmaxf(fmaxf(q0, q1), fmaxf(q2, q3)) * sl2;
      } else {
        uint32_t w[KEYS / 32];                       // ancestor bits of this chunk's keys
#pragma unroll
        for (int q = 0; q < KEYS / 32; ++q) {
          const int wi = (t0 >> 5) + q;
          w[q] = !tree ? 0xffffffffu
                       : (row_ok && wi < kMaskWords ? a.mask[(long)node * kMaskWords + wi] : 0u);
        }
        mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < KEYS; ++j) {
          const bool bit = (w[j >> 5] >> (j & 31)) & 1u;
          const bool valid = (t0 + j < kend) && bit;
          s[j] = valid ? s[j] * sl2 : -INFINITY;
          mx = fmaxf(mx, s[j]);
        }
      }
      // this chunk's P buffer was last read by the P V of chunk i - 2
      if (i >= 2 && !warp_wait(bar(BOF + 2 * t + (i & 1)), ((i - 2) >> 1) & 1)) { timed_out = true; break; }
      const bool raise = m_use != -INFINITY && mx > m_use + AT_LAZY;
      if (__any_sync(0xffffffffu, raise)) {
        // O must hold the P V of chunk i - 1 before it is rescaled
        if (!warp_wait(bar(BOF + 2 * t + ((i - 1) & 1)), ((i - 1) >> 1) & 1)) { timed_out = true; break; }
        tc_fence_after();
        const float f = raise ? ex2_approx(m_use - mx) : 1.f;
#pragma unroll
        for (int c = 0; c < DH; c += 16) {
          float v[16];
          tmem_ld16(lane_base + OCOL + c, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= f;
          tmem_st16(lane_base + OCOL + c, v);
        }
        if (raise) {
          l_acc *= f;
          m_use = mx;
        }
      }
      if (m_use == -INFINITY) m_use = mx;             // first keys of this row
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
      if (full) {
        const float nm = -m_use;
#pragma unroll
        for (int j = 0; j < KEYS; j += 4) {
          s[j] = ex2_approx(fmaf(s[j], sl2, nm));
          s[j + 1] = ex2_approx(fmaf(s[j + 1], sl2, nm));
          s[j + 2] = ex2_approx(fmaf(s[j + 2], sl2, nm));
          s[j + 3] = ex2_approx(fmaf(s[j + 3], sl2, nm));
          l0 += s[j];
          l1 += s[j + 1];
          l2 += s[j + 2];
          l3 += s[j + 3];
        }
      } else {
#pragma unroll
        for (int j = 0; j < KEYS; j += 4) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            s[j + e] = s[j + e] == -INFINITY ? 0.f : ex2_approx(s[j + e] - m_use);
          l0 += s[j];
          l1 += s[j + 1];
          l2 += s[j + 2];
          l3 += s[j + 3];
        }
      }
      l_acc += (l0 + l1) + (l2 + l3);
      // P row (bf16) into the 128-byte-swizzled K-major tile the PV MMA reads
      uint8_t* prow = pgen + (size_t)(i & 1) * PT + r * 128;
#pragma unroll
      for (int c = 0; c < KEYS / 8; ++c) {            // 16-byte unit c: atom c / 8, unit c % 8
        uint4 u;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(s[8 * c + 0], s[8 * c + 1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(s[8 * c + 2], s[8 * c + 3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(s[8 * c + 4], s[8 * c + 5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(s[8 * c + 6], s[8 * c + 7]);
        u.x = *reinterpret_cast<uint32_t*>(&p0);
        u.y = *reinterpret_cast<uint32_t*>(&p1);
        u.z = *reinterpret_cast<uint32_t*>(&p2);
        u.w = *reinterpret_cast<uint32_t*>(&p3);
        *reinterpret_cast<uint4*>(prow + (c >> 3) * PA + (((c & 7) ^ (r & 7)) << 4)) = u;
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bar(BPR + 2 * t + (i & 1)));
    }
    float o[DH];
#pragma unroll
    for (int c = 0; c < DH; ++c) o[c] = 0.f;
    if (!timed_out && nch > 0 && live) {
      if (!warp_wait(bar(BOF + 2 * t + ((nch - 1) & 1)), ((nch - 1) >> 1) & 1)) {
        timed_out = true;
      } else {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DH; c += 64) {
          float v[64];
          tmem_ld64(lane_base + OCOL + c, v);
#pragma unroll
          for (int e = 0; e < 64; ++e) o[c + e] = v[e];
        }
      }
    }
    if (row_ok) {
      const long pr = (((long)b * a.Hkv + gk) * (a.nsplit + 1) + split) * R + gr;
      float4* dst = reinterpret_cast<float4*>(a.part_o + pr * DH);
#pragma unroll
      for (int c = 0; c < DH; c += 4) dst[c / 4] = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
      a.part_ml[pr * 2] = m_use * 0.6931471805599453f;     // back to natural-log units
      a.part_ml[pr * 2 + 1] = l_acc;
    }
  }
  if (timed_out) set_flag(a.status, MEDUSA_FLAG_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && nch > 0) {                 // drain copies issued but never waited for
    if (!s_qok) mbar_wait(bar(BQ), 0, TC_TIMEOUT_NS / 16);
    for (int i = s_waited; i < s_issued; ++i)
      mbar_wait(bar(BKVF + i % ST), (i / ST) & 1, TC_TIMEOUT_NS / 16);
  }
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, tmem_cols);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode3_fn() {
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

// bf16 [z][y][x] tensor (x contiguous, x = dh), box {64, by, bz}, 128-byte swizzle.
static bool make_map3(CUtensorMap* map, const void* ptr, long x, long y, long z, int by, int bz) {
  auto fn = encode3_fn();
  if (!fn || !ptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)x, (cuuint64_t)y, (cuuint64_t)z};
  cuuint64_t strides[2] = {(cuuint64_t)x * 2, (cuuint64_t)(x * y) * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)by, (cuuint32_t)bz};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tree_attention_tc_supported(int dtype, int dh, int G, int page_size) {
  if (dtype != 1 || (dh != 64 && dh != 128)) return false;
  if (G < 1 || G > AT_ROWS || AT_ROWS % G != 0) return false;
  if (page_size > 0 && (page_size < 8 || page_size > AT_KEYS || AT_KEYS % page_size != 0)) return false;
  return true;
}

cudaError_t launch_tree_attention_tc(const AttnArgs& a, const void* q_bf16, cudaStream_t st) {
  static AttnTcArgs g;                     // ~700 bytes of tensor maps: kept off the stack
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  std::memset(&g, 0, sizeof(g));
  g.a = a;
  if (a.rows_per_block != AT_ROWS && a.rows_per_block != AT_ROWS * AT_TILES) return cudaErrorInvalidValue;
  g.nt = a.rows_per_block / AT_ROWS;
  const int H = a.dh / 64;
  // shared memory: Q tiles, two P buffers per tile, then as many K/V stages as fit in the
  // per-CTA maximum less the kernel's own static shared memory
  int optin = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    optin = 227 * 1024;
  auto kernel_for = [&](int keys) -> void (*)(AttnTcArgs) {
    if (a.dh == 128) return keys == AT_KEYS1 ? tree_attn_tc_kernel<128, AT_KEYS1> : tree_attn_tc_kernel<128, AT_KEYS>;
    return keys == AT_KEYS1 ? tree_attn_tc_kernel<64, AT_KEYS1> : tree_attn_tc_kernel<64, AT_KEYS>;
  };
  auto plan = [&](int keys, size_t& smem) {
    cudaFuncAttributes fa{};
    const size_t stat = cudaFuncGetAttributes(&fa, kernel_for(keys)) == cudaSuccess ? fa.sharedSizeBytes : 4096;
    const size_t budget = (size_t)optin > stat ? (size_t)optin - stat : 0;
    const size_t fixed = 1024 + (size_t)g.nt * H * AT_ROWS * 128 + (size_t)g.nt * 2 * AT_ROWS * keys * 2;
    const size_t kv_stage = (size_t)2 * H * keys * 128;
    const int stages = fixed < budget ? (int)std::min<size_t>(AT_STAGES, (budget - fixed) / kv_stage) : 0;
    smem = fixed + (size_t)stages * kv_stage;
    return stages;
  };
  // one query tile: 128-key chunks (half the MMA issues, waits and commits per key) when
  // two stages of them fit; two tiles keep 64-key chunks (TMEM holds 2 x 256 columns)
  size_t smem = 0;
  int keys = AT_KEYS;
  g.stages = plan(AT_KEYS, smem);
  if (g.nt == 1) {
    size_t smem1 = 0;
    const int st1 = plan(AT_KEYS1, smem1);
    if (st1 >= 2) { keys = AT_KEYS1; g.stages = st1; smem = smem1; }
  }
  if (g.stages < 2) return cudaErrorInvalidValue;
  const long nodes = (long)a.B * a.n1;
  if (!make_map3(&g.tq, q_bf16, a.dh, a.Hq, nodes, a.G, AT_ROWS / a.G)) return cudaErrorInvalidValue;
  if (a.page_table) {
    g.kbox = a.page_size;
    const long slots = (long)a.num_pages * a.page_size;
    if (!make_map3(&g.tk, a.kc, a.dh, a.Hkv, slots, 1, a.page_size)) return cudaErrorInvalidValue;
    if (!make_map3(&g.tv, a.vc, a.dh, a.Hkv, slots, 1, a.page_size)) return cudaErrorInvalidValue;
  } else {
    g.kbox = keys;
    const long slots = (long)a.B * a.capacity;
    if (!make_map3(&g.tk, a.kc, a.dh, a.Hkv, slots, 1, keys)) return cudaErrorInvalidValue;
    if (!make_map3(&g.tv, a.vc, a.dh, a.Hkv, slots, 1, keys)) return cudaErrorInvalidValue;
  }
  if (!make_map3(&g.ttk, a.tk, a.dh, a.Hkv, nodes, 1, keys)) return cudaErrorInvalidValue;
  if (!make_map3(&g.ttv, a.tv, a.dh, a.Hkv, nodes, 1, keys)) return cudaErrorInvalidValue;
  void (*kern)(AttnTcArgs) = kernel_for(keys);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nsplit + 1, a.Hkv, a.B * a.nrb);
  return launch_kernel(kern, grid, dim3(AT_WARPS * 32), smem, st, 1, g);
}

}  // namespace medusa
