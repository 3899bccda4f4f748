// Persistent tensor-core (tcgen05) tree attention for sm_103a, bf16 caches, dh = 64 or 128.
//
// The work is the same split-KV decomposition as the CUDA-core kernel in k_attn.cu
// ("Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding Heads"
// §3.4 Tree Attention, Steps 3 and 5): a unit is (prefix split or the tree keys, KV head
// g, sequence b, block of query rows; row = node x query head of g's group), and every
// unit writes one unnormalised partial (o, max, sum) per row for attn_combine_kernel.
// Here one CTA per SM walks a fixed stride of the units, so the K/V stream of the SM never
// stops for a CTA launch, and keys go in chunks of 128:
//
//   warps 8-10         producers: per unit the query tile(s) (warp 8, TMA), then the K and
//                      V chunks through two rings of 2 to 4 stages that run on across
//                      units: a K stage is freed as soon as its S products are done, a V
//                      stage after its P V products.  Contiguous caches and the tree keys
//                      come by TMA (warp 8); a paged cache is copied by all three warps
//                      with cp.async (each reads 32 page ids at once)
//   warp 11 (one lane) MMAs for two "slots", each with S (128 columns) and O (dh columns)
//                      in tensor memory: S = Q K^T, then O += P V with P read from tensor
//                      memory (the A operand), V from shared memory (MN-major)
//   warps 0-3, 4-7     two softmax warpgroups, one per slot, one query row per thread:
//                      S is read from TMEM, masked (ancestor bitmask for the tree keys),
//                      exponentiated in base 2 and written back over S as bf16 pairs: P
//                      never passes through shared memory.
//
// Slots take turns on the tensor cores: while one warpgroup exponentiates its S, the MMAs
// of the other slot run.  With more than 128 rows per group the two slots are the two
// query tiles of the unit and share every K/V chunk; with at most 128 rows both slots
// work on the same query tile and take alternate chunks, and at the end of the unit the
// first warpgroup merges the second slot's (o, max, sum) into its own before writing.
//
// The running maximum is raised lazily (only past 2^8 of headroom; O is then rescaled in
// TMEM).  Every wait is bounded; on expiry MEDUSA_FLAG_TIMEOUT is set, the CTA stops
// taking work, drains the copies it issued and frees its tensor memory.
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

constexpr int PP_ROWS = 128;     // query rows per tile (MMA M, TMEM lanes)
constexpr int PP_KEYS = 128;     // keys per chunk
constexpr int PP_MAXST = 4;      // K/V ring depth at most
constexpr int PP_PROD = 3;       // producer warps (all three copy a paged cache)
constexpr int PP_MMA_WARP = 8 + PP_PROD;
constexpr int PP_THREADS = (PP_MMA_WARP + 1) * 32;   // 8 softmax warps, producers, MMA warp
constexpr float PP_LAZY = 8.f;   // log2 headroom before O is rescaled
constexpr uint32_t PP_SLOT_COLS = 256;   // per slot: S [0, 128), O [128, 128 + dh)

struct AttnPPArgs {
  CUtensorMap tq;        // q bf16:    dims {dh, Hq, B*n1},   box {64, G, 128/G}
  CUtensorMap tk, tv;    // cache:     dims {dh, Hkv, slots}, box {64, 1, kbox}
  CUtensorMap ttk, ttv;  // tree K/V:  dims {dh, Hkv, B*n1},  box {64, 1, 128}
  AttnArgs a;
  int kbox;              // cache rows per TMA box: 128 (contiguous) or the page size
  int nt;                // 2: two query tiles per unit, one per slot; 1: one tile, alternate chunks
  int kst, vst;          // K and V ring depths
  int units;             // (nsplit + 1) * B * Hkv * nrb
};

// Barriers.  QF / QE: query tile loaded / no longer read.  KF / KE and VF / VE: K and V
// ring stages full / free.  Per slot: SF (S written), PR (P written: every thread of the
// warpgroup), OF (P V done).  MRG / MFR: the second slot's (max, sum) are in shared memory
// / consumed.  END: every MMA the CTA issued has completed.
enum {
  PB_QF = 0, PB_QE = 1, PB_KF = 2, PB_KE = PB_KF + PP_MAXST, PB_VF = PB_KE + PP_MAXST,
  PB_VE = PB_VF + PP_MAXST, PB_SF = PB_VE + PP_MAXST, PB_PR = PB_SF + 2, PB_OF = PB_PR + 2,
  PB_MRG = PB_OF + 2, PB_MFR = PB_MRG + 1, PB_END = PB_MFR + 1, PB_COUNT = PB_END + 1
};

// D[tmem] (+)= A(tmem) * B(smem desc), kind::f16: A is read from tensor memory (one row
// per lane, two bf16 per 32-bit column).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane; returns once written.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,"
      "%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// A bounded wait whose outcome is the same in every lane (TMEM accesses that follow are
// warp-collective).
__device__ __forceinline__ bool pp_warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, TC_TIMEOUT_NS));
}

// One unit of work, decoded identically by every role.
struct PPUnit {
  int split, g, b, rb;
  bool tree;
  int kbeg, kend, nch;
};

__device__ __forceinline__ PPUnit pp_unit(const AttnArgs& a, int u) {
  PPUnit w;
  const int per_split = a.B * a.Hkv * a.nrb;          // tree units come last
  w.split = u / per_split;
  int rem = u - w.split * per_split;
  w.b = rem / (a.Hkv * a.nrb);
  rem -= w.b * (a.Hkv * a.nrb);
  w.g = rem / a.nrb;
  w.rb = rem - w.g * a.nrb;
  w.tree = w.split == a.nsplit;
  int L = a.len[w.b];
  L = L < 0 ? 0 : (L > a.capacity ? a.capacity : L);
  w.kbeg = w.tree ? 0 : w.split * a.chunk;
  w.kend = w.tree ? a.n1 : min(L, w.kbeg + a.chunk);
  w.nch = w.kend > w.kbeg ? (w.kend - w.kbeg + PP_KEYS - 1) / PP_KEYS : 0;
  return w;
}

template <int DH>
__global__ void __launch_bounds__(PP_THREADS, 1) tree_attn_pp_kernel(const __grid_constant__ AttnPPArgs g) {
  constexpr int H = DH / 64;                         // 64-column halves of a head
  constexpr uint32_t QH = PP_ROWS * 128;             // one half of a Q tile: 16 KB
  constexpr uint32_t KVH = PP_KEYS * 128;            // one half of a K or V chunk: 16 KB
  constexpr uint32_t KV_CHUNK = H * KVH;             // one K (or V) chunk
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[PB_COUNT];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_kiss, s_kwait, s_viss, s_vwait, s_qiss, s_qwait, s_abort;
  __shared__ float2 s_ml[PP_ROWS];                   // second slot's (max, sum) per row
  const AttnArgs& a = g.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, R = a.n1 * G, nt = g.nt, SK = g.kst, SV = g.vst;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t qs = base, k0s = base + nt * H * QH, v0s = k0s + SK * KV_CHUNK;
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  if (tid == 0) {
    mbar_init(bar(PB_QF), 1);
    mbar_init(bar(PB_QE), 1);
    // paged caches: every lane of the producer warp arrives on a full stage (its own
    // copies, or a plain arrive next to lane 0's expected bytes for a TMA stage)
    const uint32_t fcount = a.page_table ? 32 * PP_PROD : 1;
    for (int i = 0; i < SK; ++i) {
      mbar_init(bar(PB_KF + i), fcount);
      mbar_init(bar(PB_KE + i), 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(bar(PB_VF + i), fcount);
      mbar_init(bar(PB_VE + i), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(PB_SF + s), 1);
      mbar_init(bar(PB_PR + s), PP_ROWS);
      mbar_init(bar(PB_OF + s), 1);
    }
    mbar_init(bar(PB_MRG), PP_ROWS);
    mbar_init(bar(PB_MFR), PP_ROWS);
    mbar_init(bar(PB_END), 1);
    s_kiss = s_kwait = s_viss = s_vwait = s_qiss = s_qwait = 0;
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == PP_MMA_WARP) tmem_alloc(smem_u32(&tmem_slot), 2 * PP_SLOT_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();                          // only once this CTA holds its TMEM
  const uint32_t tmem = tmem_slot;
  bool timed_out = false;
  auto aborted = [&]() { return *(volatile int*)&s_abort != 0; };

  if (warp >= 8 && warp < PP_MMA_WARP && (warp == 8 || a.page_table)) {
    // ------------------------------------------------------------ producers
    // Warp 8 loads the query tiles and issues every copy-engine load; with a paged cache
    // all producer warps copy prefix chunks (and arrive on each stage).
    const int pw = warp - 8;
    const uint64_t pol_kv = policy_evict_first(), pol_q = policy_evict_last();
    int gc = 0, qn = 0;                   // chunks and query tiles issued so far
    bool first = true;
    for (int u = blockIdx.x; u < g.units; u += gridDim.x) {
      const PPUnit w = pp_unit(a, u);
      if (w.nch == 0) continue;
      const int row0 = w.rb * PP_ROWS * nt;
      const int nta = nt == 2 ? (row0 + PP_ROWS < R ? 2 : 1) : 1;
      // The cached prefix is written by no kernel of this call: the first unit's first
      // K/V chunks go out before the wait for earlier kernels, its query tile after.
      const int pre = first && pw == 0 ? (w.tree ? 0 : min(w.nch, min(SK, SV))) : 0;
      const bool paged = !w.tree && a.page_table;
      // Page ids of a 32-page window starting at p0 (lane l holds page l), refreshed when a
      // chunk leaves it.  All lanes.
      int pref0 = -1 << 30, my_page = 0;
      auto page_window = [&](int t0, int& p0, int& mine) {
        if (t0 >= p0 && t0 + PP_KEYS <= p0 + 32 * a.page_size) return;
        p0 = t0 - t0 % a.page_size;
        const int t = p0 + lane * a.page_size;
        mine = 0;
        if (t < a.capacity) {
          mine = a.page_table[(long)w.b * a.pages_per_seq + t / a.page_size];
          if (mine < 0 || mine >= a.num_pages) {
            set_flag(a.status, MEDUSA_FLAG_PAGE_RANGE);
            mine = 0;
          }
        }
      };
      auto load_q = [&]() -> bool {
        if (pw != 0) return true;
        if (first) pdl_wait();
        first = false;
        bool ok = true;
        if (lane == 0 && qn > 0) ok = mbar_wait(bar(PB_QE), (qn - 1) & 1, TC_TIMEOUT_NS);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        if (lane == 0) {
          mbar_expect_tx(bar(PB_QF), nta * H * QH);
          for (int t = 0; t < nta; ++t) {
            const int node0 = (row0 + t * PP_ROWS) / G;
#pragma unroll
            for (int h = 0; h < H; ++h)
              tma_load_3d(qs + (t * H + h) * QH, &g.tq, h * 64, w.g * G, w.b * a.n1 + node0, bar(PB_QF), pol_q);
          }
          s_qiss = qn + 1;
        }
        ++qn;
        return true;
      };
      bool ok = pre > 0 || load_q();
      for (int i = 0; i < w.nch && ok; ++i) {
        if (i == pre && pre > 0) ok = load_q();
        if (!ok) break;
        const int c = gc + i;
        const int t0 = w.kbeg + i * PP_KEYS;
        if (paged) page_window(t0, pref0, my_page);
        // K of chunk c, then V (each into its own ring)
        for (int part = 0; part < 2 && ok; ++part) {
          const int S = part == 0 ? SK : SV;
          const int st = c % S;
          const int full = (part == 0 ? PB_KF : PB_VF) + st, empty = (part == 0 ? PB_KE : PB_VE) + st;
          bool got = true;
          if (lane == 0) got = mbar_wait(bar(empty), ((c / S) & 1) ^ 1, TC_TIMEOUT_NS);
          if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
          const uint32_t dst = (part == 0 ? k0s : v0s) + st * KV_CHUNK;
          if (paged) {
            // Paged prefix: a page holds only 16 rows of a head, so copy-engine boxes would
            // be small and many; the producer warps copy the chunk themselves, 16 bytes per
            // cp.async into the 128-byte-swizzled layout (warp pw takes the 32-row groups
            // pw, pw + 3, ...; lane l row l of a group), and each thread's arrive fires once
            // its own copies have landed.
            const char* src = static_cast<const char*>(part == 0 ? a.kc : a.vc);
            for (int grp = pw; grp < PP_KEYS / 32; grp += PP_PROD) {
              const int r = lane + 32 * grp, t = t0 + r;
              const int pg = __shfl_sync(0xffffffffu, my_page, min((t - pref0) / a.page_size, 31));
              const bool in = t < a.capacity;
              const char* row = src + (((long)pg * a.page_size + t % a.page_size) * a.Hkv + w.g) * (long)(DH * 2);
#pragma unroll
              for (int u = 0; u < DH / 8; ++u) {          // 16-byte units of the row
                const int h = u >> 3, uu = u & 7;
                cp_async16(dst + h * KVH + r * 128 + ((uu ^ (r & 7)) << 4), in ? row + u * 16 : src, in ? 16 : 0);
              }
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar(full)) : "memory");
            if (pw == 0 && lane == 0) {
              if (part == 0) s_kiss = c + 1;
              else s_viss = c + 1;
            }
            continue;
          }
          if (pw != 0 || lane != 0) {
            if (a.page_table) mbar_arrive(bar(full));    // the tree keys of a paged launch
            continue;
          }
          mbar_expect_tx(bar(full), KV_CHUNK);
          const CUtensorMap* tm = w.tree ? (part == 0 ? &g.ttk : &g.ttv) : (part == 0 ? &g.tk : &g.tv);
          if (w.tree) {
#pragma unroll
            for (int h = 0; h < H; ++h) tma_load_3d(dst + h * KVH, tm, h * 64, w.g, w.b * a.n1 + t0, bar(full), pol_kv);
          } else {
#pragma unroll
            for (int h = 0; h < H; ++h)
              tma_load_3d(dst + h * KVH, tm, h * 64, w.g, w.b * a.capacity + t0, bar(full), pol_kv);
          }
          if (part == 0) s_kiss = c + 1;
          else s_viss = c + 1;
        }
      }
      if (ok && pre == w.nch && pre > 0) ok = load_q();    // every chunk went out early
      if (!ok) {
        timed_out = lane == 0;
        break;
      }
      gc += w.nch;
      if (aborted()) break;
    }
    if (first && pw == 0) pdl_wait();
  } else if (warp == PP_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(PP_ROWS, PP_KEYS);
      const uint32_t id_pv = idesc_bf16(PP_ROWS, DH) | IDESC_B_MN_MAJOR;
      int gc = 0, qn = 0, mc = 0;
      int js0 = 0, js1 = 0;               // jobs (chunk x slot) issued per slot
      // stages of a paged cache were written by the producer warp's cp.async (the generic
      // proxy): make them visible to the tensor cores before the MMAs read them
      const bool generic = a.page_table != nullptr;
      auto wait_k = [&](int c) -> bool {
        if (!mbar_wait(bar(PB_KF + c % SK), (c / SK) & 1, TC_TIMEOUT_NS)) return false;
        s_kwait = c + 1;
        if (generic) fence_proxy_async();
        tc_fence_after();
        return true;
      };
      auto wait_v = [&](int c) -> bool {
        if (!mbar_wait(bar(PB_VF + c % SV), (c / SV) & 1, TC_TIMEOUT_NS)) return false;
        s_vwait = c + 1;
        if (generic) fence_proxy_async();
        tc_fence_after();
        return true;
      };
      auto issue_qk = [&](int slot, int tile, int c) {
        const uint32_t ks = k0s + (c % SK) * KV_CHUNK;
        const uint32_t d = tmem + slot * PP_SLOT_COLS;
#pragma unroll
        for (int h = 0; h < H; ++h)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, sw128_desc(qs + (tile * H + h) * QH) + 2 * kk, sw128_desc(ks + h * KVH) + 2 * kk,
                      id_qk, (h | kk) != 0);
        umma_commit(bar(PB_SF + slot));
      };
      auto wait_p = [&](int slot) -> bool {
        if (!mbar_wait(bar(PB_PR + slot), (slot ? js1 : js0) & 1, TC_TIMEOUT_NS)) return false;
        tc_fence_after();
        return true;
      };
      auto issue_pv = [&](int slot, int c, bool acc) {
        const uint32_t vs = v0s + (c % SV) * KV_CHUNK;
        const uint32_t d = tmem + slot * PP_SLOT_COLS + PP_KEYS;
        const uint32_t pa = tmem + slot * PP_SLOT_COLS;
#pragma unroll
        for (int kk = 0; kk < PP_KEYS / 16; ++kk)      // 16 keys per MMA: 8 columns of P
          umma_bf16_tmem_a(d, pa + 8 * kk, sw128_desc_mn(vs + kk * 2048, KVH), id_pv, acc || kk > 0);
        umma_commit(bar(PB_OF + slot));
        if (slot) ++js1;
        else ++js0;
      };
      bool dead = false;
      for (int u = blockIdx.x; u < g.units && !dead; u += gridDim.x) {
        const PPUnit w = pp_unit(a, u);
        if (w.nch == 0) continue;
        const int row0 = w.rb * PP_ROWS * nt;
        const int nta = nt == 2 ? (row0 + PP_ROWS < R ? 2 : 1) : 1;
        if (!mbar_wait(bar(PB_QF), qn & 1, TC_TIMEOUT_NS)) { dead = true; break; }
        s_qwait = ++qn;
        tc_fence_after();
        const int n = w.nch;
        if (nt == 2) {
          // every chunk goes to each active tile's slot
          if (!wait_k(gc)) { dead = true; break; }
          for (int s = 0; s < nta; ++s) issue_qk(s, s, gc);
          umma_commit(bar(PB_KE + gc % SK));
          if (n == 1) umma_commit(bar(PB_QE));
          for (int i = 0; i < n && !dead; ++i) {
            const int c = gc + i;
            if (!wait_v(c)) { dead = true; break; }
            for (int s = 0; s < nta; ++s) {
              if (!wait_p(s)) { dead = true; break; }
              issue_pv(s, c, i > 0);
              if (i + 1 < n) {
                if (s == 0 && !wait_k(c + 1)) { dead = true; break; }
                issue_qk(s, s, c + 1);
                if (s == nta - 1) {
                  umma_commit(bar(PB_KE + (c + 1) % SK));   // both tiles' S of chunk c + 1
                  if (i + 2 == n) umma_commit(bar(PB_QE));
                }
              }
            }
            if (!dead) umma_commit(bar(PB_VE + c % SV));     // both tiles' P V of chunk c
          }
        } else {
          // one tile: chunk i goes to slot i & 1; slot 1's O may be overwritten only after
          // the first warpgroup has merged it into the previous unit's partial
          if (!wait_k(gc)) { dead = true; break; }
          issue_qk(0, 0, gc);
          umma_commit(bar(PB_KE + gc % SK));
          if (n > 1) {
            if (!wait_k(gc + 1)) { dead = true; break; }
            issue_qk(1, 0, gc + 1);
            umma_commit(bar(PB_KE + (gc + 1) % SK));
          }
          if (n <= 2) umma_commit(bar(PB_QE));
          for (int i = 0; i < n; ++i) {
            const int s = i & 1, c = gc + i;
            if (!wait_v(c) || !wait_p(s)) { dead = true; break; }
            if (i == 1 && mc > 0 && !mbar_wait(bar(PB_MFR), (mc - 1) & 1, TC_TIMEOUT_NS)) { dead = true; break; }
            issue_pv(s, c, i > 1);
            umma_commit(bar(PB_VE + c % SV));
            if (i + 2 < n) {
              if (!wait_k(c + 2)) { dead = true; break; }
              issue_qk(s, 0, c + 2);
              umma_commit(bar(PB_KE + (c + 2) % SK));
              if (i + 3 == n) umma_commit(bar(PB_QE));
            }
          }
          ++mc;
        }
        gc += n;
        if (aborted()) break;
      }
      timed_out = dead;
      umma_commit(bar(PB_END));           // arrives once every MMA issued above is done
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    const int slot = warp >> 2, wl = warp & 3;
    const int r = wl * 32 + lane;                    // row within the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(wl * 32) << 16);
    const uint32_t scol = lane_base + slot * PP_SLOT_COLS;      // this slot's S / P
    const uint32_t ocol = scol + PP_KEYS;                       // this slot's O
    const float sl2 = a.scale * 1.4426950408889634f;           // scores in base-2 units
    int js = 0, mc = 0;
    int js1 = 0;                                     // slot 1's jobs (merging warpgroup)
    for (int u = blockIdx.x; u < g.units && !timed_out; u += gridDim.x) {
      const PPUnit w = pp_unit(a, u);
      const int row0 = w.rb * PP_ROWS * nt;
      const int tile = nt == 2 ? slot : 0;
      if (nt == 2 && row0 + tile * PP_ROWS >= R) continue;          // this tile has no rows
      if (nt == 1 && slot == 1 && w.nch == 0) continue;
      const int gr = row0 + tile * PP_ROWS + r;
      const bool row_ok = gr < R;
      const int node = gr / G;
      const bool live = row0 + tile * PP_ROWS + wl * 32 < R;       // the warp has rows
      const int njobs = nt == 2 ? w.nch : (w.nch + 1 - slot) / 2;
      float m_use = -INFINITY, l_acc = 0.f;
      for (int jj = 0; jj < njobs; ++jj) {
        const int i = nt == 2 ? jj : 2 * jj + slot;
        if (!pp_warp_wait(bar(PB_SF + slot), js & 1)) { timed_out = true; break; }
        tc_fence_after();
        if (live) {
          float s[PP_KEYS];
          tmem_ld64(scol, *reinterpret_cast<float(*)[64]>(s));
          tmem_ld64(scol + 64, *reinterpret_cast<float(*)[64]>(s + 64));
          const int t0 = w.kbeg + i * PP_KEYS;
          // a whole chunk of prefix keys needs no mask: the maximum is taken over the raw
          // scores and the scale is folded into the exponent's FMA below
          const bool full = !w.tree && t0 + PP_KEYS <= w.kend;
          float mx;
          if (full) {
            float q0 = s[0], q1 = s[1], q2 = s[2], q3 = s[3];
#pragma unroll
            for (int j = 4; j < PP_KEYS; j += 4) {
              q0 = fmaxf(q0, s[j]);
              q1 = fmaxf(q1, s[j + 1]);
              q2 = fmaxf(q2, s[j + 2]);
              q3 = fmaxf(q3, s[j + 3]);
            }
            mx = fmaxf(fmaxf(q0, q1), fmaxf(q2, q3)) * sl2;
          } else {
            uint32_t wbits[PP_KEYS / 32];            // ancestor bits of this chunk's keys
#pragma unroll
            for (int q = 0; q < PP_KEYS / 32; ++q) {
              const int wi = (t0 >> 5) + q;
              wbits[q] = !w.tree ? 0xffffffffu
                                 : (row_ok && wi < kMaskWords ? a.mask[(long)node * kMaskWords + wi] : 0u);
            }
            mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < PP_KEYS; ++j) {
              const bool bit = (wbits[j >> 5] >> (j & 31)) & 1u;
              const bool valid = (t0 + j < w.kend) && bit;
              s[j] = valid ? s[j] * sl2 : -INFINITY;
              mx = fmaxf(mx, s[j]);
            }
          }
          // The P V of this slot's previous chunk has completed (this S comes from a later
          // MMA of the same issuer, and its commit covers every earlier one), so O may be
          // rescaled here.
          const bool raise = m_use != -INFINITY && mx > m_use + PP_LAZY;
          if (__any_sync(0xffffffffu, raise)) {
            const float f = raise ? ex2_approx(m_use - mx) : 1.f;
#pragma unroll
            for (int c = 0; c < DH; c += 16) {
              float v[16];
              tmem_ld16(ocol + c, v);
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] *= f;
              tmem_st16(ocol + c, v);
            }
            if (raise) {
              l_acc *= f;
              m_use = mx;
            }
          }
          if (m_use == -INFINITY) m_use = mx;        // first keys of this row
          // P over the first 64 columns of S, in two stores of 64 keys
          float l0 = 0.f, l1 = 0.f;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t pk[32];
            if (full) {
              const float nm = -m_use;
#pragma unroll
              for (int j = 0; j < 64; j += 2) {
                const float p0 = ex2_approx(fmaf(s[64 * hf + j], sl2, nm));
                const float p1 = ex2_approx(fmaf(s[64 * hf + j + 1], sl2, nm));
                l0 += p0;
                l1 += p1;
                pk[j / 2] = pack_bf16x2(p0, p1);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 64; j += 2) {
                const float x0 = s[64 * hf + j], x1 = s[64 * hf + j + 1];
                const float p0 = x0 == -INFINITY ? 0.f : ex2_approx(x0 - m_use);
                const float p1 = x1 == -INFINITY ? 0.f : ex2_approx(x1 - m_use);
                l0 += p0;
                l1 += p1;
                pk[j / 2] = pack_bf16x2(p0, p1);
              }
            }
            tmem_st32(scol + 32 * hf, pk);
          }
          l_acc += l0 + l1;
        }
        tc_fence_before();
        mbar_arrive(bar(PB_PR + slot));
        ++js;
      }
      if (timed_out) break;
      // ---- the unit's partial
      const long prow = (((long)w.b * a.Hkv + w.g) * (a.nsplit + 1) + w.split) * R + gr;
      float* dst = a.part_o + prow * DH;
      if (nt == 2 || w.nch == 0) {
        if (njobs > 0 && live) {
          if (!pp_warp_wait(bar(PB_OF + slot), (js - 1) & 1)) { timed_out = true; break; }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < DH; c += 16) {
            float v[16];
            tmem_ld16(ocol + c, v);
            if (row_ok) {
#pragma unroll
              for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4*>(dst + c + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            }
          }
        } else if (row_ok) {
          for (int c = 0; c < DH; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (row_ok) {
          a.part_ml[prow * 2] = m_use * 0.6931471805599453f;     // back to natural-log units
          a.part_ml[prow * 2 + 1] = l_acc;
        }
        continue;
      }
      const int nj1 = w.nch / 2;                         // slot 1's chunks in this unit
      if (slot == 1) {
        // hand (max, sum) to the first warpgroup once it has consumed the previous ones
        if (mc > 0 && !pp_warp_wait(bar(PB_MFR), (mc - 1) & 1)) { timed_out = true; break; }
        s_ml[r] = make_float2(m_use, l_acc);
        mbar_arrive(bar(PB_MRG));
        ++mc;
        continue;
      }
      js1 += nj1;
      bool ok = pp_warp_wait(bar(PB_OF), (js - 1) & 1);
      if (ok && nj1 > 0) ok = pp_warp_wait(bar(PB_OF + 1), (js1 - 1) & 1);
      if (ok) ok = pp_warp_wait(bar(PB_MRG), mc & 1);
      if (!ok) { timed_out = true; break; }
      tc_fence_after();
      const float2 ml1 = s_ml[r];
      const float m = fmaxf(m_use, ml1.x);
      const float f0 = m_use == -INFINITY ? 0.f : ex2_approx(m_use - m);
      const float f1 = ml1.x == -INFINITY ? 0.f : ex2_approx(ml1.x - m);
      const uint32_t ocol1 = lane_base + PP_SLOT_COLS + PP_KEYS;
      if (live) {
#pragma unroll
        for (int c = 0; c < DH; c += 16) {
          float v0[16], v1[16];
          tmem_ld16(ocol + c, v0);
          if (nj1 > 0) {
            tmem_ld16(ocol1 + c, v1);            // written by this unit's P V of slot 1
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v1[e] = 0.f;
          }
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              *reinterpret_cast<float4*>(dst + c + e) =
                  make_float4(v0[e] * f0 + v1[e] * f1, v0[e + 1] * f0 + v1[e + 1] * f1,
                              v0[e + 2] * f0 + v1[e + 2] * f1, v0[e + 3] * f0 + v1[e + 3] * f1);
          }
        }
      }
      if (row_ok) {
        a.part_ml[prow * 2] = m * 0.6931471805599453f;
        a.part_ml[prow * 2 + 1] = l_acc * f0 + ml1.y * f1;
      }
      tc_fence_before();
      mbar_arrive(bar(PB_MFR));
      ++mc;
    }
  }
  if (timed_out) {
    set_flag(a.status, MEDUSA_FLAG_TIMEOUT);
    *(volatile int*)&s_abort = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    // every MMA done, then the copies issued but never waited for (bounded)
    mbar_wait(bar(PB_END), 0, TC_TIMEOUT_NS);
    if (s_qiss > s_qwait) mbar_wait(bar(PB_QF), (s_qiss - 1) & 1, TC_TIMEOUT_NS / 16);
    for (int c = s_kwait; c < s_kiss; ++c) mbar_wait(bar(PB_KF + c % SK), (c / SK) & 1, TC_TIMEOUT_NS / 16);
    for (int c = s_vwait; c < s_viss; ++c) mbar_wait(bar(PB_VF + c % SV), (c / SV) & 1, TC_TIMEOUT_NS / 16);
  }
  __syncthreads();
  if (warp == PP_MMA_WARP) tmem_dealloc(tmem, 2 * PP_SLOT_COLS);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_pp_fn() {
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
static bool make_map_pp(CUtensorMap* map, const void* ptr, long x, long y, long z, int by, int bz) {
  auto fn = encode_pp_fn();
  if (!fn || !ptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)x, (cuuint64_t)y, (cuuint64_t)z};
  cuuint64_t strides[2] = {(cuuint64_t)x * 2, (cuuint64_t)(x * y) * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)by, (cuuint32_t)bz};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tree_attention_pp_supported(int dtype, int dh, int G, int page_size) {
  if (dtype != 1 || (dh != 64 && dh != 128)) return false;
  if (G < 1 || G > PP_ROWS || PP_ROWS % G != 0) return false;
  if (page_size > 0 && (page_size < 8 || page_size > PP_KEYS || PP_KEYS % page_size != 0)) return false;
  return true;
}

int tree_attention_pp_units(int B, int Hkv, int nrb, int nsplit) { return (nsplit + 1) * B * Hkv * nrb; }

cudaError_t launch_tree_attention_pp(const AttnArgs& a, const void* q_bf16, int num_sms, cudaStream_t st) {
  static AttnPPArgs g;                     // ~700 bytes of tensor maps: kept off the stack
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  std::memset(&g, 0, sizeof(g));
  g.a = a;
  if (a.rows_per_block != PP_ROWS && a.rows_per_block != 2 * PP_ROWS) return cudaErrorInvalidValue;
  if (a.chunk % PP_KEYS != 0) return cudaErrorInvalidValue;
  g.nt = a.rows_per_block / PP_ROWS;
  g.units = tree_attention_pp_units(a.B, a.Hkv, a.nrb, a.nsplit);
  const int H = a.dh / 64;
  int optin = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    optin = 227 * 1024;
  void (*kern)(AttnPPArgs) = a.dh == 128 ? tree_attn_pp_kernel<128> : tree_attn_pp_kernel<64>;
  cudaFuncAttributes fa{};
  const size_t stat = cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.sharedSizeBytes : 4096;
  const size_t budget = (size_t)optin > stat ? (size_t)optin - stat : 0;
  const size_t fixed = 1024 + (size_t)g.nt * H * PP_ROWS * 128;
  const size_t chunk = (size_t)H * PP_KEYS * 128;             // one K or V chunk
  const int total = fixed < budget ? (int)std::min<size_t>(2 * PP_MAXST, (budget - fixed) / chunk) : 0;
  // V is needed later than K in a chunk's life, and freed later: give K the deeper ring
  g.vst = std::min(PP_MAXST, total / 2);
  g.kst = std::min(PP_MAXST, total - g.vst);
  if (g.kst < 2 || g.vst < 2) return cudaErrorInvalidValue;
  const size_t smem = fixed + (size_t)(g.kst + g.vst) * chunk;
  const long nodes = (long)a.B * a.n1;
  if (!make_map_pp(&g.tq, q_bf16, a.dh, a.Hq, nodes, a.G, PP_ROWS / a.G)) return cudaErrorInvalidValue;
  if (a.page_table) {
    g.kbox = a.page_size;
    const long slots = (long)a.num_pages * a.page_size;
    if (!make_map_pp(&g.tk, a.kc, a.dh, a.Hkv, slots, 1, a.page_size)) return cudaErrorInvalidValue;
    if (!make_map_pp(&g.tv, a.vc, a.dh, a.Hkv, slots, 1, a.page_size)) return cudaErrorInvalidValue;
  } else {
    g.kbox = PP_KEYS;
    const long slots = (long)a.B * a.capacity;
    if (!make_map_pp(&g.tk, a.kc, a.dh, a.Hkv, slots, 1, PP_KEYS)) return cudaErrorInvalidValue;
    if (!make_map_pp(&g.tv, a.vc, a.dh, a.Hkv, slots, 1, PP_KEYS)) return cudaErrorInvalidValue;
  }
  if (!make_map_pp(&g.ttk, a.tk, a.dh, a.Hkv, nodes, 1, PP_KEYS)) return cudaErrorInvalidValue;
  if (!make_map_pp(&g.ttv, a.tv, a.dh, a.Hkv, nodes, 1, PP_KEYS)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(g.units, num_sms));
  return launch_kernel(kern, dim3(grid), dim3(PP_THREADS), smem, st, 1, g);
}

}  // namespace medusa
