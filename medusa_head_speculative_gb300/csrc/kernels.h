// Internal launcher interface between the C ABI (capi.cu) and the kernel files.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/medusa.h"

namespace medusa {

typedef __nv_bfloat16 bf16;

constexpr int kMaxSeg = 10;     // LM head + up to 8 Medusa heads (+1 spare)
constexpr int kTops = 16;       // candidates kept per head (MEDUSA_MAX_TOPS)
constexpr int kMaskWords = 8;   // 256 nodes / 32

enum Epi { EPI_STORE = 0, EPI_SILU_RES = 1, EPI_RES_ADD = 2, EPI_ROPE = 3 };

// One row block of a stacked projection Y[m][out_off + r] = sum_k X[m][k] W[r][k].
struct MatSeg {
  const void* w;                 // [rows][k] weights (dtype)
  const float* x;                // CUDA-core path: fp32 activations [M][ldx]
  const __nv_bfloat16* a_hi;     // tensor-core path: bf16 activations [M][ldx]
  const __nv_bfloat16* a_lo;     // low halves of the fp32 activations, or null
  long ldx;                      // activation row stride (elements)
  int rows;
  int out_off;
  // Fused top-k (vocab projections of the heads): when `cand` is set the block's outputs
  // are not stored; instead each CTA writes, per activation row m, the best `rounds`
  // (logit, token) pairs of the rows it computed (sorted, then sentinels up to kTops) to
  // MatArgs::cand_val / cand_idx at [m][head][slot][kTops], token = row index r.  The slot
  // is the CTA's index among those covering the block: the 128-row tile for the
  // tensor-core path; for the row-dot blockIdx.x - slot0, slot0 = rowdot_cta_of(first row).
  int cand, head, rounds, slot0;
};

struct MatArgs {
  MatSeg seg[kMaxSeg];
  int nseg;
  int tile_off[kMaxSeg + 1];     // tensor-core path: first row tile of each segment
  int M, k;
  float* out;                    // out[m * ldo + out_off + r]
  long ldo;
  int epi;
  const float* res_f32;          // residual res[m * ldr + r] (fp32) ...
  const void* res_w;             // ... or in the weights' dtype
  long ldr;
  __nv_bfloat16* out_hi;         // optional bf16 hi/lo copies of out (same indexing)
  __nv_bfloat16* out_lo;
  float* kpart;                  // tensor-core path: scratch for split-K partials, or null
  size_t kpart_bytes;
  // layout of the split-K partials: kpart[z][m][kp_ld], holding output columns
  // kp_c0 .. kp_c0 + kp_ld - 1 (set by the launcher; a split of the whole output has
  // kp_c0 = 0 and kp_ld = ldo)
  long kp_ld;
  int kp_c0;
  // EPI_ROPE (tensor-core path, segments q | k | v of one head size): rotary embedding of
  // the q and k outputs at position rope_pos[m] (cos | sin rows of rope_table), then q to
  // rq (fp32, optional) and rqb (bf16, optional), k to rk and v to rv in the cache dtype
  // (bf16 when rkv_bf16, else fp32); `out` is not written.
  const int32_t* rope_pos;
  const float* rope_table;
  int rope_rows, rope_dh, rope_qcols, rope_kcols;
  float* rq;
  __nv_bfloat16* rqb;
  void* rk;
  void* rv;
  int rkv_bf16;
  uint32_t* rope_status;
  // CUDA-core row-dot only: when out_alt is set, segments from alt_from on store their
  // raw sums to out_alt[m * ldo_alt + out_off + r] instead (no epilogue), so the heads'
  // first projection and the LM head can share one launch.
  int alt_from;
  float* out_alt;
  long ldo_alt;
  // Tensor-core path, failure-path tests only (0 otherwise): the MMA thread first waits
  // on a barrier that nothing arrives on, for at most this many nanoseconds, and then
  // takes the expired-wait path.
  unsigned long long test_wait_ns;
  // fused top-k output of the segments with `cand` set: [M][cand_nh][cand_ld][kTops]
  float* cand_val;
  int32_t* cand_idx;
  int cand_nh, cand_ld;
};

// CUDA-core row-dot projection: dtype 0 = f32 weights, 1 = bf16.
cudaError_t launch_rowdot(const MatArgs& a, int dtype, cudaStream_t st);
// CTAs of that launch (one round: as many as are resident at once, >= 8 rows each).
int rowdot_grid(const MatArgs& a, int dtype);
// Row-dot CTA c computes the stacked rows [total*c/grid, total*(c+1)/grid); the CTA that
// computes row x is the largest c with floor(total*c/grid) <= x.
__host__ __device__ inline long rowdot_cta_of(long x, long total, long grid) {
  return ((x + 1) * grid + total - 1) / total - 1;
}
// Tensor-core path with fused top-k: 128-row tiles of a block (its slots).
constexpr int kCandTileRows = 128;
// Fused top-k geometry of segment si of a heads launch `a` (its `cand` flags set as
// launched): the candidate slots it writes per (activation row, head), and on the row-dot
// path the first CTA covering it (MatSeg::slot0; 0 on the tensor-core path, whose slots are
// its 128-row tiles).  False when the row-dot's launch geometry cannot be had.
bool cand_geometry(const MatArgs& a, int si, bool tensor_cores, int dtype, int* count, int* first);
// Tensor-core (tcgen05 + TMA + TMEM) projection; bf16 weights only.  Sets
// MEDUSA_FLAG_TIMEOUT in *status if a pipeline wait expires.
cudaError_t launch_umma_gemm(const MatArgs& a, uint32_t* status, cudaStream_t st);
// fp32 -> bf16 hi/lo split of n elements.
cudaError_t launch_split(const float* x, __nv_bfloat16* hi, __nv_bfloat16* lo, long n,
                         cudaStream_t st);
// X[m][:] = E[tok[m]][:], written as fp32 (xf) or bf16 (xb); one of them non-null.
cudaError_t launch_gather(const void* emb, int dtype, const int32_t* tok, int M, int d, int V,
                          float* xf, __nv_bfloat16* xb, cudaStream_t st);

// ---- heads top-k and tree
struct TopkArgs {
  const float* logits;   // [B][nh][V]
  int B, nh, V, splits, chunk;
  float* cand_val;       // [B][nh][splits][kTops]
  int32_t* cand_idx;
  int rounds[MEDUSA_MAX_HEADS + 1];   // ranks needed per head (0 = all kTops); the rest
                                      // of each list is left as sentinels
  int k0;                             // first head to select (1: the root is given and
                                      // the LM head's logits were not computed)
};
cudaError_t launch_topk_partial(const TopkArgs& a, cudaStream_t st);

// Merge of the vocab slices: per-head top-16 (head 0 = LM head) and the root token.
struct MergeArgs {
  const float* cand_val; const int32_t* cand_idx;
  int B, K, V, splits;
  const int32_t* root_in;
  int32_t* topk_tok; float* topk_val; int32_t* root_out;              // [B][K][kTops], [B]
  uint32_t* status;
  int rounds[MEDUSA_MAX_HEADS + 1];   // as TopkArgs::rounds
  int k0;                             // as TopkArgs::k0 (requires root_in when 1)
};
cudaError_t launch_topk_merge(const MergeArgs& a, cudaStream_t st);

struct TreeArgs {
  const int32_t* topk_tok; const int32_t* root; const int32_t* len;
  int B, K, V, n1;
  const int32_t* parent; const int32_t* depth; const int32_t* rank;   // device spec [n1]
  int32_t* tok; int32_t* pos;                                         // [B][n1]
  uint32_t* mask; int32_t* retrieve;                                  // [n1][8], [n1][K+1]
  uint32_t* status;
};
cudaError_t launch_tree_build(const TreeArgs& a, cudaStream_t st);
// Resident 256-thread slice top-k CTAs per SM (0 when the query fails).
int topk_partial_ctas_per_sm();

// Selection from the fused top-k candidates (MatSeg::cand): CTA (head, sequence) merges
// the head's `count[head]` slot lists into its final top list (fin_val / fin_idx,
// [B][nh][kTops]); the last CTA of a sequence (atomic counter, reset on exit) merges the
// heads, picks the root and writes the node tokens and positions.
struct CandArgs {
  const float* cand_val; const int32_t* cand_idx;     // [B][nh][ld][kTops]
  int B, nh, ld, k0;
  int count[MEDUSA_MAX_HEADS + 1];
  int rounds[MEDUSA_MAX_HEADS + 1];
  float* fin_val; int32_t* fin_idx;                  // [B][nh][kTops]
};
cudaError_t launch_cand_select(const CandArgs& c, const MergeArgs& m, const TreeArgs& tr,
                               int32_t* counter, cudaStream_t st);

// qkv [M][(Hq+2Hkv)*dh] fp32 -> q [M][Hq][dh] fp32 (RoPE; also as bf16 into qb when
// non-null), tree k (RoPE) / v in dtype.
// table: [rows][dh] = cos(p theta_i) for i < dh/2, then sin(p theta_i); built by rope_table.
cudaError_t launch_rope_split(const float* qkv, const int32_t* pos, int M, int Hq, int Hkv, int dh,
                              const float* table, int rows, uint32_t* status, int dtype, float* q,
                              __nv_bfloat16* qb, void* tk, void* tv, cudaStream_t st);
// Host: cos/sin of p * base^(-2i/dh) for p < rows, computed in double.
void rope_table(float base, int dh, int rows, float* out);

// ---- attention
struct AttnArgs {
  const float* q;
  const void* kc; const void* vc;
  const int32_t* page_table; int page_size; int pages_per_seq; int num_pages;
  const int32_t* len; int capacity;
  const void* tk; const void* tv;
  const uint32_t* mask;
  int B, n1, Hq, Hkv, G, dh;
  int nsplit, chunk;
  int rows_per_block, nrb, rpw;
  float* part_o; float* part_ml;
  float* o; __nv_bfloat16* o_hi; __nv_bfloat16* o_lo;
  uint32_t* status;
  float scale;
};
cudaError_t launch_tree_attention(const AttnArgs& a, int dtype, cudaStream_t st);
cudaError_t launch_attn_combine(const AttnArgs& a, cudaStream_t st);
// Persistent tensor-core tree attention (bf16, dh 64/128, G | 128, page size 8..128
// dividing 128): rows_per_block 128 or 256, chunk a multiple of 128; one CTA per SM at
// most (num_sms), each walking a fixed stride of the (split, KV head, sequence, row block)
// units.  q_bf16: [B*n1][Hq][dh].
bool tree_attention_pp_supported(int dtype, int dh, int G, int page_size);
cudaError_t launch_tree_attention_pp(const AttnArgs& a, const void* q_bf16, int num_sms, cudaStream_t st);
// fp32 -> bf16 (round to nearest) of n elements.
cudaError_t launch_to_bf16(const float* x, __nv_bfloat16* y, long n, cudaStream_t st);

// ---- verify
struct VerifyArgs {
  const float* logits;      // [M][V]
  const int32_t* tok; const int32_t* parent; const int32_t* depth;
  int B, n1, V, K, P, d;
  int typical; float temperature, eps, delta;       // typical: softmax statistics per row
  int reject; const float* uniforms;                // rejection sampling: [B][1 + 16 K]
  int32_t* am; float* stats;                        // [M], [M][4]
  const int32_t* retrieve; const float* hprime;     // [n1][K+1], [M][d]
  int32_t* out_tok; int32_t* n_acc; int32_t* path_nodes; float* h_next; int32_t* root_next;
  uint32_t* status;
};
cudaError_t launch_verify_stats(const VerifyArgs& a, cudaStream_t st);
cudaError_t launch_verify_accept(const VerifyArgs& a, cudaStream_t st);

struct CompactArgs {
  void* kc; void* vc;
  const int32_t* page_table; int page_size; int pages_per_seq; int num_pages;
  const int32_t* len; int32_t* len_out; int capacity;
  const void* tk; const void* tv;
  const int32_t* path_nodes; const int32_t* n_acc;
  int B, n1, Hkv, dh, K, dtype;
  uint32_t* status;
  int no_copy;              // fused commit: acceptance only (a multi-layer step compacts after)
};
cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t st);
// Compaction of up to kLayersPerLaunch backbone layers: grid (B, nl), block (b, l) copies
// sequence b's kept nodes from layer l's tree K/V into layer l's cache (base.len: the
// lengths before the step).  With write_len, the last block of a sequence (counter cnt[b],
// zero on entry, left zero) writes base.len_out[b], so len_out may alias len.
constexpr int kLayersPerLaunch = 16;
struct CompactLayersArgs {
  CompactArgs base;
  int nl, write_len;
  int32_t* cnt;
  void* kc[kLayersPerLaunch];
  void* vc[kLayersPerLaunch];
  const void* tk[kLayersPerLaunch];
  const void* tv[kLayersPerLaunch];
};
cudaError_t launch_kv_compact_layers(const CompactLayersArgs& a, cudaStream_t st);

// ---- optimized tree on the device (one CTA): acc [K][smax] doubles; fmax = N*smax + smax
// frontier entries; parent / rank [N+1] in canonical packing; expected [N+1] (optional):
// expected[n] = sum of the path products of the first n nodes added.
struct TreeGreedyArgs {
  const double* acc;
  int K, smax, N, fmax;
  int s[MEDUSA_MAX_HEADS];
  int32_t* parent;
  int32_t* rank;
  double* expected;
};
size_t tree_greedy_smem(int N, int smax);
cudaError_t launch_tree_greedy(const TreeGreedyArgs& a, cudaStream_t st);
// Fused per-row statistics + acceptance + KV compaction.  row_cnt [B*n1] and seq_cnt [B]
// zero on entry (left zero); parts: [B*n1][kVerifySlicesMax][6] float scratch.
constexpr int kVerifySlicesMax = 8;
cudaError_t launch_verify_commit(const VerifyArgs& v, const CompactArgs& c, int32_t* row_cnt,
                                 int32_t* seq_cnt, float* parts, cudaStream_t st);

// Decode loop: ring_tok[c % max_steps] = tok ([B][W]), ring_nacc[c % max_steps] = n_acc,
// then *count = c + 1, where c = *count (one CTA).
cudaError_t launch_loop_append(const int32_t* tok, const int32_t* n_acc, int B, int W, int max_steps,
                               long long* count, int32_t* ring_tok, int32_t* ring_nacc,
                               cudaStream_t st);

// Plan fields used by the workspace-free heads entry point (defined in capi.cu).
struct HeadsPlanView {
  medusa_dims dims;
  int K;
  bool tc_heads;
  int topk_splits, topk_chunk;
  uint32_t* status;
};
bool heads_plan_view(const medusa_plan* p, HeadsPlanView* v);

}  // namespace medusa
