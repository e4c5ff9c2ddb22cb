// Internal declarations shared by the translation units of libdg.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dg.h"

namespace dg {

// Tuning constant: CTAs the split-K / split-KV grids aim for (one wave on the
// 152 SMs of a GB300).  Kernels are correct for any SM count.
constexpr int kTargetCtas = 152;
constexpr int kLmBN = 256;     // vocabulary columns per LM-head tile
constexpr int kStatCols = 128; // vocabulary columns per softmax-statistics group
constexpr int kScBN = 256;     // model columns per self-conditioning tile
constexpr int kAttnRows = 64;  // query rows per attention CTA
constexpr int kAttnKeys = 64;  // keys per attention block
constexpr int kMaxAttnSplits = 64;

inline int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split of the key sequence [prefix ; canvas] of length T (prefix P) into
// chunks for the attention grid; returns the number of splits and the keys per
// split.  Head dim 128 with P a multiple of 128 takes the tensor-core kernel,
// other shapes the warp-MMA kernel; attn_max_splits bounds both for any P <= cap.
bool attn_use_tc(const dg_dims& D, int P);
void attn_split(const dg_dims& D, int T, int P, int* nsplit, int* keys_per_split);
int attn_max_splits(const dg_dims& D, int T);

// Byte offsets of every buffer in the caller's workspace.
struct WsLayout {
  size_t status, stop_at, rope;
  size_t a, q, kc, vc, o, h;
  size_t attn_o, attn_ml;
  size_t pt;
  size_t gst;  // per (row, 128-column group) statistics records
  size_t Hd, lsum, rowmax, amax, acc;
  size_t upart, gbest, gidx;
  size_t gpart, gpart_elems;  // split-K partials of the small GEMMs
  size_t u, g;
  size_t h8, hscale;          // FP8 head: h quantized per row
  size_t ref2, ref2f, rkey;   // tile storage reference per row
  // MoE FFN (n_exp > 0): normalised input, routing, permutation, tile table,
  // gathered rows, expert hidden and gated outputs (R = rows * (top_k + 1))
  size_t moe_x, moe_idx, moe_gate, moe_slot, moe_ptok, moe_pgate, moe_tiles, moe_xp, moe_gp, moe_yp;
  size_t moe_rpart, moe_rpart_elems;  // router GEMM partials
  int moe_max_tiles;
  size_t total;
};
bool ws_layout(const dg_dims& D, int32_t cap, WsLayout* L);

constexpr int kProgrammaticLaunch = 1;

// Launch with programmatic stream serialisation: the launch may begin while
// the kernel before it in the stream is still retiring (each kernel opens
// with griddepcontrol.wait, so none reads its inputs early).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Opt a kernel in to more than 48 KB of dynamic shared memory, once per
// kernel (the value is fixed per kernel), so that enqueueing a step makes no
// attribute calls and can be captured into a CUDA graph.
template <auto Kernel>
cudaError_t set_smem_once(int bytes) {
  static cudaError_t result = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return result;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (bf16, or
// with u8 set 8-bit codes; 128-byte swizzle).
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool u8 = false);

// ------------------------------------------------------------- launchers --
struct StopCtl {
  const int* stop_at;  // int32 [B] or nullptr
  int B;
  int step;
};

// D fp32 [M][N] = A[M][K] B^T (diagnostics).
cudaError_t launch_debug_gemm(const void* A, const void* Bm, float* D, int M, int N, int K,
                              int b_mn_major, int* status, cudaStream_t st);
// out bf16 [M][N] (row pitch ldo) = act(A[M][K] W[N][K]^T (+ resid)); rows of
// stopped canvases (row / C) are left untouched when ctl.stop_at is set.
// Small GEMMs that would leave SMs idle are split over K into `part`
// (fp32, ksplit x M x N, at most part_elems) and reduced by a fused epilogue.
int gemm_ksplit(int M, int N, int K);
cudaError_t launch_gemm_bf16(const void* A, const void* W, void* out, int ldo, const void* resid,
                             int ldr, int gelu, int M, int N, int K, int C, StopCtl ctl,
                             int* status, float* part, size_t part_elems, cudaStream_t st);
// Projections of a [M][d]: q (RoPE) to [B][Hq][C][hd], k (RoPE) and v to
// [B][Hkv][kv_rows][hd] at row kv_row0 + i.  With Wq == nullptr only k, v.
cudaError_t launch_qkv(const void* a, const void* Wq, const void* Wk, const void* Wv, void* q,
                       void* k, void* v, int kv_rows, int kv_row0, const float2* rope,
                       const dg_dims& D, StopCtl ctl, int* status, float* part, size_t part_elems,
                       cudaStream_t st);
// Statistics of one (row, 128-column group) of the LM head, one 32-byte
// record (a whole sector, written by one 256-bit store): the group maximum m
// of the tempered logits and l = sum exp2(t - m), S = sum exp2(t - m) (t - m)
// (log2 units), the largest raw product vmax and its column idx.
struct GroupStat {
  float m, l, S, vmax;
  int idx, pad0, pad1, pad2;
};
static_assert(sizeof(GroupStat) == 32, "one sector per record");

// LM head with the statistics epilogue.
struct LmArgs {
  const void* h;       // bf16 [M][d]
  const void* E;       // bf16 [V][d]
  const float* alpha;  // [M]
  float coef2;         // log2(e) / (sqrt(d) tau)
  float inv_sqrt_d;
  void* pt;            // bf16 [M][V]  exp(s - m_tile)
  GroupStat* gst;      // [M][NT] statistics of each 128-column group
  float* logits;       // optional fp32 [M][V]
  int M, V, d;
  int excl;            // column left out of the softmax (masked decoding's [MASK]), or -1
  // FP8 head (all null for bf16): h8 [M][d] and E8 [V][d] E4M3 codes with
  // per-row scales hscale [M] and escale [V]; the product runs on
  // tcgen05 kind::f8f6f4 and the epilogue applies the scales
  const void *h8, *E8;
  const float *hscale, *escale;
  // Tile storage reference (see RefArgs): ref2 [M] in; rkey [M] raised (an
  // order-preserving key of the group's maximum) for every group stored
  // against its own maximum, so that a row with rkey != 0 is flagged and
  // rkey holds its maximum
  const float* ref2;
  unsigned* rkey;
};
cudaError_t launch_lmhead(const LmArgs& a, StopCtl ctl, int* status, cudaStream_t st);
// The stored tiles of a row are exp2(t - R) for a per-row reference R (log2
// units of the LM head's epilogue: the scaled logit of a reference token,
// alpha (h . E_ref) log2(e) / (sqrt(d) tau)), so the contraction reads them as
// they are and one per-row factor exp2(R - m) / Z makes p0 of the result.  The
// reference is the larger of the logits of the current token and (step >= 1
// with prev_argmax given) the previous step's argmax, never of the excluded
// column, so R <= m:
// values of a group far below R underflow only where p0 < 2^-64 relative to
// the row's largest.  A group whose maximum lies more than kRefSpan above R
// (its stored values would overflow) is stored against its own maximum and
// flags the row; right after the LM head, lm_fix rewrites a flagged row
// against the row's maximum R' (the largest such group maximum), which
// becomes the row's final reference ref2f.  From there on every row's tiles
// hold exp2(t - ref2f) and p0 = tile * exp2(ref2f - m) / Z.
constexpr float kRefSpan = 64.0f;
struct RefArgs {
  const void* h;               // bf16 [M][d]
  const void* E;               // bf16 [V][d]
  const float* alpha;          // [M]
  float coef2;                 // log2(e) / (sqrt(d) tau)
  const int32_t* tokens;       // [M]
  const int32_t* prev_argmax;  // [M] or null
  int step, M, d, V;
  int excl;                    // column left out of the softmax, or -1 (never the reference)
  float* ref2;                 // out [M]
  float* ref2f;                // out [M], = ref2 (lm_fix updates flagged rows)
  unsigned* rkey;              // out [M], cleared
};
cudaError_t launch_lm_ref(const RefArgs& a, StopCtl ctl, cudaStream_t st);
// Rewrite of the flagged rows' tiles against their maximum (see kRefSpan).
struct FixArgs {
  void* pt;                    // bf16 [M][V] tiles
  const GroupStat* gst;        // [M][NT] group statistics (the maxima m, log2 units)
  const float* ref2;           // [M] the LM head's reference
  const unsigned* rkey;        // [M] 0, or the key of the row's maximum
  float* ref2f;                // [M] final reference (flagged rows: their maximum)
  int M, V;
};
cudaError_t launch_lm_fix(const FixArgs& a, StopCtl ctl, cudaStream_t st);

// ------------------------------------------------------------ MoE FFN ----
// Router and top-k per row of x (bf16 [M][d]): fp32 logits x . Wr_e, the
// top_k experts (value descending, lower index on ties) and their gates
// (softmax over the selected logits).  idx, gate [M][top_k]; the optional
// debug copies also get the logits [M][n_exp].
struct MoeRouteArgs {
  const void* x;
  const void* Wr;  // bf16 [n_exp][d]
  int* idx;
  float* gate;
  int32_t* dbg_idx;
  float *dbg_gate, *dbg_logits;
  int M, d, n_exp, top_k;
};
// The router logits run as a K-split tcgen05 GEMM into fp32 partials `part`
// (room for part_elems floats), summed by the top-k kernel.
cudaError_t launch_moe_route(const MoeRouteArgs& a, float* part, size_t part_elems, int* status, StopCtl ctl,
                             cudaStream_t st);
// part [ks][M][N] = the K-split partial products of A [M][K] and W [N][K] (bf16).
cudaError_t launch_gemm_f32_partials(const void* A, const void* W, float* part, int M, int N, int K, int ks,
                                     StopCtl ctl, int* status, cudaStream_t st);
int gemm_ksplit(int M, int N, int K);
// Expert-sorted permutation of the M * (top_k + 1) assignments (the shared
// expert, index n_exp, takes every row with gate 1): per expert, rows in
// increasing row order.  ptok / pgate [R] (source row and gate of permuted
// row p), slot [M][top_k + 1] (permuted row of each assignment), and the
// M-tile table of the grouped GEMMs: tiles[0].x = count, then per tile
// (expert, first permuted row, rows) in tiles[1 + t].
struct MoePlanArgs {
  const int* idx;
  const float* gate;
  int* ptok;
  float* pgate;
  int* slot;
  int4* tiles;
  int M, n_exp, top_k, max_tiles;
};
cudaError_t launch_moe_plan(const MoePlanArgs& a, int* status, StopCtl ctl, cudaStream_t st);
// Shared memory of the plan kernel (bytes); bounds of its one-CTA design.
int moe_plan_smem(int M, int n_exp);
constexpr int kMoeMaxRows = 4096, kMoeMaxExperts = 256, kMoeMaxTopK = 16;
// Rows of an expert per tile of the grouped expert GEMMs (their N dimension).
constexpr int kMoeTileRows = 32;
// xp[p] = x[ptok[p]] for the R permuted rows (bf16, d columns; x has M rows).
cudaError_t launch_moe_gather(const void* x, const int* ptok, void* xp, int R, int d, int M, StopCtl ctl,
                              cudaStream_t st);
// Grouped expert GEMMs over the tile table: up: gp = GELU(xp We1_e^T) (bf16
// [R][Fe]); down: yp = pgate * (gp We2_e^T) (fp32 [R][d]).
// R: rows of xp / gp / yp; groups = n_exp + 1 stacked expert matrices.
cudaError_t launch_moe_experts(const void* xp, const void* We1, const void* We2, const int4* tiles,
                               int max_tiles, int R, int groups, const float* pgate, void* gp, float* yp, int d,
                               int Fe, int* status, StopCtl ctl, cudaStream_t st);
// h[r] = bf16(h[r] + sum_j yp[slot[r][j]]), j = 0..top_k (rank order, then
// the shared expert), on the rows of active canvases (C rows per canvas).
cudaError_t launch_moe_combine(void* h, const float* yp, const int* slot, int M, int d, int top_k, int C,
                               StopCtl ctl, cudaStream_t st);
// Self-conditioning contraction u = p0 . E (split over the vocabulary).
struct ScArgs {
  const void* pt;        // bf16 [M][V]: p0
  const void* E;         // bf16 [V][d]
  float* upart;          // [S][M][d]
  int M, V, d, nsplit;
};
cudaError_t launch_selfcond(const ScArgs& a, StopCtl ctl, int* status, cudaStream_t st);
// Vocabulary splits of the self-conditioning contraction: selfcond_splits is
// the bound the workspace is sized for, selfcond_active_splits what a launch
// on the current device uses (at most the bound).
int selfcond_splits(const dg_dims& D);
int selfcond_active_splits(const dg_dims& D);
// The Gumbel-max search of the accepted rows over the stored tiles, in
// vocabulary chunks of kGumbelChunk entries (one best (score, index) per row
// and chunk; the reduce takes the best of a row's chunks).
constexpr int kGumbelChunk = 4096;
struct P0Args {
  const void* pt;        // bf16 [M][V]: the tiles, exp2(t - ref2f)
  const GroupStat* gst;  // [M][NT]  group maxima m_g (log2 units)
  const float* rowmax;   // [M]  row maximum m (log2 units)
  const float* lsum;     // [M]  Z
  const uint8_t* acc;    // [M]
  const int* amax;       // [M]  argmax of the logits (lowest index on ties)
  float* gbest;          // [NC][M]
  int* gidx;             // [NC][M]
  int M, V, C;
  uint64_t seed;
  int block, step;
  const float* ref2f;    // [M] final storage reference of the tiles (log2 units)
};
cudaError_t launch_p0_gumbel(const P0Args& a, StopCtl ctl, cudaStream_t st);

// Attention over [prefix ; canvas].
struct AttnArgs {
  const void* q;            // bf16 [B][Hq][C][hd]
  const void *Kp, *Vp;      // bf16 [B][Hkv][cap][hd]
  const void *kc, *vc;      // bf16 [B][Hkv][C][hd]
  void* o;                  // bf16 [B*C][Hq*hd]
  float* opart;             // fp32 [S][B][Hq][C][hd]
  float* ml;                // fp32 [S][B][Hq][C][2]
  int B, C, Hq, Hkv, hd, P, cap;
  int causal;               // 1: canvas query i sees canvas keys 0..i only (prefill); takes the warp-MMA kernel
};
cudaError_t launch_attention(const AttnArgs& a, StopCtl ctl, int* status, cudaStream_t st);
cudaError_t launch_attention_tc(const AttnArgs& a, StopCtl ctl, int* status, cudaStream_t st);
cudaError_t launch_attention_combine(const AttnArgs& a, int nsplit, StopCtl ctl, cudaStream_t st);
void attn_split_tc(const dg_dims& D, int T, int* nsplit, int* keys_per_split);
void attn_split_mma(const dg_dims& D, int T, int* nsplit, int* keys_per_split);

// Misc kernels.
// A token outside [0, V) is embedded as token 0 and sets DG_ERR_VALUE in *status.
// src: optional bf16 [rows][d]; when given, a = RMSNorm(src) (a deeper
// layer's input) and tokens, E, z are not read.
cudaError_t launch_embed_rmsnorm(const int32_t* tokens, const void* E, const void* z, void* a,
                                 float2* rope, const dg_dims& D, int rows, int P, StopCtl ctl,
                                 int* status, cudaStream_t st, const void* src = nullptr);
struct StatsArgs {
  const GroupStat* gst;  // [M][NT]
  int NT, M;
  double* Hd;            // [M]
  float* lsum;           // [M]  Z
  float* rowmax;         // [M]  m (log2 units)
  int* amax;             // [M]
  float* entropy;        // optional out [M]
  int* argmax_out;       // optional out [M]
};
cudaError_t launch_stats(const StatsArgs& a, StopCtl ctl, cudaStream_t st);
struct SamplerArgs {
  const double* Hd;      // [B][C]
  const int* amax;       // [B][C]
  int* prev_argmax;      // [B][C]
  int* tokens;           // [B][C]
  uint8_t* acc;          // [B][C] (workspace copy)
  uint8_t* acc_out;      // optional
  int* n_acc;            // optional [B]
  float* mean_H;         // optional [B]
  int* stop;             // optional [B]
  int* stop_at;          // [B] (workspace)
  int* n_stopped;        // canvases whose stop test fired (workspace), or nullptr
  int B, C, V;
  float b, stop_H;
  uint64_t seed;
  int block, step;
  int* accepted_log;     // optional [B][N] for the loop
  int N;
};
cudaError_t launch_sampler(const SamplerArgs& a, cudaStream_t st);
// Per-row E4M3 quantization of a bf16 matrix [R][d]: scale = absmax / 448 and
// codes of x * (448 / absmax), float32 arithmetic, round to nearest even with
// saturation; zero rows get scale 0 and zero codes.
cudaError_t launch_quantize_rows_e4m3(const void* X, int R, int d, uint8_t* Q, float* scale, cudaStream_t st);
// Masked confidence decoding of one step: per canvas, the
// min(ceil(U / (N - step)), U) masked positions of smallest Z (highest
// confidence 1 / Z) take their argmax; the accept copy is cleared (no
// Gumbel-max sampling in this mode).
struct RevealArgs {
  const double* Hd;      // [B][C] (mean entropy output)
  const float* lsum;     // [B][C] Z
  const int* amax;       // [B][C]
  int* prev_argmax;      // [B][C]
  int* tokens;           // [B][C]
  uint8_t* acc;          // [B][C] workspace copy (cleared)
  uint8_t* acc_out;      // optional: 1 where revealed at this step
  int* n_acc;            // optional [B]: positions revealed
  float* mean_H;         // optional [B]
  int* stop;             // optional [B] (0)
  int* accepted_log;     // optional [B][N]
  int B, C, mask_id, step, N;
};
cudaError_t launch_reveal(const RevealArgs& a, cudaStream_t st);
cudaError_t launch_fill_tokens(int32_t* tokens, int n, int value, cudaStream_t st);

struct ReduceArgs {
  const float* upart;    // [S][M][d]
  const float* gbest;    // [NC][M]
  const int* gidx;       // [NC][M]
  const uint8_t* acc;
  void* u;               // bf16 [M][d]
  int* tokens;           // [M]
  int* status;           // DG_ERR_VALUE if an accepted row has no finite Gumbel score
  int M, d, C, V, nsplit, nchunks;
  // per-row factor of the contraction: exp2(ref2f - rowmax) / lsum
  const float *ref2f, *rowmax, *lsum;
};
cudaError_t launch_reduce(const ReduceArgs& a, StopCtl ctl, cudaStream_t st);
cudaError_t launch_wait_timeout(int* status, cudaStream_t st);
cudaError_t launch_canvas_init(int32_t* tokens, int B, int C, int V, uint64_t seed, int block,
                               cudaStream_t st);
cudaError_t launch_loop_finish(const int* stop_at, int B, int N, int* steps_taken, int* converged,
                               const int* prev_argmax, int* xhat0, int C, cudaStream_t st);

}  // namespace dg
