/*
 * dg.h -- C ABI of the GB300 block-diffusion denoising library (libdg.so).
 *
 * The library computes the hot path of a DiffusionGemma-style uniform-state
 * text diffusion decoder on one GPU: denoising steps over a C-token canvas that
 * reads a static prefix KV cache, the annealed loop of such steps, and the
 * commit of a finished block into the cache.
 *
 * Sources of the operations (page title, then section):
 *   [TR]   "DiffusionGemma Technical Report" summary page: "Method step
 *          details" (inference steps 1-5) and the reproduction paragraph that
 *          lists the sampler hyper-parameters of the report's Table 2.
 *   [EXP]  "DiffusionGemma explained" (Gemma docs): "Uniform State Diffusion",
 *          "Architecture: incremental prefill and denoising",
 *          "Self-conditioning", "Multi-canvas sampling".
 *   [CH12] "DiffusionGemma" chapter of the diffusion docs: the KV-cache timing
 *          list, the attention-mask list and the data-flow pseudocode.
 *   [P4]   "从零拆开DiffusionGemma" news piece: the masked confidence decoder
 *          generate() of its fourth step (the second sampler below).
 *   [SURV] "文本 Diffusion 模型" survey page: §11 (DiffusionGemma: 128
 *          experts per layer, 8 routed plus one shared; throughput quoted for
 *          FP8) and §13 (router top-k, expert GEMM, token permutation); with
 *          the [TR] results paragraph (FP8 on H100), the basis of the optional
 *          FP8 LM head and MoE FFN.
 * The model is a synthetic stand-in: RMSNorm of embedding plus
 * self-conditioning, L pre-norm GQA attention layers with RoPE, a tied LM head
 * with a per-position logit sharpness alpha, and a two-matrix FFW for
 * self-conditioning.
 *
 * Conventions for every entry point:
 *  - All tensors are caller-owned DEVICE buffers unless stated otherwise; the
 *    library never allocates device memory and keeps no per-model state.
 *  - bf16 tensors are IEEE bfloat16, row-major, densely packed.  Weight
 *    matrices are stored [out][in] (the row of W that produces output n is
 *    contiguous), so y = x W^T.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call only enqueues work on `stream` and returns; the exceptions are said.
 *    A denoising step also runs part of its work (statistics, sampler, Gumbel
 *    search) on a library-owned stream of the device, forked from `stream` by
 *    an event and joined back into it within the step, so the step's work is
 *    done when `stream`'s is; under stream capture the fork and join are
 *    captured too.  The library creates that stream and two events once per
 *    device, at the first step not under capture.
 *  - Arguments are validated before anything is enqueued: on any error code no
 *    device memory has been written.
 *  - The workspace `ws` (size from dg_workspace_size, 256-byte aligned) holds
 *    intermediates between calls of one step; its first 4 bytes are a device
 *    status word that kernels set to DG_ERR_TIMEOUT if a bounded wait inside a
 *    kernel ran out, or to DG_ERR_VALUE if a device-side value check failed
 *    (read it with dg_read_status); zero the workspace (or at
 *    least that word) before its first use.  Calls sharing one workspace must
 *    not overlap on the GPU.
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DG_API __attribute__((visibility("default")))
#else
#define DG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t dg_status;
enum {
  DG_OK = 0,
  DG_ERR_ARG = 1,        /* null pointer, non-positive size, inconsistent dims */
  DG_ERR_SHAPE = 2,      /* a size the kernels do not support (see dg_dims) */
  DG_ERR_CAPACITY = 3,   /* commit would write past the cache capacity */
  DG_ERR_WORKSPACE = 4,  /* workspace too small or misaligned */
  DG_ERR_CUDA = 5,       /* a CUDA runtime call or kernel launch failed */
  DG_ERR_TIMEOUT = 6,    /* a bounded device-side wait ran out (status word) */
  DG_ERR_VALUE = 7       /* a device-side value check failed (status word): a canvas
                            token outside [0, V) reached the embedding (embedded as
                            token 0), or an accepted row had no finite Gumbel score
                            (non-finite probabilities; the row kept its token) */
};

/* Model and canvas sizes.
 *   V    vocabulary size (multiple of 8)
 *   d    model width (multiple of 64, <= 16384)
 *   C    canvas length (1..1024); B canvases are processed together
 *   Hq   query heads, Hkv key/value heads (Hq % Hkv == 0, grouped-query)
 *   hd   head dim: 32, 64 or 128
 *   F    self-conditioning FFW hidden width (multiple of 64)
 *   rope_base  RoPE base (10000); rms_eps  RMSNorm epsilon (1e-6)
 *   L    attention layers (1..64).  The stand-in's layer l takes a_l (a_0 =
 *        RMSNorm(E[x] + z)), h_l = a_l + Attn_l(a_l) Wo_l^T, a_{l+1} =
 *        RMSNorm(h_l); the LM head reads h_{L-1}; layer l attends over its own
 *        prefix cache.  L = 1 is the single-layer model.
 *   n_exp, top_k, Fe  optional mixture-of-experts FFN after each attention
 *        block [SURV] (n_exp = 0: none): n_exp routed experts (1..256) of
 *        hidden width Fe (multiple of 128), top_k (1..min(16, n_exp)) of them
 *        per token, plus one shared expert of the same shape.  Layer l then
 *        takes h_l <- h_l + sum_j g_j FFN_{e_j}(x) + FFN_shared(x) with
 *        x = RMSNorm(h_l), router logits r = x Wr_l^T (fp32), e_j the top_k
 *        experts (value descending, lower index on ties), g = softmax of their
 *        logits, FFN_e(x) = We2_e GELU(We1_e x); a_{l+1} = RMSNorm(h_l).  Needs
 *        d a multiple of 128 and B*C <= 4096.                                  */
typedef struct dg_dims {
  int32_t V, d, C, B, Hq, Hkv, hd, F;
  float rope_base, rms_eps;
  int32_t L;
  int32_t n_exp, top_k, Fe;
} dg_dims;

/* Weights (device, bf16):
 *   E  [V][d]        tied token embedding and LM head
 *   Wq [L][Hq*hd][d], Wk [L][Hkv*hd][d], Wv [L][Hkv*hd][d], Wo [L][d][Hq*hd]
 *   (one matrix per layer, stacked)
 *   W1 [F][d], W2 [d][F]
 * Optional FP8 LM head [SURV] (both NULL = bf16 head):
 *   E8 [V][d] uint8  E4M3 codes of E, E8_scale [V] float32 its per-row scales
 *   (dg_quantize_rows_e4m3 of E; E8 and E8_scale 16-byte aligned, both or neither
 *   given, else DG_ERR_ARG).  Each step then quantizes h per row the same
 *   way and takes the logits l_v = alpha s_h s_v (q_h . q_v) / sqrt(d) on the
 *   E4M3 tensor cores (fp32 accumulation); the embedding lookup and the
 *   self-conditioning contraction p0 . E keep the bf16 E.
 * MoE FFN (n_exp > 0; bf16, stacked per layer; else ignored):
 *   Wr [L][n_exp][d] router; We1 [L][n_exp + 1][Fe][d], We2 [L][n_exp + 1][d][Fe]
 *   expert matrices, index n_exp being the shared expert.                    */
typedef struct dg_model {
  dg_dims dims;
  const void *E, *Wq, *Wk, *Wv, *Wo, *W1, *W2;
  const void* E8;
  const float* E8_scale;
  const void *Wr, *We1, *We2;
} dg_model;

/* Static prefix KV cache ([CH12] "prompt / finished output block -> causal
 * encoder prefill -> written to the KV cache"; [EXP] incremental prefill).
 * K, V: bf16 [L][B][Hkv][cap][hd] (one cache per layer); rows 0..len-1 of
 * every (layer, canvas, head) are valid, keys already rotated by RoPE at their
 * absolute positions.  `len` is a host value: every canvas of the batch has
 * the same prefix length.  dg_prefill writes it from a prompt.              */
typedef struct dg_kv_cache {
  void *K, *V;
  int32_t cap;
  int32_t len;
} dg_kv_cache;

/* Canvas state of B canvases ([TR] steps 2-3):
 *   tokens       int32 [B][C]   x_t on entry, x_{t+1} on return
 *   z            bf16 [B][C][d] self-conditioning z_t on entry, z_{t+1} on return
 *   alpha        fp32 [B][C]    per-position logit sharpness (> 0)
 *   prev_argmax  int32 [B][C]   argmax of the previous step on entry (read only
 *                               when step >= 1), this step's argmax on return */
typedef struct dg_canvas {
  int32_t* tokens;
  void* z;
  const float* alpha;
  int32_t* prev_argmax;
} dg_canvas;

/* Optional copies of the intermediates of one step, for checking (every
 * pointer may be NULL).  Device buffers:
 *   a, h [B*C][d]; q [B][Hq][C][hd]; k, v [B][Hkv][C][hd]; o [B*C][Hq*hd];
 *   u [B*C][d]; g [B*C][F]  (bf16)      logits fp32 [B*C][V] (l = alpha h.E / sqrt d)
 *   MoE routing of the last layer (n_exp > 0): moe_idx int32 [B*C][top_k]
 *   (experts in rank order), moe_gate fp32 [B*C][top_k], moe_logits fp32
 *   [B*C][n_exp] (router logits), moe_x bf16 [B*C][d] (the router's input
 *   RMSNorm(h)).  h is the last layer's output (after its MoE block when there
 *   is one).                                                                 */
typedef struct dg_step_debug {
  void *a, *q, *k, *v, *o, *h, *u, *g;
  float* logits;
  int32_t* moe_idx;
  float *moe_gate, *moe_logits;
  void* moe_x;
} dg_step_debug;

/* Kernel slots of a step, in launch order, for dg_step_out.events. */
enum {
  DG_PROF_EMBED = 0,     /* embedding + self-conditioning + RMSNorm   */
  DG_PROF_QKV = 1,       /* q, k, v projections with RoPE             */
  DG_PROF_ATTN = 2,      /* attention over prefix + canvas (+ merge)  */
  DG_PROF_OPROJ = 3,     /* output projection + residual              */
  DG_PROF_LMHEAD = 4,    /* LM head + statistics (FP8: + h's codes)   */
  DG_PROF_STATS = 5,     /* merge of the statistics: entropy, argmax  */
  DG_PROF_SAMPLER = 6,   /* sort, cumulative entropy, accept, renoise */
  DG_PROF_P0 = 7,        /* Gumbel-max search of the accepted rows    */
  DG_PROF_SELFCOND = 8,  /* p0 . E on the tensor cores                */
  DG_PROF_REDUCE = 9,    /* reduction of p0 . E, sampled tokens        */
  DG_PROF_FFW1 = 10,     /* GELU(W1 u)                                */
  DG_PROF_FFW2 = 11,     /* z = W2 g                                  */
  DG_PROF_MOE = 12,      /* MoE FFN of the first layer (n_exp > 0)    */
  DG_PROF_NUM = 13
};

/* Per-step outputs (device; any pointer may be NULL except where noted):
 *   entropy  fp32 [B][C]  entropy of softmax(l / tau) in nats
 *   argmax   int32 [B][C] argmax_v l (lowest index on ties)
 *   accept   uint8 [B][C] 1 where the position was accepted
 *   n_acc    int32 [B]    accepted positions per canvas
 *   mean_H   fp32 [B]     mean entropy of the canvas
 *   stop     int32 [B]    1 when the adaptive stop test fired at this step
 *   debug    host pointer to a dg_step_debug, or NULL
 *   events   host array of 2 * DG_PROF_NUM cudaEvent_t (caller-created), or
 *            NULL: events[2k] / events[2k+1] are recorded on `stream` just
 *            before / after the kernels of slot k (for per-kernel timing);
 *            NULL entries are skipped.  Records are external, so a step
 *            captured into a CUDA graph records them at every replay.       */
typedef struct dg_step_out {
  float* entropy;
  int32_t* argmax;
  uint8_t* accept;
  int32_t* n_acc;
  float* mean_H;
  int32_t* stop;
  const dg_step_debug* debug;
  void* const* events;
} dg_step_out;

/* Sampler schedule ([TR] step 3 and Table 2): tau_s = tau0 + (tau1 - tau0) *
 * s / (N - 1) for s = 0..N-1; entropy budget b; stop when the mean entropy of
 * the canvas is <= stop_H and the argmax equals the previous step's.  Defaults
 * 0.8, 0.4, 48, 0.1, 0.005.                                                 */
typedef struct dg_sched {
  float tau0, tau1;
  int32_t N;
  float b, stop_H;
} dg_sched;

/* Temperature of step `step` (0 <= step < N) of the schedule: tau0 + (tau1 -
 * tau0) * step / (N - 1), evaluated in double and rounded to float (tau0 when
 * N == 1).  dg_denoise_canvas uses exactly this value at each step; callers
 * that run the loop step by step take theirs from here.  DG_ERR_ARG for a
 * null pointer, N <= 0, a step outside [0, N) or a non-positive tau.       */
DG_API dg_status dg_tau(const dg_sched* sched, int32_t step, float* tau);

/* Result of the denoising loop (device buffers):
 *   steps_taken int32 [B]; converged int32 [B] (1 = stopped early);
 *   accepted int32 [B][N] (accepted count per step, -1 after the canvas stopped);
 *   xhat0 int32 [B][C] (argmax of the canvas's last step: the block to commit) */
typedef struct dg_canvas_result {
  int32_t* steps_taken;
  int32_t* converged;
  int32_t* accepted;
  int32_t* xhat0;
} dg_canvas_result;

/* Human-readable name of a status code (static string). */
DG_API const char* dg_status_string(dg_status s);

/* Bytes of workspace needed for `dims` with a prefix cache of up to `cap`
 * rows.  Returns DG_ERR_ARG / DG_ERR_SHAPE for unsupported dims.             */
DG_API dg_status dg_workspace_size(const dg_dims* dims, int32_t cap, size_t* bytes);

/* Copies the device status word of `ws` to *status (synchronises `stream`). */
DG_API dg_status dg_read_status(const void* ws, int32_t* status, void* stream);

/* Initial canvas, [TR] step 2: tokens[b][i] uniform over [0, V) from the
 * Philox stream of (seed, block, canvas b, position i); also the uniform
 * token law used for renoising ([EXP] "Uniform State Diffusion").           */
DG_API dg_status dg_canvas_init(int32_t* tokens, int32_t B, int32_t C, int32_t V, uint64_t seed,
                         int32_t block, void* stream);

/* One denoising step over B canvases, [TR] step 3 (with the stop test of
 * step 4):
 *   a = RMSNorm(E[x_t] + z_t); q, k = RoPE(a Wq^T, a Wk^T) at positions
 *   len + i, v = a Wv^T; o = softmax(q [K_pre ; k]^T / sqrt hd) [V_pre ; v]
 *   (no mask: canvas queries see every canvas key and the whole prefix);
 *   h = a + o Wo^T; l = alpha h E^T / sqrt d; p0 = softmax(l / tau);
 *   positions sorted by ascending entropy are accepted while the cumulative
 *   entropy stays <= b; accepted positions take the Gumbel-max sample of
 *   l / tau, all others a uniform random token; z_{t+1} = W2 GELU(W1 (p0 E)).
 * Random draws are Philox4x64-10 keyed by (seed, block, step, canvas,
 * position).  The cache is read only.  Canvas state is updated in place.    */
DG_API dg_status dg_denoise_step(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas,
                          float tau, float b, uint64_t seed, int32_t step, int32_t block,
                          void* ws, size_t ws_bytes, dg_step_out* out, void* stream);

/* The annealed denoising loop of one block, [TR] steps 3-4: up to sched->N
 * steps with the linear temperature schedule (dg_tau); each canvas stops on
 * its own when its stop test fires and is left unchanged afterwards.
 * Stopping: when `stream` is not being captured into a CUDA graph, the call
 * reads a 4-byte count of stopped canvases from the workspace after step 1
 * (the first step at which the stop test can fire) and every 4 steps after,
 * synchronising `stream` for each read, and enqueues no further step once
 * every canvas has stopped.  Under stream capture it enqueues all N steps
 * without synchronising; their kernels return at once after every canvas
 * stopped.  canvas->tokens/z must hold the initial canvas (dg_canvas_init,
 * z = 0).                                                                  */
DG_API dg_status dg_denoise_canvas(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas,
                            const dg_sched* sched, uint64_t seed, int32_t block, void* ws,
                            size_t ws_bytes, dg_canvas_result* result, void* stream);

/* Causal prefill, [TR] step 1 and [EXP] "Architecture: incremental prefill
 * and denoising": tokens int32 [B][n] (n >= 1, any length) are appended to
 * every layer's cache at rows len..len+n-1, then cache->len += n.  The
 * encoder is the denoiser's attention stack with no self-conditioning (a_0 =
 * RMSNorm(E[x])) and a causal mask: token i attends to every cached row and to
 * the new tokens 0..i.  Per layer, k and v (RoPE at positions len + i) are
 * written to the layer's cache; below the last layer q attends (causally)
 * and h_l = a_l + o_l Wo_l^T, a_{l+1} = RMSNorm(h_l).  Tokens are processed in
 * pieces of at most C per canvas, each attending over all earlier rows, which
 * gives the same cache as one pass.  DG_ERR_CAPACITY (nothing written) if
 * len + n > cap.                                                            */
DG_API dg_status dg_prefill(const dg_model* model, dg_kv_cache* cache, const int32_t* tokens, int32_t n,
                            void* ws, size_t ws_bytes, void* stream);

/* Commit of a finished block, [TR] step 5 and [CH12] KV-cache timing (the
 * cache comes from re-encoding the finished block, not from the denoiser's
 * states): dg_prefill of the block's tokens int32 [B][C].  With one layer the
 * appended K/V depend only on each token and its position; with more, the
 * deeper layers' K/V depend on the causal attention over earlier tokens.
 * DG_ERR_CAPACITY (nothing written) if len + C > cap.                       */
DG_API dg_status dg_commit_block(const dg_model* model, dg_kv_cache* cache, const int32_t* tokens,
                          void* ws, size_t ws_bytes, void* stream);

/* Masked confidence decoding, the second sampler of the pages ([P4] the
 * "从零拆开DiffusionGemma" news piece, generate() of its fourth step, given
 * there as the masked-diffusion contrast to the uniform-state sampler):
 *
 * dg_canvas_init_masked: tokens int32 [B][C] all set to mask_id ([MASK]).
 *
 * dg_denoise_step_masked: one step of the same denoiser (a, q, k, v, o, h,
 * l = alpha h E^T / sqrt d, self-conditioning z_{t+1} = W2 GELU(W1 (p0 E)))
 * with the [MASK] token left out of the tempered softmax p0 = softmax(l / tau)
 * (it is not a prediction target: its logit counts as -inf).  Per canvas, of
 * the U positions still holding mask_id, the k = min(ceil(U / (N - step)), U)
 * with the highest confidence max_v p0_v = 1 / Z (ties to the lower
 * position) take their candidate argmax_v l_v; every other position keeps its
 * token, so revealed positions never change and step N - 1 reveals all that
 * remain.  Outputs as in dg_denoise_step: accept = revealed at this step,
 * n_acc = k, stop = 0.  mask_id in [0, V); 0 <= step < N.  The cache is read
 * only; no random draws.
 *
 * dg_denoise_canvas_masked: N = sched->N such steps at the fixed temperature
 * tau0 (the pages' generate() keeps one temperature; tau1, b and stop_H are
 * not used), enqueued without synchronising.  result: steps_taken = N,
 * converged = 0 (no adaptive stop in this mode), accepted[b][s] = positions
 * revealed at step s, xhat0 = the final canvas (every position revealed). */
DG_API dg_status dg_canvas_init_masked(int32_t* tokens, int32_t B, int32_t C, int32_t mask_id, void* stream);
DG_API dg_status dg_denoise_step_masked(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas,
                                        float tau, int32_t mask_id, int32_t step, int32_t N, void* ws,
                                        size_t ws_bytes, dg_step_out* out, void* stream);
DG_API dg_status dg_denoise_canvas_masked(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas,
                                          const dg_sched* sched, int32_t mask_id, void* ws, size_t ws_bytes,
                                          dg_canvas_result* result, void* stream);

/* Attention of the denoising step (the bidirectional attention inside
 * dg_denoise_step) for callers that cannot allocate device memory, e.g. a
 * process whose device memory is fully pre-reserved by another framework's
 * caching allocator, or embedding code that is only handed fixed buffers.
 * The pages describe no such entry point; it has no counterpart there.
 *   q  bf16 [B][Hq][C][hd] (RoPE applied); K, V bf16 [B][Hkv][cap][hd] prefix
 *   cache with rows 0..len-1 valid; k, v bf16 [B][Hkv][C][hd] canvas keys and
 *   values; o bf16 [B*C][Hq*hd] output (caller-owned).
 * Its scratch is a 16 MiB static device array inside the library (held on
 * every GPU that loads it until exit), so no workspace is passed and nothing
 * is allocated.  DG_ERR_WORKSPACE (nothing launched) if the scratch this size
 * needs exceeds 16 MiB, e.g. 2 canvases of 8 heads over 8190 prefix keys (a
 * prefix that is not a multiple of 128 takes the warp-MMA kernel, which splits
 * the keys more finely).  DG_ERR_SHAPE (nothing launched) for sizes the step
 * rejects as well: C > 1024, B*C > 2^20, B*Hq > 65535, len + C > 2^30.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and should come before any stream capture.  All
 * calls share the array: calls that overlap on the GPU race.
 * Failure of a bounded device wait: the array holds a status word that each
 * call clears on `stream` before its kernels run; a wait that runs out sets it
 * to DG_ERR_TIMEOUT and leaves `o` unwritten.  The call itself only enqueues
 * work, so it returns DG_OK in that case: read the word with
 * dg_attention_noalloc_status after the call.                              */
DG_API dg_status dg_attention_noalloc(const void* q, const void* K, const void* V, int32_t cap,
                                      int32_t len, const void* k, const void* v, void* o, int32_t B,
                                      int32_t C, int32_t Hq, int32_t Hkv, int32_t hd, void* stream);

/* Per-row E4M3 quantization [SURV] (the FP8 LM head's operands).
 *   X      bf16 [R][d] device, d a multiple of 16
 *   Q      uint8 [R][d] device (written): codes of x * (448 / absmax(row))
 *          rounded to nearest even with saturation at 448
 *   scale  float32 [R] device (written): absmax(row) / 448; x ~= code * scale.
 * Both quotients and the product are IEEE float32.  A zero row gets scale 0
 * and zero codes.  R = 0 is a no-op.  Returns DG_ERR_ARG for NULL pointers,
 * R < 0 or X / Q not 16-byte aligned, DG_ERR_SHAPE for d not a positive
 * multiple of 16.                                                            */
DG_API dg_status dg_quantize_rows_e4m3(const void* X, int32_t R, int32_t d, void* Q, float* scale,
                                       void* stream);

/* Status word of the last dg_attention_noalloc call on the current device:
 * synchronises `stream` and copies the word to *status (DG_OK, or
 * DG_ERR_TIMEOUT if a bounded wait of that call ran out).  Allocates nothing.  */
DG_API dg_status dg_attention_noalloc_status(int32_t* status, void* stream);

/* Diagnostics of the bounded device waits (not a step of the method): runs
 * one kernel whose mbarrier wait is never satisfied.  The wait gives up after
 * its limit (2 s), records DG_ERR_TIMEOUT in a library status word, and the
 * kernel returns; *status receives that word (synchronises `stream`), so a
 * caller sees DG_ERR_TIMEOUT and the context stays usable.  The tests use it
 * to check that path without a device fault.                                  */
DG_API dg_status dg_debug_wait_timeout(int32_t* status, void* stream);

/* Diagnostics of the tensor-core GEMM engine, used by the tests to check it
 * in isolation (not a step of the method).  D fp32 [M][N] = A B^T with
 * A bf16 [M][K], and B bf16 [N][K] when b_mn_major == 0, or B bf16 [K][N]
 * when b_mn_major == 1 (the layout of E in the self-conditioning contraction).
 * b_mn_major == 3 / 4 run the same products (B [N][K] / B [K][N]) on the
 * CTA-pair engine (M = 256 MMAs over two SMs) that the LM head and the
 * self-conditioning contraction use.  b_mn_major == 5 / 6 / 7 / 8 run
 * B [N][K] on the cluster split-K engine of the small projections (the K
 * slices of a tile summed in shared memory across the cluster): 128-column
 * tiles over 2 / 4 slices, 64-column tiles over 2 / 4 slices; K must then
 * hold at least one 64-wide block per slice (DG_ERR_SHAPE otherwise).
 * K, N multiples of 8.                                                        */
DG_API dg_status dg_debug_gemm(const void* A, const void* Bm, float* D, int32_t M, int32_t N, int32_t K,
                        int32_t b_mn_major, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
