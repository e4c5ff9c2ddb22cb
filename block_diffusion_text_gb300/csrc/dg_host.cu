// C-ABI entry points of libdg: argument validation, workspace layout and the
// ordered launch of the kernels of one denoising step, the annealed loop and
// the block commit.  Nothing here computes on the host.
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "dg_internal.h"

using namespace dg;

namespace {

// Status word used by the diagnostics entry point (module memory).
__device__ int g_debug_status;

bool dims_ok(const dg_dims* D) {
  if (!D) return false;
  if (D->V <= 0 || D->d <= 0 || D->C <= 0 || D->B <= 0 || D->Hq <= 0 || D->Hkv <= 0 || D->hd <= 0 ||
      D->F <= 0)
    return false;
  if (D->Hq % D->Hkv != 0) return false;
  if (!(D->rope_base > 0.f) || !(D->rms_eps >= 0.f)) return false;
  if (D->L < 1 || D->L > 64) return false;
  if (D->n_exp < 0 || D->n_exp > kMoeMaxExperts) return false;
  if (D->n_exp > 0 && (D->top_k < 1 || D->top_k > D->n_exp || D->top_k > kMoeMaxTopK || D->Fe <= 0)) return false;
  return true;
}

dg_status dims_supported(const dg_dims* D) {
  if (!dims_ok(D)) return DG_ERR_ARG;
  if (D->V % 8 != 0 || D->d % 64 != 0 || D->d > 16384 || D->F % 64 != 0) return DG_ERR_SHAPE;
  if (D->hd != 32 && D->hd != 64 && D->hd != 128) return DG_ERR_SHAPE;
  if (D->C > 1024) return DG_ERR_SHAPE;
  if ((int64_t)D->B * D->C > (1 << 20) || (int64_t)D->V > (1 << 30)) return DG_ERR_SHAPE;
  if (D->n_exp > 0 && (D->Fe % 128 != 0 || D->Fe > 16384 || D->d % 128 != 0 || (int64_t)D->B * D->C > kMoeMaxRows))
    return DG_ERR_SHAPE;
  return DG_OK;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(ws) + off);
}

dg_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DG_OK : DG_ERR_CUDA; }

#define DG_TRY(expr)                         \
  do {                                       \
    cudaError_t _e = (expr);                 \
    if (_e != cudaSuccess) return DG_ERR_CUDA; \
  } while (0)

struct StepCtx {
  const dg_model* model;
  const dg_kv_cache* cache;
  dg_canvas* canvas;
  void* ws;
  WsLayout L;
  cudaStream_t st;
};

dg_status check_model(const dg_model* m) {
  if (!m) return DG_ERR_ARG;
  dg_status s = dims_supported(&m->dims);
  if (s) return s;
  if (!m->E || !m->Wq || !m->Wk || !m->Wv || !m->Wo || !m->W1 || !m->W2) return DG_ERR_ARG;
  if (!m->E8 != !m->E8_scale) return DG_ERR_ARG;  // the FP8 head needs codes and scales
  if (reinterpret_cast<uintptr_t>(m->E8) % 16 != 0 || reinterpret_cast<uintptr_t>(m->E8_scale) % 16 != 0)
    return DG_ERR_ARG;  // TMA base; vector loads of the scales
  if (m->dims.n_exp > 0 && (!m->Wr || !m->We1 || !m->We2)) return DG_ERR_ARG;
  return DG_OK;
}

dg_status check_ws(const dg_dims& D, int32_t cap, void* ws, size_t ws_bytes, WsLayout* L) {
  if (!ws) return DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return DG_ERR_WORKSPACE;
  if (!ws_layout(D, cap, L)) return DG_ERR_SHAPE;
  if (ws_bytes < L->total) return DG_ERR_WORKSPACE;
  return DG_OK;
}

// Layer l of a stacked [L][n] bf16 weight, and a byte offset into a buffer.
const void* layer_ptr(const void* w, int l, size_t n) {
  return reinterpret_cast<const uint8_t*>(w) + (size_t)l * n * 2;
}
void* byte_ptr(void* p, size_t off) { return reinterpret_cast<uint8_t*>(p) + off; }

struct Prof {
  void* const* ev;
  cudaStream_t st;
  // Inside a stream capture an external record, which becomes an event-record
  // node of the graph (timing each replay); outside a capture a plain record
  // (the external flag is only accepted under capture).
  cudaError_t mark(int slot, int end) const {
    if (!ev || !ev[2 * slot + end]) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    const cudaEvent_t evt = reinterpret_cast<cudaEvent_t>(ev[2 * slot + end]);
    return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(evt, st, cudaEventRecordExternal)
                                               : cudaEventRecord(evt, st);
  }
};

// The MoE block of layer l on the rows h [rows][d] (in place): RMSNorm,
// router and top-k, plan, gather, the two grouped expert GEMMs, combine.
// dbg (optional) receives the routing of this layer.
dg_status enqueue_moe(const dg_model* m, int l, void* ws, const WsLayout& L, int rows, int C, StopCtl ctl,
                      int* status, const dg_step_debug* dbg, cudaStream_t st) {
  const dg_dims& D = m->dims;
  const int NE = D.n_exp, K = D.top_k, R = rows * (K + 1);
  DG_TRY(launch_embed_rmsnorm(nullptr, nullptr, nullptr, at<void>(ws, L.moe_x), nullptr, D, rows, 0, ctl, status, st,
                              at<void>(ws, L.h)));
  MoeRouteArgs ra{at<void>(ws, L.moe_x), layer_ptr(m->Wr, l, (size_t)NE * D.d), at<int>(ws, L.moe_idx),
                  at<float>(ws, L.moe_gate), dbg ? dbg->moe_idx : nullptr, dbg ? dbg->moe_gate : nullptr,
                  dbg ? dbg->moe_logits : nullptr, rows, D.d, NE, K};
  DG_TRY(launch_moe_route(ra, at<float>(ws, L.moe_rpart), L.moe_rpart_elems, status, ctl, st));
  const int max_tiles = cdiv(R, kMoeTileRows) + NE + 1;
  MoePlanArgs pa{at<int>(ws, L.moe_idx), at<float>(ws, L.moe_gate), at<int>(ws, L.moe_ptok),
                 at<float>(ws, L.moe_pgate), at<int>(ws, L.moe_slot), at<int4>(ws, L.moe_tiles), rows, NE, K,
                 max_tiles};
  DG_TRY(launch_moe_plan(pa, status, ctl, st));
  DG_TRY(launch_moe_gather(at<void>(ws, L.moe_x), at<int>(ws, L.moe_ptok), at<void>(ws, L.moe_xp), R, D.d, rows,
                           ctl, st));
  const size_t e1 = (size_t)(NE + 1) * D.Fe * D.d;  // elements of one layer's We1 (and We2)
  DG_TRY(launch_moe_experts(at<void>(ws, L.moe_xp), layer_ptr(m->We1, l, e1), layer_ptr(m->We2, l, e1),
                            at<int4>(ws, L.moe_tiles), max_tiles, R, NE + 1, at<float>(ws, L.moe_pgate),
                            at<void>(ws, L.moe_gp), at<float>(ws, L.moe_yp), D.d, D.Fe, status, ctl, st));
  DG_TRY(launch_moe_combine(at<void>(ws, L.h), at<float>(ws, L.moe_yp), at<int>(ws, L.moe_slot), rows, D.d, K, C,
                            ctl, st));
  return DG_OK;
}

// A second stream per device for the work of a step that may overlap the
// self-conditioning contraction (statistics, sampler, Gumbel search): forked
// from and joined back into the caller's stream with two events, so a step
// stays one unit of work on the caller's stream (and one fork/join in a
// captured graph).  Created once, outside stream capture; the mutex keeps the
// record/wait pairs of concurrent callers apart.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;       // held from a step's fork record to its join wait
std::mutex g_side_make_mu;  // creation of the side streams
SideStream g_side[64];

// The device's side stream, or null (no overlap) when it cannot be created
// now: the first call on a device made under stream capture.
SideStream* side_stream(cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& sd = g_side[dev];
  std::lock_guard<std::mutex> lock(g_side_make_mu);
  if (sd.s) return &sd;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
  if (cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) != cudaSuccess) {
    sd.s = nullptr;
    return nullptr;
  }
  if (cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaStreamDestroy(sd.s);
    sd.s = nullptr;
    return nullptr;
  }
  return &sd;
}

// All kernels of one denoising step, in order, on ctx.st.
// fill_rope: (re)compute the RoPE table of positions P + i; a canvas loop
// fills it at its first step only (P is fixed for the loop).
// mask_id >= 0 selects masked confidence decoding (the [MASK] token left out
// of the softmax, the reveal kernel in place of the sampler); -1 the
// uniform-state sampler.
dg_status enqueue_step(const StepCtx& c, float tau, float b, float stop_H, uint64_t seed, int step,
                       int block, const dg_step_out* out, int* accepted_log, int N, bool fill_rope,
                       int mask_id = -1) {
  const dg_dims& D = c.model->dims;
  const WsLayout& L = c.L;
  void* ws = c.ws;
  const int M = D.B * D.C, NT = cdiv(D.V, kStatCols), P = c.cache->len;
  int* status = at<int>(ws, L.status);
  int* stop_at = at<int>(ws, L.stop_at);
  StopCtl ctl{stop_at, D.B, step};
  float2* rope = at<float2>(ws, L.rope);
  const Prof pf{out ? out->events : nullptr, c.st};

  DG_TRY(pf.mark(DG_PROF_EMBED, 0));
  DG_TRY(launch_embed_rmsnorm(c.canvas->tokens, c.model->E, c.canvas->z, at<void>(ws, L.a),
                              fill_rope ? rope : nullptr, D, M,
                              P, ctl, status, c.st));
  DG_TRY(pf.mark(DG_PROF_EMBED, 1));
  // a2-a4 per layer; the profiling slots time the first layer's kernels (a
  // deeper layer's RMSNorm of h goes with its projections)
  const size_t nq = (size_t)D.Hq * D.hd, nkv = (size_t)D.Hkv * D.hd, dd = D.d;
  const size_t cache_layer = (size_t)D.B * D.Hkv * c.cache->cap * D.hd * 2;
  for (int l = 0; l < D.L; ++l) {
    const Prof pl{l == 0 ? pf.ev : nullptr, c.st};
    if (l > 0)
      DG_TRY(launch_embed_rmsnorm(nullptr, nullptr, nullptr, at<void>(ws, L.a), nullptr, D, M, P, ctl, status,
                                  c.st, at<void>(ws, L.h)));
    DG_TRY(pl.mark(DG_PROF_QKV, 0));
    DG_TRY(launch_qkv(at<void>(ws, L.a), layer_ptr(c.model->Wq, l, nq * dd), layer_ptr(c.model->Wk, l, nkv * dd),
                      layer_ptr(c.model->Wv, l, nkv * dd), at<void>(ws, L.q), at<void>(ws, L.kc),
                      at<void>(ws, L.vc), D.C, 0, rope, D, ctl, status, at<float>(ws, L.gpart), L.gpart_elems,
                      c.st));
    DG_TRY(pl.mark(DG_PROF_QKV, 1));
    AttnArgs aa{at<void>(ws, L.q), byte_ptr(c.cache->K, l * cache_layer), byte_ptr(c.cache->V, l * cache_layer),
                at<void>(ws, L.kc), at<void>(ws, L.vc), at<void>(ws, L.o), at<float>(ws, L.attn_o),
                at<float>(ws, L.attn_ml), D.B, D.C, D.Hq, D.Hkv, D.hd, P, c.cache->cap, 0};
    DG_TRY(pl.mark(DG_PROF_ATTN, 0));
    DG_TRY(launch_attention(aa, ctl, status, c.st));
    DG_TRY(pl.mark(DG_PROF_ATTN, 1));
    DG_TRY(pl.mark(DG_PROF_OPROJ, 0));
    DG_TRY(launch_gemm_bf16(at<void>(ws, L.o), layer_ptr(c.model->Wo, l, dd * nq), at<void>(ws, L.h), D.d,
                            at<void>(ws, L.a), D.d, 0, M, D.d, D.Hq * D.hd, D.C, ctl, status,
                            at<float>(ws, L.gpart), L.gpart_elems, c.st));
    DG_TRY(pl.mark(DG_PROF_OPROJ, 1));
    if (D.n_exp > 0) {
      DG_TRY(pl.mark(DG_PROF_MOE, 0));
      dg_status ms = enqueue_moe(c.model, l, ws, L, M, D.C, ctl, status,
                                 (out && out->debug && l == D.L - 1) ? out->debug : nullptr, c.st);
      if (ms) return ms;
      DG_TRY(pl.mark(DG_PROF_MOE, 1));
    }
  }
  LmArgs lm{};
  lm.h = at<void>(ws, L.h);
  lm.E = c.model->E;
  lm.alpha = c.canvas->alpha;
  lm.coef2 = (float)(1.4426950408889634 / (std::sqrt((double)D.d) * (double)tau));
  lm.inv_sqrt_d = (float)(1.0 / std::sqrt((double)D.d));
  lm.pt = at<void>(ws, L.pt);
  lm.gst = at<GroupStat>(ws, L.gst);
  lm.logits = (out && out->debug) ? out->debug->logits : nullptr;
  lm.M = M;
  lm.V = D.V;
  lm.d = D.d;
  lm.excl = mask_id;
  lm.ref2 = at<float>(ws, L.ref2);
  lm.rkey = at<unsigned>(ws, L.rkey);
  float* ref2f = at<float>(ws, L.ref2f);
  RefArgs rf{lm.h, c.model->E, c.canvas->alpha, lm.coef2, c.canvas->tokens, c.canvas->prev_argmax, step, M, D.d,
             D.V, mask_id, at<float>(ws, L.ref2), ref2f, lm.rkey};
  DG_TRY(launch_lm_ref(rf, ctl, c.st));
  // the LM head slot: the product with its statistics (and, for the FP8
  // head, the quantization of h it needs), without the reference and fix
  DG_TRY(pf.mark(DG_PROF_LMHEAD, 0));
  if (c.model->E8) {
    lm.h8 = at<void>(ws, L.h8);
    lm.hscale = at<float>(ws, L.hscale);
    lm.E8 = c.model->E8;
    lm.escale = c.model->E8_scale;
    DG_TRY(launch_quantize_rows_e4m3(lm.h, M, D.d, at<uint8_t>(ws, L.h8), at<float>(ws, L.hscale), c.st));
  }
  DG_TRY(launch_lmhead(lm, ctl, status, c.st));
  DG_TRY(pf.mark(DG_PROF_LMHEAD, 1));
  FixArgs fx{at<void>(ws, L.pt), lm.gst, lm.ref2, lm.rkey, ref2f, M, D.V};
  DG_TRY(launch_lm_fix(fx, ctl, c.st));
  // fork: statistics, sampler and Gumbel search on the side stream, the
  // contraction (which reads only the tiles) on the caller's stream
  SideStream* sd = side_stream(c.st);
  std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
  // Joins the side stream back into the caller's stream on every way out of
  // this function once the fork is recorded, an error return included, so
  // that no side-stream kernel still reads the workspace after the caller's
  // stream has passed the step.  Declared after the lock: it runs first.
  struct JoinGuard {
    SideStream* sd = nullptr;
    cudaStream_t st = nullptr;
    cudaError_t join() {
      if (!sd) return cudaSuccess;
      SideStream* s = sd;
      sd = nullptr;
      const cudaError_t e = cudaEventRecord(s->join, s->s);
      const cudaError_t w = cudaStreamWaitEvent(st, s->join, 0);
      return e != cudaSuccess ? e : w;
    }
    ~JoinGuard() { join(); }
  } side_join;
  cudaStream_t sst = c.st;
  if (sd) {
    side_lock.lock();
    DG_TRY(cudaEventRecord(sd->fork, c.st));
    side_join.sd = sd;
    side_join.st = c.st;
    DG_TRY(cudaStreamWaitEvent(sd->s, sd->fork, 0));
    sst = sd->s;
  }
  const Prof ps{pf.ev, sst};
  StatsArgs sa{lm.gst, NT, M, at<double>(ws, L.Hd), at<float>(ws, L.lsum),
               at<float>(ws, L.rowmax), at<int>(ws, L.amax), out ? out->entropy : nullptr,
               out ? out->argmax : nullptr};
  DG_TRY(ps.mark(DG_PROF_STATS, 0));
  DG_TRY(launch_stats(sa, ctl, sst));
  DG_TRY(ps.mark(DG_PROF_STATS, 1));
  SamplerArgs sp{};
  sp.Hd = at<double>(ws, L.Hd);
  sp.amax = at<int>(ws, L.amax);
  sp.prev_argmax = c.canvas->prev_argmax;
  sp.tokens = c.canvas->tokens;
  sp.acc = at<uint8_t>(ws, L.acc);
  sp.acc_out = out ? out->accept : nullptr;
  sp.n_acc = out ? out->n_acc : nullptr;
  sp.mean_H = out ? out->mean_H : nullptr;
  sp.stop = out ? out->stop : nullptr;
  sp.stop_at = stop_at;
  sp.n_stopped = at<int>(ws, L.status) + 1;
  sp.B = D.B;
  sp.C = D.C;
  sp.V = D.V;
  sp.b = b;
  sp.stop_H = stop_H;
  sp.seed = seed;
  sp.block = block;
  sp.step = step;
  sp.accepted_log = accepted_log;
  sp.N = N;
  DG_TRY(ps.mark(DG_PROF_SAMPLER, 0));
  if (mask_id < 0) {
    DG_TRY(launch_sampler(sp, sst));
  } else {
    RevealArgs rv{at<double>(ws, L.Hd), at<float>(ws, L.lsum), at<int>(ws, L.amax), c.canvas->prev_argmax,
                  c.canvas->tokens, at<uint8_t>(ws, L.acc), sp.acc_out, sp.n_acc, sp.mean_H, sp.stop,
                  accepted_log, D.B, D.C, mask_id, step, N};
    DG_TRY(launch_reveal(rv, sst));
  }
  DG_TRY(ps.mark(DG_PROF_SAMPLER, 1));
  P0Args p0{};
  p0.pt = at<void>(ws, L.pt);
  p0.gst = lm.gst;
  p0.rowmax = at<float>(ws, L.rowmax);
  p0.lsum = at<float>(ws, L.lsum);
  p0.acc = at<uint8_t>(ws, L.acc);
  p0.amax = at<int>(ws, L.amax);
  p0.gbest = at<float>(ws, L.gbest);
  p0.gidx = at<int>(ws, L.gidx);
  p0.M = M;
  p0.V = D.V;
  p0.C = D.C;
  p0.seed = seed;
  p0.block = block;
  p0.step = step;
  p0.ref2f = ref2f;
  DG_TRY(ps.mark(DG_PROF_P0, 0));
  DG_TRY(launch_p0_gumbel(p0, ctl, sst));
  DG_TRY(ps.mark(DG_PROF_P0, 1));
  ScArgs sc{};
  sc.pt = at<void>(ws, L.pt);
  sc.E = c.model->E;
  sc.upart = at<float>(ws, L.upart);
  sc.M = M;
  sc.V = D.V;
  sc.d = D.d;
  sc.nsplit = selfcond_active_splits(D);
  DG_TRY(pf.mark(DG_PROF_SELFCOND, 0));
  DG_TRY(launch_selfcond(sc, ctl, status, c.st));
  DG_TRY(pf.mark(DG_PROF_SELFCOND, 1));
  if (sd) {  // join
    DG_TRY(side_join.join());
    side_lock.unlock();
  }
  ReduceArgs ra{at<float>(ws, L.upart), at<float>(ws, L.gbest), at<int>(ws, L.gidx), at<uint8_t>(ws, L.acc),
                at<void>(ws, L.u), c.canvas->tokens, status, M, D.d, D.C, D.V, sc.nsplit,
                cdiv(D.V, kGumbelChunk), ref2f, at<float>(ws, L.rowmax), at<float>(ws, L.lsum)};
  DG_TRY(pf.mark(DG_PROF_REDUCE, 0));
  DG_TRY(launch_reduce(ra, ctl, c.st));
  DG_TRY(pf.mark(DG_PROF_REDUCE, 1));
  DG_TRY(pf.mark(DG_PROF_FFW1, 0));
  DG_TRY(launch_gemm_bf16(at<void>(ws, L.u), c.model->W1, at<void>(ws, L.g), D.F, nullptr, 0, 1, M, D.F,
                          D.d, D.C, ctl, status, at<float>(ws, L.gpart), L.gpart_elems, c.st));
  DG_TRY(pf.mark(DG_PROF_FFW1, 1));
  DG_TRY(pf.mark(DG_PROF_FFW2, 0));
  DG_TRY(launch_gemm_bf16(at<void>(ws, L.g), c.model->W2, c.canvas->z, D.d, nullptr, 0, 0, M, D.d, D.F,
                          D.C, ctl, status, at<float>(ws, L.gpart), L.gpart_elems, c.st));
  DG_TRY(pf.mark(DG_PROF_FFW2, 1));
  if (out && out->debug) {
    const dg_step_debug* g = out->debug;
    const size_t bf = 2;
    struct {
      void* dst;
      size_t off, bytes;
    } cp[] = {{g->a, L.a, bf * M * D.d},
              {g->q, L.q, bf * M * D.Hq * D.hd},
              {g->k, L.kc, bf * M * D.Hkv * D.hd},
              {g->v, L.vc, bf * M * D.Hkv * D.hd},
              {g->o, L.o, bf * M * D.Hq * D.hd},
              {g->h, L.h, bf * M * D.d},
              {g->u, L.u, bf * M * D.d},
              {g->g, L.g, bf * M * D.F}};
    for (auto& e : cp)
      if (e.dst) DG_TRY(cudaMemcpyAsync(e.dst, at<void>(ws, e.off), e.bytes, cudaMemcpyDeviceToDevice, c.st));
    if (g->moe_x && D.n_exp > 0)
      DG_TRY(cudaMemcpyAsync(g->moe_x, at<void>(ws, L.moe_x), bf * M * D.d, cudaMemcpyDeviceToDevice, c.st));
  }
  return DG_OK;
}

dg_status check_cache(const dg_dims& D, const dg_kv_cache* cache) {
  if (!cache || !cache->K || !cache->V) return DG_ERR_ARG;
  if (cache->cap < 0 || cache->len < 0 || cache->len > cache->cap) return DG_ERR_ARG;
  (void)D;
  return DG_OK;
}

dg_status check_canvas(const dg_canvas* cv) {
  if (!cv || !cv->tokens || !cv->z || !cv->alpha || !cv->prev_argmax) return DG_ERR_ARG;
  return DG_OK;
}

// Linear temperature anneal of [TR] step 3 / Table 2: tau0 at step 0, tau1 at
// step N - 1, in double, rounded once to float.
float tau_at(const dg_sched& sc, int step) {
  const double frac = sc.N > 1 ? (double)step / (double)(sc.N - 1) : 0.0;
  return (float)((double)sc.tau0 + ((double)sc.tau1 - (double)sc.tau0) * frac);
}

}  // namespace

namespace dg {

int selfcond_splits(const dg_dims& D) {
  const int n_tiles = cdiv(D.d, kScBN), m_pairs = cdiv((int64_t)D.B * D.C, 256);
  int ns = (kTargetCtas / 2) / (n_tiles * m_pairs);  // one CTA pair per (split, tile)
  const int nkb = cdiv(D.V, 64);
  if (ns > nkb) ns = nkb;
  if (ns > 64) ns = 64;
  if (ns < 1) ns = 1;
  return ns;
}

bool ws_layout(const dg_dims& D, int32_t cap, WsLayout* L) {
  if (cap < 0) return false;
  const size_t M = (size_t)D.B * D.C, NT = (size_t)cdiv(D.V, kStatCols);
  // room for the largest split count any prefix length up to cap can use
  const int ns_attn = attn_max_splits(D, cap + D.C);
  const size_t S = (size_t)selfcond_splits(D);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + (bytes ? bytes : 1), 256);
    return o;
  };
  L->status = take(256);
  L->stop_at = take(4 * D.B);
  L->rope = take(8 * (size_t)D.C * (D.hd / 2));
  L->a = take(2 * M * D.d);
  L->q = take(2 * M * D.Hq * D.hd);
  L->kc = take(2 * M * D.Hkv * D.hd);
  L->vc = take(2 * M * D.Hkv * D.hd);
  L->o = take(2 * M * D.Hq * D.hd);
  L->h = take(2 * M * D.d);
  L->attn_o = take(4 * (size_t)ns_attn * M * D.Hq * D.hd);
  L->attn_ml = take(8 * (size_t)ns_attn * M * D.Hq);
  L->pt = take(2 * M * (size_t)D.V);
  L->gst = take(sizeof(GroupStat) * NT * M);
  L->Hd = take(8 * M);
  L->lsum = take(4 * M);
  L->rowmax = take(4 * M);
  L->amax = take(4 * M);
  L->acc = take(M);
  L->upart = take(4 * S * M * D.d);
  const size_t NC = (size_t)cdiv(D.V, kGumbelChunk);
  L->gbest = take(4 * NC * M);
  L->gidx = take(4 * NC * M);
  {
    const int nq = D.Hq * D.hd, nkv = D.Hkv * D.hd;
    const int shapes[5][2] = {{nq + 2 * nkv, D.d}, {D.d, nq}, {D.F, D.d}, {D.d, D.F}, {2 * nkv, D.d}};
    size_t most = 0;
    for (auto& sh : shapes) {
      const size_t e = (size_t)gemm_ksplit((int)M, sh[0], sh[1]) * M * sh[0];
      if (e > most) most = e;
    }
    L->gpart_elems = most;
    L->gpart = take(4 * most);
  }
  L->u = take(2 * M * D.d);
  L->g = take(2 * M * D.F);
  L->h8 = take(M * D.d);
  L->hscale = take(4 * M);
  L->ref2 = take(4 * M);
  L->ref2f = take(4 * M);
  L->rkey = take(4 * M);
  if (D.n_exp > 0) {
    const size_t K = D.top_k, R = M * (K + 1);
    L->moe_max_tiles = cdiv((int64_t)R, kMoeTileRows) + D.n_exp + 1;
    L->moe_x = take(2 * M * D.d);
    L->moe_idx = take(4 * M * K);
    L->moe_gate = take(4 * M * K);
    L->moe_slot = take(4 * R);
    L->moe_ptok = take(4 * R);
    L->moe_pgate = take(4 * R);
    L->moe_tiles = take(16 * (size_t)(L->moe_max_tiles + 1));
    L->moe_xp = take(2 * R * D.d);
    L->moe_gp = take(2 * R * D.Fe);
    L->moe_yp = take(4 * R * D.d);
    L->moe_rpart_elems = (size_t)gemm_ksplit((int)M, D.n_exp, D.d) * M * D.n_exp;
    L->moe_rpart = take(4 * L->moe_rpart_elems);
  }
  L->total = off;
  return true;
}

}  // namespace dg

extern "C" {

const char* dg_status_string(dg_status s) {
  switch (s) {
    case DG_OK: return "ok";
    case DG_ERR_ARG: return "invalid argument";
    case DG_ERR_SHAPE: return "unsupported shape";
    case DG_ERR_CAPACITY: return "cache capacity exceeded";
    case DG_ERR_WORKSPACE: return "workspace too small or misaligned";
    case DG_ERR_CUDA: return "CUDA error";
    case DG_ERR_TIMEOUT: return "device wait timed out";
    case DG_ERR_VALUE: return "device value check failed (token out of range or non-finite probabilities)";
  }
  return "unknown status";
}

dg_status dg_workspace_size(const dg_dims* dims, int32_t cap, size_t* bytes) {
  if (!bytes) return DG_ERR_ARG;
  dg_status s = dims_supported(dims);
  if (s) return s;
  if (cap < 0) return DG_ERR_ARG;
  WsLayout L;
  if (!ws_layout(*dims, cap, &L)) return DG_ERR_SHAPE;
  *bytes = L.total;
  return DG_OK;
}

dg_status dg_quantize_rows_e4m3(const void* X, int32_t R, int32_t d, void* Q, float* scale, void* stream) {
  if (!X || !Q || !scale || R < 0) return DG_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(X) % 16 || reinterpret_cast<uintptr_t>(Q) % 16 ||
      reinterpret_cast<uintptr_t>(scale) % 4)
    return DG_ERR_ARG;
  if (d <= 0 || d % 16 != 0) return DG_ERR_SHAPE;
  return cuda_status(launch_quantize_rows_e4m3(X, R, d, reinterpret_cast<uint8_t*>(Q), scale,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_tau(const dg_sched* sched, int32_t step, float* tau) {
  if (!sched || !tau || sched->N <= 0 || step < 0 || step >= sched->N || !(sched->tau0 > 0.f) ||
      !(sched->tau1 > 0.f))
    return DG_ERR_ARG;
  *tau = tau_at(*sched, step);
  return DG_OK;
}

dg_status dg_read_status(const void* ws, int32_t* status, void* stream) {
  if (!ws || !status) return DG_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DG_TRY(cudaMemcpyAsync(status, ws, 4, cudaMemcpyDeviceToHost, st));
  DG_TRY(cudaStreamSynchronize(st));
  return DG_OK;
}

dg_status dg_canvas_init(int32_t* tokens, int32_t B, int32_t C, int32_t V, uint64_t seed,
                         int32_t block, void* stream) {
  if (!tokens || B <= 0 || C <= 0 || V <= 0) return DG_ERR_ARG;
  return cuda_status(launch_canvas_init(tokens, B, C, V, seed, block, reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_denoise_step(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas,
                          float tau, float b, uint64_t seed, int32_t step, int32_t block, void* ws,
                          size_t ws_bytes, dg_step_out* out, void* stream) {
  dg_status s = check_model(model);
  if (s) return s;
  if ((s = check_cache(model->dims, cache)) || (s = check_canvas(canvas))) return s;
  if (!(tau > 0.f) || !(b >= 0.f) || step < 0 || block < 0) return DG_ERR_ARG;
  StepCtx c{model, cache, canvas, ws, {}, reinterpret_cast<cudaStream_t>(stream)};
  if ((s = check_ws(model->dims, cache->cap, ws, ws_bytes, &c.L))) return s;
  // A lone step treats every canvas as still denoising.
  DG_TRY(cudaMemsetAsync(at<void>(ws, c.L.stop_at), 0x7f, 4 * (size_t)model->dims.B, c.st));
  return enqueue_step(c, tau, b, 0.005f, seed, step, block, out, nullptr, 0, true);
}

dg_status dg_denoise_canvas(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas,
                            const dg_sched* sched, uint64_t seed, int32_t block, void* ws,
                            size_t ws_bytes, dg_canvas_result* result, void* stream) {
  dg_status s = check_model(model);
  if (s) return s;
  if ((s = check_cache(model->dims, cache)) || (s = check_canvas(canvas))) return s;
  if (!sched || sched->N <= 0 || sched->N > 4096 || !(sched->tau0 > 0.f) || !(sched->tau1 > 0.f) ||
      !(sched->b >= 0.f) || block < 0)
    return DG_ERR_ARG;
  if (!result || !result->steps_taken || !result->converged || !result->accepted || !result->xhat0)
    return DG_ERR_ARG;
  StepCtx c{model, cache, canvas, ws, {}, reinterpret_cast<cudaStream_t>(stream)};
  if ((s = check_ws(model->dims, cache->cap, ws, ws_bytes, &c.L))) return s;
  const dg_dims& D = model->dims;
  int* n_stopped = at<int>(ws, c.L.status) + 1;
  DG_TRY(cudaMemsetAsync(at<void>(ws, c.L.stop_at), 0x7f, 4 * (size_t)D.B, c.st));
  DG_TRY(cudaMemsetAsync(n_stopped, 0, sizeof(int), c.st));
  DG_TRY(cudaMemsetAsync(result->accepted, 0xff, 4 * (size_t)D.B * sched->N, c.st));
  // Outside a stream capture the loop reads the count of stopped canvases
  // (4 bytes; the stream is synchronised) after step 1, the first step at
  // which the stop test can fire, and every kLoopCheck steps after, and
  // enqueues nothing more once every canvas has stopped.  Under capture it
  // enqueues all N steps; their kernels exit at once after every canvas stopped.
  constexpr int kLoopCheck = 4;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  DG_TRY(cudaStreamIsCapturing(c.st, &cap));
  const bool check = cap == cudaStreamCaptureStatusNone;
  const int N = sched->N;
  for (int step = 0; step < N; ++step) {
    s = enqueue_step(c, tau_at(*sched, step), sched->b, sched->stop_H, seed, step, block, nullptr,
                     result->accepted, N, step == 0);
    if (s) return s;
    if (check && step + 1 < N && step % kLoopCheck == 1) {
      int stopped = 0;
      DG_TRY(cudaMemcpyAsync(&stopped, n_stopped, sizeof(int), cudaMemcpyDeviceToHost, c.st));
      DG_TRY(cudaStreamSynchronize(c.st));
      if (stopped >= D.B) break;
    }
  }
  return cuda_status(launch_loop_finish(at<int>(ws, c.L.stop_at), D.B, N, result->steps_taken,
                                        result->converged, canvas->prev_argmax, result->xhat0, D.C, c.st));
}

dg_status dg_canvas_init_masked(int32_t* tokens, int32_t B, int32_t C, int32_t mask_id, void* stream) {
  if (!tokens || B <= 0 || C <= 0 || mask_id < 0 || (int64_t)B * C > (1 << 30)) return DG_ERR_ARG;
  return cuda_status(launch_fill_tokens(tokens, B * C, mask_id, reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_denoise_step_masked(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas, float tau,
                                 int32_t mask_id, int32_t step, int32_t N, void* ws, size_t ws_bytes,
                                 dg_step_out* out, void* stream) {
  dg_status s = check_model(model);
  if (s) return s;
  if ((s = check_cache(model->dims, cache)) || (s = check_canvas(canvas))) return s;
  if (!(tau > 0.f) || mask_id < 0 || mask_id >= model->dims.V || N <= 0 || step < 0 || step >= N)
    return DG_ERR_ARG;
  StepCtx c{model, cache, canvas, ws, {}, reinterpret_cast<cudaStream_t>(stream)};
  if ((s = check_ws(model->dims, cache->cap, ws, ws_bytes, &c.L))) return s;
  DG_TRY(cudaMemsetAsync(at<void>(ws, c.L.stop_at), 0x7f, 4 * (size_t)model->dims.B, c.st));
  return enqueue_step(c, tau, 0.f, 0.f, 0, step, 0, out, nullptr, N, true, mask_id);
}

dg_status dg_denoise_canvas_masked(const dg_model* model, const dg_kv_cache* cache, dg_canvas* canvas,
                                   const dg_sched* sched, int32_t mask_id, void* ws, size_t ws_bytes,
                                   dg_canvas_result* result, void* stream) {
  dg_status s = check_model(model);
  if (s) return s;
  if ((s = check_cache(model->dims, cache)) || (s = check_canvas(canvas))) return s;
  if (!sched || sched->N <= 0 || sched->N > 4096 || !(sched->tau0 > 0.f) || mask_id < 0 ||
      mask_id >= model->dims.V)
    return DG_ERR_ARG;
  if (!result || !result->steps_taken || !result->converged || !result->accepted || !result->xhat0)
    return DG_ERR_ARG;
  StepCtx c{model, cache, canvas, ws, {}, reinterpret_cast<cudaStream_t>(stream)};
  if ((s = check_ws(model->dims, cache->cap, ws, ws_bytes, &c.L))) return s;
  const dg_dims& D = model->dims;
  DG_TRY(cudaMemsetAsync(at<void>(ws, c.L.stop_at), 0x7f, 4 * (size_t)D.B, c.st));
  const int N = sched->N;
  for (int step = 0; step < N; ++step) {
    s = enqueue_step(c, sched->tau0, 0.f, 0.f, 0, step, 0, nullptr, result->accepted, N, step == 0, mask_id);
    if (s) return s;
  }
  // every canvas ran all N steps; its result is the revealed canvas itself
  DG_TRY(launch_loop_finish(at<int>(ws, c.L.stop_at), D.B, N, result->steps_taken, result->converged, nullptr,
                            nullptr, D.C, c.st));
  DG_TRY(cudaMemcpyAsync(result->xhat0, canvas->tokens, 4 * (size_t)D.B * D.C, cudaMemcpyDeviceToDevice, c.st));
  return DG_OK;
}

dg_status dg_prefill(const dg_model* model, dg_kv_cache* cache, const int32_t* tokens, int32_t n, void* ws,
                     size_t ws_bytes, void* stream) {
  dg_status s = check_model(model);
  if (s) return s;
  if ((s = check_cache(model->dims, cache))) return s;
  if (!tokens || n < 1) return DG_ERR_ARG;
  const dg_dims& D = model->dims;
  WsLayout L;
  if ((s = check_ws(D, cache->cap, ws, ws_bytes, &L))) return s;
  if ((int64_t)cache->len + n > cache->cap) return DG_ERR_CAPACITY;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  StopCtl none{nullptr, 0, 0};
  int* status = at<int>(ws, L.status);
  float2* rope = at<float2>(ws, L.rope);
  const size_t nq = (size_t)D.Hq * D.hd, nkv = (size_t)D.Hkv * D.hd, dd = D.d;
  const size_t cache_layer = (size_t)D.B * D.Hkv * cache->cap * D.hd * 2;
  // pieces of at most C tokens per canvas: the workspace holds B * C rows
  for (int32_t done = 0; done < n;) {
    const int np = n - done < D.C ? n - done : D.C;
    dg_dims Dn = D;
    Dn.C = np;
    const int len = cache->len;
    // this piece's tokens, [B][np], gathered from [B][n]
    int32_t* tk = at<int32_t>(ws, L.amax);  // free between steps: the step rewrites it
    DG_TRY(cudaMemcpy2DAsync(tk, 4 * (size_t)np, tokens + done, 4 * (size_t)n, 4 * (size_t)np, D.B,
                             cudaMemcpyDeviceToDevice, st));
    DG_TRY(launch_embed_rmsnorm(tk, model->E, nullptr, at<void>(ws, L.a), rope, Dn, D.B * np, len, none, status,
                                st));
    for (int l = 0; l < D.L; ++l) {
      const bool last = l == D.L - 1;
      if (l > 0)
        DG_TRY(launch_embed_rmsnorm(nullptr, nullptr, nullptr, at<void>(ws, L.a), nullptr, Dn, D.B * np, len, none,
                                    status, st, at<void>(ws, L.h)));
      // k, v (and below the last layer q) of the piece into the workspace
      DG_TRY(launch_qkv(at<void>(ws, L.a), last ? nullptr : layer_ptr(model->Wq, l, nq * dd),
                        layer_ptr(model->Wk, l, nkv * dd), layer_ptr(model->Wv, l, nkv * dd), at<void>(ws, L.q),
                        at<void>(ws, L.kc), at<void>(ws, L.vc), np, 0, rope, Dn, none, status,
                        at<float>(ws, L.gpart), L.gpart_elems, st));
      // ... appended to this layer's cache at rows len..len+np-1
      const size_t row_bytes = (size_t)D.hd * 2;
      for (int kv = 0; kv < 2; ++kv)
        DG_TRY(cudaMemcpy2DAsync(byte_ptr(kv ? cache->V : cache->K, l * cache_layer + (size_t)len * row_bytes),
                                 cache->cap * row_bytes, at<void>(ws, kv ? L.vc : L.kc), np * row_bytes,
                                 np * row_bytes, (size_t)D.B * D.Hkv, cudaMemcpyDeviceToDevice, st));
      if (last) break;
      // causal attention over the cached rows and the piece, then the output
      // projection with the residual
      AttnArgs aa{at<void>(ws, L.q), byte_ptr(cache->K, l * cache_layer), byte_ptr(cache->V, l * cache_layer),
                  at<void>(ws, L.kc), at<void>(ws, L.vc), at<void>(ws, L.o), at<float>(ws, L.attn_o),
                  at<float>(ws, L.attn_ml), D.B, np, D.Hq, D.Hkv, D.hd, len, cache->cap, 1};
      DG_TRY(launch_attention(aa, none, status, st));
      DG_TRY(launch_gemm_bf16(at<void>(ws, L.o), layer_ptr(model->Wo, l, dd * nq), at<void>(ws, L.h), D.d,
                              at<void>(ws, L.a), D.d, 0, D.B * np, D.d, D.Hq * D.hd, np, none, status,
                              at<float>(ws, L.gpart), L.gpart_elems, st));
      // the layer's MoE block feeds the next layer (the last layer's is not needed)
      if (D.n_exp > 0) {
        dg_status ms = enqueue_moe(model, l, ws, L, D.B * np, np, none, status, nullptr, st);
        if (ms) return ms;
      }
    }
    cache->len += np;
    done += np;
  }
  return DG_OK;
}

dg_status dg_commit_block(const dg_model* model, dg_kv_cache* cache, const int32_t* tokens, void* ws,
                          size_t ws_bytes, void* stream) {
  if (!model) return DG_ERR_ARG;
  return dg_prefill(model, cache, tokens, model->dims.C, ws, ws_bytes, stream);
}

dg_status dg_debug_gemm(const void* A, const void* Bm, float* D, int32_t M, int32_t N, int32_t K,
                        int32_t b_mn_major, void* stream) {
  if (!A || !Bm || !D || M <= 0 || N <= 0 || K <= 0 || b_mn_major < 0 || b_mn_major > 8)
    return DG_ERR_ARG;
  if (K % 8 != 0 || N % 8 != 0) return DG_ERR_SHAPE;
  if (b_mn_major >= 5 && cdiv(K, 64) < (b_mn_major == 6 || b_mn_major == 8 ? 4 : 2)) return DG_ERR_SHAPE;
  int* status = nullptr;
  DG_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_debug_status));
  return cuda_status(launch_debug_gemm(A, Bm, D, M, N, K, b_mn_major, status,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_debug_wait_timeout(int32_t* status, void* stream) {
  if (!status) return DG_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* word = nullptr;
  DG_TRY(cudaGetSymbolAddress(reinterpret_cast<void**>(&word), g_debug_status));
  DG_TRY(cudaMemsetAsync(word, 0, sizeof(int), st));
  DG_TRY(launch_wait_timeout(word, st));
  DG_TRY(cudaMemcpyAsync(status, word, sizeof(int), cudaMemcpyDeviceToHost, st));
  DG_TRY(cudaStreamSynchronize(st));
  return DG_OK;
}

}  // extern "C"
