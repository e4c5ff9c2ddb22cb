// Fused vocabulary kernel of the denoising step: the LM head with its softmax
// statistics ("DiffusionGemma Technical Report" summary, method step 3:
// p0 = softmax(l / tau), entropy, argmax) and the self-conditioning
// contraction u = p0 . E ("DiffusionGemma explained", "Self-conditioning")
// in one persistent launch, so that the embedding E is read from HBM once per
// step instead of once per product.
//
// Schedule.  The vocabulary is cut into chunks whose E rows (with the next
// chunk's) fit in L2.  Work items:
//   * LM item (chunk c, row pair mp, vocabulary tile nt): a 256 x 256 tile of
//     h E^T on a CTA pair (tcgen05 cta_group::2, M = 256, N = 256); its
//     epilogue writes, per (row, 128-column group g), the integer reference
//     k_g = ceil(max_g t) of t = s log2 e, the sums l_g = sum 2^(t - k_g),
//     S_g = sum 2^(t - k_g) (t - k_g), the group's largest logit and its
//     index, and stores the tile 2^(t - k_g) as bf16.
//   * contraction slot (row pair mp, d tile dt, vocabulary slice q): owned by
//     one CTA pair for the whole launch, it accumulates in TMEM, chunk after
//     chunk, U = sum over its slice of 2^(t - R) E_v for the rows of mp and
//     the 256 columns of dt.  R is a per-row integer reference: the maximum of
//     k_g over the first chunk's slice, raised (and the accumulator rescaled
//     by an exact power of two) only when a later chunk's slice maximum
//     exceeds it by more than kRescaleT.  The A operand is the stored tile
//     scaled in shared memory by 2^(k_g - R) (exact in bf16).
// A slot may take its slice of chunk c once the LM tiles that cover the slice
// (for its rows) have finished; LM items are claimed in chunk order from a
// global counter, at most kLookahead chunks ahead of the slowest slot, so that
// the E rows a slot reads are still in L2.  The group references of a slice
// come into shared memory by one tensor copy per slice, so the operand scaling
// needs no dependent global loads.
// Each CTA pair runs one sequence of items: its leader's producer thread
// decides the next item (the slot's next chunk when it is ready, else an LM
// item) and passes it through a small queue in shared memory to the other
// roles of both CTAs.  Items are taken in an order consistent with their
// dependencies and every CTA pair is resident, so the launch cannot deadlock;
// every wait is bounded all the same (status DG_ERR_TIMEOUT).
//
// Roles per CTA (10 warps): warp 0 TMA producer (and, in the leader, the
// scheduler), warp 1 MMA issuer (leader only), warps 2-5 LM epilogue, warps
// 6-9 contraction operand scaling, accumulator rescale and final drain.
// TMEM: 512 columns; a pair with a slot keeps the LM accumulator in columns
// 0-255 and the slot's accumulator in 256-511, a pair without one double
// buffers the LM accumulator.
#include <cfloat>
#include <climits>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

constexpr int kVBM = 128;          // rows per CTA
constexpr int kVBK = 64;           // K elements per 128-byte swizzled row
#ifndef DG_VOCAB_STAGES
#define DG_VOCAB_STAGES 6
#endif
constexpr int kVStages = DG_VOCAB_STAGES;
constexpr int kVStage = 32768;     // A 16 KB + B 16 KB per CTA
constexpr int kVThreads = 448;     // 14 warps
constexpr int kVQueue = 8;
constexpr int kConvWarps = 8;      // operand-scaling warps per CTA (two per row quarter)
constexpr int kQEmptyCount = 2 * (1 + 4 + kConvWarps);  // per CTA: MMA or producer, epilogue, scaling
constexpr float kRescaleT = 96.f;  // log2 units a slice maximum may exceed R by before a rescale
constexpr int kItemEnd = -1;
constexpr int kItemSc = 1 << 30;
#ifndef DG_VOCAB_LOOKAHEAD
#define DG_VOCAB_LOOKAHEAD 3
#endif
#ifndef DG_VOCAB_L2_MB
#define DG_VOCAB_L2_MB 88
#endif
constexpr int kLookahead = DG_VOCAB_LOOKAHEAD;  // LM chunks in flight beyond the slowest slot's
constexpr size_t kVocabL2Budget = size_t(DG_VOCAB_L2_MB) << 20;
constexpr int kMaxSliceKb = 32;    // K blocks of one slice of one chunk (<= 17 groups)
constexpr int kKgBox = 20;         // groups per row in a slice's reference copy (>= 17 + 3)
constexpr int kKgBytes = kKgBox * 4 * kVBM;

struct VLayout {
  static constexpr int kKg = kVStages * kVStage;        // two slice reference buffers
  static constexpr int kBar = kKg + 2 * ((kKgBytes + 1023) / 1024 * 1024);
  // barriers: full, scfull, conv, empty [S]; lm_tfull[2], lm_tempty[2], scdone; kgfull[2], kgempty[2];
  // qfull, qempty [Q]
  static constexpr int kNumBars = 4 * kVStages + 5 + 4 + 2 * kVQueue;
  static constexpr int kQItem = kBar + kNumBars * 8;
  static constexpr int kSlot = kQItem + kVQueue * 4;
  static constexpr int kSmem = kSlot + 16 + 1024;
};

struct VocabKParams {
  VocabPlan P;
  const float* alpha;
  float coef2, inv_sqrt_d;
  __nv_bfloat16* pt;
  float *pm, *pl, *pS, *pvmax;
  int* pidx;
  float* logits;
  float* upart;
  float* rref;
  int* lm_counter;
  int* lm_done;  // [n_nt][n_mp]: finished epilogue warps of each LM tile (8 when done)
  int* sc_done;  // [nC]: slots that issued their slice of the chunk
  int* status;
};

DG_DEV int v_chunk_tiles(const VocabPlan& P, int c) { return c < P.nC - 1 ? P.TPC : P.n_nt - c * P.TPC; }
DG_DEV int v_chunk_kb(const VocabPlan& P, int c) {
  const int len = min(P.CH, P.V - c * P.CH);
  return (len + kVBK - 1) / kVBK;
}
// LM item i (chunk-major, then row pair, then tile) -> chunk, row pair, tile.
DG_DEV void v_lm_decode(const VocabPlan& P, int i, int& c, int& mp, int& nt) {
  const int per = P.n_mp * P.TPC;
  c = i / per;
  if (c > P.nC - 1) c = P.nC - 1;
  const int r = i - c * per, tpc = v_chunk_tiles(P, c);
  mp = r / tpc;
  nt = c * P.TPC + r % tpc;
}
DG_DEV int v_lm_chunk(const VocabPlan& P, int i) {
  const int c = i / (P.n_mp * P.TPC);
  return c < P.nC - 1 ? c : P.nC - 1;
}
DG_DEV void v_slice(const VocabPlan& P, int c, int q, int& k0, int& k1) {
  const int nkb = v_chunk_kb(P, c);
  k0 = (int)((int64_t)q * nkb / P.Q);
  k1 = (int)((int64_t)(q + 1) * nkb / P.Q);
}
// The LM tiles that cover K blocks [k0, k1) of chunk c.
DG_DEV void v_slice_tiles(const VocabPlan& P, int c, int k0, int k1, int& t0, int& t1) {
  t0 = (c * P.CH + k0 * kVBK) / 256;
  t1 = (c * P.CH + k1 * kVBK - 1) / 256;
}

DG_DEV int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
DG_DEV int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
DG_DEV void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DG_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// 2^n for an integer n, exactly (0 below the normal range).
DG_DEV float pow2i(int n) { return n < -126 ? 0.f : (n > 127 ? __int_as_float(0x7f800000) : __int_as_float((n + 127) << 23)); }
DG_DEV void st_cluster_u32(uint32_t caddr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(caddr), "r"(v) : "memory");
}
DG_DEV void mbar_arrive_cluster_release(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// try_wait with cluster-scope acquire: pairs with a release.cluster arrive
// from the other CTA of the pair (the queue entries it wrote remotely).
DG_DEV bool mbar_try_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
DG_DEV bool qwait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort) {
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicExch(status, kStatusTimeout);
      *abort = 1;
      return false;
    }
  }
}
// Bounded spin until *p >= target (acquire).  False after recording a timeout.
DG_DEV bool wait_count(const int* p, int target, int* status, volatile int* abort) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    __nanosleep(128);
    if (ld_acquire(p) >= target) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicExch(status, kStatusTimeout);
      *abort = 1;
      return false;
    }
  }
}

// Queue consumption common to every role: wait for entry qi, read it, release it.
struct QReader {
  int qi = 0;
  uint32_t qph = 0;
  DG_DEV int next(uint64_t* qfull, uint64_t* qempty, const int* qitem, bool leader, bool warp_wide, int* status,
                  volatile int* abort) {
    bool ok;
    if (warp_wide)
      ok = __all_sync(0xffffffffu, qwait(&qfull[qi], qph, status, abort));
    else
      ok = qwait(&qfull[qi], qph, status, abort);
    int item = ok ? reinterpret_cast<const volatile int*>(qitem)[qi] : kItemEnd;
    if (warp_wide) __syncwarp();
    if (!warp_wide || (threadIdx.x % 32) == 0) {
      if (leader)
        mbar_arrive(&qempty[qi]);
      else
        mbar_arrive_cluster(cluster_addr(&qempty[qi], 0));
    }
    if (++qi == kVQueue) {
      qi = 0;
      qph ^= 1;
    }
    return item;
  }
};

__global__ void __launch_bounds__(kVThreads, 1)
    vocab_kernel(const __grid_constant__ CUtensorMap mH, const __grid_constant__ CUtensorMap mE,
                 const __grid_constant__ CUtensorMap mP, const __grid_constant__ CUtensorMap mEmn,
                 const __grid_constant__ CUtensorMap mKg, const VocabKParams p, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const VocabPlan& P = p.P;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + VLayout::kBar);
  uint64_t* full = bars;
  uint64_t* scfull = full + kVStages;
  uint64_t* conv = scfull + kVStages;
  uint64_t* empty = conv + kVStages;
  uint64_t* lm_tfull = empty + kVStages;
  uint64_t* lm_tempty = lm_tfull + 2;
  uint64_t* scdone = lm_tempty + 2;
  uint64_t* kgfull = scdone + 1;
  uint64_t* kgempty = kgfull + 2;
  uint64_t* qfull = kgempty + 2;
  uint64_t* qempty = qfull + kVQueue;
  int* qitem = reinterpret_cast<int*>(smem + VLayout::kQItem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + VLayout::kSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = (int)cluster_id_x();
  const bool has_slot = cid < P.n_slots;
  const int s_q = has_slot ? cid / (P.n_mp * P.n_dt) : 0;
  const int s_rem = has_slot ? cid % (P.n_mp * P.n_dt) : 0;
  const int s_mp = s_rem / P.n_dt, s_dt = s_rem % P.n_dt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&scfull[s], 1);
      mbar_init(&conv[s], 2 * kConvWarps);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&lm_tfull[a], 1);
      mbar_init(&lm_tempty[a], 8);
    }
    mbar_init(scdone, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kgfull[i], 1);
      mbar_init(&kgempty[i], kConvWarps);  // this CTA's scaling warps
    }
    for (int i = 0; i < kVQueue; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], kQEmptyCount);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  QReader qr;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch(&mH);
      tma_prefetch(&mE);
      tma_prefetch(&mP);
      tma_prefetch(&mEmn);
      tma_prefetch(&mKg);
      int stage = 0;
      uint32_t eph = 0;
      int kgb = 0;
      uint32_t kgph = 0;
      bool alive = true;
      // scheduler state (leader)
      int c_sc = 0, held = -1;
      bool lm_out = false;
      int wq = 0;
      uint32_t wqph = 0;
      auto lm_allowed = [&](int c) {
        return c <= kLookahead || ld_relaxed(p.sc_done + c - kLookahead - 1) >= P.n_slots;
      };
      // the slot's next slice is ready once the LM tiles covering it are done
      auto sc_ready = [&](int c) {
        int k0, k1, t0, t1;
        v_slice(P, c, s_q, k0, k1);
        if (k1 <= k0) return true;
        v_slice_tiles(P, c, k0, k1, t0, t1);
        for (int t = t0; t <= t1; ++t)
          if (ld_acquire(p.lm_done + t * P.n_mp + s_mp) < 8) return false;
        return true;
      };
      auto decide = [&]() -> int {
        const uint64_t t0 = globaltimer();
        while (true) {
          if (*abort) return kItemEnd;
          if (has_slot && c_sc < P.nC && sc_ready(c_sc)) return kItemSc | c_sc++;
          if (held < 0 && !lm_out) {
            const int peek = ld_relaxed(p.lm_counter);
            if (peek >= P.n_lm) {
              lm_out = true;
            } else if (lm_allowed(v_lm_chunk(P, peek))) {
              const int i = atomicAdd(p.lm_counter, 1);
              if (i >= P.n_lm)
                lm_out = true;
              else
                held = i;
            }
          }
          if (held >= 0 && lm_allowed(v_lm_chunk(P, held))) {
            const int i = held;
            held = -1;
            return i;
          }
          if (lm_out && held < 0 && (!has_slot || c_sc >= P.nC)) return kItemEnd;
          if (globaltimer() - t0 > kWaitLimitNs) {
            atomicExch(p.status, kStatusTimeout);
            *abort = 1;
            return kItemEnd;
          }
          __nanosleep(256);
        }
      };
      while (true) {
        int item;
        if (leader) {
          item = alive ? decide() : kItemEnd;
          if (!mbar_wait(&qempty[wq], wqph ^ 1, p.status, abort)) item = kItemEnd;
          qitem[wq] = item;
          st_cluster_u32(cluster_addr(&qitem[wq], 1), (uint32_t)item);
          mbar_arrive(&qfull[wq]);
          mbar_arrive_cluster_release(cluster_addr(&qfull[wq], 1));
          if (++wq == kVQueue) {
            wq = 0;
            wqph ^= 1;
          }
        } else {
          item = qr.next(qfull, qempty, qitem, false, false, p.status, abort);
        }
        if (item == kItemEnd) break;
        if (!alive) continue;
        if (!(item & kItemSc)) {
          int c, mp, nt;
          v_lm_decode(P, item, c, mp, nt);
          const int arow = mp * 2 * kVBM + (int)rank * kVBM, bcol = nt * 256 + (int)rank * 128;
          for (int kb = 0; kb < P.kd; ++kb) {
            if (!mbar_wait(&empty[stage], eph ^ 1, p.status, abort)) {
              alive = false;
              break;
            }
            uint8_t* sa = smem + stage * kVStage;
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kVStage);
            const uint32_t bar = cluster_addr(&full[stage], 0);
            tma_load_2d_pair(sa, &mH, bar, kb * kVBK, arow);
            tma_load_2d_pair(sa + kVStage / 2, &mE, bar, kb * kVBK, bcol);
            if (++stage == kVStages) {
              stage = 0;
              eph ^= 1;
            }
          }
        } else {
          const int c = item & ~kItemSc;
          int k0, k1;
          v_slice(P, c, s_q, k0, k1);
          if (k1 <= k0) {
            if (leader) atomicAdd(p.sc_done + c, 1);
            continue;
          }
          // the stored tiles and group references of the slice were written by
          // other CTAs (generic proxy): acquire the tiles' completion counts,
          // then order the async-proxy reads after them
          int t0, t1;
          v_slice_tiles(P, c, k0, k1, t0, t1);
          for (int t = t0; t <= t1 && alive; ++t)
            alive = wait_count(p.lm_done + t * P.n_mp + s_mp, 8, p.status, abort);
          if (!alive) continue;
          fence_proxy_async_global();
          const int arow = s_mp * 2 * kVBM + (int)rank * kVBM;
          const int dcol = s_dt * 256 + (int)rank * 128;
          // the slice's group references, rows of this CTA: one copy
          if (!mbar_wait(&kgempty[kgb], kgph ^ 1, p.status, abort)) {
            alive = false;
            continue;
          }
          mbar_arrive_expect_tx(&kgfull[kgb], kKgBytes);
          tma_load_2d(smem + VLayout::kKg + kgb * ((kKgBytes + 1023) / 1024 * 1024), &mKg, &kgfull[kgb],
                      ((c * P.CH + k0 * kVBK) / kStatCols) & ~3, arow);
          if (++kgb == 2) {
            kgb = 0;
            kgph ^= 1;
          }
          for (int kb = k0; kb < k1; ++kb) {
            if (!mbar_wait(&empty[stage], eph ^ 1, p.status, abort)) {
              alive = false;
              break;
            }
            uint8_t* sa = smem + stage * kVStage;
            mbar_arrive_expect_tx(&scfull[stage], kVStage);
            const int v = c * P.CH + kb * kVBK;
            tma_load_2d(sa, &mP, &scfull[stage], v, arow);
            tma_load_2d(sa + kVStage / 2, &mEmn, &scfull[stage], dcol, v);
            tma_load_2d(sa + kVStage / 2 + 8192, &mEmn, &scfull[stage], dcol + 64, v);
            if (++stage == kVStages) {
              stage = 0;
              eph ^= 1;
            }
          }
          if (leader && alive) atomicAdd(p.sc_done + c, 1);
        }
      }
      // every commit addressed to this CTA's stage barriers has landed before exit
      for (int i = 0; i < kVStages && alive; ++i) {
        if (!mbar_wait(&empty[stage], eph ^ 1, p.status, abort)) break;
        if (++stage == kVStages) {
          stage = 0;
          eph ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      constexpr uint32_t idesc_lm = idesc_bf16(2 * kVBM, 256, false);
      constexpr uint32_t idesc_sc = idesc_bf16(2 * kVBM, 256, true);
      int stage = 0;
      uint32_t full_par = 0, conv_par = 0;  // per-stage parity bits
      uint32_t tempty_use[2] = {0, 0};
      int lm_it = 0;
      bool sc_started = false, alive = true;
      while (true) {
        const int item = qr.next(qfull, qempty, qitem, true, false, p.status, abort);
        if (item == kItemEnd) break;
        if (!alive) continue;
        if (!(item & kItemSc)) {
          const int acc = has_slot ? 0 : (lm_it & 1);
          ++lm_it;
          if (!mbar_wait(&lm_tempty[acc], (tempty_use[acc] & 1) ^ 1, p.status, abort)) {
            alive = false;
            continue;
          }
          ++tempty_use[acc];
          tc_fence_after();
          const uint32_t dt = tmem + acc * 256;
          for (int kb = 0; kb < P.kd; ++kb) {
            if (!mbar_wait(&full[stage], (full_par >> stage) & 1, p.status, abort)) {
              alive = false;
              break;
            }
            full_par ^= 1u << stage;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * kVStage);
            const uint32_t sb = sa + kVStage / 2;
#pragma unroll
            for (int kk = 0; kk < kVBK / 16; ++kk)
              umma_bf16_pair(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024),
                             idesc_lm, (kb != 0 || kk != 0) ? 1u : 0u);
            umma_commit_pair(&empty[stage]);
            if (++stage == kVStages) stage = 0;
          }
          if (alive) umma_commit_pair(&lm_tfull[acc]);
        } else {
          const int c = item & ~kItemSc;
          int k0, k1;
          v_slice(P, c, s_q, k0, k1);
          const uint32_t dt = tmem + 256;
          for (int kb = k0; kb < k1; ++kb) {
            if (!mbar_wait(&conv[stage], (conv_par >> stage) & 1, p.status, abort)) {
              alive = false;
              break;
            }
            conv_par ^= 1u << stage;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * kVStage);
            const uint32_t sb = sa + kVStage / 2;
#pragma unroll
            for (int kk = 0; kk < kVBK / 16; ++kk) {
              umma_bf16_pair(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 2048, kVBK * 128, 1024),
                             idesc_sc, (sc_started || kk != 0) ? 1u : 0u);
            }
            sc_started = true;
            umma_commit_pair(&empty[stage]);
            if (++stage == kVStages) stage = 0;
          }
          if (alive) umma_commit_pair(scdone);
        }
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------ LM epilogue --
    const int qd = warp & 3;
    const int r_local = qd * 32 + lane;
    uint32_t tfull_use[2] = {0, 0};
    int lm_it = 0;
    const int NTs = P.NTs;
    while (true) {
      const int item = qr.next(qfull, qempty, qitem, leader, true, p.status, abort);
      if (item == kItemEnd) break;
      if (item & kItemSc) continue;
      const int acc = has_slot ? 0 : (lm_it & 1);
      ++lm_it;
      if (!mbar_wait_warp(&lm_tfull[acc], tfull_use[acc] & 1, p.status, abort)) break;
      ++tfull_use[acc];
      tc_fence_after();
      int c, mp, nt;
      v_lm_decode(P, item, c, mp, nt);
      const int row = mp * 2 * kVBM + (int)rank * kVBM + r_local;
      const bool ok = row < P.M;
      const int n0 = nt * 256;
      const uint32_t tb = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * 256);
      const float al = ok ? __ldg(p.alpha + row) : 1.0f;
      const float c2 = al * p.coef2;
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {
        const int g0 = n0 + g * kStatCols;
        if (g0 >= P.V) break;  // uniform over the warp
        float vmax = -FLT_MAX;
        int imax = g0;
#pragma unroll 1
        for (int cc = 0; cc < kStatCols / 32; ++cc) {
          float v[32];
          tmem_ld32(tb + g * kStatCols + cc * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = g0 + cc * 32 + j;
            if (col < P.V && v[j] > vmax) {
              vmax = v[j];
              imax = col;
            }
          }
        }
        // integer reference of the group: the stored tile is 2^(t - kg) with
        // t - kg in (-inf, 0], so scaling it by a power of two is exact
        const float kg = ceilf(vmax * c2);
        float l = 0.f, S = 0.f;
#pragma unroll 1
        for (int cc = 0; cc < kStatCols / 32; ++cc) {
          float v[32];
          tmem_ld32(tb + g * kStatCols + cc * 32, v);
          const int col0 = g0 + cc * 32;
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float t0 = fmaf(v[j], c2, -kg), t1 = fmaf(v[j + 1], c2, -kg);
            const float p0 = (col0 + j < P.V) ? exp2f(t0) : 0.f;
            const float p1 = (col0 + j + 1 < P.V) ? exp2f(t1) : 0.f;
            l += p0 + p1;
            S = fmaf(p0, t0, fmaf(p1, t1, S));
            pk[j / 2] = pack_bf16(p0, p1);
          }
          if (ok) {
            if (col0 + 32 <= P.V) {
              uint4* dst = reinterpret_cast<uint4*>(p.pt + (size_t)row * P.V + col0);
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            } else {
              const __nv_bfloat16* pb = reinterpret_cast<const __nv_bfloat16*>(pk);
              for (int j = 0; j < 32; ++j)
                if (col0 + j < P.V) p.pt[(size_t)row * P.V + col0 + j] = pb[j];
            }
            if (p.logits) {
              const float cl = al * p.inv_sqrt_d;
              for (int j = 0; j < 32; ++j)
                if (col0 + j < P.V) p.logits[(size_t)row * P.V + col0 + j] = v[j] * cl;
            }
          }
        }
        if (ok) {
          const size_t o = (size_t)row * NTs + g0 / kStatCols;
          p.pm[o] = kg;
          p.pl[o] = l;
          p.pS[o] = S;
          p.pvmax[o] = vmax;
          p.pidx[o] = imax;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(&lm_tempty[acc], 0));
      // publish the tile: its stores reach the other CTAs' TMA reads of the
      // stored tile (async proxy) and their loads of the statistics
      fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0) red_release_add(p.lm_done + nt * P.n_mp + mp, 1);
    }
  } else {
    // ------------------------------------ contraction operands and drain --
    // warps 6-9 and 10-13: two warps per quarter of the rows, each scaling half
    // of a row's 16-byte chunks; warps 6-9 also rescale and drain the TMEM
    // accumulator (their lane quarter, warp % 4, holds their rows)
    const int qd = warp & 3;
    const int half = (warp - 6) >> 2;
    const int r_local = qd * 32 + lane;
    const int row = s_mp * 2 * kVBM + (int)rank * kVBM + r_local;
    const bool ok = has_slot && row < P.M;
    const uint32_t tsc = tmem + ((uint32_t)(qd * 32) << 16) + 256u;
    int stage = 0, kgb = 0;
    uint32_t scfull_par = 0, kgph = 0;
    int n_sc = 0;
    float R = -1e30f;
    bool started = false, alive = true;
    while (true) {
      const int item = qr.next(qfull, qempty, qitem, leader, true, p.status, abort);
      if (item == kItemEnd) break;
      if (!(item & kItemSc)) {
        stage = (stage + P.kd) % kVStages;
        continue;
      }
      const int c = item & ~kItemSc;
      int k0, k1;
      v_slice(P, c, s_q, k0, k1);
      ++n_sc;
      if (!alive || k1 <= k0) continue;
      // the slice's group references for this row (one copy per slice)
      if (!mbar_wait_warp(&kgfull[kgb], kgph, p.status, abort)) {
        alive = false;
        continue;
      }
      const float* kgrow = reinterpret_cast<const float*>(smem + VLayout::kKg +
                                                          kgb * ((kKgBytes + 1023) / 1024 * 1024)) +
                           r_local * kKgBox;
      const int gbase = ((c * P.CH + k0 * kVBK) / kStatCols) & ~3;
      const int g1 = min((c * P.CH + k1 * kVBK - 1) / kStatCols, P.NT - 1);
      float m = -1e30f;
      for (int g = (c * P.CH + k0 * kVBK) / kStatCols; g <= g1; ++g) m = fmaxf(m, kgrow[g - gbase]);
      const bool need = started && ok && m > R + kRescaleT;
      if (!started) R = ok ? m : 0.f;
      if (half == 0 && __any_sync(0xffffffffu, need)) {
        // wait until the slot's previous MMAs completed, then rescale the rows
        // whose reference grows (exact powers of two)
        if (!mbar_wait_warp(scdone, (uint32_t)(n_sc - 2) & 1, p.status, abort)) {
          alive = false;
          continue;
        }
        tc_fence_after();
        const float f = need ? pow2i((int)(R - m)) : 1.0f;
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          float v[32];
          tmem_ld32(tsc + cc * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= f;
          tmem_st32(tsc + cc * 32, v);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      if (need) R = m;  // both warps of the quarter keep the same reference
      started = true;
      for (int kb = k0; kb < k1; ++kb) {
        const int g = (c * P.CH + kb * kVBK) / kStatCols;
        const float kg = (ok && g < P.NT) ? kgrow[g - gbase] : -1e30f;
        if (!mbar_wait_warp(&scfull[stage], (scfull_par >> stage) & 1, p.status, abort)) {
          alive = false;
          break;
        }
        scfull_par ^= 1u << stage;
        const float f = kg > -1e29f ? pow2i((int)(kg - R)) : 0.f;  // an exact power of two
        const __nv_bfloat162 f2 = __floats2bfloat162_rn(f, f);
        // the row's eight 16-byte chunks, visited from a row-dependent start so
        // that the lanes of a warp (rows r..r+31, 128 bytes apart) spread over
        // the banks instead of all hitting the same four
        uint4* arow = reinterpret_cast<uint4*>(smem + stage * kVStage + r_local * 128);
        uint4 x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = arow[(4 * half + j) ^ (r_local & 7)];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __nv_bfloat162* xb = reinterpret_cast<__nv_bfloat162*>(&x[j]);
#pragma unroll
          for (int e = 0; e < 4; ++e) xb[e] = __hmul2(xb[e], f2);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) arow[(4 * half + j) ^ (r_local & 7)] = x[j];
        // generic-proxy writes made visible to the tensor core's reads (the
        // leader's pair MMA reads this CTA's rows), then one arrive per warp on
        // the leader's barrier (default semantics: a cluster-scope release here
        // cost about 0.7 us per stage)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cluster_addr(&conv[stage], 0));
        if (++stage == kVStages) stage = 0;
      }
      // the reference buffer is free once every row of the slice is scaled
      __syncwarp();
      if (lane == 0) mbar_arrive(&kgempty[kgb]);
      if (++kgb == 2) {
        kgb = 0;
        kgph ^= 1;
      }
    }
    // drain the slot's sums and their references
    if (half == 0 && has_slot && alive && n_sc > 0 &&
        mbar_wait_warp(scdone, (uint32_t)(n_sc - 1) & 1, p.status, abort)) {
      tc_fence_after();
      const int ncols = min(256, P.d - s_dt * 256);
      float* dst = p.upart + ((size_t)s_q * P.M + (ok ? row : 0)) * P.d + s_dt * 256;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        float v[32];
        tmem_ld32(tsc + cc * 32, v);
        if (!ok || cc * 32 >= ncols) continue;
        if (!started) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        if (cc * 32 + 32 <= ncols) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(dst + cc * 32)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
          for (int j = 0; j < 32; ++j)
            if (cc * 32 + j < ncols) dst[cc * 32 + j] = v[j];
        }
      }
      if (ok && s_dt == 0) p.rref[(size_t)s_q * P.M + row] = started ? R : -1e30f;
    }
  }
  __syncwarp();
  if (*abort) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

int v_max_clusters() {
  static int n = -1;
  if (n < 0) {
    if (cudaFuncSetAttribute(vocab_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, VLayout::kSmem) !=
        cudaSuccess) {
      cudaGetLastError();
      n = 0;
      return n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (kTargetCtas / 2), 1, 1);
    cfg.blockDim = dim3(kVThreads, 1, 1);
    cfg.dynamicSmemBytes = VLayout::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, vocab_kernel, &cfg) != cudaSuccess || c <= 0) {
      cudaGetLastError();
      c = 0;
    }
    n = c;
  }
  return n;
}

}  // namespace

int vocab_chunk(const dg_dims& D) {
  const int64_t M = (int64_t)D.B * D.C;
  // the chunks in flight (the slowest slot's, and kLookahead more in the LM
  // head) with their stored tiles within the L2 budget
  int64_t ch = (int64_t)kVocabL2Budget / ((kLookahead + 1) * 2 * ((int64_t)D.d + M));
  // a slice of a chunk spans at most kMaxSliceKb K blocks
  const int64_t cap = (int64_t)vocab_q_bound(D) * kMaxSliceKb * kVBK;
  if (ch > cap) ch = cap;
  ch = ch / 256 * 256;
  if (ch < 256) ch = 256;
  const int64_t vr = ((int64_t)D.V + 255) / 256 * 256;
  if (ch > vr) ch = vr;
  return (int)ch;
}

int vocab_q_bound(const dg_dims& D) {
  const int pairs = cdiv((int64_t)D.B * D.C, 256) * cdiv(D.d, 256);
  int q = (kTargetCtas / 2) / pairs;
  if (q > kMaxVocabSlices) q = kMaxVocabSlices;
  return q < 1 ? 1 : q;
}

size_t vocab_sync_ints(const dg_dims& D) {
  const int nC = cdiv(D.V, vocab_chunk(D));
  return 1 + (size_t)cdiv(D.V, 256) * cdiv((int64_t)D.B * D.C, 256) + (size_t)nC;
}

bool vocab_plan(const dg_dims& D, VocabPlan* P) {
  const int ncl = v_max_clusters();
  const int M = D.B * D.C;
  P->M = M;
  P->V = D.V;
  P->d = D.d;
  P->NT = cdiv(D.V, kStatCols);
  P->NTs = stat_stride(D.V);
  P->n_mp = cdiv(M, 256);
  P->n_nt = cdiv(D.V, 256);
  P->kd = cdiv(D.d, kVBK);
  P->n_dt = cdiv(D.d, 256);
  P->CH = vocab_chunk(D);
  P->TPC = P->CH / 256;
  P->nC = cdiv(D.V, P->CH);
  const int pairs = P->n_mp * P->n_dt;
  if (ncl <= 0 || pairs > ncl) return false;
  int q = ncl / pairs;
  const int qk = (P->CH / kVBK) / 8;  // slices of at least 8 K blocks
  if (q > qk) q = qk;
  if (q > vocab_q_bound(D)) q = vocab_q_bound(D);
  if (q < 1) q = 1;
  if (cdiv(P->CH / kVBK, q) > kMaxSliceKb) return false;  // fewer pairs than the chunk was sized for
  P->Q = q;
  P->n_slots = pairs * q;
  P->n_lm = P->n_mp * P->n_nt;
  P->ncl = ncl;
  return true;
}

cudaError_t launch_vocab(const VocabArgs& a, const VocabPlan& P, StopCtl ctl, int* status, cudaStream_t st) {
  CUtensorMap mH, mE, mP, mEmn, mKg;
  if (!make_tmap_2d(&mH, a.h, (uint64_t)P.d, (uint64_t)P.M, (uint64_t)P.d * 2, kVBK, kVBM) ||
      !make_tmap_2d(&mE, a.E, (uint64_t)P.d, (uint64_t)P.V, (uint64_t)P.d * 2, kVBK, 128) ||
      !make_tmap_2d(&mP, a.pt, (uint64_t)P.V, (uint64_t)P.M, (uint64_t)P.V * 2, kVBK, kVBM) ||
      !make_tmap_2d(&mEmn, a.E, (uint64_t)P.d, (uint64_t)P.V, (uint64_t)P.d * 2, 64, kVBK) ||
      !make_tmap_2d_ex(&mKg, a.pm, (uint64_t)P.NTs, (uint64_t)P.M, (uint64_t)P.NTs * 4, kKgBox, kVBM, true))
    return cudaErrorInvalidValue;
  VocabKParams k{};
  k.P = P;
  k.alpha = a.alpha;
  k.coef2 = a.coef2;
  k.inv_sqrt_d = a.inv_sqrt_d;
  k.pt = reinterpret_cast<__nv_bfloat16*>(a.pt);
  k.pm = a.pm;
  k.pl = a.pl;
  k.pS = a.pS;
  k.pvmax = a.pvmax;
  k.pidx = a.pidx;
  k.logits = a.logits;
  k.upart = a.upart;
  k.rref = a.rref;
  k.lm_counter = a.sync;
  k.lm_done = a.sync + 1;
  k.sc_done = a.sync + 1 + (size_t)P.n_nt * P.n_mp;
  k.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * P.ncl, 1, 1);
  cfg.blockDim = dim3(kVThreads, 1, 1);
  cfg.dynamicSmemBytes = VLayout::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, vocab_kernel, mH, mE, mP, mEmn, mKg, k, ctl);
}

}  // namespace dg

extern "C" dg_status dg_vocab_plan_info(const dg_dims* dims, int32_t* info) {
  if (!dims || !info) return DG_ERR_ARG;
  dg::VocabPlan P{};
  const bool ok = dg::vocab_plan(*dims, &P);
  const int32_t v[10] = {ok ? 1 : 0, P.ncl, P.n_slots, P.Q, P.CH, P.nC, P.n_lm, P.n_mp, P.n_dt, P.kd};
  for (int i = 0; i < 10; ++i) info[i] = v[i];
  return DG_OK;
}
