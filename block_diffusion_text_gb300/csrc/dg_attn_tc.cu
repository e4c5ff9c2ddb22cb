// Tensor-core (tcgen05 + TMA) attention of the canvas queries over
// [prefix cache ; canvas] with no mask, for head dim 128 ("DiffusionGemma"
// docs chapter, attention-mask list: the canvas is a full bidirectional
// matrix that reads the prompt / finished-block KV cache).
//
// One CTA owns 128 query rows (one tile of the rows of the group's query
// heads) of one (canvas, kv head) and one chunk of the key sequence; the CTAs
// of the other tiles of the group are launched next to it and read the same
// K/V blocks through L2.  Warp roles:
//   warp 0      TMA: the Q tile once, then K/V blocks of 64 keys into a
//               4-stage ring;
//   warp 1      MMA: S = Q K^T (bf16) into double-buffered TMEM, and
//               O += P V (f16) into TMEM;
//   warps 2-3   re-encode each V block from bf16 to f16 in shared memory;
//   warps 4-11  softmax, two threads per row (warps 4-7 take the first 32
//               keys of a block, warps 8-11 the last 32; they exchange their
//               maxima through shared memory): base-2 online softmax with lazy
//               rescaling of O (only when the row maximum grows by more than
//               2^8).  P goes to double-buffered shared memory as two f16
//               parts, P = P_hi + P_lo, and O accumulates P_hi.V + P_lo.V, so
//               the probabilities enter the product to ~2^-22.
// Several key chunks per row are merged by attn_combine_kernel.
#include <cfloat>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

constexpr int kTcHD = 128;
constexpr int kTcKeys = 64;
constexpr int kTcStages = 4;
constexpr int kTcThreads = 384;
constexpr float kLazyRescale = 8.0f;  // log2 units

struct TcLayout {
  static constexpr int kQ = 128 * kTcHD * 2;       // 32 KB: two boxes of 64 columns
  static constexpr int kKV = kTcKeys * kTcHD * 2;  // 16 KB: K or V of one block
  static constexpr int kStage = 2 * kKV;           // K then V
  static constexpr int kP = 128 * kTcKeys * 2;     // 16 KB: one f16 part
  static constexpr int kOffStage = kQ;
  static constexpr int kOffP = kOffStage + kTcStages * kStage;  // [buffer][hi, lo]
  static constexpr int kOffBar = kOffP + 4 * kP;
  static constexpr int kOffRed = kOffBar + 256;  // [2 parities][2 halves][128 rows] float
  // No alignment slack: the kernel checks that dynamic shared memory starts on
  // a 1024-byte boundary (it does when the kernel has no static shared memory).
  static constexpr int kSmem = kOffRed + 2048;
};

DG_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKp,
                   const __grid_constant__ CUtensorMap mVp, const __grid_constant__ CUtensorMap mKc,
                   const __grid_constant__ CUtensorMap mVc, AttnArgs a, int nqt, int kps,
                   float scale_log2, int* status, StopCtl ctl) {
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // uniform over the CTA: return before any barrier
    if (threadIdx.x == 0) atomicExch(status, kStatusTimeout);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem;
  uint8_t* sStage = smem + TcLayout::kOffStage;
  uint8_t* sP = smem + TcLayout::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TcLayout::kOffBar);
  uint64_t* qfull = bars;
  uint64_t* kfull = bars + 1;              // [stages]
  uint64_t* vfull = kfull + kTcStages;     // [stages]
  uint64_t* vready = vfull + kTcStages;    // [stages]
  uint64_t* kvempty = vready + kTcStages;  // [stages]
  uint64_t* sfull = kvempty + kTcStages;   // [2 buffers]
  uint64_t* sfree = sfull + 2;             // [2]
  uint64_t* pready = sfree + 2;            // [2]
  uint64_t* pdone = pready + 2;            // [2]
  uint64_t* xmax = pdone + 2;              // [2]: both halves of every row posted their maximum
  uint64_t* xsum = xmax + 2;               // both halves posted their row sum
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xsum + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int qt = blockIdx.x % nqt, split = blockIdx.x / nqt;
  const int b = blockIdx.y / a.Hkv, g = blockIdx.y % a.Hkv;
  const int grp = a.Hq / a.Hkv;
  const int R = grp * a.C;  // query rows of the group
  const int row0 = qt * 128;
  const int T = a.P + a.C;
  const int k_begin = split * kps;
  const int k_end = min(T, k_begin + kps);
  const int nblk = (k_end - k_begin + kTcKeys - 1) / kTcKeys;

  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vready[s], 64);
      mbar_init(&kvempty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 256);
      mbar_init(&pready[i], 256);
      mbar_init(&pdone[i], 1);
      mbar_init(&xmax[i], 256);
    }
    mbar_init(xsum, 256);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S[buf] at buf*64, O at 128.

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch(&mQ);
      tma_prefetch(&mKp);
      tma_prefetch(&mVp);
      const int qrow = (b * a.Hq + g * grp) * a.C + row0;
      mbar_arrive_expect_tx(qfull, TcLayout::kQ);
      tma_load_2d(sQ, &mQ, qfull, 0, qrow);
      tma_load_2d(sQ + 16384, &mQ, qfull, 64, qrow);
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kTcStages;
        if (!mbar_wait(&kvempty[s], ((j / kTcStages) & 1) ^ 1, status, abort)) break;
        const int kj = k_begin + j * kTcKeys;
        const bool pre = kj < a.P;  // blocks never straddle P (P is a multiple of 64)
        const CUtensorMap* mk = pre ? &mKp : &mKc;
        const CUtensorMap* mv = pre ? &mVp : &mVc;
        const int row = pre ? (b * a.Hkv + g) * a.cap + kj : (b * a.Hkv + g) * a.C + (kj - a.P);
        uint8_t* sk = sStage + s * TcLayout::kStage;
        uint8_t* sv = sk + TcLayout::kKV;
        mbar_arrive_expect_tx(&kfull[s], TcLayout::kKV);
        tma_load_2d(sk, mk, &kfull[s], 0, row);
        tma_load_2d(sk + 8192, mk, &kfull[s], 64, row);
        mbar_arrive_expect_tx(&vfull[s], TcLayout::kKV);
        tma_load_2d(sv, mv, &vfull[s], 0, row);
        tma_load_2d(sv + 8192, mv, &vfull[s], 64, row);
      }
    }
  } else if (warp == 1) {
    constexpr uint32_t idS = idesc_bf16(128, kTcKeys, false);
    constexpr uint32_t idPV = idesc_f16(128, kTcHD, true);
    bool alive = mbar_wait(qfull, 0, status, abort);
    const uint32_t sq = smem_u32(sQ);
    auto issue_S = [&](int j) -> bool {
      const int s = j % kTcStages, bb = j & 1;
      if (!mbar_wait(&kfull[s], (j / kTcStages) & 1, status, abort)) return false;
      if (!mbar_wait(&sfree[bb], ((j >> 1) & 1) ^ 1, status, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sk = smem_u32(sStage + s * TcLayout::kStage);
#pragma unroll
        for (int kk = 0; kk < kTcHD / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(sq + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sk + (kk / 4) * 8192 + (kk % 4) * 32, 16, 1024);
          umma_bf16(tmem + bb * 64, ad, bd, idS, kk ? 1u : 0u);
        }
        umma_commit(&sfull[bb]);
      }
      __syncwarp();
      return true;
    };
    auto issue_PV = [&](int j) -> bool {
      const int s = j % kTcStages, bb = j & 1;
      if (!mbar_wait(&vready[s], (j / kTcStages) & 1, status, abort)) return false;
      if (!mbar_wait(&pready[bb], (j >> 1) & 1, status, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sv = smem_u32(sStage + s * TcLayout::kStage + TcLayout::kKV);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t sp = smem_u32(sP + (2 * bb + part) * TcLayout::kP);
#pragma unroll
          for (int kk = 0; kk < kTcKeys / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sp + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sv + kk * 2048, 8192, 1024);
            umma_bf16(tmem + 128, ad, bd, idPV, (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&pdone[bb]);
        umma_commit(&kvempty[s]);
      }
      __syncwarp();
      return true;
    };
    if (alive && nblk > 0) alive = issue_S(0);
    for (int j = 0; j < nblk && alive; ++j) {
      if (j + 1 < nblk) alive = issue_S(j + 1);
      if (alive) alive = issue_PV(j);
    }
  } else if (warp < 4) {
    // V: bf16 -> f16 in place (exact for magnitudes in the f16 range).
    const int ct = threadIdx.x - 64;
    for (int j = 0; j < nblk; ++j) {
      const int s = j % kTcStages;
      if (!mbar_wait(&vfull[s], (j / kTcStages) & 1, status, abort)) break;
      uint4* v4 = reinterpret_cast<uint4*>(sStage + s * TcLayout::kStage + TcLayout::kKV);
#pragma unroll 4
      for (int i = ct; i < TcLayout::kKV / 16; i += 64) {
        uint4 x = v4[i];
        x.x = bf16x2_to_f16x2(x.x);
        x.y = bf16x2_to_f16x2(x.y);
        x.z = bf16x2_to_f16x2(x.z);
        x.w = bf16x2_to_f16x2(x.w);
        v4[i] = x;
      }
      fence_proxy_async_smem();
      mbar_arrive(&vready[s]);
    }
  } else {
    // Softmax: thread (half, r) owns keys [32 half, 32 half + 32) of row r
    // (TMEM lane r) and columns [64 half, 64 half + 64) of its O row.
    const int half = (warp - 4) / 4;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + TcLayout::kOffRed);
    float m_run = -FLT_MAX, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk && ok; ++j) {
      const int bb = j & 1;
      if (!(ok = mbar_wait(&sfull[bb], (j >> 1) & 1, status, abort))) break;
      tc_fence_after();
      float sv[32];
      tmem_ld32(tmem + lane_base + bb * 64 + half * 32, sv);
      tc_fence_before();
      mbar_arrive(&sfree[bb]);
      const int kb = k_begin + j * kTcKeys + half * 32;
      if (kb + 32 > k_end) {  // keys past the end of the chunk do not exist
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (kb + c >= k_end) sv[c] = -FLT_MAX;
      }
      float mx;
      {
        float t16[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) t16[c] = fmaxf(sv[c], sv[c + 16]);
#pragma unroll
        for (int w = 8; w > 0; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) t16[c] = fmaxf(t16[c], t16[c + w]);
        mx = t16[0];
      }
      // Exchange with the other half of the row.  red[parity] is written again two
      // blocks later, after every thread has arrived for block j + 1, i.e. after
      // every thread has read it for block j.
      float* rp = red + bb * 256;
      rp[half * 128 + r] = mx;
      mbar_arrive(&xmax[bb]);
      if (!(ok = mbar_wait(&xmax[bb], (j >> 1) & 1, status, abort))) break;
      mx = fmaxf(mx, rp[(half ^ 1) * 128 + r]) * scale_log2;  // scale_log2 > 0
      // P buffer bb was last read by P.V of block j - 2
      if (j >= 2 && !(ok = mbar_wait(&pdone[bb], ((j - 2) >> 1) & 1, status, abort))) break;
      if (j == 0) {
        m_run = mx;
      } else {
        const bool need = mx > m_run + kLazyRescale;
        if (__any_sync(0xffffffffu, need)) {
          // O must hold P.V of block j - 1 before it is rescaled
          if (!(ok = mbar_wait(&pdone[bb ^ 1], ((j - 1) >> 1) & 1, status, abort))) break;
          tc_fence_after();
          const float corr = need ? ex2(m_run - mx) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            float o[32];
            const uint32_t ta = tmem + lane_base + 128 + half * 64 + c * 32;
            tmem_ld32(ta, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= corr;
            tmem_st32(ta, o);
          }
          tmem_wait_st();
          if (need) {
            l_run *= corr;
            m_run = mx;
          }
        }
      }
      const float nm = -m_run;
      uint8_t* prow = sP + 2 * bb * TcLayout::kP + r * 128;
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2(fmaf(sv[c8 * 8 + 2 * e], scale_log2, nm));
          const float p1 = ex2(fmaf(sv[c8 * 8 + 2 * e + 1], scale_log2, nm));
          rs[e] += p0 + p1;
          hw[e] = pack_f16(p0, p1);
          const __half2 hh = *reinterpret_cast<const __half2*>(&hw[e]);
          lw[e] = pack_f16(p0 - __low2float(hh), p1 - __high2float(hh));
        }
        const int off = ((half * 4 + c8) ^ (r & 7)) << 4;
        *reinterpret_cast<uint4*>(prow + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(prow + TcLayout::kP + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&pready[bb]);
    }
    // Row sum = both halves' partial sums, exchanged in the buffer of parity
    // nblk & 1: every thread read it for block nblk - 2 before arriving for
    // block nblk - 1, which this thread waited for.
    if (ok) {
      float* rs_x = red + (nblk & 1) * 256;
      rs_x[half * 128 + r] = l_run;
      mbar_arrive(xsum);
      ok = mbar_wait(xsum, 0, status, abort);
      if (ok) l_run += rs_x[(half ^ 1) * 128 + r];
    }
    if (ok && nblk > 0 && mbar_wait(&pdone[(nblk - 1) & 1], ((nblk - 1) >> 1) & 1, status, abort)) {
      tc_fence_after();
      const int ridx = row0 + r;
      const bool valid = ridx < R;
      const int h = g * grp + ridx / a.C, i = ridx % a.C;
      const int nsplit = gridDim.x / nqt;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const int col = half * 64 + c * 32;
        float o[32];
        tmem_ld32(tmem + lane_base + 128 + col, o);
        if (!valid) continue;
        if (nsplit == 1) {
          const float inv = 1.0f / l_run;
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                                ((size_t)b * a.C + i) * ((size_t)a.Hq * kTcHD) +
                                                (size_t)h * kTcHD + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16(o[8 * q + 0] * inv, o[8 * q + 1] * inv);
            w.y = pack_bf16(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            w.z = pack_bf16(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            w.w = pack_bf16(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            dst[q] = w;
          }
        } else {
          const size_t rowid = (((size_t)split * a.B + b) * a.Hq + h) * a.C + i;
          float4* dst = reinterpret_cast<float4*>(a.opart + rowid * kTcHD + col);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          if (c == 0 && half == 0) *reinterpret_cast<float2*>(a.ml + rowid * 2) = make_float2(m_run, l_run);
        }
      }
    }
  }
  __syncthreads();
  if (*abort) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

bool attn_use_tc(const dg_dims& D, int P) { return D.hd == kTcHD && P % kTcKeys == 0; }

void attn_split_tc(const dg_dims& D, int T, int* nsplit, int* keys_per_split) {
  const int grp = D.Hq / D.Hkv;
  const int units = cdiv((int64_t)grp * D.C, 128) * D.B * D.Hkv;
  int ns = kTargetCtas / units;  // at most one wave (one CTA per SM)
  if (ns > cdiv(T, 256)) ns = cdiv(T, 256);
  if (ns > kMaxAttnSplits) ns = kMaxAttnSplits;
  if (ns < 1) ns = 1;
  const int kps = cdiv(cdiv(T, ns), kTcKeys) * kTcKeys;
  *keys_per_split = kps;
  *nsplit = cdiv(T, kps);
}

cudaError_t launch_attention_tc(const AttnArgs& a, StopCtl ctl, int* status, cudaStream_t st) {
  dg_dims D{};
  D.B = a.B;
  D.C = a.C;
  D.Hq = a.Hq;
  D.Hkv = a.Hkv;
  D.hd = a.hd;
  const int T = a.P + a.C;
  int ns, kps;
  attn_split_tc(D, T, &ns, &kps);
  const int nqt = cdiv((int64_t)(a.Hq / a.Hkv) * a.C, 128);
  CUtensorMap mQ, mKp, mVp, mKc, mVc;
  if (!make_tmap_2d(&mQ, a.q, kTcHD, (uint64_t)a.B * a.Hq * a.C, kTcHD * 2, 64, 128) ||
      !make_tmap_2d(&mKp, a.Kp, kTcHD, (uint64_t)a.B * a.Hkv * a.cap, kTcHD * 2, 64, kTcKeys) ||
      !make_tmap_2d(&mVp, a.Vp, kTcHD, (uint64_t)a.B * a.Hkv * a.cap, kTcHD * 2, 64, kTcKeys) ||
      !make_tmap_2d(&mKc, a.kc, kTcHD, (uint64_t)a.B * a.Hkv * a.C, kTcHD * 2, 64, kTcKeys) ||
      !make_tmap_2d(&mVc, a.vc, kTcHD, (uint64_t)a.B * a.Hkv * a.C, kTcHD * 2, 64, kTcKeys))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once<attn_tc_kernel>(TcLayout::kSmem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kTcHD);
  dim3 grid(nqt * ns, a.B * a.Hkv);
  attn_tc_kernel<<<grid, kTcThreads, TcLayout::kSmem, st>>>(mQ, mKp, mVp, mKc, mVc, a, nqt, kps, scale_log2,
                                                             status, ctl);
  e = cudaGetLastError();
  if (e != cudaSuccess || ns == 1) return e;
  return launch_attention_combine(a, ns, ctl, st);
}

}  // namespace dg
