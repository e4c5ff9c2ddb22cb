// Tensor-core (tcgen05 + TMA) attention of the canvas queries over
// [prefix cache ; canvas] with no mask, for head dim 128 ("DiffusionGemma"
// docs chapter, attention-mask list: the canvas is a full bidirectional
// matrix that reads the prompt / finished-block KV cache).
//
// One CTA owns two tiles of 128 query rows (of the rows of the group's query
// heads) of one (canvas, kv head) and one chunk of the key sequence, so each
// K/V block it streams serves 256 queries.  Warp roles:
//   warp 0      TMA: both Q tiles once, then K and V blocks of 128 keys into a
//               2-stage ring;
//   warp 1      MMA: S_t = Q_t K^T into TMEM (A and B from shared memory),
//               and O_t += P_t V with P_t read from TMEM;
//   warps 2-5   softmax of tile 0, warps 6-9 softmax of tile 1: one thread
//               per query row (its TMEM lane), base-2 online softmax with
//               lazy rescaling of O (only when the row maximum grows by more
//               than 2^8).  P is written back over S in TMEM as two bf16
//               parts, P = P_hi + P_lo, and O accumulates P_hi.V + P_lo.V, so
//               the probabilities enter the product to ~2^-16.
// The MMA warp interleaves the tiles (S_0, S_1, P_0.V, next S_0, P_1.V, next
// S_1, ...), so one tile's softmax runs while the tensor core works on the
// other.  Several key chunks per row are merged by attn_combine_kernel.
#include <cfloat>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

constexpr int kTcHD = 128;
constexpr int kTcKeys = 128;  // keys per block
constexpr int kTcStages = 2;
constexpr int kTcThreads = 320;
constexpr float kLazyRescale = 8.0f;  // log2 units

struct TcLayout {
  static constexpr int kQ = 128 * kTcHD * 2;       // 32 KB per query tile: two boxes of 64 columns
  static constexpr int kBox = kTcKeys * 128;       // 64 columns of one block (128 B per key)
  static constexpr int kKV = kTcKeys * kTcHD * 2;  // 32 KB: K or V of one block, two boxes
  static constexpr int kStage = 2 * kKV;           // K then V
  static constexpr int kOffStage = 2 * kQ;
  static constexpr int kOffBar = kOffStage + kTcStages * kStage;
  // No alignment slack: the kernel checks that dynamic shared memory starts on
  // a 1024-byte boundary (it does when the kernel has no static shared memory).
  static constexpr int kSmem = kOffBar + 256;
};
// TMEM columns: S_t (fp32, 128 keys) at 128 t, overwritten by P_t as bf16
// pairs (P_hi in its first 64 columns, P_lo in the last 64); O_t at 256 + 128 t.
constexpr int kColO = 2 * kTcKeys;

DG_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKp,
                   const __grid_constant__ CUtensorMap mVp, const __grid_constant__ CUtensorMap mKc,
                   const __grid_constant__ CUtensorMap mVc, AttnArgs a, int npair, int kps,
                   float scale_log2, int* status, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // uniform over the CTA: return before any barrier
    if (threadIdx.x == 0) atomicExch(status, kStatusTimeout);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem;  // [2 tiles]
  uint8_t* sStage = smem + TcLayout::kOffStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TcLayout::kOffBar);
  uint64_t* qfull = bars;
  uint64_t* kvfull = bars + 1;             // [stages]
  uint64_t* kvempty = kvfull + kTcStages;  // [stages]
  uint64_t* sfull = kvempty + kTcStages;   // [2 tiles]: S_t of the current block is in TMEM
  uint64_t* pready = sfull + 2;            // [2 tiles][2 halves]: P_t of 64 keys written (128 threads)
  uint64_t* pvdone = pready + 4;           // [2]: O_t += P_t V of the block completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pvdone + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int pr = blockIdx.x % npair, split = blockIdx.x / npair;
  const int b = blockIdx.y / a.Hkv, g = blockIdx.y % a.Hkv;
  const int grp = a.Hq / a.Hkv;
  const int R = grp * a.C;  // query rows of the group
  const int row0 = pr * 256;
  const int T = a.P + a.C;
  const int k_begin = split * kps;
  const int k_end = min(T, k_begin + kps);
  const int nblk = (k_end - k_begin + kTcKeys - 1) / kTcKeys;

  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sfull[t], 1);
      mbar_init(&pready[2 * t], 128);
      mbar_init(&pready[2 * t + 1], 128);
      mbar_init(&pvdone[t], 1);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch(&mQ);
      tma_prefetch(&mKp);
      tma_prefetch(&mVp);
      const int qrow = (b * a.Hq + g * grp) * a.C + row0;
      mbar_arrive_expect_tx(qfull, 2 * TcLayout::kQ);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        tma_load_2d(sQ + t * TcLayout::kQ, &mQ, qfull, 0, qrow + 128 * t);
        tma_load_2d(sQ + t * TcLayout::kQ + 16384, &mQ, qfull, 64, qrow + 128 * t);
      }
      for (int j = 0; j < nblk; ++j) {
        const int s = j % kTcStages;
        if (!mbar_wait(&kvempty[s], ((j / kTcStages) & 1) ^ 1, status, abort)) break;
        const int kj = k_begin + j * kTcKeys;
        const bool pre = kj < a.P;  // blocks never straddle P (P is a multiple of the block)
        const CUtensorMap* mk = pre ? &mKp : &mKc;
        const CUtensorMap* mv = pre ? &mVp : &mVc;
        const int row = pre ? (b * a.Hkv + g) * a.cap + kj : (b * a.Hkv + g) * a.C + (kj - a.P);
        uint8_t* sk = sStage + s * TcLayout::kStage;
        uint8_t* sv = sk + TcLayout::kKV;
        mbar_arrive_expect_tx(&kvfull[s], TcLayout::kStage);
        tma_load_2d(sk, mk, &kvfull[s], 0, row);
        tma_load_2d(sk + TcLayout::kBox, mk, &kvfull[s], 64, row);
        tma_load_2d(sv, mv, &kvfull[s], 0, row);
        tma_load_2d(sv + TcLayout::kBox, mv, &kvfull[s], 64, row);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // one thread waits and issues; the MMAs need no other lane
      constexpr uint32_t idS = idesc_bf16(128, kTcKeys, false);
      constexpr uint32_t idPV = idesc_bf16(128, kTcHD, true);
      bool alive = mbar_wait(qfull, 0, status, abort);
      const uint32_t sq = smem_u32(sQ);
      auto issue_S = [&](int t, int j) {
        const uint32_t sk = smem_u32(sStage + (j % kTcStages) * TcLayout::kStage);
#pragma unroll
        for (int kk = 0; kk < kTcHD / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(sq + t * TcLayout::kQ + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sk + (kk / 4) * TcLayout::kBox + (kk % 4) * 32, 16, 1024);
          umma_bf16(tmem + kTcKeys * t, ad, bd, idS, kk ? 1u : 0u);
        }
        umma_commit(&sfull[t]);
      };
      auto issue_PV = [&](int t, int j) -> bool {
        const uint32_t sv = smem_u32(sStage + (j % kTcStages) * TcLayout::kStage + TcLayout::kKV);
        // each half of the block's keys as soon as the softmax has written its P
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait(&pready[2 * t + hf], j & 1, status, abort)) return false;
          tc_fence_after();
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int k4 = 0; k4 < kTcKeys / 32; ++k4) {
              const int kk = hf * (kTcKeys / 32) + k4;
              const uint64_t bd = sdesc_sw128(sv + kk * 2048, TcLayout::kBox, 1024);
              umma_bf16_ts(tmem + kColO + 128 * t, tmem + kTcKeys * t + (kTcKeys / 2) * part + 8 * kk, bd, idPV,
                           (j > 0 || hf > 0 || part > 0 || k4 > 0) ? 1u : 0u);
            }
          }
        }
        umma_commit(&pvdone[t]);
        if (t == 1) umma_commit(&kvempty[j % kTcStages]);
        return true;
      };
      auto wait_kv = [&](int j) -> bool {
        if (!mbar_wait(&kvfull[j % kTcStages], (j / kTcStages) & 1, status, abort)) return false;
        tc_fence_after();
        return true;
      };
      if (alive && nblk > 0 && (alive = wait_kv(0))) {
        issue_S(0, 0);
        issue_S(1, 0);
      }
      for (int j = 0; j < nblk && alive; ++j) {
        // S_t of block j + 1 overwrites P_t of block j: it is issued after the
        // P_t.V that reads it, and the tensor core runs one thread's MMAs in order.
        if (!(alive = issue_PV(0, j))) break;
        if (j + 1 < nblk) {
          if (!(alive = wait_kv(j + 1))) break;
          issue_S(0, j + 1);
        }
        if (!(alive = issue_PV(1, j))) break;
        if (j + 1 < nblk) issue_S(1, j + 1);
      }
    }
    __syncwarp();
  } else {
    // Softmax of tile t: thread r owns query row r of the tile (TMEM lane r).
    const int t = (warp - 2) / 4;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_base + kTcKeys * t;
    const uint32_t tO = tmem + lane_base + kColO + 128 * t;
    float m_run = -FLT_MAX, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk && ok; ++j) {
      if (!(ok = mbar_wait_warp(&sfull[t], j & 1, status, abort))) break;
      tc_fence_after();
      float sv[kTcKeys];
#pragma unroll
      for (int c = 0; c < kTcKeys / 32; ++c) tmem_ld32_async(tS + 32 * c, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
      tmem_wait_ld();
      const int kb = k_begin + j * kTcKeys;
      if (kb + kTcKeys > k_end) {  // keys past the end of the chunk do not exist
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c)
          if (kb + c >= k_end) sv[c] = -FLT_MAX;
      }
      float mx;
      {
        // 3-input maxima into four running values (two keys each per step)
        static_assert(kTcKeys % 8 == 0, "key block");
        float r4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
        for (int c = 4; c + 8 <= kTcKeys; c += 8) {
#pragma unroll
          for (int k = 0; k < 4; ++k) r4[k] = fmax3(r4[k], sv[c + 2 * k], sv[c + 2 * k + 1]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) r4[k] = fmaxf(r4[k], sv[kTcKeys - 4 + k]);
        mx = fmaxf(fmaxf(r4[0], r4[1]), fmaxf(r4[2], r4[3])) * scale_log2;  // scale_log2 > 0
      }
      if (j == 0) {
        m_run = mx;
      } else {
        const bool need = mx > m_run + kLazyRescale;
        if (__any_sync(0xffffffffu, need)) {
          // O_t must hold P_t.V of block j - 1 before it is rescaled
          if (!(ok = mbar_wait_warp(&pvdone[t], (j - 1) & 1, status, abort))) break;
          tc_fence_after();
          const float corr = need ? ex2(m_run - mx) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < kTcHD / 16; ++c) {  // 16 columns at a time: S is still live
            uint32_t o[16];
            tmem_ld16(tO + 16 * c, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st16(tO + 16 * c, o);
          }
          if (need) {
            l_run *= corr;
            m_run = mx;
          }
        }
      }
      // p = 2^(s * scale - m) two keys at a time (paired fp32 FMA / add / sub)
      const uint64_t scale2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_run, -m_run);
      uint64_t rs2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < kTcKeys / 32; ++c) {  // 32 keys: 16 columns of P_hi and of P_lo
        uint32_t hw[16], lw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(sv[32 * c + 2 * e], sv[32 * c + 2 * e + 1]), scale2, nm2), t0, t1);
          const float p0 = ex2(t0), p1 = ex2(t1);
          const uint64_t p2 = f2_pack(p0, p1);
          rs2[e & 1] = f2_add(rs2[e & 1], p2);
          hw[e] = pack_bf16(p0, p1);
          float l0, l1;
          f2_unpack(f2_sub(p2, f2_pack(__uint_as_float(hw[e] << 16), __uint_as_float(hw[e] & 0xffff0000u))), l0, l1);
          lw[e] = pack_bf16(l0, l1);
        }
        tmem_st16(tS + 16 * c, hw);
        tmem_st16(tS + kTcKeys / 2 + 16 * c, lw);
        if (c % 2 == 1) {  // a half of the keys is written: its P.V may start
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&pready[2 * t + c / 2]);
        }
      }
      {
        float a0, a1, b0, b1;
        f2_unpack(rs2[0], a0, a1);
        f2_unpack(rs2[1], b0, b1);
        l_run += (a0 + a1) + (b0 + b1);
      }
    }
    if (ok && nblk > 0 && mbar_wait_warp(&pvdone[t], (nblk - 1) & 1, status, abort)) {
      tc_fence_after();
      const int ridx = row0 + 128 * t + r;
      const bool valid = ridx < R;
      const int h = g * grp + ridx / a.C, i = ridx % a.C;
      const int nsplit = gridDim.x / npair;
#pragma unroll 1
      for (int c = 0; c < kTcHD / 32; ++c) {
        const int col = 32 * c;
        float o[32];
        tmem_ld32(tO + col, o);
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
          if (c == 0) *reinterpret_cast<float2*>(a.ml + rowid * 2) = make_float2(m_run, l_run);
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
    tmem_dealloc(tmem, 512);
  }
}

bool attn_use_tc(const dg_dims& D, int P) { return D.hd == kTcHD && P % kTcKeys == 0; }

void attn_split_tc(const dg_dims& D, int T, int* nsplit, int* keys_per_split) {
  const int grp = D.Hq / D.Hkv;
  const int units = cdiv(cdiv((int64_t)grp * D.C, 128), 2) * D.B * D.Hkv;  // CTAs per key chunk
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
  const int npair = cdiv(cdiv((int64_t)(a.Hq / a.Hkv) * a.C, 128), 2);
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
  dim3 grid(npair * ns, a.B * a.Hkv);
  e = launch_pdl(attn_tc_kernel, grid, dim3(kTcThreads), TcLayout::kSmem, st, mQ, mKp, mVp, mKc, mVc, a, npair,
                 kps, scale_log2, status, ctl);
  if (e != cudaSuccess || ns == 1) return e;
  return launch_attention_combine(a, ns, ctl, st);
}

}  // namespace dg
