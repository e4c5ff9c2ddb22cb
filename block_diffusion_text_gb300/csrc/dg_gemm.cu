// Tensor-core (tcgen05 + TMA + mbarrier) GEMM engine of libdg and the fused
// kernels built on it:
//   * gemm_kernel: D = A B^T with A [M][K], B [N][K] (or [K][N]) bf16, fp32
//     accumulation in TMEM, warp-specialised (TMA producer warp, MMA warp,
//     four epilogue warps), persistent over output tiles with a
//     double-buffered TMEM accumulator.  Epilogues: fp32 store (diagnostics),
//     bf16 store with residual / GELU (output projection, FFW), RoPE
//     projections (q, k, v), and the LM head statistics epilogue.
//   * gemm_ksum_kernel: the same engine split over K across a cluster of 2 or
//     4 CTAs, the slices summed in the owning CTA's shared memory before the
//     epilogue (the q, k, v projections and FFW1 at C = 256).
//   * gemm_pair_kernel: the same engine on CTA pairs (M = 256 MMAs over two
//     SMs), for the two vocabulary-sized products: the LM head and the
//     self-conditioning contraction u = p0 . E (the LM head's stored tiles
//     as A, one p0 factor per row applied in the reduce, E as the MN-major B
//     operand, split over the vocabulary).
#include <cfloat>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

constexpr int kBM = 128;  // rows per MMA (one TMEM lane per row)
constexpr int kBK = 64;   // bf16 elements per 128-byte swizzled row
constexpr int kGemmThreads = 192;

DG_DEV uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// If a role gave up (timeout), sleep long enough for copies and MMAs it may
// have left in flight to land before the CTA releases TMEM and exits.
DG_DEV void drain_if_aborted(volatile int* abort) {
  if (*abort) {
    uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
  }
}

// 256-bit global store of w[o .. o+7] (the address 32-byte aligned).
DG_DEV void st_global_v8(uint32_t* p, const uint32_t (&w)[16], int o) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[o]), "r"(w[o + 1]),
               "r"(w[o + 2]), "r"(w[o + 3]), "r"(w[o + 4]), "r"(w[o + 5]), "r"(w[o + 6]), "r"(w[o + 7])
               : "memory");
}

// ================================================================ epilogues
struct EpiF32 {
  float* out;
  int ldo;
  template <int BN, class LD>
  DG_DEV void tile(int row, bool ok, int n0, int N, LD& ld, int /*split*/) const {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      ld(c, v);
      if (!ok) continue;
      int col0 = n0 + c * 32;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < N) out[(size_t)row * ldo + col0 + j] = v[j];
    }
  }
};

// Split-K partial: the fp32 tile of one K-split, reduced by splitk_*_kernel.
struct EpiPartial {
  float* part;  // [ksplit][M][N]
  int M, N;
  template <int BN, class LD>
  DG_DEV void tile(int row, bool ok, int n0, int N_, LD& ld, int split) const {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      ld(c, v);
      const int col0 = n0 + c * 32;
      if (!ok || col0 >= N) continue;
      float* dst = part + ((size_t)split * M + row) * N + col0;
      if (col0 + 32 <= N) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          reinterpret_cast<float4*>(dst)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      } else {
        for (int j = 0; j < 32; ++j)
          if (col0 + j < N) dst[j] = v[j];
      }
    }
  }
};

struct EpiBF16 {
  __nv_bfloat16* out;
  int ldo;
  const __nv_bfloat16* resid;
  int ldr;
  int gelu;
  int C;
  StopCtl ctl;
  template <int BN, class LD>
  DG_DEV void tile(int row, bool ok, int n0, int N, LD& ld, int /*split*/) const {
    const bool active = ok && canvas_active(ctl.stop_at, row / C, ctl.step);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      ld(c, v);
      if (!active) continue;
      const int col0 = n0 + c * 32;
      if (resid) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          if (col0 + j + 8 <= N) {
            uint4 r = *reinterpret_cast<const uint4*>(resid + (size_t)row * ldr + col0 + j);
            const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(&r);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[j + e] += __bfloat162float(rb[e]);
          }
        }
      }
      if (gelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.5f * v[j] * (1.0f + erff(v[j] * 0.70710678118654752f));
      }
      if (col0 + 32 <= N) {
        uint4* dst = reinterpret_cast<uint4*>(out + (size_t)row * ldo + col0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 w;
          w.x = pack_bf16(v[8 * j + 0], v[8 * j + 1]);
          w.y = pack_bf16(v[8 * j + 2], v[8 * j + 3]);
          w.z = pack_bf16(v[8 * j + 4], v[8 * j + 5]);
          w.w = pack_bf16(v[8 * j + 6], v[8 * j + 7]);
          dst[j] = w;
        }
      } else {
        for (int j = 0; j < 32; ++j)
          if (col0 + j < N) out[(size_t)row * ldo + col0 + j] = __float2bfloat16_rn(v[j]);
      }
    }
  }
};

// q, k, v projections with RoPE on q and k.  One 128-column tile covers
// 128 / HD whole heads, so both halves of every rotated pair are in the
// thread's registers.
template <int HD>
struct EpiQKV {
  __nv_bfloat16 *q, *k, *v;
  const float2* rope;  // [C][HD/2] (cos, sin) of positions P + i
  int C, Hq, Hkv, nq, nkv, kv_rows, kv_row0;
  template <int BN, class LD>
  DG_DEV void tile(int row, bool ok, int n0, int N, LD& ld, int /*split*/) const {
    static_assert(BN % HD == 0, "tile must hold whole heads");
    float x[BN];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      float t[32];
      ld(c, t);
#pragma unroll
      for (int j = 0; j < 32; ++j) x[c * 32 + j] = t[j];
    }
    if (!ok) return;
    const int b = row / C, i = row % C;
#pragma unroll
    for (int hh = 0; hh < BN / HD; ++hh) {
      const int col0 = n0 + hh * HD;
      if (col0 >= N) break;
      const bool is_q = col0 < nq;
      const bool is_k = !is_q && col0 < nq + nkv;
      float* xv = x + hh * HD;
      if (is_q || is_k) {
        const float2* cs = rope + (size_t)i * (HD / 2);
#pragma unroll
        for (int j = 0; j < HD / 2; ++j) {
          float2 r = cs[j];
          float a0 = xv[j], a1 = xv[j + HD / 2];
          xv[j] = a0 * r.x - a1 * r.y;
          xv[j + HD / 2] = a0 * r.y + a1 * r.x;
        }
      }
      __nv_bfloat16* dst;
      if (is_q) {
        dst = q + (((size_t)b * Hq + col0 / HD) * C + i) * HD;
      } else {
        const int head = (col0 - nq - (is_k ? 0 : nkv)) / HD;
        dst = (is_k ? k : v) + (((size_t)b * Hkv + head) * kv_rows + kv_row0 + i) * HD;
      }
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int j = 0; j < HD / 8; ++j) {
        uint4 w;
        w.x = pack_bf16(xv[8 * j + 0], xv[8 * j + 1]);
        w.y = pack_bf16(xv[8 * j + 2], xv[8 * j + 3]);
        w.z = pack_bf16(xv[8 * j + 4], xv[8 * j + 5]);
        w.w = pack_bf16(xv[8 * j + 6], xv[8 * j + 7]);
        d4[j] = w;
      }
    }
  }
};

// LM head: l = alpha h.E / sqrt d, s = l / tau.  Per (row, 128-column group):
// m_g = max s (kept in log2 units), l_g = sum exp(s - m_g), S_g = sum
// exp(s - m_g) (s - m_g) log2 e, and the argmax of h.E (lowest column on
// ties); the tile values are stored as bf16 for the self-conditioning pass,
// exp(s - R) for the row's reference R (kRefSpan).
struct EpiLM {
  const float* alpha;
  float coef2;  // log2(e) / (sqrt(d) tau)
  float inv_sqrt_d;
  __nv_bfloat16* pt;
  GroupStat* gst;
  float* logits;
  int M, V;
  int excl;  // vocabulary column left out of the softmax (the [MASK] token), or -1
  const float* rowscale;  // FP8 head: per-row scale of h (else null)
  const float* colscale;  // FP8 head: per-row scale of E, i.e. per column of the tile (else null)
  const float* ref2;      // per-row storage reference R (log2 units)
  unsigned* rkey;         // raised to the key of a group maximum stored against itself
  // The accumulator of column col, scaled for the FP8 head.
  DG_DEV void scale_cols(float (&v)[32], int col0, int N) const {
    if (!colscale) return;
    if (col0 + 32 <= N) {  // 16-byte aligned (col0 is a multiple of 32)
      const float4* s4 = reinterpret_cast<const float4*>(colscale + col0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 sc = __ldg(s4 + j);
        v[4 * j] *= sc.x;
        v[4 * j + 1] *= sc.y;
        v[4 * j + 2] *= sc.z;
        v[4 * j + 3] *= sc.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= __ldg(colscale + (col0 + j < N ? col0 + j : N - 1));
    }
  }
  // Statistics per group of kStatCols columns, so that a tile may be 128 or
  // 256 columns wide.  The maximum / argmax scan and the two sums each run as
  // four independent chains (columns j mod 4, pairs (j / 2) mod 4) merged at
  // the end of the group, so that one thread's dependent adds and compares
  // overlap; chunks wholly inside the vocabulary and clear of the excluded
  // column skip the per-column tests.
  template <int BN, class LD>
  DG_DEV void tile(int row, bool ok, int n0, int N, LD& ld, int /*split*/) const {
    static_assert(BN % kStatCols == 0, "a tile holds whole statistics groups");
    const float al = (ok ? __ldg(alpha + row) : 1.0f) * (rowscale && ok ? __ldg(rowscale + row) : 1.0f);
    const float c2 = al * coef2;
    const float R2 = ok ? __ldg(ref2 + row) : 0.f;
    const int NT = (V + kStatCols - 1) / kStatCols;
#pragma unroll 1
    for (int g = 0; g < BN / kStatCols; ++g) {
      const int g0 = n0 + g * kStatCols;
      if (g0 >= N) break;  // uniform over the warp
      float vm[4] = {-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX};
      int im[4] = {g0, g0, g0, g0};
#pragma unroll 1
      for (int c = 0; c < kStatCols / 32; ++c) {
        float v[32];
        ld(g * (kStatCols / 32) + c, v);
        const int col0 = g0 + c * 32;
        scale_cols(v, col0, N);
        if (col0 + 32 <= N && (excl < col0 || excl >= col0 + 32)) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (v[j] > vm[j & 3]) {
              vm[j & 3] = v[j];
              im[j & 3] = col0 + j;
            }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = col0 + j;
            if (col < N && col != excl && v[j] > vm[j & 3]) {
              vm[j & 3] = v[j];
              im[j & 3] = col;
            }
          }
        }
      }
      // the chains' first maxima, ties to the lowest column
      float vmax = vm[0];
      int imax = im[0];
#pragma unroll
      for (int k = 1; k < 4; ++k)
        if (vm[k] > vmax || (vm[k] == vmax && im[k] < imax)) {
          vmax = vm[k];
          imax = im[k];
        }
      const float m2 = vmax * c2;
      // stored values exp2(t - R2) = p * exp2(m2 - R2), unless they would
      // overflow (then p itself, row flagged)
      const bool own = !(m2 - R2 <= kRefSpan);
      const float F = own ? 1.0f : exp2f(m2 - R2);
      if (own && ok) atomicMax(rkey + row, float_key(m2));
      float l4[4] = {0.f, 0.f, 0.f, 0.f}, S4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int c = 0; c < kStatCols / 32; ++c) {
        float v[32];
        ld(g * (kStatCols / 32) + c, v);
        const int col0 = g0 + c * 32;
        scale_cols(v, col0, N);
        const bool full = col0 + 32 <= N && (excl < col0 || excl >= col0 + 32);
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float t0 = fmaf(v[j], c2, -m2), t1 = fmaf(v[j + 1], c2, -m2);
          float p0 = exp2f(t0), p1 = exp2f(t1);
          if (!full) {
            if (col0 + j >= N || col0 + j == excl) p0 = 0.f;
            if (col0 + j + 1 >= N || col0 + j + 1 == excl) p1 = 0.f;
          }
          const int k = (j / 2) & 3;
          l4[k] += p0 + p1;
          S4[k] = fmaf(p0, t0, fmaf(p1, t1, S4[k]));
          pk[j / 2] = pack_bf16(p0 * F, p1 * F);
        }
        if (ok) {
          if (col0 + 32 <= N && V % 16 == 0) {
            // rows 32-byte aligned: two 256-bit stores (half the L1 wavefronts of
            // four 128-bit ones, each lane of the warp writing another row)
            uint32_t* dst = reinterpret_cast<uint32_t*>(pt + (size_t)row * V + col0);
            st_global_v8(dst, pk, 0);
            st_global_v8(dst + 8, pk, 8);
          } else if (col0 + 32 <= N) {
            uint4* dst = reinterpret_cast<uint4*>(pt + (size_t)row * V + col0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          } else {
            const __nv_bfloat16* pb = reinterpret_cast<const __nv_bfloat16*>(pk);
            for (int j = 0; j < 32; ++j)
              if (col0 + j < N) pt[(size_t)row * V + col0 + j] = pb[j];
          }
          if (logits) {
            const float cl = al * inv_sqrt_d;
            for (int j = 0; j < 32; ++j)
              if (col0 + j < N) logits[(size_t)row * V + col0 + j] = v[j] * cl;
          }
        }
      }
      const float l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
      const float S = (S4[0] + S4[1]) + (S4[2] + S4[3]);
      if (ok) {  // one 32-byte record: a whole sector per lane
        uint32_t rec[16];
        rec[0] = __float_as_uint(m2);
        rec[1] = __float_as_uint(l);
        rec[2] = __float_as_uint(S);
        rec[3] = __float_as_uint(vmax);
        rec[4] = (uint32_t)imax;
        rec[5] = rec[6] = rec[7] = 0u;
        st_global_v8(reinterpret_cast<uint32_t*>(gst + (size_t)row * NT + g0 / kStatCols), rec, 0);
      }
    }
  }
};

// ============================================================ GEMM kernel
template <int BN, int STAGES, bool B_MN>
struct GemmLayout {
  static constexpr int kA = kBM * kBK * 2;
  static constexpr int kB = BN * kBK * 2;
  static constexpr int kStage = kA + kB;
  static constexpr int kBar = STAGES * kStage;
  static constexpr int kSmem = kBar + 256 + 1024;
};

// B rows [0, nb0) come from mB0, [nb0, nb0 + nb1) from mB1, the rest from mB2
// (used to run the q, k, v projections as one GEMM over three weights).  A
// K-major B tile is loaded as BN / b_sub boxes of b_sub rows, each from the
// map that holds its rows (b_sub divides nb0 and nb1).
template <int BN, int STAGES, bool B_MN, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                const __grid_constant__ CUtensorMap mB1, const __grid_constant__ CUtensorMap mB2,
                int nb0, int nb1, int b_sub, int M, int N, int K, int ksplit, uint32_t b_lbo,
                uint32_t b_sbo, Epi epi, int* status, StopCtl ctl) {
  using L = GemmLayout<BN, STAGES, B_MN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int num_m = (M + kBM - 1) / kBM, num_n = (N + BN - 1) / BN;
  const int num_mn = num_m * num_n;
  const int num_tiles = num_mn * ksplit;  // tile t: split t / num_mn, (m, n) from t % num_mn
  const int nk_all = (K + kBK - 1) / kBK;
  auto krange = [&](int tile, int& kb_lo, int& kb_hi) {
    const int sp = tile / num_mn;
    kb_lo = (int)((int64_t)sp * nk_all / ksplit);
    kb_hi = (int)((int64_t)(sp + 1) * nk_all / ksplit);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The prologue above overlaps the kernel before this one when that one
  // triggers its dependents early; its results are read only from here on.
  pdl_wait();
  if (!all_stopped(ctl.stop_at, ctl.B, ctl.step)) {
    if (warp == 0) {
      if (lane == 0) {
        tma_prefetch(&mA);
        tma_prefetch(&mB0);
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        for (int tile = blockIdx.x; tile < num_tiles && alive; tile += gridDim.x) {
          const int tmn = tile % num_mn;
          const int m0 = (tmn % num_m) * kBM, n0 = (tmn / num_m) * BN;
          int kb_lo, kb_hi;
          krange(tile, kb_lo, kb_hi);
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, status, abort)) {
              alive = false;
              break;
            }
            uint8_t* sa = smem + stage * L::kStage;
            uint8_t* sb = sa + L::kA;
            mbar_arrive_expect_tx(&full[stage], L::kStage);
            tma_load_2d(sa, &mA, &full[stage], kb * kBK, m0);
            if (!B_MN) {
              for (int r = 0; r < BN; r += b_sub) {
                const int n = n0 + r;
                const CUtensorMap* mb = &mB0;
                int nb = n;
                if (n >= nb0 + nb1) {
                  mb = &mB2;
                  nb = n - nb0 - nb1;
                } else if (n >= nb0) {
                  mb = &mB1;
                  nb = n - nb0;
                }
                tma_load_2d(sb + r * 128, mb, &full[stage], kb * kBK, nb);
              }
            } else {
  #pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(sb + j * (kBK * 128), &mB0, &full[stage], n0 + 64 * j, kb * kBK);
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {  // one thread waits and issues; the MMAs need no other lane
        constexpr uint32_t idesc = idesc_bf16(kBM, BN, B_MN);
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        int it = 0;
        for (int tile = blockIdx.x; tile < num_tiles && alive; tile += gridDim.x, ++it) {
          const int acc = it & 1;
          const uint32_t aph = (it >> 1) & 1;
          if (!mbar_wait(&tempty[acc], aph ^ 1, status, abort)) break;
          tc_fence_after();
          const uint32_t dt = tmem + acc * BN;
          int kb_lo, kb_hi;
          krange(tile, kb_lo, kb_hi);
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (!mbar_wait(&full[stage], phase, status, abort)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * L::kStage);
            const uint32_t sb = sa + L::kA;
  #pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc_sw128(sb + kk * 2048, b_lbo, b_sbo)
                                       : sdesc_sw128(sb + kk * 32, 16, 1024);
              umma_bf16(dt, ad, bd, idesc, (kb != kb_lo || kk != 0) ? 1u : 0u);
            }
            umma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (alive) umma_commit(&tfull[acc]);
        }
      }
      __syncwarp();
    } else {
      const int q = warp & 3;  // TMEM lane quarter this warp may read
      const int r_local = q * 32 + lane;
      int it = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_warp(&tfull[acc], aph, status, abort)) break;
        tc_fence_after();
        const int tmn = tile % num_mn;
        const int m0 = (tmn % num_m) * kBM, n0 = (tmn / num_m) * BN;
        const int row = m0 + r_local;
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
        auto ld = [&](int c, float(&v)[32]) { tmem_ld32(tb + c * 32, v); };
        epi.template tile<BN>(row, row < M, n0, N, ld, tile / num_mn);
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
      }
    }
  }
  __syncthreads();
  drain_if_aborted(abort);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
}

// ================================================= split-K over a cluster
// The KS CTAs of a cluster (cluster dims KS x 1 x 1) compute the KS K-slices
// of one output tile, CTA rank r the slice [r nk / KS, (r + 1) nk / KS) of the
// nk 64-wide K blocks.  The sum over the slices is taken in shared memory: the
// 32 rows of epilogue warp quarter q belong to rank q KS / 4, the other ranks
// store their partial sums of those rows into the owner's receive buffer
// (remote stores, then one release arrival per lane on the owner's barrier
// for quarter q), and the owner's warp adds them to its own accumulator and
// runs the epilogue.  No fp32 partials go through global memory and no
// second launch reduces them.  One tile per cluster; a cluster barrier at the
// end keeps every CTA resident until no peer can still store into it.
template <int BN, int STAGES, int KS>
struct KsumLayout {
  static_assert(KS == 2 || KS == 4, "a quarter of the tile's rows per owner warp");
  static constexpr int kA = kBM * kBK * 2;
  static constexpr int kB = BN * kBK * 2;
  static constexpr int kStage = kA + kB;
  static constexpr int kOwned = kBM / KS;  // rows kept by each rank
  static constexpr int kLd = BN + 4;       // floats per received row (padded against bank conflicts)
  static constexpr int kRecv = (KS - 1) * kOwned * kLd * 4;
  static constexpr int kBar = STAGES * kStage + kRecv;
  static constexpr int kSmem = kBar + 256 + 1024;
};

template <int BN, int STAGES, int KS, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_ksum_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                     const __grid_constant__ CUtensorMap mB1, const __grid_constant__ CUtensorMap mB2,
                     int nb0, int nb1, int b_sub, int M, int N, int K, Epi epi, int* status, StopCtl ctl) {
  using L = KsumLayout<BN, STAGES, KS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  float* recv = reinterpret_cast<float*>(smem + STAGES * L::kStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* rbar = tfull + 1;  // [4]: the other slices of quarter q have arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rbar + 4);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = (int)cluster_ctarank();
  const int tmn = (int)cluster_id_x();
  const int num_m = (M + kBM - 1) / kBM;
  const int m0 = (tmn % num_m) * kBM, n0 = (tmn / num_m) * BN;
  const int nk = (K + kBK - 1) / kBK;
  const int kb_lo = rank * nk / KS, kb_hi = (rank + 1) * nk / KS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&rbar[q], (KS - 1) * 32);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peers' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The prologue above overlaps the kernel before this one when that one
  // triggers its dependents early; its results are read only from here on.
  pdl_wait();
  if (!all_stopped(ctl.stop_at, ctl.B, ctl.step)) {
    if (warp == 0) {
      if (lane == 0) {
        tma_prefetch(&mA);
        tma_prefetch(&mB0);
        int stage = 0;
        uint32_t phase = 0;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, status, abort)) break;
          uint8_t* sa = smem + stage * L::kStage;
          uint8_t* sb = sa + L::kA;
          mbar_arrive_expect_tx(&full[stage], L::kStage);
          tma_load_2d(sa, &mA, &full[stage], kb * kBK, m0);
          for (int r = 0; r < BN; r += b_sub) {
            const int n = n0 + r;
            const CUtensorMap* mb = &mB0;
            int nb = n;
            if (n >= nb0 + nb1) {
              mb = &mB2;
              nb = n - nb0 - nb1;
            } else if (n >= nb0) {
              mb = &mB1;
              nb = n - nb0;
            }
            tma_load_2d(sb + r * 128, mb, &full[stage], kb * kBK, nb);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16(kBM, BN, false);
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(&full[stage], phase, status, abort)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * L::kStage);
          const uint32_t sb = sa + L::kA;
  #pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sb + kk * 32, 16, 1024);
            umma_bf16(tmem, ad, bd, idesc, (kb != kb_lo || kk != 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (alive) umma_commit(tfull);
      }
      __syncwarp();
    } else {
      const int q = warp & 3;  // TMEM lane quarter this warp may read
      const int r_local = q * 32 + lane;
      const int owner = q * KS / 4;
      const int lr = r_local - owner * L::kOwned;  // row within the owner's block
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16);
      if (mbar_wait_warp(tfull, 0, status, abort)) {
        tc_fence_after();
        if (owner != rank) {
          const int slot = rank < owner ? rank : rank - 1;
          const uint32_t dst = cluster_addr(recv + ((size_t)slot * L::kOwned + lr) * L::kLd, (uint32_t)owner);
  #pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(tb + c * 32, v);
  #pragma unroll
            for (int j = 0; j < 8; ++j)
              st_cluster_v4(dst + (uint32_t)((c * 32 + 4 * j) * 4), v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
          mbar_arrive_cluster_release(cluster_addr(&rbar[q], (uint32_t)owner));
        } else if (mbar_wait_warp<true>(&rbar[q], 0, status, abort)) {
          const float* own = recv + (size_t)lr * L::kLd;
          auto ld = [&](int c, float(&v)[32]) {
            tmem_ld32(tb + c * 32, v);
  #pragma unroll
            for (int s = 0; s < KS - 1; ++s) {
              const float4* src = reinterpret_cast<const float4*>(own + (size_t)s * L::kOwned * L::kLd + c * 32);
  #pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 x = src[j];
                v[4 * j] += x.x;
                v[4 * j + 1] += x.y;
                v[4 * j + 2] += x.z;
                v[4 * j + 3] += x.w;
              }
            }
          };
          const int row = m0 + r_local;
          epi.template tile<BN>(row, row < M, n0, N, ld, 0);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync();  // no CTA leaves while a peer may still store into its shared memory
  drain_if_aborted(abort);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

// ============================================================ grouped GEMM
// The MoE expert products, D^T = W x^T per expert: A = the experts' matrices
// stacked [groups * b_rows][K] (M = 128 output features of one expert per
// tile), B = a tile of that expert's rows of the expert-sorted input [R][K]
// (N = kMoeTileRows rows).  An expert gets few rows at C = 256 (top 8 of 128:
// ~24 each), so the rows are the narrow side: a 128-row tile of them would be
// mostly padding in the MMA and in the operand loads.  The tile table
// (written on the device by the routing plan) holds the count in tiles[0].x
// and, per tile, (expert, first row, rows) in tiles[1 + t]; output tile
// (t, n) is rows [first, first + rows) x features [n, n + 128).  Tiles run
// n-major, so the row tiles of one expert, which share its weight tiles, run
// side by side.  TMEM lane f of the accumulator holds feature n + f for the
// tile's rows (its columns); the epilogue stores one row at a time, the lanes
// of a warp writing consecutive features.
struct EpiMoeUp {  // expert hidden: bf16(GELU(acc))
  __nv_bfloat16* gp;
  int ldo;
  DG_DEV void store(int feat, int first, int rows, const float (&v)[kMoeTileRows]) const {
#pragma unroll
    for (int j = 0; j < kMoeTileRows; ++j) {
      if (j >= rows) break;  // uniform over the warp
      const float x = v[j];
      gp[(size_t)(first + j) * ldo + feat] = __float2bfloat16_rn(0.5f * x * (1.0f + erff(x * 0.70710678118654752f)));
    }
  }
};
struct EpiMoeDown {  // gated expert output, fp32
  float* yp;
  const float* pgate;
  int ldo;
  DG_DEV void store(int feat, int first, int rows, const float (&v)[kMoeTileRows]) const {
#pragma unroll
    for (int j = 0; j < kMoeTileRows; ++j) {
      if (j >= rows) break;  // uniform over the warp
      yp[(size_t)(first + j) * ldo + feat] = __ldg(pgate + first + j) * v[j];
    }
  }
};

template <int STAGES, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_grouped_kernel(const __grid_constant__ CUtensorMap mW, const __grid_constant__ CUtensorMap mX,
                        const int4* __restrict__ tiles, int max_tiles, int b_rows, int N, int K, Epi epi,
                        int* status, StopCtl ctl) {
  static_assert(kMoeTileRows == 32, "one 32-column TMEM load per tile");
  constexpr int BN = kMoeTileRows;
  using L = GemmLayout<BN, STAGES, false>;  // A: 128 weight rows, B: BN rows of the input
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The prologue above reads nothing the kernel before wrote (see pdl_trigger).
  pdl_wait();
  if (!all_stopped(ctl.stop_at, ctl.B, ctl.step)) {
    const int n_mt = min(tiles[0].x, max_tiles);
    const int num_tiles = n_mt * (N / kBM);
    const int nk = (K + kBK - 1) / kBK;
    if (warp == 0) {
      if (lane == 0) {
        tma_prefetch(&mW);
        tma_prefetch(&mX);
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        for (int tile = blockIdx.x; tile < num_tiles && alive; tile += gridDim.x) {
          const int4 te = tiles[1 + tile % n_mt];
          const int wrow = te.x * b_rows + (tile / n_mt) * kBM;
          for (int kb = 0; kb < nk; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, status, abort)) {
              alive = false;
              break;
            }
            uint8_t* sa = smem + stage * L::kStage;
            mbar_arrive_expect_tx(&full[stage], L::kStage);
            tma_load_2d(sa, &mW, &full[stage], kb * kBK, wrow);
            tma_load_2d(sa + L::kA, &mX, &full[stage], kb * kBK, te.y);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16(kBM, BN, false);
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        int it = 0;
        for (int tile = blockIdx.x; tile < num_tiles && alive; tile += gridDim.x, ++it) {
          const int acc = it & 1;
          const uint32_t aph = (it >> 1) & 1;
          if (!mbar_wait(&tempty[acc], aph ^ 1, status, abort)) break;
          tc_fence_after();
          const uint32_t dt = tmem + acc * BN;
          for (int kb = 0; kb < nk; ++kb) {
            if (!mbar_wait(&full[stage], phase, status, abort)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * L::kStage);
            const uint32_t sb = sa + L::kA;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024), idesc,
                        (kb != 0 || kk != 0) ? 1u : 0u);
            umma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (alive) umma_commit(&tfull[acc]);
        }
      }
      __syncwarp();
    } else {
      const int q = warp & 3;
      int it = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_warp(&tfull[acc], aph, status, abort)) break;
        tc_fence_after();
        const int4 te = tiles[1 + tile % n_mt];
        float v[kMoeTileRows];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN), v);
        tc_fence_before();
        mbar_arrive(&tempty[acc]);  // the accumulator is in registers
        epi.store((tile / n_mt) * kBM + q * 32 + lane, te.y, te.z, v);
      }
    }
  }
  __syncthreads();
  drain_if_aborted(abort);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
}

// ====================================================== host-side helpers
static int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = kTargetCtas;
  }
  return n;
}

bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool u8) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                               const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                               const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess || !p)
      return false;
    fn = reinterpret_cast<EncodeFn>(p);
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// K-major operand X [rows][K]: box of 64 K-elements x box_rows rows.
static bool tmap_kmajor(CUtensorMap* m, const void* X, int rows, int K, int box_rows) {
  return make_tmap_2d(m, X, (uint64_t)K, (uint64_t)rows, (uint64_t)K * 2, kBK, (uint32_t)box_rows);
}
// MN-major operand X [K][N]: box of 64 N-elements x 64 K-rows.
static bool tmap_mnmajor(CUtensorMap* m, const void* X, int K, int N) {
  return make_tmap_2d(m, X, (uint64_t)N, (uint64_t)K, (uint64_t)N * 2, 64, kBK);
}

template <int BN, int STAGES, bool B_MN, class Epi>
static cudaError_t run_gemm(const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                            const CUtensorMap& mB2, int nb0, int nb1, int b_sub, int M, int N, int K,
                            uint32_t lbo, uint32_t sbo, const Epi& epi, int* status, StopCtl ctl,
                            cudaStream_t st, int ksplit = 1) {
  using L = GemmLayout<BN, STAGES, B_MN>;
  auto kern = gemm_kernel<BN, STAGES, B_MN, Epi>;
  cudaError_t e = set_smem_once<gemm_kernel<BN, STAGES, B_MN, Epi>>(L::kSmem);
  if (e != cudaSuccess) return e;
  const int tiles = cdiv(M, kBM) * cdiv(N, BN) * ksplit;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_pdl(kern, dim3(grid), dim3(kGemmThreads), L::kSmem, st, mA, mB0, mB1, mB2, nb0, nb1, b_sub, M,
                    N, K, ksplit, lbo, sbo, epi, status, ctl);
}

template <int BN, int STAGES, int KS, class Epi>
static cudaError_t run_gemm_ksum(const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                                 const CUtensorMap& mB2, int nb0, int nb1, int b_sub, int M, int N, int K,
                                 const Epi& epi, int* status, StopCtl ctl, cudaStream_t st) {
  using L = KsumLayout<BN, STAGES, KS>;
  cudaError_t e = set_smem_once<gemm_ksum_kernel<BN, STAGES, KS, Epi>>(L::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cdiv(M, kBM) * cdiv(N, BN) * KS, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_ksum_kernel<BN, STAGES, KS, Epi>, mA, mB0, mB1, mB2, nb0, nb1, b_sub, M, N,
                            K, epi, status, ctl);
}

// Shape of a cluster split-K launch: 128- or 64-column tiles, 2 or 4 K-slices
// per tile, one wave (tiles x slices <= SMs), each slice at least 4 K blocks;
// the choice with the fewest operand bytes per CTA, or {0, 0} when none fits
// or none beats an unsplit 64-column launch by a quarter.  `bn128_only` for
// epilogues that need whole 128-column tiles.  The launchers take it only
// where the GEMM would otherwise be split over K with a reduce launch: where
// unsplit 64-column tiles fit in one wave they measured as fast or faster.
struct KsumShape {
  int bn, ks;
};
static KsumShape ksum_shape(int M, int N, int K, bool bn128_only) {
  const int nk = cdiv(K, kBK), mt = cdiv(M, kBM);
  KsumShape best{0, 0};
  double best_bytes = 0;
  for (int bn : {128, 64}) {
    if (bn == 64 && bn128_only) continue;
    if (N % bn != 0) continue;
    for (int ks : {2, 4}) {
      const int ctas = mt * (N / bn) * ks;
      if (ctas > num_sms() || nk < 4 * ks) continue;
      const double bytes = (double)cdiv(nk, ks) * (kBM + bn) * kBK * 2;
      if (best.ks == 0 || bytes < best_bytes) {
        best = {bn, ks};
        best_bytes = bytes;
      }
    }
  }
  if (best.ks == 0) return best;
  const double unsplit = (double)nk * (kBM + 64) * kBK * 2;
  if (best_bytes > 0.75 * unsplit) return KsumShape{0, 0};
  return best;
}

// k64: instantiate the 64-column shapes too (not for epilogues that need
// whole 128-column tiles).
template <bool k64, class Epi>
static cudaError_t run_ksum(KsumShape sh, const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                            const CUtensorMap& mB2, int nb0, int nb1, int b_sub, int M, int N, int K, const Epi& epi,
                            int* status, StopCtl ctl, cudaStream_t st) {
  if (sh.bn == 128 && sh.ks == 2)
    return run_gemm_ksum<128, 4, 2>(mA, mB0, mB1, mB2, nb0, nb1, b_sub, M, N, K, epi, status, ctl, st);
  if (sh.bn == 128 && sh.ks == 4)
    return run_gemm_ksum<128, 4, 4>(mA, mB0, mB1, mB2, nb0, nb1, b_sub, M, N, K, epi, status, ctl, st);
  if constexpr (k64) {
    if (sh.bn == 64 && sh.ks == 2)
      return run_gemm_ksum<64, 6, 2>(mA, mB0, mB1, mB2, nb0, nb1, b_sub, M, N, K, epi, status, ctl, st);
    if (sh.bn == 64 && sh.ks == 4)
      return run_gemm_ksum<64, 6, 4>(mA, mB0, mB1, mB2, nb0, nb1, b_sub, M, N, K, epi, status, ctl, st);
  }
  return cudaErrorInvalidConfiguration;
}

// ============================================================ pair GEMM
// The same product on CTA pairs: a cluster of two CTAs computes an output
// tile of 256 rows x BN columns with M = 256 MMAs (cta_group::2).  Each CTA
// loads its 128 rows of A and its half (BN / 2 columns) of B, so a B tile is
// fetched once per pair and each SM's shared memory holds and serves a third
// less operand data per MMA than with two independent M = 128 tiles.  The
// leader (rank 0) waits for both CTAs' copies on its own `full` barrier
// (each copy signals it across the pair) and issues the MMAs; its commits
// arrive on the `empty` / `tfull` barriers of both CTAs.  Each CTA's four
// epilogue warps drain its own TMEM rows and arrive on the leader's `tempty`.
// Persistent over tiles (split, n, m-pair), one tile sequence per cluster.
template <int BN, int STAGES, bool B_MN>
struct PairLayout {
  static constexpr int kA = kBM * kBK * 2;         // this CTA's 128 rows of A
  static constexpr int kB = (BN / 2) * kBK * 2;    // this CTA's half of the B tile
  static constexpr int kStage = kA + kB;
  static constexpr int kBar = STAGES * kStage;
  static constexpr int kSmem = kBar + 256 + 1024;
};

// TAIL: when the last round of tiles would leave clusters idle (fewer
// remaining tiles than clusters), those tiles are cut into two halves of BN / 2
// columns (loaded through mBh, boxes of BN / 4 rows), so the round is shorter.
// F8: E4M3 operands (tcgen05 kind::f8f6f4): a 128-byte swizzled row then holds
// 128 elements of K instead of 64, so a stage covers twice the K.
// EW: epilogue warps per TMEM lane quarter.  With 2, each of the two warps of a
// quarter takes one half of the tile's columns (BN / 2, one statistics group
// of the LM head), so two warps per SM sub-partition hide each other's TMEM
// and exp latency; a half tile (TAIL) goes to the first warp of each quarter.
template <int BN, int STAGES, bool B_MN, class Epi, bool TAIL = false, bool F8 = false, int EW = 1>
__global__ void __launch_bounds__(64 + 128 * EW, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                     const __grid_constant__ CUtensorMap mBh, int M, int N, int K, int ksplit, Epi epi,
                     int* status, StopCtl ctl) {
  using L = PairLayout<BN, STAGES, B_MN>;
  constexpr int KBE = F8 ? 2 * kBK : kBK;  // K elements per stage
  static_assert(!B_MN || (BN / 2) % 64 == 0, "MN-major B halves are whole 64-column blocks");
  static_assert(!TAIL || !B_MN, "half tiles are loaded K-major");
  static_assert(!F8 || !B_MN, "E4M3 operands are loaded K-major");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  const int num_mp = (M + 2 * kBM - 1) / (2 * kBM), num_n = (N + BN - 1) / BN;
  const int num_mn = num_mp * num_n;
  const int num_full = num_mn * ksplit;  // tile t: split t / num_mn, m-pair and n from t % num_mn
  const int nk_all = (K + KBE - 1) / KBE;
  // work items: full tiles, then (TAIL) the last round's tiles as two halves each
  const int n_whole = num_full / ncl * ncl, n_rest = num_full - n_whole;
  const bool halves = TAIL && ksplit == 1 && n_rest > 0 && 2 * n_rest <= ncl;
  const int num_tiles = halves ? n_whole + 2 * n_rest : num_full;
  auto coords = [&](int item, int& m0, int& n0, int& kb_lo, int& kb_hi, int& width) {
    int tile = item, sub = 0;
    width = BN;
    if (halves && item >= n_whole) {
      tile = n_whole + (item - n_whole) / 2;
      sub = (item - n_whole) & 1;
      width = BN / 2;
    }
    const int sp = tile / num_mn, tmn = tile % num_mn;
    m0 = (tmn % num_mp) * 2 * kBM;
    n0 = (tmn / num_mp) * BN + sub * (BN / 2);
    kb_lo = (int)((int64_t)sp * nk_all / ksplit);
    kb_hi = (int)((int64_t)(sp + 1) * nk_all / ksplit);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8 * EW);  // 4 EW epilogue warps in each CTA
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 2 * BN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The prologue above overlaps the kernel before this one when that one
  // triggers its dependents early; its results are read only from here on.
  pdl_wait();
  if (!all_stopped(ctl.stop_at, ctl.B, ctl.step)) {
    if (warp == 0) {
      if (lane == 0) {
        tma_prefetch(&mA);
        tma_prefetch(&mB);
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        for (int tile = cid; tile < num_tiles && alive; tile += ncl) {
          int m0, n0, kb_lo, kb_hi, width;
          coords(tile, m0, n0, kb_lo, kb_hi, width);
          const int arow = m0 + (int)rank * kBM, bcol = n0 + (int)rank * (width / 2);
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, status, abort)) {
              alive = false;
              break;
            }
            uint8_t* sa = smem + stage * L::kStage;
            uint8_t* sb = sa + L::kA;
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (L::kA + (width / 2) * kBK * 2));
            const uint32_t bar = cluster_addr(&full[stage], 0);
            tma_load_2d_pair(sa, &mA, bar, kb * KBE, arow);
            if (!B_MN) {
              tma_load_2d_pair(sb, width == BN ? &mB : &mBh, bar, kb * KBE, bcol);
            } else {
  #pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tma_load_2d_pair(sb + j * (kBK * 128), &mB, bar, bcol + 64 * j, kb * kBK);
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        // Wait until the leader's MMAs released every stage, so that no commit
        // is still on its way to this CTA's barriers when it exits.
        for (int i = 0; i < STAGES && alive; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1, status, abort)) break;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    } else if (warp == 1) {
      if (leader && lane == 0) {  // one thread of the leader waits and issues for the pair
        constexpr uint32_t idesc_full = F8 ? idesc_e4m3(2 * kBM, BN) : idesc_bf16(2 * kBM, BN, B_MN);
        constexpr uint32_t idesc_half = F8 ? idesc_e4m3(2 * kBM, BN / 2) : idesc_bf16(2 * kBM, BN / 2, B_MN);
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        int it = 0;
        for (int tile = cid; tile < num_tiles && alive; tile += ncl, ++it) {
          const int acc = it & 1;
          const uint32_t aph = (it >> 1) & 1;
          if (!mbar_wait(&tempty[acc], aph ^ 1, status, abort)) break;
          tc_fence_after();
          const uint32_t dt = tmem + acc * BN;
          int m0, n0, kb_lo, kb_hi, width;
          coords(tile, m0, n0, kb_lo, kb_hi, width);
          const uint32_t idesc = width == BN ? idesc_full : idesc_half;
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            if (!mbar_wait(&full[stage], phase, status, abort)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * L::kStage);
            const uint32_t sb = sa + L::kA;
  #pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc_sw128(sb + kk * 2048, kBK * 128, 1024)
                                       : sdesc_sw128(sb + kk * 32, 16, 1024);
              if constexpr (F8)
                umma_e4m3_pair(dt, ad, bd, idesc, (kb != kb_lo || kk != 0) ? 1u : 0u);
              else
                umma_bf16_pair(dt, ad, bd, idesc, (kb != kb_lo || kk != 0) ? 1u : 0u);
            }
            umma_commit_pair(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (alive) umma_commit_pair(&tfull[acc]);
        }
      }
      __syncwarp();
    } else {
      const int q = warp & 3;  // TMEM lane quarter this warp may read
      const int half = (warp - 2) / 4;  // EW == 2: which half of the tile's columns
      const int r_local = q * 32 + lane;
      int it = 0;
      for (int tile = cid; tile < num_tiles; tile += ncl, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_warp(&tfull[acc], aph, status, abort)) break;
        tc_fence_after();
        int m0, n0, kb_lo, kb_hi, width;
        coords(tile, m0, n0, kb_lo, kb_hi, width);
        const int row = m0 + (int)rank * kBM + r_local;
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
        if constexpr (EW == 1) {
          auto ld = [&](int c, float(&v)[32]) { tmem_ld32(tb + c * 32, v); };
          if (!TAIL || width == BN)
            epi.template tile<BN>(row, row < M, n0, N, ld, tile / num_mn);
          else
            epi.template tile<BN / 2>(row, row < M, n0, N, ld, 0);
        } else {
          static_assert(EW == 2, "one or two epilogue warps per lane quarter");
          const uint32_t th = tb + (uint32_t)(half * (BN / 2));
          auto ld = [&](int c, float(&v)[32]) { tmem_ld32(th + c * 32, v); };
          if (!TAIL || width == BN)
            epi.template tile<BN / 2>(row, row < M, n0 + half * (BN / 2), N, ld, tile / num_mn);
          else if (half == 0)
            epi.template tile<BN / 2>(row, row < M, n0, N, ld, 0);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cluster_addr(&tempty[acc], 0));
      }
    }
  }
  __syncwarp();
  drain_if_aborted(abort);
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 2 * BN);
  }
}

// Clusters of two that can be resident at once with this kernel's shared
// memory (SMs per GPC may be odd, so it can be below half the SM count).
template <auto Kernel>
static int max_pair_clusters(int smem, int threads) {
  static int n = -1;
  if (n < 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (kTargetCtas / 2), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, Kernel, &cfg) != cudaSuccess || c <= 0) {
      cudaGetLastError();
      c = 0;
    }
    n = c;
  }
  return n;
}

// Clusters a pair GEMM of this many tiles may use (0 if none can launch).
template <int BN, int STAGES, bool B_MN, class Epi, bool TAIL = false, bool F8 = false, int EW = 1>
static int pair_clusters() {
  using L = PairLayout<BN, STAGES, B_MN>;
  if (set_smem_once<gemm_pair_kernel<BN, STAGES, B_MN, Epi, TAIL, F8, EW>>(L::kSmem) != cudaSuccess) return 0;
  return max_pair_clusters<gemm_pair_kernel<BN, STAGES, B_MN, Epi, TAIL, F8, EW>>(L::kSmem, 64 + 128 * EW);
}

template <int BN, int STAGES, bool B_MN, class Epi, bool TAIL = false, bool F8 = false, int EW = 1>
static cudaError_t run_gemm_pair(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mBh, int M,
                                 int N, int K, int ksplit, const Epi& epi, int* status, StopCtl ctl,
                                 cudaStream_t st) {
  using L = PairLayout<BN, STAGES, B_MN>;
  const int maxc = pair_clusters<BN, STAGES, B_MN, Epi, TAIL, F8, EW>();
  if (maxc <= 0) return cudaErrorInvalidConfiguration;
  const int tiles = cdiv(M, 2 * kBM) * cdiv(N, BN) * ksplit;
  const int ncl = tiles < maxc ? tiles : maxc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ncl, 1, 1);
  cfg.blockDim = dim3(64 + 128 * EW, 1, 1);
  cfg.dynamicSmemBytes = L::kSmem;
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
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<BN, STAGES, B_MN, Epi, TAIL, F8, EW>, mA, mB, mBh, M, N, K,
                            ksplit, epi, status, ctl);
}

cudaError_t launch_debug_gemm(const void* A, const void* Bm, float* D, int M, int N, int K,
                              int b_mn_major, int* status, cudaStream_t st) {
  CUtensorMap mA, mB;
  EpiF32 epi{D, N};
  StopCtl ctl{nullptr, 0, 0};
  if (!tmap_kmajor(&mA, A, M, K, kBM)) return cudaErrorInvalidValue;
  if (b_mn_major == 0) {
    if (!tmap_kmajor(&mB, Bm, N, K, 256)) return cudaErrorInvalidValue;
    return run_gemm<256, 4, false>(mA, mB, mB, mB, N, 0, 256, M, N, K, 0, 0, epi, status, ctl, st);
  }
  if (b_mn_major >= 5) {  // cluster split-K engine, B [N][K]
    const KsumShape sh{b_mn_major <= 6 ? 128 : 64, b_mn_major % 2 == 1 ? 2 : 4};
    if (!tmap_kmajor(&mB, Bm, N, K, sh.bn)) return cudaErrorInvalidValue;
    return run_ksum<true>(sh, mA, mB, mB, mB, N, 0, sh.bn, M, N, K, epi, status, ctl, st);
  }
  if (b_mn_major == 3) {  // CTA-pair engine, B [N][K]
    if (!tmap_kmajor(&mB, Bm, N, K, 128)) return cudaErrorInvalidValue;
    return run_gemm_pair<256, 6, false>(mA, mB, mB, M, N, K, 1, epi, status, ctl, st);
  }
  if (!tmap_mnmajor(&mB, Bm, K, N)) return cudaErrorInvalidValue;
  if (b_mn_major == 4) {  // CTA-pair engine, B [K][N]
    return run_gemm_pair<256, 6, true>(mA, mB, mB, M, N, K, 1, epi, status, ctl, st);
  }
  // 1: LBO = distance between 64-column blocks along N, SBO = between 8-row
  // groups along K (the layout the self-conditioning kernel uses); 2: swapped.
  const uint32_t lbo = b_mn_major == 1 ? kBK * 128 : 1024;
  const uint32_t sbo = b_mn_major == 1 ? 1024 : kBK * 128;
  return run_gemm<256, 4, true>(mA, mB, mB, mB, N, 0, 64, M, N, K, lbo, sbo, epi, status, ctl, st);
}

cudaError_t launch_gemm_f32_partials(const void* A, const void* W, float* part, int M, int N, int K, int ks,
                                     StopCtl ctl, int* status, cudaStream_t st) {
  CUtensorMap mA, mB;
  if (!tmap_kmajor(&mA, A, M, K, kBM) || !tmap_kmajor(&mB, W, N, K, 128)) return cudaErrorInvalidValue;
  EpiPartial ep{part, M, N};
  return run_gemm<128, 4, false>(mA, mB, mB, mB, N, 0, 128, M, N, K, 0, 0, ep, status, ctl, st, ks);
}

int gemm_ksplit(int M, int N, int K) {
  const int tiles = cdiv(M, kBM) * cdiv(N, 128);
  const int nk = cdiv(K, kBK);
  int ks = kTargetCtas / tiles;
  if (ks > nk / 2) ks = nk / 2;
  if (ks > 16) ks = 16;
  return ks < 1 ? 1 : ks;
}

// Sum of the K-split partials of one row segment of 8 columns, then the
// residual / GELU epilogue of the small GEMMs, bf16 out.
__global__ void __launch_bounds__(256)
    splitk_bf16_kernel(const float* part, int ksplit, int M, int N, __nv_bfloat16* out, int ldo,
                       const __nv_bfloat16* resid, int ldr, int gelu, int C, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.y;
  const int c8 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c8 >= N || !canvas_active(ctl.stop_at, row / C, ctl.step)) return;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int sp = 0; sp < ksplit; ++sp) {
    const float4* src = reinterpret_cast<const float4*>(part + ((size_t)sp * M + row) * N + c8);
    const float4 x = src[0], y = src[1];
    v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
    v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
  }
  if (resid) {
    uint4 r = *reinterpret_cast<const uint4*>(resid + (size_t)row * ldr + c8);
    const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(&r);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] += __bfloat162float(rb[e]);
  }
  if (gelu) {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.5f * v[e] * (1.0f + erff(v[e] * 0.70710678118654752f));
  }
  uint4 w;
  w.x = pack_bf16(v[0], v[1]);
  w.y = pack_bf16(v[2], v[3]);
  w.z = pack_bf16(v[4], v[5]);
  w.w = pack_bf16(v[6], v[7]);
  *reinterpret_cast<uint4*>(out + (size_t)row * ldo + c8) = w;
}

// Sum of the K-split partials of the q / k / v projections; RoPE on the
// (j, j + hd/2) pairs of q and k.  Thread = (row, head, j < hd/2).
struct QkvOut {
  __nv_bfloat16 *q, *k, *v;
  const float2* rope;
  int C, Hq, Hkv, nq, nkv, kv_rows, kv_row0, hd;
};
__global__ void __launch_bounds__(256)
    splitk_qkv_kernel(const float* part, int ksplit, int M, int N, QkvOut o, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.y;
  const int pidx = blockIdx.x * blockDim.x + threadIdx.x;
  const int half = o.hd / 2;
  if (pidx >= N / 2) return;
  const int head = pidx / half, j = pidx % half;
  const int col0 = head * o.hd + j, col1 = col0 + half;
  float x0 = 0.f, x1 = 0.f;
  for (int sp = 0; sp < ksplit; ++sp) {
    const float* src = part + ((size_t)sp * M + row) * N;
    x0 += src[col0];
    x1 += src[col1];
  }
  const int b = row / o.C, i = row % o.C;
  const bool is_q = col0 < o.nq;
  const bool is_k = !is_q && col0 < o.nq + o.nkv;
  if (is_q || is_k) {
    const float2 r = o.rope[(size_t)i * half + j];
    const float a0 = x0, a1 = x1;
    x0 = a0 * r.x - a1 * r.y;
    x1 = a0 * r.y + a1 * r.x;
  }
  __nv_bfloat16* dst;
  if (is_q) {
    dst = o.q + (((size_t)b * o.Hq + col0 / o.hd) * o.C + i) * o.hd;
  } else {
    const int hh = (col0 - o.nq - (is_k ? 0 : o.nkv)) / o.hd;
    dst = (is_k ? o.k : o.v) + (((size_t)b * o.Hkv + hh) * o.kv_rows + o.kv_row0 + i) * o.hd;
  }
  dst[j] = __float2bfloat16_rn(x0);
  dst[j + half] = __float2bfloat16_rn(x1);
}

cudaError_t launch_gemm_bf16(const void* A, const void* W, void* out, int ldo, const void* resid,
                             int ldr, int gelu, int M, int N, int K, int C, StopCtl ctl,
                             int* status, float* part, size_t part_elems, cudaStream_t st) {
  CUtensorMap mA, mB;
  if (!tmap_kmajor(&mA, A, M, K, kBM) || !tmap_kmajor(&mB, W, N, K, 128)) return cudaErrorInvalidValue;
  EpiBF16 epi{reinterpret_cast<__nv_bfloat16*>(out), ldo,
              reinterpret_cast<const __nv_bfloat16*>(resid), ldr, gelu, C, ctl};
  // When 64-column tiles fit in one wave and the K loop is short, they run
  // unsplit (no partials, no reduce launch), which measured faster; otherwise
  // 128-column tiles, split over K when too few to fill the GPU.
  const int tiles64 = cdiv(M, kBM) * (N / 64);
  if (N % 64 == 0 && tiles64 <= kTargetCtas && (K <= 1024 || (tiles64 >= 64 && K <= 2048))) {
    CUtensorMap mB64;
    if (!tmap_kmajor(&mB64, W, N, K, 64)) return cudaErrorInvalidValue;
    return run_gemm<64, 6, false>(mA, mB64, mB64, mB64, N, 0, 64, M, N, K, 0, 0, epi, status, ctl, st);
  }
  const int ks = gemm_ksplit(M, N, K);
  // Split over K: one wave of clusters that sum their K slices in shared
  // memory (no partials, no reduce launch) when the shape allows, else fp32
  // partials and a reduce kernel.
  const KsumShape sh = ks > 1 ? ksum_shape(M, N, K, false) : KsumShape{0, 0};
  if (sh.ks > 0) {
    CUtensorMap mBs;
    if (!tmap_kmajor(&mBs, W, N, K, sh.bn)) return cudaErrorInvalidValue;
    return run_ksum<true>(sh, mA, mBs, mBs, mBs, N, 0, sh.bn, M, N, K, epi, status, ctl, st);
  }
  if (ks > 1 && part && (size_t)ks * M * N <= part_elems && N % 8 == 0) {
    EpiPartial ep{part, M, N};
    cudaError_t e = run_gemm<128, 4, false>(mA, mB, mB, mB, N, 0, 128, M, N, K, 0, 0, ep, status, ctl, st, ks);
    if (e != cudaSuccess) return e;
    dim3 grid(cdiv(N / 8, 256), M);
    return launch_pdl(splitk_bf16_kernel, grid, dim3(256), 0, st, (const float*)part, ks, M, N,
                      reinterpret_cast<__nv_bfloat16*>(out), ldo, reinterpret_cast<const __nv_bfloat16*>(resid),
                      ldr, gelu, C, ctl);
  }
  return run_gemm<128, 4, false>(mA, mB, mB, mB, N, 0, 128, M, N, K, 0, 0, epi, status, ctl, st);
}

template <int HD>
static cudaError_t qkv_impl(const CUtensorMap& mA, const CUtensorMap& m0, const CUtensorMap& m1,
                            const CUtensorMap& m2, int nb0, int nb1, int M, int N, int K,
                            const EpiQKV<HD>& epi, int* status, StopCtl ctl, cudaStream_t st) {
  return run_gemm<128, 4, false>(mA, m0, m1, m2, nb0, nb1, HD, M, N, K, 0, 0, epi, status, ctl, st);
}

cudaError_t launch_qkv(const void* a, const void* Wq, const void* Wk, const void* Wv, void* q,
                       void* k, void* v, int kv_rows, int kv_row0, const float2* rope,
                       const dg_dims& D, StopCtl ctl, int* status, float* part, size_t part_elems,
                       cudaStream_t st) {
  const int M = D.B * D.C, nq = Wq ? D.Hq * D.hd : 0, nkv = D.Hkv * D.hd;
  CUtensorMap mA, mq, mk, mv;
  if (!tmap_kmajor(&mA, a, M, D.d, kBM)) return cudaErrorInvalidValue;
  // boxes of one head (hd rows) so that a tile may span the q / k / v weights
  if (!tmap_kmajor(&mk, Wk, nkv, D.d, D.hd) || !tmap_kmajor(&mv, Wv, nkv, D.d, D.hd))
    return cudaErrorInvalidValue;
  if (Wq && !tmap_kmajor(&mq, Wq, nq, D.d, D.hd)) return cudaErrorInvalidValue;
  const int N = nq + 2 * nkv;
  auto bf = [](void* p) { return reinterpret_cast<__nv_bfloat16*>(p); };
  const CUtensorMap& m0 = Wq ? mq : mk;
  const CUtensorMap& m1 = Wq ? mk : mv;
  const CUtensorMap& m2 = mv;
  const int nb0 = Wq ? nq : nkv, nb1 = Wq ? nkv : nkv;
  const int ks = gemm_ksplit(M, N, D.d);
  const KsumShape sh = ks > 1 ? ksum_shape(M, N, D.d, D.hd > 64) : KsumShape{0, 0};
  if (sh.ks > 0) {  // split over K, summed across the cluster (see launch_gemm_bf16)
    switch (D.hd) {
      case 32: {
        EpiQKV<32> e{bf(q), bf(k), bf(v), rope, D.C, D.Hq, D.Hkv, nq, nkv, kv_rows, kv_row0};
        return run_ksum<true>(sh, mA, m0, m1, m2, nb0, nb1, D.hd, M, N, D.d, e, status, ctl, st);
      }
      case 64: {
        EpiQKV<64> e{bf(q), bf(k), bf(v), rope, D.C, D.Hq, D.Hkv, nq, nkv, kv_rows, kv_row0};
        return run_ksum<true>(sh, mA, m0, m1, m2, nb0, nb1, D.hd, M, N, D.d, e, status, ctl, st);
      }
      case 128: {
        EpiQKV<128> e{bf(q), bf(k), bf(v), rope, D.C, D.Hq, D.Hkv, nq, nkv, kv_rows, kv_row0};
        return run_ksum<false>(sh, mA, m0, m1, m2, nb0, nb1, D.hd, M, N, D.d, e, status, ctl, st);
      }
      default:
        return cudaErrorInvalidValue;
    }
  }
  if (ks > 1 && part && (size_t)ks * M * N <= part_elems) {
    EpiPartial ep{part, M, N};
    cudaError_t e =
        run_gemm<128, 4, false>(mA, m0, m1, m2, nb0, nb1, D.hd, M, N, D.d, 0, 0, ep, status, ctl, st, ks);
    if (e != cudaSuccess) return e;
    QkvOut o{bf(q), bf(k), bf(v), rope, D.C, D.Hq, D.Hkv, nq, nkv, kv_rows, kv_row0, D.hd};
    dim3 grid(cdiv(N / 2, 256), M);
    return launch_pdl(splitk_qkv_kernel, grid, dim3(256), 0, st, (const float*)part, ks, M, N, o, ctl);
  }
  switch (D.hd) {
    case 32: {
      EpiQKV<32> e{bf(q), bf(k), bf(v), rope, D.C, D.Hq, D.Hkv, nq, nkv, kv_rows, kv_row0};
      return qkv_impl<32>(mA, m0, m1, m2, nb0, nb1, M, N, D.d, e, status, ctl, st);
    }
    case 64: {
      EpiQKV<64> e{bf(q), bf(k), bf(v), rope, D.C, D.Hq, D.Hkv, nq, nkv, kv_rows, kv_row0};
      return qkv_impl<64>(mA, m0, m1, m2, nb0, nb1, M, N, D.d, e, status, ctl, st);
    }
    case 128: {
      EpiQKV<128> e{bf(q), bf(k), bf(v), rope, D.C, D.Hq, D.Hkv, nq, nkv, kv_rows, kv_row0};
      return qkv_impl<128>(mA, m0, m1, m2, nb0, nb1, M, N, D.d, e, status, ctl, st);
    }
  }
  return cudaErrorInvalidValue;
}

// Epilogue warps per TMEM lane quarter of the LM head.  The FP8 head's main
// loop is half as long as the bf16 head's, so its epilogue bounds it: two
// warps per quarter took it from 216 to 180 us at V = 262144, d = 2816, C = 256
// (same-box A/B), while the bf16 head measured 3.5 us slower with two.
constexpr int kLmEW = 1, kLmEW8 = 2;

cudaError_t launch_lmhead(const LmArgs& a, StopCtl ctl, int* status, cudaStream_t st) {
  CUtensorMap mA, mB, mBh;  // B boxes: half a vocabulary tile (one CTA of a pair), or half of a half tile
  EpiLM epi{a.alpha, a.coef2, a.inv_sqrt_d, reinterpret_cast<__nv_bfloat16*>(a.pt), a.gst, a.logits, a.M, a.V,
            a.excl, a.hscale, a.escale, a.ref2, a.rkey};
  if (a.E8) {
    // E4M3 codes: 128 one-byte elements per 128-byte row
    if (!make_tmap_2d(&mA, a.h8, (uint64_t)a.d, (uint64_t)a.M, (uint64_t)a.d, 2 * kBK, kBM, true) ||
        !make_tmap_2d(&mB, a.E8, (uint64_t)a.d, (uint64_t)a.V, (uint64_t)a.d, 2 * kBK, kLmBN / 2, true) ||
        !make_tmap_2d(&mBh, a.E8, (uint64_t)a.d, (uint64_t)a.V, (uint64_t)a.d, 2 * kBK, kLmBN / 4, true))
      return cudaErrorInvalidValue;
    return run_gemm_pair<kLmBN, 7, false, EpiLM, true, true, kLmEW8>(mA, mB, mBh, a.M, a.V, a.d, 1, epi, status, ctl,
                                                                    st);
  }
  if (!tmap_kmajor(&mA, a.h, a.M, a.d, kBM) || !tmap_kmajor(&mB, a.E, a.V, a.d, kLmBN / 2) ||
      !tmap_kmajor(&mBh, a.E, a.V, a.d, kLmBN / 4))
    return cudaErrorInvalidValue;
  return run_gemm_pair<kLmBN, 7, false, EpiLM, true, false, kLmEW>(mA, mB, mBh, a.M, a.V, a.d, 1, epi, status, ctl,
                                                                st);
}

// ====================================================== self-conditioning
// u_split = p0[:, vocabulary split] . E[vocabulary split, :] on CTA pairs:
// A = p0 [M][V] (K-major over the vocabulary), B = E [V][d] (MN-major), fp32
// partials [split][M][d] summed by reduce_kernel.  Consecutive clusters take
// the d-tiles of one split, so the p0 columns they share are read from HBM
// once and from L2 after.
int selfcond_active_splits(const dg_dims& D) {
  const int bound = selfcond_splits(D);
  const int tiles = cdiv(D.d, kScBN) * cdiv(D.B * D.C, 2 * kBM);
  const int maxc = pair_clusters<kScBN, 7, true, EpiPartial>();
  int ns = maxc / tiles;
  if (ns > bound) ns = bound;
  return ns < 1 ? 1 : ns;
}

cudaError_t launch_selfcond(const ScArgs& a, StopCtl ctl, int* status, cudaStream_t st) {
  CUtensorMap mP, mE;
  if (!tmap_kmajor(&mP, a.pt, a.M, a.V, kBM) || !tmap_mnmajor(&mE, a.E, a.V, a.d))
    return cudaErrorInvalidValue;
  EpiPartial ep{a.upart, a.M, a.d};
  return run_gemm_pair<kScBN, 7, true>(mP, mE, mE, a.M, a.d, a.V, a.nsplit, ep, status, ctl, st);
}

// The two grouped expert GEMMs of the MoE FFN (128-column tiles; d and Fe are
// multiples of 128).
template <class Epi>
static cudaError_t run_grouped(const CUtensorMap& mW, const CUtensorMap& mX, const int4* tiles, int max_tiles,
                               int b_rows, int N, int K, const Epi& epi, int* status, StopCtl ctl,
                               cudaStream_t st) {
  constexpr int STAGES = 8;
  using L = GemmLayout<kMoeTileRows, STAGES, false>;
  cudaError_t e = set_smem_once<gemm_grouped_kernel<STAGES, Epi>>(L::kSmem);
  if (e != cudaSuccess) return e;
  const int bound = max_tiles * (N / kBM);
  const int grid = bound < num_sms() ? (bound > 0 ? bound : 1) : num_sms();
  return launch_pdl(gemm_grouped_kernel<STAGES, Epi>, dim3(grid), dim3(kGemmThreads), L::kSmem, st, mW, mX, tiles,
                    max_tiles, b_rows, N, K, epi, status, ctl);
}

cudaError_t launch_moe_experts(const void* xp, const void* We1, const void* We2, const int4* tiles,
                               int max_tiles, int R, int groups, const float* pgate, void* gp, float* yp, int d,
                               int Fe, int* status, StopCtl ctl, cudaStream_t st) {
  // row boxes reaching past row R read zeros (the tensor maps end there);
  // their results are not stored
  CUtensorMap mX, mW1, mG, mW2;
  if (!tmap_kmajor(&mX, xp, R, d, kMoeTileRows) || !tmap_kmajor(&mG, gp, R, Fe, kMoeTileRows) ||
      !tmap_kmajor(&mW1, We1, groups * Fe, d, kBM) || !tmap_kmajor(&mW2, We2, groups * d, Fe, kBM))
    return cudaErrorInvalidValue;
  cudaError_t e = run_grouped(mW1, mX, tiles, max_tiles, Fe, Fe, d,
                              EpiMoeUp{reinterpret_cast<__nv_bfloat16*>(gp), Fe}, status, ctl, st);
  if (e != cudaSuccess) return e;
  return run_grouped(mW2, mG, tiles, max_tiles, d, d, Fe, EpiMoeDown{yp, pgate, d}, status, ctl, st);
}

}  // namespace dg
