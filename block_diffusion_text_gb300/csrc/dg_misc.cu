// Memory-bound kernels of the denoising step: embedding + RMSNorm, the merge
// of the LM-head tile statistics, the entropy-bounded sampler, the reduction
// of the self-conditioning partials, canvas initialisation and the loop
// bookkeeping.
#include <cfloat>
#include <climits>

#include <cmath>

#include <cuda_fp8.h>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

// ------------------------------------------------------- embed + RMSNorm --
// a = RMSNorm(E[x] + z) with no learned gain ("DiffusionGemma" docs chapter,
// data-flow pseudocode: embed(canvas) + self_conditioning(prev); technical
// report summary, step 3).  Row blocks 0..C-1 also fill the RoPE table of
// positions P + i in double precision.
constexpr int kEmbThreads = 256;
constexpr int kEmbMaxChunks = 8;  // d <= 8 * 8 * 256

// The sum of squares is kept as an unevaluated pair of floats (error-free
// products and sums), the scale r = 1 / sqrt(mean + eps) is formed once per
// row as a float pair (~2^-44), and each x r is rounded to bf16 from a float
// pair: a is the correctly rounded bf16 of x r, the value the definition
// gives, so its rounding does not depend on the order of the sum.  (FP64
// division and square root are slow on this part; nothing here uses them.)
DG_DEV void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
DG_DEV void pair_add(float& hi, float& lo, float bhi, float blo) {  // (hi, lo) += (bhi, blo)
  float s, e;
  two_sum(hi, bhi, s, e);
  e += lo + blo;
  hi = s + e;
  lo = e - (hi - s);
}
// bf16 of hi + lo, round to nearest even: the midpoint between the two bf16
// neighbours of hi has hi's exponent, so hi - mid is exact and the sign of
// (hi - mid) + lo is that of the exact difference.
DG_DEV uint32_t bf16_of_pair(float hi, float lo) {
  const uint32_t bits = __float_as_uint(hi);
  const uint32_t t = bits >> 16;  // sign, exponent, 7 mantissa bits
  if ((bits & 0x7f800000u) == 0x7f800000u) return t | ((bits & 0xffffu) ? 0x40u : 0u);  // inf, nan
  const float mid = __uint_as_float((t << 16) | 0x8000u);
  const float dlt = (hi - mid) + lo;
  bool up = (bits >> 31) ? (dlt < 0.f) : (dlt > 0.f);  // magnitude above the midpoint
  if (dlt == 0.f) up = (t & 1u) != 0;
  return t + (up ? 1u : 0u);
}

// RoPE frequencies theta_j = base^(-2j / hd), computed on the host in double.
struct RopeTheta {
  double th[64];  // hd / 2 <= 64
};

__global__ void __launch_bounds__(kEmbThreads)
    embed_rmsnorm_kernel(const int32_t* tokens, const __nv_bfloat16* E, const __nv_bfloat16* z,
                         __nv_bfloat16* a, float2* rope, int d, int V, float eps, int C, int P, int hd,
                         RopeTheta theta, StopCtl ctl, int* status, const __nv_bfloat16* src) {
  pdl_trigger();
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.x;
  const int nch = d / 8;
  const uint4* e4;
  const uint4* z4;
  if (src) {  // a deeper layer: the residual stream h of the layer below
    e4 = reinterpret_cast<const uint4*>(src + (size_t)row * d);
    z4 = nullptr;
  } else {
    int tok = tokens[row];
    if (tok < 0 || tok >= V) {  // never gather outside E: record the bad token, embed token 0
      if (threadIdx.x == 0) atomicExch(status, kStatusValue);
      tok = 0;
    }
    e4 = reinterpret_cast<const uint4*>(E + (size_t)tok * d);
    z4 = z ? reinterpret_cast<const uint4*>(z + (size_t)row * d) : nullptr;
  }
  float x[kEmbMaxChunks][8];
  float sh = 0.f, sl = 0.f;  // sum of squares as a float pair
#pragma unroll
  for (int k = 0; k < kEmbMaxChunks; ++k) {
    const int c = threadIdx.x + k * kEmbThreads;
    if (c < nch) {
      uint4 ev = e4[c];
      const __nv_bfloat16* eb = reinterpret_cast<const __nv_bfloat16*>(&ev);
      uint4 zv = z4 ? z4[c] : make_uint4(0, 0, 0, 0);
      const __nv_bfloat16* zb = reinterpret_cast<const __nv_bfloat16*>(&zv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[k][e] = __bfloat162float(eb[e]) + __bfloat162float(zb[e]);
        const float p = x[k][e] * x[k][e];
        pair_add(sh, sl, p, fmaf(x[k][e], x[k][e], -p));
      }
    }
  }
  __shared__ float red[2][kEmbThreads / 32];
  __shared__ float rs[2];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    pair_add(sh, sl, __shfl_xor_sync(0xffffffffu, sh, o), __shfl_xor_sync(0xffffffffu, sl, o));
  if (threadIdx.x % 32 == 0) {
    red[0][threadIdx.x / 32] = sh;
    red[1][threadIdx.x / 32] = sl;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float th = red[0][0], tl = red[1][0];
    for (int w = 1; w < kEmbThreads / 32; ++w) pair_add(th, tl, red[0][w], red[1][w]);
    // m = sum / d + eps as a float pair (the remainder of a correctly rounded
    // quotient is exact under fma)
    const float fd = (float)d;
    float mh = th / fd;
    float ml = (fmaf(-mh, fd, th) + tl) / fd;
    pair_add(mh, ml, eps, 0.f);
    // r = 1 / sqrt(m): rsqrtf, then one Newton step whose residual 1 - m r0^2
    // is formed from exact products (its relative error squares: ~2^-44)
    const float r0 = rsqrtf(mh);
    const float t = r0 * r0, te = fmaf(r0, r0, -t);
    const float p = mh * t, pe = fmaf(mh, t, -p);
    const float e = ((1.0f - p) - pe) - fmaf(mh, te, ml * t);
    two_sum(r0, 0.5f * r0 * e, rs[0], rs[1]);
  }
  __syncthreads();
  const float rh = rs[0], rl = rs[1];
  auto scaled = [&](float v) {  // bf16 of v r from the float pair v rh + v rl
    const float ph = v * rh;
    return bf16_of_pair(ph, fmaf(v, rl, fmaf(v, rh, -ph)));
  };
  uint4* a4 = reinterpret_cast<uint4*>(a + (size_t)row * d);
#pragma unroll
  for (int k = 0; k < kEmbMaxChunks; ++k) {
    const int c = threadIdx.x + k * kEmbThreads;
    if (c < nch) {
      uint4 w;
      w.x = scaled(x[k][0]) | (scaled(x[k][1]) << 16);
      w.y = scaled(x[k][2]) | (scaled(x[k][3]) << 16);
      w.z = scaled(x[k][4]) | (scaled(x[k][5]) << 16);
      w.w = scaled(x[k][6]) | (scaled(x[k][7]) << 16);
      a4[c] = w;
    }
  }
  if (rope && row < C) {
    // angle (P + i) theta_j reduced modulo 2 pi in double (a few operations on
    // the slow FP64 units), then sine and cosine in float of |r| <= pi
    for (int j = threadIdx.x; j < hd / 2; j += kEmbThreads) {
      const double ang = (double)(P + row) * theta.th[j];
      const double k = rint(ang * 0.15915494309189535);  // 1 / (2 pi)
      const double r = fma(-k, 6.283185307179586, ang);
      float sn, cs;
      sincosf((float)r, &sn, &cs);
      rope[(size_t)row * (hd / 2) + j] = make_float2(cs, sn);
    }
  }
}

cudaError_t launch_embed_rmsnorm(const int32_t* tokens, const void* E, const void* z, void* a,
                                 float2* rope, const dg_dims& D, int rows, int P, StopCtl ctl,
                                 int* status, cudaStream_t st, const void* src) {
  RopeTheta th{};
  for (int j = 0; j < D.hd / 2 && j < 64; ++j) th.th[j] = std::pow((double)D.rope_base, -2.0 * j / D.hd);
  return launch_pdl(embed_rmsnorm_kernel, dim3(rows), dim3(kEmbThreads), 0, st, tokens,
                    reinterpret_cast<const __nv_bfloat16*>(E), reinterpret_cast<const __nv_bfloat16*>(z),
                    reinterpret_cast<__nv_bfloat16*>(a), rope, D.d, D.V, D.rms_eps, D.C, P, D.hd, th, ctl,
                    status, reinterpret_cast<const __nv_bfloat16*>(src));
}

// ------------------------------------------------------- tile statistics --
// Merge of the per-group (max, sum, weighted sum, argmax) of each row into the
// tempered-softmax entropy H = ln Z - S / Z, the argmax, the row maximum m and
// Z (a stored group exp(s - m_g) becomes p0 with the factor exp(m_g - m) / Z).
// The group statistics are laid out [row][group]; each row is taken by `wpr`
// warps of a CTA (all eight for long rows, one for short ones), which read it
// once with coalesced loads, merging online: running maximum R, with
// L = sum 2^(m_g - R) l_g and Q = sum 2^(m_g - R) (S_g + l_g (m_g - R)),
// rescaled when R grows.  Sums in fp32 (two accumulators per thread); the
// entropy is formed in double.
constexpr int kStatsThreads = 256;
constexpr int kStatsWarps = kStatsThreads / 32;

struct RowSum {
  float R, L, Q;
};
DG_DEV RowSum merge_rowsum(RowSum a, RowSum b) {
  if (b.L == 0.f) return a;
  if (a.L == 0.f) return b;
  const float R = fmaxf(a.R, b.R);
  const float da = a.R - R, db = b.R - R;
  const float wa = exp2f(da), wb = exp2f(db);
  return {R, wa * a.L + wb * b.L, wa * fmaf(da, a.L, a.Q) + wb * fmaf(db, b.L, b.Q)};
}
DG_DEV void add_group(RowSum& acc, float mt, float lt, float St) {
  if (mt > acc.R) {  // the running maximum grows: rescale what was summed
    if (acc.L != 0.f) {
      const float d = acc.R - mt;
      const float w = exp2f(d);
      acc.Q = w * fmaf(d, acc.L, acc.Q);
      acc.L *= w;
    }
    acc.R = mt;
  }
  const float dm = mt - acc.R;
  const float w = exp2f(dm);
  acc.L = fmaf(w, lt, acc.L);
  acc.Q = fmaf(w, fmaf(lt, dm, St), acc.Q);
}

// Reduction over the wpr warps of each row (warps r*wpr .. r*wpr + wpr - 1).
template <class T, class Op>
DG_DEV T rows_reduce(T v, Op op, T* sh, int wpr) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x / 32;
  if (threadIdx.x % 32 == 0) sh[warp] = v;
  __syncthreads();
  const int w0 = warp / wpr * wpr;
  T r = sh[w0];
  for (int w = 1; w < wpr; ++w) r = op(r, sh[w0 + w]);
  __syncthreads();
  return r;
}
DG_DEV RowSum shfl_rowsum(RowSum v, int o) {
  return {__shfl_xor_sync(0xffffffffu, v.R, o), __shfl_xor_sync(0xffffffffu, v.L, o),
          __shfl_xor_sync(0xffffffffu, v.Q, o)};
}

__global__ void __launch_bounds__(kStatsThreads) stats_kernel(StatsArgs a, int wpr, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int warp = threadIdx.x / 32;
  const int row = blockIdx.x * (kStatsWarps / wpr) + warp / wpr;
  const bool ok = row < a.M;
  const int t0 = (warp % wpr) * 32 + threadIdx.x % 32, tstep = wpr * 32;
  const size_t base = (size_t)(ok ? row : 0) * a.NT;
  __shared__ float shf[kStatsWarps];
  __shared__ int shi[kStatsWarps];
  __shared__ RowSum shr[kStatsWarps];
  RowSum acc{-FLT_MAX, 0.f, 0.f}, acc2{-FLT_MAX, 0.f, 0.f};
  float vbest = -FLT_MAX;
  int ibest = INT_MAX;
  if (ok) {
#pragma unroll 2
    for (int t = t0; t < a.NT; t += 2 * tstep) {
      const int t2 = t + tstep;
      const bool has2 = t2 < a.NT;
      const float4* r1 = reinterpret_cast<const float4*>(a.gst + base + t);
      const float4 x1 = r1[0], y1 = r1[1];
      float4 x2 = make_float4(-FLT_MAX, 0.f, 0.f, -FLT_MAX), y2 = make_float4(__int_as_float(INT_MAX), 0.f, 0.f, 0.f);
      if (has2) {
        const float4* r2 = reinterpret_cast<const float4*>(a.gst + base + t2);
        x2 = r2[0];
        y2 = r2[1];
      }
      const float m1 = x1.x, l1 = x1.y, S1 = x1.z, v1 = x1.w;
      const int i1 = __float_as_int(y1.x);
      const float m2 = x2.x, l2 = x2.y, S2 = x2.z, v2 = x2.w;
      const int i2 = __float_as_int(y2.x);
      if (v1 > vbest || (v1 == vbest && i1 < ibest)) {
        vbest = v1;
        ibest = i1;
      }
      if (v2 > vbest || (v2 == vbest && i2 < ibest)) {
        vbest = v2;
        ibest = i2;
      }
      add_group(acc, m1, l1, S1);
      if (has2) add_group(acc2, m2, l2, S2);
    }
  }
  acc = merge_rowsum(acc, acc2);
  // per row: the merged sums, and the argmax (largest value, lowest index)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = merge_rowsum(acc, shfl_rowsum(acc, o));
  if (threadIdx.x % 32 == 0) shr[warp] = acc;
  __syncthreads();
  const int w0 = warp / wpr * wpr;
  RowSum tot = shr[w0];
  for (int w = 1; w < wpr; ++w) tot = merge_rowsum(tot, shr[w0 + w]);
  const float vrow = rows_reduce(vbest, [](float x, float y) { return fmaxf(x, y); }, shf, wpr);
  const int irow =
      rows_reduce(vbest == vrow ? ibest : INT_MAX, [](int x, int y) { return x < y ? x : y; }, shi, wpr);
  if (!ok || t0 != 0) return;
  const double Z = (double)tot.L;
  const double H = log(Z) - 0.69314718055994531 * (double)tot.Q / Z;
  a.Hd[row] = H;
  a.lsum[row] = (float)Z;
  a.rowmax[row] = tot.R;
  a.amax[row] = irow;
  if (a.entropy) a.entropy[row] = (float)H;
  if (a.argmax_out) a.argmax_out[row] = irow;
}

cudaError_t launch_stats(const StatsArgs& a, StopCtl ctl, cudaStream_t st) {
  // warps per row: about 4 groups per thread, one to eight warps
  int wpr = 1;
  while (wpr < kStatsWarps && wpr * 32 * 4 < a.NT) wpr *= 2;
  const int rows_per_cta = kStatsWarps / wpr;
  return launch_pdl(stats_kernel, dim3(cdiv(a.M, rows_per_cta)), dim3(kStatsThreads), 0, st, a, wpr, ctl);
}

// ------------------------------------------- p0 and Gumbel-max sampling --
// The stored tiles of a row hold exp2(t - R) against the row's final reference
// R (kRefSpan; flagged rows were rewritten by lm_fix), so p0 = tile *
// exp2(R - m) / Z with one factor per row, which the contraction's reduce
// applies.  This pass searches, for the accepted rows only, the sample
// argmax_v (log p0_v + G_v), G_v the Gumbel noise of Philox stream 0 keyed by
// (seed, block, step, canvas, position, v), lowest index on ties (technical
// report summary, step 3: accepted positions take their predicted token; the
// Gumbel-max form of that draw is this library's reading).  The argmax token's
// p0 is 1/Z, so its perturbed score S_a = log(1/Z) + G_a is computed first; the
// largest draw is 16.64, so entries with log p0 < S_a - 16.64 - 0.02 can never
// win and skip the draw.  Rows that are not accepted are not read, nor are the
// tiles of a statistics group whose maximum (from the LM head's records) lies
// below that threshold: in the low-entropy rows that are accepted most groups
// are.
// One CTA per (row, 4096-entry chunk): larger chunks measured slower (16384:
// +2 us; 32768 with 16 loads in flight per thread: +22 us): the search wants
// many CTAs.  So did one CTA per row listing its candidate groups: quicker
// beside the long contraction at V = 262144, but a row whose accepted
// distribution leaves many groups above the threshold went through them eight
// warps at a time, and at V = 32768 (a short contraction) that lengthened the
// step.
constexpr int kP0Threads = kGumbelChunk / 32;
constexpr float kGumbelMaxDraw = 16.6355f;  // -log(-log(1 - 2^-24))

__global__ void __launch_bounds__(kP0Threads) p0_gumbel_kernel(P0Args a, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const bool gum = a.acc[row] && canvas_active(ctl.stop_at, row / a.C, ctl.step);
  if (!gum) return;  // uniform over the CTA
  const __nv_bfloat16* pt = reinterpret_cast<const __nv_bfloat16*>(a.pt) + (size_t)row * a.V;
  const int canvas = row / a.C, pos = row % a.C;
  const float mrow = a.rowmax[row], invZ = 1.0f / a.lsum[row];
  const float f = exp2f(a.ref2f[row] - mrow) * invZ;  // p0 = tile * f
  float best = -FLT_MAX;
  int bidx = INT_MAX;
  // Each warp takes 1024 contiguous entries (2 KB); load q of lane l is the
  // 16-byte chunk q * 32 + l, so a warp's load covers 512 contiguous bytes
  // (two statistics groups of 128 columns, one scale factor each).
  const int wbase = chunk * kGumbelChunk + (threadIdx.x / 32) * 1024;
  const int lane = threadIdx.x % 32;
  // the maxima of the statistics groups of this lane's four 8-entry pieces
  // (L2-resident records), read while the threshold's draw is computed
  const int NT = (a.V + kStatCols - 1) / kStatCols;
  float mg[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int v = wbase + (q * 32 + lane) * 8;
    mg[q] = v < a.V ? a.gst[(size_t)row * NT + v / kStatCols].m : -FLT_MAX;
  }
  // p0 threshold below which no entry can win the Gumbel-max search: the
  // argmax token's p0 is 1/Z, so its perturbed score S_a is known, and an
  // entry beats it only if log p0 + (largest draw) >= S_a.
  float thr = 0.f;
  if (gum) {
    const int va = a.amax[row];
    uint64_t wa[4];
    philox_block(wa, a.seed, a.block, a.step, canvas, pos, va >> 2, 0);
    const float sa = logf(invZ) + gumbel_from_word(wa[va & 3]);
    thr = expf(sa - kGumbelMaxDraw - 0.02f);
  }
  // A group whose largest p0, exp2(m_g - m) / Z (the tile holds it rounded
  // to bf16; a margin of 2^-6 covers that), is below the threshold holds no
  // candidate: its tiles are not read.
  bool need[4];
  uint4 x[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int v = wbase + (q * 32 + lane) * 8;
    need[q] = v < a.V && exp2f(mg[q] - mrow) * invZ * 1.015625f >= thr;
    if (need[q]) x[q] = *reinterpret_cast<const uint4*>(pt + v);  // V is a multiple of 8
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int vq = wbase + (q * 32 + lane) * 8;
    if (!need[q]) continue;
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&x[q]);
    float p[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) p[e] = __bfloat162float(xb[e]) * f;
#pragma unroll
    for (int g4 = 0; g4 < 2; ++g4) {
      bool any = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) any |= p[g4 * 4 + e] >= thr;
      if (!any) continue;
      uint64_t w[4];
      philox_block(w, a.seed, a.block, a.step, canvas, pos, (vq + g4 * 4) >> 2, 0);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = p[g4 * 4 + e];
        if (pv >= thr && pv > 0.f) {
          const float sc = logf(pv) + gumbel_from_word(w[e]);
          if (sc > best) {
            best = sc;
            bidx = vq + g4 * 4 + e;
          }
        }
      }
    }
  }
  // (score, lowest index) over the block
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (b2 > best || (b2 == best && i2 < bidx)) {
      best = b2;
      bidx = i2;
    }
  }
  __shared__ float sb[kP0Threads / 32];
  __shared__ int si[kP0Threads / 32];
  if (threadIdx.x % 32 == 0) {
    sb[threadIdx.x / 32] = best;
    si[threadIdx.x / 32] = bidx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kP0Threads / 32; ++k) {
      if (sb[k] > best || (sb[k] == best && si[k] < bidx)) {
        best = sb[k];
        bidx = si[k];
      }
    }
    a.gbest[(size_t)chunk * a.M + row] = best;
    a.gidx[(size_t)chunk * a.M + row] = bidx;
  }
}

cudaError_t launch_p0_gumbel(const P0Args& a, StopCtl ctl, cudaStream_t st) {
  dim3 grid(cdiv(a.V, kGumbelChunk), a.M);
  return launch_pdl(p0_gumbel_kernel, grid, dim3(kP0Threads), 0, st, a, ctl);
}

// --------------------------------------------------------------- sampler --
// Entropy-bounded acceptance ("DiffusionGemma Technical Report" summary,
// method step 3): positions sorted by ascending entropy (ties by position),
// the longest prefix whose cumulative entropy is <= b is accepted, every other
// position is renoised to a uniform random token (Philox stream 1).  Also the
// mean entropy, the accepted count and the adaptive-stop test of step 4
// (mean entropy <= stop_H and the argmax equal to the previous step's).
// One CTA per canvas, one thread per (padded) position:
//  - every global load and the Philox draw of the thread's own position are
//    issued first, so their latency overlaps the sort;
//  - (entropy as an order-preserving integer key, position) pairs are sorted
//    by a bitonic network: strides below 32 by warp shuffles, the others
//    through shared memory;
//  - the sorted entropies are summed in fixed point (units of 2^-44, exact
//    integer sums, so the result does not depend on the order of additions;
//    it differs from a double sum by < 1e-10);
//  - counts and the all-unchanged test are block ballots.
DG_DEV uint64_t order_key(double h) {
  const uint64_t b = (uint64_t)__double_as_longlong(h);
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);  // unsigned order = numeric order
}
constexpr double kFixScale = 17592186044416.0;  // 2^44
DG_DEV long long fixed_entropy(double h) {
  // |H| <= 32 for any finite entropy of V <= 2^31 tokens; anything else (not
  // finite) counts as 32 nats: never accepted, and 1024 of them cannot overflow
  return (h > -32.0 && h < 32.0) ? __double2ll_rn(h * kFixScale) : (long long)(32.0 * kFixScale);
}
DG_DEV bool sorts_before(uint64_t ka, int ia, uint64_t kb, int ib) { return ka < kb || (ka == kb && ia < ib); }

__global__ void __launch_bounds__(1024) sampler_kernel(SamplerArgs a, int npow2) {
  pdl_wait();
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  // Every canvas skips its work once it has stopped.
  if (a.stop_at[b] < a.step) return;
  __shared__ uint64_t sk[1024];
  __shared__ int si[1024];
  __shared__ long long sf[1024];
  __shared__ int stok[1024];
  __shared__ long long wsum[32];
  __shared__ long long total;
  const int base = b * a.C;
  const bool valid = t < a.C;
  // own position: entropy, argmax, previous argmax, renoise token
  double h = 0.0;
  int am = 0, prev = 0;
  if (valid) {
    h = a.Hd[base + t];
    am = a.amax[base + t];
    prev = a.prev_argmax[base + t];
    uint64_t pw[4];
    philox_block(pw, a.seed, a.block, a.step, b, t, 0, 1);
    stok[t] = uniform_token(pw[0], a.V);
    sf[t] = fixed_entropy(h);
  }
  const bool unchanged = !valid || (a.step >= 1 && prev == am);
  if (valid) a.prev_argmax[base + t] = am;
  uint64_t k = valid ? order_key(h) : ~0ull;
  int ix = t;
  const int all_unchanged = __syncthreads_and(unchanged);  // also publishes stok, sf
  // bitonic sort of (k, ix) ascending: thread t ends with the element of rank t
  for (int size = 2; size <= npow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint64_t ko;
      int io;
      if (stride >= 32) {
        sk[t] = k;
        si[t] = ix;
        __syncthreads();
        ko = sk[t ^ stride];
        io = si[t ^ stride];
        __syncthreads();
      } else {
        ko = __shfl_xor_sync(0xffffffffu, k, stride);
        io = __shfl_xor_sync(0xffffffffu, ix, stride);
      }
      // the lower index of a pair keeps the smaller element in an ascending
      // block (the larger in a descending one), the upper index the other
      const bool keep_min = ((t & stride) == 0) == ((t & size) == 0);
      const bool other_first = sorts_before(ko, io, k, ix);
      if (keep_min == other_first) {
        k = ko;
        ix = io;
      }
    }
  }
  // inclusive prefix sums of the sorted entropies (padding adds 0)
  const long long f = ix < a.C ? sf[ix] : 0ll;
  long long v = f;
  const int lane = t & 31, w = t >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) wsum[w] = v;
  __syncthreads();
  if (w == 0) {
    long long s = lane < (npow2 + 31) / 32 ? wsum[lane] : 0ll;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    wsum[lane] = s;  // inclusive totals of warps 0..lane
  }
  __syncthreads();
  if (w > 0) v += wsum[w - 1];
  if (t == a.C - 1) total = v;
  // accept the sorted prefix with cumulative entropy <= b
  const long long bfix = (long long)floor((double)a.b * kFixScale);
  const bool acc = t < a.C && v <= bfix;
  if (t < a.C) {
    const int pos = ix;
    a.acc[base + pos] = acc ? 1 : 0;
    if (a.acc_out) a.acc_out[base + pos] = acc ? 1 : 0;
    if (!acc) a.tokens[base + pos] = stok[pos];
  }
  const int n_acc = __syncthreads_count(acc);  // also publishes total
  if (t == 0) {
    const double meanH = (double)total / kFixScale / (double)a.C;
    const int stop = (a.step >= 1 && all_unchanged && meanH <= (double)a.stop_H) ? 1 : 0;
    if (a.n_acc) a.n_acc[b] = n_acc;
    if (a.mean_H) a.mean_H[b] = (float)meanH;
    if (a.stop) a.stop[b] = stop;
    if (a.accepted_log) a.accepted_log[(size_t)b * a.N + a.step] = n_acc;
    if (stop) {
      a.stop_at[b] = a.step;
      if (a.n_stopped) atomicAdd(a.n_stopped, 1);
    }
  }
}

cudaError_t launch_sampler(const SamplerArgs& a, cudaStream_t st) {
  int np = 32;
  while (np < a.C) np <<= 1;
  return launch_pdl(sampler_kernel, dim3(a.B), dim3(np), 0, st, a, np);
}

// ----------------------------------------- masked confidence decoding --
// The second sampler ("从零拆开DiffusionGemma" news piece, generate() of its
// fourth step): of the positions of a canvas still holding [MASK], the
// k = min(ceil(U / (N - step)), U) with the highest confidence take their
// candidate, the argmax; the others stay masked and revealed positions never
// change.  The confidence of a position is its largest tempered probability
// 1 / Z (the [MASK] column is left out of the softmax by the LM head), so the
// order is ascending Z, ties to the lower position.  One CTA per canvas, one
// thread per (padded) position, the bitonic network of sampler_kernel.
DG_DEV uint64_t z_key(float z) {
  // positive Z: the float's bits order like its value; anything else last
  return (z > 0.f && z < INFINITY) ? (uint64_t)__float_as_uint(z) : 0xfffffffeull;
}

__global__ void __launch_bounds__(1024) reveal_kernel(RevealArgs a, int npow2) {
  pdl_wait();
  const int b = blockIdx.x, t = threadIdx.x, base = b * a.C;
  const bool valid = t < a.C;
  __shared__ uint64_t sk[1024];
  __shared__ int si[1024];
  __shared__ long long wsum[32];
  bool unres = false;
  long long f = 0;
  if (valid) {
    unres = a.tokens[base + t] == a.mask_id;
    a.acc[base + t] = 0;
    if (a.acc_out) a.acc_out[base + t] = 0;
    a.prev_argmax[base + t] = a.amax[base + t];
    f = fixed_entropy(a.Hd[base + t]);
  }
  uint64_t k = unres ? z_key(a.lsum[base + t]) : ~0ull;
  int ix = t;
  const int U = __syncthreads_count(unres);
  for (int size = 2; size <= npow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint64_t ko;
      int io;
      if (stride >= 32) {
        sk[t] = k;
        si[t] = ix;
        __syncthreads();
        ko = sk[t ^ stride];
        io = si[t ^ stride];
        __syncthreads();
      } else {
        ko = __shfl_xor_sync(0xffffffffu, k, stride);
        io = __shfl_xor_sync(0xffffffffu, ix, stride);
      }
      const bool keep_min = ((t & stride) == 0) == ((t & size) == 0);
      const bool other_first = sorts_before(ko, io, k, ix);
      if (keep_min == other_first) {
        k = ko;
        ix = io;
      }
    }
  }
  const int remaining = a.N - a.step;
  int kk = (U + remaining - 1) / remaining;
  if (kk > U) kk = U;
  __syncthreads();  // every position's own writes above precede the reveal writes
  if (t < kk) {  // rank t < kk <= U: a masked position
    a.tokens[base + ix] = a.amax[base + ix];
    if (a.acc_out) a.acc_out[base + ix] = 1;
  }
  // mean entropy (exact fixed-point sum, as in the sampler)
  const int lane = t & 31, w = t >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) f += __shfl_xor_sync(0xffffffffu, f, o);
  if (lane == 0) wsum[w] = f;
  __syncthreads();
  if (t == 0) {
    long long tot = 0;
    for (int i = 0; i < (npow2 + 31) / 32; ++i) tot += wsum[i];
    if (a.n_acc) a.n_acc[b] = kk;
    if (a.mean_H) a.mean_H[b] = (float)((double)tot / kFixScale / (double)a.C);
    if (a.stop) a.stop[b] = 0;
    if (a.accepted_log) a.accepted_log[(size_t)b * a.N + a.step] = kk;
  }
}

cudaError_t launch_reveal(const RevealArgs& a, cudaStream_t st) {
  int np = 32;
  while (np < a.C) np <<= 1;
  return launch_pdl(reveal_kernel, dim3(a.B), dim3(np), 0, st, a, np);
}

__global__ void fill_tokens_kernel(int32_t* tokens, int n, int value) {
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n) tokens[t] = value;
}

cudaError_t launch_fill_tokens(int32_t* tokens, int n, int value, cudaStream_t st) {
  return launch_pdl(fill_tokens_kernel, dim3(cdiv(n, 256)), dim3(256), 0, st, tokens, n, value);
}

// ------------------------------------------------ self-conditioning reduce --
// u = sum of the per-split partials of p0 . E (bf16 out), and the Gumbel-max
// token of accepted positions = the best (score, lowest index) over chunks.
// Grid (M, G + 1): CTA (row, y < G) sums 128 float4 columns of the row, each
// thread one column with the loads of eight splits in flight at once (summed
// as a fixed tree per group of eight, the groups in order); CTA (row, G) picks
// the sampled token.
constexpr int kReduceCols = 128;

__global__ void __launch_bounds__(kReduceCols) reduce_kernel(ReduceArgs a, StopCtl ctl) {
  pdl_trigger();
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.x;
  const int n4 = a.d / 4;
  if ((int)blockIdx.y * kReduceCols < n4) {
    const int c = blockIdx.y * kReduceCols + threadIdx.x;
    if (c >= n4) return;
    const size_t sstride = (size_t)a.M * a.d;
    // the row's p0 factor (its tiles hold exp2(t - ref2f))
    const float fr = exp2f(a.ref2f[row] - a.rowmax[row]) / a.lsum[row];
    const float* src = a.upart + (size_t)row * a.d + 4 * c;
    float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < a.nsplit; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = s0 + k < a.nsplit ? *reinterpret_cast<const float4*>(src + (s0 + k) * sstride)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[k].x += v[k + 4].x;
        v[k].y += v[k + 4].y;
        v[k].z += v[k + 4].z;
        v[k].w += v[k + 4].w;
      }
      tot.x += (v[0].x + v[1].x) + (v[2].x + v[3].x);
      tot.y += (v[0].y + v[1].y) + (v[2].y + v[3].y);
      tot.z += (v[0].z + v[1].z) + (v[2].z + v[3].z);
      tot.w += (v[0].w + v[1].w) + (v[2].w + v[3].w);
    }
    uint2 w;
    w.x = pack_bf16(tot.x * fr, tot.y * fr);
    w.y = pack_bf16(tot.z * fr, tot.w * fr);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.u) + (size_t)row * a.d + 4 * c) = w;
    return;
  }
  // sampled token of an accepted row: the best (score, lowest index) over the
  // chunks, one warp
  if (threadIdx.x < 32 && a.acc[row] && canvas_active(ctl.stop_at, row / a.C, ctl.step)) {
    float best = -FLT_MAX;
    int bi = INT_MAX;
    for (int s = threadIdx.x; s < a.nchunks; s += 32) {
      const float v = a.gbest[(size_t)s * a.M + row];
      const int i = a.gidx[(size_t)s * a.M + row];
      if (v > best || (v == best && i < bi)) {
        best = v;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (b2 > best || (b2 == best && i2 < bi)) {
        best = b2;
        bi = i2;
      }
    }
    // no candidate only when the probabilities are not finite: keep the token
    if (threadIdx.x == 0) {
      if (bi >= 0 && bi < a.V)
        a.tokens[row] = bi;
      else
        atomicExch(a.status, kStatusValue);
    }
  }
}

cudaError_t launch_reduce(const ReduceArgs& a, StopCtl ctl, cudaStream_t st) {
  const int g = cdiv(a.d / 4, kReduceCols);
  return launch_pdl(reduce_kernel, dim3(a.M, g + 1), dim3(kReduceCols), 0, st, a, ctl);
}

// ------------------------------------------------- bounded-wait diagnostics --
// One thread waits on an mbarrier phase that nothing completes.  The bounded
// wait gives up after its limit, records DG_ERR_TIMEOUT in *status and the
// kernel returns: the path every pipeline takes when a copy or MMA it waits
// for never lands.
__global__ void wait_timeout_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, &abort_flag);
}

cudaError_t launch_wait_timeout(int* status, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

// ------------------------------------------------------- canvas + loop ----
__global__ void canvas_init_kernel(int32_t* tokens, int B, int C, int V, uint64_t seed, int block) {
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= B * C) return;
  uint64_t w[4];
  philox_block(w, seed, block, 0, t / C, t % C, 0, 2);
  tokens[t] = uniform_token(w[0], V);
}

cudaError_t launch_canvas_init(int32_t* tokens, int B, int C, int V, uint64_t seed, int block,
                               cudaStream_t st) {
  return launch_pdl(canvas_init_kernel, dim3(cdiv(B * C, 256)), dim3(256), 0, st, tokens, B, C, V, seed, block);
}

__global__ void loop_finish_kernel(const int* stop_at, int B, int N, int* steps_taken, int* converged,
                                   const int* prev_argmax, int* xhat0, int C) {
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < B) {
    const int s = stop_at[t];
    const bool conv = s < N;
    if (steps_taken) steps_taken[t] = conv ? s + 1 : N;
    if (converged) converged[t] = conv ? 1 : 0;
  }
  if (t < B * C && xhat0 && prev_argmax) xhat0[t] = prev_argmax[t];
}

cudaError_t launch_loop_finish(const int* stop_at, int B, int N, int* steps_taken, int* converged,
                               const int* prev_argmax, int* xhat0, int C, cudaStream_t st) {
  return launch_pdl(loop_finish_kernel, dim3(cdiv(B * C > B ? B * C : B, 256)), dim3(256), 0, st, stop_at, B, N,
                    steps_taken, converged, prev_argmax, xhat0, C);
}

// ------------------------------------------------- E4M3 quantization ----
// One warp per row of X (bf16 [R][d], d a multiple of 8): the row's absmax,
// then the codes of x * (448 / absmax) through the hardware's saturating
// round-to-nearest-even conversion.  Scale and its inverse are IEEE float32
// quotients, the product a float32 multiply, so the bytes are fixed by the
// definition.  A zero row gets scale 0 and zero codes.
__global__ void __launch_bounds__(256) quant_rows_e4m3_kernel(const __nv_bfloat16* __restrict__ X, int R, int d,
                                                              uint8_t* __restrict__ Q, float* __restrict__ scale) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= R) return;
  const uint4* x = reinterpret_cast<const uint4*>(X + (size_t)row * d);
  const int n8 = d / 8;
  float amax = 0.0f;
  for (int c = lane; c < n8; c += 32) {
    const uint4 u = __ldg(x + c);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  uint2* q = reinterpret_cast<uint2*>(Q + (size_t)row * d);
  if (!(amax > 0.0f)) {
    for (int c = lane; c < n8; c += 32) q[c] = make_uint2(0u, 0u);
    if (lane == 0) scale[row] = 0.0f;
    return;
  }
  const float inv = __fdiv_rn(448.0f, amax);
  if (lane == 0) scale[row] = __fdiv_rn(amax, 448.0f);
  for (int c = lane; c < n8; c += 32) {
    const uint4 u = __ldg(x + c);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      const uint32_t lo = __nv_cvt_float_to_fp8(__fmul_rn(f.x, inv), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float_to_fp8(__fmul_rn(f.y, inv), __NV_SATFINITE, __NV_E4M3);
      w[j >> 1] |= (lo | (hi << 8)) << (16 * (j & 1));
    }
    q[c] = make_uint2(w[0], w[1]);
  }
}

cudaError_t launch_quantize_rows_e4m3(const void* X, int R, int d, uint8_t* Q, float* scale, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  return launch_pdl(quant_rows_e4m3_kernel, dim3(cdiv(R, 8)), dim3(256), 0, st,
                    reinterpret_cast<const __nv_bfloat16*>(X), R, d, Q, scale);
}

// ------------------------------------------------ tile storage reference --
// R = alpha (h . E_ref) log2(e) / (sqrt(d) tau) per row, the larger of the
// values for E_ref = the current token and E_ref = the previous step's argmax
// (never the excluded column, so that R is at most the row's maximum); clears
// the row's flag.
__global__ void __launch_bounds__(128) lm_ref_kernel(RefArgs a, StopCtl ctl) {
  pdl_trigger();
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.x;
  // candidates: the current token and (from step 1) the previous step's argmax;
  // a reference only, so any column but the excluded one will do
  int t0 = min(max(a.tokens[row], 0), a.V - 1);
  int t1 = (a.step > 0 && a.prev_argmax) ? min(max(a.prev_argmax[row], 0), a.V - 1) : t0;
  if (t0 == a.excl) t0 = t1;
  if (t1 == a.excl) t1 = t0;
  if (t0 == a.excl) t0 = t1 = a.excl == 0 ? 1 : 0;
  const uint4* h = reinterpret_cast<const uint4*>(a.h) + (size_t)row * (a.d / 8);
  const uint4* e0 = reinterpret_cast<const uint4*>(a.E) + (size_t)t0 * (a.d / 8);
  const uint4* e1 = reinterpret_cast<const uint4*>(a.E) + (size_t)t1 * (a.d / 8);
  float acc0 = 0.f, acc1 = 0.f;
  for (int c = threadIdx.x; c < a.d / 8; c += blockDim.x) {
    const uint4 hv = __ldg(h + c), ev = __ldg(e0 + c), fv = __ldg(e1 + c);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&hv);
    const __nv_bfloat162* eb = reinterpret_cast<const __nv_bfloat162*>(&ev);
    const __nv_bfloat162* fb = reinterpret_cast<const __nv_bfloat162*>(&fv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = __bfloat1622float2(hb[j]), y = __bfloat1622float2(eb[j]), z = __bfloat1622float2(fb[j]);
      acc0 = fmaf(x.x, y.x, fmaf(x.y, y.y, acc0));
      acc1 = fmaf(x.x, z.x, fmaf(x.y, z.y, acc1));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    acc0 += __shfl_xor_sync(0xffffffffu, acc0, o);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, o);
  }
  __shared__ float red[2][4];
  if (threadIdx.x % 32 == 0) {
    red[0][threadIdx.x / 32] = acc0;
    red[1][threadIdx.x / 32] = acc1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float c = a.alpha[row] * a.coef2;
    const float r0 = c * ((red[0][0] + red[0][1]) + (red[0][2] + red[0][3]));
    const float r1 = c * ((red[1][0] + red[1][1]) + (red[1][2] + red[1][3]));
    const float R = fmaxf(r0, r1);  // the larger of two logits: still at most the row's maximum
    a.ref2[row] = R;
    a.ref2f[row] = R;
    a.rkey[row] = 0u;
  }
}

cudaError_t launch_lm_ref(const RefArgs& a, StopCtl ctl, cudaStream_t st) {
  return launch_pdl(lm_ref_kernel, dim3(a.M), dim3(128), 0, st, a, ctl);
}

// ------------------------------------------------ flagged-row rewrite --
// A flagged row (some group stored against its own maximum, kRefSpan) is
// rewritten against the row's maximum R' (the largest of those group maxima,
// rkey): a group stored against R scales by exp2(R - R') (< 2^-64: its
// values were negligible), one stored against its own maximum m_g by
// exp2(m_g - R'); R' becomes the row's final reference.  Needs only the group
// maxima, so it runs right after the LM head.  kFixSplit CTAs per row, each
// reading the row's flag once; those of unflagged rows return at once.
constexpr int kFixSplit = 4;
constexpr int kFixThreads = 256;
__global__ void __launch_bounds__(kFixThreads) lm_fix_kernel(FixArgs a, StopCtl ctl) {
  pdl_trigger();
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.y;
  const unsigned key = a.rkey[row];
  if (key == 0u) return;  // uniform over the CTA
  const float R = a.ref2[row], Rn = key_float(key);
  if (blockIdx.x == 0 && threadIdx.x == 0) a.ref2f[row] = Rn;
  const int NT = (a.V + kStatCols - 1) / kStatCols;
  const int per = ((a.V + kFixSplit - 1) / kFixSplit + 7) / 8 * 8;  // entries of this CTA, a multiple of 8
  const int v0 = blockIdx.x * per, v1 = min(a.V, v0 + per);
  __nv_bfloat16* pt = reinterpret_cast<__nv_bfloat16*>(a.pt) + (size_t)row * a.V;
  for (int v = v0 + threadIdx.x * 8; v < v1; v += kFixThreads * 8) {  // V is a multiple of 8
    const float mg = a.gst[(size_t)row * NT + v / kStatCols].m;
    const float f = exp2f((mg - R <= kRefSpan ? R : mg) - Rn);
    uint4 x = *reinterpret_cast<const uint4*>(pt + v);
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&x);
    uint4 y;
    y.x = pack_bf16(__bfloat162float(xb[0]) * f, __bfloat162float(xb[1]) * f);
    y.y = pack_bf16(__bfloat162float(xb[2]) * f, __bfloat162float(xb[3]) * f);
    y.z = pack_bf16(__bfloat162float(xb[4]) * f, __bfloat162float(xb[5]) * f);
    y.w = pack_bf16(__bfloat162float(xb[6]) * f, __bfloat162float(xb[7]) * f);
    *reinterpret_cast<uint4*>(pt + v) = y;
  }
}

cudaError_t launch_lm_fix(const FixArgs& a, StopCtl ctl, cudaStream_t st) {
  return launch_pdl(lm_fix_kernel, dim3(kFixSplit, a.M), dim3(kFixThreads), 0, st, a, ctl);
}

}  // namespace dg
