// Bidirectional grouped-query attention of the canvas queries over the
// static prefix cache followed by the canvas keys, with no mask
// ("DiffusionGemma" docs chapter, attention-mask list: the current canvas is
// a full bidirectional matrix and it reads the prompt / finished-block KV
// cache; "DiffusionGemma explained", denoising mode).
//
// Flash-style: each CTA owns 64 query rows of one (canvas, query head) and one
// contiguous chunk of the key sequence; K/V blocks of 64 keys are streamed
// through shared memory with cp.async double buffering, scores and P.V use
// the warp-level MMA, the softmax is online in base 2.  Scores use bf16 q, k;
// the probabilities enter P.V as two f16 parts P_hi + P_lo (V re-encoded from
// bf16 to f16, exact in the f16 range), i.e. to ~2^-22.  With several
// chunks per row the CTAs write unnormalised partials that a combine kernel
// merges with their (max, sum).
#include <cfloat>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

template <int HD>
DG_DEV int swz(int r, int c) {
  if constexpr (HD >= 64) return c ^ (r & 7);
  else return c ^ ((r >> 1) & 3);
}

template <int HD>
__global__ void __launch_bounds__(128)
    attn_kernel(AttnArgs a, int nqt, int nsplit, int kps, float scale_log2, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  constexpr int CH = HD / 8;  // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sK = sQ + kAttnRows * HD;  // [2][64][HD]
  __nv_bfloat16* sV = sK + 2 * kAttnKeys * HD;

  const int split = blockIdx.x / nqt, qt = blockIdx.x % nqt;
  const int b = blockIdx.y / a.Hq, h = blockIdx.y % a.Hq;
  const int g = h / (a.Hq / a.Hkv);
  const int T = a.P + a.C;
  const int k_begin = split * kps;
  const int k_end = min(T, k_begin + kps);
  const int q0 = qt * kAttnRows;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  const __nv_bfloat16* Q = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + h) * a.C * HD;
  const __nv_bfloat16* Kp = reinterpret_cast<const __nv_bfloat16*>(a.Kp) + ((size_t)b * a.Hkv + g) * a.cap * HD;
  const __nv_bfloat16* Vp = reinterpret_cast<const __nv_bfloat16*>(a.Vp) + ((size_t)b * a.Hkv + g) * a.cap * HD;
  const __nv_bfloat16* Kc = reinterpret_cast<const __nv_bfloat16*>(a.kc) + ((size_t)b * a.Hkv + g) * a.C * HD;
  const __nv_bfloat16* Vc = reinterpret_cast<const __nv_bfloat16*>(a.vc) + ((size_t)b * a.Hkv + g) * a.C * HD;

  for (int idx = tid; idx < kAttnRows * CH; idx += 128) {
    const int r = idx / CH, c = idx % CH;
    const bool ok = q0 + r < a.C;
    cp_async16(sQ + r * HD + swz<HD>(r, c) * 8, Q + (size_t)(ok ? q0 + r : 0) * HD + c * 8, ok);
  }
  cp_async_commit();

  auto load_kv = [&](int blk, int buf) {
    const int kb0 = k_begin + blk * kAttnKeys;
    for (int idx = tid; idx < kAttnKeys * CH; idx += 128) {
      const int r = idx / CH, c = idx % CH;
      const int j = kb0 + r;
      const bool ok = j < k_end;
      const __nv_bfloat16 *ks, *vs;
      if (!ok) {
        ks = Kc;
        vs = Vc;
      } else if (j < a.P) {
        ks = Kp + (size_t)j * HD;
        vs = Vp + (size_t)j * HD;
      } else {
        ks = Kc + (size_t)(j - a.P) * HD;
        vs = Vc + (size_t)(j - a.P) * HD;
      }
      const int so = buf * kAttnKeys * HD + r * HD + swz<HD>(r, c) * 8;
      cp_async16(sK + so, ks + c * 8, ok);
      cp_async16(sV + so, vs + c * 8, ok);
    }
    cp_async_commit();
  };

  const int nblk = (k_end - k_begin + kAttnKeys - 1) / kAttnKeys;
  load_kv(0, 0);
  cp_async_wait<1>();
  __syncthreads();

  uint32_t qa[HD / 16][4];
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    const int mat = lane / 8;
    const int r = warp * 16 + (mat % 2) * 8 + lane % 8;
    const int c = ks * 2 + mat / 2;
    ldmatrix_x4(qa[ks], sQ + r * HD + swz<HD>(r, c) * 8);
  }

  float o[HD / 8][4];
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const int tq = lane % 4;

  for (int blk = 0; blk < nblk; ++blk) {
    const int buf = blk & 1;
    if (blk + 1 < nblk) load_kv(blk + 1, buf ^ 1);
    else cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const __nv_bfloat16* cK = sK + buf * kAttnKeys * HD;
    const __nv_bfloat16* cV = sV + buf * kAttnKeys * HD;

    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t kb[4];
        const int mat = lane / 8;
        const int key = j * 16 + (mat / 2) * 8 + lane % 8;
        const int c = ks * 2 + (mat % 2);
        ldmatrix_x4(kb, cK + key * HD + swz<HD>(key, c) * 8);
        mma_bf16_16816(s[2 * j], qa[ks], kb[0], kb[1]);
        mma_bf16_16816(s[2 * j + 1], qa[ks], kb[2], kb[3]);
      }
    }
    // Keys past the chunk end do not exist; with the causal mask (prefill),
    // canvas query i sees canvas keys 0..i only.
    const int kbase = k_begin + blk * kAttnKeys;
    const int qrow = q0 + warp * 16 + lane / 4;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kbase + n * 8 + 2 * tq + (e & 1);
        const bool seen = key < k_end && (!a.causal || key - a.P <= qrow + (e >> 1) * 8);
        s[n][e] = seen ? s[n][e] * scale_log2 : -INFINITY;
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float mx = -FLT_MAX;
#pragma unroll
      for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(s[n][2 * hr], s[n][2 * hr + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[hr], mx);
      // a row that has seen no key yet (all masked so far) keeps weight 0
      const float m_sub = m_new == -INFINITY ? 0.f : m_new;
      const float corr = exp2f(m_run[hr] - m_sub);
      float rs = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        s[n][2 * hr] = exp2f(s[n][2 * hr] - m_sub);
        s[n][2 * hr + 1] = exp2f(s[n][2 * hr + 1] - m_sub);
        rs += s[n][2 * hr] + s[n][2 * hr + 1];
      }
      l_run[hr] = l_run[hr] * corr + rs;
      m_run[hr] = m_new;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        o[n][2 * hr] *= corr;
        o[n][2 * hr + 1] *= corr;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float pv[8] = {s[2 * j][0], s[2 * j][1], s[2 * j][2], s[2 * j][3],
                           s[2 * j + 1][0], s[2 * j + 1][1], s[2 * j + 1][2], s[2 * j + 1][3]};
      uint32_t pa[4], pl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pa[e] = pack_f16(pv[2 * e], pv[2 * e + 1]);
        const __half2 hh = *reinterpret_cast<const __half2*>(&pa[e]);
        pl[e] = pack_f16(pv[2 * e] - __low2float(hh), pv[2 * e + 1] - __high2float(hh));
      }
#pragma unroll
      for (int dn = 0; dn < HD / 16; ++dn) {
        uint32_t vb[4];
        const int mat = lane / 8;
        const int key = j * 16 + (mat % 2) * 8 + lane % 8;
        const int c = dn * 2 + mat / 2;
        ldmatrix_x4_trans(vb, cV + key * HD + swz<HD>(key, c) * 8);
        const uint32_t v0 = bf16x2_to_f16x2(vb[0]), v1 = bf16x2_to_f16x2(vb[1]);
        const uint32_t v2 = bf16x2_to_f16x2(vb[2]), v3 = bf16x2_to_f16x2(vb[3]);
        mma_f16_16816(o[2 * dn], pa, v0, v1);
        mma_f16_16816(o[2 * dn], pl, v0, v1);
        mma_f16_16816(o[2 * dn + 1], pa, v2, v3);
        mma_f16_16816(o[2 * dn + 1], pl, v2, v3);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }
  const int gq = lane / 4;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = q0 + warp * 16 + gq + hr * 8;
    if (i >= a.C) continue;
    if (nsplit == 1) {
      const float inv = 1.0f / l_run[hr];
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.o) +
                           ((size_t)b * a.C + i) * ((size_t)a.Hq * HD) + (size_t)h * HD;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n)
        *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * tq) =
            pack_bf16(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
    } else {
      const size_t rowid = (((size_t)split * a.B + b) * a.Hq + h) * a.C + i;
      float* dst = a.opart + rowid * HD;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n)
        *reinterpret_cast<float2*>(dst + n * 8 + 2 * tq) = make_float2(o[n][2 * hr], o[n][2 * hr + 1]);
      if (tq == 0) *reinterpret_cast<float2*>(a.ml + rowid * 2) = make_float2(m_run[hr], l_run[hr]);
    }
  }
}

// Merge of the per-chunk partials: one warp per (canvas, head, query row),
// eight rows per CTA.  Lane s holds the (max, sum) of chunks s and s + 32; the
// head dim is split over the lanes (HD / 32 consecutive floats each).
constexpr int kCombineRows = 8;

template <int HD>
__global__ void __launch_bounds__(32 * kCombineRows) attn_combine_kernel(AttnArgs a, int nsplit, StopCtl ctl) {
  pdl_trigger();
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  constexpr int VEC = HD / 32;
  const int lane = threadIdx.x % 32;
  const size_t nrows = (size_t)a.B * a.Hq * a.C;
  const size_t row = (size_t)blockIdx.x * kCombineRows + threadIdx.x / 32;  // ((b * Hq + h) * C + i)
  if (row >= nrows) return;
  float m[2], l[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int s = lane + 32 * k;
    const float2 v = s < nsplit ? *reinterpret_cast<const float2*>(a.ml + (s * nrows + row) * 2)
                                : make_float2(-FLT_MAX, 0.f);
    m[k] = v.x;
    l[k] = v.y;
  }
  float M = fmaxf(m[0], m[1]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float w[2], L = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    w[k] = lane + 32 * k < nsplit ? exp2f(m[k] - M) : 0.f;
    L += w[k] * l[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int s = 0; s < nsplit; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w[s / 32], s % 32);
    const float* src = a.opart + (s * nrows + row) * HD + lane * VEC;
    if constexpr (VEC == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += v.x * ws;
      acc[1] += v.y * ws;
      acc[2] += v.z * ws;
      acc[3] += v.w * ws;
    } else if constexpr (VEC == 2) {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] += v.x * ws;
      acc[1] += v.y * ws;
    } else {
      acc[0] += src[0] * ws;
    }
  }
  const float inv = 1.0f / L;
  const int i = (int)(row % a.C);
  const int bh = (int)(row / a.C);
  const int b = bh / a.Hq, h = bh % a.Hq;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.o) + ((size_t)b * a.C + i) * ((size_t)a.Hq * HD) +
                       (size_t)h * HD + lane * VEC;
#pragma unroll
  for (int e = 0; e < VEC; ++e) dst[e] = __float2bfloat16_rn(acc[e] * inv);
}

void attn_split_mma(const dg_dims& D, int T, int* nsplit, int* keys_per_split) {
  const int nqt = cdiv(D.C, kAttnRows);
  const int units = nqt * D.B * D.Hq;
  int target = cdiv(3 * kTargetCtas, units);
  int ns = target < cdiv(T, 256) ? target : cdiv(T, 256);
  if (ns > kMaxAttnSplits) ns = kMaxAttnSplits;
  if (ns < 1) ns = 1;
  int kps = cdiv(cdiv(T, ns), kAttnKeys) * kAttnKeys;
  *keys_per_split = kps;
  *nsplit = cdiv(T, kps);
}

void attn_split(const dg_dims& D, int T, int P, int* nsplit, int* keys_per_split) {
  if (attn_use_tc(D, P)) attn_split_tc(D, T, nsplit, keys_per_split);
  else attn_split_mma(D, T, nsplit, keys_per_split);
}

int attn_max_splits(const dg_dims& D, int T) {
  int ns1, ns2, k;
  attn_split_mma(D, T, &ns1, &k);
  attn_split_tc(D, T, &ns2, &k);
  // the split count of either kernel grows with T, so T = cap + C bounds every prefix length
  return ns1 > ns2 ? ns1 : ns2;
}

cudaError_t launch_attention_combine(const AttnArgs& a, int nsplit, StopCtl ctl, cudaStream_t st) {
  if (nsplit > 64) return cudaErrorInvalidValue;
  const dim3 grid(cdiv((int64_t)a.B * a.Hq * a.C, kCombineRows)), block(32 * kCombineRows);
  switch (a.hd) {
    case 32: return launch_pdl(attn_combine_kernel<32>, grid, block, 0, st, a, nsplit, ctl);
    case 64: return launch_pdl(attn_combine_kernel<64>, grid, block, 0, st, a, nsplit, ctl);
    case 128: return launch_pdl(attn_combine_kernel<128>, grid, block, 0, st, a, nsplit, ctl);
  }
  return cudaErrorInvalidValue;
}

template <int HD>
static cudaError_t attn_impl(const AttnArgs& a, StopCtl ctl, cudaStream_t st) {
  dg_dims D{};
  D.C = a.C;
  D.B = a.B;
  D.Hq = a.Hq;
  D.Hkv = a.Hkv;
  D.hd = a.hd;
  const int T = a.P + a.C;
  int ns, kps;
  attn_split_mma(D, T, &ns, &kps);
  const int nqt = cdiv(a.C, kAttnRows);
  const size_t smem = (size_t)(kAttnRows + 4 * kAttnKeys) * HD * 2;
  auto kern = attn_kernel<HD>;
  cudaError_t e = set_smem_once<attn_kernel<HD>>((int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  dim3 grid(nqt * ns, a.B * a.Hq);
  e = launch_pdl(kern, grid, dim3(128), smem, st, a, nqt, ns, kps, scale_log2, ctl);
  if (e != cudaSuccess || ns == 1) return e;
  return launch_attention_combine(a, ns, ctl, st);
}

cudaError_t launch_attention(const AttnArgs& a, StopCtl ctl, int* status, cudaStream_t st) {
  dg_dims D{};
  D.hd = a.hd;
  if (!a.causal && attn_use_tc(D, a.P)) return launch_attention_tc(a, ctl, status, st);
  switch (a.hd) {
    case 32: return attn_impl<32>(a, ctl, st);
    case 64: return attn_impl<64>(a, ctl, st);
    case 128: return attn_impl<128>(a, ctl, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
