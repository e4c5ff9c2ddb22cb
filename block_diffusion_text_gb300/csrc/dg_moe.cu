// Mixture-of-experts FFN of a layer (the DiffusionGemma backbone's FFN: the
// "文本 Diffusion 模型" survey page, §11 -- 128 experts per layer, 8 routed
// plus one shared -- and §13 -- router top-k, expert GEMM, token permutation;
// the "DiffusionGemma Technical Report" summary, MoE paragraph -- expert
// weight traffic is the bottleneck of a denoising step, a canvas activating
// far more experts than one token).
//
// One layer's block on the rows h [M][d], x = RMSNorm(h) (bf16, computed by
// the embedding / RMSNorm kernel):
//   route    fp32 router logits x . Wr_e, top_k experts per row (value
//            descending, lower index on ties), gates = softmax over the
//            selected logits
//   plan     one CTA: the M * (top_k + 1) assignments (the shared expert
//            takes every row) sorted by expert, rows in increasing order
//            within an expert, and the table of row tiles per expert
//            (kMoeTileRows rows each)
//   gather   the expert-sorted copy of x
//   experts  two grouped tcgen05 GEMMs (dg_gemm.cu), the expert's weights
//            as the 128-row operand and a tile of its rows as N:
//            GELU(x We1_e^T), then gate * (. We2_e^T) in fp32
//   combine  h += sum over the row's assignments in rank order, then the
//            shared expert (fp32), rounded to bf16
// Every weight matrix of an active expert is read once per layer and step
// (the tiles of an expert's rows run side by side and share its weight
// tiles), which is the HBM floor of the block.
#include <cfloat>
#include <climits>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

constexpr int kTopkRows = 8;  // rows per top-k CTA, one warp each

DG_DEV void bf16x8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 p = __bfloat1622float2(b[j]);
    f[2 * j] = p.x;
    f[2 * j + 1] = p.y;
  }
}

// Router logits from the K-split partials of the router GEMM x Wr^T (summed in
// split order), then the row's top_k: one warp per row, lane holding experts
// lane, lane + 32, ... (n_exp <= 256).
__global__ void __launch_bounds__(kTopkRows * 32) moe_topk_kernel(MoeRouteArgs a, const float* __restrict__ part,
                                                                  int ksplit, int* status, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row = blockIdx.x * kTopkRows + warp;
  if (row >= a.M) return;
  // the row's logits, summed over the K splits in order; the loads of four
  // splits of every expert of the lane are in flight at once
  float l[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) l[j] = 0.f;
  for (int sp0 = 0; sp0 < ksplit; sp0 += 4) {
    float t[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        t[j][k] = (e < a.n_exp && sp0 + k < ksplit) ? part[((size_t)(sp0 + k) * a.M + row) * a.n_exp + e] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) l[j] += t[j][k];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane + 32 * j;
    if (a.dbg_logits && e < a.n_exp) a.dbg_logits[(size_t)row * a.n_exp + e] = l[j];
  }
  uint32_t taken = 0;
  float top = 0.f, Z = 0.f;
  float sv[kMoeMaxTopK];
  int se[kMoeMaxTopK];
#pragma unroll 1
  for (int k = 0; k < a.top_k; ++k) {
    float bv = -FLT_MAX;
    int be = INT_MAX;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      if (e < a.n_exp && !((taken >> j) & 1u) && (l[j] > bv || (l[j] == bv && e < be))) {
        bv = l[j];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be < 0 || be >= a.n_exp) {  // non-finite logits: record and route to a valid expert
      if (lane == 0) atomicExch(status, kStatusValue);
      be = k;
      bv = -FLT_MAX;
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (k == 0) top = bv;
    sv[k] = bv;
    se[k] = be;
  }
  for (int k = 0; k < a.top_k; ++k) Z += expf(sv[k] - top);
  if (lane < a.top_k) {
    float v = sv[0];
    int e = se[0];
    for (int k = 1; k < a.top_k; ++k)
      if (k == lane) {
        v = sv[k];
        e = se[k];
      }
    const float g = expf(v - top) / Z;
    a.idx[(size_t)row * a.top_k + lane] = e;
    a.gate[(size_t)row * a.top_k + lane] = g;
    if (a.dbg_idx) a.dbg_idx[(size_t)row * a.top_k + lane] = e;
    if (a.dbg_gate) a.dbg_gate[(size_t)row * a.top_k + lane] = g;
  }
}

cudaError_t launch_moe_route(const MoeRouteArgs& a, float* part, size_t part_elems, int* status, StopCtl ctl,
                             cudaStream_t st) {
  int ks = gemm_ksplit(a.M, a.n_exp, a.d);
  while (ks > 1 && (size_t)ks * a.M * a.n_exp > part_elems) --ks;
  cudaError_t e = launch_gemm_f32_partials(a.x, a.Wr, part, a.M, a.n_exp, a.d, ks, ctl, status, st);
  if (e != cudaSuccess) return e;
  return launch_pdl(moe_topk_kernel, dim3(cdiv(a.M, kTopkRows)), dim3(kTopkRows * 32), 0, st, a,
                    (const float*)part, ks, status, ctl);
}

// The expert-sorted permutation and the tile table, in one CTA.  A bitmap per
// expert over the rows gives, for each assignment, its rank among the
// expert's rows (a prefix popcount), so the order is fixed by the data alone.
__global__ void __launch_bounds__(1024) moe_plan_kernel(MoePlanArgs a, int* status, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  extern __shared__ uint32_t sm_plan[];
  const int G = a.n_exp + 1, W = (a.M + 31) / 32, K1 = a.top_k + 1;
  const int R = a.M * K1;
  uint32_t* bm = sm_plan;                               // [G][W]
  int* cnt = reinterpret_cast<int*>(bm + (size_t)G * W);  // [G]
  int* off = cnt + G;                                   // [G + 1]
  int* toff = off + G + 1;                              // [G + 1]
  for (int i = threadIdx.x; i < G * W; i += blockDim.x) bm[i] = 0u;
  for (int p = threadIdx.x; p < R; p += blockDim.x) {
    a.ptok[p] = 0;
    a.pgate[p] = 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.M * a.top_k; i += blockDim.x) {
    int e = a.idx[i];
    if (e < 0 || e >= a.n_exp) {
      atomicExch(status, kStatusValue);
      e = 0;
    }
    const int t = i / a.top_k;
    atomicOr(&bm[(size_t)e * W + t / 32], 1u << (t % 32));
  }
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    const int left = a.M - 32 * w;
    bm[(size_t)a.n_exp * W + w] = left >= 32 ? 0xffffffffu : ((1u << left) - 1u);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < W; ++w) c += __popc(bm[(size_t)e * W + w]);
    cnt[e] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int o = 0, to = 0;
    for (int e = 0; e < G; ++e) {
      off[e] = o;
      toff[e] = to;
      o += cnt[e];
      to += (cnt[e] + kMoeTileRows - 1) / kMoeTileRows;
    }
    off[G] = o;
    toff[G] = to;
    a.tiles[0] = make_int4(min(to, a.max_tiles), 0, 0, 0);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    for (int j = 0; j * kMoeTileRows < cnt[e]; ++j) {
      const int ti = toff[e] + j;
      if (ti < a.max_tiles)
        a.tiles[1 + ti] = make_int4(e, off[e] + kMoeTileRows * j, min(kMoeTileRows, cnt[e] - kMoeTileRows * j), 0);
    }
  }
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    const int t = i / K1, j = i % K1;
    int e;
    float g;
    if (j < a.top_k) {
      e = a.idx[(size_t)t * a.top_k + j];
      if (e < 0 || e >= a.n_exp) e = 0;
      g = a.gate[(size_t)t * a.top_k + j];
    } else {
      e = a.n_exp;
      g = 1.0f;
    }
    const uint32_t* row = bm + (size_t)e * W;
    int rank = __popc(row[t / 32] & ((1u << (t % 32)) - 1u));
    for (int w = 0; w < t / 32; ++w) rank += __popc(row[w]);
    const int p = min(off[e] + rank, R - 1);
    a.slot[i] = p;
    a.ptok[p] = t;
    a.pgate[p] = g;
  }
}

int moe_plan_smem(int M, int n_exp) {
  const int G = n_exp + 1, W = (M + 31) / 32;
  return (G * W + 3 * (G + 1)) * 4;
}

cudaError_t launch_moe_plan(const MoePlanArgs& a, int* status, StopCtl ctl, cudaStream_t st) {
  cudaError_t e = set_smem_once<moe_plan_kernel>(moe_plan_smem(kMoeMaxRows, kMoeMaxExperts));
  if (e != cudaSuccess) return e;
  return launch_pdl(moe_plan_kernel, dim3(1), dim3(1024), (size_t)moe_plan_smem(a.M, a.n_exp), st, a, status,
                    ctl);
}

__global__ void __launch_bounds__(256) moe_gather_kernel(const uint4* __restrict__ x, const int* __restrict__ ptok,
                                                         uint4* __restrict__ xp, int R, int d8, int M, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)R * d8) return;
  const int p = (int)(i / d8), c = (int)(i % d8);
  const int t = min(max(ptok[p], 0), M - 1);
  xp[i] = __ldg(x + (size_t)t * d8 + c);
}

cudaError_t launch_moe_gather(const void* x, const int* ptok, void* xp, int R, int d, int M, StopCtl ctl,
                              cudaStream_t st) {
  const size_t n = (size_t)R * (d / 8);
  return launch_pdl(moe_gather_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st,
                    reinterpret_cast<const uint4*>(x), ptok, reinterpret_cast<uint4*>(xp), R, d / 8, M, ctl);
}

// One thread per 8 columns of a row: the row's gated expert outputs summed in
// rank order, then the shared expert, added to h and rounded once.
__global__ void __launch_bounds__(256) moe_combine_kernel(__nv_bfloat16* h, const float* __restrict__ yp,
                                                          const int* __restrict__ slot, int M, int d, int K1,
                                                          int C, StopCtl ctl) {
  pdl_wait();
  if (all_stopped(ctl.stop_at, ctl.B, ctl.step)) return;
  const int row = blockIdx.y;
  const int c8 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c8 >= d || !canvas_active(ctl.stop_at, row / C, ctl.step)) return;
  const int R = M * K1;
  // the row's slots first (one round trip), then the loads of up to eight
  // gated outputs in flight at once, summed in rank order
  int ps[kMoeMaxTopK + 1];
#pragma unroll
  for (int j = 0; j < kMoeMaxTopK + 1; ++j)
    ps[j] = j < K1 ? min(max(slot[(size_t)row * K1 + j], 0), R - 1) : 0;
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j0 = 0; j0 < kMoeMaxTopK + 1; j0 += 8) {
    if (j0 >= K1) break;
    float4 u[8], v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (j0 + k < K1) {
        const float4* src = reinterpret_cast<const float4*>(yp + (size_t)ps[j0 + k] * d + c8);
        u[k] = src[0];
        v[k] = src[1];
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (j0 + k < K1) {
        s[0] += u[k].x; s[1] += u[k].y; s[2] += u[k].z; s[3] += u[k].w;
        s[4] += v[k].x; s[5] += v[k].y; s[6] += v[k].z; s[7] += v[k].w;
      }
    }
  }
  uint4* hp = reinterpret_cast<uint4*>(h + (size_t)row * d + c8);
  float hv[8];
  bf16x8(*hp, hv);
  *hp = make_uint4(pack_bf16(hv[0] + s[0], hv[1] + s[1]), pack_bf16(hv[2] + s[2], hv[3] + s[3]),
                   pack_bf16(hv[4] + s[4], hv[5] + s[5]), pack_bf16(hv[6] + s[6], hv[7] + s[7]));
}

cudaError_t launch_moe_combine(void* h, const float* yp, const int* slot, int M, int d, int top_k, int C,
                               StopCtl ctl, cudaStream_t st) {
  dim3 grid(cdiv(d / 8, 256), M);
  return launch_pdl(moe_combine_kernel, grid, dim3(256), 0, st, reinterpret_cast<__nv_bfloat16*>(h), yp, slot, M,
                    d, top_k + 1, C, ctl);
}

}  // namespace dg
