// Device helpers shared by the kernels of libdg: inline-PTX wrappers for
// mbarriers, TMA tensor copies, tcgen05 (TMEM allocation, MMA, loads), the
// legacy warp-level MMA used by attention, and the Philox4x64-10 generator.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DG_DEV __device__ __forceinline__

namespace dg {

constexpr int kStatusTimeout = 6;  // DG_ERR_TIMEOUT
constexpr int kStatusValue = 7;    // DG_ERR_VALUE
// Upper bound of any spin on an mbarrier (ns of %globaltimer).  A healthy
// pipeline never waits more than microseconds; past this the kernel records
// DG_ERR_TIMEOUT in the status word and winds down instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

DG_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

DG_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------- programmatic launches ----
// Every kernel of the library begins with pdl_wait(): wait until the kernel
// before it in the stream has completed and its writes are visible (a no-op
// when launched without programmatic serialisation).  The short kernels on the
// step's critical path (embedding, attention merge, tile reference, flagged-row
// rewrite, reduce) call pdl_trigger() first, so that the GEMM or attention
// after them is launched while they run and its CTAs wait on the SMs they
// leave free; the long kernels do not, since CTAs of the next kernel parked
// beside them cost more than the launch latency they hide (measured).
// pdl_trigger() only allows the launch: the dependent's pdl_wait() still
// waits for this kernel's completion.  The tensor-core GEMM kernels call
// pdl_wait() after their prologue (barrier initialisation, TMEM allocation,
// cluster synchronisation), which reads nothing the kernel before wrote, so
// that the prologue of a GEMM launched early overlaps the short kernel
// before it.  No kernel that holds TMEM triggers early, so such a prologue
// never waits on TMEM held by a kernel still running.
DG_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DG_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------- mbarrier ----
DG_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
DG_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
DG_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
DG_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// kCluster: acquire at cluster scope, for phases completed by arrivals from
// other CTAs of the cluster that release their remote shared-memory stores.
template <bool kCluster = false>
DG_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if (kCluster) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}
// Bounded wait for the phase with the given parity.  Returns false (after
// recording the timeout in *status and raising *abort) if the wait ran out or
// another role of the CTA already gave up.
template <bool kCluster = false>
DG_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort) {
#pragma unroll 1
  for (int i = 0; i < 256; ++i)
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait<kCluster>(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicExch(status, kStatusTimeout);
      *abort = 1;
      return false;
    }
  }
}

// The same wait taken by a whole warp that goes on to warp-collective
// tcgen05 loads / stores: every lane gets the same answer, so the warp never
// splits between a lane that gave up and one that carries on.
template <bool kCluster = false>
DG_DEV bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* status, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait<kCluster>(bar, parity, status, abort));
}

// ------------------------------------------------------------------ TMA ----
DG_DEV void tma_prefetch(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled copy global -> shared, completion counted on `bar` (bytes).
// c0 is the innermost coordinate (elements).
DG_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// -------------------------------------------------------------- tcgen05 ----
DG_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
DG_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
DG_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
DG_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DG_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulation.
DG_DEV void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], bf16 inputs, fp32 accumulation: A (M = 128
// rows, one per TMEM lane) is read from TMEM, two bf16 of consecutive K per
// 32-bit column, so one K = 16 step spans 8 columns.
DG_DEV void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive on `bar` once all previously issued MMAs of this thread completed.
DG_DEV void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
DG_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Warp-collective: lane t of the warp receives 32 consecutive 32-bit columns
// (starting at the column of taddr) of TMEM lane (lane field of taddr) + t.
DG_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tmem_ld32 without the wait: several loads may be in flight; complete them
// with tmem_wait_ld() before reading v.
DG_DEV void tmem_ld32_async(uint32_t taddr, float (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]),
        "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]),
        "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
      : "r"(taddr)
      : "memory");
}
// Warp-collective load of 16 consecutive 32-bit columns per lane (waits).
DG_DEV void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
  tmem_wait_ld();
}
// Warp-collective store of 16 consecutive 32-bit columns per lane.
DG_DEV void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

DG_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Instruction descriptor of tcgen05.mma kind::f16 with f16 A and B (fp32 D).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4)                                  // D format: f32
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness (A, B format 0 = f16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B (format
// 0 in both fields), fp32 D, both K-major, shape M x N (K = 32 per instruction).
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4)                                  // D format: f32
         | ((uint32_t)(N >> 3) << 17)               // N / 8
         | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 D,
// A K-major, B K-major or MN-major, shape M x N (K = 16 per instruction).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | ((uint32_t)(N >> 3) << 17)               // N / 8
         | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 layout version 1).
// K-major operand: rows of 64 bf16 (128 B), 8-row groups 1024 B apart (SBO).
// MN-major operand: 64-element (128 B) wide columns of 8-row K groups; LBO is
// the byte distance between 64-element column blocks along M/N, SBO between
// 8-row groups along K.
DG_DEV uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// ------------------------------------------------------------ CTA pairs ----
// A cluster of two CTAs on two SMs runs one tcgen05 MMA of M = 256: each CTA
// holds 128 rows of A and half of the N columns of B in its own shared
// memory, and receives its 128 rows of D in its own TMEM.  CTA rank 0 (the
// leader) issues the MMAs; both CTAs allocate TMEM together.
DG_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
DG_DEV uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
DG_DEV uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of both CTAs; orders shared-memory writes before it (release)
// with reads after it (acquire) across the cluster.
DG_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address, in the cluster's shared window, of the same variable in CTA `rank`.
DG_DEV uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrive on an mbarrier of either CTA of the pair (default .release.cta
// semantics: the callers signal completed tcgen05 stores or loads, ordered by
// tcgen05.wait and tcgen05.fence::before_thread_sync; a cluster-scope
// release would add a memory barrier to every call).
DG_DEV void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// Store of four floats into the shared memory of a CTA of the cluster
// (cluster address), and an arrival on an mbarrier there that releases this
// thread's earlier stores at cluster scope (the waiter acquires them with
// mbar_wait<true>).
DG_DEV void st_cluster_v4(uint32_t caddr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
DG_DEV void mbar_arrive_cluster_release(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// 2-D tiled copy into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (cluster address).
DG_DEV void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_caddr, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_caddr), "r"(c0), "r"(c1)
      : "memory");
}
DG_DEV void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
DG_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
DG_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (M = 256 over the pair) (+)= A * B; issued by the leader only.
DG_DEV void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// The same with E4M3 operands (kind::f8f6f4): 32 bytes of K per instruction,
// as for bf16, so the shared-memory descriptors advance alike.
DG_DEV void umma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive on the mbarrier at `bar`'s offset in both CTAs of the pair once all
// previously issued pair MMAs of this thread completed.
DG_DEV void umma_commit_pair(uint64_t* bar) {
  const uint16_t mask = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// ------------------------------------------------ paired fp32 arithmetic ----
// Two fp32 lanes in one 64-bit register (sm_100 f32x2 instructions).
DG_DEV uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
DG_DEV void f2_unpack(uint64_t v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
DG_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
DG_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
DG_DEV uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
DG_DEV float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------ legacy warp-level MMA ----
DG_DEV void cp_async16(void* dst, const void* src, bool pred) {
  int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(sz)
               : "memory");
}
DG_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DG_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
DG_DEV void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
DG_DEV void ldmatrix_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
DG_DEV void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
DG_DEV void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
DG_DEV uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// Two bf16 (low, high halves of r) re-encoded as two f16 (exact for
// magnitudes in the f16 normal range).
DG_DEV uint32_t bf16x2_to_f16x2(uint32_t r) {
  return pack_f16(__uint_as_float(r << 16), __uint_as_float(r & 0xffff0000u));
}
DG_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------- Philox ------
// Philox4x64-10 (Salmon et al., SC'11): ten rounds of two 64x64->128-bit
// multiplications by the Philox constants, mixing the high halves with the
// other two counter words and the round key; the key advances by the Weyl
// constants between rounds.
DG_DEV void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += W0;
      k1 += W1;
    }
    uint64_t lo0 = M0 * c[0], hi0 = __umul64hi(M0, c[0]);
    uint64_t lo1 = M1 * c[2], hi1 = __umul64hi(M1, c[2]);
    uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}
// The Philox block of (seed, block, step, canvas, position, v >> 2, stream):
// counter = (v >> 2, pos, block << 32 | step, canvas << 32 | stream), key = (seed, 0).
// Word v & 3 of the block is the draw of vocabulary index v.
DG_DEV void philox_block(uint64_t (&out)[4], uint64_t seed, int block, int step, int canvas, int pos,
                         int64_t v4, int stream) {
  out[0] = (uint64_t)v4;
  out[1] = (uint64_t)(uint32_t)pos;
  out[2] = ((uint64_t)(uint32_t)block << 32) | (uint32_t)step;
  out[3] = ((uint64_t)(uint32_t)canvas << 32) | (uint32_t)stream;
  philox4x64_10(out, seed, 0);
}
// Uniform token in [0, V): high word of w * V.
DG_DEV int32_t uniform_token(uint64_t w, int32_t V) { return (int32_t)__umul64hi(w, (uint64_t)V); }
// Standard Gumbel noise from a 64-bit word: U = (top 23 bits + 1/2) / 2^23.
DG_DEV float gumbel_from_word(uint64_t w) {
  float u = ((float)(uint32_t)(w >> 41) + 0.5f) * (1.0f / 8388608.0f);
  return -logf(-logf(u));
}

// Canvas b is still denoising at `step` unless its stop test fired earlier.
// Order-preserving unsigned key of a float (unsigned order = numeric order;
// 0 is below every finite value) and its inverse.
DG_DEV unsigned float_key(float f) {
  const unsigned b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DG_DEV float key_float(unsigned k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }
DG_DEV bool canvas_active(const int* stop_at, int b, int step) {
  return stop_at == nullptr || stop_at[b] >= step;
}
DG_DEV bool all_stopped(const int* stop_at, int B, int step) {
  if (stop_at == nullptr) return false;
  for (int b = 0; b < B; ++b)
    if (stop_at[b] >= step) return false;
  return true;
}

}  // namespace dg
