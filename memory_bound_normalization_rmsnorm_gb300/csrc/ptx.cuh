// ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the kernels
// use: mbarriers, bulk (TMA) global->shared copies with an L2 hint, 4-byte
// cp.async completions tracked by an mbarrier, cluster special registers,
// distributed shared memory loads and the split cluster barrier.
#pragma once
#include <cstdint>

namespace gbn {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarriers
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test with a suspend-time hint: a thread whose phase is not yet
// complete may sleep up to `ns` nanoseconds (or until the phase completes)
// instead of the hardware's default interval, issuing nothing meanwhile.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Error bits a kernel may set in the library's device error word.
constexpr unsigned kErrWaitTimeout = 1u;
// Number of try_wait polls before a wait is declared lost.  Each poll may
// suspend the thread for a short hardware-defined time, so this bounds the
// wait to seconds, never forever.
constexpr uint32_t kMaxPolls = 1u << 22;

// Waits for phase `parity` of `bar`.  Gives up after max_polls polls (or at
// once when another thread of the CTA already gave up, signalled through
// *abort), records the failure in *err and returns false.  The caller then
// carries on with whatever the stage holds: every address it touches stays
// in bounds, so a lost copy yields a wrong result and an error code, never
// a fault or a hang.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          unsigned *err, volatile int *abort,
                                          uint32_t max_polls = kMaxPolls) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < max_polls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  *abort = 1;
  atomicOr(err, kErrWaitTimeout);
  return false;
}

// mbar_wait whose polls may each sleep up to `ns` nanoseconds: warps that
// wait for a stage leave the issue slots to the row groups that compute.
// Same bound in polls (so at most kMaxPolls x ns when every poll sleeps in
// full: seconds for the hints the plans use).
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, unsigned *err,
                                                volatile int *abort, uint32_t ns) {
  if (mbar_try_wait_sleep(bar, parity, ns)) return true;
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait_sleep(bar, parity, ns)) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  *abort = 1;
  atomicOr(err, kErrWaitTimeout);
  return false;
}

// ------------------------------------------------------ bulk async copies
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(pol));
  return pol;
}

// One bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory; completion is counted
// in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem,
                                         uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 4-byte asynchronous copy global -> shared (non-bulk cp.async).
__device__ __forceinline__ void cp_async_4(void *dst_smem, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   smem_addr(dst_smem)),
               "l"(src)
               : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies have
// landed.  The pending-arrival count is raised first, so the net change to
// the phase's expected arrivals is zero.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// ------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive_release();
  cluster_wait_acquire();
}
// Shared::cluster address of `local` (this CTA's shared memory) in CTA
// `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(const void *local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_addr(local)), "r"(rank));
  return remote;
}

// Asynchronous 16-byte store into another CTA's shared memory whose
// completion is counted (in bytes) on that CTA's mbarrier `remote_bar`.
// Orders nothing else: no fence over this thread's other memory traffic.
__device__ __forceinline__ void st_async_f32x4(uint32_t remote_addr, float4 v,
                                               uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(remote_addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
      : "memory");
}

// ------------------------------------------------------------ barriers
// Named barrier for `nthreads` threads (multiple of 32) with id 1..15.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------- global stores
// 16-byte streaming store (evict-first in L2): outputs are written once.
__device__ __forceinline__ void st_global_cs_v4(void *p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_global_cs_v2(void *p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y)
               : "memory");
}

// One byte to global memory if `pred` (a predicated store: no branch).
__device__ __forceinline__ void st_global_u8_if(void *p, uint32_t v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %2, 0;\n\t"
      "@q st.global.u8 [%0], %1;\n\t}" ::"l"(p),
      "r"(v), "r"(static_cast<uint32_t>(pred))
      : "memory");
}

// Two fp32 values to two E4M3 codes (round to nearest even, saturating to
// +-448), packed with `lo` in the low byte (the lower address).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------- PDL controls
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace gbn
