// kq_ptx.cuh -- thin inline-PTX wrappers for sm_103a used by the kq kernels:
// mbarriers, 1-D TMA bulk copies (global -> shared), L2 bulk prefetch,
// programmatic dependent launch, packed fp32x2 FMA, and the library's device
// error word.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kq {

// ---------------------------------------------------------------------------
// Device error word: kernels never trap.  A bounded wait that gives up, or a
// bad index found on the device, records a code here and the kernel returns.
// ---------------------------------------------------------------------------
enum : int {
  DEV_OK = 0,
  DEV_ERR_MBAR_TIMEOUT = 1,   // a TMA stage never completed within the wait bound
  DEV_ERR_EXPERT_ID = 2,      // routed expert id outside [0, n_experts)
  DEV_ERR_TMEM = 3,           // tensor-memory allocation not granted
};
// The word lives in the API translation unit; kernels receive its address.
__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, DEV_OK, code);
}

// A waiting thread sleeps inside try_wait for up to kSuspendNs (it wakes as
// soon as the phase completes), so a wait costs a few instructions instead of
// a spin.  kMaxPolls bounds the total wait at a few seconds -- far above any
// legitimate copy latency -- after which the wait is declared failed.
constexpr uint32_t kSuspendNs = 2000;
constexpr uint32_t kMaxPolls = 1u << 21;

__host__ __device__ __forceinline__ int64_t min_i64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded wait for the given phase parity; false (and the error word set) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  for (uint32_t i = 0; i < kMaxPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  record_error(err, DEV_ERR_MBAR_TIMEOUT);
  return false;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Ask L2 to fetch [src, src+bytes) (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: wait for the preceding grid's memory to be
// visible / allow the next grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// d = a * b + c on two fp32 lanes at once (round to nearest, no reassociation).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

}  // namespace kq
