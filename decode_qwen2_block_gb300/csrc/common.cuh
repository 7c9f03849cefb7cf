// Device helpers shared by the block kernels: PTX wrappers for mbarriers,
// bulk (TMA) copies, programmatic dependent launch, and bounded waits that
// record an error instead of hanging.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace blk {

// Device status codes written to the handle's status word (first one wins).
constexpr int kDevTimeout = 1;
constexpr int kDevPosition = 2;
constexpr int kDevToken = 3;     // a token id outside [0, vocab)

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---- programmatic dependent launch ----------------------------------------
// wait: blocks until the preceding kernel in the stream has completed and its
// writes are visible (a no-op when launched without the PDL attribute).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// launch_dependents: lets the next kernel's CTAs be scheduled.  Every kernel
// here calls it only after its own wait, so at most two kernels of a chain
// overlap and everything older is complete.
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// records kDevTimeout) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      set_error(err, kDevTimeout);
      return false;
    }
  }
  return true;
}

// Brings a tensor map (a kernel parameter or global memory) into the TMA
// unit's descriptor cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tmap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- bulk copies (TMA, untiled) ----------------------------------------------
// Copies `bytes` (multiple of 16, both addresses 16-byte aligned) from global
// to shared memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc,
                                         uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Hints the L2 to fetch [gsrc, gsrc + bytes) (multiple of 16, 16B aligned).
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc,
                                                 uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc),
               "r"(bytes)
               : "memory");
}

// Named barrier among `nthreads` threads (id 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- sliding window ---------------------------------------------------------
// First slot a query in slot `last` attends: with a sliding window of
// `window` slots the last `window` slots (its own included), else slot 0.
__host__ __device__ __forceinline__ int64_t window_lo(int64_t window, int64_t last) {
  return (window > 0 && last + 1 > window) ? last + 1 - window : 0;
}

// ---- small math --------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// silu(z) = z / (1 + e^-z) with the single-path fast divide: an IEEE divide
// takes a long special-case path for huge or non-finite operands, which rows
// past the end of a tile can hold.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// 8 fp16 values (one 16-byte vector) to fp32.
__device__ __forceinline__ void h8_to_f32(const uint4& v, float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Looks up (cos, sin) for position `p` and pair index `i`; clamps an
// out-of-range position and records kDevPosition.
__device__ __forceinline__ float2 rope_cs(const float2* table, int64_t len,
                                          int half_d, int64_t p, int i,
                                          int* err) {
  if (p < 0 || p >= len) {
    set_error(err, kDevPosition);
    p = p < 0 ? 0 : len - 1;
  }
  return table[p * half_d + i];
}

}  // namespace blk
