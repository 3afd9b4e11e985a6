// Device helpers shared by the tensor-core kernels: fp16 operand stores,
// instruction descriptors for fp16 MMAs, named barriers, bulk copies and a
// bounded mbarrier wait that gives up when another role has aborted.
#pragma once
#include <cstdint>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Explicit shared-memory accesses by 32-bit shared address (code that only
// has a generic pointer would otherwise go through generic loads/stores).
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds_u32x4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// max(m, |x|), NaN-propagating: a running bound on what went into fp16
// operands (checked once against the fp16 range at the end).
__device__ __forceinline__ float absmax_nan(float m, float x) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(x)));
  return r;
}

// 8 consecutive floats -> bf16 high parts and bf16 remainders (x = hi + lo to
// about 16 significant bits), stored as two 16-byte chunks.
__device__ __forceinline__ void store_bf16x8_hilo(uint32_t addr_hi, uint32_t addr_lo, const float* f) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    h[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
    const float r0 = f[2 * e] - __uint_as_float(h[e] << 16);
    const float r1 = f[2 * e + 1] - __uint_as_float(h[e] & 0xffff0000u);
    l[e] = pack_bf16x2(r0, r1);
  }
  st_shared_v4(addr_hi, h[0], h[1], h[2], h[3]);
  st_shared_v4(addr_lo, l[0], l[1], l[2], l[3]);
}

// Two packed bf16 (times d) -> two packed fp16, round to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float d) {
  return pack_f16x2(__uint_as_float(w << 16) * d, __uint_as_float(w & 0xffff0000u) * d);
}

// Instruction descriptor for kind::f16 with fp16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %3, 0;\n bar.red.or.pred po, %1, %2, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}"
      : "=r"(r)
      : "r"(id), "r"(count), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// ---- bulk (non-tensor) async copies ----
// global -> shared, completing on an mbarrier (both addresses 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// shared -> global, tracked by this thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of this thread has read its source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bounded wait on an mbarrier phase; gives up (false) after the wall-clock
// limit, recording `code` in *abort, or as soon as *abort is set by another
// thread.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, int* abort, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(abort)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(abort, 0, code);
      return false;
    }
  }
}

}  // namespace gdn
