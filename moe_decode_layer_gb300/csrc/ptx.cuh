// Thin wrappers over the sm_100-family PTX the MoE decode kernels use:
// mbarriers, 1-D bulk (TMA) copies into shared memory, L2 cache policies,
// programmatic dependent launch, the global nanosecond timer, relaxed GPU-scope
// 64-bit accesses for tagged data, and bf16 / e2m1 / e4m3 arithmetic helpers.
#pragma once
#include <cstdint>

namespace moe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Makes barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}
// Non-blocking probe: true once the phase with this parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_try_wait, with a caller-chosen suspend-time hint (ns).
__device__ __forceinline__ bool mbar_try_wait_ns(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// One bounded probe: true once the phase with this parity has completed. The
// hardware may suspend the thread for up to ~1 us inside the call.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------- bulk copies
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Global -> shared 1-D bulk copy; completion is counted in bytes on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// The same without a cache hint (data that other CTAs read too).
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Orders this thread's earlier generic-proxy accesses to global / shared memory
// before later bulk-copy (async proxy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- launch order
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- timer
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- named barriers
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ---------------------------------------------------------------- tagged data
// A tagged word is (tag << 32) | float bits, written and read as one 64-bit
// access, so a reader that sees the current tag also sees that store's value.
__device__ __forceinline__ void st_tagged(unsigned long long* p, uint32_t tag, float v) {
  unsigned long long w = (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ void ld_tagged2(const unsigned long long* p, unsigned long long& a,
                                           unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------- arithmetic
// acc += sum_i w_i * x_i over the 8 bf16 pairs of two 16-byte chunks, in order,
// with the exact bf16 x bf16 product and one fp32 rounding per step.
__device__ __forceinline__ void dot8_bf16(float& acc, const uint4 w, const uint4 x) {
  asm("{\n .reg .b16 a0, a1, b0, b1;\n"
      " mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %5;\n"
      " fma.rn.f32.bf16 %0, a0, b0, %0; fma.rn.f32.bf16 %0, a1, b1, %0;\n"
      " mov.b32 {a0, a1}, %2; mov.b32 {b0, b1}, %6;\n"
      " fma.rn.f32.bf16 %0, a0, b0, %0; fma.rn.f32.bf16 %0, a1, b1, %0;\n"
      " mov.b32 {a0, a1}, %3; mov.b32 {b0, b1}, %7;\n"
      " fma.rn.f32.bf16 %0, a0, b0, %0; fma.rn.f32.bf16 %0, a1, b1, %0;\n"
      " mov.b32 {a0, a1}, %4; mov.b32 {b0, b1}, %8;\n"
      " fma.rn.f32.bf16 %0, a0, b0, %0; fma.rn.f32.bf16 %0, a1, b1, %0;\n}\n"
      : "+f"(acc)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// acc += sum_i w_i * h_i for 8 bf16 weights and 8 fp32 values, in order.
__device__ __forceinline__ void dot8_bf16_f32(float& acc, const uint4 w, const float* h) {
  acc = fmaf(bf16lo(w.x), h[0], acc);
  acc = fmaf(bf16hi(w.x), h[1], acc);
  acc = fmaf(bf16lo(w.y), h[2], acc);
  acc = fmaf(bf16hi(w.y), h[3], acc);
  acc = fmaf(bf16lo(w.z), h[4], acc);
  acc = fmaf(bf16hi(w.z), h[5], acc);
  acc = fmaf(bf16lo(w.w), h[6], acc);
  acc = fmaf(bf16hi(w.w), h[7], acc);
}

// Round-to-nearest-even float -> bf16 bits (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// Order-preserving map of a float to an unsigned key (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Two e2m1 codes (one byte) -> two fp16 values packed low/high.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n .reg .b16 s;\n cvt.u16.u32 s, %1;\n cvt.u8.u16 t, s;\n"
      " cvt.rn.f16x2.e2m1x2 %0, t;\n}\n"
      : "=r"(r)
      : "r"(byte));
  return r;
}
// Two e4m3 bytes (low, high of a 16-bit value) -> two fp16 values packed.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("{\n .reg .b16 s;\n cvt.u16.u32 s, %1;\n cvt.rn.f16x2.e4m3x2 %0, s;\n}\n"
      : "=r"(r)
      : "r"(two_bytes));
  return r;
}

}  // namespace moe
