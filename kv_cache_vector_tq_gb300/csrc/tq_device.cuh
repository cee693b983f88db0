// Device helpers shared by the libtq kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include <cmath>

namespace tq {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kSpinLimitDev = 1u << 22;  // bounded mbarrier waits

// D += A·B with mma.m16n8k16, fp16 operands, fp32 accumulators.
// Fragment ownership (lane = 4g + t):
//   A (16x16, row): a0 = (g, 2t..2t+1), a1 = (g+8, 2t..), a2 = (g, 2t+8..), a3 = (g+8, 2t+8..)
//   B (16x8, col) : b0 = (k 2t..2t+1, n g), b1 = (k 2t+8..2t+9, n g)
//   D (16x8)      : d0 = (g, 2t), d1 = (g, 2t+1), d2 = (g+8, 2t), d3 = (g+8, 2t+1)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// fp16 hi/lo split of two fp32 values: x ≈ hi + lo with |x - hi - lo| <= 2^-22 |x|
// when hi and lo are normal numbers.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(x0, x1);
  __half2 l = __floats2half2_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = h2_bits(h);
  lo = h2_bits(l);
}

__device__ __forceinline__ uint32_t pack_f16x2(float x0, float x1) {
  return h2_bits(__floats2half2_rn(x0, x1));
}

// Extract `bits` bits at bit offset `off` of a little-endian word array (off
// and bits compile-time after unrolling; codes may straddle two words).
template <int BITS>
__device__ __forceinline__ uint32_t get_bits(const uint32_t* w, int off) {
  const int wi = off >> 5, sh = off & 31;
  uint32_t v = w[wi] >> sh;
  if (sh + BITS > 32) v |= w[wi + 1] << (32 - sh);
  return v & ((1u << BITS) - 1u);
}

template <int BITS>
__device__ __forceinline__ void put_bits(uint32_t* w, int off, uint32_t v) {
  const int wi = off >> 5, sh = off & 31;
  w[wi] |= v << sh;
  if (sh + BITS > 32) w[wi + 1] |= v >> (32 - sh);
}

// Power-of-two scale 2^e such that s·2^e lies in [16, 32) (1 for s == 0).
__device__ __forceinline__ float pow2_scale_16_32(float s) {
  if (!(s > 0.f)) return 1.f;
  int e;
  frexpf(s, &e);  // s = m·2^e, m in [0.5, 1)
  return ldexpf(1.f, 5 - e);
}

// ------------------------------------------------------------------ PTX helpers
// mbarrier, bulk asynchronous copy (global -> shared), programmatic dependent launch
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// programmatic dependent launch: wait for the preceding grid / let the next one start
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
// Shared-window address of a lane's copy of table entry `byte k of w`, for
// tables laid out as 256-byte rows (one row per index, 4-byte entries at
// lane·4): byte 0 = lane·4, byte 1 = byte k of w, upper bytes zero.
__device__ __forceinline__ uint32_t byte_row_addr(uint32_t w, uint32_t lane4, int k) {
  return __byte_perm(w, lane4, 0x5504 | (k << 4));
}
// 32-bit shared load at a window address plus a compile-time offset.
template <int OFF>
__device__ __forceinline__ uint32_t lds_at(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1+%2];\n" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace tq
