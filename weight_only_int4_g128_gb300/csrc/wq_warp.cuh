// wq_warp.cuh -- helpers of the warp-level MMA decode path (M <= 8 tokens as
// the N = 8 side of mma.sync.m16n8k16): per-lane asynchronous copies, the
// offset-code MMA operands and the activation block sums.  Used by the
// weight-streaming decode kernel (wq_gemv.cu) and the persistent chain kernel
// (wq_chain.cu).
//
// Offset codes (section "The core mismatch": W_sym = (q - 8) * scale).  One
// LOP3 turns a word of code pairs into MMA operands that carry an exact
// offset instead of (v - 8): fp16 1024 + v for the low nibble of each code
// byte, 1024 + 16 v for the high nibble (two accumulator chains); bf16
// 128 + v (its 7-bit mantissa cannot hold a nibble at bits 4..7, so those
// pairs are shifted down first).  Per 128-k block the offsets come off in
// fp32 with the block sums of the activations:
//   fp16: sum (v - 8) x = D_lo + D_hi / 16 - (1032 * sum_lo x + 72 * sum_hi x)
//   bf16: sum (v - 8) x = D - 136 * sum x
// where lo / hi are the k whose code sits in the low / high nibble of its byte.
#pragma once

#include "wq_device.cuh"

namespace wq {
namespace warp {

// 16-byte asynchronous copy global -> shared (L1 bypassed), with an L2 policy.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
// 4-byte asynchronous copy global -> shared (through L1, the only mode for
// copies under 16 bytes), with an L2 policy.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's most recent copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint16_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
// 16-byte global load cached in L2 only: data written during the same launch
// by other CTAs (after they released it) is never served from a stale L1 line.
__device__ __forceinline__ uint4 ldg_cg128(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ float4 ldg_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ float ldg_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void stg_cg_f32(float* p, float a) {
  asm volatile("st.global.cg.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// D = A * B + C, m16n8k16, fp32 accumulate; A 16 x 16 (row), B 16 x 8 (col).
template <int XK>
__device__ __forceinline__ void mma16816(float (&d)[4], const float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if (XK == kXBF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
  }
}

// Sums of one 16-byte chunk (k = 8c .. 8c+7) of an activation row, split by the
// position of k in its code word: k % 8 in {0, 1, 4, 5} (low nibble of a code
// byte) into lo, {2, 3, 6, 7} (high nibble) into hi.
template <int XK>
__device__ __forceinline__ void sum_chunk(const uint4& v, float& lo, float& hi) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  float s[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (XK == kXF16) {
      s[i] = __half2float(__ushort_as_half(static_cast<uint16_t>(u[i] & 0xFFFFu))) +
             __half2float(__ushort_as_half(static_cast<uint16_t>(u[i] >> 16)));
    } else {
      s[i] = __uint_as_float(u[i] << 16) + __uint_as_float(u[i] & 0xFFFF0000u);
    }
  }
  lo = s[0] + s[2];
  hi = s[1] + s[3];
}

// The offset code operands (see the file header).
__device__ __forceinline__ uint32_t off_lo_f16(uint32_t w) { return lop_and_or(w, 0x000F000Fu, 0x64006400u); }
__device__ __forceinline__ uint32_t off_hi_f16(uint32_t w) { return lop_and_or(w, 0x00F000F0u, 0x64006400u); }
__device__ __forceinline__ uint32_t off_bf16(uint32_t w) { return lop_and_or(w, 0x000F000Fu, 0x43004300u); }

// Swizzle of an activation tile in shared memory: logical 16-byte chunk c of
// token row m sits at chunk c ^ (bit 3 of c | (m & 1) << 1), so the eight lanes
// of a quarter warp (two token rows x four lanes t, chunks 4t + q) hit eight
// distinct bank groups.
__device__ __forceinline__ int xswz(int c, int m) { return c ^ (((c >> 3) & 1) | ((m & 1) << 1)); }

}  // namespace warp
}  // namespace wq
