// wq_device.cuh -- sm_103a device helpers for the INT4-weight GEMM family:
// mbarriers with bounded waits, TMA tile loads, tcgen05 (TMEM alloc, MMA,
// commit, ld/st), shared-memory matrix descriptors and the INT4 dequant
// bit tricks.  Everything here is hand-written inline PTX or plain CUDA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "wq_internal.h"

namespace wq {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared abort flag + time limit for every wait of one CTA.  A wait that runs
// out ORs `code` into the device status word `*status` (read back by the host
// in checked mode) and raises the CTA's abort flag.
struct WaitCtx {
  volatile int* abort;   // shared memory flag: set once any wait of the CTA gave up
  uint64_t limit_ns;     // per-wait time limit
  unsigned code;         // status bits to report on expiry
  unsigned* status;      // device status word
};

// Wait until the phase with the given parity has completed.  Returns false
// if the wait ran out of time (or another wait of this CTA already did).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      *w.abort = 1;
      atomicOr(w.status, w.code);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tile mode, completion on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Plain bulk copy global -> shared (contiguous bytes, multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// L2 cache policies for the copies: weights stream through once per call
// (evict first) while activations and outputs should stay resident (evict last).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// TMA tile store shared -> global (bulk-group completion; the source must stay
// untouched until cp.async.bulk.wait_group.read).  Elements outside the tensor
// map's bounds are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

// The same store with an L2 cache policy (e.g. evict-first for outputs nothing reads soon).
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int x, int y,
                                                  uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters: barrier over every thread of the cluster, and
// distributed shared memory loads from a peer CTA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
// Arrive on an mbarrier of a CTA in the cluster (shared::cluster address from
// mapa_shared), releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bulk copy from this CTA's shared memory to a CTA of the cluster (address from
// mapa_shared); completes `bytes` on that CTA's mbarrier (also a mapa address).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                  uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the source buffers of every committed bulk copy have been read.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Split cluster barrier: arrive (no ordering) now, wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: wait for the preceding grid in the stream (its
// memory operations become visible), and let the following grid launch early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (fp16 or bf16 operands, fp32 D).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns, one register per column.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand staged by
// TMA with 128-byte swizzling.  Rows are 128 B apart, 8-row groups 1024 B
// apart; the leading-byte offset is unused for this layout.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                         // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                         // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, A and B both fp16
// (bf16 = 0) or both bf16 (bf16 = 1), both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t bf16, uint32_t M, uint32_t N) {
  return (1u << 4) | (bf16 << 7) | (bf16 << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// INT4 -> 16-bit dequant.  A packed word holds 8 consecutive-k codes of one
// column; code j sits at bit 4*(j/2) + 16*(j%2), so one AND+OR drops two
// neighbouring codes into the two halves of a 32-bit register.
//
// binary16 trick: OR-ing a nibble v into the low mantissa bits of 1024.0
// (0x6400) gives exactly 1024 + v; a nibble in bits 4..7 gives 1024 + 16 v.
// Subtracting 1032 (resp. scaling by 1/16 and subtracting 72) yields v - 8
// exactly, in one rounding-free half2 op per pair.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop_and_or(uint32_t x, uint32_t andm, uint32_t orm) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(andm), "r"(orm));  // (a & b) | c
  return r;
}
__device__ __forceinline__ uint32_t hsub2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 8 codes -> 4 half2 registers holding (v - 8) exactly, k ascending.
__device__ __forceinline__ void dq8_f16_exact(uint32_t w, uint32_t (&o)[4]) {
  constexpr uint32_t kMagic = 0x64006400u;      // (1024.0, 1024.0)
  constexpr uint32_t kSub = 0x64086408u;        // (1032.0, 1032.0)
  constexpr uint32_t kSixteenth = 0x2C002C00u;  // (1/16, 1/16)
  constexpr uint32_t kMinus72 = 0xD480D480u;    // (-72.0, -72.0)
  const uint32_t t = w >> 8;
  o[0] = hsub2_rn(lop_and_or(w, 0x000F000Fu, kMagic), kSub);
  o[1] = hfma2_rn(lop_and_or(w, 0x00F000F0u, kMagic), kSixteenth, kMinus72);
  o[2] = hsub2_rn(lop_and_or(t, 0x000F000Fu, kMagic), kSub);
  o[3] = hfma2_rn(lop_and_or(t, 0x00F000F0u, kMagic), kSixteenth, kMinus72);
}

// 8 codes -> binary16_RN((v - 8) * s) for a half2 (s, s): one rounding (the multiply).
__device__ __forceinline__ void dq8_f16_scaled(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
  dq8_f16_exact(w, o);
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = hmul2_rn(o[i], s2);
}

// 8 codes -> 4 bf16x2 registers holding (v - 8) exactly: OR-ing a nibble into
// the mantissa of 128.0 (0x4300) gives 128 + v exactly; subtract 136.
__device__ __forceinline__ uint32_t bsub2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bmul2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ void dq8_bf16_exact(uint32_t w, uint32_t (&o)[4]) {
  constexpr uint32_t kMagic = 0x43004300u;  // (128.0, 128.0)
  constexpr uint32_t kSub = 0x43084308u;    // (136.0, 136.0)
#pragma unroll
  for (int p = 0; p < 4; ++p) o[p] = bsub2_rn(lop_and_or(w >> (4 * p), 0x000F000Fu, kMagic), kSub);
}

// Split an fp16 scale into bf16 s_hi = RN(s) and s_lo = s - s_hi, each
// broadcast to both halves of a bf16x2.  s_lo is exact in bf16: an fp16
// significand has 11 bits, s_hi keeps the top 8, the remainder needs <= 3.
struct ScaleBf16 {
  uint32_t hi2, lo2;
};
__device__ __forceinline__ ScaleBf16 split_scale_bf16(__half s) {
  const float f = __half2float(s);
  const __nv_bfloat16 hi = __float2bfloat16_rn(f);
  const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(f, __bfloat162float(hi)));
  ScaleBf16 r;
  r.hi2 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) * 0x00010001u;
  r.lo2 = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) * 0x00010001u;
  return r;
}

// 8 codes -> bfloat16_RN((v - 8) * s) with one rounding.  x = v - 8 has <= 3
// significant bits, so x * s_lo (<= 6 bits) is exact in bf16; the fused
// x * s_hi + x * s_lo is then rounded once, which is RN(x * s) because
// s_hi + s_lo == s exactly.
__device__ __forceinline__ void dq8_bf16_scaled(uint32_t w, const ScaleBf16& s, uint32_t (&o)[4]) {
  dq8_bf16_exact(w, o);
#pragma unroll
  for (int p = 0; p < 4; ++p) o[p] = bfma2_rn(o[p], s.hi2, bmul2_rn(o[p], s.lo2));
}

// fp32 -> (hi, lo) bfloat16 split: hi = bf16_RN(x), lo = bf16_RN(x - hi).
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(__fsub_rn(x, __bfloat162float(hi)));
}

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// Store one output element in the requested type (kYF16 / kYBF16 / kYF32).
__device__ __forceinline__ void store_y_any(void* Y, int yk, size_t idx, float v) {
  if (yk == kYF16) {
    reinterpret_cast<__half*>(Y)[idx] = __float2half_rn(v);
  } else if (yk == kYBF16) {
    reinterpret_cast<__nv_bfloat16*>(Y)[idx] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<float*>(Y)[idx] = v;
  }
}

// SwiGLU activation of a gate/up pair in fp32: silu(g) * u, silu(g) = g / (1 + e^-g)
// (a very negative g gives e^-g = inf and silu = -0).
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Gate/up pair interleave of the combined weight: in every 16-column group the
// first 8 columns are gate columns and the next 8 the same up columns, so
// combined column c holds projection column 8 * (c / 16) + c % 8.
__host__ __device__ __forceinline__ int pair_source_col(int c) { return 8 * (c >> 4) + (c & 7); }

}  // namespace wq
