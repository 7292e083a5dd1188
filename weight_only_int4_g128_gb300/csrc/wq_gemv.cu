// wq_gemv.cu -- the decode path (M <= 16 tokens) of the W4A16 / W4A8 GEMM,
// where the op is bound by reading the 4-bit weights from HBM.
//
// Same swap-AB arrangement as the large-M kernel (128 weight rows = the MMA's
// M = 128 TMEM lanes, 16 tokens = the MMA's N), but the per-group scale is not
// applied in the dequant.  Each 128-k block is contracted with the exact
// integers (q - 8) (exact in fp16 and bf16) into its own fp32 TMEM buffer, and
// the dequant warps promote it in fp32 ("Marlin INT4 on Ada -- how it works",
// section "The core mismatch": W_sym = (q - 8) * scale, C = C_sym +
// A_group_sum @ delta):
//     acc[n][m] += scale[g][n] * D_kb[n][m] + delta[g][n] * a_sum[m][kb]
// a_sum (the group sums of the 16 token rows) is computed in the same kernel
// by a dedicated warp from the activation tile already in shared memory, so
// the whole W4A16 GEMM is one launch.  In a thread the scale and delta of its
// row are scalars, so promotion costs 32 FMAs per 128 weights.
//
//   warp 0      TMA producer, per 128-k block: activation tile [16 x 128 k]
//               (one 3-D box = two 128-byte swizzled atoms) and the packed
//               weight tile (one contiguous 8 KB block, bulk copy); per 8
//               groups: the scale and delta rows of the tile's 128 columns
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma into a ring of 4 D buffers
//   warp 2      group sums of the activation tile
//   warps 3..6  dequant: each thread one weight row, 16 words -> 64 exact
//               (v - 8) pairs -> TMEM A-stage (two tcgen05.st of 32 columns)
//   warps 7..10 promotion: tcgen05.ld of the k-block's D, fp32 FMAs, epilogue
// Dequant and promotion run in separate warps so that neither waits on the
// other's latency chain (TMEM store / barrier round trips).
// Split-K: the K segments of one column tile form a thread-block cluster
// (gridDim.y = cluster size <= 8).  At the end every CTA leaves its fp32
// partial in shared memory; CTA r then sums, over all ranks in rank order
// (deterministic), the token rows m with m % splits == r, reading its peers'
// partials through distributed shared memory, and writes them to Y.
#include "wq_device.cuh"

namespace wq {

namespace gemv {
constexpr int kNSX = 8;     // shared-memory stages (one 128-k block each)
constexpr int kNSA = 3;     // TMEM A-stages
constexpr int kNB = 4;      // TMEM D buffers (16 fp32 columns each)
constexpr int kBT = 16;
constexpr int kXStage = kBT * kKBlock * 2;              // 4 KB
constexpr int kXAtom = kBT * 128;                       // 2 KB
constexpr int kWStage = kTileN * kWordsPerKBlock * 4;   // 8 KB
constexpr int kChunk = 8;  // groups per scale/delta chunk (the index math uses >> 3)
constexpr int kSChunk = kChunk * kTileN * 2;            // scale rows of a chunk, fp16 (2 KB)
constexpr int kDChunk = kChunk * kTileN * 4;            // delta rows of a chunk, fp32 (4 KB)
constexpr int kChunkSlots = 2;
constexpr int kDCol = kNSA * 64;                        // 192
constexpr int kTmemCols = 256;
constexpr int kThreads = 352;  // 11 warps
constexpr int kNumBars = 4 * kNSX + kNSA + kNB + 1 + 2 * kChunkSlots;
constexpr int kSmemBytes = 1024 + kNSX * (kXStage + kWStage) + kChunkSlots * (kSChunk + kDChunk) +
                           kNSX * kBT * 4 + kNumBars * 8 + 16;
constexpr int kMaxSplits = 8;  // portable cluster size
static_assert(kNB + kNSA < kNSX, "stages are released after promotion");
static_assert(kNSA < kNSX && kNB < kNSX, "mma_done is indexed by stage");
static_assert(kDCol + kNB * kBT <= kTmemCols, "TMEM budget");
static_assert(kBT * kTileN * 4 <= kNSX * kWStage, "reduction buffer reuses the weight ring");
}  // namespace gemv

__device__ __forceinline__ bool warp_wait_g(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float lo_to_f32(uint32_t u, int xk) {
  return xk == kXF16 ? __half2float(__ushort_as_half(static_cast<uint16_t>(u & 0xFFFFu)))
                     : __uint_as_float(u << 16);
}
__device__ __forceinline__ float hi_to_f32(uint32_t u, int xk) {
  return xk == kXF16 ? __half2float(__ushort_as_half(static_cast<uint16_t>(u >> 16)))
                     : __uint_as_float(u & 0xFFFF0000u);
}

template <int XK>
__global__ void __launch_bounds__(gemv::kThreads, 2)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_s,
                const __grid_constant__ CUtensorMap tm_d, const GemmParams p, unsigned* status) {
  using namespace gemv;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t sx = base;
  const uint32_t sw = sx + kNSX * kXStage;
  const uint32_t sch = sw + kNSX * kWStage;  // scale/delta chunk slots: [slot][S 2 KB | delta 4 KB]
  const uint32_t sasum = sch + kChunkSlots * (kSChunk + kDChunk);
  const uint32_t sbar = sasum + kNSX * kBT * 4;
  // Barriers.  Per stage s (k-block it, s = it % kNSX):
  //   full_x    TMA bytes of the stage landed
  //   empty_x   the stage's non-MMA readers are done (dequant, promotion, group sums)
  //   asum_full the group sums of the stage are in shared memory
  //   mma_done  the k-block's MMAs completed (one tcgen05.commit per k-block): the
  //             activation tile and the TMEM A-stage are free and D holds the result
  // full_a[a]  the TMEM A-stage a holds dequantized weights
  // empty_d[b] the promotion warps have read TMEM D buffer b
  auto full_x = [&](int s) { return sbar + 8u * s; };
  auto empty_x = [&](int s) { return sbar + 8u * (kNSX + s); };
  auto asum_full = [&](int s) { return sbar + 8u * (2 * kNSX + s); };
  auto mma_done = [&](int s) { return sbar + 8u * (3 * kNSX + s); };
  auto full_a = [&](int a) { return sbar + 8u * (4 * kNSX + a); };
  auto empty_d = [&](int b) { return sbar + 8u * (4 * kNSX + kNSA + b); };
  const uint32_t done_bar = sbar + 8u * (4 * kNSX + kNSA + kNB);
  // full_c / empty_c: scale+delta rows of 8 consecutive groups (one chunk) landed /
  // released by the promotion warps.
  auto full_c = [&](int c) { return sbar + 8u * (4 * kNSX + kNSA + kNB + 1 + c); };
  auto empty_c = [&](int c) { return sbar + 8u * (4 * kNSX + kNSA + kNB + 1 + kChunkSlots + c); };
  uint8_t* const gmisc = gbase + (sbar + 8u * kNumBars - base);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gmisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gmisc + 4);
  float* const asum_ring = reinterpret_cast<float*>(gbase + (sasum - base));
  const uint8_t* const chunk_smem = gbase + (sch - base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTileN;
  const int seg = blockIdx.y;  // == rank in the cluster (cluster dims 1 x splits x 1)
  const int kb0 = seg * p.kb_per_split;
  const int nkb = max(0, min(p.kb_total, kb0 + p.kb_per_split) - kb0);
  const bool has_delta = p.delta != nullptr;
  const uint32_t stage_tx = kXStage + kWStage;
  const uint32_t chunk_tx = kSChunk + (has_delta ? kDChunk : 0);
  // group size is 128 (group = k-block) or K (one group per column)
  const bool per_channel = p.group_size != kKBlock;
  const int g_first = per_channel ? 0 : kb0;  // first group of this K segment
  // chunk ordinal (0, 1, ...) of the k-block `it` of this segment, and its row (chunks of 8 groups)
  auto chunk_of = [&](int it) { return per_channel ? 0 : ((kb0 + it) >> 3) - (g_first >> 3); };
  auto chunk_row = [&](int it) { return per_channel ? 0 : ((kb0 + it) & 7); };
  int chunks_loaded = 0;  // producer lane: chunk ordinals [0, chunks_loaded) are issued
  // Weight-side copies of k-block `it` (producer lane only): the packed tile, and the
  // scale/delta chunk when the k-block starts a new one.
  auto weight_copies = [&](int it, const WaitCtx& wc) -> bool {
    const int o = chunk_of(it);
    if (o >= chunks_loaded) {
      const int slot = o % kChunkSlots;
      if (!mbar_wait(empty_c(slot), ((o / kChunkSlots) & 1) ^ 1, wc)) return false;
      const int grow = ((g_first >> 3) + o) * kChunk;
      const uint32_t dst = sch + slot * (kSChunk + kDChunk);
      mbar_arrive_expect_tx(full_c(slot), chunk_tx);
      tma_load_2d(dst, &tm_s, full_c(slot), n0, grow);
      if (has_delta) tma_load_2d(dst + kSChunk, &tm_d, full_c(slot), n0, grow);
      chunks_loaded = o + 1;
    }
    const int s = it % kNSX;
    mbar_arrive_expect_tx(full_x(s), stage_tx);
    // packed weight tile: one contiguous 8 KB block of the blocked layout
    bulk_load(sw + s * kWStage, p.B + (static_cast<size_t>(blockIdx.x) * p.kb_total + kb0 + it) * 2048,
              kWStage, full_x(s));
    return true;
  };
  const int pre = p.weight_prefetch ? min(kNSX, nkb) : 0;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_s);
    if (has_delta) prefetch_tensormap(&tm_d);
    for (int s = 0; s < kNSX; ++s) {
      mbar_init(full_x(s), 1);
      mbar_init(empty_x(s), 4 + 4 + 1);  // dequant warps, promotion warps, group sums
      mbar_init(asum_full(s), 32);
      mbar_init(mma_done(s), 1);
    }
    for (int a = 0; a < kNSA; ++a) mbar_init(full_a(a), 4);
    for (int b = 0; b < kNB; ++b) mbar_init(empty_d(b), 4);  // promotion warps
    for (int c = 0; c < kChunkSlots; ++c) {
      mbar_init(full_c(c), 1);
      mbar_init(empty_c(c), 4);  // promotion warps
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // Weight-side copies of the first stages go out before anything else (fresh
    // stages and chunk slots: nothing to wait for); see the note below.
    volatile int never = 0;
    const WaitCtx nowait{&never, 1000000ull, kDevTimeoutProducer, status};
    for (int it = 0; it < pre; ++it) weight_copies(it, nowait);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(gmisc), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Programmatic dependent launch: nothing before griddep_wait() touches memory
  // the preceding grid may write (X, Y).  Only the weight-side copies (packed
  // codes, scales, delta) of the first stages may be issued earlier, and only
  // when the caller enabled it (the weights must not be written by the
  // preceding kernel).
  int issued = 0;  // TMA stages the producer lane has issued
  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutProducer, status};
      griddep_wait();
      for (int it = 0; it < nkb; ++it) {
        const int s = it % kNSX;
        if (it >= pre) {
          const uint32_t prev = ((it / kNSX) & 1) ^ 1;  // phase of k-block it - kNSX
          if (!mbar_wait(empty_x(s), prev, wc)) break;
          if (!mbar_wait(mma_done(s), prev, wc)) break;
          if (!weight_copies(it, wc)) break;
        }
        // activation tile [16 x 128 k]: one 3-D box {64 k, 16 rows, 2 halves of the k-block}
        tma_load_3d(sx + s * kXStage, &tm_x, full_x(s), 0, 0, 2 * (kb0 + it));
        issued = it + 1;
      }
    } else {
      griddep_wait();
    }
  } else {
    griddep_wait();
  }
  if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMma, status};
      constexpr uint32_t idesc = idesc_f16(XK, 128, kBT);
      const uint64_t desc0 = desc_kmajor_sw128(sx);  // stage 0, k step 0
      for (int it = 0; it < nkb; ++it) {
        const int s = it % kNSX;
        const int a = it % kNSA;
        const int b = it % kNB;
        // full_a implies the stage's TMA bytes landed: the dequant warps waited on full_x
        if (!mbar_wait(full_a(a), (it / kNSA) & 1, wc)) break;
        if (!mbar_wait(empty_d(b), ((it / kNB) & 1) ^ 1, wc)) break;
        tc_fence_after();
        // descriptor start address advances in 16-byte units: stage, 64-k half, 16-k step
        const uint64_t ds = desc0 + static_cast<uint64_t>((s * kXStage) >> 4);
        const uint32_t d = tmem + kDCol + b * kBT;
        const uint32_t at = tmem + a * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          mma_ts(d, at + i * 8, ds + (((i >> 2) * kXAtom + (i & 3) * 32) >> 4), idesc, i > 0 ? 1u : 0u);
        mma_commit(mma_done(s));
      }
      mma_commit(done_bar);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- group sums
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
    const uint8_t* xring = gbase + (sx - base);
    const int r = lane >> 1;  // token row
    const int h = lane & 1;   // which 64-k half of the block
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kNSX;
      if (!warp_wait_g(full_x(s), (it / kNSX) & 1, wc)) break;
      if (has_delta) {
        const uint8_t* rowp = xring + s * kXStage + h * kXAtom + r * 128;
        float sum = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + 16 * (c ^ (r & 7)));
          sum += lo_to_f32(v.x, XK) + hi_to_f32(v.x, XK);
          sum += lo_to_f32(v.y, XK) + hi_to_f32(v.y, XK);
          sum += lo_to_f32(v.z, XK) + hi_to_f32(v.z, XK);
          sum += lo_to_f32(v.w, XK) + hi_to_f32(v.w, XK);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        if (h == 0) asum_ring[s * kBT + r] = sum;
        __syncwarp();
        mbar_arrive(asum_full(s));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_x(s));
    }
  }

  // ---------------------------------------------------------------- dequant / promotion
  float acc[kBT];
#pragma unroll
  for (int m = 0; m < kBT; ++m) acc[m] = 0.0f;
  const bool dequant = (warp >= 3 && warp <= 6);
  const bool promote = (warp >= 7 && warp <= 10);
  const int q = warp & 3;              // TMEM lane quarter this warp may access
  const int row = q * 32 + lane;       // weight row of the tile = TMEM lane
  const int n = n0 + row;
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  if (dequant) {
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
    const uint8_t* wring = gbase + (sw - base);
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kNSX;
      const int a = it % kNSA;
      if (!warp_wait_g(full_x(s), (it / kNSX) & 1, wc)) break;
      uint4 wv[4];
      const uint8_t* wrow = wring + s * kWStage + row * 64;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        wv[c] = *reinterpret_cast<const uint4*>(wrow + 16 * (c ^ ((row >> 1) & 3)));
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_x(s));
      if (it >= kNSA) {  // A-stage a was last read by the MMAs of k-block it - kNSA
        const int pk = it - kNSA;
        if (!warp_wait_g(mma_done(pk % kNSX), (pk / kNSX) & 1, wc)) break;
        tc_fence_after();
      }
      const uint32_t at = tmem + lane_base + a * 64;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint4 w0 = wv[2 * half], w1 = wv[2 * half + 1];
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t v[32];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          uint32_t o[4];
          if (XK == kXF16) dq8_f16_exact(words[w], o);
          else dq8_bf16_exact(words[w], o);
#pragma unroll
          for (int e = 0; e < 4; ++e) v[4 * w + e] = o[e];
        }
        tmem_st32(at + 32 * half, v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_a(a));
    }
  } else if (promote) {
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
    for (int j = 0; j < nkb; ++j) {
      const int b = j % kNB;
      const int sj = j % kNSX;
      if (!warp_wait_g(mma_done(sj), (j / kNSX) & 1, wc)) break;
      tc_fence_after();
      uint32_t r[kBT];
      tmem_ld16(tmem + lane_base + kDCol + b * kBT, r);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_d(b));
      const int o = chunk_of(j);
      const int slot = o % kChunkSlots;
      if (!warp_wait_g(full_c(slot), (o / kChunkSlots) & 1, wc)) break;
      const uint8_t* chunk = chunk_smem + slot * (kSChunk + kDChunk);
      const int gr = chunk_row(j);
      const float sc = __half2float(reinterpret_cast<const __half*>(chunk)[gr * kTileN + row]);
#pragma unroll
      for (int m = 0; m < kBT; ++m) acc[m] = fmaf(sc, __uint_as_float(r[m]), acc[m]);
      if (has_delta) {
        if (!warp_wait_g(asum_full(sj), (j / kNSX) & 1, wc)) break;
        const float dl = reinterpret_cast<const float*>(chunk + kSChunk)[gr * kTileN + row];
        const float4* a4 = reinterpret_cast<const float4*>(asum_ring + sj * kBT);
#pragma unroll
        for (int v = 0; v < kBT / 4; ++v) {
          const float4 t = a4[v];
          acc[4 * v + 0] = fmaf(dl, t.x, acc[4 * v + 0]);
          acc[4 * v + 1] = fmaf(dl, t.y, acc[4 * v + 1]);
          acc[4 * v + 2] = fmaf(dl, t.z, acc[4 * v + 2]);
          acc[4 * v + 3] = fmaf(dl, t.w, acc[4 * v + 3]);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(empty_x(sj));
        if (j + 1 == nkb || chunk_of(j + 1) != o) mbar_arrive(empty_c(slot));  // chunk done
      }
    }
    tc_fence_before();
  }
  const bool math = promote;

  // ---------------------------------------------------------------- split-K reduction + store
  __syncthreads();  // every role is past its loop
  griddep_launch_dependents();  // the next grid in the stream may start its setup
  const bool aborted = *abort_flag != 0;
  if (aborted && warp == 0 && lane == 0) {
    // Let every copy the producer issued land before the shared memory is reused.
    volatile int never = 0;
    const WaitCtx drain{&never, 50000000ull, kDevTimeoutProducer, status};
    for (int it = max(0, issued - kNSX); it < issued; ++it)
      mbar_wait(full_x(it % kNSX), (it / kNSX) & 1, drain);
    for (int o = max(0, chunks_loaded - kChunkSlots); o < chunks_loaded; ++o)
      mbar_wait(full_c(o % kChunkSlots), (o / kChunkSlots) & 1, drain);
  }
  __syncthreads();
  float* const red = reinterpret_cast<float*>(gbase + (sw - base));  // [16][128] fp32
  if (math) {
#pragma unroll
    for (int m = 0; m < kBT; ++m) red[m * kTileN + row] = aborted ? __int_as_float(0x7fc00000) : acc[m];
  }
  cluster_sync_all();
  if (math) {
    const int splits = p.splits;
    const uint32_t red_local = smem_u32(red) + static_cast<uint32_t>(row) * 4u;
    for (int m = seg; m < p.M; m += splits) {
      float t = 0.0f;
#pragma unroll 8
      for (int rr = 0; rr < splits; ++rr)
        t += ld_dsmem_f32(mapa_shared(red_local + static_cast<uint32_t>(m * kTileN) * 4u, rr));
      if (p.x_scale) t *= __ldg(p.x_scale + m);
      store_y_any(p.Y, p.y_kind, static_cast<size_t>(m) * p.N + n, t);
    }
  }
  cluster_sync_all();  // peers keep their shared memory until every rank has read it

  if (warp == 1) {
    volatile int never = 0;
    const WaitCtx drain{&never, 50000000ull, kDevTimeoutMma, status};
    mbar_wait(done_bar, 0, drain);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int XK>
static cudaError_t launch_gemv_xk(const CUtensorMap& tm_x, const CUtensorMap& tm_s,
                                  const CUtensorMap& tm_d, const GemmParams& p, unsigned* status,
                                  cudaStream_t st) {
  static unsigned long long attr_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_mask & bit)) {
    e = cudaFuncSetAttribute(gemv_kernel<XK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemv::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_mask |= bit;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.N / kTileN, p.splits, 1);
  cfg.blockDim = dim3(gemv::kThreads, 1, 1);
  cfg.dynamicSmemBytes = gemv::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = p.splits;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<XK>, tm_x, tm_s, tm_d, p, status);
}

int gemv_max_splits() { return gemv::kMaxSplits; }

cudaError_t launch_gemv(int x_kind, const CUtensorMap& tm_x, const CUtensorMap& tm_s,
                        const CUtensorMap& tm_d, const GemmParams& p, cudaStream_t stream) {
  unsigned* status = status_word();
  if (!status) return cudaErrorInvalidSymbol;
  if (p.splits < 1 || p.splits > gemv::kMaxSplits) return cudaErrorInvalidValue;
  return x_kind == kXBF16 ? launch_gemv_xk<kXBF16>(tm_x, tm_s, tm_d, p, status, stream)
                          : launch_gemv_xk<kXF16>(tm_x, tm_s, tm_d, p, status, stream);
}

}  // namespace wq
