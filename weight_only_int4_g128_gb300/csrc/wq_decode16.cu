// wq_decode16.cu -- the decode path (M <= 16 tokens) of the W4A16 GEMM on
// kind::f16 tensor cores, reading the fp16 / bf16 activations directly.
//
// Same swap-AB arrangement as the other kernels (128 weight rows per CTA = the
// MMA's M = 128 TMEM lanes, 16 tokens = the MMA's N), one launch per GEMM: no
// activation pre-pass sits between the preceding grid and this one.  Each
// 128-k block is contracted with the exact integers (q - 8) (exact in fp16 and
// bf16) into an fp32 TMEM buffer of its own, and the promotion warps apply the
// group's scale and correction in fp32 ("Marlin INT4 on Ada -- how it works",
// section "The core mismatch": W_sym = (q - 8) * scale, C = C_sym +
// A_group_sum @ delta):
//     acc[n][m] += scale[g][n] * D_kb[n][m] + delta[g][n] * a_sum[kb][m]
// with a_sum (the block sums of the 16 token rows) computed in the kernel by a
// dedicated warp from the activation tile already in shared memory.
//
//   warp 0      TMA producer: per pair of 128-k blocks the packed weight tiles
//               (one 16 KB bulk copy) and the activation tiles (one 3-D box of
//               4 x {64 k, 16 rows}: four 128-byte swizzled atoms); per 8 groups
//               the scale and delta rows of the tile
//   warp 1      TMEM owner; lane 0 issues the MMAs (A from TMEM, B from shared)
//   warp 2      block sums of the activation tile
//   warps 3..6  dequant: each thread one weight row, 16 words -> 64 exact
//               (v - 8) pairs -> TMEM A-stage (two tcgen05.st of 32 columns)
//   warps 7..10 promotion (tcgen05.ld of the block's D, fp32 FMAs) and epilogue
// Split-K: the K segments of one column tile form a thread-block cluster; each
// CTA stages its fp32 partials and sends every rank the rows it owns with one
// bulk shared-to-shared copy completing on the owner's mbarrier.
#include "wq_device.cuh"

namespace wq {

namespace d16 {
constexpr int kNSX = 6;                   // shared-memory stages (one 128-k block each)
constexpr int kPair = 2;                  // k-blocks per load group (one copy each of W and X)
constexpr int kNG = kNSX / kPair;         // load groups in the ring
constexpr int kNSA = 3;                   // TMEM A-stages
constexpr int kNB = 4;                    // TMEM D buffers
constexpr int kMT = 16;                   // tokens per tile = MMA N
constexpr int kXStage = kMT * kKBlock * 2;  // 4 KB: two 64-k atoms of 16 rows x 128 B
constexpr int kXAtom = kMT * 128;           // 2 KB
constexpr int kWStage = kTileN * kWordsPerKBlock * 4;  // 8 KB
constexpr int kChunk = 8;                 // groups per scale/delta chunk (index math uses >> 3)
constexpr int kSChunk = kChunk * kTileN * 2;
constexpr int kDChunk = kChunk * kTileN * 4;
constexpr int kChunkSlots = 2;
constexpr int kACol = 64;                 // TMEM columns of one A-stage (128 k of 16-bit pairs)
constexpr int kDCol0 = kNSA * kACol;      // 192
constexpr int kTmemCols = 256;
constexpr int kThreads = 352;             // 11 warps
constexpr int kMaxSplits = 8;             // portable cluster size
constexpr int kRedBytes = 8704;           // >= splits * ceil(128 / splits) * 16 * 4 for splits <= 8
constexpr int kNumBars = 2 * kNG + 3 * kNSX + kNSA + 2 * kChunkSlots + 2;
constexpr int kSmemBytes = 1024 + kNSX * (kXStage + kWStage) + kChunkSlots * (kSChunk + kDChunk) +
                           kNSX * kMT * 4 + kRedBytes + kNumBars * 8 + 16;
static_assert(kDCol0 + kNB * kMT <= kTmemCols, "TMEM budget");
static_assert(kNSA < kNSX && kNB < kNSX && kNG * kPair == kNSX, "ring and barrier phase distances");
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(kTileN * kMT * 4 <= kWStage, "partials staged in one weight stage");
}  // namespace d16

__device__ __forceinline__ bool warp_wait16(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void named_sync16(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int XK>
__device__ __forceinline__ float sum_pair(uint32_t u) {
  if (XK == kXF16)
    return __half2float(__ushort_as_half(static_cast<uint16_t>(u & 0xFFFFu))) +
           __half2float(__ushort_as_half(static_cast<uint16_t>(u >> 16)));
  return __uint_as_float(u << 16) + __uint_as_float(u & 0xFFFF0000u);
}

template <int XK>
__global__ void __launch_bounds__(d16::kThreads, 2)
    decode16_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_s,
                    const __grid_constant__ CUtensorMap tm_d, const GemmParams p, unsigned* status) {
  using namespace d16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t sx = base;                                   // activation tiles [kNSX][4 KB] (1024-aligned)
  const uint32_t sw = sx + kNSX * kXStage;                    // weight tiles [kNSX][8 KB]
  const uint32_t sch = sw + kNSX * kWStage;                   // chunk slots [2][S 2 KB | delta 4 KB]
  const uint32_t sas = sch + kChunkSlots * (kSChunk + kDChunk);  // block sums [kNSX][16] fp32
  const uint32_t sred = sas + kNSX * kMT * 4;                 // split-K partials (peers copy here)
  const uint32_t sbar = sred + kRedBytes;
  // Barriers.  Per load group g (k-blocks 2 gi, 2 gi + 1; g = gi % kNG, stages 2 g, 2 g + 1):
  //   full_w    both weight tiles landed (the dequant warps need nothing else, so
  //             with weight prefetch they may run before the preceding grid ends)
  //   full_x    both activation tiles landed (block sums, MMAs)
  // Per stage s (k-block it, s = it % kNSX):
  //   mma_done  the k-block's MMAs completed (A-stage it % kNSA free, D buffer it % kNB full)
  //   asum_full the block sums of the stage's activation tile are in shared memory
  //   pdone     the promotion warps read D buffer it % kNB and the stage's block sums:
  //             the D buffer and (with the other stage of its group) the stage are free
  // full_a[a]  A-stage a holds the k-block's weights
  // full_c/empty_c  scale + delta rows of 8 groups landed / released
  auto full_w = [&](int g) { return sbar + 8u * g; };
  auto full_x = [&](int g) { return sbar + 8u * (kNG + g); };
  auto mma_done = [&](int s) { return sbar + 8u * (2 * kNG + s); };
  auto asum_full = [&](int s) { return sbar + 8u * (2 * kNG + kNSX + s); };
  auto pdone = [&](int s) { return sbar + 8u * (2 * kNG + 2 * kNSX + s); };
  auto full_a = [&](int a) { return sbar + 8u * (2 * kNG + 3 * kNSX + a); };
  auto full_c = [&](int c) { return sbar + 8u * (2 * kNG + 3 * kNSX + kNSA + c); };
  auto empty_c = [&](int c) { return sbar + 8u * (2 * kNG + 3 * kNSX + kNSA + kChunkSlots + c); };
  const uint32_t done_bar = sbar + 8u * (kNumBars - 2);
  const uint32_t red_full = sbar + 8u * (kNumBars - 1);
  uint8_t* const gmisc = gbase + (sbar + 8u * kNumBars - base);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gmisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gmisc + 4);
  const uint8_t* const chunk_smem = gbase + (sch - base);
  float* const asum = reinterpret_cast<float*>(gbase + (sas - base));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTileN;
  const int seg = blockIdx.y;  // == rank in the cluster (cluster dims 1 x splits x 1)
  const int kb0 = seg * p.kb_per_split;
  const int nkb = max(0, min(p.kb_total, kb0 + p.kb_per_split) - kb0);
  const int ngi = (nkb + kPair - 1) / kPair;
  const bool has_delta = p.delta != nullptr;
  const uint32_t chunk_tx = kSChunk + (has_delta ? kDChunk : 0);
  const bool per_channel = p.group_size != kKBlock;  // group size 128, or one group per column
  const int g_first = per_channel ? 0 : kb0;
  auto chunk_of = [&](int it) { return per_channel ? 0 : ((kb0 + it) >> 3) - (g_first >> 3); };
  auto chunk_row = [&](int it) { return per_channel ? 0 : ((kb0 + it) & 7); };
  int chunks_loaded = 0;  // producer lane: chunk ordinals [0, chunks_loaded) are issued
  auto w_bytes = [&](int gi) { return static_cast<uint32_t>(min(kPair, nkb - kPair * gi) * kWStage); };
  // weights, scales and deltas are read once per call: keep them from evicting X and Y in L2
  const uint64_t pol_stream = l2_evict_first();
  const uint64_t pol_keep = l2_evict_last();
  auto issue_w = [&](int gi) {
    const int g = gi % kNG;
    mbar_arrive_expect_tx(full_w(g), w_bytes(gi));
    bulk_load_hint(sw + g * kPair * kWStage,
                   p.B + (static_cast<size_t>(blockIdx.x) * p.kb_total + kb0 + kPair * gi) * 2048, w_bytes(gi),
                   full_w(g), pol_stream);
  };
  // activation tiles of both k-blocks of load group gi: one 3-D box {64 k, 16 rows, 4 atoms}
  auto issue_x = [&](int gi) {
    const int g = gi % kNG;
    mbar_arrive_expect_tx(full_x(g), kPair * kXStage);
    tma_load_3d_hint(sx + g * kPair * kXStage, &tm_x, full_x(g), 0, 0, 2 * (kb0 + kPair * gi), pol_keep);
  };
  auto issue_chunk = [&](int o) {
    const int slot = o % kChunkSlots;
    const int grow = ((g_first >> 3) + o) * kChunk;
    const uint32_t dst = sch + slot * (kSChunk + kDChunk);
    mbar_arrive_expect_tx(full_c(slot), chunk_tx);
    tma_load_2d_hint(dst, &tm_s, full_c(slot), n0, grow, pol_stream);
    if (has_delta) tma_load_2d_hint(dst + kSChunk, &tm_d, full_c(slot), n0, grow, pol_stream);
  };
  // Weight-side copies of load group gi (producer lane only); every wait comes first.
  auto weight_copies = [&](int gi, const WaitCtx& wc) -> bool {
    const int last = chunk_of(min(nkb, kPair * gi + kPair) - 1);
    for (int o = chunks_loaded; o <= last; ++o)
      if (!mbar_wait(empty_c(o % kChunkSlots), ((o / kChunkSlots) & 1) ^ 1, wc)) return false;
    issue_w(gi);
    for (; chunks_loaded <= last; ++chunks_loaded) issue_chunk(chunks_loaded);
    return true;
  };
  const int pre = p.weight_prefetch ? min(kNG, ngi) : 0;
  const int splits = p.splits;
  const int rpr = (kTileN + splits - 1) / splits;
  const int own_rows = max(0, min(kTileN - seg * rpr, rpr));

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_s);
    if (has_delta) prefetch_tensormap(&tm_d);
    for (int g = 0; g < kNG; ++g) {
      mbar_init(full_w(g), 1);
      mbar_init(full_x(g), 1);
    }
    for (int s = 0; s < kNSX; ++s) {
      mbar_init(mma_done(s), 1);
      mbar_init(asum_full(s), 1);
      mbar_init(pdone(s), 4);
    }
    for (int a = 0; a < kNSA; ++a) mbar_init(full_a(a), 4);
    for (int c = 0; c < kChunkSlots; ++c) {
      mbar_init(full_c(c), 1);
      mbar_init(empty_c(c), 4);
    }
    mbar_init(done_bar, 1);
    mbar_init(red_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (splits > 1) mbar_arrive_expect_tx(red_full, static_cast<uint32_t>(own_rows * splits * kMT * 4));
  }
  if (warp == 0) {
    // Weight-side copies of the first load groups go out before anything else
    // (fresh stages and chunk slots: nothing to wait for), one group per lane.
    __syncwarp();
    if (lane < pre) issue_w(lane);
    if (lane == 0 && pre > 0) {
      const int last = chunk_of(min(nkb, kPair * pre) - 1);  // at most kChunkSlots chunks
      for (; chunks_loaded <= last; ++chunks_loaded) issue_chunk(chunks_loaded);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(gmisc), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (splits > 1) cluster_arrive_relaxed();  // barriers initialized and armed (waited before any copy)

  // Programmatic dependent launch: the next grid in the stream may be scheduled
  // now (it waits for this one to complete before it touches memory this one
  // uses).  Only two places touch global memory the preceding grid may write:
  // the producer lane's copies (X always; the weight side too unless the caller
  // enabled weight prefetch) and the stores of Y.  Both come after
  // griddep_wait(); until then the dequant warps may already turn prefetched
  // weight tiles into TMEM A-stages (shared memory and TMEM only).
  griddep_launch_dependents();

  int w_issued = pre;  // load groups whose weight tiles have been issued (producer lane)
  int x_issued = 0;    // load groups whose activation box has been issued (producer lane)
  const int q = warp & 3;         // TMEM lane quarter this warp may access
  const int row = q * 32 + lane;  // weight row of the tile = TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  float acc[kMT];
#pragma unroll
  for (int m = 0; m < kMT; ++m) acc[m] = 0.0f;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutProducer, status};
      griddep_wait();
      for (int gi = 0; gi < ngi; ++gi) {
        const int g = gi % kNG;
        if (gi >= pre) {
          const uint32_t prev = ((gi / kNG) & 1) ^ 1;  // phase of load group gi - kNG
          bool ok = true;
          for (int j = 0; j < kPair && ok; ++j) ok = mbar_wait(pdone(kPair * g + j), prev, wc);
          if (!ok || !weight_copies(gi, wc)) break;
          w_issued = gi + 1;
        }
        issue_x(gi);
        x_issued = gi + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMma, status};
      constexpr uint32_t idesc = idesc_f16(XK, 128, kMT);
      const uint64_t desc0 = desc_kmajor_sw128(sx);
      for (int it = 0; it < nkb; ++it) {
        const int s = it % kNSX;
        const int a = it % kNSA;
        const int b = it % kNB;
        // weights in A-stage a, activation tiles landed; D buffer b was last read
        // by the promotion of k-block it - kNB
        if (!mbar_wait(full_a(a), (it / kNSA) & 1, wc)) break;
        if (!mbar_wait(full_x(s / kPair), (it / kNSX) & 1, wc)) break;
        if (it >= kNB) {
          const int pk = it - kNB;
          if (!mbar_wait(pdone(pk % kNSX), (pk / kNSX) & 1, wc)) break;
        }
        tc_fence_after();
        // descriptor start address advances in 16-byte units: stage, 64-k atom, 16-k step
        const uint64_t ds = desc0 + static_cast<uint64_t>((s * kXStage) >> 4);
        const uint32_t d = tmem + kDCol0 + b * kMT;
        const uint32_t at = tmem + a * kACol;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          mma_ts(d, at + i * 8, ds + (((i >> 2) * kXAtom + (i & 3) * 32) >> 4), idesc, i > 0 ? 1u : 0u);
        mma_commit(mma_done(s));
      }
      mma_commit(done_bar);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- block sums
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
    const uint8_t* xring = gbase + (sx - base);
    const int r = lane >> 1;  // token row
    const int h = lane & 1;   // 64-k atom of the block
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kNSX;
      if (!warp_wait16(full_x(s / kPair), (it / kNSX) & 1, wc)) break;
      if (has_delta) {
        const uint8_t* rowp = xring + s * kXStage + h * kXAtom + r * 128;
        float sum = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + 16 * (c ^ (r & 7)));
          sum += (sum_pair<XK>(v.x) + sum_pair<XK>(v.y)) + (sum_pair<XK>(v.z) + sum_pair<XK>(v.w));
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        if (h == 0) asum[s * kMT + r] = sum;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(asum_full(s));
    }
  } else if (warp >= 3 && warp <= 6) {
    // ---------------------------------------------------------------- dequant
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
    const uint8_t* wring = gbase + (sw - base);
    auto load_words = [&](int it, uint4 (&wv)[4]) -> bool {
      const int s = it % kNSX;
      if (!warp_wait16(full_w(s / kPair), (it / kNSX) & 1, wc)) return false;
      const uint8_t* wrow = wring + s * kWStage + row * 64;
#pragma unroll
      for (int c = 0; c < 4; ++c) wv[c] = *reinterpret_cast<const uint4*>(wrow + 16 * (c ^ ((row >> 1) & 3)));
      return true;
    };
    uint4 wv[4];
    bool ok = nkb > 0 && load_words(0, wv);
    for (int it = 0; ok && it < nkb; ++it) {
      const int a = it % kNSA;
      if (it >= kNSA) {  // A-stage a was last read by the MMAs of k-block it - kNSA
        const int pk = it - kNSA;
        if (!warp_wait16(mma_done(pk % kNSX), (pk / kNSX) & 1, wc)) break;
        tc_fence_after();
      }
      const uint32_t at = tmem + lane_base + a * kACol;
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
      // the next k-block's words load while the stores complete
      if (it + 1 < nkb) ok = load_words(it + 1, wv);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_a(a));
    }
  } else if (warp >= 7 && warp <= 10) {
    // ---------------------------------------------------------------- promotion
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
    for (int j = 0; j < nkb; ++j) {
      const int s = j % kNSX;
      const int b = j % kNB;
      // operands that do not depend on the MMAs first: block sums, scale, delta
      float as[kMT];
      if (has_delta) {
        if (!warp_wait16(asum_full(s), (j / kNSX) & 1, wc)) break;
        const float4* a4 = reinterpret_cast<const float4*>(asum + s * kMT);
#pragma unroll
        for (int v4 = 0; v4 < kMT / 4; ++v4) {
          const float4 t = a4[v4];
          as[4 * v4] = t.x; as[4 * v4 + 1] = t.y; as[4 * v4 + 2] = t.z; as[4 * v4 + 3] = t.w;
        }
      }
      const int o = chunk_of(j);
      const int slot = o % kChunkSlots;
      if (!warp_wait16(full_c(slot), (o / kChunkSlots) & 1, wc)) break;
      const uint8_t* chunk = chunk_smem + slot * (kSChunk + kDChunk);
      const int gr = chunk_row(j);
      const float sc = __half2float(reinterpret_cast<const __half*>(chunk)[gr * kTileN + row]);
      const float dl = has_delta ? reinterpret_cast<const float*>(chunk + kSChunk)[gr * kTileN + row] : 0.0f;
      __syncwarp();
      if (lane == 0 && (j + 1 == nkb || chunk_of(j + 1) != o)) mbar_arrive(empty_c(slot));
      if (!warp_wait16(mma_done(s), (j / kNSX) & 1, wc)) break;
      tc_fence_after();
      uint32_t d[kMT];
      tmem_ld16(tmem + lane_base + kDCol0 + b * kMT, d);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pdone(s));
      if (has_delta) {
#pragma unroll
        for (int m = 0; m < kMT; ++m) acc[m] = fmaf(dl, as[m], fmaf(sc, __uint_as_float(d[m]), acc[m]));
      } else {
#pragma unroll
        for (int m = 0; m < kMT; ++m) acc[m] = fmaf(sc, __uint_as_float(d[m]), acc[m]);
      }
    }
    tc_fence_before();
  }

  // ---------------------------------------------------------------- split-K reduction + store
  __syncthreads();  // every role is past its loop
  griddep_wait();   // Y may be read or written by the preceding grid (returns at once by now)
  const bool aborted = *abort_flag != 0;
  if (aborted && warp == 0 && lane == 0) {
    // Let every copy the producer issued land before the shared memory is reused
    // or the CTA exits.
    volatile int never = 0;
    const WaitCtx drain{&never, 50000000ull, kDevTimeoutProducer, status};
    for (int gi = max(0, w_issued - kNG); gi < w_issued; ++gi) mbar_wait(full_w(gi % kNG), (gi / kNG) & 1, drain);
    for (int gi = max(0, x_issued - kNG); gi < x_issued; ++gi) mbar_wait(full_x(gi % kNG), (gi / kNG) & 1, drain);
    for (int o = max(0, chunks_loaded - kChunkSlots); o < chunks_loaded; ++o)
      mbar_wait(full_c(o % kChunkSlots), (o / kChunkSlots) & 1, drain);
  }
  if (aborted) __syncthreads();  // uniform: the flag no longer changes
  if (aborted) {
#pragma unroll
    for (int m = 0; m < kMT; ++m) acc[m] = __int_as_float(0x7fc00000);
  }
  const bool promote = warp >= 7 && warp <= 10;
  if (splits == 1) {
    if (promote) {
#pragma unroll
      for (int m = 0; m < kMT; ++m)
        if (m < p.M) store_y_any(p.Y, p.y_kind, static_cast<size_t>(m) * p.N + n0 + row, acc[m]);
    }
  } else {
    // Partials, row-major [128 rows][16 tokens], staged in the first weight stage
    // (every copy into the ring has landed and been consumed): the rows rank o
    // owns are one contiguous block.
    float* const stage = reinterpret_cast<float*>(gbase + (sw - base));
    if (promote) {
      float4* dst = reinterpret_cast<float4*>(stage + row * kMT);
#pragma unroll
      for (int v4 = 0; v4 < kMT / 4; ++v4)
        dst[v4] = make_float4(acc[4 * v4], acc[4 * v4 + 1], acc[4 * v4 + 2], acc[4 * v4 + 3]);
      fence_proxy_async_smem();  // make the generic writes visible to the bulk copies
      named_sync16(1, 128);
    }
    cluster_wait();  // every rank's barriers are initialized and armed
    if (warp == 7 && lane < splits) {
      const int o = lane;
      const int rows_o = min(kTileN - o * rpr, rpr);
      if (rows_o > 0) {
        bulk_copy_to_peer(mapa_shared(sred + static_cast<uint32_t>(seg * rpr * kMT * 4), o),
                          sw + static_cast<uint32_t>(o * rpr * kMT * 4), static_cast<uint32_t>(rows_o * kMT * 4),
                          mapa_shared(red_full, o));
      }
      bulk_commit_group();
      bulk_wait_group_read0();  // the staging buffer stays valid until the copies have read it
    }
    const float* red = reinterpret_cast<const float*>(gbase + (sred - base));
    const int total = own_rows * p.M;
    if (static_cast<int>(threadIdx.x) < total) {
      volatile int never = 0;
      const WaitCtx wred{&never, p.timeout_ns, kDevTimeoutFixup, status};
      mbar_wait(red_full, 0, wred);
    }
    for (int t = threadIdx.x; t < total; t += kThreads) {
      const int m = t / own_rows;
      const int lr = t - m * own_rows;
      float sum = 0.0f;
      for (int src = 0; src < splits; ++src) sum += red[(src * rpr + lr) * kMT + m];
      store_y_any(p.Y, p.y_kind, static_cast<size_t>(m) * p.N + n0 + seg * rpr + lr, sum);
    }
  }

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
static cudaError_t launch_decode16_xk(const CUtensorMap& tm_x, const CUtensorMap& tm_s, const CUtensorMap& tm_d,
                                      const GemmParams& p, unsigned* status, cudaStream_t st) {
  static PerContextOnce attr_set;  // redone after a context rebuild
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_set.needed(dev)) {
    e = cudaFuncSetAttribute(decode16_kernel<XK>, cudaFuncAttributeMaxDynamicSharedMemorySize, d16::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set.done(dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.N / kTileN, p.splits, 1);
  cfg.blockDim = dim3(d16::kThreads, 1, 1);
  cfg.dynamicSmemBytes = d16::kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, decode16_kernel<XK>, tm_x, tm_s, tm_d, p, status);
}

int decode16_max_splits() { return d16::kMaxSplits; }

cudaError_t launch_decode16(int x_kind, const CUtensorMap& tm_x, const CUtensorMap& tm_s, const CUtensorMap& tm_d,
                            const GemmParams& p, cudaStream_t stream) {
  unsigned* status = status_word();
  if (!status) return cudaErrorInvalidSymbol;
  if (p.splits < 1 || p.splits > d16::kMaxSplits || p.M < 1 || p.M > d16::kMT || p.x_scale)
    return cudaErrorInvalidValue;
  return x_kind == kXBF16 ? launch_decode16_xk<kXBF16>(tm_x, tm_s, tm_d, p, status, stream)
                          : launch_decode16_xk<kXF16>(tm_x, tm_s, tm_d, p, status, stream);
}

}  // namespace wq
