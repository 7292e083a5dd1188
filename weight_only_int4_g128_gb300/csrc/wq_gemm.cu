// wq_gemm.cu -- the tcgen05 W4A16 / W4A8 GEMM for sm_103a.
//
// What it computes (from "Marlin INT4 on Ada -- how it works", section "The
// core mismatch: symmetric vs asymmetric"):
//   Y[m][n] = sum_k X[m][k] * W_sym[k][n] + sum_g a_sum[m][g] * delta[g][n]
//   W_sym[k][n] = (q[k][n] - 8) * scale[g][n],  a_sum[m][g] = sum_{k in g} X[m][k]
// The second term is the zero-point correction; it is accumulated into the
// same TMEM accumulator as extra "K" steps (see below), so there is no
// second pass over Y.  The operands are fp16: bf16 activations arrive as a
// per-token power-of-two scaled fp16 copy (exact) and W4A8's int8 activations
// (HyperQwen article, "hidden mine") as fp16 (exact); the accumulator is
// multiplied by the per-token factor (2^-e, or x_scale) in the epilogue.
//
// Tiling (swap-AB): one CTA owns 128 output columns n (the MMA's M = 128,
// i.e. 128 TMEM lanes, one weight row per lane) and BT tokens (the MMA's N).
//   warp 0      TMA producer: activation tile [BT x 128 k] (one 3-D box = two
//               128-byte swizzled atoms), the packed weight tile (one
//               contiguous 8 KB block, bulk copy) and the scale row.
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma (A from TMEM,
//               B = activations from shared memory) and tcgen05.commit.
//   warps 2..9  dequant: each thread owns one weight row (a TMEM lane), turns
//               its codes into scaled fp16 values in registers and stores them
//               into a TMEM A-stage with tcgen05.st (the weights never pass
//               through shared memory once dequantized).  128- and 256-token
//               tiles: two groups of four warps take alternate stages, a thread
//               the whole 128-k row; smaller tiles: all eight warps every stage,
//               a thread one 64-k half.  Then the epilogue.
// Correction as K-augmentation: a_sum (fp32, computed once by a pre-pass) is
// split into bf16 hi/lo and laid out as extra activation columns
// [a_hi | a_lo | a_hi]; the dequant warps write the matching weight-side
// columns [d_hi | d_hi | d_lo] (delta split the same way).  Their bf16 MMAs add
// a_hi*d_hi + a_lo*d_hi + a_hi*d_lo, which is a_sum*delta up to ~2^-16
// relative.
// Epilogue: with one K segment the dequant warps convert the accumulator into
// a [BT tokens][128 columns] image over the idle activation ring and one TMA
// tensor store writes it to Y (whole 256-byte row segments).
// Split-K: gridDim.z segments of k-blocks form a thread-block cluster; the
// partials are reduced through distributed shared memory in rank order
// (deterministic) and written to Y.
//
// Every wait is bounded; on expiry the CTA records a status bit, drains what
// it issued, frees its TMEM and returns.
#include <mutex>

#include "wq_device.cuh"

namespace wq {

// Device status word: bounded waits that expire OR a code into it.
static __device__ unsigned int g_status = 0;

constexpr int kGemmThreads = 320;  // producer, MMA issuer, 8 dequant/epilogue warps
constexpr int kDqWarps = 8;

template <int BT>
struct Cfg {
  static constexpr int kXStageBytes = BT * kKBlock * 2;              // two SW128 atoms
  static constexpr int kXAtomBytes = BT * 128;                        // one box of 64 k
  static constexpr int kWStageBytes = kTileN * kWordsPerKBlock * 4;  // 8 KB
  // tiles of <= 64 tokens run two CTAs per SM (<= 113 KB shared memory, 256 TMEM columns)
  static constexpr bool kTwoPerSM = BT <= 64;
  static constexpr int kNSX = (BT >= 256) ? 3 : (BT >= 128) ? 5 : (BT >= 64) ? 4 : 6;
  // TMEM A-stages (64 columns each); at most kNSX so that the per-stage
  // mma_done barrier also tells when an A-stage is free again
  static constexpr int kNSA = kTwoPerSM ? 3 : (kNSX < 4 ? kNSX : 4);
  static constexpr int kDCol = kTwoPerSM ? 192 : 256;                // accumulator columns
  static constexpr int kTmemCols = kTwoPerSM ? 256 : 512;
  // 128- and 256-token tiles (one CTA per SM) split the dequant warps into two
  // groups that take alternate stages, each thread a whole 128-k row, and read
  // their group scales straight from S; smaller tiles (two CTAs per SM) keep all
  // eight warps on every stage (two per row) with the scale rows staged in chunks.
  static constexpr bool kGroups = BT >= 128;
  static constexpr int kChunk = 8;  // groups per scale chunk (the index math below uses >> 3)
  static constexpr int kSChunkBytes = kChunk * kTileN * 2;            // 2 KB of fp16 scale rows
  static constexpr int kChunkSlots = 2;
  static constexpr int kNumBars = 4 * kNSX + kNSA + 1 + 2 * kChunkSlots;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kNSX * (kXStageBytes + kWStageBytes) +
                                    kChunkSlots * kSChunkBytes + kNumBars * 8 + 16;
  static_assert(BT % 16 == 0 && BT >= 16 && BT <= 256, "MMA N for M=128 is 16..256, step 16");
  static_assert(kDCol + BT <= kTmemCols, "TMEM budget");
  static_assert(!kTwoPerSM || kSmemBytes + 1024 <= 116 * 1024, "two CTAs per SM");
  static_assert(kNSA * 64 <= kDCol, "TMEM budget");
  static_assert(kNSA <= kNSX, "mma_done is indexed by stage");
  // split-K: the reduction buffer red[splits][128][rpr + 4] fp32 (rows of the tile
  // per rank rounded up to 16) and the owner's output image [rpr][128] (fp32 at
  // most) after it, over the idle activation and weight rings
  static constexpr int split_rpr(int splits) { return ((BT + splits - 1) / splits + 15) & ~15; }
  static constexpr int split_bytes(int splits) {
    return splits * kTileN * (split_rpr(splits) + 4) * 4 + split_rpr(splits) * kTileN * 4;
  }
  static constexpr int split_bytes_max() {
    int m = 0;
    for (int k = 2; k <= 8; ++k) m = split_bytes(k) > m ? split_bytes(k) : m;
    return m;
  }
  static_assert(split_bytes_max() <= kNSX * (kXStageBytes + kWStageBytes),
                "split-K reduction buffer reuses the stage ring");
  // the output tile's image (fp32 at most) and the tile's per-token factors are
  // staged over the activation ring
  static constexpr int kXsOffset = BT * kTileN * 4;
  static_assert(kXsOffset + BT * 4 <= kNSX * kXStageBytes, "the output tile is staged over the activation ring");
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Epilogue image of one tile over shared memory: [BT tokens][128 columns] of
// type YK (row-major, as the TMA store of Y reads it).  This thread owns column
// `col` and writes tokens 16 c + j of its chunks c = h + 2 i; with XS each value is
// first multiplied by its token's factor, read per chunk from the factors staged
// in shared memory at xs_s (1.0 for tokens past M, which the store clips).
template <int YK, int kCh, bool XS>
__device__ __forceinline__ void write_image(uint32_t img, int col, int h, const uint32_t (&r)[kCh][16],
                                            uint32_t xs_s) {
  constexpr uint32_t es = (YK == kYF32) ? 4 : 2;
  const uint32_t base = img + static_cast<uint32_t>(col) * es;
#pragma unroll
  for (int i = 0; i < kCh; ++i) {
    const int c = h + 2 * i;
    float sc[16];
    if constexpr (XS) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(sc[4 * q]), "=f"(sc[4 * q + 1]), "=f"(sc[4 * q + 2]), "=f"(sc[4 * q + 3])
                     : "r"(xs_s + static_cast<uint32_t>(64 * c + 16 * q)));
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int ml = 16 * c + j;
      float v = __uint_as_float(r[i][j]);
      if constexpr (XS) v *= sc[j];
      const uint32_t a = base + static_cast<uint32_t>(ml) * (kTileN * es);
      if constexpr (YK == kYF16) {
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(__half_as_ushort(__float2half_rn(v))) : "memory");
      } else if constexpr (YK == kYBF16) {
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(__bfloat16_as_ushort(__float2bfloat16_rn(v))) : "memory");
      } else {
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(__float_as_uint(v)) : "memory");
      }
    }
  }
}

// All lanes wait; the warp proceeds only if every lane saw the phase complete,
// so the .sync.aligned tcgen05 ops that follow stay warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

template <int BT, int XK>
__global__ void __launch_bounds__(kGemmThreads, (BT <= 64) ? 2 : 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_aug,
                const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_y,
                const GemmParams p) {
  using C = Cfg<BT>;
  static_assert(XK == kXF16, "fp16 operands (bf16 and int8 activations arrive as fp16)");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t sx = base;
  const uint32_t sw = sx + C::kNSX * C::kXStageBytes;
  const uint32_t sch = sw + C::kNSX * C::kWStageBytes;  // scale chunk slots
  const uint32_t sbar = sch + C::kChunkSlots * C::kSChunkBytes;
  // The packed weight tile of a stage travels on its own barrier and is copied
  // one stage ahead of the stage's activation tile, so the dequant of a stage
  // overlaps the copy of its (much larger) activation tile.
  // full_x: activation tile of stage s landed; full_w: weight tile landed (a
  // correction stage has none: the producer only completes the phase);
  // empty_w: the dequant warps have read the weight tile; mma_done: the
  // k-block's MMAs completed (one tcgen05.commit per k-block; frees the
  // activation tile and the TMEM A-stage); full_a: the A-stage holds
  // dequantized weights.
  auto full_x = [&](int s) { return sbar + 8u * s; };
  auto empty_w = [&](int s) { return sbar + 8u * (C::kNSX + s); };
  auto mma_done = [&](int s) { return sbar + 8u * (2 * C::kNSX + s); };
  auto full_w = [&](int s) { return sbar + 8u * (3 * C::kNSX + s); };
  auto full_a = [&](int a) { return sbar + 8u * (4 * C::kNSX + a); };
  const uint32_t done_bar = sbar + 8u * (4 * C::kNSX + C::kNSA);
  // full_c / empty_c: scale rows of 8 consecutive groups (one chunk) landed /
  // released by the dequant warps.
  auto full_c = [&](int c) { return sbar + 8u * (4 * C::kNSX + C::kNSA + 1 + c); };
  auto empty_c = [&](int c) { return sbar + 8u * (4 * C::kNSX + C::kNSA + 1 + C::kChunkSlots + c); };
  const uint32_t misc = sbar + 8u * C::kNumBars;
  uint8_t* const gmisc = gbase + (misc - base);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gmisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gmisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(gmisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tile = p.tile_base + static_cast<int>(blockIdx.x);  // column tile fastest
  const int ntiles = p.N / kTileN;
  const int n_tile = tile % ntiles;
  const int n0 = n_tile * kTileN;
  const int m0 = (tile / ntiles) * BT;
  const int seg = blockIdx.z;
  // segment 0 carries the correction stages, so it may take fewer k-blocks
  const int kb_first = p.kb_first > 0 ? p.kb_first : p.kb_per_split;
  const int kb0 = (seg == 0) ? 0 : kb_first + (seg - 1) * p.kb_per_split;
  const int kb1 = min(p.kb_total, (seg == 0) ? kb_first : kb0 + p.kb_per_split);
  const int n_aug = (seg == 0) ? p.aug_stages : 0;
  const int n_stages = n_aug + max(0, kb1 - kb0);
  // group size is 128 (group = k-block) or K (one group per column)
  const bool per_channel = p.group_size != kKBlock;
  const int g_first = per_channel ? 0 : kb0;  // first group of this K segment
  // chunk ordinal (0, 1, ...) and row of the k-block `kb` (chunks of 8 groups)
  auto chunk_of = [&](int kb) { return per_channel ? 0 : (kb >> 3) - (g_first >> 3); };
  auto chunk_row = [&](int kb) { return per_channel ? 0 : (kb & 7); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kNSX; ++s) {
      mbar_init(full_x(s), 1);
      mbar_init(full_w(s), 1);
      mbar_init(empty_w(s), C::kGroups ? kDqWarps / 2 : kDqWarps);  // one arrive per warp reading the stage
      mbar_init(mma_done(s), 1);
    }
    for (int a = 0; a < C::kNSA; ++a) {
      mbar_init(full_a(a), C::kGroups ? kDqWarps / 2 : kDqWarps);
    }
    for (int c = 0; c < C::kChunkSlots; ++c) {
      mbar_init(full_c(c), 1);
      mbar_init(empty_c(c), kDqWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_s);
    if (p.aug_stages > 0) prefetch_tensormap(&tm_aug);
  }
  if (warp == 1) {
    tmem_alloc(misc, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Programmatic dependent launch.  Nothing here reads or writes memory a preceding
  // grid may write (X, the correction columns of the pre-pass, Y) before the wait.
  // The next grid in the stream may be scheduled at once (it waits for this one to
  // complete before it touches memory this one uses), except after a main launch
  // with a tail (tail == 2): only once every CTA of it is past its wait, so that the
  // tail launch starts after the pre-pass completed.  The tail launch (tail == 1)
  // does not wait for the main launch (they write disjoint tiles and read what the
  // pre-pass wrote); it waits before exiting, so its completion implies the main
  // launch's.
  if (p.tail == 2) {
    griddep_wait();
    griddep_launch_dependents();
  } else {
    griddep_launch_dependents();
    if (p.tail == 0) griddep_wait();
  }

  int issued = 0;         // stages whose activation tile the producer lane has issued
  int w_issued = 0;       // stages whose weight side the producer lane has issued
  int chunks_loaded = 0;  // producer lane: scale chunks [0, chunks_loaded) issued
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutProducer, &g_status};
      // A weight tile is read again by every token tile's CTA, waves apart; Y is
      // written once: weights stay in L2 ahead of the output's lines.
      const uint64_t pol_w = l2_evict_last();
      // Weight side of stage it2: the packed tile (+ a scale chunk when its k-block
      // starts one); a correction stage has no weight tile and only completes the
      // phase.  Every wait comes before the first copy of the stage.
      auto issue_w = [&](int it2) -> bool {
        const int s2 = it2 % C::kNSX;
        if (!mbar_wait(empty_w(s2), ((it2 / C::kNSX) & 1) ^ 1, wc)) return false;
        if (it2 < n_aug) {
          mbar_arrive(full_w(s2));
          return true;
        }
        const int kb = kb0 + (it2 - n_aug);
        const int o = chunk_of(kb);
        if (!C::kGroups && o >= chunks_loaded) {
          const int slot = o % C::kChunkSlots;
          if (!mbar_wait(empty_c(slot), ((o / C::kChunkSlots) & 1) ^ 1, wc)) return false;
          mbar_arrive_expect_tx(full_c(slot), C::kSChunkBytes);
          tma_load_2d(sch + slot * C::kSChunkBytes, &tm_s, full_c(slot), n0, ((g_first >> 3) + o) * C::kChunk);
          chunks_loaded = o + 1;
        }
        mbar_arrive_expect_tx(full_w(s2), C::kWStageBytes);
        // packed weight tile: one contiguous 8 KB block of the blocked layout
        bulk_load_hint(sw + s2 * C::kWStageBytes, p.B + (static_cast<size_t>(n_tile) * p.kb_total + kb) * 2048,
                       C::kWStageBytes, full_w(s2), pol_w);
        return true;
      };
      bool ok = n_stages == 0 || issue_w(0);
      if (ok) w_issued = n_stages > 0 ? 1 : 0;
      for (int it = 0; ok && it < n_stages; ++it) {
        // weight side one stage ahead
        if (it + 1 < n_stages) {
          if (!issue_w(it + 1)) break;
          w_issued = it + 2;
        }
        // activation tile [BT x 128 k]: one 3-D box {64 k, BT rows, 2 halves}
        const int s = it % C::kNSX;
        if (!mbar_wait(mma_done(s), ((it / C::kNSX) & 1) ^ 1, wc)) break;
        const uint32_t xdst = sx + s * C::kXStageBytes;
        mbar_arrive_expect_tx(full_x(s), C::kXStageBytes);
        if (it < n_aug) tma_load_3d(xdst, &tm_aug, full_x(s), 0, m0, 2 * it);
        else tma_load_3d(xdst, &tm_x, full_x(s), 0, m0, 2 * (kb0 + (it - n_aug)));
        issued = it + 1;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMma, &g_status};
      const uint32_t d_tmem = tmem + C::kDCol;
      constexpr uint32_t id_x = idesc_f16(XK, 128, BT);
      constexpr uint32_t id_aug = idesc_f16(1, 128, BT);
      const uint64_t desc0 = desc_kmajor_sw128(sx);
      for (int it = 0; it < n_stages; ++it) {
        const int s = it % C::kNSX;
        const int a = it % C::kNSA;
        if (!mbar_wait(full_a(a), (it / C::kNSA) & 1, wc)) break;
        if (!mbar_wait(full_x(s), (it / C::kNSX) & 1, wc)) break;  // activation tile landed
        tc_fence_after();
        const uint64_t ds = desc0 + static_cast<uint64_t>((s * C::kXStageBytes) >> 4);
        const uint32_t id = (it < n_aug) ? id_aug : id_x;
        const uint32_t at = tmem + a * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          mma_ts(d_tmem, at + i * 8, ds + (((i >> 2) * C::kXAtomBytes + (i & 3) * 32) >> 4), id,
                 (it > 0 || i > 0) ? 1u : 0u);
        mma_commit(mma_done(s));
      }
      mma_commit(done_bar);
    }
  } else {
    // ------------------------------------------------------------ dequant + epilogue
    // Two warps per TMEM lane quarter, h = 0 or 1.  Tiles of 128 or 256 tokens:
    // warp group h takes the stages it with it % 2 == h (see below); smaller tiles:
    // warp half h owns words [8h, 8h + 8) of each weight row (A-stage columns
    // [32h, 32h + 32)) of every stage.  In the epilogue warp h takes the
    // 16-column chunks c with c % 2 == h.
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, &g_status};
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;        // 0 or 1
    const int row = q * 32 + lane;        // weight row of the tile = TMEM lane
    const int n = n0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint8_t* wring = gbase + (sw - base);

    if constexpr (C::kGroups) {
    // Two groups of four warps (one per TMEM lane quarter) take alternate stages:
    // group h dequantizes the k-blocks it with it % 2 == h, each thread a whole
    // 128-k weight row into the stage's 64 A columns, so every barrier round trip
    // of a group is spread over two stages of MMA time.  The row's group scale
    // is read from S into a register one of the group's stages ahead.
    auto scale_of = [&](int st) -> __half {
      if (st >= n_stages || st < n_aug) return __ushort_as_half(0);
      const int kb = kb0 + (st - n_aug);
      return __ldg(p.S + static_cast<size_t>(per_channel ? 0 : kb) * p.N + n);
    };
    __half sc_next = scale_of(h);
    for (int it = h; it < n_stages; it += 2) {
      const int s = it % C::kNSX;
      const uint32_t ph = (it / C::kNSX) & 1;
      const int a = it % C::kNSA;
      const uint32_t a_tmem = tmem + lane_base + a * 64;
      const __half sc = sc_next;
      sc_next = scale_of(it + 2);
      // A-stage a was last read by the MMAs of k-block it - kNSA.  Waiting for them
      // first also makes the full_w wait below exact: a parity wait only tells the
      // current phase from the one just before it, and the previous tile of slot s
      // (k-block it - kNSX, possibly the other group's, whose copy may land after
      // this group's own earlier tiles) has been consumed once MMA it - kNSA is
      // done (MMAs complete in order and kNSA <= kNSX).
      if (it >= C::kNSA) {
        const int pk = it - C::kNSA;
        if (!warp_wait(mma_done(pk % C::kNSX), (pk / C::kNSX) & 1, wc)) break;
        tc_fence_after();
      }
      uint32_t v[64];
      if (it < n_aug) {
        // weight-side correction columns [d_hi | d_hi | d_lo | 0...] of this row,
        // prepared per call in the workspace: 128 bf16 = 64 columns, 16 vector loads.
        const uint4* src = reinterpret_cast<const uint4*>(p.delta_aug + static_cast<size_t>(n) * p.kaug + it * kKBlock);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint4 t = __ldg(src + i);
          v[4 * i + 0] = t.x;
          v[4 * i + 1] = t.y;
          v[4 * i + 2] = t.z;
          v[4 * i + 3] = t.w;
        }
        if (!warp_wait(full_w(s), ph, wc)) break;  // the producer's (empty) weight side of the stage
        if (lane == 0) mbar_arrive(empty_w(s));
      } else {
        if (!warp_wait(full_w(s), ph, wc)) break;
        const uint8_t* const slot = wring + s * C::kWStageBytes;
        // the row's four 16-byte chunks (chunk c stored at c ^ ((row / 2) % 4))
        uint4 wc4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          wc4[c] = *reinterpret_cast<const uint4*>(slot + row * 64 + 16 * (c ^ ((row >> 1) & 3)));
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_w(s));
        const uint32_t s2 = static_cast<uint32_t>(__half_as_ushort(sc)) * 0x00010001u;
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          const uint4& q4 = wc4[w >> 2];
          const uint32_t word = (w & 3) == 0 ? q4.x : (w & 3) == 1 ? q4.y : (w & 3) == 2 ? q4.z : q4.w;
          uint32_t o[4];
          dq8_f16_scaled(word, s2, o);
#pragma unroll
          for (int e = 0; e < 4; ++e) v[4 * w + e] = o[e];
        }
      }
      tmem_st32(a_tmem, *reinterpret_cast<const uint32_t(*)[32]>(&v[0]));
      tmem_st32(a_tmem + 32, *reinterpret_cast<const uint32_t(*)[32]>(&v[32]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_a(a));
    }
    } else {
    for (int it = 0; it < n_stages; ++it) {
      const int s = it % C::kNSX;
      const uint32_t ph = (it / C::kNSX) & 1;
      const int a = it % C::kNSA;
      const uint32_t a_tmem = tmem + lane_base + a * 64 + 32 * h;
      uint32_t v[32];
      if (it < n_aug) {
        // weight-side correction columns [d_hi | d_hi | d_lo | 0...] of this row,
        // prepared per call in the workspace: 64 bf16 = 32 columns, 8 vector loads.
        const uint4* src = reinterpret_cast<const uint4*>(
            p.delta_aug + static_cast<size_t>(n) * p.kaug + it * kKBlock + 64 * h);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 t = __ldg(src + i);
          v[4 * i + 0] = t.x;
          v[4 * i + 1] = t.y;
          v[4 * i + 2] = t.z;
          v[4 * i + 3] = t.w;
        }
        if (!warp_wait(full_w(s), ph, wc)) break;  // the producer's (empty) weight side of the stage
        if (lane == 0) mbar_arrive(empty_w(s));
      } else {
        if (!warp_wait(full_w(s), ph, wc)) break;
        const int kb = kb0 + (it - n_aug);
        const int o = chunk_of(kb);
        const int slot = o % C::kChunkSlots;
        if (!warp_wait(full_c(slot), (o / C::kChunkSlots) & 1, wc)) break;
        const __half sc = reinterpret_cast<const __half*>(
            gbase + (sch - base) + slot * C::kSChunkBytes)[chunk_row(kb) * kTileN + row];
        const uint8_t* wrow = wring + s * C::kWStageBytes + row * 64;
        const uint4 w0 = *reinterpret_cast<const uint4*>(wrow + 16 * ((2 * h) ^ ((row >> 1) & 3)));
        const uint4 w1 = *reinterpret_cast<const uint4*>(wrow + 16 * ((2 * h + 1) ^ ((row >> 1) & 3)));
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(empty_w(s));
          if (kb + 1 == kb1 || chunk_of(kb + 1) != o) mbar_arrive(empty_c(slot));  // chunk done
        }
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t s2 = static_cast<uint32_t>(__half_as_ushort(sc)) * 0x00010001u;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          uint32_t o[4];
          dq8_f16_scaled(words[w], s2, o);
#pragma unroll
          for (int e = 0; e < 4; ++e) v[4 * w + e] = o[e];
        }
      }
      if (it >= C::kNSA) {  // A-stage a was last read by the MMAs of k-block it - kNSA
        const int pk = it - C::kNSA;
        if (!warp_wait(mma_done(pk % C::kNSX), (pk / C::kNSX) & 1, wc)) break;
        tc_fence_after();
      }
      tmem_st32(a_tmem, v);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_a(a));
    }
    }

    // ---- epilogue (single K segment): accumulator -> Y
    warp_wait(done_bar, 0, wc);
    // Every MMA has completed, so the activation ring is idle: the tile's per-token
    // factors go next to where the image will be (1.0 past M: those rows are clipped).
    const uint32_t xs_s = sx + C::kXsOffset;
    if (p.x_scale && p.splits == 1 && !*abort_flag) {
      const int mlim = min(BT, p.M - m0);
      float* const xs_g = reinterpret_cast<float*>(gbase + C::kXsOffset);
      for (int i = threadIdx.x - 64; i < BT; i += 32 * kDqWarps) xs_g[i] = (i < mlim) ? __ldg(p.x_scale + m0 + i) : 1.0f;
    }
    named_bar_sync(1, 32 * kDqWarps);
    tc_fence_after();
    // The tile's outputs are converted into a [BT tokens][128 columns] image over
    // the (now idle) activation ring, then written by one TMA tensor store: full
    // 256-byte row segments instead of 2-byte stores scattered over BT rows of Y.
    // Tokens past M are outside the tensor map and are not written.
    const bool store_tile = !*abort_flag && p.splits == 1;  // uniform: no wait can set the flag past here
    if (store_tile) {
      const uint32_t dt = tmem + lane_base + C::kDCol;
      // this warp's 16-column chunks c = h, h + 2, ...: every TMEM load is issued
      // before the one wait, so the load latency is paid once per tile
      constexpr int kCh = BT / 32;
      uint32_t r[kCh][16];
#pragma unroll
      for (int i = 0; i < kCh; ++i) tmem_ld16(dt + 16 * (h + 2 * i), r[i]);
      tmem_wait_ld();
      // the output type and whether a per-token factor applies are decided once,
      // outside the element loop, and every element is one shared-memory store
      const bool xs_on = p.x_scale != nullptr;
      switch (p.y_kind) {
        case kYF16:
          if (xs_on) write_image<kYF16, kCh, true>(sx, row, h, r, xs_s);
          else write_image<kYF16, kCh, false>(sx, row, h, r, xs_s);
          break;
        case kYBF16:
          if (xs_on) write_image<kYBF16, kCh, true>(sx, row, h, r, xs_s);
          else write_image<kYBF16, kCh, false>(sx, row, h, r, xs_s);
          break;
        default:
          if (xs_on) write_image<kYF32, kCh, true>(sx, row, h, r, xs_s);
          else write_image<kYF32, kCh, false>(sx, row, h, r, xs_s);
          break;
      }
      fence_proxy_async_smem();  // the image's generic writes become visible to the TMA store
    }
    named_bar_sync(1, 32 * kDqWarps);
    if (store_tile && warp == 2 && lane == 0) {
      const uint32_t box = 16u * kTileN * ((p.y_kind == kYF32) ? 4u : 2u);
      const uint64_t pol_y = l2_evict_first();
      for (int b = 0; 16 * b < BT && m0 + 16 * b < p.M; ++b)
        tma_store_2d_hint(&tm_y, sx + b * box, n0, m0 + 16 * b, pol_y);
      bulk_commit_group();
      bulk_wait_group_read0();  // the image is read before the CTA's shared memory is released
    }
    tc_fence_before();
  }

  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // Let every copy the producer issued land before the CTA exits.
    volatile int never = 0;
    const WaitCtx drain{&never, 50000000ull, kDevTimeoutProducer, &g_status};
    for (int it = max(0, issued - C::kNSX); it < issued; ++it)
      mbar_wait(full_x(it % C::kNSX), (it / C::kNSX) & 1, drain);
    for (int it = max(0, w_issued - C::kNSX); it < w_issued; ++it)
      mbar_wait(full_w(it % C::kNSX), (it / C::kNSX) & 1, drain);
    for (int o = max(0, chunks_loaded - C::kChunkSlots); o < chunks_loaded; ++o)
      mbar_wait(full_c(o % C::kChunkSlots), (o / C::kChunkSlots) & 1, drain);
  }
  __syncthreads();

  // ---- split-K over a thread-block cluster (the K segments of one output tile).
  // Rows (tokens) [r*rpr, (r+1)*rpr) of the tile belong to rank r (rpr a multiple
  // of 16).  Every CTA pushes its fp32 partial of those rows into rank r's shared
  // memory with 16-byte stores (remote for the other ranks), laid out
  // red[src][row][rpr_pad] (rows are the 128 weight rows of the tile); the owner
  // sums the partials in rank order (deterministic) and stores its rows of Y.
  if (p.splits > 1) {
    const int splits = p.splits;
    const int rpr = C::split_rpr(splits);  // a multiple of 16: whole 16-row store boxes
    const int rpr_pad = rpr + 4;  // breaks shared-memory bank conflicts between rows
    const int mlim = min(BT, p.M - m0);
    const bool math = warp >= 2;
    const int q = warp & 3;
    const int h = math ? (warp - 2) >> 2 : 0;
    const int row = q * 32 + lane;
    float* const red = reinterpret_cast<float*>(gbase);  // over the (now idle) stage ring
    cluster_sync_all();  // every CTA of the cluster is past its mainloop: rings are free
    if (math) {
      tc_fence_after();
      const bool aborted = *abort_flag != 0;
      const uint32_t dt = tmem + (static_cast<uint32_t>(q * 32) << 16) + C::kDCol;
      const uint32_t red_row = smem_u32(red) + static_cast<uint32_t>((seg * kTileN + row) * rpr_pad * 4);
      // this warp's 16-column chunks c = h, h + 2, ...: every TMEM load is issued
      // before the one wait, then the partials are pushed to their owners
      constexpr int kCh = BT / 32;
      uint32_t r[kCh][16];
#pragma unroll
      for (int i = 0; i < kCh; ++i) tmem_ld16(dt + 16 * (h + 2 * i), r[i]);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < kCh; ++i) {
        const int c = h + 2 * i;
        if (16 * c >= mlim) break;
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const int ml = 16 * c + j;  // 4 consecutive rows, same owner (rpr % 4 == 0)
          if (ml < mlim) {
            const int owner = ml / rpr;
            const int local = ml - owner * rpr;
            const uint32_t la = red_row + static_cast<uint32_t>(local * 4);
            const float nanv = __int_as_float(0x7fc00000);
            const float v0 = aborted ? nanv : __uint_as_float(r[i][j]);
            const float v1 = aborted ? nanv : __uint_as_float(r[i][j + 1]);
            const float v2 = aborted ? nanv : __uint_as_float(r[i][j + 2]);
            const float v3 = aborted ? nanv : __uint_as_float(r[i][j + 3]);
            // rows this CTA owns stay in its own shared memory (a plain store);
            // the others go to their owner over the cluster
            if (owner == seg)
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(la), "f"(v0), "f"(v1), "f"(v2), "f"(v3)
                           : "memory");
            else
              st_dsmem_v4(mapa_shared(la, owner), v0, v1, v2, v3);
          }
        }
      }
      tc_fence_before();
    }
    cluster_sync_all();  // all pushes landed
    // The owner sums its rows' partials in rank order (deterministic) into an image
    // [rpr tokens][128 columns] of Y's type after the reduction buffer, which TMA
    // stores of 16-token boxes write to Y (rows past M are clipped by the map).
    const int lo = seg * rpr;
    const int hi = min(mlim, lo + rpr);
    const uint32_t img = smem_u32(red) + static_cast<uint32_t>(splits * kTileN * rpr_pad * 4);
    if (math && !*abort_flag) {
      const uint32_t ecol = static_cast<uint32_t>(row) * ((p.y_kind == kYF32) ? 4u : 2u);
      const uint32_t pitch = (p.y_kind == kYF32) ? kTileN * 4u : kTileN * 2u;
      for (int l4 = 4 * h; lo + l4 < hi; l4 += 8) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int src = 0; src < splits; ++src) {
          const float4 v = *reinterpret_cast<const float4*>(red + (src * kTileN + row) * rpr_pad + l4);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        float a4[4] = {acc.x, acc.y, acc.z, acc.w};
        if (p.x_scale) {
#pragma unroll
          for (int e = 0; e < 4; ++e) a4[e] *= (lo + l4 + e < hi) ? __ldg(p.x_scale + m0 + lo + l4 + e) : 1.0f;
        }
        const uint32_t a0 = img + static_cast<uint32_t>(l4) * pitch + ecol;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t a = a0 + static_cast<uint32_t>(e) * pitch;
          if (p.y_kind == kYF16)
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(__half_as_ushort(__float2half_rn(a4[e]))) : "memory");
          else if (p.y_kind == kYBF16)
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(__bfloat16_as_ushort(__float2bfloat16_rn(a4[e])))
                         : "memory");
          else
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(__float_as_uint(a4[e])) : "memory");
        }
      }
      fence_proxy_async_smem();  // the image's generic writes become visible to the TMA stores
    }
    __syncthreads();
    if (warp == 2 && lane == 0 && !*abort_flag && hi > lo) {
      const uint32_t box = 16u * kTileN * ((p.y_kind == kYF32) ? 4u : 2u);
      const uint64_t pol_y = l2_evict_first();
      for (int b = 0; lo + 16 * b < hi; ++b) tma_store_2d_hint(&tm_y, img + b * box, n0, m0 + lo + 16 * b, pol_y);
      bulk_commit_group();
      bulk_wait_group_read0();  // the image is read before the CTA's shared memory is released
    }
  }

  if (warp == 1) {
    // Every MMA this CTA issued has completed once the final commit arrived.
    volatile int never = 0;
    const WaitCtx drain{&never, 50000000ull, kDevTimeoutMma, &g_status};
    mbar_wait(done_bar, 0, drain);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (p.tail == 1) griddep_wait();
}

template <int BT, int XK>
static cudaError_t launch_bt(const CUtensorMap& tm_x, const CUtensorMap& tm_aug, const CUtensorMap& tm_s,
                             const CUtensorMap& tm_y, const GemmParams& p, cudaStream_t st) {
  using C = Cfg<BT>;
  static PerContextOnce attr_set;  // redone after a context rebuild
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_set.needed(dev)) {
    e = cudaFuncSetAttribute(gemm_kernel<BT, XK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set.done(dev);
  }
  cudaLaunchConfig_t cfg = {};
  const int tiles = (p.N / kTileN) * ((p.M + BT - 1) / BT);
  const int count = (p.tail == 1) ? tiles - p.tile_base : (p.tile_count > 0 ? p.tile_count : tiles);
  cfg.gridDim = dim3(count, 1, p.splits);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the K segments of a tile form a cluster
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = p.splits;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BT, XK>, tm_x, tm_aug, tm_s, tm_y, p);
}

template <int XK>
static cudaError_t launch_xk(int bt, const CUtensorMap& tm_x, const CUtensorMap& tm_aug, const CUtensorMap& tm_s,
                             const CUtensorMap& tm_y, const GemmParams& p, cudaStream_t st) {
  switch (bt) {
    case 32: return launch_bt<32, XK>(tm_x, tm_aug, tm_s, tm_y, p, st);
    case 64: return launch_bt<64, XK>(tm_x, tm_aug, tm_s, tm_y, p, st);
    case 128: return launch_bt<128, XK>(tm_x, tm_aug, tm_s, tm_y, p, st);
    case 256: return launch_bt<256, XK>(tm_x, tm_aug, tm_s, tm_y, p, st);
    default: return cudaErrorInvalidValue;
  }
}

// fp16 operands only: bf16 activations reach this kernel as their per-token scaled
// fp16 copy (the correction pre-pass), int8 ones as exact fp16.
cudaError_t launch_gemm(int bt, int x_kind, const CUtensorMap& tm_x, const CUtensorMap& tm_aug,
                        const CUtensorMap& tm_s, const CUtensorMap& tm_y, const GemmParams& p, cudaStream_t stream) {
  if (x_kind != kXF16) return cudaErrorInvalidValue;
  return launch_xk<kXF16>(bt, tm_x, tm_aug, tm_s, tm_y, p, stream);
}

// Device address of the status word (host side), looked up once per device
// and again whenever the device's context has been rebuilt (the old address
// then belongs to a context that no longer exists).
unsigned* status_word() {
  static std::mutex mu;
  static PerContextOnce looked_up;
  static unsigned* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || looked_up.needed(dev)) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(ptr);
    looked_up.done(dev);
  }
  return addr[dev];
}

// ---------------------------------------------------------------------------
// Bounded-wait probe: one thread waits on an mbarrier that nothing arrives
// on.  The wait gives up after limit_ns, records kDevTimeoutProbe in the
// status word and the kernel returns normally.
// ---------------------------------------------------------------------------
__global__ void wait_probe_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    const WaitCtx w{&abort_flag, limit_ns, kDevTimeoutProbe, &g_status};
    mbar_wait(smem_u32(&bar), 0, w);
  }
}

cudaError_t launch_wait_probe(unsigned long long limit_ns, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_status(unsigned int* out) {
  return cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
}

cudaError_t clear_status() {
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
}

size_t gemm_smem_bytes(int bt) {
  switch (bt) {
    case 32: return Cfg<32>::kSmemBytes;
    case 64: return Cfg<64>::kSmemBytes;
    case 128: return Cfg<128>::kSmemBytes;
    case 256: return Cfg<256>::kSmemBytes;
    default: return 0;
  }
}

}  // namespace wq
