// wq_gemv.cu -- the weight-streaming decode path (M <= 8 tokens) of the W4A16
// GEMM: each lane streams its own weight-code chunks from HBM into a per-warp
// shared-memory ring (asynchronous copies), loads them into registers,
// dequantizes them there and contracts them with warp-level MMAs, so no
// dequantized weight is ever written to shared or tensor memory.
//
// Why not the tcgen05 pipeline here: with at most 8 tokens the MMA's N is tiny
// and the work is the weight stream (the opening of "Marlin INT4 on Ada -- how
// it works": with no reuse across outputs, the weight reads bound the kernel).
// A tcgen05 MMA takes its weight operand from TMEM or shared memory, so every
// dequantized 128 x 128 block (32 KB of fp16) must first be stored there; on
// this part that staging, not HBM, paces a per-SM pipeline at ~275 ns per 8 KB
// block.  A warp-level MMA takes the weight fragment from registers, where the
// dequant leaves it.
//
// Arithmetic (section "The core mismatch": W_sym = (q - 8) * scale, C = C_sym +
// A_group_sum @ delta).  The MMA operands are the codes with an exact offset,
// one LOP3 per code pair: fp16 1024 + v for the low nibble of each code byte
// and 1024 + 16 v for the high nibble (two accumulator chains), bf16 128 + v.
// Per 128-k block, in fp32:
//     D = D_lo + D_hi / 16 - (1032 * sum_lo x + 72 * sum_hi x)   (= sum (v - 8) x)
//     acc[n][m] += scale[g][n] * D[n][m] + delta[g][n] * a_sum[kb][m]
// (bf16: D = D_all - 136 * sum x), with the activation sums over the block's
// low / high-nibble k formed while the activation tile is staged.  The 8 token
// slots are the MMA's N = 8; slots past M read zeros.
//
// W4A8 rows run through the same kernel: the int8 activations are turned into
// fp16 (exact, |x| <= 127) as they are staged, so every offset-code product
// and block sum is an integer below 2^24 and each block's D is exact in fp32;
// the per-token scale multiplies the result at the store.
//
// A grouped (mixture-of-experts) launch runs the same kernel over all experts:
// blockIdx.z is the expert, whose token rows, weights, scales and delta the CTA
// offsets to; an expert without tokens returns at once.
//
// A gate/up pair weight (16-column groups of 8 gate and the same 8 up columns)
// puts a gate row and its up row 8 rows apart in one m16 strip, which the MMA
// accumulator hands to the same lane: that instance stores silu(gate) * up.
//
// Work split: one CTA per (128-row column tile, K segment); warp w owns rows
// 16 w .. 16 w + 15 of the tile (one m16 strip) for the whole segment.  The K
// segments of a tile form a thread-block cluster and are reduced through
// distributed shared memory (each rank owns a contiguous block of rows).
//
// Order of k inside an MMA.  The sum over k does not depend on the order in
// which k enters an MMA, as long as the weight and activation fragments use the
// same order.  The packed layout gives lane (g, t) of the warp the 16-byte chunk
// t of its rows: words 4t .. 4t+3, i.e. k = 32t .. 32t+31 of the block, each
// word holding four (even k, odd k) code pairs.  MMA step s = 4h + p (h = 0, 1;
// p = 0..3) takes pair p of words 4t + 2h (fragment k 2t, 2t+1) and 4t + 2h + 1
// (fragment k 2t+8, 2t+9); the activation fragment takes x at the same physical
// k: 32t + 16h + 2p (+ 8).  One chunk of codes per row and one 64-byte run of
// the activation row per lane cover a whole k-block with no shuffles.
#include "wq_warp.cuh"

namespace wq {

namespace gv {
constexpr int kWarps = 8;                 // one 16-row strip of the 128-row tile each
constexpr int kThreads = kWarps * 32;
constexpr int kMT = 8;                    // token slots = MMA N
constexpr int kMaxM = kMT;
constexpr int kMaxSplits = 8;             // portable cluster size
constexpr int kMaxSmem = 113 * 1024;      // two CTAs per SM
constexpr int kUint4PerBlock = kTileN * kWordsPerKBlock / 4;  // 512
constexpr int kRingSlot = 2 * 32 * 16;    // one k-block of one warp: 2 row halves x 32 lanes x 16 B
constexpr int kRingDepth = 8;             // k-blocks of codes in flight per warp
// k-blocks requested before the preceding grid has finished (weight prefetch):
// enough to cover the hand-off, few enough that the activation loads issued
// right after it do not queue behind a whole ring of weight traffic.
constexpr int kPreWait = 3;

// Shared memory of one CTA.  Offsets in bytes from the 128-aligned base.
struct Layout {
  int ring;    // per-warp code rings [8][depth][2][32][16 B]; reused for the partials
  int xs;      // activations [M][kbps * 128] 16-bit, 16-byte chunks swizzled, then one zero k-block
  int asum;    // per (k-block, token slot): block sum and code-offset term, [kbps][2][8] fp32
  int ssc;     // scales [gseg][128] fp16
  int sdl;     // delta [gseg][128] fp32
  int red;     // split-K partials from every rank [splits][rpr][8] fp32
  int bars;    // sd_full, red_full mbarriers, abort flag
  int bytes;   // total (with 128 bytes of alignment slack)
};

__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }

// Weight rows of a column tile whose split-K reduction rank r owns: rows
// [r * rpr, (r + 1) * rpr).  A gate/up pair rounds rpr up to 16 rows so that the
// gate row and its up row 8 rows further on always fall to the same owner.
__host__ __device__ inline int reduce_rows(int splits, bool pair) {
  const int rpr = (kTileN + splits - 1) / splits;
  return pair ? (rpr + 15) & ~15 : rpr;
}

__host__ __device__ inline Layout layout(int M, int kbps, int splits, int gseg, bool has_delta, int depth,
                                         bool pair) {
  Layout L;
  const int rpr = reduce_rows(splits, pair);
  int off = 0;
  L.ring = off;
  off = align128(off + kWarps * depth * kRingSlot);  // >= the partials [128][8] fp32
  L.xs = off;
  off = align128(off + (M * kbps + 1) * kKBlock * 2);
  L.asum = off;
  off = align128(off + kbps * 2 * kMT * 4);
  L.ssc = off;
  off = align128(off + gseg * kTileN * 2);
  L.sdl = off;
  if (has_delta) off = align128(off + gseg * kTileN * 4);
  L.red = off;
  if (splits > 1) off = align128(off + splits * rpr * kMT * 4);
  L.bars = off;
  off = align128(off + 32);
  L.bytes = off + 128;
  return L;
}
}  // namespace gv

// The per-lane copies, offset-code operands, MMA, block sums and activation
// swizzle of this path are in wq_warp.cuh.
using namespace warp;

// Eight int8 activations (one 8-byte load) as the 16-byte chunk of their fp16
// values, element e in half e of the chunk (|x| <= 128: exact).
__device__ __forceinline__ uint4 i8x8_to_f16x8(uint2 w) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t word = (i < 2) ? w.x : w.y;
    const int sh = 16 * (i & 1);
    const __half2 h = __halves2half2(__short2half_rn(static_cast<short>(static_cast<int8_t>(word >> sh))),
                                     __short2half_rn(static_cast<short>(static_cast<int8_t>(word >> (sh + 8)))));
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// MINB: CTAs per SM the registers are budgeted for -- 2 for a plain GEMM (one
// wave of two CTAs per SM), 3 for a grouped launch, whose many short CTAs (one
// per column tile and expert) then fit in one wave.
template <int XK, int D, int MINB, bool PAIR, bool XS>
__global__ void __launch_bounds__(gv::kThreads, MINB) gemv_kernel(const GemmParams p, unsigned* status) {
  using namespace gv;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* const sm = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int tile = blockIdx.x;
  const int n0 = tile * kTileN;
  const int seg = blockIdx.y;  // == rank in the cluster (cluster dims 1 x splits x 1)
  const int splits = p.splits;
  const int kbps = p.kb_per_split;
  const int kb0 = seg * kbps;
  const int nkb = min(p.kb_total, kb0 + kbps) - kb0;
  const bool has_delta = p.delta != nullptr;
  const int N = p.N;
  // This CTA's problem: the whole GEMM, or (grouped launch) expert blockIdx.z's
  // token rows and weights.  An expert without tokens has nothing to do.
  int M = p.M;
  const uint8_t* Xp = static_cast<const uint8_t*>(p.X);
  const float* Xsp = p.x_scale;  // XS: X holds int8 rows (W4A8), this their per-token scales
  uint8_t* Yp = static_cast<uint8_t*>(p.Y);
  const uint32_t* Bp = p.B;
  const __half* Sp = p.S;
  const float* Dp = p.delta;
  if (p.experts > 0) {
    const int e = blockIdx.z;
    const int r0 = p.goff[e];
    M = p.goff[e + 1] - r0;
    if (M <= 0) return;
    Xp += static_cast<size_t>(r0) * p.K * (XS ? 1 : 2);
    if (XS) Xsp += r0;
    Yp += static_cast<size_t>(r0) * N * (p.y_kind == kYF32 ? 4 : 2);
    Bp += e * p.b_stride;
    Sp += e * p.sd_stride;
    if (has_delta) Dp += e * p.sd_stride;
  }
  const bool per_channel = p.G == 1;  // one group spans the whole K
  const int g0 = per_channel ? 0 : kb0;
  const int gseg = per_channel ? 1 : nkb;
  const Layout L = layout(M, kbps, splits, per_channel ? 1 : kbps, has_delta, D, PAIR);
  constexpr bool pair = PAIR;  // gate/up pair weight, SwiGLU epilogue
  const int rpr = reduce_rows(splits, pair);
  const int own_rows = max(0, min(kTileN - seg * rpr, rpr));

  uint8_t* const xs = sm + L.xs;
  float* const asum = reinterpret_cast<float*>(sm + L.asum);
  const __half* const ssc = reinterpret_cast<const __half*>(sm + L.ssc);
  const float* const sdl = reinterpret_cast<const float*>(sm + L.sdl);
  const uint32_t sd_full = base + L.bars;
  const uint32_t red_full = base + L.bars + 8;
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sm + L.bars + 16);
  const int xstride = kbps * kKBlock * 2;  // bytes per token row of the tile

  const uint32_t sd_bytes = static_cast<uint32_t>(gseg * kTileN * (has_delta ? 6 : 2));
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(sd_full, 1);
    mbar_init(red_full, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && splits > 1)
    mbar_arrive_expect_tx(red_full, static_cast<uint32_t>(own_rows * splits * kMT * 4));
  if (splits > 1) cluster_arrive_relaxed();  // barriers initialized and armed (waited before any copy)

  // Scale and delta rows of the segment's groups: one bulk copy per row.  Like
  // the codes, they are only ever written by the pack, so with weight prefetch
  // they are requested before the preceding grid has finished.
  const uint64_t pol_stream = l2_evict_first();
  // The lanes of warp 0 issue the copies side by side (one group row each), so
  // no thread is held up issuing them one after the other.
  auto issue_sd = [&]() {
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(sd_full, sd_bytes);
      __syncwarp();
      for (int r = lane; r < gseg; r += 32) {
        const size_t src = static_cast<size_t>(g0 + r) * N + n0;
        bulk_load_hint(base + L.ssc + r * kTileN * 2, Sp + src, kTileN * 2, sd_full, pol_stream);
        if (has_delta) bulk_load_hint(base + L.sdl + r * kTileN * 4, Dp + src, kTileN * 4, sd_full, pol_stream);
      }
    }
  };

  // Codes: rows rA = 16 warp + g and rB = rA + 8 of the tile, logical chunk t
  // (stored at slot t ^ ((r / 2) % 4); both rows share the slot).
  const int rA = 16 * warp + g;
  const int rB = rA + 8;
  const uint4* const blk0 =
      reinterpret_cast<const uint4*>(Bp) + (static_cast<size_t>(tile) * p.kb_total + kb0) * kUint4PerBlock;
  const int offA = rA * 4 + (t ^ ((g >> 1) & 3));
  const int offB = offA + 32;
  // Ring of this warp: slot d holds k-block (d mod D) as [row half][lane][16 B];
  // each lane copies and later reads only its own two chunks, so the copies
  // need no barrier: the lane's own wait_group orders them.
  const uint32_t ring = base + L.ring + static_cast<uint32_t>(warp * D * kRingSlot + lane * 16);
  auto issue_kb = [&](int kb, int slot) {
    const uint4* src = blk0 + static_cast<size_t>(kb) * kUint4PerBlock;
    cp_async16(ring + slot * kRingSlot, src + offA, pol_stream);
    cp_async16(ring + slot * kRingSlot + 512, src + offB, pol_stream);
  };
  // One copy group per ring slot d in [d0, d1) (empty past the segment).
  auto issue_codes = [&](int d0, int d1) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (d >= d0 && d < d1) {
        if (d < nkb) issue_kb(d, d);
        cp_async_commit();
      }
    }
  };
  constexpr int kPre = kPreWait < D ? kPreWait : D;
  if (p.weight_prefetch) {
    issue_sd();
    issue_codes(0, kPre);
  }
  griddep_launch_dependents();
  griddep_wait();  // X written by the preceding grid is visible from here on

  // ---- stage the activation rows of the segment and their 128-k block sums;
  // token slots past M read a zero k-block instead.  The activation loads go
  // out first, the rest of the code ring right behind them.
  {
    const int per_tok = nkb * 16;  // 16-byte chunks per token row of the segment
    const int total = M * per_tok;
    if (threadIdx.x < 16)
      *reinterpret_cast<uint4*>(xs + M * xstride + 16 * threadIdx.x) = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < kbps * 2 * kMT; i += kThreads)
      if (i % kMT >= M) asum[i] = 0.0f;
    const uint8_t* const xg = Xp;
    constexpr int kU = 8;  // one round trip for up to 16 k-blocks x 8 tokens x 16 chunks
    for (int b = 0; b < total; b += kThreads * kU) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = b + u * kThreads + threadIdx.x;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (idx < total) {
          const int m = idx / per_tok;
          const int rem = idx - m * per_tok;
          if constexpr (XS) {
            v[u] = i8x8_to_f16x8(
                *reinterpret_cast<const uint2*>(xg + static_cast<size_t>(m) * p.K + kb0 * kKBlock + rem * 8));
          } else {
            v[u] = *reinterpret_cast<const uint4*>(xg + (static_cast<size_t>(m) * p.K + kb0 * kKBlock) * 2 + rem * 16);
          }
        }
      }
      if (b == 0) {
        if (!p.weight_prefetch) {
          issue_sd();
          issue_codes(0, kPre);
        }
        issue_codes(kPre, D);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx0 = b + u * kThreads;
        if (idx0 >= total) break;  // uniform
        const int idx = idx0 + threadIdx.x;
        float lo = 0.0f, hi = 0.0f;
        int m = 0, rem = 0;
        if (idx < total) {
          m = idx / per_tok;
          rem = idx - m * per_tok;
          *reinterpret_cast<uint4*>(xs + m * xstride + 16 * xswz(rem, m)) = v[u];
          sum_chunk<XK>(v[u], lo, hi);
        }
        // the 16 chunks of one (token, k-block) are 16 consecutive lanes
#pragma unroll
        for (int sh = 1; sh < 16; sh <<= 1) {
          lo += __shfl_xor_sync(0xffffffffu, lo, sh);
          hi += __shfl_xor_sync(0xffffffffu, hi, sh);
        }
        if (idx < total && (rem & 15) == 0) {
          // block sum, and the offset the MMA's codes carry: fp16 codes are
          // 1024 + v (lo k) or (1024 + 16 v) / 16 = 64 + v (hi k), so
          // sum (v - 8) x = D - 1032 lo - 72 hi; bf16 codes are 128 + v
          const int kb = rem >> 4;
          asum[kb * 2 * kMT + m] = lo + hi;
          asum[kb * 2 * kMT + kMT + m] = (XK == kXF16) ? fmaf(1032.0f, lo, 72.0f * hi) : 136.0f * (lo + hi);
        }
      }
    }
  }
  __syncthreads();
  {
    const WaitCtx wsd{abort_flag, p.timeout_ns, kDevTimeoutProducer, status};
    mbar_wait(sd_full, 0, wsd);
  }

  // ---- main loop: per k-block 8 MMA steps in two chains, then the promotion
  float tot[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const int sw = (t >> 1) | ((g & 1) << 1);  // xswz for this lane's chunks 4t + q: flips the low bits of q
  // token slot g: its row of the tile, or the zero k-block (not advanced) past M
  const uint8_t* const xrow = xs + (g < M ? g * xstride : M * xstride) + 64 * t;
  const int xstep = g < M ? kKBlock * 2 : 0;
  int slot = 0;
  for (int i = 0; i < nkb; ++i) {
    cp_async_wait<D - 1>();  // k-block i (group i) has landed
    const uint4 a = lds128(ring + slot * kRingSlot);
    const uint4 c = lds128(ring + slot * kRingSlot + 512);
    uint32_t xr[16];
    const uint8_t* const row = xrow + i * xstep;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * (q ^ sw));
      xr[4 * q] = v.x;
      xr[4 * q + 1] = v.y;
      xr[4 * q + 2] = v.z;
      xr[4 * q + 3] = v.w;
    }
    // Each step's fragments: pair p of words 4t + 2h (k 2t, 2t+1) and
    // 4t + 2h + 1 (k 2t+8, 2t+9), rows g and g + 8, as offset codes.  fp16:
    // steps with p even (low nibbles, 1024 + v) and p odd (high nibbles,
    // 1024 + 16 v) accumulate into separate chains; bf16: chains by h.
    const uint32_t wa[2][2] = {{a.x, a.y}, {a.z, a.w}};  // [h][fragment k half], row g
    const uint32_t wc[2][2] = {{c.x, c.y}, {c.z, c.w}};  // row g + 8
    // The ring slot has been read (the code words are in registers): refill it
    // with k-block i + D.
    asm volatile("" ::"r"(wa[0][0]), "r"(wa[1][1]), "r"(wc[0][0]), "r"(wc[1][1]) : "memory");
    if (i + D < nkb) issue_kb(i + D, slot);
    cp_async_commit();
    slot = (slot + 1 == D) ? 0 : slot + 1;
    float acc[2][4];
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      // issue order alternates the two chains: fp16 chains by p, so h outer;
      // bf16 chains by h, so p outer
      const int h = (XK == kXBF16) ? (st & 1) : (st >> 2);
      const int pp = (XK == kXBF16) ? (st >> 1) : (st & 3);
      {
        uint32_t f[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = (j & 1) ? wc[h][j >> 1] : wa[h][j >> 1];  // f0 row g, f1 row g+8, f2, f3 the k+8 half
          if (XK == kXBF16) f[j] = off_bf16(w >> (4 * pp));
          else f[j] = (pp & 1) ? off_hi_f16(pp >= 2 ? w >> 8 : w) : off_lo_f16(pp >= 2 ? w >> 8 : w);
        }
        const int ch = (XK == kXBF16) ? h : (pp & 1);
        const bool first = (XK == kXBF16) ? (pp == 0) : (h == 0 && pp < 2);
        if (first) mma16816<XK>(acc[ch], zero4, f[0], f[1], f[2], f[3], xr[8 * h + pp], xr[8 * h + 4 + pp]);
        else mma16816<XK>(acc[ch], acc[ch], f[0], f[1], f[2], f[3], xr[8 * h + pp], xr[8 * h + 4 + pp]);
      }
    }
    const int gl = per_channel ? 0 : i;
    const float sA = __half2float(ssc[gl * kTileN + rA]);
    const float sB = __half2float(ssc[gl * kTileN + rB]);
    // sum_k (v - 8) x for the block: the offset codes' product minus the offset term
    const float2 ofs = *reinterpret_cast<const float2*>(asum + i * 2 * kMT + kMT + 2 * t);
    float d[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float o = (e & 1) ? ofs.y : ofs.x;
      d[e] = (XK == kXBF16 ? acc[0][e] + acc[1][e] : fmaf(acc[1][e], 0.0625f, acc[0][e])) - o;
    }
    if (has_delta) {
      const float dA = sdl[gl * kTileN + rA];
      const float dB = sdl[gl * kTileN + rB];
      const float2 as = *reinterpret_cast<const float2*>(asum + i * 2 * kMT + 2 * t);
      tot[0] = fmaf(dA, as.x, fmaf(sA, d[0], tot[0]));
      tot[1] = fmaf(dA, as.y, fmaf(sA, d[1], tot[1]));
      tot[2] = fmaf(dB, as.x, fmaf(sB, d[2], tot[2]));
      tot[3] = fmaf(dB, as.y, fmaf(sB, d[3], tot[3]));
    } else {
      tot[0] = fmaf(sA, d[0], tot[0]);
      tot[1] = fmaf(sA, d[1], tot[1]);
      tot[2] = fmaf(sB, d[2], tot[2]);
      tot[3] = fmaf(sB, d[3], tot[3]);
    }
  }
  cp_async_wait<0>();  // nothing of this thread is in flight (the trailing groups are empty)

  // ---- split-K reduction + store
  __syncthreads();  // every warp is done with its ring and the activation tile
  const bool aborted = *abort_flag != 0;
  if (aborted) {
    if (threadIdx.x == 0) {
      // let the scale / delta copies land before the shared memory is reused or the CTA exits
      volatile int never = 0;
      const WaitCtx drain{&never, 50000000ull, kDevTimeoutProducer, status};
      mbar_wait(sd_full, 0, drain);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) tot[e] = __int_as_float(0x7fc00000);
    __syncthreads();
  }
  if (splits == 1) {
    if constexpr (pair) {
      // row rA is a gate column and rB = rA + 8 the up column of the same output
      const int j = ((n0 + 16 * warp) >> 1) + g;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = 2 * t + e;
        if (tok < M) store_y_any(Yp, p.y_kind, static_cast<size_t>(tok) * (N >> 1) + j, silu_mul(tot[e], tot[2 + e]));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = 2 * t + (e & 1);
        const int row = (e < 2) ? rA : rB;
        if (tok < M)
          store_y_any(Yp, p.y_kind, static_cast<size_t>(tok) * N + n0 + row, XS ? tot[e] * Xsp[tok] : tot[e]);
      }
    }
    return;
  }
  // Partials, row-major [128 rows][8 tokens], in the ring area: the rows rank o
  // owns are one contiguous block.
  float* const part = reinterpret_cast<float*>(sm + L.ring);
  *reinterpret_cast<float2*>(part + rA * kMT + 2 * t) = make_float2(tot[0], tot[1]);
  *reinterpret_cast<float2*>(part + rB * kMT + 2 * t) = make_float2(tot[2], tot[3]);
  fence_proxy_async_smem();  // the generic writes become visible to the bulk copies
  __syncthreads();
  cluster_wait();  // every rank's barriers are initialized and armed
  if (warp == 0) {
    if (lane < splits) {
      const int o = lane;
      const int rows_o = min(kTileN - o * rpr, rpr);
      if (rows_o > 0) {
        bulk_copy_to_peer(mapa_shared(base + L.red + static_cast<uint32_t>(seg * rpr * kMT * 4), o),
                          base + L.ring + static_cast<uint32_t>(o * rpr * kMT * 4),
                          static_cast<uint32_t>(rows_o * kMT * 4), mapa_shared(red_full, o));
      }
      bulk_commit_group();
      bulk_wait_group_read0();  // the partials stay valid until the copies have read them
    }
  }
  const float* const red = reinterpret_cast<const float*>(sm + L.red);
  const int total = own_rows * M;
  if (static_cast<int>(threadIdx.x) < total) {
    volatile int never = 0;
    const WaitCtx wred{&never, p.timeout_ns, kDevTimeoutFixup, status};
    mbar_wait(red_full, 0, wred);
  }
  if constexpr (pair) {
    // own_rows is a multiple of 16: pairs (16 * (i / 8) + i % 8, that row + 8)
    const int npair = own_rows >> 1;
    for (int i = threadIdx.x; i < npair * M; i += kThreads) {
      const int m = i / npair;
      const int pi = i - m * npair;
      const int lr = 16 * (pi >> 3) + (pi & 7);
      float gs = 0.0f, us = 0.0f;
      for (int src = 0; src < splits; ++src) {
        gs += red[(src * rpr + lr) * kMT + m];
        us += red[(src * rpr + lr + 8) * kMT + m];
      }
      store_y_any(Yp, p.y_kind, static_cast<size_t>(m) * (N >> 1) + ((n0 + seg * rpr) >> 1) + pi, silu_mul(gs, us));
    }
  } else {
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int m = i / own_rows;
      const int lr = i - m * own_rows;
      float sum = 0.0f;
      for (int src = 0; src < splits; ++src) sum += red[(src * rpr + lr) * kMT + m];
      store_y_any(Yp, p.y_kind, static_cast<size_t>(m) * N + n0 + seg * rpr + lr, XS ? sum * Xsp[m] : sum);
    }
  }
}

// Split of K over a thread-block cluster for the weight-streaming path: the
// most K segments (at most 8, the portable cluster size) that still give one
// wave of two CTAs per SM, so that every SM streams with 16 warps.  Returns 0
// when the problem is not for this path (M > 8) or no split fits the shared
// memory limit.
int gemv_plan(int M, int N, int K, int group_size, bool has_delta, int* splits_out, int* kbps_out, bool pair) {
  if (M < 1 || M > gv::kMaxM) return 0;
  const int kb = K / kKBlock;
  const int tiles = N / kTileN;
  int best = -1;
  for (int s = 1; s <= gv::kMaxSplits && s <= kb; ++s) {
    const int kbps = (kb + s - 1) / s;
    const int sp = (kb + kbps - 1) / kbps;
    const int gseg = (group_size == K) ? 1 : kbps;
    if (gv::layout(M, kbps, sp, gseg, has_delta, gv::kRingDepth, pair).bytes > gv::kMaxSmem) continue;
    if (best < 0 || tiles * sp <= 2 * kNumSMs) best = sp;
  }
  if (best < 0) return 0;
  *splits_out = best;
  *kbps_out = (kb + best - 1) / best;
  return 1;
}

// Whether a launch with these segments fits the shared memory limit.
bool gemv_plan_fits(int M, int kbps, int splits, bool per_channel, bool has_delta, bool pair) {
  return M >= 1 && M <= gv::kMaxM &&
         gv::layout(M, kbps, splits, per_channel ? 1 : kbps, has_delta, gv::kRingDepth, pair).bytes <= gv::kMaxSmem;
}

template <int XK, int D, int MINB, bool PAIR, bool XS = false>
static cudaError_t launch_gemv_t(const GemmParams& p, unsigned* status, cudaStream_t st) {
  static PerContextOnce attr_set;  // redone after a context rebuild
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_set.needed(dev)) {
    e = cudaFuncSetAttribute(gemv_kernel<XK, D, MINB, PAIR, XS>, cudaFuncAttributeMaxDynamicSharedMemorySize, gv::kMaxSmem);
    if (e != cudaSuccess) return e;
    attr_set.done(dev);
  }
  const int gseg = (p.G == 1) ? 1 : p.kb_per_split;
  const gv::Layout L = gv::layout(p.M, p.kb_per_split, p.splits, gseg, p.delta != nullptr, D, PAIR);
  if (L.bytes > gv::kMaxSmem) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.N / kTileN, p.splits, p.experts > 0 ? p.experts : 1);
  cfg.blockDim = dim3(gv::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L.bytes;
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
  return cudaLaunchKernelEx(&cfg, gemv_kernel<XK, D, MINB, PAIR, XS>, p, status);
}

cudaError_t launch_gemv(int x_kind, const GemmParams& p, cudaStream_t stream) {
  unsigned* status = status_word();
  if (!status) return cudaErrorInvalidSymbol;
  if (p.splits < 1 || p.splits > gv::kMaxSplits || p.M < 1 || p.M > gv::kMaxM || (p.x_scale && p.swiglu) || !p.X ||
      p.experts < 0 || p.experts > kMaxExperts ||
      p.kb_per_split < 1 || (p.splits - 1) * p.kb_per_split >= p.kb_total)
    return cudaErrorInvalidValue;
  if (p.x_scale) {  // W4A8 rows as fp16
    if (x_kind != kXF16) return cudaErrorInvalidValue;
    if (p.experts > 0) return launch_gemv_t<kXF16, gv::kRingDepth, 3, false, true>(p, status, stream);
    return launch_gemv_t<kXF16, gv::kRingDepth, 2, false, true>(p, status, stream);
  }
  if (p.experts > 0) {
    if (p.swiglu) return cudaErrorInvalidValue;
    if (x_kind == kXBF16) return launch_gemv_t<kXBF16, gv::kRingDepth, 3, false>(p, status, stream);
    return launch_gemv_t<kXF16, gv::kRingDepth, 3, false>(p, status, stream);
  }
  if (p.swiglu) {
    if (x_kind == kXBF16) return launch_gemv_t<kXBF16, gv::kRingDepth, 2, true>(p, status, stream);
    return launch_gemv_t<kXF16, gv::kRingDepth, 2, true>(p, status, stream);
  }
  if (x_kind == kXBF16) return launch_gemv_t<kXBF16, gv::kRingDepth, 2, false>(p, status, stream);
  return launch_gemv_t<kXF16, gv::kRingDepth, 2, false>(p, status, stream);
}

}  // namespace wq
