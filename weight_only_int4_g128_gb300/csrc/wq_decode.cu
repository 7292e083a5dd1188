// wq_decode.cu -- the decode path (M <= 16 tokens) of the W4A16 / W4A8 GEMM,
// where the op is bound by reading the 4-bit weights from HBM.
//
// Swap-AB as in the large-M kernel: 128 weight rows per CTA are the MMA's
// M = 128 TMEM lanes, the tokens are the MMA's N.  What differs is the operand
// type: the tensor cores run kind::f8f6f4 (e4m3 x e4m3, fp32 accumulate), which
// takes K = 32 per instruction, so a 128-k block costs 4 MMAs instead of 8.
//
//  * Weights.  The e4m3 byte whose bit pattern is the 4-bit code v (0..15) has
//    the value v * 2^-9 exactly (v < 8: subnormals m * 2^-9; v >= 8: exponent
//    field 1, (8 + m) * 2^-9).  Dequantizing is therefore only moving nibbles
//    into bytes (two byte permutes per 8 codes); scale and zero are applied in
//    fp32 after each 128-k block.
//  * Activations.  A pre-pass splits every 128-k block of every activation row
//    into three e4m3 components with a power-of-two scale sigma of its own:
//    x / sigma = c1 + c2/16 + c3/256 up to 2^-12 relative (about one bit finer
//    than fp16), and stores the block's fp32 sum of x and the factor
//    f = sigma * 2^9.  The 48 = 3 x 16 component rows are the MMA's N.
//  * Per 128-k block (group g) the kernel has D[n][3m+c] = sum_k v[k][n] *
//    c_c[m][k] * 2^-9 in TMEM, and the promotion warps accumulate in fp32
//        acc[n][m] += s[g][n] * f[m] * (D1 + D2/16 + D3/256) + zero[g][n] * asum[m]
//    with zero = delta - 8 s ("Marlin INT4 on Ada -- how it works", section "The
//    core mismatch": C = C_sym + A_group_sum @ delta, W_sym = (q - 8) * scale,
//    rewritten as s * sum v x + (delta - 8 s) * sum x).  For W4A8 the per-token
//    activation scale is folded into f and asum by the pre-pass.
//
//   warp 0      TMA producer: per pair of 128-k blocks the packed weight tiles
//               (one 16 KB bulk copy: the blocked layout keeps a tile's k-blocks
//               contiguous, and copies this large stream about twice as fast as
//               8 KB ones) and the activation components (one 3-D box of 2 x 56
//               rows x 128 B: 48 component rows + one row carrying the block's
//               sums and factors, padded); per 8 groups the scale and delta rows
//   warp 1      TMEM owner; lane 0 issues the MMAs (A from TMEM, B from shared)
//   warps 2..5  dequant: each thread one weight row, 16 words -> 32 e4m3 words
//               -> TMEM A-stage (one tcgen05.st of 32 columns)
//   warps 6..9  promotion (tcgen05.ld of the block's D, fp32 FMAs) and epilogue
// Split-K: the K segments of one column tile form a thread-block cluster
// (gridDim.y = cluster size <= 8).  Each CTA stages its fp32 partials in its
// own shared memory and sends each rank the rows that rank owns with one bulk
// copy, which completes on the owner's mbarrier; an owner waits only for its
// own rows, adds the partials in rank order and writes Y.
#include <cuda_fp8.h>

#include "wq_device.cuh"

namespace wq {

namespace dec {
constexpr int kNSX = 6;                   // shared-memory stages (one 128-k block each)
constexpr int kNSA = 3;                   // TMEM A-stages
constexpr int kNB = 3;                    // TMEM D buffers
constexpr int kMT = 16;                   // tokens per tile
constexpr int kComp = 3;                  // e4m3 components per activation
constexpr int kBN = kComp * kMT;          // MMA N = 48
constexpr int kBRows = 56;                // + the sums/factors row (48), padded to 7 KB
constexpr int kBStage = kBRows * 128;     // 7 KB, 1024-aligned
constexpr int kPair = 2;                  // k-blocks per load group (one copy each of W and B)
constexpr int kNG = 3;                    // load groups in the ring
constexpr int kWStage = kTileN * kWordsPerKBlock * 4;  // 8 KB
constexpr int kChunk = 8;                 // groups per scale/delta chunk (index math uses >> 3)
constexpr int kSChunk = kChunk * kTileN * 2;
constexpr int kDChunk = kChunk * kTileN * 4;
constexpr int kChunkSlots = 2;
constexpr int kACol = 32;                 // TMEM columns of one A-stage (128 e4m3 per lane)
constexpr int kDCol0 = kNSA * kACol;      // first D column
constexpr int kTmemCols = 256;
constexpr int kThreads = 320;             // 10 warps
constexpr int kMaxSplits = 8;             // portable cluster size
constexpr int kRedBytes = 8704;           // >= splits * ceil(128 / splits) * 16 * 4 for splits <= 8
constexpr int kNumBars = kNG + 2 * kNSX + kNSA + 2 * kChunkSlots + 2;
constexpr int kSmemBytes = 1024 + kNSX * (kBStage + kWStage) + kChunkSlots * (kSChunk + kDChunk) +
                           kRedBytes + kNumBars * 8 + 16;
static_assert(kBStage % 1024 == 0 && kBN < kBRows, "B stage");
static_assert(kNG * kPair == kNSX, "ring = load groups x pair");
static_assert(kDCol0 + kNB * kBN <= kTmemCols, "TMEM budget");
static_assert(kNSA < kNSX && kNB < kNSX, "barrier phase distances");
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");

constexpr int red_bytes(int splits) { return splits * ((kTileN + splits - 1) / splits) * kMT * 4; }
static_assert(red_bytes(2) <= kRedBytes && red_bytes(3) <= kRedBytes && red_bytes(4) <= kRedBytes &&
                  red_bytes(5) <= kRedBytes && red_bytes(6) <= kRedBytes && red_bytes(7) <= kRedBytes &&
                  red_bytes(8) <= kRedBytes,
              "reduction buffer");

// Instruction descriptor for kind::f8f6f4 with e4m3 A and B (format code 0),
// fp32 accumulator, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
}  // namespace dec

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f8f6f4.
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// Pre-pass: one warp per (token row m < 16, 128-k block kb); lane l holds
// k = 128 kb + 4 l .. + 3.
//   X8 rows 3 m + c (c = 0, 1, 2), bytes [128 kb, 128 kb + 128): e4m3
//       components of x[m][k] / sigma, sigma = 2^(e - 8) with max |x| < 2^e
//       (token-major, so that M tokens occupy the first 3 M rows)
//   X8 row 48, bytes [128 kb, 128 kb + 128): fp32 asum[16] = xs[m] * sum x,
//       then fp32 f[16] = xs[m] * sigma * 2^9 (xs = W4A8 token scale, else 1;
//       f = NaN when the block holds inf or NaN)
// Rows m >= M are written as zeros.
// ---------------------------------------------------------------------------
template <int XK>
__device__ __forceinline__ void load4(const void* X, size_t idx, float (&v)[4]) {
  if (XK == kXI8) {
    const char4 c = *reinterpret_cast<const char4*>(static_cast<const int8_t*>(X) + idx);
    v[0] = c.x; v[1] = c.y; v[2] = c.z; v[3] = c.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(X) + idx);
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (XK == kXF16) {
        v[2 * i] = __half2float(__ushort_as_half(static_cast<uint16_t>(w[i] & 0xFFFFu)));
        v[2 * i + 1] = __half2float(__ushort_as_half(static_cast<uint16_t>(w[i] >> 16)));
      } else {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }
}

__device__ __forceinline__ uint32_t e4m3_rn(float x) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

// One (128-k block, token) of the activation operand: this lane's 4 values v
// (k = 128 kb + 4 lane .. + 3) become three exact e4m3 components under a
// power-of-two block factor; lane 0 stores the block's sum and factor, both
// times the token's scale xs.
__device__ __forceinline__ void prep_block(const float (&v)[4], int m, int kb, int K, float xs, uint8_t* X8) {
  const int lane = threadIdx.x & 31;
  const size_t o = static_cast<size_t>(kb) * kKBlock + lane * 4;
  uint32_t* const r1 = reinterpret_cast<uint32_t*>(X8 + static_cast<size_t>(3 * m) * K + o);
  uint32_t* const r2 = reinterpret_cast<uint32_t*>(X8 + static_cast<size_t>(3 * m + 1) * K + o);
  uint32_t* const r3 = reinterpret_cast<uint32_t*>(X8 + static_cast<size_t>(3 * m + 2) * K + o);
  float* const srow = reinterpret_cast<float*>(X8 + static_cast<size_t>(dec::kBN) * K + static_cast<size_t>(kb) * kKBlock);
  float amax = 0.0f;
  int bad = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = fabsf(v[i]);
    bad |= !(a <= 3.402823466e38f);
    amax = fmaxf(amax, a);
  }
  float sum = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
    bad |= __shfl_xor_sync(0xffffffffu, bad, sh);
    sum += __shfl_xor_sync(0xffffffffu, sum, sh);
  }
  // sigma = 2^(e - 8) with amax < 2^e, so |x| / sigma < 256 (e4m3 saturates at 448)
  float inv = 1.0f, f = 512.0f;
  if (!bad && amax > 0.0f) {
    int e = 0;
    frexpf(amax, &e);
    inv = ldexpf(1.0f, 8 - e);
    f = ldexpf(1.0f, e + 1);  // sigma * 2^9
  }
  uint32_t b1 = 0, b2 = 0, b3 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x = v[i] * inv;  // exact: power-of-two scale
    const uint32_t c1 = e4m3_rn(x);
    const float t1 = (x - e4m3_to_f32(c1)) * 16.0f;  // exact residual
    const uint32_t c2 = e4m3_rn(t1);
    const float t2 = (t1 - e4m3_to_f32(c2)) * 16.0f;
    const uint32_t c3 = e4m3_rn(t2);
    b1 |= c1 << (8 * i);
    b2 |= c2 << (8 * i);
    b3 |= c3 << (8 * i);
  }
  *r1 = b1;
  *r2 = b2;
  *r3 = b3;
  if (lane == 0) {
    srow[m] = sum * xs;
    srow[dec::kMT + m] = bad ? __int_as_float(0x7fc00000) : f * xs;
  }
}

// Token slots past M: zero components, sum and factor.
__device__ __forceinline__ void prep_block_zero(int m, int kb, int K, uint8_t* X8) {
  const int lane = threadIdx.x & 31;
  const size_t o = static_cast<size_t>(kb) * kKBlock + lane * 4;
#pragma unroll
  for (int c = 0; c < 3; ++c) *reinterpret_cast<uint32_t*>(X8 + static_cast<size_t>(3 * m + c) * K + o) = 0u;
  if (lane == 0) {
    float* const srow = reinterpret_cast<float*>(X8 + static_cast<size_t>(dec::kBN) * K + static_cast<size_t>(kb) * kKBlock);
    srow[m] = 0.0f;
    srow[dec::kMT + m] = 0.0f;
  }
}

template <int XK>
__global__ void __launch_bounds__(256) decode_prep_kernel(const void* X, int M, int K, const float* x_scale,
                                                          uint8_t* X8) {
  const int nkb = K / kKBlock;
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);  // (kb, m) pair, m fastest
  const int lane = threadIdx.x & 31;
  const int m = wid & (dec::kMT - 1);
  const int kb = wid >> 4;
  // The decode kernel that follows may be scheduled at once: it waits for this
  // grid to complete before it reads X8.  X may be written by the preceding
  // grid, and X8 may still be read by it, so nothing is touched before the wait.
  griddep_launch_dependents();
  griddep_wait();
  if (kb >= nkb) return;
  if (m >= M) {
    prep_block_zero(m, kb, K, X8);
    return;
  }
  float v[4];
  load4<XK>(X, static_cast<size_t>(m) * K + static_cast<size_t>(kb) * kKBlock + lane * 4, v);
  prep_block(v, m, kb, K, x_scale ? x_scale[m] : 1.0f, X8);
}

// Per-token int8 quantization of fp16 rows (HyperQwen W4A8 article, "why
// W4A8": activations quantized per token; absmax / 127, round half to even,
// clamp to [-127, 127]) fused with the activation operand above: one CTA per
// token slot computes the row's absmax, writes x_scale[m], and turns the codes
// of every k-block into e4m3 components.  The codes and scale are the ones
// quantize_per_token_kernel produces; they are never written out.
__device__ __forceinline__ float quant_code(float x, float xs) {
  if (!(xs > 0.0f)) return 0.0f;
  return fminf(fmaxf(rintf(__fdiv_rn(x, xs)), -127.0f), 127.0f);
}

__device__ __forceinline__ float row_absmax_f16(const __half* row, int K, float* red) {
  float amax = 0.0f;
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + k);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(__half2float(__ushort_as_half(static_cast<uint16_t>(w[i] & 0xFFFFu)))));
      amax = fmaxf(amax, fabsf(__half2float(__ushort_as_half(static_cast<uint16_t>(w[i] >> 16)))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  float v = 0.0f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) v = fmaxf(v, red[i]);
  return v;
}

__global__ void __launch_bounds__(256) decode_prep_quant_kernel(const __half* X, int M, int K, float* x_scale,
                                                                uint8_t* X8) {
  __shared__ float red[8];
  const int m = blockIdx.x;  // token slot of the tile
  const int nkb = K / kKBlock;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();
  griddep_wait();  // as decode_prep_kernel
  if (m >= M) {
    for (int kb = warp; kb < nkb; kb += 8) prep_block_zero(m, kb, K, X8);
    return;
  }
  const __half* const row = X + static_cast<size_t>(m) * K;
  const float xs = __fdiv_rn(row_absmax_f16(row, K, red), 127.0f);
  if (threadIdx.x == 0) x_scale[m] = xs;
  for (int kb = warp; kb < nkb; kb += 8) {
    float v[4];
    load4<kXF16>(row, static_cast<size_t>(kb) * kKBlock + lane * 4, v);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = quant_code(v[i], xs);
    prep_block(v, m, kb, K, xs, X8);
  }
}

// The same quantization for the large-M path: one CTA per row writes the codes
// as fp16 (exact) for the fp16 tensor-core GEMM, and x_scale[m].
__global__ void __launch_bounds__(256) quant_f16_kernel(const __half* X, int K, __half* X16, float* x_scale) {
  __shared__ float red[8];
  const int m = blockIdx.x;
  griddep_launch_dependents();
  griddep_wait();  // X may be written by the preceding grid, X16 read by it
  const __half* const row = X + static_cast<size_t>(m) * K;
  const float xs = __fdiv_rn(row_absmax_f16(row, K, red), 127.0f);
  if (threadIdx.x == 0) x_scale[m] = xs;
  __half* const out = X16 + static_cast<size_t>(m) * K;
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + k);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = quant_code(__half2float(__ushort_as_half(static_cast<uint16_t>(w[i] & 0xFFFFu))), xs);
      const float hi = quant_code(__half2float(__ushort_as_half(static_cast<uint16_t>(w[i] >> 16))), xs);
      const __half2 h2 = __floats2half2_rn(lo, hi);  // integers |c| <= 127: exact
      o[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(out + k) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Promotion loop of the decode kernel (warps 6..9): per 128-k block, read the
// block's D (G groups of 16 fp32 columns: tokens 0 .. 16 G / 3), combine the
// three components, and accumulate s * f * D + zero * asum in fp32.  Barrier
// addresses follow the kernel's layout (see decode_kernel).
template <int G>
__device__ __forceinline__ void promote_loop(const GemmParams& p, uint32_t tmem_lane, const uint8_t* bring,
                                             const uint8_t* chunk_smem, uint32_t sbar, int nkb, int kb0, int row,
                                             volatile int* abort_flag, unsigned* status, float (&acc)[dec::kMT]) {
  using namespace dec;
  constexpr int T = (16 * G) / 3;  // tokens whose three columns are loaded
  auto full_g = [&](int g) { return sbar + 8u * g; };
  auto mma_done = [&](int s) { return sbar + 8u * (kNG + s); };
  auto pdone = [&](int s) { return sbar + 8u * (kNG + kNSX + s); };
  auto full_c = [&](int c) { return sbar + 8u * (kNG + 2 * kNSX + kNSA + c); };
  auto empty_c = [&](int c) { return sbar + 8u * (kNG + 2 * kNSX + kNSA + kChunkSlots + c); };
  const bool per_channel = p.group_size != kKBlock;
  const int g_first = per_channel ? 0 : kb0;
  auto chunk_of = [&](int it) { return per_channel ? 0 : ((kb0 + it) >> 3) - (g_first >> 3); };
  auto chunk_row = [&](int it) { return per_channel ? 0 : ((kb0 + it) & 7); };
  const bool has_delta = p.delta != nullptr;
  const int lane = threadIdx.x & 31;
  const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
  for (int j = 0; j < nkb; ++j) {
    const int s = j % kNSX;
    const int b = j % kNB;
    // operands that do not depend on the MMAs first: the block's sums and factors
    // (the TMA copy that wrote them completed full_g) and the row's scale and delta
    if (!warp_wait(full_g(s / kPair), (j / kNSX) & 1, wc)) break;
    float as[kMT], fs[kMT];
    const float4* srow = reinterpret_cast<const float4*>(bring + s * kBStage + kBN * 128);
#pragma unroll
    for (int v4 = 0; v4 < (T + 3) / 4; ++v4) {
      const float4 t = srow[v4];
      const float4 u = srow[kMT / 4 + v4];
      as[4 * v4] = t.x; as[4 * v4 + 1] = t.y; as[4 * v4 + 2] = t.z; as[4 * v4 + 3] = t.w;
      fs[4 * v4] = u.x; fs[4 * v4 + 1] = u.y; fs[4 * v4 + 2] = u.z; fs[4 * v4 + 3] = u.w;
    }
    const int o = chunk_of(j);
    const int slot = o % kChunkSlots;
    if (!warp_wait(full_c(slot), (o / kChunkSlots) & 1, wc)) break;
    const uint8_t* chunk = chunk_smem + slot * (kSChunk + kDChunk);
    const int gr = chunk_row(j);
    const float sc = __half2float(reinterpret_cast<const __half*>(chunk)[gr * kTileN + row]);
    const float dl = has_delta ? reinterpret_cast<const float*>(chunk + kSChunk)[gr * kTileN + row] : 0.0f;
    const float zero = fmaf(-8.0f, sc, dl);  // delta - 8 s: the zero point
    __syncwarp();
    if (lane == 0 && (j + 1 == nkb || chunk_of(j + 1) != o)) mbar_arrive(empty_c(slot));
    if (!warp_wait(mma_done(s), (j / kNSX) & 1, wc)) break;
    tc_fence_after();
    uint32_t d[16 * G];
    const uint32_t dcol = tmem_lane + kDCol0 + b * kBN;
#pragma unroll
    for (int g = 0; g < G; ++g) tmem_ld16(dcol + 16 * g, *reinterpret_cast<uint32_t(*)[16]>(d + 16 * g));
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(pdone(s));
#pragma unroll
    for (int m = 0; m < T; ++m) {
      const float val = fmaf(__uint_as_float(d[3 * m + 2]), 1.0f / 256.0f,
                             fmaf(__uint_as_float(d[3 * m + 1]), 1.0f / 16.0f, __uint_as_float(d[3 * m])));
      acc[m] = fmaf(zero, as[m], fmaf(sc * fs[m], val, acc[m]));
    }
  }
}

// ---------------------------------------------------------------------------
// The decode GEMM kernel.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(dec::kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_d, const GemmParams p, unsigned* status) {
  using namespace dec;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t sb = base;                                   // B tiles [kNSX][7 KB] (1024-aligned)
  const uint32_t sw = sb + kNSX * kBStage;                    // weight tiles [kNSX][8 KB]
  const uint32_t sch = sw + kNSX * kWStage;                   // chunk slots [2][S 2 KB | delta 4 KB]
  const uint32_t sred = sch + kChunkSlots * (kSChunk + kDChunk);  // split-K partials (peers push here)
  const uint32_t sbar = sred + kRedBytes;
  // Barriers.  Per load group g (k-blocks 2 gi, 2 gi + 1; g = gi % kNG, stages 2 g, 2 g + 1):
  //   full_g    both weight tiles + both B tiles landed
  // Per stage s (k-block it, s = it % kNSX):
  //   mma_done  the k-block's MMAs completed (A-stage it % kNSA free, D buffer it % kNB full)
  //   pdone     the promotion warps read D buffer it % kNB and the stage's sums/factors row:
  //             the D buffer and (together with the other stage of its group) the stage are free
  // full_a[a]  A-stage a holds the k-block's weights
  // full_c/empty_c  scale + delta rows of 8 groups landed / released
  auto full_g = [&](int g) { return sbar + 8u * g; };
  auto mma_done = [&](int s) { return sbar + 8u * (kNG + s); };
  auto pdone = [&](int s) { return sbar + 8u * (kNG + kNSX + s); };
  auto full_a = [&](int a) { return sbar + 8u * (kNG + 2 * kNSX + a); };
  auto full_c = [&](int c) { return sbar + 8u * (kNG + 2 * kNSX + kNSA + c); };
  auto empty_c = [&](int c) { return sbar + 8u * (kNG + 2 * kNSX + kNSA + kChunkSlots + c); };
  const uint32_t done_bar = sbar + 8u * (kNumBars - 2);
  const uint32_t red_full = sbar + 8u * (kNumBars - 1);  // partials of this CTA's rows pushed by every rank
  uint8_t* const gmisc = gbase + (sbar + 8u * kNumBars - base);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gmisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gmisc + 4);
  const uint8_t* const chunk_smem = gbase + (sch - base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTileN;
  const int seg = blockIdx.y;  // == rank in the cluster (cluster dims 1 x splits x 1)
  const int kb0 = seg * p.kb_per_split;
  const int nkb = max(0, min(p.kb_total, kb0 + p.kb_per_split) - kb0);
  const bool has_delta = p.delta != nullptr;
  const int ngi = (nkb + kPair - 1) / kPair;  // load groups (pairs of k-blocks) of this segment
  const uint32_t chunk_tx = kSChunk + (has_delta ? kDChunk : 0);
  const bool per_channel = p.group_size != kKBlock;  // group size 128, or one group per column
  const int g_first = per_channel ? 0 : kb0;
  auto chunk_of = [&](int it) { return per_channel ? 0 : ((kb0 + it) >> 3) - (g_first >> 3); };
  int chunks_loaded = 0;  // producer lane: chunk ordinals [0, chunks_loaded) are issued
  auto group_tx = [&](int gi) { return static_cast<uint32_t>(min(kPair, nkb - kPair * gi) * kWStage + kPair * kBStage); };
  auto issue_w = [&](int gi) {  // the pair's weight tiles: one bulk copy
    const int g = gi % kNG;
    bulk_load(sw + g * kPair * kWStage, p.B + (static_cast<size_t>(blockIdx.x) * p.kb_total + kb0 + kPair * gi) * 2048,
              static_cast<uint32_t>(min(kPair, nkb - kPair * gi) * kWStage), full_g(g));
  };
  auto issue_chunk = [&](int o) {
    const int slot = o % kChunkSlots;
    const int grow = ((g_first >> 3) + o) * kChunk;
    const uint32_t dst = sch + slot * (kSChunk + kDChunk);
    mbar_arrive_expect_tx(full_c(slot), chunk_tx);
    tma_load_2d(dst, &tm_s, full_c(slot), n0, grow);
    if (has_delta) tma_load_2d(dst + kSChunk, &tm_d, full_c(slot), n0, grow);
  };
  // Weight-side copies of load group gi (producer lane only).  Every wait comes
  // before the first copy, so a failed wait leaves no copy of this group issued.
  auto weight_copies = [&](int gi, const WaitCtx& wc) -> bool {
    const int last = chunk_of(min(nkb, kPair * gi + kPair) - 1);
    for (int o = chunks_loaded; o <= last; ++o)
      if (!mbar_wait(empty_c(o % kChunkSlots), ((o / kChunkSlots) & 1) ^ 1, wc)) return false;
    mbar_arrive_expect_tx(full_g(gi % kNG), group_tx(gi));
    issue_w(gi);
    for (; chunks_loaded <= last; ++chunks_loaded) issue_chunk(chunks_loaded);
    return true;
  };
  const int pre = p.weight_prefetch ? min(kNG, ngi) : 0;  // load groups whose weights go out first

  const int splits = p.splits;
  const int rpr = (kTileN + splits - 1) / splits;           // weight rows owned by each rank
  const int own_rows = max(0, min(kTileN - seg * rpr, rpr));  // rows this CTA reduces and stores
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tm_b);
    prefetch_tensormap(&tm_s);
    if (has_delta) prefetch_tensormap(&tm_d);
    for (int g = 0; g < kNG; ++g) mbar_init(full_g(g), 1);
    for (int s = 0; s < kNSX; ++s) {
      mbar_init(mma_done(s), 1);
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
    // every rank (this one included) sends own_rows x 16 fp32 partials
    if (splits > 1) mbar_arrive_expect_tx(red_full, static_cast<uint32_t>(own_rows * splits * kMT * 4));
  }
  if (warp == 0) {
    // Weight-side copies of the first load groups go out before anything else
    // (fresh stages and chunk slots: nothing to wait for), one group per lane.
    __syncwarp();
    if (lane < pre) {
      mbar_arrive_expect_tx(full_g(lane), group_tx(lane));
      issue_w(lane);
    }
    if (lane == 0 && pre > 0) {
      // at most kChunkSlots chunks: the first kNSX < 2 * kChunk k-blocks
      const int last = chunk_of(min(nkb, kPair * pre) - 1);
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
  if (splits > 1) cluster_arrive_relaxed();  // this CTA's barriers are initialized (waited before any push)

  // Programmatic dependent launch.  The next grid in the stream may be scheduled
  // now (every grid that follows waits for this one to complete before it reads
  // or writes memory this one uses), so its CTAs take over SM slots as soon as
  // ours exit.  Nothing before griddep_wait() touches memory the preceding grid
  // may write (the activation components, Y); only the weight-side copies of the
  // first stages may be issued earlier, and only when the caller enabled it (the
  // weights must not be written by a preceding grid).
  griddep_launch_dependents();
  griddep_wait();

  int issued = 0;  // load groups whose B box the producer lane has issued
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
      for (int gi = 0; gi < ngi; ++gi) {
        const int g = gi % kNG;
        if (gi >= pre) {
          const uint32_t prev = ((gi / kNG) & 1) ^ 1;  // phase of load group gi - kNG (stages full)
          bool ok = true;
          for (int j = 0; j < kPair && ok; ++j)
            ok = mbar_wait(pdone(kPair * g + j), prev, wc);
          if (!ok || !weight_copies(gi, wc)) break;
        }
        // activation components + sums/factors rows of both k-blocks: one 3-D box
        // {128 B, 56 rows, 2 k-blocks} (a k-block past K reads as zeros)
        tma_load_3d(sb + g * kPair * kBStage, &tm_b, full_g(g), 0, 0, kb0 + kPair * gi);
        issued = gi + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMma, status};
      constexpr uint32_t idesc = idesc_e4m3(128, kBN);
      const uint64_t desc0 = desc_kmajor_sw128(sb);
      for (int it = 0; it < nkb; ++it) {
        const int s = it % kNSX;
        const int a = it % kNSA;
        const int b = it % kNB;
        // full_a implies the stage's bytes landed; D buffer b was last read by the
        // promotion of k-block it - kNB
        if (!mbar_wait(full_a(a), (it / kNSA) & 1, wc)) break;
        if (it >= kNB) {
          const int pk = it - kNB;
          if (!mbar_wait(pdone(pk % kNSX), (pk / kNSX) & 1, wc)) break;
        }
        tc_fence_after();
        const uint64_t ds = desc0 + static_cast<uint64_t>((s * kBStage) >> 4);
        const uint32_t d = tmem + kDCol0 + b * kBN;
        const uint32_t at = tmem + a * kACol;
#pragma unroll
        for (int i = 0; i < 4; ++i) mma_ts_f8(d, at + i * 8, ds + ((i * 32) >> 4), idesc, i > 0 ? 1u : 0u);
        mma_commit(mma_done(s));
      }
      mma_commit(done_bar);
    }
  } else if (warp <= 5) {
    // ---------------------------------------------------------------- dequant
    const WaitCtx wc{abort_flag, p.timeout_ns, kDevTimeoutMath, status};
    const uint8_t* wring = gbase + (sw - base);
    // the weight words of k-block it: 16 words of this thread's row (swizzled 16-byte chunks)
    auto load_words = [&](int it, uint4 (&wv)[4]) -> bool {
      const int s = it % kNSX;
      if (!warp_wait(full_g(s / kPair), (it / kNSX) & 1, wc)) return false;
      const uint8_t* wrow = wring + s * kWStage + row * 64;
#pragma unroll
      for (int c = 0; c < 4; ++c) wv[c] = *reinterpret_cast<const uint4*>(wrow + 16 * (c ^ ((row >> 1) & 3)));
      return true;
    };
    uint4 wv[4];
    bool ok = nkb > 0 && load_words(0, wv);
    for (int it = 0; ok && it < nkb; ++it) {
      const int a = it % kNSA;
      // code j of a word sits at bit 4*(j/2) + 16*(j%2): t holds codes 0,4,1,5 and
      // u codes 2,6,3,7 in its bytes; two permutes restore k order.
      uint32_t v[32];
      const uint32_t words[16] = {wv[0].x, wv[0].y, wv[0].z, wv[0].w, wv[1].x, wv[1].y, wv[1].z, wv[1].w,
                                  wv[2].x, wv[2].y, wv[2].z, wv[2].w, wv[3].x, wv[3].y, wv[3].z, wv[3].w};
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        const uint32_t t = words[w] & 0x0F0F0F0Fu;
        const uint32_t u = (words[w] >> 4) & 0x0F0F0F0Fu;
        v[2 * w] = __byte_perm(t, u, 0x6420);
        v[2 * w + 1] = __byte_perm(t, u, 0x7531);
      }
      if (it >= kNSA) {  // A-stage a was last read by the MMAs of k-block it - kNSA
        const int pk = it - kNSA;
        if (!warp_wait(mma_done(pk % kNSX), (pk / kNSX) & 1, wc)) break;
        tc_fence_after();
      }
      tmem_st32(tmem + lane_base + a * kACol, v);
      // the next k-block's words load while the store completes
      if (it + 1 < nkb) ok = load_words(it + 1, wv);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_a(a));
    }
  } else {
    // ---------------------------------------------------------------- promotion
    // Only the first 3 M columns of D are live: load and combine 16, 32 or 48.
    const int groups = (3 * p.M + 15) / 16;
    if (groups == 1)
      promote_loop<1>(p, tmem + lane_base, gbase + (sb - base), chunk_smem, sbar, nkb, kb0, row, abort_flag, status, acc);
    else if (groups == 2)
      promote_loop<2>(p, tmem + lane_base, gbase + (sb - base), chunk_smem, sbar, nkb, kb0, row, abort_flag, status, acc);
    else
      promote_loop<3>(p, tmem + lane_base, gbase + (sb - base), chunk_smem, sbar, nkb, kb0, row, abort_flag, status, acc);
    tc_fence_before();
  }

  // ---------------------------------------------------------------- split-K reduction + store
  __syncthreads();  // every role is past its loop
  const bool aborted = *abort_flag != 0;
  if (aborted && warp == 0 && lane == 0) {
    // Let every copy the producer issued land before the shared memory is reused
    // or the CTA exits.  Stages whose weight tile was prefetched but whose
    // activation box was not issued get it now, so that their barrier completes.
    for (int gi = issued; gi < pre; ++gi)
      tma_load_3d(sb + (gi % kNG) * kPair * kBStage, &tm_b, full_g(gi % kNG), 0, 0, kb0 + kPair * gi);
    issued = max(issued, pre);
    volatile int never = 0;
    const WaitCtx drain{&never, 50000000ull, kDevTimeoutProducer, status};
    for (int gi = max(0, issued - kNG); gi < issued; ++gi) mbar_wait(full_g(gi % kNG), (gi / kNG) & 1, drain);
    for (int o = max(0, chunks_loaded - kChunkSlots); o < chunks_loaded; ++o)
      mbar_wait(full_c(o % kChunkSlots), (o / kChunkSlots) & 1, drain);
  }
  if (aborted) __syncthreads();  // uniform: the flag no longer changes
  if (aborted) {
#pragma unroll
    for (int m = 0; m < kMT; ++m) acc[m] = __int_as_float(0x7fc00000);
  }
  const bool promote = warp >= 6;
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
      named_barrier_sync(1, 128);
    }
    cluster_wait();  // every rank's barriers are initialized and armed
    if (warp == 6 && lane < splits) {
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
      // wait until every rank's copy of this CTA's rows landed (bounded)
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

// ---------------------------------------------------------------------------
// Host launchers.
// ---------------------------------------------------------------------------
static cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a = {};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

cudaError_t launch_decode_prep_quant(const __half* X, int M, int K, float* x_scale, uint8_t* X8,
                                     cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dec::kMT, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_prep_quant_kernel, X, M, K, x_scale, X8);
}

cudaError_t launch_quant_f16(const __half* X, int M, int K, __half* X16, float* x_scale, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_f16_kernel, X, K, X16, x_scale);
}

cudaError_t launch_decode_prep(const void* X, int x_kind, int M, int K, const float* x_scale, uint8_t* X8,
                               cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((dec::kMT * (K / kKBlock) + 7) / 8, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (x_kind) {
    case kXF16: return cudaLaunchKernelEx(&cfg, decode_prep_kernel<kXF16>, X, M, K, x_scale, X8);
    case kXBF16: return cudaLaunchKernelEx(&cfg, decode_prep_kernel<kXBF16>, X, M, K, x_scale, X8);
    case kXI8: return cudaLaunchKernelEx(&cfg, decode_prep_kernel<kXI8>, X, M, K, x_scale, X8);
    default: return cudaErrorInvalidValue;
  }
}

int decode_max_splits() { return dec::kMaxSplits; }
int decode_b_rows() { return dec::kBRows; }

cudaError_t launch_decode(const CUtensorMap& tm_b, const CUtensorMap& tm_s, const CUtensorMap& tm_d,
                          const GemmParams& p, cudaStream_t stream) {
  unsigned* status = status_word();
  if (!status) return cudaErrorInvalidSymbol;
  if (p.splits < 1 || p.splits > dec::kMaxSplits || p.M < 1 || p.M > dec::kMT)
    return cudaErrorInvalidValue;
  static PerContextOnce attr_set;  // redone after a context rebuild
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_set.needed(dev)) {
    e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dec::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set.done(dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.N / kTileN, p.splits, 1);
  cfg.blockDim = dim3(dec::kThreads, 1, 1);
  cfg.dynamicSmemBytes = dec::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = p.splits;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attr();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_kernel, tm_b, tm_s, tm_d, p, status);
}

}  // namespace wq
