// wq_chain.cu -- a list of W4A16 decode GEMMs (at most 8 token rows) in one
// persistent launch: the chain kernel.
//
// Why.  One decode GEMM per launch pays a fixed latency on top of its weight
// stream: the hand-off from the preceding grid, the activation rows landing
// behind the weight traffic, the split-K reduction and the last CTAs' exit.
// For the projections of a decode layer that is as long as the stream itself
// (section "Gaps and follow-ups" of "Marlin INT4 on Ada -- how it works" names
// the launch-latency floor of small-batch decode).  Here every CTA of one
// launch walks the whole list, so the weight stream of the next GEMM starts
// while the current one reduces, and a GEMM whose activations are an earlier
// GEMM's output (the down projection after the gate/up pair) waits only for
// the producer tiles that cover its own k-range.
//
// Arithmetic (section "The core mismatch": W_sym = (q - 8) * scale,
// C = C_sym + A_group_sum @ delta), per 128-k block and in fp32:
//     acc[n][m] += scale[g][n] * sum_k (v - 8) x  +  delta[g][n] * a_sum[kb][m]
// with warp-level MMAs on offset codes (wq_warp.cuh): the 8 token slots are the
// MMA's N, slots past M read a zero block.
//
// Work split (stream-K).  The k-blocks of GEMM l, numbered tile-major
// (f = tile * kb + k, which is also the index of the packed 8 KB block), are cut
// into C_l = min(grid, tiles * kb) contiguous ranges of q = T / C_l or q + 1
// k-blocks (the first T % C_l ranges the longer ones), range c going to CTA c, so
// every CTA slot streams the same share of every GEMM.  Compute warp w of a CTA
// owns rows 16 w .. 16 w + 15 of whichever tile it is in.  Each CTA writes its
// part of a tile (its partial [8 tokens][128 rows], fp32) to its slot (index =
// CTA - first CTA of the tile) and increments the tile's counter; the CTA that
// brings the counter to the number of sharers adds the slots in slot order from
// 0.0f (so the sum does not depend on which CTA came last), stores the tile and
// resets the counter.
//
// Roles.  Eight compute warps stream, multiply and accumulate.  At the end of a
// tile they only write the partial and signal a ninth, fixup warp (two hand-off
// mbarriers, full / empty), which fences, counts the arrival and, as the last
// sharer, sums and stores the tile: a fence by a thread waits for that thread's
// copies in flight, and the fixup warp has none, so the weight stream of the
// compute warps never drains at a tile boundary.  The CTA's final tile, when
// nothing is in flight any more, is reduced by the compute warps themselves.
//
// Weights: each lane streams its two 16-byte code chunks per k-block into a
// per-warp ring kD k-blocks deep, in the CTA's own order across GEMM boundaries,
// so the next GEMM's first k-blocks arrive while the current one finishes.  The
// range is processed in windows of up to lmax k-blocks; a window's activation
// rows (a cyclic run of K: consecutive positions of a range are consecutive k,
// wrapping to the next tile) are staged once in shared memory with their block
// sums, together with the scale and delta rows of its positions (small per-lane
// copies of those per k-block cost a quarter of the streaming rate, measured).

// Dependencies.  The warp that stores a tile of a GEMM that a later GEMM reads
// publishes it: the stores are fenced, then one thread writes the call's
// generation number into the tile's done word with release semantics.  Before
// staging a window, the compute warps of a consumer poll (acquire loads, a time
// limit) the done words of the producer tiles that wrote the window's columns.
// Every CTA walks the list in order and a wait only ever targets tiles of an
// earlier GEMM, whose sharers never wait on a later one, so with all CTAs
// resident (a cooperative launch) every wait ends.  A wait that runs out of time
// sets a status bit and the CTA goes on (its results are then wrong, and the
// status word says so).
//
// Generations.  The control word ctl[0] counts completed calls; it only changes
// after every CTA of a launch has finished, so it can be read at any point of the
// launch.  Done words are compared with it plus one, so the words of earlier
// calls never match and nothing has to be cleared between calls.  The last CTA
// to finish (a counter in ctl[1], reset by that CTA) increments it.  Arrival
// counters are reset by the CTA that completes the tile.  The control words sit
// at fixed offsets, so a workspace zeroed once serves any number of calls and
// chains.
//
// Measured on the decode MLP of hidden size 4096 (pair 2 x 11008 with SwiGLU,
// then down 11008 -> 4096, 4 tokens): 34.6 us per block against 27.1 us for the
// fused-SwiGLU call followed by the down call.  The k-block loop runs at about the
// single-GEMM kernel's rate; the start (the first window's activations and scale
// rows, ~6 us) and the producer-to-consumer boundary (~8 us: the last tiles' sums
// through L2, the done words, the consumer's window) are what the separate calls
// do not pay.
#include "wq_chain.h"
#include "wq_warp.cuh"

namespace wq {

namespace chn {
constexpr int kComputeWarps = 8;           // warp w: rows 16 w .. 16 w + 15 of the tile
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 32;  // + the fixup warp
constexpr int kMT = 8;                     // token slots = MMA N
constexpr int kD = 6;                      // ring depth: k-blocks in flight per warp
constexpr int kPre = 3;                    // of them requested before the first activation window
constexpr int kSlot = 1024;                // codes of one k-block of one warp: 2 row halves x 32 lanes x 16 B
constexpr int kRing = kComputeWarps * kD * kSlot;
constexpr int kMaxSmem = 113 * 1024;       // two CTAs per SM
constexpr int kMaxWindow = 128;            // k-blocks of a window (the done-word polls use 2 per k-block)
constexpr int kPartFloats = kTileN * kMT;  // one partial slot [8 tokens][128 rows]
constexpr int kUint4PerBlock = kTileN * kWordsPerKBlock / 4;  // 16-byte chunks of one packed 8 KB block

__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }
__host__ __device__ inline int xs_bytes(int M, int lmax) { return align128((M * lmax + 1) * kKBlock * 2); }
__host__ __device__ inline int asum_bytes(int lmax) { return align128(lmax * 2 * kMT * 4); }
// scale rows [lmax][128] fp16 and delta rows [lmax][128] fp32 of the window's k-blocks
__host__ __device__ inline int ssc_bytes(int lmax) { return align128(lmax * kTileN * 2); }
__host__ __device__ inline int sdl_bytes(int lmax) { return align128(lmax * kTileN * 4); }
__host__ __device__ inline int smem_bytes(int M, int lmax) {
  return 128 + kRing + xs_bytes(M, lmax) + asum_bytes(lmax) + ssc_bytes(lmax) + sdl_bytes(lmax) + 128;
}
}  // namespace chn

namespace {

// Range of CTA c in GEMM G: [a, b), empty for c >= G.ctas.  The T k-blocks are cut
// into C ranges of q = T / C or q + 1 k-blocks, the first r = T % C of them longer:
// range c starts at c q + min(c, r).
__device__ __forceinline__ int range_start(const ChainGemm& G, int c) { return c * G.q + min(c, G.r); }
__device__ __forceinline__ void chain_range(const ChainGemm& G, int c, int& a, int& b) {
  if (c >= G.ctas) {
    a = b = 0;
    return;
  }
  a = range_start(G, c);
  b = range_start(G, c + 1);
}
// The CTA whose range holds position f.
__device__ __forceinline__ int chain_owner(const ChainGemm& G, int f) {
  const int long_end = G.r * (G.q + 1);  // the longer ranges come first
  return f < long_end ? f / (G.q + 1) : G.r + (f - long_end) / G.q;
}

// Position of a CTA in its list of k-blocks.
struct Cursor {
  int l;     // GEMM (== n once the list is done)
  int f;     // position in the GEMM
  int end;   // end of the CTA's range in it
  int tile;  // f / kb
  int k;     // f % kb
};

// The first k-block of the CTA in GEMM l or later (l == n when there is none).
__device__ __noinline__ Cursor cursor_seek(const ChainParams& p, int c, int l) {
  Cursor u;
  for (; l < p.n; ++l) {
    int a, b;
    chain_range(p.g[l], c, a, b);
    if (a < b) {
      u.l = l;
      u.f = a;
      u.end = b;
      u.tile = a / p.g[l].kb;
      u.k = a - u.tile * p.g[l].kb;
      return u;
    }
  }
  u.l = p.n;
  u.f = u.end = u.tile = u.k = 0;
  return u;
}

// Steps past the current k-block; true when that left the GEMM.
__device__ __forceinline__ bool cursor_next(const ChainParams& p, int c, Cursor& u) {
  if (++u.f == u.end) {
    u = cursor_seek(p, c, u.l + 1);
    return true;
  }
  if (++u.k == p.g[u.l].kb) {
    u.k = 0;
    ++u.tile;
  }
  return false;
}

// Stages a window: the activation rows of k-blocks k0, k0 + 1, ... (lx of them,
// cyclic in K) with their block sums (asum[s][0][m] = sum x, asum[s][1][m] = the
// offset term of the codes, see wq_warp.cuh), and the scale and delta rows of the
// window's L positions (tile t0, k-block k0 onwards, wrapping to the next tile):
// ssc[j][128] fp16, sdl[j][128] fp32.  All loads of a batch are in flight together.
template <int XK>
__device__ __forceinline__ void chain_stage(const ChainGemm& G, int M, int t0, int k0, int lx, int L, uint8_t* xs,
                                         int xstride, float* asum, __half* ssc, float* sdl) {
  using namespace chn;
  const uint8_t* const X = static_cast<const uint8_t*>(G.X);
  const int per_tok = lx * 16;  // 16-byte chunks per token row of the window
  const int xtotal = M * per_tok;  // a multiple of 16: a 16-lane group is all X or all scale rows
  const int per_pos = G.delta != nullptr ? 48 : 16;  // 16-byte chunks of one position's scale + delta rows
  const int total = xtotal + L * per_pos;
  constexpr int kU = 8;
  for (int b = 0; b < total; b += kComputeThreads * kU) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int idx = b + u * kComputeThreads + threadIdx.x;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < xtotal) {
        const int m = idx / per_tok;
        const int rem = idx - m * per_tok;
        int kk = k0 + (rem >> 4);
        if (kk >= G.kb) kk -= G.kb;
        v[u] = warp::ldg_cg128(X + (static_cast<size_t>(m) * G.K + kk * kKBlock) * 2 + (rem & 15) * 16);
      } else if (idx < total) {
        const int j = (idx - xtotal) / per_pos;
        const int ch = (idx - xtotal) - j * per_pos;
        const int q = k0 + j;
        const int tile = t0 + q / G.kb;
        const int kk = q - (q / G.kb) * G.kb;
        const size_t row = static_cast<size_t>(G.per_channel ? 0 : kk) * G.N + static_cast<size_t>(tile) * kTileN;
        v[u] = ch < 16 ? warp::ldg_cg128(G.S + row + 8 * ch) : warp::ldg_cg128(G.delta + row + 4 * (ch - 16));
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int idx0 = b + u * kComputeThreads;
      if (idx0 >= total) break;  // uniform
      const int idx = idx0 + threadIdx.x;
      float lo = 0.0f, hi = 0.0f;
      int m = 0, rem = 0;
      if (idx < xtotal) {
        m = idx / per_tok;
        rem = idx - m * per_tok;
        *reinterpret_cast<uint4*>(xs + m * xstride + 16 * warp::xswz(rem, m)) = v[u];
        warp::sum_chunk<XK>(v[u], lo, hi);
      } else if (idx < total) {
        const int j = (idx - xtotal) / per_pos;
        const int ch = (idx - xtotal) - j * per_pos;
        if (ch < 16) *reinterpret_cast<uint4*>(ssc + j * kTileN + 8 * ch) = v[u];
        else *reinterpret_cast<uint4*>(sdl + j * kTileN + 4 * (ch - 16)) = v[u];
      }
      // the 16 chunks of one (token, k-block) are 16 consecutive lanes
#pragma unroll
      for (int sh = 1; sh < 16; sh <<= 1) {
        lo += __shfl_xor_sync(0xffffffffu, lo, sh);
        hi += __shfl_xor_sync(0xffffffffu, hi, sh);
      }
      if (idx < xtotal && (rem & 15) == 0) {
        const int s = rem >> 4;
        asum[s * 2 * kMT + m] = lo + hi;
        asum[s * 2 * kMT + kMT + m] = (XK == kXF16) ? fmaf(1032.0f, lo, 72.0f * hi) : 136.0f * (lo + hi);
      }
    }
  }
}

// The fixup warp's wait on a hand-off barrier: it sleeps between polls, so that it
// takes no issue slots from the compute warps of its scheduler.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(100);
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      *w.abort = 1;
      atomicOr(w.status, w.code);
      return false;
    }
  }
}

// Barrier of the eight compute warps (named barrier 1; the fixup warp is not in it).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(chn::kComputeThreads) : "memory"); }

// A lane's four accumulators (rows rA, rB x tokens 2t, 2t+1) to / from a partial
// slot [8 tokens][128 rows]; tokens past M are neither written nor read.
__device__ __forceinline__ void put_partial(float* slot, const float (&v)[4], int M, int rA, int rB, int t) {
  if (2 * t < M) {
    warp::stg_cg_f32(slot + 2 * t * kTileN + rA, v[0]);
    warp::stg_cg_f32(slot + 2 * t * kTileN + rB, v[2]);
  }
  if (2 * t + 1 < M) {
    warp::stg_cg_f32(slot + (2 * t + 1) * kTileN + rA, v[1]);
    warp::stg_cg_f32(slot + (2 * t + 1) * kTileN + rB, v[3]);
  }
}
__device__ __forceinline__ void get_partial(const float* slot, float (&v)[4], int M, int rA, int rB, int t) {
  v[0] = v[1] = v[2] = v[3] = 0.0f;
  if (2 * t < M) {
    v[0] = warp::ldg_cg_f32(slot + 2 * t * kTileN + rA);
    v[2] = warp::ldg_cg_f32(slot + 2 * t * kTileN + rB);
  }
  if (2 * t + 1 < M) {
    v[1] = warp::ldg_cg_f32(slot + (2 * t + 1) * kTileN + rA);
    v[3] = warp::ldg_cg_f32(slot + (2 * t + 1) * kTileN + rB);
  }
}

// Sums over the nc partial slots of a tile of NCH runs of four consecutive elements
// (src[i], one run per lane's chunk; nch of them used), each in slot order from
// 0.0f, so every CTA that completes a tile forms the same sums.  B slots of all
// chunks are loaded before they are added.
template <int NCH, int B>
__device__ __forceinline__ void sum_slots(const float* const (&src)[NCH], int nch, int nc, float4 (&acc)[NCH]) {
#pragma unroll
  for (int i = 0; i < NCH; ++i) acc[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int j0 = 0; j0 < nc; j0 += B) {
    float4 v[B][NCH];
#pragma unroll
    for (int b = 0; b < B; ++b)
#pragma unroll
      for (int i = 0; i < NCH; ++i)
        if (j0 + b < nc && i < nch) v[b][i] = warp::ldg_cg_f4(src[i] + (j0 + b) * chn::kPartFloats);
#pragma unroll
    for (int b = 0; b < B; ++b)
#pragma unroll
      for (int i = 0; i < NCH; ++i)
        if (j0 + b < nc && i < nch) {
          acc[i].x += v[b][i].x;
          acc[i].y += v[b][i].y;
          acc[i].z += v[b][i].z;
          acc[i].w += v[b][i].w;
        }
  }
}

// The fixup warp's store of a tile from its nc partial slots: plain, Y[m][n0 + r];
// a gate/up pair, Y[m][n0 / 2 + 8 (r / 16) + r % 8] = silu(gate row r) * up row r + 8
// for the rows r with r % 16 < 8.  Lane l takes the runs of four rows of token m at
// rows 4l .. 4l + 3 (plain), or, for the pair, the runs e = l + 32 i < 16 M: token
// e / 16, gate rows 4q .. 4q + 3 with q = 4 (pc / 2) + pc % 2, pc = e % 16, and the up
// rows 8 further on.  Four runs per pass, one slot per batch (the kernel's register
// budget: with 9 warps per CTA and two CTAs per SM, a scheduler holds 5 warps).
__device__ __forceinline__ void fix_store(const ChainGemm& G, int tile, const float* part, int nc, int M, int lane) {
  const int n0 = tile * kTileN;
  const float* src[4];
  float4 acc[4];
  if (!G.pair) {
    for (int m0 = 0; m0 < M; m0 += 4) {
      const int nch = min(4, M - m0);
#pragma unroll
      for (int i = 0; i < 4; ++i) src[i] = part + (m0 + i) * kTileN + 4 * lane;
      sum_slots<4, 1>(src, nch, nc, acc);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < nch) {
          const size_t o = static_cast<size_t>(m0 + i) * G.N + n0 + 4 * lane;
          store_y_any(G.Y, G.y_kind, o, acc[i].x);
          store_y_any(G.Y, G.y_kind, o + 1, acc[i].y);
          store_y_any(G.Y, G.y_kind, o + 2, acc[i].z);
          store_y_any(G.Y, G.y_kind, o + 3, acc[i].w);
        }
      }
    }
  } else {
    for (int e0 = lane; e0 < M * 16; e0 += 64) {  // two runs (gate and up) per element
      const int ne = (e0 + 32 < M * 16) ? 2 : 1;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int e = e0 + 32 * i;
        const int pc = e & 15;
        const int q = 4 * (pc >> 1) + (pc & 1);
        src[2 * i] = part + (e >> 4) * kTileN + 4 * q;
        src[2 * i + 1] = src[2 * i] + 8;
      }
      sum_slots<4, 1>(src, 2 * ne, nc, acc);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i < ne) {
          const int e = e0 + 32 * i;
          const int pc = e & 15;
          const int q = 4 * (pc >> 1) + (pc & 1);
          const size_t o = static_cast<size_t>(e >> 4) * (G.N >> 1) + (n0 >> 1) + 8 * (q >> 2) + 4 * (q & 3);
          const float4 gv = acc[2 * i], uv = acc[2 * i + 1];
          store_y_any(G.Y, G.y_kind, o, silu_mul(gv.x, uv.x));
          store_y_any(G.Y, G.y_kind, o + 1, silu_mul(gv.y, uv.y));
          store_y_any(G.Y, G.y_kind, o + 2, silu_mul(gv.z, uv.z));
          store_y_any(G.Y, G.y_kind, o + 3, silu_mul(gv.w, uv.w));
        }
      }
    }
  }
}

}  // namespace

template <int XK>
__global__ void __launch_bounds__(chn::kThreads, 2)
    chain_kernel(const __grid_constant__ ChainParams p, unsigned* status) {
  using namespace chn;
  using namespace warp;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* const sm = smem_raw + (base - raw);

  const int warp_id = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int c = blockIdx.x;
  const int M = p.M;
  const int lmax = p.lmax;
  const int xstride = lmax * kKBlock * 2;  // bytes per token row of the window
  uint8_t* const xs = sm + kRing;
  float* const asum = reinterpret_cast<float*>(sm + kRing + xs_bytes(M, lmax));
  __half* const ssc = reinterpret_cast<__half*>(sm + kRing + xs_bytes(M, lmax) + asum_bytes(lmax));
  float* const sdl = reinterpret_cast<float*>(sm + kRing + xs_bytes(M, lmax) + asum_bytes(lmax) + ssc_bytes(lmax));
  const int misc_off = kRing + xs_bytes(M, lmax) + asum_bytes(lmax) + ssc_bytes(lmax) + sdl_bytes(lmax);
  // The last 128 bytes: the compute -> fixup hand-off barriers full[2] and empty[2]
  // (slot b of flush i is i % 2), the CTA's abort flag, and misc words: misc[1] the
  // last-sharer flag of the compute warps' own reduction, misc[2] the last GEMM in
  // which the CTA has k-blocks.
  const uint32_t full_bar = base + misc_off;        // + 8 b
  const uint32_t empty_bar = base + misc_off + 16;  // + 8 b
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sm + misc_off + 32);
  volatile unsigned* const misc = reinterpret_cast<volatile unsigned*>(sm + misc_off + 40);

  if (threadIdx.x == 0) {
    mbar_init(full_bar, kComputeWarps);
    mbar_init(full_bar + 8, kComputeWarps);
    mbar_init(empty_bar, 1);
    mbar_init(empty_bar + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // token slots past M: a zero k-block and zero sums (the staging writes rows < M only)
  if (threadIdx.x < 16)
    *reinterpret_cast<uint4*>(xs + M * xstride + 16 * threadIdx.x) = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < lmax * 2 * kMT; i += kThreads)
    if (i % kMT >= M) asum[i] = 0.0f;

  // The last GEMM in which this CTA has k-blocks: its last tile is the CTA's final
  // segment, which the compute warps reduce themselves (their rings are empty by then).
  if (threadIdx.x == 0) {
    int last_l = -1;
    for (int l = 0; l < p.n; ++l) {
      int a, b;
      chain_range(p.g[l], c, a, b);
      if (a < b) last_l = l;
    }
    misc[2] = static_cast<unsigned>(last_l);
  }

  // Codes: rows rA = 16 warp + g and rB = rA + 8 of the tile, logical chunk t
  // (stored at slot t ^ ((r / 2) % 4) of the packed block; both rows share it).
  const int rA = 16 * warp_id + g;
  const int rB = rA + 8;
  const int offA = rA * 4 + (t ^ ((g >> 1) & 3));
  const int offB = offA + 32;
  const uint32_t ring_w = base + static_cast<uint32_t>(warp_id * kD * kSlot);
  const uint64_t pol = l2_evict_first();
  const bool compute = warp_id < kComputeWarps;

  // The issue cursor runs kD k-blocks ahead of the consumer, across GEMMs.
  Cursor iu = cursor_seek(p, c, 0);
  auto issue = [&](int s) {
    if (iu.l < p.n) {
      const ChainGemm& G = p.g[iu.l];
      const uint32_t dst = ring_w + static_cast<uint32_t>(s * kSlot);
      // packed block of (tile, k) = position f: the GEMM's blocks are stored tile-major
      const uint4* src = reinterpret_cast<const uint4*>(G.B) + static_cast<size_t>(iu.f) * kUint4PerBlock;
      cp_async16(dst + lane * 16, src + offA, pol);
      cp_async16(dst + 512 + lane * 16, src + offB, pol);
      cursor_next(p, c, iu);
    }
    cp_async_commit();  // one group per slot, empty past the list
  };
  // Weights are only ever written by the pack: with the caller's promise
  // (weight prefetch) the first k-blocks are requested before the preceding grid
  // has finished.  The rest of the ring follows the first activation window, so
  // that those loads do not queue behind a whole ring of weight traffic.
  if (compute && p.weight_prefetch) {
#pragma unroll 1
    for (int d = 0; d < kPre; ++d) issue(d);
  }
  griddep_launch_dependents();
  griddep_wait();  // activations written by the preceding grid are visible from here on
  if (compute && !p.weight_prefetch) {
#pragma unroll 1
    for (int d = 0; d < kPre; ++d) issue(d);
  }
  __syncthreads();

  if (!compute) {
    // ---- the fixup warp: the split-K arrival, sum and store of every segment of
    // the CTA but the final one, in the compute warps' order, off their path
    const WaitCtx wctx{abort_flag, p.timeout_ns, kDevTimeoutChain, status};
    // The generation word only changes after every CTA has finished: it can be read
    // at any point of the launch.
    const unsigned target = *reinterpret_cast<volatile const unsigned*>(p.ctl) + 1u;
    const int last_l = static_cast<int>(misc[2]);
    int i = 0;
    for (int l = 0; l <= last_l; ++l) {
      const ChainGemm& G = p.g[l];
      int a, b;
      chain_range(G, c, a, b);
      if (a >= b) continue;
      const int t1 = (b - 1) / G.kb;
      for (int tile = a / G.kb; tile <= t1; ++tile, ++i) {
        if (l == last_l && tile == t1) break;
        const int bi = i & 1;
        mbar_wait_sleep(full_bar + 8 * bi, (i >> 1) & 1, wctx);
        const int f0 = tile * G.kb;
        const int c0 = chain_owner(G, f0);
        const int nc = chain_owner(G, f0 + G.kb - 1) - c0 + 1;
        unsigned last = 1u;
        if (nc > 1) {
          if (lane == 0) {
            __threadfence();  // the compute warps' partials (ordered before the barrier) first
            const unsigned old = atomicAdd(p.cnt + G.flag_off + tile, 1u);
            last = (old == static_cast<unsigned>(nc - 1)) ? 1u : 0u;
            if (last) atomicExch(p.cnt + G.flag_off + tile, 0u);
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) __threadfence();
        }
        if (last && nc <= G.maxc) {
          const float* const part = p.part + G.part_off + static_cast<size_t>(tile) * G.maxc * kPartFloats;
          fix_store(G, tile, part, nc, M, lane);
          if (G.dependents) {
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(p.done + G.flag_off + tile, target);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar + 8 * bi);
      }
    }
  } else {
    // Final segment of the CTA: partial, arrival and the sum in slot order by the
    // last sharer, all by the compute warps.  Returns whether this CTA holds the
    // tile's result in tot (then it stores it).
    auto reduce_final = [&](const ChainGemm& G, int tile, float (&tot)[4]) -> bool {
      const int f0 = tile * G.kb;
      const int c0 = chain_owner(G, f0);
      const int nc = chain_owner(G, f0 + G.kb - 1) - c0 + 1;
      if (nc == 1) return true;
      const int j = c - c0;
      const bool ok = nc <= G.maxc && j >= 0 && j < nc;  // the plan's bound
      float* const part = p.part + G.part_off + static_cast<size_t>(tile) * G.maxc * kPartFloats;
      if (ok) put_partial(part + j * kPartFloats, tot, M, rA, rB, t);
      __threadfence();  // (the ring is empty: nothing of this thread is in flight)
      compute_sync();
      if (threadIdx.x == 0) {
        unsigned last = 0u;
        if (ok) {
          const unsigned old = atomicAdd(p.cnt + G.flag_off + tile, 1u);
          last = (old == static_cast<unsigned>(nc - 1)) ? 1u : 0u;
          if (last) atomicExch(p.cnt + G.flag_off + tile, 0u);
        } else {
          atomicOr(status, kDevTimeoutChain);
        }
        misc[1] = last;
      }
      compute_sync();
      if (misc[1] == 0u) return false;
      __threadfence();
      // the sum in slot order from 0.0f (as the fixup warp forms it), 8 slots per batch
      float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int j0 = 0; j0 < nc; j0 += 8) {
        float v[8][4];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int jj = j0 + b;
          if (jj < nc && jj != j) get_partial(part + jj * kPartFloats, v[b], M, rA, rB, t);
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int jj = j0 + b;
          if (jj < nc)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] += (jj == j) ? tot[e] : v[b][e];
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) tot[e] = s[e];
      return true;
    };

    auto store_final = [&](const ChainGemm& G, int tile, const float (&tot)[4]) {
      const int n0 = tile * kTileN;
      if (G.pair) {
        // row rA is a gate column and rB = rA + 8 the up column of the same output
        const int jc = ((n0 + 16 * warp_id) >> 1) + g;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = 2 * t + e;
          if (tok < M)
            store_y_any(G.Y, G.y_kind, static_cast<size_t>(tok) * (G.N >> 1) + jc, silu_mul(tot[e], tot[2 + e]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = 2 * t + (e & 1);
          const int row = (e < 2) ? rA : rB;
          if (tok < M) store_y_any(G.Y, G.y_kind, static_cast<size_t>(tok) * G.N + n0 + row, tot[e]);
        }
      }
      if (G.dependents) {
        __threadfence();  // the stores are visible GPU-wide before the done word
        compute_sync();
        if (threadIdx.x == 0)
          st_release_gpu(p.done + G.flag_off + tile, *reinterpret_cast<volatile const unsigned*>(p.ctl) + 1u);
      }
    };

    // Waits until the producer tiles that wrote columns [128 k, 128 k + 128) of
    // this GEMM's X, for the window's k-blocks, are stored (one poll per tile).
    auto wait_window = [&](const ChainGemm& G, int k0, int lx) {
      const ChainGemm& P = p.g[G.src];
      const int per = P.pair ? 2 : 1;  // producer tiles per 128 columns
      if (static_cast<int>(threadIdx.x) < lx * per) {
        const int s = static_cast<int>(threadIdx.x) / per;
        int kk = k0 + s;
        if (kk >= G.kb) kk -= G.kb;
        const unsigned* const w = p.done + P.flag_off + kk * per + (static_cast<int>(threadIdx.x) - s * per);
        const uint64_t t0 = globaltimer_ns();
        const unsigned target = *reinterpret_cast<volatile const unsigned*>(p.ctl) + 1u;
        while (ld_acquire_gpu(w) != target) {
          if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicOr(status, kDevTimeoutChain);
            break;
          }
          __nanosleep(64);
        }
        __threadfence();
      }
    };

    // ---- the compute warps: the CTA's k-blocks, GEMM after GEMM
    Cursor cu = cursor_seek(p, c, 0);
    int slot = 0, prem = 0, xslot = 0, lx = 1, nfl = 0, wpos = 0, final_tile = -1;
    bool primed = false;
    float tot[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float zero4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int sw = (t >> 1) | ((g & 1) << 1);  // xswz for this lane's chunks 4t + q: flips the low bits of q
    // token slot g: its row of the window, or the zero k-block (not advanced) past M
    // (shared-space addresses: 32-bit, which keeps the loop within its registers)
    const uint32_t xrow = smem_u32(xs) + static_cast<uint32_t>((g < M ? g * xstride : M * xstride) + 64 * t);
    const uint32_t asum_s = smem_u32(asum) + 8u * t;        // + 64 xslot: (sum, offset) of tokens 2t, 2t+1
    const uint32_t ssc_s = smem_u32(ssc) + 2u * rA;          // + 256 wpos: the scale of row rA (rB: + 16)
    const uint32_t sdl_s = smem_u32(sdl) + 4u * rA;          // + 512 wpos: the delta of row rA (rB: + 32)
    const int xstep = g < M ? kKBlock * 2 : 0;
    while (cu.l < p.n) {
      const ChainGemm& G = p.g[cu.l];
      if (prem == 0) {  // a new window: up to lmax k-blocks of the range
        const int L = min(lmax, cu.end - cu.f);
        lx = min(L, G.kb);
        if (G.src >= 0) wait_window(G, cu.k, lx);
        compute_sync();  // every warp is done with the previous window
        chain_stage<XK>(G, M, cu.tile, cu.k, lx, L, xs, xstride, asum, ssc, sdl);
        compute_sync();
        if (!primed) {
#pragma unroll 1
          for (int d = kPre; d < kD; ++d) issue(d);
          primed = true;
        }
        prem = L;
        xslot = 0;
        wpos = 0;
      }
      // The k-blocks up to the end of the window or of the tile, whichever is first.
      const int run = min(prem, min(G.kb - cu.k, cu.end - cu.f));
      const bool has_delta = G.delta != nullptr;
#pragma unroll 1
      for (int it = 0; it < run; ++it) {
        cp_async_wait<kD - 1>();  // this slot's group (this lane's copies) has landed
        const uint32_t sl = ring_w + static_cast<uint32_t>(slot * kSlot);
        const uint4 a = lds128(sl + lane * 16);
        const uint4 cc = lds128(sl + 512 + lane * 16);
        // The slot has been read into registers: refill it with the k-block kD further on.
        asm volatile("" ::"r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(cc.x), "r"(cc.y), "r"(cc.z), "r"(cc.w)
                     : "memory");
        issue(slot);
        slot = (slot + 1 == kD) ? 0 : slot + 1;
        // the scale and delta rows of this position of the window
        const float sA = __half2float(__ushort_as_half(lds_u16(ssc_s + 256u * wpos)));
        const float sB = __half2float(__ushort_as_half(lds_u16(ssc_s + 256u * wpos + 16u)));
        const float dA = has_delta ? lds_f32(sdl_s + 512u * wpos) : 0.0f;
        const float dB = has_delta ? lds_f32(sdl_s + 512u * wpos + 32u) : 0.0f;
        ++wpos;

        uint32_t xr[16];
        const uint32_t row = xrow + static_cast<uint32_t>(xslot * xstep);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = lds128(row + 16u * (q ^ sw));
          xr[4 * q] = v.x;
          xr[4 * q + 1] = v.y;
          xr[4 * q + 2] = v.z;
          xr[4 * q + 3] = v.w;
        }
        // MMA step s = 4h + p takes pair p of words 4t + 2h (k 2t, 2t+1 of the
        // fragment) and 4t + 2h + 1 (k 2t+8, 2t+9), rows g and g + 8; the activation
        // fragment takes x at the same physical k (32t + 16h + 2p (+ 8)).  fp16:
        // low-nibble (p even) and high-nibble (p odd) steps accumulate separately;
        // bf16: the chains are the two h.
        const uint32_t wa[2][2] = {{a.x, a.y}, {a.z, a.w}};
        const uint32_t wc[2][2] = {{cc.x, cc.y}, {cc.z, cc.w}};
        float acc[2][4];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const int h = (XK == kXBF16) ? (st & 1) : (st >> 2);
          const int pp = (XK == kXBF16) ? (st >> 1) : (st & 3);
          uint32_t f[4];
#pragma unroll
          for (int jf = 0; jf < 4; ++jf) {
            const uint32_t w = (jf & 1) ? wc[h][jf >> 1] : wa[h][jf >> 1];
            if (XK == kXBF16) f[jf] = off_bf16(w >> (4 * pp));
            else f[jf] = (pp & 1) ? off_hi_f16(pp >= 2 ? w >> 8 : w) : off_lo_f16(pp >= 2 ? w >> 8 : w);
          }
          const int ch = (XK == kXBF16) ? h : (pp & 1);
          const bool first = (XK == kXBF16) ? (pp == 0) : (h == 0 && pp < 2);
          if (first) mma16816<XK>(acc[ch], zero4, f[0], f[1], f[2], f[3], xr[8 * h + pp], xr[8 * h + 4 + pp]);
          else mma16816<XK>(acc[ch], acc[ch], f[0], f[1], f[2], f[3], xr[8 * h + pp], xr[8 * h + 4 + pp]);
        }
        const float2 ofs = lds_f2(asum_s + 64u * xslot + 32u);
        float d[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float o = (e & 1) ? ofs.y : ofs.x;
          d[e] = (XK == kXBF16 ? acc[0][e] + acc[1][e] : fmaf(acc[1][e], 0.0625f, acc[0][e])) - o;
        }
        if (has_delta) {
          const float2 as = lds_f2(asum_s + 64u * xslot);
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
        if (++xslot == lx) xslot = 0;
      }
      prem -= run;
      cu.f += run;
      cu.k += run;
      if (cu.k == G.kb || cu.f == cu.end) {  // the CTA's part of this tile is done
        if (cu.f == cu.end && cu.l == static_cast<int>(misc[2])) {
          final_tile = cu.tile;  // reduced after the loop, where few registers are live
          break;
        } else {
          // hand the partial to the fixup warp: its slot in the workspace, then the barrier
          const int bi = nfl & 1;
          if (nfl >= 2)
            mbar_wait(base + misc_off + 16 + 8 * bi, ((nfl >> 1) - 1) & 1,
                      WaitCtx{reinterpret_cast<volatile int*>(sm + misc_off + 32), p.timeout_ns, kDevTimeoutChain,
                              status});
          const int j = c - chain_owner(G, cu.tile * G.kb);
          if (j >= 0 && j < G.maxc)
            put_partial(p.part + G.part_off + (static_cast<size_t>(cu.tile) * G.maxc + j) * kPartFloats, tot, M,
                        rA, rB, t);
          __syncwarp();
          if (lane == 0) mbar_arrive(base + misc_off + 8 * bi);
          ++nfl;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) tot[e] = 0.0f;
      }
      if (cu.f == cu.end) {  // the next GEMM starts a new window
        cu = cursor_seek(p, c, cu.l + 1);
        prem = 0;
      } else if (cu.k == G.kb) {
        cu.k = 0;
        ++cu.tile;
      }
    }
    cp_async_wait<0>();  // nothing of this thread is in flight (the trailing groups are empty)
    if (final_tile >= 0) {
      const ChainGemm& G = p.g[misc[2]];
      if (reduce_final(G, final_tile, tot)) store_final(G, final_tile, tot);
    }
  }

  // The last CTA to finish advances the generation for the next call.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(p.ctl + 1, 1u);
    if (old == gridDim.x - 1) {
      atomicExch(p.ctl + 1, 0u);
      __threadfence();
      atomicAdd(p.ctl, 1u);
    }
  }
}

// ---------------------------------------------------------------- host side

namespace {

int chain_lmax(int M) {
  int best = 1;
  for (int l = 1; l <= chn::kMaxWindow; ++l)
    if (chn::smem_bytes(M, l) <= chn::kMaxSmem) best = l;
  return best;
}

template <int XK>
cudaError_t chain_attr(int dev) {
  static PerContextOnce attr_set;  // redone after a context rebuild
  if (!attr_set.needed(dev)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(chain_kernel<XK>, cudaFuncAttributeMaxDynamicSharedMemorySize, chn::kMaxSmem);
  if (e == cudaSuccess) attr_set.done(dev);
  return e;
}

}  // namespace

cudaError_t chain_geometry(int x_kind, int M, ChainGeom* out) {
  if (M < 1 || M > kChainMaxM || (x_kind != kXF16 && x_kind != kXBF16)) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // one cached geometry per (device, activation type, M), redone after a context rebuild
  struct Entry {
    unsigned long long ctx;
    ChainGeom geo;
  };
  static Entry cache[16][2][kChainMaxM + 1];
  const unsigned long long ctx = current_context_id();
  const int xi = x_kind == kXBF16 ? 1 : 0;
  if (dev >= 0 && dev < 16 && ctx != 0 && cache[dev][xi][M].ctx == ctx) {
    *out = cache[dev][xi][M].geo;
    return cudaSuccess;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = x_kind == kXBF16 ? chain_attr<kXBF16>(dev) : chain_attr<kXF16>(dev);
  if (e != cudaSuccess) return e;
  ChainGeom geo;
  geo.lmax = chain_lmax(M);
  geo.smem = chn::smem_bytes(M, geo.lmax);
  int per_sm = 0;
  e = x_kind == kXBF16
          ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_kernel<kXBF16>, chn::kThreads, geo.smem)
          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_kernel<kXF16>, chn::kThreads, geo.smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  geo.ctas = (per_sm < 2 ? per_sm : 2) * sms;
  if (dev >= 0 && dev < 16 && ctx != 0) cache[dev][xi][M] = Entry{ctx, geo};
  *out = geo;
  return cudaSuccess;
}

static size_t align256z(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t chain_plan(ChainParams& p, const ChainGeom& geo) {
  p.lmax = geo.lmax;
  int flags = 0;
  long long parts = 0;
  for (int l = 0; l < p.n; ++l) {
    ChainGemm& G = p.g[l];
    G.kb = G.K / kKBlock;
    G.tiles = G.N / kTileN;
    G.total = static_cast<long long>(G.kb) * G.tiles;
    G.ctas = static_cast<int>(G.total < geo.ctas ? G.total : geo.ctas);
    G.q = static_cast<int>(G.total / G.ctas);
    G.r = static_cast<int>(G.total % G.ctas);
    // Ranges hold at least q = T / C k-blocks, so a tile of kb consecutive positions
    // meets at most 1 + ceil((kb - 1) / q) of them.
    const long long minlen = G.q;
    long long maxc = 2 + (G.kb - 1) / minlen;
    if (maxc > G.ctas) maxc = G.ctas;
    G.maxc = static_cast<int>(maxc);
    G.flag_off = flags;
    flags += G.tiles;
    G.part_off = parts;
    if (G.maxc > 1) parts += static_cast<long long>(G.tiles) * G.maxc * chn::kPartFloats;
    G.dependents = 0;
  }
  for (int l = 0; l < p.n; ++l)
    if (p.g[l].src >= 0) p.g[p.g[l].src].dependents = 1;
  if (flags > kChainMaxTiles) return 0;
  return kChainPartOffset + align256z(static_cast<size_t>(parts) * 4);
}

// The control words sit at the same offsets for every chain, ahead of the partial
// slots, so a workspace that one chain has used (its counters back at zero, its done
// words at earlier generations) serves any other.
void chain_bind_workspace(ChainParams& p, void* ws) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  p.ctl = reinterpret_cast<unsigned*>(b);
  p.cnt = reinterpret_cast<unsigned*>(b + 256);
  p.done = reinterpret_cast<unsigned*>(b + 256 + static_cast<size_t>(kChainMaxTiles) * 4);
  p.part = reinterpret_cast<float*>(b + kChainPartOffset);
}

template <int XK>
static cudaError_t launch_chain_t(const ChainParams& p, const ChainGeom& geo, unsigned* status, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = chain_attr<XK>(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(geo.ctas, 1, 1);
  cfg.blockDim = dim3(chn::kThreads, 1, 1);
  cfg.dynamicSmemBytes = geo.smem;
  cfg.stream = st;
  // Cooperative: the CTAs wait on one another's tiles, so all of them must be
  // resident at once (the launch fails otherwise).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, chain_kernel<XK>, p, status);
}

cudaError_t launch_chain(int x_kind, const ChainParams& p, const ChainGeom& geo, cudaStream_t stream) {
  unsigned* status = status_word();
  if (!status) return cudaErrorInvalidSymbol;
  if (p.n < 1 || p.n > kChainMaxGemms || p.M < 1 || p.M > kChainMaxM || p.lmax < 1 || p.lmax > chn::kMaxWindow ||
      geo.smem > chn::kMaxSmem || geo.ctas < 1 || !p.ctl)
    return cudaErrorInvalidValue;
  return x_kind == kXBF16 ? launch_chain_t<kXBF16>(p, geo, status, stream)
                          : launch_chain_t<kXF16>(p, geo, status, stream);
}

}  // namespace wq
