// wq_chain.h -- the persistent decode chain (a list of W4A16 GEMMs with at most
// 8 token rows run by one cooperative launch); declarations shared by the C
// entry point (wq_api.cu) and the kernel (wq_chain.cu).  Not part of the C ABI.
#pragma once

#include "wq_internal.h"

namespace wq {

// Status bit: a chain GEMM gave up waiting for the tiles of its producer.
constexpr unsigned kDevTimeoutChain = 1u << 5;
constexpr int kChainMaxGemms = 8;
constexpr int kChainMaxM = 8;
// Workspace: control words [0, 256), arrival counters and done words of up to
// kChainMaxTiles tiles per chain at fixed offsets, then the partial slots.
constexpr int kChainMaxTiles = 1 << 16;
constexpr size_t kChainPartOffset = 256 + 2 * static_cast<size_t>(kChainMaxTiles) * 4;

// One GEMM of a chain.  The host fills the first block; chain_plan the rest.
struct ChainGemm {
  const void* X;         // [M][K] activations (the Y of GEMM src when src >= 0)
  const uint32_t* B;     // packed weights (wq_pack_w4a16 / wq_pack_w4a16_pair layout)
  const __half* S;       // [G][N] group scales
  const float* delta;    // [G][N] zero-point residual, or null
  void* Y;               // [M][N] (pair: [M][N / 2])
  int y_kind;
  int N, K;              // weight columns (a pair: both projections) and depth
  int per_channel;       // one group spans K
  int pair;              // gate/up pair weight: Y = silu(gate) * up
  int src;               // producer GEMM of X, or -1
  // derived by chain_plan
  int kb;                // K / 128
  int tiles;             // N / 128
  int dependents;        // a later GEMM reads this Y: publish each finished tile
  int ctas;              // CTAs sharing the GEMM's k-blocks (min(grid, kb * tiles))
  int q, r;              // range lengths: the first r ranges hold q + 1 k-blocks, the rest q
  int maxc;              // most CTAs that can share one tile
  int flag_off;          // first tile word of this GEMM (arrival counters, done flags)
  long long total;       // k-blocks of the GEMM, tile-major: position f = tile * kb + k
  long long part_off;    // first float of this GEMM's partial slots [tiles][maxc][128][8]
};

struct ChainParams {
  int n;                 // GEMMs in the list
  int M;                 // token rows (1..8), the same for every GEMM
  int lmax;              // k-blocks of one staged activation window
  int weight_prefetch;   // copy weights before waiting on the preceding grid
  float* part;           // split tiles' partial sums
  unsigned* cnt;         // per-tile arrival counters (left at zero by every call)
  unsigned* done;        // per-tile done words: the call's generation once the tile is stored
  unsigned* ctl;         // [0] generation of the call, [1] CTAs finished (left at zero)
  unsigned long long timeout_ns;
  ChainGemm g[kChainMaxGemms];
};

// Launch geometry on the current device: the grid (every CTA co-resident), the
// activation window and the dynamic shared memory of one CTA.
struct ChainGeom {
  int ctas;
  int lmax;
  int smem;
};
cudaError_t chain_geometry(int x_kind, int M, ChainGeom* out);
// Fills the derived fields of p.g[0 .. p.n) and p.lmax for a grid of geo.ctas
// CTAs; returns the workspace bytes the chain needs (the fixed control region,
// then the partial slots), or 0 when its tiles exceed kChainMaxTiles.
size_t chain_plan(ChainParams& p, const ChainGeom& geo);
// Points p.ctl / cnt / done / part into the workspace laid out by chain_plan.
void chain_bind_workspace(ChainParams& p, void* ws);
cudaError_t launch_chain(int x_kind, const ChainParams& p, const ChainGeom& geo, cudaStream_t stream);

}  // namespace wq
