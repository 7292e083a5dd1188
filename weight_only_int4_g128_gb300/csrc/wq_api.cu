// wq_api.cu -- the extern "C" entry points of libwq.so: argument checks,
// shape heuristics, TMA tensor maps, workspace carving and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <cstring>
#include <mutex>

#include "wq.h"
#include "wq_internal.h"
#include "wq_chain.h"

namespace {

thread_local char t_err[512] = "";
std::atomic<int> g_weight_prefetch{0};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(WQ_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_device() {
  static int cache[64];  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev >= 0 && dev < 64 && cache[dev] == 1) return WQ_OK;
  if (!wq_device_supported(dev)) {
    if (dev >= 0 && dev < 64) cache[dev] = 2;
    return fail(WQ_ERR_ARCH, "device %d is not an sm_103 GPU", dev);
  }
  if (dev >= 0 && dev < 64) cache[dev] = 1;
  return WQ_OK;
}

bool checked_mode() {
  static int v = -1;
  if (v < 0) {
    const char* s = getenv("WQ_CHECKED");
    v = (s && s[0] && s[0] != '0') ? 1 : 0;
  }
  return v == 1;
}

unsigned long long timeout_ns() {
  static unsigned long long v = 0;
  if (v == 0) {
    const char* s = getenv("WQ_WAIT_LIMIT_MS");
    long long ms = s ? atoll(s) : 2000;
    if (ms <= 0 || ms > 10000) ms = 2000;
    v = static_cast<unsigned long long>(ms) * 1000000ull;
  }
  return v;
}

int after_launch(cudaError_t e, const char* where, cudaStream_t st) {
  if (e != cudaSuccess) return cuda_fail(e, where);
  if (checked_mode()) {
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, where);
    unsigned int status = 0;
    e = wq::read_status(&status);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (status) return fail(WQ_ERR_TIMEOUT, "%s: bounded device wait expired (status 0x%x)", where, status);
  }
  return WQ_OK;
}

int norm_group(int K, int group_size, int* gs_out) {
  int gs = (group_size == -1) ? K : group_size;
  if (gs != 128 && gs != K)
    return fail(WQ_ERR_UNSUPPORTED_SHAPE, "group_size %d: only 128 or K (-1) are supported", group_size);
  if (gs <= 0 || K % gs != 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "K %% group_size != 0");
  *gs_out = gs;
  return WQ_OK;
}

int check_kn(int K, int N) {
  if (K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0)
    return fail(WQ_ERR_UNSUPPORTED_SHAPE, "K=%d N=%d: both must be positive multiples of 128", K, N);
  return WQ_OK;
}

// ---------------------------------------------------------------- tensor maps
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// 2-D row-major tensor [rows][cols] of `esize`-byte elements; box [box_rows][box_cols].
int make_map(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* ptr, uint64_t rows,
             uint64_t cols, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle sw) {
  EncodeFn enc = get_encode();
  if (!enc) return fail(WQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return WQ_OK;
}

// Activations [rows][K] as a 3-D tensor {64 k, rows, K/64 halves-of-k-blocks} so
// that one box {64, box_rows, 2} fetches a whole 128-k block as two 128-byte
// swizzled atoms placed one after the other in shared memory (box_atoms = 4:
// two consecutive 128-k blocks).
int make_map_x3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t rows, uint64_t K,
                 uint32_t box_rows, uint32_t box_atoms = 2) {
  EncodeFn enc = get_encode();
  if (!enc) return fail(WQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {64, rows, K / 64};
  cuuint64_t strides[2] = {K * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_atoms};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WQ_ERR_CUDA, "cuTensorMapEncodeTiled (3-D activations) failed (%d)", static_cast<int>(r));
  return WQ_OK;
}

// Decode activation components [rows][K] bytes as a 3-D tensor {128 bytes of a
// k-block, rows, K/128 k-blocks}: one box {128, rows, 2} fetches two k-blocks'
// tiles, each rows x 128 B with 128-byte swizzling, one after the other.
int make_map_b3d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t K) {
  EncodeFn enc = get_encode();
  if (!enc) return fail(WQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {128, rows, K / 128};
  cuuint64_t strides[2] = {K, 128};
  cuuint32_t box[3] = {128, static_cast<cuuint32_t>(rows), 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WQ_ERR_CUDA, "cuTensorMapEncodeTiled (decode components) failed (%d)", static_cast<int>(r));
  return WQ_OK;
}

// ---------------------------------------------------------------- heuristics
struct Plan {
  bool gemv;      // M <= 16: decode pre-pass + decode kernel
  int bt;         // token tile
  int splits;
  int kb_per_split;
  int kb_first;   // large M: k-blocks of segment 0 (which also runs the correction stages)
  int kaug;       // large-M correction length (0 without correction or for the decode kernel)
  // large M, one K segment per tile: the last, partial wave of tiles as a second
  // launch split along K (0 tiles: none)
  int tail_tiles, tail_splits, tail_kbps, tail_kb_first;
  size_t off_aug, off_daug, off_x16, off_xs;  // byte offsets into the workspace (large M)
  size_t off_x8;                      // byte offset into the workspace (decode)
  size_t bytes;
};

constexpr int kMaxClusterSplits = 8;  // K segments of one tile form a portable cluster

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// x_kind: the activations' type, or -1 for the most any activation type needs
// (the public size query, which takes no type).
Plan make_plan(int variant, int M, int N, int K, int gs, int x_kind) {
  Plan p{};
  const int G = K / gs;
  const int kb = K / 128;
  const int ntiles = N / 128;
  p.gemv = (M <= 16);
  p.bt = p.gemv ? 16 : (M <= 32) ? 32 : (M <= 64) ? 64 : (M <= 128) ? 128 : 256;
  const int mtiles = (M + p.bt - 1) / p.bt;
  const int tiles = ntiles * mtiles;
  // CTA slots per wave: the decode kernel and the 16/32-token tiles fit two per SM.
  const int slots = (p.bt <= 64) ? 2 * wq::kNumSMs : wq::kNumSMs;
  // As many K segments as still fit in one wave; the segments of a tile form
  // one thread-block cluster and are reduced through distributed shared memory.
  int splits = slots / tiles;
  if (splits < 1) splits = 1;
  const int max_splits = p.gemv ? wq::decode_max_splits() : kMaxClusterSplits;
  if (splits > max_splits) splits = max_splits;
  if (splits > kb) splits = kb;
  p.kb_per_split = (kb + splits - 1) / splits;
  p.splits = (kb + p.kb_per_split - 1) / p.kb_per_split;
  p.kb_first = p.kb_per_split;
  const bool corr = variant == WQ_VARIANT_W4A16 || variant == WQ_VARIANT_W4A8_ASYM;
  const bool int8x = variant == WQ_VARIANT_W4A8 || variant == WQ_VARIANT_W4A8_ASYM;
  p.kaug = (!p.gemv && corr) ? ((3 * G + 127) / 128) * 128 : 0;
  const int n_aug = p.kaug / 128;
  // Segment 0 also runs the n_aug correction stages: spread the stages (k-blocks
  // plus correction) evenly over the segments, segment 0 taking that many fewer
  // k-blocks.
  auto balance = [&](int& segs, int& kbps, int& kb_first) {
    if (segs <= 1 || n_aug == 0) return;
    const int per = (kb + n_aug + segs - 1) / segs;
    if (per - n_aug < 1) return;
    kb_first = per - n_aug;
    kbps = per;
    segs = 1 + (kb - kb_first + per - 1) / per;
  };
  if (!p.gemv) balance(p.splits, p.kb_per_split, p.kb_first);
  // Equal tiles leave the last wave partly empty: with T tiles over S CTA slots the
  // call takes ceil(T / S) tile times.  When the last wave holds at most half the
  // slots, its tiles go to a second launch, split along K so that they fill it
  // (a cluster per tile, as above), and take a fraction of a tile time.
  // Measured on this part, a K-split tile pays ~10 us more than a whole one (the
  // cluster reduction), and a partial last wave otherwise lets the next call's
  // pre-pass start on the idle SMs: the tail launch pays off only for long K
  // segments (c3's K = 17408: -3.6 %; K = 5120: +2 to +6 %), so it is used from
  // 96 k-blocks on.
  if (!p.gemv && p.splits == 1 && tiles > slots && kb >= 96) {
    const int rest = tiles % slots;
    if (rest > 0 && 2 * rest <= slots) {
      int ts = slots / rest;
      if (ts > kMaxClusterSplits) ts = kMaxClusterSplits;
      if (ts > kb) ts = kb;
      const int kbps = (kb + ts - 1) / ts;
      ts = (kb + kbps - 1) / kbps;
      if (ts > 1) {
        p.tail_tiles = rest;
        p.tail_splits = ts;
        p.tail_kbps = kbps;
        p.tail_kb_first = kbps;  // (balancing the tail's segments measured 1.5 % slower on c3)
      }
    }
  }
  size_t off = 0;
  p.off_aug = off;
  if (p.kaug) off = align256(off + static_cast<size_t>(M) * p.kaug * 2);
  p.off_daug = off;
  if (p.kaug) off = align256(off + static_cast<size_t>(N) * p.kaug * 2);
  // large M: W4A8's int8 rows as fp16, or bf16 rows as per-token scaled fp16 (+ the factors)
  const bool conv = !p.gemv && !int8x && x_kind != wq::kXF16;
  p.off_x16 = off;
  if ((int8x && !p.gemv) || conv) off = align256(off + static_cast<size_t>(M) * K * 2);
  p.off_xs = off;
  if (conv) off = align256(off + static_cast<size_t>(M) * 4);
  // decode W4A8: e4m3 activation components + per-block sums/factors row, padded: [56][K]
  // bytes (the W4A16 decode kernel reads the activations directly)
  p.off_x8 = off;
  if (p.gemv && int8x) off = align256(off + static_cast<size_t>(wq::decode_b_rows()) * K);
  p.bytes = off;
  return p;
}

// One launch of the weight-streaming decode kernel (M <= 8) on a plan from
// gemv_plan; pair: N columns of a gate/up pair weight, Y [M][N/2] = silu(gate) * up.
int launch_gemv_call(const void* X, int x_kind, const uint32_t* Bpacked, const void* S, const float* delta, void* Y,
                     int y_kind, int M, int N, int K, int gs, int splits, int kbps, bool pair, cudaStream_t st,
                     const char* name, const float* x_scale = nullptr) {
  wq::GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.group_size = gs;
  p.G = K / gs;
  p.kb_total = K / 128;
  p.kb_per_split = kbps;
  p.splits = splits;
  p.X = X;
  p.B = Bpacked;
  p.S = static_cast<const __half*>(S);
  p.delta = delta;
  p.Y = Y;
  p.y_kind = y_kind;
  p.timeout_ns = timeout_ns();
  p.weight_prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
  p.swiglu = pair ? 1 : 0;
  p.x_scale = x_scale;
  return after_launch(wq::launch_gemv(x_kind, p, st), name, st);
}

// ---------------------------------------------------------------- GEMM core
// quant_in (W4A8 variants only): X is fp16 [M][K], quantized per token by the
// activation pre-pass, which also writes x_scale (then an output).
int gemm_core(const void* X, int x_kind, const uint32_t* Bpacked, const void* S, const float* delta,
              const float* x_scale, void* Y, int y_kind, int M, int N, int K, int gs, int variant,
              void* ws, size_t ws_bytes, cudaStream_t st, const char* name, bool quant_in = false) {
  const Plan plan = make_plan(variant, M, N, K, gs, x_kind);
  if (plan.bytes > 0 && (!ws || ws_bytes < plan.bytes))
    return fail(WQ_ERR_WORKSPACE, "%s: workspace of %zu bytes given, %zu needed", name, ws_bytes, plan.bytes);
  if (ws && !aligned16(ws)) return fail(WQ_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", name);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const int G = K / gs;
  cudaError_t e;

  const bool int8x = variant == WQ_VARIANT_W4A8 || variant == WQ_VARIANT_W4A8_ASYM;
  const bool corr = delta && (variant == WQ_VARIANT_W4A16 || variant == WQ_VARIANT_W4A8_ASYM);
  if (plan.gemv && !int8x) {
    // decode W4A16: one launch, activations read directly.  Up to 8 tokens the
    // weight-streaming kernel (warp-level MMAs on register-dequantized weights)
    // takes every problem whose segment fits its shared memory; 9..16 tokens,
    // where the MMA work doubles, and the rest go to the tcgen05 decode kernel.
    int gv_splits = 0, gv_kbps = 0;
    if (wq::gemv_plan(M, N, K, gs, delta != nullptr, &gv_splits, &gv_kbps))
      return launch_gemv_call(X, x_kind, Bpacked, S, delta, Y, y_kind, M, N, K, gs, gv_splits, gv_kbps, false, st,
                              name);
    CUtensorMap tm_x, tm_s, tm_d;
    const CUtensorMapDataType xdt =
        x_kind == wq::kXBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    int rc = make_map_x3d(&tm_x, xdt, X, M, K, 16, 4);
    if (rc) return rc;
    rc = make_map(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, S, G, N, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
    if (delta) {
      rc = make_map(&tm_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, delta, G, N, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc) return rc;
    } else {
      tm_d = tm_s;  // unused
    }
    wq::GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.group_size = gs;
    p.G = G;
    p.kb_total = K / 128;
    p.kb_per_split = plan.kb_per_split;
    p.splits = plan.splits;
    p.B = Bpacked;
    p.S = static_cast<const __half*>(S);
    p.delta = delta;
    p.Y = Y;
    p.y_kind = y_kind;
    p.timeout_ns = timeout_ns();
    p.weight_prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
    e = wq::launch_decode16(x_kind, tm_x, tm_s, tm_d, p, st);
    return after_launch(e, name, st);
  }
  if (plan.gemv) {
    // decode W4A8 with at most 8 tokens: the weight-streaming kernel reads the
    // int8 rows (fp16 rows are first quantized per token into the workspace)
    // and applies the per-token scale at its store -- when its plan keeps one
    // wave of two CTAs per SM; otherwise (long K segments whose activation
    // tile does not fit) the e4m3 decode kernel below is faster
    int gv_splits = 0, gv_kbps = 0;
    if (wq::gemv_plan(M, N, K, gs, corr, &gv_splits, &gv_kbps) && (N / 128) * gv_splits <= 2 * wq::kNumSMs) {
      const void* xq = X;
      if (quant_in) {
        int8_t* x8q = reinterpret_cast<int8_t*>(wsb + plan.off_x8);  // M * K bytes <= the e4m3 rows' room
        e = wq::launch_quantize_per_token(static_cast<const __half*>(X), x8q, const_cast<float*>(x_scale), M, K, st);
        if (e != cudaSuccess) return cuda_fail(e, "per-token quantization");
        xq = x8q;
      }
      return launch_gemv_call(xq, wq::kXF16, Bpacked, S, corr ? delta : nullptr, Y, y_kind, M, N, K, gs, gv_splits,
                              gv_kbps, false, st, name, x_scale);
    }
    // decode W4A8: activation pre-pass (e4m3 components, block sums and factors), then the GEMM
    uint8_t* x8 = wsb + plan.off_x8;
    const int pk = int8x ? wq::kXI8 : x_kind;
    e = quant_in ? wq::launch_decode_prep_quant(static_cast<const __half*>(X), M, K, const_cast<float*>(x_scale), x8, st)
                 : wq::launch_decode_prep(X, pk, M, K, x_scale, x8, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode activation pre-pass");
    CUtensorMap tm_b, tm_s, tm_d;
    int rc = make_map_b3d(&tm_b, x8, wq::decode_b_rows(), K);
    if (rc) return rc;
    rc = make_map(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, S, G, N, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
    if (corr) {
      rc = make_map(&tm_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, delta, G, N, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc) return rc;
    } else {
      tm_d = tm_s;  // unused
    }
    wq::GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.group_size = gs;
    p.G = G;
    p.kb_total = K / 128;
    p.kb_per_split = plan.kb_per_split;
    p.splits = plan.splits;
    p.B = Bpacked;
    p.S = static_cast<const __half*>(S);
    p.delta = corr ? delta : nullptr;
    p.Y = Y;
    p.y_kind = y_kind;
    p.timeout_ns = timeout_ns();
    p.weight_prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
    p.x_scale = nullptr;  // folded into the pre-pass factors
    e = wq::launch_decode(tm_b, tm_s, tm_d, p, st);
    return after_launch(e, name, st);
  }

  const void* xg = X;
  if (int8x) {
    __half* x16 = reinterpret_cast<__half*>(wsb + plan.off_x16);
    e = quant_in ? wq::launch_quant_f16(static_cast<const __half*>(X), M, K, x16, const_cast<float*>(x_scale), st)
                 : wq::launch_i8_to_f16(static_cast<const int8_t*>(X), x16, static_cast<long long>(M) * K, st);
    if (e != cudaSuccess) return cuda_fail(e, "int8 -> fp16 pre-pass");
    xg = x16;
  }
  __nv_bfloat16* aug = reinterpret_cast<__nv_bfloat16*>(wsb + plan.off_aug);
  __nv_bfloat16* daug = reinterpret_cast<__nv_bfloat16*>(wsb + plan.off_daug);
  // bf16 rows: the GEMM runs on fp16 operands, reading a per-token scaled fp16
  // copy of X that the pre-pass writes, and undoes the scale in its epilogue
  const bool conv = !int8x && x_kind == wq::kXBF16;
  __half* x16c = conv ? reinterpret_cast<__half*>(wsb + plan.off_x16) : nullptr;
  float* xsc = conv ? reinterpret_cast<float*>(wsb + plan.off_xs) : nullptr;
  if (plan.kaug || conv) {
    // group sums of the activations the GEMM reads (for W4A8 the int8 rows as fp16,
    // exact; for bf16 rows the scaled fp16 copy written here)
    e = wq::launch_corr_prep(xg, x_kind, delta, M, K, N, gs, G, plan.kaug, aug, daug, x16c, xsc, st);
    if (e != cudaSuccess) return cuda_fail(e, "correction pre-pass");
  }
  int gk = x_kind;  // the GEMM's operand type
  if (conv) {
    xg = x16c;
    gk = wq::kXF16;
    x_scale = xsc;
  }

  CUtensorMap tm_x, tm_aug, tm_s, tm_d;
  const CUtensorMapDataType xdt =
      gk == wq::kXBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  int rc = make_map_x3d(&tm_x, xdt, xg, M, K, plan.bt);
  if (rc) return rc;
  if (plan.kaug) {
    rc = make_map_x3d(&tm_aug, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, aug, M, plan.kaug, plan.bt);
    if (rc) return rc;
  } else {
    tm_aug = tm_x;  // unused
  }
  // scale and delta rows: 8 group rows of 128 columns per copy (rows past G read as zero)
  rc = make_map(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, S, G, N, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc) return rc;
  if (corr) {
    rc = make_map(&tm_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, delta, G, N, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  } else {
    tm_d = tm_s;  // unused
  }

  wq::GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.group_size = gs;
  p.G = G;
  p.kb_total = K / 128;
  p.kb_per_split = plan.kb_per_split;
  p.kb_first = plan.kb_first;
  p.splits = plan.splits;
  p.aug_stages = plan.kaug / 128;
  p.kaug = plan.kaug;
  p.B = Bpacked;
  p.S = static_cast<const __half*>(S);
  p.delta = corr ? delta : nullptr;
  p.delta_aug = plan.kaug ? daug : nullptr;
  p.x_scale = x_scale;
  p.Y = Y;
  p.y_kind = y_kind;
  p.timeout_ns = timeout_ns();
  p.weight_prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
  // Y for the epilogue's tile stores: [M][N], boxes of {128 columns, 16 tokens}
  CUtensorMap tm_y;
  const CUtensorMapDataType ydt = y_kind == wq::kYF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : y_kind == wq::kYBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  rc = make_map(&tm_y, ydt, y_kind == wq::kYF32 ? 4 : 2, Y, M, N, 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc) return rc;
  const int tiles = (N / 128) * ((M + plan.bt - 1) / plan.bt);
  p.tile_base = 0;
  p.tile_count = tiles - plan.tail_tiles;
  p.tail = plan.tail_tiles > 0 ? 2 : 0;
  e = wq::launch_gemm(plan.bt, gk, tm_x, tm_aug, tm_s, tm_y, p, st);
  if (e == cudaSuccess && plan.tail_tiles > 0) {
    // the last, partial wave: its own launch, each tile split along K
    p.tile_base = p.tile_count;
    p.tile_count = plan.tail_tiles;
    p.tail = 1;
    p.splits = plan.tail_splits;
    p.kb_per_split = plan.tail_kbps;
    p.kb_first = plan.tail_kb_first;
    e = wq::launch_gemm(plan.bt, gk, tm_x, tm_aug, tm_s, tm_y, p, st);
  }
  return after_launch(e, name, st);
}

int y_kind_of(int y_dtype) {
  switch (y_dtype) {
    case WQ_DTYPE_F16: return wq::kYF16;
    case WQ_DTYPE_BF16: return wq::kYBF16;
    case WQ_DTYPE_F32: return wq::kYF32;
    default: return -1;
  }
}

}  // namespace

namespace wq {
unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

size_t gemm_workspace_bytes(int variant, int x_dtype, int M, int N, int K, int group_size) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 || N % 128) return 0;
  const int gs = (group_size == -1) ? K : group_size;
  if (gs != 128 && gs != K) return 0;
  if (variant < WQ_VARIANT_W4A16 || variant > WQ_VARIANT_W4A8_ASYM) return 0;
  return make_plan(variant, M, N, K, gs, x_dtype == WQ_DTYPE_F16 ? kXF16 : x_dtype == WQ_DTYPE_BF16 ? kXBF16 : -1)
      .bytes;
}

int set_last_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}
}  // namespace wq

extern "C" {

int wq_device_supported(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return (major == 10 && minor == 3) ? 1 : 0;
}

const char* wq_last_error(void) { return t_err; }

int wq_set_option(int option, long long value) {
  if (option == WQ_OPTION_WEIGHT_PREFETCH) {
    if (value != 0 && value != 1) return fail(WQ_ERR_INVALID_ARG, "wq_set_option: value must be 0 or 1");
    g_weight_prefetch.store(static_cast<int>(value), std::memory_order_relaxed);
    return WQ_OK;
  }
  return fail(WQ_ERR_INVALID_ARG, "wq_set_option: unknown option %d", option);
}

int wq_get_option(int option, long long* value) {
  if (!value) return fail(WQ_ERR_INVALID_ARG, "wq_get_option: null pointer");
  if (option == WQ_OPTION_WEIGHT_PREFETCH) {
    *value = g_weight_prefetch.load(std::memory_order_relaxed);
    return WQ_OK;
  }
  return fail(WQ_ERR_INVALID_ARG, "wq_get_option: unknown option %d", option);
}

const char* wq_version(void) { return "wq 0.1.0 (sm_103a, tcgen05)"; }

// Gate/up pair GEMM, output width N (the pair weight has 2N columns): the
// weight-streaming kernel with the SwiGLU epilogue when it takes the problem
// (no workspace); else the GEMM's own scratch, then the fp32 product [M][2N].
struct SwigluPlan {
  bool fused;
  int splits, kbps;
  size_t off_prod, bytes;
};

SwigluPlan make_swiglu_plan(int M, int N, int K, int gs, bool has_delta, int x_kind) {
  SwigluPlan sp{};
  const int Nc = 2 * N;
  sp.fused = wq::gemv_plan(M, Nc, K, gs, has_delta, &sp.splits, &sp.kbps, true) != 0;
  if (sp.fused) return sp;
  const int variant = has_delta ? WQ_VARIANT_W4A16 : WQ_VARIANT_W4A16_SYM;
  sp.off_prod = align256(make_plan(variant, M, Nc, K, gs, x_kind).bytes);
  sp.bytes = sp.off_prod + static_cast<size_t>(M) * Nc * 4;
  return sp;
}

size_t wq_workspace_size(int variant, int M, int N, int K, int group_size) {
  const bool pair = variant == WQ_VARIANT_W4A16_SWIGLU || variant == WQ_VARIANT_W4A16_SWIGLU_SYM;
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 || N % (pair ? 64 : 128)) return 0;
  int gs = (group_size == -1) ? K : group_size;
  if (gs != 128 && gs != K) return 0;
  if (pair) return make_swiglu_plan(M, N, K, gs, variant == WQ_VARIANT_W4A16_SWIGLU, -1).bytes;
  if (variant < WQ_VARIANT_W4A16 || variant > WQ_VARIANT_W4A8_ASYM) return 0;
  return make_plan(variant, M, N, K, gs, -1).bytes;
}

int wq_pack_w4a16_pair(const uint8_t* q_gate, const void* scale_gate, const void* zero_gate, const uint8_t* q_up,
                       const void* scale_up, const void* zero_up, uint32_t* Bpacked, void* S, float* delta, int K,
                       int N, int group_size, void* stream) {
  if (N <= 0 || N % 64) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_pack_w4a16_pair: N=%d (a multiple of 64)", N);
  int rc = check_kn(K, 2 * N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (!q_gate || !scale_gate || !zero_gate || !q_up || !scale_up || !zero_up || !Bpacked || !S || !delta)
    return fail(WQ_ERR_INVALID_ARG, "wq_pack_w4a16_pair: null pointer");
  if ((rc = check_device())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = wq::launch_pack_pair(q_gate, static_cast<const __half*>(scale_gate),
                                       static_cast<const __half*>(zero_gate), q_up,
                                       static_cast<const __half*>(scale_up), static_cast<const __half*>(zero_up),
                                       Bpacked, static_cast<__half*>(S), delta, K, N, gs, st);
  return after_launch(e, "wq_pack_w4a16_pair", st);
}

int wq_gemm_w4a16_swiglu(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S, const float* delta,
                         void* Y, int y_dtype, int M, int N, int K, int group_size, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (M < 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_gemm_w4a16_swiglu: M=%d", M);
  if (N <= 0 || N % 64) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_gemm_w4a16_swiglu: N=%d (a multiple of 64)", N);
  int rc = check_kn(K, 2 * N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (x_dtype != WQ_DTYPE_F16 && x_dtype != WQ_DTYPE_BF16)
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_swiglu: x_dtype must be F16 or BF16");
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_swiglu: bad y_dtype %d", y_dtype);
  if (M == 0) return WQ_OK;
  if (!X || !Bpacked || !S || !Y) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_swiglu: null pointer");
  if (!aligned16(X) || !aligned16(Bpacked) || !aligned16(Y) || !aligned16(S) || (delta && !aligned16(delta)))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_swiglu: X, Bpacked, S, delta and Y must be 16-byte aligned");
  const SwigluPlan sp =
      make_swiglu_plan(M, N, K, gs, delta != nullptr, x_dtype == WQ_DTYPE_BF16 ? wq::kXBF16 : wq::kXF16);
  if (sp.bytes > 0 && (!workspace || workspace_bytes < sp.bytes))
    return fail(WQ_ERR_WORKSPACE, "wq_gemm_w4a16_swiglu: workspace of %zu bytes given, %zu needed", workspace_bytes,
                sp.bytes);
  if (workspace && !aligned16(workspace))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_swiglu: workspace must be 16-byte aligned");
  if ((rc = check_device())) return rc;
  const int xk = x_dtype == WQ_DTYPE_BF16 ? wq::kXBF16 : wq::kXF16;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (sp.fused)
    return launch_gemv_call(X, xk, Bpacked, S, delta, Y, yk, M, 2 * N, K, gs, sp.splits, sp.kbps, true, st,
                            "wq_gemm_w4a16_swiglu");
  // the pair product in fp32, then the activation in one elementwise pass
  float* prod = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + sp.off_prod);
  rc = gemm_core(X, xk, Bpacked, S, delta, nullptr, prod, wq::kYF32, M, 2 * N, K, gs,
                 delta ? WQ_VARIANT_W4A16 : WQ_VARIANT_W4A16_SYM, workspace, sp.off_prod, st, "wq_gemm_w4a16_swiglu");
  if (rc) return rc;
  return after_launch(wq::launch_swiglu_pairs(prod, Y, yk, M, N, st), "wq_gemm_w4a16_swiglu", st);
}

int wq_pack_w4a16(const uint8_t* q, const void* scale, const void* zero, uint32_t* Bpacked, void* S,
                  float* delta, int K, int N, int group_size, void* stream) {
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (!q || !scale || !zero || !Bpacked || !S || !delta)
    return fail(WQ_ERR_INVALID_ARG, "wq_pack_w4a16: null pointer");
  if ((rc = check_device())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = wq::launch_pack(q, static_cast<const __half*>(scale), static_cast<const __half*>(zero), 0,
                                  Bpacked, static_cast<__half*>(S), delta, K, N, gs, st);
  return after_launch(e, "wq_pack_w4a16", st);
}

int wq_pack_w4a8(const uint8_t* q, const void* scale_signed, uint32_t* Bpacked, void* S_abs, int K, int N,
                 int group_size, void* stream) {
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (!q || !scale_signed || !Bpacked || !S_abs) return fail(WQ_ERR_INVALID_ARG, "wq_pack_w4a8: null pointer");
  if ((rc = check_device())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = wq::launch_pack(q, static_cast<const __half*>(scale_signed), nullptr, 1, Bpacked,
                                  static_cast<__half*>(S_abs), nullptr, K, N, gs, st);
  return after_launch(e, "wq_pack_w4a8", st);
}

int wq_unpack_w4(const uint32_t* Bpacked, uint8_t* q, int K, int N, void* stream) {
  int rc = check_kn(K, N);
  if (rc) return rc;
  if (!Bpacked || !q) return fail(WQ_ERR_INVALID_ARG, "wq_unpack_w4: null pointer");
  if ((rc = check_device())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return after_launch(wq::launch_unpack(Bpacked, q, K, N, st), "wq_unpack_w4", st);
}

int wq_dequant_w4(const uint32_t* Bpacked, const void* S, void* W, int w_dtype, int K, int N, int group_size,
                  void* stream) {
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (!Bpacked || !S || !W) return fail(WQ_ERR_INVALID_ARG, "wq_dequant_w4: null pointer");
  if (w_dtype != WQ_DTYPE_F16 && w_dtype != WQ_DTYPE_BF16)
    return fail(WQ_ERR_INVALID_ARG, "wq_dequant_w4: w_dtype must be F16 or BF16");
  if ((rc = check_device())) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return after_launch(wq::launch_dequant(Bpacked, static_cast<const __half*>(S), W,
                                         w_dtype == WQ_DTYPE_BF16 ? wq::kXBF16 : wq::kXF16, K, N, gs, st),
                      "wq_dequant_w4", st);
}

int wq_quantize_per_token(const void* x, int8_t* Xq, float* x_scale, int M, int K, void* stream) {
  if (M < 0 || K <= 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_quantize_per_token: M=%d K=%d", M, K);
  if (M == 0) return WQ_OK;
  if (!x || !Xq || !x_scale) return fail(WQ_ERR_INVALID_ARG, "wq_quantize_per_token: null pointer");
  int rc = check_device();
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return after_launch(wq::launch_quantize_per_token(static_cast<const __half*>(x), Xq, x_scale, M, K, st),
                      "wq_quantize_per_token", st);
}

int wq_gemm_w4a16(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S, const float* delta,
                  void* Y, int y_dtype, int M, int N, int K, int group_size, void* workspace,
                  size_t workspace_bytes, void* stream) {
  if (M < 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_gemm_w4a16: M=%d", M);
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (x_dtype != WQ_DTYPE_F16 && x_dtype != WQ_DTYPE_BF16)
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16: x_dtype must be F16 or BF16");
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16: bad y_dtype %d", y_dtype);
  if (M == 0) return WQ_OK;
  if (!X || !Bpacked || !S || !Y) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16: null pointer");
  if (!aligned16(X) || !aligned16(Bpacked) || !aligned16(Y) || !aligned16(S) || (delta && !aligned16(delta)))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16: X, Bpacked, S, delta and Y must be 16-byte aligned");
  if ((rc = check_device())) return rc;
  const int variant = delta ? WQ_VARIANT_W4A16 : WQ_VARIANT_W4A16_SYM;
  return gemm_core(X, x_dtype == WQ_DTYPE_BF16 ? wq::kXBF16 : wq::kXF16, Bpacked, S, delta, nullptr, Y, yk, M, N,
                   K, gs, variant, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                   "wq_gemm_w4a16");
}

static size_t y_elem_bytes(int y_dtype) { return y_dtype == WQ_DTYPE_F32 ? 4 : 2; }

namespace {
// The pipelined host-buffer GEMM: two copy streams and the events that order
// them against the caller's stream, per device.  Created on the first large
// call on a device (and again after its context has been rebuilt); no memory is
// allocated.
constexpr int kHostChunksMax = 4;
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t x_in[kHostChunksMax] = {}, y_ready[kHostChunksMax] = {};
};
std::mutex g_host_mu;  // held while a pipelined call is enqueued (the streams and events are shared)
HostPipe g_host_pipe[64];
wq::PerContextOnce g_host_pipe_made;

int host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "wq_gemm_w4a16_host: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(WQ_ERR_CUDA, "wq_gemm_w4a16_host: device %d", dev);
  HostPipe& hp = g_host_pipe[dev];
  if (g_host_pipe_made.needed(dev)) {
    hp = HostPipe{};
    e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming);
    for (int c = 0; c < kHostChunksMax && e == cudaSuccess; ++c) {
      e = cudaEventCreateWithFlags(&hp.x_in[c], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.y_ready[c], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(e, "wq_gemm_w4a16_host: copy streams");
    g_host_pipe_made.done(dev);
  }
  *out = &hp;
  return WQ_OK;
}
}  // namespace

size_t wq_host_workspace_size(int variant, int M, int N, int K, int group_size, int y_dtype) {
  if (variant != WQ_VARIANT_W4A16 && variant != WQ_VARIANT_W4A16_SYM) return 0;
  if (y_kind_of(y_dtype) < 0 || M <= 0 || N <= 0 || K <= 0 || K % 128 || N % 128) return 0;
  const int gs = (group_size == -1) ? K : group_size;
  if (gs != 128 && gs != K) return 0;
  return align256(static_cast<size_t>(M) * K * 2) + align256(static_cast<size_t>(M) * N * y_elem_bytes(y_dtype)) +
         make_plan(variant, M, N, K, gs, -1).bytes;
}

int wq_gemm_w4a16_host(const void* X_host, int x_dtype, const uint32_t* Bpacked, const void* S, const float* delta,
                       void* Y_host, int y_dtype, int M, int N, int K, int group_size, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (M < 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_gemm_w4a16_host: M=%d", M);
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (x_dtype != WQ_DTYPE_F16 && x_dtype != WQ_DTYPE_BF16)
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_host: x_dtype must be F16 or BF16");
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_host: bad y_dtype %d", y_dtype);
  if (M == 0) return WQ_OK;
  if (!X_host || !Bpacked || !S || !Y_host) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_host: null pointer");
  if (!aligned16(Bpacked) || !aligned16(S) || (delta && !aligned16(delta)))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_host: Bpacked, S and delta must be 16-byte aligned");
  const int variant = delta ? WQ_VARIANT_W4A16 : WQ_VARIANT_W4A16_SYM;
  const size_t x_bytes = static_cast<size_t>(M) * K * 2;
  const size_t y_bytes = static_cast<size_t>(M) * N * y_elem_bytes(y_dtype);
  const size_t need = wq_host_workspace_size(variant, M, N, K, gs, y_dtype);
  if (!workspace || workspace_bytes < need)
    return fail(WQ_ERR_WORKSPACE, "wq_gemm_w4a16_host: workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_host: workspace must be 256-byte aligned");
  if ((rc = check_device())) return rc;
  uint8_t* const ws = static_cast<uint8_t*>(workspace);
  void* const Xd = ws;
  void* const Yd = ws + align256(x_bytes);
  uint8_t* const gws = ws + align256(x_bytes) + align256(y_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int xk = x_dtype == WQ_DTYPE_BF16 ? wq::kXBF16 : wq::kXF16;
  const size_t gws_bytes = workspace_bytes - (gws - ws);
  const int chunks = (M >= 2048) ? (M / 1024 < kHostChunksMax ? M / 1024 : kHostChunksMax) : 1;
  if (chunks == 1) {
    cudaError_t e = cudaMemcpyAsync(Xd, X_host, x_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "wq_gemm_w4a16_host: copy of X to the device");
    rc = gemm_core(Xd, xk, Bpacked, S, delta, nullptr, Yd, yk, M, N, K, gs, variant, gws, gws_bytes, st,
                   "wq_gemm_w4a16_host");
    if (rc) return rc;
    e = cudaMemcpyAsync(Y_host, Yd, y_bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "wq_gemm_w4a16_host: copy of Y to the host");
    return WQ_OK;
  }
  // Large M: token-row chunks (a multiple of 256 rows) in a pipeline, so that the
  // copy of chunk c + 1's activations and of chunk c - 1's outputs overlap chunk
  // c's GEMM.  Copies in run on one internal stream, copies out on another, the
  // GEMMs on the caller's stream; events order each chunk's three steps, and the
  // caller's stream waits for the last copy out before anything enqueued after
  // this call (so Y_host is complete once that stream is synchronized).
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostPipe* hp = nullptr;
  if ((rc = host_pipe(&hp))) return rc;
  const int rows = ((M + chunks - 1) / chunks + 255) & ~255;
  const size_t ysz = y_elem_bytes(y_dtype);
  cudaError_t e = cudaEventRecord(hp->start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->start, 0);  // earlier work on st is done with Xd
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "wq_gemm_w4a16_host: stream fork");
  int c = 0;
  for (int r0 = 0; r0 < M && rc == WQ_OK; r0 += rows, ++c) {
    const int mc = (M - r0 < rows) ? M - r0 : rows;
    uint8_t* const xc = static_cast<uint8_t*>(Xd) + static_cast<size_t>(r0) * K * 2;
    uint8_t* const yc = static_cast<uint8_t*>(Yd) + static_cast<size_t>(r0) * N * ysz;
    e = cudaMemcpyAsync(xc, static_cast<const uint8_t*>(X_host) + static_cast<size_t>(r0) * K * 2,
                        static_cast<size_t>(mc) * K * 2, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->x_in[c], hp->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->x_in[c], 0);
    if (e != cudaSuccess) {
      rc = cuda_fail(e, "wq_gemm_w4a16_host: copy of X to the device");
      break;
    }
    rc = gemm_core(xc, xk, Bpacked, S, delta, nullptr, yc, yk, mc, N, K, gs, variant, gws, gws_bytes, st,
                   "wq_gemm_w4a16_host");
    if (rc) break;
    e = cudaEventRecord(hp->y_ready[c], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->y_ready[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(Y_host) + static_cast<size_t>(r0) * N * ysz, yc,
                          static_cast<size_t>(mc) * N * ysz, cudaMemcpyDeviceToHost, hp->out);
    if (e != cudaSuccess) rc = cuda_fail(e, "wq_gemm_w4a16_host: copy of Y to the host");
  }
  // join the copy streams back into the caller's stream, also after an error
  cudaError_t ej = cudaEventRecord(hp->done, hp->out);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, hp->done, 0);
  if (ej == cudaSuccess) ej = cudaEventRecord(hp->start, hp->in);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, hp->start, 0);
  if (rc) return rc;
  if (ej != cudaSuccess) return cuda_fail(ej, "wq_gemm_w4a16_host: stream join");
  return WQ_OK;
}

int wq_gemm_w4a8(const int8_t* Xq, const float* x_scale, const uint32_t* Bpacked, const void* S_abs, void* Y,
                 int y_dtype, int M, int N, int K, int group_size, void* workspace, size_t workspace_bytes,
                 void* stream) {
  if (M < 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_gemm_w4a8: M=%d", M);
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8: bad y_dtype %d", y_dtype);
  if (M == 0) return WQ_OK;
  if (!Xq || !x_scale || !Bpacked || !S_abs || !Y) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8: null pointer");
  if (!aligned16(Xq) || !aligned16(Bpacked) || !aligned16(Y) || !aligned16(S_abs))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8: Xq, Bpacked, S_abs and Y must be 16-byte aligned");
  if ((rc = check_device())) return rc;
  return gemm_core(Xq, wq::kXF16, Bpacked, S_abs, nullptr, x_scale, Y, yk, M, N, K, gs, WQ_VARIANT_W4A8,
                   workspace, workspace_bytes, static_cast<cudaStream_t>(stream), "wq_gemm_w4a8");
}

int wq_gemm_w4a16_grouped(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S, const float* delta,
                          void* Y, int y_dtype, const int* expert_offsets, int experts, int N, int K,
                          int group_size, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  if (x_dtype != WQ_DTYPE_F16 && x_dtype != WQ_DTYPE_BF16)
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: x_dtype must be F16 or BF16");
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: bad y_dtype %d", y_dtype);
  if (experts < 1 || experts > wq::kMaxExperts)
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: experts=%d (1..%d)", experts, wq::kMaxExperts);
  if (!expert_offsets) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: null expert_offsets");
  if (expert_offsets[0] != 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: expert_offsets[0] != 0");
  int max_m = 0;
  for (int e = 0; e < experts; ++e) {
    const int me = expert_offsets[e + 1] - expert_offsets[e];
    if (me < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: expert_offsets decrease at %d", e);
    max_m = me > max_m ? me : max_m;
  }
  const int M = expert_offsets[experts];
  if (M == 0) return WQ_OK;
  if (!X || !Bpacked || !S || !Y) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: null pointer");
  if (!aligned16(X) || !aligned16(Bpacked) || !aligned16(S) || !aligned16(Y) || (delta && !aligned16(delta)))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a16_grouped: X, Bpacked, S, delta and Y must be 16-byte aligned");
  const int variant = delta ? WQ_VARIANT_W4A16 : WQ_VARIANT_W4A16_SYM;
  const int G = K / gs;
  const long long b_stride = static_cast<long long>(K) * N / 8;
  const long long sd_stride = static_cast<long long>(G) * N;
  const int xk = x_dtype == WQ_DTYPE_BF16 ? wq::kXBF16 : wq::kXF16;
  const size_t ysz = (yk == wq::kYF32) ? 4 : 2;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // One launch over all experts when each has at most 8 tokens (the
  // weight-streaming kernel, one K segment per tile); else one GEMM per expert.
  int g_splits = 0, g_kbps = 0;
  if (wq::gemv_plan(max_m, N, K, gs, delta != nullptr, &g_splits, &g_kbps) &&
      wq::gemv_plan_fits(max_m, K / 128, 1, gs == K, delta != nullptr)) {
    if ((rc = check_device())) return rc;
    wq::GemmParams p{};
    p.M = max_m;
    p.N = N;
    p.K = K;
    p.group_size = gs;
    p.G = G;
    p.kb_total = K / 128;
    p.kb_per_split = K / 128;
    p.splits = 1;
    p.X = X;
    p.B = Bpacked;
    p.S = static_cast<const __half*>(S);
    p.delta = delta;
    p.Y = Y;
    p.y_kind = yk;
    p.timeout_ns = timeout_ns();
    p.weight_prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
    p.experts = experts;
    p.b_stride = b_stride;
    p.sd_stride = sd_stride;
    for (int e = 0; e <= experts; ++e) p.goff[e] = expert_offsets[e];
    return after_launch(wq::launch_gemv(xk, p, st), "wq_gemm_w4a16_grouped", st);
  }
  // every expert's workspace need is checked before anything is enqueued
  size_t need = 0;
  for (int e = 0; e < experts; ++e) {
    const int me = expert_offsets[e + 1] - expert_offsets[e];
    if (me > 0) {
      const size_t b = make_plan(variant, me, N, K, gs, xk).bytes;
      need = b > need ? b : need;
    }
  }
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(WQ_ERR_WORKSPACE, "wq_gemm_w4a16_grouped: workspace of %zu bytes given, %zu needed", workspace_bytes,
                need);
  if ((rc = check_device())) return rc;
  for (int e = 0; e < experts; ++e) {
    const int r0 = expert_offsets[e];
    const int me = expert_offsets[e + 1] - r0;
    if (me == 0) continue;
    rc = gemm_core(static_cast<const uint8_t*>(X) + static_cast<size_t>(r0) * K * 2, xk, Bpacked + e * b_stride,
                   static_cast<const __half*>(S) + e * sd_stride, delta ? delta + e * sd_stride : nullptr, nullptr,
                   static_cast<uint8_t*>(Y) + static_cast<size_t>(r0) * N * ysz, yk, me, N, K, gs, variant, workspace,
                   workspace_bytes, st, "wq_gemm_w4a16_grouped");
    if (rc) return rc;
  }
  return WQ_OK;
}

int wq_gemm_w4a8_grouped(const int8_t* Xq, const float* x_scale, const uint32_t* Bpacked, const void* S,
                         const float* delta, void* Y, int y_dtype, const int* expert_offsets, int experts, int N,
                         int K, int group_size, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_grouped: bad y_dtype %d", y_dtype);
  if (experts < 1 || experts > wq::kMaxExperts)
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_grouped: experts=%d (1..%d)", experts, wq::kMaxExperts);
  if (!expert_offsets) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_grouped: null expert_offsets");
  if (expert_offsets[0] != 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_grouped: expert_offsets[0] != 0");
  for (int e = 0; e < experts; ++e)
    if (expert_offsets[e + 1] < expert_offsets[e])
      return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_grouped: expert_offsets decrease at %d", e);
  if (expert_offsets[experts] == 0) return WQ_OK;
  if (!Xq || !x_scale || !Bpacked || !S || !Y) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_grouped: null pointer");
  if (!aligned16(Xq) || !aligned16(Bpacked) || !aligned16(S) || !aligned16(Y) || (delta && !aligned16(delta)) ||
      (reinterpret_cast<uintptr_t>(x_scale) & 3u))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_grouped: Xq, Bpacked, S, delta and Y must be 16-byte aligned, "
                                    "x_scale 4-byte aligned");
  const int variant = delta ? WQ_VARIANT_W4A8_ASYM : WQ_VARIANT_W4A8;
  const long long b_stride = static_cast<long long>(K) * N / 8;
  const long long sd_stride = static_cast<long long>(K / gs) * N;
  const size_t ysz = (yk == wq::kYF32) ? 4 : 2;
  int max_m = 0;
  for (int e = 0; e < experts; ++e) {
    const int me = expert_offsets[e + 1] - expert_offsets[e];
    max_m = me > max_m ? me : max_m;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int g_splits = 0, g_kbps = 0;
  if (wq::gemv_plan(max_m, N, K, gs, delta != nullptr, &g_splits, &g_kbps) &&
      wq::gemv_plan_fits(max_m, K / 128, 1, gs == K, delta != nullptr)) {
    // every expert has at most 8 tokens: one weight-streaming launch over all
    // experts reads the int8 rows and applies the per-token scale at its store
    if ((rc = check_device())) return rc;
    wq::GemmParams p{};
    p.M = max_m;
    p.N = N;
    p.K = K;
    p.group_size = gs;
    p.G = K / gs;
    p.kb_total = K / 128;
    p.kb_per_split = K / 128;
    p.splits = 1;
    p.X = Xq;
    p.B = Bpacked;
    p.S = static_cast<const __half*>(S);
    p.delta = delta;
    p.x_scale = x_scale;
    p.Y = Y;
    p.y_kind = yk;
    p.timeout_ns = timeout_ns();
    p.weight_prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
    p.experts = experts;
    p.b_stride = b_stride;
    p.sd_stride = sd_stride;
    for (int i = 0; i <= experts; ++i) p.goff[i] = expert_offsets[i];
    return after_launch(wq::launch_gemv(wq::kXF16, p, st), "wq_gemm_w4a8_grouped", st);
  }
  // every expert's workspace need is checked before anything is enqueued
  size_t need = 0;
  for (int e = 0; e < experts; ++e) {
    const int me = expert_offsets[e + 1] - expert_offsets[e];
    if (me > 0) {
      const size_t b = make_plan(variant, me, N, K, gs, -1).bytes;
      need = b > need ? b : need;
    }
  }
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(WQ_ERR_WORKSPACE, "wq_gemm_w4a8_grouped: workspace of %zu bytes given, %zu needed", workspace_bytes,
                need);
  if ((rc = check_device())) return rc;
  for (int e = 0; e < experts; ++e) {
    const int r0 = expert_offsets[e];
    const int me = expert_offsets[e + 1] - r0;
    if (me == 0) continue;
    rc = gemm_core(Xq + static_cast<size_t>(r0) * K, wq::kXF16, Bpacked + e * b_stride,
                   static_cast<const __half*>(S) + e * sd_stride, delta ? delta + e * sd_stride : nullptr,
                   x_scale + r0, static_cast<uint8_t*>(Y) + static_cast<size_t>(r0) * N * ysz, yk, me, N, K, gs,
                   variant, workspace, workspace_bytes, st, "wq_gemm_w4a8_grouped");
    if (rc) return rc;
  }
  return WQ_OK;
}

int wq_gemm_w4a8_asym(const int8_t* Xq, const float* x_scale, const uint32_t* Bpacked, const void* S,
                      const float* delta, void* Y, int y_dtype, int M, int N, int K, int group_size,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_gemm_w4a8_asym: M=%d", M);
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_asym: bad y_dtype %d", y_dtype);
  if (M == 0) return WQ_OK;
  if (!Xq || !x_scale || !Bpacked || !S || !Y) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_asym: null pointer");
  if (!aligned16(Xq) || !aligned16(Bpacked) || !aligned16(Y) || !aligned16(S) || (delta && !aligned16(delta)))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_asym: Xq, Bpacked, S, delta and Y must be 16-byte aligned");
  if ((rc = check_device())) return rc;
  return gemm_core(Xq, wq::kXF16, Bpacked, S, delta, x_scale, Y, yk, M, N, K, gs,
                   delta ? WQ_VARIANT_W4A8_ASYM : WQ_VARIANT_W4A8, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), "wq_gemm_w4a8_asym");
}

int wq_gemm_w4a8_fp16(const void* X, const uint32_t* Bpacked, const void* S, const float* delta, float* x_scale,
                      void* Y, int y_dtype, int M, int N, int K, int group_size, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (M < 0) return fail(WQ_ERR_UNSUPPORTED_SHAPE, "wq_gemm_w4a8_fp16: M=%d", M);
  int rc = check_kn(K, N);
  if (rc) return rc;
  int gs;
  if ((rc = norm_group(K, group_size, &gs))) return rc;
  const int yk = y_kind_of(y_dtype);
  if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_fp16: bad y_dtype %d", y_dtype);
  if (M == 0) return WQ_OK;
  if (!X || !x_scale || !Bpacked || !S || !Y) return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_fp16: null pointer");
  if (!aligned16(X) || !aligned16(Bpacked) || !aligned16(Y) || !aligned16(S) || (delta && !aligned16(delta)) ||
      (reinterpret_cast<uintptr_t>(x_scale) & 3u))
    return fail(WQ_ERR_INVALID_ARG, "wq_gemm_w4a8_fp16: X, Bpacked, S, delta and Y must be 16-byte aligned, "
                                    "x_scale 4-byte aligned");
  if ((rc = check_device())) return rc;
  return gemm_core(X, wq::kXF16, Bpacked, S, delta, x_scale, Y, yk, M, N, K, gs,
                   delta ? WQ_VARIANT_W4A8_ASYM : WQ_VARIANT_W4A8, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), "wq_gemm_w4a8_fp16", true);
}

int wq_device_status(unsigned int* status, int reset, void* stream) {
  if (!status) return fail(WQ_ERR_INVALID_ARG, "wq_device_status: null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "wq_device_status");
  e = wq::read_status(status);
  if (e != cudaSuccess) return cuda_fail(e, "wq_device_status");
  if (reset) {
    e = wq::clear_status();
    if (e != cudaSuccess) return cuda_fail(e, "wq_device_status");
  }
  return *status ? fail(WQ_ERR_TIMEOUT, "device status 0x%x", *status) : WQ_OK;
}

int wq_debug_wait_probe(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(WQ_ERR_INVALID_ARG, "wq_debug_wait_probe: limit must be in (0, 10 s]");
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = wq::launch_wait_probe(limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wq_debug_wait_probe");
  return WQ_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- persistent decode chain
namespace {

// Checks a chain's arguments (pointers only when check_ptrs) and fills the
// host-given fields of p; nothing here touches the device.
int chain_args(const wq_chain_gemm* gemms, int n, int M, int x_dtype, wq::ChainParams* p, bool check_ptrs,
               const char* name) {
  if (!gemms || n < 1 || n > wq::kChainMaxGemms)
    return fail(WQ_ERR_INVALID_ARG, "%s: n=%d (a list of 1..%d GEMMs)", name, n, wq::kChainMaxGemms);
  if (M < 0 || M > wq::kChainMaxM)
    return fail(WQ_ERR_UNSUPPORTED_SHAPE, "%s: M=%d (at most %d token rows)", name, M, wq::kChainMaxM);
  if (x_dtype != WQ_DTYPE_F16 && x_dtype != WQ_DTYPE_BF16)
    return fail(WQ_ERR_INVALID_ARG, "%s: x_dtype must be F16 or BF16", name);
  memset(p, 0, sizeof(*p));
  p->n = n;
  p->M = M;
  for (int i = 0; i < n; ++i) {
    const wq_chain_gemm& s = gemms[i];
    if (s.pair != 0 && s.pair != 1) return fail(WQ_ERR_INVALID_ARG, "%s: GEMM %d: pair must be 0 or 1", name, i);
    if (s.pair && (s.N <= 0 || s.N % 64))
      return fail(WQ_ERR_UNSUPPORTED_SHAPE, "%s: GEMM %d: N=%d (a multiple of 64 for a pair)", name, i, s.N);
    const int ncols = s.pair ? 2 * s.N : s.N;
    int rc = check_kn(s.K, ncols);
    if (rc) return rc;
    int gs;
    if ((rc = norm_group(s.K, s.group_size, &gs))) return rc;
    const int yk = y_kind_of(s.y_dtype);
    if (yk < 0) return fail(WQ_ERR_INVALID_ARG, "%s: GEMM %d: bad y_dtype %d", name, i, s.y_dtype);
    if (static_cast<long long>(ncols / 128) * (s.K / 128) >= (1ll << 31))
      return fail(WQ_ERR_UNSUPPORTED_SHAPE, "%s: GEMM %d: too many k-blocks", name, i);
    if (s.src < -1 || s.src >= i)
      return fail(WQ_ERR_INVALID_ARG, "%s: GEMM %d: src=%d (-1 or an earlier GEMM)", name, i, s.src);
    const void* X = s.X;
    if (s.src >= 0) {
      const wq_chain_gemm& q = gemms[s.src];
      if (q.N != s.K)
        return fail(WQ_ERR_UNSUPPORTED_SHAPE, "%s: GEMM %d: K=%d differs from the output width %d of GEMM %d", name,
                    i, s.K, q.N, s.src);
      if (q.y_dtype != x_dtype)
        return fail(WQ_ERR_INVALID_ARG, "%s: GEMM %d reads GEMM %d's Y, whose y_dtype is not x_dtype", name, i,
                    s.src);
      if (s.X && s.X != q.Y)
        return fail(WQ_ERR_INVALID_ARG, "%s: GEMM %d: X must be NULL or GEMM %d's Y", name, i, s.src);
      X = q.Y;
    }
    if (check_ptrs) {
      if (!X || !s.Bpacked || !s.S || !s.Y) return fail(WQ_ERR_INVALID_ARG, "%s: GEMM %d: null pointer", name, i);
      if (!aligned16(X) || !aligned16(s.Bpacked) || !aligned16(s.S) || !aligned16(s.Y) ||
          (s.delta && !aligned16(s.delta)))
        return fail(WQ_ERR_INVALID_ARG, "%s: GEMM %d: X, Bpacked, S, delta and Y must be 16-byte aligned", name, i);
    }
    wq::ChainGemm& G = p->g[i];
    G.X = X;
    G.B = s.Bpacked;
    G.S = static_cast<const __half*>(s.S);
    G.delta = s.delta;
    G.Y = s.Y;
    G.y_kind = yk;
    G.N = ncols;
    G.K = s.K;
    G.per_channel = gs == s.K ? 1 : 0;
    G.pair = s.pair;
    G.src = s.src;
  }
  return WQ_OK;
}

int x_kind_of(int x_dtype) { return x_dtype == WQ_DTYPE_BF16 ? wq::kXBF16 : wq::kXF16; }

}  // namespace

size_t wq_chain_workspace_size(const wq_chain_gemm* gemms, int n, int M, int x_dtype) {
  wq::ChainParams p;
  if (chain_args(gemms, n, M, x_dtype, &p, false, "wq_chain_workspace_size") || M == 0) return 0;
  if (check_device()) return 0;
  wq::ChainGeom geo;
  if (wq::chain_geometry(x_kind_of(x_dtype), M, &geo) != cudaSuccess) return 0;
  return wq::chain_plan(p, geo);
}

int wq_gemm_w4a16_chain(const wq_chain_gemm* gemms, int n, int M, int x_dtype, void* workspace,
                        size_t workspace_bytes, void* stream) {
  static const char* name = "wq_gemm_w4a16_chain";
  wq::ChainParams p;
  int rc = chain_args(gemms, n, M, x_dtype, &p, true, name);
  if (rc) return rc;
  if (M == 0) return WQ_OK;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(WQ_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", name);
  if ((rc = check_device())) return rc;
  wq::ChainGeom geo;
  cudaError_t e = wq::chain_geometry(x_kind_of(x_dtype), M, &geo);
  if (e != cudaSuccess) return cuda_fail(e, name);
  const size_t need = wq::chain_plan(p, geo);
  if (need == 0)
    return fail(WQ_ERR_UNSUPPORTED_SHAPE, "%s: more than %d output tiles of 128 columns in one chain", name,
                wq::kChainMaxTiles);
  if (!workspace || workspace_bytes < need)
    return fail(WQ_ERR_WORKSPACE, "%s: workspace of %zu bytes given, %zu needed", name, workspace_bytes, need);
  wq::chain_bind_workspace(p, workspace);
  p.timeout_ns = timeout_ns();
  p.weight_prefetch = g_weight_prefetch.load(std::memory_order_relaxed);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return after_launch(wq::launch_chain(x_kind_of(x_dtype), p, geo, st), name, st);
}
