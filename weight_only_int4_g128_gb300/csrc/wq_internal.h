// wq_internal.h -- declarations shared by the library's translation units
// (not part of the public C ABI; see include/wq.h for that).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace wq {

constexpr int kTileN = 128;        // weight rows (output columns) per CTA = MMA M
constexpr int kKBlock = 128;       // K elements per pipeline stage
constexpr int kWordsPerKBlock = kKBlock / 8;
constexpr int kNumSMs = 152;
constexpr int kMaxExperts = 64;    // experts of one grouped GEMM call

// Status bits written by kernels into the device status word.
constexpr unsigned kDevTimeoutProducer = 1u << 0;
constexpr unsigned kDevTimeoutMma = 1u << 1;
constexpr unsigned kDevTimeoutMath = 1u << 2;
constexpr unsigned kDevTimeoutFixup = 1u << 3;
constexpr unsigned kDevTimeoutProbe = 1u << 4;

enum XKind { kXF16 = 0, kXBF16 = 1, kXI8 = 2 };
enum YKind { kYF16 = 0, kYBF16 = 1, kYF32 = 2 };


struct GemmParams {
  int M, N, K;
  int group_size;        // K for one group per column
  int G;                 // number of groups
  int kb_total;          // K / 128
  int kb_per_split;      // k-blocks per split segment
  int kb_first;          // large-M kernel: k-blocks of segment 0, which also runs the
                         // correction stages (0: kb_per_split like the others)
  int splits;            // number of K segments (one thread-block cluster per tile)
  int aug_stages;        // correction stages (Kaug / 128), 0 when there is no correction
  int kaug;              // padded correction length (multiple of 128)
  const void* X;         // [M][K] activations (weight-streaming decode kernel)
  const uint32_t* B;     // packed weights, blocked layout (one 8 KB block per tile, k-block)
  const __half* S;       // [G][N] group scales
  const float* delta;    // [G][N] zero-point residual, or null
  const __nv_bfloat16* delta_aug;  // [N][kaug] correction columns (large-M kernel)
  const float* x_scale;  // [M] per-token activation scale (W4A8), or null
  void* Y;               // [M][N]
  int y_kind;
  unsigned long long timeout_ns;
  int weight_prefetch;   // issue weight copies before waiting on the preceding grid
  // Large-M kernel: this launch covers tiles [tile_base, tile_base + gridDim.x) of
  // the (column tile fastest) tile order.  tail = 1: the launch finishes the last,
  // partial wave of tiles of the launch just before it on the stream (same call,
  // split along K): it starts without waiting for that launch, which (tail = 2) let
  // it start only after the call's pre-pass had completed, and waits for it before
  // exiting.
  int tile_base;
  int tile_count;  // tiles of a main launch (0: all of them); a tail launch takes the rest
  int tail;
  // Grouped (mixture-of-experts) launch of the weight-streaming decode kernel:
  // blockIdx.z = expert e, whose token rows are goff[e] .. goff[e+1] of X and Y
  // and whose weights sit b_stride words / sd_stride elements after expert 0's.
  // experts == 0: a plain GEMM.
  int experts;
  long long b_stride, sd_stride;
  int goff[kMaxExperts + 1];
  // Gate/up pair (weight-streaming decode kernel): the N columns are the
  // pair-interleaved gate and up projections (each 16-column group: 8 gate
  // columns, then the same 8 up columns) and Y is [M][N/2] = silu(gate) * up.
  int swiglu;
};

// Identifier of the calling thread's current CUDA context, unique for the life
// of the process (the context a device gets after cudaDeviceReset has a new
// one); 0 when no context is current yet or the driver cannot tell.
unsigned long long current_context_id();
// Workspace bytes of one GEMM call with activations of x_dtype (WQ_DTYPE_*):
// wq_workspace_size() returns the most over the activation types.
size_t gemm_workspace_bytes(int variant, int x_dtype, int M, int N, int K, int group_size);

// A per-device set-up step (a kernel attribute, a device symbol's address)
// that has to be redone when the device's context is rebuilt, e.g. after
// cudaDeviceReset.  Concurrent callers may both redo the step; that is harmless.
struct PerContextOnce {
  unsigned long long ctx[64] = {};
  bool needed(int dev) const {
    const unsigned long long id = current_context_id();
    return dev < 0 || dev >= 64 || id == 0 || ctx[dev] != id;
  }
  void done(int dev) {
    if (dev >= 0 && dev < 64) ctx[dev] = current_context_id();
  }
};

// Record the message for wq_last_error() on this thread and return `code`.
int set_last_error(int code, const char* fmt, ...);

// Host-side launchers (wq_gemm.cu, wq_decode.cu).
cudaError_t launch_decode_prep(const void* X, int x_kind, int M, int K, const float* x_scale, uint8_t* X8,
                               cudaStream_t stream);
cudaError_t launch_decode_prep_quant(const __half* X, int M, int K, float* x_scale, uint8_t* X8,
                                     cudaStream_t stream);
cudaError_t launch_quant_f16(const __half* X, int M, int K, __half* X16, float* x_scale, cudaStream_t stream);
cudaError_t launch_decode(const CUtensorMap& tm_b, const CUtensorMap& tm_s, const CUtensorMap& tm_d,
                          const GemmParams& p, cudaStream_t stream);
int decode_max_splits();
cudaError_t launch_decode16(int x_kind, const CUtensorMap& tm_x, const CUtensorMap& tm_s, const CUtensorMap& tm_d,
                            const GemmParams& p, cudaStream_t stream);
int decode16_max_splits();
cudaError_t launch_gemv(int x_kind, const GemmParams& p, cudaStream_t stream);
// pair: a gate/up pair weight (SwiGLU epilogue), whose split-K ownership is rounded to 16 rows
int gemv_plan(int M, int N, int K, int group_size, bool has_delta, int* splits, int* kb_per_split,
              bool pair = false);
bool gemv_plan_fits(int M, int kbps, int splits, bool per_channel, bool has_delta, bool pair = false);
int decode_b_rows();  // rows of the activation-component tensor (3 x 16 components + sums/factors)
unsigned* status_word();
// tm_y: Y [M][N] with boxes of {128 columns, 16 tokens} (the epilogue's TMA stores).
cudaError_t launch_gemm(int bt, int x_kind, const CUtensorMap& tm_x, const CUtensorMap& tm_aug,
                        const CUtensorMap& tm_s, const CUtensorMap& tm_y, const GemmParams& p, cudaStream_t stream);
size_t gemm_smem_bytes(int bt);

// Pre-pass kernels (wq_kernels.cu).
// Correction columns (kaug > 0) and, for bf16 X (x_kind == kXBF16), the per-token
// scaled fp16 copy x16 [M][K] with its factors xs [M] that the GEMM reads instead.
cudaError_t launch_corr_prep(const void* X, int x_kind, const float* delta, int M, int K, int N, int group_size,
                             int G, int kaug, __nv_bfloat16* aug, __nv_bfloat16* delta_aug, __half* x16, float* xs,
                             cudaStream_t stream);
cudaError_t launch_i8_to_f16(const int8_t* Xq, __half* X16, long long count, cudaStream_t stream);
cudaError_t launch_pack_pair(const uint8_t* q_gate, const __half* scale_gate, const __half* zero_gate,
                             const uint8_t* q_up, const __half* scale_up, const __half* zero_up, uint32_t* Bpacked,
                             __half* S, float* delta, int K, int N, int group_size, cudaStream_t stream);
cudaError_t launch_swiglu_pairs(const float* Yc, void* Y, int y_kind, int M, int N, cudaStream_t stream);
cudaError_t launch_pack(const uint8_t* q, const __half* scale, const __half* zero, int fold,
                        uint32_t* Bpacked, __half* S, float* delta, int K, int N, int group_size,
                        cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t* Bpacked, uint8_t* q, int K, int N, cudaStream_t stream);
cudaError_t launch_dequant(const uint32_t* Bpacked, const __half* S, void* W, int w_kind, int K,
                           int N, int group_size, cudaStream_t stream);
cudaError_t launch_quantize_per_token(const __half* x, int8_t* Xq, float* x_scale, int M, int K,
                                      cudaStream_t stream);
cudaError_t launch_wait_probe(unsigned long long limit_ns, cudaStream_t stream);
cudaError_t read_status(unsigned int* out);
cudaError_t clear_status();

}  // namespace wq
