/*
 * wq.h -- C ABI of the GB300 (sm_103a) group-quantized INT4-weight GEMM
 * library (libwq.so).
 *
 * The operation ("Marlin INT4 on Ada -- how it works", TinyLoop docs, section
 * "The core mismatch: symmetric vs asymmetric"):
 *
 *   asymmetric weight    W[k][n]     = q[k][n] * scale[g][n] + zero[g][n]
 *   symmetric weight     W_sym[k][n] = (q[k][n] - 8) * scale[g][n]
 *   residual             delta[g][n] = zero[g][n] + 8 * scale[g][n]
 *   product              Y = X @ W = X @ W_sym + A_group_sum @ delta
 *                        A_group_sum[m][g] = sum over k in group g of X[m][k]
 *
 * with codes q in [0, 15], g = k / group_size, and group_size = K meaning one
 * group per column (section "How the dispatcher chooses").  The W4A8 entry
 * follows the HyperQwen W4A8 article (kwkr.cn): activations quantized per
 * token to int8, weights with signed fp16 group scales folded at pack time
 * (section "hidden mine: the negative group scale bug").
 *
 * Conventions for every entry point:
 *  - Pointers named as device buffers must be device memory of the current
 *    CUDA device; the caller allocates and owns every buffer.  The library
 *    never allocates, frees or synchronizes (unless WQ_CHECKED=1 is set in
 *    the environment, which adds a stream synchronize and a device-status
 *    check after each launch).
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Work is enqueued asynchronously on it.
 *  - Return value: WQ_OK or one of the WQ_ERR_* codes below; on error no work
 *    has been enqueued (except WQ_ERR_CUDA / WQ_ERR_TIMEOUT, which report a
 *    failure of work already enqueued) and wq_last_error() describes it.
 *  - Shapes: K and N multiples of 128 (the kernel tile; the same rule as the
 *    pages' Marlin preconditions), M >= 0 (M == 0 is a no-op), group_size 128
 *    or K (-1 is accepted as K).  Other shapes return WQ_ERR_UNSUPPORTED_SHAPE.
 *  - Device pointers that a kernel reads with TMA or vector loads must be
 *    16-byte aligned: X, Xq, Bpacked, S, delta, Y, the workspace.  Otherwise
 *    WQ_ERR_INVALID_ARG.
 *  - Only sm_103 devices are supported (WQ_ERR_ARCH otherwise).
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define WQ_OK 0
#define WQ_ERR_INVALID_ARG 1       /* null or misaligned pointer, bad dtype, negative size */
#define WQ_ERR_UNSUPPORTED_SHAPE 2 /* K or N not a multiple of 128, bad group size */
#define WQ_ERR_WORKSPACE 3         /* workspace missing or smaller than wq_workspace_size() */
#define WQ_ERR_ARCH 4              /* current device is not sm_103 */
#define WQ_ERR_CUDA 5              /* a CUDA runtime call or launch failed */
#define WQ_ERR_TIMEOUT 6           /* a bounded device-side wait expired (checked mode) */

/* element types */
#define WQ_DTYPE_F16 0
#define WQ_DTYPE_BF16 1
#define WQ_DTYPE_F32 2

/* options for wq_set_option / wq_get_option */
#define WQ_OPTION_WEIGHT_PREFETCH 1 /* 0 (default) or 1, see wq_set_option */

/* workspace variants for wq_workspace_size */
#define WQ_VARIANT_W4A16 0      /* wq_gemm_w4a16 with delta (asymmetric) */
#define WQ_VARIANT_W4A16_SYM 1  /* wq_gemm_w4a16 with delta == NULL */
#define WQ_VARIANT_W4A8 2       /* wq_gemm_w4a8 */
#define WQ_VARIANT_W4A8_ASYM 3  /* wq_gemm_w4a8_asym with delta (zero-point weights) */
#define WQ_VARIANT_W4A16_SWIGLU 4      /* wq_gemm_w4a16_swiglu with delta; N = output width */
#define WQ_VARIANT_W4A16_SWIGLU_SYM 5  /* wq_gemm_w4a16_swiglu with delta == NULL */

/*
 * Load-time pack of asymmetric W4A16 weights ("Marlin INT4 on Ada", section
 * "The pipeline, end to end": codes packed 8 x int4 per uint32, and
 * delta = zero + 8 * scale per group and column).
 *   q        [K][N] uint8 device, one code 0..15 per byte (row k, column n).
 *   scale    [G][N] fp16 device, G = K / group_size.
 *   zero     [G][N] fp16 device.
 *   Bpacked  K*N/8 uint32 device, output, in this library's blocked layout:
 *            the word for column n and codes k = 8w..8w+7 holds q[8w + j][n],
 *            code j in bits [4*(j/2) + 16*(j%2), +4); words are grouped in
 *            blocks of 128 columns x 128 k (2048 words), block index
 *            (n/128)*(K/128) + 8w/128, and inside a block row r = n%128 holds
 *            its 16 words as four 16-byte chunks, chunk c = (w%16)/4 stored at
 *            word offset r*16 + 4*(c ^ ((r/2)%4)) + w%4.  Each block is the
 *            weight tile one GEMM pipeline stage copies in a single transfer.
 *   S        [G][N] fp16 device, output: a copy of scale.
 *   delta    [G][N] fp32 device, output: fp32(zero) + 8*fp32(scale), rounded
 *            once (exact for operands of similar magnitude).
 * Codes outside 0..15 are reduced to their low 4 bits.
 */
int wq_pack_w4a16(const uint8_t* q, const void* scale, const void* zero, uint32_t* Bpacked,
                  void* S, float* delta, int K, int N, int group_size, void* stream);

/*
 * Load-time pack of W4A8 weights with signed group scales (HyperQwen article,
 * section "hidden mine"): for every (g, n) with scale < 0, scale -> -scale and
 * each code v of the group -> min(16 - v, 15).  Exact except the code v = 0
 * (value -8), which becomes +7 instead of +8.
 *   q             [K][N] uint8 device, uint4b8 codes (value = v - 8).
 *   scale_signed  [G][N] fp16 device.
 *   Bpacked       K*N/8 uint32 device, output (layout as wq_pack_w4a16).
 *   S_abs         [G][N] fp16 device, output: the folded (non-negative) scales.
 */
int wq_pack_w4a8(const uint8_t* q, const void* scale_signed, uint32_t* Bpacked, void* S_abs,
                 int K, int N, int group_size, void* stream);

/*
 * Load-time pack of a gate/up projection pair for the fused SwiGLU GEMM
 * ("Marlin INT4 on Ada", section "Gaps and follow-ups": the fused SwiGLU
 * dispatch runs mlp_gate and mlp_up in one kernel).  The two asymmetric
 * [K][N] weights become one [K][2N] weight packed as wq_pack_w4a16 packs it,
 * with the columns interleaved in groups of 16: combined columns 16i .. 16i+7
 * are gate columns 8i .. 8i+7 and combined columns 16i+8 .. 16i+15 the same up
 * columns.  S and delta follow the same column order.
 *   q_gate, q_up           [K][N] uint8 device codes 0..15.
 *   scale_gate, zero_gate, scale_up, zero_up   [G][N] fp16 device.
 *   Bpacked                K*2N/8 uint32 device, output.
 *   S, delta               [G][2N] fp16 / fp32 device, outputs.
 * N must be a multiple of 64 (so that 2N is a multiple of 128), else
 * WQ_ERR_UNSUPPORTED_SHAPE.
 */
int wq_pack_w4a16_pair(const uint8_t* q_gate, const void* scale_gate, const void* zero_gate, const uint8_t* q_up,
                       const void* scale_up, const void* zero_up, uint32_t* Bpacked, void* S, float* delta, int K,
                       int N, int group_size, void* stream);

/* Inverse of the packing: Bpacked (blocked layout) -> q [K][N] uint8 codes. */
int wq_unpack_w4(const uint32_t* Bpacked, uint8_t* q, int K, int N, void* stream);

/*
 * Dequantized symmetric weights: W[k][n] = RN((q - 8) * S[g][n]) rounded once to
 * w_dtype (WQ_DTYPE_F16 or WQ_DTYPE_BF16).  With WQ_DTYPE_F16 these are the
 * values the large-M GEMM feeds to the tensor cores, for fp16 and bf16
 * activations alike; WQ_DTYPE_BF16 gives the same product rounded to bf16.
 * W is [K][N] device, output.
 */
int wq_dequant_w4(const uint32_t* Bpacked, const void* S, void* W, int w_dtype, int K, int N,
                  int group_size, void* stream);

/*
 * W4A16 GEMM with the fused zero-point correction:
 *   Y[m][n] = sum_k X[m][k] * W_sym[k][n] + (A_group_sum @ delta)[m][n]
 *   X        [M][K] device, fp16 or bf16 (x_dtype), row-major.
 *   Bpacked  K*N/8 uint32 device (from wq_pack_w4a16).
 *   S        [G][N] fp16 device.
 *   delta    [G][N] fp32 device, or NULL for symmetric weights (no correction).
 *   Y        [M][N] device, output, overwritten (y_dtype F16, BF16 or F32).
 *   workspace / workspace_bytes: device scratch of at least
 *            wq_workspace_size(variant, M, N, K, group_size) bytes (may be NULL
 *            when that is 0; it is 0 for W4A16 with M <= 16).  No
 *            initialization is needed.  Calls that may run concurrently must
 *            use different workspaces.
 * Accumulation is fp32.  The weights are dequantized as RN((q-8)*scale) in
 * fp16 for M > 16 (in the activation type's exact offset form with the scale
 * applied in fp32 per 128-k block for M <= 16); the correction is added in
 * the same accumulator.  bf16 activations with M > 16 are first copied into
 * the workspace as fp16 after a per-token power-of-two scale (exact: fp16
 * holds every bf16 significand in range), which the GEMM undoes exactly at its
 * store, so large-M bf16 calls keep fp16's 11-bit weights.
 */
int wq_gemm_w4a16(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S,
                  const float* delta, void* Y, int y_dtype, int M, int N, int K, int group_size,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * W4A8 GEMM (symmetric, folded weights):
 *   Y[m][n] = x_scale[m] * sum_k Xq[m][k] * (q[k][n] - 8) * S_abs[g][n]
 *   Xq       [M][K] int8 device (per-token quantized activations).
 *   x_scale  [M] fp32 device.
 *   Bpacked, S_abs from wq_pack_w4a8.  Other arguments as wq_gemm_w4a16.
 * sm_103a has no int8 tcgen05 MMA, so the int8 activations and the
 * (q - 8) * scale weights are fed to the fp16 tensor-core path; int8 values
 * are exact in fp16.
 */
int wq_gemm_w4a8(const int8_t* Xq, const float* x_scale, const uint32_t* Bpacked,
                 const void* S_abs, void* Y, int y_dtype, int M, int N, int K, int group_size,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Fused SwiGLU pair GEMM on a wq_pack_w4a16_pair weight:
 *   Y[m][n] = silu(G[m][n]) * U[m][n],  silu(g) = g / (1 + exp(-g)),
 * with G = X @ W_gate and U = X @ W_up the W4A16 products of wq_gemm_w4a16
 * (zero-point correction included when delta is given; delta NULL gives the
 * symmetric weights (q - 8) * scale).  Both products and the activation are
 * in fp32; Y is rounded once to y_dtype.
 *   X        [M][K] fp16/bf16 device.
 *   Bpacked, S, delta: from wq_pack_w4a16_pair (2N columns).
 *   Y        [M][N] device.
 *   N        the width of each projection (a multiple of 64, else
 *            WQ_ERR_UNSUPPORTED_SHAPE).
 *   workspace  wq_workspace_size(WQ_VARIANT_W4A16_SWIGLU (delta given) or
 *            WQ_VARIANT_W4A16_SWIGLU_SYM, M, N, K, group_size) bytes: 0 when
 *            M <= 8 and the weight-streaming kernel takes the problem (one
 *            launch, the activation in its epilogue); otherwise the GEMM's
 *            scratch plus the fp32 pair product [M][2N], activated by one
 *            elementwise launch after the GEMM.
 */
int wq_gemm_w4a16_swiglu(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S, const float* delta,
                         void* Y, int y_dtype, int M, int N, int K, int group_size, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Persistent decode chain: a list of W4A16 GEMMs over the same M <= 8 token
 * rows, run by ONE cooperative launch, in which a GEMM may take an earlier
 * GEMM's output as its activations (a decode layer's MLP: the gate/up pair with
 * SwiGLU, then the down projection).  Each GEMM computes what wq_gemm_w4a16
 * (pair == 0) or wq_gemm_w4a16_swiglu (pair == 1) computes ("Marlin INT4 on
 * Ada -- how it works", section "The core mismatch": Y = X @ W_sym +
 * A_group_sum @ delta, fp32 accumulation, Y rounded once to y_dtype); the
 * launch-latency floor of small-batch decode (section "Gaps and follow-ups" of
 * the same page) is paid once per list instead of once per GEMM.  The k-blocks
 * of every GEMM are shared evenly by all CTAs (stream-K ranges); a tile shared
 * by several CTAs is summed in a fixed order, so repeated calls give bitwise
 * identical results.  A GEMM that reads an earlier output starts each part of
 * its work once the producer tiles it reads are stored; its weights stream in
 * before that.
 *   gemms[i].X       [M][K] device activations of x_dtype (F16 or BF16); NULL
 *                    or gemms[src].Y when src >= 0.
 *   gemms[i].src     -1, or the index (< i) of the GEMM whose Y is this X: that
 *                    GEMM's output width N must equal this K and its y_dtype must
 *                    be x_dtype.
 *   Bpacked, S, delta  from wq_pack_w4a16 (pair 0) or wq_pack_w4a16_pair
 *                    (pair 1); delta NULL: symmetric weights.
 *   Y, y_dtype       [M][N] device output (F16, BF16 or F32).  Outputs must not
 *                    overlap one another or any input.
 *   N, K, group_size N the output width (pair: each projection's width, a
 *                    multiple of 64; otherwise a multiple of 128); K a multiple
 *                    of 128; group_size 128 or K (-1).
 *   n                1..8 GEMMs with at most 65536 output tiles of 128 columns
 *                    in all (pair: 2N columns).  M: 1..8 token rows (0: no-op;
 *                    larger M goes to the single-GEMM entries,
 *                    WQ_ERR_UNSUPPORTED_SHAPE here).
 *   workspace        wq_chain_workspace_size(gemms, n, M, x_dtype) bytes of
 *                    device memory, 256-byte aligned, ZEROED once before its
 *                    first use and then passed unchanged to later calls: each
 *                    call leaves its counters and control words as the next
 *                    call needs them, and any chain may reuse a workspace large
 *                    enough for it.  Calls that share a workspace must not run
 *                    at the same time (different streams).  After a call that
 *                    reports WQ_ERR_TIMEOUT (status bit 5: a GEMM's wait for its
 *                    producer's tiles expired), zero the workspace again.
 * The launch needs every CTA resident at once (two per SM); a device that is
 * shared with other work still runs it, later.  WQ_ERR_CUDA if the launch is
 * refused.  The weight-prefetch option (wq_set_option) applies as for the
 * decode GEMMs.  Measured on a GB300 for a decode MLP block (hidden 4096,
 * intermediate 11008, 4 tokens) it takes 34.6 us, against 27.1 us for
 * wq_gemm_w4a16_swiglu followed by wq_gemm_w4a16: use it where one launch per
 * list matters more than the time.
 */
typedef struct wq_chain_gemm {
  const void* X;
  int src;
  const uint32_t* Bpacked;
  const void* S;
  const float* delta;
  void* Y;
  int y_dtype;
  int N;
  int K;
  int group_size;
  int pair;
} wq_chain_gemm;

/* Bytes of workspace wq_gemm_w4a16_chain needs on the current device (0 for an
 * invalid list, M == 0 or an unsupported device). */
size_t wq_chain_workspace_size(const wq_chain_gemm* gemms, int n, int M, int x_dtype);

int wq_gemm_w4a16_chain(const wq_chain_gemm* gemms, int n, int M, int x_dtype, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Grouped (mixture-of-experts) W4A16 GEMM: the token rows of X are sorted by
 * expert, and expert e multiplies rows expert_offsets[e] .. expert_offsets[e+1]
 * by its own weights (the grouped GEMM of the SGLang W4A8 MoE article, section
 * "task split": one GEMM per group, tiled along K):
 *   Y[r][n] = sum_k X[r][k] W_e[k][n]   for r in expert e's rows,
 * each W_e the asymmetric (delta given) or symmetric weight of wq_gemm_w4a16.
 *   X, Y          [M][K] / [M][N] device, M = expert_offsets[experts].
 *   Bpacked       experts x (K*N/8 words) device: wq_pack_w4a16 outputs
 *                 stacked, expert-major.
 *   S, delta      experts x [G][N] device (delta NULL: symmetric).
 *   expert_offsets HOST int array of experts + 1 entries, offsets[0] == 0,
 *                 non-decreasing; experts in 1..64.  Read at the call and
 *                 passed by value in the launch parameters: a CUDA graph that
 *                 captures the call replays the offsets it was captured with.
 *   workspace     the largest wq_workspace_size(variant, tokens of one
 *                 expert, N, K, group_size) over the experts (0 when every
 *                 expert has <= 8 tokens).
 * With at most 8 tokens per expert this is one launch over all experts (an
 * expert without tokens costs nothing); otherwise one GEMM per expert.
 * Other arguments as wq_gemm_w4a16.
 */
int wq_gemm_w4a16_grouped(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S, const float* delta,
                          void* Y, int y_dtype, const int* expert_offsets, int experts, int N, int K,
                          int group_size, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Grouped (mixture-of-experts) W4A8 GEMM, the SGLang W4A8 MoE article's own
 * case (section "task split": one GEMM per group): the int8 token rows of Xq
 * are sorted by expert and expert e multiplies rows expert_offsets[e] ..
 * expert_offsets[e+1] by its own weights,
 *   Y[r][n] = x_scale[r] * sum_k Xq[r][k] W_e[k][n]   for r in expert e's rows,
 * W_e either the folded symmetric weight of wq_gemm_w4a8 (delta NULL; S and
 * Bpacked from wq_pack_w4a8) or the zero-point weight of wq_gemm_w4a8_asym
 * (delta given; from wq_pack_w4a16).
 *   Xq, x_scale   [M][K] int8 / [M] fp32 device, M = expert_offsets[experts].
 *   Bpacked, S, delta: one weight per expert, stacked expert-major as in
 *                 wq_gemm_w4a16_grouped.
 *   expert_offsets HOST int array as in wq_gemm_w4a16_grouped.
 *   workspace     the largest wq_workspace_size(variant, tokens of one
 *                 expert, N, K, group_size) over the experts, variant
 *                 WQ_VARIANT_W4A8_ASYM with delta, WQ_VARIANT_W4A8 without
 *                 (not used when every expert has <= 8 tokens).
 * With at most 8 tokens per expert: one weight-streaming launch over all
 * experts, which reads the int8 rows and applies the per-token scale at its
 * store.  Otherwise one W4A8 GEMM (activation pre-pass + GEMM) per expert that
 * has tokens, every expert's workspace need checked before anything is
 * enqueued.  All on `stream`.  Other arguments as wq_gemm_w4a16.
 */
int wq_gemm_w4a8_grouped(const int8_t* Xq, const float* x_scale, const uint32_t* Bpacked, const void* S,
                         const float* delta, void* Y, int y_dtype, const int* expert_offsets, int experts, int N,
                         int K, int group_size, void* workspace, size_t workspace_bytes, void* stream);

/*
 * W4A8 GEMM with zero-point (asymmetric) uint4 weights (HyperQwen W4A8
 * article, section "int8 tensor cores: how the numbers were verified", item
 * 2: int8 activations against uint4 codes with a zero point; the weight is
 * q * scale + zero as "Marlin INT4 on Ada", section "The core mismatch",
 * defines it):
 *   Y[m][n] = x_scale[m] * sum_k Xq[m][k] * (q[k][n] * scale[g][n] + zero[g][n])
 *           = x_scale[m] * (sum_k Xq[m][k] (q - 8) scale + sum_g a_sum[m][g] delta[g][n])
 * with a_sum the group sums of the int8 rows (exact in fp32).
 *   Xq, x_scale as wq_gemm_w4a8.
 *   Bpacked, S, delta from wq_pack_w4a16 (codes unfolded, scales with their
 *            signs, delta = zero + 8 scale); delta NULL gives the symmetric
 *            product with those scales (the same as wq_gemm_w4a8).
 *   workspace: wq_workspace_size(WQ_VARIANT_W4A8_ASYM, ...) bytes (or
 *            WQ_VARIANT_W4A8 with delta == NULL).  Other arguments as
 *            wq_gemm_w4a16.
 */
int wq_gemm_w4a8_asym(const int8_t* Xq, const float* x_scale, const uint32_t* Bpacked, const void* S,
                      const float* delta, void* Y, int y_dtype, int M, int N, int K, int group_size,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * W4A8 GEMM on fp16 activations quantized per token inside the call
 * (HyperQwen W4A8 article, section "why W4A8": activations quantized per token
 * to int8).  x_scale[m] = RN32(max_k |X[m][k]| / 127) and the codes
 * clamp(round_half_even(RN32(X / x_scale)), -127, 127) are exactly those of
 * wq_quantize_per_token; Y is then that of wq_gemm_w4a8_asym (delta given) or
 * wq_gemm_w4a8 (delta NULL), bit for bit.  The quantization is the GEMM's own
 * activation pre-pass: for the e4m3 decode kernel (M <= 16) it splits the
 * codes into e4m3 components on the way (the codes are never written out),
 * for the weight-streaming kernel (M <= 8, when its plan keeps one wave) it
 * writes them to the workspace, for larger M as fp16.
 *   X        [M][K] fp16 device.
 *   x_scale  [M] fp32 device, output: the per-token scales.
 *   Bpacked, S, delta: from wq_pack_w4a16 (zero-point weights; delta may be
 *            NULL) or wq_pack_w4a8 (folded symmetric weights, delta NULL).
 *   workspace: wq_workspace_size(WQ_VARIANT_W4A8_ASYM, ...) bytes with delta,
 *            wq_workspace_size(WQ_VARIANT_W4A8, ...) without.
 */
int wq_gemm_w4a8_fp16(const void* X, const uint32_t* Bpacked, const void* S, const float* delta, float* x_scale,
                      void* Y, int y_dtype, int M, int N, int K, int group_size, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Per-token int8 quantization of fp16 activations (HyperQwen article, "why
 * W4A8": activations quantized per token):
 *   x_scale[m] = fp32_RN(max_k |x[m][k]| / 127)
 *   Xq[m][k]   = clamp(rint(fp32_RN(x[m][k] / x_scale[m])), -127, 127)
 * An all-zero row gives x_scale = 0 and zero codes.  Any K >= 1.
 */
int wq_quantize_per_token(const void* x, int8_t* Xq, float* x_scale, int M, int K, void* stream);

/*
 * Process-wide launch options.
 *   WQ_OPTION_WEIGHT_PREFETCH: the decode kernel (M <= 16) is launched with
 *   programmatic dependent launch, so its setup overlaps the tail of the
 *   preceding kernel in the stream; it waits for that kernel before touching
 *   X or Y.  With this option set to 1 it also starts copying its first weight
 *   tiles (Bpacked, S, delta) before that wait.  Only enable it when the
 *   kernel launched just before each GEMM on the stream does not write the
 *   weights (the usual serving loop, where weights are packed once).
 * Returns WQ_ERR_INVALID_ARG for an unknown option or value.
 */
int wq_set_option(int option, long long value);
int wq_get_option(int option, long long* value);

/*
 * wq_gemm_w4a16 without a workspace argument, for callers that cannot
 * allocate device memory where they make the call (inside a framework that
 * forbids allocations outside its own allocator, host code that runs during
 * CUDA stream capture, latency-critical loops where cudaMalloc could
 * synchronize).  The pages have no counterpart to this entry point.
 *   Arguments and result as wq_gemm_w4a16.  The scratch comes from a 16 MiB
 *   array of device memory inside the library image (held by every GPU that
 *   loads the library until the process exits); problems that need more
 *   return WQ_ERR_WORKSPACE without launching.  The need is that of this
 *   call's activation type: about (M + N) * K/128 * 4 bytes of correction
 *   columns for M > 16 with delta, plus M * K * 2 bytes of scaled fp16
 *   activations when they are bf16 (so bf16 problems above about 8M
 *   activation elements are refused).
 *   The arguments are checked first, as wq_gemm_w4a16 checks them, then the
 *   size.  Nothing is allocated or freed.  The first call on a device looks
 *   up the array's device address (cudaGetSymbolAddress), and so does the
 *   first call after the device's context has been rebuilt (cudaDeviceReset);
 *   make that first call before capturing a stream.  All calls on a device
 *   share the array and it keeps the last call's contents (no call needs any
 *   of it to start at zero), so calls whose kernels may overlap on the GPU
 *   (different streams) race on it.
 */
int wq_gemm_w4a16_noalloc(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S,
                          const float* delta, void* Y, int y_dtype, int M, int N, int K,
                          int group_size, void* stream);

/*
 * W4A16 GEMM between host buffers: X is copied host -> device, the GEMM runs
 * as wq_gemm_w4a16 ("Marlin INT4 on Ada -- how it works", section "The
 * pipeline, end to end": Y = X @ W_sym + A_group_sum @ delta), and Y is
 * copied device -> host, all enqueued on `stream` with cudaMemcpyAsync.
 * Pinned (page-locked) host buffers let the copies run asynchronously; the
 * call returns before the work completes, so read Y_host after synchronizing
 * the stream.  The copies to and from the host are this library's addition.
 *   X_host   [M][K] host memory, fp16 or bf16 (x_dtype), row-major.
 *   Y_host   [M][N] host memory, output (y_dtype F16, BF16 or F32).
 *   Bpacked, S, delta: device, as wq_gemm_w4a16.
 *   workspace / workspace_bytes: device scratch of at least
 *            wq_host_workspace_size(...) bytes, 256-byte aligned: the device
 *            copies of X and Y, then the GEMM's own workspace.
 * All arguments are checked before anything is enqueued.
 * With M >= 2048 the call pipelines token-row chunks (up to four, multiples of
 * 256 rows): the copy of a chunk's X runs on one internal stream, its GEMM on
 * `stream`, the copy of its Y on a second internal stream, ordered by events,
 * so copies overlap the neighbouring chunks' GEMMs.  The two copy streams and
 * their events are created once per device on the first such call (no memory
 * is allocated); `stream` waits for the last copy before any later work, so
 * Y_host is complete once `stream` is synchronized.  Concurrent calls from
 * several host threads are serialized while they are enqueued.
 */
int wq_gemm_w4a16_host(const void* X_host, int x_dtype, const uint32_t* Bpacked, const void* S,
                       const float* delta, void* Y_host, int y_dtype, int M, int N, int K,
                       int group_size, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace wq_gemm_w4a16_host needs (0 for an unsupported problem);
 * variant WQ_VARIANT_W4A16 or WQ_VARIANT_W4A16_SYM. */
size_t wq_host_workspace_size(int variant, int M, int N, int K, int group_size, int y_dtype);

/* Bytes of workspace the GEMM needs for this problem (0 if none): the most any
 * activation type needs (bf16 activations with M > 16 need M * K * 2 + M * 4
 * bytes more than fp16 ones, for their scaled fp16 copy). */
size_t wq_workspace_size(int variant, int M, int N, int K, int group_size);

/* 1 if `device` is an sm_103 GPU this library can run on, else 0. */
int wq_device_supported(int device);

/* Description of the last error on this thread ("" if none). */
const char* wq_last_error(void);

/* Library version string. */
const char* wq_version(void);

/*
 * Synchronizes `stream`, then reads the device status word of the current
 * device into *status (bit 0..3: a bounded wait in the GEMM expired, bit 4:
 * the wait probe expired, bit 5: a chain GEMM's wait for its producer expired)
 * and clears it if `reset` is nonzero.  Returns
 * WQ_ERR_TIMEOUT if any bit was set, else WQ_OK.
 */
int wq_device_status(unsigned int* status, int reset, void* stream);

/*
 * Test aid: launches one thread that waits on a barrier nothing will ever
 * complete, with a limit of limit_ns nanoseconds (<= 10 s).  The kernel gives
 * up, sets bit 4 of the device status word and returns normally.
 */
int wq_debug_wait_probe(unsigned long long limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H_ */
