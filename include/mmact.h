/*
 * mmact.h -- C ABI of the fused GEMM / implicit-GEMM conv + bias + activation
 * library for GB300 (sm_103a).  libmmact.so exports exactly these symbols.
 *
 * Operations
 *   C = act(A x B + bias)                        mmact_gemm, mmact_gemm_split
 *   C = act(A x B + bias + R)                    mmact_gemm_residual
 *     "MatmulLeakyRelu fusion walkthrough" (pyasc examples/05_matmul_leakyrelu):
 *     overview formula C = A x B + Bias then LeakyReLU, computed in one kernel;
 *     sample spec table (A [M,K], B [K,N] row-major and not transposed, bias
 *     fp32 [1,N], C fp32).  ReLU: "ops-nn fused_matmul_relu" article, the
 *     fused call on 4096^3 and its two-call fallback (matmul into a device
 *     temporary, then relu).
 *   y = act(conv2d(x, w, bias))                  mmact_conv2d, mmact_conv2d_split,
 *                                                mmact_conv2d_nhwc (channels-last)
 *   y = act(conv2d(x, w, bias) + R)              mmact_conv2d_residual, mmact_conv2d_nhwc_residual
 *     "multimodal-ops Fused ConvTanh" article: y = tanh(conv2d(x, filter,
 *     bias)) with strides / pads / dilations; the convolution is an implicit
 *     GEMM whose A operand is the filter [Co x Ci*kh*kw] and whose B operand is
 *     the input features [Ci*kh*kw x Ho*Wo], so the result is already laid out
 *     [Co, Ho*Wo] per image (NCHW) -- section "how the two kernels split the
 *     work".  The *_split variants are that article's two-kernel "half fusion"
 *     (fp32 workspace in device memory, then a separate activation pass), kept
 *     as a measured ablation.
 *
 * Activations (all evaluated in fp32 on the fp32 accumulator plus the fp32
 * bias, then rounded to the output dtype with round-to-nearest-even):
 *   MMACT_ACT_NONE        z
 *   MMACT_ACT_RELU        z > 0 ? z : 0
 *   MMACT_ACT_LEAKY_RELU  z > 0 ? z : alpha * z
 *   MMACT_ACT_TANH        (e^z - e^-z) / (e^z + e^-z)
 *   MMACT_ACT_SIGMOID     1 / (1 + e^-z)       (the Fused ConvTanh article's twin
 *                         operator, Fused ConvSigmoid)
 *   MMACT_ACT_GELU        z/2 * (1 + erf(z / sqrt(2)))   (the fused_matmul_relu
 *                         article's matmul + GELU / Sigmoid / Tanh family; exact
 *                         erf form, the pages print no formula)
 *
 * Conventions for every entry point
 *   - Tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) on
 *     the current CUDA device.  The caller owns every buffer; the library
 *     never allocates, frees or retains them.
 *   - All tensors are dense and row-major (C order).  16-byte alignment is
 *     required of A, B, C, x, y, w and workspace; 4-byte alignment of bias.
 *   - bias may be NULL (treated as all zeros).  Any other pointer may be NULL
 *     only when its tensor has no elements.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous: they validate arguments on the host,
 *     enqueue kernels on `stream` and return.  A status other than MMACT_OK
 *     means nothing was enqueued.
 *   - Errors that arise inside a kernel (a bounded wait that ran out) are
 *     recorded in a per-device status word; mmact_get_last_error() reads and
 *     clears it.
 *   - Thread safety: calls may come from several host threads; the only
 *     shared state is the per-device status word and one-time kernel set-up.
 */
#ifndef MMACT_H
#define MMACT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MMACT_OK = 0,
    MMACT_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum, bad geometry */
    MMACT_ERR_UNSUPPORTED = 2,   /* valid request the library does not handle (alignment, dtype pair) */
    MMACT_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    MMACT_ERR_TIMEOUT = 4        /* a kernel's bounded wait ran out (reported by get_last_error) */
} mmact_status;

typedef enum {
    MMACT_ACT_NONE = 0,
    MMACT_ACT_RELU = 1,
    MMACT_ACT_LEAKY_RELU = 2,
    MMACT_ACT_TANH = 3,
    MMACT_ACT_SIGMOID = 4,
    MMACT_ACT_GELU = 5
} mmact_act;

typedef enum {
    MMACT_F16 = 0,
    MMACT_BF16 = 1,
    MMACT_F32 = 2,   /* as an input: fp32 values used to fp32 accuracy (split precision, below) */
    MMACT_TF32 = 3   /* input only: fp32 values rounded to tf32 (10 fraction bits) by the tensor core */
} mmact_dtype;

/*
 * fp32 inputs (the Fused ConvTanh article evaluates fp32 cases beside fp16 and
 * bf16).  MMACT_F32 inputs are computed in split precision: every input value
 * v is split into two bf16 values hi = rn(v) and lo = rn(v - hi), and each
 * product as xh*wh + xl*wh + xh*wl (three tensor-core products accumulated in
 * the same fp32 accumulator), which leaves an error of about 2^-15 of
 * sum_k |x_k w_k| -- inside the fp32-output tolerance 2e-3 + 2e-3 |y|.  It
 * runs on the general gather kernel (three MMAs per K step; several times
 * slower than 16-bit inputs).  MMACT_TF32 inputs (mmact_conv2d_nhwc only) are
 * the fast one-pass alternative: each operand keeps 10 fraction bits, so the
 * error is up to about 2^-9 * sum_k |x_k w_k|.
 */

/*
 * Fused single-kernel GEMM + bias + activation:  C = act(A x B + bias).
 *   A     [M, K] ab_dtype (F16, BF16, or F32 in split precision), row-major
 *   B     [K, N] ab_dtype, row-major (N contiguous; not transposed)
 *   bias  [N] fp32, or NULL
 *   C     [M, N] c_dtype (F32, F16 or BF16), row-major; fully overwritten
 *   alpha LeakyReLU slope (ignored by the other activations)
 * Accumulation is fp32 on the tensor cores.  M == 0 or N == 0 enqueues
 * nothing; K == 0 gives C = act(bias).  16-bit A/B require K % 8 == 0 and
 * N % 8 == 0 (16-byte row pitch) else MMACT_ERR_UNSUPPORTED; F32 A/B need
 * only 4-byte alignment (any K, N; C stays 16-byte aligned); TF32 is
 * MMACT_ERR_UNSUPPORTED here.  M, N, K < 2^31.
 */
mmact_status mmact_gemm(const void *A, const void *B, const float *bias, void *C,
                        int64_t M, int64_t N, int64_t K,
                        mmact_dtype ab_dtype, mmact_dtype c_dtype,
                        mmact_act act, float alpha, void *stream);

/*
 * Fused GEMM + bias + residual + activation:  C = act(A x B + bias + R).
 * The element-wise add of a residual tensor fused into the matmul epilogue,
 * from the ops-nn fused_matmul_relu article's fusion families (the "math"
 * family: matmul + add + bias, so a residual path is accumulated on chip
 * instead of making a round trip through HBM); R is added to the fp32
 * accumulator before the activation, the order residual networks use.
 *   R  [M, N] in c_dtype, row-major, 16-byte aligned; read, never written.
 *      R == C (in-place residual update) is allowed; any other overlap of
 *      R and C returns MMACT_ERR_INVALID_ARG.  R may be NULL only if M*N == 0.
 * Everything else as mmact_gemm (K == 0 gives C = act(bias + R)).
 */
mmact_status mmact_gemm_residual(const void *A, const void *B, const float *bias, const void *R,
                                 void *C, int64_t M, int64_t N, int64_t K,
                                 mmact_dtype ab_dtype, mmact_dtype c_dtype,
                                 mmact_act act, float alpha, void *stream);

/*
 * Two-kernel ablation of mmact_gemm.  Kernel 1 writes z = A x B + bias in fp32
 * to `workspace` ([M, N] fp32, caller-allocated, M*N*4 bytes, 16-byte
 * aligned); kernel 2 reads it, applies act in fp32 and writes C.  Same result
 * contract as mmact_gemm; the workspace holds z afterwards.
 */
mmact_status mmact_gemm_split(const void *A, const void *B, const float *bias, void *C,
                              int64_t M, int64_t N, int64_t K,
                              mmact_dtype ab_dtype, mmact_dtype c_dtype,
                              mmact_act act, float alpha, float *workspace, void *stream);

/*
 * Fused or two-kernel GEMM, decided per shape at run time (the ops-nn
 * fused_matmul_relu article's run-time decision between the fused call and
 * its fallback, matmul into a device temporary then the activation).  The
 * rule comes from a measured grid of fused against split times on GB300:
 * the split path is taken for GELU on an output of at most 65536 elements
 * (one or two tiles: the fused epilogue's few warps are latency-bound on the
 * activation, the split's activation pass spreads over the GPU), the fused
 * kernel everywhere else (faster by up to 3x there, or within a few per cent
 * on mid-sized GELU outputs).  `workspace`
 * ([M, N] fp32, 16-byte aligned) may be NULL: then the fused kernel always
 * runs.  Everything else as mmact_gemm / mmact_gemm_split.
 */
mmact_status mmact_gemm_auto(const void *A, const void *B, const float *bias, void *C,
                             int64_t M, int64_t N, int64_t K,
                             mmact_dtype ab_dtype, mmact_dtype c_dtype,
                             mmact_act act, float alpha, float *workspace, void *stream);

/* Which path mmact_gemm_auto takes with a workspace: *split = 1 for the two-kernel
 * split, 0 for the fused kernel (host only).  MMACT_ERR_INVALID_ARG for bad arguments. */
mmact_status mmact_gemm_auto_choice(int64_t M, int64_t N, int64_t K, mmact_dtype ab_dtype,
                                    mmact_dtype c_dtype, mmact_act act, int *split);

/*
 * Fused implicit-GEMM conv2d + bias + activation:  y = act(conv2d(x, w) + bias).
 *   x    [N, C, H, W] in_dtype (F16, BF16, or F32 in split precision), NCHW
 *   w    [Co, C, kh, kw] in_dtype
 *   bias [Co] fp32, or NULL
 *   y    [N, Co, Ho, Wo] out_dtype (F32, F16 or BF16), NCHW; fully overwritten
 *   strides   = {sh, sw} >= 1
 *   pads      = {top, bottom, left, right} >= 0 (zero padding)
 *   dilations = {dh, dw} >= 1
 *   Ho = floor((H + top + bottom - dh*(kh-1) - 1) / sh) + 1, Wo likewise;
 *   a geometry with Ho < 1 or Wo < 1 is MMACT_ERR_INVALID_ARG.
 * N == 0 or Co == 0 enqueues nothing; C == 0 gives y = act(bias).
 */
mmact_status mmact_conv2d(const void *x, const void *w, const float *bias, void *y,
                          int64_t N, int64_t C, int64_t H, int64_t W,
                          int64_t Co, int64_t kh, int64_t kw,
                          const int32_t strides[2], const int32_t pads[4],
                          const int32_t dilations[2],
                          mmact_dtype in_dtype, mmact_dtype out_dtype,
                          mmact_act act, float alpha, void *stream);

/*
 * mmact_conv2d with a residual tensor added before the activation:
 *   y = act(conv2d(x, w) + bias + R), the conv form of mmact_gemm_residual
 *   (the fused_matmul_relu article's element-wise add fused into the
 *   preceding computation, as in residual networks).
 *   R  [N, Co, Ho, Wo] in out_dtype (y's shape), 16-byte aligned; read, never
 *      written.  R == y is allowed; any other overlap of R and y returns
 *      MMACT_ERR_INVALID_ARG.  R may be NULL only if y is empty.
 * Everything else as mmact_conv2d (C == 0 gives y = act(bias + R)).
 */
mmact_status mmact_conv2d_residual(const void *x, const void *w, const float *bias, const void *R,
                                   void *y, int64_t N, int64_t C, int64_t H, int64_t W,
                                   int64_t Co, int64_t kh, int64_t kw,
                                   const int32_t strides[2], const int32_t pads[4],
                                   const int32_t dilations[2],
                                   mmact_dtype in_dtype, mmact_dtype out_dtype,
                                   mmact_act act, float alpha, void *stream);

/*
 * Two-kernel ablation of mmact_conv2d: kernel 1 writes z (conv + bias, fp32)
 * to `workspace` ([N, Co, Ho, Wo] fp32, caller-allocated, 16-byte aligned),
 * kernel 2 applies act and writes y.
 */
mmact_status mmact_conv2d_split(const void *x, const void *w, const float *bias, void *y,
                                int64_t N, int64_t C, int64_t H, int64_t W,
                                int64_t Co, int64_t kh, int64_t kw,
                                const int32_t strides[2], const int32_t pads[4],
                                const int32_t dilations[2],
                                mmact_dtype in_dtype, mmact_dtype out_dtype,
                                mmact_act act, float alpha, float *workspace, void *stream);

/*
 * mmact_conv2d or mmact_conv2d_split, decided per geometry at run time as for
 * mmact_gemm_auto.  The split path is taken for GELU over a contraction
 * C*kh*kw of at most 288 with Co >= 64, and when the fused kernel would store a 16-bit
 * output element by element (the output row pitch Ho*Wo*2 is not a
 * multiple of 16 bytes and neither the tensor-memory nor the vectorised
 * producer applies), where the split's fp32 intermediate is stored by TMA.
 * `workspace` ([N, Co, Ho, Wo] fp32) may be NULL: then the fused kernel runs.
 */
mmact_status mmact_conv2d_auto(const void *x, const void *w, const float *bias, void *y,
                               int64_t N, int64_t C, int64_t H, int64_t W,
                               int64_t Co, int64_t kh, int64_t kw,
                               const int32_t strides[2], const int32_t pads[4],
                               const int32_t dilations[2],
                               mmact_dtype in_dtype, mmact_dtype out_dtype,
                               mmact_act act, float alpha, float *workspace, void *stream);

/* Which path mmact_conv2d_auto takes with a workspace (*split: 1 split, 0 fused; host only). */
mmact_status mmact_conv2d_auto_choice(int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co,
                                      int64_t kh, int64_t kw, const int32_t strides[2],
                                      const int32_t pads[4], const int32_t dilations[2],
                                      mmact_dtype in_dtype, mmact_dtype out_dtype, mmact_act act,
                                      int *split);

/*
 * Largest M*N accepted by mmact_gemm_split_noalloc (fp32 elements of its
 * built-in scratch array: 16 MiB per device).
 */
#define MMACT_NOALLOC_MAX_ELEMENTS 4194304

/*
 * mmact_gemm_split for callers that cannot allocate device memory when they
 * call the library.  (The pages have no counterpart: this entry point exists
 * for deployment, not for the method.)  Some callers are only handed their
 * input and output buffers by a host framework, run under a framework
 * allocator that already owns the device budget, or sit in a latency-critical
 * loop where cudaMalloc / cudaFree could block or synchronise the device;
 * they cannot supply the M*N fp32 workspace the split path needs.  This entry
 * point takes the same arguments as mmact_gemm_split minus `workspace`, and
 * uses a fixed scratch array compiled into the library instead; it calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - Limit: M*N <= MMACT_NOALLOC_MAX_ELEMENTS, else MMACT_ERR_UNSUPPORTED
 *     (nothing enqueued).  Every GPU that loads the library holds the 16 MiB
 *     array until the process exits.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress, with that device current) and caches it
 *     for that device's current CUDA context; make that first call before any
 *     stream capture.  A call in a new context (after cudaDeviceReset) looks
 *     the address up again, so the same rule applies to it.
 *   - Sharing: all calls on a device share the one array, which keeps the
 *     last call's intermediate values.  Nothing in it needs clearing: the
 *     first kernel overwrites every element it uses before the second reads
 *     it.  Calls whose kernels may overlap on the GPU (different streams, or
 *     several host threads without ordering) race on the array; order them,
 *     e.g. on one stream.
 * Argument checks are those of mmact_gemm_split and come first (a bad
 * pointer, dtype or activation returns MMACT_ERR_INVALID_ARG whatever the
 * size); the size limit is checked next, and the scratch address is looked
 * up only for a call that will run.  All other behaviour, layouts and errors
 * are those of mmact_gemm_split.
 */
mmact_status mmact_gemm_split_noalloc(const void *A, const void *B, const float *bias, void *C,
                                      int64_t M, int64_t N, int64_t K,
                                      mmact_dtype ab_dtype, mmact_dtype c_dtype,
                                      mmact_act act, float alpha, void *stream);

/*
 * Channels-last fused conv2d + bias + activation (the layout-converting
 * member of the fused_matmul_relu article's fusion families applied to the
 * Fused ConvTanh operator):  y = act(conv2d(x, w) + bias).
 *   x    [N, H, W, C] in_dtype (F16, BF16, F32 in split precision, or TF32),
 *        channels innermost (NHWC)
 *   w    [Co, kh, kw, C] in_dtype, channels innermost
 *   bias [Co] fp32, or NULL
 *   y    [N, Ho, Wo, Co] out_dtype (F32, F16 or BF16), NHWC; fully overwritten
 * strides / pads / dilations and Ho, Wo as for mmact_conv2d.  TF32 inputs
 * (fp32 storage) run on the tensor cores as tf32 with the operands fed by
 * TMA: each operand keeps 10 fraction bits, so |error| <= about
 * 2^-9 * sum_k |x_k w_k| beyond the fp32 accumulation.  F32 inputs run in
 * split precision on the general gather kernel (fp32 accuracy, slower).
 * Requires C * sizeof(in_dtype) % 16 == 0 and Co % 8 == 0 (16-byte channel
 * rows), else MMACT_ERR_UNSUPPORTED.  N == 0 or Co == 0 enqueues nothing;
 * C == 0 gives y = act(bias).
 */
mmact_status mmact_conv2d_nhwc(const void *x, const void *w, const float *bias, void *y,
                               int64_t N, int64_t C, int64_t H, int64_t W,
                               int64_t Co, int64_t kh, int64_t kw,
                               const int32_t strides[2], const int32_t pads[4],
                               const int32_t dilations[2],
                               mmact_dtype in_dtype, mmact_dtype out_dtype,
                               mmact_act act, float alpha, void *stream);

/*
 * mmact_conv2d_nhwc with a residual tensor added before the activation:
 *   y = act(conv2d(x, w) + bias + R), R [N, Ho, Wo, Co] in out_dtype (y's
 *   shape), 16-byte aligned; R == y allowed, other overlaps rejected with
 *   MMACT_ERR_INVALID_ARG.  F32 (split precision) inputs are
 *   MMACT_ERR_UNSUPPORTED here.  Everything else as mmact_conv2d_nhwc.
 */
mmact_status mmact_conv2d_nhwc_residual(const void *x, const void *w, const float *bias, const void *R,
                                        void *y, int64_t N, int64_t C, int64_t H, int64_t W,
                                        int64_t Co, int64_t kh, int64_t kw,
                                        const int32_t strides[2], const int32_t pads[4],
                                        const int32_t dilations[2],
                                        mmact_dtype in_dtype, mmact_dtype out_dtype,
                                        mmact_act act, float alpha, void *stream);

/*
 * Output spatial size of a conv geometry (host only, no CUDA call).  Writes
 * Ho and Wo (host pointers) and returns MMACT_OK, or MMACT_ERR_INVALID_ARG for
 * a bad geometry (non-positive kernel/stride/dilation, negative pad or size,
 * or an empty output).
 */
mmact_status mmact_conv2d_out_shape(int64_t H, int64_t W, int64_t kh, int64_t kw,
                                    const int32_t strides[2], const int32_t pads[4],
                                    const int32_t dilations[2], int64_t *Ho, int64_t *Wo);

/*
 * Diagnostic: which B-tile producer mmact_conv2d (and mmact_conv2d_split)
 * would use for this NCHW geometry.  The choice depends only on the shape and
 * dtypes.  Returns a mmact_conv_producer value, or -1 when the arguments are
 * invalid, C == 0, or the problem is too large for the library.
 *   MMACT_CONV_GATHER  per-element im2col gather (any geometry; every F32-input conv)
 *   MMACT_CONV_VECTOR  16-byte chunk loads from global memory + byte picks
 *                      (W % 8 == 0, horizontal stride 1 or 2, filter rows a
 *                      multiple of 16 bytes, output rows TMA-storable)
 *   MMACT_CONV_WINDOW  as VECTOR, but each K block's input window is first
 *                      loaded into shared memory by one TMA box (when that
 *                      window fits in 24 KB)
 *   MMACT_CONV_TMEM    the im2col operand is assembled in tensor memory, one
 *                      output pixel per TMEM lane, from each K block's input
 *                      window (staged by TMA); the filter is the MMA's
 *                      shared-memory operand (16-bit inputs, W % 8 == 0,
 *                      C*kh*kw % 8 == 0, a window of at most 40 KB, and
 *                      lcm(64, kh*kw) <= 3136).  Taken whenever it applies,
 *                      unless mmact_set_conv_tmem(1) turned it off.
 */
typedef enum {
    MMACT_CONV_GATHER = 0,
    MMACT_CONV_VECTOR = 1,
    MMACT_CONV_WINDOW = 2,
    MMACT_CONV_TMEM = 3
} mmact_conv_producer;
int mmact_conv2d_producer(int64_t N, int64_t C, int64_t H, int64_t W, int64_t Co, int64_t kh,
                          int64_t kw, const int32_t strides[2], const int32_t pads[4],
                          const int32_t dilations[2], mmact_dtype in_dtype, mmact_dtype out_dtype);

/*
 * Synchronises `stream`, then reports and clears the current device's kernel
 * status word: MMACT_OK, MMACT_ERR_TIMEOUT (a bounded wait inside a kernel ran
 * out; the kernel skipped its remaining work and left its outputs
 * unspecified), or MMACT_ERR_CUDA (the stream reported a CUDA error).
 */
mmact_status mmact_get_last_error(void *stream);

/*
 * Upper bound, in nanoseconds, on every wait inside the pipelined kernels
 * (default 2e9).  A wait that runs out makes the kernel stop, release its
 * tensor memory and record MMACT_ERR_TIMEOUT.  Applies to launches made after
 * the call.  0 restores the default.
 */
void mmact_set_wait_timeout_ns(uint64_t ns);

/*
 * Diagnostic: enqueue one tiny kernel on `stream` that waits on an mbarrier
 * nothing ever arrives at, bounded by `timeout_ns`; it records
 * MMACT_ERR_TIMEOUT in the status word and returns.  Used to check the
 * timeout-reporting path without any fault.
 */
mmact_status mmact_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/*
 * Tuning and testing aid: force the N-extent of the GEMM output tile (64, 128,
 * 192, 224 or 256; 0 = automatic choice).  Applies to later mmact_gemm* calls in the
 * process.  Returns MMACT_ERR_INVALID_ARG for other values.
 */
mmact_status mmact_set_gemm_tile_n(int tile_n);

/*
 * Tuning and testing aid (no counterpart in the pages, whose operators split
 * work over cores by output blocks only): the split-K GEMM kernel.  For GEMMs with few
 * 128 x 256 output tiles (small M) mmact_gemm, mmact_gemm_residual,
 * mmact_gemm_split and mmact_gemm_split_noalloc may run each tile on a
 * thread-block cluster of 2 or 4 CTAs, each CTA accumulating 1/2 or 1/4 of
 * the K blocks, the partial fp32 tiles summed across the cluster before the
 * same residual + bias + activation epilogue (the sum over K stays in fp32).
 * split_k: 0 = chosen per shape (the default), 1 = never, 2 or 4 = always
 * with that factor when K has at least that many 64-wide blocks.  Applies to
 * later calls in the process.  Returns MMACT_ERR_INVALID_ARG for other values.
 */
mmact_status mmact_set_gemm_split_k(int split_k);

/*
 * Tuning and testing aid (no counterpart in the pages: a GB300 execution
 * choice for the same operator): the CTA-pair GEMM kernel, which runs 256 x 256
 * output tiles on two SMs with one M = 256 tcgen05.mma per pair
 * (cta_group::2), each SM holding half of A and half of B.  mode: 0 = chosen
 * per shape (the default: when the persistent kernel would use 256-wide
 * tiles and the pair grid needs no more waves), 1 = never, 2 = for every
 * mmact_gemm-family call that does not take the split-K kernel.  Applies to later calls in the
 * process.  Returns MMACT_ERR_INVALID_ARG for other values.
 */
mmact_status mmact_set_gemm_pair(int mode);

/*
 * Tuning and testing aid (no counterpart in the pages: a GB300 execution
 * choice for the same operator): whether mmact_conv2d, mmact_conv2d_residual
 * and mmact_conv2d_split use the tensor-memory im2col kernel
 * (MMACT_CONV_TMEM) where it applies.  mode: 0 = yes (the default), 1 = never
 * (the window / vector / gather producers).  Applies to later calls in the
 * process.  Returns MMACT_ERR_INVALID_ARG for other values.
 */
mmact_status mmact_set_conv_tmem(int mode);

/*
 * L2 cache policy of the CTA-pair GEMM kernel (diagnostic; no counterpart in
 * the pages).  The kernel rasters its 256 x 256 tiles in groups of 8 M
 * blocks: every wave of tiles in a group reads the same A rows, while a B
 * column strip is read by the tiles of one wave only.  mode 1 (the default)
 * loads A with the L2 evict-last policy, so that the group's A rows stay in
 * L2 across its waves, and stores C with evict-first (C is not read back);
 * mode 0 issues the same copies without cache hints.  Results are identical.
 * Returns MMACT_ERR_INVALID_ARG for other values.
 */
mmact_status mmact_set_gemm_l2_policy(int mode);

/*
 * Tensor-map cache counters (diagnostic; no counterpart in the pages).  Every
 * call encodes up to four TMA tensor maps on the host; an encoded map depends
 * only on its address, shape, strides, box and dtype, so the library keeps up
 * to 256 per host thread (64 sets of 4), keyed by all of them, and a call that repeats an
 * earlier call's tensors and shapes copies them instead of encoding again.
 * Writes the process-wide number of cache hits and of encodes so far (either
 * pointer may be null).  Never fails.
 */
mmact_status mmact_tensor_map_cache_stats(uint64_t *hits, uint64_t *encodes);

/* The GEMM kernels an mmact_gemm-family call can run. */
typedef enum {
    MMACT_GEMM_KERNEL_NONE = 0,        /* empty output or K = 0: the bias/activation fill only */
    MMACT_GEMM_KERNEL_PERSISTENT = 1,  /* one SM per 128 x BN tile, persistent grid */
    MMACT_GEMM_KERNEL_PAIR = 2,        /* 256 x 256 tiles on CTA pairs (cta_group::2) */
    MMACT_GEMM_KERNEL_SPLIT_K = 3      /* 128 x 256 tiles on clusters of 2 or 4 CTAs, K split */
} mmact_gemm_kernel;

/*
 * Which kernel an mmact_gemm-family call of this shape on the current device
 * would run (an mmact_gemm_kernel value in *kernel), under the current
 * settings of mmact_set_gemm_split_k, mmact_set_gemm_pair and
 * mmact_set_gemm_tile_n; has_residual != 0 for mmact_gemm_residual.  Returns
 * MMACT_ERR_INVALID_ARG for a null kernel or a negative extent,
 * MMACT_ERR_CUDA when the device cannot be queried.
 */
mmact_status mmact_gemm_kernel_choice(int64_t M, int64_t N, int64_t K, int has_residual, int *kernel);

/*
 * The split-K factor (0 = none, 2 or 4) that an mmact_gemm-family call of
 * this shape on the current device would use under the current setting of
 * mmact_set_gemm_split_k and mmact_set_gemm_tile_n.  Writes it to *split_k.
 * Returns MMACT_ERR_INVALID_ARG for a null split_k or a negative extent,
 * MMACT_ERR_CUDA when the device cannot be queried.
 */
mmact_status mmact_gemm_split_k_choice(int64_t M, int64_t N, int64_t K, int *split_k);

/* Human-readable name of a status code (static string, never NULL). */
const char *mmact_status_string(mmact_status status);

/* ABI version of this header: 1. */
int mmact_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MMACT_H */
