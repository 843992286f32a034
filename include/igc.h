/*
 * igc.h -- C ABI of the GB300 (sm_103a) tensor-core GEMM / implicit-GEMM
 * convolution library (libigc.so).
 *
 * Pages the operations follow (cited by title and section):
 *  [P1] "TVM在CUDA GPU上跑GEMM的全套张量化实现：WMMA/DP4A/IMMA + TensorIR调度 +
 *       INT8/FP16多精度支持": §2.1 (tensor-core MMA with "row.col" operands: A
 *       row-major, B column-major), §2.3 (INT8 GEMM with input zero points,
 *       C = (A_q - zp_A)(B_q - zp_B), fused quantise / dequantise), §4.1 (the GEMM
 *       compute definition C[i,j] = sum_k A[i,k] * B[k,j] on fp16 operands),
 *       §4.4 (destination passing: caller-allocated inputs and outputs, mod(a, b, c)).
 *  [P3] "如何使用 TensorCores 优化卷积" (TVM tutorial "How to optimize convolution
 *       using TensorCores"), section "准备和算法" (3x3 convolution, zero padding
 *       Apad, reduction over input channels and the filter window, fp16 operands
 *       cast to float32 before the multiply-add) and "生成 CUDA 内核" (the built
 *       function is called as func(a, w, c) on caller-owned device arrays).
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller owns every buffer.  Pointers named "device" must be
 *    device memory of the current CUDA device (e.g. torch tensors' data_ptr()).
 *    The library allocates no device memory; gemm_s8_zp takes its scratch as a
 *    caller-provided workspace.
 *  - Asynchrony: compute calls enqueue work on `stream` (NULL = legacy default
 *    stream) and return without synchronising.  A non-IGC_OK return means
 *    nothing was enqueued (except IGC_ERR_CUDA, where a launch failed).
 *  - Errors: no exceptions cross the ABI.  Argument errors are detected on the
 *    host before any launch.  Kernel-side pipeline waits are bounded: if one
 *    gives up, the kernel records it in a device status word and exits;
 *    igc_check_device_status() reports it as IGC_ERR_DEVICE_TIMEOUT.
 *  - Alignment: operand base pointers must be 16-byte aligned and operand row
 *    strides (in bytes) multiples of 16 (TMA rules), else IGC_ERR_MISALIGNED.
 *    Outputs may have any alignment; outputs whose base and row stride are
 *    16-byte aligned are written by TMA bulk tensor stores, others by direct
 *    stores.
 *  - Device: an sm_103 GPU (GB300); any other returns IGC_ERR_UNSUPPORTED.
 *  - Calls are stateless and re-entrant; concurrent calls on different streams
 *    are independent (each gemm_s8_zp call needs its own workspace).  The
 *    schedule of a call depends only on its arguments and the device, unless
 *    the calling thread itself forced one through the test hooks of
 *    igc_debug.h (thread-local: they never reach another thread's calls).
 *  - Launch: kernels use programmatic dependent launch -- a kernel may start
 *    while the previous kernel in the stream finishes, and waits for it before
 *    touching memory -- so stream order is kept as with plain launches.  Calls
 *    may be captured in CUDA graphs; make one call of each operation on the
 *    device first (per-kernel set-up runs once, outside the capture).
 */
#ifndef IGC_H
#define IGC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *igc_stream_t;

/* status codes */
#define IGC_OK 0
#define IGC_ERR_INVALID_ARG 1    /* null required pointer, negative size, ld < K, no output */
#define IGC_ERR_MISALIGNED 2     /* operand pointer / row stride breaks the 16-byte TMA rules */
#define IGC_ERR_UNSUPPORTED 3    /* shape or device outside what the kernels implement */
#define IGC_ERR_CUDA 4           /* a CUDA runtime / driver call failed */
#define IGC_ERR_DEVICE_TIMEOUT 5 /* a kernel's bounded pipeline wait gave up */
#define IGC_ERR_WORKSPACE 6      /* workspace pointer null or smaller than required */

/* output element types for gemm_f16 / gemm_bf16 */
#define IGC_F32 0
#define IGC_F16 1
#define IGC_BF16 2

/*
 * gemm_f16 -- C = A * B, fp16 operands, fp32 accumulation ([P1] §4.1, §2.1).
 *
 *   C[i,j] = sum_{k<K} A[i,k] * Bt[j,k]      0 <= i < M, 0 <= j < N
 *
 *  A    device, fp16, M x K row-major, row stride lda >= K elements.
 *  Bt   device, fp16, B stored column-major: N x K row-major (K contiguous),
 *       row stride ldb >= K elements.
 *  C    device, M x N row-major, row stride ldc >= N elements, element type
 *       c_dtype: IGC_F32 (the fp32 accumulator) or IGC_F16 (round to nearest
 *       even of the fp32 accumulator; overflow gives +-inf).  May be NULL if
 *       C_f32_check is given.
 *  C_f32_check  device fp32 M x N (row stride ldc32 >= N) or NULL: an extra
 *       copy of the fp32 accumulator, so that an fp16 C can be checked as the
 *       exact rounding of it.
 *  Sizes: M, N, K >= 0; M == 0 or N == 0 is a no-op; K == 0 writes zeros.
 *  Alignment: A, Bt 16-byte aligned; lda, ldb multiples of 8.
 *  Accuracy: per element |C - exact| <= 2e-3 * sum_k |A[i,k] * Bt[j,k]| (fp32
 *  accumulation in the tensor cores, order unspecified), plus the fp16
 *  rounding of C when c_dtype is IGC_F16.
 */
int gemm_f16(int64_t M, int64_t N, int64_t K,
             const void *A, int64_t lda,
             const void *Bt, int64_t ldb,
             void *C, int64_t ldc, int c_dtype,
             float *C_f32_check, int64_t ldc32,
             igc_stream_t stream);

/*
 * gemm_bf16 -- gemm_f16 with bf16 operands ([P1] §3.3: the f16 -> bf16 swap of
 * the tensor intrinsic), fp32 accumulation on the same tensor pipe.
 *
 *   C[i,j] = sum_{k<K} A[i,k] * Bt[j,k]
 *
 *  A, Bt as for gemm_f16 but bf16.  C is IGC_F32 (the accumulator) or IGC_BF16
 *  (round to nearest even of the fp32 accumulator); C_f32_check as for
 *  gemm_f16.  Sizes, alignment and accuracy bound as for gemm_f16, plus the
 *  bf16 rounding of C when c_dtype is IGC_BF16.
 */
int gemm_bf16(int64_t M, int64_t N, int64_t K,
              const void *A, int64_t lda,
              const void *Bt, int64_t ldb,
              void *C, int64_t ldc, int c_dtype,
              float *C_f32_check, int64_t ldc32,
              igc_stream_t stream);

/*
 * gemm_s8_zp -- INT8 GEMM with input zero points and requantisation
 * ([P1] §2.3: C = (A_q - zp_A)(B_q - zp_B) accumulated in int32, then the
 * dequantise / requantise step of the four-term fusion).
 *
 *   C32[i,j] = sum_{k<K} (A_q[i,k] - zA_i) * (B_q[k,j] - zB_j)     (int32, wraps mod 2^32)
 *   C8[i,j]  = clamp(rne(fp32(C32[i,j]) * scale_j), -128, 127)
 *
 *  A       device, M x K row-major bytes, uint8 (a_signed = 0) or int8 (a_signed = 1),
 *          row stride lda >= K bytes.
 *  Bt      device, B stored column-major: N x K row-major bytes, uint8 or int8
 *          (b_signed), row stride ldb >= K bytes.
 *  zA      per-tensor zero point of A, used when zA_row is NULL.
 *  zA_row  device int32[M] per-row zero points, or NULL.
 *  zB      per-tensor zero point of B, used when zB_col is NULL.
 *  zB_col  device int32[N] per-column zero points, or NULL.
 *  C32     device int32 M x N row-major (row stride ldc32 >= N), or NULL.
 *  C8      device int8 M x N row-major (row stride ldc8 >= N), or NULL.  At
 *          least one of C32 / C8 must be given.
 *  scale   per-tensor fp32 scale, used when scale_col is NULL.
 *  scale_col  device fp32[N] per-column scales, or NULL.
 *  workspace  device scratch of at least gemm_s8_zp_workspace_size(M, N, K)
 *          bytes, 256-byte aligned, owned by the caller, not shared with a
 *          concurrent call.  It holds the operands shifted to [-128, 127] and
 *          widened to fp16, and their row / column sums (whole, or per 1024-k
 *          chunk with one completion flag per 128 rows and chunk when the
 *          GEMM kernel converts the operands itself); nothing in it need
 *          survive between calls.
 *  Rounding: fp32(C32) rounds to nearest even; the product is one fp32
 *  multiply rounded to nearest even; the integer rounding is half-to-even; a
 *  NaN product gives 0.  Results are bit-exact (no tolerance).
 *  Sizes: M, N, K >= 0; M == 0 or N == 0 is a no-op; K == 0 writes zeros.
 *  Alignment: A, Bt 16-byte aligned; lda, ldb multiples of 16.
 */
int gemm_s8_zp(int64_t M, int64_t N, int64_t K,
               const void *A, int a_signed, int64_t lda,
               const void *Bt, int b_signed, int64_t ldb,
               int32_t zA, const int32_t *zA_row,
               int32_t zB, const int32_t *zB_col,
               int32_t *C32, int64_t ldc32,
               int8_t *C8, int64_t ldc8,
               float scale, const float *scale_col,
               void *workspace, size_t workspace_bytes,
               igc_stream_t stream);

/* Bytes of workspace gemm_s8_zp needs for an M x N x K problem (0 if any size < 0). */
size_t gemm_s8_zp_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * gemm_s8_zp is these two phases in sequence; they are exported so that a
 * caller can prepare a constant operand (e.g. quantised weights Bt) once and
 * reuse it, and so that each phase can be timed on its own.
 *
 * gemm_s8_zp_prepare -- the operand pre-pass: for each non-NULL operand,
 * writes its values shifted to [-128, 127] (minus 128 for uint8, unchanged
 * for int8) as fp16 into the workspace, with the row sums of the shifted
 * values.  A == NULL keeps the workspace's prepared A; Bt == NULL keeps B.
 * At least one must be non-NULL.  Arguments as for gemm_s8_zp; the
 * workspace must be sized for the same (M, N, K).
 *
 * gemm_s8_zp_run -- the tcgen05 GEMM over the prepared workspace with the
 * fused zero-point correction and requantisation; a_signed / b_signed must
 * be those the operands were prepared with.  Outputs and rounding as for
 * gemm_s8_zp.  The workspace is only read.
 */
int gemm_s8_zp_prepare(int64_t M, int64_t N, int64_t K,
                       const void *A, int a_signed, int64_t lda,
                       const void *Bt, int b_signed, int64_t ldb,
                       void *workspace, size_t workspace_bytes,
                       igc_stream_t stream);

int gemm_s8_zp_run(int64_t M, int64_t N, int64_t K, int a_signed, int b_signed,
                   int32_t zA, const int32_t *zA_row,
                   int32_t zB, const int32_t *zB_col,
                   int32_t *C32, int64_t ldc32,
                   int8_t *C8, int64_t ldc8,
                   float scale, const float *scale_col,
                   const void *workspace, size_t workspace_bytes,
                   igc_stream_t stream);

/*
 * gemm_s8_zp_dequant -- INT8 GEMM with zero points and a dequantised float
 * output, the "dequantize(C) + add_bias" half of [P1] §2.3's four-term fusion:
 *
 *   C32[i,j] = sum_{k<K} (A_q[i,k] - zA_i) * (B_q[k,j] - zB_j)          (int32)
 *   Y[i,j]   = ((fp32(C32[i,j]) * scale_row_i) * scale_col_j) + bias_j  (fp32)
 *
 * Each step is one fp32 operation rounded to nearest even, in this order, with
 * no fused multiply-add; a NULL scale_row / scale_col / bias vector skips its
 * step (scale 1, bias 0).  scale_row is device float[M] (the per-row scale of
 * A), scale_col and bias device float[N] (per-column scale of B, bias).
 * Y is device fp32 M x N row-major (row stride ldy >= N).  The other arguments,
 * the workspace, alignment and sizes are as for gemm_s8_zp, except that K must
 * be >= 1 (IGC_ERR_UNSUPPORTED otherwise).  Results are bit-exact.
 */
int gemm_s8_zp_dequant(int64_t M, int64_t N, int64_t K,
                       const void *A, int a_signed, int64_t lda,
                       const void *Bt, int b_signed, int64_t ldb,
                       int32_t zA, const int32_t *zA_row,
                       int32_t zB, const int32_t *zB_col,
                       const float *scale_row, const float *scale_col, const float *bias,
                       float *Y, int64_t ldy,
                       void *workspace, size_t workspace_bytes,
                       igc_stream_t stream);

/*
 * gemm_s8_zp_noalloc -- gemm_s8_zp without a caller-provided workspace, for
 * callers that cannot allocate device memory: for example code running
 * inside a host framework that owns all device memory through its own pool
 * and forbids direct cudaMalloc, or a service that must not allocate once it
 * is serving because an allocation could fail or stall in the middle of a
 * request.  (The pages have no counterpart of this entry point.)
 *
 * Same arguments, results and rounding as gemm_s8_zp, minus the workspace.
 * Its scratch is a fixed array of IGC_NOALLOC_SCRATCH_BYTES in the library's
 * device image; every GPU that loads the library holds that memory until the
 * process exits.  The call allocates nothing (no cudaMalloc, cudaFree or any
 * allocating library routine); the caller still provides inputs and outputs.
 *  - Problems whose gemm_s8_zp_workspace_size(M, N, K) exceeds
 *    IGC_NOALLOC_SCRATCH_BYTES are rejected with IGC_ERR_WORKSPACE before
 *    anything is enqueued (e.g. 2048^3 fits, 4096^3 does not).
 *  - When the array is reserved: the library's int8 kernels and this array
 *    sit in one device module, which CUDA loads on a device the first time
 *    the process uses it there (with lazy module loading, CUDA's default):
 *    the first call of this entry point, or any earlier gemm_s8_zp /
 *    gemm_s8_zp_prepare / gemm_s8_zp_run / gemm_s8_zp_dequant call.  That
 *    first use reserves the IGC_NOALLOC_SCRATCH_BYTES on the device and can
 *    fail if the device is full.  A caller that must not allocate while
 *    serving therefore makes one call per device at start-up, before its
 *    memory pool claims the GPU; later calls reserve nothing more.
 *  - The first call on a device also looks up the device address of the
 *    scratch array (cudaGetSymbolAddress, with that device current) and
 *    caches it once the lookup succeeds (a failed lookup returns
 *    IGC_ERR_CUDA and is tried again on the next call); make that first call
 *    before any stream capture.
 *  - Arguments are checked in gemm_s8_zp's order before the size: a bad
 *    argument returns IGC_ERR_INVALID_ARG / IGC_ERR_MISALIGNED whatever the
 *    size, and K == 0 (all outputs zero) needs no scratch.
 *  - Every call shares the one array and leaves its contents behind; each
 *    call rewrites everything it later reads, so nothing needs clearing.
 *    Calls that overlap on the GPU (e.g. on two streams at once) race on the
 *    scratch and give wrong results: serialise them.
 */
#define IGC_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int gemm_s8_zp_noalloc(int64_t M, int64_t N, int64_t K,
                       const void *A, int a_signed, int64_t lda,
                       const void *Bt, int b_signed, int64_t ldb,
                       int32_t zA, const int32_t *zA_row,
                       int32_t zB, const int32_t *zB_col,
                       int32_t *C32, int64_t ldc32,
                       int8_t *C8, int64_t ldc8,
                       float scale, const float *scale_col,
                       igc_stream_t stream);

/*
 * conv2d_nhwc_f16_implicit -- 2-D convolution (cross-correlation, no kernel
 * flip) as an implicit GEMM ([P3] "准备和算法"): no im2col tensor is built;
 * the A operand is gathered by TMA in im2col mode.
 *
 *   y[n,p,q,k] = sum_{r<R} sum_{s<S} sum_{c<C}
 *                xpad(n, p*stride_h + r - pad_h, q*stride_w + s - pad_w, c) * w[k,r,s,c]
 *
 *  with xpad = x inside [0,H) x [0,W) and 0 outside (zero padding), fp32
 *  accumulation, P = (H + 2*pad_h - R)/stride_h + 1, Q likewise.
 *
 *  x    device fp16 NHWC, N x H x W x C, dense.
 *  w    device fp16 KRSC, K x R x S x C, dense (= a K x (R*S*C) K-major matrix).
 *  y    device fp16 NHWC (N x P x Q x K), dense, round to nearest even.  May be
 *       NULL if y_f32_check is given.
 *  y_f32_check  device fp32 N x P x Q x K or NULL: copy of the fp32 accumulator.
 *  Supported: C a multiple of 8 (16-byte pixel rows), strides 1..8, padding
 *  with pad - (filter - 1) in [-128, 127] (the TMA im2col box corners), dense
 *  tensors, N*H*W*C < 2^31 and N*P*Q*K < 2^31; else IGC_ERR_UNSUPPORTED.
 *  When C is not a multiple of 128 the weights must be finite (padded channels
 *  meet the next tap's weights with a zero input).
 *  N == 0 is a no-op.  Accuracy as for gemm_f16 with the sum over the taps.
 */
int conv2d_nhwc_f16_implicit(int N, int H, int W, int C, int K, int R, int S,
                             int pad_h, int pad_w, int stride_h, int stride_w,
                             const void *x, const void *w,
                             void *y, float *y_f32_check,
                             igc_stream_t stream);

/*
 * conv2d_nhwc_s8_zp -- INT8 convolution as an implicit GEMM with input zero
 * points and requantisation: the pages' im2col lowering of the convolution
 * ([P1] §2.2) applied to the INT8 path ([P1] §2.3), with [P3]'s padded input.
 *
 *   y32[n,p,q,k] = sum_{r<R} sum_{s<S} sum_{c<C}
 *                  (xpad(n, p*stride_h + r - pad_h, q*stride_w + s - pad_w, c) - zX)
 *                  * (w[k,r,s,c] - zW_k)                               (int32, wraps)
 *   y8[n,p,q,k]  = clamp(rne(fp32(y32) * scale_k), -128, 127)
 *
 *  xpad is x inside [0,H) x [0,W) and zX outside: with asymmetric quantisation
 *  the input's real zero is its zero point, so padded taps contribute nothing.
 *  x       device NHWC bytes, uint8 (x_signed = 0) or int8 (x_signed = 1), dense.
 *  zX      per-tensor zero point of x; must be a value of x's type.
 *  w       device KRSC bytes, uint8 or int8 (w_signed), dense.
 *  zW / zW_k  per-tensor zero point of w, or device int32[K] per output channel.
 *  y32, y8 device NPQK int32 / int8 outputs (at least one non-NULL), dense.
 *  scale / scale_k  per-tensor fp32 scale, or device float[K] per output channel.
 *  workspace  device scratch of conv2d_nhwc_s8_zp_workspace_size(...) bytes,
 *          256-byte aligned, caller-owned: the padded, shifted input (fp16),
 *          the shifted weights (fp16) and the sums of both.
 *  Rounding and exactness as for gemm_s8_zp (bit-exact).  Supported: C a
 *  multiple of 8, strides 1..8, R, S <= 32, R*S*C < 2^24, x and w 16-byte
 *  aligned; N == 0 is a no-op.
 */
int conv2d_nhwc_s8_zp(int N, int H, int W, int C, int K, int R, int S,
                      int pad_h, int pad_w, int stride_h, int stride_w,
                      const void *x, int x_signed, int32_t zX,
                      const void *w, int w_signed, int32_t zW, const int32_t *zW_k,
                      int32_t *y32, int8_t *y8,
                      float scale, const float *scale_k,
                      void *workspace, size_t workspace_bytes,
                      igc_stream_t stream);

/* Bytes of workspace conv2d_nhwc_s8_zp needs (0 if the shape is invalid or unsupported). */
size_t conv2d_nhwc_s8_zp_workspace_size(int N, int H, int W, int C, int K, int R, int S,
                                        int pad_h, int pad_w, int stride_h, int stride_w);

/* Static description of a status code (never NULL). */
const char *igc_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns IGC_OK, IGC_ERR_DEVICE_TIMEOUT if a kernel's
 * bounded wait gave up since the last check (details via
 * igc_last_device_status()), or IGC_ERR_CUDA if the synchronisation failed.
 */
int igc_check_device_status(igc_stream_t stream);

/* Raw status word read by the last igc_check_device_status() call:
 * (code << 56) | (wait site << 32) | block index; 0 when none. */
uint64_t igc_last_device_status(void);

/*
 * Limit, in nanoseconds, of every kernel-side pipeline wait launched after
 * this call (default 2e9; values < 1000 are raised to 1000).  Returns the
 * previous limit.  Process-wide: it is the one setting shared by all threads
 * (a safety limit on how long a broken pipeline may wait, not a tuning knob;
 * it does not change any result).
 */
uint64_t igc_set_wait_limit_ns(uint64_t limit_ns);

/*
 * igc_plan_gemm -- the schedule a GEMM call would run with, computed on the
 * host by the decisions the launch makes (no device work; with clusters > 0 no
 * GPU is needed).
 *
 *  op        IGC_PLAN_GEMM_F16, IGC_PLAN_GEMM_BF16 or IGC_PLAN_GEMM_S8 (gemm_f16,
 *            gemm_bf16, gemm_s8_zp / gemm_s8_zp_run / gemm_s8_zp_dequant).
 *  M, N, K   the problem (all >= 1).
 *  clusters  CTA pairs that run at once (76 on GB300), or <= 0 for the current
 *            device's.
 *  out       int32[8], written: [0] tile width (columns of B per CTA pair),
 *            [1] pipeline stage depth in k (64 or 128), [2] m-tiles of 256 rows,
 *            [3] n-tiles, [4] first column-half unit (= tiles when the last
 *            round is not split), [5] work units, [6] CTAs launched, [7] leading
 *            units per CTA pair whose operand panels are prefetched into L2.
 *  The calling thread's igc_set_tile_width / igc_set_stage_depth overrides
 *  (igc_debug.h) apply.
 *  Returns IGC_OK, IGC_ERR_INVALID_ARG (null out, size < 1, unknown op),
 *  IGC_ERR_UNSUPPORTED (sizes beyond 2^31 - 1) or a device error when clusters
 *  <= 0 and no usable device is present.
 */
#define IGC_PLAN_GEMM_F16 0
#define IGC_PLAN_GEMM_BF16 1
#define IGC_PLAN_GEMM_S8 2
int igc_plan_gemm(int op, int64_t M, int64_t N, int64_t K, int clusters, int32_t *out);

/* Library version, "major.minor.patch". */
const char *igc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IGC_H */
