/*
 * qmm.h -- C ABI of the GB300 (sm_103a) integer-quantised matmul library.
 *
 * Four operations, each an integer matmul whose dequantisation is fused into
 * the kernel so that no dequantised (float) copy of a quantised operand is
 * ever written to memory:
 *   qmm_w8_dequant           float activations x int8 weight, scale/zero point
 *   qmm_a8w8                 int8 x int8 -> exact int32 -> row/column scales
 *   matmul_integer           ONNX MatMulInteger with zero points, shared B
 *   dynamic_quantize_linear  ONNX DynamicQuantizeLinear to uint8
 *
 * Conventions for every entry point:
 *  - Tensors are caller-owned DEVICE pointers, row-major and contiguous in the
 *    last dimension, on the current CUDA device. The library never allocates
 *    device or host memory and never takes ownership.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and runs asynchronously; the call returns after the launch.
 *  - Scales and zero points are device pointers too, so a chain of calls
 *    (e.g. dynamic_quantize_linear then matmul_integer) needs no host sync.
 *  - Arguments are validated before anything is launched; an invalid call
 *    returns QMM_ERR_INVALID_ARG (malformed) or QMM_ERR_UNSUPPORTED (well
 *    formed but outside what the kernels implement) and enqueues nothing.
 *  - The CUDA last-error state is cleared before each launch and read after
 *    it; a launch failure returns QMM_ERR_CUDA (qmm_last_cuda_error() gives
 *    the cudaError_t value).
 *  - Kernels never trap or spin without bound. A device-side wait that runs
 *    out (about one second) records a code in a device error word and the
 *    kernel returns; qmm_check_device_error() reports it as QMM_ERR_TIMEOUT.
 *  - Integer results wrap modulo 2^32 (two's complement); nothing saturates
 *    except the uint8 outputs of dynamic_quantize_linear.
 *  - Shapes use int64_t; each dimension must fit in int32 (< 2^31).
 *
 * The operations follow five public web pages; each declaration names the
 * page (title) and the section it implements.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QMM_OK = 0,
  QMM_ERR_INVALID_ARG = 1,
  QMM_ERR_UNSUPPORTED = 2,
  QMM_ERR_CUDA = 3,
  QMM_ERR_TIMEOUT = 4
} qmm_status;

/* Element types (values of the *_dtype arguments). */
typedef enum {
  QMM_F32 = 0,
  QMM_BF16 = 1,
  QMM_S8 = 2,
  QMM_U8 = 3,
  QMM_S32 = 4
} qmm_dtype;

/*
 * Form (a): int8-weight matmul with the affine dequantisation factored out.
 * TrainDeeploy PR #53, "feat(PULPOpen): matmul that dequantises an int8
 * weight in-kernel", section "The kernel":
 *     C[m,n] = scale_n * ( sum_k A[m,k]*B[k,n]  -  zp_n * sum_k A[m,k] )
 * i.e. sum_k A[m,k] * scale_n*(B[k,n] - zp_n) with one correction multiply per
 * output instead of one per multiply-accumulate.
 *
 *  A           [M,K] activations, a_dtype QMM_F32 or QMM_BF16
 *  B           [K,N] int8 weight
 *  scale       device float[scale_count], scale_count 1 (per tensor) or N (per column)
 *  zero_point  device int32[zp_count], zp_count 0 (no zero point), 1 or N; may be
 *              NULL when zp_count is 0
 *  C           [M,N] output, c_dtype QMM_F32 or QMM_BF16 (round to nearest even)
 * Kernels: for bf16 A with 1 <= M <= 16 (the decode shape; K % 8 == 0,
 * N % 16 == 0, A and B 16-byte aligned) a weight-streaming tensor-core GEMV
 * fed by TMA; otherwise a CUDA-core tiled kernel. Accumulation is fp32.
 * Accuracy: |C - exact| <= 1e-3 * sum_k |A[m,k]*scale_n*(B[k,n]-zp_n)| + 1e-6,
 * plus half an ulp of the output type.
 */
qmm_status qmm_w8_dequant(const void* A, int a_dtype, const int8_t* B, int64_t M, int64_t K, int64_t N,
                          const float* scale, int64_t scale_count, const int32_t* zero_point, int64_t zp_count,
                          void* C, int c_dtype, void* stream);

/*
 * qmm_w8_dequant_ws: the same operation, for large M (prefill) on the
 * tensor cores when a workspace is supplied. A pre-pass writes the int8
 * weight as exact bf16 into the workspace once (and the activations' row sums
 * when there is a zero point); an SM-pair GEMM (tcgen05 cta_group::2) then
 * multiplies bf16 activations by it with one fp32 accumulation over K and
 * applies scale_n * (acc - zp_n * rowsum(A)[m]) in its epilogue. fp32
 * activations are split into two bf16 parts (hi + lo, about 2^-16 relative)
 * along a doubled K that rereads the weight. Same accuracy bound as above.
 *
 * For 3 to 16 bf16 rows (K % 8 == 0, N % 16 == 0) the workspace serves the
 * decode GEMV instead: a pre-pass scales each activation row by the power of
 * two that puts its largest magnitude in [2^14, 2^15) and stores it as exact
 * fp16 (values below 2^-17 of the row maximum lose low bits, far inside the
 * bound above), and the GEMV multiplies fp16 activations by the weight
 * widened to fp16 in registers, undoing the row scale in its epilogue.
 *
 *  workspace   at least qmm_w8_dequant_workspace_bytes(a_dtype, M, K, N) bytes,
 *              16-byte aligned, caller-owned.
 * The size function returns 0 when neither path applies (M < 64 other than the
 * decode rows above, K or N not a multiple of 16); the call then runs
 * qmm_w8_dequant and ignores the workspace. The same happens for an unaligned
 * A (bf16: 16 bytes) or B.
 */
size_t qmm_w8_dequant_workspace_bytes(int a_dtype, int64_t M, int64_t K, int64_t N);
qmm_status qmm_w8_dequant_ws(const void* A, int a_dtype, const int8_t* B, int64_t M, int64_t K, int64_t N,
                             const float* scale, int64_t scale_count, const int32_t* zero_point, int64_t zp_count,
                             void* C, int c_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Form (b): A8W8 matmul-dequant. PyPTO PR #1920, "Feature/a8w8 matmul dequant
 * fusion", the walkthrough's sequence diagram (INT8 matmul into an INT32
 * accumulator, cast to FP32, act_scale on rows, weight_scale on columns, cast
 * to out_dtype) and the review comments on 1-D scales ([M] scales rows,
 * [N] scales columns, never a last-dimension broadcast):
 *     acc = sum_k A[m,k]*B[k,n]              (exact, int32, wrapping)
 *     C   = out( ((float)acc * act_scale[m]) * weight_scale[n] )
 * each float step a single fp32 multiply rounded to nearest even.
 *
 *  A             [M,K] int8;  B [K,N] int8
 *  act_scale     device float[act_count], act_count 1 (scalar) or M
 *  weight_scale  device float[w_count], w_count 1 or N
 *  C             [M,N], c_dtype QMM_F32 or QMM_BF16
 * Kernel: exact integer GEMM on the tcgen05 tensor cores with the scaling in
 * the epilogue. sm_103a has no 8-bit integer MMA kind, so the product runs on
 * fp16 copies of the bytes (exact) in K-chunks short enough for the fp32
 * accumulator to stay exact, drained into an int32 sum. Results are
 * bit-identical to the float32 chain above.
 */
qmm_status qmm_a8w8(const int8_t* A, const int8_t* B, int64_t M, int64_t K, int64_t N, const float* act_scale,
                    int64_t act_count, const float* weight_scale, int64_t w_count, void* C, int c_dtype,
                    void* stream);

/*
 * qmm_a8w8_ws: the same operation and bit-identical results as qmm_a8w8, with
 * a caller-provided workspace that lets large problems run in two passes: a
 * bandwidth-bound pre-pass writes exact fp16 copies of A and B into the
 * workspace once, and the GEMM then stages fp16 tiles with TMA straight into
 * the tensor-core layout on SM pairs, instead of converting every operand
 * tile once for each output tile that uses it.
 *
 *  workspace        device scratch of at least qmm_a8w8_workspace_bytes(M, K, N)
 *                   bytes, 16-byte aligned, caller-owned; contents on entry do
 *                   not matter, contents on return are unspecified.
 * qmm_a8w8_workspace_bytes returns 0 when the two-pass path does not apply to
 * the shape (M < 256, or K or N not a multiple of 16); the call then runs
 * qmm_a8w8 and ignores the workspace (which may be NULL). The same happens
 * when A or B is not 16-byte aligned.
 */
size_t qmm_a8w8_workspace_bytes(int64_t M, int64_t K, int64_t N);
qmm_status qmm_a8w8_ws(const int8_t* A, const int8_t* B, int64_t M, int64_t K, int64_t N, const float* act_scale,
                       int64_t act_count, const float* weight_scale, int64_t w_count, void* C, int c_dtype,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * The two passes of qmm_a8w8_ws as separate calls, for callers that time or
 * schedule them apart, or that run several products on the same packed
 * operands (e.g. the same A and B with different scales):
 *   qmm_a8w8_pack    writes the fp16 copies of A and B into the workspace;
 *   qmm_a8w8_packed  runs the SM-pair GEMM and the fused scaling on them.
 * qmm_a8w8_pack(...) followed by qmm_a8w8_packed(...) on one stream gives the
 * same result as qmm_a8w8_ws. Both return QMM_ERR_UNSUPPORTED when
 * qmm_a8w8_workspace_bytes(M, K, N) is 0; pack requires 16-byte-aligned A and
 * B. The workspace must not be modified between the two calls.
 */
qmm_status qmm_a8w8_pack(const int8_t* A, const int8_t* B, int64_t M, int64_t K, int64_t N, void* workspace,
                         size_t workspace_bytes, void* stream);
qmm_status qmm_a8w8_packed(int64_t M, int64_t K, int64_t N, const float* act_scale, int64_t act_count,
                           const float* weight_scale, int64_t w_count, void* C, int c_dtype, const void* workspace,
                           size_t workspace_bytes, void* stream);


/*
 * qmm_a8w8 from HOST buffers, with the copies overlapped with the work: the
 * same operation and bit-identical results as qmm_a8w8_ws, for callers whose
 * operands and result live in host memory.
 *
 *  hA, hB                 host int8 [M,K] and [K,N]
 *  h_act_scale            host float[act_count], 1 or M
 *  h_weight_scale         host float[w_count], 1 or N
 *  hC                     host [M,N] float (QMM_F32) or bf16 bits (QMM_BF16)
 *  workspace              device, at least qmm_a8w8_host_workspace_bytes(...)
 *                         bytes, 16-byte aligned: the device copies of the
 *                         operands, scales and result, then the two-pass
 *                         path's workspace
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to run asynchronously; they must stay valid and unchanged until
 * the work on `stream` completes (hC is written by then).
 * Where the two-pass path applies (qmm_a8w8_workspace_bytes(M, K, N) > 0), the
 * copies in run on one internal copy stream, the pre-passes and GEMMs on
 * `stream` as soon as their operands have arrived, and the copies of C back on
 * a second internal stream as soon as each part is written, so the copies in
 * both directions overlap the GEMMs. From 512 rows and 1024 columns on the
 * work is 2 x 2 blocks (A in two row panels, B in two column panels copied as
 * pitched panels; each block's C goes back as a pitched copy), so the first
 * GEMM needs a quarter of each operand; below that, all of B and then A's row
 * panels, sized so each panel's pair tiles fill whole waves. Elsewhere the
 * call copies in, runs qmm_a8w8 and copies out on `stream`. Calls on one
 * device enqueue one at a time (the internal streams and events are shared).
 * Errors: as qmm_a8w8_ws, plus QMM_ERR_CUDA when a copy cannot be enqueued.
 */
size_t qmm_a8w8_host_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t act_count, int64_t w_count,
                                     int c_dtype);
qmm_status qmm_a8w8_host(const int8_t* hA, const int8_t* hB, int64_t M, int64_t K, int64_t N,
                         const float* h_act_scale, int64_t act_count, const float* h_weight_scale, int64_t w_count,
                         void* hC, int c_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Accumulating A8W8. PyPTO PR #1920, "What Changed", "A8W8 matmul-dequant-acc
 * op" (an INT32 accumulator input beside the INT8 operands, [M] or [M,1]
 * activation scales, [N] or [1,N] weight scales, FP32 or BF16 output, a_trans /
 * b_trans dimension inference), lowered there to matmul_acc (gemv_acc for
 * M == 1), the cast and the two scale multiplies:
 *     acc = acc_in[m,n] + sum_k A[m,k]*B[k,n]   (exact, int32, wrapping)
 *     C   = out( ((float)acc * act_scale[m]) * weight_scale[n] )
 * the float steps exactly those of qmm_a8w8 (which this equals for acc_in 0).
 *
 *  A          int8, [M,K] row-major, or [K,M] when a_trans = 1
 *  B          int8, [K,N] row-major, or [N,K] when b_trans = 1
 *  acc_in     device int32 [M,N] row-major, or NULL (zero)
 *  acc_out    device int32 [M,N] or NULL: receives acc (before any scaling),
 *             e.g. to pass a partial sum over part of K to the next call;
 *             may be the same array as acc_in (each element is read before
 *             it is written), may not overlap it otherwise
 *  act_scale, act_count, weight_scale, w_count, C, c_dtype   as in qmm_a8w8;
 *             C may be NULL when acc_out is given (then only acc_out is
 *             written and the scales are not read)
 *  workspace  at least qmm_a8w8_acc_workspace_bytes(M, K, N) bytes, 16-byte
 *             aligned, caller-owned (NULL allowed when that size is 0)
 * Any M, K, N >= 0 and any alignment of A, B. Kernels: a pre-pass writes
 * exact fp16 copies of A and B (transposing a transposed operand, rows padded
 * to 16 bytes), then the SM-pair tensor-core GEMM with the accumulator and the
 * scaling in its epilogue. K = 0 passes acc_in through (one elementwise kernel).
 * Errors: QMM_ERR_INVALID_ARG for a bad flag, count, null pointer or too small
 * a workspace, and when both C and acc_out are NULL.
 */
size_t qmm_a8w8_acc_workspace_bytes(int64_t M, int64_t K, int64_t N);
qmm_status qmm_a8w8_acc(const int8_t* A, int a_trans, const int8_t* B, int b_trans, int64_t M, int64_t K, int64_t N,
                        const int32_t* acc_in, int32_t* acc_out, const float* act_scale, int64_t act_count,
                        const float* weight_scale, int64_t w_count, void* C, int c_dtype, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Form (c): MatMulInteger with zero points. ROCm hip-ep PR #1248,
 * "feat(onnx-to-hip): lower quantized integer conv and matmul", section
 * "What", MatMulInteger paragraph:
 *     C[b,m,n] = sum_k (A[b,m,k] - a_zp) * (B[b,k,n] - b_zp)     (int32, wrapping)
 * ranks 2-4 with the batch dimensions flattened into `batch` by the caller;
 * a rank-2 B (or one whose batch dims are all 1) is one matrix shared by all
 * batches: pass b_batch_stride = 0. A size-1 batch on A is expanded: pass
 * a_batch_stride = 0.
 *
 *  A               [batch][M][K] 8-bit, a_dtype QMM_S8 or QMM_U8
 *  B               [batch][K][N] 8-bit, b_dtype QMM_S8 or QMM_U8
 *  a_batch_stride  elements between A batches (M*K for a dense batch, 0 = broadcast)
 *  b_batch_stride  elements between B batches (K*N, or 0 = shared rank-2 B)
 *  a_zero_point    device array of a_dtype: a_zp_count 0 (none), 1 (scalar) or M (per row)
 *  b_zero_point    device array of b_dtype: b_zp_count 0, 1 or N (per column)
 *  C               [batch][M][N] int32, contiguous
 * Computed as sum ab - a_zp*colsum(B) - b_zp*rowsum(A) + K*a_zp*b_zp, exact
 * modulo 2^32, with the row/column sums taken in the same pass as the product.
 */
qmm_status matmul_integer(const void* A, int a_dtype, const void* B, int b_dtype, int64_t batch, int64_t M,
                          int64_t K, int64_t N, int64_t a_batch_stride, int64_t b_batch_stride,
                          const void* a_zero_point, int64_t a_zp_count, const void* b_zero_point,
                          int64_t b_zp_count, int32_t* C, void* stream);

/*
 * matmul_integer_ws: the same operation and results as matmul_integer, run in
 * two passes when a workspace is supplied: the pre-pass writes exact fp16
 * copies of A and B together with rowsum(A) (when b_zp is given) and
 * colsum(B) (when a_zp is given), then the SM-pair GEMM reads fp16 tiles with
 * TMA and applies the zero-point expansion with the precomputed sums.
 *
 *  workspace   at least matmul_integer_workspace_bytes(batch, M, K, N,
 *              a_batch_stride, b_batch_stride) bytes, 16-byte aligned.
 * The size function returns 0 when the two-pass path does not apply: M < 256
 * after folding a dense batch over a shared B into M, K or N not a multiple
 * of 16, or batch strides other than 0 or dense. The call then runs
 * matmul_integer and ignores the workspace; likewise for unaligned A or B.
 */
size_t matmul_integer_workspace_bytes(int64_t batch, int64_t M, int64_t K, int64_t N, int64_t a_batch_stride,
                                      int64_t b_batch_stride);
qmm_status matmul_integer_ws(const void* A, int a_dtype, const void* B, int b_dtype, int64_t batch, int64_t M,
                             int64_t K, int64_t N, int64_t a_batch_stride, int64_t b_batch_stride,
                             const void* a_zero_point, int64_t a_zp_count, const void* b_zero_point,
                             int64_t b_zp_count, int32_t* C, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * ConvInteger. ROCm hip-ep PR #1248, "What", ConvInteger paragraph: rank-4
 * NCHW, and rank-3 NCL widened to a unit spatial row (the caller passes H = 1,
 * kH = 1 and zero top/bottom pads; the result is then [N, M, 1, oW]); a
 * scalar activation zero point; a scalar or per-output-channel weight zero
 * point. With Cg = C / group, Mg = M / group and g = m / Mg:
 *   y[n,m,oh,ow] = sum_{c<Cg, kh, kw} (xs[n, g*Cg + c, oh*sh + kh*dh - pt, ow*sw + kw*dw - pl])
 *                                     * (w[m,c,kh,kw] - w_zp[m])           (exact, int32, wrapping)
 * where xs = x - x_zp inside the input and 0 at padded positions (the page
 * leaves the pad value open; this is the convolution of the shifted tensors).
 *
 *  x            [N,C,H,W] 8-bit (x_dtype QMM_U8 / QMM_S8), device
 *  w            [M,C/group,kH,kW] 8-bit (w_dtype), device
 *  pads         host int64[4] {top, left, bottom, right} (ONNX order), or NULL (all 0)
 *  strides      host int64[2] {h, w}, or NULL (1, 1)
 *  dilations    host int64[2] {h, w}, or NULL (1, 1)
 *  group        >= 1, dividing C and M
 *  x_zero_point device, one value of x's type, or NULL (0)
 *  w_zero_point device, w_zp_count (0, 1 or M) values of w's type
 *  y            device int32 [N,M,oH,oW], oH = (H + pt + pb - dh*(kH-1) - 1)/sh + 1 (same for W)
 *  workspace    at least conv_integer_workspace_bytes(...) bytes, 16-byte aligned
 * Kernels, when each group has a whole number of 64-channel blocks (C/group %
 * 64 == 0), oH*oW % 4 == 0, strides <= 8 and the padded window's bounding box
 * is within 128 pixels of the input's edges: an implicit GEMM. x - x_zp is
 * written as fp16 channels-innermost (NHWC) and w - w_zp as fp16 in (kh, kw,
 * c) order; the SM-pair GEMM gathers each stage's 128 output pixels x 64
 * channels of one tap with an im2col tensor copy (padding reads as zero, i.e.
 * as x_zp before the shift) and stores the exact sums into NCHW. Otherwise:
 * the weight as exact fp16 with its row sums, an im2col pre-pass that writes
 * each image's [C*kH*kW, oH*oW] matrix as exact fp16 (padded positions
 * holding x_zp) with its column sums, then the SM-pair MatMulInteger GEMM with
 * A = the weight (per-row zero point w_zp), B = the im2col matrix (zero point
 * x_zp), one batch per (image, group), its rows written straight into NCHW.
 * conv_integer_workspace_bytes sizes the route the call will take.
 * Errors: QMM_ERR_INVALID_ARG for a bad dtype, geometry (group not dividing C
 * and M, non-positive extents, strides or dilations, negative pads), zero-point
 * count, null pointer or too small a workspace; QMM_ERR_UNSUPPORTED above
 * 65535 (image, group) pairs per call. An empty output (N = 0, or a kernel wider than the
 * padded input) launches nothing.
 */
size_t conv_integer_workspace_bytes(int64_t N, int64_t C, int64_t H, int64_t W, int64_t M, int64_t kH, int64_t kW,
                                    const int64_t* pads, const int64_t* strides, const int64_t* dilations,
                                    int64_t group);
qmm_status conv_integer(const void* x, int x_dtype, const void* w, int w_dtype, int64_t N, int64_t C, int64_t H,
                        int64_t W, int64_t M, int64_t kH, int64_t kW, const int64_t* pads, const int64_t* strides,
                        const int64_t* dilations, int64_t group, const void* x_zero_point, const void* w_zero_point,
                        int64_t w_zp_count, int32_t* y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The chain DynamicQuantizeLinear -> MatMulInteger -> dequantise, in one call.
 * ROCm hip-ep PR #1248, "Why" and "What": a graph using MatMulInteger casts,
 * scales and adds the bias after it. Each step below is one fp32 operation
 * rounded to nearest even:
 *   (y, y_scale, y_zp) = DynamicQuantizeLinear(x)            (as dynamic_quantize_linear)
 *   acc[m,n] = sum_k (y[m,k] - y_zp) * (W[k,n] - w_zp[n])    (exact, int32, wrapping)
 *   C[m,n]   = f32(f32(acc) * f32(y_scale * w_scale[n]))  (+ bias[n], one more rounding)
 *
 *  x             device float [M,K]
 *  W             device 8-bit [K,N] (w_dtype QMM_S8 or QMM_U8)
 *  w_scale       device float[w_scale_count], 1 or N
 *  w_zero_point  device, w_zp_count (0, 1 or N) values of W's type
 *  bias          device float[N], or NULL
 *  C             device float [M,N]
 *  y_scale, y_zero_point  device float[1] / uint8[1] receiving the quantiser's
 *                scale and zero point, or NULL (then kept in the workspace)
 *  workspace     at least dynamic_quantize_matmul_workspace_bytes(M, K, N), 16-byte aligned
 * Kernels: the quantiser's min/max pass; the weight as exact fp16 with its
 * column sums; the quantize pass writing y straight into the GEMM's fp16 A
 * operand with y's row sums (no uint8 tensor in between); the SM-pair
 * MatMulInteger GEMM whose epilogue applies the zero points, the multiplier
 * and the bias and stores fp32 (no int32 tensor in between).
 * Errors: QMM_ERR_INVALID_ARG for a bad dtype, count, null pointer or too small
 * a workspace; QMM_ERR_UNSUPPORTED for K = 0. M = 0 or N = 0 launches nothing.
 */
size_t dynamic_quantize_matmul_workspace_bytes(int64_t M, int64_t K, int64_t N);
qmm_status dynamic_quantize_matmul(const float* x, int64_t M, int64_t K, const void* W, int w_dtype, int64_t N,
                                   const float* w_scale, int64_t w_scale_count, const void* w_zero_point,
                                   int64_t w_zp_count, const float* bias, float* C, float* y_scale,
                                   uint8_t* y_zero_point, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same chain on a weight packed once. TrainDeeploy PR #53, first
 * paragraph: the weight is a frozen constant, so its exact fp16 copy and
 * column sums need not be redone on every call.
 *   dynamic_quantize_matmul_pack_weight  writes, into `packed` (device, at
 *       least dynamic_quantize_matmul_weight_bytes(K, N) bytes, 16-byte
 *       aligned, caller-owned), W [K,N] of w_dtype as exact fp16 rows of
 *       pitch N rounded up to 8, then colsum(W) as int32[N];
 *   dynamic_quantize_matmul_packed  runs the quantiser on x and the GEMM with
 *       its epilogue on that buffer: the same results, bit for bit, as
 *       dynamic_quantize_matmul on the unpacked W. K, N and w_dtype must be
 *       the ones the buffer was packed with, and the buffer must not change
 *       in between (neither is checked on the device). The workspace holds
 *       y's fp16 copy, its row sums and the quantiser's partials:
 *       dynamic_quantize_matmul_packed_workspace_bytes(M, K) bytes, 16-byte
 *       aligned. The zero points and the scales stay arguments of each call.
 * Errors: as dynamic_quantize_matmul, plus QMM_ERR_INVALID_ARG for a null,
 * unaligned or too short packed buffer. The size functions return 0 for an
 * empty or out-of-range extent.
 */
size_t dynamic_quantize_matmul_weight_bytes(int64_t K, int64_t N);
qmm_status dynamic_quantize_matmul_pack_weight(const void* W, int w_dtype, int64_t K, int64_t N, void* packed,
                                               size_t packed_bytes, void* stream);
size_t dynamic_quantize_matmul_packed_workspace_bytes(int64_t M, int64_t K);
qmm_status dynamic_quantize_matmul_packed(const float* x, int64_t M, int64_t K, const void* packed,
                                          size_t packed_bytes, int w_dtype, int64_t N, const float* w_scale,
                                          int64_t w_scale_count, const void* w_zero_point, int64_t w_zp_count,
                                          const float* bias, float* C, float* y_scale, uint8_t* y_zero_point,
                                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Form (d): DynamicQuantizeLinear, uint8 only. ROCm hip-ep PR #1248, section
 * "What", DynamicQuantizeLinear paragraph (reduce to a scalar min and max,
 * scale (max-min)/255 with a zero range selecting scale 1, ties-to-even zero
 * point, quantize), with the range widened to include 0:
 *     lo = min(0, min x); hi = max(0, max x)
 *     scale = (hi - lo) == 0 ? 1 : (hi - lo) / 255
 *     zp    = sat_u8(rne(-lo / scale))
 *     y     = sat_u8(rne(x / scale) + zp)
 * every step one IEEE fp32 operation (true division), ties to even.
 *
 *  x             [n] float32 (NaN/Inf inputs are outside the domain: undefined)
 *  y             [n] uint8 output
 *  y_scale       device float[1] output
 *  y_zero_point  device uint8[1] output
 *  row_sums      optional device int32[n / row_len]: the sum of each run of
 *                row_len elements of y (the rowsum(A) of a following
 *                matmul_integer); NULL to skip. Requires n % row_len == 0.
 *  workspace     device scratch of at least
 *                dynamic_quantize_linear_workspace_bytes(n) bytes, 16-byte
 *                aligned, caller-owned; its contents on entry do not matter.
 * n == 0 writes scale 1 and zero point 0.
 */
size_t dynamic_quantize_linear_workspace_bytes(int64_t n);
qmm_status dynamic_quantize_linear(const float* x, int64_t n, uint8_t* y, float* y_scale, uint8_t* y_zero_point,
                                   int32_t* row_sums, int64_t row_len, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * dynamic_quantize_linear_noalloc: the same operation and results as
 * dynamic_quantize_linear, for callers that cannot allocate device memory and
 * so cannot supply a workspace -- e.g. a plugin inside a host framework that
 * owns all device memory, an engine whose memory is fixed at start-up, or a
 * host thread that must not call cudaMalloc because it can synchronise the
 * device. The pages have no counterpart; this is a library convenience.
 *
 * The scratch for the (min, max) partials is a fixed 8 KiB array inside the
 * library (room for 1024 partials, which covers every n); every GPU that loads
 * the library keeps it until the process exits. The call allocates nothing.
 * The first call on a device looks the array's device address up (once, with
 * that device current), so make that first call before any stream capture.
 * All calls share the array: calls whose kernels overlap on the GPU race and
 * give wrong results -- order them on one stream. Nothing in the array needs
 * to start at zero. Arguments as for dynamic_quantize_linear (minus the
 * workspace); QMM_ERR_UNSUPPORTED if the partials would not fit the array.
 * This entry point does not update qmm_last_kernel()/qmm_last_cuda_error().
 */
qmm_status dynamic_quantize_linear_noalloc(const float* x, int64_t n, uint8_t* y, float* y_scale,
                                           uint8_t* y_zero_point, int32_t* row_sums, int64_t row_len,
                                           void* stream);

/*
 * Failure-path test hook (no operation of the pages). Runs qmm_a8w8_packed
 * with one fault planted on the host side of the launch: the first SM pair
 * issues neither the arrival nor the copies of its first operand stage, so
 * that pair's MMA issuer waits for data that never comes. Its wait runs out
 * after wait_limit_ns (1 us .. 100 ms; the pair's other waits after four
 * times that), the pair records site 0x401 (operand stage never filled) in the
 * device error word, abandons its tiles, drains, frees its tensor memory and
 * returns; every other pair computes its tiles as usual. Nothing traps and
 * the context stays usable: qmm_check_device_error() then returns
 * QMM_ERR_TIMEOUT with qmm_last_device_error() == 0x401. The output tiles
 * of the stalled pair are left unwritten. Arguments as for
 * qmm_a8w8_packed; QMM_ERR_INVALID_ARG for a limit outside the range.
 */
qmm_status qmm_test_a8w8_packed_stall(int64_t M, int64_t K, int64_t N, const float* act_scale, int64_t act_count,
                                      const float* weight_scale, int64_t w_count, void* C, int c_dtype,
                                      const void* workspace, size_t workspace_bytes, uint64_t wait_limit_ns,
                                      void* stream);

/*
 * Measurement aid (no operation of the pages): enqueue one launch of a kernel
 * that issues nothing but warp-level integer MMAs (mma.sync m16n8k32,
 * s8 x s8 -> s32, register operands, eight independent accumulators per warp)
 * on every SM, `iters` rounds per warp. *ops receives the integer operations
 * the launch performs (2*16*8*32 per MMA); divided by the launch's
 * event-timed duration it gives the rate of the legacy int8 tensor path, the
 * denominator of an "% of int8 tensor peak" figure. QMM_ERR_INVALID_ARG when
 * iters < 1 or ops is NULL.
 */
qmm_status qmm_int8_mma_peak_launch(int iters, double* ops, void* stream);

/*
 * Decode form (a) on a weight packed once. TrainDeeploy PR #53 ("matmul that
 * dequantises an int8 weight in-kernel", section "The kernel"): the same
 * operation and tolerance as qmm_w8_dequant for bf16 activations, 1 <= M <= 16
 * rows, with the int8 weight W [K,N] first re-laid out once (as for any frozen
 * weight) into the order the decode kernel's tensor-core fragments read it:
 * the same K x N bytes (K padded to 16, N to 64), each biased by 128, so that
 * a warp reads each 16-row step as one contiguous KB and widens every byte to
 * fp16 with about one instruction. The per-call work reads the packed weight
 * once and never forms a dequantised copy.
 *   qmm_w8_decode_pack_bytes(K, N)       bytes of the packed weight (0: shape
 *                                        unsupported: K or N not a multiple of 8)
 *   qmm_w8_pack_decode_weight(W, K, N, packed, bytes, stream)
 *                                        W int8 [K,N] device -> packed (caller-owned,
 *                                        16-byte aligned device memory)
 *   qmm_w8_dequant_packed_workspace_bytes(M, K)
 *                                        the activations' fp16 copy (rows padded to 8 or 16)
 *   qmm_w8_dequant_packed(A, M, K, N, packed, bytes, scale, scale_count,
 *                         zero_point, zp_count, C, c_dtype, workspace, bytes, stream)
 *       A bf16 [M,K] (16-byte aligned), scale / zero_point / C as for
 *       qmm_w8_dequant. QMM_ERR_UNSUPPORTED outside 1 <= M <= 16, K % 8, N % 8;
 *       QMM_ERR_INVALID_ARG for short or unaligned buffers.
 */
size_t qmm_w8_decode_pack_bytes(int64_t K, int64_t N);
qmm_status qmm_w8_pack_decode_weight(const int8_t* W, int64_t K, int64_t N, void* packed, size_t packed_bytes,
                                     void* stream);
size_t qmm_w8_dequant_packed_workspace_bytes(int64_t M, int64_t K);
qmm_status qmm_w8_dequant_packed(const void* A, int64_t M, int64_t K, int64_t N, const void* packed,
                                 size_t packed_bytes, const float* scale, int64_t scale_count,
                                 const int32_t* zero_point, int64_t zp_count, void* C, int c_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Human-readable name of a status. Never NULL. */
const char* qmm_status_string(int status);

/* Name of the kernel(s) the last successful call on this host thread launched
 * (a test hook: it shows which path actually ran). Never NULL. */
const char* qmm_last_kernel(void);

/* cudaError_t of the last call that returned QMM_ERR_CUDA on this thread. */
int qmm_last_cuda_error(void);

/* Synchronise `stream`, then read and clear the device error word of the
 * current device: QMM_OK if no kernel timed out since the last check,
 * QMM_ERR_TIMEOUT if one did (qmm_last_device_error() gives its site code),
 * QMM_ERR_CUDA if the synchronisation failed. */
qmm_status qmm_check_device_error(void* stream);
unsigned qmm_last_device_error(void);

/* Number of streaming multiprocessors of the current device (0 on error). */
int qmm_num_sms(void);

/* ABI version of this header: 1. */
int qmm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
