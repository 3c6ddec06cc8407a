// Host-side launch interfaces of the sm_103a kernels (internal to the library).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace qmm {

// ---------------------------------------------------------------------------
// Exact 8-bit GEMM on tcgen05 (A8W8 and MatMulInteger epilogues).
// ---------------------------------------------------------------------------
struct GemmArgs {
  const uint8_t* A;        // [batch][M][K] 8-bit, row-major
  const uint8_t* B;        // [batch][K][N] 8-bit, row-major
  long long a_bstride;     // elements between batches of A (0 = one A for all)
  long long b_bstride;     // elements between batches of B (0 = shared B)
  int batch, M, K, N;
  // epilogue, A8W8: C = bf16/f32( f32(acc) * act_scale[m] * weight_scale[n] )
  void* C;                 // [batch][M][N]
  int c_f32;               // A8W8 only: 1 = f32 out, 0 = bf16 out
  const float* act_scale;  int act_count;   // 1 or M
  const float* w_scale;    int w_count;     // 1 or N
  // epilogue, MatMulInteger: C = acc - za*colsum(B) - zb*rowsum(A) + K*za*zb (int32, wrapping)
  const void* a_zp;        int a_zp_count;  // 0 (none), 1, or per row
  const void* b_zp;        int b_zp_count;  // 0 (none), 1, or N
  int zp_row_mod;          // row index modulus for per-row a_zp / act_scale
  unsigned* err;           // device error word
};

// mmi = MatMulInteger epilogue (int32 out); otherwise A8W8 (s8 x s8 only).
// chunk_k: K-chunk length between exact drains (multiple of 64).
cudaError_t launch_gemm_tc(const GemmArgs& a, bool a_u8, bool b_u8, bool mmi, int chunk_k, cudaStream_t s,
                           const char** kernel_name);

// The same GEMM on a CTA pair (tcgen05 cta_group::2, 256 x 256 pair tiles).
// Requires 16-byte-aligned operand rows (the TMA path) and M >= 256.
cudaError_t launch_gemm_tc_pair(const GemmArgs& a, bool a_u8, bool b_u8, bool mmi, int chunk_k, int c_vec,
                                cudaStream_t s, const char** kernel_name);

// The same GEMM on SM pairs from exact fp16 copies of the operands (made by
// the pre-pass below), with the MatMulInteger row/column sums precomputed.
struct GemmF16Args {
  const void* A16;         // fp16 [batch][M][K] (or one [M][K] when a_bstride == 0)
  const void* B16;         // fp16 [batch][K][N] (or one [K][N] when b_bstride == 0)
  long long a_bstride;     // elements between batches (0 = shared)
  long long b_bstride;
  int batch, M, K, N;
  void* C;                 // [batch][M][N]
  int c_f32;
  const float* act_scale;  int act_count;
  const float* w_scale;    int w_count;
  const void* a_zp;        int a_zp_count;
  const void* b_zp;        int b_zp_count;
  const int* rowsum;       // MatMulInteger with b_zp: rowsum(A), [batch or 1][M]; form (a): fp32 row sums
  const int* colsum;       // MatMulInteger with a_zp: colsum(B), [batch or 1][N]
  int zp_row_mod;
  unsigned* err;
  // form (a) (bf16 A x bf16 copy of the int8 weight, fp32 accumulation): the
  // weight's K coordinate wraps at fa_kwrap when A holds [hi | lo] halves of
  // fp32 activations (0: no wrap); scale = w_scale/w_count, zp = b_zp (int32)
  int fa_kwrap;
  // row pitches of the fp16 copies in elements (0: dense, K for A and N for B;
  // otherwise a multiple of 8, the operand padded on the right)
  int a_pitch, b_pitch;
  // accumulating A8W8: int32 [M][N] added to the exact product before the
  // scaling (wrapping), and/or written with the combined sums; with C null only
  // acc_out is written (act_scale / w_scale unused)
  const int* acc_in;
  int* acc_out;
  // MatMulInteger followed by the dequantisation of a DynamicQuantizeLinear
  // chain (f32 out): C = f32(f32(acc) * f32(act_scale[0] * w_scale[n])) (+ bias[n])
  const float* bias;
  // A's batch index is b % a_bmod when a_bmod > 0 (a weight shared by every
  // image, one slice per convolution group); per-row zero points and row sums
  // are then indexed (b % a_bmod) * M + row
  int a_bmod;
  // implicit-GEMM convolution (launch_gemm_f16pair_conv): B is gathered per
  // stage from an fp16 NHWC input by im2col tensor copies instead of read from
  // B16. K runs over (tap row r, tap column s, 64-channel block) with the
  // channel block fastest, N over the output pixels of one image (oh * oW +
  // ow), and batch b is image b / cv_G, group b % cv_G.
  int cv_oW, cv_sh, cv_sw, cv_pt, cv_pl, cv_dh, cv_dw, cv_kW;
  int cv_cb;   // 64-channel blocks per group
  int cv_G, cv_Cg;
  // failure-path test hook (0 = off): the first cluster issues neither the
  // arrival nor the copies of its first ring stage, so its MMA thread's wait
  // for that stage runs out after wait_ns (the other roles' waits after
  // 4 * wait_ns) and the kernel takes its abort path
  int stall_test;
  unsigned long long wait_ns;   // 0: the default limit of every wait
};
cudaError_t launch_gemm_f16pair(const GemmF16Args& a, bool a_u8, bool b_u8, bool mmi, int chunk_k, cudaStream_t s,
                                const char** kernel_name);
// ConvInteger as an implicit GEMM on the same engine: A = the fp16 weight
// [G][Mg][K] in (r, s, c) order, B = im2col copies of the fp16 NHWC input
// described by tx (rank 4, {C, W, H, N}, 64 channels x 128 pixels, 128-byte
// swizzle), C int32 [N * G][Mg][P]; the operands already hold x - x_zp and
// w - w_zp, so the epilogue stores the exact sums unchanged.
// Pair-tile width (output pixels) the convolution launch uses for these
// arguments: 256, 224 or 192. The im2col map's pixel box must be half of it.
int conv_tile_width(const GemmF16Args& a);
cudaError_t launch_gemm_f16pair_conv(const GemmF16Args& a, const CUtensorMap& tx, cudaStream_t s,
                                     const char** kernel_name);

// Form (a) on the same engine: C = scale[n] * (A @ W - zp[n] * rowsum(A)[m]),
// A bf16 [M][K_eff] (K_eff = a.K: the weight's w_k, or 2*Kp for split fp32
// activations), W the bf16 copy [w_k][N]; one fp32 accumulation over K_eff.
cudaError_t launch_gemm_w8_bf16pair(const GemmF16Args& a, int w_k, cudaStream_t s, const char** kernel_name);

// Form (a) pre-pass: int8 -> exact bf16 (byte counts multiples of 16); fp32 row
// sums of bf16 rows (K % 8 == 0); fp32 rows -> [hi | lo] bf16 halves of width
// Kp each (optional fp32 row sums).
cudaError_t launch_convert_s8_bf16(const void* src, void* dst, long long bytes, cudaStream_t s);
cudaError_t launch_rowsum_bf16(const void* A, long long rows, int K, float* rowsum, cudaStream_t s);
cudaError_t launch_split_f32(const float* A, long long rows, int K, int Kp, void* out, float* rowsum,
                             cudaStream_t s);

// General pre-pass plane: an 8-bit [rows][cols] matrix at a byte pitch, copied
// (trans = 0: dst[r][c] = src[r][c]) or transposed (trans = 1: dst[c][r] =
// src[r][c]) into exact fp16 at an element pitch that is a multiple of 8.
struct ConvPlane {
  const void* src;
  long long src_pitch;     // bytes between source rows
  int rows, cols;          // source extent
  int trans;
  __half* dst;
  long long dst_pitch;     // fp16 elements between destination rows
};
// Both planes in one launch (a plane with rows or cols 0 is skipped).
cudaError_t launch_convert_planes(const ConvPlane& a, bool au, const ConvPlane& b, bool bu, cudaStream_t s);
// The accumulating A8W8 with an empty K: acc = acc_in (or 0); acc_out = acc,
// C = out(f32(acc) * act_scale[m] * w_scale[n]) where C is given.
cudaError_t launch_acc_only(const int* acc_in, int* acc_out, int M, int N, const float* act_scale, int act_count,
                            const float* w_scale, int w_count, void* C, int c_f32, cudaStream_t s);

// DynamicQuantizeLinear of `rows` rows of `row_len` floats into exact fp16 rows
// at `pitch` (the A operand of the following GEMM) with the rows' sums of y.
cudaError_t launch_dql_rows_f16(const float* x, long long rows, long long row_len, __half* y16, long long pitch,
                                float* y_scale, uint8_t* y_zp, int32_t* row_sums, float* partials,
                                int num_partials, cudaStream_t s);
// colsum[c] = sum over the rows of an 8-bit [rows][cols] matrix (dense; zeroed here).
cudaError_t launch_colsum(const void* src, bool u8, int rows, int cols, int* colsum, cudaStream_t s);

// ConvInteger pre-pass (conv.cu). im2col of an 8-bit NCHW input into fp16
// col[n][k][p] (k = (c*kH + kh)*kW + kw over all C input channels, p = oh*oW +
// ow, rows `pitch` elements apart), padded positions holding the activation
// zero point, and, when colsum is given, colsum[n*G + g][p] = the sum of group
// g's k rows (from per-group channel sums of x held in sum_scratch, of
// im2col_sum_scratch_bytes).
struct Im2colArgs {
  const void* x;           // [Nb][C][H][W]
  int Nb, C, H, W;
  int kH, kW, pt, pl, sh, sw, dh, dw, oH, oW;
  int G;                   // groups
  const void* xzp;         // device: the activation zero point (one byte of the x type), or null (0)
  __half* col;
  long long pitch;
  int* colsum;             // or null
};
size_t im2col_sum_scratch_bytes(long long Nb, long long G, long long H, long long W);
cudaError_t launch_im2col(const Im2colArgs& a, bool x_u8, int* sum_scratch, cudaStream_t s);
// Implicit-GEMM ConvInteger pre-passes (conv.cu): x [Nb][C][HW] (8-bit) ->
// x16 [Nb][HW][C] fp16 holding x - x_zp (xzp: a device byte of the x type, or
// null for 0); w [M][Cg][kH][kW] -> w16 [M][(r*kW + s)*Cg + c] fp16 holding
// w - w_zp[m] (wzp: device bytes of the w type, wzp_count 0, 1 or M). Every
// difference lies in [-255, 255], exact in fp16.
// Both in one launch (the weight's CTAs ride along in an extra z slice).
cudaError_t launch_conv_operands(const void* x, bool xu, int Nb, int C, int HW, const void* xzp, __half* x16,
                                 const void* w, bool wu, int M, int Cg, int kH, int kW, const void* wzp,
                                 int wzp_count, __half* w16, cudaStream_t s);
// rows x cols 8-bit (dense) -> fp16 at `pitch`, with optional int32 row sums.
cudaError_t launch_rows_pitched(const void* src, bool u8, int rows, int cols, __half* dst, long long pitch,
                                int* rowsum, cudaStream_t s);

// Pre-pass: 8-bit rows -> exact fp16 (one warp per row; optional row sums), and
// 8-bit [mats][rows][cols] -> fp16 with column sums (colsum zeroed here).
cudaError_t launch_convert_rows(const void* src, bool u8, __half* dst, long long rows, int row_bytes, int* rowsum,
                                cudaStream_t s);
cudaError_t launch_convert_cols(const void* src, bool u8, __half* dst, int mats, int rows, int cols, int* colsum,
                                cudaStream_t s);
// Both operands without sums in one launch, staged through shared memory by
// bulk asynchronous copies (byte counts multiples of 16, 16-byte aligned).
cudaError_t launch_convert_bulk(const void* A, bool au, __half* A16, long long a_bytes, const void* B, bool bu,
                                __half* B16, long long b_bytes, unsigned* err, cudaStream_t s);
// Both operands without sums in one launch (byte counts multiples of 16).
cudaError_t launch_convert_flat(const void* A, bool au, __half* A16, long long a_bytes, const void* B, bool bu,
                                __half* B16, long long b_bytes, cudaStream_t s);

// Largest exact chunk length for the operand signedness (fp32 sums <= 2^24).
int gemm_default_chunk_k(bool a_u8, bool b_u8);

// ---------------------------------------------------------------------------
// Decode GEMV: bf16 A [M<=16][K] x int8 W [K][N], per-column or scalar scale/zp.
// ---------------------------------------------------------------------------
struct GemvArgs {
  const uint16_t* A;       // bf16 bits [M][K]
  const int8_t* W;         // [K][N]
  int M, K, N;
  const float* scale; int scale_count;        // 1 or N
  const int32_t* zp;  int zp_count;           // 0, 1 or N
  void* C; int c_f32;                         // [M][N] bf16 (0) or f32 (1)
  unsigned* err;                              // device error word
  // fp16 route (A16 non-null): the activations as fp16 [M][Kp] (Kp = K rounded
  // up to 16), row m scaled by 2^s_m and its K order permuted inside every
  // 16-element group, as launch_gemv_prep writes them; inv[m] = 2^-s_m
  const uint16_t* A16;
  const float* inv;
  int Kp;
};
bool gemv_supported(long long M, long long K, long long N, const void* A, const void* W);
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, const char** kernel_name);
// The fp16 route's pre-pass (one CTA per row; bf16 A [M][K], K % 8 == 0): a
// power-of-two row scale 2^s_m that puts the row's largest magnitude in
// [2^14, 2^15) (exact, and inside fp16's range), then fp16 copies of the
// scaled values (exact for every bf16 value down to 2^-17 of the row maximum)
// in the K order the GEMV's fragments read: inside each group of 16, element
// q holds k = q with bits 0 and 1 swapped. Workspace: gemv_f16_workspace_bytes.
size_t gemv_f16_workspace_bytes(long long M, long long K);
cudaError_t launch_gemv_prep(const uint16_t* A, int M, int K, void* workspace, cudaStream_t s);
// The fp16 route: the GEMV launched as a programmatic dependent of the prep
// (its weight stream starts before the prep ends); A16 / inv / Kp point into
// the prep's workspace.
cudaError_t launch_gemv_f16(GemvArgs a, void* workspace, cudaStream_t s, const char** kernel_name);

// Decode GEMV on a weight packed once (gemv_packed.cu): the packed layout holds
// each lane's MMA fragments in order, biased, K padded to 16 and N to 64.
size_t gemv_packed_weight_bytes(long long K, long long N);
// workspace of the activations' fp16 copy: M padded to 8 or 16 rows of Kp
size_t gemv_packed_workspace_bytes(long long M, long long K);
cudaError_t launch_gemv_pack(const int8_t* W, long long K, long long N, void* packed, cudaStream_t s);
// 1 <= M <= 16, K % 8 == 0, N % 8 == 0; g.W unused (the packed weight is given)
cudaError_t launch_gemv_packed(const GemvArgs& g, const void* packed, void* workspace, cudaStream_t s,
                               const char** kernel_name);

// ---------------------------------------------------------------------------
// Decode-shaped form (a) for M <= 4 on the CUDA cores: TMA-staged weight,
// packed fp32 FMAs, CTA pairs splitting K and reducing through distributed
// shared memory (one launch, no workspace).
// ---------------------------------------------------------------------------
struct GemvSimtArgs {
  const void* A; int a_bf16;   // [M][K] bf16 (1) or f32 (0)
  const int8_t* W;             // [K][N]
  int M, K, N;
  const float* scale; int scale_count;        // 1 or N
  const int32_t* zp;  int zp_count;           // 0, 1 or N
  void* C; int c_f32;
};
bool gemv_simt_supported(long long M, long long K, long long N, int a_bf16, const void* A, const void* W);
cudaError_t launch_gemv_simt(const GemvSimtArgs& p, unsigned* err, cudaStream_t s, const char** kernel_name);

// ---------------------------------------------------------------------------
// Decode-shaped accumulating A8W8 (M <= 16), dp4a on the CUDA cores.
// ---------------------------------------------------------------------------
struct GemvAccArgs {
  const int8_t* A;             // [M][K] (after the a_trans copy)
  const int8_t* B;             // [N][K] (b_trans) or [K][N]
  int M, K, N;
  const int* acc_in;           // [M][N] or null
  int* acc_out;                // [M][N] or null
  const float* act_scale; int act_count;
  const float* w_scale; int w_count;
  void* C; int c_f32;          // [M][N] or null
};
bool gemv_acc_supported(long long M, long long K, long long N, int b_trans, const void* A, const void* B);
size_t gemv_acc_workspace_bytes(long long M, long long K, long long N);
cudaError_t launch_gemv_acc(GemvAccArgs p, int a_trans, int b_trans, void* ws, cudaStream_t s,
                            const char** kernel_name);

// ---------------------------------------------------------------------------
// Generic CUDA-core form (a): float A (f32 or bf16) x int8 B, any shape.
// ---------------------------------------------------------------------------
struct W8SimtArgs {
  const void* A; int a_bf16;   // [M][K]
  const int8_t* B;             // [K][N]
  int M, K, N;
  const float* scale; int scale_count;
  const int32_t* zp;  int zp_count;
  void* C; int c_f32;
};
cudaError_t launch_w8_simt(const W8SimtArgs& a, cudaStream_t s, const char** kernel_name);

// ---------------------------------------------------------------------------
// DynamicQuantizeLinear: two-pass grid min/max + vectorised quantize.
// ---------------------------------------------------------------------------
constexpr int kDqlMaxPartials = 1024;
int dql_num_partials(long long n);
cudaError_t launch_dql(const float* x, long long n, uint8_t* y, float* y_scale, uint8_t* y_zp, int32_t* row_sums,
                       long long row_len, float* partials, int num_partials, cudaStream_t s,
                       const char** kernel_name);

int num_sms();
// The unique id of the calling thread's current CUDA context; false when no
// context is current (or the driver offers no such query).
bool current_context_id(unsigned long long* id);

}  // namespace qmm
