// The library's C ABI (include/qmm.h): argument validation, kernel selection,
// launch-error handling, the device error word, and the per-thread record of
// which kernel ran.
//
// Error handling follows the launch convention of ROCm hip-ep PR #1248
// ("What", last paragraph): the CUDA last-error state is cleared before a
// launch and read back after it.
#include "kernels.h"
#include "tma.h"
#include "../../include/qmm.h"

#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace qmm {

// Device error word: a timed-out wait inside a kernel records its site here.
__device__ unsigned g_qmm_error_word;

namespace {

constexpr int kMaxDevices = 64;

thread_local const char* t_last_kernel = "none";
thread_local int t_last_cuda_error = 0;
thread_local unsigned t_last_device_error = 0;

std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
unsigned long long g_err_ctx[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

// Device address of the error word in the current context. The address is
// cached per device together with the context it was taken in: after a
// cudaDeviceReset the primary context (and the module holding the word) is
// made anew and the address is looked up again.
unsigned* err_word() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  unsigned long long ctx = 0;
  const bool have = current_context_id(&ctx);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d] || !have || ctx != g_err_ctx[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qmm_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<unsigned*>(p);
    g_err_ctx[d] = current_context_id(&ctx) ? ctx : 0;   // the lookup made the context current
  }
  return g_err_ptr[d];
}

bool dim_ok(int64_t v) { return v >= 0 && v <= (int64_t)INT_MAX; }

qmm_status finish_launch(cudaError_t e, const char* name) {
  if (e != cudaSuccess) {
    t_last_cuda_error = (int)e;
    return QMM_ERR_CUDA;
  }
  t_last_kernel = name;
  return QMM_OK;
}

// Chunk length between exact drains of the tensor-core accumulator. The
// environment variable QMM_CHUNK_K may only shorten it (a multiple of 64):
// it exists to exercise the drain path with more chunks per tile.
int chunk_k_for(bool a_u8, bool b_u8) {
  const int dflt = gemm_default_chunk_k(a_u8, b_u8);
  const char* env = std::getenv("QMM_CHUNK_K");
  if (env) {
    const int v = std::atoi(env);
    if (v >= 64 && v % 64 == 0 && v < dflt) return v;
  }
  return dflt;
}


// ---------------------------------------------------------------------------
// Pre-pass path: operands converted once to exact fp16 copies in a caller
// workspace (with the MatMulInteger row/column sums), then the SM-pair GEMM
// stages fp16 tiles with TMA. Used for 16-byte-aligned rows, M >= 256 (after
// folding a batch) and batches that are dense or shared.
// Workspace: [A16: rowsA*K fp16][B16: matsB*K*N fp16][rowsum: rowsA int32]
// [colsum: matsB*N int32], each region 256-byte aligned.
struct PrepassPlan {
  bool use = false;
  int64_t rowsA = 0, matsB = 0;
  size_t off_b = 0, off_rs = 0, off_cs = 0, bytes = 0;
};

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

PrepassPlan prepass_plan(int64_t gb, int64_t gm, int64_t K, int64_t N, int64_t a_bstride, int64_t b_bstride,
                         int64_t M) {
  PrepassPlan pl;
  if (K <= 0 || K % 16 != 0 || N % 16 != 0 || gm < 256) return pl;
  if (gb > 1 && ((a_bstride != 0 && a_bstride != M * K) || (b_bstride != 0 && b_bstride != K * N))) return pl;
  pl.rowsA = (gb > 1 && a_bstride != 0) ? gb * gm : gm;
  pl.matsB = (gb > 1 && b_bstride != 0) ? gb : 1;
  pl.off_b = round256((size_t)pl.rowsA * K * 2);
  pl.off_rs = pl.off_b + round256((size_t)pl.matsB * K * N * 2);
  pl.off_cs = pl.off_rs + round256((size_t)pl.rowsA * 4);
  pl.bytes = pl.off_cs + round256((size_t)pl.matsB * N * 4);
  pl.use = true;
  return pl;
}

// Fold a shared B with a densely batched A into one GEMM of batch*M rows.
void fold_batch(int64_t batch, int64_t M, int64_t K, int64_t a_bstride, int64_t b_bstride, int64_t* gb,
                int64_t* gm) {
  *gb = batch;
  *gm = M;
  if (batch > 1 && b_bstride == 0 && a_bstride == M * K) {
    *gm = batch * M;
    *gb = 1;
  }
}

// A second stream per device for a pre-pass that does not depend on the one on
// the caller's stream (B's conversion beside A's): forked after the caller's
// earlier work, joined before the GEMM. The events are reused, so a mutex
// covers the enqueueing from fork to join.
struct AuxStream {
  bool ready = false;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};
AuxStream g_aux[kMaxDevices];

AuxStream* aux_stream() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  AuxStream& a = g_aux[d];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!a.ready) {
    if (cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    a.ready = true;
  }
  return &a;
}

// Runs side(aux stream) and primary(s) concurrently, s continuing after both;
// when no side stream can be made, both run in order on s.
template <class Side, class Primary>
cudaError_t fork_join(cudaStream_t s, Side side, Primary primary) {
  AuxStream* ax = aux_stream();
  if (!ax) {
    cudaError_t e = side(s);
    return e == cudaSuccess ? primary(s) : e;
  }
  std::lock_guard<std::mutex> lk(ax->mu);
  cudaError_t e = cudaEventRecord(ax->fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ax->s, ax->fork, 0);
  if (e != cudaSuccess) return e;   // nothing forked
  // Once forked, s always waits for the side stream again, whatever failed in
  // between: a stream capture stays joined, and s never runs ahead of side
  // work that uses the same workspace. The first error is returned.
  const cudaError_t es = side(ax->s);
  const cudaError_t er = cudaEventRecord(ax->join, ax->s);
  const cudaError_t ep = es == cudaSuccess ? primary(s) : cudaSuccess;
  const cudaError_t ew = er == cudaSuccess ? cudaStreamWaitEvent(s, ax->join, 0) : er;
  for (cudaError_t x : {es, ep, er, ew})
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

// The pre-pass: fp16 copies of A and B (and the sums the zero points need).
cudaError_t run_pack(const PrepassPlan& pl, const void* A, bool au, const void* B, bool bu, bool need_rs,
                     bool need_cs, void* ws, int K, int N, cudaStream_t s) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  __half* a16 = reinterpret_cast<__half*>(base);
  __half* b16 = reinterpret_cast<__half*>(base + pl.off_b);
  int* rs = reinterpret_cast<int*>(base + pl.off_rs);
  int* cs = reinterpret_cast<int*>(base + pl.off_cs);
  if (!need_rs && !need_cs)   // one launch for both operands, staged by bulk copies
    return launch_convert_bulk(A, au, a16, pl.rowsA * K, B, bu, b16, pl.matsB * K * N, err_word(), s);
  // with sums, A's and B's conversions are separate kernels: run them side by side
  auto side = [&](cudaStream_t st) {
    return need_cs ? launch_convert_cols(B, bu, b16, (int)pl.matsB, K, N, cs, st)
                   : launch_convert_flat(nullptr, au, nullptr, 0, B, bu, b16, pl.matsB * K * N, st);
  };
  auto primary = [&](cudaStream_t st) {
    return need_rs ? launch_convert_rows(A, au, a16, pl.rowsA, K, rs, st)
                   : launch_convert_flat(A, au, a16, pl.rowsA * K, nullptr, bu, nullptr, 0, st);
  };
  return fork_join(s, side, primary);
}

// The GEMM on packed operands.
cudaError_t run_packed_gemm(const PrepassPlan& pl, const void* ws, GemmF16Args& f, bool au, bool bu, bool mmi,
                            int chunk, cudaStream_t s) {
  const uint8_t* base = static_cast<const uint8_t*>(ws);
  f.A16 = base;
  f.B16 = base + pl.off_b;
  f.rowsum = reinterpret_cast<const int*>(base + pl.off_rs);
  f.colsum = reinterpret_cast<const int*>(base + pl.off_cs);
  const char* gname = "none";
  return launch_gemm_f16pair(f, au, bu, mmi, chunk, s, &gname);
}

const char* kPackName = "f16_prepass";
const char* kPackedA8W8 = "gemm_tc05_pair_f16ops_a8w8";
const char* kPackedMMI = "gemm_tc05_pair_f16ops_matmul_integer";
const char* kTwoPassA8W8 = "f16_prepass+gemm_tc05_pair_f16ops_a8w8";
const char* kTwoPassMMI = "f16_prepass+gemm_tc05_pair_f16ops_matmul_integer";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

// Form (a) for large M on the SM-pair GEMM: the int8 weight converted once to
// exact bf16 in a workspace, the activations' row sums (for a zero point), and
// for fp32 activations their [hi | lo] bf16 split. Workspace:
// [W16: K*N bf16][rowsum: M fp32][A': M*2*Kp bf16 (fp32 activations only)].
struct W8Plan {
  bool use = false;
  int Kp = 0;
  size_t off_rs = 0, off_a = 0, bytes = 0;
};
constexpr int64_t kW8PrefillMinM = 64;

W8Plan w8_plan(int a_dtype, int64_t M, int64_t K, int64_t N) {
  W8Plan pl;
  if (M < kW8PrefillMinM || K <= 0 || K % 16 != 0 || N % 16 != 0) return pl;
  if (a_dtype != QMM_F32 && a_dtype != QMM_BF16) return pl;
  pl.Kp = (int)((K + 63) / 64 * 64);
  pl.off_rs = round256((size_t)K * N * 2);
  pl.off_a = pl.off_rs + round256((size_t)M * 4);
  pl.bytes = pl.off_a + (a_dtype == QMM_F32 ? round256((size_t)M * 2 * pl.Kp * 2) : 0);
  pl.use = true;
  return pl;
}
// Accumulating A8W8 (PyPTO PR #1920's tensor.a8w8_matmul_dequant_acc, with
// its a_trans / b_trans): both operands converted, and transposed where they
// are stored transposed, into fp16 copies whose rows are padded to 16 bytes;
// then the SM-pair GEMM with the accumulator epilogue. Workspace:
// [A16: M x Kp fp16][B16: K x Np fp16], Kp and Np rounded up to multiples of 8.
struct AccPlan {
  int64_t Kp = 0, Np = 0;
  size_t off_b = 0, bytes = 0;
};

AccPlan acc_plan(int64_t M, int64_t K, int64_t N) {
  AccPlan pl;
  if (M <= 0 || K <= 0 || N <= 0) return pl;
  pl.Kp = (K + 7) / 8 * 8;
  pl.Np = (N + 7) / 8 * 8;
  pl.off_b = round256((size_t)M * pl.Kp * 2);
  pl.bytes = pl.off_b + round256((size_t)K * pl.Np * 2);
  return pl;
}
// ConvInteger (ROCm hip-ep PR #1248, "What", ConvInteger paragraph) as the
// exact MatMulInteger GEMM: A = the weight [M][C/G*kH*kW] (shared by every
// image, one slice per group), B = each image's im2col matrix, C = y in NCHW.
// Workspace: [W16: M x Kgp fp16][col: N x C*kH*kW x Pp fp16][rowsum(W): M
// int32][colsum(col): N*G x P int32][channel sums of x: N*G x H*W int32], Kgp
// and Pp rounded up to multiples of 8.
struct ConvPlan {
  bool ok = false;
  int oH = 0, oW = 0;
  int64_t P = 0, Pp = 0, Kg = 0, Kgp = 0;
  int64_t pt = 0, pl = 0, pb = 0, pr = 0, sh = 1, sw = 1, dh = 1, dw = 1;
  size_t off_col = 0, off_rs = 0, off_cs = 0, off_s = 0, bytes = 0;
  // implicit-GEMM route: [w16: M x Kg fp16][x16: N x H x W x C fp16]
  bool im2col_tma = false;
  int lower[2] = {0, 0}, upper[2] = {0, 0};   // bounding-box corners, W then H
  size_t off_x16 = 0;
};

ConvPlan conv_plan(int64_t N, int64_t C, int64_t H, int64_t W, int64_t M, int64_t kH, int64_t kW,
                   const int64_t* pads, const int64_t* strides, const int64_t* dilations, int64_t G) {
  ConvPlan pl;
  if (!dim_ok(N) || !dim_ok(C) || !dim_ok(H) || !dim_ok(W) || !dim_ok(M) || !dim_ok(kH) || !dim_ok(kW)) return pl;
  if (C < 1 || H < 1 || W < 1 || M < 1 || kH < 1 || kW < 1 || G < 1 || C % G != 0 || M % G != 0) return pl;
  if (pads) {
    pl.pt = pads[0];
    pl.pl = pads[1];
    pl.pb = pads[2];
    pl.pr = pads[3];
  }
  if (strides) {
    pl.sh = strides[0];
    pl.sw = strides[1];
  }
  if (dilations) {
    pl.dh = dilations[0];
    pl.dw = dilations[1];
  }
  const int64_t lim = 1 << 20;
  if (pl.pt < 0 || pl.pl < 0 || pl.pb < 0 || pl.pr < 0 || pl.pt > lim || pl.pl > lim || pl.pb > lim || pl.pr > lim)
    return pl;
  if (pl.sh < 1 || pl.sw < 1 || pl.dh < 1 || pl.dw < 1 || pl.sh > lim || pl.sw > lim || pl.dh > lim || pl.dw > lim)
    return pl;
  const int64_t oH = (H + pl.pt + pl.pb - pl.dh * (kH - 1) - 1) / pl.sh + 1;
  const int64_t oW = (W + pl.pl + pl.pr - pl.dw * (kW - 1) - 1) / pl.sw + 1;
  const int64_t eh = H + pl.pt + pl.pb - pl.dh * (kH - 1), ew = W + pl.pl + pl.pr - pl.dw * (kW - 1);
  pl.oH = eh >= 1 ? (int)oH : 0;   // a kernel wider than the padded input: empty output
  pl.oW = ew >= 1 ? (int)oW : 0;
  pl.P = (int64_t)pl.oH * pl.oW;
  pl.Kg = C / G * kH * kW;
  if (C * kH * kW > (int64_t)INT_MAX || pl.P > (int64_t)INT_MAX || N * G > (int64_t)INT_MAX) return pl;
  pl.Kgp = (pl.Kg + 7) / 8 * 8;
  pl.Pp = (pl.P + 7) / 8 * 8;
  pl.off_col = round256((size_t)M * pl.Kgp * 2);
  pl.off_rs = pl.off_col + round256((size_t)N * C * kH * kW * pl.Pp * 2);
  pl.off_cs = pl.off_rs + round256((size_t)M * 4);
  pl.off_s = pl.off_cs + round256((size_t)N * G * pl.P * 4);
  pl.bytes = pl.off_s + round256(im2col_sum_scratch_bytes(N, G, H, W));
  pl.ok = true;
  // The implicit GEMM (im2col tensor copies of an fp16 NHWC input) applies when
  // a group's channels come in whole 64-channel boxes, the traversal strides
  // and the window's bounding-box corners fit the copy's fields, and output
  // rows are 16-byte multiples (the TMA-store epilogue). Otherwise the
  // materialised im2col matrix above is used.
  const int64_t Cg = C / G;
  const int64_t lw = -pl.pl, lh = -pl.pt;
  const int64_t uw = (int64_t)(pl.oW - 1) * pl.sw - pl.pl - (W - 1);
  const int64_t uh = (int64_t)(pl.oH - 1) * pl.sh - pl.pt - (H - 1);
  if (pl.P > 0 && Cg % 64 == 0 && pl.P % 4 == 0 && pl.sh <= 8 && pl.sw <= 8 && lw >= -128 && lh >= -128 &&
      uw >= -128 && uw <= 127 && uh >= -128 && uh <= 127 && (kW - 1) * pl.dw <= 32767 && (kH - 1) * pl.dh <= 32767 &&
      N * H * W * C <= ((int64_t)1 << 40)) {
    pl.im2col_tma = true;
    pl.lower[0] = (int)lw;
    pl.lower[1] = (int)lh;
    pl.upper[0] = (int)uw;
    pl.upper[1] = (int)uh;
    pl.off_x16 = round256((size_t)M * pl.Kg * 2);
    pl.bytes = pl.off_x16 + round256((size_t)N * H * W * C * 2);
  }
  return pl;
}
// The DynamicQuantizeLinear -> MatMulInteger -> dequantise chain. Workspace:
// [DQL partials][A16: M x Kp fp16][B16: K x Np fp16][rowsum(y): M int32]
// [colsum(W): N int32][y_scale: f32, y_zp: u8], Kp and Np rounded up to 8.
struct DqmPlan {
  int64_t Kp = 0, Np = 0;
  size_t off_a = 0, off_b = 0, off_rs = 0, off_cs = 0, off_sz = 0, bytes = 0;
};

// with_weight = false leaves out the weight's fp16 copy and column sums (they
// live in a buffer packed once by dynamic_quantize_matmul_pack_weight)
DqmPlan dqm_plan(int64_t M, int64_t K, int64_t N, bool with_weight = true) {
  DqmPlan pl;
  pl.Kp = (K + 7) / 8 * 8;
  pl.Np = (N + 7) / 8 * 8;
  pl.off_a = round256(dynamic_quantize_linear_workspace_bytes(M * K));
  pl.off_b = pl.off_a + round256((size_t)M * pl.Kp * 2);
  pl.off_rs = pl.off_b + (with_weight ? round256((size_t)K * pl.Np * 2) : 0);
  pl.off_cs = pl.off_rs + round256((size_t)M * 4);
  pl.off_sz = pl.off_cs + (with_weight ? round256((size_t)N * 4) : 0);
  pl.bytes = pl.off_sz + 256;
  return pl;
}

// The packed weight of the chain: W as exact fp16 [K][Np] (Np = N rounded up
// to 8, pad columns unspecified), then colsum(W) as int32[N].
struct DqmWeight {
  int64_t Np = 0;
  size_t off_cs = 0, bytes = 0;
};

DqmWeight dqm_weight(int64_t K, int64_t N) {
  DqmWeight w;
  w.Np = (N + 7) / 8 * 8;
  w.off_cs = round256((size_t)K * w.Np * 2);
  w.bytes = w.off_cs + round256((size_t)N * 4);
  return w;
}

// W -> exact fp16 copy with pitch Np plus its column sums, on stream st
cudaError_t dqm_convert_weight(const void* W, bool wu, int64_t K, int64_t N, int64_t Np, __half* b16, int* cs,
                               cudaStream_t st) {
  if (N % 16 == 0 && aligned16(W)) return launch_convert_cols(W, wu, b16, 1, (int)K, (int)N, cs, st);
  const ConvPlane none{nullptr, 0, 0, 0, 0, nullptr, 0};
  const ConvPlane pb{W, N, (int)K, (int)N, 0, b16, Np};
  cudaError_t e = launch_convert_planes(none, false, pb, wu, st);
  return e == cudaSuccess ? launch_colsum(W, wu, (int)K, (int)N, cs, st) : e;
}
}  // namespace

bool current_context_id(unsigned long long* id) {
  using CtxGetCurrentFn = CUresult (*)(CUcontext*);
  using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext c = nullptr;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c) return false;
  return get_id(c, id) == CUDA_SUCCESS;
}

int num_sms() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    g_sms[d] = n;
  }
  return g_sms[d];
}

}  // namespace qmm

using namespace qmm;

extern "C" {

const char* qmm_status_string(int s) {
  switch (s) {
    case QMM_OK: return "QMM_OK";
    case QMM_ERR_INVALID_ARG: return "QMM_ERR_INVALID_ARG";
    case QMM_ERR_UNSUPPORTED: return "QMM_ERR_UNSUPPORTED";
    case QMM_ERR_CUDA: return "QMM_ERR_CUDA";
    case QMM_ERR_TIMEOUT: return "QMM_ERR_TIMEOUT";
    default: return "QMM_UNKNOWN_STATUS";
  }
}

const char* qmm_last_kernel(void) { return t_last_kernel; }
int qmm_last_cuda_error(void) { return t_last_cuda_error; }
unsigned qmm_last_device_error(void) { return t_last_device_error; }
int qmm_num_sms(void) { return num_sms(); }
int qmm_abi_version(void) { return 1; }

qmm_status qmm_check_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    t_last_cuda_error = (int)e;
    return QMM_ERR_CUDA;
  }
  unsigned* w = err_word();
  if (!w) return QMM_ERR_CUDA;
  unsigned v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    t_last_cuda_error = (int)e;
    return QMM_ERR_CUDA;
  }
  t_last_device_error = v;
  if (v != 0) {
    cudaMemset(w, 0, sizeof(unsigned));
    return QMM_ERR_TIMEOUT;
  }
  return QMM_OK;
}

qmm_status qmm_w8_dequant(const void* A, int a_dtype, const int8_t* B, int64_t M, int64_t K, int64_t N,
                          const float* scale, int64_t scale_count, const int32_t* zero_point, int64_t zp_count,
                          void* C, int c_dtype, void* stream) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  if (a_dtype != QMM_F32 && a_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (scale_count != 1 && scale_count != N) return QMM_ERR_INVALID_ARG;
  if (zp_count != 0 && zp_count != 1 && zp_count != N) return QMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (!scale || !C || (K > 0 && (!A || !B)) || (zp_count > 0 && !zero_point)) return QMM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  const char* name = "none";
  if (gemv_simt_supported(M, K, N, a_dtype == QMM_BF16, A, B)) {   // one to four rows: CUDA cores, CTA pairs
    GemvSimtArgs g{};
    g.A = A;
    g.a_bf16 = a_dtype == QMM_BF16;
    g.W = B;
    g.M = (int)M;
    g.K = (int)K;
    g.N = (int)N;
    g.scale = scale;
    g.scale_count = (int)scale_count;
    g.zp = zero_point;
    g.zp_count = (int)zp_count;
    g.C = C;
    g.c_f32 = c_dtype == QMM_F32;
    unsigned* err = err_word();
    if (!err) return QMM_ERR_CUDA;
    return finish_launch(launch_gemv_simt(g, err, s, &name), name);
  }
  if (a_dtype == QMM_BF16 && gemv_supported(M, K, N, A, B)) {
    GemvArgs g{};
    g.A = static_cast<const uint16_t*>(A);
    g.W = B;
    g.M = (int)M;
    g.K = (int)K;
    g.N = (int)N;
    g.scale = scale;
    g.scale_count = (int)scale_count;
    g.zp = zero_point;
    g.zp_count = (int)zp_count;
    g.C = C;
    g.c_f32 = c_dtype == QMM_F32;
    g.err = err_word();
    if (!g.err) return QMM_ERR_CUDA;
    return finish_launch(launch_gemv(g, s, &name), name);
  }
  if ((M + 63) / 64 > 65535) return QMM_ERR_UNSUPPORTED;
  W8SimtArgs w{};
  w.A = A;
  w.a_bf16 = a_dtype == QMM_BF16;
  w.B = B;
  w.M = (int)M;
  w.K = (int)K;
  w.N = (int)N;
  w.scale = scale;
  w.scale_count = (int)scale_count;
  w.zp = zero_point;
  w.zp_count = (int)zp_count;
  w.C = C;
  w.c_f32 = c_dtype == QMM_F32;
  return finish_launch(launch_w8_simt(w, s, &name), name);
}

// Decode shapes of 3 to 16 bf16 rows take the GEMV's fp16 route when a
// workspace is given (the activations pre-scaled to fp16 there); one or two
// rows keep the CUDA-core pair kernel, which is faster for them.
bool gemv_f16_shape(int a_dtype, int64_t M, int64_t K, int64_t N) {
  return a_dtype == QMM_BF16 && M >= 3 && M <= 16 && K >= 8 && K % 8 == 0 && N >= 16 && N % 16 == 0;
}

size_t qmm_w8_decode_pack_bytes(int64_t K, int64_t N) {
  if (K < 8 || N < 8 || !dim_ok(K) || !dim_ok(N) || K % 8 != 0 || N % 8 != 0) return 0;
  return gemv_packed_weight_bytes(K, N);
}

qmm_status qmm_w8_pack_decode_weight(const int8_t* W, int64_t K, int64_t N, void* packed, size_t packed_bytes,
                                     void* stream) {
  const size_t need = qmm_w8_decode_pack_bytes(K, N);
  if (need == 0) return QMM_ERR_UNSUPPORTED;
  if (!W || !packed || !aligned16(packed) || packed_bytes < need) return QMM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  return finish_launch(launch_gemv_pack(W, K, N, packed, s), "gemv_w8_pack");
}

size_t qmm_w8_dequant_packed_workspace_bytes(int64_t M, int64_t K) {
  if (M < 1 || M > 16 || K < 8 || !dim_ok(K) || K % 8 != 0) return 0;
  return gemv_packed_workspace_bytes(M, K);
}

qmm_status qmm_w8_dequant_packed(const void* A, int64_t M, int64_t K, int64_t N, const void* packed,
                                 size_t packed_bytes, const float* scale, int64_t scale_count,
                                 const int32_t* zero_point, int64_t zp_count, void* C, int c_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (M < 1 || M > 16 || K < 8 || N < 8 || !dim_ok(K) || !dim_ok(N) || K % 8 != 0 || N % 8 != 0)
    return QMM_ERR_UNSUPPORTED;
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (scale_count != 1 && scale_count != N) return QMM_ERR_INVALID_ARG;
  if (zp_count != 0 && zp_count != 1 && zp_count != N) return QMM_ERR_INVALID_ARG;
  if (!A || !aligned16(A) || !scale || !C || (zp_count > 0 && !zero_point)) return QMM_ERR_INVALID_ARG;
  if (!packed || !aligned16(packed) || packed_bytes < gemv_packed_weight_bytes(K, N)) return QMM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < gemv_packed_workspace_bytes(M, K))
    return QMM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  GemvArgs g{};
  g.A = static_cast<const uint16_t*>(A);
  g.M = (int)M;
  g.K = (int)K;
  g.N = (int)N;
  g.scale = scale;
  g.scale_count = (int)scale_count;
  g.zp = zero_point;
  g.zp_count = (int)zp_count;
  g.C = C;
  g.c_f32 = c_dtype == QMM_F32;
  const char* name = "none";
  return finish_launch(launch_gemv_packed(g, packed, workspace, s, &name), name);
}

size_t qmm_w8_dequant_workspace_bytes(int a_dtype, int64_t M, int64_t K, int64_t N) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return 0;
  if (a_dtype != QMM_F32 && a_dtype != QMM_BF16) return 0;
  if (gemv_f16_shape(a_dtype, M, K, N)) return gemv_f16_workspace_bytes(M, K);
  const W8Plan pl = w8_plan(a_dtype, M, K, N);
  return pl.use ? pl.bytes : 0;
}

qmm_status qmm_w8_dequant_ws(const void* A, int a_dtype, const int8_t* B, int64_t M, int64_t K, int64_t N,
                             const float* scale, int64_t scale_count, const int32_t* zero_point, int64_t zp_count,
                             void* C, int c_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (dim_ok(M) && dim_ok(K) && dim_ok(N) && gemv_f16_shape(a_dtype, M, K, N) && gemv_supported(M, K, N, A, B) &&
      workspace && aligned16(workspace) && workspace_bytes >= gemv_f16_workspace_bytes(M, K)) {
    if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
    if (scale_count != 1 && scale_count != N) return QMM_ERR_INVALID_ARG;
    if (zp_count != 0 && zp_count != 1 && zp_count != N) return QMM_ERR_INVALID_ARG;
    if (!scale || !C || (zp_count > 0 && !zero_point)) return QMM_ERR_INVALID_ARG;
    unsigned* err = err_word();
    if (!err) return QMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    GemvArgs g{};
    g.A = static_cast<const uint16_t*>(A);
    g.W = B;
    g.M = (int)M;
    g.K = (int)K;
    g.N = (int)N;
    g.scale = scale;
    g.scale_count = (int)scale_count;
    g.zp = zero_point;
    g.zp_count = (int)zp_count;
    g.C = C;
    g.c_f32 = c_dtype == QMM_F32;
    g.err = err;
    const char* name = "none";
    cudaError_t e = launch_gemv_prep(g.A, g.M, g.K, workspace, s);
    if (e == cudaSuccess) e = launch_gemv_f16(g, workspace, s, &name);
    return finish_launch(e, zp_count > 0 ? "gemv_f16_prep+gemv_w8_f16_tma_zp" : "gemv_f16_prep+gemv_w8_f16_tma");
  }
  const W8Plan pl = (dim_ok(M) && dim_ok(K) && dim_ok(N)) ? w8_plan(a_dtype, M, K, N) : W8Plan{};
  const bool a_ok = a_dtype == QMM_F32 ? (reinterpret_cast<uintptr_t>(A) % 4) == 0 : aligned16(A);
  if (!pl.use || N == 0 || !a_ok || !aligned16(B))
    return qmm_w8_dequant(A, a_dtype, B, M, K, N, scale, scale_count, zero_point, zp_count, C, c_dtype, stream);
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (scale_count != 1 && scale_count != N) return QMM_ERR_INVALID_ARG;
  if (zp_count != 0 && zp_count != 1 && zp_count != N) return QMM_ERR_INVALID_ARG;
  if (!scale || !C || !A || !B || (zp_count > 0 && !zero_point)) return QMM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  uint8_t* base = static_cast<uint8_t*>(workspace);
  float* rowsum = zp_count > 0 ? reinterpret_cast<float*>(base + pl.off_rs) : nullptr;
  cudaError_t e = launch_convert_s8_bf16(B, base, K * N, s);
  GemmF16Args f{};
  f.batch = 1;
  f.M = (int)M;
  f.N = (int)N;
  f.B16 = base;
  if (e == cudaSuccess) {
    if (a_dtype == QMM_F32) {
      e = launch_split_f32(static_cast<const float*>(A), M, (int)K, pl.Kp, base + pl.off_a, rowsum, s);
      f.A16 = base + pl.off_a;
      f.K = 2 * pl.Kp;
      f.fa_kwrap = pl.Kp;
    } else {
      if (rowsum) e = launch_rowsum_bf16(A, M, (int)K, rowsum, s);
      f.A16 = A;
      f.K = (int)K;
      f.fa_kwrap = 0;
    }
  }
  f.C = C;
  f.c_f32 = c_dtype == QMM_F32;
  f.w_scale = scale;
  f.w_count = (int)scale_count;
  f.b_zp = zero_point;
  f.b_zp_count = (int)zp_count;
  f.rowsum = reinterpret_cast<const int*>(rowsum);
  f.zp_row_mod = (int)M;
  f.err = err;
  const char* name = "none";
  if (e == cudaSuccess) e = launch_gemm_w8_bf16pair(f, (int)K, s, &name);
  return finish_launch(e, "w8_bf16_prepass+gemm_tc05_pair_w8_bf16");
}

qmm_status qmm_a8w8(const int8_t* A, const int8_t* B, int64_t M, int64_t K, int64_t N, const float* act_scale,
                    int64_t act_count, const float* weight_scale, int64_t w_count, void* C, int c_dtype,
                    void* stream) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (act_count != 1 && act_count != M) return QMM_ERR_INVALID_ARG;
  if (w_count != 1 && w_count != N) return QMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (!act_scale || !weight_scale || !C || (K > 0 && (!A || !B))) return QMM_ERR_INVALID_ARG;
  const long long tiles = ((M + 127) / 128) * ((N + 255) / 256);
  if (tiles > INT_MAX) return QMM_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  if (K == 0) {   // empty sum: acc = 0, so every output is +0
    const size_t bytes = (size_t)M * (size_t)N * (c_dtype == QMM_F32 ? 4 : 2);
    return finish_launch(cudaMemsetAsync(C, 0, bytes, s), "memset_zero");
  }
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  GemmArgs g{};
  g.A = reinterpret_cast<const uint8_t*>(A);
  g.B = reinterpret_cast<const uint8_t*>(B);
  g.a_bstride = 0;
  g.b_bstride = 0;
  g.batch = 1;
  g.M = (int)M;
  g.K = (int)K;
  g.N = (int)N;
  g.C = C;
  g.c_f32 = c_dtype == QMM_F32;
  g.act_scale = act_scale;
  g.act_count = (int)act_count;
  g.w_scale = weight_scale;
  g.w_count = (int)w_count;
  g.zp_row_mod = (int)M;
  g.err = err;
  const char* name = "none";
  return finish_launch(launch_gemm_tc(g, false, false, false, chunk_k_for(false, false), s, &name), name);
}

qmm_status matmul_integer(const void* A, int a_dtype, const void* B, int b_dtype, int64_t batch, int64_t M,
                          int64_t K, int64_t N, int64_t a_batch_stride, int64_t b_batch_stride,
                          const void* a_zero_point, int64_t a_zp_count, const void* b_zero_point,
                          int64_t b_zp_count, int32_t* C, void* stream) {
  if (!dim_ok(batch) || !dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  if ((a_dtype != QMM_S8 && a_dtype != QMM_U8) || (b_dtype != QMM_S8 && b_dtype != QMM_U8))
    return QMM_ERR_INVALID_ARG;
  if (a_batch_stride < 0 || b_batch_stride < 0) return QMM_ERR_INVALID_ARG;
  if (a_zp_count != 0 && a_zp_count != 1 && a_zp_count != M) return QMM_ERR_INVALID_ARG;
  if (b_zp_count != 0 && b_zp_count != 1 && b_zp_count != N) return QMM_ERR_INVALID_ARG;
  if (batch == 0 || M == 0 || N == 0) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (!C || (K > 0 && (!A || !B)) || (a_zp_count > 0 && !a_zero_point) || (b_zp_count > 0 && !b_zero_point))
    return QMM_ERR_INVALID_ARG;
  if (batch * M > (int64_t)INT_MAX) return QMM_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  if (K == 0) {   // empty sums: every output is 0
    return finish_launch(cudaMemsetAsync(C, 0, (size_t)batch * M * N * sizeof(int32_t), s), "memset_zero");
  }
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  // A shared B with a densely batched A is one GEMM with the batch folded into M.
  int64_t gb = batch, gm = M;
  if (batch > 1 && b_batch_stride == 0 && a_batch_stride == M * K) {
    gm = batch * M;
    gb = 1;
  }
  const long long tiles = gb * ((gm + 127) / 128) * ((N + 255) / 256);
  if (tiles > INT_MAX) return QMM_ERR_UNSUPPORTED;
  GemmArgs g{};
  g.A = static_cast<const uint8_t*>(A);
  g.B = static_cast<const uint8_t*>(B);
  g.a_bstride = gb > 1 ? a_batch_stride : 0;
  g.b_bstride = gb > 1 ? b_batch_stride : 0;
  g.batch = (int)gb;
  g.M = (int)gm;
  g.K = (int)K;
  g.N = (int)N;
  g.C = C;
  g.a_zp = a_zero_point;
  g.a_zp_count = (int)a_zp_count;
  g.b_zp = b_zero_point;
  g.b_zp_count = (int)b_zp_count;
  g.zp_row_mod = (int)M;
  g.err = err;
  const bool au = a_dtype == QMM_U8, bu = b_dtype == QMM_U8;
  const char* name = "none";
  return finish_launch(launch_gemm_tc(g, au, bu, true, chunk_k_for(au, bu), s, &name), name);
}

size_t qmm_a8w8_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return 0;
  const PrepassPlan pl = prepass_plan(1, M, K, N, 0, 0, M);
  return pl.use ? pl.bytes : 0;
}

qmm_status qmm_a8w8_ws(const int8_t* A, const int8_t* B, int64_t M, int64_t K, int64_t N, const float* act_scale,
                       int64_t act_count, const float* weight_scale, int64_t w_count, void* C, int c_dtype,
                       void* workspace, size_t workspace_bytes, void* stream) {
  const PrepassPlan pl = (dim_ok(M) && dim_ok(K) && dim_ok(N)) ? prepass_plan(1, M, K, N, 0, 0, M) : PrepassPlan{};
  if (!pl.use || M == 0 || N == 0 || !aligned16(A) || !aligned16(B))
    return qmm_a8w8(A, B, M, K, N, act_scale, act_count, weight_scale, w_count, C, c_dtype, stream);
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (act_count != 1 && act_count != M) return QMM_ERR_INVALID_ARG;
  if (w_count != 1 && w_count != N) return QMM_ERR_INVALID_ARG;
  if (!act_scale || !weight_scale || !C || !A || !B) return QMM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  GemmF16Args f{};
  f.batch = 1;
  f.M = (int)M;
  f.K = (int)K;
  f.N = (int)N;
  f.C = C;
  f.c_f32 = c_dtype == QMM_F32;
  f.act_scale = act_scale;
  f.act_count = (int)act_count;
  f.w_scale = weight_scale;
  f.w_count = (int)w_count;
  f.zp_row_mod = (int)M;
  f.err = err;
  cudaError_t e = run_pack(pl, A, false, B, false, false, false, workspace, (int)K, (int)N, s);
  if (e == cudaSuccess) e = run_packed_gemm(pl, workspace, f, false, false, false, chunk_k_for(false, false), s);
  return finish_launch(e, kTwoPassA8W8);
}

size_t matmul_integer_workspace_bytes(int64_t batch, int64_t M, int64_t K, int64_t N, int64_t a_batch_stride,
                                      int64_t b_batch_stride) {
  if (!dim_ok(batch) || !dim_ok(M) || !dim_ok(K) || !dim_ok(N) || batch * M > (int64_t)INT_MAX) return 0;
  int64_t gb, gm;
  fold_batch(batch, M, K, a_batch_stride, b_batch_stride, &gb, &gm);
  const PrepassPlan pl = prepass_plan(gb, gm, K, N, a_batch_stride, b_batch_stride, M);
  return pl.use ? pl.bytes : 0;
}

qmm_status matmul_integer_ws(const void* A, int a_dtype, const void* B, int b_dtype, int64_t batch, int64_t M,
                             int64_t K, int64_t N, int64_t a_batch_stride, int64_t b_batch_stride,
                             const void* a_zero_point, int64_t a_zp_count, const void* b_zero_point,
                             int64_t b_zp_count, int32_t* C, void* workspace, size_t workspace_bytes, void* stream) {
  PrepassPlan pl;
  int64_t gb = batch, gm = M;
  if (dim_ok(batch) && dim_ok(M) && dim_ok(K) && dim_ok(N) && batch * M <= (int64_t)INT_MAX &&
      a_batch_stride >= 0 && b_batch_stride >= 0) {
    fold_batch(batch, M, K, a_batch_stride, b_batch_stride, &gb, &gm);
    pl = prepass_plan(gb, gm, K, N, a_batch_stride, b_batch_stride, M);
  }
  if (!pl.use || batch == 0 || M == 0 || N == 0 || !aligned16(A) || !aligned16(B))
    return matmul_integer(A, a_dtype, B, b_dtype, batch, M, K, N, a_batch_stride, b_batch_stride, a_zero_point,
                          a_zp_count, b_zero_point, b_zp_count, C, stream);
  if ((a_dtype != QMM_S8 && a_dtype != QMM_U8) || (b_dtype != QMM_S8 && b_dtype != QMM_U8))
    return QMM_ERR_INVALID_ARG;
  if (a_zp_count != 0 && a_zp_count != 1 && a_zp_count != M) return QMM_ERR_INVALID_ARG;
  if (b_zp_count != 0 && b_zp_count != 1 && b_zp_count != N) return QMM_ERR_INVALID_ARG;
  if (!C || !A || !B || (a_zp_count > 0 && !a_zero_point) || (b_zp_count > 0 && !b_zero_point))
    return QMM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  if (gb * ((gm + 255) / 256) * ((N + 255) / 256) > INT_MAX) return QMM_ERR_UNSUPPORTED;
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  GemmF16Args f{};
  f.a_bstride = (gb > 1 && a_batch_stride != 0) ? gm * K : 0;
  f.b_bstride = (gb > 1 && b_batch_stride != 0) ? K * N : 0;
  f.batch = (int)gb;
  f.M = (int)gm;
  f.K = (int)K;
  f.N = (int)N;
  f.C = C;
  f.a_zp = a_zero_point;
  f.a_zp_count = (int)a_zp_count;
  f.b_zp = b_zero_point;
  f.b_zp_count = (int)b_zp_count;
  f.zp_row_mod = (int)M;
  f.err = err;
  const bool au = a_dtype == QMM_U8, bu = b_dtype == QMM_U8;
  cudaError_t e = run_pack(pl, A, au, B, bu, b_zp_count > 0, a_zp_count > 0, workspace, (int)K, (int)N, s);
  if (e == cudaSuccess) e = run_packed_gemm(pl, workspace, f, au, bu, true, chunk_k_for(au, bu), s);
  return finish_launch(e, kTwoPassMMI);
}

qmm_status qmm_a8w8_pack(const int8_t* A, const int8_t* B, int64_t M, int64_t K, int64_t N, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  const PrepassPlan pl = prepass_plan(1, M, K, N, 0, 0, M);
  if (!pl.use) return QMM_ERR_UNSUPPORTED;
  if (!A || !B || !aligned16(A) || !aligned16(B)) return QMM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  return finish_launch(run_pack(pl, A, false, B, false, false, false, workspace, (int)K, (int)N, s), kPackName);
}

namespace {
qmm_status a8w8_packed_impl(int64_t M, int64_t K, int64_t N, const float* act_scale, int64_t act_count,
                            const float* weight_scale, int64_t w_count, void* C, int c_dtype, const void* workspace,
                            size_t workspace_bytes, void* stream, int stall_test, uint64_t wait_ns) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  const PrepassPlan pl = prepass_plan(1, M, K, N, 0, 0, M);
  if (!pl.use) return QMM_ERR_UNSUPPORTED;
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (act_count != 1 && act_count != M) return QMM_ERR_INVALID_ARG;
  if (w_count != 1 && w_count != N) return QMM_ERR_INVALID_ARG;
  if (!act_scale || !weight_scale || !C) return QMM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  GemmF16Args f{};
  f.batch = 1;
  f.M = (int)M;
  f.K = (int)K;
  f.N = (int)N;
  f.C = C;
  f.c_f32 = c_dtype == QMM_F32;
  f.act_scale = act_scale;
  f.act_count = (int)act_count;
  f.w_scale = weight_scale;
  f.w_count = (int)w_count;
  f.zp_row_mod = (int)M;
  f.err = err;
  f.stall_test = stall_test;
  f.wait_ns = wait_ns;
  return finish_launch(run_packed_gemm(pl, workspace, f, false, false, false, chunk_k_for(false, false), s),
                       kPackedA8W8);
}
}  // namespace

qmm_status qmm_a8w8_packed(int64_t M, int64_t K, int64_t N, const float* act_scale, int64_t act_count,
                           const float* weight_scale, int64_t w_count, void* C, int c_dtype, const void* workspace,
                           size_t workspace_bytes, void* stream) {
  return a8w8_packed_impl(M, K, N, act_scale, act_count, weight_scale, w_count, C, c_dtype, workspace,
                          workspace_bytes, stream, 0, 0);
}

qmm_status qmm_test_a8w8_packed_stall(int64_t M, int64_t K, int64_t N, const float* act_scale, int64_t act_count,
                                      const float* weight_scale, int64_t w_count, void* C, int c_dtype,
                                      const void* workspace, size_t workspace_bytes, uint64_t wait_limit_ns,
                                      void* stream) {
  if (wait_limit_ns < 1000 || wait_limit_ns > 100000000ull) return QMM_ERR_INVALID_ARG;
  return a8w8_packed_impl(M, K, N, act_scale, act_count, weight_scale, w_count, C, c_dtype, workspace,
                          workspace_bytes, stream, 1, wait_limit_ns);
}

// ---------------------------------------------------------------------------
// A8W8 from host buffers: the copies pipelined with the two-pass GEMM.
// ---------------------------------------------------------------------------
namespace {

constexpr int kHostMaxPanels = 8;

// Device layout of the host call's workspace: the operands, scales and output
// on the device, then the two-pass path's workspace.
struct HostPlan {
  bool two_pass = false;
  int64_t Mp = 0;   // rows per panel
  int panels = 0;
  size_t off_b = 0, off_act = 0, off_w = 0, off_c = 0, off_pack = 0, bytes = 0;
  PrepassPlan pl;
};

HostPlan host_plan(int64_t M, int64_t K, int64_t N, int64_t act_count, int64_t w_count, int c_dtype) {
  HostPlan h;
  const size_t celem = c_dtype == QMM_F32 ? 4 : 2;
  h.off_b = round256((size_t)M * K);
  h.off_act = h.off_b + round256((size_t)K * N);
  h.off_w = h.off_act + round256((size_t)std::max<int64_t>(act_count, 1) * 4);
  h.off_c = h.off_w + round256((size_t)std::max<int64_t>(w_count, 1) * 4);
  h.off_pack = h.off_c + round256((size_t)M * N * celem);
  h.pl = prepass_plan(1, M, K, N, 0, 0, M);
  h.two_pass = h.pl.use;
  h.bytes = h.off_pack + (h.two_pass ? h.pl.bytes : 0);
  if (h.two_pass) {
    // row panels whose pair tiles fill whole waves of the resident pairs: the
    // copy of panel i + 1 and the read-back of panel i - 1 overlap panel i's GEMM
    const int64_t n_tiles = (N + 223) / 224;   // pair tiles across N at the narrower tile width
    const int64_t pairs = std::max(1, num_sms() / 2);
    int64_t Mp = std::max<int64_t>(1, pairs / n_tiles) * 256;
    Mp = std::max(Mp, (M + kHostMaxPanels - 1) / kHostMaxPanels);
    Mp = (Mp + 255) / 256 * 256;
    h.Mp = Mp;
    h.panels = (int)((M + Mp - 1) / Mp);
  }
  return h;
}

// Per device: the copy streams and events of the pipeline, made once. A mutex
// serialises the enqueueing of calls on one device (the events are reused).
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done = nullptr, b_in = nullptr;
  cudaEvent_t in[kHostMaxPanels] = {}, out[kHostMaxPanels] = {};
  std::mutex mu;
};
HostPipe g_pipe[kMaxDevices];

cudaError_t host_pipe(int dev, HostPipe** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  HostPipe& h = g_pipe[dev];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!h.ready) {
    const unsigned ef = cudaEventDisableTiming;
    cudaError_t e = cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.start, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.done, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.b_in, ef);
    for (int i = 0; i < kHostMaxPanels && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&h.in[i], ef);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.out[i], ef);
    }
    if (e != cudaSuccess) return e;
    h.ready = true;
  }
  *out = &h;
  return cudaSuccess;
}

}  // namespace

size_t qmm_a8w8_host_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t act_count, int64_t w_count,
                                     int c_dtype) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N) || M == 0 || N == 0) return 0;
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return 0;
  return host_plan(M, K, N, act_count, w_count, c_dtype).bytes;
}

qmm_status qmm_a8w8_host(const int8_t* hA, const int8_t* hB, int64_t M, int64_t K, int64_t N,
                         const float* h_act_scale, int64_t act_count, const float* h_weight_scale, int64_t w_count,
                         void* hC, int c_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
  if (act_count != 1 && act_count != M) return QMM_ERR_INVALID_ARG;
  if (w_count != 1 && w_count != N) return QMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (!h_act_scale || !h_weight_scale || !hC || (K > 0 && (!hA || !hB))) return QMM_ERR_INVALID_ARG;
  const HostPlan hp = host_plan(M, K, N, act_count, w_count, c_dtype);
  if (!workspace || !aligned16(workspace) || workspace_bytes < hp.bytes) return QMM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  int8_t* dA = reinterpret_cast<int8_t*>(base);
  int8_t* dB = reinterpret_cast<int8_t*>(base + hp.off_b);
  float* dAct = reinterpret_cast<float*>(base + hp.off_act);
  float* dW = reinterpret_cast<float*>(base + hp.off_w);
  uint8_t* dC = base + hp.off_c;
  const size_t celem = c_dtype == QMM_F32 ? 4 : 2;
  const int8_t* cA = static_cast<const int8_t*>(hA);
  uint8_t* cC = static_cast<uint8_t*>(hC);
  cudaGetLastError();
  if (!hp.two_pass) {
    // outside the two-pass path: copy in, one fused kernel, copy out
    cudaError_t e = cudaMemcpyAsync(dA, hA, (size_t)M * K, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dB, hB, (size_t)K * N, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dAct, h_act_scale, (size_t)act_count * 4, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dW, h_weight_scale, (size_t)w_count * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return finish_launch(e, "none");
    const qmm_status st = qmm_a8w8(dA, dB, M, K, N, dAct, act_count, dW, w_count, dC, c_dtype, stream);
    if (st != QMM_OK) return st;
    const char* name = t_last_kernel;
    e = cudaMemcpyAsync(hC, dC, (size_t)M * N * celem, cudaMemcpyDeviceToHost, s);
    return finish_launch(e, name);
  }
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  HostPipe* hpipe = nullptr;
  cudaError_t e = host_pipe(current_device(), &hpipe);
  if (e != cudaSuccess) return finish_launch(e, "none");
  std::lock_guard<std::mutex> lk(hpipe->mu);
  uint8_t* pbase = base + hp.off_pack;
  __half* a16 = reinterpret_cast<__half*>(pbase);
  __half* b16 = reinterpret_cast<__half*>(pbase + hp.pl.off_b);
  if (M >= 512 && N >= 1024) {
    // 2 x 2 blocks: A in two row panels and B in two column panels, so the
    // first block's GEMM needs only a quarter of each operand and its rows of C
    // go back while the remaining operands are still coming in (row panels
    // alone wait for the whole of B first). Every block has a dense device
    // buffer; B's column panels come in and C's blocks go out as pitched copies.
    const int64_t M1 = std::min(M, ((M + 1) / 2 + 255) / 256 * 256);
    const int64_t N1 = std::min(N, ((N + 1) / 2 + 255) / 256 * 256);
    const int64_t r0s[2] = {0, M1}, rws[2] = {M1, M - M1}, c0s[2] = {0, N1}, cls[2] = {N1, N - N1};
    auto c_block = [&](int i, int j) { return dC + (size_t)(r0s[i] * N + rws[i] * c0s[j]) * celem; };
    const char* gname = "none";
    const uint8_t* cB = static_cast<const uint8_t*>(static_cast<const void*>(hB));
    e = cudaEventRecord(hpipe->start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hpipe->h2d, hpipe->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hpipe->d2h, hpipe->start, 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dW, h_weight_scale, (size_t)w_count * 4, cudaMemcpyHostToDevice, hpipe->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dAct, h_act_scale, (size_t)act_count * 4, cudaMemcpyHostToDevice, hpipe->h2d);
    // in: A0, B0, B1, A1 (events in[0], in[2], in[3], in[1])
    auto copy_a = [&](int i) {
      cudaError_t x = cudaMemcpyAsync(dA + r0s[i] * K, cA + r0s[i] * K, (size_t)rws[i] * K, cudaMemcpyHostToDevice,
                                      hpipe->h2d);
      return x == cudaSuccess ? cudaEventRecord(hpipe->in[i], hpipe->h2d) : x;
    };
    auto copy_b = [&](int j) {
      cudaError_t x = cudaMemcpy2DAsync(dB + K * c0s[j], (size_t)cls[j], cB + c0s[j], (size_t)N, (size_t)cls[j],
                                        (size_t)K, cudaMemcpyHostToDevice, hpipe->h2d);
      return x == cudaSuccess ? cudaEventRecord(hpipe->in[2 + j], hpipe->h2d) : x;
    };
    if (e == cudaSuccess) e = copy_a(0);
    if (e == cudaSuccess) e = copy_b(0);
    if (e == cudaSuccess) e = copy_b(1);
    if (e == cudaSuccess) e = copy_a(1);
    // on the caller's stream, in the order the operands arrive: each panel's
    // conversion, each block's GEMM, and each block of C back on the second
    // copy stream as soon as it is written
    auto convert_a = [&](int i) {
      cudaError_t x = cudaStreamWaitEvent(s, hpipe->in[i], 0);
      return x == cudaSuccess ? launch_convert_bulk(dA + r0s[i] * K, false, a16 + r0s[i] * K, rws[i] * K, nullptr,
                                                    false, nullptr, 0, err, s)
                              : x;
    };
    auto convert_b = [&](int j) {
      cudaError_t x = cudaStreamWaitEvent(s, hpipe->in[2 + j], 0);
      return x == cudaSuccess ? launch_convert_bulk(nullptr, false, nullptr, 0, dB + K * c0s[j], false,
                                                    b16 + K * c0s[j], K * cls[j], err, s)
                              : x;
    };
    int nb = 0;
    auto block = [&](int i, int j) {
      GemmF16Args f{};
      f.A16 = a16 + r0s[i] * K;
      f.B16 = b16 + K * c0s[j];
      f.batch = 1;
      f.M = (int)rws[i];
      f.K = (int)K;
      f.N = (int)cls[j];
      f.C = c_block(i, j);
      f.c_f32 = c_dtype == QMM_F32;
      f.act_scale = dAct + (act_count == 1 ? 0 : r0s[i]);
      f.act_count = (int)act_count;
      f.w_scale = dW + (w_count == 1 ? 0 : c0s[j]);
      f.w_count = (int)w_count;
      f.zp_row_mod = (int)rws[i];
      f.err = err;
      cudaError_t x = launch_gemm_f16pair(f, false, false, false, chunk_k_for(false, false), s, &gname);
      if (x == cudaSuccess) x = cudaEventRecord(hpipe->out[nb], s);
      if (x == cudaSuccess) x = cudaStreamWaitEvent(hpipe->d2h, hpipe->out[nb], 0);
      ++nb;
      if (x == cudaSuccess)
        x = cudaMemcpy2DAsync(cC + (size_t)(r0s[i] * N + c0s[j]) * celem, (size_t)N * celem, c_block(i, j),
                              (size_t)cls[j] * celem, (size_t)cls[j] * celem, (size_t)rws[i], cudaMemcpyDeviceToHost,
                              hpipe->d2h);
      return x;
    };
    if (e == cudaSuccess) e = convert_a(0);
    if (e == cudaSuccess) e = convert_b(0);
    if (e == cudaSuccess) e = block(0, 0);
    if (e == cudaSuccess) e = convert_b(1);
    if (e == cudaSuccess) e = block(0, 1);
    if (e == cudaSuccess) e = convert_a(1);
    if (e == cudaSuccess) e = block(1, 0);
    if (e == cudaSuccess) e = block(1, 1);
    if (e == cudaSuccess) e = cudaEventRecord(hpipe->done, hpipe->d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hpipe->done, 0);
    return finish_launch(e, "h2d_pipelined+f16_prepass+gemm_tc05_pair_f16ops_a8w8");
  }
  // copies in, on the copy stream after the caller's earlier work: B and the
  // scales, then A panel by panel
  e = cudaEventRecord(hpipe->start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hpipe->h2d, hpipe->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hpipe->d2h, hpipe->start, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dB, hB, (size_t)K * N, cudaMemcpyHostToDevice, hpipe->h2d);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dW, h_weight_scale, (size_t)w_count * 4, cudaMemcpyHostToDevice, hpipe->h2d);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dAct, h_act_scale, (size_t)act_count * 4, cudaMemcpyHostToDevice, hpipe->h2d);
  if (e == cudaSuccess) e = cudaEventRecord(hpipe->b_in, hpipe->h2d);
  for (int i = 0; i < hp.panels && e == cudaSuccess; ++i) {
    const int64_t r0 = i * hp.Mp, rows = std::min(hp.Mp, M - r0);
    e = cudaMemcpyAsync(dA + r0 * K, cA + r0 * K, (size_t)rows * K, cudaMemcpyHostToDevice, hpipe->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(hpipe->in[i], hpipe->h2d);
  }
  // on the caller's stream: B's conversion as soon as B has arrived (while the
  // first panel of A is still being copied), then per panel its pre-pass and
  // GEMM; its rows of C go back on the second copy stream as soon as written
  const char* gname = "none";
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hpipe->b_in, 0);
  if (e == cudaSuccess) e = launch_convert_bulk(nullptr, false, nullptr, 0, dB, false, b16, K * N, err, s);
  for (int i = 0; i < hp.panels && e == cudaSuccess; ++i) {
    const int64_t r0 = i * hp.Mp, rows = std::min(hp.Mp, M - r0);
    e = cudaStreamWaitEvent(s, hpipe->in[i], 0);
    if (e == cudaSuccess)
      e = launch_convert_bulk(dA + r0 * K, false, a16 + r0 * K, rows * K, nullptr, false, nullptr, 0, err, s);
    GemmF16Args f{};
    f.A16 = a16 + r0 * K;
    f.B16 = b16;
    f.batch = 1;
    f.M = (int)rows;
    f.K = (int)K;
    f.N = (int)N;
    f.C = dC + (size_t)r0 * N * celem;
    f.c_f32 = c_dtype == QMM_F32;
    f.act_scale = dAct + (act_count == 1 ? 0 : r0);
    f.act_count = (int)act_count;
    f.w_scale = dW;
    f.w_count = (int)w_count;
    f.zp_row_mod = (int)rows;
    f.err = err;
    if (e == cudaSuccess) e = launch_gemm_f16pair(f, false, false, false, chunk_k_for(false, false), s, &gname);
    if (e == cudaSuccess) e = cudaEventRecord(hpipe->out[i], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hpipe->d2h, hpipe->out[i], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(cC + (size_t)r0 * N * celem, dC + (size_t)r0 * N * celem, (size_t)rows * N * celem,
                          cudaMemcpyDeviceToHost, hpipe->d2h);
  }
  // the caller's stream resumes once the last rows are back
  if (e == cudaSuccess) e = cudaEventRecord(hpipe->done, hpipe->d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hpipe->done, 0);
  return finish_launch(e, "h2d_pipelined+f16_prepass+gemm_tc05_pair_f16ops_a8w8");
}

size_t qmm_a8w8_acc_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return 0;
  const size_t general = acc_plan(M, K, N).bytes;
  if (M < 1 || M > 16 || K < 1 || N < 1) return general;
  return std::max(general, gemv_acc_workspace_bytes(M, K, N));   // the decode path's needs
}

qmm_status qmm_a8w8_acc(const int8_t* A, int a_trans, const int8_t* B, int b_trans, int64_t M, int64_t K, int64_t N,
                        const int32_t* acc_in, int32_t* acc_out, const float* act_scale, int64_t act_count,
                        const float* weight_scale, int64_t w_count, void* C, int c_dtype, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  if ((a_trans != 0 && a_trans != 1) || (b_trans != 0 && b_trans != 1)) return QMM_ERR_INVALID_ARG;
  if (!C && !acc_out) return QMM_ERR_INVALID_ARG;
  if (C) {
    if (c_dtype != QMM_F32 && c_dtype != QMM_BF16) return QMM_ERR_INVALID_ARG;
    if (act_count != 1 && act_count != M) return QMM_ERR_INVALID_ARG;
    if (w_count != 1 && w_count != N) return QMM_ERR_INVALID_ARG;
  }
  if (M == 0 || N == 0) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (C && (!act_scale || !weight_scale)) return QMM_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B)) return QMM_ERR_INVALID_ARG;
  if (((M + 255) / 256) * ((N + 223) / 224) > (int64_t)INT_MAX) return QMM_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  const int c_f32 = C ? (c_dtype == QMM_F32) : 0;
  if (K == 0)   // empty product: the accumulator passes through
    return finish_launch(launch_acc_only(acc_in, acc_out, (int)M, (int)N, act_scale, (int)act_count, weight_scale,
                                         (int)w_count, C, c_f32, s),
                         "acc_passthrough");
  const AccPlan pl = acc_plan(M, K, N);
  if (!workspace || !aligned16(workspace) || workspace_bytes < qmm_a8w8_acc_workspace_bytes(M, K, N))
    return QMM_ERR_INVALID_ARG;
  // decode shapes (PyPTO PR #1920's gemv_acc for a logical M of 1): a weight-streaming dp4a kernel
  if (gemv_acc_supported(M, K, N, b_trans, A, B)) {
    GemvAccArgs g{};
    g.A = A;
    g.B = B;
    g.M = (int)M;
    g.K = (int)K;
    g.N = (int)N;
    g.acc_in = acc_in;
    g.acc_out = acc_out;
    g.act_scale = act_scale;
    g.act_count = (int)act_count;
    g.w_scale = weight_scale;
    g.w_count = (int)w_count;
    g.C = C;
    g.c_f32 = c_f32;
    const char* name = "none";
    return finish_launch(launch_gemv_acc(g, a_trans, b_trans, workspace, s, &name), name);
  }
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  __half* a16 = reinterpret_cast<__half*>(base);
  __half* b16 = reinterpret_cast<__half*>(base + pl.off_b);
  cudaError_t e;
  if (!a_trans && !b_trans && K % 16 == 0 && N % 16 == 0 && aligned16(A) && aligned16(B)) {
    e = launch_convert_bulk(A, false, a16, M * K, B, false, b16, K * N, err, s);   // dense copies: Kp = K, Np = N
  } else {
    const ConvPlane pa{A, a_trans ? M : K, (int)(a_trans ? K : M), (int)(a_trans ? M : K), a_trans, a16, pl.Kp};
    const ConvPlane pb{B, b_trans ? K : N, (int)(b_trans ? N : K), (int)(b_trans ? K : N), b_trans, b16, pl.Np};
    e = launch_convert_planes(pa, false, pb, false, s);
  }
  GemmF16Args f{};
  f.A16 = a16;
  f.B16 = b16;
  f.batch = 1;
  f.M = (int)M;
  f.K = (int)K;
  f.N = (int)N;
  f.a_pitch = (int)pl.Kp;
  f.b_pitch = (int)pl.Np;
  f.C = C;
  f.c_f32 = c_f32;
  f.act_scale = act_scale;
  f.act_count = (int)act_count;
  f.w_scale = weight_scale;
  f.w_count = (int)w_count;
  f.acc_in = acc_in;
  f.acc_out = acc_out;
  f.zp_row_mod = (int)M;
  f.err = err;
  const char* gname = "none";
  if (e == cudaSuccess) e = launch_gemm_f16pair(f, false, false, false, chunk_k_for(false, false), s, &gname);
  return finish_launch(e, "f16_prepass+gemm_tc05_pair_f16ops_a8w8_acc");
}

size_t conv_integer_workspace_bytes(int64_t N, int64_t C, int64_t H, int64_t W, int64_t M, int64_t kH, int64_t kW,
                                    const int64_t* pads, const int64_t* strides, const int64_t* dilations,
                                    int64_t group) {
  const ConvPlan pl = conv_plan(N, C, H, W, M, kH, kW, pads, strides, dilations, group);
  return (pl.ok && N > 0 && pl.P > 0) ? pl.bytes : 0;
}

qmm_status conv_integer(const void* x, int x_dtype, const void* w, int w_dtype, int64_t N, int64_t C, int64_t H,
                        int64_t W, int64_t M, int64_t kH, int64_t kW, const int64_t* pads, const int64_t* strides,
                        const int64_t* dilations, int64_t group, const void* x_zero_point, const void* w_zero_point,
                        int64_t w_zp_count, int32_t* y, void* workspace, size_t workspace_bytes, void* stream) {
  if ((x_dtype != QMM_S8 && x_dtype != QMM_U8) || (w_dtype != QMM_S8 && w_dtype != QMM_U8)) return QMM_ERR_INVALID_ARG;
  const ConvPlan pl = conv_plan(N, C, H, W, M, kH, kW, pads, strides, dilations, group);
  if (!pl.ok) return QMM_ERR_INVALID_ARG;
  if (w_zp_count != 0 && w_zp_count != 1 && w_zp_count != M) return QMM_ERR_INVALID_ARG;
  if (N == 0 || pl.P == 0) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (!x || !w || !y || (w_zp_count > 0 && !w_zero_point)) return QMM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  const int64_t Mg = M / group, batch = N * group;
  if (N * group > 65535 || (C * kH * kW + 31) / 32 > 65535) return QMM_ERR_UNSUPPORTED;
  if (batch * ((Mg + 255) / 256) * ((pl.P + 223) / 224) > (int64_t)INT_MAX) return QMM_ERR_UNSUPPORTED;
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  const bool xu = x_dtype == QMM_U8, wu = w_dtype == QMM_U8;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  __half* w16 = reinterpret_cast<__half*>(base);
  if (pl.im2col_tma) {
    // implicit GEMM: the shifted operands in fp16, the input channels-innermost,
    // then the pair GEMM gathering each stage's windows with im2col copies
    __half* x16 = reinterpret_cast<__half*>(base + pl.off_x16);
    const int Cg = (int)(C / group);
    cudaError_t e = launch_conv_operands(x, xu, (int)N, (int)C, (int)(H * W), x_zero_point, x16, w, wu, (int)M, Cg,
                                         (int)kH, (int)kW, w_zero_point, (int)w_zp_count, w16, s);
    GemmF16Args f{};
    f.A16 = w16;
    f.a_bstride = group > 1 ? Mg * pl.Kg : 0;
    f.a_bmod = group > 1 ? (int)group : 0;
    f.batch = (int)batch;
    f.M = (int)Mg;
    f.K = (int)pl.Kg;
    f.N = (int)pl.P;
    f.C = y;
    f.zp_row_mod = (int)Mg;
    f.err = err;
    f.cv_oW = pl.oW;
    f.cv_sh = (int)pl.sh;
    f.cv_sw = (int)pl.sw;
    f.cv_pt = (int)pl.pt;
    f.cv_pl = (int)pl.pl;
    f.cv_dh = (int)pl.dh;
    f.cv_dw = (int)pl.dw;
    f.cv_kW = (int)kW;
    f.cv_cb = Cg / 64;
    f.cv_G = (int)group;
    f.cv_Cg = Cg;
    // each copy gathers the pixel rows of one CTA's half of the pair tile
    CUtensorMap tx{};
    if (e == cudaSuccess) {
      const uint64_t dims[4] = {(uint64_t)C, (uint64_t)W, (uint64_t)H, (uint64_t)N};
      const uint64_t strides[3] = {(uint64_t)C * 2, (uint64_t)W * C * 2, (uint64_t)H * W * C * 2};
      const uint32_t es[4] = {1u, (uint32_t)pl.sw, (uint32_t)pl.sh, 1u};
      e = make_tmap_im2col(&tx, x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, dims, strides, pl.lower, pl.upper, 64,
                           (uint32_t)(conv_tile_width(f) / 2), es, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    const char* gname = "none";
    if (e == cudaSuccess) e = launch_gemm_f16pair_conv(f, tx, s, &gname);
    return finish_launch(e, "conv_f16_nhwc+gemm_tc05_pair_f16ops_conv_im2col");
  }
  __half* col = reinterpret_cast<__half*>(base + pl.off_col);
  int* rs = reinterpret_cast<int*>(base + pl.off_rs);
  int* cs = reinterpret_cast<int*>(base + pl.off_cs);
  // rowsum(W) serves the x_zp term, colsum(col) the w_zp term
  cudaError_t e = launch_rows_pitched(w, wu, (int)M, (int)pl.Kg, w16, pl.Kgp, x_zero_point ? rs : nullptr, s);
  if (e == cudaSuccess) {
    Im2colArgs a{};
    a.x = x;
    a.Nb = (int)N;
    a.C = (int)C;
    a.H = (int)H;
    a.W = (int)W;
    a.kH = (int)kH;
    a.kW = (int)kW;
    a.pt = (int)pl.pt;
    a.pl = (int)pl.pl;
    a.sh = (int)pl.sh;
    a.sw = (int)pl.sw;
    a.dh = (int)pl.dh;
    a.dw = (int)pl.dw;
    a.oH = pl.oH;
    a.oW = pl.oW;
    a.G = (int)group;
    a.xzp = x_zero_point;
    a.col = col;
    a.pitch = pl.Pp;
    a.colsum = w_zp_count > 0 ? cs : nullptr;
    e = launch_im2col(a, xu, reinterpret_cast<int*>(base + pl.off_s), s);
  }
  GemmF16Args f{};
  f.A16 = w16;
  f.B16 = col;
  f.a_pitch = (int)pl.Kgp;
  f.b_pitch = (int)pl.Pp;
  f.a_bstride = group > 1 ? Mg * pl.Kgp : 0;
  f.a_bmod = group > 1 ? (int)group : 0;
  f.b_bstride = pl.Kg * pl.Pp;
  f.batch = (int)batch;
  f.M = (int)Mg;
  f.K = (int)pl.Kg;
  f.N = (int)pl.P;
  f.C = y;
  f.a_zp = w_zero_point;
  f.a_zp_count = (int)w_zp_count;
  f.b_zp = x_zero_point;
  f.b_zp_count = x_zero_point ? 1 : 0;
  f.rowsum = rs;
  f.colsum = cs;
  f.zp_row_mod = (int)Mg;
  f.err = err;
  const char* gname = "none";
  if (e == cudaSuccess) e = launch_gemm_f16pair(f, wu, xu, true, chunk_k_for(wu, xu), s, &gname);
  return finish_launch(e, "im2col_f16+gemm_tc05_pair_f16ops_matmul_integer");
}

size_t dynamic_quantize_matmul_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N) || M == 0 || K == 0 || N == 0) return 0;
  return dqm_plan(M, K, N).bytes;
}

namespace {

// Host checks shared by the chain's two entry points; QMM_OK means "go on",
// with *nothing = true for an empty output (nothing to launch).
qmm_status dqm_check(int64_t M, int64_t K, int64_t N, int w_dtype, int64_t w_scale_count, int64_t w_zp_count,
                     bool* nothing) {
  *nothing = false;
  if (!dim_ok(M) || !dim_ok(K) || !dim_ok(N)) return QMM_ERR_INVALID_ARG;
  if (w_dtype != QMM_S8 && w_dtype != QMM_U8) return QMM_ERR_INVALID_ARG;
  if (w_scale_count != 1 && w_scale_count != N) return QMM_ERR_INVALID_ARG;
  if (w_zp_count != 0 && w_zp_count != 1 && w_zp_count != N) return QMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    *nothing = true;
    return QMM_OK;
  }
  if (K == 0) return QMM_ERR_UNSUPPORTED;
  if (((M + 255) / 256) * ((N + 223) / 224) > (int64_t)INT_MAX || M * K / 32768 > (int64_t)INT_MAX)
    return QMM_ERR_UNSUPPORTED;
  return QMM_OK;
}

// The chain's GEMM: acc from y's fp16 copy (rows of pitch Kp) and W's (pitch
// Np), zero points and sums applied, times y_scale * w_scale[n], plus bias.
cudaError_t dqm_gemm(const __half* a16, int64_t Kp, const __half* b16, int64_t Np, const int* rs, const int* cs,
                     const float* ys, const uint8_t* yz, bool wu, int64_t M, int64_t K, int64_t N,
                     const float* w_scale, int64_t w_scale_count, const void* w_zero_point, int64_t w_zp_count,
                     const float* bias, float* C, unsigned* err, cudaStream_t s) {
  GemmF16Args f{};
  f.A16 = a16;
  f.B16 = b16;
  f.a_pitch = (int)Kp;
  f.b_pitch = (int)Np;
  f.batch = 1;
  f.M = (int)M;
  f.K = (int)K;
  f.N = (int)N;
  f.C = C;
  f.a_zp = yz;
  f.a_zp_count = 1;
  f.b_zp = w_zero_point;
  f.b_zp_count = (int)w_zp_count;
  f.rowsum = rs;
  f.colsum = cs;
  f.act_scale = ys;
  f.act_count = 1;
  f.w_scale = w_scale;
  f.w_count = (int)w_scale_count;
  f.bias = bias;
  f.zp_row_mod = (int)M;
  f.err = err;
  const char* gname = "none";
  return launch_gemm_f16pair(f, true, wu, true, chunk_k_for(true, wu), s, &gname);
}

}  // namespace

qmm_status dynamic_quantize_matmul(const float* x, int64_t M, int64_t K, const void* W, int w_dtype, int64_t N,
                                   const float* w_scale, int64_t w_scale_count, const void* w_zero_point,
                                   int64_t w_zp_count, const float* bias, float* C, float* y_scale,
                                   uint8_t* y_zero_point, void* workspace, size_t workspace_bytes, void* stream) {
  bool nothing = false;
  const qmm_status chk = dqm_check(M, K, N, w_dtype, w_scale_count, w_zp_count, &nothing);
  if (chk != QMM_OK) return chk;
  if (nothing) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (!x || !W || !w_scale || !C || (w_zp_count > 0 && !w_zero_point)) return QMM_ERR_INVALID_ARG;
  const DqmPlan pl = dqm_plan(M, K, N);
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  const bool wu = w_dtype == QMM_U8;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  __half* a16 = reinterpret_cast<__half*>(base + pl.off_a);
  __half* b16 = reinterpret_cast<__half*>(base + pl.off_b);
  int* rs = reinterpret_cast<int*>(base + pl.off_rs);
  int* cs = reinterpret_cast<int*>(base + pl.off_cs);
  float* ys = y_scale ? y_scale : reinterpret_cast<float*>(base + pl.off_sz);
  uint8_t* yz = y_zero_point ? y_zero_point : base + pl.off_sz + 16;
  // the weight (exact fp16 copy and column sums, the y_zp term) on a side stream,
  // beside the activations' DynamicQuantizeLinear straight into the fp16
  // operand with rowsum(y)
  auto side = [&](cudaStream_t st) { return dqm_convert_weight(W, wu, K, N, pl.Np, b16, cs, st); };
  auto primary = [&](cudaStream_t st) {
    return launch_dql_rows_f16(x, M, K, a16, pl.Kp, ys, yz, rs, reinterpret_cast<float*>(base),
                               dql_num_partials(M * K), st);
  };
  cudaError_t e = fork_join(s, side, primary);
  if (e == cudaSuccess)
    e = dqm_gemm(a16, pl.Kp, b16, pl.Np, rs, cs, ys, yz, wu, M, K, N, w_scale, w_scale_count, w_zero_point,
                 w_zp_count, bias, C, err, s);
  return finish_launch(e, "dql_f16+gemm_tc05_pair_f16ops_matmul_integer_dequant");
}

size_t dynamic_quantize_matmul_weight_bytes(int64_t K, int64_t N) {
  if (!dim_ok(K) || !dim_ok(N) || K == 0 || N == 0) return 0;
  return dqm_weight(K, N).bytes;
}

qmm_status dynamic_quantize_matmul_pack_weight(const void* W, int w_dtype, int64_t K, int64_t N, void* packed,
                                               size_t packed_bytes, void* stream) {
  if (!dim_ok(K) || !dim_ok(N) || K == 0 || N == 0) return QMM_ERR_INVALID_ARG;
  if (w_dtype != QMM_S8 && w_dtype != QMM_U8) return QMM_ERR_INVALID_ARG;
  const DqmWeight pw = dqm_weight(K, N);
  if (!W || !packed || !aligned16(packed) || packed_bytes < pw.bytes) return QMM_ERR_INVALID_ARG;
  cudaGetLastError();
  uint8_t* base = static_cast<uint8_t*>(packed);
  const cudaError_t e = dqm_convert_weight(W, w_dtype == QMM_U8, K, N, pw.Np, reinterpret_cast<__half*>(base),
                                           reinterpret_cast<int*>(base + pw.off_cs), static_cast<cudaStream_t>(stream));
  return finish_launch(e, "dqm_weight_f16");
}

size_t dynamic_quantize_matmul_packed_workspace_bytes(int64_t M, int64_t K) {
  if (!dim_ok(M) || !dim_ok(K) || M == 0 || K == 0) return 0;
  return dqm_plan(M, K, 0, false).bytes;
}

qmm_status dynamic_quantize_matmul_packed(const float* x, int64_t M, int64_t K, const void* packed,
                                          size_t packed_bytes, int w_dtype, int64_t N, const float* w_scale,
                                          int64_t w_scale_count, const void* w_zero_point, int64_t w_zp_count,
                                          const float* bias, float* C, float* y_scale, uint8_t* y_zero_point,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  bool nothing = false;
  const qmm_status chk = dqm_check(M, K, N, w_dtype, w_scale_count, w_zp_count, &nothing);
  if (chk != QMM_OK) return chk;
  if (nothing) {
    t_last_kernel = "none";
    return QMM_OK;
  }
  if (!x || !w_scale || !C || (w_zp_count > 0 && !w_zero_point)) return QMM_ERR_INVALID_ARG;
  const DqmWeight pw = dqm_weight(K, N);
  if (!packed || !aligned16(packed) || packed_bytes < pw.bytes) return QMM_ERR_INVALID_ARG;
  const DqmPlan pl = dqm_plan(M, K, N, false);
  if (!workspace || !aligned16(workspace) || workspace_bytes < pl.bytes) return QMM_ERR_INVALID_ARG;
  unsigned* err = err_word();
  if (!err) return QMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  uint8_t* base = static_cast<uint8_t*>(workspace);
  const uint8_t* wbase = static_cast<const uint8_t*>(packed);
  __half* a16 = reinterpret_cast<__half*>(base + pl.off_a);
  int* rs = reinterpret_cast<int*>(base + pl.off_rs);
  float* ys = y_scale ? y_scale : reinterpret_cast<float*>(base + pl.off_sz);
  uint8_t* yz = y_zero_point ? y_zero_point : base + pl.off_sz + 16;
  cudaError_t e = launch_dql_rows_f16(x, M, K, a16, pl.Kp, ys, yz, rs, reinterpret_cast<float*>(base),
                                      dql_num_partials(M * K), s);
  if (e == cudaSuccess)
    e = dqm_gemm(a16, pl.Kp, reinterpret_cast<const __half*>(wbase), pw.Np,
                 rs, reinterpret_cast<const int*>(wbase + pw.off_cs), ys, yz, w_dtype == QMM_U8, M, K, N, w_scale,
                 w_scale_count, w_zero_point, w_zp_count, bias, C, err, s);
  return finish_launch(e, "dql_f16+gemm_tc05_pair_f16ops_matmul_integer_dequant_packed");
}

size_t dynamic_quantize_linear_workspace_bytes(int64_t n) {
  long long p = (n + 32767) / 32768;
  if (p < 1) p = 1;
  if (p > kDqlMaxPartials) p = kDqlMaxPartials;
  return (size_t)p * 2 * sizeof(float);
}

qmm_status dynamic_quantize_linear(const float* x, int64_t n, uint8_t* y, float* y_scale, uint8_t* y_zero_point,
                                   int32_t* row_sums, int64_t row_len, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  if (n < 0) return QMM_ERR_INVALID_ARG;
  if (!y_scale || !y_zero_point || (n > 0 && (!x || !y))) return QMM_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % 16) != 0) return QMM_ERR_INVALID_ARG;
  if (workspace_bytes < dynamic_quantize_linear_workspace_bytes(n)) return QMM_ERR_INVALID_ARG;
  if (row_sums) {
    if (row_len <= 0 || n % row_len != 0) return QMM_ERR_INVALID_ARG;
    if (n / row_len > (int64_t)INT_MAX) return QMM_ERR_UNSUPPORTED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  const int parts = dql_num_partials(n);
  const char* name = "none";
  return finish_launch(launch_dql(x, n, y, y_scale, y_zero_point, row_sums, row_len,
                                  static_cast<float*>(workspace), parts, s, &name),
                       name);
}

}  // extern "C"
