// DynamicQuantizeLinear for callers that cannot allocate device memory.
//
// dynamic_quantize_linear() needs a small scratch buffer for its per-CTA
// (min, max) partials and takes it from the caller. Some callers have no way
// to provide one: a plugin running inside a host framework that owns all
// device memory and exposes no allocator to it, an engine whose device
// memory is fixed once at start-up, or a latency-critical host thread that
// must not call cudaMalloc (which can synchronise the whole device). This
// entry point runs the same two kernels with the scratch taken from a
// fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (8 KiB) until the process exits. Host code cannot use the
// variable's name as a device address, so the address is looked up once per
// device with cudaGetSymbolAddress, on the first call made with that device
// current (and again if that device's context has been made anew, as after a
// cudaDeviceReset, since the array may then sit elsewhere). That first call
// should therefore come before any stream capture.
// All calls share the one array and it keeps the last call's contents; this
// is harmless because pass 1 writes every partial that pass 2 reads, so
// nothing in it needs to start at zero. Calls whose kernels overlap on the
// GPU (different streams without ordering) race on the array and give wrong
// results; order them on one stream.
#include "kernels.h"
#include "../../include/qmm.h"

#include <climits>
#include <mutex>

namespace qmm {
namespace {

// Room for kDqlMaxPartials (min, max) pairs: the most partials any n uses.
constexpr int kNoAllocFloats = 2 * kDqlMaxPartials;
static __device__ __align__(256) float g_dql_scratch[kNoAllocFloats];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDev] = {};
unsigned long long g_scratch_ctx[kMaxDev] = {};

// Device address of g_dql_scratch for the current device: looked up on the
// first call, and again whenever the device's current context is not the one
// the cached address was taken in.
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  const bool have = current_context_id(&ctx);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev] || !have || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dql_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(p);
    g_scratch_ctx[dev] = current_context_id(&ctx) ? ctx : 0;   // the lookup made the context current
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace qmm

extern "C" qmm_status dynamic_quantize_linear_noalloc(const float* x, int64_t n, uint8_t* y, float* y_scale,
                                                      uint8_t* y_zero_point, int32_t* row_sums, int64_t row_len,
                                                      void* stream) {
  using namespace qmm;
  if (n < 0) return QMM_ERR_INVALID_ARG;
  if (!y_scale || !y_zero_point || (n > 0 && (!x || !y))) return QMM_ERR_INVALID_ARG;
  if (row_sums) {
    if (row_len <= 0 || n % row_len != 0) return QMM_ERR_INVALID_ARG;
    if (n / row_len > (int64_t)INT_MAX) return QMM_ERR_UNSUPPORTED;
  }
  // The scratch holds at most kDqlMaxPartials partials; refuse anything that would need more.
  const int parts = dql_num_partials(n);
  if (parts < 1 || parts > kDqlMaxPartials ||
      dynamic_quantize_linear_workspace_bytes(n) > sizeof(float) * (size_t)kNoAllocFloats)
    return QMM_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  cudaGetLastError();
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e == cudaSuccess) {
    const char* name = "none";
    e = launch_dql(x, n, y, y_scale, y_zero_point, row_sums, row_len, scratch, parts,
                   static_cast<cudaStream_t>(stream), &name);
  }
  return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}
