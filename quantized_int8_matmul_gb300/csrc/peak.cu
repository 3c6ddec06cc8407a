// Measurement aid, not an operation of the method: the throughput of the
// legacy warp-level integer tensor path (mma.sync m16n8k32, s8 x s8 -> s32)
// on this GPU, the denominator of a "fraction of the int8 tensor peak". Every
// warp issues `iters` rounds of eight independent MMAs on register operands,
// so the launch measures the MMA pipe alone (no memory traffic).
#include "kernels.h"
#include "../../include/qmm.h"

namespace qmm {
namespace peak {

constexpr int kILP = 8;
constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 4;

__global__ void __launch_bounds__(kThreads) imma_kernel(int iters, uint32_t seed, int* sink) {
  const uint32_t a0 = seed ^ threadIdx.x, a1 = a0 * 3u, a2 = a0 * 5u, a3 = a0 * 7u, b0 = a0 * 11u, b1 = a0 * 13u;
  int d[kILP][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kILP; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+r"(d[j][0]), "+r"(d[j][1]), "+r"(d[j][2]), "+r"(d[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < kILP; ++j) s += d[j][0] ^ d[j][1] ^ d[j][2] ^ d[j][3];
  if (s == 0x7fffffff && sink) *sink = s;   // keeps the MMAs live; practically never taken
}

}  // namespace peak
}  // namespace qmm

extern "C" qmm_status qmm_int8_mma_peak_launch(int iters, double* ops, void* stream) {
  using namespace qmm;
  if (iters < 1 || !ops) return QMM_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms < 1) return QMM_ERR_CUDA;
  const int blocks = sms * peak::kBlocksPerSm;
  cudaGetLastError();
  peak::imma_kernel<<<blocks, peak::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(iters, 0x9E3779B9u, nullptr);
  if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
  const double warps = (double)blocks * peak::kThreads / 32.0;
  *ops = warps * iters * peak::kILP * 2.0 * 16 * 8 * 32;
  return QMM_OK;
}
