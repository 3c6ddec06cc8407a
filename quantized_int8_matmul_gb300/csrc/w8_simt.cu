// Form (a) on CUDA cores for any shape: float activations (fp32 or bf16)
// times an int8 weight with a per-tensor (or per-column) scale and zero point,
//   C[m,n] = scale_n * (sum_k A[m,k]*B[k,n] - zp_n * sum_k A[m,k]),
// the factoring of TrainDeeploy PR #53 ("matmul that dequantises an int8
// weight in-kernel", section "The kernel"): the int8 weight is read as int8,
// widened in registers, and the correction costs one multiply per output.
// With zp == 0 the correction vanishes and this is the fp32 loop with an
// int8 load (same section).
//
// 64x64 output tile per CTA, 256 threads, 4x4 outputs per thread, K tile 32
// staged in shared memory (A as float, B as float widened from int8).
#include "common.cuh"
#include "kernels.h"

namespace qmm {
namespace w8 {

constexpr int TM = 64, TN = 64, TK = 32;

__global__ void __launch_bounds__(256) w8_simt_kernel(const W8SimtArgs p) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x & 15;   // column group
  const int ty = threadIdx.x >> 4;   // row group
  const int m0 = blockIdx.y * TM;
  const int n0 = blockIdx.x * TN;

  float acc[4][4];
  float rsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  const float* Af = reinterpret_cast<const float*>(p.A);
  const __nv_bfloat16* Ah = reinterpret_cast<const __nv_bfloat16*>(p.A);

  for (int k0 = 0; k0 < p.K; k0 += TK) {
    for (int e = threadIdx.x; e < TM * TK; e += 256) {
      const int r = e / TK, c = e % TK;
      const int m = m0 + r, k = k0 + c;
      float v = 0.f;
      if (m < p.M && k < p.K) v = p.a_bf16 ? __bfloat162float(Ah[(size_t)m * p.K + k]) : Af[(size_t)m * p.K + k];
      As[c][r] = v;
    }
    for (int e = threadIdx.x; e < TK * TN; e += 256) {
      const int r = e / TN, c = e % TN;
      const int k = k0 + r, n = n0 + c;
      Bs[r][c] = (k < p.K && n < p.N) ? (float)p.B[(size_t)k * p.N + n] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rsum[i] += a[i];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= p.N) continue;
      const float sc = p.scale[p.scale_count == 1 ? 0 : n];
      float v = acc[i][j];
      if (p.zp_count > 0) {
        const float zp = (float)p.zp[p.zp_count == 1 ? 0 : n];
        v = __fsub_rn(v, __fmul_rn(zp, rsum[i]));
      }
      v = __fmul_rn(sc, v);
      if (p.c_f32)
        reinterpret_cast<float*>(p.C)[(size_t)m * p.N + n] = v;
      else
        reinterpret_cast<__nv_bfloat16*>(p.C)[(size_t)m * p.N + n] = __float2bfloat16_rn(v);
    }
  }
}

}  // namespace w8

cudaError_t launch_w8_simt(const W8SimtArgs& a, cudaStream_t s, const char** kernel_name) {
  const dim3 grid((a.N + w8::TN - 1) / w8::TN, (a.M + w8::TM - 1) / w8::TM);
  *kernel_name = "w8_dequant_simt";
  w8::w8_simt_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace qmm
