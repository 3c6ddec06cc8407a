// Decode-shaped form (a) for one to four activation rows on the CUDA cores:
//   C[m,n] = scale_n * (sum_k A[m,k]*W[k,n] - zp_n * sum_k A[m,k])
// (TrainDeeploy PR #53, "The kernel": the int8 weight is dequantised inside the
// kernel and the zero point is applied once per output through the row sum of
// A). The weight stream K*N is read once, so the kernel is built around the
// fewest instructions per weight byte:
//  * a thread owns 16 adjacent columns and reads each weight row with one
//    16-byte load; the bytes, biased to unsigned, go into the low mantissa of
//    2^23 by one byte permute each and one packed fp32 subtract per pair makes
//    them exact floats (|w| <= 128);
//  * packed fp32 FMAs (f32x2) accumulate a[m][k] * w for two columns at a time;
//  * the 8 warps of a block sit side by side on 4096 adjacent columns and read
//    the same rows, so each row is read as one contiguous 4 KB run; blocks
//    split K and write fp32 partial sums, which a second kernel adds in a fixed
//    order before applying the zero point and the scale. Results do not depend
//    on timing.
// About 2.5 instructions per weight byte for one row (the tensor-core GEMV
// needs ~4 for fragment handling), so HBM rather than issue sets the pace.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <climits>

namespace qmm {
namespace gvs {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCols = 16;                       // columns per thread
constexpr int kBlockCols = kWarps * 32 * kCols; // 4096 columns per block: the warps side by side
constexpr int kMaxSplits = 64;                  // K splits across blocks

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}

__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

template <bool BF16>
__device__ __forceinline__ float load_a(const void* A, size_t i) {
  if (BF16) return __uint_as_float((uint32_t)__ldg(static_cast<const unsigned short*>(A) + i) << 16);
  return __ldg(static_cast<const float*>(A) + i);
}

template <int MT, bool BF16>
__global__ void __launch_bounds__(kThreads) gemv_simt_kernel(const GemvSimtArgs p, int k_per_block,
                                                             float* __restrict__ part, float* __restrict__ rpart) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = blockIdx.x * kBlockCols;
  const int n0 = nb + (warp * 32 + lane) * kCols;
  const int k0 = blockIdx.y * k_per_block;
  const int k1 = min(p.K, k0 + k_per_block);
  unsigned long long acc[MT][kCols / 2];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < kCols / 2; ++j) acc[m][j] = 0ull;
  float rs[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) rs[m] = 0.f;
  const unsigned long long bias = pack2(-8388736.f, -8388736.f);   // 2^23 + 128
  const bool live = n0 < p.N;
  const int8_t* wcol = p.W + n0;
  // U rows per batch, double-buffered: the next batch's loads are in flight
  // while the current batch is converted and accumulated
  constexpr int U = MT <= 2 ? 4 : 2;
  uint4 w[2][U];
  float a[2][U][MT];
  auto load = [&](int buf, int kb) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = kb + u;
      const bool in = k < k1;
#pragma unroll
      for (int m = 0; m < MT; ++m) a[buf][u][m] = (in && m < p.M) ? load_a<BF16>(p.A, (size_t)m * p.K + k) : 0.f;
      w[buf][u] = (in && live) ? ldg_nc_v4(wcol + (size_t)k * p.N) : make_uint4(0u, 0u, 0u, 0u);   // a is 0 there too
    }
  };
  auto compute = [&](int buf) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int m = 0; m < MT; ++m) rs[m] += a[buf][u][m];
      const uint32_t uw[4] = {w[buf][u].x ^ 0x80808080u, w[buf][u].y ^ 0x80808080u, w[buf][u].z ^ 0x80808080u,
                              w[buf][u].w ^ 0x80808080u};
      unsigned long long v[kCols / 2];
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) {
        const uint32_t word = uw[j >> 1];
        const int b = (j & 1) * 2;
        const uint32_t lo = prmt(word, 0x4B000000u, 0x7440u | (uint32_t)b);
        const uint32_t hi = prmt(word, 0x4B000000u, 0x7440u | (uint32_t)(b + 1));
        v[j] = fadd2(((unsigned long long)hi << 32) | lo, bias);   // exact: two int8 values as floats
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const unsigned long long aa = pack2(a[buf][u][m], a[buf][u][m]);
#pragma unroll
        for (int j = 0; j < kCols / 2; ++j) acc[m][j] = ffma2(aa, v[j], acc[m][j]);
      }
    }
  };
  if (k0 < k1) load(0, k0);
  int kb = k0;
  for (; kb + U < k1; kb += 2 * U) {
    load(1, kb + U);
    compute(0);
    if (kb + 2 * U < k1) load(0, kb + 2 * U);
    compute(1);
  }
  if (kb < k1) compute(0);
  if (live) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m >= p.M) continue;
      float* dst = part + ((size_t)blockIdx.y * p.M + m) * p.N + n0;
#pragma unroll
      for (int j = 0; j < kCols / 2; j += 2)
        st_global_v4_hint(dst + 2 * j, (uint32_t)acc[m][j], (uint32_t)(acc[m][j] >> 32), (uint32_t)acc[m][j + 1],
                          (uint32_t)(acc[m][j + 1] >> 32), l2_policy_evict_first());
    }
  }
  // the row sums of A over this block's K range (every thread of the block has them)
  if (blockIdx.x == 0 && threadIdx.x == 0)
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (m < p.M) rpart[blockIdx.y * p.M + m] = rs[m];
}

__global__ void __launch_bounds__(kThreads) gemv_simt_finish_kernel(const GemvSimtArgs p, int splits,
                                                                    const float* __restrict__ part,
                                                                    const float* __restrict__ rpart) {
  const long long total = (long long)p.M * p.N;
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < total;
       i += (long long)gridDim.x * kThreads) {
    const int m = (int)(i / p.N), n = (int)(i - (long long)m * p.N);
    float s = 0.f, r = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
      s += __ldg(part + ((size_t)sp * p.M + m) * p.N + n);
      r += __ldg(rpart + sp * p.M + m);
    }
    float v = s;
    if (p.zp_count > 0) v = __fsub_rn(v, __fmul_rn((float)__ldg(p.zp + (p.zp_count == 1 ? 0 : n)), r));
    v = __fmul_rn(__ldg(p.scale + (p.scale_count == 1 ? 0 : n)), v);
    if (p.c_f32) static_cast<float*>(p.C)[i] = v;
    else static_cast<__nv_bfloat16*>(p.C)[i] = __float2bfloat16_rn(v);
  }
}

// Two waves of blocks: K is split so that the column blocks times the splits
// fill every SM to the kernel's occupancy twice (at least 32 rows per block).
template <int MT, bool BF16>
int launch_main(const GemvSimtArgs& p, float* part, float* rpart, cudaStream_t s) {
  auto kern = gemv_simt_kernel<MT, BF16>;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, 0) != cudaSuccess || occ < 1) occ = 1;
  const int sms = std::max(1, num_sms());
  const int nblk = (p.N + kBlockCols - 1) / kBlockCols;
  int splits = std::max(1, std::min(kMaxSplits, (2 * occ * sms + nblk - 1) / nblk));
  splits = std::max(1, std::min(splits, p.K / 32));
  const int kpb = (p.K + splits - 1) / splits;
  splits = (p.K + kpb - 1) / kpb;
  kern<<<dim3((unsigned)nblk, (unsigned)splits), kThreads, 0, s>>>(p, kpb, part, rpart);
  return splits;
}

template <bool BF16>
int launch_rows(const GemvSimtArgs& p, float* part, float* rpart, cudaStream_t s) {
  if (p.M == 1) return launch_main<1, BF16>(p, part, rpart, s);
  if (p.M == 2) return launch_main<2, BF16>(p, part, rpart, s);
  return launch_main<4, BF16>(p, part, rpart, s);
}

}  // namespace gvs

bool gemv_simt_supported(long long M, long long K, long long N, const void* W) {
  return M == 1 && K >= 1 && K <= INT_MAX && N >= 16 && N % 16 == 0 && N <= INT_MAX &&
         (reinterpret_cast<uintptr_t>(W) % 16) == 0;
}

size_t gemv_simt_workspace_bytes(long long M, long long N) {
  using namespace gvs;
  return (size_t)kMaxSplits * M * N * sizeof(float) + 256 + (size_t)kMaxSplits * M * sizeof(float);
}

cudaError_t launch_gemv_simt(const GemvSimtArgs& p, void* ws, cudaStream_t s, const char** kernel_name) {
  using namespace gvs;
  const int sms = std::max(1, num_sms());
  float* part = static_cast<float*>(ws);
  float* rpart = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                          (((size_t)kMaxSplits * p.M * p.N * sizeof(float) + 255) & ~(size_t)255));
  const int splits = p.a_bf16 ? launch_rows<true>(p, part, rpart, s) : launch_rows<false>(p, part, rpart, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long total = (long long)p.M * p.N;
  const int fg = (int)std::max<long long>(1, std::min<long long>((total + kThreads - 1) / kThreads, 4LL * sms));
  gemv_simt_finish_kernel<<<fg, kThreads, 0, s>>>(p, splits, part, rpart);
  *kernel_name = "gemv_w8_simt_f32x2";
  return cudaGetLastError();
}

}  // namespace qmm
