// DynamicQuantizeLinear to uint8, as lowered in ROCm hip-ep PR #1248
// ("feat(onnx-to-hip): lower quantized integer conv and matmul", section
// "What", DynamicQuantizeLinear paragraph): reduce the input to a scalar
// minimum and maximum, take scale = (max - min)/255 (scale 1 when the range is
// zero) and a ties-to-even zero point, then quantize.
//
// The range includes 0: lo = min(0, min x), hi = max(0, max x), which keeps
// zero exactly representable and the zero point inside [0, 255].
// Every float step is a single IEEE operation rounded to nearest even:
//   r = hi - lo; scale = r == 0 ? 1 : r / 255; zp = sat_u8(rne(-lo / scale));
//   y = sat_u8(rne(x / scale) + zp)
// with true division (__fdiv_rn), never a reciprocal multiply.
//
// Two passes over x (HBM-bound):
//   pass 1: each CTA reduces a contiguous chunk to a (min, max) partial;
//   pass 2: every CTA reduces all partials (order-free: min/max are exact),
//           derives scale and zero point, CTA 0 publishes them, and the grid
//           quantizes with 16-byte loads and 4-byte stores. Pass 2 walks the
//           chunks in reverse so its first reads hit what pass 1 left in L2.
//   Optionally pass 2 also writes the sum of each row of y (row_len elements),
//   the rowsum(A) a following MatMulInteger needs for its zero-point term.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace qmm {
namespace dql {

constexpr int THREADS = 256;
constexpr int UNROLL = 8;               // 16-byte loads in flight per thread
constexpr long long CHUNK_MIN = 32768;   // elements per pass-1 CTA at least

__device__ __forceinline__ void block_minmax(float& lo, float& hi) {
  __shared__ float slo[THREADS / 32], shi[THREADS / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    slo[w] = lo;
    shi[w] = hi;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    lo = threadIdx.x < THREADS / 32 ? slo[threadIdx.x] : 0.f;
    hi = threadIdx.x < THREADS / 32 ? shi[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void chunk_range(long long n, int parts, int b, long long& beg, long long& end) {
  // chunk boundaries on multiples of 4 elements so vector loads stay aligned
  const long long n4 = (n + 3) / 4;
  beg = (n4 * b / parts) * 4;
  end = (n4 * (b + 1) / parts) * 4;
  if (end > n) end = n;
  if (beg > n) beg = n;
}

__global__ void __launch_bounds__(THREADS) dql_minmax_kernel(const float* __restrict__ x, long long n, int vec,
                                                             float* __restrict__ partials) {
  long long beg, end;
  chunk_range(n, gridDim.x, blockIdx.x, beg, end);
  float lo = 0.f, hi = 0.f;   // the range always includes 0
  if (vec) {
    // UNROLL independent 16-byte loads in flight per thread
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const long long e4 = end / 4;
    long long i = beg / 4 + threadIdx.x;
    for (; i + (UNROLL - 1) * THREADS < e4; i += UNROLL * THREADS) {
      float4 v[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) v[u] = __ldg(x4 + i + u * THREADS);
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        lo = fminf(lo, fminf(fminf(v[u].x, v[u].y), fminf(v[u].z, v[u].w)));
        hi = fmaxf(hi, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
      }
    }
    for (; i < e4; i += THREADS) {
      const float4 v = __ldg(x4 + i);
      lo = fminf(lo, fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
      hi = fmaxf(hi, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
    }
    for (long long j = e4 * 4 + threadIdx.x; j < end; j += THREADS) {
      const float v = __ldg(x + j);
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
  } else {
    for (long long i = beg + threadIdx.x; i < end; i += THREADS) {
      const float v = __ldg(x + i);
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
  }
  block_minmax(lo, hi);
  if (threadIdx.x == 0) {
    partials[2 * blockIdx.x] = lo;
    partials[2 * blockIdx.x + 1] = hi;
  }
}

struct ScaleZp {
  float scale;
  float zp;       // integer-valued, in [0, 255]
};

__device__ __forceinline__ ScaleZp reduce_partials(const float* __restrict__ partials, int num_partials) {
  __shared__ ScaleZp s_out;
  float lo = 0.f, hi = 0.f;
  for (int i = threadIdx.x; i < num_partials; i += THREADS) {
    lo = fminf(lo, partials[2 * i]);
    hi = fmaxf(hi, partials[2 * i + 1]);
  }
  block_minmax(lo, hi);
  if (threadIdx.x == 0) {
    const float r = __fsub_rn(hi, lo);
    const float scale = (r == 0.f) ? 1.f : __fdiv_rn(r, 255.f);
    float zp = rintf(__fdiv_rn(-lo, scale));
    zp = fminf(fmaxf(zp, 0.f), 255.f);
    s_out.scale = scale;
    s_out.zp = zp;
  }
  __syncthreads();
  return s_out;
}

// x / scale, correctly rounded to nearest even, by Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/scale),
// q = RN(x*r) is within an ulp of x/scale, e = x - q*scale is exact as one
// FMA, and RN(q + e*r) is the correctly rounded quotient (a quotient of two
// floats is never exactly halfway between two floats). The residual e is only
// exact while it stays out of the subnormal range: for a quotient of at least
// 1/4 (smaller ones quantize to 0 either way) that holds when scale >= 2^-100,
// i.e. r <= 2^100. Outside that range (and when 1/scale is not a normal float)
// the callers fall back to IEEE division.
__device__ __forceinline__ float div_markstein(float x, float scale, float r) {
  const float q = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q, scale, x);
  return __fmaf_rn(e, r, q);
}

__device__ __forceinline__ uint32_t quant1(float v, float scale, int zp) {
  float q = rintf(__fdiv_rn(v, scale));
  q = fminf(fmaxf(q, -1024.f), 1024.f);   // keeps the int conversion in range; saturation follows
  int y = __float2int_rn(q) + zp;
  y = min(max(y, 0), 255);
  return (uint32_t)y;
}

// Same as quant1, with the division done by div_markstein (r = RN(1/scale)).
__device__ __forceinline__ uint32_t quant1r(float v, float scale, float r, int zp) {
  float q = rintf(div_markstein(v, scale, r));
  q = fminf(fmaxf(q, -1024.f), 1024.f);
  int y = __float2int_rn(q) + zp;
  y = min(max(y, 0), 255);
  return (uint32_t)y;
}

__device__ __forceinline__ uint32_t quant4(const float4 v, float scale, float r, int zp) {
  if (r != 0.f)
    return quant1r(v.x, scale, r, zp) | (quant1r(v.y, scale, r, zp) << 8) | (quant1r(v.z, scale, r, zp) << 16) |
           (quant1r(v.w, scale, r, zp) << 24);
  return quant1(v.x, scale, zp) | (quant1(v.y, scale, zp) << 8) | (quant1(v.z, scale, zp) << 16) |
         (quant1(v.w, scale, zp) << 24);
}

// RN(1/scale) when it is a normal float no larger than 2^100 (the residual of
// div_markstein is then exact), else 0 (= use IEEE division).
__device__ __forceinline__ float safe_recip(float scale) {
  const float r = __frcp_rn(scale);
  return (isfinite(r) && fabsf(r) >= 1.17549435e-38f && fabsf(r) <= 0x1p100f) ? r : 0.f;
}

__global__ void __launch_bounds__(THREADS) dql_quantize_kernel(const float* __restrict__ x, long long n, int vec,
                                                               const float* __restrict__ partials,
                                                               int num_partials, int num_chunks,
                                                               uint8_t* __restrict__ y, float* y_scale,
                                                               uint8_t* y_zp) {
  const ScaleZp sz = reduce_partials(partials, num_partials);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *y_scale = sz.scale;
    *y_zp = (uint8_t)(int)sz.zp;
  }
  const int zp = (int)sz.zp;
  const float rcp = safe_recip(sz.scale);
  // reverse chunk order: start where pass 1 finished
  for (int c = (int)gridDim.x - 1 - (int)blockIdx.x; c >= 0 && c < num_chunks; c -= (int)gridDim.x) {
    long long beg, end;
    chunk_range(n, num_chunks, c, beg, end);
    if (vec) {
      const float4* x4 = reinterpret_cast<const float4*>(x);
      uint32_t* y4 = reinterpret_cast<uint32_t*>(y);
      const long long e4 = end / 4;
      long long i = beg / 4 + threadIdx.x;
      for (; i + (UNROLL - 1) * THREADS < e4; i += UNROLL * THREADS) {
        float4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) v[u] = __ldg(x4 + i + u * THREADS);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) y4[i + u * THREADS] = quant4(v[u], sz.scale, rcp, zp);
      }
      for (; i < e4; i += THREADS) y4[i] = quant4(__ldg(x4 + i), sz.scale, rcp, zp);
      for (long long i = (end / 4) * 4 + threadIdx.x; i < end; i += THREADS)
        y[i] = (uint8_t)quant1(__ldg(x + i), sz.scale, zp);
    } else {
      for (long long i = beg + threadIdx.x; i < end; i += THREADS) y[i] = (uint8_t)quant1(__ldg(x + i), sz.scale, zp);
    }
  }
}

// Quantize whole rows, one warp per row, and write each row's sum of y.
__global__ void __launch_bounds__(THREADS) dql_quantize_rows_kernel(const float* __restrict__ x, long long rows,
                                                                    long long row_len, int vec,
                                                                    const float* __restrict__ partials,
                                                                    int num_partials, uint8_t* __restrict__ y,
                                                                    float* y_scale, uint8_t* y_zp,
                                                                    int32_t* __restrict__ row_sums) {
  const ScaleZp sz = reduce_partials(partials, num_partials);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *y_scale = sz.scale;
    *y_zp = (uint8_t)(int)sz.zp;
  }
  const int zp = (int)sz.zp;
  const float rcp = safe_recip(sz.scale);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total_warps = (long long)gridDim.x * (THREADS / 32);
  // reverse row order, as in the flat kernel
  for (long long wr = (long long)(gridDim.x - 1 - blockIdx.x) * (THREADS / 32) + warp; wr < rows;
       wr += total_warps) {
    const float* xr = x + wr * row_len;
    uint8_t* yr = y + wr * row_len;
    int s = 0;
    if (vec) {
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      uint32_t* y4 = reinterpret_cast<uint32_t*>(yr);
      const long long r4 = row_len / 4;
      long long i = lane;
      for (; i + (UNROLL - 1) * 32 < r4; i += UNROLL * 32) {
        float4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) v[u] = __ldg(x4 + i + u * 32);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
          const uint32_t w = quant4(v[u], sz.scale, rcp, zp);
          y4[i + u * 32] = w;
          s += (int)__dp4a(w, 0x01010101u, 0u);
        }
      }
      for (; i < r4; i += 32) {
        const uint32_t w = quant4(__ldg(x4 + i), sz.scale, rcp, zp);
        y4[i] = w;
        s += (int)__dp4a(w, 0x01010101u, 0u);
      }
    } else {
      for (long long i = lane; i < row_len; i += 32) {
        const uint32_t q = quant1(__ldg(xr + i), sz.scale, zp);
        yr[i] = (uint8_t)q;
        s += (int)q;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) row_sums[wr] = s;
  }
}

// The same row quantization written as exact fp16 values (0..255) into an
// operand copy whose rows are `pitch` elements apart, with each row's sum of
// y: the A operand of a following MatMulInteger GEMM, without the uint8 tensor
// in between.
__global__ void __launch_bounds__(THREADS) dql_quantize_rows_f16_kernel(const float* __restrict__ x, long long rows,
                                                                        long long row_len, int vec,
                                                                        const float* __restrict__ partials,
                                                                        int num_partials, __half* __restrict__ y16,
                                                                        long long pitch, float* y_scale,
                                                                        uint8_t* y_zp,
                                                                        int32_t* __restrict__ row_sums) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const ScaleZp sz = reduce_partials(partials, num_partials);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *y_scale = sz.scale;
    *y_zp = (uint8_t)(int)sz.zp;
  }
  const int zp = (int)sz.zp;
  const float rcp = safe_recip(sz.scale);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total_warps = (long long)gridDim.x * (THREADS / 32);
  for (long long wr = (long long)(gridDim.x - 1 - blockIdx.x) * (THREADS / 32) + warp; wr < rows;
       wr += total_warps) {
    const float* xr = x + wr * row_len;
    __half* yr = y16 + wr * pitch;
    int s = 0;
    if (vec) {   // x rows 16-byte aligned, row_len % 4 == 0: 4 values -> one 8-byte store
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      uint2* y4 = reinterpret_cast<uint2*>(yr);
      const long long r4 = row_len / 4;
      long long i = lane;
      for (; i + (UNROLL - 1) * 32 < r4; i += UNROLL * 32) {
        float4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) v[u] = __ldg(x4 + i + u * 32);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
          const uint32_t w = quant4(v[u], sz.scale, rcp, zp);
          uint2 h;
          bytes_to_half4<true>(w, h.x, h.y);
          y4[i + u * 32] = h;
          s += (int)__dp4a(w, 0x01010101u, 0u);
        }
      }
      for (; i < r4; i += 32) {
        const uint32_t w = quant4(__ldg(x4 + i), sz.scale, rcp, zp);
        uint2 h;
        bytes_to_half4<true>(w, h.x, h.y);
        y4[i] = h;
        s += (int)__dp4a(w, 0x01010101u, 0u);
      }
    } else {
      for (long long i = lane; i < row_len; i += 32) {
        const uint32_t q = quant1(__ldg(xr + i), sz.scale, zp);
        yr[i] = __int2half_rn((int)q);   // 0..255: exact
        s += (int)q;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) row_sums[wr] = s;
  }
}

}  // namespace dql

int dql_num_partials(long long n) {
  long long p = (n + dql::CHUNK_MIN - 1) / dql::CHUNK_MIN;
  if (p < 1) p = 1;
  const long long cap = std::min<long long>(kDqlMaxPartials, 4LL * std::max(1, num_sms()));
  return (int)std::min<long long>(p, cap);
}

cudaError_t launch_dql(const float* x, long long n, uint8_t* y, float* y_scale, uint8_t* y_zp, int32_t* row_sums,
                       long long row_len, float* partials, int num_partials, cudaStream_t s,
                       const char** kernel_name) {
  using namespace dql;
  const int vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (reinterpret_cast<uintptr_t>(y) % 4 == 0);
  dql_minmax_kernel<<<num_partials, THREADS, 0, s>>>(x, n, vec, partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (row_sums) {
    const long long rows = n / row_len;
    const int rvec = vec && (row_len % 4 == 0);
    const long long want = (rows + (THREADS / 32) - 1) / (THREADS / 32);
    const int grid = (int)std::max<long long>(1, std::min<long long>(want, 8LL * num_sms()));
    *kernel_name = "dql_minmax+dql_quantize_rows";
    dql_quantize_rows_kernel<<<grid, THREADS, 0, s>>>(x, rows, row_len, rvec, partials, num_partials, y, y_scale,
                                                       y_zp, row_sums);
  } else {
    *kernel_name = "dql_minmax+dql_quantize";
    dql_quantize_kernel<<<num_partials, THREADS, 0, s>>>(x, n, vec, partials, num_partials, num_partials, y,
                                                          y_scale, y_zp);
  }
  return cudaGetLastError();
}

}  // namespace qmm

namespace qmm {

cudaError_t launch_dql_rows_f16(const float* x, long long rows, long long row_len, __half* y16, long long pitch,
                                float* y_scale, uint8_t* y_zp, int32_t* row_sums, float* partials,
                                int num_partials, cudaStream_t s) {
  using namespace dql;
  if (rows <= 0 || row_len <= 0) return cudaSuccess;
  dql_minmax_kernel<<<num_partials, THREADS, 0, s>>>(x, rows * row_len, reinterpret_cast<uintptr_t>(x) % 16 == 0,
                                                     partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (row_len % 4 == 0) && (pitch % 4 == 0) &&
                  (reinterpret_cast<uintptr_t>(y16) % 8 == 0);
  const long long want = (rows + (THREADS / 32) - 1) / (THREADS / 32);
  const int grid = (int)std::max<long long>(1, std::min<long long>(want, 8LL * num_sms()));
  dql_quantize_rows_f16_kernel<<<grid, THREADS, 0, s>>>(x, rows, row_len, vec, partials, num_partials, y16, pitch,
                                                         y_scale, y_zp, row_sums);
  return cudaGetLastError();
}

}  // namespace qmm
