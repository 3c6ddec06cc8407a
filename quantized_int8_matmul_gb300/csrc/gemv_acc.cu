// Decode-shaped accumulating A8W8 (M <= 16): PyPTO PR #1920 lowers
// a8w8_matmul_dequant_acc to gemv_acc when the logical M is 1 (the review
// comments on choosing tile.gemv_acc). The weight stream K*N is read once, so
// the work is HBM-bound; the products are int8 x int8 summed exactly in int32
// (wrapping) with dp4a on the CUDA cores, then the A8W8 epilogue:
//   acc = acc_in + sum_k a*b;  C = out(f32(acc) * act_scale[m] * weight_scale[n]).
//
// Two kernels, one per weight layout:
//  * B stored [N][K] (b_trans): a warp owns 4 columns; its lanes stride K with
//    16-byte loads of each column's contiguous row, dp4a against 16-byte loads
//    of the activation rows, reduce across the warp and run the epilogue.
//  * B stored [K][N]: a thread owns 4 adjacent columns and reads 4 rows x 4
//    bytes per step; six byte permutes turn them into 4 words of 4 k-values per
//    column for dp4a. The 8 warps of a block split K and reduce through shared
//    memory; blocks split K further and add their partial sums with int32
//    atomics into a buffer that holds acc_in, which a last small kernel turns
//    into C.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <climits>

namespace qmm {
namespace gva {

constexpr int kThreads = 256;

__device__ __forceinline__ void store_out(const GemvAccArgs& p, int m, int n, uint32_t acc) {
  const size_t i = (size_t)m * p.N + n;
  if (p.acc_out) p.acc_out[i] = (int)acc;
  if (!p.C) return;
  float v = __int2float_rn((int)acc);
  v = __fmul_rn(v, __ldg(p.act_scale + (p.act_count == 1 ? 0 : m)));
  v = __fmul_rn(v, __ldg(p.w_scale + (p.w_count == 1 ? 0 : n)));
  if (p.c_f32) static_cast<float*>(p.C)[i] = v;
  else static_cast<__nv_bfloat16*>(p.C)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ int dp4a_s8(uint32_t a, uint32_t b, int c) { return __dp4a((int)a, (int)b, c); }

// ---------------------------------------------------------------------------
// B [N][K]: one warp per 4 columns over all of K (K % 16 == 0, rows 16-byte aligned)
// ---------------------------------------------------------------------------
template <int MT>
__global__ void __launch_bounds__(kThreads) gemv_acc_kmajor_kernel(const GemvAccArgs p) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int n0 = (int)(warp * 4);
  if (n0 >= p.N) return;
  const int8_t* A = p.A;
  const int8_t* B = p.B;
  int acc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[m][j] = 0;
  const int K = p.K;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 2
  for (int k = lane * 16; k < K; k += 32 * 16) {
    uint4 b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = (n0 + j < p.N) ? ldg_nc_v4(B + (size_t)(n0 + j) * K + k) : zero;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < p.M) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(A + (size_t)m * K + k));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int t = acc[m][j];
          t = dp4a_s8(a.x, b[j].x, t);
          t = dp4a_s8(a.y, b[j].y, t);
          t = dp4a_s8(a.z, b[j].z, t);
          t = dp4a_s8(a.w, b[j].w, t);
          acc[m][j] = t;
        }
      }
    }
  }
  // every lane ends with every sum (int32 addition wraps, as the exact sum does)
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], o);
  // lane t writes output (m, j) = (t / 4, t % 4); a second pass covers M > 8
#pragma unroll
  for (int base = 0; base < MT * 4; base += 32) {
    const int t = base + lane;
    uint32_t v = 0u;
#pragma unroll
    for (int q = 0; q < MT * 4; ++q)
      if (q == t) v = (uint32_t)acc[q >> 2][q & 3];
    const int m = t >> 2, n = n0 + (t & 3);
    if (t < MT * 4 && m < p.M && n < p.N) {
      if (p.acc_in) v += (uint32_t)__ldg(p.acc_in + (size_t)m * p.N + n);
      store_out(p, m, n, v);
    }
  }
}

// ---------------------------------------------------------------------------
// B [K][N]: thread = 4 adjacent columns, warp = 128 columns, the block's 8
// warps split the block's K range (N % 4 == 0, K % 4 == 0, 4-byte alignment)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void transpose4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3, uint32_t (&c)[4]) {
  const uint32_t t0 = prmt(r0, r1, 0x5140u), t1 = prmt(r0, r1, 0x7362u);
  const uint32_t t2 = prmt(r2, r3, 0x5140u), t3 = prmt(r2, r3, 0x7362u);
  c[0] = prmt(t0, t2, 0x5410u);
  c[1] = prmt(t0, t2, 0x7632u);
  c[2] = prmt(t1, t3, 0x5410u);
  c[3] = prmt(t1, t3, 0x7632u);
}

template <int CPT>
struct RowLoad;
template <>
struct RowLoad<4> {
  static __device__ __forceinline__ void get(const int8_t* p, uint32_t (&w)[1]) {
    w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
  }
};
template <>
struct RowLoad<8> {
  static __device__ __forceinline__ void get(const int8_t* p, uint32_t (&w)[2]) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = v.x;
    w[1] = v.y;
  }
};
template <>
struct RowLoad<16> {
  static __device__ __forceinline__ void get(const int8_t* p, uint32_t (&w)[4]) {
    const uint4 v = ldg_nc_v4(p);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
};

// CPT adjacent columns per thread (CPT-byte loads per row), MT activation rows.
template <int MT, int CPT>
__global__ void __launch_bounds__(kThreads) gemv_acc_nmajor_kernel(const GemvAccArgs p, int k_per_block,
                                                                   int* __restrict__ R) {
  constexpr int W = CPT / 4;        // words per row and thread
  constexpr int BW = 32 * CPT;      // columns per block
  __shared__ int red[MT][BW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = blockIdx.x * BW;
  const int n0 = nb + lane * CPT;
  const int kb0 = blockIdx.y * k_per_block;
  const int kb1 = min(p.K, kb0 + k_per_block);
  const int kw = ((kb1 - kb0 + 31) / 32) * 4;   // rows per warp, a multiple of 4
  const int k0 = kb0 + warp * kw, k1 = min(kb1, k0 + kw);
  for (int i = threadIdx.x; i < MT * BW; i += kThreads) red[i / BW][i % BW] = 0;
  __syncthreads();
  int acc[MT][CPT];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < CPT; ++j) acc[m][j] = 0;
  if (n0 < p.N) {
    const int8_t* B = p.B + n0;
#pragma unroll 2
    for (int k = k0; k < k1; k += 4) {
      uint32_t r[4][W];
#pragma unroll
      for (int i = 0; i < 4; ++i) RowLoad<CPT>::get(B + (size_t)(k + i) * p.N, r[i]);
      uint32_t c[W][4];
#pragma unroll
      for (int w = 0; w < W; ++w) transpose4(r[0][w], r[1][w], r[2][w], r[3][w], c[w]);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
          const uint32_t a = __ldg(reinterpret_cast<const uint32_t*>(p.A + (size_t)m * p.K + k));
#pragma unroll
          for (int j = 0; j < CPT; ++j) acc[m][j] = dp4a_s8(a, c[j >> 2][j & 3], acc[m][j]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < CPT; ++j)
      if (m < p.M && acc[m][j] != 0) atomicAdd(&red[m][lane * CPT + j], acc[m][j]);
  __syncthreads();
  for (int i = threadIdx.x; i < MT * BW; i += kThreads) {
    const int m = i / BW, n = nb + (i % BW);
    if (m < p.M && n < p.N) atomicAdd(R + (size_t)m * p.N + n, red[m][i % BW]);
  }
}

template <int MT, int CPT>
void launch_nmajor(const GemvAccArgs& p, int* R, int sms, cudaStream_t s) {
  constexpr int BW = 32 * CPT;
  const int nblk = (p.N + BW - 1) / BW;
  // blocks: BW-column blocks x K splits, about four blocks per SM
  int ks = (int)std::max<long long>(1, std::min<long long>((4LL * sms + nblk - 1) / nblk, (p.K + 127) / 128));
  ks = std::min(ks, 65535);
  const int kpb = ((p.K + ks - 1) / ks + 3) / 4 * 4;
  ks = (p.K + kpb - 1) / kpb;
  gemv_acc_nmajor_kernel<MT, CPT><<<dim3((unsigned)nblk, (unsigned)ks), kThreads, 0, s>>>(p, kpb, R);
}

template <int MT>
void launch_nmajor_cols(const GemvAccArgs& p, int* R, int sms, cudaStream_t s) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(p.B);
  // the widest loads the row length and alignment allow, within 64 accumulators a thread
  if (MT * 16 <= 64 && p.N % 16 == 0 && b % 16 == 0) return launch_nmajor<MT, (MT * 16 <= 64 ? 16 : 4)>(p, R, sms, s);
  if (MT * 8 <= 64 && p.N % 8 == 0 && b % 8 == 0) return launch_nmajor<MT, (MT * 8 <= 64 ? 8 : 4)>(p, R, sms, s);
  launch_nmajor<MT, 4>(p, R, sms, s);
}

// R = acc_in (or 0) before the partial sums are added.
__global__ void __launch_bounds__(kThreads) init_kernel(const int* __restrict__ acc_in, int* __restrict__ R,
                                                        long long n) {
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < n; i += (long long)gridDim.x * kThreads)
    R[i] = acc_in ? __ldg(acc_in + i) : 0;
}

__global__ void __launch_bounds__(kThreads) finish_kernel(const GemvAccArgs p, const int* __restrict__ R) {
  const long long n = (long long)p.M * p.N;
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < n; i += (long long)gridDim.x * kThreads)
    store_out(p, (int)(i / p.N), (int)(i % p.N), (uint32_t)R[i]);
}

// int8 [K][M] -> [M][K] (the activations of a_trans; M <= 16).
__global__ void __launch_bounds__(kThreads) transpose_a_kernel(const int8_t* __restrict__ src, int K, int M,
                                                               int8_t* __restrict__ dst) {
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < (long long)K * M;
       i += (long long)gridDim.x * kThreads) {
    const int k = (int)(i / M), m = (int)(i % M);
    dst[(size_t)m * K + k] = src[i];
  }
}

}  // namespace gva

bool gemv_acc_supported(long long M, long long K, long long N, int b_trans, const void* A, const void* B) {
  if (M < 1 || M > 16 || K < 1 || N < 1 || K > INT_MAX || N > INT_MAX) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(A), b = reinterpret_cast<uintptr_t>(B);
  if (b_trans) return K % 16 == 0 && b % 16 == 0 && a % 16 == 0;
  return K % 4 == 0 && N % 4 == 0 && b % 4 == 0 && a % 4 == 0;
}

size_t gemv_acc_workspace_bytes(long long M, long long K, long long N) {
  return (size_t)(((M * K + 255) / 256) * 256) + (size_t)M * N * 4;
}

cudaError_t launch_gemv_acc(GemvAccArgs p, int a_trans, int b_trans, void* ws, cudaStream_t s,
                            const char** kernel_name) {
  using namespace gva;
  uint8_t* base = static_cast<uint8_t*>(ws);
  cudaError_t e = cudaSuccess;
  const int sms = std::max(1, num_sms());
  if (a_trans) {   // the activations as [M][K]
    int8_t* at = reinterpret_cast<int8_t*>(base);
    const long long n = (long long)p.K * p.M;
    transpose_a_kernel<<<(int)std::min<long long>((n + kThreads - 1) / kThreads, 4LL * sms), kThreads, 0, s>>>(
        p.A, p.K, p.M, at);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.A = at;
  }
  const int mt = p.M <= 1 ? 1 : p.M <= 2 ? 2 : p.M <= 4 ? 4 : p.M <= 8 ? 8 : 16;
  if (b_trans) {
    *kernel_name = "gemv_acc_a8w8_kmajor";
    const long long warps = ((long long)p.N + 3) / 4;
    const long long blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks > INT_MAX) return cudaErrorInvalidValue;
    switch (mt) {
      case 1: gemv_acc_kmajor_kernel<1><<<(int)blocks, kThreads, 0, s>>>(p); break;
      case 2: gemv_acc_kmajor_kernel<2><<<(int)blocks, kThreads, 0, s>>>(p); break;
      case 4: gemv_acc_kmajor_kernel<4><<<(int)blocks, kThreads, 0, s>>>(p); break;
      case 8: gemv_acc_kmajor_kernel<8><<<(int)blocks, kThreads, 0, s>>>(p); break;
      default: gemv_acc_kmajor_kernel<16><<<(int)blocks, kThreads, 0, s>>>(p); break;
    }
    return cudaGetLastError();
  }
  *kernel_name = "gemv_acc_a8w8_nmajor";
  int* R = reinterpret_cast<int*>(base + ((((size_t)p.M * p.K) + 255) / 256) * 256);
  const long long mn = (long long)p.M * p.N;
  const int eg = (int)std::max<long long>(1, std::min<long long>((mn + kThreads - 1) / kThreads, 4LL * sms));
  init_kernel<<<eg, kThreads, 0, s>>>(p.acc_in, R, mn);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (mt) {
    case 1: launch_nmajor_cols<1>(p, R, sms, s); break;
    case 2: launch_nmajor_cols<2>(p, R, sms, s); break;
    case 4: launch_nmajor_cols<4>(p, R, sms, s); break;
    case 8: launch_nmajor_cols<8>(p, R, sms, s); break;
    default: launch_nmajor_cols<16>(p, R, sms, s); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  finish_kernel<<<eg, kThreads, 0, s>>>(p, R);
  return cudaGetLastError();
}

}  // namespace qmm
