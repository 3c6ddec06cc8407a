// Decode-shaped accumulating A8W8 (M <= 16): PyPTO PR #1920 lowers
// a8w8_matmul_dequant_acc to gemv_acc when the logical M is 1 (the review
// comments on choosing tile.gemv_acc). The weight stream K*N is read once, so
// the work is HBM-bound; the products are int8 x int8 summed exactly in int32
// (wrapping) with dp4a on the CUDA cores, then the A8W8 epilogue:
//   acc = acc_in + sum_k a*b;  C = out(f32(acc) * act_scale[m] * weight_scale[n]).
//
// Kernels by weight layout:
//  * B stored [N][K] (b_trans), up to 3 rows: a warp owns 4 columns; its
//    lanes stride K with 16-byte loads of each column's contiguous row, dp4a
//    against 16-byte loads of the activation rows, reduce across the warp and
//    run the epilogue.
//  * B stored [N][K], 4 to 16 rows: the products on the tensor cores
//    (gemv_acc_kmajor_tc_kernel, below), exact through fp32 partial sums of
//    at most 1024 k.
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

// ---------------------------------------------------------------------------
// B [N][K], 2..16 rows: the products on the tensor cores. dp4a costs one
// instruction per 4 bytes per activation row, which outgrows the weight
// stream as the rows increase; mma.sync.m16n8k16 (fp16 in, fp32 accumulate)
// takes 8 rows per instruction. Both operands hold the 8-bit integers
// exactly as fp16; every product is at most 2^14 in magnitude, so an fp32
// partial sum over at most 1024 k (2^24) is exact in any order, and each
// warp moves its partial sums into wrapping int32 every 1024 k.
//
// CTA: 64 columns, 8 warps = 4 groups of 16 columns x 2 contiguous halves of
// K. Lane (g, t) loads, per step, the CH contiguous bytes k0 + CH t .. of
// columns c0 + g and c0 + g + 8. The MMA's k order is permuted (the same way
// for both operands): MMA j of the step takes, in lane (g, t)'s k slots
// 2t, 2t+1 / 2t+8, 2t+9, the physical k = k0 + CH t + 4j + 0, 1 / + 2, 3 --
// byte word j of the lane's chunk -- so the loaded bytes are the A fragment
// as they are. The activations come as fp16 rows (acc_prep_kernel, exact),
// read just before their MMAs (every CTA reads the same rows: L1 keeps them).
// Each column row is read by one warp front to back; how many contiguous
// bytes of a row a warp requests at once sets the speed (8192 x 28672, 8
// rows: 16-byte pieces in alternating 64-k steps of the two halves 66 us,
// contiguous halves 57 us, 32-byte pieces 54 us).
// ---------------------------------------------------------------------------
constexpr int kTcCols = 64, kTcKPad = 256;   // activation rows padded to the longest step
// Up to 3 rows stay on dp4a (8192 x 28672: 42 us for 1 or 2 rows, near the
// copy rate); from 4 rows on the tensor cores are faster (4 rows: 52 against
// 54 us; 8: 54 against 75; 16: 60 against 123).
constexpr int kTcMinRows = 4;

__host__ __device__ constexpr long long tc_padded_k(long long K) { return (K + kTcKPad - 1) / kTcKPad * kTcKPad; }

// A (int8 [M][K], or [K][M] with a_trans) as exact fp16 [M][Kp], zero past K.
__global__ void __launch_bounds__(kThreads) acc_prep_kernel(const int8_t* __restrict__ A, int a_trans, int M, int K,
                                                            int Kp, __half* __restrict__ A16) {
  asm volatile("griddepcontrol.launch_dependents;");   // the GEMV starts its weight stream meanwhile
  const long long total = (long long)M * Kp;
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < total;
       i += (long long)gridDim.x * kThreads) {
    const int m = (int)(i / Kp), k = (int)(i % Kp);
    int v = 0;
    if (k < K) v = a_trans ? A[(size_t)k * M + m] : A[(size_t)m * K + k];
    A16[i] = __int2half_rn(v);
  }
}

__device__ __forceinline__ void mma_f16_f32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// CH: bytes of each of its two columns a lane loads per step (16, 32 or 64);
// a step is 4 CH of k, CH / 4 MMAs.
template <int MT, int D, int CH>
__global__ void __launch_bounds__(kThreads, 3) gemv_acc_kmajor_tc_kernel(const GemvAccArgs p,
                                                                         const __half* __restrict__ A16, int Kp) {
  constexpr int KS = 4 * CH;          // k per step
  constexpr int NL = CH / 16;         // 16-byte loads per column per step
  constexpr int NJ = CH / 4;          // MMAs per step
  constexpr int FLUSH = 1024 / KS;    // steps per exact fp32 partial
  __shared__ int red[4][MT * 4][32];   // the second K half's int32 sums, per column group
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int cg = warp & 3, kh = warp >> 2;
  const int c0 = blockIdx.x * kTcCols + cg * 16 + g;   // this lane's columns: c0 and c0 + 8
  const bool v0 = c0 < p.N, v1 = c0 + 8 < p.N;
  const int8_t* b0p = p.B + (size_t)(v0 ? c0 : 0) * p.K + CH * t;
  const int8_t* b1p = p.B + (size_t)(v1 ? c0 + 8 : 0) * p.K + CH * t;
  const int steps_all = Kp / KS;
  const int half0 = (steps_all + 1) / 2;
  const int s_beg = kh ? half0 : 0;                   // this warp's contiguous half of the steps
  const int nst = kh ? steps_all - half0 : half0;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  // step j's weight chunks (K % 16 == 0: each 16-byte piece lies wholly inside or past K)
  auto load_w = [&](uint4 (&w)[2][NL], int j) {
    const int k0 = (s_beg + j) * KS;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const bool in = k0 + CH * t + 16 * l < p.K;
      w[0][l] = (v0 && in) ? ldg_nc_v4(b0p + k0 + 16 * l) : zero;
      w[1][l] = (v1 && in) ? ldg_nc_v4(b1p + k0 + 16 * l) : zero;
    }
  };
  uint4 ring[D][2][NL];
#pragma unroll
  for (int d = 0; d < D; ++d)
    if (d < nst) load_w(ring[d], d);
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the fp16 activations are written

  bool live[MT];
  const __half* arow[MT];
#pragma unroll
  for (int nt = 0; nt < MT; ++nt) {
    const int m = 8 * nt + g;
    live[nt] = m < p.M;
    arow[nt] = A16 + (size_t)(live[nt] ? m : 0) * Kp + CH * t;
  }
  float facc[MT][4];
  uint32_t iacc[MT][4];
#pragma unroll
  for (int nt = 0; nt < MT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      facc[nt][e] = 0.f;
      iacc[nt][e] = 0u;
    }
  for (int base = 0; base < nst; base += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int j = base + d;
      if (j < nst) {
        const int k0 = (s_beg + j) * KS;
#pragma unroll
        for (int l = 0; l < NL; ++l) {   // 16 weight bytes per column: MMAs 4l .. 4l + 3
          uint4 act[MT][2];
#pragma unroll
          for (int nt = 0; nt < MT; ++nt) {
            act[nt][0] = live[nt] ? __ldg(reinterpret_cast<const uint4*>(arow[nt] + k0 + 16 * l)) : zero;
            act[nt][1] = live[nt] ? __ldg(reinterpret_cast<const uint4*>(arow[nt] + k0 + 16 * l + 8)) : zero;
          }
          const uint32_t w0[4] = {ring[d][0][l].x, ring[d][0][l].y, ring[d][0][l].z, ring[d][0][l].w};
          const uint32_t w1[4] = {ring[d][1][l].x, ring[d][1][l].y, ring[d][1][l].z, ring[d][1][l].w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            uint32_t a[4];
            bytes_to_half4<false>(w0[jj], a[0], a[2]);   // column c0:     k slots 2t, 2t+1 | 2t+8, 2t+9
            bytes_to_half4<false>(w1[jj], a[1], a[3]);   // column c0 + 8
#pragma unroll
            for (int nt = 0; nt < MT; ++nt) {
              const uint4& x = act[nt][jj >> 1];
              const uint32_t bl = (jj & 1) ? x.z : x.x, bh = (jj & 1) ? x.w : x.y;
              mma_f16_f32(facc[nt], a, bl, bh);
            }
          }
        }
        if (j + D < nst) load_w(ring[d], j + D);
        if ((j + 1) % FLUSH == 0) {   // 1024 k summed: move the exact partials to int32
#pragma unroll
          for (int nt = 0; nt < MT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              iacc[nt][e] += (uint32_t)__float2int_rn(facc[nt][e]);
              facc[nt][e] = 0.f;
            }
        }
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < MT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) iacc[nt][e] += (uint32_t)__float2int_rn(facc[nt][e]);
  // the second K half adds into the first (int32, wrapping: any order is exact)
  if (kh == 1)
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) red[cg][nt * 4 + e][lane] = (int)iacc[nt][e];
  __syncthreads();
  if (kh == 1) return;
  // lane (g, t) holds, per row tile nt: (column c0 | c0 + 8) x (row 8 nt + 2t | + 1)
#pragma unroll
  for (int nt = 0; nt < MT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = 8 * nt + 2 * t + (e & 1);
      const int n = c0 + ((e & 2) ? 8 : 0);
      if (m < p.M && n < p.N) {
        uint32_t v = iacc[nt][e] + (uint32_t)red[cg][nt * 4 + e][lane];
        if (p.acc_in) v += (uint32_t)__ldg(p.acc_in + (size_t)m * p.N + n);
        store_out(p, m, n, v);
      }
    }
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
  const size_t dp4a = (size_t)(((M * K + 255) / 256) * 256) + (size_t)M * N * 4;
  return std::max(dp4a, (size_t)M * (size_t)gva::tc_padded_k(K) * 2);   // the tensor-core route's fp16 rows
}

cudaError_t launch_gemv_acc(GemvAccArgs p, int a_trans, int b_trans, void* ws, cudaStream_t s,
                            const char** kernel_name) {
  using namespace gva;
  uint8_t* base = static_cast<uint8_t*>(ws);
  cudaError_t e = cudaSuccess;
  const int sms = std::max(1, num_sms());
  if (b_trans && p.M >= kTcMinRows) {
    // the tensor-core route: the activations as fp16 rows, then the GEMV,
    // launched as the prep's programmatic dependent
    const int Kp = (int)tc_padded_k(p.K);
    __half* a16 = reinterpret_cast<__half*>(base);
    const long long n = (long long)p.M * Kp;
    acc_prep_kernel<<<(int)std::min<long long>((n + kThreads - 1) / kThreads, 4LL * sms), kThreads, 0, s>>>(
        p.A, a_trans, p.M, p.K, Kp, a16);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *kernel_name = "gemv_acc_prep+gemv_acc_a8w8_kmajor_tc";
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.N + kTcCols - 1) / kTcCols), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const __half* ca16 = a16;
    // 32 contiguous bytes per lane and column for 8 rows; 16 rows (twice the
    // accumulators) keep 16-byte pieces three steps deep within 80 registers
    if (p.M <= 8) return cudaLaunchKernelEx(&cfg, gemv_acc_kmajor_tc_kernel<1, 2, 32>, p, ca16, Kp);
    return cudaLaunchKernelEx(&cfg, gemv_acc_kmajor_tc_kernel<2, 3, 16>, p, ca16, Kp);
  }
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
