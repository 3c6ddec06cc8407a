// Decode-shaped form (a): C[m,n] = scale_n * (sum_k A[m,k]*W[k,n] - zp_n * sum_k A[m,k])
// for a few activation rows (M <= 16, bf16) against a streamed int8 weight
// W [K,N] (row-major, N contiguous). The dequantised weight is never formed:
// int8 is widened to bf16 in registers (exact) and fed to the tensor cores,
// and the zero point is applied once per output through the factoring of
// TrainDeeploy PR #53 ("matmul that dequantises an int8 weight in-kernel",
// section "The kernel"). The small-M dispatch to this kernel follows the
// decode path of PyPTO PR #1920 (reviews on choosing tile.gemv when M == 1).
//
// The weight stream is the whole cost (K*N bytes), so the kernel is built
// around keeping HBM busy:
//  * each lane issues 16-byte loads of four consecutive K rows of W
//    (16 columns each), so a warp moves 2 KB of W per 16-K step and every
//    byte is loaded exactly once;
//  * the contraction uses mma.sync m16n8k16 (bf16 in, fp32 accumulate) with
//    the activation rows as the MMA's M (zero-padded to 16). Inside each
//    16-K step the K order is permuted -- fragment k index 2t,2t+1,2t+8,2t+9
//    of lane t maps to actual k 4t..4t+3 -- applied identically to A and W,
//    so a lane's four loaded rows are exactly the K values its fragments need
//    and no data moves between lanes;
//  * K is split over a cluster of 4 CTAs (8 warps each); warps reduce through
//    shared memory and the cluster reduces through distributed shared memory,
//    so there is no global workspace and the sum order is fixed.
#include "common.cuh"
#include "kernels.h"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace qmm {
namespace gemv {

constexpr int NWARP = 8;
constexpr int NTHR = NWARP * 32;
constexpr int CL = 4;          // CTAs per cluster = K splits
constexpr int BNW = 128;       // columns per CTA
constexpr int NTILE = BNW / 8; // n8 tiles per warp

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte `b` of the biased word (x ^ 0x80) as an exact float: the byte goes into
// the low mantissa bits of 2^23 and 2^23 + 128 is subtracted.
__device__ __forceinline__ float biased_byte_to_float(uint32_t xb, int b) {
  const uint32_t bits = prmt(xb, 0x4B000000u, 0x7440u | (uint32_t)b);
  return __uint_as_float(bits) - 8388736.0f;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct StepRegs {
  uint4 w[4];    // W rows k0+4t+i, columns 16g .. 16g+15 (int8)
  uint2 a_lo;    // A row g,   k0+4t .. k0+4t+3 (bf16)
  uint2 a_hi;    // A row g+8
};

__device__ __forceinline__ void load_step(const GemvArgs& p, int step, int n_col, int g, int t, StepRegs& r) {
  const int k = step * 16 + 4 * t;
  const bool k_ok = k < p.K;                 // K % 4 == 0: the 4 rows are all in or all out
  const bool n_ok = n_col < p.N;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    r.w[i] = (k_ok && n_ok) ? ldg_nc_v4(p.W + (size_t)(k + i) * p.N + n_col) : make_uint4(0, 0, 0, 0);
  r.a_lo = (k_ok && g < p.M) ? __ldg(reinterpret_cast<const uint2*>(p.A + (size_t)g * p.K + k)) : make_uint2(0, 0);
  r.a_hi = (k_ok && g + 8 < p.M) ? __ldg(reinterpret_cast<const uint2*>(p.A + (size_t)(g + 8) * p.K + k))
                                 : make_uint2(0, 0);
}

template <bool HAS_ZP>
__device__ __forceinline__ void compute_step(const StepRegs& r, float (&acc)[NTILE][4], float (&rs)[4]) {
  // A fragment with the permuted K order: a0/a2 = row g, a1/a3 = row g+8.
  const uint32_t a[4] = {r.a_lo.x, r.a_hi.x, r.a_lo.y, r.a_hi.y};
  uint32_t xb[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    xb[i][0] = r.w[i].x ^ 0x80808080u;
    xb[i][1] = r.w[i].y ^ 0x80808080u;
    xb[i][2] = r.w[i].z ^ 0x80808080u;
    xb[i][3] = r.w[i].w ^ 0x80808080u;
  }
#pragma unroll
  for (int j = 0; j < NTILE; ++j) {
    const int wq = j >> 2, b = j & 3;
    const uint32_t b0 = pack_bf16x2(biased_byte_to_float(xb[0][wq], b), biased_byte_to_float(xb[1][wq], b));
    const uint32_t b1 = pack_bf16x2(biased_byte_to_float(xb[2][wq], b), biased_byte_to_float(xb[3][wq], b));
    mma_bf16(acc[j], a, b0, b1);
  }
  if (HAS_ZP) {
    const uint32_t ones = 0x3F803F80u;   // bf16 (1, 1): the tile accumulates sum_k A[m,k]
    mma_bf16(rs, a, ones, ones);
  }
}

template <bool HAS_ZP>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NTHR, 2) gemv_kernel(const GemvArgs p) {
  constexpr int NACC = NTILE * 4 + (HAS_ZP ? 4 : 0);
  __shared__ float red[4][NACC][32];        // staged warp reduction (4 writer warps per round)
  cg::cluster_group cluster = cg::this_cluster();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int rank = (int)cluster.block_rank();
  const int nb = blockIdx.x / CL;
  const int n_col = nb * BNW + 16 * g;

  const int steps = (p.K + 15) / 16;
  const int s_beg = (int)(((long long)steps * rank) / CL);
  const int s_end = (int)(((long long)steps * (rank + 1)) / CL);

  float acc[NTILE][4];
  float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NTILE; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  // Two steps of loads in flight per warp.
  StepRegs r0, r1;
  int s = s_beg + warp;
  if (s < s_end) load_step(p, s, n_col, g, t, r0);
  if (s + NWARP < s_end) load_step(p, s + NWARP, n_col, g, t, r1);
  for (; s < s_end; s += NWARP) {
    StepRegs r2;
    if (s + 2 * NWARP < s_end) load_step(p, s + 2 * NWARP, n_col, g, t, r2);
    compute_step<HAS_ZP>(r0, acc, rs);
    r0 = r1;
    r1 = r2;
  }

  // Warp reduction inside the CTA, fixed order: 4..7 -> 0..3, then 2,3 -> 0,1, then 1 -> 0.
  auto put = [&](int slot) {
#pragma unroll
    for (int j = 0; j < NTILE; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) red[slot][j * 4 + e][lane] = acc[j][e];
    if (HAS_ZP)
#pragma unroll
      for (int e = 0; e < 4; ++e) red[slot][NTILE * 4 + e][lane] = rs[e];
  };
  auto take = [&](int slot) {
#pragma unroll
    for (int j = 0; j < NTILE; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] += red[slot][j * 4 + e][lane];
    if (HAS_ZP)
#pragma unroll
      for (int e = 0; e < 4; ++e) rs[e] += red[slot][NTILE * 4 + e][lane];
  };
#pragma unroll 1
  for (int half = NWARP / 2; half >= 1; half >>= 1) {
    if (warp >= half && warp < 2 * half) put(warp - half);
    __syncthreads();
    if (warp < half) take(warp);
    __syncthreads();
  }
  if (warp == 0) put(0);

  // Cluster reduction: rank 0 adds ranks 1..CL-1 in order through DSMEM.
  cluster.sync();
  if (rank == 0 && warp == 0) {
#pragma unroll 1
    for (int rr = 1; rr < CL; ++rr) {
      float(*peer)[NACC][32] = cluster.map_shared_rank(red, rr);
#pragma unroll
      for (int j = 0; j < NTILE; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] += peer[0][j * 4 + e][lane];
      if (HAS_ZP)
#pragma unroll
        for (int e = 0; e < 4; ++e) rs[e] += peer[0][NTILE * 4 + e][lane];
    }
  }
  cluster.sync();   // peers keep their shared memory alive until rank 0 has read it

  if (rank == 0 && warp == 0) {
    // Fragment element e of tile j: row g + 8*(e>>1), fragment column 2t + (e&1),
    // which is actual column nb*128 + 16*(2t + (e&1)) + j.
#pragma unroll
    for (int j = 0; j < NTILE; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = g + 8 * (e >> 1);
        const int n = nb * BNW + 16 * (2 * t + (e & 1)) + j;
        if (m < p.M && n < p.N) {
          const float sc = __ldg(p.scale + (p.scale_count == 1 ? 0 : n));
          float v = acc[j][e];
          if (HAS_ZP) {
            const float zp = (float)__ldg(p.zp + (p.zp_count == 1 ? 0 : n));
            v = __fsub_rn(v, __fmul_rn(zp, rs[e & 2]));
          }
          v = __fmul_rn(sc, v);
          if (p.c_f32)
            reinterpret_cast<float*>(p.C)[(size_t)m * p.N + n] = v;
          else
            reinterpret_cast<__nv_bfloat16*>(p.C)[(size_t)m * p.N + n] = __float2bfloat16_rn(v);
        }
      }
    }
  }
}

}  // namespace gemv

bool gemv_supported(long long M, long long K, long long N, const void* A, const void* W) {
  return M >= 1 && M <= 16 && K >= 4 && K % 4 == 0 && N % 16 == 0 && (reinterpret_cast<uintptr_t>(A) % 8) == 0 &&
         (reinterpret_cast<uintptr_t>(W) % 16) == 0;
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, const char** kernel_name) {
  using namespace gemv;
  const int nblocks = (a.N + BNW - 1) / BNW;
  const dim3 grid(nblocks * CL);
  if (a.zp_count > 0) {
    *kernel_name = "gemv_w8_bf16_mma_zp";
    gemv_kernel<true><<<grid, NTHR, 0, s>>>(a);
  } else {
    *kernel_name = "gemv_w8_bf16_mma";
    gemv_kernel<false><<<grid, NTHR, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace qmm
