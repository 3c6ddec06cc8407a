// Decode-shaped form (a) against a weight packed once for the decode stream:
//   C[m,n] = scale_n * (sum_k A[m,k]*W[k,n] - zp_n * sum_k A[m,k])
// for 1..16 bf16 activation rows. The dequantised weight is never formed: each
// weight byte becomes an exact fp16 value in registers and feeds the tensor
// cores, and the zero point costs one multiply per output through the
// factoring of TrainDeeploy PR #53 ("matmul that dequantises an int8 weight
// in-kernel", section "The kernel"). The same page's follow-up makes the point
// that the win is reading a quarter of the bytes, so everything here serves
// the weight stream, which on this part only reaches the memory's read
// ceiling through plain register loads (TMA and cp.async streams stop near
// 4.8 and 3 TB/s) with enough of them in flight -- which in turn needs the
// per-byte instruction count low, or the warps spend their time converting
// instead of keeping loads in flight.
//
// The packed weight (qmm_w8_pack_decode_weight, the same K x N bytes, made
// once for a frozen weight) stores each lane's MMA fragments in order:
// per 64-column slab c and 16-row step s, lane l = 4g + t owns 32 bytes, and
// for fragment i (columns 64c + 8g + 2i and + 1, rows 16s + 4t .. + 3) they
// are the 8 bytes
//   [W[r0][c0], W[r1][c0], W[r0][c1], W[r1][c1], W[r2][c0], W[r3][c0], W[r2][c1], W[r3][c1]]
// each XORed with 0x80 (biased to unsigned). A step is 1 KB contiguous per
// warp (two 16-byte loads per lane), and every 16-bit half of an MMA A
// register is one byte permute into the mantissa of 1024 plus one half2
// subtraction away: about one instruction per weight byte, no interleaving,
// no address predicates (K and N are padded in the packed layout).
//
// The activations enter as fp16 copies of the bf16 rows scaled by a power of
// two per row (exact: the largest magnitude lands in [2^14, 2^15)). A row of
// up to 8192 values is prepared inside every CTA, into its shared memory,
// while its first weight loads are in flight; larger row sets are prepared by
// a small kernel the GEMV overlaps through programmatic dependent launch. The
// MMAs read each step's activation fragment just before use, from shared
// memory or from L1 (every CTA on an SM reads the same rows), so the register
// ring holds weight bytes only.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <utility>

namespace qmm {
namespace gvp {

constexpr int SLAB = 64;        // columns per CTA
constexpr int STEP = 16;        // K rows per warp step
constexpr int STEP_BYTES = 1024;

__host__ __device__ constexpr long long padded_k(long long K) { return (K + STEP - 1) / STEP * STEP; }
__host__ __device__ constexpr long long padded_n(long long N) { return (N + SLAB - 1) / SLAB * SLAB; }
// Byte offset of step s of slab c: each slab's steps contiguous.
__host__ __device__ __forceinline__ long long step_offset(long long c, long long s, long long steps) {
  return (c * steps + s) * STEP_BYTES;
}

// One thread per 8-byte fragment group: 4 rows x 2 columns of W, biased
// (rows past K and columns past N read as 0).
__global__ void __launch_bounds__(256) pack_kernel(const int8_t* __restrict__ W, int K, int N, long long steps,
                                                   long long groups, uint8_t* __restrict__ out) {
  for (long long u = (long long)blockIdx.x * 256 + threadIdx.x; u < groups; u += (long long)gridDim.x * 256) {
    const int i = (int)(u & 3);
    const int l = (int)((u >> 2) & 31);
    const long long s = (u >> 7) % steps;
    const long long c = (u >> 7) / steps;
    const int g = l >> 2, t = l & 3;
    const long long c0 = c * SLAB + 8 * g + 2 * i;
    const long long r0 = s * STEP + 4 * t;
    uint32_t b[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long r = r0 + j;
      const bool rv = r < K;
      const uint32_t v0 = (rv && c0 < N) ? (uint32_t)(uint8_t)__ldg(W + r * N + c0) : 0u;
      const uint32_t v1 = (rv && c0 + 1 < N) ? (uint32_t)(uint8_t)__ldg(W + r * N + c0 + 1) : 0u;
      // rows 0,1 -> bytes 0..3; rows 2,3 -> bytes 4..7; within a pair: [ra c0, rb c0, ra c1, rb c1]
      const int base = (j >> 1) * 4 + (j & 1);
      b[base] = v0;
      b[base + 2] = v1;
    }
    const uint32_t lo = (b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24)) ^ 0x80808080u;
    const uint32_t hi = (b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24)) ^ 0x80808080u;
    *reinterpret_cast<uint2*>(out + step_offset(c, s, steps) + l * 32 + i * 8) = make_uint2(lo, hi);
  }
}

// Power-of-two row scale: s puts the row's largest magnitude mx in
// [2^14, 2^15); 0 for an all-zero or non-finite row; clamped to [-100, 100]
// so that 2^s and 2^-s are normal floats.
__device__ __forceinline__ int row_shift(float mx) {
  const uint32_t ex = (__float_as_uint(mx) >> 23) & 0xFFu;
  return (mx > 0.f && ex != 0xFFu) ? max(-100, min(100, 14 - ((int)ex - 127))) : 0;
}

// One CTA per activation row: a power-of-two scale 2^s that puts the row's
// largest magnitude in [2^14, 2^15), then the scaled fp16 row in natural K
// order, zero-padded to Kp. (The GEMV reads no row past M.)
__global__ void __launch_bounds__(256) prep_kernel(const uint16_t* __restrict__ A, int K, int Kp,
                                                   uint16_t* __restrict__ A16, float* __restrict__ inv) {
  asm volatile("griddepcontrol.launch_dependents;");   // the GEMV starts its weight stream meanwhile
  __shared__ float red[8];
  const int row = blockIdx.x;
  uint16_t* d = A16 + (size_t)row * Kp;
  const uint16_t* a = A + (size_t)row * K;
  float mx = 0.f;
  for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {   // K % 8 == 0: 16-byte loads
    const uint4 v = *reinterpret_cast<const uint4*>(a + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mx = fmaxf(mx, fabsf(__uint_as_float(w[i] << 16)));
      mx = fmaxf(mx, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i]);
  const int sh = row_shift(mx);
  const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
  if (threadIdx.x == 0) inv[row] = __uint_as_float((uint32_t)(127 - sh) << 23);
  // K % 8 == 0: every 8-element group is wholly inside the row or wholly padding
  for (int k0 = threadIdx.x * 8; k0 < Kp; k0 += 256 * 8) {
    const uint4 v = k0 < K ? *reinterpret_cast<const uint4*>(a + k0) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __fmul_rn(__uint_as_float(w[q] << 16), up);
      const float hi = __fmul_rn(__uint_as_float(w[q] & 0xFFFF0000u), up);
      const __half2 h2 = __floats2half2_rn(lo, hi);
      out[q] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(d + k0) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Bytes 0, 1 (HI: 2, 3) of a word of biased bytes as an exact fp16 pair: each
// byte in the low mantissa bits of 1024 (fp16 0x6400, ulp 1), then 1024 + 128
// subtracted -- the byte's signed value.
template <bool HI>
__device__ __forceinline__ uint32_t biased_pair_to_half2(uint32_t x) {
  const uint32_t h = prmt(x, 0x64646464u, HI ? 0x4342u : 0x4140u);
  const __half2 v =
      __hsub2(*reinterpret_cast<const __half2*>(&h), __half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// The activation fragments, read just before their MMAs: every CTA on the SM
// reads the same rows, so they are kept in L1.
__device__ __forceinline__ uint2 ldg_v2_l1(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::evict_last.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// One warp step of one lane: its 32 packed weight bytes (loaded D steps
// ahead) and its activation fragments (read just before the MMAs).
template <int MT>
struct Step {
  uint4 w[2];
  uint32_t b[MT][2];   // activation rows 8 nt + g, k 4t..4t+3
};

template <int MT, bool ZP>
__device__ __forceinline__ void compute_step(const Step<MT>& st, float (&acc)[4][MT][4], float (&rs)[MT][4]) {
  const uint32_t wd[8] = {st.w[0].x, st.w[0].y, st.w[0].z, st.w[0].w, st.w[1].x, st.w[1].y, st.w[1].z, st.w[1].w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t a[4];
    a[0] = biased_pair_to_half2<false>(wd[2 * i]);       // MMA row g:     k 2t, 2t+1
    a[1] = biased_pair_to_half2<true>(wd[2 * i]);        // MMA row g + 8: k 2t, 2t+1
    a[2] = biased_pair_to_half2<false>(wd[2 * i + 1]);   // MMA row g:     k 2t+8, 2t+9
    a[3] = biased_pair_to_half2<true>(wd[2 * i + 1]);    // MMA row g + 8: k 2t+8, 2t+9
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) mma_f16(acc[i][nt], a, st.b[nt][0], st.b[nt][1]);
  }
  if (ZP) {
    const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) mma_f16(rs[nt], ones, st.b[nt][0], st.b[nt][1]);
  }
}

template <int MT, bool ZP>
struct Sizes {
  static constexpr int NACC = 4 * MT * 4;                  // MMA accumulators per lane
  static constexpr int NV = NACC + (ZP ? 2 * MT : 0);      // + row sums
};

struct PackedArgs {
  const uint8_t* Wp;       // packed weight
  const uint16_t* A;       // bf16 bits [M][K] (the in-CTA prep reads these)
  const uint16_t* A16;     // [M][Kp] fp16 (written by prep_kernel), row pitch Kp
  const float* inv;        // [M] 2^-s per row
  int M, K, N, Kp;
  const float* scale; int scale_count;
  const int32_t* zp;  int zp_count;
  void* C; int c_f32;
};

// Eight bf16 values scaled by 2^s (exact) and rounded to fp16.
__device__ __forceinline__ uint4 bf16x8_to_scaled_f16(const uint4 v, const float up) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2 h2 = __floats2half2_rn(__fmul_rn(__uint_as_float(w[q] << 16), up),
                                         __fmul_rn(__uint_as_float(w[q] & 0xFFFF0000u), up));
    o[q] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The prep inside each CTA (rows 0..M-1 only): every CTA finds each row's
// largest magnitude over all of K (so the CTAs of a split K share one scale
// per row, as with prep_kernel), then writes its own K range of the rows as
// scaled fp16 into shared memory, rows `pitch` halves apart, and 2^-s into
// inv_s. The fp16 values are those prep_kernel writes.
template <int NW>
__device__ __forceinline__ void prep_in_cta(const PackedArgs& p, int k_beg, int k_len, uint16_t* act, int pitch,
                                            float* inv_s) {
  __shared__ float rmax[NW][8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int m = 0; m < p.M; ++m) {
    const uint16_t* a = p.A + (size_t)m * p.K;
    float mx = 0.f;
    for (int k = tid * 8; k < p.K; k += NW * 32 * 8) {   // K % 8 == 0: 16-byte loads
      const uint4 v = *reinterpret_cast<const uint4*>(a + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mx = fmaxf(mx, fabsf(__uint_as_float(w[i] << 16)));
        mx = fmaxf(mx, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) rmax[warp][m] = mx;
  }
  __syncthreads();
  for (int m = 0; m < p.M; ++m) {
    float mx = rmax[0][m];
#pragma unroll
    for (int w = 1; w < NW; ++w) mx = fmaxf(mx, rmax[w][m]);
    const int sh = row_shift(mx);
    const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
    if (tid == 0) inv_s[m] = __uint_as_float((uint32_t)(127 - sh) << 23);
    const uint16_t* a = p.A + (size_t)m * p.K;
    for (int k = tid * 8; k < k_len; k += NW * 32 * 8) {   // groups of 8 wholly inside K or wholly padding
      const int kg = k_beg + k;
      const uint4 v = kg < p.K ? *reinterpret_cast<const uint4*>(a + kg) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(act + (size_t)m * pitch + k) = bf16x8_to_scaled_f16(v, up);
    }
  }
  __syncthreads();
}

__device__ __forceinline__ uint2 lds_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Shared-memory pitch (halves) of the in-CTA prep's rows: 16 halves of
// padding put consecutive rows 8 banks apart.
__host__ __device__ constexpr int act_pitch(int k_len) { return k_len + 16; }

// grid (slabs, S), cluster (1, S, 1): CTA (slab, ks) covers columns
// [64 slab, 64 slab + 64) and K steps [ks * spc, (ks + 1) * spc); its NW
// warps take the steps in turn, each keeping D steps of loads in flight.
// FP: the rows are prepared inside the CTA (prep_in_cta) instead of by
// prep_kernel; at most 8 rows.
template <int MT, bool ZP, int NW, int D, int MINB, bool FP>
__global__ void __launch_bounds__(NW * 32, MINB) gemv_packed_kernel(const PackedArgs p, const int spc) {
  static_assert(!FP || MT == 1, "in-CTA prep: up to 8 rows");
  constexpr int NV = Sizes<MT, ZP>::NV;
  extern __shared__ __align__(16) uint16_t act_s[];   // FP: [M][act_pitch(spc * STEP)] fp16
  __shared__ float inv_s[8];
  __shared__ float red[NW / 2][NV][32];   // the warp reduction (half the warps' values in flight)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int slab = blockIdx.x, ks = blockIdx.y;
  const int steps_all = p.Kp / STEP;
  const int s_beg = ks * spc;
  const int nsteps = max(0, min(steps_all, s_beg + spc) - s_beg);
  // this lane's bytes of the weight, and its activation rows
  const uint8_t* wp = p.Wp + (size_t)lane * 32;
  const uint16_t* arow[MT];
#pragma unroll
  for (int nt = 0; nt < MT; ++nt) arow[nt] = p.A16 + (size_t)(8 * nt + g) * p.Kp + 4 * t + (size_t)s_beg * STEP;

  float acc[4][MT][4];
  float rs[MT][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) acc[i][nt][0] = acc[i][nt][1] = acc[i][nt][2] = acc[i][nt][3] = 0.f;
#pragma unroll
  for (int nt = 0; nt < MT; ++nt) rs[nt][0] = rs[nt][1] = rs[nt][2] = rs[nt][3] = 0.f;

  // The first D steps' weight loads go out before the wait for the prep grid
  // (whose output the activation loads read).
  Step<MT> ring[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    const int st = warp + d * NW;
    if (st < nsteps) {
      const uint8_t* q = wp + step_offset(slab, s_beg + st, steps_all);
      ring[d].w[0] = ldg_nc_v4(q);
      ring[d].w[1] = ldg_nc_v4(q + 16);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  bool live[MT];   // activation rows past M are zero: not loaded
#pragma unroll
  for (int nt = 0; nt < MT; ++nt) live[nt] = 8 * nt + g < p.M;
  const int pitch = act_pitch(spc * STEP);
  uint32_t act_lane = 0;   // FP: this lane's row g, k 4t, in shared memory
  if (FP) {
    prep_in_cta<NW>(p, s_beg * STEP, nsteps * STEP, act_s, pitch, inv_s);
    act_lane = smem_u32(act_s) + (uint32_t)((g * pitch + 4 * t) * 2);
  }
  for (int base = warp; base < nsteps; base += D * NW) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int st = base + d * NW;
      if (st < nsteps) {
        // the activation fragments: rows read by every CTA on the SM, so hot in L1
#pragma unroll
          for (int nt = 0; nt < MT; ++nt) {
            const uint2 v = !live[nt] ? make_uint2(0u, 0u)
                            : FP      ? lds_v2(act_lane + (uint32_t)(st * STEP * 2))
                                      : ldg_v2_l1(arow[nt] + st * STEP);
            ring[d].b[nt][0] = v.x;
            ring[d].b[nt][1] = v.y;
          }
        compute_step<MT, ZP>(ring[d], acc, rs);
        const int nx = st + D * NW;   // refill the slot just used
        if (nx < nsteps) {
          const uint8_t* q = wp + step_offset(slab, s_beg + nx, steps_all);
          ring[d].w[0] = ldg_nc_v4(q);
          ring[d].w[1] = ldg_nc_v4(q + 16);
        }
      }
    }
  }

  // NW warps -> warp 0, fixed order (the upper half adds into the lower half).
  float v[NV];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int nt = 0; nt < MT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[(i * MT + nt) * 4 + e] = acc[i][nt][e];
  if (ZP)
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) {
      v[Sizes<MT, ZP>::NACC + 2 * nt] = rs[nt][0];
      v[Sizes<MT, ZP>::NACC + 2 * nt + 1] = rs[nt][1];
    }
#pragma unroll 1
  for (int half = NW / 2; half >= 1; half >>= 1) {
    if (warp >= half && warp < 2 * half)
#pragma unroll
      for (int i = 0; i < NV; ++i) red[warp - half][i][lane] = v[i];
    __syncthreads();
    if (warp < half)
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] += red[warp][i][lane];
    __syncthreads();
  }
  // With a split K, the cluster's CTAs (the K slices of this slab) add up in
  // rank order in rank 0; every CTA keeps its shared memory until rank 0 has
  // read it.
  const int S = (int)gridDim.y;
  if (S > 1) {
    if (warp == 0)
#pragma unroll
      for (int i = 0; i < NV; ++i) red[0][i][lane] = v[i];
    cluster_sync_all();
    if (ks == 0 && warp == 0) {
      for (int r = 1; r < S; ++r) {
        const uint32_t rb = mapa_shared(smem_u32(&red[0][0][lane]), (uint32_t)r);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          float x;
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(rb + (uint32_t)(i * 32 * 4)));
          v[i] += x;
        }
      }
    }
  }
  const int col = slab * SLAB + 8 * g;
  if (ks == 0 && warp == 0 && col < p.N) {
    // lane (g, t) holds columns col + 2i + cp of activation rows 8 nt + 2t + rp
    // (accumulator element rp + 2 cp of fragment i); N % 8 == 0, so its eight
    // columns are all in range
    const bool c_vec = (reinterpret_cast<uintptr_t>(p.C) % 16) == 0;
#pragma unroll
    for (int nt = 0; nt < MT; ++nt) {
#pragma unroll
      for (int rp = 0; rp < 2; ++rp) {
        const int m = 8 * nt + 2 * t + rp;
        if (m >= p.M) continue;
        const float inv = FP ? inv_s[m] : p.inv[m];
        const float rsum = ZP ? v[Sizes<MT, ZP>::NACC + 2 * nt + rp] : 0.f;
        float o[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int n = col + c;
          float r = v[((c >> 1) * MT + nt) * 4 + rp + 2 * (c & 1)];
          if (ZP) {
            const float zp = (float)__ldg(p.zp + (p.zp_count == 1 ? 0 : n));
            r = __fsub_rn(r, __fmul_rn(zp, rsum));
          }
          r = __fmul_rn(r, inv);   // undo the row's power-of-two scale (exact)
          o[c] = __fmul_rn(__ldg(p.scale + (p.scale_count == 1 ? 0 : n)), r);
        }
        const size_t off = (size_t)m * p.N + col;
        if (!c_vec) {
          for (int c = 0; c < 8; ++c) {
            if (p.c_f32)
              static_cast<float*>(p.C)[off + c] = o[c];
            else
              static_cast<__nv_bfloat16*>(p.C)[off + c] = __float2bfloat16_rn(o[c]);
          }
        } else if (p.c_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.C) + off);
          dst[0] = make_float4(o[0], o[1], o[2], o[3]);
          dst[1] = make_float4(o[4], o[5], o[6], o[7]);
        } else {
          uint32_t h[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[2 * q], o[2 * q + 1]);
            h[q] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.C) + off) = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
    }
  }
  if (S > 1) cluster_sync_all();
}

// Largest shared-memory share of the in-CTA prep's rows per CTA (one row of
// 8192). Shared memory takes its capacity from L1, which also holds the
// weight stream's loads in flight: with 4 rows (64 KB per CTA, three CTAs per
// SM) the 8192 x 28672 decode took 68 us against 51 us through prep_kernel,
// with 2 rows (33 KB) the two routes tied, with 1 row the in-CTA prep saved
// about 2 us (the prep kernel's latency before the first MMA).
constexpr int kFpSmemMax = 16 * 1024 + 512;

template <int MT, bool ZP, int NW, int D, int MINB, bool FP>
cudaError_t launch_impl(const PackedArgs& a, cudaStream_t s) {
  auto kern = gemv_packed_kernel<MT, ZP, NW, D, MINB, FP>;
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> per_sm_of;   // (device, dynamic smem bytes) -> CTAs per SM
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int steps_all = a.Kp / STEP;
  // the in-CTA prep's rows for the whole K: the most any split of K needs
  const int smem_full = FP ? a.M * act_pitch(a.Kp) * 2 : 0;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = per_sm_of.find({dev, smem_full});
    if (it == per_sm_of.end()) {
      int n = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NW * 32, smem_full);
      if (e != cudaSuccess) return e;
      it = per_sm_of.emplace(std::make_pair(dev, smem_full), std::max(1, n)).first;
    }
    per_sm = it->second;
  }
  const long long slots = (long long)per_sm * std::max(1, num_sms());
  const int slabs = (int)(padded_n(a.N) / SLAB);
  // Split K over a cluster only while all CTAs still fit in one wave and
  // every warp keeps at least 2 * D steps.
  int S = 1;
  while (S < 8 && (long long)slabs * 2 * S <= slots && steps_all / (2 * S) >= 2 * D * NW) S *= 2;
  const int spc = (steps_all + S - 1) / S;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the prep
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)slabs, (unsigned)S, 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = FP ? (size_t)a.M * act_pitch(spc * STEP) * 2 : 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = FP ? 1 : 2;   // no prep kernel to overlap with the in-CTA prep
  e = cudaLaunchKernelEx(&cfg, kern, a, spc);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The in-CTA prep applies to rows whose whole-K fp16 copy fits the per-CTA
// shared-memory share.
bool prep_fits_in_cta(int M, int Kp) { return M <= 8 && (long long)M * act_pitch(Kp) * 2 <= kFpSmemMax; }

}  // namespace gvp

size_t gemv_packed_weight_bytes(long long K, long long N) {
  if (K <= 0 || N <= 0) return 0;
  return (size_t)gvp::padded_k(K) * (size_t)gvp::padded_n(N);
}

size_t gemv_packed_workspace_bytes(long long M, long long K) {
  if (M <= 0 || M > 16 || K <= 0) return 0;
  const long long Mp = M <= 8 ? 8 : 16;
  return (size_t)((Mp * gvp::padded_k(K) * 2 + 255) / 256 * 256) + (size_t)((Mp * 4 + 255) / 256 * 256);
}

cudaError_t launch_gemv_pack(const int8_t* W, long long K, long long N, void* packed, cudaStream_t s) {
  using namespace gvp;
  const long long steps = padded_k(K) / STEP;
  const long long groups = (padded_n(N) / SLAB) * steps * 128;   // 8-byte groups: 32 lanes x 4 fragments per step
  const int grid = (int)std::max<long long>(1, std::min<long long>((groups + 255) / 256, 16LL * std::max(1, num_sms())));
  pack_kernel<<<grid, 256, 0, s>>>(W, (int)K, (int)N, steps, groups, static_cast<uint8_t*>(packed));
  return cudaGetLastError();
}

cudaError_t launch_gemv_packed(const GemvArgs& g, const void* packed, void* workspace, cudaStream_t s,
                               const char** kernel_name) {
  using namespace gvp;
  if (g.M < 1 || g.M > 16 || g.K < 8 || g.K % 8 != 0 || g.N < 8 || g.N % 8 != 0) return cudaErrorInvalidValue;
  const int Mp = g.M <= 8 ? 8 : 16;
  const int Kp = (int)padded_k(g.K);
  const bool fp = prep_fits_in_cta(g.M, Kp);
  uint16_t* a16 = static_cast<uint16_t*>(workspace);
  float* inv = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ((size_t)Mp * Kp * 2 + 255) / 256 * 256);
  if (!fp) {
    prep_kernel<<<g.M, 256, 0, s>>>(g.A, g.K, Kp, a16, inv);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  PackedArgs a{};
  a.Wp = static_cast<const uint8_t*>(packed);
  a.A = g.A;
  a.A16 = a16;
  a.inv = inv;
  a.M = g.M;
  a.K = g.K;
  a.N = g.N;
  a.Kp = Kp;
  a.scale = g.scale;
  a.scale_count = g.scale_count;
  a.zp = g.zp;
  a.zp_count = g.zp_count;
  a.C = g.C;
  a.c_f32 = g.c_f32;
  const bool zp = g.zp_count > 0;
  if (fp) {
    *kernel_name = zp ? "gemv_w8_packed_rows_in_cta_zp" : "gemv_w8_packed_rows_in_cta";
    return zp ? launch_impl<1, true, 8, 4, 3, true>(a, s) : launch_impl<1, false, 8, 4, 3, true>(a, s);
  }
  if (g.M <= 8) {
    *kernel_name = zp ? "gemv_prep_rows+gemv_w8_packed_zp" : "gemv_prep_rows+gemv_w8_packed";
    return zp ? launch_impl<1, true, 8, 4, 3, false>(a, s) : launch_impl<1, false, 8, 4, 3, false>(a, s);
  }
  *kernel_name = zp ? "gemv_prep_rows+gemv_w8_packed_m16_zp" : "gemv_prep_rows+gemv_w8_packed_m16";
  return zp ? launch_impl<2, true, 8, 2, 3, false>(a, s) : launch_impl<2, false, 8, 2, 3, false>(a, s);
}

}  // namespace qmm
