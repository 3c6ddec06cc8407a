// Decode-shaped form (a): C[m,n] = scale_n * (sum_k A[m,k]*W[k,n] - zp_n * sum_k A[m,k])
// for a few activation rows (M <= 16, bf16) against a streamed int8 weight
// W [K,N] (row-major, N contiguous). The dequantised weight is never formed:
// int8 is widened to bf16 in registers (exact) and fed to the tensor cores,
// and the zero point is applied once per output through the factoring of
// TrainDeeploy PR #53 ("matmul that dequantises an int8 weight in-kernel",
// section "The kernel"). The small-M dispatch to this kernel follows the
// decode path of PyPTO PR #1920 (reviews on choosing tile.gemv when M == 1).
//
// The weight stream (K*N bytes, read once) is the whole cost, so the kernel
// is built to keep HBM busy:
//  * one producer warp streams stages of W (256 k-rows x 64 columns, 16 KB,
//    64-byte swizzle) and of A (16 rows x 256 k, bf16, rows >= M zero-filled
//    by the copy) into a 5-stage shared-memory ring with TMA
//    (cp.async.bulk.tensor), so ~120 KB per SM are in flight without costing
//    registers;
//  * sixteen consumer warps each take one 16-deep K step of every stage and
//    run mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the activation rows
//    as the MMA's M (zero-padded to 16) and 8 n8 tiles covering 64 columns;
//  * the K order inside a step is permuted, identically for A and W: lane t of
//    a warp handles rows rb(t) + {0, 2, 8, 10} with rb = {0, 1, 4, 5}, which
//    gives the four row-groups of a half-warp distinct (row bit 0, row bit 2)
//    and so makes the 8-byte shared-memory reads of the swizzled stage
//    conflict-free;
//  * persistent CTAs walk 64-column blocks of N (fine enough to balance the
//    SMs) over the full K; the warps' partial sums are reduced through shared
//    memory in a fixed order.
#include "common.cuh"
#include "kernels.h"
#include "tma.h"

#include <algorithm>

namespace qmm {
namespace gemv {

constexpr int NCW = 16;                   // consumer warps, one 16-deep K step of a stage each
constexpr int NTHR = (NCW + 1) * 32;      // + one producer warp
constexpr int BNW = 64;                   // columns per block
constexpr int BKS = 16 * NCW;             // K rows per stage (256)
constexpr int NST = 5;                    // ring stages
constexpr int W_BYTES = BKS * BNW;        // 16 KB
constexpr int A_BOX = 16 * 64 * 2;        // one A box: 16 rows x 64 k bf16 (2 KB)
constexpr int A_BOXES = BKS / 64;
constexpr int STAGE = W_BYTES + A_BOXES * A_BOX;
constexpr int NTILE = BNW / 8;            // n8 tiles per warp
constexpr int NACC_MAX = NTILE * 4 + 4;

struct Shared {
  float red[NCW / 2][NACC_MAX][32];       // staged warp reduction
  uint64_t full[NST];
  uint64_t empty[NST];
  int abort_flag;
};

constexpr size_t SMEM_BYTES = (size_t)NST * STAGE + sizeof(Shared) + 1024;

enum : unsigned { SITE_FULL = 0x200, SITE_EMPTY = 0x201, SITE_DRAIN = 0x202 };

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

// Two floats that are small integers (|x| <= 128, so at most 8 significant
// bits) have all-zero low 16 bits: their bf16 values are exactly their top
// halves, so packing them is one byte permute (no rounding step needed).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return prmt(__float_as_uint(lo), __float_as_uint(hi), 0x7632u);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Bytes 0, 1 (HI: 2, 3) of a word of biased bytes as an fp16 pair: each byte
// goes into the low mantissa bits of 1024 (fp16 0x6400, ulp 1) and 1024 + 128
// is subtracted -- exact, the byte's signed value.
template <bool HI>
__device__ __forceinline__ uint32_t biased_pair_to_half2(uint32_t x) {
  const uint32_t h = prmt(x, 0x64646464u, HI ? 0x4342u : 0x4140u);
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// A[row][k] of the stage: 64-k boxes, 128-byte swizzle (16-byte chunk c of
// row r stored at chunk position c ^ (r % 8)).
__device__ __forceinline__ uint32_t a_addr(uint32_t a_base, int row, int k) {
  const int box = k >> 6, kk = k & 63;
  return a_base + (uint32_t)box * A_BOX + (uint32_t)row * 128u + ((uint32_t)((kk >> 3) ^ (row & 7)) << 4) +
         (uint32_t)(kk & 7) * 2u;
}

// Shared-memory offsets (within a stage) of one lane's operands for its warp's
// 16-deep K step: stage rows 16*warp + rb(t) + {0, 2, 8, 10}, rb = {0, 1, 4, 5}.
// They are the same for every stage, so they are computed once.
//  W stage: 64-byte rows, 64-byte swizzle (16-byte chunk c of row r stored at
//  chunk position c ^ ((r >> 1) & 3)); this lane reads 8 bytes (columns 8g..8g+7).
//  A stage: four 64-k boxes (see a_addr); this lane reads rows g and g + 8.
struct StepOffsets {
  uint32_t w[4];
  uint32_t a[8];   // [h * 4 + i]: row g + 8h, k = kb + {0, 2, 8, 10}[i]
};

__device__ __forceinline__ StepOffsets step_offsets(int warp, int g, int t) {
  StepOffsets o;
  const int kb = 16 * warp + (t & 1) + 4 * (t >> 1);
  const int ro[4] = {0, 2, 8, 10};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = kb + ro[i];
    o.w[i] = (uint32_t)r * 64u + ((uint32_t)((g >> 1) ^ ((r >> 1) & 3)) << 4) + (uint32_t)(g & 1) * 8u;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i) o.a[h * 4 + i] = a_addr((uint32_t)W_BYTES, g + 8 * h, kb + ro[i]);
  return o;
}

// One 16-deep K step of this warp on the stage at `sbase`.
template <bool HAS_ZP>
__device__ __forceinline__ void compute_step(uint32_t sbase, const StepOffsets& o, float (&acc)[NTILE][4],
                                             float (&rs)[4]) {
  uint32_t a[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {        // h = 0: row g (a0, a2); h = 1: row g + 8 (a1, a3)
    const uint32_t k0 = lds_u16(sbase + o.a[h * 4 + 0]);
    const uint32_t k1 = lds_u16(sbase + o.a[h * 4 + 1]);
    const uint32_t k2 = lds_u16(sbase + o.a[h * 4 + 2]);
    const uint32_t k3 = lds_u16(sbase + o.a[h * 4 + 3]);
    a[h] = prmt(k0, k1, 0x5410u);
    a[2 + h] = prmt(k2, k3, 0x5410u);
  }
  uint32_t xb[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint2 w = lds_v2(sbase + o.w[i]);
    xb[i][0] = w.x ^ 0x80808080u;
    xb[i][1] = w.y ^ 0x80808080u;
  }
#pragma unroll
  for (int j = 0; j < NTILE; ++j) {
    const int wq = j >> 2, b = j & 3;
    const uint32_t b0 = pack_bf16x2(biased_byte_to_float(xb[0][wq], b), biased_byte_to_float(xb[1][wq], b));
    const uint32_t b1 = pack_bf16x2(biased_byte_to_float(xb[2][wq], b), biased_byte_to_float(xb[3][wq], b));
    mma_bf16(acc[j], a, b0, b1);
  }
  if (HAS_ZP) {
    const uint32_t ones = 0x3F803F80u;   // bf16 (1, 1): this tile accumulates sum_k A[m,k]
    mma_bf16(rs, a, ones, ones);
  }
}

// The fp16 route's 16-deep K step: A (fp16, K-permuted by the prep so that the
// fragment's k order matches the rows this lane reads of W) with one
// ldmatrix; W rows rb + {0, 2} give b0 and rb + {8, 10} give b1 of every n8
// tile: the two rows' words interleaved byte by byte, each byte pair turned
// into an exact fp16 pair.
template <bool HAS_ZP>
__device__ __forceinline__ void compute_step_f16(uint32_t sbase, const StepOffsets& o, uint32_t a_ld,
                                                 float (&acc)[NTILE][4], float (&rs)[4]) {
  uint32_t a[4];
  ldmatrix_x4(a, sbase + a_ld);
  uint32_t x[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint2 w = lds_v2(sbase + o.w[i]);
    x[i][0] = w.x ^ 0x80808080u;
    x[i][1] = w.y ^ 0x80808080u;
  }
#pragma unroll
  for (int wq = 0; wq < 2; ++wq) {
    const uint32_t p01[2] = {prmt(x[0][wq], x[1][wq], 0x5140u), prmt(x[0][wq], x[1][wq], 0x7362u)};
    const uint32_t p23[2] = {prmt(x[2][wq], x[3][wq], 0x5140u), prmt(x[2][wq], x[3][wq], 0x7362u)};
#pragma unroll
    for (int b = 0; b < 4; ++b) {   // byte b of the words: tile 4 * wq + b
      const uint32_t b0 = (b & 1) ? biased_pair_to_half2<true>(p01[b >> 1]) : biased_pair_to_half2<false>(p01[b >> 1]);
      const uint32_t b1 = (b & 1) ? biased_pair_to_half2<true>(p23[b >> 1]) : biased_pair_to_half2<false>(p23[b >> 1]);
      mma_f16(acc[4 * wq + b], a, b0, b1);
    }
  }
  if (HAS_ZP) {
    const uint32_t ones = 0x3C003C00u;   // fp16 (1, 1): this tile accumulates sum_k A[m,k]
    mma_f16(rs, a, ones, ones);
  }
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory"); }

template <bool HAS_ZP, bool F16>
__global__ void __launch_bounds__(NTHR, 1)
    gemv_tma_kernel(const GemvArgs p, const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                    unsigned* err) {
  constexpr int NACC = NTILE * 4 + (HAS_ZP ? 4 : 0);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  Shared& sm = *reinterpret_cast<Shared*>(smem_raw + (sbase - raw) + NST * STAGE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nblocks = (p.N + BNW - 1) / BNW;
  const int spt = (p.K + BKS - 1) / BKS;   // stages per block
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], NCW);
    }
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();

  if (warp == NCW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmA);
      auto load_a = [&](int slot, int s) {
#pragma unroll
        for (int b = 0; b < A_BOXES; ++b)
          tma_load_2d(sbase + (uint32_t)slot * STAGE + W_BYTES + b * A_BOX, &tmA, s * BKS + 64 * b, 0,
                      &sm.full[slot]);
      };
      // fp16 route: the first ring's weight copies go out before the wait for
      // the prep grid (whose output A is); their activation copies after it
      const int my_blocks = blockIdx.x < nblocks ? (nblocks - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
      const int pre = F16 ? min(NST, my_blocks * spt) : 0;
      int it = 0;
      bool ok = true;
      for (int nb = blockIdx.x; nb < nblocks && ok; nb += gridDim.x) {
        for (int s = 0; s < spt; ++s, ++it) {
          const int slot = it % NST;
          if (it >= NST && !mbar_wait(&sm.empty[slot], (uint32_t)(((it / NST) - 1) & 1), &sm.abort_flag, err, SITE_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + (uint32_t)slot * STAGE;
          mbar_arrive_expect_tx(&sm.full[slot], STAGE);
          tma_load_2d(dst, &tmW, nb * BNW, s * BKS, &sm.full[slot]);
          if (it >= pre) load_a(slot, s);
          if (it == pre - 1) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int j = 0; j < pre; ++j) load_a(j, j % spt);
          }
        }
      }
      // Before the CTA exits, wait (bounded) until every copy issued has landed.
      for (int j = (it > NST ? it - NST : 0); j < it; ++j)
        mbar_wait(&sm.full[j % NST], (uint32_t)((j / NST) & 1), nullptr, err, SITE_DRAIN);
    }
    __syncwarp();
    return;
  }

  // ---------------- consumers ----------------
  const int g = lane >> 2;
  const int t = lane & 3;
  const StepOffsets so = step_offsets(warp, g, t);
  // fp16 route: this lane's ldmatrix row (matrix lane/8: rows +8 for odd, k +8
  // for the upper two) in the A box of this warp's 16-deep K step
  uint32_t a_ld = 0;
  if (F16) {
    const int q = lane >> 3, row = (q & 1) * 8 + (lane & 7);
    const int chunk = 2 * (warp & 3) + (q >> 1);
    a_ld = (uint32_t)W_BYTES + (uint32_t)(warp >> 2) * A_BOX + (uint32_t)row * 128u +
           ((uint32_t)(chunk ^ (row & 7)) << 4);
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the prep's row scales, read in the epilogue
  }
  int it = 0;
  bool ok = true;
  for (int nb = blockIdx.x; nb < nblocks; nb += gridDim.x) {
    float acc[NTILE][4];
    float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NTILE; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    for (int s = 0; s < spt; ++s, ++it) {
      const int slot = it % NST;
      if (ok) ok = mbar_wait(&sm.full[slot], (uint32_t)((it / NST) & 1), &sm.abort_flag, err, SITE_FULL);
      if (ok) {
        if (F16)
          compute_step_f16<HAS_ZP>(sbase + (uint32_t)slot * STAGE, so, a_ld, acc, rs);
        else
          compute_step<HAS_ZP>(sbase + (uint32_t)slot * STAGE, so, acc, rs);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }

    // Reduce the eight warps' partials in a fixed order: 4..7 -> 0..3, 2,3 -> 0,1, 1 -> 0.
#pragma unroll 1
    for (int half = NCW / 2; half >= 1; half >>= 1) {
      if (warp >= half && warp < 2 * half) {
#pragma unroll
        for (int j = 0; j < NTILE; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) sm.red[warp - half][j * 4 + e][lane] = acc[j][e];
        if (HAS_ZP)
#pragma unroll
          for (int e = 0; e < 4; ++e) sm.red[warp - half][NTILE * 4 + e][lane] = rs[e];
      }
      consumer_bar();
      if (warp < half) {
#pragma unroll
        for (int j = 0; j < NTILE; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] += sm.red[warp][j * 4 + e][lane];
        if (HAS_ZP)
#pragma unroll
          for (int e = 0; e < 4; ++e) rs[e] += sm.red[warp][NTILE * 4 + e][lane];
      }
      consumer_bar();
    }
    (void)NACC;

    if (warp == 0 && ok) {
      // Fragment element e of tile j: row g + 8*(e>>1), fragment column 2t + (e&1),
      // which is actual column nb*64 + 8*(2t + (e&1)) + j.
#pragma unroll
      for (int j = 0; j < NTILE; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = g + 8 * (e >> 1);
          const int n = nb * BNW + 8 * (2 * t + (e & 1)) + j;
          if (m < p.M && n < p.N) {
            const float sc = __ldg(p.scale + (p.scale_count == 1 ? 0 : n));
            float v = acc[j][e];
            if (HAS_ZP) {
              const float zp = (float)__ldg(p.zp + (p.zp_count == 1 ? 0 : n));
              v = __fsub_rn(v, __fmul_rn(zp, rs[e & 2]));
            }
            if (F16) v = __fmul_rn(v, p.inv[m]);   // undo the row's power-of-two scale (exact)
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
}

template <bool HAS_ZP, bool F16>
cudaError_t launch_impl(const GemvArgs& a, const CUtensorMap& tw, const CUtensorMap& ta, cudaStream_t s) {
  auto kern = gemv_tma_kernel<HAS_ZP, F16>;
  static unsigned attr_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || !(attr_mask & (1u << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 32) attr_mask |= 1u << dev;
  }
  const int nblocks = (a.N + BNW - 1) / BNW;
  const int grid = std::min(nblocks, num_sms());
  if (!F16) {
    kern<<<grid, NTHR, SMEM_BYTES, s>>>(a, tw, ta, a.err);
    return cudaGetLastError();
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the prep
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NTHR, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, tw, ta, a.err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The fp16 route's pre-pass: one CTA per activation row.
__global__ void __launch_bounds__(256) gemv_prep_kernel(const uint16_t* __restrict__ A, int K, int Kp,
                                                        uint16_t* __restrict__ A16, float* __restrict__ inv) {
  asm volatile("griddepcontrol.launch_dependents;");   // the GEMV starts its weight stream meanwhile
  __shared__ float red[8];
  const int row = blockIdx.x;
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
  // s: the row maximum times 2^s lies in [2^14, 2^15); 0 for an all-zero or
  // non-finite row; kept within [-100, 100] so 2^s and 2^-s are normal floats
  int sh = 0;
  const uint32_t ex = (__float_as_uint(mx) >> 23) & 0xFFu;
  if (mx > 0.f && ex != 0xFFu) sh = max(-100, min(100, 14 - ((int)ex - 127)));
  const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
  if (threadIdx.x == 0) inv[row] = __uint_as_float((uint32_t)(127 - sh) << 23);
  uint16_t* d = A16 + (size_t)row * Kp;
  for (int gq = threadIdx.x; gq < Kp / 16; gq += 256) {
    uint32_t out[8];
#pragma unroll
    for (int q = 0; q < 16; q += 2) {
      uint16_t hv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int qq = q + u;
        const int k = 16 * gq + ((qq & ~3) | ((qq & 1) << 1) | ((qq >> 1) & 1));   // bits 0 and 1 swapped
        const float x = k < K ? __uint_as_float((uint32_t)a[k] << 16) : 0.f;
        hv[u] = __half_as_ushort(__float2half_rn(__fmul_rn(x, up)));
      }
      out[q / 2] = (uint32_t)hv[0] | ((uint32_t)hv[1] << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(d + 16 * gq);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

}  // namespace gemv

bool gemv_supported(long long M, long long K, long long N, const void* A, const void* W) {
  return M >= 1 && M <= 16 && K >= 8 && K % 8 == 0 && N >= 16 && N % 16 == 0 &&
         (reinterpret_cast<uintptr_t>(A) % 16) == 0 && (reinterpret_cast<uintptr_t>(W) % 16) == 0;
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, const char** kernel_name) {
  using namespace gemv;
  CUtensorMap tw, ta;
  cudaError_t e = make_tmap_2d(&tw, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)a.N, (uint64_t)a.K,
                               (uint64_t)a.N, BNW, BKS, CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&ta, a.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, 64,
                   16, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  if (a.zp_count > 0) {
    *kernel_name = "gemv_w8_bf16_tma_zp";
    return launch_impl<true, false>(a, tw, ta, s);
  }
  *kernel_name = "gemv_w8_bf16_tma";
  return launch_impl<false, false>(a, tw, ta, s);
}

size_t gemv_f16_workspace_bytes(long long M, long long K) {
  if (M <= 0 || K <= 0) return 0;
  const long long Kp = (K + 15) / 16 * 16;
  return (size_t)((M * Kp * 2 + 255) / 256 * 256) + (size_t)((M * 4 + 255) / 256 * 256);
}

namespace gemv {
struct PrepLayout {
  int Kp;
  uint16_t* a16;
  float* inv;
};
PrepLayout prep_layout(int M, int K, void* ws) {
  PrepLayout l;
  l.Kp = (K + 15) / 16 * 16;
  l.a16 = static_cast<uint16_t*>(ws);
  l.inv = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ((size_t)M * l.Kp * 2 + 255) / 256 * 256);
  return l;
}
}  // namespace gemv

cudaError_t launch_gemv_prep(const uint16_t* A, int M, int K, void* workspace, cudaStream_t s) {
  using namespace gemv;
  if (M <= 0 || K <= 0 || K % 8 != 0) return cudaErrorInvalidValue;
  const PrepLayout l = prep_layout(M, K, workspace);
  gemv_prep_kernel<<<M, 256, 0, s>>>(A, K, l.Kp, l.a16, l.inv);
  return cudaGetLastError();
}

cudaError_t launch_gemv_f16(GemvArgs a, void* workspace, cudaStream_t s, const char** kernel_name) {
  using namespace gemv;
  const PrepLayout l = prep_layout(a.M, a.K, workspace);
  a.A16 = l.a16;
  a.inv = l.inv;
  a.Kp = l.Kp;
  CUtensorMap tw, ta;
  cudaError_t e = make_tmap_2d(&tw, a.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)a.N, (uint64_t)a.K,
                               (uint64_t)a.N, BNW, BKS, CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&ta, l.a16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)l.Kp, (uint64_t)a.M, (uint64_t)l.Kp * 2,
                   64, 16, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  if (a.zp_count > 0) {
    *kernel_name = "gemv_w8_f16_tma_zp";
    return launch_impl<true, true>(a, tw, ta, s);
  }
  *kernel_name = "gemv_w8_f16_tma";
  return launch_impl<false, true>(a, tw, ta, s);
}

}  // namespace qmm
