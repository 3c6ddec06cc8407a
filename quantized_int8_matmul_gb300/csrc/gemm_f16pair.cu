// Exact 8-bit GEMM on SM pairs from fp16 copies of the operands (made once by
// the pre-pass in convert.cu). The arithmetic is that of gemm_tc.cu: operands
// are 8-bit integers held exactly in fp16, tcgen05.mma kind::f16 sums their
// products exactly in fp32 over K-chunks no longer than 2^24 / max|product|,
// and each chunk is folded into wrapping int32 sums in TMEM (the INT32
// accumulator of PyPTO PR #1920's sequence diagram; the wrapping int32 of
// MatMulInteger in ROCm hip-ep PR #1248, "What"). Epilogues: A8W8 row-then-
// column scaling (PyPTO PR #1920), or the MatMulInteger zero-point expansion
//   acc - za*colsum(B)[n] - zb*rowsum(A)[m] + K*za*zb
// with the sums taken from the pre-pass.
//
// Because nothing is converted here, the main loop is TMA -> shared memory ->
// tensor core: per 64-deep K stage each SM receives 32 KB by TMA and its MMA
// reads 32 KB, and no thread touches operand bytes.
//
// Cluster of 2 CTAs (256 x 256 pair tile; each CTA: 128 rows of A, 128
// columns of B, its 128 x 256 accumulator in its own TMEM), 320 threads:
//  * warp 9 (producer): TMA copies of this CTA's fp16 A rows (box 64 x 128,
//    128-byte swizzle: the K-major MMA layout) and B columns (two boxes of
//    64 k x 64 n: the MN-major layout) into a 6-stage ring. Both CTAs' copies
//    complete on the even CTA's `full` barrier (cta_group::2 form).
//  * warp 8: TMEM allocation for the pair; in the even CTA one lane issues
//    the pair MMAs (M=256, N=256, K=16) and commits to both CTAs' barriers.
//  * warps 0-7: drain each K-chunk's fp32 accumulator into int32 running sums
//    held in registers (each thread: one row, 128 columns), then run the
//    epilogue from those registers.
// TMEM holds two fp32 accumulators (columns [0,256) and [256,512)); K-chunks
// alternate between them, so the tensor core fills one while the other is
// drained and never waits for a drain or an epilogue.
// Every wait is bounded (see common.cuh).
#include "common.cuh"
#include "kernels.h"
#include "tma.h"

#include <algorithm>
#include <mutex>

namespace qmm {
namespace gemmf {

// Pair tile: 256 rows x BN columns, BN = 256 or 224 (192 too for the
// convolution; a template parameter, chosen per problem by the launcher to
// fill the last wave of tiles). Each CTA stages two 64-column B boxes (128
// columns) and the MMA reads BN/2; the convolution's im2col copy delivers
// exactly BN/2 pixel rows.
constexpr int BM = 128;
constexpr int BMP = 2 * BM;
constexpr int BN_MAX = 256;
constexpr int BK = 64;
constexpr int NS = 6;                   // stages in the ring (5 with the TMA-store epilogue)
constexpr int STG_BYTES = 2 * 32 * 64;  // per drain warp: two 32-row x 64-byte C staging buffers
constexpr int STG_TOTAL = 8 * STG_BYTES;
constexpr int NEW = 8;                  // drain / epilogue warps
constexpr int NT = NEW * 32 + 64;       // + MMA warp + producer warp
constexpr int CPW_MAX = BN_MAX / 2;     // accumulator columns per drain warp (two warps per TMEM lane quarter)
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BYTES = BK * 128 * 2;   // two 64-column boxes: 16 KB
constexpr int B_BOX = 64 * BK * 2;      // one 64-column B box: 8 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;     // one accumulator buffer
constexpr int PAIR_ARRIVALS = 2 * NEW;

struct Shared {
  uint64_t full[NS];      // even CTA: one arrival (expect_tx) + both CTAs' copy bytes
  uint64_t empty[NS];     // the pair's commit
  uint64_t acc_full[2];   // per accumulator buffer: the pair's commit
  uint64_t acc_empty[2];  // even CTA: one arrival per drain warp of both CTAs
  uint64_t teardown;
  uint64_t accld[NEW][2];   // accumulating A8W8: per drain warp, its two acc_in staging buffers
  uint32_t tmem_base;
  int abort_flag;
  // per drain warp, the current tile's operands of its CPW columns:
  // A8W8 weight_scale (float bits) / MatMulInteger b_zp, and colsum(B)
  uint32_t col_op[NEW][CPW_MAX];
  int col_sum[NEW][CPW_MAX];
  // MatMulInteger with dequantisation: the per-column multiplier and bias
  float col_scale[NEW][CPW_MAX];
  float col_bias[NEW][CPW_MAX];
};

// Ring stages of an instantiation: the MatMulInteger ones (4-byte outputs) and
// the accumulating A8W8 one give one stage to per-warp staging buffers (C for
// the TMA-store epilogue, acc_in for the accumulator's TMA loads).
template <bool TS>
__host__ __device__ constexpr int ring_stages() { return TS ? NS - 1 : NS; }
template <bool TS>
constexpr size_t smem_bytes() {
  return (size_t)ring_stages<TS>() * STAGE_BYTES + (TS ? STG_TOTAL : 0) + sizeof(Shared) + 1024;
}
static_assert(smem_bytes<false>() <= 232448 && smem_bytes<true>() <= 232448, "shared memory per CTA");

enum : unsigned {
  SITE_EMPTY = 0x400, SITE_FULL = 0x401, SITE_ACC_FULL = 0x402, SITE_ACC_EMPTY = 0x403, SITE_TEARDOWN = 0x404,
  SITE_FINAL = 0x405, SITE_ACCLD = 0x407
};

struct TileCoord {
  int b, m0, n0;   // m0: this CTA's first row; n0: the pair tile's first column
};

template <int BN>
__device__ __forceinline__ TileCoord tile_coord(const GemmF16Args& p, int tile_local, int cid, int ncl, int rank) {
  const int m_tiles = (p.M + BMP - 1) / BMP;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tile_id = cid + tile_local * ncl;
  const int per_batch = m_tiles * n_tiles;
  TileCoord c;
  c.b = tile_id / per_batch;
  const int r = tile_id - c.b * per_batch;
  const int mt = r / n_tiles;
  c.m0 = mt * BMP + rank * BM;
  c.n0 = (r - mt * n_tiles) * BN;
  return c;
}

// TMA copy completing on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
      : "memory");
}

// Im2col tensor copy (rank 4, {C, W, H, N}) completing on an mbarrier of
// either CTA of the pair: the pixels from base (w, h) of image n onwards, each
// shifted by the tap offsets (ow, oh), channels [c, c + box).
__device__ __forceinline__ void tma_im2col_4d_pair(uint32_t dst, const void* tmap, int c, int w, int h, int n,
                                                   uint16_t ow, uint16_t oh, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.im2col.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6], {%7, %8};" ::"r"(dst),
      "l"(tmap), "r"(c), "r"(w), "r"(h), "r"(n), "r"(bar_cluster), "h"(ow), "h"(oh)
      : "memory");
}

// Per-tile operands of this warp's CPW columns, staged in shared memory by
// the warp itself.
template <int CPW, bool BU, bool MMI, bool FA, bool ACC = false, bool DQ = false>
__device__ __forceinline__ void stage_columns(const GemmF16Args& p, Shared& sm, const TileCoord tc, int warp, int h,
                                              int lane) {
  const int* colsum = (MMI && p.a_zp_count > 0) ? p.colsum + (p.b_bstride ? (size_t)tc.b * p.N : 0) : nullptr;
  const float ys = DQ ? __ldg(p.act_scale) : 0.f;
  for (int col = lane; col < CPW; col += 32) {
    const int n = tc.n0 + h * CPW + col;
    uint32_t op = 0u;
    int cs = 0;
    if (n < p.N) {
      if (FA) {
        op = __float_as_uint(__ldg(p.w_scale + (p.w_count == 1 ? 0 : n)));
        if (p.b_zp_count > 0) cs = __ldg((const int*)p.b_zp + (p.b_zp_count == 1 ? 0 : n));
      } else if (!MMI) {
        if (!ACC || p.C) op = __float_as_uint(__ldg(p.w_scale + (p.w_count == 1 ? 0 : n)));
      } else {
        if (p.b_zp_count > 0) {
          const int zi = p.b_zp_count == 1 ? 0 : n;
          op = BU ? (uint32_t)__ldg((const uint8_t*)p.b_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.b_zp + zi);
        }
        if (colsum) cs = __ldg(colsum + n);
      }
    }
    sm.col_op[warp][col] = op;
    sm.col_sum[warp][col] = cs;
    if (DQ) {
      sm.col_scale[warp][col] = n < p.N ? __fmul_rn(ys, __ldg(p.w_scale + (p.w_count == 1 ? 0 : n))) : 0.f;
      sm.col_bias[warp][col] = (n < p.N && p.bias) ? __ldg(p.bias + n) : 0.f;
    }
  }
  __syncwarp();
}

// Epilogue of one tile from the int32 sums in registers (this thread: one row,
// this warp's CPW columns): dequantise (A8W8; with ACC, first add acc_in and
// store the combined int32 sums to acc_out) or apply the zero-point expansion
// (MatMulInteger), store C. c_vec bit 0: C rows take 16-byte vectors; bit 1:
// so do acc_in / acc_out rows.
template <int CPW, bool AU, bool BU, bool MMI, bool FA, bool ACC = false, bool DQ = false>
__device__ __forceinline__ void epilogue(const GemmF16Args& p, const Shared& sm, uint32_t (&sums)[CPW],
                                         const TileCoord tc, int warp, int q, int h, int lane, int c_vec) {
  const int row = tc.m0 + q * 32 + lane;
  if (row >= p.M) return;
  const size_t crow = ((size_t)tc.b * p.M + (size_t)row) * (size_t)p.N;
  const uint64_t pol = l2_policy_evict_first();
  const int ag = p.a_bmod ? tc.b % p.a_bmod : 0;   // weight slice of a grouped batch
  const int mz = ag * p.M + row % p.zp_row_mod;
  float as = 0.f;
  uint32_t za = 0u, rs = 0u;
  if (FA) {
    // form (a): scale_n * (sum_k a*w - zp_n * sum_k a), in fp32
    const float rsum = p.b_zp_count > 0 ? __ldg(reinterpret_cast<const float*>(p.rowsum) + row) : 0.f;
#pragma unroll
    for (int g = 0; g < CPW / 16; ++g) {
      const int nb = tc.n0 + h * CPW + g * 16;
      if (nb >= p.N) break;
      const bool full = (nb + 16 <= p.N) && (c_vec & 1);
      uint32_t* o = &sums[g * 16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float zp = (float)sm.col_sum[warp][g * 16 + i];
        const float v = __fmaf_rn(-zp, rsum, __uint_as_float(o[i]));
        o[i] = __float_as_uint(__fmul_rn(v, __uint_as_float(sm.col_op[warp][g * 16 + i])));
      }
      if (p.c_f32) {
        float* out = reinterpret_cast<float*>(p.C) + crow + nb;
        if (full) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) st_global_v4_hint(out + i, o[i], o[i + 1], o[i + 2], o[i + 3], pol);
        } else {
          for (int i = 0; i < 16; ++i)
            if (nb + i < p.N) out[i] = __uint_as_float(o[i]);
        }
      } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + crow + nb;
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
          pk[i] = *reinterpret_cast<uint32_t*>(&b2);
        }
        if (full) {
          st_global_v4_hint(out, pk[0], pk[1], pk[2], pk[3], pol);
          st_global_v4_hint(out + 8, pk[4], pk[5], pk[6], pk[7], pol);
        } else {
          for (int i = 0; i < 16; ++i)
            if (nb + i < p.N) out[i] = __float2bfloat16_rn(__uint_as_float(o[i]));
        }
      }
    }
    return;
  }
  if (!MMI) {
    if (!ACC || p.C) as = __ldg(p.act_scale + (p.act_count == 1 ? 0 : mz));
  } else {
    if (p.a_zp_count > 0) {
      const int zi = p.a_zp_count == 1 ? 0 : mz;
      za = AU ? (uint32_t)__ldg((const uint8_t*)p.a_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.a_zp + zi);
    }
    if (p.b_zp_count > 0)
      rs = (uint32_t)__ldg(p.rowsum + (size_t)(p.a_bstride ? (p.a_bmod ? ag : tc.b) : 0) * p.M + row);
  }
  const uint32_t kzz = (uint32_t)p.K * za;
#pragma unroll
  for (int g = 0; g < CPW / 16; ++g) {
    const int nb = tc.n0 + h * CPW + g * 16;
    if (nb >= p.N) break;
    const bool full = (nb + 16 <= p.N) && (c_vec & 1);
    uint32_t* o = &sums[g * 16];
    if (ACC) {   // the sums already hold acc_in (loaded before the tile's first chunk)
      const bool full_acc = (nb + 16 <= p.N) && (c_vec & 2);
      if (p.acc_out) {
        int* dst = p.acc_out + crow + nb;
        if (full_acc) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) st_global_v4_hint(dst + i, o[i], o[i + 1], o[i + 2], o[i + 3], pol);
        } else {
          for (int i = 0; i < 16; ++i)
            if (nb + i < p.N) dst[i] = (int)o[i];
        }
      }
      if (!p.C) continue;
    }
    if (!MMI) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float v = __int2float_rn((int)o[i]);
        v = __fmul_rn(v, as);
        o[i] = __float_as_uint(__fmul_rn(v, __uint_as_float(sm.col_op[warp][g * 16 + i])));
      }
      if (p.c_f32) {
        float* out = reinterpret_cast<float*>(p.C) + crow + nb;
        if (full) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) st_global_v4_hint(out + i, o[i], o[i + 1], o[i + 2], o[i + 3], pol);
        } else {
          for (int i = 0; i < 16; ++i)
            if (nb + i < p.N) out[i] = __uint_as_float(o[i]);
        }
      } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + crow + nb;
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
          pk[i] = *reinterpret_cast<uint32_t*>(&b2);
        }
        if (full) {
          st_global_v4_hint(out, pk[0], pk[1], pk[2], pk[3], pol);
          st_global_v4_hint(out + 8, pk[4], pk[5], pk[6], pk[7], pol);
        } else {
          for (int i = 0; i < 16; ++i)
            if (nb + i < p.N) out[i] = __float2bfloat16_rn(__uint_as_float(o[i]));
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t zb = sm.col_op[warp][g * 16 + i];
        const uint32_t cs = (uint32_t)sm.col_sum[warp][g * 16 + i];
        o[i] = o[i] - za * cs - zb * rs + kzz * zb;
        if (DQ) {   // cast, one multiply by y_scale * w_scale[n], then the bias
          float v = __fmul_rn(__int2float_rn((int)o[i]), sm.col_scale[warp][g * 16 + i]);
          if (p.bias) v = __fadd_rn(v, sm.col_bias[warp][g * 16 + i]);
          o[i] = __float_as_uint(v);
        }
      }
      int32_t* out = reinterpret_cast<int32_t*>(p.C) + crow + nb;
      if (full) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) st_global_v4_hint(out + i, o[i], o[i + 1], o[i + 2], o[i + 3], pol);
      } else {
        for (int i = 0; i < 16; ++i)
          if (nb + i < p.N) out[i] = (int)o[i];
      }
    }
  }
}

// MatMulInteger epilogue (int32 out, or fp32 with the dequantising step)
// through TMA stores: per 16-column group the warp's 32 rows x 64 bytes go to
// one of its two staging buffers (64-byte swizzle: chunk j of row r at chunk
// j ^ ((r >> 1) & 3), conflict-free), and one lane stores the box; rows and
// columns outside C are not written. nst counts this warp's stores.
template <int CPW, bool AU, bool BU, bool DQ>
__device__ __forceinline__ void epilogue_tma(const GemmF16Args& p, const Shared& sm, uint32_t (&sums)[CPW],
                                             const TileCoord tc, int warp, int q, int h, int lane, uint32_t stg,
                                             const CUtensorMap* tmC, int& nst) {
  const int row0 = tc.m0 + q * 32;
  if (row0 >= p.M) return;
  const int row = row0 + lane;
  const bool rv = row < p.M;
  const int ag = p.a_bmod ? tc.b % p.a_bmod : 0;
  uint32_t za = 0u, rs = 0u;
  if (rv && p.a_zp_count > 0) {
    const int zi = p.a_zp_count == 1 ? 0 : ag * p.M + row % p.zp_row_mod;
    za = AU ? (uint32_t)__ldg((const uint8_t*)p.a_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.a_zp + zi);
  }
  if (rv && p.b_zp_count > 0)
    rs = (uint32_t)__ldg(p.rowsum + (size_t)(p.a_bstride ? (p.a_bmod ? ag : tc.b) : 0) * p.M + row);
  const uint32_t kzz = (uint32_t)p.K * za;
  const uint32_t swz = (uint32_t)((lane >> 1) & 3);
#pragma unroll
  for (int g = 0; g < CPW / 16; ++g) {
    const int nb = tc.n0 + h * CPW + g * 16;
    if (nb >= p.N) break;
    uint32_t* o = &sums[g * 16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t zb = sm.col_op[warp][g * 16 + i];
      const uint32_t cs = (uint32_t)sm.col_sum[warp][g * 16 + i];
      o[i] = o[i] - za * cs - zb * rs + kzz * zb;
      if (DQ) {   // cast, one multiply by y_scale * w_scale[n], then the bias
        float v = __fmul_rn(__int2float_rn((int)o[i]), sm.col_scale[warp][g * 16 + i]);
        if (p.bias) v = __fadd_rn(v, sm.col_bias[warp][g * 16 + i]);
        o[i] = __float_as_uint(v);
      }
    }
    const int buf = nst & 1;
    if (nst >= 2) {   // the store that used this buffer has read it
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
    const uint32_t b = stg + (uint32_t)buf * (32 * 64);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st_shared_v4(b + (uint32_t)lane * 64u + ((uint32_t)j ^ swz) * 16u, o[4 * j], o[4 * j + 1], o[4 * j + 2],
                   o[4 * j + 3]);
    fence_proxy_async_smem();   // the generic-proxy writes, visible to the copy engine
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmC, b, nb, row0, tc.b);
      bulk_commit();
    }
    ++nst;
  }
}

// Accumulating A8W8 epilogue with acc_in arriving by TMA: per 16-column group
// one lane copies the warp's 32 rows x 16 int32 of acc_in into a staging
// buffer (64-byte swizzle, two buffers, the next group's copy in flight while
// this one is used), every lane adds its row's 16 values to its sums, then
// acc_out (optional) and the scaled C are stored as in the plain epilogue.
// Coalesced box copies replace 28 per-lane 16-byte loads of separate rows,
// which filled the load queue and held up the drains. nacc counts this warp's
// copies (buffer = count & 1, phase parity = (count >> 1) & 1).
template <int CPW>
__device__ __forceinline__ void epilogue_acc_tma(const GemmF16Args& p, Shared& sm, uint32_t (&sums)[CPW],
                                                 const TileCoord tc, int warp, int q, int h, int lane, int c_vec,
                                                 uint32_t stg, const CUtensorMap* tm_acc, int& nacc) {
  const int row0 = tc.m0 + q * 32;
  if (row0 >= p.M) return;   // warp-uniform
  const int row = row0 + lane;
  const bool rv = row < p.M;
  const size_t crow = ((size_t)tc.b * p.M + (size_t)(rv ? row : 0)) * (size_t)p.N;
  const uint64_t pol = l2_policy_evict_first();
  const float as = (p.C && rv) ? __ldg(p.act_scale + (p.act_count == 1 ? 0 : row % p.zp_row_mod)) : 0.f;
  const int n_first = tc.n0 + h * CPW;
  const int ng = p.N > n_first ? min(CPW / 16, (p.N - n_first + 15) / 16) : 0;
  auto issue = [&](int gi) {
    if (lane == 0) {
      const int k = nacc + gi, buf = k & 1;
      mbar_arrive_expect_tx(&sm.accld[warp][buf], 32u * 16u * 4u);
      tma_load_3d(stg + (uint32_t)buf * 2048u, tm_acc, n_first + 16 * gi, row0, tc.b, &sm.accld[warp][buf]);
    }
  };
  if (ng > 0) issue(0);
  if (ng > 1) issue(1);
  const uint32_t swz = (uint32_t)((lane >> 1) & 3);
#pragma unroll
  for (int g = 0; g < CPW / 16; ++g) {
    if (g >= ng) break;
    const int nb = n_first + g * 16;
    const int k = nacc + g, buf = k & 1;
    uint32_t* o = &sums[g * 16];
    if (mbar_wait(&sm.accld[warp][buf], (uint32_t)((k >> 1) & 1), &sm.abort_flag, p.err, SITE_ACCLD)) {
      const uint32_t b = stg + (uint32_t)buf * 2048u + (uint32_t)lane * 64u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 x = ld_shared_v4(b + (((uint32_t)j ^ swz) << 4));
        o[4 * j] += x.x;
        o[4 * j + 1] += x.y;
        o[4 * j + 2] += x.z;
        o[4 * j + 3] += x.w;
      }
    }
    fence_proxy_async_smem();   // this buffer's reads are done before the next copy overwrites it
    __syncwarp();
    if (g + 2 < ng) issue(g + 2);
    if (!rv) continue;
    const bool full_acc = (nb + 16 <= p.N) && (c_vec & 2);
    if (p.acc_out) {
      int* dst = p.acc_out + crow + nb;
      if (full_acc) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) st_global_v4_hint(dst + i, o[i], o[i + 1], o[i + 2], o[i + 3], pol);
      } else {
        for (int i = 0; i < 16; ++i)
          if (nb + i < p.N) dst[i] = (int)o[i];
      }
    }
    if (!p.C) continue;
    const bool full = (nb + 16 <= p.N) && (c_vec & 1);
    float f[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      f[i] = __fmul_rn(__fmul_rn(__int2float_rn((int)o[i]), as), __uint_as_float(sm.col_op[warp][g * 16 + i]));
    if (p.c_f32) {
      float* out = reinterpret_cast<float*>(p.C) + crow + nb;
      if (full) {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          st_global_v4_hint(out + i, __float_as_uint(f[i]), __float_as_uint(f[i + 1]), __float_as_uint(f[i + 2]),
                            __float_as_uint(f[i + 3]), pol);
      } else {
        for (int i = 0; i < 16; ++i)
          if (nb + i < p.N) out[i] = f[i];
      }
    } else {
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + crow + nb;
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        pk[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      if (full) {
        st_global_v4_hint(out, pk[0], pk[1], pk[2], pk[3], pol);
        st_global_v4_hint(out + 8, pk[4], pk[5], pk[6], pk[7], pol);
      } else {
        for (int i = 0; i < 16; ++i)
          if (nb + i < p.N) out[i] = __float2bfloat16_rn(f[i]);
      }
    }
  }
  nacc += ng;
}

// Accumulating A8W8: start this thread's running sums (one row, CPW columns)
// from the caller's int32 accumulator (0 outside the problem). Issued before
// the wait for the tile's first chunk, so the loads overlap the MMAs.
template <int CPW>
__device__ __forceinline__ void preload_acc(const GemmF16Args& p, const TileCoord tc, int q, int h, int lane,
                                            uint32_t (&sums)[CPW], int c_vec) {
  const int row = tc.m0 + q * 32 + lane;
  const bool rv = p.acc_in && row < p.M;
  const int* src = rv ? p.acc_in + ((size_t)tc.b * p.M + (size_t)row) * (size_t)p.N : nullptr;
  const uint64_t pol = l2_policy_evict_first();   // read once: keep the operand tiles in L2
#pragma unroll
  for (int g = 0; g < CPW / 16; ++g) {
    const int nb = tc.n0 + h * CPW + g * 16;
    if (rv && nb + 16 <= p.N && (c_vec & 2)) {
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const uint4 x = ldg_nc_v4_hint(src + nb + i, pol);
        sums[g * 16 + i] = x.x;
        sums[g * 16 + i + 1] = x.y;
        sums[g * 16 + i + 2] = x.z;
        sums[g * 16 + i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) sums[g * 16 + i] = (rv && nb + i < p.N) ? (uint32_t)__ldg(src + nb + i) : 0u;
    }
  }
}

template <int BN, bool AU, bool BU, bool MMI, bool FA, bool ACC, bool DQ, bool CV>
__global__ void __launch_bounds__(NT, 1)
    gemm_f16pair_kernel(const GemmF16Args p, const int cs, const int c_vec, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC) {
  constexpr bool TS = MMI;                 // 4-byte outputs leave through the TMA-store epilogue
  constexpr bool STG = MMI || ACC;         // per-warp staging buffers (C out, or acc_in in)
  constexpr int kNS = ring_stages<STG>();
  constexpr int BNH = BN / 2;   // B columns of each CTA
  constexpr int CPW = BN / 2;   // accumulator columns per drain warp
  static_assert(BN % 32 == 0 && BN <= BN_MAX && BNH <= 128, "pair tile width");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sbase_ptr = smem_raw + (sbase - raw);
  const uint32_t stg_base = sbase + (uint32_t)(kNS * STAGE_BYTES);   // C staging (TS), 1024-byte aligned
  Shared& sm = *reinterpret_cast<Shared*>(sbase_ptr + kNS * STAGE_BYTES + (STG ? STG_TOTAL : 0));

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x();
  const int ncl = (int)nclusters_x();

  const int m_tiles = (p.M + BMP - 1) / BMP;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int num_tiles = p.batch * m_tiles * n_tiles;
  const int my_tiles = (cid < num_tiles) ? (num_tiles - cid + ncl - 1) / ncl : 0;
  const int spt = (p.K + BK - 1) / BK;
  const int cpt = (spt + cs - 1) / cs;
  const int total_stages = my_tiles * spt;
  const int total_chunks = my_tiles * cpt;

  if (t == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], PAIR_ARRIVALS);
    }
    mbar_init(&sm.teardown, 1);
    for (int i = 0; i < NEW; ++i) {
      mbar_init(&sm.accld[i][0], 1);
      mbar_init(&sm.accld[i][1], 1);
    }
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == NEW) {
    tmem_alloc_pair(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  // wait limits: the MMA thread's, and every other role's (longer under the
  // stall test, so that the MMA thread's wait is the one that runs out first)
  const uint64_t lim = p.wait_ns ? p.wait_ns : kWaitLimitNs;
  const uint64_t lim2 = p.stall_test ? 4 * lim : lim;
  // launched as a programmatic dependent of the pre-pass: everything above ran
  // while it finished; nothing below reads its output before it completes
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == NEW) {
    // ---------------- pair MMA issuer (even CTA) ----------------
    if (rank == 0 && lane == 0) {
      // B is MN-major (64-column boxes of [K][N] rows) except for the implicit
      // convolution, whose im2col copies deliver pixel rows of 64 channels (K-major)
      const uint32_t idesc = FA ? idesc_bf16_f32(BMP, BN, false, true) : idesc_f16_f32(BMP, BN, false, !CV);
      int g = 0, d = 0;
      bool ok = true;
      for (int tl = 0; tl < my_tiles && ok; ++tl) {
        for (int c = 0; c < cpt && ok; ++c) {
          const int ab = d & 1;   // accumulator buffer of this chunk
          if (d >= 2) {
            ok = mbar_wait_cluster(&sm.acc_empty[ab], (uint32_t)(((d >> 1) - 1) & 1), &sm.abort_flag, p.err,
                                   SITE_ACC_EMPTY, lim);
            if (!ok) break;
          }
          tc_fence_after();
          const uint32_t tacc = tbase + (uint32_t)ab * ACC_COLS;
          const int s_beg = c * cs;
          const int s_end = min(spt, s_beg + cs);
          for (int s = s_beg; s < s_end; ++s, ++g) {
            const int slot = g % kNS;
            ok = mbar_wait_cluster(&sm.full[slot], (uint32_t)((g / kNS) & 1), &sm.abort_flag, p.err, SITE_FULL,
                                   lim);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_addr = sbase + (uint32_t)slot * STAGE_BYTES;
            const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              const uint64_t ad = sdesc_sw128(a_addr + (uint32_t)j * 32u, 16u, 1024u);
              // B: 64-column boxes 8 KB apart (LBO), 8-row k groups 1 KB apart (SBO)
              const uint64_t bd = CV ? sdesc_sw128(b_addr + (uint32_t)j * 32u, 16u, 1024u)
                                     : sdesc_sw128(b_addr + (uint32_t)j * 2048u, (uint32_t)B_BOX, 1024u);
              tc_mma_f16_pair(tacc, ad, bd, idesc, (s > s_beg || j > 0) ? 1u : 0u);
            }
            tc_commit_pair_mc(&sm.empty[slot], 0x3);
          }
          if (!ok) break;
          tc_commit_pair_mc(&sm.acc_full[ab], 0x3);
          ++d;
        }
      }
    }
    __syncwarp();
  } else if (warp == NEW + 1) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      const uint32_t full_leader0 = mapa_shared(smem_u32(&sm.full[0]), 0);
      int tl = 0, s = 0;
      TileCoord tc = tile_coord<BN>(p, 0, cid, ncl, (int)rank);
      int g = 0;
      for (; g < total_stages; ++g) {
        const int slot = g % kNS;
        if (g >= kNS &&
            !mbar_wait(&sm.empty[slot], (uint32_t)(((g / kNS) - 1) & 1), &sm.abort_flag, p.err, SITE_EMPTY, lim2))
          break;
        if (p.stall_test && cid == 0 && g == 0) {   // test hook: this stage never fills
          if (++s == spt) {
            s = 0;
            tc = tile_coord<BN>(p, ++tl, cid, ncl, (int)rank);
          }
          continue;
        }
        const uint32_t bar = full_leader0 + (uint32_t)slot * 8u;
        // the convolution's B box is BNH pixel rows of 128 bytes (the other
        // instantiations always fill both 64-column boxes)
        if (rank == 0) mbar_arrive_expect_tx(&sm.full[slot], 2u * (CV ? (uint32_t)(A_BYTES + 128 * BNH) : STAGE_BYTES));
        const uint32_t dst = sbase + (uint32_t)slot * STAGE_BYTES;
        const int ab = p.a_bstride ? (p.a_bmod ? tc.b % p.a_bmod : tc.b) : 0, bb = p.b_bstride ? tc.b : 0;
        const int nc = tc.n0 + (int)rank * BNH;
        tma_load_3d_pair(dst, &tmA, s * BK, tc.m0, ab, bar);
        if (CV) {
          // K stage s: tap (r, sx) and 64-channel block cb of the group; the
          // CTA's 128 pixels start at output pixel nc of image b / G (a start
          // past the image's last pixel loads pixels that are never stored)
          const int tap = s / p.cv_cb, cb = s - tap * p.cv_cb;
          const int r = tap / p.cv_kW, sx = tap - r * p.cv_kW;
          const int img = tc.b / p.cv_G, grp = tc.b - img * p.cv_G;
          const int px = nc < p.N ? nc : 0;
          const int oh = px / p.cv_oW, ow = px - oh * p.cv_oW;
          tma_im2col_4d_pair(dst + A_BYTES, &tmB, grp * p.cv_Cg + cb * 64, ow * p.cv_sw - p.cv_pl,
                             oh * p.cv_sh - p.cv_pt, img, (uint16_t)(sx * p.cv_dw), (uint16_t)(r * p.cv_dh), bar);
        } else {
          const int kb = (FA && p.fa_kwrap) ? (s * BK) % p.fa_kwrap : s * BK;   // [hi | lo] halves reread W
          tma_load_3d_pair(dst + A_BYTES, &tmB, nc, kb, bb, bar);
          tma_load_3d_pair(dst + A_BYTES + B_BOX, &tmB, nc + 64, kb, bb, bar);
        }
        if (++s == spt) {
          s = 0;
          tc = tile_coord<BN>(p, ++tl, cid, ncl, (int)rank);
        }
      }
      // The even CTA's `full` barriers count both CTAs' bytes: once the phases
      // of the last stages complete, no copy of either CTA is in flight.
      if (rank == 0)
        for (int j = (g > kNS ? g - kNS : 0); j < g; ++j)
          mbar_wait_cluster(&sm.full[j % kNS], (uint32_t)((j / kNS) & 1), nullptr, p.err, SITE_FINAL, lim2);
    }
    __syncwarp();
  } else {
    // ---------------- drain / epilogue warps ----------------
    const int q = warp & 3;
    const int h = warp >> 2;
    const uint32_t acc_empty_leader0 = mapa_shared(smem_u32(&sm.acc_empty[0]), 0);
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    uint32_t sums[CPW];
    int nst = 0;    // TMA stores this warp has issued
    int nacc = 0;   // acc_in copies this warp has issued
    int tl = 0, c = 0;
    TileCoord tc = tile_coord<BN>(p, 0, cid, ncl, (int)rank);
    if (my_tiles > 0) stage_columns<CPW, BU, MMI, FA, ACC, DQ>(p, sm, tc, warp, h, lane);
    for (int d = 0; d < total_chunks; ++d) {
      const int ab = d & 1;
      // acc_in joins the sums before the first chunk, or in the epilogue by TMA (c_vec bit 2)
      if (ACC && c == 0 && !(c_vec & 4)) preload_acc<CPW>(p, tc, q, h, lane, sums, c_vec);
      if (!mbar_wait_cluster(&sm.acc_full[ab], (uint32_t)((d >> 1) & 1), &sm.abort_flag, p.err, SITE_ACC_FULL,
                             lim2))
        break;
      tc_fence_after();
      const uint32_t t_acc = tbase + lane_off + (uint32_t)ab * ACC_COLS + (uint32_t)(h * CPW);
      // exact fp32 chunk sums -> int32, into the running sums (wrapping)
#pragma unroll
      for (int g = 0; g < CPW / 16; ++g) {
        uint32_t acc[16];
        tmem_ld16(t_acc + g * 16, acc);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (FA) {   // form (a): one fp32 accumulation over all of K; the launcher makes it one chunk
            sums[g * 16 + i] = acc[i];
          } else {
            const uint32_t v = (uint32_t)__float2int_rn(__uint_as_float(acc[i]));
            sums[g * 16 + i] = (c == 0 && (!ACC || (c_vec & 4))) ? v : sums[g * 16 + i] + v;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote_cta(acc_empty_leader0 + (uint32_t)ab * 8u);
      if (c == cpt - 1) {
        if (TS && (c_vec & 1))
          epilogue_tma<CPW, AU, BU, DQ>(p, sm, sums, tc, warp, q, h, lane, stg_base + (uint32_t)warp * STG_BYTES,
                                        &tmC, nst);
        else if (ACC && (c_vec & 4))
          epilogue_acc_tma<CPW>(p, sm, sums, tc, warp, q, h, lane, c_vec, stg_base + (uint32_t)warp * STG_BYTES,
                                &tmC, nacc);
        else
          epilogue<CPW, AU, BU, MMI, FA, ACC, DQ>(p, sm, sums, tc, warp, q, h, lane, c_vec);
        __syncwarp();   // the warp's staged operands are read: restage for the next tile
        if (tl + 1 < my_tiles)
          stage_columns<CPW, BU, MMI, FA, ACC, DQ>(p, sm, tile_coord<BN>(p, tl + 1, cid, ncl, (int)rank), warp,
                                                   h, lane);
      }
      if (++c == cpt) {
        c = 0;
        ++tl;
        tc = tile_coord<BN>(p, tl, cid, ncl, (int)rank);
      }
    }
    if (TS && lane == 0 && nst > 0) bulk_wait_all();   // this warp's stores are complete
    tc_fence_before();
  }

  __syncthreads();
  if (t == 0 && sm.abort_flag)
    st_shared_cluster_u32(mapa_shared(smem_u32(&sm.abort_flag), rank ^ 1u), 1u);
  if (warp == NEW && rank == 0) {
    tc_fence_after();
    if (lane == 0) {
      tc_commit_pair_mc(&sm.teardown, 0x1);
      mbar_wait(&sm.teardown, 0u, nullptr, p.err, SITE_TEARDOWN, lim2);
    }
    __syncwarp();
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == NEW) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, TMEM_COLS);
  }
}

struct DeviceLaunchInfo {
  bool attr_set = false;
  int max_clusters = 0;
};

template <int BN, bool AU, bool BU, bool MMI, bool FA = false, bool ACC = false, bool DQ = false, bool CV = false>
cudaError_t launch_one(const GemmF16Args& a, int cs, int c_vec, const CUtensorMap& ta, const CUtensorMap& tb,
                       const CUtensorMap& tc, cudaStream_t s) {
  constexpr size_t SMEM_BYTES = smem_bytes<MMI || ACC>();
  auto kern = gemm_f16pair_kernel<BN, AU, BU, MMI, FA, ACC, DQ, CV>;
  static std::mutex mu;
  static DeviceLaunchInfo info[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the pre-pass's tail
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!info[dev].attr_set) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(2 * 64, 1, 1);
      e = cudaOccupancyMaxActiveClusters(&info[dev].max_clusters, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (info[dev].max_clusters < 1) return cudaErrorInvalidConfiguration;
      info[dev].attr_set = true;
    }
    max_clusters = info[dev].max_clusters;
  }
  const int m_tiles = (a.M + BMP - 1) / BMP;
  const int n_tiles = (a.N + BN - 1) / BN;
  const long long tiles = (long long)a.batch * m_tiles * n_tiles;
  const int ncl = (int)std::min<long long>(tiles, (long long)max_clusters);
  cfg.gridDim = dim3(2 * ncl, 1, 1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, cs, c_vec, ta, tb, tc);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// fp16 operand maps: A as {K, M, batch} (box 64 x 128), B as {N, K, batch}
// (box 64 x 64), both with 128-byte swizzle; rows a_pitch / b_pitch elements
// apart (the columns past K or N are never read: the copies there are zeros).
cudaError_t make_maps(const GemmF16Args& a, CUtensorMap* ta, CUtensorMap* tb) {
  const uint64_t ab = a.a_bstride ? (uint64_t)(a.a_bmod ? a.a_bmod : a.batch) : 1;
  const uint64_t bb = a.b_bstride ? (uint64_t)a.batch : 1;
  const uint64_t ap = a.a_pitch ? (uint64_t)a.a_pitch : (uint64_t)a.K;
  const uint64_t bp = a.b_pitch ? (uint64_t)a.b_pitch : (uint64_t)a.N;
  const uint64_t as = 2ull * (a.a_bstride ? (uint64_t)a.a_bstride : (uint64_t)a.M * ap);
  const uint64_t bs = 2ull * (a.b_bstride ? (uint64_t)a.b_bstride : (uint64_t)a.K * bp);
  cudaError_t e = make_tmap_3d(ta, a.A16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)a.K, (uint64_t)a.M, ab, 2ull * ap,
                               as, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  return make_tmap_3d(tb, a.B16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)a.N, (uint64_t)a.K, bb, 2ull * bp, bs,
                      64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
}


// Pair-tile width: the one whose tiles fill the last wave best. The cost of a
// width is its number of waves (tiles over the pairs that run at once) times
// the tile width plus a fixed per-tile overhead (about 16 columns' worth of
// MMA time: pipeline fill, the last drain and epilogue).
int choose_tile_width(const GemmF16Args& a) {
  const long long clusters = std::max(1, num_sms() / 2);
  const long long m_tiles = (a.M + BMP - 1) / BMP;
  int best = 256;
  long long best_cost = -1;
  for (int bn : {256, 224}) {
    const long long tiles = (long long)a.batch * m_tiles * ((a.N + bn - 1) / bn);
    const long long waves = (tiles + clusters - 1) / clusters;
    const long long cost = waves * (bn + 16);
    if (best_cost < 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

template <int BN>
cudaError_t dispatch(const GemmF16Args& a, bool a_u8, bool b_u8, bool mmi, int cs, int c_vec, const CUtensorMap& ta,
                     const CUtensorMap& tb, const CUtensorMap& tc, cudaStream_t s) {
  if (!mmi) {
    // the accumulator epilogue's extra loads fit the register budget at the
    // 224-column width only (the 256-column one spills)
    if (a.acc_in || a.acc_out || !a.C) return launch_one<224, false, false, false, false, true>(a, cs, c_vec, ta, tb, tc, s);
    return launch_one<BN, false, false, false>(a, cs, c_vec, ta, tb, tc, s);
  }
  if (a.act_scale) {   // dequantising MatMulInteger: A is the quantised activation (uint8); 224 columns
    if (!a_u8) return cudaErrorInvalidValue;   // fit the extra epilogue operands without spilling
    if (b_u8) return launch_one<224, true, true, true, false, false, true>(a, cs, c_vec, ta, tb, tc, s);
    return launch_one<224, true, false, true, false, false, true>(a, cs, c_vec, ta, tb, tc, s);
  }
  if (!a_u8 && !b_u8) return launch_one<BN, false, false, true>(a, cs, c_vec, ta, tb, tc, s);
  if (a_u8 && !b_u8) return launch_one<BN, true, false, true>(a, cs, c_vec, ta, tb, tc, s);
  if (!a_u8 && b_u8) return launch_one<BN, false, true, true>(a, cs, c_vec, ta, tb, tc, s);
  return launch_one<BN, true, true, true>(a, cs, c_vec, ta, tb, tc, s);
}

}  // namespace gemmf

cudaError_t launch_gemm_f16pair(const GemmF16Args& a, bool a_u8, bool b_u8, bool mmi, int chunk_k, cudaStream_t s,
                                const char** kernel_name) {
  using namespace gemmf;
  const int cs = chunk_k / BK;
  const int celem = (mmi || a.c_f32) ? 4 : 2;
  const bool acc_al = ((reinterpret_cast<uintptr_t>(a.acc_in) | reinterpret_cast<uintptr_t>(a.acc_out)) % 16) == 0;
  int c_vec = (((reinterpret_cast<uintptr_t>(a.C) % 16) == 0) && (((long long)a.N * celem) % 16 == 0) ? 1 : 0) |
                    ((acc_al && a.N % 4 == 0) ? 2 : 0);
  CUtensorMap ta{}, tb{}, tc{};
  cudaError_t e = make_maps(a, &ta, &tb);
  if (e != cudaSuccess) return e;
  if (mmi && (c_vec & 1)) {   // C as {N, M, batch} int32 / fp32, box 16 x 32, for the TMA-store epilogue
    e = make_tmap_3d(&tc, a.C, CU_TENSOR_MAP_DATA_TYPE_INT32, (uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.batch,
                     4ull * (uint64_t)a.N, 4ull * (uint64_t)a.M * (uint64_t)a.N, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (e != cudaSuccess) return e;
  }
  // accumulating A8W8: acc_in as {N, M, batch} int32, box 16 x 32, copied in by
  // the epilogue (c_vec bit 2) when its rows are 16-byte multiples
  if (!mmi && a.acc_in && (reinterpret_cast<uintptr_t>(a.acc_in) % 16) == 0 && a.N % 4 == 0) {
    e = make_tmap_3d(&tc, a.acc_in, CU_TENSOR_MAP_DATA_TYPE_INT32, (uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.batch,
                     4ull * (uint64_t)a.N, 4ull * (uint64_t)a.M * (uint64_t)a.N, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (e != cudaSuccess) return e;
    c_vec |= 4;
  }
  *kernel_name = mmi ? (a.act_scale ? "gemm_tc05_pair_f16ops_matmul_integer_dequant"
                           : "gemm_tc05_pair_f16ops_matmul_integer")
                     : ((a.acc_in || a.acc_out || !a.C) ? "gemm_tc05_pair_f16ops_a8w8_acc" : "gemm_tc05_pair_f16ops_a8w8");
  if (choose_tile_width(a) == 224) return dispatch<224>(a, a_u8, b_u8, mmi, cs, c_vec, ta, tb, tc, s);
  return dispatch<256>(a, a_u8, b_u8, mmi, cs, c_vec, ta, tb, tc, s);
}

// The convolution's pair-tile width, by the cost model of choose_tile_width
// over 256, 224 and 192 columns (output pixels): its problems are often a few
// tiles short of whole waves (3x3 8x256x56x56: 104, 112 or 136 tiles on 76
// SM pairs, all two waves; 192 makes them the shortest).
int conv_tile_width(const GemmF16Args& a) {
  const long long clusters = std::max(1, num_sms() / 2);
  const long long m_tiles = (a.M + gemmf::BMP - 1) / gemmf::BMP;
  int best = 256;
  long long best_cost = -1;
  for (int bn : {256, 224, 192}) {
    const long long tiles = (long long)a.batch * m_tiles * ((a.N + bn - 1) / bn);
    const long long cost = (tiles + clusters - 1) / clusters * (bn + 16);
    if (best_cost < 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

cudaError_t launch_gemm_f16pair_conv(const GemmF16Args& a, const CUtensorMap& tx, cudaStream_t s,
                                     const char** kernel_name) {
  using namespace gemmf;
  // |(x - x_zp)(w - w_zp)| <= 255^2: the u8 x u8 chunk keeps every fp32 sum exact
  const int cs = gemm_default_chunk_k(true, true) / BK;
  const int c_vec = (((reinterpret_cast<uintptr_t>(a.C) % 16) == 0) && (((long long)a.N * 4) % 16 == 0)) ? 1 : 0;
  if (!c_vec) return cudaErrorInvalidValue;   // the TMA-store epilogue needs 16-byte rows
  // A: the fp16 weight {K, Mg, groups} (box 64 x 128, 128-byte swizzle)
  const uint64_t ab = a.a_bstride ? (uint64_t)(a.a_bmod ? a.a_bmod : a.batch) : 1;
  const uint64_t ap = a.a_pitch ? (uint64_t)a.a_pitch : (uint64_t)a.K;
  const uint64_t as = 2ull * (a.a_bstride ? (uint64_t)a.a_bstride : (uint64_t)a.M * ap);
  CUtensorMap ta{}, tc{};
  cudaError_t e = make_tmap_3d(&ta, a.A16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)a.K, (uint64_t)a.M, ab,
                               2ull * ap, as, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tc, a.C, CU_TENSOR_MAP_DATA_TYPE_INT32, (uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.batch,
                   4ull * (uint64_t)a.N, 4ull * (uint64_t)a.M * (uint64_t)a.N, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  *kernel_name = "gemm_tc05_pair_f16ops_conv_im2col";
  // the im2col map's pixel box is conv_tile_width(a) / 2 (the caller builds it)
  switch (conv_tile_width(a)) {
    case 192: return launch_one<192, false, false, true, false, false, false, true>(a, cs, c_vec, ta, tx, tc, s);
    case 224: return launch_one<224, false, false, true, false, false, false, true>(a, cs, c_vec, ta, tx, tc, s);
    default: return launch_one<256, false, false, true, false, false, false, true>(a, cs, c_vec, ta, tx, tc, s);
  }
}

cudaError_t launch_gemm_w8_bf16pair(const GemmF16Args& a, int w_k, cudaStream_t s, const char** kernel_name) {
  using namespace gemmf;
  const int cs = (a.K + BK - 1) / BK;   // one chunk: fp32 accumulation over all of K
  const int celem = a.c_f32 ? 4 : 2;
  const int c_vec = ((reinterpret_cast<uintptr_t>(a.C) % 16) == 0) && (((long long)a.N * celem) % 16 == 0);
  // A: {K_eff, M} with K_eff = a.K; W: {N, w_k} (its true K rows: coordinates
  // past them, in the padding of split activations, read as zeros)
  CUtensorMap ta{}, tb{};
  GemmF16Args wa = a;
  wa.K = w_k;
  cudaError_t e = make_maps(a, &ta, &tb);
  CUtensorMap unused{}, tc{};
  if (e == cudaSuccess) e = make_maps(wa, &unused, &tb);
  if (e != cudaSuccess) return e;
  *kernel_name = "gemm_tc05_pair_w8_bf16";
  if (choose_tile_width(a) == 224) return launch_one<224, false, false, false, true>(a, cs, c_vec, ta, tb, tc, s);
  return launch_one<256, false, false, false, true>(a, cs, c_vec, ta, tb, tc, s);
}

}  // namespace qmm
