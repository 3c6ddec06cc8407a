// Exact 8-bit x 8-bit GEMM on the sm_103a tensor cores (tcgen05), with the
// dequantisation fused into the epilogue.
//
// The sm_103a tensor core has no 8-bit integer MMA kind, so the contraction
// runs on tcgen05.mma kind::f16 with fp16 operands: every int8 and uint8 value
// is exact in fp16, every product of two of them is exact in fp32, and an fp32
// sum of such products stays exact while its magnitude stays within 2^24. K is
// therefore split into chunks no longer than 2^24 / max|product| (1024 for
// s8 x s8, 512 for u8 x s8, 256 for u8 x u8). After each chunk the fp32 TMEM
// accumulator is converted to int32 (exact) and added, wrapping, into a running
// int32 sum that also lives in TMEM. The result is the exact int32 product
// sum_k A*B modulo 2^32 -- the INT32 accumulator of the A8W8 lowering
// (PyPTO PR #1920, "Feature/a8w8 matmul dequant fusion", sequence diagram) and
// the wrapping int32 of MatMulInteger (ROCm hip-ep PR #1248, "What",
// MatMulInteger paragraph).
//
// Epilogues, applied in registers as the tile leaves TMEM:
//  * A8W8: cast the int32 sum to fp32, multiply by act_scale[m] (rows), then by
//    weight_scale[n] (columns), then round to the output type (PyPTO PR #1920,
//    sequence diagram and the review comments on 1-D scales).
//  * MatMulInteger: sum_k (a-za)(b-zb) = acc - za*colsum(B)[n] - zb*rowsum(A)[m]
//    + K*za*zb, exact modulo 2^32. rowsum(A) and colsum(B) are computed by the
//    converter warps from the same bytes they convert, in the same pass.
//
// CTA organisation (one persistent CTA per SM, 288 threads):
//  * warps 0-7 ("workers"): load 8-bit tiles from global memory into
//    registers (two stages of prefetch), convert them to fp16 and write them to
//    shared memory in the canonical 128-byte-swizzled layouts the MMA reads
//    (A K-major, B MN-major); keep the row/column sums; drain the TMEM
//    accumulator after each K-chunk; run the epilogue and store C.
//  * warp 8: allocates TMEM and, from one lane, issues the MMAs
//    (M=128, N=256, K=16 per instruction) and the commits.
// Tile: 128 x 256 outputs, K stage 64, 4 shared-memory stages (48 KB each).
// TMEM: columns [0,256) the fp32 chunk accumulator, [256,512) the int32 sums.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace qmm {
namespace gemm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int NS = 4;                  // shared-memory stages
constexpr int LOOKAHEAD = NS - 1;      // stages produced past a chunk before it is drained
constexpr int NWW = 8;                 // worker warps
constexpr int NW = NWW * 32;
constexpr int NT = NW + 32;
constexpr int A_BYTES = BM * BK * 2;   // fp16 A stage: 16 KB
constexpr int B_BYTES = BK * BN * 2;   // fp16 B stage: 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SUM_RING = LOOKAHEAD + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SUM_COL = 256;      // TMEM columns [256, 512): running int32 sums

struct Shared {
  int part[NWW][BN];
  int rowsum[SUM_RING][BM];
  int colsum[SUM_RING][BN];
  uint64_t full[NS];
  uint64_t empty[NS];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t red_bar;
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = (size_t)NS * STAGE_BYTES + sizeof(Shared) + 1024;

// Error-site codes recorded on a timed-out wait.
enum : unsigned {
  SITE_EMPTY = 0x100, SITE_FULL = 0x101, SITE_ACC_FULL = 0x102, SITE_ACC_EMPTY = 0x103,
  SITE_RED = 0x104, SITE_TEARDOWN = 0x105
};

struct TileCoord {
  int b, m0, n0;
};

__device__ __forceinline__ TileCoord tile_coord(const GemmArgs& p, int tile_local) {
  const int m_tiles = (p.M + BM - 1) / BM;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tile_id = blockIdx.x + tile_local * gridDim.x;
  const int per_batch = m_tiles * n_tiles;
  TileCoord c;
  c.b = tile_id / per_batch;
  const int r = tile_id - c.b * per_batch;
  const int mt = r / n_tiles;
  c.m0 = mt * BM;
  c.n0 = (r - mt * n_tiles) * BN;
  return c;
}

// Gather 16 bytes of a row, zero outside [0, limit); byte-wise (any alignment).
__device__ __forceinline__ uint4 load16_bytes(const uint8_t* row, int col, int limit, bool row_ok) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (row_ok) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (col + i < limit) w[i >> 2] |= (uint32_t)__ldg(row + col + i) << (8 * (i & 3));
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Issue this thread's loads of one K-stage: 2 pieces of A (16 bytes each, rows
// t/4 and 64 + t/4, k-quarter t%4) and 4 pieces of B (k rows t/16 + 16j,
// 16 columns at (t%16)*16).
template <bool VEC>
__device__ __forceinline__ void load_stage(const GemmArgs& p, int gidx, int total, int spt, uint4 (&v)[6],
                                           int t) {
  if (gidx >= total) return;
  const int tl = gidx / spt;
  const int s = gidx - tl * spt;
  const TileCoord tc = tile_coord(p, tl);
  const uint8_t* Ab = p.A + (long long)tc.b * p.a_bstride;
  const uint8_t* Bb = p.B + (long long)tc.b * p.b_bstride;
  const int k0 = s * BK;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int row = tc.m0 + (t >> 2) + 64 * j;
    const int k = k0 + (t & 3) * 16;
    if (VEC) {
      v[j] = (row < p.M && k < p.K) ? ldg_nc_v4(Ab + (size_t)row * p.K + k) : make_uint4(0, 0, 0, 0);
    } else {
      v[j] = load16_bytes(Ab + (size_t)row * p.K, k, p.K, row < p.M);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k = k0 + (t >> 4) + 16 * j;
    const int n = tc.n0 + (t & 15) * 16;
    if (VEC) {
      v[2 + j] = (k < p.K && n < p.N) ? ldg_nc_v4(Bb + (size_t)k * p.N + n) : make_uint4(0, 0, 0, 0);
    } else {
      v[2 + j] = load16_bytes(Bb + (size_t)k * p.N, n, p.N, k < p.K);
    }
  }
}

// Convert this thread's pieces to fp16 and write them into the stage:
//  A: K-major, 128-byte swizzle. Row r of the 128-row tile is 128 bytes
//     (64 fp16 along K); 8-row groups form 1024-byte atoms; the 16-byte chunk
//     c of row r sits at chunk position c ^ (r % 8).
//  B: MN-major, 128-byte swizzle. K row k holds 64 fp16 along N per atom;
//     atom (k/8, n/64) starts at (k/8)*4096 + (n/64)*1024; chunk c = (n%64)/8
//     of row k%8 sits at chunk position c ^ (k % 8).
template <bool AU, bool BU>
__device__ __forceinline__ void store_stage(uint32_t a_base, uint32_t b_base, const uint4 (&v)[6], int t) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = (t >> 2) + 64 * j;
    const int kq = t & 3;
    uint32_t hv[8];
    bytes_to_half4<AU>(v[j].x, hv[0], hv[1]);
    bytes_to_half4<AU>(v[j].y, hv[2], hv[3]);
    bytes_to_half4<AU>(v[j].z, hv[4], hv[5]);
    bytes_to_half4<AU>(v[j].w, hv[6], hv[7]);
    const uint32_t rb = a_base + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
    st_shared_v4(rb + ((uint32_t)((kq * 2 + 0) ^ (r & 7)) << 4), hv[0], hv[1], hv[2], hv[3]);
    st_shared_v4(rb + ((uint32_t)((kq * 2 + 1) ^ (r & 7)) << 4), hv[4], hv[5], hv[6], hv[7]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k = (t >> 4) + 16 * j;
    const int nq = t & 15;
    uint32_t hv[8];
    bytes_to_half4<BU>(v[2 + j].x, hv[0], hv[1]);
    bytes_to_half4<BU>(v[2 + j].y, hv[2], hv[3]);
    bytes_to_half4<BU>(v[2 + j].z, hv[4], hv[5]);
    bytes_to_half4<BU>(v[2 + j].w, hv[6], hv[7]);
    const uint32_t kb =
        b_base + (uint32_t)(k >> 3) * 4096u + (uint32_t)(nq >> 2) * 1024u + (uint32_t)(k & 7) * 128u;
    st_shared_v4(kb + ((uint32_t)(((nq & 3) * 2 + 0) ^ (k & 7)) << 4), hv[0], hv[1], hv[2], hv[3]);
    st_shared_v4(kb + ((uint32_t)(((nq & 3) * 2 + 1) ^ (k & 7)) << 4), hv[4], hv[5], hv[6], hv[7]);
  }
}

template <bool U>
__device__ __forceinline__ int dp4a_ones(uint32_t w, int acc) {
  if (U) return (int)__dp4a(w, 0x01010101u, (unsigned)acc);
  return __dp4a((int)w, 0x01010101, acc);
}

// An mbarrier used as a bounded barrier among the 256 worker threads.
__device__ __forceinline__ bool worker_sync(Shared& sm, int& phase, unsigned* err) {
  mbar_arrive(&sm.red_bar);
  const bool ok = mbar_wait(&sm.red_bar, (uint32_t)(phase & 1), &sm.abort_flag, err, SITE_RED);
  ++phase;
  return ok;
}

// Epilogue of one tile: read the final int32 sums back from TMEM (this warp's
// 32 rows, its 128-column half, 32 columns at a time), apply the fused
// dequantisation / zero-point correction, and store C.
template <bool AU, bool BU, bool MMI>
__device__ __forceinline__ void epilogue(const GemmArgs& p, Shared& sm, uint32_t tbase, int tile_local, int q,
                                         int h, int lane, int c_vec) {
  const TileCoord tc = tile_coord(p, tile_local);
  const int slot = tile_local % SUM_RING;
  const int rloc = q * 32 + lane;
  const int row = tc.m0 + rloc;
  const bool row_ok = row < p.M;
  const uint32_t lane_off = (uint32_t)(q * 32) << 16;
  const size_t crow = ((size_t)tc.b * p.M + (size_t)(row_ok ? row : 0)) * (size_t)p.N;

  float as = 0.f;
  uint32_t za = 0u, rs = 0u;
  if (!MMI) {
    if (row_ok) as = __ldg(p.act_scale + (p.act_count == 1 ? 0 : row % p.zp_row_mod));
  } else {
    if (p.a_zp_count > 0 && row_ok) {
      const int zi = p.a_zp_count == 1 ? 0 : row % p.zp_row_mod;
      za = AU ? (uint32_t)__ldg((const uint8_t*)p.a_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.a_zp + zi);
    }
    if (p.b_zp_count > 0) rs = (uint32_t)sm.rowsum[slot][rloc];
  }

#pragma unroll 1
  for (int g = 0; g < 4; ++g) {
    uint32_t tot[32];
    tmem_ld32(tbase + lane_off + SUM_COL + (uint32_t)(h * 128 + g * 32), tot);   // warp-collective
    const int nb = tc.n0 + h * 128 + g * 32;
    if (!row_ok || nb >= p.N) continue;
    const bool full = (nb + 32 <= p.N) && c_vec;
    if (!MMI) {
      float f[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int n = nb + i;
        const float ws = (n < p.N) ? __ldg(p.w_scale + (p.w_count == 1 ? 0 : n)) : 0.f;
        float v = __int2float_rn((int)tot[i]);
        v = __fmul_rn(v, as);
        f[i] = __fmul_rn(v, ws);
      }
      if (p.c_f32) {
        float* out = reinterpret_cast<float*>(p.C) + crow + nb;
        if (full) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(out + i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
        } else {
          for (int i = 0; i < 32; ++i)
            if (nb + i < p.N) out[i] = f[i];
        }
      } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C) + crow + nb;
        if (full) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            __nv_bfloat162 b0 = __floats2bfloat162_rn(f[i + 0], f[i + 1]);
            __nv_bfloat162 b1 = __floats2bfloat162_rn(f[i + 2], f[i + 3]);
            __nv_bfloat162 b2 = __floats2bfloat162_rn(f[i + 4], f[i + 5]);
            __nv_bfloat162 b3 = __floats2bfloat162_rn(f[i + 6], f[i + 7]);
            w.x = *reinterpret_cast<uint32_t*>(&b0);
            w.y = *reinterpret_cast<uint32_t*>(&b1);
            w.z = *reinterpret_cast<uint32_t*>(&b2);
            w.w = *reinterpret_cast<uint32_t*>(&b3);
            *reinterpret_cast<uint4*>(out + i) = w;
          }
        } else {
          for (int i = 0; i < 32; ++i)
            if (nb + i < p.N) out[i] = __float2bfloat16_rn(f[i]);
        }
      }
    } else {
      uint32_t o[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int n = nb + i;
        uint32_t zb = 0u, cs = 0u;
        if (p.b_zp_count > 0 && n < p.N) {
          const int zi = p.b_zp_count == 1 ? 0 : n;
          zb = BU ? (uint32_t)__ldg((const uint8_t*)p.b_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.b_zp + zi);
        }
        if (p.a_zp_count > 0) cs = (uint32_t)sm.colsum[slot][h * 128 + g * 32 + i];
        o[i] = tot[i] - za * cs - zb * rs + (uint32_t)p.K * za * zb;
      }
      int32_t* out = reinterpret_cast<int32_t*>(p.C) + crow + nb;
      if (full) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<int4*>(out + i) = make_int4((int)o[i], (int)o[i + 1], (int)o[i + 2], (int)o[i + 3]);
      } else {
        for (int i = 0; i < 32; ++i)
          if (nb + i < p.N) out[i] = (int)o[i];
      }
    }
  }
}

template <bool AU, bool BU, bool MMI, bool VEC>
__global__ void __launch_bounds__(NT, 1) gemm_tc_kernel(const GemmArgs p, const int cs, const int c_vec) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sbase_ptr = smem_raw + (sbase - raw);
  Shared& sm = *reinterpret_cast<Shared*>(sbase_ptr + NS * STAGE_BYTES);

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;

  const int m_tiles = (p.M + BM - 1) / BM;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int num_tiles = p.batch * m_tiles * n_tiles;
  const int my_tiles =
      ((int)blockIdx.x < num_tiles) ? (num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int spt = (p.K + BK - 1) / BK;       // K stages per tile
  const int cpt = (spt + cs - 1) / cs;       // K chunks per tile
  const int total_stages = my_tiles * spt;
  const int total_chunks = my_tiles * cpt;

  if (t == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm.full[i], NW);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, NW);
    mbar_init(&sm.red_bar, NW);
    mbar_init(&sm.teardown, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == NWW) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;

  if (warp == NWW) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(BM, BN, false, true);
      int g = 0;
      int d = 0;
      bool ok = true;
      for (int tl = 0; tl < my_tiles && ok; ++tl) {
        for (int c = 0; c < cpt && ok; ++c) {
          if (d > 0) {
            ok = mbar_wait(&sm.acc_empty, (uint32_t)((d - 1) & 1), &sm.abort_flag, p.err, SITE_ACC_EMPTY);
            if (!ok) break;
          }
          tc_fence_after();
          const int s_beg = c * cs;
          const int s_end = min(spt, s_beg + cs);
          for (int s = s_beg; s < s_end; ++s, ++g) {
            const int slot = g % NS;
            ok = mbar_wait(&sm.full[slot], (uint32_t)((g / NS) & 1), &sm.abort_flag, p.err, SITE_FULL);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_addr = sbase + (uint32_t)slot * STAGE_BYTES;
            const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              const uint64_t ad = sdesc_sw128(a_addr + (uint32_t)j * 32u, 16u, 1024u);
              const uint64_t bd = sdesc_sw128(b_addr + (uint32_t)j * 8192u, 1024u, 4096u);
              tc_mma_f16(tbase, ad, bd, idesc, (s > s_beg || j > 0) ? 1u : 0u);
            }
            tc_commit(&sm.empty[slot]);
          }
          if (!ok) break;
          tc_commit(&sm.acc_full);
          ++d;
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- workers ----------------
    const int q = warp & 3;      // TMEM lane quarter this warp may access
    const int h = warp >> 2;     // column half of the 256-column tile
    const bool need_rs = MMI && p.b_zp_count > 0;
    const bool need_cs = MMI && p.a_zp_count > 0;
    int red_phase = 0;
    int drain_d = 0;
    bool ok = true;

    int rs_acc[2] = {0, 0};
    uint32_t ce[4] = {0u, 0u, 0u, 0u}, co[4] = {0u, 0u, 0u, 0u};
    int col32[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) col32[i] = 0;

    uint4 cur[6], nx1[6], nx2[6];
    load_stage<VEC>(p, 0, total_stages, spt, cur, t);
    load_stage<VEC>(p, 1, total_stages, spt, nx1, t);

    // Drain chunk d of this CTA's chunk sequence: convert the fp32 chunk sum
    // to int32 and fold it into the running sums (TMEM columns 256..511); on a
    // tile's last chunk, also run the epilogue.
    auto drain = [&](int d) -> bool {
      if (!mbar_wait(&sm.acc_full, (uint32_t)(d & 1), &sm.abort_flag, p.err, SITE_ACC_FULL)) return false;
      tc_fence_after();
      const int tl = d / cpt;
      const int c = d - tl * cpt;
      const uint32_t lane_off = (uint32_t)(q * 32) << 16;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        const uint32_t col = (uint32_t)(h * 128 + g * 32);
        uint32_t acc[32];
        uint32_t sum[32];
        tmem_ld32(tbase + lane_off + col, acc);
        if (c > 0) {
          tmem_ld32(tbase + lane_off + SUM_COL + col, sum);
#pragma unroll
          for (int i = 0; i < 32; ++i) sum[i] += (uint32_t)__float2int_rn(__uint_as_float(acc[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) sum[i] = (uint32_t)__float2int_rn(__uint_as_float(acc[i]));
        }
        tmem_st32(tbase + lane_off + SUM_COL + col, sum);
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_empty);
      if (c == cpt - 1) epilogue<AU, BU, MMI>(p, sm, tbase, tl, q, h, lane, c_vec);
      return true;
    };

    for (int g = 0; g < total_stages && ok; ++g) {
      load_stage<VEC>(p, g + 2, total_stages, spt, nx2, t);
      const int slot = g % NS;
      if (g >= NS) {
        ok = mbar_wait(&sm.empty[slot], (uint32_t)(((g / NS) - 1) & 1), &sm.abort_flag, p.err, SITE_EMPTY);
        if (!ok) break;
      }
      const uint32_t a_addr = sbase + (uint32_t)slot * STAGE_BYTES;
      store_stage<AU, BU>(a_addr, a_addr + A_BYTES, cur, t);
      fence_proxy_async_smem();
      mbar_arrive(&sm.full[slot]);

      const int tl = g / spt;
      const int s = g - tl * spt;
      if (need_rs) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          rs_acc[j] = dp4a_ones<AU>(cur[j].x, rs_acc[j]);
          rs_acc[j] = dp4a_ones<AU>(cur[j].y, rs_acc[j]);
          rs_acc[j] = dp4a_ones<AU>(cur[j].z, rs_acc[j]);
          rs_acc[j] = dp4a_ones<AU>(cur[j].w, rs_acc[j]);
        }
      }
      if (need_cs) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w[4] = {cur[2 + j].x, cur[2 + j].y, cur[2 + j].z, cur[2 + j].w};
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint32_t u = BU ? w[qq] : (w[qq] ^ 0x80808080u);
            ce[qq] += prmt(u, 0u, 0x4240u);   // bytes 0 and 2 into 16-bit lanes
            co[qq] += prmt(u, 0u, 0x4341u);   // bytes 1 and 3
          }
        }
        // 16-bit lanes take at most 257 additions of 255: fold every 64 stages.
        if ((s & 63) == 63 || s == spt - 1) {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            col32[4 * qq + 0] += (int)(ce[qq] & 0xFFFFu);
            col32[4 * qq + 2] += (int)(ce[qq] >> 16);
            col32[4 * qq + 1] += (int)(co[qq] & 0xFFFFu);
            col32[4 * qq + 3] += (int)(co[qq] >> 16);
            ce[qq] = 0u;
            co[qq] = 0u;
          }
        }
      }
      if (s == spt - 1 && (need_rs || need_cs)) {
        // Tile finished: reduce this tile's row and column sums into shared memory.
        const int ring = tl % SUM_RING;
        if (need_rs) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            int v = rs_acc[j];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if ((t & 3) == 0) sm.rowsum[ring][(t >> 2) + 64 * j] = v;
            rs_acc[j] = 0;
          }
        }
        if (need_cs) {
          const int bias = BU ? 0 : 128 * 4 * spt;   // every added byte carried +128
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            int v = col32[i] - bias;
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (lane < 16) sm.part[warp][(t & 15) * 16 + i] = v;
            col32[i] = 0;
          }
          ok = worker_sync(sm, red_phase, p.err);
          if (!ok) break;
          int v = 0;
#pragma unroll
          for (int w = 0; w < NWW; ++w) v += sm.part[w][t];
          sm.colsum[ring][t] = v;
        }
        ok = worker_sync(sm, red_phase, p.err);
        if (!ok) break;
      }

      while (ok && drain_d < total_chunks) {
        const int dtl = drain_d / cpt;
        const int dc = drain_d - dtl * cpt;
        const int last_stage = dtl * spt + min((dc + 1) * cs, spt) - 1;
        if (last_stage + LOOKAHEAD > g) break;
        ok = drain(drain_d);
        ++drain_d;
      }
#pragma unroll
      for (int i = 0; i < 6; ++i) {
        cur[i] = nx1[i];
        nx1[i] = nx2[i];
      }
    }
    while (ok && drain_d < total_chunks) {
      ok = drain(drain_d);
      ++drain_d;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == NWW) {
    tc_fence_after();
    if (sm.abort_flag) {
      // After an abort, wait (bounded) for any MMA still in flight before freeing TMEM.
      if (lane == 0) {
        tc_commit(&sm.teardown);
        mbar_wait(&sm.teardown, 0u, nullptr, p.err, SITE_TEARDOWN);
      }
      __syncwarp();
    }
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

template <bool AU, bool BU, bool MMI, bool VEC>
cudaError_t launch_one(const GemmArgs& a, int cs, int c_vec, cudaStream_t s) {
  auto kern = gemm_tc_kernel<AU, BU, MMI, VEC>;
  static unsigned attr_set_mask = 0;   // per instantiation, one bit per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || !(attr_set_mask & (1u << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 32) attr_set_mask |= 1u << dev;
  }
  const int m_tiles = (a.M + BM - 1) / BM;
  const int n_tiles = (a.N + BN - 1) / BN;
  const long long tiles = (long long)a.batch * m_tiles * n_tiles;
  const int grid = (int)std::min<long long>(tiles, (long long)num_sms());
  kern<<<grid, NT, SMEM_BYTES, s>>>(a, cs, c_vec);
  return cudaGetLastError();
}

}  // namespace gemm

int gemm_default_chunk_k(bool a_u8, bool b_u8) {
  // largest multiple of 64 with chunk * max|a*b| <= 2^24
  if (a_u8 && b_u8) return 256;    // 65025 * 256  < 2^24
  if (a_u8 || b_u8) return 512;    // 32640 * 512  < 2^24
  return 1024;                     // 16384 * 1024 = 2^24
}

cudaError_t launch_gemm_tc(const GemmArgs& a, bool a_u8, bool b_u8, bool mmi, int chunk_k, cudaStream_t s,
                           const char** kernel_name) {
  using namespace gemm;
  const int cs = chunk_k / BK;
  const uintptr_t ua = reinterpret_cast<uintptr_t>(a.A), ub = reinterpret_cast<uintptr_t>(a.B);
  const bool vec = (a.K % 16 == 0) && (a.N % 16 == 0) && (ua % 16 == 0) && (ub % 16 == 0) &&
                   (a.a_bstride % 16 == 0) && (a.b_bstride % 16 == 0);
  const int celem = (mmi || a.c_f32) ? 4 : 2;
  const int c_vec = ((reinterpret_cast<uintptr_t>(a.C) % 16) == 0) && (((long long)a.N * celem) % 16 == 0);
  if (!mmi) {
    *kernel_name = vec ? "gemm_tc05_exact_a8w8" : "gemm_tc05_exact_a8w8_bytewise";
    return vec ? launch_one<false, false, false, true>(a, cs, c_vec, s)
               : launch_one<false, false, false, false>(a, cs, c_vec, s);
  }
  *kernel_name = vec ? "gemm_tc05_exact_matmul_integer" : "gemm_tc05_exact_matmul_integer_bytewise";
#define QMM_DISPATCH(AU, BU)                                                                   \
  if (a_u8 == AU && b_u8 == BU)                                                                \
    return vec ? launch_one<AU, BU, true, true>(a, cs, c_vec, s)                              \
               : launch_one<AU, BU, true, false>(a, cs, c_vec, s);
  QMM_DISPATCH(false, false)
  QMM_DISPATCH(true, false)
  QMM_DISPATCH(false, true)
  QMM_DISPATCH(true, true)
#undef QMM_DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace qmm
