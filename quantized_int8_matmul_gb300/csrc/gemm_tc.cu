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
// CTA organisation (one persistent CTA per SM, 320 threads):
//  * warp 9 (producer): one lane copies 8-bit tiles of A (128 rows x 64 k) and
//    B (64 k x 256 columns) from global memory into a 4-stage shared-memory
//    staging ring with TMA (cp.async.bulk.tensor, completion counted on the
//    stage's mbarrier); out-of-range rows and columns arrive as zeros.
//  * warps 0-7 ("workers"): read a staged stage with 16-byte shared loads,
//    convert the bytes to fp16 (byte in the mantissa of 1024, bias subtracted)
//    and write them into a 2-stage ring in the canonical 128-byte-swizzled
//    layouts the MMA reads (A K-major, B MN-major, so B is never transposed);
//    keep the row/column sums; drain the TMEM accumulator after each K-chunk;
//    run the epilogue and store C.
//  * warp 8: allocates TMEM and, from one lane, issues the MMAs
//    (M=128, N=256, K=16 per instruction) and the commits.
// Tile: 128 x 256 outputs, K stage 64; fp16 stage 48 KB, int8 stage 24 KB.
// TMEM: columns [0,256) the fp32 chunk accumulator, [256,512) the int32 sums.
#include "common.cuh"
#include "kernels.h"
#include "tma.h"

#include <algorithm>

namespace qmm {
namespace gemm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int NS = 2;                  // fp16 shared-memory stages read by the MMA
constexpr int NI = 4;                  // int8 staging stages filled by TMA
constexpr int LOOKAHEAD = NS - 1;      // stages produced past a chunk before it is drained
constexpr int NWW = 8;                 // worker warps
constexpr int NW = NWW * 32;
constexpr int NT = NW + 64;            // + MMA warp + TMA producer warp
constexpr int A_BYTES = BM * BK * 2;   // fp16 A stage: 16 KB
constexpr int B_BYTES = BK * BN * 2;   // fp16 B stage: 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int I8_A = BM * BK;          // int8 A staging: 128 rows x 64 bytes
constexpr int I8_B = BK * BN;          // int8 B staging: 64 rows x 256 bytes
constexpr int I8_STAGE = I8_A + I8_B;  // 24 KB
constexpr int SUM_RING = LOOKAHEAD + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SUM_COL = 256;      // TMEM columns [256, 512): running int32 sums

struct Shared {
  int part[NWW][BN];
  int rowsum[SUM_RING][BM];
  int colsum[SUM_RING][BN];
  // per-tile epilogue operands, staged when the tile's first stage is converted:
  // A8W8: weight_scale[n] (as float bits) and act_scale[m]; MatMulInteger:
  // b_zp[n] and a_zp[m] (as int)
  uint32_t col_op[SUM_RING][BN];
  uint32_t row_op[SUM_RING][BM];
  uint64_t full[NS];
  uint64_t empty[NS];
  uint64_t i8_full[NI];
  uint64_t i8_empty[NI];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t red_bar;
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = (size_t)NS * STAGE_BYTES + (size_t)NI * I8_STAGE + sizeof(Shared) + 1024;

// Error-site codes recorded on a timed-out wait.
enum : unsigned {
  SITE_EMPTY = 0x100, SITE_FULL = 0x101, SITE_ACC_FULL = 0x102, SITE_ACC_EMPTY = 0x103,
  SITE_RED = 0x104, SITE_TEARDOWN = 0x105, SITE_I8_FULL = 0x106, SITE_I8_EMPTY = 0x107, SITE_I8_DRAIN = 0x108
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

// Piece assignment of worker thread t (0..255) in one 64-deep K stage:
//  A: 2 pieces of 16 bytes, rows t/4 and 64 + t/4 of the tile, k bytes (t%4)*16.
//  B: 4 pieces of 16 bytes, k rows 2*(t/32) + ((t/4)&1) + 16j, columns 16*nq with
//     nq = (t&3) | ((t&31)/8)*4. A quarter-warp then writes two k rows of one
//     64-column atom, i.e. 8 distinct 16-byte slots of the swizzle pattern, so
//     the shared-memory stores are free of bank conflicts.
__device__ __forceinline__ int a_row(int t, int j) { return (t >> 2) + 64 * j; }
__device__ __forceinline__ int a_kq(int t) { return t & 3; }
__device__ __forceinline__ int b_nq(int t) { return (t & 3) | (((t & 31) >> 3) << 2); }
__device__ __forceinline__ int b_krow(int t, int j) { return 2 * (t >> 5) + ((t >> 2) & 1) + 16 * j; }

// Where a worker's loads stand: the tile and stage being loaded, this thread's
// first A and B piece pointers at that stage (the second A piece is 64 rows
// further, B piece j is 16*j rows further), and which pieces lie inside.
struct LoadCursor {
  int tl, s, k0;             // local tile index, stage in tile, k of the stage
  int b, m0, n0;             // tile coordinates
  const uint8_t* pa;
  const uint8_t* pb;
  bool a_ok0, a_ok1, b_ok;
};

__device__ __forceinline__ void cursor_tile(const GemmArgs& p, int tl, int t, LoadCursor& c) {
  const TileCoord tc = tile_coord(p, tl);
  c.tl = tl;
  c.s = 0;
  c.k0 = 0;
  c.b = tc.b;
  c.m0 = tc.m0;
  c.n0 = tc.n0;
  const int row = tc.m0 + a_row(t, 0);
  c.a_ok0 = row < p.M;
  c.a_ok1 = row + 64 < p.M;
  c.pa = p.A + (long long)tc.b * p.a_bstride + (size_t)row * p.K + a_kq(t) * 16;
  const int n = tc.n0 + b_nq(t) * 16;
  c.b_ok = n < p.N;
  c.pb = p.B + (long long)tc.b * p.b_bstride + (size_t)b_krow(t, 0) * p.N + n;
}

__device__ __forceinline__ void cursor_advance(const GemmArgs& p, int spt, int t, LoadCursor& c) {
  if (++c.s == spt) {
    cursor_tile(p, c.tl + 1, t, c);
    return;
  }
  c.k0 += BK;
  c.pa += BK;
  c.pb += (size_t)BK * p.N;
}

// Issue this thread's six 16-byte loads for the cursor's stage (zeros outside the matrices).
template <bool VEC>
__device__ __forceinline__ void load_pieces(const GemmArgs& p, const LoadCursor& c, int t, uint4 (&v)[6]) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  if (VEC) {
    const bool kfull = c.k0 + BK <= p.K;   // every piece of the stage is inside K
    const bool ka = kfull || c.k0 + a_kq(t) * 16 < p.K;
    v[0] = (c.a_ok0 && ka) ? ldg_nc_v4(c.pa) : z;
    v[1] = (c.a_ok1 && ka) ? ldg_nc_v4(c.pa + (size_t)64 * p.K) : z;
    const size_t bstep = (size_t)16 * p.N;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = c.b_ok && (kfull || c.k0 + b_krow(t, j) < p.K);
      v[2 + j] = ok ? ldg_nc_v4(c.pb + j * bstep) : z;
    }
  } else {
    const uint8_t* Ab = p.A + (long long)c.b * p.a_bstride;
    const uint8_t* Bb = p.B + (long long)c.b * p.b_bstride;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int row = c.m0 + a_row(t, j);
      v[j] = load16_bytes(Ab + (size_t)row * p.K, c.k0 + a_kq(t) * 16, p.K, row < p.M);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = c.k0 + b_krow(t, j);
      v[2 + j] = load16_bytes(Bb + (size_t)k * p.N, c.n0 + b_nq(t) * 16, p.N, k < p.K);
    }
  }
}

// Shared-memory byte offsets (within a stage) of this thread's 12 16-byte stores.
//  A: K-major, 128-byte swizzle. Row r of the 128-row tile is 128 bytes
//     (64 fp16 along K); 8-row groups form 1024-byte atoms; the 16-byte chunk
//     c of row r sits at chunk position c ^ (r % 8).
//  B: MN-major, 128-byte swizzle. K row k holds 64 fp16 along N per atom;
//     atom (k/8, n/64) starts at (k/8)*4096 + (n/64)*1024; chunk c = (n%64)/8
//     of row k%8 sits at chunk position c ^ (k % 8).
struct StoreOffsets {
  uint32_t a0, a1;   // A piece 0, chunks 0 and 1 (piece 1: +8192, 64 rows = 8 atoms further)
  uint32_t b0, b1;   // B piece 0, chunks 0 and 1 (piece j: +8192*j, 16 k rows further)
};

__device__ __forceinline__ StoreOffsets store_offsets(int t) {
  StoreOffsets o;
  const int r = a_row(t, 0);
  const uint32_t rb = (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
  o.a0 = rb + ((uint32_t)((a_kq(t) * 2 + 0) ^ (r & 7)) << 4);
  o.a1 = rb + ((uint32_t)((a_kq(t) * 2 + 1) ^ (r & 7)) << 4);
  const int nq = b_nq(t);
  const int k = b_krow(t, 0);
  const uint32_t kb = (uint32_t)A_BYTES + (uint32_t)(k >> 3) * 4096u + (uint32_t)(nq >> 2) * 1024u +
                      (uint32_t)(k & 7) * 128u;
  o.b0 = kb + ((uint32_t)(((nq & 3) * 2 + 0) ^ (k & 7)) << 4);
  o.b1 = kb + ((uint32_t)(((nq & 3) * 2 + 1) ^ (k & 7)) << 4);
  return o;
}

// Convert this thread's pieces to fp16 and write them into the stage at `base`.
template <bool AU, bool BU>
__device__ __forceinline__ void store_stage(uint32_t base, const StoreOffsets& o, const uint4 (&v)[6]) {
#pragma unroll
  for (int j = 0; j < 6; ++j) {
    uint32_t hv[8];
    const bool isa = j < 2;
    if (isa) {
      bytes_to_half4<AU>(v[j].x, hv[0], hv[1]);
      bytes_to_half4<AU>(v[j].y, hv[2], hv[3]);
      bytes_to_half4<AU>(v[j].z, hv[4], hv[5]);
      bytes_to_half4<AU>(v[j].w, hv[6], hv[7]);
    } else {
      bytes_to_half4<BU>(v[j].x, hv[0], hv[1]);
      bytes_to_half4<BU>(v[j].y, hv[2], hv[3]);
      bytes_to_half4<BU>(v[j].z, hv[4], hv[5]);
      bytes_to_half4<BU>(v[j].w, hv[6], hv[7]);
    }
    const uint32_t off = isa ? (uint32_t)j * 8192u : (uint32_t)(j - 2) * 8192u;
    st_shared_v4(base + (isa ? o.a0 : o.b0) + off, hv[0], hv[1], hv[2], hv[3]);
    st_shared_v4(base + (isa ? o.a1 : o.b1) + off, hv[4], hv[5], hv[6], hv[7]);
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
// 32 rows, its 128-column half, 16 columns at a time), apply the fused
// dequantisation / zero-point correction, and store C. Outputs are written
// with an evict-first L2 policy so they do not push the operands out of L2.
template <bool AU, bool BU, bool MMI>
__device__ __noinline__ void epilogue(const GemmArgs& p, Shared& sm, uint32_t tbase, int tile_local, int q, int h,
                                      int lane, int c_vec) {
  const TileCoord tc = tile_coord(p, tile_local);
  const int slot = tile_local % SUM_RING;
  const int rloc = q * 32 + lane;
  const int row = tc.m0 + rloc;
  const bool row_ok = row < p.M;
  const uint32_t lane_off = (uint32_t)(q * 32) << 16;
  const size_t crow = ((size_t)tc.b * p.M + (size_t)(row_ok ? row : 0)) * (size_t)p.N;
  const uint64_t pol = l2_policy_evict_first();

  uint32_t hold[16];   // second half of a 32-column TMEM load
  const float as = __uint_as_float(sm.row_op[slot][rloc]);         // A8W8: act_scale of this row
  const uint32_t za = sm.row_op[slot][rloc];                        // MatMulInteger: a_zp of this row
  const uint32_t rs = (MMI && p.b_zp_count > 0) ? (uint32_t)sm.rowsum[slot][rloc] : 0u;

#pragma unroll 1
  for (int g = 0; g < 8; ++g) {
    uint32_t tot[16];
    if ((g & 1) == 0) {
      uint32_t t32[32];
      tmem_ld32(tbase + lane_off + SUM_COL + (uint32_t)(h * 128 + g * 16), t32);   // warp-collective
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        tot[i] = t32[i];
        hold[i] = t32[16 + i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) tot[i] = hold[i];
    }
    const int nb = tc.n0 + h * 128 + g * 16;
    if (!row_ok || nb >= p.N) continue;
    const bool full = (nb + 16 <= p.N) && c_vec;
    uint32_t o[16];
    if (!MMI) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float ws = __uint_as_float(sm.col_op[slot][h * 128 + g * 16 + i]);
        float v = __int2float_rn((int)tot[i]);
        v = __fmul_rn(v, as);
        o[i] = __float_as_uint(__fmul_rn(v, ws));
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
        const uint32_t zb = sm.col_op[slot][h * 128 + g * 16 + i];
        const uint32_t cs = (p.a_zp_count > 0) ? (uint32_t)sm.colsum[slot][h * 128 + g * 16 + i] : 0u;
        o[i] = tot[i] - za * cs - zb * rs + (uint32_t)p.K * za * zb;
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

template <bool AU, bool BU, bool MMI, bool VEC>
__global__ void __launch_bounds__(NT, 1)
    gemm_tc_kernel(const GemmArgs p, const int cs, const int c_vec, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sbase_ptr = smem_raw + (sbase - raw);
  const uint32_t i8base = sbase + NS * STAGE_BYTES;   // int8 staging ring
  Shared& sm = *reinterpret_cast<Shared*>(sbase_ptr + NS * STAGE_BYTES + NI * I8_STAGE);

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
    for (int i = 0; i < NI; ++i) {
      mbar_init(&sm.i8_full[i], 1);
      mbar_init(&sm.i8_empty[i], NW);
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
  } else if (warp == NWW + 1) {
    // ---------------- TMA producer: int8 tiles of A and B into the staging ring ----------------
    if (VEC && lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int tl = 0, s = 0, g = 0;
      TileCoord tc = tile_coord(p, 0);
      for (; g < total_stages; ++g) {
        const int slot = g & (NI - 1);
        if (g >= NI &&
            !mbar_wait(&sm.i8_empty[slot], (uint32_t)(((g / NI) - 1) & 1), &sm.abort_flag, p.err, SITE_I8_EMPTY))
          break;
        const uint32_t dst = i8base + (uint32_t)slot * I8_STAGE;
        mbar_arrive_expect_tx(&sm.i8_full[slot], I8_STAGE);
        tma_load_3d(dst, &tmA, s * BK, tc.m0, p.a_bstride ? tc.b : 0, &sm.i8_full[slot]);
        tma_load_3d(dst + I8_A, &tmB, tc.n0, s * BK, p.b_bstride ? tc.b : 0, &sm.i8_full[slot]);
        if (++s == spt) {
          s = 0;
          tc = tile_coord(p, ++tl);
        }
      }
      // Before the CTA may exit, wait (bounded) until the copies issued have landed.
      for (int j = (g > NI ? g - NI : 0); j < g; ++j)
        mbar_wait(&sm.i8_full[j & (NI - 1)], (uint32_t)((j / NI) & 1), nullptr, p.err, SITE_I8_DRAIN);
    }
    __syncwarp();
  } else {
    // ---------------- workers ----------------
    const int q = warp & 3;      // TMEM lane quarter this warp may access
    const int h = warp >> 2;     // column half of the 256-column tile
    const bool need_rs = MMI && p.b_zp_count > 0;
    const bool need_cs = MMI && p.a_zp_count > 0;
    int red_phase = 0;
    bool ok = true;

    // next chunk to drain, and the last stage it contains
    int dr_d = 0, dr_tl = 0, dr_c = 0;
    int dr_last = min(cs, spt) - 1;

    int rs_acc[2] = {0, 0};
    uint32_t ce[4] = {0u, 0u, 0u, 0u}, co[4] = {0u, 0u, 0u, 0u};
    // Column sums accumulate in sm.part[warp][column]: lane t (k-row parity 0)
    // owns the 16 columns b_nq(t)*16.. of its warp's row.
    const bool cs_owner = ((t >> 2) & 1) == 0;
    if (need_cs && cs_owner) {
#pragma unroll
      for (int i = 0; i < 16; ++i) sm.part[warp][b_nq(t) * 16 + i] = 0;
    }

    const StoreOffsets so = store_offsets(t);
    // this thread's six 16-byte pieces in an int8 staging stage (A rows +64, B rows +16 per piece)
    const uint32_t ia0 = (uint32_t)a_row(t, 0) * 64u + (uint32_t)a_kq(t) * 16u;
    const uint32_t ib0 = (uint32_t)I8_A + (uint32_t)b_krow(t, 0) * 256u + (uint32_t)b_nq(t) * 16u;
    LoadCursor lc;                 // direct byte loads (unaligned shapes only)
    if (!VEC) cursor_tile(p, 0, t, lc);
    int st_tl = 0, st_s = 0;     // tile and stage being stored

    // Drain chunk dr_d: convert the fp32 chunk sum to int32 and fold it into the
    // running sums (TMEM columns 256..511); on a tile's last chunk, run the epilogue.
    auto drain = [&]() -> bool {
      if (!mbar_wait(&sm.acc_full, (uint32_t)(dr_d & 1), &sm.abort_flag, p.err, SITE_ACC_FULL)) return false;
      tc_fence_after();
      const uint32_t lane_off = (uint32_t)(q * 32) << 16;
      const uint32_t t_acc = tbase + lane_off + (uint32_t)(h * 128);
      const uint32_t t_sum = t_acc + SUM_COL;
      // 16-column groups: accumulator and running sum in one load-wait, asynchronous store
#pragma unroll 1
      for (int g = 0; g < 8; ++g) {
        uint32_t acc[16];
        uint32_t sum[16];
        if (dr_c > 0) {
          tmem_ld16x2(t_acc + g * 16, acc, t_sum + g * 16, sum);
#pragma unroll
          for (int i = 0; i < 16; ++i) sum[i] += (uint32_t)__float2int_rn(__uint_as_float(acc[i]));
        } else {
          tmem_ld16(t_acc + g * 16, acc);
#pragma unroll
          for (int i = 0; i < 16; ++i) sum[i] = (uint32_t)__float2int_rn(__uint_as_float(acc[i]));
        }
        tmem_st16_async(t_sum + g * 16, sum);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.acc_empty);
      if (dr_c == cpt - 1) epilogue<AU, BU, MMI>(p, sm, tbase, dr_tl, q, h, lane, c_vec);
      // advance to the next chunk
      ++dr_d;
      if (++dr_c == cpt) {
        dr_c = 0;
        ++dr_tl;
      }
      dr_last = dr_tl * spt + min((dr_c + 1) * cs, spt) - 1;
      return true;
    };

    // One producer step: prefetch stage g+2 into `nxt`, then convert and publish stage g from `cur`.
    auto step = [&](int g) -> bool {
      uint4 cur[6];
      if (VEC) {
        const int is = g & (NI - 1);
        if (!mbar_wait(&sm.i8_full[is], (uint32_t)((g / NI) & 1), &sm.abort_flag, p.err, SITE_I8_FULL)) return false;
        const uint32_t src = i8base + (uint32_t)is * I8_STAGE;
        cur[0] = ld_shared_v4(src + ia0);
        cur[1] = ld_shared_v4(src + ia0 + 64u * 64u);
#pragma unroll
        for (int j = 0; j < 4; ++j) cur[2 + j] = ld_shared_v4(src + ib0 + (uint32_t)j * 16u * 256u);
        // The slot is released only after these registers have been consumed
        // (below), so no read of it can still be in flight when TMA refills it.
      } else {
        load_pieces<false>(p, lc, t, cur);
        cursor_advance(p, spt, t, lc);
      }
      const int slot = g & (NS - 1);
      if (g >= NS) {
        if (!mbar_wait(&sm.empty[slot], (uint32_t)(((g / NS) - 1) & 1), &sm.abort_flag, p.err, SITE_EMPTY))
          return false;
      }
      store_stage<AU, BU>(sbase + (uint32_t)slot * STAGE_BYTES, so, cur);
      fence_proxy_async_smem();
      mbar_arrive(&sm.full[slot]);
      if (VEC) mbar_arrive(&sm.i8_empty[g & (NI - 1)]);   // int8 bytes consumed: TMA may refill the slot

      if (st_s == 0) {
        // Stage this tile's per-column and per-row epilogue operands; the
        // epilogue reads them after the whole K loop, so the loads are hidden.
        const TileCoord tc = tile_coord(p, st_tl);
        const int ring = st_tl % SUM_RING;
        const int n = tc.n0 + t;
        const int m = tc.m0 + (t & (BM - 1));
        if (!MMI) {
          sm.col_op[ring][t] = __float_as_uint(n < p.N ? __ldg(p.w_scale + (p.w_count == 1 ? 0 : n)) : 0.f);
          if (t < BM)
            sm.row_op[ring][t] = __float_as_uint(m < p.M ? __ldg(p.act_scale + (p.act_count == 1 ? 0 : m % p.zp_row_mod)) : 0.f);
        } else {
          uint32_t zb = 0u, za = 0u;
          if (p.b_zp_count > 0 && n < p.N) {
            const int zi = p.b_zp_count == 1 ? 0 : n;
            zb = BU ? (uint32_t)__ldg((const uint8_t*)p.b_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.b_zp + zi);
          }
          sm.col_op[ring][t] = zb;
          if (t < BM) {
            if (p.a_zp_count > 0 && m < p.M) {
              const int zi = p.a_zp_count == 1 ? 0 : m % p.zp_row_mod;
              za = AU ? (uint32_t)__ldg((const uint8_t*)p.a_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.a_zp + zi);
            }
            sm.row_op[ring][t] = za;
          }
        }
      }
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
        // A 16-bit lane holds at most 257 additions of 255. Combining the two lanes
        // of a column doubles the count, so fold every 32 stages (2 lanes x 4 rows
        // x 32 stages = 256 additions) and at the tile end into the owner's 32-bit
        // slots in shared memory.
        if ((st_s & 31) == 31 || st_s == spt - 1) {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint32_t e = ce[qq] + __shfl_xor_sync(0xffffffffu, ce[qq], 4);   // lanes of both k-row parities
            const uint32_t o = co[qq] + __shfl_xor_sync(0xffffffffu, co[qq], 4);
            ce[qq] = 0u;
            co[qq] = 0u;
            if (cs_owner) {
              int* dst = &sm.part[warp][b_nq(t) * 16 + 4 * qq];
              dst[0] += (int)(e & 0xFFFFu);
              dst[2] += (int)(e >> 16);
              dst[1] += (int)(o & 0xFFFFu);
              dst[3] += (int)(o >> 16);
            }
          }
        }
      }
      if (st_s == spt - 1) {
        // Tile finished: reduce this tile's row and column sums into shared memory,
        // and make them and the staged epilogue operands visible to all workers.
        const int ring = st_tl % SUM_RING;
        if (need_rs) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            int v = rs_acc[j];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if ((t & 3) == 0) sm.rowsum[ring][a_row(t, j)] = v;
            rs_acc[j] = 0;
          }
        }
        if (need_cs) {
          if (!worker_sync(sm, red_phase, p.err)) return false;
          // every byte added was biased by +128 (signed B): 2 lanes x 4 rows per stage
          int v = BU ? 0 : -(128 * 2 * 4 * spt) * NWW;
#pragma unroll
          for (int w = 0; w < NWW; ++w) v += sm.part[w][t];
          sm.colsum[ring][t] = v;
        }
        if (!worker_sync(sm, red_phase, p.err)) return false;
        if (need_cs && cs_owner) {   // everyone has read sm.part: clear this lane's slots for the next tile
#pragma unroll
          for (int i = 0; i < 16; ++i) sm.part[warp][b_nq(t) * 16 + i] = 0;
        }
      }
      if (++st_s == spt) {
        st_s = 0;
        ++st_tl;
      }
      return true;
    };

    // After the last stage, the remaining chunks are drained by the same call site.
    for (int g = 0; ok && (g < total_stages || dr_d < total_chunks); ++g) {
      if (g < total_stages) ok = step(g);
      while (ok && dr_d < total_chunks && (g >= total_stages || dr_last + LOOKAHEAD <= g)) ok = drain();
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
cudaError_t launch_one(const GemmArgs& a, int cs, int c_vec, const CUtensorMap& ta, const CUtensorMap& tb,
                       cudaStream_t s) {
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
  kern<<<grid, NT, SMEM_BYTES, s>>>(a, cs, c_vec, ta, tb);
  return cudaGetLastError();
}

// Tensor maps of the int8 operands for the TMA producer: A as {K, M, batch}
// (box 64 x 128), B as {N, K, batch} (box 256 x 64); a batch stride of 0 is a
// single matrix shared by every batch.
cudaError_t make_operand_maps(const GemmArgs& a, CUtensorMap* ta, CUtensorMap* tb) {
  const uint64_t ab = a.a_bstride ? (uint64_t)a.batch : 1, bb = a.b_bstride ? (uint64_t)a.batch : 1;
  const uint64_t as = a.a_bstride ? (uint64_t)a.a_bstride : (uint64_t)a.M * a.K;
  const uint64_t bs = a.b_bstride ? (uint64_t)a.b_bstride : (uint64_t)a.K * a.N;
  cudaError_t e = make_tmap_3d(ta, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)a.K, (uint64_t)a.M, ab,
                               (uint64_t)a.K, as, BK, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return make_tmap_3d(tb, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)a.N, (uint64_t)a.K, bb, (uint64_t)a.N, bs, BN,
                      BK, CU_TENSOR_MAP_SWIZZLE_NONE);
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
  // Large aligned problems run on SM pairs (half of B per SM in shared memory).
  if (vec && a.M >= 256) return launch_gemm_tc_pair(a, a_u8, b_u8, mmi, chunk_k, c_vec, s, kernel_name);
  CUtensorMap ta{}, tb{};
  if (vec) {
    const cudaError_t e = make_operand_maps(a, &ta, &tb);
    if (e != cudaSuccess) return e;
  }
  if (!mmi) {
    *kernel_name = vec ? "gemm_tc05_exact_a8w8" : "gemm_tc05_exact_a8w8_bytewise";
    return vec ? launch_one<false, false, false, true>(a, cs, c_vec, ta, tb, s)
               : launch_one<false, false, false, false>(a, cs, c_vec, ta, tb, s);
  }
  *kernel_name = vec ? "gemm_tc05_exact_matmul_integer" : "gemm_tc05_exact_matmul_integer_bytewise";
#define QMM_DISPATCH(AU, BU)                                                                   \
  if (a_u8 == AU && b_u8 == BU)                                                                \
    return vec ? launch_one<AU, BU, true, true>(a, cs, c_vec, ta, tb, s)                      \
               : launch_one<AU, BU, true, false>(a, cs, c_vec, ta, tb, s);
  QMM_DISPATCH(false, false)
  QMM_DISPATCH(true, false)
  QMM_DISPATCH(false, true)
  QMM_DISPATCH(true, true)
#undef QMM_DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace qmm
