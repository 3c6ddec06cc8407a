// Exact 8-bit x 8-bit GEMM on a pair of SMs (tcgen05 cta_group::2), with the
// dequantisation fused into the epilogue. Same arithmetic as gemm_tc.cu: the
// bytes become exact fp16 values, tcgen05.mma kind::f16 accumulates exact fp32
// sums over K-chunks no longer than 2^24 / max|product|, and each chunk is
// folded into wrapping int32 sums in TMEM (the INT32 accumulator of PyPTO PR
// #1920's sequence diagram; the wrapping int32 of MatMulInteger in ROCm hip-ep
// PR #1248, "What"). The epilogues are the A8W8 row-then-column scaling and the
// MatMulInteger zero-point expansion
//   sum_k (a-za)(b-zb) = acc - za*colsum(B)[n] - zb*rowsum(A)[m] + K*za*zb.
//
// Why a pair: on sm_103a the conversion to fp16 makes shared memory, not the
// tensor core, the limit of the single-SM kernel (each SM stages, reads,
// writes and feeds to the MMA all of its 256-column B tile). In a pair tile of
// 256 x 256 outputs each CTA owns 128 rows of A and 128 columns of B; one MMA
// of M=256 reads A from each CTA and both halves of B, and each CTA's TMEM
// holds its own 128 rows x 256 columns. Per 64-deep K stage an SM therefore
// moves 96 KB through shared memory instead of 144 KB for the same MACs.
//
// CTA organisation (cluster of 2 CTAs, 576 threads each, one CTA per SM):
//  * warp 17 (producer): TMA copies of this CTA's int8 A rows (128 x 64) and
//    B columns (64 x 128) into a 4-stage staging ring.
//  * warps 0-15 (workers): convert staged bytes to fp16 in the canonical
//    128-byte-swizzled layouts (A K-major, B MN-major), 4-stage ring; the row
//    sums of their A rows and the column sums of their B columns; drain the
//    TMEM accumulator after each K-chunk; run the epilogue and store C.
//  * warp 16: allocates TMEM for the pair (with the peer's warp 16); in the even
//    CTA, one lane issues the pair MMAs (M=256, N=256, K=16) and the commits,
//    which arrive on the barriers of both CTAs.
// A stage is published to the MMA by one arrival per worker warp of either
// CTA on the even CTA's `full` barrier; chunk drains likewise arrive on the
// even CTA's `acc_empty`. Those arrivals release at CTA scope: each hands over
// shared memory of the arriving CTA, already made visible to the async proxy
// (the tensor core) by fence.proxy.async, or TMEM reads already waited for.
// MatMulInteger's column sums are exchanged between the two CTAs once per tile
// through distributed shared memory (cluster-scope release), guarded by a
// full/empty barrier pair. Every wait is bounded (see common.cuh).
#include "common.cuh"
#include "kernels.h"
#include "tma.h"

#include <algorithm>
#include <cstdlib>
#include <mutex>

namespace qmm {
namespace gemm2 {

constexpr int BM = 128;                // A rows per CTA
constexpr int BMP = 2 * BM;            // rows per pair tile
constexpr int BN = 256;                // columns per pair tile
constexpr int BNH = BN / 2;            // B columns staged by each CTA
constexpr int BK = 64;
constexpr int NS = 4;                  // fp16 stages read by the MMA
constexpr int NI = 4;                  // int8 staging stages filled by TMA
constexpr int LOOKAHEAD = NS - 1;      // stages produced past a chunk before it is drained
constexpr int NWW = 16;                // worker warps
constexpr int NW = NWW * 32;
constexpr int NT = NW + 64;            // + MMA warp + TMA producer warp
constexpr int PPT = 512 / NW;          // 16-byte pieces of A, and of B, per worker thread per stage
constexpr int CPW = 1024 / NWW;        // accumulator columns per worker warp in drains and epilogues
constexpr int A_BYTES = BM * BK * 2;   // fp16 A: 16 KB
constexpr int B_BYTES = BK * BNH * 2;  // fp16 B half: 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int I8_A = BM * BK;          // 8 KB
constexpr int I8_B = BK * BNH;         // 8 KB
constexpr int I8_STAGE = I8_A + I8_B;
constexpr int SUM_RING = LOOKAHEAD + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SUM_COL = 256;      // TMEM columns [256, 512): running int32 sums
constexpr int PAIR_ARRIVALS = 2 * NWW; // one arrival per worker warp of both CTAs
static_assert((NS & (NS - 1)) == 0 && (NI & (NI - 1)) == 0, "ring sizes are powers of two");
static_assert(NWW == 8 || NWW == 16, "worker warps: 8 or 16");

struct Shared {
  int part[NWW][BNH];               // column-sum partials of this CTA's B half, per warp
  int rowsum[SUM_RING][BM];
  int colsum[SUM_RING][BN];         // both halves: this CTA's and the peer's
  uint32_t col_op[SUM_RING][BN];    // weight_scale[n] bits or b_zp[n]
  uint32_t row_op[SUM_RING][BM];    // act_scale[m] bits or a_zp[m]
  uint64_t full[NS];                // used in the even CTA: PAIR_ARRIVALS per phase
  uint64_t empty[NS];               // completed by the pair's commit
  uint64_t i8_full[NI];
  uint64_t i8_empty[NI];
  uint64_t acc_full;                // completed by the pair's commit
  uint64_t acc_empty;               // used in the even CTA: PAIR_ARRIVALS per phase
  uint64_t cs_full[SUM_RING];       // column sums of a tile present: 2 x BNH thread arrivals
  uint64_t cs_empty[SUM_RING];      // both epilogues done with a slot: PAIR_ARRIVALS
  uint64_t red_bar;
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = (size_t)NS * STAGE_BYTES + (size_t)NI * I8_STAGE + sizeof(Shared) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

enum : unsigned {
  SITE_EMPTY = 0x300, SITE_FULL = 0x301, SITE_ACC_FULL = 0x302, SITE_ACC_EMPTY = 0x303, SITE_RED = 0x304,
  SITE_TEARDOWN = 0x305, SITE_I8_FULL = 0x306, SITE_I8_EMPTY = 0x307, SITE_I8_DRAIN = 0x308,
  SITE_CS_FULL = 0x309, SITE_CS_EMPTY = 0x30a, SITE_FINAL = 0x30b
};

struct TileCoord {
  int b, m0, n0;   // m0: this CTA's first row; n0: the pair tile's first column
};

__device__ __forceinline__ TileCoord tile_coord(const GemmArgs& p, int tile_local, int cid, int ncl, int rank) {
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

// Piece assignment of worker thread t (0..NW-1) in one 64-deep K stage: the
// stage holds 512 pieces of 16 bytes of A and 512 of B; each thread takes PPT
// of each.
//  A: rows t/4 + j*NW/4, k bytes (t%4)*16. A quarter-warp reads rows 2p, 2p+1
//     (64-byte staging rows: 8 distinct bank groups) and writes 8 distinct
//     swizzle slots.
//  B (the 64 x 128 half): k rows 2*(t/16) + (t/4)%2 + j*NW/8, columns 16*nq
//     with nq = (t%8) ^ 4*((t/8)%2). A quarter-warp reads 8 different 16-byte
//     columns of two 128-byte staging rows (8 bank groups) and writes, for two
//     consecutive k rows, 4 chunk pairs each, which the swizzle puts in 8
//     distinct slots: both shared-memory sides are free of bank conflicts.
__device__ __forceinline__ int a_row(int t, int j) { return (t >> 2) + (NW / 4) * j; }
__device__ __forceinline__ int a_kq(int t) { return t & 3; }
__device__ __forceinline__ int b_nq(int t) { return (t & 7) ^ (((t >> 3) & 1) << 2); }
__device__ __forceinline__ int b_krow(int t, int j) { return 2 * (t >> 4) + ((t >> 2) & 1) + (NW / 8) * j; }
// byte steps between a thread's pieces: int8 staging (A, B) and fp16 stage (A, B)
constexpr uint32_t I8_A_STEP = (NW / 4) * 64u, I8_B_STEP = (NW / 8) * 128u;
constexpr uint32_t F16_A_STEP = (NW / 4) * 128u, F16_B_STEP = (NW / 8) * 256u;

// Shared-memory byte offsets (within a stage) of this thread's first A and B
// pieces, chunks 0 and 1; piece j of each is j * F16_A_STEP / F16_B_STEP further.
//  A: K-major, 128-byte swizzle: row r is 128 bytes (64 fp16 along K), 8-row
//     groups form 1024-byte atoms, 16-byte chunk c of row r sits at c ^ (r % 8).
//  B: MN-major, 128-byte swizzle: atom (k/8, n/64) at (k/8)*2048 + (n/64)*1024,
//     chunk c = (n%64)/8 of row k%8 at c ^ (k % 8).
struct StoreOffsets {
  uint32_t a0, a1, b0, b1;
};

__device__ __forceinline__ StoreOffsets store_offsets(int t) {
  StoreOffsets o;
  const int r = a_row(t, 0);
  const uint32_t rb = (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
  o.a0 = rb + ((uint32_t)((a_kq(t) * 2 + 0) ^ (r & 7)) << 4);
  o.a1 = rb + ((uint32_t)((a_kq(t) * 2 + 1) ^ (r & 7)) << 4);
  const int nq = b_nq(t);
  const int k = b_krow(t, 0);
  const uint32_t kb = (uint32_t)A_BYTES + (uint32_t)(k >> 3) * 2048u + (uint32_t)(nq >> 2) * 1024u +
                      (uint32_t)(k & 7) * 128u;
  o.b0 = kb + ((uint32_t)(((nq & 3) * 2 + 0) ^ (k & 7)) << 4);
  o.b1 = kb + ((uint32_t)(((nq & 3) * 2 + 1) ^ (k & 7)) << 4);
  return o;
}

template <bool AU, bool BU>
__device__ __forceinline__ void store_stage(uint32_t base, const StoreOffsets& o, const uint4 (&v)[2 * PPT]) {
#pragma unroll
  for (int j = 0; j < 2 * PPT; ++j) {
    uint32_t hv[8];
    const bool isa = j < PPT;
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
    const uint32_t off = isa ? (uint32_t)j * F16_A_STEP : (uint32_t)(j - PPT) * F16_B_STEP;
    st_shared_v4(base + (isa ? o.a0 : o.b0) + off, hv[0], hv[1], hv[2], hv[3]);
    st_shared_v4(base + (isa ? o.a1 : o.b1) + off, hv[4], hv[5], hv[6], hv[7]);
  }
}

template <bool U>
__device__ __forceinline__ int dp4a_ones(uint32_t w, int acc) {
  if (U) return (int)__dp4a(w, 0x01010101u, (unsigned)acc);
  return __dp4a((int)w, 0x01010101, acc);
}

__device__ __forceinline__ bool worker_sync(Shared& sm, int& phase, unsigned* err) {
  mbar_arrive(&sm.red_bar);
  const bool ok = mbar_wait(&sm.red_bar, (uint32_t)(phase & 1), &sm.abort_flag, err, SITE_RED);
  ++phase;
  return ok;
}

// Epilogue of one tile (this CTA's 128 rows x 256 columns): read the final
// int32 sums from TMEM (this warp's 32 rows, its CPW-column slice, 16 columns
// at a time), apply the fused dequantisation / zero-point correction, store C.
template <bool AU, bool BU, bool MMI>
__device__ __noinline__ void epilogue(const GemmArgs& p, Shared& sm, uint32_t tbase, const TileCoord tc, int tile_local,
                                      int q, int h, int lane, int c_vec, bool need_cs, uint32_t peer) {
  const int slot = tile_local % SUM_RING;
  const int rloc = q * 32 + lane;
  const int row = tc.m0 + rloc;
  const bool row_ok = row < p.M;
  const uint32_t lane_off = (uint32_t)(q * 32) << 16;
  const size_t crow = ((size_t)tc.b * p.M + (size_t)(row_ok ? row : 0)) * (size_t)p.N;
  const uint64_t pol = l2_policy_evict_first();
  bool cs_ok = true;
  if (need_cs)
    cs_ok = mbar_wait_cluster(&sm.cs_full[slot], (uint32_t)((tile_local / SUM_RING) & 1), &sm.abort_flag, p.err,
                              SITE_CS_FULL);

  uint32_t hold[16];
  const float as = __uint_as_float(sm.row_op[slot][rloc]);
  const uint32_t za = sm.row_op[slot][rloc];
  const uint32_t rs = (MMI && p.b_zp_count > 0) ? (uint32_t)sm.rowsum[slot][rloc] : 0u;

#pragma unroll 1
  for (int g = 0; g < CPW / 16; ++g) {
    uint32_t tot[16];
    if ((g & 1) == 0) {
      uint32_t t32[32];
      tmem_ld32(tbase + lane_off + SUM_COL + (uint32_t)(h * CPW + g * 16), t32);   // warp-collective
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        tot[i] = t32[i];
        hold[i] = t32[16 + i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) tot[i] = hold[i];
    }
    const int nb = tc.n0 + h * CPW + g * 16;
    if (!row_ok || nb >= p.N || !cs_ok) continue;
    const bool full = (nb + 16 <= p.N) && c_vec;
    uint32_t o[16];
    if (!MMI) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float ws = __uint_as_float(sm.col_op[slot][h * CPW + g * 16 + i]);
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
        const uint32_t zb = sm.col_op[slot][h * CPW + g * 16 + i];
        const uint32_t cs = (p.a_zp_count > 0) ? (uint32_t)sm.colsum[slot][h * CPW + g * 16 + i] : 0u;
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
  if (need_cs) {
    // this warp is done with the slot's column sums, in this CTA's copy; tell both CTAs
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_cluster(smem_u32(&sm.cs_empty[slot]));
      mbar_arrive_cluster(mapa_shared(smem_u32(&sm.cs_empty[slot]), peer));
    }
  }
}

template <bool AU, bool BU, bool MMI>
__global__ void __launch_bounds__(NT, 1)
    gemm_tc2_kernel(const GemmArgs p, const int cs, const int c_vec, const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sbase_ptr = smem_raw + (sbase - raw);
  const uint32_t i8base = sbase + NS * STAGE_BYTES;
  Shared& sm = *reinterpret_cast<Shared*>(sbase_ptr + NS * STAGE_BYTES + NI * I8_STAGE);

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
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
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm.full[i], PAIR_ARRIVALS);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < NI; ++i) {
      mbar_init(&sm.i8_full[i], 1);
      mbar_init(&sm.i8_empty[i], NWW);
    }
    for (int i = 0; i < SUM_RING; ++i) {
      mbar_init(&sm.cs_full[i], 2 * BNH);
      mbar_init(&sm.cs_empty[i], PAIR_ARRIVALS);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, PAIR_ARRIVALS);
    mbar_init(&sm.red_bar, NW);
    mbar_init(&sm.teardown, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == NWW) {
    tmem_alloc_pair(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();   // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;

  if (warp == NWW) {
    // ---------------- pair MMA issuer (even CTA) ----------------
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = idesc_f16_f32(BMP, BN, false, true);
      int g = 0;
      int d = 0;
      bool ok = true;
      for (int tl = 0; tl < my_tiles && ok; ++tl) {
        for (int c = 0; c < cpt && ok; ++c) {
          if (d > 0) {
            ok = mbar_wait_cluster(&sm.acc_empty, (uint32_t)((d - 1) & 1), &sm.abort_flag, p.err, SITE_ACC_EMPTY);
            if (!ok) break;
          }
          tc_fence_after();
          const int s_beg = c * cs;
          const int s_end = min(spt, s_beg + cs);
          for (int s = s_beg; s < s_end; ++s, ++g) {
            const int slot = g & (NS - 1);
            ok = mbar_wait_cluster(&sm.full[slot], (uint32_t)((g / NS) & 1), &sm.abort_flag, p.err, SITE_FULL);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_addr = sbase + (uint32_t)slot * STAGE_BYTES;
            const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              const uint64_t ad = sdesc_sw128(a_addr + (uint32_t)j * 32u, 16u, 1024u);
              const uint64_t bd = sdesc_sw128(b_addr + (uint32_t)j * 4096u, 1024u, 2048u);
              tc_mma_f16_pair(tbase, ad, bd, idesc, (s > s_beg || j > 0) ? 1u : 0u);
            }
            tc_commit_pair_mc(&sm.empty[slot], 0x3);
          }
          if (!ok) break;
          tc_commit_pair_mc(&sm.acc_full, 0x3);
          ++d;
        }
      }
    }
    __syncwarp();
  } else if (warp == NWW + 1) {
    // ---------------- TMA producer: this CTA's int8 A rows and B columns ----------------
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int tl = 0, s = 0, g = 0;
      TileCoord tc = tile_coord(p, 0, cid, ncl, (int)rank);
      for (; g < total_stages; ++g) {
        const int slot = g & (NI - 1);
        if (g >= NI &&
            !mbar_wait(&sm.i8_empty[slot], (uint32_t)(((g / NI) - 1) & 1), &sm.abort_flag, p.err, SITE_I8_EMPTY))
          break;
        const uint32_t dst = i8base + (uint32_t)slot * I8_STAGE;
        mbar_arrive_expect_tx(&sm.i8_full[slot], I8_STAGE);
        tma_load_3d(dst, &tmA, s * BK, tc.m0, p.a_bstride ? tc.b : 0, &sm.i8_full[slot]);
        tma_load_3d(dst + I8_A, &tmB, tc.n0 + (int)rank * BNH, s * BK, p.b_bstride ? tc.b : 0, &sm.i8_full[slot]);
        if (++s == spt) {
          s = 0;
          tc = tile_coord(p, ++tl, cid, ncl, (int)rank);
        }
      }
      for (int j = (g > NI ? g - NI : 0); j < g; ++j)
        mbar_wait(&sm.i8_full[j & (NI - 1)], (uint32_t)((j / NI) & 1), nullptr, p.err, SITE_I8_DRAIN);
    }
    __syncwarp();
  } else {
    // ---------------- workers ----------------
    const int q = warp & 3;
    const int h = warp >> 2;     // column slice [h*CPW, (h+1)*CPW) of the tile
    const bool need_rs = MMI && p.b_zp_count > 0;
    const bool need_cs = MMI && p.a_zp_count > 0;
    const uint32_t full_leader0 = mapa_shared(smem_u32(&sm.full[0]), 0);
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(&sm.acc_empty), 0);
    int red_phase = 0;
    bool ok = true;

    int dr_d = 0, dr_tl = 0, dr_c = 0;
    int dr_last = min(cs, spt) - 1;

    int rs_acc[PPT];
#pragma unroll
    for (int j = 0; j < PPT; ++j) rs_acc[j] = 0;
    uint32_t ce[4] = {0u, 0u, 0u, 0u}, co[4] = {0u, 0u, 0u, 0u};
    // Column sums of this CTA's B half accumulate in sm.part[warp][column]:
    // lanes 0-7 own the 16 columns b_nq(lane)*16.. of their warp's row.
    const bool cs_owner = lane < 8;
    if (need_cs && cs_owner) {
#pragma unroll
      for (int i = 0; i < 16; ++i) sm.part[warp][b_nq(t) * 16 + i] = 0;
    }

    const StoreOffsets so = store_offsets(t);
    const uint32_t ia0 = (uint32_t)a_row(t, 0) * 64u + (uint32_t)a_kq(t) * 16u;
    const uint32_t ib0 = (uint32_t)I8_A + (uint32_t)b_krow(t, 0) * 128u + (uint32_t)b_nq(t) * 16u;
    int st_tl = 0, st_s = 0;

    auto drain = [&]() -> bool {
      if (!mbar_wait_cluster(&sm.acc_full, (uint32_t)(dr_d & 1), &sm.abort_flag, p.err, SITE_ACC_FULL))
        return false;
      tc_fence_after();
      const uint32_t lane_off = (uint32_t)(q * 32) << 16;
      const uint32_t t_acc = tbase + lane_off + (uint32_t)(h * CPW);
      const uint32_t t_sum = t_acc + SUM_COL;
#pragma unroll 1
      for (int g = 0; g < CPW / 16; ++g) {
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
      __syncwarp();
      if (lane == 0) mbar_arrive_remote_cta(acc_empty_leader);
      if (dr_c == cpt - 1)
        epilogue<AU, BU, MMI>(p, sm, tbase, tile_coord(p, dr_tl, cid, ncl, (int)rank), dr_tl, q, h, lane, c_vec,
                              need_cs, peer);
      ++dr_d;
      if (++dr_c == cpt) {
        dr_c = 0;
        ++dr_tl;
      }
      dr_last = dr_tl * spt + min((dr_c + 1) * cs, spt) - 1;
      return true;
    };

    auto step = [&](int g) -> bool {
      uint4 cur[2 * PPT];
      const int is = g & (NI - 1);
      if (!mbar_wait(&sm.i8_full[is], (uint32_t)((g / NI) & 1), &sm.abort_flag, p.err, SITE_I8_FULL)) return false;
      const uint32_t src = i8base + (uint32_t)is * I8_STAGE;
#pragma unroll
      for (int j = 0; j < PPT; ++j) {
        cur[j] = ld_shared_v4(src + ia0 + (uint32_t)j * I8_A_STEP);
        cur[PPT + j] = ld_shared_v4(src + ib0 + (uint32_t)j * I8_B_STEP);
      }
      const int slot = g & (NS - 1);
      if (g >= NS) {
        if (!mbar_wait_cluster(&sm.empty[slot], (uint32_t)(((g / NS) - 1) & 1), &sm.abort_flag, p.err, SITE_EMPTY))
          return false;
      }
      store_stage<AU, BU>(sbase + (uint32_t)slot * STAGE_BYTES, so, cur);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_remote_cta(full_leader0 + (uint32_t)slot * 8u);
        mbar_arrive(&sm.i8_empty[is]);   // the warp's int8 bytes are consumed: TMA may refill the slot
      }

      if (st_s == 0) {
        const TileCoord tc = tile_coord(p, st_tl, cid, ncl, (int)rank);
        const int ring = st_tl % SUM_RING;
        const int n = tc.n0 + t;
        const int m = tc.m0 + (t & (BM - 1));
        if (!MMI) {
          if (t < BN)
            sm.col_op[ring][t] = __float_as_uint(n < p.N ? __ldg(p.w_scale + (p.w_count == 1 ? 0 : n)) : 0.f);
          if (t < BM)
            sm.row_op[ring][t] =
                __float_as_uint(m < p.M ? __ldg(p.act_scale + (p.act_count == 1 ? 0 : m % p.zp_row_mod)) : 0.f);
        } else {
          uint32_t zb = 0u, za = 0u;
          if (p.b_zp_count > 0 && n < p.N && t < BN) {
            const int zi = p.b_zp_count == 1 ? 0 : n;
            zb = BU ? (uint32_t)__ldg((const uint8_t*)p.b_zp + zi) : (uint32_t)(int)__ldg((const int8_t*)p.b_zp + zi);
          }
          if (t < BN) sm.col_op[ring][t] = zb;
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
        for (int j = 0; j < PPT; ++j) {
          rs_acc[j] = dp4a_ones<AU>(cur[j].x, rs_acc[j]);
          rs_acc[j] = dp4a_ones<AU>(cur[j].y, rs_acc[j]);
          rs_acc[j] = dp4a_ones<AU>(cur[j].z, rs_acc[j]);
          rs_acc[j] = dp4a_ones<AU>(cur[j].w, rs_acc[j]);
        }
      }
      if (need_cs) {
#pragma unroll
        for (int j = 0; j < PPT; ++j) {
          const uint32_t w[4] = {cur[PPT + j].x, cur[PPT + j].y, cur[PPT + j].z, cur[PPT + j].w};
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint32_t u = BU ? w[qq] : (w[qq] ^ 0x80808080u);
            ce[qq] += prmt(u, 0u, 0x4240u);   // bytes 0 and 2 into 16-bit lanes
            co[qq] += prmt(u, 0u, 0x4341u);   // bytes 1 and 3
          }
        }
        // A 16-bit lane holds at most 257 additions of 255. The four lanes of a
        // warp that share columns (lane ^ 12, ^ 16, ^ 28) are combined before the
        // fold, so fold every 32 stages (4 lanes x PPT <= 2 pieces x 32 stages
        // <= 256 additions) and at the tile end.
        if ((st_s & 31) == 31 || st_s == spt - 1) {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            uint32_t e = ce[qq] + __shfl_xor_sync(0xffffffffu, ce[qq], 12);
            uint32_t o = co[qq] + __shfl_xor_sync(0xffffffffu, co[qq], 12);
            e += __shfl_xor_sync(0xffffffffu, e, 16);
            o += __shfl_xor_sync(0xffffffffu, o, 16);
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
        const int ring = st_tl % SUM_RING;
        if (need_rs) {
#pragma unroll
          for (int j = 0; j < PPT; ++j) {
            int v = rs_acc[j];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if ((t & 3) == 0) sm.rowsum[ring][a_row(t, j)] = v;
            rs_acc[j] = 0;
          }
        }
        if (need_cs) {
          if (!worker_sync(sm, red_phase, p.err)) return false;
          if (t < BNH) {
            // every byte added was biased by +128 (signed B), one per k row of the tile
            int v = BU ? 0 : -(128 * BK * spt);
#pragma unroll
            for (int w = 0; w < NWW; ++w) v += sm.part[w][t];
            // both CTAs' epilogues of the tile SUM_RING tiles back must be done with this slot
            if (st_tl >= SUM_RING &&
                !mbar_wait_cluster(&sm.cs_empty[ring], (uint32_t)(((st_tl / SUM_RING) - 1) & 1), &sm.abort_flag,
                                   p.err, SITE_CS_EMPTY))
              return false;
            const int col = (int)rank * BNH + t;
            sm.colsum[ring][col] = v;
            st_shared_cluster_u32(mapa_shared(smem_u32(&sm.colsum[ring][col]), peer), (uint32_t)v);
            mbar_arrive(&sm.cs_full[ring]);
            mbar_arrive_cluster(mapa_shared(smem_u32(&sm.cs_full[ring]), peer));
          }
        }
        if (!worker_sync(sm, red_phase, p.err)) return false;
        if (need_cs && cs_owner) {
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

    for (int g = 0; ok && (g < total_stages || dr_d < total_chunks); ++g) {
      if (g < total_stages) ok = step(g);
      while (ok && dr_d < total_chunks && (g >= total_stages || dr_last + LOOKAHEAD <= g)) ok = drain();
    }
    // The pair's commits of the last stages also arrive on this CTA's `empty`
    // barriers: let them land before the CTA may leave.
    for (int g = (total_stages > NS ? total_stages - NS : 0); ok && g < total_stages; ++g)
      ok = mbar_wait_cluster(&sm.empty[g & (NS - 1)], (uint32_t)((g / NS) & 1), &sm.abort_flag, p.err, SITE_FINAL);
    tc_fence_before();
  }

  __syncthreads();
  if (t == 0 && sm.abort_flag) st_shared_cluster_u32(mapa_shared(smem_u32(&sm.abort_flag), peer), 1u);
  if (warp == NWW && rank == 0) {
    // every pair MMA this CTA issued has completed before the pair frees TMEM
    tc_fence_after();
    if (lane == 0) {
      tc_commit_pair_mc(&sm.teardown, 0x1);
      mbar_wait(&sm.teardown, 0u, nullptr, p.err, SITE_TEARDOWN);
    }
    __syncwarp();
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == NWW) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, TMEM_COLS);
  }
}

struct DeviceLaunchInfo {
  bool attr_set = false;
  int max_clusters = 0;
};

template <bool AU, bool BU, bool MMI>
cudaError_t launch_one(const GemmArgs& a, int cs, int c_vec, const CUtensorMap& ta, const CUtensorMap& tb,
                       cudaStream_t s) {
  auto kern = gemm_tc2_kernel<AU, BU, MMI>;
  static std::mutex mu;
  static DeviceLaunchInfo info[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, cs, c_vec, ta, tb);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Tensor maps of the int8 operands: A as {K, M, batch} with box 64 x 128 (a
// CTA's rows), B as {N, K, batch} with box 128 x 64 (a CTA's column half). A
// batch stride of 0 is a single matrix shared by every batch.
cudaError_t make_operand_maps(const GemmArgs& a, CUtensorMap* ta, CUtensorMap* tb) {
  const uint64_t ab = a.a_bstride ? (uint64_t)a.batch : 1, bb = a.b_bstride ? (uint64_t)a.batch : 1;
  const uint64_t as = a.a_bstride ? (uint64_t)a.a_bstride : (uint64_t)a.M * a.K;
  const uint64_t bs = a.b_bstride ? (uint64_t)a.b_bstride : (uint64_t)a.K * a.N;
  cudaError_t e = make_tmap_3d(ta, a.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)a.K, (uint64_t)a.M, ab,
                               (uint64_t)a.K, as, BK, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return make_tmap_3d(tb, a.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)a.N, (uint64_t)a.K, bb, (uint64_t)a.N, bs,
                      BNH, BK, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace gemm2

cudaError_t launch_gemm_tc_pair(const GemmArgs& a, bool a_u8, bool b_u8, bool mmi, int chunk_k, int c_vec,
                                cudaStream_t s, const char** kernel_name) {
  using namespace gemm2;
  const int cs = chunk_k / BK;
  CUtensorMap ta{}, tb{};
  cudaError_t e = make_operand_maps(a, &ta, &tb);
  if (e != cudaSuccess) return e;
  if (!mmi) {
    *kernel_name = "gemm_tc05_pair_exact_a8w8";
    return launch_one<false, false, false>(a, cs, c_vec, ta, tb, s);
  }
  *kernel_name = "gemm_tc05_pair_exact_matmul_integer";
  if (!a_u8 && !b_u8) return launch_one<false, false, true>(a, cs, c_vec, ta, tb, s);
  if (a_u8 && !b_u8) return launch_one<true, false, true>(a, cs, c_vec, ta, tb, s);
  if (!a_u8 && b_u8) return launch_one<false, true, true>(a, cs, c_vec, ta, tb, s);
  return launch_one<true, true, true>(a, cs, c_vec, ta, tb, s);
}

}  // namespace qmm
