// Decode-shaped form (a) for one or two activation rows on the CUDA cores
// (templates cover up to four):
//   C[m,n] = scale_n * (sum_k A[m,k]*W[k,n] - zp_n * sum_k A[m,k])
// (TrainDeeploy PR #53, "The kernel": the int8 weight is dequantised inside the
// kernel and the zero point is applied once per output through the row sum of
// A). The weight stream K*N is read once, so the kernel keeps HBM busy with
// copies that cost no registers and spends as few instructions per weight byte
// as it can, in one launch:
//  * clusters of two CTAs own 128-column blocks of W in turn (persistent); the
//    two CTAs of a pair take the two halves of K;
//  * in each CTA one producer warp streams stages of 256 weight rows x 128
//    columns and the matching 256 columns of A into a TMA ring;
//  * the consumer warps take rows of a stage: a lane owns 16 adjacent columns
//    (one 16-byte shared load per row); the bytes, biased to unsigned, go into
//    the low mantissa of 2^23 by one byte permute each, and one packed fp32
//    subtract per pair makes them exact floats; packed fp32 FMAs (f32x2)
//    accumulate a[m][k] * w two columns at a time;
//  * at the end of a column block each CTA reduces its warps in a fixed order;
//    the odd CTA hands its sums to the even one through distributed shared
//    memory, which adds them (K half 0, then half 1) and applies the zero point
//    and the scale. Results do not depend on timing.
// Every wait is bounded (see common.cuh).
#include "common.cuh"
#include "kernels.h"
#include "tma.h"

#include <algorithm>
#include <climits>
#include <mutex>

namespace qmm {
namespace gvs {

constexpr int kMaxRows = 4;
constexpr int kCols = 16;                      // columns per lane
constexpr int kBlockCols = 8 * kCols;          // 128 columns per column block (8 lanes across)
constexpr int kStageRows = 256;                // weight rows per stage
constexpr int kStages = 5;
constexpr int kWBytes = kStageRows * kBlockCols;   // 32 KB
constexpr int kABytes = kMaxRows * kStageRows * 4; // A slice, f32 worst case: 4 KB
constexpr int kStageBytes = kWBytes + kABytes;

// consumer warps: 16 for one or two activation rows (more warps to hide the
// conversion chain), 8 for four (their accumulators need the registers)
template <int MT>
__host__ __device__ constexpr int consumer_warps() { return MT <= 2 ? 16 : 8; }

enum : unsigned { SITE_FULL = 0x600, SITE_EMPTY = 0x601, SITE_DRAIN = 0x602, SITE_XFULL = 0x603, SITE_XEMPTY = 0x604 };

struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t xfull;     // even CTA: the odd CTA's sums have arrived (8 arrivals)
  uint64_t xempty;    // odd CTA: the even CTA has consumed them (8 arrivals)
  int abort_flag;
  float xsum[kMaxRows][kBlockCols];    // even CTA: the odd CTA's sums of the current column block
  float xrs[kMaxRows];                 // even CTA: the odd CTA's row sums of A
  float rs_warp[16][kMaxRows];
  unsigned long long red[16 * kMaxRows / 2][8][kCols / 2];   // [warp x rows][column lane][column pair]
};

constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + sizeof(Shared) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}

__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_addr, float v) {
  st_shared_cluster_u32(cluster_addr, __float_as_uint(v));
}

template <int CW>
__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory"); }

template <int MT, bool BF16>
__global__ void __launch_bounds__((consumer_warps<MT>() + 1) * 32, 1)
    gemv_pair_kernel(const GemvSimtArgs p, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmA, int k_half, unsigned* err) {
  constexpr int kCW = consumer_warps<MT>();
  constexpr int kRowsPerWarp = kStageRows / kCW;   // 16 or 32, in rounds of 4 (one per row lane group)
  constexpr int esz = BF16 ? 2 : 4;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  Shared& sm = *reinterpret_cast<Shared*>(smem_raw + (sbase - raw) + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x(), ncl = (int)nclusters_x();
  const int nblk = (p.N + kBlockCols - 1) / kBlockCols;
  const int k_lo = (int)rank * k_half, k_hi = min(p.K, k_lo + k_half);
  const int spb = k_hi > k_lo ? (k_hi - k_lo + kStageRows - 1) / kStageRows : 0;   // stages per column block
  const int my_blocks = cid < nblk ? (nblk - cid + ncl - 1) / ncl : 0;
  const int total = my_blocks * spb;
  const uint32_t a_bytes = (uint32_t)(kStageRows * p.M * esz);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kCW);
    }
    mbar_init(&sm.xfull, 8);
    mbar_init(&sm.xempty, 8);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  cluster_sync_all();   // both CTAs' barriers exist before any remote arrive

  if (warp == kCW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmA);
      int i = 0;
      for (; i < total; ++i) {
        const int slot = i % kStages;
        if (i >= kStages &&
            !mbar_wait(&sm.empty[slot], (uint32_t)(((i / kStages) - 1) & 1), &sm.abort_flag, err, SITE_EMPTY))
          break;
        const int cb = cid + (i / spb) * ncl, k = k_lo + (i % spb) * kStageRows;
        const uint32_t dst = sbase + (uint32_t)slot * kStageBytes;
        mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)kWBytes + a_bytes);
        tma_load_2d(dst, &tmW, cb * kBlockCols, k, &sm.full[slot]);
        tma_load_2d(dst + kWBytes, &tmA, k, 0, &sm.full[slot]);
      }
      // Before the CTA exits, wait (bounded) until every copy issued has landed.
      for (int j = (i > kStages ? i - kStages : 0); j < i; ++j)
        mbar_wait(&sm.full[j % kStages], (uint32_t)((j / kStages) & 1), nullptr, err, SITE_DRAIN);
    }
    __syncwarp();
  } else {
    // ---------------- consumers ----------------
    const int cs = lane & 7, rg = lane >> 3;   // column lane (16 columns), row lane group
    const unsigned long long bias = pack2(-8388736.f, -8388736.f);   // 2^23 + 128
    const uint32_t peer_xsum = mapa_shared(smem_u32(&sm.xsum[0][0]), 0);
    const uint32_t peer_xrs = mapa_shared(smem_u32(&sm.xrs[0]), 0);
    const uint32_t peer_xfull = mapa_shared(smem_u32(&sm.xfull), 0);
    const uint32_t peer_xempty = mapa_shared(smem_u32(&sm.xempty), 1);
    int it = 0;
    bool ok = true;
    for (int u = 0; u < my_blocks; ++u) {
      const int cb = cid + u * ncl;
      unsigned long long acc[MT][kCols / 2];
      float rs[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        rs[m] = 0.f;
#pragma unroll
        for (int j = 0; j < kCols / 2; ++j) acc[m][j] = 0ull;
      }
      for (int s = 0; s < spb; ++s, ++it) {
        const int slot = it % kStages;
        if (ok) ok = mbar_wait(&sm.full[slot], (uint32_t)((it / kStages) & 1), &sm.abort_flag, err, SITE_FULL);
        if (ok) {
          const uint32_t stage = sbase + (uint32_t)slot * kStageBytes;
#pragma unroll 2
          for (int rr = 0; rr < kRowsPerWarp; rr += 4) {
            const int r = warp * kRowsPerWarp + rr + rg;
            float a[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint32_t aa = stage + kWBytes + (uint32_t)((m * kStageRows + r) * esz);
              a[m] = m < p.M ? (BF16 ? __uint_as_float(lds_u16(aa) << 16) : __uint_as_float(lds_u32(aa))) : 0.f;
              rs[m] += a[m];
            }
            const uint4 w = ld_shared_v4(stage + (uint32_t)(r * kBlockCols + cs * kCols));
            const uint32_t uw[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
            unsigned long long v[kCols / 2];
#pragma unroll
            for (int j = 0; j < kCols / 2; ++j) {
              const uint32_t word = uw[j >> 1];
              const int b = (j & 1) * 2;
              const uint32_t lo = prmt(word, 0x4B000000u, 0x7440u | (uint32_t)b);
              const uint32_t hi = prmt(word, 0x4B000000u, 0x7440u | (uint32_t)(b + 1));
              v[j] = fadd2(((unsigned long long)hi << 32) | lo, bias);   // exact: two int8 values as floats
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const unsigned long long a2 = pack2(a[m], a[m]);
#pragma unroll
              for (int j = 0; j < kCols / 2; ++j) acc[m][j] = ffma2(a2, v[j], acc[m][j]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }
      // (1) the warp's four row groups, in a fixed order (xor 8, then 16)
#pragma unroll
      for (int o = 8; o <= 16; o <<= 1)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          rs[m] += __shfl_xor_sync(0xffffffffu, rs[m], o);
#pragma unroll
          for (int j = 0; j < kCols / 2; ++j) {
            const unsigned long long x = acc[m][j];
            const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)x, o);
            const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(x >> 32), o);
            acc[m][j] = fadd2(x, ((unsigned long long)hi << 32) | lo);
          }
        }
      // (2) the warps, in a fixed order, into warp 0 lanes 0..7
      consumer_bar<kCW>();   // the previous column block's reduction buffer has been read
      if (lane < 8) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int j = 0; j < kCols / 2; ++j) sm.red[warp * MT + m][lane][j] = acc[m][j];
      }
      if (lane == 0)
#pragma unroll
        for (int m = 0; m < MT; ++m) sm.rs_warp[warp][m] = rs[m];
      consumer_bar<kCW>();
      if (warp != 0) continue;   // warp 0 finishes the column block; lanes 0..7 hold its 128 columns
      const bool owner = lane < 8;
      if (owner) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
          for (int j = 0; j < kCols / 2; ++j) acc[m][j] = sm.red[m][lane][j];
          rs[m] = sm.rs_warp[0][m];
          for (int w = 1; w < kCW; ++w) {
#pragma unroll
            for (int j = 0; j < kCols / 2; ++j) acc[m][j] = fadd2(acc[m][j], sm.red[w * MT + m][lane][j]);
            rs[m] += sm.rs_warp[w][m];
          }
        }
      }
      // (3) the pair: the odd CTA hands its sums to the even CTA
      if (rank == 1) {
        if (u > 0 && ok)
          ok = mbar_wait_cluster(&sm.xempty, (uint32_t)((u - 1) & 1), &sm.abort_flag, err, SITE_XEMPTY);
        if (ok && owner) {
#pragma unroll
          for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int j = 0; j < kCols / 2; ++j) {
              const uint32_t at = peer_xsum + (uint32_t)((m * kBlockCols + lane * kCols + 2 * j) * 4);
              st_cluster_f32(at, __uint_as_float((uint32_t)acc[m][j]));
              st_cluster_f32(at + 4, __uint_as_float((uint32_t)(acc[m][j] >> 32)));
            }
            if (lane == 0) st_cluster_f32(peer_xrs + (uint32_t)(m * 4), rs[m]);
          }
        }
        if (owner) mbar_arrive_cluster(peer_xfull);   // releases the stores above at cluster scope
        __syncwarp();
        continue;
      }
      if (ok) ok = mbar_wait_cluster(&sm.xfull, (uint32_t)(u & 1), &sm.abort_flag, err, SITE_XFULL);
      if (ok && owner) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m >= p.M) continue;
          const float r = rs[m] + sm.xrs[m];   // rowsum(A)[m]: K half 0, then half 1
#pragma unroll
          for (int j = 0; j < kCols / 2; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = lane * kCols + 2 * j + h;
              const int n = cb * kBlockCols + c;
              if (n >= p.N) continue;
              float v = __uint_as_float((uint32_t)(acc[m][j] >> (32 * h))) + sm.xsum[m][c];
              if (p.zp_count > 0) v = __fsub_rn(v, __fmul_rn((float)__ldg(p.zp + (p.zp_count == 1 ? 0 : n)), r));
              v = __fmul_rn(__ldg(p.scale + (p.scale_count == 1 ? 0 : n)), v);
              const size_t o = (size_t)m * p.N + n;
              if (p.c_f32) static_cast<float*>(p.C)[o] = v;
              else static_cast<__nv_bfloat16*>(p.C)[o] = __float2bfloat16_rn(v);
            }
          }
        }
      }
      if (owner) mbar_arrive_cluster(peer_xempty);   // the odd CTA may overwrite the buffer
      __syncwarp();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sm.abort_flag) st_shared_cluster_u32(mapa_shared(smem_u32(&sm.abort_flag), rank ^ 1u), 1u);
  cluster_sync_all();   // neither CTA leaves while the other may still reach its shared memory
}

struct DeviceInfo {
  bool set = false;
  int max_clusters = 0;
};

template <int MT, bool BF16>
cudaError_t launch_main(const GemvSimtArgs& p, const CUtensorMap& tw, const CUtensorMap& ta, unsigned* err,
                        cudaStream_t s) {
  auto kern = gemv_pair_kernel<MT, BF16>;
  constexpr int threads = (consumer_warps<MT>() + 1) * 32;
  static std::mutex mu;
  static DeviceInfo info[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!info[dev].set) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(2 * 64, 1, 1);
      e = cudaOccupancyMaxActiveClusters(&info[dev].max_clusters, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (info[dev].max_clusters < 1) return cudaErrorInvalidConfiguration;
      info[dev].set = true;
    }
    max_clusters = info[dev].max_clusters;
  }
  const int nblk = (p.N + kBlockCols - 1) / kBlockCols;
  const int ncl = std::max(1, std::min(nblk, max_clusters));
  const int k_half = ((p.K + 1) / 2 + kStageRows - 1) / kStageRows * kStageRows;
  cfg.gridDim = dim3(2 * ncl, 1, 1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p, tw, ta, k_half, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gvs

bool gemv_simt_supported(long long M, long long K, long long N, int a_bf16, const void* A, const void* W) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(A), w = reinterpret_cast<uintptr_t>(W);
  // one or two rows: at four the tensor-core GEMV is faster (the accumulators of
  // four rows leave the CUDA-core kernel too few warps to hide its latency)
  return M >= 1 && M <= 2 && K >= 1 && K <= INT_MAX && N >= 16 && N % 16 == 0 && N <= INT_MAX &&
         K % (a_bf16 ? 8 : 4) == 0 && a % 16 == 0 && w % 16 == 0;
}

cudaError_t launch_gemv_simt(const GemvSimtArgs& p, unsigned* err, cudaStream_t s, const char** kernel_name) {
  using namespace gvs;
  CUtensorMap tw{}, ta{};
  cudaError_t e = make_tmap_2d(&tw, p.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)p.N, (uint64_t)p.K, (uint64_t)p.N,
                               kBlockCols, kStageRows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&ta, p.A, p.a_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   (uint64_t)p.K, (uint64_t)p.M, (uint64_t)p.K * (p.a_bf16 ? 2 : 4), kStageRows, (uint32_t)p.M,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  *kernel_name = "gemv_w8_pair_simt_f32x2";
  const int mt = p.M == 1 ? 1 : p.M == 2 ? 2 : 4;
  if (p.a_bf16)
    return mt == 1 ? launch_main<1, true>(p, tw, ta, err, s)
           : mt == 2 ? launch_main<2, true>(p, tw, ta, err, s)
                     : launch_main<4, true>(p, tw, ta, err, s);
  return mt == 1 ? launch_main<1, false>(p, tw, ta, err, s)
         : mt == 2 ? launch_main<2, false>(p, tw, ta, err, s)
                   : launch_main<4, false>(p, tw, ta, err, s);
}

}  // namespace qmm
