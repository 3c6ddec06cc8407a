// Operand pre-pass for the fp16-operand GEMM: 8-bit integer matrices become
// exact fp16 copies (every int8 and uint8 value is an fp16 value), with the
// row sums of A and the column sums of B that the MatMulInteger zero-point
// expansion needs (sum_k (a-za)(b-zb) = sum ab - za*colsum(B) - zb*rowsum(A)
// + K*za*zb; ROCm hip-ep PR #1248, "What"). The pass reads each byte once and
// writes two; the GEMM that follows then stages fp16 tiles with TMA straight
// into the tensor core's layout, instead of converting every operand tile once
// per output tile that uses it.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <climits>

namespace qmm {
namespace conv {

// 16 bytes -> 16 exact fp16 values (8 words), byte order preserved.
template <bool U>
__device__ __forceinline__ void convert16(const uint4 v, uint32_t (&h)[8]) {
  bytes_to_half4<U>(v.x, h[0], h[1]);
  bytes_to_half4<U>(v.y, h[2], h[3]);
  bytes_to_half4<U>(v.z, h[4], h[5]);
  bytes_to_half4<U>(v.w, h[6], h[7]);
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <bool U>
__device__ __forceinline__ int dp4a_sum(uint32_t w, int acc) {
  if (U) return (int)__dp4a(w, 0x01010101u, (unsigned)acc);
  return __dp4a((int)w, 0x01010101, acc);
}

// ---------------------------------------------------------------------------
// A and B together, no sums, staged through shared memory by bulk copies: each
// CTA (one per SM) walks 16 KB input blocks of the concatenation [A | B]; one
// thread copies a block in with cp.async.bulk (completion counted on an
// mbarrier), all threads convert it to a 32 KB fp16 block in shared memory, and
// one thread copies that out with cp.async.bulk. Three blocks are in flight per
// SM, which keeps HBM busy without per-thread loads.
constexpr int kBlkIn = 16384;
constexpr int kBlkOut = 2 * kBlkIn;
constexpr int kBulkStages = 3;
constexpr int kBulkThreads = 256;
constexpr size_t kBulkSmem = (size_t)kBulkStages * (kBlkIn + kBlkOut) + 1024;
enum : unsigned { SITE_BULK_FULL = 0x500 };

// Block `blk` of the concatenation: source, destination and byte count.
struct BulkBlock {
  const uint8_t* src;
  __half* dst;
  uint32_t bytes;
  bool second;
};
__device__ __forceinline__ BulkBlock bulk_block(long long blk, const uint8_t* A, __half* A16, long long a_bytes,
                                                long long a_blocks, const uint8_t* B, __half* B16, long long b_bytes) {
  BulkBlock r;
  const bool sec = blk >= a_blocks;
  const long long off = (sec ? blk - a_blocks : blk) * kBlkIn;
  const long long total = sec ? b_bytes : a_bytes;
  r.src = (sec ? B : A) + off;
  r.dst = (sec ? B16 : A16) + off;
  r.bytes = (uint32_t)min((long long)kBlkIn, total - off);
  r.second = sec;
  return r;
}

template <bool UA, bool UB>
__global__ void __launch_bounds__(kBulkThreads, 1)
    convert_bulk_kernel(const uint8_t* __restrict__ A, __half* __restrict__ A16, long long a_bytes,
                        const uint8_t* __restrict__ B, __half* __restrict__ B16, long long b_bytes, unsigned* err) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kBulkStages];
  __shared__ int abort_flag;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t in0 = base, out0 = base + kBulkStages * kBlkIn;
  const int t = threadIdx.x;
  const long long a_blocks = (a_bytes + kBlkIn - 1) / kBlkIn;
  const long long nblocks = a_blocks + (b_bytes + kBlkIn - 1) / kBlkIn;
  const long long my = (blockIdx.x < nblocks) ? (nblocks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (t == 0) {
    for (int i = 0; i < kBulkStages; ++i) mbar_init(&full[i], 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  auto issue_load = [&](long long i) {
    const int s = (int)(i % kBulkStages);
    const BulkBlock b = bulk_block(blockIdx.x + i * gridDim.x, A, A16, a_bytes, a_blocks, B, B16, b_bytes);
    mbar_arrive_expect_tx(&full[s], b.bytes);
    bulk_load(in0 + (uint32_t)s * kBlkIn, b.src, b.bytes, &full[s]);
  };
  if (t == 0)
    for (long long i = 0; i < my && i < kBulkStages; ++i) issue_load(i);
  for (long long i = 0; i < my; ++i) {
    const int s = (int)(i % kBulkStages);
    const BulkBlock b = bulk_block(blockIdx.x + i * gridDim.x, A, A16, a_bytes, a_blocks, B, B16, b_bytes);
    const bool ok = mbar_wait(&full[s], (uint32_t)((i / kBulkStages) & 1), &abort_flag, err, SITE_BULK_FULL);
    // the output buffer of this stage was last stored kBulkStages blocks ago
    if (t == 0) bulk_wait_read<kBulkStages - 1>();
    __syncthreads();
    if (ok) {
      const uint32_t src = in0 + (uint32_t)s * kBlkIn, dst = out0 + (uint32_t)s * kBlkOut;
      // 8 input bytes per thread and step: conflict-free 8-byte loads and 16-byte stores
#pragma unroll 4
      for (uint32_t o = (uint32_t)t * 8u; o < b.bytes; o += kBulkThreads * 8u) {
        const uint2 v = ld_shared_v2(src + o);
        uint32_t h[4];
        if (b.second) {
          bytes_to_half4<UB>(v.x, h[0], h[1]);
          bytes_to_half4<UB>(v.y, h[2], h[3]);
        } else {
          bytes_to_half4<UA>(v.x, h[0], h[1]);
          bytes_to_half4<UA>(v.y, h[2], h[3]);
        }
        st_shared_v4(dst + 2u * o, h[0], h[1], h[2], h[3]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0) {
      if (ok) {
        bulk_store(b.dst, out0 + (uint32_t)s * kBlkOut, 2u * b.bytes);
        bulk_commit();
      }
      if (i + kBulkStages < my) issue_load(i + kBulkStages);
    }
  }
  if (t == 0) {
    bulk_wait_all();
    // a load issued but not consumed (only after an abort) must land before exit
    for (long long i = (my > kBulkStages ? my - kBulkStages : 0); i < my; ++i)
      mbar_wait(&full[i % kBulkStages], (uint32_t)((i / kBulkStages) & 1), nullptr, err, SITE_BULK_FULL);
  }
}

// A and B together, no sums: 16-byte chunks [0, nA) of A then [0, nB) of B,
// grid-stride with four chunks (four loads) in flight per thread.
template <bool UA, bool UB>
__global__ void __launch_bounds__(256) convert_flat_kernel(const uint8_t* __restrict__ A, __half* __restrict__ A16,
                                                           long long nA, const uint8_t* __restrict__ B,
                                                           __half* __restrict__ B16, long long nB) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const long long total = nA + nB;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long c = i + j * stride;
      if (c < total) v[j] = ldg_nc_v4(c < nA ? A + 16 * c : B + 16 * (c - nA));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long c = i + j * stride;
      if (c >= total) break;
      uint32_t h[8];
      __half* d;
      if (c < nA) {
        convert16<UA>(v[j], h);
        d = A16 + 16 * c;
      } else {
        convert16<UB>(v[j], h);
        d = B16 + 16 * (c - nA);
      }
      st_global_v4(d, h[0], h[1], h[2], h[3]);
      st_global_v4(d + 8, h[4], h[5], h[6], h[7]);
    }
  }
}

// One warp per row (grid-stride over rows): row r of `rows` rows of
// `row_bytes` bytes (a multiple of 16, rows 16-byte aligned) becomes fp16 in
// dst; with ROWSUM, rowsum[r] = sum of the row's values (int32, wrapping).
template <bool U, bool ROWSUM>
__global__ void __launch_bounds__(256) convert_rows_kernel(const uint8_t* __restrict__ src, __half* __restrict__ dst,
                                                           long long rows, int row_bytes, int* __restrict__ rowsum) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int chunks = row_bytes >> 4;
  for (long long r = warp0; r < rows; r += nwarps) {
    const uint8_t* s = src + r * row_bytes;
    __half* d = dst + r * row_bytes;
    int acc = 0;
    for (int c0 = lane; c0 < chunks; c0 += 128) {   // four chunks (loads) in flight per lane
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (c0 + 32 * j < chunks) v[j] = ldg_nc_v4(s + 16 * (c0 + 32 * j));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 32 * j;
        if (c >= chunks) break;
        uint32_t h[8];
        convert16<U>(v[j], h);
        st_global_v4(d + 16 * c, h[0], h[1], h[2], h[3]);
        st_global_v4(d + 16 * c + 8, h[4], h[5], h[6], h[7]);
        if (ROWSUM) {
          acc = dp4a_sum<U>(v[j].x, acc);
          acc = dp4a_sum<U>(v[j].y, acc);
          acc = dp4a_sum<U>(v[j].z, acc);
          acc = dp4a_sum<U>(v[j].w, acc);
        }
      }
    }
    if (ROWSUM) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) rowsum[r] = acc;
    }
  }
}

// Column sums with the conversion: thread (column chunk cc, row block rb)
// converts rows [rb*R, rb*R + R) of 16 columns and adds its 16 partial column
// sums into colsum (zeroed beforehand) with atomics. `mats` matrices of
// `rows` x `cols` bytes each (batch of B), colsum is [mats][cols].
constexpr int kColRows = 32;   // rows per task at most (fewer when the matrix is small)

// Rows per task: as many as keep every SM busy with a few waves of tasks, a
// multiple of 4 in [4, kColRows] (a 1024 x 1024 weight gets 4: 64 CTAs instead of 8
// with 32).
int col_rows_per_task(long long mats, int rows, int cols) {
  const long long target = (long long)num_sms() * 1024;
  const long long work = mats * (long long)rows * (cols / 16);
  long long r = (work + target - 1) / target;
  r = (r + 3) / 4 * 4;
  return (int)std::max<long long>(4, std::min<long long>(kColRows, r));
}

template <bool U>
__global__ void __launch_bounds__(256) convert_cols_kernel(const uint8_t* __restrict__ src, __half* __restrict__ dst,
                                                           int mats, int rows, int cols, int* __restrict__ colsum,
                                                           int rpt) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const int cchunks = cols >> 4;
  const int rblocks = (rows + rpt - 1) / rpt;
  const long long tasks = (long long)mats * rblocks * cchunks;
  for (long long task = (long long)blockIdx.x * blockDim.x + threadIdx.x; task < tasks;
       task += (long long)gridDim.x * blockDim.x) {
    const int cc = (int)(task % cchunks);
    const long long rest = task / cchunks;
    const int rb = (int)(rest % rblocks);
    const int m = (int)(rest / rblocks);
    const size_t base = (size_t)m * rows * cols;
    int sum[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) sum[i] = 0;
    const int r_end = min(rows, (rb + 1) * rpt);
#pragma unroll 4
    for (int r = rb * rpt; r < r_end; ++r) {
      const size_t off = base + (size_t)r * cols + 16 * (size_t)cc;
      const uint4 v = ldg_nc_v4(src + off);
      uint32_t h[8];
      convert16<U>(v, h);
      st_global_v4(dst + off, h[0], h[1], h[2], h[3]);
      st_global_v4(dst + off + 8, h[4], h[5], h[6], h[7]);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t b = (w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
        sum[i] += U ? (int)b : (int)(int8_t)b;
      }
    }
    int* cs = colsum + (size_t)m * cols + 16 * (size_t)cc;
#pragma unroll
    for (int i = 0; i < 16; ++i) atomicAdd(cs + i, sum[i]);
  }
}

int grid_for(long long work_items, int per_block) {
  const long long blocks = (work_items + per_block - 1) / per_block;
  return (int)std::max<long long>(1, std::min<long long>(blocks, (long long)num_sms() * 8));
}

}  // namespace conv

cudaError_t launch_convert_rows(const void* src, bool u8, __half* dst, long long rows, int row_bytes, int* rowsum,
                                cudaStream_t s) {
  using namespace conv;
  if (rows <= 0 || row_bytes <= 0) return cudaSuccess;
  const int grid = grid_for(rows * 32, 256);
  const uint8_t* p = static_cast<const uint8_t*>(src);
  if (rowsum) {
    if (u8) convert_rows_kernel<true, true><<<grid, 256, 0, s>>>(p, dst, rows, row_bytes, rowsum);
    else convert_rows_kernel<false, true><<<grid, 256, 0, s>>>(p, dst, rows, row_bytes, rowsum);
  } else {
    if (u8) convert_rows_kernel<true, false><<<grid, 256, 0, s>>>(p, dst, rows, row_bytes, nullptr);
    else convert_rows_kernel<false, false><<<grid, 256, 0, s>>>(p, dst, rows, row_bytes, nullptr);
  }
  return cudaGetLastError();
}

cudaError_t launch_convert_flat(const void* A, bool au, __half* A16, long long a_bytes, const void* B, bool bu,
                                __half* B16, long long b_bytes, cudaStream_t s) {
  using namespace conv;
  const long long nA = a_bytes / 16, nB = b_bytes / 16;
  if (nA + nB <= 0) return cudaSuccess;
  const int grid = grid_for((nA + nB + 3) / 4, 256);
  const uint8_t* a = static_cast<const uint8_t*>(A);
  const uint8_t* b = static_cast<const uint8_t*>(B);
  if (au && bu) convert_flat_kernel<true, true><<<grid, 256, 0, s>>>(a, A16, nA, b, B16, nB);
  else if (au) convert_flat_kernel<true, false><<<grid, 256, 0, s>>>(a, A16, nA, b, B16, nB);
  else if (bu) convert_flat_kernel<false, true><<<grid, 256, 0, s>>>(a, A16, nA, b, B16, nB);
  else convert_flat_kernel<false, false><<<grid, 256, 0, s>>>(a, A16, nA, b, B16, nB);
  return cudaGetLastError();
}

namespace conv {
// Launch one instantiation; the dynamic shared-memory opt-in is recorded per
// instantiation and device.
template <bool UA, bool UB>
cudaError_t launch_bulk(int grid, const uint8_t* a, __half* A16, long long a_bytes, const uint8_t* b, __half* B16,
                        long long b_bytes, unsigned* err, cudaStream_t s) {
  static unsigned attr_dev_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 32 || !(attr_dev_mask & (1u << dev))) {
    const cudaError_t e =
        cudaFuncSetAttribute(convert_bulk_kernel<UA, UB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmem);
    if (e != cudaSuccess) return e;
    if (dev < 32) attr_dev_mask |= 1u << dev;
  }
  convert_bulk_kernel<UA, UB><<<grid, kBulkThreads, kBulkSmem, s>>>(a, A16, a_bytes, b, B16, b_bytes, err);
  return cudaGetLastError();
}
}  // namespace conv

cudaError_t launch_convert_bulk(const void* A, bool au, __half* A16, long long a_bytes, const void* B, bool bu,
                                __half* B16, long long b_bytes, unsigned* err, cudaStream_t s) {
  using namespace conv;
  if (a_bytes + b_bytes <= 0) return cudaSuccess;
  const long long nblocks = (a_bytes + kBlkIn - 1) / kBlkIn + (b_bytes + kBlkIn - 1) / kBlkIn;
  const int grid = (int)std::max<long long>(1, std::min<long long>(nblocks, (long long)num_sms()));
  const uint8_t* a = static_cast<const uint8_t*>(A);
  const uint8_t* b = static_cast<const uint8_t*>(B);
  if (au && bu) return launch_bulk<true, true>(grid, a, A16, a_bytes, b, B16, b_bytes, err, s);
  if (au) return launch_bulk<true, false>(grid, a, A16, a_bytes, b, B16, b_bytes, err, s);
  if (bu) return launch_bulk<false, true>(grid, a, A16, a_bytes, b, B16, b_bytes, err, s);
  return launch_bulk<false, false>(grid, a, A16, a_bytes, b, B16, b_bytes, err, s);
}

cudaError_t launch_convert_cols(const void* src, bool u8, __half* dst, int mats, int rows, int cols, int* colsum,
                                cudaStream_t s) {
  using namespace conv;
  if (mats <= 0 || rows <= 0 || cols <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(colsum, 0, sizeof(int) * (size_t)mats * cols, s);
  if (e != cudaSuccess) return e;
  const int rpt = col_rows_per_task(mats, rows, cols);
  const long long tasks = (long long)mats * ((rows + rpt - 1) / rpt) * (cols / 16);
  const int grid = grid_for(tasks, 256);
  const uint8_t* p = static_cast<const uint8_t*>(src);
  if (u8) convert_cols_kernel<true><<<grid, 256, 0, s>>>(p, dst, mats, rows, cols, colsum, rpt);
  else convert_cols_kernel<false><<<grid, 256, 0, s>>>(p, dst, mats, rows, cols, colsum, rpt);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// General planes: operands at any pitch, stored as they are or transposed
// (PyPTO PR #1920's a_trans / b_trans: A held as [K][M], B as [N][K]), become
// fp16 [rows][K] and [K][cols] copies whose rows are padded to 16 bytes. One
// CTA per 64 x 64 source tile; each thread reads one 16-byte chunk of a source
// row. A copy converts the chunk and writes it out; a transpose passes the tile
// through shared memory and each thread writes 16 values of one destination
// row.
// ---------------------------------------------------------------------------
namespace conv {

constexpr int kPT = 64;

// Bytes [c, c+16) of source row r; zero where outside the plane. vec: the
// plane's base and pitch are 16-byte multiples (c is one already).
__device__ __forceinline__ uint4 load_chunk(const uint8_t* src, long long pitch, int rows, int cols, int r, int c,
                                            bool vec) {
  if (r >= rows || c >= cols) return make_uint4(0u, 0u, 0u, 0u);
  const uint8_t* p = src + (long long)r * pitch + c;
  if (vec && c + 16 <= cols) return ldg_nc_v4(p);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  for (int i = 0; i < 16 && c + i < cols; ++i) w[i >> 2] |= (uint32_t)__ldg(p + i) << (8 * (i & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The first n (<= 16) of 16 fp16 values (h: pairs, element 0 in the low half)
// to d; a full chunk is two 16-byte stores (d is then 16-byte aligned).
__device__ __forceinline__ void store_halves(__half* d, const uint32_t (&h)[8], int n) {
  if (n == 16) {
    st_global_v4(d, h[0], h[1], h[2], h[3]);
    st_global_v4(d + 8, h[4], h[5], h[6], h[7]);
    return;
  }
  for (int i = 0; i < n; ++i) d[i] = __ushort_as_half((unsigned short)(h[i >> 1] >> (16 * (i & 1))));
}

template <bool U>
__device__ __forceinline__ void plane_tile(const ConvPlane& p, long long tile, uint8_t (*st)[kPT + 4]) {
  const int ct = (p.cols + kPT - 1) / kPT;
  const int r0 = (int)(tile / ct) * kPT, c0 = (int)(tile % ct) * kPT;
  const int t = threadIdx.x;
  const uint8_t* src = static_cast<const uint8_t*>(p.src);
  const bool vec = ((reinterpret_cast<uintptr_t>(src) | (uintptr_t)p.src_pitch) & 15u) == 0;
  const int lr = t >> 2, lc = (t & 3) * 16;
  const uint4 v = load_chunk(src, p.src_pitch, p.rows, p.cols, r0 + lr, c0 + lc, vec);
  uint32_t h[8];
  if (!p.trans) {
    if (r0 + lr < p.rows && c0 + lc < p.cols) {
      convert16<U>(v, h);
      store_halves(p.dst + (long long)(r0 + lr) * p.dst_pitch + c0 + lc, h, min(16, p.cols - c0 - lc));
    }
    return;
  }
  uint32_t* row = reinterpret_cast<uint32_t*>(&st[lr][lc]);
  row[0] = v.x;
  row[1] = v.y;
  row[2] = v.z;
  row[3] = v.w;
  __syncthreads();
  // destination row c0 + cc (a source column), values from source rows r0 + rg ..
  const int cc = t & 63, rg = (t >> 6) * 16;
  if (c0 + cc >= p.cols || r0 + rg >= p.rows) return;
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    w[j] = (uint32_t)st[rg + 4 * j][cc] | ((uint32_t)st[rg + 4 * j + 1][cc] << 8) |
           ((uint32_t)st[rg + 4 * j + 2][cc] << 16) | ((uint32_t)st[rg + 4 * j + 3][cc] << 24);
  convert16<U>(make_uint4(w[0], w[1], w[2], w[3]), h);
  store_halves(p.dst + (long long)(c0 + cc) * p.dst_pitch + r0 + rg, h, min(16, p.rows - r0 - rg));
}

template <bool UA, bool UB>
__global__ void __launch_bounds__(256) convert_planes_kernel(const ConvPlane a, const ConvPlane b, long long tiles_a) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  __shared__ uint8_t st[kPT][kPT + 4];
  if ((long long)blockIdx.x < tiles_a) plane_tile<UA>(a, (long long)blockIdx.x, st);
  else plane_tile<UB>(b, (long long)blockIdx.x - tiles_a, st);
}

long long plane_tiles(const ConvPlane& p) {
  if (p.rows <= 0 || p.cols <= 0) return 0;
  return (long long)((p.rows + kPT - 1) / kPT) * ((p.cols + kPT - 1) / kPT);
}

// acc = acc_in (or 0) at every output; acc_out and the scaled C from it.
__global__ void __launch_bounds__(256) acc_only_kernel(const int* __restrict__ acc_in, int* __restrict__ acc_out,
                                                       int M, int N, const float* __restrict__ as, int ac,
                                                       const float* __restrict__ ws, int wc, void* C, int c_f32) {
  const long long total = (long long)M * N;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int acc = acc_in ? __ldg(acc_in + i) : 0;
    if (acc_out) acc_out[i] = acc;
    if (!C) continue;
    const int m = (int)(i / N), n = (int)(i - (long long)m * N);
    float v = __int2float_rn(acc);
    v = __fmul_rn(v, __ldg(as + (ac == 1 ? 0 : m)));
    v = __fmul_rn(v, __ldg(ws + (wc == 1 ? 0 : n)));
    if (c_f32) static_cast<float*>(C)[i] = v;
    else static_cast<__nv_bfloat16*>(C)[i] = __float2bfloat16_rn(v);
  }
}

// colsum[c] += the sum of rows [r0, r0 + 64) of column c (one thread per column).
template <bool U>
__global__ void __launch_bounds__(256) colsum_kernel(const uint8_t* __restrict__ src, int rows, int cols,
                                                     int* __restrict__ colsum) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= cols) return;
  const int r0 = blockIdx.y * 64, r1 = min(rows, r0 + 64);
  int acc = 0;
#pragma unroll 8
  for (int r = r0; r < r1; ++r) {
    const uint32_t v = __ldg(src + (long long)r * cols + c);
    acc += U ? (int)v : (int)(int8_t)(uint8_t)v;
  }
  atomicAdd(colsum + c, acc);
}

}  // namespace conv

cudaError_t launch_colsum(const void* src, bool u8, int rows, int cols, int* colsum, cudaStream_t s) {
  using namespace conv;
  if (cols <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(colsum, 0, sizeof(int) * (size_t)cols, s);
  if (e != cudaSuccess || rows <= 0) return e;
  if ((rows + 63) / 64 > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((cols + 255) / 256), (unsigned)((rows + 63) / 64));
  const uint8_t* p = static_cast<const uint8_t*>(src);
  if (u8) colsum_kernel<true><<<grid, 256, 0, s>>>(p, rows, cols, colsum);
  else colsum_kernel<false><<<grid, 256, 0, s>>>(p, rows, cols, colsum);
  return cudaGetLastError();
}

cudaError_t launch_convert_planes(const ConvPlane& a, bool au, const ConvPlane& b, bool bu, cudaStream_t s) {
  using namespace conv;
  const long long ta = plane_tiles(a), tb = plane_tiles(b);
  if (ta + tb == 0) return cudaSuccess;
  if (ta + tb > INT_MAX) return cudaErrorInvalidValue;
  const int grid = (int)(ta + tb);
  if (au && bu) convert_planes_kernel<true, true><<<grid, 256, 0, s>>>(a, b, ta);
  else if (au) convert_planes_kernel<true, false><<<grid, 256, 0, s>>>(a, b, ta);
  else if (bu) convert_planes_kernel<false, true><<<grid, 256, 0, s>>>(a, b, ta);
  else convert_planes_kernel<false, false><<<grid, 256, 0, s>>>(a, b, ta);
  return cudaGetLastError();
}

cudaError_t launch_acc_only(const int* acc_in, int* acc_out, int M, int N, const float* act_scale, int act_count,
                            const float* w_scale, int w_count, void* C, int c_f32, cudaStream_t s) {
  using namespace conv;
  if (M <= 0 || N <= 0) return cudaSuccess;
  conv::acc_only_kernel<<<grid_for((long long)M * N, 256), 256, 0, s>>>(acc_in, acc_out, M, N, act_scale, act_count,
                                                                        w_scale, w_count, C, c_f32);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// Form (a) pre-pass: the int8 weight as exact bf16, and the activations' row
// sums (the zero-point correction of TrainDeeploy PR #53, "The kernel") or,
// for fp32 activations, a split into two bf16 parts.
// ---------------------------------------------------------------------------
namespace conv {

// Four int8 (bytes of w) -> four exact bf16, as two bf16x2 words: the byte,
// biased to unsigned, sits in the low mantissa bits of 2^23 (fp32 0x4B000000),
// the bias is subtracted in fp32 (exact), and the top halves of the fp32 words
// are the bf16 values (integers of magnitude <= 256 have at most 8 significant
// bits, so dropping the low half loses nothing).
__device__ __forceinline__ void s8_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  float f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(0x4B000000u | ((u >> (8 * i)) & 0xFFu)) - 8388736.0f;
  lo = prmt(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632u);
  hi = prmt(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632u);
}

__global__ void __launch_bounds__(256) convert_s8_bf16_kernel(const uint8_t* __restrict__ src,
                                                              uint32_t* __restrict__ dst, long long n16) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i + j * stride < n16) v[j] = ldg_nc_v4(src + 16 * (i + j * stride));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long c = i + j * stride;
      if (c >= n16) break;
      uint32_t h[8];
      s8_to_bf16x4(v[j].x, h[0], h[1]);
      s8_to_bf16x4(v[j].y, h[2], h[3]);
      s8_to_bf16x4(v[j].z, h[4], h[5]);
      s8_to_bf16x4(v[j].w, h[6], h[7]);
      st_global_v4(dst + 8 * c, h[0], h[1], h[2], h[3]);
      st_global_v4(dst + 8 * c + 4, h[4], h[5], h[6], h[7]);
    }
  }
}

// fp32 row sums of bf16 rows (one warp per row).
__global__ void __launch_bounds__(256) rowsum_bf16_kernel(const uint16_t* __restrict__ A, long long rows, int K,
                                                          float* __restrict__ rowsum) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = warp0; r < rows; r += nwarps) {
    const uint16_t* a = A + r * K;
    float acc = 0.f;
    for (int k = lane * 8; k < K; k += 256) {   // 16-byte loads (K % 8 == 0)
      const uint4 v = ldg_nc_v4(a + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) acc += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xFFFF0000u);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) rowsum[r] = acc;
  }
}

// fp32 rows [M][K] -> bf16 [M][2*Kp]: the first Kp columns hold hi = RN_bf16(a),
// the next Kp columns lo = RN_bf16(a - hi) (zero padded from K to Kp, a multiple
// of 64), so that hi + lo equals a to about 2^-16 relative; with rowsum, the fp32
// row sums of a (one warp per row).
__global__ void __launch_bounds__(256) split_f32_kernel(const float* __restrict__ A, long long rows, int K, int Kp,
                                                        uint16_t* __restrict__ out, float* __restrict__ rowsum) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = warp0; r < rows; r += nwarps) {
    const float* a = A + r * K;
    uint16_t* hi = out + r * 2 * (long long)Kp;
    uint16_t* lo = hi + Kp;
    float acc = 0.f;
    for (int k = lane; k < Kp; k += 32) {
      const float x = k < K ? __ldg(a + k) : 0.f;
      const __nv_bfloat16 h = __float2bfloat16_rn(x);
      const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
      hi[k] = *reinterpret_cast<const uint16_t*>(&h);
      lo[k] = *reinterpret_cast<const uint16_t*>(&l);
      acc += x;
    }
    if (rowsum) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) rowsum[r] = acc;
    }
  }
}

}  // namespace conv

cudaError_t launch_convert_s8_bf16(const void* src, void* dst, long long bytes, cudaStream_t s) {
  using namespace conv;
  const long long n16 = bytes / 16;
  if (n16 <= 0) return cudaSuccess;
  convert_s8_bf16_kernel<<<grid_for((n16 + 3) / 4, 256), 256, 0, s>>>(static_cast<const uint8_t*>(src),
                                                                       static_cast<uint32_t*>(dst), n16);
  return cudaGetLastError();
}

cudaError_t launch_rowsum_bf16(const void* A, long long rows, int K, float* rowsum, cudaStream_t s) {
  using namespace conv;
  if (rows <= 0) return cudaSuccess;
  rowsum_bf16_kernel<<<grid_for(rows * 32, 256), 256, 0, s>>>(static_cast<const uint16_t*>(A), rows, K, rowsum);
  return cudaGetLastError();
}

cudaError_t launch_split_f32(const float* A, long long rows, int K, int Kp, void* out, float* rowsum,
                             cudaStream_t s) {
  using namespace conv;
  if (rows <= 0) return cudaSuccess;
  split_f32_kernel<<<grid_for(rows * 32, 256), 256, 0, s>>>(A, rows, K, Kp, static_cast<uint16_t*>(out), rowsum);
  return cudaGetLastError();
}

}  // namespace qmm
