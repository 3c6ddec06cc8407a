// ConvInteger pre-pass. ROCm hip-ep PR #1248 ("What", ConvInteger paragraph)
// defines the operator on rank-4 NCHW (rank-3 NCL through a unit spatial row)
// with a scalar activation zero point and a scalar or per-output-channel
// weight zero point. Here it becomes the exact integer GEMM of the library:
// for each image n and group g,
//   y[n, g*Mg + m, p] = sum_k (w[g*Mg + m, k] - w_zp) * (col[n, g, k, p] - x_zp)
// with k running over the group's (channel, kh, kw) taps and p over output
// pixels, so A = the weight [M][C/G*kH*kW] (shared by every image), B = the
// im2col matrix of each image, and the output rows land directly in NCHW.
// A padded position holds x_zp in col, so its shifted value is 0 and the
// zero-point expansion of the GEMM epilogue (sum ab - w_zp*colsum(col) -
// x_zp*rowsum(w) + K*w_zp*x_zp) stays exact with the sums taken here.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <climits>

namespace qmm {
namespace convk {

constexpr int kThreads = 256;
constexpr int kPix = 8;       // output pixels per thread (one 16-byte fp16 store per tap)
constexpr int kTaps = 32;     // taps (k rows) per thread

__device__ __forceinline__ void st_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <bool U>
__device__ __forceinline__ int byte_value(uint32_t v) {
  return U ? (int)v : (int)(int8_t)(uint8_t)v;
}

// Gather form (any geometry): one thread takes kPix consecutive output pixels
// of image blockIdx.z for kTaps consecutive taps starting at blockIdx.y *
// kTaps, reading each input byte straight from global memory. Used when the
// input rows a band of output rows needs do not fit in shared memory.
template <bool U>
__global__ void __launch_bounds__(kThreads) im2col_gather_kernel(const Im2colArgs a) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const int P = a.oH * a.oW;
  const int p0 = (blockIdx.x * kThreads + threadIdx.x) * kPix;
  if (p0 >= P) return;
  const int n = blockIdx.z;
  const int khw = a.kH * a.kW;
  const int Kt = a.C * khw;
  const int k_beg = blockIdx.y * kTaps;
  const int k_end = min(Kt, k_beg + kTaps);
  int ih0[kPix], iw0[kPix];
#pragma unroll
  for (int j = 0; j < kPix; ++j) {
    const int p = min(p0 + j, P - 1);
    const int oh = p / a.oW, ow = p - oh * a.oW;
    ih0[j] = oh * a.sh - a.pt;
    iw0[j] = ow * a.sw - a.pl;
  }
  const int npix = min(kPix, P - p0);
  const uint8_t* xn = static_cast<const uint8_t*>(a.x) + (long long)n * a.C * a.H * a.W;
  const uint32_t zb = a.xzp ? (uint32_t)__ldg(static_cast<const uint8_t*>(a.xzp)) : 0u;
  for (int k = k_beg; k < k_end; ++k) {
    const int c = k / khw, r = k - c * khw;
    const int kh = r / a.kW, kw = r - kh * a.kW;
    const uint8_t* xc = xn + (long long)c * a.H * a.W;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < kPix; ++j) {
      const int ih = ih0[j] + kh * a.dh, iw = iw0[j] + kw * a.dw;
      const uint32_t v = ((unsigned)ih < (unsigned)a.H && (unsigned)iw < (unsigned)a.W)
                             ? (uint32_t)__ldg(xc + (long long)ih * a.W + iw)
                             : zb;
      w[j >> 2] |= v << (8 * (j & 3));
    }
    uint32_t h[4];
    bytes_to_half4<U>(w[0], h[0], h[1]);
    bytes_to_half4<U>(w[1], h[2], h[3]);
    __half* dst = a.col + ((long long)n * Kt + k) * a.pitch + p0;
    if (npix == kPix) {
      st_v4(dst, h[0], h[1], h[2], h[3]);
    } else {
      for (int j = 0; j < npix; ++j) dst[j] = __ushort_as_half((unsigned short)(h[j >> 1] >> (16 * (j & 1))));
    }
  }
}

// Staged form: block (band of R output rows, cpb channels, image). The input
// rows the band reads, for all its channels, are copied into shared memory
// (one warp per row, lanes along it) with the padding in place: x_zp outside
// the input, `ws` bytes per row with the left pad included. Each thread then
// owns fixed 8-pixel groups of the band: it works out their eight shared-memory
// offsets once and walks channels x kh x kw, each tap one 16-byte store of 8
// fp16 values.
template <bool U>
__global__ void __launch_bounds__(kThreads) im2col_staged_kernel(const Im2colArgs a, int R, int ws, int cpb) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  extern __shared__ uint8_t sx[];
  const int n = blockIdx.z;
  const int oh0 = blockIdx.x * R;
  const int oh1 = min(a.oH, oh0 + R);
  const int ih_lo = oh0 * a.sh - a.pt;
  const int nrows = (oh1 - 1 - oh0) * a.sh + (a.kH - 1) * a.dh + 1;
  const int c_beg = blockIdx.y * cpb;
  const int nc = min(cpb, a.C - c_beg);
  const uint8_t zb = a.xzp ? __ldg(static_cast<const uint8_t*>(a.xzp)) : (uint8_t)0;
  const uint8_t* xb = static_cast<const uint8_t*>(a.x) + ((long long)n * a.C + c_beg) * a.H * a.W;
  const int plane = nrows * ws;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int row = warp; row < nc * nrows; row += kThreads / 32) {
    const int ci = row / nrows, rr = row - ci * nrows;
    const int ih = ih_lo + rr;
    uint8_t* dst = sx + ci * plane + rr * ws;
    if ((unsigned)ih >= (unsigned)a.H) {
      for (int cc = lane; cc < ws; cc += 32) dst[cc] = zb;
      continue;
    }
    const uint8_t* src = xb + ((long long)ci * a.H + ih) * a.W - a.pl;
#pragma unroll 4
    for (int cc = lane; cc < ws; cc += 32) {
      const int iw = cc - a.pl;
      dst[cc] = ((unsigned)iw < (unsigned)a.W) ? __ldg(src + cc) : zb;
    }
  }
  __syncthreads();
  const int p_beg = oh0 * a.oW, p_end = oh1 * a.oW;
  const int g_beg = p_beg & ~(kPix - 1);
  const int ngroups = (p_end - g_beg + kPix - 1) / kPix;
  const int khw = a.kH * a.kW;
  const long long Kt = (long long)a.C * khw;
  const int tap_h = a.dh * ws;   // shared-memory step of one kh
  // with fewer groups than threads, the block's channels are split among
  // `lanes` threads per group
  const int lanes = max(1, min(nc, kThreads / ngroups));
  const int cl = threadIdx.x / ngroups;
  if (lanes > 1 && cl >= lanes) return;
  const int gstep = lanes > 1 ? ngroups : kThreads;
  for (int gi = lanes > 1 ? threadIdx.x - cl * ngroups : threadIdx.x; gi < ngroups; gi += gstep) {
    const int pg = g_beg + gi * kPix;
    int off[kPix];
    bool valid[kPix];
    int oh = pg / a.oW, ow = pg - oh * a.oW;
#pragma unroll
    for (int j = 0; j < kPix; ++j) {
      valid[j] = pg + j >= p_beg && pg + j < p_end;
      off[j] = valid[j] ? (oh - oh0) * a.sh * ws + ow * a.sw : 0;
      if (++ow == a.oW) {
        ow = 0;
        ++oh;
      }
    }
    const bool full = pg >= p_beg && pg + kPix <= p_end;
    for (int ci = lanes > 1 ? cl : 0; ci < nc; ci += lanes) {
      const uint8_t* sc = sx + ci * plane;
      __half* dst = a.col + ((long long)n * Kt + (long long)(c_beg + ci) * khw) * a.pitch + pg;
      for (int kh = 0; kh < a.kH; ++kh, sc += tap_h) {
        const uint8_t* st = sc;
        for (int kw = 0; kw < a.kW; ++kw, st += a.dw, dst += a.pitch) {
          uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            w0 |= (uint32_t)st[off[j]] << (8 * j);
            w1 |= (uint32_t)st[off[j + 4]] << (8 * j);
          }
          uint32_t h[4];
          bytes_to_half4<U>(w0, h[0], h[1]);
          bytes_to_half4<U>(w1, h[2], h[3]);
          if (full) {
            st_v4(dst, h[0], h[1], h[2], h[3]);
          } else {
#pragma unroll
            for (int j = 0; j < kPix; ++j)
              if (valid[j]) dst[j] = __ushort_as_half((unsigned short)(h[j >> 1] >> (16 * (j & 1))));
          }
        }
      }
    }
  }
}

// Per-group channel sums of x: S[n*G + g][h*W + w] = sum of x[n, c, h, w] over
// the group's channels. Block: 32 positions x 8 channel slices.
template <bool U>
__global__ void __launch_bounds__(kThreads) chansum_kernel(const uint8_t* __restrict__ x, int C, int HW, int G,
                                                           int* __restrict__ S) {
  __shared__ int part[kThreads / 32][33];
  const int lane = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int hw = blockIdx.x * 32 + lane;
  const int g = blockIdx.y, n = blockIdx.z, Cg = C / G;
  int acc = 0;
  if (hw < HW) {
    const uint8_t* xp = x + ((long long)n * C + (long long)g * Cg) * HW + hw;
#pragma unroll 8
    for (int c = sl; c < Cg; c += kThreads / 32) acc += byte_value<U>(__ldg(xp + (long long)c * HW));
  }
  part[sl][lane] = acc;
  __syncthreads();
  if (sl == 0 && hw < HW) {
    int t = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) t += part[i][lane];
    S[((long long)n * G + g) * HW + hw] = t;
  }
}

// colsum[n*G + g][p] = sum over the taps of the window of output pixel p of the
// group's channel sums, a padded position counting Cg * x_zp (Cg copies of the
// pad value).
template <bool U>
__global__ void __launch_bounds__(kThreads) window_colsum_kernel(const int* __restrict__ S, const Im2colArgs a,
                                                                 int* __restrict__ colsum) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  const int P = a.oH * a.oW;
  const int p = blockIdx.x * kThreads + threadIdx.x;
  if (p >= P) return;
  const long long ng = blockIdx.y;
  const int Cg = a.C / a.G;
  const int zp = a.xzp ? byte_value<U>(__ldg(static_cast<const uint8_t*>(a.xzp))) : 0;
  const int pad = Cg * zp;
  const int oh = p / a.oW, ow = p - oh * a.oW;
  const int* Sn = S + ng * a.H * a.W;
  int t = 0;
  for (int kh = 0; kh < a.kH; ++kh) {
    const int ih = oh * a.sh - a.pt + kh * a.dh;
    for (int kw = 0; kw < a.kW; ++kw) {
      const int iw = ow * a.sw - a.pl + kw * a.dw;
      t += ((unsigned)ih < (unsigned)a.H && (unsigned)iw < (unsigned)a.W) ? __ldg(Sn + (long long)ih * a.W + iw) : pad;
    }
  }
  colsum[ng * P + p] = t;
}

// One block per row: fp16 copy at `pitch` and the row's sum.
template <bool U>
__global__ void __launch_bounds__(kThreads) rows_pitched_kernel(const uint8_t* __restrict__ src, int cols,
                                                                __half* __restrict__ dst, long long pitch,
                                                                int* __restrict__ rowsum) {
  __shared__ int part[kThreads / 32];
  const int r = blockIdx.x;
  const uint8_t* s = src + (long long)r * cols;
  __half* d = dst + (long long)r * pitch;
  int acc = 0;
#pragma unroll 4
  for (int c = threadIdx.x; c < cols; c += kThreads) {
    const int v = byte_value<U>(__ldg(s + c));
    d[c] = __int2half_rn(v);   // |v| <= 255: exact in fp16
    acc += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (rowsum && threadIdx.x == 0) {
    int t = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) t += part[i];
    rowsum[r] = t;
  }
}

}  // namespace convk

namespace convk {
constexpr int kStagedSmemMax = 48 * 1024;

template <bool U>
cudaError_t im2col_one(const Im2colArgs& a, int* S, cudaStream_t s) {
  using namespace convk;
  const long long P = (long long)a.oH * a.oW;
  const long long Kt = (long long)a.C * a.kH * a.kW;
  // staged form: R output rows per block (about 1024 pixels), if their input rows fit
  // staged form: R output rows (about 1024 pixels) and up to 8 channels per
  // block, if their input rows fit in shared memory
  const long long ws = ((long long)(a.oW - 1) * a.sw + (long long)(a.kW - 1) * a.dw + 1 + 3) & ~3ll;
  int R = (int)std::max<long long>(1, std::min<long long>(a.oH, 1024 / std::max(1, a.oW)));
  auto rows_for = [&](int r) { return (long long)(r - 1) * a.sh + (long long)(a.kH - 1) * a.dh + 1; };
  while (R > 1 && rows_for(R) * ws > kStagedSmemMax) R /= 2;
  int cpb = 8;
  while (cpb > 1 && cpb * rows_for(R) * ws > kStagedSmemMax) cpb /= 2;
  cpb = std::min(cpb, a.C);
  if (ws <= kStagedSmemMax && cpb * rows_for(R) * ws <= kStagedSmemMax) {
    const long long gx = (a.oH + R - 1) / R, gy = (a.C + cpb - 1) / cpb;
    if (gx > INT_MAX || gy > 65535) return cudaErrorInvalidValue;
    const size_t smem = (size_t)(cpb * rows_for(R) * ws);
    im2col_staged_kernel<U><<<dim3((unsigned)gx, (unsigned)gy, (unsigned)a.Nb), kThreads, smem, s>>>(a, R, (int)ws,
                                                                                                      cpb);
  } else {
    const long long gx = (P + (long long)kThreads * kPix - 1) / ((long long)kThreads * kPix);
    const long long gy = (Kt + kTaps - 1) / kTaps;
    if (gx > INT_MAX || gy > 65535) return cudaErrorInvalidValue;
    im2col_gather_kernel<U><<<dim3((unsigned)gx, (unsigned)gy, (unsigned)a.Nb), kThreads, 0, s>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !a.colsum) return e;
  const long long HW = (long long)a.H * a.W;
  if ((HW + 31) / 32 > INT_MAX || a.G > 65535 || (long long)a.Nb * a.G > 65535) return cudaErrorInvalidValue;
  chansum_kernel<U><<<dim3((unsigned)((HW + 31) / 32), (unsigned)a.G, (unsigned)a.Nb), kThreads, 0, s>>>(
      static_cast<const uint8_t*>(a.x), a.C, (int)HW, a.G, S);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  window_colsum_kernel<U><<<dim3((unsigned)((P + kThreads - 1) / kThreads), (unsigned)(a.Nb * a.G)), kThreads, 0,
                            s>>>(S, a, a.colsum);
  return cudaGetLastError();
}
}  // namespace convk

// ---------------------------------------------------------------------------
// Implicit-GEMM route: the operands with their zero points already taken out,
// as fp16 (every difference of two 8-bit values lies in [-255, 255]). The
// input becomes channels-innermost (NHWC) so that an im2col tensor copy can
// gather a 64-channel slice of 128 output pixels' windows per stage; padding
// then reads as 0, i.e. as x_zp before the shift.
// ---------------------------------------------------------------------------
namespace convk {

template <bool U>
__device__ __forceinline__ int zp_value(const void* zp, int i) {
  return U ? (int)static_cast<const uint8_t*>(zp)[i] : (int)static_cast<const int8_t*>(zp)[i];
}

// The weight's share of the launch below: one thread per element of
// w16 [M][(r*kW + s)*Cg + c].
struct ConvW16 {
  const uint8_t* w;
  int M, Cg, kH, kW;
  const void* wzp;
  int wzp_count;
  __half* w16;
};

template <bool U>
__device__ __forceinline__ void conv_w16_elements(const ConvW16& a, long long first, long long count) {
  const long long Kg = (long long)a.kH * a.kW * a.Cg;
  const long long total = (long long)a.M * Kg;
  for (long long idx = first + threadIdx.x; idx < total && idx < first + count; idx += kThreads) {
    const int m = (int)(idx / Kg);
    const int k = (int)(idx - (long long)m * Kg);
    const int tap = k / a.Cg, c = k - tap * a.Cg;
    const int r = tap / a.kW, sx = tap - r * a.kW;
    const int zp = a.wzp_count == 0 ? 0 : zp_value<U>(a.wzp, a.wzp_count == 1 ? 0 : m);
    const int v = byte_value<U>(a.w[(((size_t)m * a.Cg + c) * a.kH + r) * a.kW + sx]);
    a.w16[idx] = __int2half_rn(v - zp);
  }
}

// Rows (channels) 4i..4i+3 of four consecutive pixels, one word per row ->
// one word per pixel holding its four channels (byte i = row i).
__device__ __forceinline__ void transpose4x4(const uint32_t (&r)[4], uint32_t (&c)[4]) {
  const uint32_t t0 = prmt(r[0], r[1], 0x5140u), t1 = prmt(r[0], r[1], 0x7362u);
  const uint32_t t2 = prmt(r[2], r[3], 0x5140u), t3 = prmt(r[2], r[3], 0x7362u);
  c[0] = prmt(t0, t2, 0x5410u);
  c[1] = prmt(t0, t2, 0x7632u);
  c[2] = prmt(t1, t3, 0x5410u);
  c[3] = prmt(t1, t3, 0x7632u);
}

// Four bytes (channels) minus the zero point as two exact fp16 pairs: each
// byte, biased to unsigned, goes into the low mantissa bits of 1024 (ulp 1)
// and 1024 + bias + zp is subtracted (every value involved is an integer
// below 2048, so the subtraction is exact).
template <bool U>
__device__ __forceinline__ void shifted_half4(uint32_t w, __half2 off, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = U ? w : (w ^ 0x80808080u);
  const uint32_t l = prmt(u, 0x64646464u, 0x4140u), h = prmt(u, 0x64646464u, 0x4342u);
  const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&l), off);
  const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&h), off);
  lo = *reinterpret_cast<const uint32_t*>(&a);
  hi = *reinterpret_cast<const uint32_t*>(&b);
}

constexpr int kXPix = 256;              // pixels per CTA of conv_x16_kernel
constexpr int kXPitch = kXPix + 4;      // shared row pitch (65 words): consecutive rows one bank apart

// One CTA per 256 pixels x 64 channels of one image: the channel rows come in
// with 16-byte loads into shared memory; each thread then takes a 4-pixel x
// 8-channel block (eight 32-bit reads, conflict-free), transposes it in
// registers and writes each pixel's 8 shifted channels as one 16-byte store,
// four lanes covering 32 channels of a pixel (64 contiguous bytes). The CTAs
// of the z slices from Nb on instead convert the weight, w_per elements each
// (at most two per thread), so both operands take one launch.
template <bool U, bool WU>
__global__ void __launch_bounds__(kThreads) conv_x16_kernel(const uint8_t* __restrict__ x, int C, int HW, int Nb,
                                                            const void* xzp, __half* __restrict__ x16, bool vec,
                                                            const ConvW16 wa, long long w_per) {
  asm volatile("griddepcontrol.launch_dependents;");   // a dependent GEMM may start its prologue
  if ((int)blockIdx.z >= Nb) {
    const long long cta = ((long long)(blockIdx.z - Nb) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    conv_w16_elements<WU>(wa, cta * w_per, w_per);
    return;
  }
  __shared__ __align__(16) uint8_t tile[64][kXPitch];
  const int p0 = blockIdx.x * kXPix, c0 = blockIdx.y * 64, n = blockIdx.z;
  const int tid = threadIdx.x;
  {
    const int col = (tid & 15) * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = (tid >> 4) + 16 * j;
      const uint8_t* src = x + ((size_t)n * C + c0 + row) * HW + p0 + col;
      uint32_t* d = reinterpret_cast<uint32_t*>(&tile[row][col]);
      if (vec && p0 + col + 16 <= HW) {
        const uint4 v = ldg_nc_v4(src);
        d[0] = v.x;
        d[1] = v.y;
        d[2] = v.z;
        d[3] = v.w;
      } else {
        for (int i = 0; i < 16; ++i) tile[row][col + i] = (p0 + col + i < HW) ? src[i] : (uint8_t)0;
      }
    }
  }
  __syncthreads();
  const int zp = xzp ? zp_value<U>(xzp, 0) : 0;
  const __half off = __int2half_rn((U ? 1024 : 1152) + zp);
  const __half2 off2 = __halves2half2(off, off);
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int job = 0; job < 2; ++job) {
    // a warp step: 4 channel octets x 8 pixel quads; with the 65-word row pitch
    // lane (co, pq) reads bank 8 (co mod 4) + pq (+ const): all 32 distinct
    const int co = 4 * job + (lane & 3);   // channels 8 co .. 8 co + 7 of the block
    const int pq = 8 * warp + (lane >> 2);   // pixels 4 pq .. 4 pq + 3 of the tile
    uint32_t r0[4], r1[4], c0w[4], c1w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r0[i] = *reinterpret_cast<const uint32_t*>(&tile[8 * co + i][4 * pq]);
      r1[i] = *reinterpret_cast<const uint32_t*>(&tile[8 * co + 4 + i][4 * pq]);
    }
    transpose4x4(r0, c0w);
    transpose4x4(r1, c1w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int p = p0 + 4 * pq + j;
      if (p < HW) {
        uint32_t h[4];
        shifted_half4<U>(c0w[j], off2, h[0], h[1]);
        shifted_half4<U>(c1w[j], off2, h[2], h[3]);
        st_v4(x16 + ((size_t)n * HW + p) * C + c0 + 8 * co, h[0], h[1], h[2], h[3]);
      }
    }
  }
}

}  // namespace convk

cudaError_t launch_conv_operands(const void* x, bool xu, int Nb, int C, int HW, const void* xzp, __half* x16,
                                 const void* w, bool wu, int M, int Cg, int kH, int kW, const void* wzp,
                                 int wzp_count, __half* w16, cudaStream_t s) {
  using namespace convk;
  if (Nb <= 0 || C <= 0 || HW <= 0 || M <= 0) return cudaSuccess;
  if (C % 64 != 0 || Nb >= 65535 || C / 64 > 65535) return cudaErrorInvalidValue;
  const bool vec = HW % 16 == 0 && (reinterpret_cast<uintptr_t>(x) % 16) == 0;
  // z >= Nb: the weight, over enough slices for at most two elements per
  // thread (each is a gathered byte: a thread's loads would otherwise queue
  // one DRAM round trip after another)
  const long long slice = (long long)((HW + kXPix - 1) / kXPix) * (C / 64);
  const long long wtotal = (long long)M * kH * kW * Cg;
  const long long wneed = (wtotal + 2LL * kThreads - 1) / (2LL * kThreads);   // CTAs at two elements per thread
  const long long wz = std::max(1LL, std::min((wneed + slice - 1) / slice, 65535LL - Nb));
  const dim3 grid((HW + kXPix - 1) / kXPix, C / 64, (unsigned)(Nb + wz));
  const long long wctas = slice * wz;
  const long long w_per = ((wtotal + wctas - 1) / wctas + kThreads - 1) / kThreads * kThreads;
  ConvW16 wa{static_cast<const uint8_t*>(w), M, Cg, kH, kW, wzp, wzp_count, w16};
  const uint8_t* p = static_cast<const uint8_t*>(x);
  if (xu && wu) conv_x16_kernel<true, true><<<grid, kThreads, 0, s>>>(p, C, HW, Nb, xzp, x16, vec, wa, w_per);
  else if (xu) conv_x16_kernel<true, false><<<grid, kThreads, 0, s>>>(p, C, HW, Nb, xzp, x16, vec, wa, w_per);
  else if (wu) conv_x16_kernel<false, true><<<grid, kThreads, 0, s>>>(p, C, HW, Nb, xzp, x16, vec, wa, w_per);
  else conv_x16_kernel<false, false><<<grid, kThreads, 0, s>>>(p, C, HW, Nb, xzp, x16, vec, wa, w_per);
  return cudaGetLastError();
}

size_t im2col_sum_scratch_bytes(long long Nb, long long G, long long H, long long W) {
  return (size_t)Nb * G * H * W * sizeof(int);
}

cudaError_t launch_im2col(const Im2colArgs& a, bool x_u8, int* sum_scratch, cudaStream_t s) {
  const long long P = (long long)a.oH * a.oW;
  const long long Kt = (long long)a.C * a.kH * a.kW;
  if (a.Nb <= 0 || P <= 0 || Kt <= 0) return cudaSuccess;
  if (a.Nb > 65535) return cudaErrorInvalidValue;
  return x_u8 ? convk::im2col_one<true>(a, sum_scratch, s) : convk::im2col_one<false>(a, sum_scratch, s);
}

cudaError_t launch_rows_pitched(const void* src, bool u8, int rows, int cols, __half* dst, long long pitch,
                                int* rowsum, cudaStream_t s) {
  using namespace convk;
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const uint8_t* p = static_cast<const uint8_t*>(src);
  if (u8) rows_pitched_kernel<true><<<rows, kThreads, 0, s>>>(p, cols, dst, pitch, rowsum);
  else rows_pitched_kernel<false><<<rows, kThreads, 0, s>>>(p, cols, dst, pitch, rowsum);
  return cudaGetLastError();
}

}  // namespace qmm
