// Tensor-memory-accelerator (TMA) descriptors for the kernels, built on the
// host with the driver's cuTensorMapEncodeTiled. The driver entry point is
// looked up at run time through the CUDA runtime, so the library itself does
// not link against the driver library (it still loads on a host without one).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace qmm {

// Encode a 2-D row-major tensor map: `inner` elements per row (contiguous),
// `outer` rows, `row_bytes` between rows, a box of box_inner x box_outer
// elements, the given swizzle. Out-of-bounds elements of a box read as zero.
// Returns cudaErrorInvalidValue on any failure (including no driver).
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                         uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swizzle);

// 3-D variant: dims {inner, mid, outer} with strides {mid_bytes, outer_bytes}
// between consecutive mid and outer indices, box {box_inner, box_mid, 1}.
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                         uint64_t mid, uint64_t outer, uint64_t mid_bytes, uint64_t outer_bytes,
                         uint32_t box_inner, uint32_t box_mid, CUtensorMapSwizzle swizzle);

// Im2col variant (rank 3 to 5, channels innermost: {C, W, N}, {C, W, H, N} or
// {C, W, H, D, N}): dims and elem_strides have `rank` entries, strides_bytes
// rank - 1; lower / upper are the bounding-box corners of the base pixel
// positions, innermost spatial dimension first (rank - 2 entries). A copy
// delivers `pixels` rows of `channels` elements; elements outside the tensor
// read as zero.
cudaError_t make_tmap_im2col(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank,
                             const uint64_t* dims, const uint64_t* strides_bytes, const int* lower, const int* upper,
                             uint32_t channels, uint32_t pixels, const uint32_t* elem_strides,
                             CUtensorMapSwizzle swizzle);

}  // namespace qmm
