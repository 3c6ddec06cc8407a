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

}  // namespace qmm
