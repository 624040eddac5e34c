// Host-side creation of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query; no libcuda link needed).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace q4k {

// 3-D uint8 tensor: dims[0] innermost (bytes), strides[i] = byte stride of
// dims[i+1]; box[i] elements per dimension; out-of-range elements read as 0.
// Returns false when the driver rejects the description.
bool encode_tmap_u8_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                       const uint64_t strides[2], const uint32_t box[3]);

// 2-D tensor of `dtype` elements: dim0 innermost, row stride in bytes;
// box0 x box1 elements per copy, with the given shared-memory swizzle.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
                    uint64_t dim1, uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle);

}  // namespace q4k
