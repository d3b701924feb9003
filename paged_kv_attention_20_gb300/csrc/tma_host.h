// Host-side tensor-map encoding (cuTensorMapEncodeTiled resolved through the
// runtime's driver entry point, so the library needs no libcuda link).
#pragma once

#include <cuda.h>
#include <cstdint>

namespace pa {

// 3-D map over 16-bit elements: dims {d0 (contiguous), d1, d2}, byte strides
// of dims 1 and 2, box {b0, b1, b2}.  Returns false if the driver entry point
// is missing or the encoding is rejected.
bool encode_map_3d(CUtensorMap *map, const void *base, bool bf16, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                   CUtensorMapSwizzle swizzle);

// 2-D map over 16-bit elements: dims {d0 (contiguous), d1}, byte stride of dim 1, box {b0, b1}.
bool encode_map_2d(CUtensorMap *map, const void *base, bool bf16, uint64_t d0, uint64_t d1, uint64_t stride1,
                   uint32_t b0, uint32_t b1, CUtensorMapSwizzle swizzle);

bool tma_available();

}  // namespace pa
