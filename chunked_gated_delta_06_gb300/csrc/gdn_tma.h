// gdn_tma.h -- host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so libgdn.so does not link
// libcuda directly).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdn {

// 3-D bf16 tensor map over rows of `inner` elements (128, or 64 for 64 x 64
// tiles): dims {inner, d1, d2} with byte strides {stride1, stride2} for dims 1
// and 2; box {64, 1, box2}; 128-byte swizzle, out-of-range elements read as
// zero.  Returns false on failure.
bool encode_rows_bf16(CUtensorMap *map, const void *base, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box2,
                      uint64_t inner = 128);

}  // namespace gdn
