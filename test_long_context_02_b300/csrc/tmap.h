// TMA tensor-map encoding (host side).
#pragma once
#include <cstdint>
#include <cuda.h>

namespace ttt {

// 2-D bf16 map over a row-major [outer][pitch_elems] array, box {64, box_outer},
// 128-byte swizzle, out-of-range elements read as zero.  False if the driver
// entry point is unavailable or the encoder rejects the arguments.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
              uint32_t box_outer);

}  // namespace ttt
