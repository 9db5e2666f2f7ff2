// tmap.h -- host-side TMA tensor-map encoding with a cache.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace bi {

// 2D bf16 tensor [outer][inner] with a row stride of `stride` elements, tiled in boxes
// of box_inner x box_outer with the given shared-memory swizzle (32, 64 or 128 bytes).
// Returns false if the descriptor cannot be encoded (alignment, stride, driver).
bool tmap_2d_bf16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                  uint64_t stride, uint32_t box_inner, uint32_t box_outer, int swizzle_bytes);

}  // namespace bi
