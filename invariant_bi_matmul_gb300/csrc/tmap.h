// tmap.h -- host-side TMA tensor-map encoding with a cache.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace bi {

// 2D bf16 tensor [outer][inner] with a row stride of `stride` elements, tiled in boxes
// of box_inner x box_outer with the given shared-memory swizzle (32, 64 or 128 bytes).
// f16: the elements are IEEE binary16 instead (same size, same layout).
// Returns false if the descriptor cannot be encoded (alignment, stride, driver).
bool tmap_2d_bf16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                  uint64_t stride, uint32_t box_inner, uint32_t box_outer, int swizzle_bytes,
                  bool f16 = false);

// The same tensor viewed in rank 3 as (box_inner-wide column, row, column block), so one
// copy of box (box_inner, box_outer, box_blocks) lands as box_blocks consecutive
// [box_outer x box_inner] tiles in shared memory (K-blocks of a K-major operand).
// Requires inner % box_inner == 0 (the view never reaches past a row).
bool tmap_kblocked_bf16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                        uint64_t stride, uint32_t box_inner, uint32_t box_outer,
                        uint32_t box_blocks, int swizzle_bytes, bool f16 = false);

// 2D byte tensor [outer][inner_bytes] (row stride stride_bytes, a multiple of 16), boxes of
// box_inner bytes x box_outer rows, no swizzle; bytes outside the tensor read as 0.
bool tmap_2d_u8(CUtensorMap* out, const void* ptr, uint64_t inner_bytes, uint64_t outer,
                uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer);
// 3D bf16 tensor [d2][d1][d0] with element strides stride1 (between d1 rows) and
// stride2 (between d2 slabs), boxes box0 x box1 x box2 landing densely in shared memory,
// 128-byte swizzle; elements outside the tensor read as 0.  No cache.
bool tmap_3d_bf16(CUtensorMap* out, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1,
                  uint32_t box2);
// The same for 16-bit elements (inner and box_inner in elements).
bool tmap_2d_u16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                 uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer);

}  // namespace bi
