// Host-side TMA tensor-map encoding for 2-D and 3-D bf16 tensors.
#pragma once

#include <cuda.h>

#include <cstdint>

namespace mla {

// A [rows, inner] bf16 tensor with `row_stride_bytes` between rows, read in
// boxes of box_rows x box_inner elements, written to shared memory with the
// given swizzle (box_inner * 2 must equal the swizzle width: 128 or 64
// bytes; 0 = no swizzle).  Elements outside the tensor read as zero.
// Returns false if the encoding fails (bad alignment or sizes).
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                       int swizzle_bytes);

// A [planes, rows, inner] bf16 tensor, boxes of 1 x box_rows x box_inner with
// 128-byte swizzle (box_inner = 64).  Loads outside the tensor read zero;
// stores are clipped to it.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t planes, uint64_t row_stride_bytes, uint64_t plane_stride_bytes,
                       uint32_t box_inner, uint32_t box_rows);
// The same for fp32 elements (box_inner = 32).
bool make_tmap_f32_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                      uint64_t planes, uint64_t row_stride_bytes, uint64_t plane_stride_bytes,
                      uint32_t box_inner, uint32_t box_rows);

// A 4-D bf16 tensor (dims[0] innermost, 64 elements per box row, 128-byte
// swizzle) with byte strides for dims 1..3 in any order; boxes land in shared
// memory with box[3] outermost.
bool make_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4]);

}  // namespace mla
