// Host helpers shared by the tensor-core kernels: TMA tensor maps and the SM count.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace moe {

// 2-D bf16 map over [outer, inner] (inner contiguous), box [box_outer, box_inner], 128-byte swizzle.
bool make_map_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer);
// The same over rows `row_stride_bytes` apart (a column slice of a wider matrix).
bool make_map_2d_strided(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                         uint32_t box_inner, uint32_t box_outer);
// The same with 64-byte swizzle (box_inner x 2 bytes = 64: 16-byte units of a
// row permuted by bits 7-8 of their shared-memory address).
bool make_map_2d_strided_sw64(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
// 3-D bf16 map over [d2, d1, d0] (d0 contiguous), box [1, box1, box0], 128-byte swizzle.
bool make_map_3d(CUtensorMap *m, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                 uint32_t box1);
// fp32 versions (outputs written by TMA stores).
bool make_map_2d_f32(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                     uint32_t box_outer);
bool make_map_3d_f32(CUtensorMap *m, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                     uint32_t box1);
// Streaming multiprocessors of the current device.
int sm_count();

}  // namespace moe
