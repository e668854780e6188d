// Host helpers for the CUDA entry points: tensor validation and TMA
// descriptor encoding (through the driver entry point, so that the library
// itself does not link libcuda and loads on machines without a GPU driver).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.h"

namespace bd {

// Checks a bf16/fp32 strided tensor: non-NULL, 16-byte aligned base, byte
// strides multiples of 16 for dims with extent > 1, rows > 0.
int32_t check_tensor(const bd_tensor* t, const char* name, int elem_bytes, int64_t B, int64_t C,
                     int64_t H, bool need_tma);

// Encodes a 5-D tiled TMA map over bf16 [B, C, rows, heads, d] with a box of
// box_rows rows x 64 columns of one head, 128-byte swizzle, zero fill out of bounds.
int32_t make_tmap_bf16(CUtensorMap* map, const bd_tensor* t, int64_t B, int64_t C, int64_t heads,
                       int64_t d, const char* name, int box_rows = 128);

// Encodes a 5-D tiled TMA map over fp32 [B, C, rows, heads, d] with a box of
// box_rows rows x box_cols columns of one head (for reduce-adds): 16 columns take
// the 64-byte swizzle, 32 columns the 128-byte swizzle.
int32_t make_tmap_f32_reduce(CUtensorMap* map, const bd_tensor* t, int64_t B, int64_t C, int64_t heads, int64_t d,
                             const char* name, int box_cols = 16, int box_rows = 128);

// Encodes a 5-D tiled TMA map over bf16 [B, C, rows, heads, d] whose box is whole
// rows of d columns for box_heads heads x box_rows rows, unswizzled (row-major in
// shared memory: head-row h of row r at (r * box_heads + h) * d elements).
int32_t make_tmap_rows_bf16(CUtensorMap* map, const bd_tensor* t, int64_t B, int64_t C, int64_t heads, int64_t d,
                            const char* name, int box_heads, int box_rows);

// Number of SMs of the current device (cached per device).
int32_t sm_count(int* out);

int32_t cuda_fail(cudaError_t e, const char* what);

}  // namespace bd
