// Internal declarations shared by the host orchestration and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include "../../include/quail.h"

namespace quail {

// Kernels launched by the current classify call on this thread (reset at the
// call's start; read back through quail_launch_count).
void count_launch();

// fp32 tensor [planes, rows, cols] (cols contiguous; row stride ld, plane
// stride plane_ld elements) for tile stores of box_cols x box_rows x 1, with
// the 128-byte swizzle (box_cols * 4 must be 128). False if the encoding fails.
bool encode_3d_f32_store(void* tm, void* ptr, uint64_t cols, uint64_t rows, uint64_t planes, uint64_t ld,
                         uint64_t plane_ld, uint32_t box_cols, uint32_t box_rows);

// bf16 tensor of the same shape for tile stores of box_cols x box_rows x
// planes (every plane at once), without swizzle (box_cols * 2 a multiple of 16).
bool encode_3d_bf16_store(void* tm, void* ptr, uint64_t cols, uint64_t rows, uint64_t planes, uint64_t ld,
                          uint64_t plane_ld, uint32_t box_cols, uint32_t box_rows);

// Device error word indices.
constexpr int kErrCode = 0;
constexpr int kErrDetail = 1;

}  // namespace quail
