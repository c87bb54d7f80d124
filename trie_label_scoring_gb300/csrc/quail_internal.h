// Internal declarations shared by the host orchestration and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include "../../include/quail.h"

namespace quail {

// Kernels launched by the current classify call on this thread (reset at the
// call's start; read back through quail_launch_count).
void count_launch();

// Device error word indices.
constexpr int kErrCode = 0;
constexpr int kErrDetail = 1;

}  // namespace quail
