// Internal declarations shared by the host orchestration and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include "../../include/quail.h"

namespace quail {

// Device error word indices.
constexpr int kErrCode = 0;
constexpr int kErrDetail = 1;

}  // namespace quail
