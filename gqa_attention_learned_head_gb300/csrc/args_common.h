// args_common.h -- what every kernel family's launch interface shares: the
// fixed head dimension and page size.  Internal to libsinkattn.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sinkattn {

constexpr int kHeadDim = 64;
constexpr int kPageSize = 16;

}  // namespace sinkattn
