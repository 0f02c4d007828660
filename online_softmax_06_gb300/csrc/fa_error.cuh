// fa_error.cuh -- the device error word and the limits of the kernels'
// bounded waits.
#pragma once

#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Kernels OR FA_DEVERR_* bits into the device error word instead of trapping.
// The word lives in fa_api.cu; kernels receive its device address as an
// argument (see device_error_word() in launch.h).
__device__ __forceinline__ void record_device_error(int *word, int bits)
{
    if (word != nullptr)
        atomicOr(word, bits);
}

// A pipeline wait gives up after this much wall time...
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
// ...or after this many polls, whichever comes first.
constexpr uint32_t kWaitMaxPolls = 1u << 30;

}  // namespace fa
