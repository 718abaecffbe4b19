// Shared definitions of the CUDA library: status word and small helpers.
#pragma once

#include <cstdint>

#include "../../include/attn_b300.h"

namespace attn {

// Device status word: the first failure a kernel records since the host last
// read it (0 = none).  Kernels record instead of trapping, so the context
// stays usable and the host can report the failure.
__device__ int g_status;

__device__ __forceinline__ void record_status(int code) { atomicCAS(&g_status, 0, code); }

// Limit of the waits in a kernel's wind-down after a failure: copies and MMAs a
// CTA has already issued must land before it releases tensor memory and exits,
// so these waits never use less than this, whatever limit the pipeline waits use.
constexpr unsigned long long kDrainTimeoutNs = 2000000000ull;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace attn
