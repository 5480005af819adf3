// Host-side helpers shared by the translation units of libfrt.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "frt.h"

namespace frt {

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline cudaStream_t as_cuda(frt_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Maps the result of a launch to a status without synchronising.
inline frt_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? FRT_OK : FRT_ERR_CUDA;
}

// Number of SMs of the current device (cached per device ordinal).
int sm_count();

// Adds n to the count of kernels this library has launched (or recorded
// into a stream capture); see frt_launch_count.
void note_launches(int n);

}  // namespace frt
