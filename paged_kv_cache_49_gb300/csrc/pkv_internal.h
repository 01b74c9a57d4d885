// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/pkv.h"

namespace pkv {

// Record a CUDA error for pkv_last_cuda_error (per host thread).
void record_cuda_error(cudaError_t e);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace pkv
