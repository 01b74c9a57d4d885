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

// Read-only inputs of a following kernel that the append kernel warms in L2
// while it runs (used by pkv_decode_step for the attention's inputs).
struct L2Warm {
    const void* ptr[3];
    size_t bytes[3];
};

// pkv_append's launch, optionally warming L2 with `warm` (may be null).
// early: launched with programmatic stream serialization, allowed only right
// behind a kernel of this library that writes none of the append's inputs
// (the step's block copy): the kernel loads its rows first and waits for
// that kernel before storing.
pkv_status launch_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                         void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                         int block_tokens, uint32_t* device_error, void* stream, const L2Warm* warm,
                         bool early);

}  // namespace pkv
