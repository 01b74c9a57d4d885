// KV append (slot scatter) and copy-on-write block copy, plus the library's
// small runtime entry points (version, status strings, device error word).
//
// Append: cs2680 Lecture 10, §10.3 -- a sequence grows by writing one slot of
// the block its table names for the new position. Block copy: "KV cache
// systems", copy-on-write paragraph -- the first writer of a shared block
// gets a copy of the whole block. Both are pure data movement: each thread
// moves 16-byte vectors, so every warp reads and writes whole 32-byte
// sectors of the 256-byte token rows.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

namespace {
thread_local char g_last_error[256] = "no CUDA error";
}

void record_cuda_error(cudaError_t e) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

namespace ops {

constexpr int kThreads = 256;

// One thread per 16-byte vector of one (token, KV head) row of K or V.
// vec_per_row = head_dim / 8. Launched early behind a step's block copy, it
// loads its rows and slots while the copy runs and waits for the copy only
// before its first store (a token may land in a block the copy fills).
__global__ void __launch_bounds__(kThreads)
append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
              const int64_t* __restrict__ slots, long long rows, int hkv, int vec_per_row, int bt,
              long long slot_limit, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
              uint32_t* err, L2Warm warm) {
    griddep_launch_dependents();  // the attention of a decode step may start its prologue
    const long long per_tensor = rows * vec_per_row;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const char* base = static_cast<const char*>(warm.ptr[r]);
        const long long lines = static_cast<long long>((warm.bytes[r] + 127) / 128);
        for (long long l = gtid; base && l < lines; l += stride) prefetch_l2(base + l * 128);
    }
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < 2 * per_tensor;
         i += stride) {
        const bool is_v = i >= per_tensor;
        const long long j = is_v ? i - per_tensor : i;
        const long long row = j / vec_per_row;  // token * hkv + head
        const int vec = static_cast<int>(j - row * vec_per_row);
        const long long tok = row / hkv;
        const int head = static_cast<int>(row - tok * hkv);
        const uint4 val = is_v ? __ldg(v + j) : __ldg(k + j);
        const long long slot = __ldg(slots + tok);
        griddep_wait();  // the block copies this step launched before us are done
        if (slot < 0) continue;
        if (slot >= slot_limit) {
            if (err && vec == 0 && head == 0 && !is_v) atomicOr(err, PKV_DEVERR_SLOT);
            continue;
        }
        const long long blk = slot / bt;
        const long long pos = slot - blk * bt;
        const long long dst = ((blk * hkv + head) * bt + pos) * vec_per_row + vec;
        if (is_v) v_cache[dst] = val;
        else k_cache[dst] = val;
    }
}

// grid.y = pair, grid.z = 0 (K) / 1 (V); blocks stride over one cache block.
__global__ void __launch_bounds__(kThreads)
copy_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ pairs,
            int num_blocks, long long vec_per_block, uint32_t* err) {
    griddep_launch_dependents();
    const int pr = blockIdx.y;
    const int src = __ldg(pairs + 2 * pr);
    const int dst = __ldg(pairs + 2 * pr + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (err && blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0) atomicOr(err, PKV_DEVERR_BLOCK_ID);
        return;
    }
    uint4* cache = blockIdx.z == 0 ? k_cache : v_cache;
    const uint4* s = cache + static_cast<long long>(src) * vec_per_block;
    uint4* d = cache + static_cast<long long>(dst) * vec_per_block;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < vec_per_block;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        d[i] = s[i];
}

}  // namespace ops
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_version(void) { return 100; }

const char* pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_EINVAL: return "invalid argument";
        case PKV_ENOMEM: return "too few free pages";
        case PKV_ERANGE: return "value out of range";
        case PKV_ECUDA: return "CUDA error";
        case PKV_ENOSPC: return "append past the reserved pages";
        case PKV_EUNSUPPORTED: return "unsupported geometry";
        case PKV_ESTATE: return "inconsistent block-manager state";
        default: return "unknown status";
    }
}

const char* pkv_last_cuda_error(void) { return g_last_error; }

pkv_status pkv_read_device_error(uint32_t* device_error, uint32_t* host_value, int clear, void* stream) {
    if (!device_error || !host_value) return PKV_EINVAL;
    cudaStream_t st = as_stream(stream);
    cudaError_t e = cudaMemcpyAsync(host_value, device_error, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(device_error, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

}  // extern "C"

namespace pkv {

// The decode-attention kernel runs with most of each SM's memory as shared
// memory; giving the cache kernels the same preference spares the SMs a
// reconfiguration between the kernels of a decode step.
static void prefer_shared_carveout() {
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(ops::append_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        cudaFuncSetAttribute(ops::copy_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        cudaGetLastError();  // a refused preference is harmless
    });
}

pkv_status launch_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                         void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                         int block_tokens, uint32_t* device_error, void* stream, const L2Warm* warm,
                         bool early) {
    if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 8 || head_dim % 8 != 0 ||
        block_tokens < 1)
        return PKV_EINVAL;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
    prefer_shared_carveout();
    const int vec_per_row = head_dim / 8;
    const long long rows = static_cast<long long>(num_tokens) * num_kv_heads;
    const long long work = 2 * rows * vec_per_row;
    const int grid = static_cast<int>(std::min<long long>((work + ops::kThreads - 1) / ops::kThreads, 65535));
    const L2Warm none = {{nullptr, nullptr, nullptr}, {0, 0, 0}};
    // early: programmatic stream serialization behind the step's block copy
    // (whose kernel lets dependents start at once); the kernel waits for it
    // before storing.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(ops::kThreads);
    cfg.stream = as_stream(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, ops::append_kernel, static_cast<const uint4*>(k),
                                       static_cast<const uint4*>(v), slot_mapping, rows, num_kv_heads, vec_per_row,
                                       block_tokens, static_cast<long long>(num_blocks) * block_tokens,
                                       static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), device_error,
                                       warm ? *warm : none);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

}  // namespace pkv

extern "C" {

pkv_status pkv_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                      void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                      uint32_t* device_error, void* stream) {
    return launch_append(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, num_kv_heads, head_dim,
                         PKV_BLOCK_TOKENS, device_error, stream, nullptr, false);
}

pkv_status pkv_append_ex(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                         void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                         int block_tokens, uint32_t* device_error, void* stream) {
    return launch_append(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, num_kv_heads, head_dim,
                         block_tokens, device_error, stream, nullptr, false);
}

pkv_status pkv_block_copy(void* k_cache, void* v_cache, const int32_t* src_dst_pairs, int num_pairs,
                          int num_blocks, int num_kv_heads, int head_dim, uint32_t* device_error,
                          void* stream) {
    return pkv_block_copy_ex(k_cache, v_cache, src_dst_pairs, num_pairs, num_blocks, num_kv_heads, head_dim,
                             PKV_BLOCK_TOKENS, device_error, stream);
}

pkv_status pkv_block_copy_ex(void* k_cache, void* v_cache, const int32_t* src_dst_pairs, int num_pairs,
                             int num_blocks, int num_kv_heads, int head_dim, int block_tokens,
                             uint32_t* device_error, void* stream) {
    if (num_pairs < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 8 || head_dim % 8 != 0 ||
        block_tokens < 1)
        return PKV_EINVAL;
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs > 65535) return PKV_ERANGE;
    if (!k_cache || !v_cache || !src_dst_pairs) return PKV_EINVAL;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
    prefer_shared_carveout();
    const long long vec_per_block = static_cast<long long>(num_kv_heads) * block_tokens * head_dim / 8;
    const int gx = static_cast<int>(std::min<long long>((vec_per_block + ops::kThreads - 1) / ops::kThreads, 64));
    dim3 grid(gx, num_pairs, 2);
    ops::copy_kernel<<<grid, ops::kThreads, 0, as_stream(stream)>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src_dst_pairs, num_blocks, vec_per_block,
        device_error);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

}  // extern "C"
