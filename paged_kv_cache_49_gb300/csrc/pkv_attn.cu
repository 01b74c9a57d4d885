// Paged decode attention for sm_103a: the launches and the C ABI around
// decode_kernel (pkv_decode_kernel.cuh), the host-buffer step with its staging
// kernel, and cascade attention (prefix_kernel, cascade_merge_kernel).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"
#include "pkv_decode_kernel.cuh"

namespace pkv {
namespace attn {

// ---------------------------------------------------------------------------
// host side

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// View of a cache as token rows (num_blocks * Hkv * block_tokens rows of 128
// bf16), 3-D: {64 columns, rows, 2 column halves} with the halves 128 bytes
// apart, so that one box of {64, min(16, block tokens), 2} brings that many
// rows of one (block, KV head) -- 4 KB, or 2 KB for 8-token blocks -- laid out
// in shared memory as the two halves one after the other, each in the
// 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* base, int num_blocks, int hkv, int block_tokens) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t rows = static_cast<cuuint64_t>(num_blocks) * hkv * block_tokens;
    cuuint64_t dims[3] = {64, rows, 2};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDim) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(block_tokens < kTok ? block_tokens : kTok), 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);

// The instantiation for a block size (8, 16, 32 or 64 tokens), skipped tiles
// (16-token blocks only) and merge slots (1 or 2), else null.
template <int S>
KernelFn kernel_for_slots(int block_tokens, bool skip) {
    if (skip) return block_tokens == PKV_BLOCK_TOKENS ? decode_kernel<PKV_BLOCK_TOKENS, true, S> : nullptr;
    switch (block_tokens) {
        case 8: return decode_kernel<8, false, S>;
        case 16: return decode_kernel<16, false, S>;
        case 32: return decode_kernel<32, false, S>;
        case 64: return decode_kernel<64, false, S>;
        default: return nullptr;
    }
}

KernelFn kernel_for(int block_tokens, bool skip, int slots) {
    return slots == 1 ? kernel_for_slots<1>(block_tokens, skip) : kernel_for_slots<2>(block_tokens, skip);
}

// The CUDA-core variant of the consumer math (16-token blocks), for group
// sizes 4 and 8, else null.
KernelFn kernel_fma_for(int slots, int group) {
    if (group == 4) return slots == 1 ? decode_kernel<PKV_BLOCK_TOKENS, false, 1, 4> : decode_kernel<PKV_BLOCK_TOKENS, false, 2, 4>;
    if (group == 8) return slots == 1 ? decode_kernel<PKV_BLOCK_TOKENS, false, 1, 8> : decode_kernel<PKV_BLOCK_TOKENS, false, 2, 8>;
    return nullptr;
}

struct DeviceInfo {
    bool ok = false;
    int sm_count = 0;
};

// Per device, once: allow every instantiation its largest dynamic shared memory.
DeviceInfo device_info() {
    static std::mutex mu;
    static std::vector<DeviceInfo> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return {};
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1);
    DeviceInfo& d = cache[dev];
    if (d.ok) return d;
    cudaError_t e = cudaSuccess;
    for (int slots : {1, 2})
        for (int bt : {8, 16, 32, 64})
            for (bool skip : {false, true}) {
                const KernelFn fn = kernel_for(bt, skip, slots);
                if (e == cudaSuccess && fn)
                    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem_bytes(PKV_ATTN_MAX_SEQS, skip, slots)));
            }
    for (int slots : {1, 2})
        for (int group : {4, 8})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kernel_fma_for(slots, group), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes(PKV_ATTN_MAX_SEQS, false, slots)));
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return {};
    }
    d.ok = true;
    return d;
}

// The launch shape for a batch of num_seqs: every CTA that fits at once (the
// shared-memory prefix sum grows with num_seqs). Two merge slots while two
// CTAs per SM still fit with them, else one when that keeps two per SM.
struct KernelConfig {
    int grid = 0;  // 0 on error
    int slots = 2;
    size_t smem = 0;
    KernelFn fn = nullptr;
};

KernelConfig config_for(int num_seqs, int block_tokens = PKV_BLOCK_TOKENS, bool skip = false) {
    const DeviceInfo d = device_info();
    if (!d.ok || !kernel_for(block_tokens, skip, 2)) return {};
    // Cached per (device, block size, skip, shared memory size), so that a
    // call made while a stream is being captured into a graph issues no CUDA
    // query.
    static std::mutex mu;
    static std::map<std::pair<int, size_t>, KernelConfig> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const std::pair<int, size_t> key{(dev * 128 + block_tokens) * 2 + (skip ? 1 : 0), smem_bytes(num_seqs, skip, 2)};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    KernelConfig best;
    for (int slots : {2, 1}) {
        KernelConfig c;
        c.slots = slots;
        c.fn = kernel_for(block_tokens, skip, slots);
        c.smem = smem_bytes(num_seqs, skip, slots);
        int per_sm = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c.fn, kThreads, c.smem);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return {};
        }
        c.grid = std::min(d.sm_count * per_sm, kMaxCtas);
        if (c.grid > best.grid) best = c;
        if (per_sm >= 2) break;
    }
    if (best.grid < 1) return {};
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = best;
    return best;
}

int grid_for(int num_seqs, int block_tokens = PKV_BLOCK_TOKENS, bool skip = false) {
    return config_for(num_seqs, block_tokens, skip).grid;
}

struct Launch {
    CUtensorMap tm_k, tm_v;
    Params prm;
    int grid;
    int slots;
    size_t smem;
    KernelFn fn;
};

// The default grid: every CTA that fits, unless the block tables bound the
// batch's work (its cost units, tiles plus the per-run charge, with every row
// full) to fewer than kMinCostPerCta per CTA: a tiny batch spread over every
// CTA cuts each run into one-tile pieces whose cross-CTA merges cost more
// than the tiles (4 sequences of at most 13 tiles: 14.3 µs on 304 CTAs, 12.3
// µs on 128; one KV head, 6 sequences: 20.5 µs against 18.4 µs on 8-64).
constexpr int kMinCostPerCta = 4;

int default_grid(int resident, int num_seqs, int num_kv_heads, int max_blocks_per_seq, int block_tokens) {
    const long long row_tiles = (static_cast<long long>(max_blocks_per_seq) * block_tokens + kTok - 1) / kTok;
    const long long bound = static_cast<long long>(num_kv_heads) * num_seqs * (row_tiles + kPieceCost);
    const long long want = (bound + kMinCostPerCta - 1) / kMinCostPerCta;
    return static_cast<int>(std::max<long long>(1, std::min<long long>(resident, want)));
}

// Validate pkv_attn_decode's arguments and build its launch.
pkv_status prepare(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                   int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_q_heads,
                   int num_kv_heads, int head_dim, int num_blocks, float scale, int num_ctas, void* workspace,
                   size_t workspace_bytes, void* out, Launch* L, int block_tokens = PKV_BLOCK_TOKENS) {
    if (!kernel_for(block_tokens, false, 2)) return PKV_EUNSUPPORTED;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace || !out)
        return PKV_EINVAL;
    if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || num_blocks < 1 ||
        max_blocks_per_seq < 1 || num_ctas < 0 || num_ctas > kMaxCtas || !std::isfinite(scale))
        return PKV_EINVAL;
    if (num_seqs > PKV_ATTN_MAX_SEQS || head_dim != PKV_ATTN_HEAD_DIM ||
        num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > PKV_ATTN_MAX_GROUP)
        return PKV_EUNSUPPORTED;
    if (static_cast<long long>(num_blocks) * num_kv_heads * block_tokens >= (1ll << 31) ||
        static_cast<long long>(num_seqs) * max_blocks_per_seq >= (1ll << 31) ||
        static_cast<long long>(max_blocks_per_seq) * block_tokens >= (1ll << 31) ||
        static_cast<long long>(num_kv_heads) * num_seqs * ((static_cast<long long>(max_blocks_per_seq) * block_tokens + kTok - 1) / kTok + kPieceCost) >= (1ll << 30))
        return PKV_ERANGE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return PKV_EINVAL;
    const KernelConfig kc = config_for(num_seqs, block_tokens);
    if (kc.grid < 1) return PKV_ECUDA;
    int grid = num_ctas > 0 ? num_ctas : default_grid(kc.grid, num_seqs, num_kv_heads, max_blocks_per_seq, block_tokens);
    if (workspace_bytes < kWsFixed + kWsPerCta) return PKV_EINVAL;
    const long long fit = static_cast<long long>((workspace_bytes - kWsFixed) / kWsPerCta);
    if (grid > fit) {
        if (num_ctas > 0) return PKV_EINVAL;
        grid = static_cast<int>(fit);
    }
    if (!make_cache_map(&L->tm_k, k_cache, num_blocks, num_kv_heads, block_tokens) ||
        !make_cache_map(&L->tm_v, v_cache, num_blocks, num_kv_heads, block_tokens))
        return PKV_ECUDA;
    Params& prm = L->prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = num_kv_heads;
    prm.group = num_q_heads / num_kv_heads;
    prm.max_blocks = max_blocks_per_seq;
    prm.cap_tokens = max_blocks_per_seq * block_tokens;
    prm.num_blocks = num_blocks;
    prm.scale_log2 = scale * 1.4426950408889634f;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    prm.err = reinterpret_cast<uint32_t*>(ws);
    prm.counters = reinterpret_cast<int*>(ws + kWsHeader);
    prm.group_counters = prm.counters + kMaxCtas;
    prm.partials = reinterpret_cast<float*>(ws + kWsFixed);
    prm.skip_tiles = nullptr;
    prm.side = nullptr;
    prm.stop_tiles = -1;
    L->grid = grid;
    L->slots = kc.slots;
    L->fn = kc.fn;
    L->smem = kc.smem;
    return PKV_OK;
}

// early: launch with programmatic stream serialization, so that the kernel's
// prologue overlaps the previous kernel on the stream (see griddep_wait).
pkv_status launch(const Launch& L, cudaStream_t stream, bool early) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, L.fn, L.tm_k, L.tm_v, L.prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

// Bring a step's packed inputs from pinned host memory that the device
// addresses directly into device memory, in 16-byte words: every load
// crosses the host link at once, all issued before any is stored (four per
// thread), where a copy engine takes several times as long for a step's few
// MB. Of the block tables only each row's entries up to ceil(context_len /
// 16) cross (the kernels never read past them): a batch padded to its
// longest row (the 70B batch: 256 rows of 8,192 entries, 8 MB, of which 0.6
// MB are live) would otherwise move mostly padding.
//  - blocks [0, dense_blocks): the words outside the table region, grid-
//    stride;
//  - the other blocks: one warp per task of up to kStageRowWords words of
//    one table row (row r's tasks r * row_tasks ..), which reads the row's
//    context length from the host buffer first.
constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 4;
constexpr int kStageRowWords = 32 * kStageUnroll;  // 2 KB of one row per warp task

struct StageArgs {
    const uint4* src;
    uint4* dst;
    size_t n16;                          // words in the packed buffer
    size_t tab_lo, tab_hi;               // the table region, in words
    size_t tab_byte0;                    // its first byte
    const int32_t* ctx;                  // context lengths in the host buffer (device view)
    int rows, row_entries, row_tasks;    // table rows, entries per row, warp tasks per row
    int dense_blocks;
};

__global__ void __launch_bounds__(kStageThreads) stage_kernel(const StageArgs a) {
    if (static_cast<int>(blockIdx.x) < a.dense_blocks) {
        const size_t n = a.n16 - (a.tab_hi - a.tab_lo);  // words outside the table region
        const size_t stride = static_cast<size_t>(a.dense_blocks) * kStageThreads;
        auto at = [&](size_t i) { return i < a.tab_lo ? i : i + (a.tab_hi - a.tab_lo); };
        size_t i = static_cast<size_t>(blockIdx.x) * kStageThreads + threadIdx.x;
        for (; i + (kStageUnroll - 1) * stride < n; i += kStageUnroll * stride) {
            uint4 v[kStageUnroll];
#pragma unroll
            for (int u = 0; u < kStageUnroll; ++u) v[u] = a.src[at(i + u * stride)];
#pragma unroll
            for (int u = 0; u < kStageUnroll; ++u) a.dst[at(i + u * stride)] = v[u];
        }
        for (; i < n; i += stride) a.dst[at(i)] = a.src[at(i)];
        return;
    }
    const int lane = threadIdx.x & 31;
    const long long task = (static_cast<long long>(blockIdx.x) - a.dense_blocks) * (kStageThreads / 32) + (threadIdx.x >> 5);
    if (task >= static_cast<long long>(a.rows) * a.row_tasks) return;
    const int r = static_cast<int>(task / a.row_tasks);
    const int c = static_cast<int>(task - static_cast<long long>(r) * a.row_tasks);
    const int len = a.ctx[r];
    const int live = len <= 0 ? 0 : min((len + PKV_BLOCK_TOKENS - 1) / PKV_BLOCK_TOKENS, a.row_entries);
    if (live == 0) return;
    const size_t byte_lo = a.tab_byte0 + static_cast<size_t>(r) * a.row_entries * 4;
    const size_t w_lo = byte_lo / 16 + static_cast<size_t>(c) * kStageRowWords;  // this task's first word
    const size_t w_end = (byte_lo + static_cast<size_t>(live) * 4 + 15) / 16;     // past the row's last live word
    if (w_lo >= w_end) return;
    size_t w[kStageUnroll];
    uint4 v[kStageUnroll];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
        w[u] = w_lo + u * 32 + lane;
        if (w[u] < w_end) v[u] = a.src[w[u]];
    }
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u)
        if (w[u] < w_end) a.dst[w[u]] = v[u];
}

}  // namespace attn
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_attn_default_ctas(int num_seqs) {
    if (num_seqs < 1 || num_seqs > PKV_ATTN_MAX_SEQS) return 0;
    return attn::grid_for(num_seqs);
}

int pkv_attn_launch_ctas(int num_seqs, int num_kv_heads, int max_blocks_per_seq, int block_tokens) {
    if (num_seqs < 1 || num_seqs > PKV_ATTN_MAX_SEQS || num_kv_heads < 1 || max_blocks_per_seq < 1 ||
        !attn::kernel_for(block_tokens, false, 2))
        return 0;
    const int resident = attn::grid_for(num_seqs, block_tokens);
    if (resident < 1) return 0;
    return attn::default_grid(resident, num_seqs, num_kv_heads, max_blocks_per_seq, block_tokens);
}

size_t pkv_attn_workspace_size(int num_seqs, int num_kv_heads) {
    if (num_seqs <= 0 || num_kv_heads <= 0 || num_seqs > PKV_ATTN_MAX_SEQS) return 0;
    const int grid = attn::grid_for(num_seqs);
    if (grid < 1) return 0;
    return attn::workspace_bytes(grid);
}

size_t pkv_attn_workspace_fixed_bytes(void) { return attn::kWsFixed; }

pkv_status pkv_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < attn::kWsHeader) return PKV_EINVAL;
    const cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, as_stream(stream));
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

pkv_status pkv_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int num_blocks, float scale,
                           int num_ctas, void* workspace, size_t workspace_bytes, void* out,
                           void* stream) {
    attn::Launch L;
    const pkv_status st = attn::prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                        num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, scale,
                                        num_ctas, workspace, workspace_bytes, out, &L);
    if (st != PKV_OK) return st;
    return attn::launch(L, as_stream(stream), false);
}

pkv_status pkv_attn_decode_cuda_cores(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int num_blocks, float scale, int num_ctas,
                                      void* workspace, size_t workspace_bytes, void* out, void* stream) {
    attn::Launch L;
    pkv_status st = attn::prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                  num_q_heads, num_kv_heads, head_dim, num_blocks, scale, num_ctas, workspace,
                                  workspace_bytes, out, &L);
    if (st != PKV_OK) return st;
    const attn::KernelFn fn = attn::kernel_fma_for(L.slots, num_q_heads / num_kv_heads);
    if (!fn) return PKV_EUNSUPPORTED;
    if (num_ctas == 0) {  // every CTA of this instantiation that fits at once
        const attn::DeviceInfo d = attn::device_info();
        int per_sm = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, attn::kThreads, L.smem);
        if (e != cudaSuccess || per_sm < 1 || !d.ok) {
            if (e != cudaSuccess) record_cuda_error(e);
            return PKV_ECUDA;
        }
        L.grid = std::min(L.grid, d.sm_count * per_sm);
    }
    L.fn = fn;
    return attn::launch(L, as_stream(stream), false);
}

pkv_status pkv_attn_decode_wait_test(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_dim, int num_blocks, float scale, int num_ctas,
                                     void* workspace, size_t workspace_bytes, void* out, int stop_tiles,
                                     void* stream) {
    if (stop_tiles < 0) return PKV_EINVAL;
    attn::Launch L;
    const pkv_status st = attn::prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                        num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, scale,
                                        num_ctas, workspace, workspace_bytes, out, &L);
    if (st != PKV_OK) return st;
    L.prm.stop_tiles = stop_tiles;
    return attn::launch(L, as_stream(stream), false);
}

pkv_status pkv_attn_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                              int head_dim, int num_blocks, int block_tokens, float scale, int num_ctas,
                              void* workspace, size_t workspace_bytes, void* out, void* stream) {
    attn::Launch L;
    const pkv_status st = attn::prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                        num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, scale,
                                        num_ctas, workspace, workspace_bytes, out, &L, block_tokens);
    if (st != PKV_OK) return st;
    return attn::launch(L, as_stream(stream), false);
}

}  // extern "C"

namespace {

// The checks of pkv_decode_step that come before anything is enqueued; on
// success L holds the attention launch.
pkv_status check_step(const void* k_new, const void* v_new, const int64_t* slot_mapping, int num_new_tokens,
                      const int32_t* src_dst_pairs, int num_pairs, void* k_cache, void* v_cache, int num_blocks,
                      const void* q, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                      int head_dim, float scale, int num_ctas, void* workspace, size_t workspace_bytes,
                      void* out, attn::Launch* L) {
    if (num_new_tokens < 0 || num_pairs < 0) return PKV_EINVAL;
    const pkv_status st =
        attn::prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                      num_kv_heads, head_dim, num_blocks, scale, num_ctas, workspace, workspace_bytes, out, L);
    if (st != PKV_OK) return st;
    if (num_pairs > 65535) return PKV_ERANGE;
    if ((num_pairs > 0 && !src_dst_pairs) || (num_new_tokens > 0 && (!k_new || !v_new || !slot_mapping)))
        return PKV_EINVAL;
    if (num_new_tokens > 0 && (!aligned16(k_new) || !aligned16(v_new))) return PKV_EINVAL;
    return PKV_OK;
}

// The launches of a checked step: block copy, append (warming L2 with the
// attention's cold inputs while it runs), attention launched early.
pkv_status enqueue_step(const attn::Launch& L, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                        int num_new_tokens, const int32_t* src_dst_pairs, int num_pairs, void* k_cache,
                        void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                        uint32_t* device_error, void* stream) {
    pkv_status st = PKV_OK;
    if (num_pairs > 0) {
        st = pkv_block_copy(k_cache, v_cache, src_dst_pairs, num_pairs, num_blocks, num_kv_heads, head_dim,
                            device_error, stream);
        if (st != PKV_OK) return st;
    }
    if (num_new_tokens > 0) {
        const attn::Params& p = L.prm;
        const L2Warm warm = {{p.block_tables, p.q, p.context_lens},
                             {static_cast<size_t>(p.num_seqs) * p.max_blocks * 4,
                              static_cast<size_t>(p.num_seqs) * p.num_q_heads * head_dim * 2,
                              static_cast<size_t>(p.num_seqs) * 4}};
        // behind the step's block copies the append starts early and waits
        // for them before its stores (it reads nothing they write)
        st = launch_append(k_new, v_new, slot_mapping, num_new_tokens, k_cache, v_cache, num_blocks, num_kv_heads,
                           head_dim, PKV_BLOCK_TOKENS, device_error, stream, &warm, num_pairs > 0);
        if (st != PKV_OK) return st;
    }
    return attn::launch(L, as_stream(stream), num_pairs > 0 || num_new_tokens > 0);
}

size_t align_up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

pkv_status pkv_decode_step(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                           int num_new_tokens, const int32_t* src_dst_pairs, int num_pairs,
                           void* k_cache, void* v_cache, int num_blocks, const void* q,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, float scale, int num_ctas, void* workspace,
                           size_t workspace_bytes, void* out, uint32_t* device_error, void* stream) {
    attn::Launch L;
    const pkv_status st = check_step(k_new, v_new, slot_mapping, num_new_tokens, src_dst_pairs, num_pairs, k_cache,
                                     v_cache, num_blocks, q, block_tables, max_blocks_per_seq, context_lens,
                                     num_seqs, num_q_heads, num_kv_heads, head_dim, scale, num_ctas, workspace,
                                     workspace_bytes, out, &L);
    if (st != PKV_OK) return st;
    return enqueue_step(L, k_new, v_new, slot_mapping, num_new_tokens, src_dst_pairs, num_pairs, k_cache, v_cache,
                        num_blocks, num_kv_heads, head_dim, device_error, stream);
}

pkv_status pkv_step_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                           int num_pairs, pkv_step_layout_t* layout) {
    if (!layout || num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || max_blocks_per_seq < 1 ||
        num_pairs < 0)
        return PKV_EINVAL;
    if (num_seqs > PKV_ATTN_MAX_SEQS || num_pairs > 65535) return PKV_ERANGE;
    const size_t B = static_cast<size_t>(num_seqs);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up256(off + bytes);
        return at;
    };
    layout->q = take(B * num_q_heads * head_dim * 2);
    layout->k_new = take(B * num_kv_heads * head_dim * 2);
    layout->v_new = take(B * num_kv_heads * head_dim * 2);
    layout->slot_mapping = take(B * 8);
    layout->block_tables = take(B * max_blocks_per_seq * 4);
    layout->context_lens = take(B * 4);
    layout->src_dst_pairs = take(static_cast<size_t>(num_pairs) * 8);  // last: no other offset depends on it
    layout->bytes = off;
    return PKV_OK;
}

pkv_status pkv_decode_step_host(const void* host_packed, void* device_staging, int num_pairs, void* k_cache,
                                void* v_cache, int num_blocks, int max_blocks_per_seq, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, float scale, int num_ctas,
                                void* workspace, size_t workspace_bytes, void* device_out, void* host_out,
                                uint32_t* device_error, void* stream) {
    if (!host_packed || !device_staging || !host_out || !device_out) return PKV_EINVAL;
    if (reinterpret_cast<uintptr_t>(device_staging) & 255u) return PKV_EINVAL;
    pkv_step_layout_t lay;
    pkv_status st = pkv_step_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_pairs,
                                    &lay);
    if (st != PKV_OK) return st;
    uint8_t* d = static_cast<uint8_t*>(device_staging);
    const void* q = d + lay.q;
    const void* k_new = d + lay.k_new;
    const void* v_new = d + lay.v_new;
    const int64_t* slots = reinterpret_cast<const int64_t*>(d + lay.slot_mapping);
    const int32_t* pairs = num_pairs > 0 ? reinterpret_cast<const int32_t*>(d + lay.src_dst_pairs) : nullptr;
    const int32_t* tables = reinterpret_cast<const int32_t*>(d + lay.block_tables);
    const int32_t* ctx = reinterpret_cast<const int32_t*>(d + lay.context_lens);
    // Host buffers that are pinned memory the device can address are used in
    // place: the inputs are staged by a kernel that reads them across the host
    // link, and the output rows go straight to host_out (the attention's
    // stores cross the link as it finishes pieces). Pageable buffers take a
    // copy each way.
    auto device_view = [](const void* h) -> void* {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, h) == cudaSuccess)
            return pa.type == cudaMemoryTypeHost ? pa.devicePointer : nullptr;
        cudaGetLastError();  // pageable memory: not an error here
        return nullptr;
    };
    void* direct = device_view(host_out);
    const void* src = device_view(host_packed);
    if (reinterpret_cast<uintptr_t>(src) & 15u) src = nullptr;
    attn::Launch L;
    st = check_step(k_new, v_new, slots, num_seqs, pairs, num_pairs, k_cache, v_cache, num_blocks, q, tables,
                    max_blocks_per_seq, ctx, num_seqs, num_q_heads, num_kv_heads, head_dim, scale, num_ctas,
                    workspace, workspace_bytes, direct ? direct : device_out, &L);
    if (st != PKV_OK) return st;
    cudaStream_t s = as_stream(stream);
    cudaError_t e = cudaSuccess;
    if (src) {
        attn::StageArgs a;
        a.src = static_cast<const uint4*>(src);
        a.dst = static_cast<uint4*>(device_staging);
        a.n16 = lay.bytes / 16;  // lay.bytes and every field offset are multiples of 256
        a.tab_lo = lay.block_tables / 16;
        a.tab_hi = lay.context_lens / 16;  // the table region, with its padding to 256 bytes
        a.tab_byte0 = lay.block_tables;
        a.ctx = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(src) + lay.context_lens);
        a.rows = num_seqs;
        a.row_entries = max_blocks_per_seq;
        // a row's words can start mid-word: one word more than its length
        a.row_tasks = static_cast<int>((static_cast<size_t>(max_blocks_per_seq) * 4 / 16 + 1 + attn::kStageRowWords - 1) /
                                       attn::kStageRowWords);
        const size_t per_block = static_cast<size_t>(attn::kStageThreads) * attn::kStageUnroll;
        const size_t dense = a.n16 - (a.tab_hi - a.tab_lo);
        a.dense_blocks = static_cast<int>(std::max<size_t>(1, std::min<size_t>((dense + per_block - 1) / per_block, 4096)));
        const size_t tasks = static_cast<size_t>(a.rows) * a.row_tasks;
        const size_t task_blocks = (tasks + attn::kStageThreads / 32 - 1) / (attn::kStageThreads / 32);
        attn::stage_kernel<<<static_cast<unsigned>(a.dense_blocks + task_blocks), attn::kStageThreads, 0, s>>>(a);
        e = cudaGetLastError();
    } else {
        e = cudaMemcpyAsync(device_staging, host_packed, lay.bytes, cudaMemcpyHostToDevice, s);
    }
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    st = enqueue_step(L, k_new, v_new, slots, num_seqs, pairs, num_pairs, k_cache, v_cache, num_blocks,
                      num_kv_heads, head_dim, device_error, stream);
    if (st != PKV_OK || direct) return st;
    e = cudaMemcpyAsync(host_out, device_out, static_cast<size_t>(num_seqs) * num_q_heads * head_dim * 2,
                        cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Cascade attention: shared prefix blocks read once for all their sharers.
//
// Sequences that share their leading blocks (a prompt forked into parallel
// samples, requests of one prefix group) would otherwise each stream the same
// prefix from HBM ("KV cache systems" and cs2680 Lecture 10, §10.4: the shared
// blocks are one copy in memory; here they are also one read). A decode step
// over such a batch runs three kernels:
//  1. prefix_kernel: for every group, KV head and 32-row chunk of the group's
//     query rows (sharers x heads of the GQA group), one pass over at most 64
//     shared tiles, all four consumer warps reading every tile for 8 rows
//     each; each pass leaves fp32 partials (output, max, sum) per row.
//  2. decode_kernel with skip_tiles: the private rest of every sequence; a
//     sequence with skipped tiles leaves its fp32 result in `side`.
//  3. cascade_merge_kernel: per grouped (sequence, KV head), the log-sum-exp
//     merge of its prefix partials and its private result, in a fixed order.
// The pages speak of sharing the memory only; sharing the reads is this
// library's own step, and it changes only the order of the sums.

namespace pkv {
namespace attn {

constexpr int kPfxRows = 32;     // query rows per prefix item: 8 per consumer warp
constexpr int kPfxTiles = 64;    // shared tiles per prefix item at most
constexpr int kPfxThreads = kConsumers + 32;
constexpr int kPfxStages = 8;       // ring depth of the prefix pass
constexpr int kPfxCtasPerSm = 3;    // resident prefix CTAs per SM (shared memory and registers)
constexpr int kPfxOffBar = kPfxStages * kStageBytes;
constexpr size_t kPfxSmem = 1024 + kPfxOffBar + 2 * kPfxStages * 8 + 64;

struct PrefixParams {
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    int max_blocks;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int num_blocks;
    float scale_log2;
    const int32_t* members;  // sequence ids of each group's sharers, group after group
    const int4* items;       // x: first sharer (index into members), y: valid rows,
                             // z: KV head | tiles << 16, w: first shared tile
    int num_items;
    uint32_t* err;
    float* wpart;            // [num_items][kPfxRows][kORow]
};

__global__ void __launch_bounds__(kPfxThreads, kPfxCtasPerSm)
prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const PrefixParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = p.group;
    const int Hkv = p.num_kv_heads;
    const uint32_t bar0 = smem_u32(smem + kPfxOffBar);
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kPfxStages + i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kPfxOffBar + 2 * kPfxStages * 8);
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (tid == 0) {
        for (int i = 0; i < kPfxStages; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), kConsumerWarps);  // every consumer warp reads every stage
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        const uint64_t policy = policy_evict_first();
        int stage = 0, issued = 0;
        uint32_t sphase = 0;
        for (int it = blockIdx.x; it < p.num_items; it += gridDim.x) {
            const int4 item = p.items[it];
            const int g = item.z & 0xffff, n = item.z >> 16;
            const int32_t* row = p.block_tables + static_cast<size_t>(__ldg(p.members + item.x)) * p.max_blocks;
            for (int j0 = 0; j0 < n; j0 += 32) {
                int y0 = 0;
                if (j0 + lane < n) {
                    int bid = __ldg(row + item.w + j0 + lane);
                    if (bid < 0 || bid >= p.num_blocks) {
                        if (p.err) atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
                        bid = 0;
                    }
                    y0 = (bid * Hkv + g) * kTok;
                }
                const int cnt = min(32, n - j0);
                for (int jj = 0; jj < cnt; ++jj) {
                    const int ya = __shfl_sync(0xffffffffu, y0, jj);
                    if (lane == 0 && mbar_wait(empty_bar(stage), sphase ^ 1u, abort_flag, p.err)) {
                        const uint32_t fb = full_bar(stage);
                        mbar_arrive_expect_tx(fb, kStageBytes);
                        const uint32_t dst = smem_u32(smem + stage * kStageBytes);
                        tma_load_3d(dst, &tm_k, 0, ya, 0, fb, policy);
                        tma_load_3d(dst + kBlockBytes, &tm_v, 0, ya, 0, fb, policy);
                        ++issued;
                    }
                    if (++stage == kPfxStages) { stage = 0; sphase ^= 1u; }
                }
            }
        }
        if (lane == 0) {  // no copy may land after the CTA exits (bounded waits; after an abort, a grace period first)
            if (*abort_flag) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < kDrainGraceNs) {
                }
            }
            volatile int never = 0;
            for (int i = max(0, issued - kPfxStages); i < issued; ++i)
                mbar_wait(full_bar(i % kPfxStages), static_cast<uint32_t>((i / kPfxStages) & 1), &never, nullptr);
        }
        return;
    }

    // consumer warps: rows 8 * warp + (0..7) of each item
    const int r = lane >> 2;
    const int c = lane & 3;
    const uint32_t k_row_off = static_cast<uint32_t>(lane & 15) * 128u;
    const int k_sw = lane & 7;
    const int k_hi = lane >> 4;
    const int v_mat = lane >> 3;
    const uint32_t v_row_off = static_cast<uint32_t>((lane & 7) + ((v_mat >> 1) << 3)) * 128u;
    const int v_sw = lane & 7;
    const float NEG_INF = -INFINITY;
    int gi = 0;  // the CTA's tile count so far: stage gi % kPfxStages
    for (int it = blockIdx.x; it < p.num_items; it += gridDim.x) {
        const int4 item = p.items[it];
        const int g = item.z & 0xffff, n = item.z >> 16;
        const int row = 8 * warp + r;  // this lane's query row (mma column) in the item
        const bool valid_row = row < item.y;
        uint32_t qb[16];
        {
            const int seq = valid_row ? __ldg(p.members + item.x + row / G) : 0;
            const uint32_t* qg = reinterpret_cast<const uint32_t*>(
                p.q + (static_cast<size_t>(seq) * p.num_q_heads + static_cast<size_t>(g) * G + row % G) * kDim) + c;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qb[2 * ks] = valid_row ? __ldg(qg + ks * 8) : 0u;
                qb[2 * ks + 1] = valid_row ? __ldg(qg + ks * 8 + 4) : 0u;
            }
        }
        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
        float o[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        for (int t = 0; t < n; ++t, ++gi) {
            const int st = gi % kPfxStages;
            // released only once seen landed (an abort's early return must not free a stage in flight)
            const bool landed = mbar_wait(full_bar(st), static_cast<uint32_t>((gi / kPfxStages) & 1), abort_flag, p.err);
            const uint32_t sk = smem_u32(smem + st * kStageBytes);
            const uint32_t sv = sk + kBlockBytes;
            float sa[4] = {0.f, 0.f, 0.f, 0.f};
            float sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int chunk = ((ks & 3) << 1) | k_hi;
                uint32_t a[4];
                ldmatrix_x4(a, sk + (ks >> 2) * kHalfBytes + k_row_off + ((chunk ^ k_sw) << 4));
                if (ks & 1) mma_bf16_16816(sb, a, qb[2 * ks], qb[2 * ks + 1]);
                else mma_bf16_16816(sa, a, qb[2 * ks], qb[2 * ks + 1]);
            }
            // shared tiles are whole blocks: all 16 tokens are valid
            const float x0 = (sa[0] + sb[0]) * p.scale_log2, x1 = (sa[1] + sb[1]) * p.scale_log2;
            const float x2 = (sa[2] + sb[2]) * p.scale_log2, x3 = (sa[3] + sb[3]) * p.scale_log2;
            float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
            }
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            const uint32_t p01 = pack_bf16x2(ex2(x0 - mn0), ex2(x1 - mn1));
            const uint32_t p23 = pack_bf16x2(ex2(x2 - mn0), ex2(x3 - mn1));
            l0 = l0 * al0 + bf16_lo(p01) + bf16_lo(p23);
            l1 = l1 * al1 + bf16_hi(p01) + bf16_hi(p23);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                o[j][0] *= al0;
                o[j][1] *= al1;
                o[j][2] *= al0;
                o[j][3] *= al1;
            }
            const uint32_t pb0 = movmatrix_trans(p01);
            const uint32_t pb1 = movmatrix_trans(p23);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int chunk = ((j & 3) << 1) | (v_mat & 1);
                uint32_t a[4];
                ldmatrix_x4_trans(a, sv + (j >> 2) * kHalfBytes + v_row_off + ((chunk ^ v_sw) << 4));
                mma_bf16_16816(o[j], a, pb0, pb1);
            }
            fence_proxy_async_shared();  // this lane's reads of the stage, before the copy that will replace it
            __syncwarp();
            if (lane == 0 && landed) mbar_arrive(empty_bar(st));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        // rows 8w + 2c and 8w + 2c + 1: dims 16j + r (o[j][0..1]) and 16j + r + 8 (o[j][2..3])
        float* w0 = p.wpart + (static_cast<size_t>(it) * kPfxRows + 8 * warp + 2 * c) * kORow;
        float* w1 = w0 + kORow;
        if (8 * warp + 2 * c < item.y) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                w0[16 * j + r] = o[j][0];
                w0[16 * j + r + 8] = o[j][2];
            }
            if (r == 0) {
                w0[kDim] = m0;
                w0[kDim + 1] = l0;
            }
        }
        if (8 * warp + 2 * c + 1 < item.y) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                w1[16 * j + r] = o[j][1];
                w1[16 * j + r + 8] = o[j][3];
            }
            if (r == 0) {
                w1[kDim] = m1;
                w1[kDim + 1] = l1;
            }
        }
    }
}

struct MergeParams {
    const float* wpart;
    const float* side;
    __nv_bfloat16* out;
    const int4* targets;  // x: sequence, y: KV head | shared tiles << 16,
                          // z: first prefix item, w: prefix items | first row << 16
    const int32_t* context_lens;
    int cap_tokens;
    int num_targets;
    int num_q_heads;
    int group;
};

// One warp per grouped (sequence, KV head): lane l owns dims [4l, 4l + 4) of
// every head; the partials are merged in a fixed order (prefix items, then
// the private result), four partials and four heads per batch of loads.
__global__ void __launch_bounds__(128) cascade_merge_kernel(const MergeParams p) {
    const int warp_id = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp_id >= p.num_targets) return;
    const int4 tg = p.targets[warp_id];
    const int s = tg.x, g = tg.y & 0xffff;
    const int ctx = min(__ldg(p.context_lens + s), p.cap_tokens);
    const bool has_private = (ctx + kTok - 1) / kTok > (tg.y >> 16);  // the private pass left a result
    const int n_items = tg.w & 0xffff, row0 = tg.w >> 16;
    const int G = p.group;
    const int np = n_items + (has_private ? 1 : 0);
    const int d0 = lane * 4;
    const float NEG_INF = -INFINITY;
    auto part_ptr = [&](int k, int h) -> const float* {
        if (k < n_items) return p.wpart + (static_cast<size_t>(tg.z + k) * kPfxRows + row0 + h) * kORow;
        return p.side + ((static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(g) * G + h) * kORow);
    };
    float Mr[kMaxG], Lr[kMaxG];
    float4 Ar[kMaxG];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
        Mr[h] = NEG_INF;
        Lr[h] = 0.f;
        Ar[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i = 0; i < np; i += 4) {
#pragma unroll
        for (int hb = 0; hb < kMaxG; hb += 4) {
            if (hb < G) {
                float mk[4][4], lk[4][4];
                float4 ok[4][4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (i + k < np && hb + h < G) {
                            const float* pp = part_ptr(i + k, hb + h);
                            mk[k][h] = __ldcg(pp + kDim);
                            lk[k][h] = __ldcg(pp + kDim + 1);
                            ok[k][h] = __ldcg(reinterpret_cast<const float4*>(pp + d0));
                        } else {
                            mk[k][h] = NEG_INF;
                            lk[k][h] = 0.f;
                            ok[k][h] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int H = hb + h;
                    if (H < G) {
                        float mn = Mr[H];
#pragma unroll
                        for (int k = 0; k < 4; ++k) mn = fmaxf(mn, mk[k][h]);
                        const float a = ex2(Mr[H] - mn);
                        float L = Lr[H] * a;
                        float4 A = make_float4(Ar[H].x * a, Ar[H].y * a, Ar[H].z * a, Ar[H].w * a);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float b = ex2(mk[k][h] - mn);
                            L += b * lk[k][h];
                            A.x += b * ok[k][h].x;
                            A.y += b * ok[k][h].y;
                            A.z += b * ok[k][h].z;
                            A.w += b * ok[k][h].w;
                        }
                        Mr[H] = mn;
                        Lr[H] = L;
                        Ar[H] = A;
                    }
                }
            }
        }
    }
    __nv_bfloat16* out_base = p.out + (static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(g) * G) * kDim + d0;
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
        if (h < G) {
            const float inv = 1.f / Lr[h];
            uint2 w2;
            w2.x = pack_bf16x2(Ar[h].x * inv, Ar[h].y * inv);
            w2.y = pack_bf16x2(Ar[h].z * inv, Ar[h].w * inv);
            *reinterpret_cast<uint2*>(out_base + static_cast<size_t>(h) * kDim) = w2;
        }
    }
}

// Host-side layout of a cascade plan inside the caller's workspace.
struct CascadeLayout {
    size_t decode_bytes, side_off, skip_off, members_off, items_off, targets_off, wpart_off, total;
    int num_items, num_targets, total_members;
    int chunk_tiles;  // shared tiles per prefix item (8..kPfxTiles)
};

pkv_status cascade_layout(int num_seqs, int num_q_heads, int num_kv_heads, int num_groups,
                          const int32_t* group_offsets, const int32_t* group_shared_blocks, CascadeLayout* L) {
    if (num_seqs < 1 || num_seqs > PKV_ATTN_MAX_SEQS || num_kv_heads < 1 || num_q_heads < 1 ||
        num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > PKV_ATTN_MAX_GROUP || num_groups < 0 ||
        (num_groups > 0 && (!group_offsets || !group_shared_blocks)))
        return PKV_EINVAL;
    const int G = num_q_heads / num_kv_heads;
    long long items = 0, targets = 0, passes = 0;
    if (num_groups > 0 && group_offsets[0] != 0) return PKV_EINVAL;
    for (int gr = 0; gr < num_groups; ++gr) {
        const int m = group_offsets[gr + 1] - group_offsets[gr];
        const int sh = group_shared_blocks[gr];
        if (m < 1 || sh < 1) return PKV_EINVAL;
        if (sh > 0xffff) return PKV_ERANGE;
        passes += static_cast<long long>(num_kv_heads) * ((static_cast<long long>(m) * G + kPfxRows - 1) / kPfxRows) * sh;
        targets += static_cast<long long>(m) * num_kv_heads;
    }
    const int total_members = num_groups > 0 ? group_offsets[num_groups] : 0;
    if (total_members > num_seqs) return PKV_ERANGE;
    // Cut shared prefixes into items of 8..64 tiles, aiming at about one item
    // per two CTA slots: a small batch gets short items (parallel reads), a
    // large one long items (fewer partials to merge, and fewer CTAs taken
    // from the concurrent private pass). Measured on a 16 x 8 fan-out: 64-tile
    // items 76 us, 21-tile items 80 us; on a 7-request group 8-tile items
    // 32 us, 64-tile items 55 us.
    const DeviceInfo dev = device_info();
    if (!dev.ok) return PKV_ECUDA;
    const long long slots = static_cast<long long>(kPfxCtasPerSm) * dev.sm_count;
    int chunk = static_cast<int>(std::min<long long>(kPfxTiles, std::max<long long>(8, (2 * passes + slots - 1) / slots)));
    L->chunk_tiles = chunk;
    for (int gr = 0; gr < num_groups; ++gr) {
        const int m = group_offsets[gr + 1] - group_offsets[gr];
        const long long chunks = (static_cast<long long>(m) * G + kPfxRows - 1) / kPfxRows;
        items += num_kv_heads * chunks * ((group_shared_blocks[gr] + chunk - 1) / chunk);
    }
    if (items > (1 << 28)) return PKV_ERANGE;
    const int grid = grid_for(num_seqs);
    if (grid < 1) return PKV_ECUDA;
    L->decode_bytes = align256(workspace_bytes(grid));
    L->side_off = L->decode_bytes;
    L->skip_off = L->side_off + align256(static_cast<size_t>(num_seqs) * num_q_heads * kORow * 4);
    L->members_off = L->skip_off + align256(static_cast<size_t>(num_seqs) * 4);
    L->items_off = L->members_off + align256(static_cast<size_t>(total_members) * 4 + 4);
    L->targets_off = L->items_off + align256(static_cast<size_t>(items) * 16 + 16);
    L->wpart_off = L->targets_off + align256(static_cast<size_t>(targets) * 16 + 16);
    L->total = L->wpart_off + static_cast<size_t>(items) * kPfxRows * kORow * 4;
    L->num_items = static_cast<int>(items);
    L->num_targets = static_cast<int>(targets);
    L->total_members = total_members;
    return PKV_OK;
}

// Per device, once: the side stream the prefix pass runs on, concurrently
// with the private pass, and the two events that fork it from and join it to
// the caller's stream.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

bool side_stream(SideStream* out) {
    static std::mutex mu;
    static std::vector<SideStream> per_dev;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(per_dev.size()) <= dev) per_dev.resize(dev + 1);
    SideStream& ss = per_dev[dev];
    if (!ss.stream) {
        e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            ss = SideStream{};
            return false;
        }
    }
    *out = ss;
    return true;
}

}  // namespace attn
}  // namespace pkv

extern "C" {

size_t pkv_attn_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int num_groups,
                                       const int32_t* group_offsets, const int32_t* group_shared_blocks) {
    attn::CascadeLayout L;
    if (attn::cascade_layout(num_seqs, num_q_heads, num_kv_heads, num_groups, group_offsets, group_shared_blocks,
                             &L) != PKV_OK)
        return 0;
    return L.total;
}

size_t pkv_cascade_staging_size(int num_seqs, int num_q_heads, int num_kv_heads, int num_groups,
                                const int32_t* group_offsets, const int32_t* group_shared_blocks) {
    attn::CascadeLayout L;
    if (attn::cascade_layout(num_seqs, num_q_heads, num_kv_heads, num_groups, group_offsets, group_shared_blocks,
                             &L) != PKV_OK)
        return 0;
    return L.wpart_off - L.skip_off;
}

pkv_status pkv_cascade_plan(int num_seqs, int num_q_heads, int num_kv_heads, int num_groups,
                            const int32_t* group_offsets, const int32_t* group_members,
                            const int32_t* group_shared_blocks, void* workspace, size_t workspace_bytes,
                            void* host_staging, size_t staging_bytes, void* stream) {
    attn::CascadeLayout L;
    pkv_status st = attn::cascade_layout(num_seqs, num_q_heads, num_kv_heads, num_groups, group_offsets,
                                         group_shared_blocks, &L);
    if (st != PKV_OK) return st;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total) return PKV_EINVAL;
    if (!host_staging || (num_groups > 0 && !group_members)) return PKV_EINVAL;
    const size_t upload = L.wpart_off - L.skip_off;
    if (staging_bytes < upload) return PKV_EINVAL;
    const int G = num_q_heads / num_kv_heads;
    uint8_t* h = static_cast<uint8_t*>(host_staging);
    std::memset(h, 0, upload);
    int32_t* skip = reinterpret_cast<int32_t*>(h);
    int32_t* members = reinterpret_cast<int32_t*>(h + (L.members_off - L.skip_off));
    int4* items = reinterpret_cast<int4*>(h + (L.items_off - L.skip_off));
    int4* targets = reinterpret_cast<int4*>(h + (L.targets_off - L.skip_off));
    std::vector<char> seen(num_seqs, 0);
    int ni = 0, nt = 0;
    for (int gr = 0; gr < num_groups; ++gr) {
        const int b = group_offsets[gr], e = group_offsets[gr + 1];
        const int sh = group_shared_blocks[gr];
        const int m = e - b;
        for (int k = b; k < e; ++k) {
            const int sq = group_members[k];
            if (sq < 0 || sq >= num_seqs || seen[sq]) return PKV_EINVAL;  // one group per sequence
            seen[sq] = 1;
            members[k] = sq;
            skip[sq] = sh;
        }
        const int chunks = (m * G + attn::kPfxRows - 1) / attn::kPfxRows;
        const int tchunks = (sh + L.chunk_tiles - 1) / L.chunk_tiles;
        for (int g = 0; g < num_kv_heads; ++g) {
            for (int rc = 0; rc < chunks; ++rc) {
                const int first_item = ni;
                for (int tc = 0; tc < tchunks; ++tc) {
                    const int t0 = tc * L.chunk_tiles;
                    const int n = std::min(L.chunk_tiles, sh - t0);
                    items[ni++] = make_int4(b + rc * attn::kPfxRows / G, std::min(attn::kPfxRows, m * G - rc * attn::kPfxRows),
                                            g | (n << 16), t0);
                }
                // the sharers whose rows this chunk holds
                for (int mi = rc * attn::kPfxRows / G; mi < std::min(m, (rc + 1) * attn::kPfxRows / G); ++mi) {
                    const int sq = group_members[b + mi];
                    targets[nt++] = make_int4(sq, g | (sh << 16), first_item,
                                              tchunks | ((mi * G - rc * attn::kPfxRows) << 16));
                }
            }
        }
    }
    if (ni != L.num_items || nt != L.num_targets) return PKV_ESTATE;
    const cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(workspace) + L.skip_off, h, upload,
                                          cudaMemcpyHostToDevice, as_stream(stream));
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

pkv_status pkv_attn_decode_cascade(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                   float scale, int num_groups, const int32_t* group_offsets,
                                   const int32_t* group_shared_blocks, void* workspace, size_t workspace_bytes,
                                   void* out, void* stream) {
    attn::CascadeLayout CL;
    pkv_status st = attn::cascade_layout(num_seqs, num_q_heads, num_kv_heads, num_groups, group_offsets,
                                         group_shared_blocks, &CL);
    if (st != PKV_OK) return st;
    if (!workspace || workspace_bytes < CL.total) return PKV_EINVAL;
    for (int gr = 0; gr < num_groups; ++gr)
        if (group_shared_blocks[gr] > max_blocks_per_seq) return PKV_EINVAL;
    attn::Launch L;
    st = attn::prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                       num_kv_heads, head_dim, num_blocks, scale, 0, workspace, CL.decode_bytes, out, &L);
    if (st != PKV_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = as_stream(stream);
    const attn::DeviceInfo dev = attn::device_info();
    if (!dev.ok) return PKV_ECUDA;
    attn::SideStream side;
    if (CL.num_items > 0 && !attn::side_stream(&side)) return PKV_ECUDA;
    auto cuda_ok = [](cudaError_t e) {
        if (e != cudaSuccess) record_cuda_error(e);
        return e == cudaSuccess;
    };
    if (CL.num_items > 0) {
        // the prefix pass runs on the side stream, concurrently with the private pass
        if (!cuda_ok(cudaEventRecord(side.fork, s)) || !cuda_ok(cudaStreamWaitEvent(side.stream, side.fork, 0)))
            return PKV_ECUDA;
        static std::once_flag once;
        static cudaError_t attr_err = cudaSuccess;
        std::call_once(once, [] {
            attr_err = cudaFuncSetAttribute(attn::prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(attn::kPfxSmem));
        });
        if (attr_err != cudaSuccess) {
            record_cuda_error(attr_err);
            return PKV_ECUDA;
        }
        attn::PrefixParams pp;
        pp.q = static_cast<const __nv_bfloat16*>(q);
        pp.block_tables = block_tables;
        pp.max_blocks = max_blocks_per_seq;
        pp.num_q_heads = num_q_heads;
        pp.num_kv_heads = num_kv_heads;
        pp.group = num_q_heads / num_kv_heads;
        pp.num_blocks = num_blocks;
        pp.scale_log2 = scale * 1.4426950408889634f;
        pp.members = reinterpret_cast<const int32_t*>(ws + CL.members_off);
        pp.items = reinterpret_cast<const int4*>(ws + CL.items_off);
        pp.num_items = CL.num_items;
        pp.err = L.prm.err;
        pp.wpart = reinterpret_cast<float*>(ws + CL.wpart_off);
        const int grid = std::min(CL.num_items, attn::kPfxCtasPerSm * dev.sm_count);
        attn::prefix_kernel<<<grid, attn::kPfxThreads, attn::kPfxSmem, side.stream>>>(L.tm_k, L.tm_v, pp);
        if (!cuda_ok(cudaGetLastError()) || !cuda_ok(cudaEventRecord(side.join, side.stream))) return PKV_ECUDA;
    }
    // the private pass: every sequence's tiles after its group's shared ones
    L.prm.skip_tiles = reinterpret_cast<const int32_t*>(ws + CL.skip_off);
    L.prm.side = reinterpret_cast<float*>(ws + CL.side_off);
    const attn::KernelConfig kc = attn::config_for(num_seqs, PKV_BLOCK_TOKENS, true);
    if (kc.grid < 1) return PKV_ECUDA;
    L.fn = kc.fn;
    L.grid = std::min(L.grid, kc.grid);
    L.smem = kc.smem;
    st = attn::launch(L, s, false);
    if (CL.num_items > 0 && !cuda_ok(cudaStreamWaitEvent(s, side.join, 0))) return PKV_ECUDA;  // join first
    if (st != PKV_OK || CL.num_targets == 0) return st;
    attn::MergeParams mp;
    mp.wpart = reinterpret_cast<const float*>(ws + CL.wpart_off);
    mp.side = L.prm.side;
    mp.out = static_cast<__nv_bfloat16*>(out);
    mp.targets = reinterpret_cast<const int4*>(ws + CL.targets_off);
    mp.context_lens = context_lens;
    mp.cap_tokens = max_blocks_per_seq * PKV_BLOCK_TOKENS;
    mp.num_targets = CL.num_targets;
    mp.num_q_heads = num_q_heads;
    mp.group = num_q_heads / num_kv_heads;
    attn::cascade_merge_kernel<<<(CL.num_targets + 3) / 4, 128, 0, s>>>(mp);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of pkv_attn_decode.
//
// For callers that cannot allocate device memory themselves -- for example a
// plugin loaded into a host program that owns every device allocation and
// gives plugins no allocator, or a latency-critical loop that must never pay
// for cudaMalloc / cudaFree. Instead of a caller-provided workspace, the
// partial results and the merge counters live in one file-scope device array
// that every GPU loading this library holds until the process exits.

namespace pkv {
namespace attn {

constexpr int kStaticMaxCtas = 512;  // partial slots: 2 per CTA
// three counters per CTA: one per split pair (by its first CTA), two per
// two-level merge group
constexpr size_t kStaticCounterBytes = align256(static_cast<size_t>(kStaticMaxCtas) * 3 * 4);
// header | counters | partial slots (4,331,776 bytes): the first two are
// cleared by each call in one memset.
constexpr size_t kStaticScratchBytes = kWsHeader + kStaticCounterBytes +
                                       static_cast<size_t>(kStaticMaxCtas) * kWsPerCta;
static_assert(kStaticScratchBytes == 4331776, "the static scratch size stated in pkv.h");

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch for the current device, looked up once
// per device (the host-side name of the array is only a stand-in).
uint8_t* static_scratch_address() {
    static std::mutex mu;
    static std::vector<uint8_t*> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(addr.size()) <= dev) addr.resize(dev + 1, nullptr);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return nullptr;
        }
        addr[dev] = static_cast<uint8_t*>(p);
    }
    return addr[dev];
}

}  // namespace attn
}  // namespace pkv

extern "C" pkv_status pkv_attn_decode_static(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, int max_blocks_per_seq,
                                             const int32_t* context_lens, int num_seqs, int num_q_heads,
                                             int num_kv_heads, int head_dim, int num_blocks, float scale,
                                             uint32_t* device_error, void* out, void* stream) {
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_EINVAL;
    if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || num_blocks < 1 || max_blocks_per_seq < 1 ||
        !std::isfinite(scale))
        return PKV_EINVAL;
    if (num_seqs > PKV_ATTN_MAX_SEQS || head_dim != PKV_ATTN_HEAD_DIM || num_q_heads % num_kv_heads != 0 ||
        num_q_heads / num_kv_heads > PKV_ATTN_MAX_GROUP)
        return PKV_EUNSUPPORTED;
    if (static_cast<long long>(num_blocks) * num_kv_heads * PKV_BLOCK_TOKENS >= (1ll << 31) ||
        static_cast<long long>(num_seqs) * max_blocks_per_seq >= (1ll << 31) ||
        static_cast<long long>(max_blocks_per_seq) * PKV_BLOCK_TOKENS >= (1ll << 31) ||
        static_cast<long long>(num_kv_heads) * num_seqs * (max_blocks_per_seq + attn::kPieceCost) >= (1ll << 30))
        return PKV_ERANGE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PKV_EINVAL;
    const attn::KernelConfig kc = attn::config_for(num_seqs);
    if (kc.grid < 1) return PKV_ECUDA;
    uint8_t* scratch = attn::static_scratch_address();
    if (!scratch) return PKV_ECUDA;
    const int grid = attn::default_grid(kc.grid < attn::kStaticMaxCtas ? kc.grid : attn::kStaticMaxCtas, num_seqs,
                                        num_kv_heads, max_blocks_per_seq, PKV_BLOCK_TOKENS);

    CUtensorMap tm_k, tm_v;
    if (!attn::make_cache_map(&tm_k, k_cache, num_blocks, num_kv_heads, PKV_BLOCK_TOKENS) ||
        !attn::make_cache_map(&tm_v, v_cache, num_blocks, num_kv_heads, PKV_BLOCK_TOKENS))
        return PKV_ECUDA;

    // The counters must start at zero; a previous call leaves them at zero
    // unless it was cut short, so clear them (and the internal error word).
    cudaError_t e = cudaMemsetAsync(scratch, 0, attn::kWsHeader + attn::kStaticCounterBytes, as_stream(stream));
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }

    attn::Params prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.num_seqs = num_seqs;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = num_kv_heads;
    prm.group = num_q_heads / num_kv_heads;
    prm.max_blocks = max_blocks_per_seq;
    prm.cap_tokens = max_blocks_per_seq * PKV_BLOCK_TOKENS;
    prm.num_blocks = num_blocks;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.err = device_error ? device_error : reinterpret_cast<uint32_t*>(scratch);
    prm.counters = reinterpret_cast<int*>(scratch + attn::kWsHeader);
    prm.group_counters = prm.counters + attn::kStaticMaxCtas;
    prm.partials = reinterpret_cast<float*>(scratch + attn::kWsHeader + attn::kStaticCounterBytes);
    prm.skip_tiles = nullptr;
    prm.side = nullptr;
    prm.stop_tiles = -1;

    void* args[] = {&tm_k, &tm_v, &prm};
    e = cudaLaunchKernel(reinterpret_cast<const void*>(kc.fn), dim3(grid), dim3(attn::kThreads), args, kc.smem,
                         as_stream(stream));
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PKV_ECUDA;
    }
    return PKV_OK;
}
