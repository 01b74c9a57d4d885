/*
 * pkv.h -- C ABI of libpkv: paged KV cache decode on GB300 (sm_103a).
 *
 * The KV cache of one attention layer is a preallocated pool of fixed-size
 * blocks of 16 tokens; each sequence reaches its tokens through a block table
 * that maps logical block i to a physical block id (cs2680 Lecture 10, §10.3
 * "PagedAttention: the KV cache as virtual memory"; "The inference server":
 * the KV cache is one arena allocated at start-up, with no allocator on the
 * hot path).
 *
 * Device-side layout (all bf16 buffers hold IEEE bfloat16 values, row-major):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][16][head_dim]
 *                      token t of a sequence, KV head g, lives at
 *                      [table[t / 16]][g][t % 16][:]
 *   q, out           : [num_seqs][num_q_heads][head_dim]
 *   k, v (append)    : [num_tokens][num_kv_heads][head_dim]
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq]; entries past
 *                      ceil(context_len / 16) in a row are never read
 *   context_lens     : int32 [num_seqs]
 *   slot_mapping     : int64 [num_tokens]; slot = block * 16 + (pos % 16)
 *   src_dst_pairs    : int32 [num_pairs][2]
 * Query head h uses KV head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: the caller owns every device buffer and stream; the library
 * allocates no device memory and frees nothing it did not create. Every
 * device call is asynchronous on the given stream (a cudaStream_t passed as
 * void*; NULL = the legacy default stream) and returns after the launch.
 *
 * Errors: calls return a pkv_status. Argument errors found on the host return
 * before anything is launched. Errors that only the device can see (a block
 * id or slot outside the pool, a context longer than its table row, a bounded
 * wait that ran out) never fault the GPU: the kernel skips the access, ORs a
 * PKV_DEVERR_* bit into a device-side 32-bit error word, and carries on; the
 * host reads that word with pkv_read_device_error.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int pkv_status;

#define PKV_OK 0
#define PKV_EINVAL (-1)      /* bad argument (null pointer, shape, alignment) */
#define PKV_ENOMEM (-2)      /* too few free pages: admission or fork refused */
#define PKV_ERANGE (-3)      /* id or length outside the valid range */
#define PKV_ECUDA (-4)       /* a CUDA runtime call failed */
#define PKV_ENOSPC (-5)      /* append past the pages a sequence reserved */
#define PKV_EUNSUPPORTED (-6) /* geometry the library does not handle */
#define PKV_ESTATE (-7)      /* block manager found its own state inconsistent */

/* Bits of the device-side error word. */
#define PKV_DEVERR_BLOCK_ID 0x1u  /* block id outside [0, num_blocks) in a table or pair */
#define PKV_DEVERR_SLOT 0x2u      /* slot outside [0, num_blocks * 16) */
#define PKV_DEVERR_CONTEXT 0x4u   /* context_len > 16 * max_blocks_per_seq */
#define PKV_DEVERR_TIMEOUT 0x8u   /* an internal wait gave up; the output is invalid */

#define PKV_BLOCK_TOKENS 16
#define PKV_ATTN_HEAD_DIM 128   /* head_dim of pkv_attn_decode */
#define PKV_ATTN_MAX_GROUP 8    /* max num_q_heads / num_kv_heads */
#define PKV_ATTN_MAX_SEQS 4096  /* max num_seqs of one pkv_attn_decode call */
#define PKV_ATTN_MAX_CTAS 2048  /* max num_ctas of one pkv_attn_decode call */

/* Library version (major * 10000 + minor * 100 + patch). */
int pkv_version(void);

/* Static description of a status code. */
const char* pkv_status_string(pkv_status status);

/* Message of the last CUDA error seen by this thread inside the library. */
const char* pkv_last_cuda_error(void);

/* Copy the device error word to *host_value (synchronises the stream); if
 * clear != 0, reset it to zero afterwards. */
pkv_status pkv_read_device_error(uint32_t* device_error, uint32_t* host_value,
                                 int clear, void* stream);

/*
 * pkv_append -- write each new token's K and V into its cache slot.
 *
 * cs2680 Lecture 10, §10.3: a sequence grows by one token by writing one slot
 * of its last block (or of the next block it owns); the slot is
 * table[pos / 16] * 16 + pos % 16, computed on the host by
 * pkv_bm_prepare_append.
 *   k, v          : device bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping  : device int64 [num_tokens]; a negative slot marks a padding
 *                   row and writes nothing ("The inference server": padding
 *                   rows of a bucketed batch are discarded)
 *   k_cache, v_cache : device bf16 pool, layout above
 *   device_error  : device uint32 error word, or NULL
 * Slots must be distinct (two rows writing one slot race). head_dim must be a
 * multiple of 8; every bf16 pointer 16-byte aligned. A slot >= num_blocks * 16
 * is skipped and sets PKV_DEVERR_SLOT.
 */
pkv_status pkv_append(const void* k, const void* v, const int64_t* slot_mapping,
                      int num_tokens, void* k_cache, void* v_cache, int num_blocks,
                      int num_kv_heads, int head_dim, uint32_t* device_error,
                      void* stream);

/* pkv_append with a cache of block_tokens-token blocks (8, 16, 32 or 64):
 * k_cache, v_cache are [num_blocks][num_kv_heads][block_tokens][head_dim] and
 * slot = block * block_tokens + pos % block_tokens. */
pkv_status pkv_append_ex(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                         void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                         int block_tokens, uint32_t* device_error, void* stream);

/*
 * pkv_block_copy -- copy-on-write of whole blocks.
 *
 * "KV cache systems", copy-on-write paragraph, and cs2680 Lecture 10, §10.4:
 * the first writer of a shared block gets a private copy of it. For each pair
 * (src, dst), physical block dst of both caches becomes a copy of block src
 * (all KV heads, all 16 rows). Destinations must be distinct and no
 * destination may also be a source in the same call. Pairs with an id
 * outside [0, num_blocks) are skipped and set PKV_DEVERR_BLOCK_ID.
 *   src_dst_pairs : device int32 [num_pairs][2]
 */
pkv_status pkv_block_copy(void* k_cache, void* v_cache, const int32_t* src_dst_pairs,
                          int num_pairs, int num_blocks, int num_kv_heads, int head_dim,
                          uint32_t* device_error, void* stream);

/* pkv_block_copy for caches of block_tokens-token blocks (8, 16, 32 or 64). */
pkv_status pkv_block_copy_ex(void* k_cache, void* v_cache, const int32_t* src_dst_pairs, int num_pairs,
                             int num_blocks, int num_kv_heads, int head_dim, int block_tokens,
                             uint32_t* device_error, void* stream);

/*
 * pkv_attn_workspace_size -- bytes of device scratch pkv_attn_decode needs for
 * num_seqs sequences and num_kv_heads KV heads on the current device (with
 * the default num_ctas). The workspace holds the error word (its first 4
 * bytes), a fixed 24 KiB of counters (three per possible CTA: one for a pair
 * split across CTAs, two for the groups of a pair split among more than
 * eight CTAs, which merges in two levels), then two fp32 partial results per
 * CTA. The counters' place and size do not depend on the call, so one
 * workspace serves calls of any batch, KV-head count and num_ctas that fit
 * in it. Returns 0 for invalid arguments or when no device is present.
 */
size_t pkv_attn_workspace_size(int num_seqs, int num_kv_heads);

/* Zero a workspace (asynchronously, on stream). Needed once after it is
 * allocated, and again after a call that set PKV_DEVERR_TIMEOUT; every
 * pkv_attn_decode leaves its counters at zero. */
pkv_status pkv_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Bytes at the start of every attention workspace that must hold zeros
 * between calls: the 256-byte header (error word) and the merge counters
 * (the same for every batch, KV-head count and grid). The bytes after them
 * are scratch whose content never matters to the next call. */
size_t pkv_attn_workspace_fixed_bytes(void);

/*
 * pkv_attn_decode -- single-token decode attention through block tables.
 *
 * For every sequence s and query head h (KV head g = h / (Hq / Hkv)):
 *   x_t = scale * <q[s,h], K[table[s][t/16]][g][t%16]>,  t < context_lens[s]
 *   out[s,h] = sum_t softmax(x)_t * V[table[s][t/16]][g][t%16]
 * (cs2680 Lecture 10, §10.3, step three: attention reads through the block
 * table, with the same FLOPs and bytes as over a contiguous cache; "The
 * inference server": attention takes a block table and a length tensor, both
 * fixed-shape, so growth changes values, not shapes.)
 * bf16 inputs and output, fp32 accumulation and softmax; the output is
 * rounded to nearest even. context_lens[s] <= 0 gives a zero output row.
 *   q, out        : device bf16 [num_seqs][num_q_heads][128]
 *   block_tables  : device int32 [num_seqs][max_blocks_per_seq]
 *   context_lens  : device int32 [num_seqs]
 *   num_ctas      : number of persistent CTAs (at most PKV_ATTN_MAX_CTAS, and
 *                   as many as the workspace holds partial slots for), 0 =
 *                   as many as fit at once on the device, or fewer when the
 *                   block tables bound the batch's work to under 4 tiles (16
 *                   tokens of one KV head, plus 3 per sequence and KV head)
 *                   per CTA; the context of all
 *                   (sequence, KV head) pairs is split evenly among them and
 *                   partial results of a pair split across CTAs are merged in
 *                   the same launch
 *   workspace     : device scratch of at least
 *                   pkv_attn_workspace_size(num_seqs, num_kv_heads) bytes,
 *                   zeroed once by pkv_attn_workspace_init; its first 4 bytes
 *                   are the device error word. Calls that share a workspace
 *                   must not overlap on the GPU.
 * Limits: head_dim == 128, num_q_heads % num_kv_heads == 0,
 * num_q_heads / num_kv_heads <= 8, 1 <= num_seqs <= 4096,
 * num_blocks * num_kv_heads * 16 < 2^31, num_seqs * max_blocks_per_seq < 2^31
 * and num_kv_heads * num_seqs * (ceil(max_blocks_per_seq * block tokens / 16)
 * + 3) < 2^30 (PKV_ERANGE otherwise; the + 3 is the work partition's charge
 * per (sequence, KV head) run). A block id outside [0, num_blocks)
 * is never dereferenced: block 0 is read in its place and PKV_DEVERR_BLOCK_ID
 * is set (the output is then invalid); context_lens above
 * 16 * max_blocks_per_seq are clamped and set PKV_DEVERR_CONTEXT.
 */
pkv_status pkv_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int num_blocks, float scale,
                           int num_ctas, void* workspace, size_t workspace_bytes,
                           void* out, void* stream);

/*
 * pkv_attn_decode_cuda_cores -- pkv_attn_decode with the per-tile math (the
 * dot products of the query heads with each key, and the probability-
 * weighted sum of the values) on the FP32 CUDA cores instead of the tensor
 * cores; everything else (work split, copies, online softmax, merges) is the
 * same kernel. For measuring the tensor-core choice: cs2680 Lecture 10,
 * §10.3, step three says paging leaves the arithmetic unchanged, so which
 * unit runs it is this library's decision. Group sizes
 * num_q_heads / num_kv_heads of 4 and 8 only (PKV_EUNSUPPORTED otherwise);
 * arguments, layouts and limits as pkv_attn_decode. The probabilities stay in
 * fp32 here (the tensor-core kernel rounds them to bf16 for the mma), so the
 * two agree within the attention tolerance, not bit for bit.
 */
pkv_status pkv_attn_decode_cuda_cores(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int num_blocks, float scale, int num_ctas,
                                      void* workspace, size_t workspace_bytes, void* out, void* stream);

/*
 * pkv_attn_decode_wait_test -- pkv_attn_decode for tests of the bounded-wait
 * path only; its output is invalid. CTA 0's producer issues the copies of its
 * first stop_tiles (>= 0) tiles and then stops, as if they never came: the
 * consumer waiting on the next tile gives up after the wait limit (1 s),
 * ORs PKV_DEVERR_TIMEOUT into the workspace's error word and raises the CTA's
 * abort flag; the CTA then runs to its end without waiting, after waiting
 * (bounded) for every copy it did issue. Nothing faults or hangs: this is
 * how a kernel of this library ends when a copy never completes (cs2680
 * Lecture 10, §10.5: a serving engine refuses or preempts instead of
 * crashing). Zero the workspace with pkv_attn_workspace_init before its next
 * use. Other arguments as pkv_attn_decode.
 */
pkv_status pkv_attn_decode_wait_test(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_dim, int num_blocks, float scale, int num_ctas,
                                     void* workspace, size_t workspace_bytes, void* out, int stop_tiles,
                                     void* stream);

/*
 * pkv_attn_decode_ex -- pkv_attn_decode over a cache of block_tokens-token
 * blocks (8, 16, 32 or 64; PKV_EUNSUPPORTED otherwise): token t of a sequence
 * is row t % block_tokens of block table[t / block_tokens]. The block size
 * trades tail waste and table length against the kernel's contiguous runs
 * (cs2680 Lecture 10, §10.3, block-size table and Exercise 3: achieved
 * attention bandwidth as a function of contiguous run length). A 128-dim
 * head's block is block_tokens * 256 contiguous bytes; the kernel reads 16
 * tokens at a time (two 8-token blocks when block_tokens is 8).
 */
pkv_status pkv_attn_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                              int head_dim, int num_blocks, int block_tokens, float scale, int num_ctas,
                              void* workspace, size_t workspace_bytes, void* out, void* stream);

/*
 * Cascade attention -- pkv_attn_decode for a batch whose sequences share
 * leading blocks, reading each shared block once for all its sharers instead
 * of once per sequence. The pages share those blocks in memory ("KV cache
 * systems", copy-on-write and prefix-hit paragraphs; cs2680 Lecture 10,
 * §10.4: forked samples and prefix groups); sharing their reads is this
 * library's own step. The result equals pkv_attn_decode's within floating-
 * point reassociation (the sums are split at the shared/private boundary).
 *
 * Groups (host arrays, read during the calls only): group i has the sharers
 * group_members[group_offsets[i] .. group_offsets[i + 1]) (sequence indices
 * of the batch, each in at most one group, at least one per group) whose
 * block tables agree on their first group_shared_blocks[i] >= 1 entries, and
 * every sharer's context_len is at least 16 * group_shared_blocks[i]
 * (violations of the last rule set PKV_DEVERR_CONTEXT). 16-token blocks only.
 *
 * pkv_attn_cascade_workspace_size: bytes of device workspace for such a batch
 *   (0 on invalid arguments). Zero it once with pkv_attn_workspace_init.
 * pkv_cascade_plan: lays the groups out for the kernels and copies that
 *   description into the workspace on `stream` (one host-to-device copy of
 *   at most staging_bytes from host_staging, which the caller owns: pinned
 *   memory, unchanged until the copy has run). Call it whenever the groups
 *   change; it reads no device data.
 * pkv_attn_decode_cascade: the attention itself, with the same groups as
 *   the plan: the prefix pass runs on a side stream the library owns (one
 *   per device), forked from `stream` and joined back to it by events, while
 *   the private pass runs on `stream`; the merge follows on `stream`.
 *   Arguments otherwise as pkv_attn_decode (the persistent grid is sized
 *   automatically); out rows of grouped sequences are written by the merge.
 *   Calls on one device must not overlap on the GPU. Worth it when the
 *   shared bytes saved are large: a 16-prompt x 8-sample fan-out (1.06 GB
 *   saved) runs about twice as fast, a 7-request prefix group (59 MB saved,
 *   mostly L2-resident) slower than pkv_attn_decode.
 */
size_t pkv_attn_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int num_groups,
                                       const int32_t* group_offsets, const int32_t* group_shared_blocks);

/* Bytes of host staging pkv_cascade_plan needs for these groups (0 on invalid arguments). */
size_t pkv_cascade_staging_size(int num_seqs, int num_q_heads, int num_kv_heads, int num_groups,
                                const int32_t* group_offsets, const int32_t* group_shared_blocks);

pkv_status pkv_cascade_plan(int num_seqs, int num_q_heads, int num_kv_heads, int num_groups,
                            const int32_t* group_offsets, const int32_t* group_members,
                            const int32_t* group_shared_blocks, void* workspace, size_t workspace_bytes,
                            void* host_staging, size_t staging_bytes, void* stream);

pkv_status pkv_attn_decode_cascade(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int num_blocks, float scale,
                                   int num_groups, const int32_t* group_offsets,
                                   const int32_t* group_shared_blocks, void* workspace,
                                   size_t workspace_bytes, void* out, void* stream);

/*
 * pkv_decode_step -- one decode step of one attention layer in one call:
 * pkv_block_copy(src_dst_pairs), then pkv_append(k_new, v_new,
 * slot_mapping), then pkv_attn_decode, on `stream`. "The inference server":
 * the decode step is schedule, copy the block tables and lengths into the
 * step's buffers, run -- with fixed-shape arguments. The arguments mean what
 * they mean in the three calls (slot_mapping and src_dst_pairs come from
 * pkv_bm_prepare_append); num_pairs or num_new_tokens may be 0.
 * All arguments are checked before anything is launched. The attention
 * kernel is launched so that its prologue (reading context_lens and
 * block_tables, planning its split) overlaps the append; it waits for the
 * append before reading the cache. Hence context_lens, block_tables and q
 * must not be written by the copy or append of the same step (they are not,
 * by construction). device_error receives copy and append errors; attention
 * errors go to the workspace's error word as in pkv_attn_decode.
 */
pkv_status pkv_decode_step(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                           int num_new_tokens, const int32_t* src_dst_pairs, int num_pairs,
                           void* k_cache, void* v_cache, int num_blocks, const void* q,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, float scale, int num_ctas, void* workspace,
                           size_t workspace_bytes, void* out, uint32_t* device_error, void* stream);

/*
 * pkv_step_layout -- where the inputs of one decode step sit in one packed
 * buffer for pkv_decode_step_host, in this order, each 256-byte aligned:
 * q [num_seqs][Hq][D] bf16, k_new and v_new [num_seqs][Hkv][D] bf16,
 * slot_mapping [num_seqs] int64, block_tables [num_seqs][max_blocks_per_seq]
 * int32, context_lens [num_seqs] int32, src_dst_pairs [num_pairs][2] int32
 * (last, so that no other offset depends on num_pairs); bytes = the
 * buffer's size. One new token per sequence (slot -1 for a padding row).
 */
typedef struct pkv_step_layout_t {
    size_t q, k_new, v_new, slot_mapping, block_tables, context_lens, src_dst_pairs;
    size_t bytes;
} pkv_step_layout_t;

pkv_status pkv_step_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                           int max_blocks_per_seq, int num_pairs, pkv_step_layout_t* layout);

/*
 * pkv_decode_step_host -- pkv_decode_step with its inputs and output in host
 * memory: host_packed (laid out by pkv_step_layout) is brought into
 * device_staging (device, layout.bytes, 256-byte aligned), the step itself
 * reads its inputs from there and writes attention rows to device_out
 * (device, [num_seqs][Hq][D] bf16), then one copy of those rows goes into
 * host_out. When host_packed is pinned host memory the device can address
 * (cudaHostAlloc / cudaHostRegister) and 16-byte aligned, a staging kernel
 * reads it across the host link (faster than a copy engine for a step's few
 * MB), and of each block-table row only the entries up to
 * ceil(context_len / 16) cross (no kernel reads past them; the rest of the
 * row in device_staging keeps what it held); otherwise one asynchronous copy
 * brings the whole buffer. When host_out is such
 * memory, the attention writes the rows there directly and device_out is not
 * touched (it must still be a valid device pointer). Everything is enqueued
 * on `stream` and checked before anything is enqueued: host_packed must not
 * change, and host_out must not be read, until the stream has passed the
 * step (e.g. after cudaStreamSynchronize). This is the call through which a
 * host program that keeps its step inputs in host memory drives a step.
 */
pkv_status pkv_decode_step_host(const void* host_packed, void* device_staging, int num_pairs,
                                void* k_cache, void* v_cache, int num_blocks, int max_blocks_per_seq,
                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                float scale, int num_ctas, void* workspace, size_t workspace_bytes,
                                void* device_out, void* host_out, uint32_t* device_error,
                                void* stream);

/* Number of persistent CTAs that fit on the current device at once for
 * num_seqs sequences: the most pkv_attn_decode launches when num_ctas == 0
 * (it launches fewer for a batch whose tables bound its work to a few tiles
 * per CTA); 0 on error. */
int pkv_attn_default_ctas(int num_seqs);

/* Number of CTAs pkv_attn_decode / pkv_attn_decode_ex launch when num_ctas
 * == 0, for num_seqs sequences, num_kv_heads KV heads, tables of
 * max_blocks_per_seq entries and blocks of block_tokens tokens (8, 16, 32 or
 * 64): pkv_attn_default_ctas(num_seqs), or fewer when the tables bound the
 * batch's work to under 4 cost units per CTA. 0 on bad arguments. */
int pkv_attn_launch_ctas(int num_seqs, int num_kv_heads, int max_blocks_per_seq, int block_tokens);

/*
 * pkv_attn_decode_static -- pkv_attn_decode without a workspace argument, for
 * callers that cannot allocate device memory themselves (for example a plugin
 * inside a host program that owns every device allocation and offers no
 * allocator, or a latency-critical loop that must never call cudaMalloc or
 * cudaFree). The pages describe no such variant: it has no counterpart there.
 *
 * Same computation, layouts and limits as pkv_attn_decode (num_seqs above
 * PKV_ATTN_MAX_SEQS is refused with PKV_EUNSUPPORTED), plus:
 *  - at most 512 persistent CTAs (the default grid, capped);
 *  - the scratch (counters and fp32 partials, 4,331,776 bytes, about 4.1 MiB)
 *    is one static device array inside this library; every GPU that loads
 *    the library holds it until the process exits. This call allocates and
 *    frees nothing: it clears the counters with an asynchronous memset on
 *    `stream`, then launches the kernel;
 *  - the first call on a device looks up that array's device address (a
 *    one-time set-up per device, with the device current); make that first
 *    call before any stream capture;
 *  - all calls share the one array, so calls that can overlap on the GPU
 *    (different streams, or other host threads) race and give wrong results:
 *    order them on one stream;
 *  - device-side errors are ORed into *device_error when it is non-NULL
 *    (a caller-owned device uint32); with NULL they are not reported.
 */
pkv_status pkv_attn_decode_static(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int num_blocks, float scale,
                                  uint32_t* device_error, void* out, void* stream);

/* ---------------------------------------------------------------------------
 * Host block manager.
 *
 * Owns the free list, the per-block reference counts and each sequence's
 * block table; it never touches device memory (freeing a sequence changes
 * ownership only -- "Reserve the page a request has not written yet",
 * "Separate the pool from its owners").
 *
 * Policy:
 *  - admission reserves ceil((prompt_len + max_new) / 16) pages at once and
 *    is refused (PKV_ENOMEM, no state change) when fewer pages are free
 *    ("Pick a reservation policy you can explain"); every call that changes
 *    state runs under one mutex, so reserve-and-admit is one decision even
 *    with concurrent callers;
 *  - members of a prefix group share the complete pages of their common
 *    prefix (prefix_len / 16 pages, charged once); the rest of each
 *    request's reservation is private ("Charge shared pages once");
 *  - fork: children share the parent's written blocks by reference count
 *    (cs2680 Lecture 10, §10.4); each child reserves private pages for the
 *    rest of its allowance and, when the parent's last written block is
 *    partial, one spare page for the copy-on-write of that block;
 *  - copy-on-write: a sequence that writes into a block with refcount > 1
 *    takes a spare page as its own copy and reports the (src, dst) pair; a
 *    writer that sees refcount 1 writes in place ("KV cache systems",
 *    copy-on-write paragraph);
 *  - free pages are handed out in free_order (ascending ids if NULL); a
 *    released page is the next one handed out.
 *
 * Options of pkv_bm_create_ex (all off in pkv_bm_create):
 *  - incremental: admission reserves only the prompt's pages,
 *    ceil(prompt_len / block_tokens), and leaves at least watermark_blocks
 *    pages available; a token that starts a new block, or a write into a
 *    shared block, takes a page when pkv_bm_prepare_append reaches it, and a
 *    step whose pages are not all available fails with PKV_ENOMEM and no
 *    state change. The caller then preempts a sequence (pkv_bm_preempt, the
 *    newest running one by pkv_bm_newest_running) and retries; the
 *    preempted sequence keeps its token count and is later re-admitted by
 *    pkv_bm_resume onto fresh pages for its KV to be recomputed (cs2680
 *    Lecture 10, §10.5: on-demand pages run out, a watermark keeps
 *    preemption rare, a preempted sequence is recomputed; "Reserve the page
 *    a request has not written yet", "Pick a reservation policy you can
 *    explain"). Fork under this policy reserves nothing.
 *  - prefix_cache: pkv_bm_admit_tokens indexes every complete prompt block
 *    by its exact token prefix and reuses indexed blocks for a later prompt
 *    from its first block up to its first mismatch (a block is reusable iff
 *    all its tokens and all earlier blocks match: 8,000 matching tokens
 *    reuse 500 blocks of 16). A released indexed block stays cached instead
 *    of returning to the free list; a cached block in use is never evicted,
 *    and allocation, once the free list is empty, evicts the least recently
 *    released idle cached block that no cached block extends ("KV cache
 *    systems", prefix-hit and eviction paragraphs). Idle cached blocks count
 *    as available to every admission and step.
 * A call that returns an error changes no state.
 * ------------------------------------------------------------------------- */
typedef struct pkv_bm pkv_bm;

typedef struct pkv_bm_stats_t {
    int32_t num_blocks;
    int32_t free_blocks;   /* on the free list */
    int32_t used_blocks;   /* refcount > 0 */
    int32_t shared_blocks; /* refcount > 1 */
    int32_t spare_blocks;  /* reserved for a future copy-on-write */
    int32_t num_seqs;
    int64_t ref_sum;       /* sum of refcounts == sum of table lengths */
    int64_t cow_copies;    /* copy-on-write pairs reported so far */
    int32_t cached_blocks;      /* in the prefix index */
    int32_t cached_idle_blocks; /* in the prefix index with refcount 0 */
    int32_t preempted_seqs;
    int32_t available_blocks;   /* free_blocks + cached_idle_blocks */
    int64_t cache_hits;         /* blocks reused by pkv_bm_admit_tokens so far */
    int64_t evictions;          /* cached blocks evicted so far */
} pkv_bm_stats_t;

/* free_order: host int32 permutation of [0, num_blocks), or NULL. Returns NULL
 * on invalid arguments. block_tokens: 8, 16, 32 or 64 (16 is the size the
 * pages use and the one the other calls assume). */
pkv_bm* pkv_bm_create(int num_blocks, int block_tokens, const int32_t* free_order);
/* As pkv_bm_create, with the policy options above (incremental and
 * prefix_cache: 0 or non-zero; watermark_blocks >= 0, used by admission and
 * resume only). */
pkv_bm* pkv_bm_create_ex(int num_blocks, int block_tokens, const int32_t* free_order,
                         int incremental, int watermark_blocks, int prefix_cache);
void pkv_bm_destroy(pkv_bm* bm);

/* group < 0: no sharing (prefix_len ignored). group >= 0: 0 <= prefix_len <=
 * prompt_len, and every member of a group must pass the same prefix_len. The
 * sequence starts with context length prompt_len (its prompt KV is written by
 * prefill, outside this library). */
pkv_status pkv_bm_admit(pkv_bm* bm, int prompt_len, int max_new, int group,
                        int prefix_len, int* seq_id);

/* Admission with the prompt's token ids (host int32 [prompt_len], read
 * during the call only) on a manager created with prefix_cache: the
 * sequence's leading complete blocks that are cached are shared, not
 * charged, and *reused_blocks (may be NULL) receives their number; its other
 * complete prompt blocks are indexed. PKV_EINVAL without prefix_cache. */
pkv_status pkv_bm_admit_tokens(pkv_bm* bm, const int32_t* tokens, int prompt_len, int max_new,
                               int* seq_id, int* reused_blocks);

/* child_ids: host int32 [n]. All-or-nothing. The parent must be running. */
pkv_status pkv_bm_fork(pkv_bm* bm, int parent_seq, int n, int32_t* child_ids);

/* For each listed sequence (distinct ids, processed in order): the slot of
 * its next token and, where that token lands in a shared block, one
 * copy-on-write pair; then its context length grows by one.
 *   slot_mapping_out : host int64 [n]
 *   cow_pairs_out    : host int32 [n][2] (at most one pair per sequence)
 *   n_pairs_out      : number of pairs written
 * Sequences must be running. Full reservation: PKV_ENOSPC if a sequence has
 * no reserved slot left. Incremental: PKV_ENOMEM if the step needs more pages
 * than are available. Either way nothing changes. */
pkv_status pkv_bm_prepare_append(pkv_bm* bm, const int32_t* seq_ids, int n,
                                 int64_t* slot_mapping_out, int32_t* cow_pairs_out,
                                 int* n_pairs_out);

/* Ends a sequence (running or preempted) and releases its references. */
pkv_status pkv_bm_free(pkv_bm* bm, int seq_id);

/* Preemption by recompute: releases a running sequence's references (its
 * table becomes empty) and keeps its context length; *released_blocks (may
 * be NULL) receives its former table length. */
pkv_status pkv_bm_preempt(pkv_bm* bm, int seq_id, int* released_blocks);

/* Re-admits a preempted sequence on fresh private pages (its context length
 * rounded up under incremental, its full allowance otherwise), leaving the
 * watermark available; the caller recomputes the KV of its context_len
 * tokens into them. PKV_ENOMEM leaves it preempted. */
pkv_status pkv_bm_resume(pkv_bm* bm, int seq_id);

/* Slots (block id * block_tokens + offset) of a running sequence's token
 * positions [first, first + n) into slots_out (host int64 [n]): where a
 * prefill, or the recompute after pkv_bm_resume, writes their KV with
 * pkv_append. Positions must lie within the sequence's table (PKV_EINVAL
 * otherwise). A position in a block shared with other sequences is shared
 * too: writing it changes their KV. */
pkv_status pkv_bm_slots(pkv_bm* bm, int seq_id, int first, int n, int64_t* slots_out);

/* Id of the most recently admitted running sequence, -1 if none. */
int pkv_bm_newest_running(pkv_bm* bm);

/* Block table of one sequence into out[0 .. capacity); *length = its length.
 * PKV_ERANGE if capacity is too small. */
pkv_status pkv_bm_block_table(pkv_bm* bm, int seq_id, int32_t* out, int capacity,
                              int* length);

pkv_status pkv_bm_context_len(pkv_bm* bm, int seq_id, int* context_len);

/* Padded batch view: tables_out int32 [n][width] (unused entries -1) and
 * context_lens_out int32 [n], ready to copy to the device for
 * pkv_attn_decode. PKV_ERANGE if a table is longer than width; PKV_EINVAL if
 * a sequence is unknown or preempted. */
pkv_status pkv_bm_batch_tables(pkv_bm* bm, const int32_t* seq_ids, int n,
                               int32_t* tables_out, int width, int32_t* context_lens_out);

pkv_status pkv_bm_stats(pkv_bm* bm, pkv_bm_stats_t* stats);

/* Reference count of a physical block (-1 if out of range). */
int pkv_bm_refcount(pkv_bm* bm, int block);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
