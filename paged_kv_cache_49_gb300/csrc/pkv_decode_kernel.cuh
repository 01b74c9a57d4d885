// Paged decode attention for sm_103a: the device code (decode_kernel and its
// helpers), included by pkv_attn.cu, which holds the launches and the C ABI.
//
// What it computes (cs2680 Lecture 10, §10.3, step three; "KV cache systems",
// block-table indirection paragraph): for every sequence s and query head h,
// softmax(scale * q[s,h] . K_t) weighted sum of V_t over the sequence's
// context, where token t lives in physical block table[s][t / 16], row t % 16.
//
// How (GB300 design):
//  * Work split. The context of every (sequence, KV head) pair is a run of
//    16-token blocks; all runs are laid end to end, in (sequence, KV head)
//    order, and the whole line is cut into gridDim.x ranges of equal cost
//    (a tile costs 1, each run kPieceCost more), one per persistent CTA.
//    Every CTA derives the same split on the device from context_lens (a
//    prefix sum over sequences), so the call needs no host-side knowledge of
//    the lengths and is balanced whatever the length mix. A pair cut by a
//    range boundary becomes two or more pieces; each piece leaves an fp32
//    partial (max, sum, unnormalised output) and the CTA that finishes a
//    pair's last piece merges them with a log-sum-exp rescale ("last arrival
//    merges": one atomic counter per pair, no waiting on other CTAs, reset by
//    the merger; pairs cut among more than eight CTAs merge in two levels).
//  * Roles. Warp 4 produces: it walks the range, reads block ids from the
//    table, and issues TMA tile loads (two 16 x 64 bf16 boxes per 4 KiB K or V
//    block, 128-byte swizzle, L2 evict-first) into an 8-stage ring of shared
//    memory, one block of K and V per stage; the query rows of a piece arrive
//    by one bulk copy into a 2-slot ring. Warps 0-3 consume the ring's blocks,
//    block i of the CTA's stream going to warp i % 4. Warp 5 merges: at the
//    end of a piece the consumers drop their softmax states into a merge slot
//    (two slots, or one for batches whose prefix sums leave room for no more)
//    and move on; the merge warp combines them and writes the output row (or
//    the partial, then the cross-CTA merge), so the ring keeps streaming
//    across piece boundaries. A pair of one tile is finished by its owner
//    consumer warp without the merge warp.
//  * Math, per block and consumer warp: S^T[16 tokens x 8 heads] = K Q^T on
//    the tensor cores (mma.sync m16n8k16, bf16 in, fp32 out, K fragments by
//    ldmatrix from the swizzled stage), an online softmax in fp32 (max over
//    tokens by shuffles, exp2 in the log2 domain), P cast to bf16 and
//    transposed in registers (movmatrix), then O^T[128 dims x 8 heads] +=
//    V^T P^T (V fragments by ldmatrix.trans). The GQA group of up to 8 query
//    heads is the mma's N dimension, so each K/V byte is read once for the
//    whole group. The softmax denominator sums the bf16-rounded weights that
//    multiply V, so the output is an exact convex combination of V rows up to
//    fp32 rounding.
//  * Tokens past the context in the last block are masked: their scores are
//    set to -inf and their V values to zero before the mma, so unwritten
//    (even non-finite) slots never reach the output.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>
#include <cstdint>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace attn {

constexpr int kTok = 16;  // tokens per tile, the kernel's unit of work (cache blocks hold kBT tokens)
constexpr int kDim = PKV_ATTN_HEAD_DIM;  // head dim
constexpr int kMaxG = PKV_ATTN_MAX_GROUP;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMergeWarp = kConsumerWarps + 1;
constexpr int kThreads = kConsumers + 64;
constexpr int kStages = 8;
static_assert(kStages % kConsumerWarps == 0, "each stage must map to one consumer warp");
static_assert((kConsumerWarps & (kConsumerWarps - 1)) == 0, "consumer warp count is a power of two");
constexpr int kQSlots = 2;
// After an abort, how long the producer waits before its drain (see there).
constexpr uint64_t kDrainGraceNs = 100000;  // 100 us
// Work partition cost of one (sequence, KV head) run beyond its tiles, in
// tiles: what a piece's fixed work (its query rows, the hand-over between
// consumer warps, the merge warp's combine and any cross-CTA merge) costs a
// CTA, next to streaming one 8 KB tile at its share of HBM bandwidth.
constexpr int kPieceCost = 3;
// Pairs split into more pieces than this merge in two levels (see the merge
// warp).
constexpr int kMergeGroup = 8;
constexpr int kHalfBytes = kTok * 64 * 2;  // one 16 x 64 bf16 box
constexpr int kBlockBytes = 2 * kHalfBytes;  // one K (or V) block of one KV head
// A stage's K (and V) tile in shared memory: 16 token rows of two 64-column
// halves, each row 128 bytes in the 128-byte swizzle, in atoms of 8 rows of
// one half. With blocks of 16 tokens or more the halves are 2 KB apart and
// the two 8-row atoms of a half adjacent (one box: both halves of 16 rows);
// with 8-token blocks the rows 0-7 and 8-15 come from two blocks, one box
// each ({64, 8, 2}: both halves of 8 rows), so there the 8-row groups are 2
// KB apart and the halves adjacent.
template <int kBT>
struct TileLayout {
    static constexpr uint32_t kHalf = kBT >= kTok ? kHalfBytes : kHalfBytes / 2;   // between the halves
    static constexpr uint32_t kRows8 = kBT >= kTok ? kHalfBytes / 2 : kHalfBytes;  // between rows 0-7 and 8-15
};
constexpr int kStageBytes = 2 * kBlockBytes;
constexpr int kQBytes = kMaxG * kDim * 2;
constexpr int kORow = 132;  // floats per head row of merge buffers and partials
constexpr int kPartialFloats = kMaxG * kORow;
constexpr int kMergeOFloats = kConsumerWarps * kMaxG * kORow;  // one merge slot
constexpr int kMergeMLFloats = kConsumerWarps * kMaxG;

constexpr int kOffStages = 0;
constexpr int kOffQ = kOffStages + kStages * kStageBytes;
constexpr int kOffO = kOffQ + kQSlots * kQBytes;
// The rest of the layout depends on the number of merge slots S (consumer
// warps' piece states waiting for the merge warp): 2 lets the consumers
// finish a piece while the merge warp combines the previous one; 1 saves
// 16.9 KB, which keeps two CTAs per SM for batches whose prefix sums would
// otherwise push a CTA past half of the SM's shared memory.
template <int S>
struct Layout {
    static constexpr int kOffM = kOffO + S * kMergeOFloats * 4;
    static constexpr int kOffL = kOffM + S * kMergeMLFloats * 4;
    static constexpr int kOffBar = kOffL + S * kMergeMLFloats * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kQSlots + 2 * S;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffScan = kOffMisc + 128;
};

// Slots (ints) of the small shared-memory area misc[]
constexpr int kMiscAbort = 0;    // the CTA's abort flag
constexpr int kMiscEnds = 2;     // [2], [3]: the CTA's range [lo, hi) of tiles
constexpr int kMiscEarly = 4;    // [4]: first-piece tiles copied by the merge warp, [5]: 1 if its query rows too
constexpr int kMiscWarpTot = 8;  // [8, 8 + warps): per-warp sums of the plan
constexpr int kMiscFirst = 16;   // [16, 20): the walk's first piece: sequence (or -1), run, block, line position

__host__ __device__ constexpr int off_scan(int slots) {
    return slots == 1 ? Layout<1>::kOffScan : Layout<2>::kOffScan;
}

// Dynamic shared memory: the fixed part, the prefix sum (4 bytes per
// sequence), each sequence's last-tile token count (1 byte per sequence) and,
// when leading tiles are skipped (the private pass of cascade attention), each
// sequence's skipped tile count (4 bytes per sequence).
__host__ __device__ constexpr size_t skip_offset(int num_seqs, int slots) {
    return (off_scan(slots) + 5 * static_cast<size_t>(num_seqs) + 3) & ~size_t(3);
}
constexpr size_t smem_bytes(int num_seqs, bool skip, int slots) {
    return 1024 + (skip ? skip_offset(num_seqs, slots) + 4 * static_cast<size_t>(num_seqs)
                        : off_scan(slots) + 5 * static_cast<size_t>(num_seqs));
}

constexpr size_t kWsHeader = 256;

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Most persistent CTAs of one launch: the workspace keeps three counters for
// each possible CTA (below), so that their place never depends on the launch.
constexpr int kMaxCtas = PKV_ATTN_MAX_CTAS;

// Counters, per CTA c: [c] counts the pieces of the split pair whose first
// piece is c's (a CTA's range ends inside at most one pair, so each split
// pair has its own counter), [kMaxCtas + 2c + slot] counts the pieces of a
// two-level merge group whose first piece is c's. Every launch leaves them at
// zero. Their region has one size for every launch shape, so no launch ever
// places a counter over memory that another launch (another batch or grid)
// used for partials.
constexpr size_t kWsCounterBytes = align256(static_cast<size_t>(kMaxCtas) * 3 * 4);

// Per CTA: two fp32 partial slots.
constexpr size_t kWsPerCta = 2 * kPartialFloats * 4;

// Workspace: header (error word), the counters, then the CTAs' partial slots.
constexpr size_t kWsFixed = kWsHeader + kWsCounterBytes;

inline size_t workspace_bytes(int grid) { return kWsFixed + static_cast<size_t>(grid) * kWsPerCta; }

struct Params {
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int max_blocks;
    int cap_tokens;  // max_blocks * block tokens: longest context a table row can hold
    int num_blocks;
    float scale_log2;
    uint32_t* err;
    int* counters;        // [kMaxCtas]: pieces counted per split pair, by the pair's first CTA
    float* partials;
    int* group_counters;  // [kMaxCtas][2]: pieces counted per group of a two-level merge
    // Cascade attention's private pass (both null otherwise): per sequence,
    // leading tiles to skip (computed elsewhere), and where a sequence with
    // skipped tiles leaves its unnormalised fp32 result instead of an output
    // row ([num_seqs * num_q_heads][kORow]: output, max, sum).
    const int32_t* skip_tiles;
    float* side;
    // Tests of the bounded-wait path only (-1 otherwise): CTA 0's producer
    // issues the copies of its first stop_tiles tiles and skips the rest, so
    // that a consumer's wait on the next one runs out.
    int stop_tiles;
};

// Position in the line of (sequence, KV head) block runs.
struct Cursor {
    int s, g, blk;
};

__device__ __forceinline__ int run_blocks(const int* scan, int s) {
    return scan[s] - (s > 0 ? scan[s - 1] : 0);
}

// Smallest i in [0, n) for which pred(i) holds, for a predicate that is
// false below some index and true from there on, and true at n - 1. The whole
// warp calls it. Each round splits the interval into 32 chunks, one per lane,
// and keeps the first chunk whose last index satisfies the predicate: 64
// sequences take two rounds of one shared-memory read per lane, where a
// binary search takes six dependent reads (about 100 cycles each on the
// start-up path, where every step is serial).
template <class Pred>
__device__ __forceinline__ int warp_first_true(int n, Pred pred) {
    const int lane = static_cast<int>(threadIdx.x & 31);
    int lo = 0, len = n;
    while (len > 1) {
        const int step = (len + 31) >> 5;
        const int i = min(lo + (lane + 1) * step, lo + len) - 1;
        const int c = __ffs(__ballot_sync(0xffffffffu, pred(i))) - 1;
        lo += c * step;
        len = min(step, len - c * step);
    }
    return lo;
}

// a / b for 0 <= a < 2^30 and b >= 1 whose quotient is small (below the KV
// head count where it is used): a single-precision estimate, then corrected
// to the exact quotient. Shorter than an integer division on the start-up
// path, where only one thread needs it.
__device__ __forceinline__ int div_small(int a, int b) {
    int q = static_cast<int>(__fdividef(static_cast<float>(a), static_cast<float>(b)));
    while (q > 0 && q * b > a) --q;
    while ((q + 1) * b <= a) ++q;
    return q;
}

// Position x of the line (x < total) as a cursor. The whole warp calls it.
// Positions on the line, and cost positions of the work partition, are
// 32-bit: the host rejects launches whose line could reach 2^30 cost units.
__device__ __forceinline__ Cursor locate(const int* scan, int n, int hkv, int x) {
    Cursor c;
    // the sequence: smallest s with hkv * scan[s] > x, i.e. scan[s] > floor(x / hkv)
    c.s = warp_first_true(n, [&](int i) { return hkv * scan[i] > x; });
    const int nb = run_blocks(scan, c.s);
    const int off = x - hkv * (scan[c.s] - nb);  // in [0, hkv * nb)
    // the run, off / nb: lanes 1 .. hkv - 1 count the run starts at or below
    // off (a division beyond 32 KV heads)
    const int lane = static_cast<int>(threadIdx.x & 31);
    c.g = hkv <= 32 ? __popc(__ballot_sync(0xffffffffu, lane >= 1 && lane < hkv && lane * nb <= off)) : off / nb;
    c.blk = off - c.g * nb;
    return c;
}

__device__ __forceinline__ void advance(Cursor& c, const int* scan, int n, int hkv, int len) {
    c.blk += len;
    if (c.blk == run_blocks(scan, c.s)) {
        c.blk = 0;
        if (++c.g == hkv) {
            c.g = 0;
            do { ++c.s; } while (c.s < n && run_blocks(scan, c.s) == 0);
        }
    }
}

// One piece: blocks [blk, blk + len) of the run of (sequence s, KV head g),
// whose run has nb blocks; start = its position on the line.
struct Piece {
    int s, g, blk, nb, len;
    int start;
};

// The pieces of one CTA's range in processing order: the range's last piece
// first, then the others from the start of the range. A pair split between
// neighbouring CTAs is the last piece of one and the first piece of the
// next, so both halves are processed early and their merge overlaps the
// streaming instead of landing on the kernel's tail.
struct PieceWalk {
    const int* scan;
    int n, hkv;
    int range_lo, split, x, end;
    int part;
    Cursor c;

    // first: the first piece as the plan found it (sequence, run, block,
    // line position), or first[0] = -1 when the plan left it to the search.
    __device__ PieceWalk(const int* scan_, int n_, int hkv_, int lo, int hi, const int* first)
        : scan(scan_), n(n_), hkv(hkv_), range_lo(lo), part(0) {
        end = hi;
        if (first[0] >= 0) {
            c.s = first[0];
            c.g = first[1];
            c.blk = first[2];
            split = first[3];
        } else {
            const Cursor last = locate(scan, n, hkv, hi - 1);
            const int nb = run_blocks(scan, last.s);
            const int seg = hkv * (scan[last.s] - nb) + last.g * nb;
            split = seg > lo ? seg : lo;
            c = locate(scan, n, hkv, split);
        }
        x = split;
    }

    __device__ bool next(Piece& pc) {
        if (x >= end) {
            if (part == 1 || split <= range_lo) return false;
            part = 1;
            x = range_lo;
            end = split;
            c = locate(scan, n, hkv, x);
        }
        const int nb = run_blocks(scan, c.s);
        pc.s = c.s;
        pc.g = c.g;
        pc.blk = c.blk;
        pc.nb = nb;
        pc.len = min(nb - c.blk, end - x);
        pc.start = x;
        advance(c, scan, n, hkv, pc.len);
        x += pc.len;
        return true;
    }
};

// ---- CUDA-core variant of the consumer math ----------------------------------
// The same pieces, rings, online softmax and merge hand-off as the tensor-core
// consumers, with the dot products and the P.V update on the FP32 pipe, so
// that the choice of tensor cores for the GQA group tile can be measured
// against it. G (the group size, 4 or 8) is a compile-time constant here.
// Lane l owns head dims [4l, 4l + 4) of every query head of the group, for
// K.q as for P.V: its q values (4 x G, pre-scaled into the log2 domain) stay
// in registers. Per round of 32 / G tokens, each lane forms the partial dot
// products of those tokens x G heads over its dims (32 values) and a
// butterfly reduce-scatter over the warp (five exchange rounds) leaves lane L
// with the whole score of token L / G, head L % G. The probabilities and the
// per-head rescale factors reach every lane through the K half of the warp's
// current stage, which is dead once the scores are formed.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < o; ++j) {
            const float keep = up ? v[o + j] : v[j];
            const float send = up ? v[j] : v[o + j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

template <int kSlots, int G>
__device__ __forceinline__ void fma_consumer_warp(const Params& p, uint8_t* smem, const int* scan,
                                                  const uint8_t* tail, int range_lo, int range_hi, const int* first,
                                                  int warp, int lane, volatile int* abort_flag, uint32_t bar0) {
    static_assert(G == 4 || G == 8, "CUDA-core variant: group sizes 4 and 8");
    using LY = Layout<kSlots>;
    constexpr int kTpc = 32 / G;         // tokens per reduce-scatter round
    constexpr int kRounds = kTok / kTpc; // rounds per tile
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kStages + i); };
    auto qfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
    auto qempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + kQSlots + i); };
    auto mfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * kQSlots + i); };
    auto mempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * kQSlots + kSlots + i); };
    float* sm_o = reinterpret_cast<float*>(smem + kOffO);
    float* sm_m = reinterpret_cast<float*>(smem + LY::kOffM);
    float* sm_l = reinterpret_cast<float*>(smem + LY::kOffL);
    const int B = p.num_seqs, Hkv = p.num_kv_heads;
    const int d0 = 4 * lane;
    // dims [d0, d0 + 4) of a token row: box d0 / 64, 16-byte chunk (d0 % 64) / 8 (XOR-swizzled by the row), byte 0 or 8
    const int box_off = (d0 >> 6) * kHalfBytes;
    const int chunk = (d0 & 63) >> 3;
    const int sub = (d0 & 7) * 2;
    const int my_head = lane % G;
    const int my_tok = lane / G;
    const float NEG_INF = -INFINITY;

    PieceWalk walk(scan, B, Hkv, range_lo, range_hi, first);
    Piece pc;
    int gidx0 = 0, qslot = 0, piece = 0;
    uint32_t qphase = 0;
    while (walk.next(pc)) {
        const int s = pc.s, blk0 = pc.blk, nb = pc.nb, len = pc.len;
        const int last_valid = tail[s];
        const int first = (warp - static_cast<int>(gidx0 % kConsumerWarps)) & (kConsumerWarps - 1);
        const bool mine = first < len;

        float q[G][4];
        auto take_q = [&](int h, uint2 w) {
            q[h][0] = bf16_lo(w.x) * p.scale_log2;
            q[h][1] = bf16_hi(w.x) * p.scale_log2;
            q[h][2] = bf16_lo(w.y) * p.scale_log2;
            q[h][3] = bf16_hi(w.y) * p.scale_log2;
        };
        if (len >= kConsumerWarps) {
            const bool landed = mbar_wait(qfull_bar(qslot), qphase, abort_flag, p.err);
            const uint8_t* qs = smem + kOffQ + qslot * kQBytes + d0 * 2;
            uint32_t held = 0;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint2 w = *reinterpret_cast<const uint2*>(qs + h * kDim * 2);
                held ^= w.x ^ w.y;
                take_q(h, w);
            }
            const uint32_t z = __reduce_or_sync(0xffffffffu, zero_after(held));  // 0, once all lanes hold theirs
            if (lane == 0 && landed) mbar_arrive(qempty_bar(qslot) + z);
            if (++qslot == kQSlots) { qslot = 0; qphase ^= 1u; }
        } else if (mine) {
            const __nv_bfloat16* qg = p.q + (static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(pc.g) * G) * kDim + d0;
#pragma unroll
            for (int h = 0; h < G; ++h) take_q(h, __ldg(reinterpret_cast<const uint2*>(qg + h * kDim)));
        }

        float m_own = NEG_INF;  // running max of head my_head
        float l_own = 0.f;      // this lane's share of head my_head's sum
        float o[G][4];
#pragma unroll
        for (int h = 0; h < G; ++h) o[h][0] = o[h][1] = o[h][2] = o[h][3] = 0.f;

        for (int jb = first; jb < len; jb += kConsumerWarps) {  // block gi goes to warp gi % 4, as in the tensor-core consumers
            const int gi = gidx0 + jb;
            const int st = static_cast<int>(gi % kStages);
            const bool landed = mbar_wait(full_bar(st), static_cast<uint32_t>((gi / kStages) & 1), abort_flag, p.err);
            const int valid = (blk0 + jb == nb - 1) ? last_valid : kTok;
            uint8_t* stage = smem + kOffStages + st * kStageBytes;
            const uint8_t* sk = stage + box_off;
            const uint8_t* sv = stage + kBlockBytes + box_off;

            float sc[kRounds];
#pragma unroll
            for (int c = 0; c < kRounds; ++c) {
                float part[32];
#pragma unroll
                for (int tl = 0; tl < kTpc; ++tl) {
                    const int t = c * kTpc + tl;
                    const uint2 kw = *reinterpret_cast<const uint2*>(sk + t * 128 + (((chunk ^ (t & 7)) << 4) | sub));
                    const float k0 = bf16_lo(kw.x), k1 = bf16_hi(kw.x), k2 = bf16_lo(kw.y), k3 = bf16_hi(kw.y);
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        part[tl * G + h] = fmaf(k3, q[h][3], fmaf(k2, q[h][2], fmaf(k1, q[h][1], k0 * q[h][0])));
                }
                sc[c] = reduce_scatter32(part, lane);  // token c * kTpc + my_tok, head my_head
            }
            float bm = NEG_INF;
#pragma unroll
            for (int c = 0; c < kRounds; ++c) {
                if (c * kTpc + my_tok >= valid) sc[c] = NEG_INF;
                bm = fmaxf(bm, sc[c]);
            }
#pragma unroll
            for (int off = G; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
            const float mn = fmaxf(m_own, bm);
            const float al = ex2(m_own - mn);
            m_own = mn;
            // probabilities [16 tokens][G heads], then the G rescale factors,
            // over the stage's first K box (every lane's K reads are done)
            __syncwarp();
            float* pb = reinterpret_cast<float*>(stage);
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < kRounds; ++c) {
                const float pv = ex2(sc[c] - mn);
                lsum += pv;
                pb[c * 32 + lane] = pv;  // = pb[token * G + head]
            }
            l_own = l_own * al + lsum;
            if (lane < G) pb[kTok * G + lane] = al;
            __syncwarp();
#pragma unroll
            for (int h = 0; h < G; h += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(pb + kTok * G + h);
                const float a[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    o[h + u][0] *= a[u];
                    o[h + u][1] *= a[u];
                    o[h + u][2] *= a[u];
                    o[h + u][3] *= a[u];
                }
            }
#pragma unroll
            for (int t = 0; t < kTok; ++t) {
                uint2 vw = *reinterpret_cast<const uint2*>(sv + t * 128 + (((chunk ^ (t & 7)) << 4) | sub));
                if (t >= valid) vw = make_uint2(0u, 0u);  // unwritten slots past the context never reach the output
                const float v0 = bf16_lo(vw.x), v1 = bf16_hi(vw.x), v2 = bf16_lo(vw.y), v3 = bf16_hi(vw.y);
#pragma unroll
                for (int h = 0; h < G; h += 4) {
                    const float4 p4 = *reinterpret_cast<const float4*>(pb + t * G + h);
                    const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        o[h + u][0] = fmaf(pr[u], v0, o[h + u][0]);
                        o[h + u][1] = fmaf(pr[u], v1, o[h + u][1]);
                        o[h + u][2] = fmaf(pr[u], v2, o[h + u][2]);
                        o[h + u][3] = fmaf(pr[u], v3, o[h + u][3]);
                    }
                }
            }
            fence_proxy_async_shared();  // this lane's reads of the stage, before the copy that will replace it
            __syncwarp();
            if (lane == 0 && landed) mbar_arrive(empty_bar(st));
        }
        gidx0 += len;

        if (mine) {  // the whole sum of head my_head in every lane of that head
#pragma unroll
            for (int off = G; off < 32; off <<= 1) l_own += __shfl_xor_sync(0xffffffffu, l_own, off);
        }
        if (nb == 1) {  // a pair of one tile: its owner warp writes the rows
            if (mine) {
                __nv_bfloat16* dst = p.out + (static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(pc.g) * G) * kDim + d0;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float inv = 1.f / __shfl_sync(0xffffffffu, l_own, h);
                    uint2 w2;
                    w2.x = pack_bf16x2(o[h][0] * inv, o[h][1] * inv);
                    w2.y = pack_bf16x2(o[h][2] * inv, o[h][3] * inv);
                    *reinterpret_cast<uint2*>(dst + h * kDim) = w2;
                }
            }
            continue;
        }
        const int ms = piece % kSlots;
        mbar_wait(mempty_bar(ms), static_cast<uint32_t>(((piece / kSlots) & 1) ^ 1), abort_flag, p.err);
        if (mine) {
#pragma unroll
            for (int h = 0; h < G; ++h)
                *reinterpret_cast<float4*>(sm_o + ms * kMergeOFloats + (warp * kMaxG + h) * kORow + d0) =
                    make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
            if (lane < G) {
                sm_m[ms * kMergeMLFloats + warp * kMaxG + lane] = m_own;
                sm_l[ms * kMergeMLFloats + warp * kMaxG + lane] = l_own;
            }
        }
        mbar_arrive(mfull_bar(ms));
        ++piece;
    }
}

// kBT: tokens per cache block (8, 16, 32 or 64). A 16-token tile is rows
// [(t mod kBT/16) * 16, +16) of block table[t / (kBT/16)] when kBT >= 16, and
// the two 8-row blocks table[2t], table[2t + 1] when kBT == 8.
// kSkip: the private pass of cascade attention (per-sequence skipped tiles,
// fp32 results for grouped sequences); a separate instantiation, so that the
// plain kernel carries none of its branches. kSlots: merge slots (1 or 2).
// kFmaG: 0 for the tensor-core consumers; 4 or 8 for the CUDA-core variant
// of their math compiled for that group size (16-token blocks only).
// One tile's copies into a stage: K then V, 16 token rows each as one box
// of both 64-column halves (blocks of 16 tokens or more), or, with 8-token
// blocks, as two boxes of 8 rows and both halves, rows 0-7 from the block at
// ya and rows 8-15 from the block at yb (TileLayout).
template <int kBT>
__device__ __forceinline__ void issue_tile(uint32_t dst, const CUtensorMap* tm_k, const CUtensorMap* tm_v, int ya,
                                           int yb, uint32_t fb, uint64_t policy) {
    tma_load_3d(dst, tm_k, 0, ya, 0, fb, policy);
    tma_load_3d(dst + kBlockBytes, tm_v, 0, ya, 0, fb, policy);
    if constexpr (kBT < kTok) {
        tma_load_3d(dst + TileLayout<kBT>::kRows8, tm_k, 0, yb, 0, fb, policy);
        tma_load_3d(dst + kBlockBytes + TileLayout<kBT>::kRows8, tm_v, 0, yb, 0, fb, policy);
    }
}

template <int kBT, bool kSkip, int kSlots, int kFmaG = 0>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int B = p.num_seqs;
    const int Hkv = p.num_kv_heads;
    const int G = p.group;

    using LY = Layout<kSlots>;
    int* scan = reinterpret_cast<int*>(smem + LY::kOffScan);
    uint8_t* tail = smem + LY::kOffScan + 4 * static_cast<size_t>(B);  // tokens in each sequence's last tile
    int* skip = kSkip ? reinterpret_cast<int*>(smem + skip_offset(B, kSlots)) : nullptr;
    auto skipped = [&](int s) { return skip ? skip[s] : 0; };
    int* misc = reinterpret_cast<int*>(smem + LY::kOffMisc);
    volatile int* abort_flag = misc + kMiscAbort;
    int* warp_tot = misc + kMiscWarpTot;  // kThreads / 32 of them
    const int* first = misc + kMiscFirst;
    float* sm_o = reinterpret_cast<float*>(smem + kOffO);
    float* sm_m = reinterpret_cast<float*>(smem + LY::kOffM);
    float* sm_l = reinterpret_cast<float*>(smem + LY::kOffL);
    const uint32_t bar0 = smem_u32(smem + LY::kOffBar);
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (kStages + i); };
    auto qfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
    auto qempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + kQSlots + i); };
    auto mfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * kQSlots + i); };
    auto mempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * kQSlots + kSlots + i); };

    if (warp == kProducerWarp && lane == 0) {  // fetch the TMA descriptors while the plan runs
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        for (int i = 0; i < kQSlots; ++i) {
            mbar_init(qfull_bar(i), 1);
            mbar_init(qempty_bar(i), kConsumerWarps);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(mfull_bar(i), kConsumers);
            mbar_init(mempty_bar(i), 32);
        }
        misc[0] = 0;
        misc[kMiscEarly] = 0;
        misc[kMiscEarly + 1] = 0;
        misc[kMiscFirst] = -1;
        fence_barrier_init();
    }

    // ---- plan: inclusive prefix sum of block-run lengths over sequences ----
    // The work partition deals out cost, not tiles: tile x of run r = s * hkv
    // + g sits at cost position x + kPieceCost * r, so that each run is
    // followed by a gap of kPieceCost positions that hold no tile. CTA b takes
    // the tiles whose cost position lies in [b, b + 1) * cchunk: equal shares
    // of tiles plus per-run overhead, so that a CTA whose range is cut into
    // many short pieces streams fewer tiles. Each end of that range is found
    // by the thread holding the sequence whose cost span contains it, while
    // it writes the prefix sum: no search of the prefix sum and no third
    // block barrier stand between the context lengths and the first copy.
    int* ends = misc + kMiscEnds;
    int cchunk;
    {
        const int per = (B + kThreads - 1) / kThreads;
        const int lo = min(B, tid * per);
        const int hi = min(B, lo + per);
        const int cap = p.cap_tokens;
        int local = 0;
        for (int s = lo; s < hi; ++s) {
            const int c = __ldg(p.context_lens + s);
            if (c > cap && p.err) atomicOr(p.err, PKV_DEVERR_CONTEXT);
            const int cc = min(c, cap);
            const int all = cc > 0 ? (cc + kTok - 1) / kTok : 0;
            int sk = 0;
            if (skip) {
                sk = __ldg(p.skip_tiles + s);
                if (sk < 0 || sk > all) {  // more skipped tiles than the context holds
                    if (p.err) atomicOr(p.err, PKV_DEVERR_CONTEXT);
                    sk = sk < 0 ? 0 : all;
                }
                skip[s] = sk;
            }
            scan[s] = all - sk;  // the run length; the second pass turns it into the prefix
            tail[s] = static_cast<uint8_t>(cc - kTok * (all - 1));  // 1..16 (unused when all == 0)
            local += all - sk;
        }
        int v = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += n;
        }
        if (lane == 31) warp_tot[warp] = v;
        __syncthreads();
        int run = v - local, per_head = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int t = warp_tot[w];
            per_head += t;
            if (w < warp) run += t;
        }
        const int cost_total = Hkv * (per_head + kPieceCost * B);
        cchunk = (cost_total + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
        const int y_lo = static_cast<int>(blockIdx.x) * cchunk;
        const int y_hi = y_lo + cchunk;
        for (int s = lo; s < hi; ++s) {
            const int before = run;
            run += scan[s];
            scan[s] = run;
            // Sequence s spans cost positions [c0, c0 + hkv * (nb + kPieceCost)):
            // run g's tiles at c0 + g * (nb + kPieceCost) + j for j < nb, then
            // its gap. The range end at y is the first tile at or after y.
            const int nb = run - before;
            const int c0 = Hkv * (before + kPieceCost * s);
            const int c1 = c0 + Hkv * (nb + kPieceCost);
            auto tile_at = [&](int y) {
                const int off = y - c0;
                const int g = div_small(off, nb + kPieceCost);
                return Hkv * before + g * nb + min(off - g * (nb + kPieceCost), nb);
            };
            if (y_lo >= c0 && y_lo < c1) ends[0] = tile_at(y_lo);
            if (y_hi >= c0 && y_hi < c1) {
                const int off = y_hi - c0;
                const int g = div_small(off, nb + kPieceCost);
                const int r = min(off - g * (nb + kPieceCost), nb);  // tiles of run g before the end
                const int hi_t = Hkv * before + g * nb + r;
                ends[1] = hi_t;
                // The walk's first piece is the part of the range in the run
                // holding tile hi_t - 1 (run g, or the last tile of run g -
                // 1). When that run is this sequence's, this thread records
                // the piece, so that no warp searches for it, and how many of
                // its tiles the merge warp (idle until the first piece ends)
                // copies right after the plan (once the step's earlier kernels
                // are done, when launched behind them): the producer's own
                // first copies come several microseconds later, most of it cold
                // instruction fetch.
                if (nb > 0 && (r > 0 || g > 0)) {
                    const int gl = r > 0 ? g : g - 1;
                    const int seg = Hkv * before + gl * nb;  // the run's first tile
                    const int split = y_lo >= c0 ? max(seg, tile_at(y_lo)) : seg;
                    const int len = hi_t - split;
                    if (len > 0) {
                        misc[kMiscFirst] = s;
                        misc[kMiscFirst + 1] = gl;
                        misc[kMiscFirst + 2] = split - seg;
                        misc[kMiscFirst + 3] = split;
                        int n = min(len, kStages);
                        if (blockIdx.x == 0 && p.stop_tiles >= 0) n = min(n, p.stop_tiles);
                        misc[kMiscEarly] = n;
                        misc[kMiscEarly + 1] = n > 0 && len >= kConsumerWarps;
                    }
                }
            }
        }
        if (tid == 0) {  // an end past the last cost position: the line's end
            if (y_lo >= cost_total) ends[0] = Hkv * per_head;
            if (y_hi >= cost_total) ends[1] = Hkv * per_head;
        }
        __syncthreads();
    }
    const int range_lo = ends[0];
    const int range_hi = ends[1];

    // The merge warp, idle until the first piece ends, warms L2 with the
    // block-table entries and query rows of this CTA's range -- two
    // contiguous spans, from the range's first tile to its last, each capped
    // at kWarmBytes -- so that the producer's reads of them after its first
    // piece are L2 hits rather than dependent DRAM round trips.
    if (warp == kMergeWarp && range_lo < range_hi) {
        // The first piece's first tiles (up to the ring's depth) and query
        // rows, when the plan found the piece: lane j reads tile j's table
        // entries and copies it into stage j, where the producer would have
        // put it. Only the tiles can hold what the step's earlier kernels
        // (block copy, append) wrote: their copies wait for those kernels
        // (a no-op for an ordinary launch).
        const int n_first = misc[kMiscEarly];
        if (n_first > 0) {
            const int s = first[0], gl = first[1];
            const uint64_t policy = policy_evict_first();
            if (lane == 0 && misc[kMiscEarly + 1]) {
                mbar_arrive_expect_tx(qfull_bar(0), G * kDim * 2);
                bulk_load(smem_u32(smem + kOffQ),
                          p.q + (static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(gl) * G) * kDim,
                          G * kDim * 2, qfull_bar(0));
            }
            const bool mine = lane < n_first;
            int ya = 0, yb = 0;
            if (mine) {
                const int32_t* row = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
                const int sk0 = skipped(s);
                const int t = sk0 + first[2] + lane;  // the tile's index within the sequence
                auto checked = [&](int bid) {
                    if (bid < 0 || bid >= p.num_blocks) {
                        if (p.err) atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
                        bid = 0;  // read a valid block instead; the output is flagged invalid
                    }
                    return bid;
                };
                if constexpr (kBT >= kTok) {
                    ya = (checked(__ldg(row + t / (kBT / kTok))) * Hkv + gl) * kBT + (t % (kBT / kTok)) * kTok;
                } else {
                    const int seq_blocks = (kTok * (sk0 + run_blocks(scan, s) - 1) + tail[s] + kBT - 1) / kBT;
                    const int b0 = checked(__ldg(row + 2 * t));
                    const int b1 = 2 * t + 1 < seq_blocks ? checked(__ldg(row + 2 * t + 1)) : b0;
                    ya = (b0 * Hkv + gl) * kBT;
                    yb = (b1 * Hkv + gl) * kBT;
                }
            }
            griddep_wait();
            if (mine) {
                mbar_arrive_expect_tx(full_bar(lane), kStageBytes);
                issue_tile<kBT>(smem_u32(smem + kOffStages + lane * kStageBytes), &tm_k, &tm_v, ya, yb, full_bar(lane),
                                policy);
            }
        }
        constexpr size_t kWarmBytes = 256 * 1024;
        const Cursor a = locate(scan, B, Hkv, range_lo);
        const Cursor z = locate(scan, B, Hkv, range_hi - 1);
        auto warm = [&](const char* lo, const char* hi) {
            if (hi - lo > static_cast<ptrdiff_t>(kWarmBytes)) hi = lo + kWarmBytes;
            const char* line = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(lo) & ~uintptr_t(127));
            for (const char* x = line + lane * 128; x < hi; x += 32 * 128) prefetch_l2(x);
        };
        warm(reinterpret_cast<const char*>(p.block_tables + static_cast<size_t>(a.s) * p.max_blocks +
                                           (skipped(a.s) + a.blk) * kTok / kBT),
             reinterpret_cast<const char*>(p.block_tables + static_cast<size_t>(z.s) * p.max_blocks +
                                           ((skipped(z.s) + z.blk + 1) * kTok + kBT - 1) / kBT));
        warm(reinterpret_cast<const char*>(p.q + (static_cast<size_t>(a.s) * p.num_q_heads +
                                                  static_cast<size_t>(a.g) * G) * kDim),
             reinterpret_cast<const char*>(p.q + (static_cast<size_t>(z.s) * p.num_q_heads +
                                                  static_cast<size_t>(z.g + 1) * G) * kDim));
    }

    // Everything above but the merge warp's tile copies (which wait for
    // them) reads only inputs that the kernels of a decode step (block copy,
    // append) do not write. Of what follows, only the producer's tile loads
    // read what they wrote (the KV cache): the producer reads its first
    // piece's query rows and table entries first, then waits for those
    // kernels (when launched early) just before its first tile load. Every
    // other thread waits here, so that the grid never completes before the
    // kernels it was launched behind.
    if (warp != kProducerWarp) griddep_wait();

    // Sequences with no context get a zero output row (sequence s by CTA
    // s mod gridDim.x, merge warp).
    if (warp == kMergeWarp) {
        const int row_vec = p.num_q_heads * kDim / 8;
        for (int s = blockIdx.x; s < B; s += gridDim.x) {
            if (run_blocks(scan, s) != 0) continue;
            uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(s) * p.num_q_heads * kDim);
            for (int i = lane; i < row_vec; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
        }
    }
    if (range_lo >= range_hi) {
        if (warp == kProducerWarp) griddep_wait();
        return;
    }

    if (warp == kProducerWarp) {
        // ======================= producer warp =======================
        const uint64_t policy = policy_evict_first();
        PieceWalk walk(scan, B, Hkv, range_lo, range_hi, first);
        Piece pc;
        int stage = 0, qslot = 0;
        uint32_t sphase = 0, qphase = 0;
        int tile = 0;  // position in the CTA's stream of tiles
        const int stop_at = (p.stop_tiles >= 0 && blockIdx.x == 0) ? p.stop_tiles : INT_MAX;
        int issued = 0, q_issued = 0;  // copies issued into the stage ring and the query ring
        // Tiles [0, n_early) and, if q_early, the first query rows are
        // copied by the merge warp: skipped here, counted in the drain.
        const int n_early = misc[kMiscEarly];
        bool q_early = misc[kMiscEarly + 1] != 0;
        bool waited = false;  // griddep_wait done by this thread
        while (walk.next(pc)) {
            const int len = pc.len;
            if (len >= kConsumerWarps) {  // short pieces: the consumers read their query rows themselves
                if (lane == 0) {
                    if (q_early) {
                        q_early = false;
                        ++q_issued;
                    } else if (mbar_wait(qempty_bar(qslot), qphase ^ 1u, abort_flag, p.err)) {
                        fence_proxy_async_shared();  // the consumers' reads of the slot, before the copy over it
                        mbar_arrive_expect_tx(qfull_bar(qslot), G * kDim * 2);
                        const __nv_bfloat16* src =
                            p.q + (static_cast<size_t>(pc.s) * p.num_q_heads + static_cast<size_t>(pc.g) * G) * kDim;
                        bulk_load(smem_u32(smem + kOffQ + qslot * kQBytes), src, G * kDim * 2, qfull_bar(qslot));
                        ++q_issued;
                    }
                }
                if (++qslot == kQSlots) { qslot = 0; qphase ^= 1u; }
            }
            const int32_t* row = p.block_tables + static_cast<size_t>(pc.s) * p.max_blocks;
            const int sk0 = skipped(pc.s);  // the run starts at the sequence's tile sk0
            const int seq_blocks = (kTok * (sk0 + pc.nb - 1) + tail[pc.s] + kBT - 1) / kBT;  // valid table entries
            auto block_id = [&](int e) {
                int bid = __ldg(row + e);
                if (bid < 0 || bid >= p.num_blocks) {
                    if (p.err) atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
                    bid = 0;  // read a valid block instead; the output is flagged invalid
                }
                return bid;
            };
            for (int j0 = 0; j0 < len; j0 += 32) {
                int y0 = 0, y1 = 0;  // token-row coordinates of the tile's rows 0 and 8
                if (j0 + lane < len) {
                    const int t = sk0 + pc.blk + j0 + lane;  // tile index within the sequence
                    if constexpr (kBT >= kTok) {
                        y0 = (block_id(t / (kBT / kTok)) * Hkv + pc.g) * kBT + (t % (kBT / kTok)) * kTok;
                    } else {
                        const int b0 = block_id(2 * t);
                        const int b1 = 2 * t + 1 < seq_blocks ? block_id(2 * t + 1) : b0;  // past the end: masked
                        y0 = (b0 * Hkv + pc.g) * kBT;
                        y1 = (b1 * Hkv + pc.g) * kBT;
                    }
                }
                const int n = min(32, len - j0);
                for (int jj = 0; jj < n; ++jj) {
                    const int ya = __shfl_sync(0xffffffffu, y0, jj);
                    const int yb = __shfl_sync(0xffffffffu, y1, jj);
                    if (lane == 0) {
                        if (!waited) {
                            griddep_wait();
                            waited = true;
                        }
                        // tiles in [n_early, stop_at) only (stop_at: tests of the bounded waits)
                        if (static_cast<unsigned>(tile - n_early) < static_cast<unsigned>(stop_at - n_early) &&
                            mbar_wait(empty_bar(stage), sphase ^ 1u, abort_flag, p.err)) {
                            const uint32_t fb = full_bar(stage);
                            mbar_arrive_expect_tx(fb, kStageBytes);
                            issue_tile<kBT>(smem_u32(smem + kOffStages + stage * kStageBytes), &tm_k, &tm_v, ya, yb, fb,
                                            policy);
                            ++issued;
                        }
                    }
                    if (++stage == kStages) { stage = 0; sphase ^= 1u; }
                    ++tile;
                }
            }
        }
        // No copy may land in shared memory after the CTA has exited. Without
        // an abort every copy issued was waited on by a consumer warp, and
        // the wait below for the last copies into each ring (bounded) returns
        // at once. After an abort a consumer may have given up on a copy
        // still in flight, and the issued copies need not be a prefix of the
        // stream (a wait that gave up leaves a stage's phases one behind, and
        // a later parity wait on that stage can pass for the phase before),
        // so the producer first waits a grace period far longer than any copy
        // takes to land.
        if (!waited) griddep_wait();
        if (lane == 0) {
            if (*abort_flag) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < kDrainGraceNs) {
                }
            }
            volatile int never = 0;
            issued += n_early;
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(full_bar(i % kStages), static_cast<uint32_t>((i / kStages) & 1), &never, nullptr);
            for (int i = max(0, q_issued - kQSlots); i < q_issued; ++i)
                mbar_wait(qfull_bar(i % kQSlots), static_cast<uint32_t>((i / kQSlots) & 1), &never, nullptr);
        }
        return;
    }

    if (warp == kMergeWarp) {
        // ========================= merge warp =========================
        // Lane l owns dims [4l, 4l + 4) of every head of the piece.
        const float NEG_INF = -INFINITY;
        const int d0 = lane * 4;
        PieceWalk walk(scan, B, Hkv, range_lo, range_hi, first);
        Piece pc;
        int piece = 0;
        int gidx0 = 0;  // the CTA's block count before this piece, as the consumers count it
        while (walk.next(pc)) {
            const int s = pc.s, g = pc.g, nb = pc.nb;
            // consumer warps that hold blocks of this piece (all of them unless it is short)
            unsigned owners = 0;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w)
                if (((w - gidx0 % kConsumerWarps) & (kConsumerWarps - 1)) < pc.len) owners |= 1u << w;
            gidx0 += pc.len;
            if (nb == 1) continue;  // finished by its owner consumer warp
            // the CTAs holding pieces of this pair, from its cost positions
            const int seg_cost = Hkv * (scan[s] - nb) + g * nb + kPieceCost * (s * Hkv + g);
            const int i0 = seg_cost / cchunk;
            const int i1 = (seg_cost + nb - 1) / cchunk;
            const int pieces = i1 - i0 + 1;
            const int ms = piece % kSlots;
            mbar_wait(mfull_bar(ms), static_cast<uint32_t>((piece / kSlots) & 1), abort_flag, p.err);
            const float* mo = sm_o + ms * kMergeOFloats;
            const float* mm = sm_m + ms * kMergeMLFloats;
            const float* ml = sm_l + ms * kMergeMLFloats;
            __nv_bfloat16* out_base =
                p.out + (static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(g) * G) * kDim + d0;
            // Partial slots: a CTA holds at most two split pieces, one that
            // continues into the next CTA (slot 1) and one that ends a pair
            // begun in an earlier CTA (slot 0).
            const bool continues = pc.start + pc.len == range_hi && pc.blk + pc.len < nb;
            float* part = p.partials + (static_cast<size_t>(blockIdx.x) * 2 + (continues ? 1 : 0)) * kPartialFloats;
            // The pair's finished result for head h: a bf16 output row, or, for
            // a sequence whose leading tiles another pass covers, its
            // unnormalised fp32 result for the cascade merge.
            const bool to_side = kSkip && skipped(s) > 0;
            float* side_base = to_side ? p.side + (static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(g) * G) * kORow
                                       : nullptr;
            auto emit = [&](int h, float4 acc, float M, float L) {
                if (to_side) {
                    float* sd = side_base + static_cast<size_t>(h) * kORow;
                    *reinterpret_cast<float4*>(sd + d0) = acc;
                    if (lane == 0) {
                        sd[kDim] = M;
                        sd[kDim + 1] = L;
                    }
                } else {
                    const float inv = 1.f / L;
                    uint2 w2;
                    w2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                    w2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                    *reinterpret_cast<uint2*>(out_base + static_cast<size_t>(h) * kDim) = w2;
                }
            };
            // Four heads at a time: every shared-memory read of the four
            // heads' warp states is issued before any of them is used.
#pragma unroll
            for (int hb = 0; hb < kMaxG; hb += 4) {
                if (hb < G) {
                    float mk[kConsumerWarps][4], lk[kConsumerWarps][4];
                    float4 ok[kConsumerWarps][4];
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh) {
                            const int h = hb + hh;
                            if (((owners >> w) & 1u) && h < G) {  // warps without blocks of the piece wrote nothing
                                mk[w][hh] = mm[w * kMaxG + h];
                                lk[w][hh] = ml[w * kMaxG + h];
                                ok[w][hh] = *reinterpret_cast<const float4*>(mo + (w * kMaxG + h) * kORow + d0);
                            } else {
                                mk[w][hh] = NEG_INF;
                                lk[w][hh] = 0.f;
                                ok[w][hh] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                    }
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        const int h = hb + hh;
                        if (h < G) {
                            float M = NEG_INF;
#pragma unroll
                            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mk[w][hh]);
                            float L = 0.f;
                            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int w = 0; w < kConsumerWarps; ++w) {
                                if (!((owners >> w) & 1u)) continue;
                                const float f = ex2(mk[w][hh] - M);
                                L += f * lk[w][hh];
                                acc.x += f * ok[w][hh].x;
                                acc.y += f * ok[w][hh].y;
                                acc.z += f * ok[w][hh].z;
                                acc.w += f * ok[w][hh].w;
                            }
                            if (pieces == 1) {
                                emit(h, acc, M, L);
                            } else {
                                *reinterpret_cast<float4*>(part + h * kORow + d0) = acc;
                                if (lane == 0) {
                                    part[h * kORow + kDim] = M;
                                    part[h * kORow + kDim + 1] = L;
                                }
                            }
                        }
                    }
                }
            }
            mbar_arrive(mempty_bar(ms));  // the consumers may reuse this slot
            if (pieces > 1) {
                // Publish this piece's partial (every lane's stores, ordered
                // before lane 0's release by the warp barrier) and count it;
                // the last piece to arrive acquires the others' and merges.
                // A pair of more than kMergeGroup pieces merges in two levels:
                // the last arrival of each group of kMergeGroup consecutive
                // pieces merges the group into the slot of its first piece,
                // and the last group to finish merges the groups, so that no
                // single warp walks dozens of partials at the kernel's end.
                // group level: base = the group's first CTA, count = its
                // pieces; pair level: base = i0, stride kMergeGroup (two
                // levels) or 1, count = the groups or the pieces
                bool group_level = pieces > kMergeGroup;
                int base = i0, count = pieces;
                if (group_level) {
                    base = i0 + (static_cast<int>(blockIdx.x) - i0) / kMergeGroup * kMergeGroup;
                    count = min(kMergeGroup, i1 - base + 1);
                    if (count == 1) {  // a lone last piece is its group's result already
                        base = i0;
                        count = (pieces + kMergeGroup - 1) / kMergeGroup;
                        group_level = false;
                    }
                }
                while (true) {
                    const int stride = pieces > kMergeGroup && !group_level ? kMergeGroup : 1;
                    int* ctr = group_level ? p.group_counters + 2 * base + (base == i1 ? 0 : 1)
                                           : p.counters + i0;
                    __syncwarp();
                    int old = 0;
                    if (lane == 0) old = atom_add_acq_rel_gpu(ctr, 1);
                    old = __shfl_sync(0xffffffffu, old, 0);
                    __syncwarp();
                    if (old != count - 1) break;  // not the last arrival: done
                    // An online log-sum-exp pass over the count partials at
                    // CTAs base + n * stride, four heads at a time and four
                    // partials per batch: each batch's loads are all issued
                    // before any of them is used, so P partials cost about
                    // P / 4 round trips to L2 per four heads, not P. A group's
                    // result replaces its first piece's partial; the pair's
                    // final result is emitted.
                    float* gp = p.partials + (static_cast<size_t>(base) * 2 + (base == i1 ? 0 : 1)) * kPartialFloats;
#pragma unroll
                    for (int hb = 0; hb < kMaxG; hb += 4) {
                        if (hb < G) {
                            float Mr[4], Lr[4];
                            float4 Ar[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                Mr[h] = NEG_INF;
                                Lr[h] = 0.f;
                                Ar[h] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                            for (int n = 0; n < count; n += 4) {
                                float mk[4][4], lk[4][4];
                                float4 ok[4][4];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const int cta = base + (n + k) * stride;
                                    const float* pi = p.partials +
                                        (static_cast<size_t>(cta) * 2 + (cta == i1 ? 0 : 1)) * kPartialFloats;
#pragma unroll
                                    for (int h = 0; h < 4; ++h) {
                                        if (n + k < count && hb + h < G) {
                                            mk[k][h] = __ldcg(pi + (hb + h) * kORow + kDim);
                                            lk[k][h] = __ldcg(pi + (hb + h) * kORow + kDim + 1);
                                            ok[k][h] = __ldcg(reinterpret_cast<const float4*>(pi + (hb + h) * kORow + d0));
                                        } else {
                                            mk[k][h] = NEG_INF;
                                            lk[k][h] = 0.f;
                                            ok[k][h] = make_float4(0.f, 0.f, 0.f, 0.f);
                                        }
                                    }
                                }
#pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    float mn = Mr[h];
#pragma unroll
                                    for (int k = 0; k < 4; ++k) mn = fmaxf(mn, mk[k][h]);
                                    const float a = ex2(Mr[h] - mn);
                                    float L = Lr[h] * a;
                                    float4 A = make_float4(Ar[h].x * a, Ar[h].y * a, Ar[h].z * a, Ar[h].w * a);
#pragma unroll
                                    for (int k = 0; k < 4; ++k) {
                                        const float b = ex2(mk[k][h] - mn);  // 0 for absent pieces
                                        L += b * lk[k][h];
                                        A.x += b * ok[k][h].x;
                                        A.y += b * ok[k][h].y;
                                        A.z += b * ok[k][h].z;
                                        A.w += b * ok[k][h].w;
                                    }
                                    Mr[h] = mn;
                                    Lr[h] = L;
                                    Ar[h] = A;
                                }
                            }
                            __syncwarp();  // every lane's loads of gp's rows precede lane 0's stores
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const int H = hb + h;
                                if (H < G) {
                                    if (!group_level) {
                                        emit(H, Ar[h], Mr[h], Lr[h]);
                                    } else {
                                        *reinterpret_cast<float4*>(gp + H * kORow + d0) = Ar[h];
                                        if (lane == 0) {
                                            gp[H * kORow + kDim] = Mr[h];
                                            gp[H * kORow + kDim + 1] = Lr[h];
                                        }
                                    }
                                }
                            }
                        }
                    }
                    if (lane == 0) *ctr = 0;  // ready for the next launch
                    if (!group_level) break;
                    // then count the group at the pair level
                    base = i0;
                    count = (pieces + kMergeGroup - 1) / kMergeGroup;
                    group_level = false;
                }
            }
            ++piece;
        }
        return;
    }

    // ========================= consumer warps =========================
    if constexpr (kFmaG > 0) {
        static_assert(kBT == kTok && !kSkip, "the CUDA-core variant serves the plain 16-token kernel");
        fma_consumer_warp<kSlots, kFmaG>(p, smem, scan, tail, range_lo, range_hi, first, warp, lane, abort_flag, bar0);
        return;
    }
    const int r = lane >> 2;  // mma group id: token row / head column owner
    const int c = lane & 3;   // thread in group
    const uint32_t stage_base = smem_u32(smem + kOffStages);
    // ldmatrix address pieces (row of the 16 x 16 tile each lane points at)
    using TL = TileLayout<kBT>;
    const uint32_t k_row_off = static_cast<uint32_t>((lane & 15) >> 3) * TL::kRows8 + static_cast<uint32_t>(lane & 7) * 128u;
    const int k_sw = lane & 7;
    const int k_hi = lane >> 4;
    const int v_mat = lane >> 3;
    const uint32_t v_row_off = static_cast<uint32_t>(v_mat >> 1) * TL::kRows8 + static_cast<uint32_t>(lane & 7) * 128u;
    const int v_sw = lane & 7;
    const float NEG_INF = -INFINITY;

    PieceWalk walk(scan, B, Hkv, range_lo, range_hi, first);
    Piece pc;
    int gidx0 = 0;
    int qslot = 0, piece = 0;
    uint32_t qphase = 0;
    while (walk.next(pc)) {
        const int s = pc.s, blk0 = pc.blk, nb = pc.nb, len = pc.len;
        const int last_valid = tail[s];  // tokens in the run's last tile
        // A piece shorter than the consumer warp count has blocks for some
        // warps only; the others skip it but for the merge-slot handshake.
        const int first = (warp - static_cast<int>(gidx0 % kConsumerWarps)) & (kConsumerWarps - 1);
        const bool mine = first < len;

        // ---- query fragments (B operand of S^T = K Q^T) ----
        // Full pieces: from the shared-memory ring the producer fills. Short
        // pieces: each warp that has a block reads its fragments straight
        // from global memory (L2-warm), so that no warp waits on a query copy
        // for a piece it takes no part in.
        uint32_t qb[16];
        if (len >= kConsumerWarps) {
            // A slot (or stage, below) is released only once this warp saw
            // its copy land: after an abort a wait gives up early, and
            // releasing then would let the producer copy into a slot whose
            // previous copy is still in flight.
            const bool landed = mbar_wait(qfull_bar(qslot), qphase, abort_flag, p.err);
            const uint8_t* qs = smem + kOffQ + qslot * kQBytes + r * (kDim * 2) + c * 4;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qb[2 * ks] = r < G ? *reinterpret_cast<const uint32_t*>(qs + ks * 32) : 0u;
                qb[2 * ks + 1] = r < G ? *reinterpret_cast<const uint32_t*>(qs + ks * 32 + 16) : 0u;
            }
            // The slot may be refilled as soon as it is released: every lane
            // first holds its fragments (the release below waits on a value
            // computed from all of them, so on every load having returned),
            // else the producer's next bulk copy can land under loads still
            // in flight.
            uint32_t held = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) held ^= qb[i];
            const uint32_t z = __reduce_or_sync(0xffffffffu, zero_after(held));  // 0, once all lanes hold theirs
            if (lane == 0 && landed) mbar_arrive(qempty_bar(qslot) + z);
            if (++qslot == kQSlots) { qslot = 0; qphase ^= 1u; }
        } else if (mine) {
            const uint32_t* qg = reinterpret_cast<const uint32_t*>(
                p.q + (static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(pc.g) * G + r) * kDim) + c;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qb[2 * ks] = r < G ? __ldg(qg + ks * 8) : 0u;
                qb[2 * ks + 1] = r < G ? __ldg(qg + ks * 8 + 4) : 0u;
            }
        }

        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
        float o[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

        // Block gi of this CTA's stream goes to warp gi % 4, so every stage
        // (gi % 8) is always consumed by the same warp, which waits on each of
        // its phases in turn. Handing blocks out per piece instead would let a
        // warp wait on a stage whose previous fill, owned by another warp, is
        // still in flight (TMA fills complete out of order); a parity wait
        // would then see the previous phase's parity and pass too early.
        for (int jb = first; jb < len; jb += kConsumerWarps) {
            const int gi = gidx0 + jb;
            const int st = static_cast<int>(gi % kStages);
            const bool landed = mbar_wait(full_bar(st), static_cast<uint32_t>((gi / kStages) & 1), abort_flag, p.err);
            const int valid = (blk0 + jb == nb - 1) ? last_valid : kTok;
            const uint32_t sk = stage_base + st * kStageBytes;
            const uint32_t sv = sk + kBlockBytes;

            // S^T = K Q^T : two accumulators halve the dependent mma chain.
            float sa[4] = {0.f, 0.f, 0.f, 0.f};
            float sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int chunk = ((ks & 3) << 1) | k_hi;
                uint32_t a[4];
                ldmatrix_x4(a, sk + (ks >> 2) * TL::kHalf + k_row_off + ((chunk ^ k_sw) << 4));
                if (ks & 1) mma_bf16_16816(sb, a, qb[2 * ks], qb[2 * ks + 1]);
                else mma_bf16_16816(sa, a, qb[2 * ks], qb[2 * ks + 1]);
            }
            float x0 = (sa[0] + sb[0]) * p.scale_log2;  // token r,   head 2c
            float x1 = (sa[1] + sb[1]) * p.scale_log2;  // token r,   head 2c+1
            float x2 = (sa[2] + sb[2]) * p.scale_log2;  // token r+8, head 2c
            float x3 = (sa[3] + sb[3]) * p.scale_log2;  // token r+8, head 2c+1
            uint32_t vmask01 = 0xffffffffu, vmask23 = 0xffffffffu;
            if (valid < kTok) {
                if (r >= valid) x0 = x1 = NEG_INF;
                if (r + 8 >= valid) x2 = x3 = NEG_INF;
                vmask01 = (2 * c < valid ? 0x0000ffffu : 0u) | (2 * c + 1 < valid ? 0xffff0000u : 0u);
                vmask23 = (2 * c + 8 < valid ? 0x0000ffffu : 0u) | (2 * c + 9 < valid ? 0xffff0000u : 0u);
            }
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
            const uint32_t p01 = pack_bf16x2(ex2(x0 - mn0), ex2(x1 - mn1));  // token r
            const uint32_t p23 = pack_bf16x2(ex2(x2 - mn0), ex2(x3 - mn1));  // token r+8
            l0 = l0 * al0 + bf16_lo(p01) + bf16_lo(p23);
            l1 = l1 * al1 + bf16_hi(p01) + bf16_hi(p23);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                o[j][0] *= al0;
                o[j][1] *= al1;
                o[j][2] *= al0;
                o[j][3] *= al1;
            }
            const uint32_t pb0 = movmatrix_trans(p01);  // P^T rows: tokens 2c, 2c+1; column: head r
            const uint32_t pb1 = movmatrix_trans(p23);  // tokens 2c+8, 2c+9

            // O^T += V^T P^T over the 8 16-dim tiles of the head.
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int chunk = ((j & 3) << 1) | (v_mat & 1);
                uint32_t a[4];
                ldmatrix_x4_trans(a, sv + (j >> 2) * TL::kHalf + v_row_off + ((chunk ^ v_sw) << 4));
                a[0] &= vmask01;
                a[1] &= vmask01;
                a[2] &= vmask23;
                a[3] &= vmask23;
                mma_bf16_16816(o[j], a, pb0, pb1);
            }
            fence_proxy_async_shared();  // this lane's reads of the stage, before the copy that will replace it
            __syncwarp();
            if (lane == 0 && landed) mbar_arrive(empty_bar(st));
        }
        gidx0 += len;

        // ---- a pair of one tile: its owner warp finishes it alone ----
        // Its state is the whole result (the merge warp's combine of a single
        // warp's state gives the same numbers), so it skips the merge-slot
        // hand-over, which for batches of short sequences is the chain every
        // piece waits on; the merge warp skips such pieces too.
        if (nb == 1) {
            if (mine) {
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
                }
                const size_t row0 = static_cast<size_t>(s) * p.num_q_heads + static_cast<size_t>(pc.g) * G + 2 * c;
                if (kSkip && skipped(s) > 0) {  // the cascade's unnormalised fp32 result
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (2 * c + h < G) {
                            float* sd = p.side + (row0 + h) * kORow;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                sd[16 * j + r] = o[j][h];
                                sd[16 * j + r + 8] = o[j][h + 2];
                            }
                            if (r == 0) {
                                sd[kDim] = h ? m1 : m0;
                                sd[kDim + 1] = h ? l1 : l0;
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (2 * c + h < G) {
                            const float inv = 1.f / (h ? l1 : l0);
                            __nv_bfloat16* dst = p.out + (row0 + h) * kDim;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                dst[16 * j + r] = __float2bfloat16_rn(o[j][h] * inv);
                                dst[16 * j + r + 8] = __float2bfloat16_rn(o[j][h + 2] * inv);
                            }
                        }
                    }
                }
            }
            continue;
        }

        // ---- hand this warp's state for the piece to the merge warp ----
        // (a warp without blocks in the piece writes nothing: the merge warp
        // knows from the piece's geometry which warps contributed)
        const int ms = piece % kSlots;
        if (mine) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
        }
        mbar_wait(mempty_bar(ms), static_cast<uint32_t>(((piece / kSlots) & 1) ^ 1), abort_flag, p.err);
        if (mine) {
            float* o0 = sm_o + ms * kMergeOFloats + (warp * kMaxG + 2 * c) * kORow + r;
            float* o1 = o0 + kORow;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                o0[16 * j] = o[j][0];
                o1[16 * j] = o[j][1];
                o0[16 * j + 8] = o[j][2];
                o1[16 * j + 8] = o[j][3];
            }
            if (r == 0) {
                sm_m[ms * kMergeMLFloats + warp * kMaxG + 2 * c] = m0;
                sm_m[ms * kMergeMLFloats + warp * kMaxG + 2 * c + 1] = m1;
                sm_l[ms * kMergeMLFloats + warp * kMaxG + 2 * c] = l0;
                sm_l[ms * kMergeMLFloats + warp * kMaxG + 2 * c + 1] = l1;
            }
        }
        mbar_arrive(mfull_bar(ms));
        ++piece;
    }
}

}  // namespace attn
}  // namespace pkv
