// decode.cu -- split-KV flash-decode over a linear, paged or ring KV cache.
//
// What is computed (vibevoice.c, "The kernels that matter" and "Attention
// backends"; talker_multiframe, NarrowStep fields; Voxtral Realtime notes,
// "Encoder KV cache"): for every request b, query row r and query head h,
// softmax(scale * q . k_t) over the valid key positions t, applied to v_t.
// The keys of each (request, KV head) are cut into pieces; each piece keeps
// an online softmax state (running max m, sum l, output O) and the pieces'
// states are merged in a fixed order.  Both are exact reformulations.
//
// GB300 mapping:
//   * Work unit = (request, KV head, row block): the query rows of the GQA
//     group (q_rows x group: up to 8 as the N dimension of one mma.sync tile,
//     up to 32 as its M dimension; a larger group is cut into 16-row units)
//     share every K/V tile, so every cache position is read from HBM once per
//     unit.  Groups of 64 or more rows over a linear slot-major bf16 cache
//     (prefill chunks) go to the tcgen05 chunk kernel (chunk.cu) instead.
//   * The kernel is persistent: two CTAs per SM (one for 32-row units).
//     Every CTA computes, from the
//     device-side seq_lens and positions, how many 16-key chunks each unit
//     needs, and takes an equal contiguous share of all units' chunks laid end
//     to end.  The share is balanced whatever the lengths are (ragged batches
//     included), and each CTA streams its share through one deep TMA ring,
//     paying the pipeline ramp once.  A CTA's share covers pieces ("segments")
//     of one or more units; a unit wholly inside one CTA is written straight
//     to the output; the others leave fp32 partial states in the workspace
//     and are merged by the CTAs that store the last ones (atomic counters
//     tell them): parts in CTA order, eight at a time, then those groups'
//     states in order.  Launches whose units may span very many CTAs, or
//     whose few units may each span more than eight, leave those units to a
//     small merge kernel instead.
//   * A producer warp streams tiles of 16-key chunks: 64 keys for bf16, 128
//     for E4M3 (whose rows are half as wide).  A tile whose slots are
//     consecutive (linear cache; a ring away from its wrap point) is one TMA
//     box per tensor; otherwise a chunk whose 16 slots are consecutive (a page
//     of >= 16 slots) is a 16-row box; any other chunk is gathered row by row
//     with 16-byte cp.async.  Boxes bring whole head rows (128-byte blocks,
//     the "halves" of a bf16 row of 128) and land 128-byte-swizzled.  Page ids
//     are fetched 32 at a time, one per lane, ahead of the tiles that use them.
//   * Four consumer warps each own one chunk (two for E4M3) of every tile:
//     S = Q K^T and O += P V on the tensor cores (mma.sync m16n8k16, bf16 in
//     -- f16 for E4M3 caches, converted in registers -- fp32 accumulate), the
//     mask and online softmax in fp32 registers with quad shuffles, exp2 with
//     log2(e) folded into the scale.  For bf16 caches P enters P V as two bf16
//     halves, hi + lo (vibevoice.c, "Attention backends": one rounding of P is
//     too coarse), so P keeps ~16 bits; for E4M3 one f16 rounding (11 bits).
//     At the end of a segment the four warps merge through shared memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace gqa {
namespace dec {

constexpr int kChunk = 16;                   // key positions per chunk
constexpr int kWarps = 4;                    // consumer warps = chunks per tile
constexpr int kThreads = (kWarps + 1) * 32;  // + one producer warp
constexpr int kProducerWarp = kWarps;
constexpr int kMaxTableEntries = 256;        // (request, row block) pairs per launch
constexpr int kMinChunksPerCta = 8;          // smallest share of key chunks per CTA
// A CTA that moves from one unit to the next pays for a second segment
// (merge of its warps, partial store, new q): in the share arithmetic every
// unit is followed by this many chunks of nothing, so such a CTA gets that
// much less real work.
constexpr int kUnitGapChunks = 12;
constexpr int kGroupParts = 8;               // partial states merged by one CTA at a time
// Lazy rescale of the running output: a row's reference maximum moves only
// when a chunk's scores pass it by more than this (log2 units), so P stays
// <= 2^8 (exact range of f16 and of the bf16 hi + lo split) and the warp
// skips the rescale of O whenever none of its rows moved.
constexpr float kRescaleLog2 = 8.0f;
// merge kernel CTA: four warps.  Beside two split CTAs (165 registers, three
// warps on two of the SM's four sub-partitions) one no longer fits, so merge
// CTAs take SMs as split CTAs leave them.
constexpr int kMergeWarps = 4;
// A launch whose units may span more CTAs than this (by the host's bound)
// leaves units of more than kGroupParts parts to the merge kernel: there one
// CTA per query row merges all parts with every load in flight, which beats
// two levels of counters and L2 round trips inside the split kernel.
constexpr int kMergeKernelParts = 128;
// bf16 tiles of a share fetched into L2 before the PDL wait (FP8 tiles hold
// twice the keys: half as many, the same first 512 key positions)
constexpr int kPrefetchTiles = 8;

struct Params {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_cache;
    const __nv_bfloat16 *v_cache;
    int64_t num_slots;
    int kind;
    int slots_per_seq;
    const int32_t *block_table;
    int block_size;
    int max_blocks;
    const int32_t *seq_lens;
    const int32_t *positions;
    int batch;   // requests in this launch
    int b_base;  // index of this launch's first request (linear / ring slot arithmetic)
    int q_rows, n_q_heads, n_kv_heads, group, rows;
    int window, max_seq_len;
    float scale_log2;
    int row_blocks;
    int rb_rows;  // query rows per unit (8, 16 or 32)
    int grid;     // CTAs of the split kernel
    __nv_bfloat16 *out;
    float *ws_o;
    float *ws_lse;
    int32_t *ws_count;   // per unit: merged groups so far (zero between calls)
    int32_t *ws_gcount;  // per partial slot that starts a group: parts stored so far
    KvPlace place;       // where a head's row of a slot lives (slot-major or head-major)
    bool merge_kernel;   // units of more than kGroupParts parts go to the merge kernel
    // fused append (nullptr: none): the step's rows, bf16 [batch * q_rows][n_kv_heads][HD],
    // row b * q_rows + r being the key at position seq_len_b - q_rows + r, and their slots
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    const int64_t *slot_mapping;
    const float *rope_inv_freq;  // [HD / 2] (nullptr: no rotary embedding)
    const float *k_ref;          // FP8 fused append: the cache's key reference [Hkv][HD], or nullptr
    // seq_lens, positions and block_table may be read before the previous
    // kernel completes (ATTN_DECODE_TABLES_EARLY)
    bool tables_early;
    // ... and the cache too (ATTN_DECODE_CACHE_EARLY): the producer issues the
    // first tiles of its share that hold none of the step's new rows before
    // it waits for the previous kernel
    bool cache_early;
    int32_t *err;
};

// MT = 0: up to 8 query rows per unit; keys are the M dimension of the
//         mma (S^T = K Q^T, O^T = V^T P^T), rows the N dimension of 8.
// MT = 1, 2: 16 or 32 rows per unit; rows are the M dimension.
// FP8: the cache holds 1-byte E4M3 elements (head_dim 128: one 128-byte block
// per head row) instead of bf16.
template <int HD, int MT, bool FP8 = false>
struct Geo {
    static constexpr int RB = MT == 0 ? 8 : 16 * MT;        // rows per unit
    static constexpr int kCtasPerSm = MT == 2 ? 1 : 2;
    static constexpr int kElem = FP8 ? 1 : 2;               // bytes per cache element
    static constexpr int kHalves = HD * kElem / 128;        // 128-byte column blocks
    static constexpr int kChunkBytes = kHalves * kChunk * 128;
    // chunks per tile: E4M3 rows are half as wide, so an FP8 tile holds 128
    // keys (each consumer warp takes two chunks of it) and a producer step
    // moves as many bytes as a bf16 one
    static constexpr int kCPT = FP8 ? 2 * kWarps : kWarps;
    static constexpr int kSubs = kCPT / kWarps;   // chunks of a tile per consumer warp
    static constexpr int kTileRows = kCPT * kChunk;
    static constexpr int kTileBytes = kCPT * kChunkBytes;  // K (or V) of one tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    // At the end of a segment each warp parks its O rows (RB x HD fp32) in
    // its own rows of the stage that held the segment's last tile (K and V,
    // 2 * kHalves pieces of 16 x 128 B, which it has finished reading); only
    // 32-row units need a dedicated area.  Row maxima and sums always have one.
    static constexpr bool kParkInStage = RB * HD * 4 <= 2 * kSubs * kHalves * kChunk * 128;
    // + per row and warp: max, sum, combined weight; per row: log-sum-exp
    static constexpr int kMergeBytes = (kParkInStage ? 0 : kWarps * RB * HD * 4) + (3 * kWarps + 1) * RB * 4;
    static constexpr int kTableBytes = (4 * kMaxTableEntries + 1) * 4;
    // q rows and row positions of a segment, staged by the producer, two
    // segments deep; rows padded by 16 bytes so the 8 rows of a fragment load
    // fall in different banks
    static constexpr int kQStride = HD * 2 + 16;
    static constexpr int kQBytes = 2 * RB * kQStride + 2 * RB * 4 + HD / 2 * 4;  // + rope table
    // as many stages as the shared memory of kCtasPerSm CTAs allows (max 8)
    static constexpr int kBudget = (kCtasPerSm == 2 ? 115712 : 232448) - 1024 - kMergeBytes -
                                   kTableBytes - kQBytes - 1024;
    static constexpr int kStages = kBudget / kStageBytes > 8 ? 8 : kBudget / kStageBytes;
    static constexpr int kOffMerge = kStages * kStageBytes;
    static constexpr int kOffBars = kOffMerge + kMergeBytes;
    // full[kStages], empty[kStages], q_full[2], q_empty[2]
    static constexpr int kOffInfo = kOffBars + (2 * kStages + 4) * 8;
    // info: t0[kStages][kCPT], mask[kStages][kCPT], whole[kStages], last[4]
    static constexpr int kOffTable = kOffInfo + ((2 * kStages * kCPT + kStages + 4) * 4 + 15) / 16 * 16;
    // tables: cnt[E], clo[E], seqlen[B], Pb[B + 1] with E, B <= kMaxTableEntries
    static constexpr int kOffQ = (kOffTable + kTableBytes + 15) / 16 * 16;
    static constexpr size_t kSmem = 1024 + kOffQ + kQBytes;
    static_assert(kStages >= 3 || MT == 2, "three stages for up to 16 rows");
    static_assert(kStages >= 2, "at least a double-buffered ring");
    static_assert(!FP8 || HD == 128, "FP8 caches have 128-element heads");
};

constexpr int kTileRows = kWarps * kChunk;  // key positions of a bf16 tile (64)

// 4D tiled TMA load / L2 prefetch (head-major caches: {columns, rows, halves,
// block x head}).
__device__ __forceinline__ void tma_load_4d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                                 int z, int w, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int x, int y, int z,
                                                int w) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

// Four E4M3 codes (one 32-bit word, lowest byte first) -> two f16x2 words:
// lo from bytes 0, 1 and hi from bytes 2, 3 (exact).  The word is split into
// its 16-bit halves by register naming, so no shift is needed.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// Rotary embedding of one interleaved pair held as bf16x2 (low half = x[2i]):
// rotated by the float32 angle pos * inv_freq in float32, rounded to bf16.
__device__ __forceinline__ uint32_t rope_pair(uint32_t w, int pos, float inv_freq) {
    const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
    float sn, cs;
    sincosf((float)pos * inv_freq, &sn, &cs);
    return pack_bf16x2(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
}

// A stage holds the K and V of one tile (64 keys bf16, 128 keys E4M3), each in
// one of two 128-byte-swizzled layouts (an 8-row group always spans 1024
// aligned bytes):
//   whole tile (one TMA box of all rows): [half][tile rows][128 B]
//   chunked    (16-row boxes / rows)    : [chunk][half][16 rows][128 B]
// Chunk c's rows start at chunk_base() and its halves are half_stride() apart.
template <int HALVES>
__device__ __forceinline__ uint32_t chunk_base(bool whole, int c) {
    return whole ? (uint32_t)c * (kChunk * 128) : (uint32_t)c * (HALVES * kChunk * 128);
}
template <int TILE_ROWS>
__device__ __forceinline__ uint32_t half_stride(bool whole) {
    return whole ? (uint32_t)(TILE_ROWS * 128) : (uint32_t)(kChunk * 128);
}
// Offset of 16-byte piece c16 (0 .. row bytes / 16 - 1) of row `key` (0 .. 15)
// of a chunk.
__device__ __forceinline__ uint32_t piece_offset(uint32_t hstride, int key, int c16) {
    const int half = c16 >> 3, cc = c16 & 7;
    return half * hstride + key * 128 + ((cc ^ (key & 7)) << 4);
}

// Where a warp parks 16-byte unit u (0 .. HD/4-1) of output row `row` for the
// end-of-segment merge.  The FP8 paths hold whole 16-byte runs of a row per
// thread and permute the units inside each row so that their stores do not
// collide in shared-memory banks; the merge reads through the same map.
template <int MT, bool FP8>
__device__ __forceinline__ int park_unit(int row, int u) {
    if constexpr (!FP8) return u;
    else if constexpr (MT == 0) return u ^ ((row >> 1) & 3);
    else return u ^ ((2 * (u >> 3) + (row & 1)) & 7);
}

// Whether every key t0 .. t0 + 15 of a chunk is visible to query rows at
// positions pmin .. pmax: all present (mask16), inside the sequence and the
// ring, causal for the earliest row and inside the window of the latest.
__device__ __forceinline__ bool chunk_open(uint32_t mask16, int t0, int seq_len, int ring_lo,
                                           int window, int pmin, int pmax) {
    const int t1 = t0 + kChunk - 1;
    return mask16 == 0xFFFFu && t1 < seq_len && t1 <= pmin && t0 >= ring_lo &&
           (window <= 0 || pmax - t0 < window);
}

// Key chunk range of unit (request b, row block rb): chunk c covers positions
// 16c .. 16c+15.  Also returns the request's effective seq_len.
__device__ __forceinline__ void unit_range(const Params &p, int b, int rb, int &c_lo, int &c_hi,
                                           int &seq_len_out, bool report) {
    int seq_len = p.seq_lens[b];
    if (seq_len > p.max_seq_len || seq_len < 0 ||
        (p.kind == ATTN_CACHE_LINEAR && seq_len > p.slots_per_seq)) {
        if (report) report_error(p.err, ATTN_ERR_BOUNDS);
        seq_len = max(0, min(seq_len, p.max_seq_len));
        if (p.kind == ATTN_CACHE_LINEAR) seq_len = min(seq_len, p.slots_per_seq);
    }
    seq_len_out = seq_len;
    const int row0 = rb * p.rb_rows, row1 = min(p.rows, row0 + p.rb_rows);
    int pmin = INT32_MAX, pmax = -1;
    for (int r = row0 / p.group; r <= (row1 - 1) / p.group; ++r) {
        const int pos = p.positions[(int64_t)b * p.q_rows + r];
        pmin = min(pmin, pos);
        pmax = max(pmax, pos);
    }
    const int hi = min(seq_len, pmax + 1);
    int lo = 0;
    if (p.window > 0) lo = max(lo, pmin - p.window + 1);
    if (p.kind == ATTN_CACHE_RING) lo = max(lo, seq_len - p.slots_per_seq);
    if (pmin < 0 || hi <= lo) {
        c_lo = c_hi = 0;
        return;
    }
    c_lo = lo / kChunk;
    c_hi = (hi + kChunk - 1) / kChunk;
}

// Shared tables every CTA builds: per (request, row block) chunk count and
// first chunk, per request effective seq_len, and Pb[b] = chunks of all
// units of requests before b (units ordered (request, KV head, row block)).
struct Tables {
    int *cnt, *clo, *seqlen, *Pb;
};

// Builds the tables every CTA of a launch computes alike: each (request, row
// block)'s chunk count and first chunk, each request's effective seq_len, and
// the prefix Pb.  All nthreads threads of the block take part; ends with a
// block barrier.  report: this block reports out-of-range seq_lens.
__device__ __forceinline__ void build_tables(const Params &p, const Tables &tb, int nthreads,
                                             bool report) {
    const int B = p.batch, RBc = p.row_blocks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < B * RBc; i += nthreads) {
        const int b = i / RBc, rb = i - (i / RBc) * RBc;
        int clo, chi, sl;
        unit_range(p, b, rb, clo, chi, sl, report && rb == 0);
        tb.cnt[i] = chi - clo;
        tb.clo[i] = clo;
        if (rb == 0) tb.seqlen[b] = sl;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        if (lane == 0) tb.Pb[0] = 0;
        for (int base = 0; base < B; base += 32) {
            const int b = base + lane;
            int v = 0;
            if (b < B)
                for (int rb = 0; rb < RBc; ++rb) {
                    const int n = tb.cnt[b * RBc + rb];
                    v += n > 0 ? n + kUnitGapChunks : 0;
                }
            v *= p.n_kv_heads;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += n;
            }
            if (b < B) tb.Pb[b + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
}

// One contiguous piece of one unit's chunks handled by this CTA.
struct Segment {
    int b, kvh, rb;
    int c_begin, c_end;  // chunk range inside the unit's key range
    int unit;
    int first, last;     // the CTAs that hold the unit's pieces
    bool whole;          // the piece is the whole unit
    bool head;           // the piece starts the unit
};

// The segments of global range [g, g_end), in order.  The range is in the
// order of all units' chunks laid end to end, each unit followed by
// kUnitGapChunks chunks that hold nothing (skipped).
struct SegmentWalker {
    int g, g_end;
    int L;  // chunks (with gaps) per CTA
    __device__ bool next(const Params &p, const Tables &t, Segment &s) {
        const int B = p.batch, RBc = p.row_blocks;
        while (g < g_end) {
            // request: the largest b with Pb[b] <= g (requests with no chunks are skipped)
            int lo = 0, hi = B;  // invariant: Pb[lo] <= g < Pb[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (t.Pb[mid] <= g)
                    lo = mid;
                else
                    hi = mid;
            }
            const int b = lo;
            const int per_head = (t.Pb[b + 1] - t.Pb[b]) / p.n_kv_heads;
            int off = g - t.Pb[b];
            const int kvh = off / per_head;
            off -= kvh * per_head;
            int rb = 0;
            auto span = [&](int e) { return t.cnt[e] > 0 ? t.cnt[e] + kUnitGapChunks : 0; };
            while (off >= span(b * RBc + rb)) off -= span(b * RBc + rb++);
            const int n_u = t.cnt[b * RBc + rb];
            const int unit_start = g - off;
            if (off >= n_u) {  // in the unit's gap
                g = min(g_end, unit_start + n_u + kUnitGapChunks);
                continue;
            }
            const int seg_end = min(g_end, unit_start + n_u);
            s.b = b;
            s.kvh = kvh;
            s.rb = rb;
            s.c_begin = t.clo[b * RBc + rb] + off;
            s.c_end = s.c_begin + (seg_end - g);
            s.unit = (b * p.n_kv_heads + kvh) * RBc + rb;
            s.first = unit_start / L;
            s.last = (unit_start + n_u - 1) / L;
            s.whole = (off == 0 && seg_end == unit_start + n_u);
            s.head = off == 0;
            g = seg_end;
            return true;
        }
        return false;
    }
};

// Merge `parts` fp32 partial states of unit u's rows, stored at workspace
// slots s0, s0 + stride, ... (in that order, the order that fixes the
// result), either into the bf16 output (final) or, as one partial state, back
// into slot s0.  Partial states hold O / l and the base-2 log-sum-exp.  Run by
// the four consumer warps, each thread two output pieces (row, 4 columns) at
// a time; for each it reads the log-sum-exps and pieces of up to kGroupParts
// parts in one round (more parts go kGroupParts at a time, the running sums
// rescaled to the new maximum).  Slot s0's log-sum-exps, which every thread
// of a row reads, are overwritten only after the consumer barrier.  Ends with
// that barrier.
template <int HD, int RB>
__device__ __forceinline__ void merge_partials(const Params &p, const Segment &u, int64_t s0,
                                               int stride, int parts, bool final, int ctid) {
    constexpr int kItems = RB * (HD / 4) / (kWarps * 32);  // output pieces per thread
    constexpr int kPair = (kItems >= 2 && RB <= 8) ? 2 : 1;  // registers: pairs for 8-row units
    static_assert(kItems * kWarps * 32 == RB * (HD / 4) && kItems % kPair == 0, "whole items");
    const int row0 = u.rb * RB, row1 = min(p.rows, row0 + RB);
    float lse_out[kItems];
#pragma unroll
    for (int q0 = 0; q0 < kItems; q0 += kPair) {
        float M[kPair], Lsum[kPair];
        float4 acc[kPair];
#pragma unroll
        for (int q = 0; q < kPair; ++q) {
            M[q] = -INFINITY;
            Lsum[q] = 0.f;
            acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int c0 = 0; c0 < parts; c0 += kGroupParts) {
            float l[kPair][kGroupParts];
            float4 v[kPair][kGroupParts];
#pragma unroll
            for (int q = 0; q < kPair; ++q) {
                const int idx = ctid + (q0 + q) * (kWarps * 32);
                const int row = idx / (HD / 4), d = (idx % (HD / 4)) * 4;
                const bool live = row0 + row < row1;
#pragma unroll
                for (int k = 0; k < kGroupParts; ++k) {
                    const int c = c0 + k;
                    l[q][k] = -INFINITY;
                    v[q][k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (live && c < parts) {
                        const int64_t slot = s0 + (int64_t)c * stride;
                        l[q][k] = __ldcg(p.ws_lse + slot * RB + row);
                        v[q][k] = __ldcg(
                            reinterpret_cast<const float4 *>(p.ws_o + (slot * RB + row) * HD + d));
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kPair; ++q) {
                float Mn = M[q];
#pragma unroll
                for (int k = 0; k < kGroupParts; ++k) Mn = fmaxf(Mn, l[q][k]);
                if (Mn == -INFINITY) continue;  // no part so far holds a key
                if (M[q] != -INFINITY && Mn != M[q]) {
                    const float rs = fast_exp2(M[q] - Mn);
                    Lsum[q] *= rs;
                    acc[q].x *= rs;
                    acc[q].y *= rs;
                    acc[q].z *= rs;
                    acc[q].w *= rs;
                }
                M[q] = Mn;
#pragma unroll
                for (int k = 0; k < kGroupParts; ++k) {
                    const float f = fast_exp2(l[q][k] - Mn);  // -inf gives 0
                    Lsum[q] += f;
                    acc[q].x += f * v[q][k].x;
                    acc[q].y += f * v[q][k].y;
                    acc[q].z += f * v[q][k].z;
                    acc[q].w += f * v[q][k].w;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kPair; ++q) {
            const int idx = ctid + (q0 + q) * (kWarps * 32);
            const int row = idx / (HD / 4), d = (idx % (HD / 4)) * 4;
            const int i = row0 + row;
            lse_out[q0 + q] = Lsum[q] > 0.f ? M[q] + __log2f(Lsum[q]) : -INFINITY;
            if (i >= row1) continue;
            const float inv = Lsum[q] > 0.f ? 1.f / Lsum[q] : 0.f;
            if (final) {
                const int r = i / p.group, g = i - (i / p.group) * p.group;
                __nv_bfloat16 *dst =
                    p.out + (((int64_t)u.b * p.q_rows + r) * p.n_q_heads + u.kvh * p.group + g) * HD +
                    d;
                uint2 packed;
                packed.x = pack_bf16x2(acc[q].x * inv, acc[q].y * inv);
                packed.y = pack_bf16x2(acc[q].z * inv, acc[q].w * inv);
                *reinterpret_cast<uint2 *>(dst) = packed;
            } else {
                // this thread alone reads (row, d) of slot s0: the overwrite is safe
                *reinterpret_cast<float4 *>(p.ws_o + (s0 * RB + row) * HD + d) =
                    make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
            }
        }
    }
    if (!final) {
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");  // all reads of slot s0 done
#pragma unroll
        for (int q = 0; q < kItems; ++q) {
            const int idx = ctid + q * (kWarps * 32);
            const int row = idx / (HD / 4), d = (idx % (HD / 4)) * 4;
            if (d == 0 && row0 + row < row1) p.ws_lse[s0 * RB + row] = lse_out[q];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}

// ROPE: the fused append's rotary embedding (its code is compiled only into
// the kernels that need it).  FP8: an E4M3 cache (vibevoice.c, "KV cache"),
// read as stored: scores from f16 q and f16 keys (the E4M3 -> f16 conversion
// is exact), P V from f16 weights and values, fp32 accumulation.
template <int HD, int MT, bool ROPE, bool FP8>
__global__ void __launch_bounds__(kThreads, Geo<HD, MT, FP8>::kCtasPerSm)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_k64,
                        const __grid_constant__ CUtensorMap tm_v64, const Params p) {
    using G = Geo<HD, MT, FP8>;
    constexpr int RB = G::RB;
    constexpr int kStages = G::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    float *mo = reinterpret_cast<float *>(smem + G::kOffMerge);  // [kWarps][RB][HD] (if !kParkInStage)
    float *mm = mo + (G::kParkInStage ? 0 : kWarps * RB * HD);   // [kWarps][RB]
    float *ml = mm + kWarps * RB;                                // [kWarps][RB]
    float *wgt = ml + kWarps * RB;                               // [RB][kWarps]
    float *rlse = wgt + kWarps * RB;                             // [RB]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + G::kOffBars);
    uint64_t *empty = full + kStages;
    uint64_t *q_full = empty + kStages;  // [2]: a segment's q rows and positions landed
    uint64_t *q_empty = q_full + 2;      // [2]: the consumers have read them
    uint8_t *qbuf = smem + G::kOffQ;     // [2][RB][kQStride]
    int *posbuf = reinterpret_cast<int *>(qbuf + 2 * RB * G::kQStride);  // [2][RB]
    float *rope_if = reinterpret_cast<float *>(posbuf + 2 * RB);        // [HD / 2]
    constexpr int kCPT = G::kCPT;
    int *info_t0 = reinterpret_cast<int *>(smem + G::kOffInfo);  // [kStages][kCPT]
    uint32_t *info_mask = reinterpret_cast<uint32_t *>(info_t0 + kStages * kCPT);
    int *info_whole = reinterpret_cast<int *>(info_mask + kStages * kCPT);  // [kStages]
    int *s_last = info_whole + kStages;
    Tables tb;
    tb.cnt = reinterpret_cast<int *>(smem + G::kOffTable);
    tb.clo = tb.cnt + kMaxTableEntries;
    tb.seqlen = tb.clo + kMaxTableEntries;
    tb.Pb = tb.seqlen + kMaxTableEntries;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 32);       // one arrival per producer lane (+ TMA bytes)
            mbar_init(&empty[s], kWarps);  // one arrival per consumer warp
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&q_full[s], 32);
            mbar_init(&q_empty[s], kWarps);
        }
        fence_barrier_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        // the maps are launch parameters: fetch them while the previous kernel drains
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_k64);
        prefetch_tensormap(&tm_v64);
    }
    // Everything may come from the previous kernel (the cache, q, the new rows,
    // and unless the caller says otherwise seq_lens and positions), and it may
    // still read this call's out and workspace: wait for it before those.
    if (!p.tables_early) pdl_wait();

    // ---- tables: chunk counts of every (request, row block), then Pb
    const int B = p.batch, RBc = p.row_blocks;
    build_tables(p, tb, kThreads, blockIdx.x == 0);
    const int N = tb.Pb[B];
    // equal shares, but at least kMinChunksPerCta so small problems do not
    // spread a few keys over every SM
    const int L = max(kMinChunksPerCta, (N + p.grid - 1) / p.grid);
    const int g0 = min(N, (int)blockIdx.x * L), g1 = min(N, g0 + L);
    if (p.tables_early) {
        // The share is known before the previous kernel has finished: start
        // the DRAM reads of its first tiles into L2 now (whole 64-slot tiles
        // of linear and ring caches; pages would need block-table reads
        // first, which cost more than they hide), so the wait below overlaps
        // their latency.  A prefetch writes nothing; a line the previous
        // kernel rewrites is refetched.
        if (warp == kProducerWarp && lane == 0 && p.kind != ATTN_CACHE_PAGED) {
            constexpr int kTiles = kPrefetchTiles / G::kSubs;
            SegmentWalker walk{g0, g1, L};
            Segment sg;
            int issued = 0;
            while (issued < kTiles && walk.next(p, tb, sg)) {
                const int bg = p.b_base + sg.b;
                for (int c = sg.c_begin; c < sg.c_end && issued < kTiles;
                     c += kCPT, ++issued) {
                    const int z = sg.kvh * G::kHalves;
                    int j = c * kChunk;  // first position of the tile
                    if (p.kind == ATTN_CACHE_RING) {
                        j %= p.slots_per_seq;
                        if (j + G::kTileRows > p.slots_per_seq) continue;  // wraps: gathered later
                    }
                    if (p.place.rows != 0) {  // head-major: block = request
                        if (j + G::kTileRows > p.slots_per_seq) continue;
                        const int w = bg * p.n_kv_heads + sg.kvh;
                        tma_prefetch_4d(&tm_k64, 0, j, 0, w);
                        tma_prefetch_4d(&tm_v64, 0, j, 0, w);
                        continue;
                    }
                    const int y = (int)((int64_t)bg * p.slots_per_seq + j);
                    tma_prefetch_3d(&tm_k64, 0, y, z);
                    tma_prefetch_3d(&tm_v64, 0, y, z);
                }
            }
        }
        // with the cache final too, the producer waits inside its loop, after
        // issuing the first tiles that need nothing from the previous kernel
        if (!(p.cache_early && warp == kProducerWarp)) pdl_wait();
    }
    pdl_launch_dependents();
    if (blockIdx.x == 0 && warp != kProducerWarp) {
        // units with no valid key get zeros (no CTA visits them)
        for (int i = threadIdx.x; i < B * RBc; i += kWarps * 32) {
            if (tb.cnt[i] != 0) continue;
            const int b = i / RBc, rb = i - (i / RBc) * RBc;
            for (int row = rb * RB; row < min(p.rows, (rb + 1) * RB); ++row) {
                const int r = row / p.group, g = row - r * p.group;
                for (int kvh = 0; kvh < p.n_kv_heads; ++kvh) {
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        p.out + (((int64_t)b * p.q_rows + r) * p.n_q_heads + kvh * p.group + g) * HD);
                    for (int d = 0; d < HD / 8; ++d) dst[d] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
    }

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // Lane c (mod kCPT) describes chunk c of each tile; the warp agrees
        // on the tile's form with ballots, so a tile costs a few dozen
        // instructions on the issuing path.
        const bool paged = p.kind == ATTN_CACHE_PAGED;
        const bool paged_tma = paged && (p.block_size % kChunk == 0);
        const int64_t num_pages = paged ? p.num_slots / p.block_size : 0;
        const bool bhsd = p.place.rows != 0;  // head-major: boxes stay inside one block
        const int c = lane & (kCPT - 1);
        const bool fused = p.k_new != nullptr;
        const uint64_t kv_policy = l2_policy_evict_first();  // every K/V byte is read once
        SegmentWalker walk{g0, g1, L};
        Segment sg;
        int tile = 0;  // tiles issued by this CTA (stage / phase counter)
        int seg = 0;   // segments started (q staging buffer / phase counter)
        bool ok = true;
        bool waited = !p.cache_early;  // passed pdl_wait (the consumers have)
        while (ok && walk.next(p, tb, sg)) {
            const int bg = p.b_base + sg.b;  // request index in the whole cache
            const int seq_len = tb.seqlen[sg.b];
            const int new_lo = seq_len - p.q_rows;  // first of the step's new keys
            const int n_tiles = (sg.c_end - sg.c_begin + kCPT - 1) / kCPT;
            // Fast path: a linear or ring tile of four present chunks whose 64
            // positions sit in 64 consecutive slots and hold none of the
            // step's new rows is one box per tensor.  Every lane reaches the
            // same decision with a few integer operations: no ballots, so
            // the producer keeps ahead of the stream (its general path costs
            // ~1,000 cycles a tile).  Returns false for a tile it cannot take.
            auto whole_tile_fast = [&](int it, int st) -> bool {
                const int chunk0 = sg.c_begin + it * kCPT;
                if (paged || chunk0 + kCPT > sg.c_end) return false;
                constexpr int kRows = G::kTileRows;
                const int T0 = chunk0 * kChunk;
                const bool no_new = !fused || T0 + kRows <= new_lo || T0 >= seq_len;
                int j0 = T0;
                bool fits = !bhsd || T0 + kRows <= p.slots_per_seq;
                if (p.kind == ATTN_CACHE_RING) {
                    j0 = T0 % p.slots_per_seq;
                    fits = j0 + kRows <= p.slots_per_seq;
                }
                const int64_t s00 = (int64_t)bg * p.slots_per_seq + j0;
                if (!(no_new && fits && s00 + kRows <= p.num_slots)) return false;
                uint8_t *kst = stages + st * G::kStageBytes;
                uint8_t *vst = kst + G::kTileBytes;
                if (lane == 0) info_whole[st] = 1;
                if (lane < kCPT) {
                    info_t0[st * kCPT + lane] = T0 + lane * kChunk;
                    info_mask[st * kCPT + lane] = 0xFFFFu;
                }
                if (lane == 0) mbar_expect_tx(&full[st], 2 * G::kTileBytes);
                __syncwarp();
                if (lane < 2) {
                    if (bhsd)  // block = request, row = position in its window
                        tma_load_4d_hint(lane ? vst : kst, lane ? &tm_v64 : &tm_k64, 0, j0, 0,
                                         bg * p.n_kv_heads + sg.kvh, &full[st], kv_policy);
                    else
                        tma_load_3d_hint(lane ? vst : kst, lane ? &tm_v64 : &tm_k64, 0, (int)s00,
                                         sg.kvh * G::kHalves, &full[st], kv_policy);
                }
                __syncwarp();
                mbar_arrive(&full[st]);
                return true;
            };
            int it0 = 0;
            if (!waited) {
                // the first tiles of the share, into fresh stages, before the
                // previous kernel completes (the cache is final: the step's new
                // rows, which it may still be writing, are never among them)
                while (it0 < n_tiles && tile < kStages && whole_tile_fast(it0, tile)) {
                    ++it0;
                    ++tile;
                }
                pdl_wait();
                waited = true;
            }
            {
                // stage the segment's q rows and row positions for the consumers
                const int qi = seg & 1;
                if (seg >= 2 && !mbar_wait(&q_empty[qi], ((seg >> 1) - 1) & 1, p.err)) {
                    ok = false;
                    break;
                }
                const int qrow0 = sg.rb * RB, nrows = min(p.rows, qrow0 + RB) - qrow0;
                constexpr int kPieces = HD / 8;  // 16-byte pieces of a q row
                uint8_t *qdst = qbuf + qi * RB * G::kQStride;
                for (int pc = lane; pc < nrows * kPieces; pc += 32) {
                    const int rr = pc / kPieces, c16 = pc - rr * kPieces;
                    const int i = qrow0 + rr, r = i / p.group, g = i - r * p.group;
                    cp_async_16(qdst + rr * G::kQStride + c16 * 16,
                                p.q + (((int64_t)sg.b * p.q_rows + r) * p.n_q_heads +
                                       sg.kvh * p.group + g) * HD + c16 * 8);
                }
                for (int rr = lane; rr < nrows; rr += 32)
                    cp_async_4(posbuf + qi * RB + rr,
                               p.positions + (int64_t)sg.b * p.q_rows + (qrow0 + rr) / p.group);
                cp_async_arrive_noinc(&q_full[qi]);
                ++seg;
            }
            const int32_t *bt = paged ? p.block_table + (int64_t)sg.b * p.max_blocks : nullptr;
            // raw table entry at page index pi (range-checked when used)
            auto table_at = [&](int pi) -> int { return pi < p.max_blocks ? bt[pi] : -1; };
            auto slot_of = [&](int t) -> int64_t {  // slot of position t, or -1
                int64_t s;
                if (p.kind == ATTN_CACHE_LINEAR) {
                    s = (int64_t)bg * p.slots_per_seq + t;
                } else if (paged) {
                    const int v = table_at(t / p.block_size);
                    if (v < 0 || v >= num_pages) return -1;
                    s = (int64_t)v * p.block_size + t % p.block_size;
                } else {
                    s = (int64_t)bg * p.slots_per_seq + t % p.slots_per_seq;
                }
                return (s >= 0 && s < p.num_slots) ? s : -1;
            };
            // page ids of two consecutive 32-page windows, one per lane; the
            // second is fetched a window ahead of its use
            int win = -1, pg_cur = -1, pg_next = -1;
            for (int it = it0; it < n_tiles && ok; ++it, ++tile) {
                const int st = tile % kStages;
                if (tile >= kStages) ok = mbar_wait(&empty[st], ((tile / kStages) - 1) & 1, p.err);
                if (!ok) break;
                uint8_t *kst = stages + st * G::kStageBytes;
                uint8_t *vst = kst + G::kTileBytes;
                const int chunk0 = sg.c_begin + it * kCPT;
                if (whole_tile_fast(it, st)) continue;
                const int chunk = chunk0 + c;
                const int t0 = chunk * kChunk;
                // slot0 >= 0: first of 16 consecutive slots (TMA box); -1: a
                // contiguous chunk whose page is out of range (box aimed
                // outside the tensor, zero-filled, keys masked); -2: gathered
                // row by row; -3: absent
                int64_t slot0 = -3;
                if (paged_tma) {
                    const int pi0 = chunk0 * kChunk / p.block_size;
                    if (win < 0 || pi0 >= win + 64) {
                        win = pi0;
                        pg_cur = table_at(win + lane);
                        pg_next = table_at(win + 32 + lane);
                    } else if (pi0 >= win + 32) {
                        win += 32;
                        pg_cur = pg_next;
                        pg_next = table_at(win + 32 + lane);
                    }
                    const int rel = t0 / p.block_size - win;  // < 64 for a present chunk
                    const int va = __shfl_sync(0xffffffffu, pg_cur, rel & 31);
                    const int vb = __shfl_sync(0xffffffffu, pg_next, rel & 31);
                    const int v = rel < 32 ? va : vb;
                    if (chunk < sg.c_end)
                        slot0 = (v < 0 || v >= num_pages)
                                    ? -1
                                    : (int64_t)v * p.block_size + t0 % p.block_size;
                    // Fast path: pages smaller than a tile, every chunk of the
                    // tile present, on a page in range and without the step's
                    // new rows: one 16-row box per chunk and tensor, with no
                    // ballots (head-major coordinates straight from the page id)
                    const bool plain = chunk < sg.c_end && v >= 0 && v < num_pages &&
                                       !(fused && t0 + kChunk > new_lo && t0 < seq_len);
                    if (p.block_size < G::kTileRows && __all_sync(0xffffffffu, plain)) {
                        if (lane == 0) info_whole[st] = 0;
                        if (lane < kCPT) {
                            info_t0[st * kCPT + lane] = t0;
                            info_mask[st * kCPT + lane] = 0xFFFFu;
                        }
                        if (lane == 0) mbar_expect_tx(&full[st], kCPT * 2 * G::kChunkBytes);
                        __syncwarp();
                        if (lane < kCPT) {
                            const uint32_t off = chunk_base<G::kHalves>(false, lane);
                            if (bhsd) {
                                const int y = t0 % p.block_size, w = v * p.n_kv_heads + sg.kvh;
                                tma_load_4d_hint(kst + off, &tm_k, 0, y, 0, w, &full[st], kv_policy);
                                tma_load_4d_hint(vst + off, &tm_v, 0, y, 0, w, &full[st], kv_policy);
                            } else {
                                tma_load_3d_hint(kst + off, &tm_k, 0, (int)slot0, sg.kvh * G::kHalves,
                                                 &full[st], kv_policy);
                                tma_load_3d_hint(vst + off, &tm_v, 0, (int)slot0, sg.kvh * G::kHalves,
                                                 &full[st], kv_policy);
                            }
                        }
                        __syncwarp();
                        mbar_arrive(&full[st]);
                        continue;
                    }
                }
                // a chunk holding any of the step's new keys (fused append) is
                // gathered, the new rows taken from k_new / v_new
                const bool has_new = fused && chunk < sg.c_end && t0 + kChunk > new_lo &&
                                     t0 < seq_len;
                if (has_new) {
                    slot0 = -2;
                } else if (!paged_tma && chunk < sg.c_end) {
                    if (p.kind == ATTN_CACHE_LINEAR) {
                        slot0 = (int64_t)bg * p.slots_per_seq + t0;
                    } else if (paged) {
                        slot0 = -2;
                    } else {
                        const int j0 = t0 % p.slots_per_seq;
                        slot0 = (j0 + kChunk <= p.slots_per_seq)
                                    ? (int64_t)bg * p.slots_per_seq + j0
                                    : -2;
                    }
                }
                // head-major: a box must not cross the end of its block
                if (bhsd && slot0 >= 0 && slot0 % p.place.rows + kChunk > p.place.rows) slot0 = -2;
                if (lane < kCPT && slot0 == -1 && t0 < seq_len) report_error(p.err, ATTN_ERR_BOUNDS);
                const unsigned lanes = (1u << kCPT) - 1;
                const unsigned boxed = __ballot_sync(0xffffffffu, slot0 >= -1) & lanes;
                const unsigned gathered = __ballot_sync(0xffffffffu, slot0 == -2) & lanes;
                const int64_t slot00 = __shfl_sync(0xffffffffu, slot0, 0);
                // a tile whose slots are consecutive is one box per tensor;
                // otherwise each boxed chunk is a 16-row box
                const bool whole_tile =
                    __all_sync(0xffffffffu, slot0 == slot00 + (int64_t)c * kChunk) && slot00 >= 0 &&
                    (!bhsd || slot00 % p.place.rows + G::kTileRows <= p.place.rows);
                // gathered chunks: lane l copies row l % 16 of K (l < 16) or V
                uint32_t gmask = 0;
                bool issued_cp = false, issued_st = false;
                for (unsigned bits = gathered; bits; bits &= bits - 1) {
                    const int gc = __ffs(bits) - 1;
                    const int gt0 = (chunk0 + gc) * kChunk;
                    const int r = lane & (kChunk - 1), tensor = lane >> 4;
                    const int t = gt0 + r;
                    const bool is_new = fused && t >= new_lo && t < seq_len;
                    const int64_t s = is_new ? 0 : slot_of(t);
                    const unsigned valid = __ballot_sync(0xffffffffu, is_new || s >= 0) & 0xFFFFu;
                    if (lane < kChunk && !is_new && s < 0 && t < seq_len)
                        report_error(p.err, ATTN_ERR_BOUNDS);
                    if (lane == gc) gmask = valid;
                    // a new key comes from the step's rows; a masked row reads
                    // slot 0 (any valid slot will do)
                    const uint8_t *src =
                        is_new ? reinterpret_cast<const uint8_t *>(
                                     (tensor ? p.v_new : p.k_new) +
                                     ((int64_t)(sg.b * p.q_rows + (t - new_lo)) * p.n_kv_heads +
                                      sg.kvh) * HD)
                               : reinterpret_cast<const uint8_t *>(tensor ? p.v_cache : p.k_cache) +
                                     p.place.head_offset(s < 0 ? 0 : s, sg.kvh);
                    uint8_t *dst = tensor ? vst : kst;
                    if (FP8 && is_new) continue;  // encoded below, a piece per lane
#pragma unroll 4
                    for (int c16 = 0; c16 < HD * G::kElem / 16; ++c16)
                        cp_async_16_hint(dst + chunk_base<G::kHalves>(false, gc) +
                                        piece_offset(half_stride<G::kTileRows>(false), r, c16),
                                    src + c16 * 16, kv_policy);
                    issued_cp = true;
                }
                if (FP8 && fused) {
                    // E4M3 cache: the step's new rows of the gathered chunks are
                    // encoded on the way in, as the FP8 append encodes them (K minus
                    // the reference, the difference in fp32; nearest even,
                    // saturating): one 16-element piece of one row per lane
                    for (unsigned bits = gathered; bits; bits &= bits - 1) {
                        const int gc = __ffs(bits) - 1;
                        const int gt0 = (chunk0 + gc) * kChunk;
                        const int n0 = max(gt0, new_lo), n1 = min(gt0 + kChunk, seq_len);
                        constexpr int kPieces = HD / 16;
                        for (int task = lane; task < max(0, n1 - n0) * 2 * kPieces; task += 32) {
                            const int pc = task % kPieces, tr = task / kPieces;
                            const int tensor = tr & 1, t = n0 + (tr >> 1);
                            const uint4 *src = reinterpret_cast<const uint4 *>(
                                (tensor ? p.v_new : p.k_new) +
                                ((int64_t)(sg.b * p.q_rows + (t - new_lo)) * p.n_kv_heads + sg.kvh) *
                                    HD + pc * 16);
                            const uint4 a = __ldg(src), b = __ldg(src + 1);
                            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                            float x[16];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                x[2 * i] = __uint_as_float(w[i] << 16);
                                x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                            }
                            if (tensor == 0 && p.k_ref) {
                                const float4 *r4 =
                                    reinterpret_cast<const float4 *>(p.k_ref + sg.kvh * HD + pc * 16);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float4 rv = __ldg(r4 + i);
                                    x[4 * i] = __fsub_rn(x[4 * i], rv.x);
                                    x[4 * i + 1] = __fsub_rn(x[4 * i + 1], rv.y);
                                    x[4 * i + 2] = __fsub_rn(x[4 * i + 2], rv.z);
                                    x[4 * i + 3] = __fsub_rn(x[4 * i + 3], rv.w);
                                }
                            }
                            uint32_t code[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                code[i] = f32x2_to_e4m3x2(x[4 * i], x[4 * i + 1]) |
                                          (f32x2_to_e4m3x2(x[4 * i + 2], x[4 * i + 3]) << 16);
                            *reinterpret_cast<uint4 *>(
                                (tensor ? vst : kst) + chunk_base<G::kHalves>(false, gc) +
                                piece_offset(half_stride<G::kTileRows>(false), t - gt0, pc)) =
                                make_uint4(code[0], code[1], code[2], code[3]);
                            issued_st = true;
                        }
                    }
                }
                if (lane == 0) info_whole[st] = whole_tile ? 1 : 0;
                if (lane < kCPT) {
                    info_t0[st * kCPT + lane] = slot0 == -3 ? -1 : t0;
                    info_mask[st * kCPT + lane] =
                        slot0 >= 0 ? 0xFFFFu : (slot0 == -1 ? 0u : gmask);
                }
                const uint32_t tma_bytes = __popc(boxed) * 2 * G::kChunkBytes;
                if (lane == 0 && tma_bytes) mbar_expect_tx(&full[st], tma_bytes);
                __syncwarp();
                // slot-major: boxes {columns, rows, halves} of the caches viewed
                // as [kv head * halves + half][slot][columns]; head-major: boxes
                // {columns, rows, halves, 1} of [block * heads + head][half][row][columns]
                if (whole_tile) {
                    if (lane < 2) {
                        if (bhsd)
                            tma_load_4d_hint(lane ? vst : kst, lane ? &tm_v64 : &tm_k64, 0,
                                             (int)(slot00 % p.place.rows), 0,
                                             (int)(slot00 / p.place.rows) * p.n_kv_heads + sg.kvh,
                                             &full[st], kv_policy);
                        else
                            tma_load_3d_hint(lane ? vst : kst, lane ? &tm_v64 : &tm_k64, 0,
                                             (int)slot00, sg.kvh * G::kHalves, &full[st],
                                             kv_policy);
                    }
                } else if (lane < kCPT && slot0 >= -1) {
                    const uint32_t off = chunk_base<G::kHalves>(false, lane);
                    if (bhsd) {
                        // an out-of-range page aims above row 0: zero-filled
                        const int y = slot0 < 0 ? -kChunk : (int)(slot0 % p.place.rows);
                        const int w = slot0 < 0 ? sg.kvh
                                                : (int)(slot0 / p.place.rows) * p.n_kv_heads + sg.kvh;
                        tma_load_4d_hint(kst + off, &tm_k, 0, y, 0, w, &full[st], kv_policy);
                        tma_load_4d_hint(vst + off, &tm_v, 0, y, 0, w, &full[st], kv_policy);
                    } else {
                        const int y = slot0 < 0 ? -kChunk : (int)slot0;
                        tma_load_3d_hint(kst + off, &tm_k, 0, y, sg.kvh * G::kHalves, &full[st],
                                         kv_policy);
                        tma_load_3d_hint(vst + off, &tm_v, 0, y, sg.kvh * G::kHalves, &full[st],
                                         kv_policy);
                    }
                }
                __syncwarp();
                if (issued_cp && !issued_st) {
                    cp_async_arrive_noinc(&full[st]);
                } else {
                    // rows stored by this thread itself are published by a
                    // release arrive (after its own copies, if any, have landed)
                    if (issued_cp) asm volatile("cp.async.wait_all;" ::: "memory");
                    mbar_arrive(&full[st]);
                }
            }
        }
        if (!waited) pdl_wait();
        // the gathered rows of this thread must land before it leaves
        asm volatile("cp.async.wait_all;" ::: "memory");
        // No box may still be landing when the CTA exits: the last tile of
        // each stage has completed (normally the consumers have waited for it
        // already; after a wait that gave up, this wait is bounded too).
        if (lane == 0)
            for (int t = max(0, tile - kStages); t < tile; ++t)
                if (!mbar_wait(&full[t % kStages], (t / kStages) & 1, p.err)) break;
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int gq = lane >> 2, tq = lane & 3;
    const int ctid = threadIdx.x;  // 0 .. 127
    constexpr bool rope = ROPE;
    if (rope) {
        for (int i = ctid; i < HD / 2; i += kWarps * 32) rope_if[i] = p.rope_inv_freq[i];
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
    }
    if (FP8 && p.k_new != nullptr) {
        // fused append into an E4M3 cache: each thread encodes 16 elements of
        // a row into one 16-byte piece, as the FP8 append does
        const int pieces = p.n_kv_heads * HD / 16;  // of one row of one tensor
        const int64_t total = (int64_t)p.batch * p.q_rows * pieces * 2;
        for (int64_t idx = (int64_t)blockIdx.x * (kWarps * 32) + ctid; idx < total;
             idx += (int64_t)p.grid * (kWarps * 32)) {
            const int64_t row = idx / (2 * pieces);
            const int rem = (int)(idx - row * 2 * pieces);
            const int tensor = rem / pieces, pc = rem - tensor * pieces;
            const int64_t slot = p.slot_mapping[row];
            if (slot < 0 || slot >= p.num_slots) {
                if (rem == 0) report_error(p.err, ATTN_ERR_BOUNDS);
                continue;
            }
            const uint4 *src =
                reinterpret_cast<const uint4 *>(tensor ? p.v_new : p.k_new) + (row * pieces + pc) * 2;
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float x[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                x[2 * i] = __uint_as_float(w[i] << 16);
                x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
            if (tensor == 0 && p.k_ref) {
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = __fsub_rn(x[i], __ldg(p.k_ref + pc * 16 + i));
            }
            uint32_t code[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                code[i] = f32x2_to_e4m3x2(x[4 * i], x[4 * i + 1]) |
                          (f32x2_to_e4m3x2(x[4 * i + 2], x[4 * i + 3]) << 16);
            const int h = pc / (HD / 16), pp = pc - h * (HD / 16);
            uint8_t *dst = reinterpret_cast<uint8_t *>(
                               const_cast<__nv_bfloat16 *>(tensor ? p.v_cache : p.k_cache)) +
                           p.place.head_offset(slot, h) + pp * 16;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(code[0], code[1], code[2], code[3]);
        }
    }
    if (!FP8 && p.k_new != nullptr) {
        // fused append: the step's rows into their cache slots, for later
        // steps (this launch reads them from k_new / v_new); 16-byte pieces
        const int pieces = p.n_kv_heads * HD / 8;  // of one row of one tensor
        const int64_t total = (int64_t)p.batch * p.q_rows * pieces * 2;
        for (int64_t idx = (int64_t)blockIdx.x * (kWarps * 32) + ctid; idx < total;
             idx += (int64_t)p.grid * (kWarps * 32)) {
            const int64_t row = idx / (2 * pieces);
            const int rem = (int)(idx - row * 2 * pieces);
            const int tensor = rem / pieces, pc = rem - tensor * pieces;
            const int64_t slot = p.slot_mapping[row];
            if (slot < 0 || slot >= p.num_slots) {
                if (rem == 0) report_error(p.err, ATTN_ERR_BOUNDS);
                continue;
            }
            const uint4 *src =
                reinterpret_cast<const uint4 *>(tensor ? p.v_new : p.k_new) + row * pieces + pc;
            const int h = pc / (HD / 8), pp = pc - h * (HD / 8);
            uint4 *dst = reinterpret_cast<uint4 *>(
                reinterpret_cast<uint8_t *>(const_cast<__nv_bfloat16 *>(tensor ? p.v_cache
                                                                                : p.k_cache)) +
                p.place.head_offset(slot, h) + pp * 16);
            uint4 w = __ldg(src);
            if (rope && tensor == 0) {
                // key row b*q_rows + r sits at position seq_len_b - q_rows + r
                const int b = (int)(row / p.q_rows), r = (int)(row - (int64_t)b * p.q_rows);
                const int pos = tb.seqlen[b] - p.q_rows + r;
                const int i0 = (pc % (HD / 8)) * 4;  // first pair of the piece in its head
                w.x = rope_pair(w.x, pos, rope_if[i0]);
                w.y = rope_pair(w.y, pos, rope_if[i0 + 1]);
                w.z = rope_pair(w.z, pos, rope_if[i0 + 2]);
                w.w = rope_pair(w.w, pos, rope_if[i0 + 3]);
            }
            *dst = w;
        }
    }
    SegmentWalker walk{g0, g1, L};
    Segment sg;
    int tile = 0;
    int seg = 0;
    bool ok = true;
    // Partial segments merged by this CTA's end-of-share pass (a share cuts
    // at most its first and its last unit), so that no fence or atomic
    // stalls the stream in between.
    Segment pend0, pend1;
    int n_pend = 0;
    while (ok && walk.next(p, tb, sg)) {
        const int b = sg.b, kvh = sg.kvh;
        const int row0 = sg.rb * RB;
        const int row1 = min(p.rows, row0 + RB);
        const int seq_len = tb.seqlen[b];
        const int ring_lo = p.kind == ATTN_CACHE_RING ? seq_len - p.slots_per_seq : 0;
        const int window = p.window;
        const int n_tiles = (sg.c_end - sg.c_begin + kCPT - 1) / kCPT;
        // the stage of the segment's last tile: its consumers keep it until
        // the warps' states have been merged through it
        const int st_last = (tile + n_tiles - 1) % kStages;
        // wl: the layout flag of stage st_last (read once per segment end)
        auto park = [&](bool wl, int w, int row) -> float * {
            if constexpr (!G::kParkInStage) {
                return mo + ((size_t)w * RB + row) * HD;
            } else {
                // pieces: (chunk of the warp, K / V, half) of 16 x 128 B each
                constexpr int kRowsPerPiece = kChunk * 128 / (HD * 4);
                const int piece = row / kRowsPerPiece;
                const int sub = piece / (2 * G::kHalves), rest = piece - sub * 2 * G::kHalves;
                const int tensor = rest / G::kHalves, h = rest - tensor * G::kHalves;
                uint8_t *base = stages + st_last * G::kStageBytes + tensor * G::kTileBytes +
                                chunk_base<G::kHalves>(wl, w + sub * kWarps) +
                                h * half_stride<G::kTileRows>(wl);
                return reinterpret_cast<float *>(base + (row - piece * kRowsPerPiece) * HD * 4);
            }
        };
        if constexpr (MT == 0) {
            // ---- up to 8 rows: S^T = K Q^T (keys x rows), O^T = V^T P^T (d x rows)
            // Q^T as the B operand: thread holds row gq, d pairs 2tq (+8) of each k-step
            // q rows and positions staged by the producer (a padding row uses
            // the unit's first row; its scores are masked and never stored)
            const int qi = seg & 1;
            ok = mbar_wait(&q_full[qi], (seg >> 1) & 1, p.err);
            __syncwarp();
            if (!ok) break;
            const uint8_t *qs = qbuf + qi * RB * G::kQStride;
            uint32_t qb[HD / 16][2];
            {
                const int qr = row0 + gq < row1 ? gq : 0;
                const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qs + qr * G::kQStride);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    if constexpr (FP8) {
                        // k-step kk pairs with bytes 4 (kk % 4) .. + 3 of piece
                        // tq + 4 (kk / 4) of a key row (see the score loop):
                        // the same dims of q, as f16
                        const int w = 8 * (tq + 4 * (kk >> 2)) + 2 * (kk & 3);
                        qb[kk][0] = bf16x2_to_f16x2(qrow[w]);
                        qb[kk][1] = bf16x2_to_f16x2(qrow[w + 1]);
                    } else {
                        qb[kk][0] = qrow[kk * 8 + tq];
                        qb[kk][1] = qrow[kk * 8 + 4 + tq];
                    }
                }
                if (rope) {  // word w of a row is pair w
                    const int qpos = posbuf[qi * RB + qr];
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        qb[kk][0] = rope_pair(qb[kk][0], qpos, rope_if[kk * 8 + tq]);
                        qb[kk][1] = rope_pair(qb[kk][1], qpos, rope_if[kk * 8 + 4 + tq]);
                    }
                }
            }
            // this thread's S^T columns are rows 2tq and 2tq+1
            int cpos[2];
            bool cvalid[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                cvalid[e] = row0 + 2 * tq + e < row1;
                cpos[e] = posbuf[qi * RB + (cvalid[e] ? 2 * tq + e : 0)];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qi]);
            ++seg;
            float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
            float o[HD / 16][4];  // m-tile md: (d = 16md + gq (+8), rows 2tq, 2tq+1)
#pragma unroll
            for (int n = 0; n < HD / 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            for (int it = 0; it < n_tiles; ++it, ++tile) {
                const int st = tile % kStages;
                ok = mbar_wait(&full[st], (tile / kStages) & 1, p.err);
                __syncwarp();  // reconverge before the warp-collective ldmatrix / mma
                if (!ok) break;
#pragma unroll 1
                for (int sub = 0; sub < G::kSubs; ++sub) {  // this warp's chunks of the tile
                const int ci = warp + sub * kWarps;
                const int t0 = info_t0[st * kCPT + ci];
                if (t0 >= 0) {
                    const uint32_t mask16 = info_mask[st * kCPT + ci];
                    const bool whole = info_whole[st] != 0;
                    const uint32_t hs = half_stride<G::kTileRows>(whole);
                    const uint32_t kbase =
                        smem_u32(stages + st * G::kStageBytes) + chunk_base<G::kHalves>(whole, ci);
                    const uint32_t vbase = kbase + G::kTileBytes;
                    if (rope && t0 + kChunk > seq_len - p.q_rows && t0 < seq_len) {
                        // new keys of the step, gathered unrotated from k_new:
                        // rotate them in place (word w of a row is pair w)
                        const int t_end = min(t0 + kChunk, seq_len);
                        for (int t = max(t0, seq_len - p.q_rows); t < t_end; ++t)
                            for (int w = lane; w < HD / 2; w += 32) {
                                const uint32_t a =
                                    kbase + piece_offset(hs, t - t0, w >> 2) + (w & 3) * 4;
                                st_shared_u32(a, rope_pair(ld_shared_u32(a), t, rope_if[w]));
                            }
                        __syncwarp();
                    }
                    const int m = lane >> 3;
                    float sacc[4] = {0.f, 0.f, 0.f, 0.f};  // (key gq | gq+8) x (row 2tq | 2tq+1)
                    // odd k-steps accumulate apart: two chains of dependent mma
                    // instead of one, added at the end
                    float sodd[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (FP8) {
                        // A = K, keys gq and gq + 8: k-step kk takes word kk % 4 of
                        // 16-byte piece tq + 4 (kk / 4) of each key row, its two
                        // low codes as k = 2tq, 2tq + 1 and its two high codes as
                        // k = 2tq + 8, 2tq + 9
                        uint32_t kw[2][8];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 lo = ld_shared_v4(kbase + piece_offset(hs, gq + 8 * h, tq));
                            const uint4 hi =
                                ld_shared_v4(kbase + piece_offset(hs, gq + 8 * h, tq + 4));
                            kw[h][0] = lo.x, kw[h][1] = lo.y, kw[h][2] = lo.z, kw[h][3] = lo.w;
                            kw[h][4] = hi.x, kw[h][5] = hi.y, kw[h][6] = hi.z, kw[h][7] = hi.w;
                        }
#pragma unroll
                        for (int kk = 0; kk < HD / 16; ++kk) {
                            uint32_t a[4];
                            e4m3x4_to_f16x2x2(kw[0][kk], a[0], a[2]);
                            e4m3x4_to_f16x2x2(kw[1][kk], a[1], a[3]);
                            mma_f16_16816((kk & 1) ? sodd : sacc, a, qb[kk][0], qb[kk][1]);
                        }
                    } else {
                        const int key = (m & 1) * 8 + (lane & 7);
#pragma unroll
                        for (int kk = 0; kk < HD / 16; ++kk) {
                            uint32_t a[4];
                            ldmatrix_x4(a[0], a[1], a[2], a[3],
                                        kbase + piece_offset(hs, key, kk * 2 + (m >> 1)));
                            mma_bf16_16816((kk & 1) ? sodd : sacc, a, qb[kk][0], qb[kk][1]);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[e] += sodd[e];
                    // the whole chunk visible to every row of the warp: no mask (a
                    // padding row repeats the unit's first row and position; its
                    // results are never stored)
                    if (__all_sync(0xffffffffu,
                                   chunk_open(mask16, t0, seq_len, ring_lo, window,
                                              min(cpos[0], cpos[1]), max(cpos[0], cpos[1])))) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) sacc[e] *= p.scale_log2;
                    } else {
#pragma unroll
                        for (int e = 0; e < 2; ++e)  // row 2tq + e: elements e (key gq), e+2 (key gq+8)
#pragma unroll
                            for (int hk = 0; hk < 2; ++hk) {
                                const int n = gq + hk * 8;
                                const int t = t0 + n, pos = cpos[e];
                                const bool valid = cvalid[e] && ((mask16 >> n) & 1u) &&
                                                   t < seq_len && t <= pos && t >= ring_lo &&
                                                   (window <= 0 || pos - t < window);
                                sacc[e + 2 * hk] =
                                    valid ? sacc[e + 2 * hk] * p.scale_log2 : -INFINITY;
                            }
                    }
                    float alpha[2];
                    bool moved = false;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float mx = fmaxf(sacc[e], sacc[e + 2]);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float m_old = m_run[e];
                        const float m_new = mx > m_old + kRescaleLog2 ? mx : m_old;
                        const float m_use = m_new == -INFINITY ? 0.f : m_new;
                        alpha[e] = m_new == m_old ? 1.f : fast_exp2(m_old - m_use);
                        moved |= m_new != m_old;
                        const float p0 = fast_exp2(sacc[e] - m_use);
                        const float p1 = fast_exp2(sacc[e + 2] - m_use);
                        sacc[e] = p0;
                        sacc[e + 2] = p1;
                        l_run[e] = l_run[e] * alpha[e] + (p0 + p1);
                        m_run[e] = m_new;
                    }
                    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                        for (int n = 0; n < HD / 16; ++n) {
                            o[n][0] *= alpha[0];
                            o[n][1] *= alpha[1];
                            o[n][2] *= alpha[0];
                            o[n][3] *= alpha[1];
                        }
                    }
                    if constexpr (FP8) {
                        // P^T in f16 (one rounding: 11 significant bits)
                        const uint32_t bh0 = movmatrix_trans(pack_f16x2(sacc[0], sacc[1]));
                        const uint32_t bh1 = movmatrix_trans(pack_f16x2(sacc[2], sacc[3]));
                        // A = V^T: this thread supplies keys 2tq, 2tq+1 (k = 2tq,
                        // 2tq+1) and 2tq+8, 2tq+9, all from 16-byte piece gq; rows
                        // gq and gq + 8 of m-tile md are dims 16 gq + 2 md and + 1
                        uint32_t vw[4][4];
#pragma unroll
                        for (int kr = 0; kr < 4; ++kr) {
                            const uint4 v = ld_shared_v4(
                                vbase + piece_offset(hs, 2 * tq + (kr & 1) + 8 * (kr >> 1), gq));
                            vw[kr][0] = v.x, vw[kr][1] = v.y, vw[kr][2] = v.z, vw[kr][3] = v.w;
                        }
#pragma unroll
                        for (int md = 0; md < HD / 16; ++md) {
                            // bytes 2md, 2md+1 of the piece, interleaved key by key
                            const uint32_t sel = (md & 1) ? 0x7362u : 0x5140u;
                            const uint32_t x = __byte_perm(vw[0][md >> 1], vw[1][md >> 1], sel);
                            const uint32_t y = __byte_perm(vw[2][md >> 1], vw[3][md >> 1], sel);
                            uint32_t a[4];
                            e4m3x4_to_f16x2x2(x, a[0], a[1]);
                            e4m3x4_to_f16x2x2(y, a[2], a[3]);
                            mma_f16_16816(o[md], a, bh0, bh1);
                        }
                    } else {
                    // P^T fragments: transpose the (key x row) blocks of keys 0-7 and 8-15
                    uint32_t h0, l0, h1, l1;
                    split_bf16x2(sacc[0], sacc[1], h0, l0);
                    split_bf16x2(sacc[2], sacc[3], h1, l1);
                    const uint32_t bh0 = movmatrix_trans(h0), bl0 = movmatrix_trans(l0);
                    const uint32_t bh1 = movmatrix_trans(h1), bl1 = movmatrix_trans(l1);
                    {
                        const int key = (m >> 1) * 8 + (lane & 7);
#pragma unroll
                        for (int md = 0; md < HD / 16; ++md) {
                            uint32_t a[4];
                            ldmatrix_x4_trans(a[0], a[1], a[2], a[3],
                                              vbase + piece_offset(hs, key, md * 2 + (m & 1)));
                            mma_bf16_16816(o[md], a, bh0, bh1);
                            mma_bf16_16816(o[md], a, bl0, bl1);
                        }
                    }
                    }
                }
                }  // sub
                __syncwarp();
                if (lane == 0 && it + 1 < n_tiles) mbar_arrive(&empty[st]);
            }
            // the row sums are spread over the 8 lanes that share tq
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = l_run[e];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                l_run[e] = l;
            }
            __syncwarp();  // the warp's reads of the last tile are done
            const bool wl = info_whole[st_last] != 0;
            if constexpr (FP8) {
                // rows 2tq + e hold dims 16 gq .. 16 gq + 15 here: 16-byte stores
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = 2 * tq + e;
                    float *dst = park(wl, warp, row);
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd)
                        *reinterpret_cast<float4 *>(dst + 4 * park_unit<MT, FP8>(row, 4 * gq + qd)) =
                            make_float4(o[2 * qd][e], o[2 * qd][e + 2], o[2 * qd + 1][e],
                                        o[2 * qd + 1][e + 2]);
                }
            } else {
#pragma unroll
                for (int md = 0; md < HD / 16; ++md)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = 2 * tq + (e & 1);
                        const int d = md * 16 + gq + (e >> 1) * 8;
                        park(wl, warp, row)[d] = o[md][e];
                    }
            }
            if (gq == 0) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    mm[warp * RB + 2 * tq + e] = m_run[e];
                    ml[warp * RB + 2 * tq + e] = l_run[e];
                }
            }
        } else {
            // q rows and positions staged by the producer, as in the MT = 0 path
            const int qi = seg & 1;
            ok = mbar_wait(&q_full[qi], (seg >> 1) & 1, p.err);
            __syncwarp();
            if (!ok) break;
            const uint8_t *qs = qbuf + qi * RB * G::kQStride;
            uint32_t qa[MT][HD / 16][4];
            int rpos[MT][2];
            bool rvalid[MT][2];
    #pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
    #pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int rr = mt * 16 + gq + hr * 8;
                    rvalid[mt][hr] = row0 + rr < row1;
                    const int rc = rvalid[mt][hr] ? rr : 0;
                    rpos[mt][hr] = posbuf[qi * RB + rc];
                    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qs + rc * G::kQStride);
    #pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        if constexpr (FP8) {  // the score loop's dim order, as f16
                            const int w = 8 * (tq + 4 * (kk >> 2)) + 2 * (kk & 3);
                            qa[mt][kk][hr] = bf16x2_to_f16x2(qrow[w]);
                            qa[mt][kk][2 + hr] = bf16x2_to_f16x2(qrow[w + 1]);
                        } else {
                            qa[mt][kk][hr] = qrow[kk * 8 + tq];
                            qa[mt][kk][2 + hr] = qrow[kk * 8 + 4 + tq];
                        }
                    }
                    if (rope) {  // word w of a row is pair w
    #pragma unroll
                        for (int kk = 0; kk < HD / 16; ++kk) {
                            qa[mt][kk][hr] =
                                rope_pair(qa[mt][kk][hr], rpos[mt][hr], rope_if[kk * 8 + tq]);
                            qa[mt][kk][2 + hr] = rope_pair(qa[mt][kk][2 + hr], rpos[mt][hr],
                                                           rope_if[kk * 8 + 4 + tq]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qi]);
            ++seg;
            float m_run[MT][2], l_run[MT][2];
            float o[MT][HD / 8][4];
    #pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                m_run[mt][0] = m_run[mt][1] = -INFINITY;
                l_run[mt][0] = l_run[mt][1] = 0.f;
    #pragma unroll
                for (int n = 0; n < HD / 8; ++n)
                    o[mt][n][0] = o[mt][n][1] = o[mt][n][2] = o[mt][n][3] = 0.f;
            }
            for (int it = 0; it < n_tiles; ++it, ++tile) {
                const int st = tile % kStages;
                ok = mbar_wait(&full[st], (tile / kStages) & 1, p.err);
                __syncwarp();  // reconverge before the warp-collective ldmatrix / mma
                if (!ok) break;
#pragma unroll 1
                for (int sub = 0; sub < G::kSubs; ++sub) {  // this warp's chunks of the tile
                const int ci = warp + sub * kWarps;
                const int t0 = info_t0[st * kCPT + ci];
                if (t0 >= 0) {
                    const uint32_t mask16 = info_mask[st * kCPT + ci];
                    const bool whole = info_whole[st] != 0;
                    const uint32_t hs = half_stride<G::kTileRows>(whole);
                    const uint32_t kbase =
                        smem_u32(stages + st * G::kStageBytes) + chunk_base<G::kHalves>(whole, ci);
                    const uint32_t vbase = kbase + G::kTileBytes;
                    if (rope && t0 + kChunk > seq_len - p.q_rows && t0 < seq_len) {
                        // new keys of the step, gathered unrotated from k_new:
                        // rotate them in place (word w of a row is pair w)
                        const int t_end = min(t0 + kChunk, seq_len);
                        for (int t = max(t0, seq_len - p.q_rows); t < t_end; ++t)
                            for (int w = lane; w < HD / 2; w += 32) {
                                const uint32_t a =
                                    kbase + piece_offset(hs, t - t0, w >> 2) + (w & 3) * 4;
                                st_shared_u32(a, rope_pair(ld_shared_u32(a), t, rope_if[w]));
                            }
                        __syncwarp();
                    }
                    float s[MT][2][4];
    #pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
    #pragma unroll
                        for (int j = 0; j < 2; ++j)
                            s[mt][j][0] = s[mt][j][1] = s[mt][j][2] = s[mt][j][3] = 0.f;
                    if constexpr (FP8) {
                        // B = K^T, keys gq (n-tile 0) and gq + 8 (n-tile 1), read
                        // as in the MT = 0 score loop
                        uint32_t kw[2][8];
    #pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 lo = ld_shared_v4(kbase + piece_offset(hs, gq + 8 * h, tq));
                            const uint4 hi =
                                ld_shared_v4(kbase + piece_offset(hs, gq + 8 * h, tq + 4));
                            kw[h][0] = lo.x, kw[h][1] = lo.y, kw[h][2] = lo.z, kw[h][3] = lo.w;
                            kw[h][4] = hi.x, kw[h][5] = hi.y, kw[h][6] = hi.z, kw[h][7] = hi.w;
                        }
    #pragma unroll
                        for (int kk = 0; kk < HD / 16; ++kk) {
                            uint32_t b00, b01, b10, b11;
                            e4m3x4_to_f16x2x2(kw[0][kk], b00, b01);
                            e4m3x4_to_f16x2x2(kw[1][kk], b10, b11);
    #pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                mma_f16_16816(s[mt][0], qa[mt][kk], b00, b01);
                                mma_f16_16816(s[mt][1], qa[mt][kk], b10, b11);
                            }
                        }
                    } else {
                        const int m = lane >> 3;
                        const int key = (m >> 1) * 8 + (lane & 7);
    #pragma unroll
                        for (int kk = 0; kk < HD / 16; ++kk) {
                            uint32_t b00, b01, b10, b11;
                            ldmatrix_x4(b00, b01, b10, b11,
                                        kbase + piece_offset(hs, key, kk * 2 + (m & 1)));
    #pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                mma_bf16_16816(s[mt][0], qa[mt][kk], b00, b01);
                                mma_bf16_16816(s[mt][1], qa[mt][kk], b10, b11);
                            }
                        }
                    }
                    // the whole chunk visible to every row of the warp: no mask
                    int pmin = rpos[0][0], pmax = rpos[0][0];
    #pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
    #pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            pmin = min(pmin, rpos[mt][hr]);
                            pmax = max(pmax, rpos[mt][hr]);
                        }
                    const bool open = __all_sync(
                        0xffffffffu, chunk_open(mask16, t0, seq_len, ring_lo, window, pmin, pmax));
                    uint32_t pa[MT][4], pl[MT][4];  // P as bf16 hi + lo
    #pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        if (open) {
    #pragma unroll
                            for (int j = 0; j < 2; ++j)
    #pragma unroll
                                for (int e = 0; e < 4; ++e) s[mt][j][e] *= p.scale_log2;
                        } else {
    #pragma unroll
                            for (int hr = 0; hr < 2; ++hr)
    #pragma unroll
                                for (int j = 0; j < 2; ++j)
    #pragma unroll
                                    for (int e = 0; e < 2; ++e) {
                                        const int n = j * 8 + tq * 2 + e;
                                        const int t = t0 + n, pos = rpos[mt][hr];
                                        const bool valid =
                                            rvalid[mt][hr] && ((mask16 >> n) & 1u) &&
                                            t < seq_len && t <= pos && t >= ring_lo &&
                                            (window <= 0 || pos - t < window);
                                        s[mt][j][hr * 2 + e] =
                                            valid ? s[mt][j][hr * 2 + e] * p.scale_log2
                                                  : -INFINITY;
                                    }
                        }
    #pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            float mx = fmaxf(fmaxf(s[mt][0][hr * 2], s[mt][0][hr * 2 + 1]),
                                             fmaxf(s[mt][1][hr * 2], s[mt][1][hr * 2 + 1]));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                            const float m_old = m_run[mt][hr];
                            const float m_new = mx > m_old + kRescaleLog2 ? mx : m_old;
                            const float m_use = m_new == -INFINITY ? 0.f : m_new;
                            float sum = 0.f;
    #pragma unroll
                            for (int j = 0; j < 2; ++j)
    #pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const float pv = fast_exp2(s[mt][j][hr * 2 + e] - m_use);
                                    s[mt][j][hr * 2 + e] = pv;
                                    sum += pv;
                                }
                            if (__any_sync(0xffffffffu, m_new != m_old)) {
                                const float alpha =
                                    m_new == m_old ? 1.f : fast_exp2(m_old - m_use);
                                l_run[mt][hr] *= alpha;
    #pragma unroll
                                for (int n = 0; n < HD / 8; ++n) {
                                    o[mt][n][hr * 2] *= alpha;
                                    o[mt][n][hr * 2 + 1] *= alpha;
                                }
                            }
                            l_run[mt][hr] += sum;
                            m_run[mt][hr] = m_new;
                        }
                        if constexpr (FP8) {  // P in f16, one rounding
                            pa[mt][0] = pack_f16x2(s[mt][0][0], s[mt][0][1]);
                            pa[mt][1] = pack_f16x2(s[mt][0][2], s[mt][0][3]);
                            pa[mt][2] = pack_f16x2(s[mt][1][0], s[mt][1][1]);
                            pa[mt][3] = pack_f16x2(s[mt][1][2], s[mt][1][3]);
                        } else {
                            split_bf16x2(s[mt][0][0], s[mt][0][1], pa[mt][0], pl[mt][0]);
                            split_bf16x2(s[mt][0][2], s[mt][0][3], pa[mt][1], pl[mt][1]);
                            split_bf16x2(s[mt][1][0], s[mt][1][1], pa[mt][2], pl[mt][2]);
                            split_bf16x2(s[mt][1][2], s[mt][1][3], pa[mt][3], pl[mt][3]);
                        }
                    }
                    if constexpr (FP8) {
                        // B = V: this thread supplies keys 2tq, 2tq+1, 2tq+8, 2tq+9
                        // of column n = gq; n-tile j's column gq is dim 16 gq + j,
                        // byte j of 16-byte piece gq
                        uint32_t vw[4][4];
    #pragma unroll
                        for (int kr = 0; kr < 4; ++kr) {
                            const uint4 v = ld_shared_v4(
                                vbase + piece_offset(hs, 2 * tq + (kr & 1) + 8 * (kr >> 1), gq));
                            vw[kr][0] = v.x, vw[kr][1] = v.y, vw[kr][2] = v.z, vw[kr][3] = v.w;
                        }
    #pragma unroll
                        for (int jj = 0; jj < HD / 16; ++jj) {  // n-tiles 2jj, 2jj + 1
                            const uint32_t sel = (jj & 1) ? 0x7362u : 0x5140u;
                            const uint32_t x = __byte_perm(vw[0][jj >> 1], vw[1][jj >> 1], sel);
                            const uint32_t y = __byte_perm(vw[2][jj >> 1], vw[3][jj >> 1], sel);
                            uint32_t x0, x1, y0, y1;
                            e4m3x4_to_f16x2x2(x, x0, x1);
                            e4m3x4_to_f16x2x2(y, y0, y1);
    #pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                mma_f16_16816(o[mt][2 * jj], pa[mt], x0, y0);
                                mma_f16_16816(o[mt][2 * jj + 1], pa[mt], x1, y1);
                            }
                        }
                    } else {
                        const int m = lane >> 3;
                        const int key = (m & 1) * 8 + (lane & 7);
    #pragma unroll
                        for (int dn = 0; dn < HD / 16; ++dn) {
                            uint32_t v0, v1, v2, v3;
                            ldmatrix_x4_trans(v0, v1, v2, v3,
                                              vbase + piece_offset(hs, key, dn * 2 + (m >> 1)));
    #pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                mma_bf16_16816(o[mt][dn * 2], pa[mt], v0, v1);
                                mma_bf16_16816(o[mt][dn * 2 + 1], pa[mt], v2, v3);
                                mma_bf16_16816(o[mt][dn * 2], pl[mt], v0, v1);
                                mma_bf16_16816(o[mt][dn * 2 + 1], pl[mt], v2, v3);
                            }
                        }
                    }
                }
                }  // sub
                __syncwarp();
                if (lane == 0 && it + 1 < n_tiles) mbar_arrive(&empty[st]);
            }
            // ---- end of segment: merge the four warps through shared memory
    #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
    #pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    float l = l_run[mt][hr];
                    l += __shfl_xor_sync(0xffffffffu, l, 1);
                    l += __shfl_xor_sync(0xffffffffu, l, 2);
                    l_run[mt][hr] = l;
                }
            __syncwarp();  // the warp's reads of the last tile are done
            const bool wl = info_whole[st_last] != 0;
    #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
    #pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int row = mt * 16 + gq + hr * 8;
                    float *dst = park(wl, warp, row);
                    if constexpr (FP8) {
                        // columns 2tq, 2tq + 1 of n-tile j are dims 32 tq + j and
                        // 32 tq + 16 + j: this thread holds dims 32 tq .. 32 tq + 31
    #pragma unroll
                        for (int qd = 0; qd < 4; ++qd) {
                            *reinterpret_cast<float4 *>(
                                dst + 4 * park_unit<MT, FP8>(row, 8 * tq + qd)) =
                                make_float4(o[mt][4 * qd][hr * 2], o[mt][4 * qd + 1][hr * 2],
                                            o[mt][4 * qd + 2][hr * 2], o[mt][4 * qd + 3][hr * 2]);
                            *reinterpret_cast<float4 *>(
                                dst + 4 * park_unit<MT, FP8>(row, 8 * tq + 4 + qd)) =
                                make_float4(o[mt][4 * qd][hr * 2 + 1], o[mt][4 * qd + 1][hr * 2 + 1],
                                            o[mt][4 * qd + 2][hr * 2 + 1],
                                            o[mt][4 * qd + 3][hr * 2 + 1]);
                        }
                    } else {
    #pragma unroll
                        for (int n = 0; n < HD / 8; ++n)
                            *reinterpret_cast<float2 *>(dst + n * 8 + tq * 2) =
                                make_float2(o[mt][n][hr * 2], o[mt][n][hr * 2 + 1]);
                    }
                    if (tq == 0) {
                        mm[warp * RB + row] = m_run[mt][hr];
                        ml[warp * RB + row] = l_run[mt][hr];
                    }
                }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
        // per row: each warp's weight exp2(m_w - M) / sum and the row's log-sum-exp
        if (ctid < RB) {
            const int row = ctid;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * RB + row]);
            float f[kWarps], Lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = mm[w * RB + row];
                f[w] = (M == -INFINITY || mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
                Lsum += ml[w * RB + row] * f[w];
            }
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) wgt[row * kWarps + w] = f[w] * inv;
            rlse[row] = Lsum > 0.f ? M + __log2f(Lsum) : -INFINITY;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
        {
            // every output piece of the unit: all parked loads in flight at once
            constexpr int kItems = RB * (HD / 4) / (kWarps * 32);
            static_assert(kItems * kWarps * 32 == RB * (HD / 4), "whole items per thread");
            const bool wl = info_whole[st_last] != 0;
            float4 acc[kItems];
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                const int idx = ctid + k * (kWarps * 32);
                const int row = idx / (HD / 4), d = (idx % (HD / 4)) * 4;
                const float4 wt = *reinterpret_cast<const float4 *>(wgt + row * kWarps);
                float4 v[kWarps];
#pragma unroll
                for (int w = 0; w < kWarps; ++w)
                    v[w] = *reinterpret_cast<const float4 *>(park(wl, w, row) +
                                                             4 * park_unit<MT, FP8>(row, d >> 2));
                const float ww[4] = {wt.x, wt.y, wt.z, wt.w};
                acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    acc[k].x += ww[w] * v[w].x;
                    acc[k].y += ww[w] * v[w].y;
                    acc[k].z += ww[w] * v[w].z;
                    acc[k].w += ww[w] * v[w].w;
                }
            }
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                const int idx = ctid + k * (kWarps * 32);
                const int row = idx / (HD / 4), d = (idx % (HD / 4)) * 4;
                const int i = row0 + row;
                if (i >= row1) continue;
                if (sg.whole) {
                    const int r = i / p.group, g = i - (i / p.group) * p.group;
                    __nv_bfloat16 *dst =
                        p.out + (((int64_t)b * p.q_rows + r) * p.n_q_heads + kvh * p.group + g) * HD +
                        d;
                    uint2 packed;
                    packed.x = pack_bf16x2(acc[k].x, acc[k].y);
                    packed.y = pack_bf16x2(acc[k].z, acc[k].w);
                    *reinterpret_cast<uint2 *>(dst) = packed;
                } else {
                    // partial slot (unit, this CTA): unit + blockIdx.x is unique
                    const int64_t slot = ((int64_t)sg.unit + blockIdx.x) * RB + row;
                    *reinterpret_cast<float4 *>(p.ws_o + slot * HD + d) = acc[k];
                    if (d == 0) p.ws_lse[slot] = rlse[row];
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");  // parked rows read
        if (lane == 0) mbar_arrive(&empty[st_last]);
        if (!sg.whole && (!p.merge_kernel || sg.last - sg.first < kGroupParts)) {
            if (n_pend == 0)
                pend0 = sg;
            else
                pend1 = sg;
            n_pend = min(n_pend + 1, 2);
        }
    }
    if (n_pend == 0) return;
    // ---- end of share: merges of units split over several CTAs.  Parts
    // first..last of a unit form groups of kGroupParts consecutive CTAs; the
    // CTA that stores a group's last part (counter at the group's first slot)
    // merges the group, in CTA order, into that slot; the CTA that completes
    // a unit's last group (per-unit counter) merges the groups in order into
    // the bf16 output.  A unit of at most kGroupParts parts is one group
    // merged straight to the output.  Ordering: the consumer barrier puts every
    // thread's partial stores before thread 0's counter update, whose release
    // (gpu scope, cumulative) publishes them; the CTA whose update completes a
    // group acquires the others' by the same update, and the barrier after it
    // orders its threads' loads after that acquire.
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
    for (int k = 0; k < n_pend; ++k) {
        const Segment &u = k == 0 ? pend0 : pend1;
        const int n = u.last - u.first + 1;
        const int gf = u.first + (((int)blockIdx.x - u.first) / kGroupParts) * kGroupParts;
        const int gl = min(u.last, gf + kGroupParts - 1);
        const int64_t gslot = (int64_t)u.unit + gf;
        // one flag per (segment, level), each written once: a thread still
        // reading one flag never sees the next decision
        if (ctid == 0) {
            int32_t *cnt = n <= kGroupParts ? p.ws_count + u.unit : p.ws_gcount + gslot;
            s_last[2 * k] = atom_add_acq_rel_gpu(cnt, 1) == gl - gf ? 1 : 0;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
        if (!s_last[2 * k]) continue;  // uniform across the consumer warps
        if (n <= kGroupParts) {
            merge_partials<HD, RB>(p, u, gslot, 1, n, true, ctid);
            if (ctid == 0) p.ws_count[u.unit] = 0;  // ready for the next call
            continue;
        }
        merge_partials<HD, RB>(p, u, gslot, 1, gl - gf + 1, false, ctid);
        // (merge_partials ends with the consumer barrier: its stores precede
        // the release below)
        const int groups = (n + kGroupParts - 1) / kGroupParts;
        if (ctid == 0) {
            p.ws_gcount[gslot] = 0;
            s_last[2 * k + 1] = atom_add_acq_rel_gpu(p.ws_count + u.unit, 1) == groups - 1 ? 1 : 0;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
        if (!s_last[2 * k + 1]) continue;
        merge_partials<HD, RB>(p, u, (int64_t)u.unit + u.first, kGroupParts, groups, true, ctid);
        if (ctid == 0) p.ws_count[u.unit] = 0;
    }
}

// Merge kernel, for launches whose units may span very many CTAs (long
// contexts over few units): one CTA per
// (request, KV head, query row of the group); its warps take the parts
// round-robin (online max / sum per warp), and the warps' states are combined
// in a fixed order, so the result does not depend on timing.
template <int HD, int RB>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const Params p) {
    constexpr int PER = HD / 32;
    __shared__ float sm_m[kMergeWarps], sm_l[kMergeWarps];
    __shared__ __align__(16) float sm_o[kMergeWarps][HD];
    __shared__ int t_cnt[kMaxTableEntries], t_clo[kMaxTableEntries], t_seq[kMaxTableEntries],
        t_pb[kMaxTableEntries + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int b = cta / (p.rows * p.n_kv_heads);
    const int rem = cta - b * p.rows * p.n_kv_heads;
    const int kvh = rem / p.rows;
    const int i = rem - kvh * p.rows;
    const int rb = i / RB, row = i - rb * RB;
    const int unit = (b * p.n_kv_heads + kvh) * p.row_blocks + rb;
    // Release the next kernel at once: a following split kernel then takes
    // each SM as this call's split CTAs leave it and plans and prefetches its
    // first tiles while this merge waits, and it waits itself for this
    // kernel to complete, which comes after this call's split kernel has.
    // Everything issued before that split kernel has completed before this
    // kernel starts (the split kernel releases it only after its own wait).
    pdl_launch_dependents();
    // The CTAs that hold the unit, from the split kernel's own tables: this
    // kernel's predecessor is that split kernel, which releases it only after
    // waiting for its own predecessor, so seq_lens and positions are final and
    // the tables can be built while the split kernel is still running.
    const Tables tb{t_cnt, t_clo, t_seq, t_pb};
    build_tables(p, tb, kMergeWarps * 32, false);
    int first = 0, last = -1;
    {
        const int RBc = p.row_blocks;
        const int N = tb.Pb[p.batch];
        const int L = max(kMinChunksPerCta, (N + p.grid - 1) / p.grid);
        const int n_u = tb.cnt[b * RBc + rb];
        if (n_u > 0) {
            const int per_head = (tb.Pb[b + 1] - tb.Pb[b]) / p.n_kv_heads;
            int start = tb.Pb[b] + kvh * per_head;
            for (int r = 0; r < rb; ++r) {
                const int n = tb.cnt[b * RBc + r];
                start += n > 0 ? n + kUnitGapChunks : 0;
            }
            first = start / L;
            last = (start + n_u - 1) / L;
        }
    }
    pdl_wait();  // the partial states come from the split kernel
    // no keys (zero-filled) or few parts (merged by the split kernel)
    if (last - first < kGroupParts) return;
    // Each warp takes parts first + warp + kMergeWarps * k; a batch of kBatch
    // of them is loaded at once (all loads in flight), then folded into the
    // warp's state.
    float m = -INFINITY, l = 0.f;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    constexpr int kBatch = 10;
    for (int c0 = first + warp; c0 <= last; c0 += kBatch * kMergeWarps) {
        float lse[kBatch];
        float v[kBatch][PER];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int c = c0 + k * kMergeWarps;
            lse[k] = -INFINITY;
#pragma unroll
            for (int e = 0; e < PER; ++e) v[k][e] = 0.f;
            if (c <= last) {
                const int64_t slot = ((int64_t)unit + c) * RB + row;
                lse[k] = __ldcg(p.ws_lse + slot);
                const float *src = p.ws_o + slot * HD + lane * PER;
                if constexpr (PER == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                    v[k][0] = t.x;
                    v[k][1] = t.y;
                    v[k][2] = t.z;
                    v[k][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                    v[k][0] = t.x;
                    v[k][1] = t.y;
                }
            }
        }
        float mb = m;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) mb = fmaxf(mb, lse[k]);
        if (mb == -INFINITY) continue;
        const float fo = fast_exp2(m - mb);  // m == -inf gives 0
        l *= fo;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] *= fo;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float f = fast_exp2(lse[k] - mb);  // -inf gives 0
            l += f;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] += f * v[k][e];
        }
        m = mb;
    }
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
    }
#pragma unroll
    for (int e = 0; e < PER; ++e) sm_o[warp][lane * PER + e] = acc[e];
    __syncthreads();
    if (warp != 0) return;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, sm_m[w]);
    float Lsum = 0.f;
    float o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            if (sm_m[w] == -INFINITY) continue;
            const float f = fast_exp2(sm_m[w] - M);
            Lsum += f * sm_l[w];
#pragma unroll
            for (int e = 0; e < PER; ++e) o[e] += f * sm_o[w][lane * PER + e];
        }
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    const int r = i / p.group, g = i - r * p.group;
    __nv_bfloat16 *dst =
        p.out + (((int64_t)b * p.q_rows + r) * p.n_q_heads + kvh * p.group + g) * HD + lane * PER;
    if constexpr (PER == 4) {
        uint2 packed;
        packed.x = pack_bf16x2(o[0] * inv, o[1] * inv);
        packed.y = pack_bf16x2(o[2] * inv, o[3] * inv);
        *reinterpret_cast<uint2 *>(dst) = packed;
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(o[0] * inv, o[1] * inv);
    }
}

template <int HD, int MT, bool ROPE, bool FP8>
int launch_split(const Params &p, const CUtensorMap &tk, const CUtensorMap &tv,
                 const CUtensorMap &tk64, const CUtensorMap &tv64, cudaStream_t stream) {
    using G = Geo<HD, MT, FP8>;
    static_assert(G::kSmem * G::kCtasPerSm + 1024 * (G::kCtasPerSm - 1) <= 232448,
                  "shared memory budget");
    auto kern = decode_split_kernel<HD, MT, ROPE, FP8>;
    const size_t smem = G::kSmem;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return ATTN_ERR_CUDA;
        }
        configured_device = dev;
    }
    if (launch_pdl(kern, dim3(p.grid), dim3(kThreads), smem, stream, tk, tv, tk64, tv64, p) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    if (p.merge_kernel) {
        const unsigned ctas = (unsigned)((int64_t)p.batch * p.rows * p.n_kv_heads);
        if (launch_pdl(decode_merge_kernel<HD, G::RB>, dim3(ctas), dim3(kMergeWarps * 32), 0,
                       stream, p) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace dec

int plan_decode(const attn_kv_cache *cache, int batch, int q_rows, int n_q_heads, int n_kv_heads,
                int head_dim, int max_seq_len, int window, DecodePlan *plan) {
    const int group = n_q_heads / n_kv_heads;
    plan->head_dim = head_dim;
    plan->rows = q_rows * group;
    // 32-row units run one CTA per SM (their registers); a group of more than
    // 32 rows (a prefill chunk: R x G rows) is cut into 16-row units instead,
    // two CTAs per SM: twice the warps to hide the mma latency, each K/V tile
    // read by more units (from L2): measured 1.26x on 29-row chunks of 28/4.
    plan->m_tiles = plan->rows <= 8 ? 0 : (plan->rows <= 16 || plan->rows > 32) ? 1 : 2;
    const int rb_rows = plan->m_tiles == 0 ? 8 : 16 * plan->m_tiles;
    plan->row_blocks = (plan->rows + rb_rows - 1) / rb_rows;
    // persistent grid: two CTAs per SM (one when a unit holds 32 rows)
    plan->grid = device_sm_count() * (plan->m_tiles == 2 ? 1 : 2);
    // Requests per launch: the (request, row block) tables live in shared memory.
    plan->batch_per_launch = std::max(1, dec::kMaxTableEntries / plan->row_blocks);
    plan->batch_per_launch = std::min(plan->batch_per_launch, std::max(batch, 1));
    const size_t units = (size_t)plan->batch_per_launch * n_kv_heads * plan->row_blocks;
    // A launch whose keys (by the host bound) give fewer than kMinChunksPerCta
    // chunks to every CTA of the full grid launches only the CTAs that can get
    // work: the others would still be launched, plan and wait for the previous
    // kernel, and hold their SMs from the next launch meanwhile.
    {
        int64_t keys_bound = max_seq_len;
        if (window > 0) keys_bound = std::min<int64_t>(keys_bound, (int64_t)window + q_rows - 1);
        if (cache->kind == ATTN_CACHE_RING)
            keys_bound = std::min<int64_t>(keys_bound, cache->slots_per_seq);
        const int64_t chunks_bound =
            (int64_t)units * ((keys_bound + dec::kChunk - 1) / dec::kChunk + 1 + dec::kUnitGapChunks);
        const int64_t needed = (chunks_bound + dec::kMinChunksPerCta - 1) / dec::kMinChunksPerCta;
        plan->grid = (int)std::max<int64_t>(1, std::min<int64_t>(plan->grid, needed));
    }
    // partial slots: unit + cta < units + grid; one counter per unit and one
    // per partial slot (a group's counter sits at its first part's slot).
    // The counters come first, in a region sized by a bound that depends on
    // n_kv_heads and the GPU alone (units <= max(tables, row blocks) x Hkv,
    // grid <= 2 x SMs): every shape of one model then keeps its counters
    // inside the same region, which every call leaves at zero, and its
    // partial states after it, so one workspace serves calls of any shape.
    const size_t slots = units + plan->grid;
    const size_t units_bound =
        (size_t)std::max(dec::kMaxTableEntries, plan->row_blocks) * n_kv_heads;
    const size_t slots_bound = units_bound + 2 * (size_t)device_sm_count();
    plan->counter_offset = 0;
    plan->counter_bytes = ((units_bound + slots_bound) * sizeof(int32_t) + 255) & ~size_t(255);
    plan->partial_offset = plan->counter_bytes;
    const size_t partial = slots * rb_rows * ((size_t)head_dim + 1) * sizeof(float);
    plan->workspace = plan->partial_offset + partial;
    // How many CTAs can a unit span?  Its chunks are at most the key bound /
    // 16 + 1 and every CTA takes at least kMinChunksPerCta.
    int64_t keys = max_seq_len;
    if (window > 0) keys = std::min<int64_t>(keys, (int64_t)window + q_rows - 1);
    if (cache->kind == ATTN_CACHE_RING) keys = std::min<int64_t>(keys, cache->slots_per_seq);
    const int64_t max_chunks = (keys + dec::kChunk - 1) / dec::kChunk + 1;
    const int64_t max_parts = (max_chunks + dec::kMinChunksPerCta - 1) / dec::kMinChunksPerCta + 1;
    // Few units (fewer than one per kGroupParts CTAs) with more than
    // kGroupParts parts each go to the merge kernel too: two levels of
    // counters inside the split kernel cost more than the kernel boundary.
    plan->merge_kernel = max_parts > dec::kMergeKernelParts ||
                         (max_parts > dec::kGroupParts &&
                          units * dec::kGroupParts <= (size_t)plan->grid);
    // A group of 64 or more query rows (a prefill chunk) over a linear
    // slot-major bf16 cache is a dense contraction: the tcgen05 chunk kernel.
    plan->chunk = cache->kind == ATTN_CACHE_LINEAR && cache->layout == ATTN_LAYOUT_BSHD &&
                  cache->dtype == ATTN_KV_BF16 && plan->rows >= 64 && group <= 128;
    plan->chunk_offset = (plan->workspace + 255) & ~size_t(255);
    if (plan->chunk) {
        plan_chunk(batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len, window,
                   &plan->cp);
        plan->workspace = plan->chunk_offset + plan->cp.workspace;
    }
    return ATTN_OK;
}

int launch_decode(const DecodePlan &plan, const void *q, const attn_kv_cache *cache,
                  const int32_t *seq_lens, const int32_t *positions, int batch, int q_rows,
                  int max_seq_len, int window, int n_q_heads, int n_kv_heads, float scale,
                  void *out, void *workspace, int32_t *err, cudaStream_t stream,
                  const void *k_new, const void *v_new, const int64_t *slot_mapping,
                  const float *rope_inv_freq, bool tables_early, bool cache_early) {
    if (plan.chunk && rope_inv_freq == nullptr) {
        // the step's rows, when given, are fused into the chunk kernel: taken
        // from k_new / v_new and written to the cache by the same launch
        return launch_chunk(plan.cp, q, cache, seq_lens, positions, batch, q_rows, max_seq_len,
                            window, n_q_heads, n_kv_heads, plan.head_dim, scale, out,
                            static_cast<uint8_t *>(workspace) + plan.chunk_offset, err, stream,
                            k_new, v_new, slot_mapping);
    }
    // TMA maps over the caches viewed as [n_kv_heads * halves][num_slots][cols]
    // (a half is 128 bytes of one head's row: 64 bf16 or 128 E4M3 columns): a
    // box of {cols, rows, halves} brings the whole head row of `rows` slots.
    const bool fp8 = cache->dtype == ATTN_KV_FP8_E4M3;
    const int esize = fp8 ? 1 : 2;
    const int halves = plan.head_dim * esize / 128;
    const uint32_t cols = 128 / esize;
    const KvPlace place = kv_place(cache, n_kv_heads, plan.head_dim, esize);
    // rows of a whole-tile box: 64 keys (bf16), 128 (E4M3, whose tiles hold 8 chunks)
    const uint32_t tile_rows = fp8 ? 2 * dec::kTileRows : dec::kTileRows;
    CUtensorMap tk, tv, tk64, tv64;
    bool maps_ok;
    if (place.rows == 0) {
        const uint64_t dims[3] = {cols, (uint64_t)cache->num_slots, (uint64_t)n_kv_heads * halves};
        const uint64_t strides[2] = {(uint64_t)n_kv_heads * plan.head_dim * esize, 128};
        const uint32_t box[3] = {cols, (uint32_t)dec::kChunk, (uint32_t)halves};
        const uint32_t box64[3] = {cols, tile_rows, (uint32_t)halves};
        maps_ok = encode_tensor_map(&tk, cache->k, 3, dims, strides, box, true, fp8) &&
                  encode_tensor_map(&tv, cache->v, 3, dims, strides, box, true, fp8) &&
                  encode_tensor_map(&tk64, cache->k, 3, dims, strides, box64, true, fp8) &&
                  encode_tensor_map(&tv64, cache->v, 3, dims, strides, box64, true, fp8);
    } else {
        // [block * heads + head][row][half][columns], iterated {columns, row, half,
        // block-head} so a box lands as [half][rows][128 B].  Boxes taller than
        // a block are encoded at the block's height and never issued (the
        // kernel boxes only chunks and tiles that lie inside one block).
        const uint64_t row_bytes = (uint64_t)plan.head_dim * esize;
        const uint64_t rows = (uint64_t)place.rows;
        const uint64_t dims[4] = {cols, rows, (uint64_t)halves,
                                  (uint64_t)(cache->num_slots / place.rows) * n_kv_heads};
        const uint64_t strides[3] = {row_bytes, 128, rows * row_bytes};
        const uint32_t r16 = (uint32_t)std::min<uint64_t>(rows, dec::kChunk);
        const uint32_t r64 = (uint32_t)std::min<uint64_t>(rows, tile_rows);
        const uint32_t box[4] = {cols, r16, (uint32_t)halves, 1};
        const uint32_t box64[4] = {cols, r64, (uint32_t)halves, 1};
        maps_ok = encode_tensor_map(&tk, cache->k, 4, dims, strides, box, true, fp8) &&
                  encode_tensor_map(&tv, cache->v, 4, dims, strides, box, true, fp8) &&
                  encode_tensor_map(&tk64, cache->k, 4, dims, strides, box64, true, fp8) &&
                  encode_tensor_map(&tv64, cache->v, 4, dims, strides, box64, true, fp8);
    }
    if (!maps_ok) {
        note_cuda_error(cudaErrorInvalidValue);
        return ATTN_ERR_CUDA;
    }
    const int rb_rows = plan.m_tiles == 0 ? 8 : 16 * plan.m_tiles;
    const size_t units = (size_t)plan.batch_per_launch * n_kv_heads * plan.row_blocks;
    const size_t slots = units + plan.grid;
    for (int b0 = 0; b0 < batch; b0 += plan.batch_per_launch) {
        const int nb = std::min(plan.batch_per_launch, batch - b0);
        const int64_t qo = (int64_t)b0 * q_rows * n_q_heads * plan.head_dim;
        dec::Params p;
        p.q = static_cast<const __nv_bfloat16 *>(q) + qo;
        p.k_cache = static_cast<const __nv_bfloat16 *>(cache->k);
        p.v_cache = static_cast<const __nv_bfloat16 *>(cache->v);
        p.num_slots = cache->num_slots;
        p.kind = cache->kind;
        p.slots_per_seq = cache->slots_per_seq;
        p.block_table = cache->block_table
                            ? cache->block_table + (int64_t)b0 * cache->max_blocks_per_seq
                            : nullptr;
        p.block_size = cache->block_size;
        p.max_blocks = cache->max_blocks_per_seq;
        p.seq_lens = seq_lens + b0;
        p.positions = positions + (int64_t)b0 * q_rows;
        const int64_t new_off = (int64_t)b0 * q_rows * n_kv_heads * plan.head_dim;
        p.k_new = k_new ? static_cast<const __nv_bfloat16 *>(k_new) + new_off : nullptr;
        p.v_new = v_new ? static_cast<const __nv_bfloat16 *>(v_new) + new_off : nullptr;
        p.slot_mapping = slot_mapping ? slot_mapping + (int64_t)b0 * q_rows : nullptr;
        p.rope_inv_freq = rope_inv_freq;
        p.k_ref = fp8 ? cache->k_ref : nullptr;
        p.tables_early = tables_early || cache_early;
        // Early tile loads are left out when the merge kernel follows (few
        // units over long contexts): measured, they slowed those calls by 5%
        // (their DRAM traffic delays the previous call's merge, which gates
        // this call's start), while calls without it gained 5-8%.
        p.cache_early = cache_early && !plan.merge_kernel;
        p.batch = nb;
        p.b_base = b0;
        p.q_rows = q_rows;
        p.n_q_heads = n_q_heads;
        p.n_kv_heads = n_kv_heads;
        p.group = n_q_heads / n_kv_heads;
        p.rows = plan.rows;
        p.window = window;
        p.max_seq_len = max_seq_len;
        p.scale_log2 = scale * 1.4426950408889634f;
        p.row_blocks = plan.row_blocks;
        p.rb_rows = rb_rows;
        p.grid = plan.grid;
        p.out = static_cast<__nv_bfloat16 *>(out) + qo;
        p.err = err;
        p.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                           plan.partial_offset);
        p.ws_lse = p.ws_o + slots * rb_rows * plan.head_dim;
        p.ws_count = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) +
                                                 plan.counter_offset);
        p.ws_gcount = p.ws_count + units;
        p.merge_kernel = plan.merge_kernel;
        p.place = place;
        int rc;
        const bool r = rope_inv_freq != nullptr;
#define GQA_SPLIT(D, M)                                                                         \
    (r ? dec::launch_split<D, M, true, false>(p, tk, tv, tk64, tv64, stream) \
       : dec::launch_split<D, M, false, false>(p, tk, tv, tk64, tv64, stream))
#define GQA_SPLIT_FP8(M) \
    dec::launch_split<128, M, false, true>(p, tk, tv, tk64, tv64, stream)
        if (fp8)  // head_dim 128, no fused append (refused before the launch)
            rc = plan.m_tiles == 0 ? GQA_SPLIT_FP8(0)
                 : plan.m_tiles == 1 ? GQA_SPLIT_FP8(1)
                                     : GQA_SPLIT_FP8(2);
        else if (plan.head_dim == 128)
            rc = plan.m_tiles == 0 ? GQA_SPLIT(128, 0)
                 : plan.m_tiles == 1 ? GQA_SPLIT(128, 1)
                                     : GQA_SPLIT(128, 2);
        else
            rc = plan.m_tiles == 0 ? GQA_SPLIT(64, 0)
                 : plan.m_tiles == 1 ? GQA_SPLIT(64, 1)
                                     : GQA_SPLIT(64, 2);
#undef GQA_SPLIT
#undef GQA_SPLIT_FP8
        if (rc != ATTN_OK) return rc;
    }
    return ATTN_OK;
}

}  // namespace gqa
