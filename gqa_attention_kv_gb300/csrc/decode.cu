// decode.cu -- split-KV flash-decode over a linear, paged or ring KV cache.
//
// What is computed (vibevoice.c, "The kernels that matter" and "Attention
// backends"; talker_multiframe, NarrowStep fields; Voxtral Realtime notes,
// "Encoder KV cache"): for every request b, query row r and query head h,
// softmax(scale * q . k_t) over the valid key positions t, applied to v_t.
// The keys of each request are cut into splits; each split keeps an online
// softmax state (running max m, sum l, output O) and a second kernel merges
// the splits' states.  Both are exact reformulations of the softmax.
//
// GB300 mapping:
//   * One CTA = (split, KV head, row block, request).  All query rows of the
//     GQA group (q_rows x group rows, padded to 16 or 32) are the M dimension
//     of one mma.sync tile, so every cache position is read from HBM once for
//     the whole group.
//   * A producer warp streams the split's keys in tiles of 64 positions (four
//     16-position chunks) into a multi-stage shared-memory ring.  A chunk
//     whose 16 slots are consecutive (linear cache; a page of >= 16 slots; a
//     ring away from its wrap point) is one 2D TMA box per 64 columns, landing
//     128-byte-swizzled; any other chunk is gathered row by row with 16-byte
//     cp.async into the same swizzled layout.  Completion is tracked by an
//     mbarrier per stage (TMA bytes + one arrival per producer lane).
//   * Four consumer warps each own one chunk of every tile: S = Q K^T and
//     O += P V on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
//     accumulate), the mask and online softmax in fp32 registers with quad
//     shuffles, exp2 with log2(e) folded into the scale.  P enters P V as
//     two bf16 halves, hi + lo (vibevoice.c, "Attention backends": one
//     rounding of P is too coarse), so P keeps ~16 bits.
//   * The four warps' states are merged in shared memory; the CTA writes the
//     final bf16 row (one split) or an fp32 partial (O / l, m + log2 l).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gqa {
namespace dec {

constexpr int kChunk = 16;                        // key positions per chunk
constexpr int kWarps = 4;                         // consumer warps = chunks per tile
constexpr int kThreads = (kWarps + 1) * 32;       // + one producer warp
constexpr int kProducerWarp = kWarps;
constexpr int kMaxStagedPages = 512;              // page-table entries staged per CTA
constexpr int kMaxChunksPerSplit = 256;
constexpr int kStages = 3;

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
    int batch, q_rows, n_q_heads, n_kv_heads, group, rows;
    int window, max_seq_len;
    float scale_log2;
    int nsplit, row_blocks;
    __nv_bfloat16 *out;
    float *ws_o;
    float *ws_lse;
    int32_t *err;
};

template <int HD>
struct Geo {
    static constexpr int kHalves = HD / 64;                 // 128-byte column blocks
    static constexpr int kChunkBytes = kHalves * kChunk * 128;
    static constexpr int kTileBytes = kWarps * kChunkBytes;  // K (or V) of one tile
    static constexpr int kStageBytes = 2 * kTileBytes;
};

// Byte offset of 16-byte piece `c16` (0 .. HD/8-1) of row `row` inside a chunk
// laid out as [half][16 rows][128 B] with the 128-byte swizzle.
__device__ __forceinline__ uint32_t chunk_offset(int row, int c16) {
    const int half = c16 >> 3, cc = c16 & 7;
    return (uint32_t)(half * (kChunk * 128) + row * 128 + ((cc ^ (row & 7)) << 4));
}

struct SplitRange {
    int seq_len;
    int ring_lo;
    int c_begin, c_end;  // chunk range of this CTA
};

// Key range of this CTA's split.  Chunk c covers positions 16c .. 16c+15.
__device__ __forceinline__ SplitRange split_range(const Params &p, int b, int row0, int row1,
                                                  int split, bool report) {
    SplitRange s;
    int seq_len = p.seq_lens[b];
    if (seq_len > p.max_seq_len || seq_len < 0 ||
        (p.kind == ATTN_CACHE_LINEAR && seq_len > p.slots_per_seq)) {
        if (report) report_error(p.err, ATTN_ERR_BOUNDS);
        seq_len = max(0, min(seq_len, p.max_seq_len));
        if (p.kind == ATTN_CACHE_LINEAR) seq_len = min(seq_len, p.slots_per_seq);
    }
    int pmin = INT32_MAX, pmax = -1;
    for (int r = row0 / p.group; r <= (row1 - 1) / p.group; ++r) {
        const int pos = p.positions[(int64_t)b * p.q_rows + r];
        pmin = min(pmin, pos);
        pmax = max(pmax, pos);
    }
    int hi = min(seq_len, pmax + 1);
    int lo = 0;
    if (p.window > 0) lo = max(lo, pmin - p.window + 1);
    s.ring_lo = 0;
    if (p.kind == ATTN_CACHE_RING) {
        s.ring_lo = seq_len - p.slots_per_seq;
        lo = max(lo, s.ring_lo);
    }
    s.seq_len = seq_len;
    if (pmin < 0 || hi <= lo) {
        s.c_begin = s.c_end = 0;
        return s;
    }
    const int c0 = lo / kChunk, c1 = (hi + kChunk - 1) / kChunk;
    const int per = (c1 - c0 + p.nsplit - 1) / p.nsplit;
    s.c_begin = min(c1, c0 + split * per);
    s.c_end = min(c1, s.c_begin + per);
    return s;
}

template <int HD, int MT>
__global__ void __launch_bounds__(kThreads, MT == 1 ? 2 : 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using G = Geo<HD>;
    constexpr int RB = 16 * MT;  // rows per CTA
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + kStages * G::kStageBytes);
    uint64_t *empty = full + kStages;
    int *info_t0 = reinterpret_cast<int *>(empty + kStages);       // [kStages][kWarps]
    uint32_t *info_mask = reinterpret_cast<uint32_t *>(info_t0 + kStages * kWarps);
    int *pages = reinterpret_cast<int *>(info_mask + kStages * kWarps);  // [kMaxStagedPages]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.row_blocks;
    const int rb = blockIdx.y - kvh * p.row_blocks;
    const int b = blockIdx.z;
    const int row0 = rb * RB;
    const int row1 = min(p.rows, row0 + RB);

    pdl_wait();  // the cache, positions and seq_lens may come from the previous kernel
    pdl_launch_dependents();
    const SplitRange sr = split_range(p, b, row0, row1, split, threadIdx.x == 0 && split == 0);
    const int n_chunks = sr.c_end - sr.c_begin;
    const int n_tiles = (n_chunks + kWarps - 1) / kWarps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 32);       // one arrival per producer lane (+ TMA bytes)
            mbar_init(&empty[s], kWarps);  // one arrival per consumer warp
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const bool paged = p.kind == ATTN_CACHE_PAGED;
        int page0 = 0;
        bool staged = false;
        if (paged && n_chunks > 0) {
            page0 = (sr.c_begin * kChunk) / p.block_size;
            const int page1 = (sr.c_end * kChunk - 1) / p.block_size;
            const int np = page1 - page0 + 1;
            staged = np <= kMaxStagedPages;
            if (staged) {
                const int32_t *bt = p.block_table + (int64_t)b * p.max_blocks;
                for (int i = lane; i < np; i += 32) {
                    const int pi = page0 + i;
                    pages[i] = pi < p.max_blocks ? bt[pi] : -1;
                }
            }
            __syncwarp();
        }
        const int64_t num_pages = paged ? p.num_slots / p.block_size : 0;
        auto page_of = [&](int t) -> int64_t {  // page id holding position t, or -1
            const int pi = t / p.block_size;
            if (pi >= p.max_blocks) return -1;
            const int v = staged ? pages[pi - page0]
                                 : p.block_table[(int64_t)b * p.max_blocks + pi];
            return (v < 0 || v >= num_pages) ? -1 : (int64_t)v;
        };
        // slot of position t, or -1 if it is out of bounds
        auto slot_of = [&](int t) -> int64_t {
            int64_t s;
            if (p.kind == ATTN_CACHE_LINEAR) {
                s = (int64_t)b * p.slots_per_seq + t;
            } else if (paged) {
                const int64_t pg = page_of(t);
                if (pg < 0) return -1;
                s = pg * p.block_size + t % p.block_size;
            } else {
                s = (int64_t)b * p.slots_per_seq + t % p.slots_per_seq;
            }
            return (s >= 0 && s < p.num_slots) ? s : -1;
        };
        const int64_t row_elems = (int64_t)p.n_kv_heads * HD;
        bool ok = true;
        for (int it = 0; it < n_tiles && ok; ++it) {
            const int st = it % kStages;
            if (it >= kStages) ok = mbar_wait(&empty[st], ((it / kStages) - 1) & 1, p.err);
            if (!ok) break;
            uint8_t *kst = stages + st * G::kStageBytes;
            uint8_t *vst = kst + G::kTileBytes;
            // Describe the tile's chunks: a chunk whose 16 slots are
            // consecutive starts at slot0[c] >= 0 (one TMA box per 64
            // columns); slot0[c] == -1 marks a contiguous chunk whose page is
            // out of bounds (the box is aimed outside the tensor, zero-filled,
            // and its keys masked); slot0[c] == -2 is gathered row by row.
            int64_t slot0[kWarps];
            uint32_t tma_bytes = 0;
            bool issued_cp = false;
#pragma unroll
            for (int c = 0; c < kWarps; ++c) {
                const int chunk = sr.c_begin + it * kWarps + c;
                slot0[c] = -3;  // absent
                if (chunk >= sr.c_end) {
                    if (lane == 0) info_t0[st * kWarps + c] = -1;
                    continue;
                }
                const int t0 = chunk * kChunk;
                int64_t s0 = -2;
                if (p.kind == ATTN_CACHE_LINEAR) {
                    s0 = (int64_t)b * p.slots_per_seq + t0;
                } else if (paged) {
                    if (p.block_size % kChunk == 0) {
                        const int64_t pg = page_of(t0);
                        s0 = pg < 0 ? -1 : pg * p.block_size + t0 % p.block_size;
                    }
                } else {
                    const int j0 = t0 % p.slots_per_seq;
                    if (j0 + kChunk <= p.slots_per_seq) s0 = (int64_t)b * p.slots_per_seq + j0;
                }
                slot0[c] = s0;
                uint32_t mask;
                if (s0 != -2) {
                    mask = 0xFFFFu;
                    if (s0 == -1) {
                        mask = 0;
                        if (t0 < sr.seq_len) report_error(p.err, ATTN_ERR_BOUNDS);
                    }
                    tma_bytes += 2 * G::kChunkBytes;
                } else {
                    mask = 0;
                    for (int r = 0; r < kChunk; ++r) {
                        const int64_t s = slot_of(t0 + r);
                        if (s >= 0) mask |= 1u << r;
                        else if (t0 + r < sr.seq_len) report_error(p.err, ATTN_ERR_BOUNDS);
                    }
                    if (lane != 0) {
                        // lanes 1..31 gather the chunk's K and V rows
                        constexpr int kPieces = kChunk * (HD / 8);
                        for (int pc = lane - 1; pc < 2 * kPieces; pc += 31) {
                            const int tensor = pc / kPieces;
                            const int rem = pc - tensor * kPieces;
                            const int r = rem / (HD / 8), c16 = rem % (HD / 8);
                            int64_t s = slot_of(t0 + r);
                            if (s < 0) s = 0;  // masked row: read any valid slot
                            const __nv_bfloat16 *src = (tensor ? p.v_cache : p.k_cache) +
                                                       s * row_elems + (int64_t)kvh * HD + c16 * 8;
                            uint8_t *dst =
                                (tensor ? vst : kst) + c * G::kChunkBytes + chunk_offset(r, c16);
                            cp_async_16(dst, src);
                            issued_cp = true;
                        }
                    }
                }
                if (lane == 0) {
                    info_t0[st * kWarps + c] = t0;
                    info_mask[st * kWarps + c] = mask;
                }
            }
            if (lane == 0) {
                if (tma_bytes) mbar_expect_tx(&full[st], tma_bytes);
#pragma unroll
                for (int c = 0; c < kWarps; ++c) {
                    if (slot0[c] < -1) continue;
                    const int y = slot0[c] < 0 ? -kChunk : (int)slot0[c];
#pragma unroll
                    for (int h = 0; h < G::kHalves; ++h) {
                        const int x = kvh * HD + h * 64;
                        tma_load_2d(kst + c * G::kChunkBytes + h * kChunk * 128, &tm_k, x, y,
                                    &full[st]);
                        tma_load_2d(vst + c * G::kChunkBytes + h * kChunk * 128, &tm_v, x, y,
                                    &full[st]);
                    }
                }
                mbar_arrive(&full[st]);
            } else if (issued_cp) {
                cp_async_arrive_noinc(&full[st]);
            } else {
                mbar_arrive(&full[st]);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int gq = lane >> 2, tq = lane & 3;
        uint32_t qa[MT][HD / 16][4];
        int rpos[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int i = row0 + mt * 16 + gq + hr * 8;
                const bool valid = i < row1;
                const int r = valid ? i / p.group : 0;
                const int g = valid ? i - r * p.group : 0;
                rpos[mt][hr] = valid ? p.positions[(int64_t)b * p.q_rows + r] : -1;
                const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                    p.q + (((int64_t)b * p.q_rows + r) * p.n_q_heads + kvh * p.group + g) * HD);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    qa[mt][kk][hr] = valid ? __ldg(qrow + kk * 8 + tq) : 0u;
                    qa[mt][kk][2 + hr] = valid ? __ldg(qrow + kk * 8 + 4 + tq) : 0u;
                }
            }
        }
        float m_run[MT][2], l_run[MT][2];
        float o[MT][HD / 8][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            m_run[mt][0] = m_run[mt][1] = -INFINITY;
            l_run[mt][0] = l_run[mt][1] = 0.f;
#pragma unroll
            for (int n = 0; n < HD / 8; ++n) o[mt][n][0] = o[mt][n][1] = o[mt][n][2] = o[mt][n][3] = 0.f;
        }
        const int seq_len = sr.seq_len, ring_lo = sr.ring_lo, window = p.window;
        bool ok = true;
        for (int it = 0; it < n_tiles && ok; ++it) {
            const int st = it % kStages;
            ok = mbar_wait(&full[st], (it / kStages) & 1, p.err);
            __syncwarp();  // reconverge before the warp-collective ldmatrix / mma
            if (!ok) break;
            const int t0 = info_t0[st * kWarps + warp];
            if (t0 >= 0) {
                const uint32_t mask16 = info_mask[st * kWarps + warp];
                const uint32_t kbase = smem_u32(stages + st * G::kStageBytes + warp * G::kChunkBytes);
                const uint32_t vbase = kbase + G::kTileBytes;
                float s[MT][2][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) s[mt][j][0] = s[mt][j][1] = s[mt][j][2] = s[mt][j][3] = 0.f;
                {
                    const int m = lane >> 3;
                    const int key = (m >> 1) * 8 + (lane & 7);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        uint32_t b00, b01, b10, b11;
                        ldmatrix_x4(b00, b01, b10, b11, kbase + chunk_offset(key, kk * 2 + (m & 1)));
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            mma_bf16_16816(s[mt][0], qa[mt][kk], b00, b01);
                            mma_bf16_16816(s[mt][1], qa[mt][kk], b10, b11);
                        }
                    }
                }
                uint32_t pa[MT][4], pl[MT][4];  // P as bf16 hi + lo
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int pos = rpos[mt][hr];
                        float mx = -INFINITY;
#pragma unroll
                        for (int j = 0; j < 2; ++j)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int n = j * 8 + tq * 2 + e;
                                const int t = t0 + n;
                                const bool valid = ((mask16 >> n) & 1u) && t < seq_len && t <= pos &&
                                                   t >= ring_lo && (window <= 0 || pos - t < window);
                                const float v = valid ? s[mt][j][hr * 2 + e] * p.scale_log2 : -INFINITY;
                                s[mt][j][hr * 2 + e] = v;
                                mx = fmaxf(mx, v);
                            }
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                        const float m_new = fmaxf(m_run[mt][hr], mx);
                        const float m_use = m_new == -INFINITY ? 0.f : m_new;
                        const float alpha = fast_exp2(m_run[mt][hr] - m_use);
                        float sum = 0.f;
#pragma unroll
                        for (int j = 0; j < 2; ++j)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float pv = fast_exp2(s[mt][j][hr * 2 + e] - m_use);
                                s[mt][j][hr * 2 + e] = pv;
                                sum += pv;
                            }
                        l_run[mt][hr] = l_run[mt][hr] * alpha + sum;
                        m_run[mt][hr] = m_new;
#pragma unroll
                        for (int n = 0; n < HD / 8; ++n) {
                            o[mt][n][hr * 2] *= alpha;
                            o[mt][n][hr * 2 + 1] *= alpha;
                        }
                    }
                    split_bf16x2(s[mt][0][0], s[mt][0][1], pa[mt][0], pl[mt][0]);
                    split_bf16x2(s[mt][0][2], s[mt][0][3], pa[mt][1], pl[mt][1]);
                    split_bf16x2(s[mt][1][0], s[mt][1][1], pa[mt][2], pl[mt][2]);
                    split_bf16x2(s[mt][1][2], s[mt][1][3], pa[mt][3], pl[mt][3]);
                }
                {
                    const int m = lane >> 3;
                    const int key = (m & 1) * 8 + (lane & 7);
#pragma unroll
                    for (int dn = 0; dn < HD / 16; ++dn) {
                        uint32_t v0, v1, v2, v3;
                        ldmatrix_x4_trans(v0, v1, v2, v3, vbase + chunk_offset(key, dn * 2 + (m >> 1)));
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
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        // quad-reduce the row sums
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float l = l_run[mt][hr];
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                l_run[mt][hr] = l;
            }
        __syncwarp();
        __syncthreads();  // (1) all stages consumed: the stage memory is free
        float *mo = reinterpret_cast<float *>(stages);          // [kWarps][RB][HD]
        float *mm = mo + kWarps * RB * HD;                       // [kWarps][RB]
        float *ml = mm + kWarps * RB;                            // [kWarps][RB]
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = mt * 16 + gq + hr * 8;
                float *dst = mo + ((size_t)warp * RB + row) * HD;
#pragma unroll
                for (int n = 0; n < HD / 8; ++n) {
                    *reinterpret_cast<float2 *>(dst + n * 8 + tq * 2) =
                        make_float2(o[mt][n][hr * 2], o[mt][n][hr * 2 + 1]);
                }
                if (tq == 0) {
                    mm[warp * RB + row] = m_run[mt][hr];
                    ml[warp * RB + row] = l_run[mt][hr];
                }
            }
        asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");  // consumers only
        // combine the four warps and write the CTA's result
        const int ctid = threadIdx.x;  // 0 .. 127
        for (int idx = ctid; idx < RB * (HD / 4); idx += kWarps * 32) {
            const int row = idx / (HD / 4), d = (idx % (HD / 4)) * 4;
            const int i = row0 + row;
            if (i >= row1) continue;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * RB + row]);
            float L = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float mw = mm[w * RB + row];
                    if (mw == -INFINITY) continue;
                    const float f = fast_exp2(mw - M);
                    L += ml[w * RB + row] * f;
                    const float4 v = *reinterpret_cast<const float4 *>(mo + ((size_t)w * RB + row) * HD + d);
                    acc.x += f * v.x;
                    acc.y += f * v.y;
                    acc.z += f * v.z;
                    acc.w += f * v.w;
                }
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const int r = i / p.group, g = i - (i / p.group) * p.group;
            if (p.nsplit == 1) {
                __nv_bfloat16 *dst =
                    p.out + (((int64_t)b * p.q_rows + r) * p.n_q_heads + kvh * p.group + g) * HD + d;
                uint2 packed;
                packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                *reinterpret_cast<uint2 *>(dst) = packed;
            } else {
                const int64_t unit = ((int64_t)b * p.n_kv_heads + kvh) * p.row_blocks + rb;
                const int64_t slot = (unit * p.nsplit + split) * RB + row;
                *reinterpret_cast<float4 *>(p.ws_o + slot * HD + d) =
                    make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                if (d == 0) p.ws_lse[slot] = L > 0.f ? M + __log2f(L) : -INFINITY;
            }
        }
        return;
    }
    __syncwarp();
    __syncthreads();  // producer's side of barrier (1)
}

// Merge the splits' partial states.  One CTA per (request, KV head, query
// row of the group); its warps take the splits round-robin, each keeping an
// online (max, sum, output) state, and the warps' states are combined in a
// fixed order, so the result does not depend on timing.
constexpr int kMergeWarps = 8;

template <int HD, int RB>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const Params p) {
    constexpr int PER = HD / 32;
    __shared__ float sm_m[kMergeWarps], sm_l[kMergeWarps];
    __shared__ __align__(16) float sm_o[kMergeWarps][HD];
    pdl_wait();  // the partial states come from the split kernel
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int b = cta / (p.rows * p.n_kv_heads);
    const int rem = cta - b * p.rows * p.n_kv_heads;
    const int kvh = rem / p.rows;
    const int i = rem - kvh * p.rows;
    const int rb = i / RB, row = i - rb * RB;
    const int64_t unit = ((int64_t)b * p.n_kv_heads + kvh) * p.row_blocks + rb;
    const int64_t base = unit * p.nsplit * RB + row;  // slot of split s: base + s*RB
    float m = -INFINITY, l = 0.f;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int s = warp; s < p.nsplit; s += kMergeWarps) {
        const int64_t slot = base + (int64_t)s * RB;
        const float lse = p.ws_lse[slot];
        float v[PER];
        const float *src = p.ws_o + slot * HD + lane * PER;
        if constexpr (PER == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(src);
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2 *>(src);
            v[0] = t.x; v[1] = t.y;
        }
        if (lse == -INFINITY) continue;
        if (lse > m) {
            const float f = fast_exp2(m - lse);
            l *= f;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] *= f;
            m = lse;
        }
        const float f = fast_exp2(lse - m);
        l += f;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] += f * v[e];
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
    float L = 0.f;
    float o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            if (sm_m[w] == -INFINITY) continue;
            const float f = fast_exp2(sm_m[w] - M);
            L += f * sm_l[w];
#pragma unroll
            for (int e = 0; e < PER; ++e) o[e] += f * sm_o[w][lane * PER + e];
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
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

template <int HD>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)kStages * Geo<HD>::kStageBytes + 2 * kStages * sizeof(uint64_t) +
           2 * kStages * kWarps * sizeof(int) + kMaxStagedPages * sizeof(int);
}

template <int HD, int MT>
int launch_split(const Params &p, const CUtensorMap &tk, const CUtensorMap &tv,
                 cudaStream_t stream) {
    static_assert(kStages * Geo<HD>::kStageBytes >=
                      (size_t)kWarps * 16 * MT * HD * 4 + 2 * kWarps * 16 * MT * 4,
                  "merge area must fit in the stage memory");
    auto kern = decode_split_kernel<HD, MT>;
    const size_t smem = smem_bytes<HD>();
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
    dim3 grid(p.nsplit, p.n_kv_heads * p.row_blocks, p.batch);
    if (launch_pdl(kern, grid, dim3(kThreads), smem, stream, tk, tv, p) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (p.nsplit > 1) {
        const unsigned ctas = (unsigned)((int64_t)p.batch * p.rows * p.n_kv_heads);
        if (launch_pdl(decode_merge_kernel<HD, 16 * MT>, dim3(ctas), dim3(kMergeWarps * 32), 0,
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
    plan->m_tiles = plan->rows <= 16 ? 1 : 2;
    const int rb_rows = 16 * plan->m_tiles;
    plan->row_blocks = (plan->rows + rb_rows - 1) / rb_rows;
    // Longest key range one request can need.
    int64_t keys = max_seq_len;
    if (window > 0) keys = std::min<int64_t>(keys, (int64_t)window + q_rows - 1);
    if (cache->kind == ATTN_CACHE_RING) keys = std::min<int64_t>(keys, cache->slots_per_seq);
    const int64_t max_chunks = (keys + dec::kChunk - 1) / dec::kChunk + 1;
    const int64_t units = (int64_t)batch * n_kv_heads * plan->row_blocks;
    const int64_t slots = (int64_t)device_sm_count() * 2;  // two CTAs per SM
    // At least two waves of CTAs, each split >= 4 chunks (64 keys) and
    // <= kMaxChunksPerSplit chunks; then round up to fill the last wave.
    int64_t lo = (max_chunks + dec::kMaxChunksPerSplit - 1) / dec::kMaxChunksPerSplit;
    int64_t hi = std::max<int64_t>(1, max_chunks / 4);
    hi = std::max(hi, lo);
    int64_t n = (2 * slots + units - 1) / std::max<int64_t>(units, 1);
    n = std::min(std::max(n, lo), hi);
    if (n > 1) {
        int64_t best = n;
        double best_eff = 0.0;
        for (int64_t c = n; c <= std::min<int64_t>(hi, 2 * n); ++c) {
            const double w = (double)(units * c) / (double)slots;
            const double eff = w / std::ceil(w);
            if (eff > best_eff + 1e-9) {
                best_eff = eff;
                best = c;
            }
        }
        n = best;
    }
    plan->nsplit = (int)n;
    plan->workspace =
        n > 1 ? (size_t)units * n * rb_rows * ((size_t)head_dim + 1) * sizeof(float) + 256 : 0;
    return ATTN_OK;
}

int launch_decode(const DecodePlan &plan, const void *q, const attn_kv_cache *cache,
                  const int32_t *seq_lens, const int32_t *positions, int batch, int q_rows,
                  int max_seq_len, int window, int n_q_heads, int n_kv_heads, float scale,
                  void *out, void *workspace, int32_t *err, cudaStream_t stream) {
    dec::Params p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_cache = static_cast<const __nv_bfloat16 *>(cache->k);
    p.v_cache = static_cast<const __nv_bfloat16 *>(cache->v);
    p.num_slots = cache->num_slots;
    p.kind = cache->kind;
    p.slots_per_seq = cache->slots_per_seq;
    p.block_table = cache->block_table;
    p.block_size = cache->block_size;
    p.max_blocks = cache->max_blocks_per_seq;
    p.seq_lens = seq_lens;
    p.positions = positions;
    p.batch = batch;
    p.q_rows = q_rows;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = n_q_heads / n_kv_heads;
    p.rows = plan.rows;
    p.window = window;
    p.max_seq_len = max_seq_len;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.nsplit = plan.nsplit;
    p.row_blocks = plan.row_blocks;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.err = err;
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    if (plan.nsplit > 1) {
        const int rb_rows = 16 * plan.m_tiles;
        const size_t units = (size_t)batch * n_kv_heads * plan.row_blocks;
        const size_t entries = units * plan.nsplit * rb_rows;
        p.ws_o = static_cast<float *>(workspace);
        p.ws_lse = p.ws_o + entries * plan.head_dim;
    }
    // TMA maps over the caches viewed as [num_slots, n_kv_heads * head_dim].
    CUtensorMap tk, tv;
    const uint64_t dims[2] = {(uint64_t)n_kv_heads * plan.head_dim, (uint64_t)cache->num_slots};
    const uint64_t strides[1] = {(uint64_t)n_kv_heads * plan.head_dim * 2};
    const uint32_t box[2] = {64, (uint32_t)dec::kChunk};
    if (!encode_tensor_map(&tk, cache->k, 2, dims, strides, box, true) ||
        !encode_tensor_map(&tv, cache->v, 2, dims, strides, box, true))
        return ATTN_ERR_CUDA;
    if (plan.head_dim == 128)
        return plan.m_tiles == 1 ? dec::launch_split<128, 1>(p, tk, tv, stream)
                                 : dec::launch_split<128, 2>(p, tk, tv, stream);
    return plan.m_tiles == 1 ? dec::launch_split<64, 1>(p, tk, tv, stream)
                             : dec::launch_split<64, 2>(p, tk, tv, stream);
}

}  // namespace gqa
