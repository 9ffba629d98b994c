// chunk.cu -- a prefill chunk against a linear KV cache on tcgen05 tensor cores.
//
// What is computed (vibevoice.c, "Prefill attention" and its streaming
// backend, which feeds the decoder 29 prompt rows at a time; talker_multiframe,
// NarrowStep fields: several query rows per request at positions[r]): for
// request b, chunk row r at position positions[b*R + r] and query head h, the
// softmax over keys t <= position (t < seq_lens[b]; i - t < window when one is
// set) of scale * q . k_t applied to v_t, with KV head h / G.  It is the
// K-row decode of the same arguments; this kernel serves it when the rows of
// one KV group are many (R x G >= 64) and the cache is linear and slot-major.
//
// GB300 mapping.  The R x G query rows of one (request, KV head) are packed
// into the M dimension of 128-row tcgen05 tiles: tile row m holds chunk row
// m / G of the tile's rows and group head m % G, so every K/V tile of the
// group is loaded once for all its heads and rows (G rows per position; 128 /
// G positions per tile, the remaining rows padding).  A CTA takes two such
// tiles and a range of key tiles: the key range of a (request, KV head) is
// split over CTAs so that the few groups of a chunk still fill the GPU; each
// CTA leaves a partial state per row (O / l in f16 and the base-2 log-sum-
// exp in fp32), and chunk_merge_kernel combines the splits in a fixed order.
// One split writes the bf16 rows itself.  Under attn_decode_append the step's
// own rows are taken from k_new / v_new and written to the cache by the same
// launch.
//
// The warp roles, rings, TMEM columns and the ping-pong of the two tiles are
// those of the prefill kernel (prefill.cu): warp 0 issues TMA, warp 1 the
// tcgen05.mma (S_a = Q_a K^T in bf16, O_a += P_a V in f16 with P rounded once
// and V rewritten to f16 in shared memory by warps 2 and 3), warps 4..11 run
// the softmax of one tile row per thread.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace gqa {
namespace chk {

constexpr int kBM = 128;       // rows per tile (two tiles per CTA)
constexpr int kBN = 128;       // keys per tile
constexpr int kThreads = 384;  // 3 warpgroups
// Registers: launched at 168 a thread, the TMA / MMA / V-conversion warpgroup
// drops to 96 and the two softmax warpgroups rise to 200 (4x32x96 + 8x32x200 =
// 63,488 <= 384x168; 96 + 200 + 200 <= 512 per sub-partition lane slot).  This
// split spills the least of those measured (88 / 208 reloaded 224 bytes).
constexpr uint32_t kRegsControl = 96;
constexpr uint32_t kRegsSoftmax = 200;
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMergeWarps = 8;

template <int HD>
struct Cfg {
    static constexpr int kHalves = HD / 64;
    // rings: three K stages, two V (measured 1.4% faster than two and three at
    // D = 128; K's depth gates how far ahead the tiles are requested)
    static constexpr int kKStages = HD == 128 ? 3 : 4;
    static constexpr int kVStages = HD == 128 ? 2 : 4;
    static constexpr int kQBytes = kBM * HD * 2;  // one Q tile
    static constexpr int kKBytes = kBN * HD * 2;
    static constexpr int kVBytes = kBN * HD * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKBytes;
    static constexpr int kOffBar = kOffV + kVStages * kVBytes;
    static constexpr int kNumBars = 2 * kKStages + 3 * kVStages + 10;
    static constexpr size_t kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
};

struct Params {
    int batch, q_rows, window, n_kv_heads, group, head_dim;
    int rt;       // chunk rows per tile: 128 / group
    int n_pairs;  // tile pairs along the chunk rows
    int n_split;  // CTAs along the key range of one (request, KV head, pair)
    int slots_per_seq, max_seq_len;
    const int32_t *seq_lens;   // [batch]
    const int32_t *positions;  // [batch * q_rows]
    float scale_log2;
    uint16_t *ws_o;  // n_split > 1: [slot][256][HD] f16, slot = ((b*Hkv + kvh)*pairs + pair)*splits + s
    float *ws_lse;   // [slot][256]
    __nv_bfloat16 *out;  // [batch, q_rows, n_q_heads, HD]
    // The step's own rows (fused append), or null: row b * q_rows + r is the
    // key at position seq_lens[b] - q_rows + r; its slot is slot_mapping[row].
    const __nv_bfloat16 *k_new, *v_new;  // [batch * q_rows, Hkv, HD]
    const int64_t *slot_mapping;
    int64_t num_slots;
    __nv_bfloat16 *k_cache, *v_cache;  // linear slot-major: slot s, head h at (s * Hkv + h) * HD
    int32_t *err;
};

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            int w, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// The request's keys: seq_lens[b], range-checked as the decode checks it.
__device__ __forceinline__ int request_keys(const Params &p, int b, bool report) {
    int n = p.seq_lens[b];
    if (n < 0 || n > p.max_seq_len || n > p.slots_per_seq) {
        if (report) report_error(p.err, ATTN_ERR_BOUNDS);
        n = max(0, min(n, min(p.max_seq_len, p.slots_per_seq)));
    }
    return n;
}

// Key tiles [kt0, kt0 + n_kt) of split s for the rows whose positions span
// [p_lo, p_hi] of a request holding n_keys keys.
__device__ __forceinline__ void split_range(const Params &p, int p_lo, int p_hi, int n_keys,
                                            int s, int &kt0, int &n_kt) {
    const int key_hi = min(n_keys, p_hi + 1);
    const int key_lo = p.window > 0 ? max(0, p_lo - p.window + 1) : 0;
    const int lo = key_lo / kBN;
    const int hi = key_hi > key_lo ? (key_hi + kBN - 1) / kBN : lo;
    const int per = (hi - lo + p.n_split - 1) / p.n_split;
    kt0 = lo + s * per;
    n_kt = max(0, min(per, hi - kt0));
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_ws,
                 const Params p) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *k_full = bars;                   // [kKStages]
    uint64_t *k_empty = k_full + C::kKStages;  // [kKStages]
    uint64_t *v_full = k_empty + C::kKStages;  // [kVStages]
    uint64_t *v_empty = v_full + C::kVStages;  // [kVStages]
    uint64_t *q_full = v_empty + C::kVStages;
    uint64_t *s_full = q_full + 1;  // [2]
    uint64_t *p_full = s_full + 2;  // [2 tiles][2 key halves]
    uint64_t *o_done = p_full + 4;
    uint64_t *mma_done = o_done + 1;
    uint64_t *v_conv = mma_done + 1;  // [kVStages]: V tile now f16
    uint64_t *k_patch = v_conv + C::kVStages;  // a K tile holding the step's rows is patched
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
    __shared__ int s_pos[2];  // min and max position of the CTA's rows

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // block: ((b * Hkv + kvh) * n_split + split) * n_pairs + pair
    const int pair = (int)(blockIdx.x % p.n_pairs);
    int rest = (int)(blockIdx.x / p.n_pairs);
    const int split = rest % p.n_split;
    rest /= p.n_split;
    const int kvh = rest % p.n_kv_heads;
    const int b = rest / p.n_kv_heads;
    const int G = p.group, R = p.q_rows;
    const int r_first = pair * 2 * p.rt;                 // first chunk row of the pair
    const int r_end = min(R, r_first + 2 * p.rt);        // one past its last
    const int used = p.rt * G;                           // tile rows that hold queries

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
            mbar_init(&v_conv[s], 64);  // every thread of warps 2 and 3
        }
        mbar_init(q_full, 1);
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&p_full[i], 128);
        mbar_init(o_done, 1);
        mbar_init(mma_done, 1);
        mbar_init(k_patch, 64);  // every thread of warps 2 and 3
        fence_barrier_init();
        s_pos[0] = INT32_MAX;
        s_pos[1] = -1;
    }
    // Tile rows past the packed queries are never written by TMA: zero them
    // (generic stores, made visible to the tensor core's proxy below).
    if (used < kBM) {
        for (int i = threadIdx.x; i < 2 * C::kHalves * (kBM - used) * 8; i += kThreads) {
            const int piece = i & 7, row = used + (i >> 3) % (kBM - used);
            const int th = (i >> 3) / (kBM - used);  // tile * halves + half
            *reinterpret_cast<uint4 *>(sQ + th * (kBM * 128) + row * 128 + piece * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // q, the cache, seq_lens and positions may come from the previous kernel
    pdl_launch_dependents();
    // the span of positions of the pair's rows (bounds the key range)
    for (int r = r_first + (int)threadIdx.x; r < r_end; r += kThreads) {
        const int pos = p.positions[(int64_t)b * R + r];
        atomicMin(&s_pos[0], pos);
        atomicMax(&s_pos[1], pos);
    }
    const int n_keys = request_keys(p, b, kvh == 0 && split == 0 && pair == 0 && threadIdx.x == 0);
    __syncthreads();
    int kt0, n_kt;
    split_range(p, s_pos[0], s_pos[1], n_keys, split, kt0, n_kt);
    const uint32_t tmem = *tmem_slot;
    // With the step's rows fused in, the keys at positions new_lo .. n_keys - 1
    // come from k_new / v_new: a K or V tile holding any of them is patched in
    // shared memory after its copy lands (the cache may still hold older rows
    // there: this launch writes them for later steps).
    const bool fused = p.k_new != nullptr;
    const int new_lo = n_keys - R;
    auto tile_new = [&](int j) {
        const int key0 = (kt0 + j) * kBN;
        return fused && key0 < n_keys && key0 + kBN > new_lo;
    };

    if (warp < 4) {
    setmaxnreg_dec<kRegsControl>();
    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            // both tiles' boxes of rt positions x G heads x 64 columns (rows
            // past the chunk's end are zero-filled by the copy)
            mbar_arrive_expect_tx(q_full, 2 * C::kHalves * used * 128);
            for (int a = 0; a < 2; ++a)
                for (int hf = 0; hf < C::kHalves; ++hf)
                    tma_load_4d(sQ + a * C::kQBytes + hf * (kBM * 128), &tm_q, hf * 64, kvh * G,
                                r_first + a * p.rt, b, q_full);
            int kj = 0, vj = 0;
            bool ok = true;
            while (ok && (kj < n_kt || vj < n_kt)) {
                if (kj < n_kt && (kj <= vj + 1 || vj >= n_kt)) {
                    const int st = kj % C::kKStages;
                    if (kj >= C::kKStages)
                        ok = mbar_wait(&k_empty[st], ((kj / C::kKStages) - 1) & 1, p.err);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&k_full[st], C::kKBytes);
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(sK + st * C::kKBytes + hf * (kBN * 128), &tm_k,
                                    kvh * HD + hf * 64, (kt0 + kj) * kBN, b, &k_full[st]);
                    ++kj;
                } else {
                    const int st = vj % C::kVStages;
                    if (vj >= C::kVStages)
                        ok = mbar_wait(&v_empty[st], ((vj / C::kVStages) - 1) & 1, p.err);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&v_full[st], C::kVBytes);
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(sV + st * C::kVBytes + hf * (kBN * 128), &tm_v,
                                    kvh * HD + hf * 64, (kt0 + vj) * kBN, b, &v_full[st]);
                    ++vj;
                }
            }
            // No copy may still be landing when the CTA exits: the last K and
            // V tile of each stage have completed (normally the MMAs have
            // read them already; after a wait that gave up, bounded too).
            bool landed = true;
            for (int j = max(0, kj - C::kKStages); landed && j < kj; ++j)
                landed = mbar_wait(&k_full[j % C::kKStages], (j / C::kKStages) & 1, p.err);
            for (int j = max(0, vj - C::kVStages); landed && j < vj; ++j)
                landed = mbar_wait(&v_full[j % C::kVStages], (j / C::kVStages) & 1, p.err);
            if (landed) mbar_wait(q_full, 0, p.err);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_f16_f32(kBM, HD, 0, 1);
            const uint64_t q_desc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t k_desc0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t v_desc0 = smem_desc_sw128(smem_u32(sV), kBN * 128, 1024);
            auto issue_qk = [&](int a, int kst) {
                const uint64_t qd = q_desc + (uint64_t)((a * C::kQBytes) >> 4);
                const uint64_t kd = k_desc0 + (uint64_t)((kst * C::kKBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
                    tc_mma_ss(tmem + a * 128, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[a]);
            };
            auto issue_pv_half = [&](int a, int vst, int hh, bool first) {
                const uint64_t vd = v_desc0 + (uint64_t)((vst * C::kVBytes) >> 4);
                const uint32_t p_tmem = tmem + a * 128;
                const uint32_t o_tmem = tmem + 256 + a * HD;
#pragma unroll
                for (int k4 = 0; k4 < kBN / 32; ++k4) {
                    const int kk = hh * (kBN / 32) + k4;
                    tc_mma_ts(o_tmem, p_tmem + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4),
                              idesc_pv, (!first || k4 > 0) ? 1u : 0u);
                }
            };
            // K tile j is ready when its copy lands or, holding the step's
            // rows, when warps 2 and 3 have patched them in (k_patch completes
            // once per such tile, in tile order)
            int n_patched = 0;
            auto k_ready = [&](int j, int st, int ph) -> bool {
                if (!tile_new(j)) return mbar_wait(&k_full[st], ph, p.err);
                return mbar_wait(k_patch, (n_patched++) & 1, p.err);
            };
            bool ok = mbar_wait(q_full, 0, p.err) && (n_kt == 0 || k_ready(0, 0, 0));
            if (ok && n_kt > 0) {
                tc_fence_after();
                issue_qk(0, 0);
                issue_qk(1, 0);
                tc_commit(&k_empty[0]);
            }
            int vst = 0, vph = 0, kst = 0, kph = 0;
            for (int j = 0; j < n_kt && ok; ++j) {
                ok = mbar_wait(&v_conv[vst], vph, p.err);  // V(j) landed and is f16
                const bool more = j + 1 < n_kt;
                if (more && ++kst == C::kKStages) {
                    kst = 0;
                    kph ^= 1;
                }
                for (int a = 0; a < 2 && ok; ++a) {
                    for (int hh = 0; hh < 2 && ok; ++hh) {
                        ok = mbar_wait(&p_full[a * 2 + hh], j & 1, p.err);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv_half(a, vst, hh, j == 0 && hh == 0);
                    }
                    if (!ok) break;
                    if (a == 1) tc_commit(&v_empty[vst]);
                    if (more) {
                        if (a == 0) {
                            ok = k_ready(j + 1, kst, kph);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        issue_qk(a, kst);
                        if (a == 1) tc_commit(&k_empty[kst]);
                    }
                }
                if (++vst == C::kVStages) {
                    vst = 0;
                    vph ^= 1;
                }
            }
            tc_commit(o_done);
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, p.err);
        }
    } else {
        // ---------------------------------------------------------- V to f16
        // as in the prefill kernel: each V tile rewritten in place, a
        // magnitude of 2^16 or more saturated and reported.  A tile holding
        // the step's rows takes them from k_new / v_new: K as soon as its
        // copy lands (every thread patches its share, fences and arrives on
        // k_patch, which the MMA warp waits for instead), V after the
        // conversion, each thread over the pieces it has just converted
        // itself (piece i of a tile is thread i % 64's), so no thread waits
        // for another.
        const int ct = threadIdx.x - 64;  // 0 .. 63
        if (fused) {
            // The step's rows into the cache for later steps (this launch
            // reads them from k_new / v_new), before the first V tile lands:
            // rows blockIdx.x, + gridDim.x, ..., each tensor's row a run of
            // 16-byte pieces at its slot.
            const int64_t n_new = (int64_t)p.batch * R;
            const int pieces = p.n_kv_heads * HD / 8;
            for (int64_t row = blockIdx.x; row < n_new; row += gridDim.x) {
                const int64_t slot = p.slot_mapping[row];
                if (slot < 0 || slot >= p.num_slots) {
                    if (ct == 0) report_error(p.err, ATTN_ERR_BOUNDS);
                    continue;
                }
                const uint4 *ks = reinterpret_cast<const uint4 *>(p.k_new) + row * pieces;
                const uint4 *vs = reinterpret_cast<const uint4 *>(p.v_new) + row * pieces;
                uint4 *kd = reinterpret_cast<uint4 *>(p.k_cache) + slot * pieces;
                uint4 *vd = reinterpret_cast<uint4 *>(p.v_cache) + slot * pieces;
                for (int pc = ct; pc < pieces; pc += 64) {
                    kd[pc] = __ldg(ks + pc);
                    vd[pc] = __ldg(vs + pc);
                }
            }
        }
        int vst = 0, vph = 0;
        bool ok = true;
        // the step's row at key t (new_lo <= t < n_keys) as 16-byte pieces
        auto new_row = [&](const __nv_bfloat16 *rows, int t) {
            return reinterpret_cast<const uint4 *>(
                rows + (((int64_t)b * R + (t - new_lo)) * p.n_kv_heads + kvh) * HD);
        };
        for (int j = 0; j < n_kt && ok; ++j) {
            const bool nw = tile_new(j);
            const int key0 = (kt0 + j) * kBN;
            if (nw) {
                // K(j) is issued before V(j); its stage is not refilled before
                // the MMA warp, which waits for this patch, has read it
                const int kst = j % C::kKStages;
                ok = mbar_wait(&k_full[kst], (j / C::kKStages) & 1, p.err);
                __syncwarp();
                if (!ok) break;
                // rows r0 .. r1 - 1 of the [half][128 rows][128 B] swizzled tile
                const uint32_t kb = smem_u32(sK + kst * C::kKBytes);
                const int r0 = max(key0, new_lo) - key0, r1 = min(key0 + kBN, n_keys) - key0;
                constexpr int kPieces = HD / 8;  // 16-byte pieces of a head row
                for (int i = ct; i < (r1 - r0) * kPieces; i += 64) {
                    const int r = r0 + i / kPieces, pc = i % kPieces;
                    st_shared_v4(kb + (pc >> 3) * (kBN * 128) + r * 128 + (((pc & 7) ^ (r & 7)) << 4),
                                 __ldg(new_row(p.k_new, key0 + r) + pc));
                }
                fence_proxy_async_smem();
                mbar_arrive(k_patch);
            }
            ok = mbar_wait(&v_full[vst], vph, p.err);
            __syncwarp();
            if (!ok) break;
            const uint32_t base = smem_u32(sV + vst * C::kVBytes);
            float amax = 0.f;
#pragma unroll 4
            for (int i = ct; i < C::kVBytes / 16; i += 64) {
                uint4 w = ld_shared_v4(base + i * 16);
                uint32_t *u = &w.x;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x0 = __uint_as_float(u[e] << 16);
                    const float x1 = __uint_as_float(u[e] & 0xFFFF0000u);
                    amax = max3(amax, fabsf(x0), fabsf(x1));
                    u[e] = pack_f16x2_sat(x0, x1);
                }
                st_shared_v4(base + i * 16, w);
            }
            if (nw) {
                // the step's rows of this tile, converted the same way: this
                // thread's pieces of row r are those of rows r = ct / 8 mod 8,
                // swizzled position ct % 8 (logical piece (ct % 8) ^ (r % 8))
                const int r0 = max(key0, new_lo) - key0, r1 = min(key0 + kBN, n_keys) - key0;
                const int rr = ct >> 3, c = (ct & 7) ^ rr;
                for (int r = r0 + ((rr - r0) & 7); r < r1; r += 8) {
                    const uint4 *src = new_row(p.v_new, key0 + r);
                    for (int hf = 0; hf < C::kHalves; ++hf) {
                        uint4 w = __ldg(src + hf * 8 + c);
                        uint32_t *u = &w.x;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = __uint_as_float(u[e] << 16);
                            const float x1 = __uint_as_float(u[e] & 0xFFFF0000u);
                            amax = max3(amax, fabsf(x0), fabsf(x1));
                            u[e] = pack_f16x2_sat(x0, x1);
                        }
                        st_shared_v4(base + (hf * (kBN * 8) + r * 8 + (ct & 7)) * 16, w);
                    }
                }
            }
            if (!(amax < 65536.f)) report_error(p.err, ATTN_ERR_UNSUPPORTED);
            fence_proxy_async_smem();
            mbar_arrive(&v_conv[vst]);
            if (++vst == C::kVStages) {
                vst = 0;
                vph ^= 1;
            }
        }
    }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ---------------------------------------------------------- softmax
        const int a = (warp - 4) >> 2;     // which tile
        const int quad = warp & 3;         // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;  // tile row = TMEM lane
        int qi = -1;  // the row's position (-1: a padding row, which sees no key)
        {
            const int r = r_first + a * p.rt + row / G;  // chunk row
            if (row < used && r < r_end) qi = p.positions[(int64_t)b * R + r];
        }
        const int key_cap = min(qi, n_keys - 1);  // last key this row may see
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const uint32_t s_tmem = tmem + a * 128 + lane_base;
        const uint32_t o_tmem = tmem + 256 + a * HD + lane_base;
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kt; ++j) {
            ok = mbar_wait(&s_full[a], j & 1, p.err);
            __syncwarp();
            if (!ok) break;
            tc_fence_after();
            float s[kBN];
            {
                uint32_t(&u)[kBN] = *reinterpret_cast<uint32_t(*)[kBN]>(s);
                tmem_ld_32x32b_x32(s_tmem + 0, *reinterpret_cast<uint32_t(*)[32]>(u + 0));
                tmem_ld_32x32b_x32(s_tmem + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
                tmem_ld_32x32b_x32(s_tmem + 64, *reinterpret_cast<uint32_t(*)[32]>(u + 64));
                tmem_ld_32x32b_x32(s_tmem + 96, *reinterpret_cast<uint32_t(*)[32]>(u + 96));
                tmem_wait_ld();
                tmem_regs_after_wait(u);
            }
            const int key0 = (kt0 + j) * kBN;
            const bool needs_mask =
                key0 + kBN - 1 > key_cap || (p.window > 0 && qi - key0 >= p.window);
            if (needs_mask) {
                // the row sees columns lo <= c <= hi (c = key - key0): one
                // compare with an immediate (two with a window) and a select
                const int hi = key_cap - key0;
                if (p.window > 0) {
                    const int lo = qi - p.window + 1 - key0;
#pragma unroll
                    for (int c = 0; c < kBN; ++c) s[c] = (c <= hi && c >= lo) ? s[c] : -INFINITY;
                } else {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) s[c] = c <= hi ? s[c] : -INFINITY;
                }
            }
            float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int c = 4; c + 8 <= kBN; c += 8) {  // columns 4 .. kBN - 5
                mx0 = max3(mx0, s[c], s[c + 1]);
                mx1 = max3(mx1, s[c + 2], s[c + 3]);
                mx2 = max3(mx2, s[c + 4], s[c + 5]);
                mx3 = max3(mx3, s[c + 6], s[c + 7]);
            }
            mx0 = max3(mx0, s[kBN - 4], s[kBN - 3]);  // the last four columns
            mx1 = max3(mx1, s[kBN - 2], s[kBN - 1]);
            const float mx = max3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
            float alpha = 1.f;
            if (mx > m_run + kRescaleThreshold || m_run == -INFINITY) {
                const float m_new = mx == -INFINITY ? m_run : mx;
                alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
                m_run = m_new;
            }
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t orow[32];
                    tmem_ld_32x32b_x32(o_tmem + c0, orow);
                    tmem_wait_ld();
                    tmem_regs_after_wait(orow);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tmem_st_32x32b_x32(o_tmem + c0, orow);
                }
            }
            const float mref = m_run == -INFINITY ? 0.f : m_run;
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < kBN; c0 += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float x0, x1;
                    fma2(x0, x1, s[c0 + 2 * e], s[c0 + 2 * e + 1], sl2, sl2, -mref, -mref);
                    const float p0 = fast_exp2(x0);
                    const float p1 = fast_exp2(x1);
                    add2(sum0, sum1, sum0, sum1, p0, p1);
                    pk[e] = pack_f16x2(p0, p1);
                }
                // P over its own S columns: 32 keys in 16 columns
                tmem_st_32x32b_x16(s_tmem + c0 / 2, pk);
                if (c0 == kBN / 2 - 32 || c0 == kBN - 32) {
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&p_full[a * 2 + (c0 >= kBN / 2 ? 1 : 0)]);
                }
            }
            l_run = l_run * alpha + (sum0 + sum1);
        }
        // epilogue: the row's O / l (bf16 when the key range is not split,
        // else an f16 partial state with its fp32 base-2 log-sum-exp)
        if (ok) ok = mbar_wait(o_done, 0, p.err);
        __syncwarp();
        tc_fence_after();
        const bool any = l_run > 0.f;  // O in TMEM was written (n_kt > 0, a key seen)
        const float inv = any ? 1.f / l_run : 0.f;
        const int64_t slot = (((int64_t)b * p.n_kv_heads + kvh) * p.n_pairs + pair) * p.n_split +
                             split;
        const int m = a * kBM + row;
        const int r = r_first + a * p.rt + row / G, gh = row % G;  // chunk row, group head
        const bool live = row < used && r < r_end;
        __nv_bfloat16 *dst =
            p.out + (((int64_t)b * R + r) * (p.n_kv_heads * G) + kvh * G + gh) * HD;
        // A split's partial O (normalised by its own sum, so |O| <= max |v|,
        // inside f16's range as the V conversion requires) is kept in f16:
        // 2^-11 relative, a quarter of the output's bf16 step, for half the
        // bytes written here and read by the merge.  It goes through shared
        // memory (the K ring for tile 0, the V ring for tile 1: the last MMA
        // has read them) as 128-byte swizzled rows of 64 columns, and TMA
        // writes whole lines of it; a row per thread stored straight to
        // global memory would write into 32 lines per instruction.
        uint8_t *stage = a == 0 ? sK : sV;
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t orow[32];
            if (n_kt > 0) {  // CTA-uniform: the TMEM rows were accumulated into
                tmem_ld_32x32b_x32(o_tmem + c0, orow);
                tmem_wait_ld();
                tmem_regs_after_wait(orow);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) orow[e] = 0u;
            }
            // O / l of this row (zero when no key was seen: inv is 0)
            auto v = [&](int e) { return any ? __uint_as_float(orow[e]) * inv : 0.f; };
            if (p.n_split == 1) {
                if (live) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<uint4 *>(dst + c0 + q4 * 8) =
                            make_uint4(pack_bf16x2(v(8 * q4), v(8 * q4 + 1)),
                                       pack_bf16x2(v(8 * q4 + 2), v(8 * q4 + 3)),
                                       pack_bf16x2(v(8 * q4 + 4), v(8 * q4 + 5)),
                                       pack_bf16x2(v(8 * q4 + 6), v(8 * q4 + 7)));
                }
            } else {
                // columns c0 .. c0 + 31: four 16-byte pieces of box c0 / 64
                const uint32_t base = smem_u32(stage + (c0 / 64) * (kBM * 128) + row * 128);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int piece = ((c0 & 63) >> 3) + q4;
                    st_shared_v4(base + ((piece ^ (row & 7)) << 4),
                                 make_uint4(pack_f16x2(v(8 * q4), v(8 * q4 + 1)),
                                            pack_f16x2(v(8 * q4 + 2), v(8 * q4 + 3)),
                                            pack_f16x2(v(8 * q4 + 4), v(8 * q4 + 5)),
                                            pack_f16x2(v(8 * q4 + 6), v(8 * q4 + 7))));
                }
            }
        }
        if (p.n_split > 1) {
            p.ws_lse[slot * 2 * kBM + m] = any ? m_run + __log2f(l_run) : -INFINITY;
            fence_proxy_async_smem();
            if (a == 0)
                asm volatile("bar.sync 1, 128;" ::: "memory");
            else
                asm volatile("bar.sync 2, 128;" ::: "memory");
            if (quad == 0 && lane == 0) {
                for (int t = 0; t < HD / 64; ++t)
                    tma_store_2d(&tm_ws, stage + t * (kBM * 128), t * 64,
                                 (int)(slot * 2 * kBM + a * kBM));
                tma_store_commit();
                tma_store_wait_all();
            }
        }
    }
    __syncwarp();  // lanes 1..31 of the TMA and MMA warps wait here for lane 0
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// One warp per packed row of a (request, KV head, pair): the splits' partial
// states in split order, weights from the log-sum-exps, one bf16 rounding.
// Up to 32 splits are read in one round (each lane one split's log-sum-exp,
// every lane its columns of all of them, f16): no load waits for another.
// More splits go 32 at a time, the running sums rescaled to the new maximum.
template <int HD>
__global__ void __launch_bounds__(kMergeWarps * 32) chunk_merge_kernel(const Params p) {
    constexpr int PER = HD / 32;
    pdl_wait();  // the partial states come from the chunk kernel
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kMergeWarps + warp;  // (group slot, m)
    const int m = (int)(gw % (2 * kBM));
    const int64_t grp = gw / (2 * kBM);  // ((b * Hkv + kvh) * pairs + pair)
    const int pair = (int)(grp % p.n_pairs);
    const int64_t bk = grp / p.n_pairs;
    if (bk >= (int64_t)p.batch * p.n_kv_heads) return;
    const int kvh = (int)(bk % p.n_kv_heads), b = (int)(bk / p.n_kv_heads);
    const int G = p.group;
    const int a = m / kBM, row = m % kBM;
    const int r = pair * 2 * p.rt + a * p.rt + row / G, gh = row % G;
    if (row >= p.rt * G || r >= p.q_rows) return;
    const float *lse = p.ws_lse + grp * p.n_split * 2 * kBM + m;  // split s at s * 2 kBM
    const uint16_t *o = p.ws_o + (grp * p.n_split * 2 * kBM + m) * HD + lane * PER;
    constexpr int kRound = 32;
    float M = -INFINITY, L = 0.f, acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int s0 = 0; s0 < p.n_split; s0 += kRound) {
        const int n = min(kRound, p.n_split - s0);
        // every load of the round issued before any is used
        const float l = lane < n ? __ldcg(lse + (int64_t)(s0 + lane) * 2 * kBM) : -INFINITY;
        uint32_t raw[kRound][PER / 2];
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
#pragma unroll
            for (int e = 0; e < PER / 2; ++e) raw[k][e] = 0u;
            if (k < n) {
                const uint16_t *src = o + (int64_t)(s0 + k) * 2 * kBM * HD;
                if constexpr (PER == 4) {
                    const uint2 t = __ldcg(reinterpret_cast<const uint2 *>(src));
                    raw[k][0] = t.x;
                    raw[k][1] = t.y;
                } else {
                    raw[k][0] = __ldcg(reinterpret_cast<const unsigned int *>(src));
                }
            }
        }
        float mr = l;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, d));
        const float Mn = fmaxf(M, mr);
        if (Mn == -INFINITY) continue;  // no split so far saw a key
        if (M != -INFINITY && Mn != M) {
            const float rs = fast_exp2(M - Mn);
            L *= rs;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] *= rs;
        }
        M = Mn;
        const float w = l == -INFINITY ? 0.f : fast_exp2(l - M);  // this lane's split
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            const float f = __shfl_sync(0xffffffffu, w, k);
            if (k < n) {
                L += f;
#pragma unroll
                for (int e = 0; e < PER / 2; ++e) {
                    const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&raw[k][e]));
                    acc[2 * e] += f * v.x;
                    acc[2 * e + 1] += f * v.y;
                }
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16 *dst =
        p.out + (((int64_t)b * p.q_rows + r) * (p.n_kv_heads * G) + kvh * G + gh) * HD + lane * PER;
    if constexpr (PER == 4) {
        uint2 w2;
        w2.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        w2.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(dst) = w2;
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}

template <int HD>
int launch(const Params &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
           const CUtensorMap &tw, cudaStream_t stream) {
    auto kern = chunk_kernel<HD>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        const cudaError_t e = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<HD>::kSmem);
        if (e != cudaSuccess) {
            note_cuda_error(e);
            return ATTN_ERR_CUDA;
        }
        configured_device = dev;
    }
    const int64_t groups = (int64_t)p.batch * p.n_kv_heads * p.n_pairs;
    const unsigned grid = (unsigned)(groups * p.n_split);
    if (launch_pdl(kern, dim3(grid), dim3(kThreads), Cfg<HD>::kSmem, stream, tq, tk, tv, tw, p) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    if (p.n_split > 1) {
        const unsigned mgrid = (unsigned)((groups * 2 * kBM + kMergeWarps - 1) / kMergeWarps);
        if (launch_pdl(chunk_merge_kernel<HD>, dim3(mgrid), dim3(kMergeWarps * 32), 0, stream,
                       p) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace chk

// Chunk plan: rows per tile, pairs and splits (see kernels.h).
void plan_chunk(int batch, int q_rows, int n_q_heads, int n_kv_heads, int head_dim,
                int max_seq_len, int window, ChunkPlan *plan) {
    const int G = n_q_heads / n_kv_heads;
    plan->rt = chk::kBM / G;
    plan->n_pairs = (q_rows + 2 * plan->rt - 1) / (2 * plan->rt);
    const int64_t groups = (int64_t)batch * n_kv_heads * plan->n_pairs;
    // key tiles a pair may need: its rows' keys (bounded by max_seq_len, and
    // by the window plus the pair's rows)
    int64_t keys = max_seq_len;
    if (window > 0) keys = std::min<int64_t>(keys, (int64_t)window + 2 * plan->rt + chk::kBN);
    const int64_t tiles = (keys + chk::kBN - 1) / chk::kBN + 1;
    // enough CTAs to fill the SMs (one CTA each), at least two key tiles apiece
    int64_t split = std::max<int64_t>(1, device_sm_count() / std::max<int64_t>(groups, 1));
    split = std::min<int64_t>(split, std::max<int64_t>(1, tiles / 2));
    plan->n_split = (int)split;
    // per split and packed row: head_dim f16 of O, one fp32 log-sum-exp
    plan->workspace = plan->n_split > 1 ? (size_t)groups * plan->n_split * 2 * chk::kBM *
                                              ((size_t)head_dim * 2 + sizeof(float))
                                        : 0;
}

int launch_chunk(const ChunkPlan &plan, const void *q, const attn_kv_cache *cache,
                 const int32_t *seq_lens, const int32_t *positions, int batch, int q_rows,
                 int max_seq_len, int window, int n_q_heads, int n_kv_heads, int head_dim,
                 float scale, void *out, void *workspace, int32_t *err, cudaStream_t stream,
                 const void *k_new, const void *v_new, const int64_t *slot_mapping) {
    chk::Params p;
    p.batch = batch;
    p.q_rows = q_rows;
    p.window = window;
    p.n_kv_heads = n_kv_heads;
    p.group = n_q_heads / n_kv_heads;
    p.head_dim = head_dim;
    p.rt = plan.rt;
    p.n_pairs = plan.n_pairs;
    p.n_split = plan.n_split;
    p.slots_per_seq = cache->slots_per_seq;
    p.max_seq_len = max_seq_len;
    p.seq_lens = seq_lens;
    p.positions = positions;
    p.scale_log2 = scale * 1.4426950408889634f;
    const size_t groups = (size_t)batch * n_kv_heads * plan.n_pairs;
    p.ws_o = static_cast<uint16_t *>(workspace);
    p.ws_lse = p.ws_o ? reinterpret_cast<float *>(p.ws_o + groups * plan.n_split * 2 * chk::kBM *
                                                               head_dim)
                      : nullptr;
    p.out = static_cast<__nv_bfloat16 *>(out);
    const bool fused = k_new != nullptr && v_new != nullptr && slot_mapping != nullptr;
    p.k_new = fused ? static_cast<const __nv_bfloat16 *>(k_new) : nullptr;
    p.v_new = fused ? static_cast<const __nv_bfloat16 *>(v_new) : nullptr;
    p.slot_mapping = fused ? slot_mapping : nullptr;
    p.num_slots = cache->num_slots;
    p.k_cache = static_cast<__nv_bfloat16 *>(cache->k);
    p.v_cache = static_cast<__nv_bfloat16 *>(cache->v);
    p.err = err;
    // q viewed as {head_dim, n_q_heads, q_rows, batch}: a box of {64, G, rt, 1}
    // lands as rt x G rows of 128 bytes, the packed tile rows.
    CUtensorMap tq, tk, tv;
    const uint64_t dq[4] = {(uint64_t)head_dim, (uint64_t)n_q_heads, (uint64_t)q_rows,
                            (uint64_t)batch};
    const uint64_t sq[3] = {(uint64_t)head_dim * 2, (uint64_t)n_q_heads * head_dim * 2,
                            (uint64_t)q_rows * n_q_heads * head_dim * 2};
    const uint32_t bq[4] = {64, (uint32_t)p.group, (uint32_t)plan.rt, 1};
    // the linear cache viewed per request: {Hkv * D, slots_per_seq, batch}
    const uint64_t dk[3] = {(uint64_t)n_kv_heads * head_dim, (uint64_t)cache->slots_per_seq,
                            (uint64_t)batch};
    const uint64_t sk[2] = {(uint64_t)n_kv_heads * head_dim * 2,
                            (uint64_t)cache->slots_per_seq * n_kv_heads * head_dim * 2};
    const uint32_t bk[3] = {64, (uint32_t)chk::kBN, 1};
    if (!encode_tensor_map(&tq, q, 4, dq, sq, bq, true) ||
        !encode_tensor_map(&tk, cache->k, 3, dk, sk, bk, true) ||
        !encode_tensor_map(&tv, cache->v, 3, dk, sk, bk, true)) {
        note_cuda_error(cudaErrorInvalidValue);
        return ATTN_ERR_CUDA;
    }
    // the splits' partial O viewed as {head_dim, slot * 256 + row} f16: a
    // box of {64, 128} is one staged 128-row tile of 64 columns (unused, and
    // the K map passed in its place, when the key range is not split)
    CUtensorMap tw = tk;
    if (plan.n_split > 1) {
        const uint64_t dw[2] = {(uint64_t)head_dim, groups * plan.n_split * 2 * chk::kBM};
        const uint64_t sw[1] = {(uint64_t)head_dim * 2};
        const uint32_t bw[2] = {64, (uint32_t)chk::kBM};
        if (!encode_tensor_map_f16(&tw, p.ws_o, 2, dw, sw, bw)) {
            note_cuda_error(cudaErrorInvalidValue);
            return ATTN_ERR_CUDA;
        }
    }
    return head_dim == 128 ? chk::launch<128>(p, tq, tk, tv, tw, stream)
                           : chk::launch<64>(p, tq, tk, tv, tw, stream);
}

}  // namespace gqa
