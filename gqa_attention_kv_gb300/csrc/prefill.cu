// prefill.cu -- causal GQA flash-attention prefill on tcgen05 tensor cores.
//
// What is computed (vibevoice.c, "Prefill attention" and "Attention
// backends"; Voxtral Realtime notes, "Offline Encoder"): for each sequence,
// query head h and position i, softmax(scale * q_i . k_t) over t <= i (and
// i - t < window when a window is set) applied to v_t, with query head h
// reading KV head h / (n_q_heads / n_kv_heads).  The online softmax over key
// tiles is an exact reformulation.
//
// GB300 mapping.  One CTA = two consecutive 128-row query tiles (Q0, Q1) of
// one head; both walk the same key tiles, so every K/V tile is loaded once for
// 256 query rows, and the two tiles ping-pong: while one softmax warpgroup
// works on its scores the tensor core computes the other tile's QK^T and PV.
// When such pairs would not fill the SMs (short sequences), a CTA takes one
// tile (Q0) and its critical chain of key tiles runs alone, faster per tile.
//
//   warp 0      TMA producer: Q0, Q1 once; then K tiles (2-stage ring) and V
//               tiles (3-stage ring) of 128 keys, 128-byte swizzled, through
//               3D tensor maps (rows past the sequence end are zero-filled).
//   warp 1      allocates all 512 TMEM columns; lane 0 issues every
//               tcgen05.mma (kind::f16, fp32 accumulate):
//                 S_a = Q_a K^T            M=128 N=128 K=D   bf16, A, B from smem
//                 O_a += P_a V             M=128 N=D   K=128 f16, A from TMEM
//               TMEM columns: S_a/P_a at 128a, O_a at 256 + D a.
//   warps 2..3  rewrite every V tile in place from bf16 to f16 (same
//               positions, so the swizzle is unchanged) before P V reads it.
//   warps 4..7  softmax for Q0, warps 8..11 for Q1.  Thread = query row = TMEM
//               lane.  tcgen05.ld of its S row, mask (only on tiles that
//               cross the diagonal or the window edge; a tile none of the
//               query tile's rows sees is skipped by the MMA issuer and the
//               softmax alike), running max / sum in
//               fp32, P written back over its S columns rounded once to f16
//               (vibevoice.c, "Attention backends": P V takes its operands in
//               FP16, because one bf16 rounding of P is too coarse; f16 keeps
//               11 significant bits), O rescaled in TMEM only when the running
//               max grew by more than 2^8 (the result is unchanged; rescaling
//               is lazy; P stays below 2^8).  P is released in two halves of
//               64 keys, so PV on the first half runs while the second is
//               exponentiated.
//               Epilogue: O / l -> bf16 -> shared (over Q_a) -> TMA store,
//               clipped at the sequence end.
//
// Ordering facts the schedule relies on: tcgen05.mma operations of one thread
// execute in issue order, so S_a(j+1) = Q_a K^T, issued after O_a += P_a(j) V,
// overwrites P_a(j)'s columns only after that MMA has read them; and the
// commit that signals S_a(j+1) also covers O_a += P_a(j) V, so a softmax
// warpgroup that sees S_a(j+1) may rescale O_a.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gqa {
namespace pre {

constexpr int kBM = 128;          // query rows per tile (two tiles per CTA)
constexpr int kBN = 128;          // keys per tile
constexpr int kThreads = 384;     // 3 warpgroups
// Registers: launched at 168 per thread (384 x 168 = 64,512; three warps of
// 168 fit one SM sub-partition's 16,384).  The TMA / MMA / V-conversion
// warpgroup then drops to 88 and the two softmax warpgroups rise to 208:
// 4x32x88 + 8x32x208 = 64,512, exactly the launch total, and 88 + 208 + 208
// <= 512 per sub-partition lane slot.
constexpr uint32_t kRegsControl = 88;
constexpr uint32_t kRegsSoftmax = 208;
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int HD>
struct Cfg {
    static constexpr int kHalves = HD / 64;
    static constexpr int kKStages = HD == 128 ? 2 : 4;
    static constexpr int kVStages = HD == 128 ? 3 : 4;
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
    int batch, seq_len, window, n_q_heads, n_kv_heads, group;
    int n_pairs;  // CTAs along the sequence (256 query rows each, 128 when single)
    int single;   // 1: one Q tile per CTA (the second tile is absent)
    float scale_log2;
    int32_t *err;
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const Params p) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *k_full = bars;                          // [kKStages]
    uint64_t *k_empty = k_full + C::kKStages;         // [kKStages]
    uint64_t *v_full = k_empty + C::kKStages;         // [kVStages]
    uint64_t *v_empty = v_full + C::kVStages;         // [kVStages]
    uint64_t *q_full = v_empty + C::kVStages;
    uint64_t *s_full = q_full + 1;                    // [2]
    uint64_t *p_full = s_full + 2;                    // [2 tiles][2 key halves]
    uint64_t *o_done = p_full + 4;
    uint64_t *mma_done = o_done + 1;
    uint64_t *v_conv = mma_done + 1;                  // [kVStages]: V tile now f16
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Longest query tiles first: the linear block id walks pairs from the end.
    const int per_pair = p.n_q_heads * p.batch;
    const int pair = p.n_pairs - 1 - (int)(blockIdx.x / per_pair);
    const int rest = blockIdx.x % per_pair;
    const int h = rest % p.n_q_heads;
    const int b = rest / p.n_q_heads;
    const int g = h / p.group;
    const int rows = p.single ? kBM : 2 * kBM;  // query rows of this CTA
    const int q0 = pair * rows;
    const int key_hi = min(p.seq_len, q0 + rows);  // exclusive
    const int key_lo = p.window > 0 ? max(0, q0 - p.window + 1) : 0;
    const int kt0 = key_lo / kBN;
    const int n_kt = (key_hi + kBN - 1) / kBN - kt0;
    // The G heads of a KV group read the same K/V tiles; each starts its walk
    // over them at a different tile (the order of the tiles does not change
    // the result of the online softmax), so the CTAs resident at one time do
    // not all ask L2 for the same lines at once.
    const int rot = n_kt > 0 ? (int)(((int64_t)(h % p.group) * n_kt) / p.group) : 0;
    auto tile_of = [&](int j) { const int t = j + rot; return kt0 + (t >= n_kt ? t - n_kt : t); };
    // Tile j is dead for query tile a when no row of a may see any of its
    // keys: all keys after a's last row, all before the window of a's first
    // row, or a's rows all past the sequence.  Its S and P V are never
    // computed: the MMA issuer and the softmax warps both skip it.
    auto live = [&](int a, int j) -> bool {
        const int qa = q0 + a * kBM, key0 = tile_of(j) * kBN;
        return (a == 0 || !p.single) && qa < p.seq_len && key0 <= qa + kBM - 1 &&
               (p.window <= 0 || qa - (key0 + kBN - 1) < p.window);
    };

    // The next kernel may start its own prologue on SMs this grid leaves
    // free; it reads nothing of ours before its programmatic-launch wait.
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        // kernel parameters, not written by the previous kernel
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_o);
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
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // q, k, v may come from the previous kernel; out may be read by it
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
    // Each role's registers are set inside its own branch: code after a join
    // of different setmaxnreg values is compiled for the smaller one.
    setmaxnreg_dec<kRegsControl>();
    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            const int n_q = p.single ? 1 : 2;
            mbar_arrive_expect_tx(q_full, n_q * C::kQBytes);
            for (int a = 0; a < n_q; ++a)
                for (int hf = 0; hf < C::kHalves; ++hf)
                    tma_load_3d(sQ + a * C::kQBytes + hf * (kBM * 128), &tm_q, h * HD + hf * 64,
                                q0 + a * kBM, b, q_full);
            // K runs ahead of V: K(j) feeds QK^T one tile before V(j) feeds PV.
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
                                    g * HD + hf * 64, tile_of(kj) * kBN, b, &k_full[st]);
                    ++kj;
                } else {
                    const int st = vj % C::kVStages;
                    if (vj >= C::kVStages)
                        ok = mbar_wait(&v_empty[st], ((vj / C::kVStages) - 1) & 1, p.err);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&v_full[st], C::kVBytes);
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(sV + st * C::kVBytes + hf * (kBN * 128), &tm_v,
                                    g * HD + hf * 64, tile_of(vj) * kBN, b, &v_full[st]);
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
            // Descriptors are built once; a k-step adds its byte offset >> 4 to
            // the start-address field (no carry: shared addresses < 256 KB).
            const uint64_t q_desc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t k_desc0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
            // V tile: keys are rows (K), head_dim contiguous (N): MN-major.
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
            // O_a += P_a V for keys 64h .. 64h+63 of the tile (P as f16: 16
            // keys per 8 TMEM columns)
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
            bool ok = mbar_wait(q_full, 0, p.err) && (n_kt == 0 || mbar_wait(&k_full[0], 0, p.err));
            if (ok && n_kt > 0) {
                tc_fence_after();
                if (live(0, 0)) issue_qk(0, 0);
                if (live(1, 0)) issue_qk(1, 0);
                tc_commit(&k_empty[0]);
            }
            // stage indices and phases of the K and V rings, stepped without division
            int vst = 0, vph = 0, kst = 0, kph = 0;
            // live tiles of query tile 0 / 1 whose P V is issued (two scalars:
            // an array indexed by a would live in local memory)
            int n_pv0 = 0, n_pv1 = 0;
            for (int j = 0; j < n_kt && ok; ++j) {
                ok = mbar_wait(&v_conv[vst], vph, p.err);  // V(j) landed and is f16
                const bool more = j + 1 < n_kt;
                if (more && ++kst == C::kKStages) {
                    kst = 0;
                    kph ^= 1;
                }
                for (int a = 0; a < 2 && ok; ++a) {
                    if (live(a, j)) {
                        const int n_pv = a ? n_pv1 : n_pv0;
                        // each half of P as soon as the softmax has written it
                        for (int hh = 0; hh < 2 && ok; ++hh) {
                            ok = mbar_wait(&p_full[a * 2 + hh], n_pv & 1, p.err);
                            if (!ok) break;
                            tc_fence_after();
                            issue_pv_half(a, vst, hh, n_pv == 0 && hh == 0);
                        }
                        if (a) ++n_pv1; else ++n_pv0;
                        if (!ok) break;
                    }
                    if (a == 1) tc_commit(&v_empty[vst]);
                    if (more) {
                        if (a == 0) {
                            ok = mbar_wait(&k_full[kst], kph, p.err);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        if (live(a, j + 1)) issue_qk(a, kst);
                        if (a == 1) tc_commit(&k_empty[kst]);
                    }
                }
                if (++vst == C::kVStages) {
                    vst = 0;
                    vph ^= 1;
                }
            }
            tc_commit(o_done);
            // All issued MMAs complete before TMEM is released.
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, p.err);
        }
    } else {
        // ---------------------------------------------------------- V to f16
        // Each V tile is rewritten in place, bf16 -> f16 (exact for
        // magnitudes in [2^-14, 2^16); below that f16 keeps 2^-24 absolute
        // precision).  A magnitude of 2^16 or more has no f16: it saturates to
        // 65504 and the error word gets ATTN_ERR_UNSUPPORTED.  The writes are
        // made visible to the tensor core's proxy before the arrive.
        const int ct = threadIdx.x - 64;  // 0 .. 63
        int vst = 0, vph = 0;
        bool ok = true;
        for (int j = 0; j < n_kt && ok; ++j) {
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
        const int a = (warp - 4) >> 2;        // which query tile
        const int quad = warp & 3;            // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;     // row inside the tile
        const int qa0 = q0 + a * kBM;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const uint32_t s_tmem = tmem + a * 128 + lane_base;
        const uint32_t o_tmem = tmem + 256 + a * HD + lane_base;
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int n_s = 0;  // live tiles whose S this warp has read
        for (int j = 0; j < n_kt; ++j) {
            if (!live(a, j)) continue;
            ok = mbar_wait(&s_full[a], n_s & 1, p.err);
            __syncwarp();  // reconverge before the warp-collective tcgen05.ld
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
            const int key0 = tile_of(j) * kBN;
            const bool needs_mask =
                key0 + kBN - 1 > qa0 || (p.window > 0 && qa0 + kBM - 1 - key0 >= p.window);
            if (needs_mask) {
                // row sees columns lo <= c <= hi (c = key - key0): per element
                // one compare with an immediate (two with a window) and a select
                const int hi = qa0 + row - key0;
                if (p.window > 0) {
                    const int lo = hi - p.window + 1;
#pragma unroll
                    for (int c = 0; c < kBN; ++c) s[c] = (c <= hi && c >= lo) ? s[c] : -INFINITY;
                } else {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) s[c] = c <= hi ? s[c] : -INFINITY;
                }
            }
            // row max of the raw scores: three-input max, four independent chains
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
            // lazy rescale: keep the reference max unless it grew by > 2^8
            float alpha = 1.f;
            if (mx > m_run + kRescaleThreshold || m_run == -INFINITY) {
                const float m_new = mx == -INFINITY ? m_run : mx;
                alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
                m_run = m_new;
            }
            // O_a += P V of the previous tile is complete (covered by s_full)
            if (n_s > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
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
                    // keys of this half are in TMEM: let PV start on them
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&p_full[a * 2 + (c0 >= kBN / 2 ? 1 : 0)]);
                }
            }
            l_run = l_run * alpha + (sum0 + sum1);
            ++n_s;
        }
        // epilogue: wait for the last PV, normalise, store through shared memory
        if (ok) ok = mbar_wait(o_done, 0, p.err);
        __syncwarp();
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        uint8_t *stage = sQ + a * C::kQBytes;
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t orow[32];
            tmem_ld_32x32b_x32(o_tmem + c0, orow);
            tmem_wait_ld();
            tmem_regs_after_wait(orow);
            uint32_t packed[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                packed[e] = pack_bf16x2(__uint_as_float(orow[2 * e]) * inv,
                                        __uint_as_float(orow[2 * e + 1]) * inv);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int cc = (c0 / 8) + q4;  // 16-byte piece index along head_dim
                const int half = cc >> 3, c8 = cc & 7;
                uint8_t *dst = stage + half * (kBM * 128) + row * 128 + ((c8 ^ (row & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[q4 * 4 + 0], packed[q4 * 4 + 1],
                                                             packed[q4 * 4 + 2], packed[q4 * 4 + 3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (a == 0)
            asm volatile("bar.sync 1, 128;" ::: "memory");
        else
            asm volatile("bar.sync 2, 128;" ::: "memory");
        if (quad == 0 && lane == 0 && ok && qa0 < p.seq_len && (a == 0 || !p.single)) {
            for (int hf = 0; hf < C::kHalves; ++hf)
                tma_store_3d(&tm_o, stage + hf * (kBM * 128), h * HD + hf * 64, qa0, b);
            tma_store_commit();
            tma_store_wait_all();
        }
    }
    __syncwarp();  // lanes 1..31 of the TMA and MMA warps wait here for lane 0
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int HD>
int launch(const Params &p, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
           const CUtensorMap &to, cudaStream_t stream) {
    auto kern = prefill_kernel<HD>;
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
    const unsigned grid = (unsigned)p.n_pairs * p.n_q_heads * p.batch;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), Cfg<HD>::kSmem, stream, tq, tk, tv, to,
                      p) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

}  // namespace pre

int launch_prefill(const void *q, const void *k, const void *v, int batch, int seq_len,
                   int window, int n_q_heads, int n_kv_heads, int head_dim, float scale,
                   void *out, int32_t *err, cudaStream_t stream) {
    pre::Params p;
    p.batch = batch;
    p.seq_len = seq_len;
    p.window = window;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = n_q_heads / n_kv_heads;
    // Two Q tiles per CTA share every K/V tile and ping-pong on the tensor
    // core; when those CTAs would not fill the SMs (short sequences), each CTA
    // takes one tile instead: twice the CTAs, and the longest CTA's chain of
    // key tiles runs alone (~1 us a tile instead of ~1.5 for the pair).
    const int64_t pair_ctas =
        (int64_t)((seq_len + 2 * pre::kBM - 1) / (2 * pre::kBM)) * n_q_heads * batch;
    p.single = pair_ctas < device_sm_count() ? 1 : 0;
    p.n_pairs = p.single ? (seq_len + pre::kBM - 1) / pre::kBM
                         : (seq_len + 2 * pre::kBM - 1) / (2 * pre::kBM);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    CUtensorMap tq, tk, tv, to;
    const uint64_t dq[3] = {(uint64_t)n_q_heads * head_dim, (uint64_t)seq_len, (uint64_t)batch};
    const uint64_t sq[2] = {(uint64_t)n_q_heads * head_dim * 2,
                            (uint64_t)seq_len * n_q_heads * head_dim * 2};
    const uint64_t dk[3] = {(uint64_t)n_kv_heads * head_dim, (uint64_t)seq_len, (uint64_t)batch};
    const uint64_t sk[2] = {(uint64_t)n_kv_heads * head_dim * 2,
                            (uint64_t)seq_len * n_kv_heads * head_dim * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!encode_tensor_map(&tq, q, 3, dq, sq, box, true) ||
        !encode_tensor_map(&tk, k, 3, dk, sk, box, true) ||
        !encode_tensor_map(&tv, v, 3, dk, sk, box, true) ||
        !encode_tensor_map(&to, out, 3, dq, sq, box, true))
        return ATTN_ERR_CUDA;
    return head_dim == 128 ? pre::launch<128>(p, tq, tk, tv, to, stream)
                           : pre::launch<64>(p, tq, tk, tv, to, stream);
}

}  // namespace gqa
