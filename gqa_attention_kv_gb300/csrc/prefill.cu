// prefill.cu -- causal GQA flash-attention prefill on tcgen05 tensor cores.
//
// What is computed (vibevoice.c, "Prefill attention" and "Attention
// backends"; Voxtral Realtime notes, "Offline Encoder"): for each sequence,
// query head h and position i, softmax(scale * q_i . k_t) over t <= i (and
// i - t < window when a window is set) applied to v_t, with query head h
// reading KV head h / (n_q_heads / n_kv_heads).  The online softmax over key
// tiles is an exact reformulation.
//
// GB300 mapping (one CTA = one 128-row query tile of one head):
//   warp 0       TMA producer: the Q tile once, then K/V tiles of 128 keys
//                into a two-stage ring (128-byte swizzle, 3D tensor maps, so
//                rows past the sequence end are zero-filled).
//   warp 1       allocates TMEM; lane 0 issues every tcgen05.mma:
//                S = Q K^T (M=128, N=128, K=head_dim) into one of two TMEM
//                buffers, then O += P V (M=128, N=head_dim, K=128) into the
//                TMEM accumulator.  QK^T of tile j+1 is issued before PV of
//                tile j so the tensor core works while the softmax runs.
//   warps 2..5   softmax: thread = query row = TMEM lane.  Reads its S row
//                with tcgen05.ld, masks, keeps the running max / sum in fp32,
//                writes P into swizzled shared tiles as two bf16 halves,
//                hi + lo (vibevoice.c, "Attention backends": one rounding of
//                P is too coarse; PV then runs once per half), and rescales
//                its O row in TMEM only when the running max grew by more
//                than 2^8 (the result is the same; rescaling is lazy).
//                At the end: O / l -> bf16 -> shared -> TMA store.
// Tiles wholly above the diagonal or before the window are never loaded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gqa {
namespace pre {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per tile
constexpr int kThreads = 192;     // 6 warps
constexpr int kSoftmaxWarp0 = 2;
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kPLo = kBM * kBN * 2;        // byte offset of the P lo tile after P hi

template <int HD>
struct Cfg {
    static constexpr int kHalves = HD / 64;
    static constexpr int kStages = HD == 128 ? 2 : 3;
    static constexpr int kQBytes = kBM * HD * 2;
    static constexpr int kKBytes = kBN * HD * 2;
    static constexpr int kVBytes = kBN * HD * 2;
    static constexpr int kPBytes = 2 * kBM * kBN * 2;  // P as bf16 hi + lo
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQBytes;
    static constexpr int kOffP = kOffKV + kStages * (kKBytes + kVBytes);
    static constexpr int kOffBar = kOffP + kPBytes;
    static constexpr int kNumBars = 2 * kStages + 8;
    static constexpr size_t kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
};

struct Params {
    int batch, seq_len, window, n_q_heads, n_kv_heads, group;
    int n_qtiles;
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
    uint8_t *sKV = smem + C::kOffKV;
    uint8_t *sP = smem + C::kOffP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *kv_full = bars;                      // [kStages]
    uint64_t *kv_empty = bars + C::kStages;        // [kStages]
    uint64_t *q_full = bars + 2 * C::kStages;
    uint64_t *s_full = q_full + 1;                 // [2]
    uint64_t *s_free = s_full + 2;                 // [2]
    uint64_t *p_full = s_free + 2;
    uint64_t *o_ready = p_full + 1;
    uint64_t *mma_done = o_ready + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Longest query tiles first: the linear block id walks tiles from the end.
    const int per_tile = p.n_q_heads * p.batch;
    const int qt = p.n_qtiles - 1 - (int)(blockIdx.x / per_tile);
    const int rest = blockIdx.x % per_tile;
    const int h = rest % p.n_q_heads;
    const int b = rest / p.n_q_heads;
    const int g = h / p.group;
    const int q0 = qt * kBM;
    const int key_hi = min(p.seq_len, q0 + kBM);  // exclusive
    const int key_lo = p.window > 0 ? max(0, q0 - p.window + 1) : 0;
    const int kt0 = key_lo / kBN;
    const int n_kt = (key_hi + kBN - 1) / kBN - kt0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(&s_free[0], 128);
        mbar_init(&s_free[1], 128);
        mbar_init(p_full, 128);
        mbar_init(o_ready, 1);
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
    const uint32_t tmem_s0 = tmem, tmem_s1 = tmem + 128, tmem_o = tmem + 256;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            mbar_arrive_expect_tx(q_full, C::kQBytes);
            for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_3d(sQ + hf * (kBM * 128), &tm_q, h * HD + hf * 64, q0, b, q_full);
            for (int j = 0; j < n_kt; ++j) {
                const int st = j % C::kStages;
                if (j >= C::kStages &&
                    !mbar_wait(&kv_empty[st], ((j / C::kStages) - 1) & 1, p.err))
                    break;
                uint8_t *sk = sKV + st * (C::kKBytes + C::kVBytes);
                uint8_t *sv = sk + C::kKBytes;
                const int key0 = (kt0 + j) * kBN;
                mbar_arrive_expect_tx(&kv_full[st], C::kKBytes + C::kVBytes);
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    tma_load_3d(sk + hf * (kBN * 128), &tm_k, g * HD + hf * 64, key0, b, &kv_full[st]);
                    tma_load_3d(sv + hf * (kBN * 128), &tm_v, g * HD + hf * 64, key0, b, &kv_full[st]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, HD, 0, 1);
            const uint32_t q_addr = smem_u32(sQ);
            const uint32_t p_addr = smem_u32(sP);
            bool ok = mbar_wait(q_full, 0, p.err);
            auto issue_qk = [&](int j) -> bool {
                const int st = j % C::kStages, sb = j & 1;
                if (!mbar_wait(&kv_full[st], (j / C::kStages) & 1, p.err)) return false;
                if (j >= 2 && !mbar_wait(&s_free[sb], ((j >> 1) - 1) & 1, p.err)) return false;
                tc_fence_after();
                const uint32_t k_addr = smem_u32(sKV + st * (C::kKBytes + C::kVBytes));
                const uint32_t d_tmem = sb ? tmem_s1 : tmem_s0;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                    const uint64_t a = smem_desc_sw128(q_addr + off, 16, 1024);
                    const uint64_t bdesc =
                        smem_desc_sw128(k_addr + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024);
                    tc_mma_ss(d_tmem, a, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[sb]);
                return true;
            };
            if (ok && n_kt > 0) ok = issue_qk(0);
            for (int j = 0; j < n_kt && ok; ++j) {
                if (j + 1 < n_kt && !issue_qk(j + 1)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(p_full, j & 1, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int st = j % C::kStages;
                const uint32_t v_addr = smem_u32(sKV + st * (C::kKBytes + C::kVBytes) + C::kKBytes);
#pragma unroll
                for (int part = 0; part < 2; ++part) {  // P hi, then P lo
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint64_t a = smem_desc_sw128(
                            p_addr + part * kPLo + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
                        // V tile: keys are rows (K), head_dim contiguous (N): MN-major.
                        const uint64_t bdesc =
                            smem_desc_sw128(v_addr + kk * 16 * 128, kBN * 128, 1024);
                        tc_mma_ss(tmem_o, a, bdesc, idesc_pv,
                                  (j > 0 || kk > 0 || part > 0) ? 1u : 0u);
                    }
                }
                tc_commit(o_ready);
                tc_commit(&kv_empty[st]);
            }
            // All issued MMAs complete before TMEM is released.
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, p.err);
        }
    } else {
        // ---------------------------------------------------------- softmax
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;
        const int qi = q0 + row;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kt && ok; ++j) {
            const int sb = j & 1;
            ok = mbar_wait(&s_full[sb], (j >> 1) & 1, p.err);
            __syncwarp();  // reconverge before the warp-collective tcgen05.ld
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[kBN];
            {
                const uint32_t base = (sb ? tmem_s1 : tmem_s0) + lane_base;
                tmem_ld_32x32b_x32(base + 0, *reinterpret_cast<uint32_t(*)[32]>(sr + 0));
                tmem_ld_32x32b_x32(base + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
                tmem_ld_32x32b_x32(base + 64, *reinterpret_cast<uint32_t(*)[32]>(sr + 64));
                tmem_ld_32x32b_x32(base + 96, *reinterpret_cast<uint32_t(*)[32]>(sr + 96));
                tmem_wait_ld();
            }
            tc_fence_before();
            mbar_arrive(&s_free[sb]);
            // mask and row max (scaled to log2 units)
            const int key0 = (kt0 + j) * kBN;
            const bool needs_mask = key0 + kBN - 1 > q0 || (p.window > 0 && q0 + kBM - 1 - key0 >= p.window);
            float mx = -INFINITY;
            float s[kBN];
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                float v = __uint_as_float(sr[c]) * p.scale_log2;
                if (needs_mask) {
                    const int t = key0 + c;
                    const bool valid = t <= qi && (p.window <= 0 || qi - t < p.window);
                    v = valid ? v : -INFINITY;
                }
                s[c] = v;
                mx = fmaxf(mx, v);
            }
            // lazy rescale: keep the old reference max unless it grew by > 2^8
            float m_use = m_run;
            float alpha = 1.f;
            if (mx > m_run + kRescaleThreshold || m_run == -INFINITY) {
                m_use = mx == -INFINITY ? m_run : mx;
                alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_use);
            }
            const float mref = m_use == -INFINITY ? 0.f : m_use;
            float sum = 0.f;
            uint32_t pk[kBN / 2], pl[kBN / 2];
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
                const float p0 = fast_exp2(s[c] - mref);
                const float p1 = fast_exp2(s[c + 1] - mref);
                sum += p0 + p1;
                split_bf16x2(p0, p1, pk[c / 2], pl[c / 2]);
            }
            l_run = l_run * alpha + sum;
            m_run = m_use;
            // PV of the previous tile must be done before P and O are touched.
            if (j > 0) ok = mbar_wait(o_ready, (j - 1) & 1, p.err);
            __syncwarp();
            if (!ok) break;
            tc_fence_after();
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t orow[32];
                    tmem_ld_32x32b_x32(tmem_o + lane_base + c0, orow);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tmem_st_32x32b_x32(tmem_o + lane_base + c0, orow);
                }
                tmem_wait_st();
            }
            // P row -> shared, K-major with the 128-byte swizzle (two 64-key halves)
#pragma unroll
            for (int cc = 0; cc < kBN / 8; ++cc) {
                const int half = cc >> 3, c8 = cc & 7;
                uint8_t *dst = sP + half * (kBM * 128) + row * 128 + ((c8 ^ (row & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) =
                    make_uint4(pk[cc * 4 + 0], pk[cc * 4 + 1], pk[cc * 4 + 2], pk[cc * 4 + 3]);
                *reinterpret_cast<uint4 *>(dst + kPLo) =
                    make_uint4(pl[cc * 4 + 0], pl[cc * 4 + 1], pl[cc * 4 + 2], pl[cc * 4 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // epilogue: wait for the last PV, normalise, store
        if (ok && n_kt > 0) ok = mbar_wait(o_ready, (n_kt - 1) & 1, p.err);
        __syncwarp();
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t orow[32];
            tmem_ld_32x32b_x32(tmem_o + lane_base + c0, orow);
            tmem_wait_ld();
            uint32_t packed[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                packed[e] = pack_bf16x2(__uint_as_float(orow[2 * e]) * inv,
                                        __uint_as_float(orow[2 * e + 1]) * inv);
            // staging tile for the TMA store: [half][128 rows][128 B], swizzled (reuses Q)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int cc = (c0 / 8) + q4;  // 16-byte piece index along head_dim
                const int half = cc >> 3, c8 = cc & 7;
                uint8_t *dst = sQ + half * (kBM * 128) + row * 128 + ((c8 ^ (row & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[q4 * 4 + 0], packed[q4 * 4 + 1],
                                                             packed[q4 * 4 + 2], packed[q4 * 4 + 3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == kSoftmaxWarp0 && lane == 0 && ok) {
            for (int hf = 0; hf < C::kHalves; ++hf)
                tma_store_3d(&tm_o, sQ + hf * (kBM * 128), h * HD + hf * 64, q0, b);
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
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Cfg<HD>::kSmem) != cudaSuccess)
            return ATTN_ERR_CUDA;
        configured_device = dev;
    }
    const unsigned grid = (unsigned)p.n_qtiles * p.n_q_heads * p.batch;
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
    p.n_qtiles = (seq_len + pre::kBM - 1) / pre::kBM;
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
