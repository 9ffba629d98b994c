// append.cu -- KV append: cache[slot_mapping[i]] = new[i] for K and V.
//
// The step's new K/V rows are written into the slots the engine reserved for
// them before attention reads the cache (Voxtral Realtime -- Architecture &
// Design Notes, "Encoder KV cache": writes happen before attention;
// talker_multiframe, NarrowStep fields: slot_mapping[r] is the slot reserved
// for the frame).  It is a pure copy: each thread moves 16-byte pieces, and
// consecutive threads move consecutive pieces of one row, so both the read of
// the new rows and the write into the slot are coalesced.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gqa {

// Pieces a lane moves at once, all loads issued before any store: the bytes
// in flight, not the thread count, set the copy rate.
constexpr int kAppendUnroll = 4;

// One warp per (row, tensor): the row's slot read once, its head rows moved
// as 16-byte pieces by the lanes, kAppendUnroll per lane in flight.  The
// index arithmetic is 32-bit per row (a 64-bit division per piece made the
// copy issue-bound).
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4 *__restrict__ k_new,
                                                        const uint4 *__restrict__ v_new,
                                                        const int64_t *__restrict__ slot_mapping,
                                                        int64_t n, uint8_t *__restrict__ k_cache,
                                                        uint8_t *__restrict__ v_cache,
                                                        int64_t num_slots, KvPlace place,
                                                        int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int pph_shift = place.head_bytes == 256 ? 4 : 3;  // pieces per head: 16 or 8
    const int ppt = place.n_kv_heads << pph_shift;           // pieces of one row of one tensor
    const int64_t items = 2 * n;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t it = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
         it += nwarps) {
        const int64_t row = it >> 1;
        const int tensor = (int)(it & 1);
        const int64_t slot = __ldg(slot_mapping + row);
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0 && tensor == 0) report_error(err, ATTN_ERR_BOUNDS);
            continue;
        }
        const uint4 *src = (tensor == 0 ? k_new : v_new) + row * ppt;
        // head h's row of the slot: head 0's, then one head stride per head
        uint8_t *base = (tensor == 0 ? k_cache : v_cache) + place.head_offset(slot, 0);
        const int64_t head_stride = (place.rows == 0 ? 1 : place.rows) * (int64_t)place.head_bytes;
        for (int p0 = lane; p0 < ppt; p0 += 32 * kAppendUnroll) {
            uint4 val[kAppendUnroll];
#pragma unroll
            for (int u = 0; u < kAppendUnroll; ++u) {
                const int pc = p0 + 32 * u;
                if (pc < ppt) val[u] = __ldg(src + pc);
            }
#pragma unroll
            for (int u = 0; u < kAppendUnroll; ++u) {
                const int pc = p0 + 32 * u;
                if (pc < ppt) {
                    const int h = pc >> pph_shift, pp = pc & ((1 << pph_shift) - 1);
                    *reinterpret_cast<uint4 *>(base + h * head_stride + pp * 16) = val[u];
                }
            }
        }
    }
}

// FP8 cache (vibevoice.c, "KV cache"): each thread writes one 16-byte piece
// of a cache row, 16 E4M3 codes, from 32 bytes of bf16 input; a K element is
// shifted by the reference vector first, the difference formed in fp32.
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const float4 *__restrict__ k_ref, const int64_t *__restrict__ slot_mapping, int64_t n,
    uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache, int64_t num_slots,
    KvPlace place, int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int pieces_per_head = place.head_bytes / 16;  // 16 codes per piece
    const int pieces_per_row = place.n_kv_heads * pieces_per_head;
    const int64_t per_row = 2ll * pieces_per_row;
    const int64_t total = n * per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    constexpr int kU = kAppendUnroll / 2;  // each piece reads 32 bytes
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < total;
         base += stride * kU) {
        uint4 a[kU], b[kU];
        int piece_of[kU], tensor_of[kU];
        uint8_t *dst[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t idx = base + u * stride;
            dst[u] = nullptr;
            if (idx >= total) continue;
            const int64_t row = idx / per_row;
            const int rem = (int)(idx - row * per_row);
            const int tensor = rem / pieces_per_row;  // 0: K, 1: V
            const int piece = rem - tensor * pieces_per_row;
            const int64_t slot = __ldg(slot_mapping + row);
            if (slot < 0 || slot >= num_slots) {
                if (rem == 0) report_error(err, ATTN_ERR_BOUNDS);
                continue;
            }
            // 16 bf16 inputs: two 16-byte loads
            const uint4 *src = (tensor == 0 ? k_new : v_new) + (row * pieces_per_row + piece) * 2;
            a[u] = __ldg(src);
            b[u] = __ldg(src + 1);
            piece_of[u] = piece;
            tensor_of[u] = tensor;
            const int h = piece / pieces_per_head, pp = piece - h * pieces_per_head;
            dst[u] = (tensor == 0 ? k_cache : v_cache) + place.head_offset(slot, h) + pp * 16;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (dst[u] == nullptr) continue;
            const uint32_t w[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
            float x[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                x[2 * i] = __uint_as_float(w[i] << 16);
                x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
            if (tensor_of[u] == 0 && k_ref != nullptr) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 r = __ldg(k_ref + piece_of[u] * 4 + i);
                    x[4 * i] = __fsub_rn(x[4 * i], r.x);
                    x[4 * i + 1] = __fsub_rn(x[4 * i + 1], r.y);
                    x[4 * i + 2] = __fsub_rn(x[4 * i + 2], r.z);
                    x[4 * i + 3] = __fsub_rn(x[4 * i + 3], r.w);
                }
            }
            uint32_t c[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                c[i] = f32x2_to_e4m3x2(x[4 * i], x[4 * i + 1]) |
                       (f32x2_to_e4m3x2(x[4 * i + 2], x[4 * i + 3]) << 16);
            *reinterpret_cast<uint4 *>(dst[u]) = make_uint4(c[0], c[1], c[2], c[3]);
        }
    }
}

// Reference vector: ref[e] = mean over n rows of k[i][e].  Block: 32 columns
// x 8 row lanes; each thread sums every 8th row in fp64, the 8 partial sums
// are added in a fixed order, so the result does not depend on timing.
__global__ void __launch_bounds__(256) kv_reference_kernel(const __nv_bfloat16 *__restrict__ k,
                                                           int64_t n, int row_elems,
                                                           float *__restrict__ ref) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ double part[8][32];
    const int col = blockIdx.x * 32 + (threadIdx.x & 31), lane_row = threadIdx.x >> 5;
    double acc = 0.0;
    if (col < row_elems)
        for (int64_t i = lane_row; i < n; i += 8)
            acc += (double)__bfloat162float(k[i * row_elems + col]);
    part[lane_row][threadIdx.x & 31] = acc;
    __syncthreads();
    if (lane_row == 0 && col < row_elems) {
        double s = 0.0;
#pragma unroll
        for (int r = 0; r < 8; ++r) s += part[r][threadIdx.x];
        ref[col] = (float)(s / (double)n);
    }
}

int launch_kv_reference(const void *k, int64_t n, int row_elems, float *ref,
                        cudaStream_t stream) {
    const unsigned blocks = (unsigned)((row_elems + 31) / 32);
    const cudaError_t e = launch_pdl(kv_reference_kernel, dim3(blocks), dim3(256), 0, stream,
                                     static_cast<const __nv_bfloat16 *>(k), n, row_elems, ref);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_kv_append_fp8(const void *k_new, const void *v_new, const float *k_ref,
                         const int64_t *slot_mapping, int64_t n, void *k_cache, void *v_cache,
                         int64_t num_slots, const KvPlace &place, int32_t *err,
                         cudaStream_t stream) {
    if (n <= 0) return ATTN_OK;
    const int pieces = place.n_kv_heads * place.head_bytes / 16;  // 16 codes per piece
    const int64_t total = n * 2ll * pieces;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const cudaError_t e = launch_pdl(
        kv_append_fp8_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
        reinterpret_cast<const float4 *>(k_ref), slot_mapping, n,
        static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), num_slots, place, err);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping, int64_t n,
                     void *k_cache, void *v_cache, int64_t num_slots, const KvPlace &place,
                     int32_t *err, cudaStream_t stream) {
    if (n <= 0) return ATTN_OK;
    // one warp per (row, tensor), eight warps a block, at most eight blocks an SM
    const int threads = 256;
    int64_t blocks = (2 * n + 7) / 8;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const cudaError_t e = launch_pdl(
        kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping, n,
        static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), num_slots, place, err);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace gqa
