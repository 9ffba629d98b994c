// append.cu -- KV append: cache[slot_mapping[i]] = new[i] for K and V.
//
// The step's new K/V rows are written into the slots the engine reserved for
// them before attention reads the cache (Voxtral Realtime -- Architecture &
// Design Notes, "Encoder KV cache": writes happen before attention;
// talker_multiframe, NarrowStep fields: slot_mapping[r] is the slot reserved
// for the frame).  It is a pure copy: each thread moves 16-byte pieces, and
// consecutive threads move consecutive pieces of one row, so both the read of
// the new rows and the write into the slot are coalesced.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gqa {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4 *__restrict__ k_new,
                                                        const uint4 *__restrict__ v_new,
                                                        const int64_t *__restrict__ slot_mapping,
                                                        int64_t n, uint4 *__restrict__ k_cache,
                                                        uint4 *__restrict__ v_cache,
                                                        int64_t num_slots, int pieces_per_row,
                                                        int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t per_row = 2ll * pieces_per_row;
    const int64_t total = n * per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += stride) {
        const int64_t row = idx / per_row;
        const int rem = (int)(idx - row * per_row);
        const int tensor = rem / pieces_per_row;  // 0: K, 1: V
        const int piece = rem - tensor * pieces_per_row;
        const int64_t slot = __ldg(slot_mapping + row);
        if (slot < 0 || slot >= num_slots) {
            if (rem == 0) report_error(err, ATTN_ERR_BOUNDS);
            continue;
        }
        const uint4 *src = tensor == 0 ? k_new : v_new;
        uint4 *dst = tensor == 0 ? k_cache : v_cache;
        dst[slot * pieces_per_row + piece] = __ldg(src + row * pieces_per_row + piece);
    }
}

int launch_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping, int64_t n,
                     void *k_cache, void *v_cache, int64_t num_slots, int row_bytes,
                     int32_t *err, cudaStream_t stream) {
    if (n <= 0) return ATTN_OK;
    const int pieces = row_bytes / 16;
    const int64_t total = n * 2ll * pieces;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const cudaError_t e = launch_pdl(
        kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping, n,
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_slots, pieces, err);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace gqa
