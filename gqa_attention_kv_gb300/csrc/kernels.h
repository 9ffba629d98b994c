// kernels.h -- host-side launchers shared between the C ABI and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/attn_kv.h"

namespace gqa {

int device_sm_count();

// The last CUDA runtime error a launch in this thread ran into (cudaSuccess if
// none); attn_last_cuda_error() reports it to the caller.
void note_cuda_error(cudaError_t e);

// Launch with programmatic stream serialisation: the kernel may begin while
// its predecessor on the stream finishes; it must call pdl_wait() before
// touching memory the predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
    if (e != cudaSuccess) note_cuda_error(e);
    return e;
}

// Encode a 2D/3D tensor map of bf16 (or, with bytes, 8-bit) elements, with
// 128-byte swizzle (returns false on failure).
bool encode_tensor_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                       const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128,
                       bool bytes = false);
// The same over f16 elements, 128-byte swizzled (boxes of 64 columns).
bool encode_tensor_map_f16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                           const uint64_t *strides_bytes, const uint32_t *box);

// Where head h's row of cache slot s starts, in bytes (attn_kv_cache's layouts):
// slot-major (rows == 0) or head-major inside blocks of `rows` slots.
struct KvPlace {
    int64_t rows;    // 0: ATTN_LAYOUT_BSHD; else the block size of ATTN_LAYOUT_BHSD
    int n_kv_heads;
    int head_bytes;  // head_dim x element size
    __host__ __device__ __forceinline__ int64_t head_offset(int64_t s, int h) const {
        return rows == 0 ? (s * n_kv_heads + h) * head_bytes
                         : (((s / rows) * n_kv_heads + h) * rows + s % rows) * head_bytes;
    }
};

// The placement a cache descriptor asks for (element size esize bytes).
inline KvPlace kv_place(const attn_kv_cache *c, int n_kv_heads, int head_dim, int esize) {
    KvPlace p;
    p.rows = c->layout == ATTN_LAYOUT_BHSD
                 ? (c->kind == ATTN_CACHE_PAGED ? c->block_size : c->slots_per_seq)
                 : 0;
    p.n_kv_heads = n_kv_heads;
    p.head_bytes = head_dim * esize;
    return p;
}

int launch_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping, int64_t n,
                     void *k_cache, void *v_cache, int64_t num_slots, const KvPlace &place,
                     int32_t *err, cudaStream_t stream);

// FP8 cache append: row_elems = n_kv_heads * head_dim (a multiple of 16);
// k_ref float32 [row_elems] or nullptr.
int launch_kv_append_fp8(const void *k_new, const void *v_new, const float *k_ref,
                         const int64_t *slot_mapping, int64_t n, void *k_cache, void *v_cache,
                         int64_t num_slots, const KvPlace &place, int32_t *err,
                         cudaStream_t stream);

// ref[e] = mean over n rows of the bf16 matrix k[n][row_elems], as float32.
int launch_kv_reference(const void *k, int64_t n, int row_elems, float *ref,
                        cudaStream_t stream);

// Chunk plan (many query rows per KV group over a linear slot-major bf16
// cache, chunk.cu): rt chunk rows per 128-row tcgen05 tile, n_pairs tile
// pairs, n_split CTAs along each key range, and the partial states (n_split >
// 1: f16 O, fp32 log-sum-exp) the merge combines.
struct ChunkPlan {
    int rt, n_pairs, n_split;
    size_t workspace;
};

void plan_chunk(int batch, int q_rows, int n_q_heads, int n_kv_heads, int head_dim,
                int max_seq_len, int window, ChunkPlan *plan);

// k_new / v_new / slot_mapping non-null: the step's rows are taken from
// k_new / v_new and written to the cache by the same launch (attn_decode_append).
int launch_chunk(const ChunkPlan &plan, const void *q, const attn_kv_cache *cache,
                 const int32_t *seq_lens, const int32_t *positions, int batch, int q_rows,
                 int max_seq_len, int window, int n_q_heads, int n_kv_heads, int head_dim,
                 float scale, void *out, void *workspace, int32_t *err, cudaStream_t stream,
                 const void *k_new = nullptr, const void *v_new = nullptr,
                 const int64_t *slot_mapping = nullptr);

// Decode plan: a persistent grid of one CTA per SM; requests are processed
// in launches of at most batch_per_launch (the per-request tables live in
// shared memory).
struct DecodePlan {
    int head_dim;
    int m_tiles;          // 0: <= 8 rows per unit (keys as MMA rows); 1, 2: 16-row tiles
    int rows;             // q_rows * group
    int row_blocks;       // units along the query rows of one KV head
    int grid;             // CTAs of the split kernel
    int batch_per_launch;
    size_t workspace;     // bytes of scratch: merge counters + fp32 partial states
    size_t counter_offset, counter_bytes;  // the counters, which must be zero between calls
    size_t partial_offset;                 // the partial states (after the counters)
    bool merge_kernel;    // units spanning very many CTAs are merged by a second kernel
    // Many rows per KV group over a linear slot-major bf16 cache go to the
    // tcgen05 chunk kernel instead (not with a fused rotary embedding, which
    // stays on the split kernel: the workspace covers both).
    bool chunk;
    ChunkPlan cp;
    size_t chunk_offset;  // the chunk's partial states, after the split kernel's scratch
};

int plan_decode(const attn_kv_cache *cache, int batch, int q_rows, int n_q_heads, int n_kv_heads,
                int head_dim, int max_seq_len, int window, DecodePlan *plan);

// Every host-side check attn_decode makes before it looks at the workspace;
// on success (and batch > 0) fills *plan.  Returns the attn_status.
int validate_decode(const void *q, const attn_kv_cache *cache, const int32_t *seq_lens,
                    const int32_t *positions, int batch, int q_rows, int max_seq_len, int window,
                    int n_q_heads, int n_kv_heads, int head_dim, float scale, const void *out,
                    DecodePlan *plan);

// k_new / v_new / slot_mapping non-null: the step's rows are appended by the
// same launch (attn_decode_append).
int launch_decode(const DecodePlan &plan, const void *q, const attn_kv_cache *cache,
                  const int32_t *seq_lens, const int32_t *positions, int batch, int q_rows,
                  int max_seq_len, int window, int n_q_heads, int n_kv_heads, float scale,
                  void *out, void *workspace, int32_t *err, cudaStream_t stream,
                  const void *k_new = nullptr, const void *v_new = nullptr,
                  const int64_t *slot_mapping = nullptr, const float *rope_inv_freq = nullptr,
                  bool tables_early = false, bool cache_early = false);

int launch_prefill(const void *q, const void *k, const void *v, int batch, int seq_len,
                   int window, int n_q_heads, int n_kv_heads, int head_dim, float scale,
                   void *out, int32_t *err, cudaStream_t stream);

}  // namespace gqa
