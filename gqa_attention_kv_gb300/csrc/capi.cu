// capi.cu -- the extern "C" entry points declared in include/attn_kv.h:
// argument validation (every host-checkable problem is refused before a
// launch), tensor-map encoding, and dispatch to the kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "kernels.h"

namespace gqa {

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

void note_cuda_error(cudaError_t e) {
    g_last_cuda_error = e;
    cudaGetLastError();  // launch errors are not sticky; clear the runtime's copy
}

cudaError_t last_cuda_error() { return g_last_cuda_error; }

int device_sm_count() {
    static std::atomic<int> counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int c = counts[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
            c = 148;
        counts[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool encode_tensor_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                       const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128,
                       bool bytes) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    CUresult r = fn(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    (cuuint32_t)rank,
                    const_cast<void *>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    // an E4M3 head row is 128 bytes: a 256-byte fill would also pull
                    // the next head's row, which another CTA reads much later
                    bytes ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tensor_map_f16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                           const uint64_t *strides_bytes, const uint32_t *box) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void *>(base), gd,
              gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gqa

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool heads_ok(int n_q_heads, int n_kv_heads, int head_dim) {
    return n_kv_heads >= 1 && n_q_heads >= 1 && n_q_heads % n_kv_heads == 0 &&
           (head_dim == 64 || head_dim == 128);
}

// The layout fields: a known layout, and for the head-major one whole blocks.
int check_layout(const attn_kv_cache *c) {
    if (c->layout == ATTN_LAYOUT_BSHD) return ATTN_OK;
    if (c->layout != ATTN_LAYOUT_BHSD) return ATTN_ERR_UNSUPPORTED;
    const int64_t rows = c->kind == ATTN_CACHE_PAGED ? c->block_size : c->slots_per_seq;
    if (c->kind != ATTN_CACHE_LINEAR && c->kind != ATTN_CACHE_PAGED && c->kind != ATTN_CACHE_RING)
        return ATTN_ERR_SHAPE;
    if (rows < 1 || c->num_slots % rows != 0) return ATTN_ERR_SHAPE;
    return ATTN_OK;
}

// Validation shared by attn_decode and attn_decode_workspace_size.
int check_decode_shape(const attn_kv_cache *cache, int batch, int q_rows, int n_q_heads,
                       int n_kv_heads, int head_dim, int max_seq_len, int window) {
    if (!cache) return ATTN_ERR_NULL;
    if (batch < 0 || q_rows < 1 || max_seq_len < 1) return ATTN_ERR_SHAPE;
    if (!heads_ok(n_q_heads, n_kv_heads, head_dim)) {
        if (n_kv_heads >= 1 && n_q_heads >= 1 && n_q_heads % n_kv_heads == 0)
            return ATTN_ERR_UNSUPPORTED;  // head_dim other than 64 / 128
        return ATTN_ERR_SHAPE;
    }
    if (cache->num_slots < 1 || cache->num_slots >= (int64_t(1) << 31)) return ATTN_ERR_SHAPE;
    if (cache->dtype != ATTN_KV_BF16 && cache->dtype != ATTN_KV_FP8_E4M3)
        return ATTN_ERR_UNSUPPORTED;
    if (cache->dtype == ATTN_KV_FP8_E4M3 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (int rc = check_layout(cache); rc != ATTN_OK) return rc;
    if (cache->layout == ATTN_LAYOUT_BHSD &&
        (cache->num_slots / (cache->kind == ATTN_CACHE_PAGED ? cache->block_size
                                                              : cache->slots_per_seq)) *
                n_kv_heads >= (int64_t(1) << 31))
        return ATTN_ERR_SHAPE;
    switch (cache->kind) {
    case ATTN_CACHE_LINEAR:
        if (cache->slots_per_seq < 1 ||
            (int64_t)batch * cache->slots_per_seq > cache->num_slots)
            return ATTN_ERR_SHAPE;
        break;
    case ATTN_CACHE_PAGED:
        if (cache->block_size < 1 || cache->max_blocks_per_seq < 1) return ATTN_ERR_SHAPE;
        if ((int64_t)cache->max_blocks_per_seq * cache->block_size < max_seq_len)
            return ATTN_ERR_SHAPE;
        break;
    case ATTN_CACHE_RING:
        // Writes land before attention, so a ring must keep the window of the
        // step's first row alive while the step's rows are written
        // (Voxtral notes, "Encoder KV cache": the buffer is twice the window).
        if (window <= 0 || cache->slots_per_seq < 1) return ATTN_ERR_SHAPE;
        if ((int64_t)cache->slots_per_seq < (int64_t)window + q_rows - 1) return ATTN_ERR_SHAPE;
        if ((int64_t)batch * cache->slots_per_seq > cache->num_slots) return ATTN_ERR_SHAPE;
        break;
    default:
        return ATTN_ERR_SHAPE;
    }
    return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping, int64_t n,
                   const attn_kv_cache *cache, int n_kv_heads, int head_dim, int32_t *err_word,
                   attn_stream_t stream) {
    if (!cache) return ATTN_ERR_NULL;
    if (n < 0 || n_kv_heads < 1) return ATTN_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128) return ATTN_ERR_UNSUPPORTED;
    if (n == 0) return ATTN_OK;
    if (!k_new || !v_new || !slot_mapping || !cache->k || !cache->v) return ATTN_ERR_NULL;
    if (cache->num_slots < 1) return ATTN_ERR_SHAPE;
    if (int rc = check_layout(cache); rc != ATTN_OK) return rc;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(cache->k) || !aligned16(cache->v))
        return ATTN_ERR_ALIGN;
    if (cache->dtype == ATTN_KV_FP8_E4M3) {
        if (head_dim != 128) return ATTN_ERR_UNSUPPORTED;
        if (cache->k_ref && !aligned16(cache->k_ref)) return ATTN_ERR_ALIGN;
        return gqa::launch_kv_append_fp8(k_new, v_new, cache->k_ref, slot_mapping, n, cache->k,
                                         cache->v, cache->num_slots,
                                         gqa::kv_place(cache, n_kv_heads, head_dim, 1), err_word,
                                         reinterpret_cast<cudaStream_t>(stream));
    }
    if (cache->dtype != ATTN_KV_BF16) return ATTN_ERR_UNSUPPORTED;
    return gqa::launch_kv_append(k_new, v_new, slot_mapping, n, cache->k, cache->v,
                                 cache->num_slots, gqa::kv_place(cache, n_kv_heads, head_dim, 2),
                                 err_word, reinterpret_cast<cudaStream_t>(stream));
}

int attn_kv_reference(const void *k, int64_t n, int n_kv_heads, int head_dim, float *ref,
                      attn_stream_t stream) {
    if (n < 1 || n_kv_heads < 1 || head_dim < 1) return ATTN_ERR_SHAPE;
    if ((int64_t)n_kv_heads * head_dim >= (int64_t(1) << 31)) return ATTN_ERR_SHAPE;
    if (!k || !ref) return ATTN_ERR_NULL;
    if (!aligned16(k) || !aligned16(ref)) return ATTN_ERR_ALIGN;
    return gqa::launch_kv_reference(k, n, n_kv_heads * head_dim, ref,
                                    reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_decode_workspace_size(const attn_kv_cache *cache, int batch, int q_rows,
                                  int n_q_heads, int n_kv_heads, int head_dim, int max_seq_len,
                                  int window) {
    if (check_decode_shape(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len,
                           window) != ATTN_OK)
        return (size_t)-1;
    if (batch == 0) return 0;
    gqa::DecodePlan plan;
    gqa::plan_decode(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len, window,
                     &plan);
    return plan.workspace;
}

int attn_decode_kernel_launches(const attn_kv_cache *cache, int batch, int q_rows, int n_q_heads,
                                int n_kv_heads, int head_dim, int max_seq_len, int window,
                                int with_append, int with_rope, unsigned flags) {
    if ((flags & ~(ATTN_DECODE_TABLES_EARLY | ATTN_DECODE_CACHE_EARLY)) != 0) return -1;
    if (check_decode_shape(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len,
                           window) != ATTN_OK)
        return -1;
    if (batch == 0) return 0;
    gqa::DecodePlan plan;
    gqa::plan_decode(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len, window,
                     &plan);
    if (plan.chunk && !with_rope) return 1 + (plan.cp.n_split > 1 ? 1 : 0);
    const int splits = (batch + plan.batch_per_launch - 1) / plan.batch_per_launch;
    return splits * (plan.merge_kernel ? 2 : 1);
}

}  // extern "C"

namespace gqa {

int validate_decode(const void *q, const attn_kv_cache *cache, const int32_t *seq_lens,
                    const int32_t *positions, int batch, int q_rows, int max_seq_len, int window,
                    int n_q_heads, int n_kv_heads, int head_dim, float scale, const void *out,
                    DecodePlan *plan) {
    int rc = check_decode_shape(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim,
                                max_seq_len, window);
    if (rc != ATTN_OK) return rc;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_SHAPE;
    if (batch == 0) return ATTN_OK;
    if (!q || !seq_lens || !positions || !out || !cache->k || !cache->v) return ATTN_ERR_NULL;
    if (cache->kind == ATTN_CACHE_PAGED && !cache->block_table) return ATTN_ERR_NULL;
    if (!aligned16(q) || !aligned16(out) || !aligned16(cache->k) || !aligned16(cache->v))
        return ATTN_ERR_ALIGN;
    plan_decode(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len, window, plan);
    return ATTN_OK;
}

}  // namespace gqa

extern "C" {

int attn_decode(const void *q, const attn_kv_cache *cache, const int32_t *seq_lens,
                const int32_t *positions, int batch, int q_rows, int max_seq_len, int window,
                int n_q_heads, int n_kv_heads, int head_dim, float scale, void *out,
                void *workspace, size_t workspace_bytes, int32_t *err_word,
                attn_stream_t stream) {
    gqa::DecodePlan plan;
    const int rc = gqa::validate_decode(q, cache, seq_lens, positions, batch, q_rows, max_seq_len,
                                        window, n_q_heads, n_kv_heads, head_dim, scale, out,
                                        &plan);
    if (rc != ATTN_OK || batch == 0) return rc;
    if (plan.workspace > 0) {
        if (!workspace) return ATTN_ERR_NULL;
        if (workspace_bytes < plan.workspace) return ATTN_ERR_WORKSPACE;
        if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
    }
    return gqa::launch_decode(plan, q, cache, seq_lens, positions, batch, q_rows, max_seq_len,
                              window, n_q_heads, n_kv_heads, scale, out, workspace, err_word,
                              reinterpret_cast<cudaStream_t>(stream));
}

int attn_decode_append(const void *q, const void *k_new, const void *v_new,
                       const int64_t *slot_mapping, const float *rope_inv_freq,
                       const attn_kv_cache *cache,
                       const int32_t *seq_lens, const int32_t *positions, int batch, int q_rows,
                       int max_seq_len, int window, int n_q_heads, int n_kv_heads, int head_dim,
                       float scale, void *out, void *workspace, size_t workspace_bytes,
                       int32_t *err_word, unsigned flags, attn_stream_t stream) {
    int rc = check_decode_shape(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim,
                                max_seq_len, window);
    if (rc != ATTN_OK) return rc;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_SHAPE;
    if ((flags & ~(ATTN_DECODE_TABLES_EARLY | ATTN_DECODE_CACHE_EARLY)) != 0)
        return ATTN_ERR_UNSUPPORTED;
    // FP8 caches: the rows are encoded as attn_kv_append encodes them; the
    // rotary embedding is not combined with them here
    if (cache->dtype == ATTN_KV_FP8_E4M3 && rope_inv_freq) return ATTN_ERR_UNSUPPORTED;
    if (cache->dtype == ATTN_KV_FP8_E4M3 && cache->k_ref && !aligned16(cache->k_ref))
        return ATTN_ERR_ALIGN;
    if (batch == 0) return ATTN_OK;
    if (!q || !k_new || !v_new || !slot_mapping || !seq_lens || !positions || !out ||
        !cache->k || !cache->v)
        return ATTN_ERR_NULL;
    if (cache->kind == ATTN_CACHE_PAGED && !cache->block_table) return ATTN_ERR_NULL;
    if (!aligned16(q) || !aligned16(out) || !aligned16(cache->k) || !aligned16(cache->v) ||
        !aligned16(k_new) || !aligned16(v_new))
        return ATTN_ERR_ALIGN;
    gqa::DecodePlan plan;
    gqa::plan_decode(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len, window,
                     &plan);
    if (plan.workspace > 0) {
        if (!workspace) return ATTN_ERR_NULL;
        if (workspace_bytes < plan.workspace) return ATTN_ERR_WORKSPACE;
        if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
    }
    return gqa::launch_decode(plan, q, cache, seq_lens, positions, batch, q_rows, max_seq_len,
                              window, n_q_heads, n_kv_heads, scale, out, workspace, err_word,
                              reinterpret_cast<cudaStream_t>(stream), k_new, v_new, slot_mapping,
                              rope_inv_freq, (flags & ATTN_DECODE_TABLES_EARLY) != 0,
                              (flags & ATTN_DECODE_CACHE_EARLY) != 0);
}

int attn_prefill(const void *q, const void *k, const void *v, int batch, int seq_len, int window,
                 int n_q_heads, int n_kv_heads, int head_dim, float scale, void *out,
                 int32_t *err_word, attn_stream_t stream) {
    if (batch < 0 || seq_len < 0) return ATTN_ERR_SHAPE;
    if (!heads_ok(n_q_heads, n_kv_heads, head_dim)) {
        if (n_kv_heads >= 1 && n_q_heads >= 1 && n_q_heads % n_kv_heads == 0)
            return ATTN_ERR_UNSUPPORTED;
        return ATTN_ERR_SHAPE;
    }
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_SHAPE;
    if (batch == 0 || seq_len == 0) return ATTN_OK;
    if (!q || !k || !v || !out) return ATTN_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_ALIGN;
    const int64_t tiles = ((int64_t)seq_len + 127) / 128 * n_q_heads * (int64_t)batch;
    if (tiles >= (int64_t(1) << 31)) return ATTN_ERR_SHAPE;
    return gqa::launch_prefill(q, k, v, batch, seq_len, window, n_q_heads, n_kv_heads, head_dim,
                               scale, out, err_word, reinterpret_cast<cudaStream_t>(stream));
}

const char *attn_status_string(int status) {
    switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "inconsistent or out-of-range sizes";
    case ATTN_ERR_UNSUPPORTED:
        return "unsupported request (head_dim other than 64 / 128, an FP8 cache where it is not "
               "implemented, an unknown dtype or flag)";
    case ATTN_ERR_WORKSPACE: return "workspace too small";
    case ATTN_ERR_BOUNDS: return "slot, page or position outside its buffer";
    case ATTN_ERR_TIMEOUT: return "a bounded device wait gave up";
    case ATTN_ERR_CUDA: return "the CUDA runtime rejected a launch";
    case ATTN_ERR_ALIGN: return "a base pointer is not 16-byte aligned";
    default: return "unknown status";
    }
}

const char *attn_version(void) { return "gqa_attention_kv_gb300 0.1.0 (sm_103a)"; }

const char *attn_last_cuda_error(void) {
    return cudaGetErrorString(gqa::last_cuda_error());
}

}  // extern "C"
