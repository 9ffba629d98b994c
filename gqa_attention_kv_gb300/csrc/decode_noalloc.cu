// decode_noalloc.cu -- attn_decode_noalloc: the decode entry point for callers
// that cannot allocate device memory.
//
// attn_decode needs a scratch buffer for the partial softmax states of its
// cache splits, and it asks the caller for it.  Some callers cannot provide
// one: a host that hands the library only its input and output tensors and
// has no device allocator of its own, or a real-time loop that must never
// call cudaMalloc (which can synchronise the whole device).  This entry point
// takes the same arguments minus the workspace and uses a fixed scratch array
// that lives in this file as a device global.  It allocates nothing.
//
// Facts a caller needs:
//   * The array holds kNoallocScratchBytes (ATTN_DECODE_NOALLOC_SCRATCH_BYTES)
//     on every GPU that loads this library, until the process exits.
//   * Shapes whose attn_decode_workspace_size exceeds it are refused with
//     ATTN_ERR_WORKSPACE before any launch.
//   * The first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and keeps it; make that
//     first call before capturing a stream into a CUDA graph.
//   * All calls share the one array.  Two calls whose kernels overlap on the
//     GPU (different streams, no ordering between them) race on it and give
//     wrong results; order them on one stream or with events.
//   * The decode keeps one counter per (request, KV head, row block) in its
//     scratch, which must start at zero; each call clears them with a stream
//     memset (no allocation) before its kernel runs.  Everything else a
//     previous call left in the array is overwritten before it is read.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "kernels.h"

namespace {

constexpr size_t kNoallocScratchBytes = ATTN_DECODE_NOALLOC_SCRATCH_BYTES;

// The shared scratch.  In host code this name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch on the current device, looked up once.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        p = g_scratch_ptr[dev].load(std::memory_order_acquire);
        if (p == nullptr) {
            if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return ATTN_ERR_CUDA;
            }
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_decode_noalloc(const void *q, const attn_kv_cache *cache,
                                   const int32_t *seq_lens, const int32_t *positions, int batch,
                                   int q_rows, int max_seq_len, int window, int n_q_heads,
                                   int n_kv_heads, int head_dim, float scale, void *out,
                                   int32_t *err_word, attn_stream_t stream) {
    const size_t need = attn_decode_workspace_size(cache, batch, q_rows, n_q_heads, n_kv_heads,
                                                   head_dim, max_seq_len, window);
    if (need == (size_t)-1) {
        // Invalid arguments: let attn_decode report exactly which.
        return attn_decode(q, cache, seq_lens, positions, batch, q_rows, max_seq_len, window,
                           n_q_heads, n_kv_heads, head_dim, scale, out, nullptr, 0, err_word,
                           stream);
    }
    if (need > kNoallocScratchBytes) return ATTN_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&scratch);
        if (rc != ATTN_OK) return rc;
        gqa::DecodePlan plan;
        gqa::plan_decode(cache, batch, q_rows, n_q_heads, n_kv_heads, head_dim, max_seq_len,
                         window, &plan);
        const cudaError_t e =
            cudaMemsetAsync(static_cast<unsigned char *>(scratch) + plan.counter_offset, 0,
                            plan.counter_bytes, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) {
            gqa::note_cuda_error(e);
            return ATTN_ERR_CUDA;
        }
    }
    return attn_decode(q, cache, seq_lens, positions, batch, q_rows, max_seq_len, window,
                       n_q_heads, n_kv_heads, head_dim, scale, out, scratch,
                       need > 0 ? kNoallocScratchBytes : 0, err_word, stream);
}
