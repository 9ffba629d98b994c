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
//     (cudaGetSymbolAddress, with that device current) and keeps it for that
//     device's current context; make that first call before capturing a
//     stream into a CUDA graph.  An address belongs to one context: when the
//     device's context is replaced (after cudaDeviceReset, say), the next call
//     looks it up again.
//   * The scratch used is the current device's: the stream must belong to it.
//   * All calls share the one array.  Two calls whose kernels overlap on the
//     GPU (different streams, no ordering between them) race on it and give
//     wrong results; order them on one stream or with events.
//   * The decode keeps one counter per (request, KV head, row block) in its
//     scratch, which must start at zero; each call clears them with one
//     stream memset (no allocation) before its kernels run, after every host
//     check has passed (a refused call enqueues nothing).  The memset is not
//     among the kernels attn_decode_kernel_launches counts.  Everything else a
//     previous call left in the array is overwritten before it is read.
#include <cuda.h>
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
struct ScratchAddress {
    unsigned long long ctx_id = 0;  // the context the address belongs to (0: none yet)
    void *ptr = nullptr;
};
ScratchAddress g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

using CtxGetCurrent = CUresult (*)(CUcontext *);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long *);

// The unique id of the calling thread's current context (0 if unknown).
unsigned long long current_context_id() {
    static CtxGetCurrent get_current = nullptr;
    static CtxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault,
                                             &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CtxGetCurrent>(a);
            get_id = reinterpret_cast<CtxGetId>(b);
        }
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch in the current device's current context,
// looked up once per context.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    // 0 when no context is current yet: the lookup below then makes the
    // device's primary context current, and a later call records its id
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddress &a = g_scratch[dev];
    if (a.ptr == nullptr || ctx == 0 || a.ctx_id != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
        a.ptr = p;
        a.ctx_id = ctx;
    }
    *out = a.ptr;
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_decode_noalloc(const void *q, const attn_kv_cache *cache,
                                   const int32_t *seq_lens, const int32_t *positions, int batch,
                                   int q_rows, int max_seq_len, int window, int n_q_heads,
                                   int n_kv_heads, int head_dim, float scale, void *out,
                                   int32_t *err_word, attn_stream_t stream) {
    // every host check first: a refused call enqueues nothing
    gqa::DecodePlan plan;
    const int rc = gqa::validate_decode(q, cache, seq_lens, positions, batch, q_rows, max_seq_len,
                                        window, n_q_heads, n_kv_heads, head_dim, scale, out,
                                        &plan);
    if (rc != ATTN_OK || batch == 0) return rc;
    if (plan.workspace > kNoallocScratchBytes) return ATTN_ERR_WORKSPACE;
    void *scratch = nullptr;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (plan.workspace > 0) {
        const int ra = scratch_address(&scratch);
        if (ra != ATTN_OK) return ra;
        const cudaError_t e = cudaMemsetAsync(static_cast<unsigned char *>(scratch) +
                                                  plan.counter_offset,
                                              0, plan.counter_bytes, s);
        if (e != cudaSuccess) {
            gqa::note_cuda_error(e);
            return ATTN_ERR_CUDA;
        }
    }
    return gqa::launch_decode(plan, q, cache, seq_lens, positions, batch, q_rows, max_seq_len,
                              window, n_q_heads, n_kv_heads, scale, out, scratch, err_word, s);
}
