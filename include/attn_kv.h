/*
 * attn_kv.h -- C ABI of the GB300 grouped-query attention library.
 *
 * Three operations on one decoder KV cache, each a few kernel launches on the
 * caller's stream:
 *
 *   attn_kv_append  write new K/V rows into the cache slots a slot_mapping names
 *   attn_decode     causal decode attention, 1..K query rows per request, over a
 *                   linear, paged (block-table) or ring-buffer (sliding-window)
 *                   cache, as a split-KV flash-decode plus a merge of the
 *                   partial softmax states
 *   attn_prefill    causal (optionally windowed) GQA prefill attention
 *
 * Sources for the operations (cited by page title and section):
 *   - vibevoice.c, "The kernels that matter", "Attention backends", "Paged KV
 *     cache", "The decode step is one submission": split-KV decode whose
 *     partial softmax states a second kernel merges, all query heads of a GQA
 *     group reading a cache position once, a device-side page table, and the
 *     step's moving parts (where new K/V land, how far attention walks) read
 *     from device memory so a captured CUDA graph replays.
 *   - Voxtral Realtime -- Architecture & Design Notes, "KV cache", "SDPA",
 *     "Attention layout", "Encoder KV cache": [B, S, H, D] caches, GQA by head
 *     ratio, ring buffers sized 2x the window, the analytic ring position and
 *     the sliding-window mask  valid = (t >= 0) & (pos - t >= 0) &
 *     (pos - t < window).
 *   - talker_multiframe (vLLM-Omni NPU worker), "How a frame advances without
 *     the host" and the NarrowStep fields: K sequential query rows per request
 *     with positions, slot_mapping, seq_lens and an unchanged block table.
 *
 * Conventions shared by every entry point:
 *   - All tensors are bf16 (16-bit words) unless stated otherwise, row-major,
 *     last dimension contiguous, in DEVICE memory, and owned by the caller.
 *     Every base pointer must be 16-byte aligned (ATTN_ERR_ALIGN otherwise).
 *   - The library never allocates, frees or synchronises, and launches only on
 *     the stream it is given (never the legacy default stream unless the
 *     caller passes 0).
 *   - Host-checkable problems (null pointers, bad sizes, unsupported shapes,
 *     too small a workspace) return a nonzero attn_status BEFORE any launch.
 *   - Data-dependent problems found on the device (a slot, page or position
 *     outside its buffer) never fault: the offending row or key is skipped and,
 *     when err_word is not NULL, the first such error code is stored there
 *     (atomically; a zero word stays zero when nothing went wrong).  Every
 *     device-side wait is bounded; one that gives up stores ATTN_ERR_TIMEOUT.
 *     The caller clears *err_word and reads it back when it wants to know.
 *   - A return of ATTN_ERR_CUDA means a launch was rejected by the runtime.
 *   - Head mapping: query head h reads KV head h / (n_q_heads / n_kv_heads).
 *   - head_dim must be 64 or 128.
 */
#ifndef GQA_ATTN_KV_H
#define GQA_ATTN_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *attn_stream_t; /* a cudaStream_t */

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,        /* a required pointer is NULL */
    ATTN_ERR_SHAPE = 2,       /* sizes inconsistent or out of range */
    ATTN_ERR_UNSUPPORTED = 3, /* a valid request this build does not implement; on the device
                                 (err_word): a value outside the range a kernel supports */
    ATTN_ERR_WORKSPACE = 4,   /* workspace smaller than attn_decode_workspace_size */
    ATTN_ERR_BOUNDS = 5,      /* device: slot / page / position outside its buffer */
    ATTN_ERR_TIMEOUT = 6,     /* device: a bounded wait gave up */
    ATTN_ERR_CUDA = 7,        /* the CUDA runtime rejected a launch */
    ATTN_ERR_ALIGN = 8        /* a base pointer is not 16-byte aligned */
} attn_status;

typedef enum {
    ATTN_CACHE_LINEAR = 0, /* request b, position t -> slot b*slots_per_seq + t */
    ATTN_CACHE_PAGED = 1,  /* -> block_table[b][t / block_size]*block_size + t % block_size */
    ATTN_CACHE_RING = 2    /* -> slot b*slots_per_seq + t % slots_per_seq (ring of that size) */
} attn_cache_kind;

typedef enum {
    ATTN_LAYOUT_BSHD = 0, /* slot-major: element (slot, head, d) at (slot*n_kv_heads + head)*head_dim + d */
    ATTN_LAYOUT_BHSD = 1  /* head-major inside each block of `rows` slots (see attn_kv_cache) */
} attn_kv_layout;

typedef enum {
    ATTN_KV_BF16 = 0,    /* 16-bit bf16 elements */
    ATTN_KV_FP8_E4M3 = 1 /* 8-bit E4M3 elements, K stored relative to k_ref */
} attn_kv_dtype;

/*
 * One layer's KV cache.  k and v are [num_slots, n_kv_heads, head_dim]
 * elements of the cache's dtype (the pages' [B, S, H, D] layout with requests
 * and positions flattened into slots).  The struct itself is read on the host
 * during the call only.
 *
 *   LINEAR: slots_per_seq = capacity of each request's window.
 *   PAGED : block_table is a DEVICE int32 [batch, max_blocks_per_seq] array of
 *           page ids; page p covers slots p*block_size .. p*block_size +
 *           block_size - 1.  block_size >= 1.  The table may change between
 *           calls (a captured graph follows it).
 *   RING  : slots_per_seq = ring size R; position t of request b lives in slot
 *           b*R + t % R.  A ring holds the last R positions written.
 *
 * dtype ATTN_KV_FP8_E4M3 (vibevoice.c, "KV cache": the cache stored as 8-bit
 * floats to halve its size, K relative to a per-layer reference vector): each
 * element is one byte in the E4M3 format of the OCP 8-bit floating point
 * specification (bias 7, no infinities, 0x7F / 0xFF NaN, largest finite 448),
 * with no scale factor.  attn_kv_append stores
 *     k_cache = E4M3(float32(k) - k_ref[head][d]),  v_cache = E4M3(float32(v)),
 * rounding to nearest even and saturating to +-448; k_ref (float32
 * [n_kv_heads][head_dim], device; NULL: no shift) is usually the mean of the
 * first prefill chunk's keys (attn_kv_reference).  Subtracting one vector from
 * every key of a head adds the same amount to all of a query row's scores, so
 * attention reads the stored keys as they are and needs no k_ref.  FP8 caches
 * require head_dim 128.
 *
 * layout ATTN_LAYOUT_BHSD (Voxtral notes, "KV cache": the CUDA path keeps its
 * static and ring caches as [B, H, S, D]): the slots form blocks of `rows`
 * consecutive slots -- rows = slots_per_seq for LINEAR and RING (a block is a
 * request), block_size for PAGED (a block is a page) -- and each block stores
 * its heads one after another: element (slot s, head h, d) lives at
 *     ((s / rows) * n_kv_heads + h) * rows + s % rows) * head_dim + d.
 * Slot numbers, slot_mapping and block tables mean exactly what they mean for
 * the slot-major layout; only the placement differs, so one KV head's keys of
 * a block are contiguous.  num_slots must be a multiple of rows.
 * A zero-initialised struct is a bf16, slot-major cache.
 */
typedef struct {
    int32_t kind;               /* attn_cache_kind */
    void *k;                    /* [num_slots, n_kv_heads, head_dim] of dtype */
    void *v;                    /* [num_slots, n_kv_heads, head_dim] of dtype */
    int64_t num_slots;
    int32_t slots_per_seq;      /* LINEAR capacity, RING size; unused for PAGED */
    const int32_t *block_table; /* PAGED only, device */
    int32_t block_size;         /* PAGED only */
    int32_t max_blocks_per_seq; /* PAGED only: row length of block_table */
    int32_t dtype;              /* attn_kv_dtype */
    const float *k_ref;         /* FP8 only: float32 [n_kv_heads, head_dim], device, or NULL */
    int32_t layout;             /* attn_kv_layout */
} attn_kv_cache;

/*
 * attn_kv_append -- cache.k[slot_mapping[i]] = k_new[i]; same for v.
 *
 * Source: the step writes its new K/V before attention reads them (Voxtral
 * notes, "Encoder KV cache": writes happen before attention), into the slot the
 * engine reserved for each new row (talker_multiframe, NarrowStep field
 * slot_mapping[r]); the slot is a device value so a replayed graph lands each
 * step's row in its own place (vibevoice.c, "The decode step is one
 * submission").
 *
 *   k_new, v_new  bf16 [n, n_kv_heads, head_dim], device
 *   slot_mapping  int64 [n], device; a slot outside [0, cache->num_slots) skips
 *                 its row and stores ATTN_ERR_BOUNDS in *err_word
 *   n             rows to write (0 is a no-op)
 * Copies are bit-exact.  With a slot repeated inside one call, which row lands
 * is unspecified.  Slots are absolute: cache->kind matters only for the
 * head-major layout, whose block size it selects.  For an FP8
 * cache the rows are converted as attn_kv_cache states (bit-exact against
 * that definition), and k_new / v_new stay bf16.
 */
int attn_kv_append(const void *k_new, const void *v_new, const int64_t *slot_mapping, int64_t n,
                   const attn_kv_cache *cache, int n_kv_heads, int head_dim, int32_t *err_word,
                   attn_stream_t stream);

/*
 * attn_kv_reference -- the FP8 cache's reference vector: ref[h][d] = mean over
 * the n rows of k[i][h][d] (vibevoice.c, "KV cache": a per-layer reference
 * built from the first prefill chunk).
 *
 *   k     bf16 [n, n_kv_heads, head_dim], device, 16-byte aligned; n >= 1
 *   ref   float32 [n_kv_heads, head_dim], device, written: the sum is taken in
 *         fp64 in a fixed order and divided by n, then rounded once to
 *         float32, so the result does not depend on timing.
 */
int attn_kv_reference(const void *k, int64_t n, int n_kv_heads, int head_dim, float *ref,
                      attn_stream_t stream);

/*
 * attn_decode_workspace_size -- bytes of device scratch attn_decode needs for
 * this shape: merge counters, then partial softmax states of the key pieces
 * different CTAs handle (fp32; a prefill chunk's partial O in f16).  A call accepts any workspace at least this
 * large.  Returns (size_t)-1 for arguments attn_decode would reject.
 *
 * The workspace must be zero-filled before its first use; every call that
 * completes leaves the counters at zero again, so a workspace kept for later
 * calls needs no clearing (after a call that reported ATTN_ERR_TIMEOUT,
 * zero it again).  The counters sit at the start, in a region whose size
 * depends only on n_kv_heads and the GPU (for groups of up to 256 row
 * blocks), with the partial states after it: one workspace, sized for the
 * largest shape, serves calls of every batch size, row count and context of
 * a model without clearing.
 */
size_t attn_decode_workspace_size(const attn_kv_cache *cache, int batch, int q_rows,
                                  int n_q_heads, int n_kv_heads, int head_dim, int max_seq_len,
                                  int window);

/*
 * attn_decode_kernel_launches -- how many kernels one call with these
 * arguments launches on the stream (host only; nothing is launched):
 * attn_decode when with_append is 0, attn_decode_append when it is 1, with a
 * rotary embedding when with_rope is 1, with attn_decode_append's flags (no
 * flag changes the count today; an unknown flag gives -1).  A split-kernel
 * call launches one split kernel per group of requests the shared-memory
 * tables hold, each followed by the merge kernel when units of this shape may
 * be split over enough CTAs to need it.  A group of 64 or more query rows (q_rows x
 * n_q_heads / n_kv_heads) over a linear slot-major bf16 cache, without a
 * rotary embedding, is a prefill chunk: the tcgen05 chunk kernel (which, for
 * attn_decode_append, also takes the step's rows from k_new / v_new and writes
 * them to the cache), and its merge kernel when the key range is split over
 * CTAs.  Returns -1 for arguments attn_decode would reject, 0 for
 * batch 0.
 */
int attn_decode_kernel_launches(const attn_kv_cache *cache, int batch, int q_rows, int n_q_heads,
                                int n_kv_heads, int head_dim, int max_seq_len, int window,
                                int with_append, int with_rope, unsigned flags);

/*
 * attn_decode -- causal decode attention for q_rows query rows per request.
 *
 * Source: vibevoice.c, "The kernels that matter" / "Attention backends"
 * (split-KV decode whose partial softmax states are merged by a second kernel;
 * the heads of a GQA group read each cache position once); talker_multiframe,
 * NarrowStep fields (K sequential query rows per request, positions[r],
 * seq_lens[r] = keys written, the block table); Voxtral notes, "Encoder KV
 * cache" (the sliding-window mask and the ring).
 *
 *   q          bf16 [batch, q_rows, n_q_heads, head_dim], device
 *   cache      the layer's cache (see attn_kv_cache)
 *   seq_lens   int32 [batch], device: keys written for each request, this
 *              step's rows included
 *   positions  int32 [batch*q_rows], device: absolute position of each query
 *              row.  Row (b, r) attends key position t iff
 *                  0 <= t < seq_lens[b],  t <= positions[b*q_rows + r],
 *                  window <= 0 or positions[...] - t < window,
 *                  RING: t >= seq_lens[b] - slots_per_seq (still in the ring).
 *              For LINEAR and PAGED caches a step's rows are normally
 *              positions seq_len - q_rows + r.
 *   batch, q_rows   >= 1 (batch 0 is a no-op)
 *   max_seq_len     host-side upper bound of seq_lens[]; it sizes the grid
 *              (the split count) only, so a graph captured for one bound
 *              replays for any seq_lens up to it.  Keys beyond it are not read.
 *   window     sliding window in positions; <= 0 means none.  RING requires
 *              window > 0 and slots_per_seq >= window + q_rows - 1.
 *   scale      multiplies q.k before the natural-base softmax; finite and > 0
 *   out        bf16 [batch, q_rows, n_q_heads, head_dim], device; rounded
 *              once from fp32 (round to nearest even).  A row with no valid
 *              key gets zeros.
 *   workspace  device scratch of at least attn_decode_workspace_size(...)
 *              bytes, 16-byte aligned, zero-filled before its first use (see
 *              attn_decode_workspace_size).  Calls whose kernels overlap on
 *              the GPU need separate workspaces.
 *   An FP8 cache (head_dim 128) is read as stored: the decode converts keys
 *   and values to f16 (exact), takes q in f16 (|q| must stay below 65504;
 *   magnitudes under 2^-14 lose precision) and the softmax weights in f16,
 *   and accumulates in fp32.
 *   A group of 64 or more query rows (q_rows x n_q_heads / n_kv_heads) over a
 *   linear slot-major bf16 cache is a prefill chunk and computes as
 *   attn_prefill does: P V from f16 softmax weights and f16 values, with the
 *   same range rule for v (a magnitude of 2^16 or more is saturated and
 *   reported as ATTN_ERR_UNSUPPORTED in *err_word).
 */
int attn_decode(const void *q, const attn_kv_cache *cache, const int32_t *seq_lens,
                const int32_t *positions, int batch, int q_rows, int max_seq_len, int window,
                int n_q_heads, int n_kv_heads, int head_dim, float scale, void *out,
                void *workspace, size_t workspace_bytes, int32_t *err_word,
                attn_stream_t stream);

/*
 * attn_decode_append -- the step's KV append and its decode in one launch.
 *
 * Source: vibevoice.c, "The decode step is one submission" (the new K/V row
 * lands at a device-side slot inside the captured step, before attention);
 * talker_multiframe, NarrowStep fields (a step writes its K rows, then
 * attends).  Same result as
 *     attn_kv_append(k_new, v_new, slot_mapping, batch * q_rows, cache, ...);
 *     attn_decode(q, cache, seq_lens, positions, ...);
 * when the step's rows follow the position contract: new row b*q_rows + r is
 * the key at position seq_lens[b] - q_rows + r, and slot_mapping of that row
 * is its slot in the cache.  The decode takes those keys from k_new / v_new
 * directly, so it never waits for the cache writes; the cache rows are
 * written by the same launch for later steps.
 *
 *   k_new, v_new   bf16 [batch * q_rows, n_kv_heads, head_dim], device,
 *                  16-byte aligned
 *   slot_mapping   int64 [batch * q_rows], device.  A slot outside
 *                  [0, num_slots) is skipped and reported as ATTN_ERR_BOUNDS
 *                  in *err_word.
 *   rope_inv_freq  float32 [head_dim / 2], device, or NULL for none: rotary
 *                  embedding of q and k_new before use (Voxtral notes,
 *                  "RoPE" and "Shared Patterns"): the interleaved pairs
 *                  (x[2i], x[2i+1]) of every head of a row at position p are
 *                  rotated by the float32 angle p * rope_inv_freq[i], in
 *                  float32, and rounded to bf16; the cache receives the
 *                  rotated keys.  q row (b, r) uses positions[b*q_rows + r],
 *                  new key row b*q_rows + r the position seq_lens[b] - q_rows + r.
 *   flags          0, or ATTN_DECODE_TABLES_EARLY: seq_lens, positions and the
 *                  block table are not written by any kernel that may still
 *                  be running when this call is issued (normally: not by the
 *                  kernel issued just before it), so the call may read them
 *                  (and plan its work) while that kernel finishes, under
 *                  programmatic dependent launch, and bring the first tiles
 *                  of its cache reads into L2 meanwhile.  Everything else is
 *                  still read after the previous kernel completes.
 *                  ATTN_DECODE_CACHE_EARLY (implies TABLES_EARLY): in
 *                  addition, no cache slot other than the ones this call
 *                  appends is written by a kernel that may still be running,
 *                  so the call may also start loading the first cache tiles
 *                  of its work into shared memory before the previous kernel
 *                  completes (the step's own rows are taken from k_new /
 *                  v_new after it).  Normal in a decode loop whose previous
 *                  kernel produces q, k_new and v_new; wrong if that kernel
 *                  wrote other rows of this cache.
 *   Every other argument, the workspace and the statuses are attn_decode's.
 *   An FP8 cache receives the rows encoded exactly as attn_kv_append encodes
 *   them (K minus k_ref), and the decode reads those codes; rope_inv_freq must
 *   then be NULL (ATTN_ERR_UNSUPPORTED otherwise).
 */
#define ATTN_DECODE_TABLES_EARLY 1u
#define ATTN_DECODE_CACHE_EARLY 2u
int attn_decode_append(const void *q, const void *k_new, const void *v_new,
                       const int64_t *slot_mapping, const float *rope_inv_freq,
                       const attn_kv_cache *cache,
                       const int32_t *seq_lens, const int32_t *positions, int batch, int q_rows,
                       int max_seq_len, int window, int n_q_heads, int n_kv_heads, int head_dim,
                       float scale, void *out, void *workspace, size_t workspace_bytes,
                       int32_t *err_word, unsigned flags, attn_stream_t stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to it.
 *
 * attn_decode asks the caller for scratch space.  A caller that has no device
 * allocator (it receives only its input and output tensors from its host), or
 * that must never call cudaMalloc in its decode loop (an allocation can
 * synchronise the whole device), calls this instead: same arguments without
 * the workspace; the scratch is a fixed device array of
 * ATTN_DECODE_NOALLOC_SCRATCH_BYTES inside the library, present on every GPU
 * that loads the library until the process exits.  Nothing is allocated.
 *
 *   Returns ATTN_ERR_WORKSPACE, before any launch, when
 *   attn_decode_workspace_size(...) for these arguments exceeds that size;
 *   otherwise the same statuses as attn_decode, every host check made before
 *   anything is enqueued.
 *   The array used is the CURRENT device's: the stream must belong to the
 *   current device.  The first call on a device looks up the array's device
 *   address, which belongs to the device's current context (a replaced
 *   context, after cudaDeviceReset for instance, is looked up again); make
 *   that first call before capturing a stream into a CUDA graph.
 *   All calls share the array: calls whose kernels overlap on the GPU race
 *   and give wrong results, so order them (one stream, or events).  Each
 *   call enqueues one memset on the stream (no allocation), clearing the
 *   part of the array that must start at zero, before its kernels; that
 *   memset is not counted by attn_decode_kernel_launches.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int attn_decode_noalloc(const void *q, const attn_kv_cache *cache, const int32_t *seq_lens,
                        const int32_t *positions, int batch, int q_rows, int max_seq_len,
                        int window, int n_q_heads, int n_kv_heads, int head_dim, float scale,
                        void *out, int32_t *err_word, attn_stream_t stream);

/*
 * attn_prefill -- causal GQA self-attention over whole sequences.
 *
 * Source: vibevoice.c, "Prefill attention" and "Attention backends" (causal
 * attention with both contractions on the tensor cores and the heads of a GQA
 * group sharing K/V tiles); Voxtral notes, "Offline Encoder" (causal SDPA over
 * the whole input, head_dim 64, and the 750-frame sliding window that only
 * matters beyond 750 frames).
 *
 *   q    bf16 [batch, seq_len, n_q_heads, head_dim], device
 *   k, v bf16 [batch, seq_len, n_kv_heads, head_dim], device
 *   Query i of a sequence attends keys t of the same sequence with t <= i and,
 *   when window > 0, i - t < window.  scale (finite, > 0) multiplies q.k.
 *   out  bf16 [batch, seq_len, n_q_heads, head_dim], device, rounded once.
 *   Q K^T takes q and k as bf16.  P V takes the softmax weights rounded once to
 *   f16 and v converted to f16 (vibevoice.c, "Attention backends": P V in
 *   FP16, since one bf16 rounding of P is too coarse); fp32 accumulation.  The
 *   conversion of v is exact for magnitudes in [2^-14, 2^16) and keeps an
 *   absolute precision of 2^-24 below; a v element of magnitude 2^16 or more
 *   has no f16 value: it is saturated to +-65504 and ATTN_ERR_UNSUPPORTED is
 *   stored in *err_word.
 */
int attn_prefill(const void *q, const void *k, const void *v, int batch, int seq_len, int window,
                 int n_q_heads, int n_kv_heads, int head_dim, float scale, void *out,
                 int32_t *err_word, attn_stream_t stream);

/* Human-readable name of an attn_status. */
const char *attn_status_string(int status);

/* Library version string. */
const char *attn_version(void);

/* Text of the last CUDA runtime error that made a call of this thread return
 * ATTN_ERR_CUDA ("no error" if there was none). */
const char *attn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_KV_H */
