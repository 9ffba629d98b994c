"""GB300 grouped-query attention over a decoder KV cache.

A thin ctypes binding over the C ABI in ``include/attn_kv.h`` (library
``libgqa_attn_kv.so``, built in-tree by ``gqa_attention_kv_gb300.build``).
Every function here only marshals arguments -- pointers, sizes and the
current CUDA stream -- and calls the entry point of the same name; all work
runs in the library's kernels.  There is no fallback: if the library is
missing or a call is refused, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .synth import LINEAR, PAGED, RING  # noqa: F401  (cache-kind constants)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_attn_kv.so")

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_NULL", 2: "ATTN_ERR_SHAPE", 3: "ATTN_ERR_UNSUPPORTED",
                4: "ATTN_ERR_WORKSPACE", 5: "ATTN_ERR_BOUNDS", 6: "ATTN_ERR_TIMEOUT",
                7: "ATTN_ERR_CUDA", 8: "ATTN_ERR_ALIGN"}
for _code, _name in STATUS_NAMES.items():
    globals()[_name] = _code
ATTN_DECODE_TABLES_EARLY = 1  # attn_decode_append flags (include/attn_kv.h)
ATTN_DECODE_CACHE_EARLY = 2
ATTN_KV_BF16, ATTN_KV_FP8_E4M3 = 0, 1  # cache element types (attn_kv_dtype)
ATTN_LAYOUT_BSHD, ATTN_LAYOUT_BHSD = 0, 1  # cache layouts (attn_kv_layout)

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        extra = ""
        if status == 7:  # ATTN_ERR_CUDA
            extra = f": {lib().attn_last_cuda_error().decode()}"
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({attn_status_string(status)}{extra})")


class _Cache(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("num_slots", ctypes.c_int64), ("slots_per_seq", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("block_size", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_ref", ctypes.c_void_p), ("layout", ctypes.c_int32)]


def lib():
    """The loaded library (ctypes.CDLL).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m gqa_attention_kv_gb300.build` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            cp = ctypes.POINTER(_Cache)
            L.attn_kv_append.argtypes = [p, p, p, i64, cp, i32, i32, p, p]
            L.attn_kv_append.restype = i32
            L.attn_decode_workspace_size.argtypes = [cp, i32, i32, i32, i32, i32, i32, i32]
            L.attn_decode_workspace_size.restype = sz
            L.attn_decode_kernel_launches.argtypes = [cp, i32, i32, i32, i32, i32, i32, i32,
                                                      i32, i32, ctypes.c_uint]
            L.attn_decode_kernel_launches.restype = i32
            L.attn_decode.argtypes = [p, cp, p, p, i32, i32, i32, i32, i32, i32, i32,
                                      ctypes.c_float, p, p, sz, p, p]
            L.attn_decode.restype = i32
            L.attn_decode_append.argtypes = [p, p, p, p, p, cp, p, p, i32, i32, i32, i32, i32,
                                             i32, i32, ctypes.c_float, p, p, sz, p,
                                             ctypes.c_uint, p]
            L.attn_decode_append.restype = i32
            L.attn_decode_noalloc.argtypes = [p, cp, p, p, i32, i32, i32, i32, i32, i32, i32,
                                              ctypes.c_float, p, p, p]
            L.attn_decode_noalloc.restype = i32
            L.attn_kv_reference.argtypes = [p, i64, i32, i32, p, p]
            L.attn_kv_reference.restype = i32
            L.attn_prefill.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, ctypes.c_float, p,
                                       p, p]
            L.attn_prefill.restype = i32
            L.attn_status_string.argtypes = [i32]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_version.restype = ctypes.c_char_p
            L.attn_last_cuda_error.restype = ctypes.c_char_p
            _lib = L
    return _lib


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_version() -> str:
    return lib().attn_version().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, where):
    if rc != ATTN_OK:
        raise AttnError(rc, where)


class KVCache:
    """One layer's cache: k, v [num_slots, n_kv_heads, head_dim] on the device,
    bf16, or uint8 E4M3 codes for an FP8 cache (dtype ATTN_KV_FP8_E4M3, whose
    keys are stored relative to k_ref, float32 [n_kv_heads, head_dim] or None).
    layout ATTN_LAYOUT_BHSD: k, v are [num_slots // rows, n_kv_heads, rows,
    head_dim] (rows = slots_per_seq, or block_size when paged); slots are
    numbered as in the slot-major layout.

    kind LINEAR: slots_per_seq = per-request capacity.
    kind PAGED : block_table int32 [batch, max_blocks_per_seq] (device), block_size.
    kind RING  : slots_per_seq = ring size.
    """

    def __init__(self, kind, k, v, slots_per_seq=0, block_table=None, block_size=0,
                 dtype=ATTN_KV_BF16, k_ref=None, layout=ATTN_LAYOUT_BSHD):
        self.kind, self.k, self.v = int(kind), k, v
        self.slots_per_seq = int(slots_per_seq)
        self.block_table = block_table
        self.block_size = int(block_size)
        self.dtype = int(dtype)
        self.k_ref = k_ref
        self.layout = int(layout)

    @property
    def n_kv_heads(self):
        return self.k.shape[1]

    @property
    def head_dim(self):
        return self.k.shape[-1]

    @property
    def num_slots(self):
        return self.k.shape[0] * (self.k.shape[2] if self.layout == ATTN_LAYOUT_BHSD else 1)

    def struct(self) -> _Cache:
        bt = self.block_table
        return _Cache(self.kind, self.k.data_ptr(), self.v.data_ptr(), self.num_slots,
                      self.slots_per_seq, None if bt is None else bt.data_ptr(),
                      self.block_size, 0 if bt is None else bt.shape[-1], self.dtype,
                      None if self.k_ref is None else self.k_ref.data_ptr(), self.layout)


def attn_kv_append(k_new, v_new, slot_mapping, cache: KVCache, err=None, stream=None):
    """cache.k[slot_mapping[i]] = k_new[i] (same for v); slot_mapping int64 [n]."""
    c = cache.struct()
    rc = lib().attn_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                              slot_mapping.shape[0], ctypes.byref(c), cache.n_kv_heads,
                              cache.head_dim, _ptr(err), _stream(stream))
    _check(rc, "attn_kv_append")


def attn_kv_reference(k, ref=None, stream=None):
    """Per-head mean of bf16 keys k [n, Hkv, D] as float32 [Hkv, D] (the FP8
    cache's reference vector).  Writes into ref if given."""
    import torch

    n, Hkv, D = k.shape
    if ref is None:
        ref = torch.empty(Hkv, D, dtype=torch.float32, device=k.device)
    rc = lib().attn_kv_reference(_ptr(k), n, Hkv, D, _ptr(ref), _stream(stream))
    _check(rc, "attn_kv_reference")
    return ref


def attn_decode_workspace_size(cache: KVCache, batch, q_rows, n_q_heads, max_seq_len,
                               window=0) -> int:
    c = cache.struct()
    n = lib().attn_decode_workspace_size(ctypes.byref(c), batch, q_rows, n_q_heads,
                                         cache.n_kv_heads, cache.head_dim, max_seq_len, window)
    if n == ctypes.c_size_t(-1).value:
        raise AttnError(ATTN_ERR_SHAPE, "attn_decode_workspace_size")
    return int(n)


def attn_decode_kernel_launches(cache: KVCache, batch, q_rows, n_q_heads, max_seq_len,
                                window=0, with_append=False, with_rope=False,
                                tables_early=False) -> int:
    """Kernels one attn_decode (with_append: attn_decode_append; with_rope:
    with a rotary embedding; tables_early: with ATTN_DECODE_TABLES_EARLY)
    call of this shape launches (host-side plan; nothing runs on the device)."""
    c = cache.struct()
    n = lib().attn_decode_kernel_launches(ctypes.byref(c), batch, q_rows, n_q_heads,
                                          cache.n_kv_heads, cache.head_dim, max_seq_len, window,
                                          int(bool(with_append)), int(bool(with_rope)),
                                          ATTN_DECODE_TABLES_EARLY if tables_early else 0)
    if n < 0:
        raise AttnError(ATTN_ERR_SHAPE, "attn_decode_kernel_launches")
    return int(n)


def attn_decode(q, cache: KVCache, seq_lens, positions, max_seq_len, window, scale, out=None,
                workspace=None, err=None, stream=None):
    """Decode attention.  q bf16 [B, R, Hq, D]; seq_lens int32 [B]; positions int32 [B*R].
    Returns out (bf16 [B, R, Hq, D]).  A workspace (zero-filled uint8 device
    tensor of at least attn_decode_workspace_size bytes) is allocated if not
    given; one kept across calls needs no clearing."""
    import torch

    B, R, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    need = attn_decode_workspace_size(cache, B, R, Hq, max_seq_len, window)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    c = cache.struct()
    rc = lib().attn_decode(_ptr(q), ctypes.byref(c), _ptr(seq_lens), _ptr(positions), B, R,
                           int(max_seq_len), int(window), Hq, cache.n_kv_heads, D, float(scale),
                           _ptr(out), _ptr(workspace),
                           0 if workspace is None else workspace.numel() * workspace.element_size(),
                           _ptr(err), _stream(stream))
    _check(rc, "attn_decode")
    return out


def attn_decode_append(q, k_new, v_new, slot_mapping, cache: KVCache, seq_lens, positions,
                       max_seq_len, window, scale, out=None, workspace=None, err=None,
                       stream=None, rope_inv_freq=None, tables_early=False, cache_early=False):
    """The step's KV append and its decode in one launch: same result as
    attn_kv_append(k_new, v_new, slot_mapping, cache) then attn_decode(...)
    when new row b*R + r is the key at position seq_lens[b] - R + r.
    k_new / v_new bf16 [B*R, Hkv, D]; slot_mapping int64 [B*R].  With
    rope_inv_freq (float32 [D/2] on the device), q and k_new are first rotated
    at their positions (interleaved pairs).  tables_early: seq_lens,
    positions and the block table were not written by the kernel launched
    just before on this stream (ATTN_DECODE_TABLES_EARLY); cache_early: nor
    are the cache's other rows (ATTN_DECODE_CACHE_EARLY, implies tables_early)."""
    import torch

    B, R, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    need = attn_decode_workspace_size(cache, B, R, Hq, max_seq_len, window)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    c = cache.struct()
    rc = lib().attn_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(rope_inv_freq),
        ctypes.byref(c), _ptr(seq_lens),
        _ptr(positions), B, R, int(max_seq_len), int(window), Hq, cache.n_kv_heads, D,
        float(scale), _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(err),
        (ATTN_DECODE_TABLES_EARLY if tables_early else 0) |
        (ATTN_DECODE_CACHE_EARLY if cache_early else 0), _stream(stream))
    _check(rc, "attn_decode_append")
    return out


def attn_prefill(q, k, v, window, scale, out=None, err=None, stream=None):
    """Causal prefill.  q bf16 [B, T, Hq, D], k/v bf16 [B, T, Hkv, D] -> out [B, T, Hq, D]."""
    import torch

    B, T, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    rc = lib().attn_prefill(_ptr(q), _ptr(k), _ptr(v), B, T, int(window), Hq, k.shape[2], D,
                            float(scale), _ptr(out), _ptr(err), _stream(stream))
    _check(rc, "attn_prefill")
    return out


def attn_decode_noalloc(q, cache: KVCache, seq_lens, positions, max_seq_len, window, scale,
                        out=None, err=None, stream=None):
    """attn_decode without a workspace argument, for callers that cannot
    allocate device memory: the library uses its own fixed scratch array
    (ATTN_DECODE_NOALLOC_SCRATCH_BYTES per GPU).  Calls that overlap on the
    GPU share that array and race; order them on one stream."""
    import torch

    f = lib().attn_decode_noalloc
    B, R, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    c = cache.struct()
    rc = f(_ptr(q), ctypes.byref(c), _ptr(seq_lens), _ptr(positions), B, R, int(max_seq_len),
           int(window), Hq, cache.n_kv_heads, D, float(scale), _ptr(out), _ptr(err),
           _stream(stream))
    _check(rc, "attn_decode_noalloc")
    return out
