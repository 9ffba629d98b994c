"""fp64 CPU oracle for grouped-query attention over a decoder KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's ``smoke()`` check and
the benchmark's CPU-baseline leg may import this module.  The product path
(the CUDA library and its Python binding) never reaches it, and the two share
no code: the arithmetic lives in ``attn_oracle.c`` (plain loops, fp64), this
file only compiles it with gcc and marshals numpy arrays.

bf16 tensors are passed as ``numpy.uint16`` bit patterns (use ``bf16_bits``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "_attn_oracle.so")
_lock = threading.Lock()
_lib = None

LINEAR, PAGED, RING = 0, 1, 2
OK, EMPTY_KEYSET, BAD_ARGS = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into an in-tree shared object (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = f64
            lib.oracle_ring_abs_pos.argtypes = [i64, i64, i64]
            lib.oracle_ring_abs_pos.restype = i64
            lib.oracle_threads.restype = i32
            lib.oracle_kv_append.argtypes = [p, p, i64, i64, p, p, p, i64]
            lib.oracle_kv_append.restype = i64
            lib.oracle_decode.argtypes = [p, i32, i32, i32, i32, i32, i32, p, p, i64, i64, p,
                                          i32, i32, p, p, i32, f64, p]
            lib.oracle_decode.restype = i32
            lib.oracle_decode_weights.argtypes = [p, i32, i32, i32, i32, i32, i32, p, p, i64, i64,
                                                  p, i32, i32, p, p, i32, f64, i32, i32, i32, p,
                                                  p, i64]
            lib.oracle_decode_weights.restype = i64
            lib.oracle_prefill.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, f64, p, i32, p]
            lib.oracle_rope_bf16.argtypes = [p, i64, i32, i32, p, p, p]
            lib.oracle_rope_bf16.restype = None
            lib.oracle_prefill.restype = i32
            lib.oracle_fp8_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_fp8_e4m3_to_f64.restype = f64
            lib.oracle_f32_to_fp8_e4m3.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_fp8_e4m3.restype = ctypes.c_uint8
            lib.oracle_fp8_e4m3_to_bf16.argtypes = [ctypes.c_uint8]
            lib.oracle_fp8_e4m3_to_bf16.restype = ctypes.c_uint16
            lib.oracle_kv_append_fp8.argtypes = [p, p, i64, i64, p, p, p, p, i64]
            lib.oracle_kv_append_fp8.restype = i64
            lib.oracle_kv_reference.argtypes = [p, i64, i64, p]
            lib.oracle_kv_reference.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 tensors are passed as uint16 bit patterns, got {a.dtype}")
    return a


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor (any device) -> numpy uint16 bit patterns."""
    import torch

    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def threads() -> int:
    return int(_load().oracle_threads())


def ring_abs_pos(j: int, total_written: int, ring: int) -> int:
    """Absolute position held by ring slot j after total_written rows were stored."""
    return int(_load().oracle_ring_abs_pos(j, total_written, ring))


def kv_append(k_cache, v_cache, k_new, v_new, slot_mapping) -> int:
    """In place: cache[slot_mapping[i]] = new[i] in row order.  Returns skipped rows."""
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags.c_contiguous:
            raise TypeError("caches must be C-contiguous uint16 arrays")
    num_slots = k_cache.shape[0]
    row = int(np.prod(k_cache.shape[1:]))
    kn, vn = _u16(k_new), _u16(v_new)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return int(_load().oracle_kv_append(_ptr(k_cache), _ptr(v_cache), num_slots, row, _ptr(kn),
                                        _ptr(vn), _ptr(sm), sm.shape[0]))


def rope(x, positions, inv_freq) -> np.ndarray:
    """Rotary embedding of interleaved pairs: x bf16 [n, heads, D] (tensor or
    uint16 bits), positions int [n], inv_freq float32 [D/2].  Returns uint16
    bf16 bits of the rotated rows (oracle_rope_bf16)."""
    xb = _u16(x)
    n, heads, D = xb.shape
    pos = _i32(positions).reshape(-1)
    inv = np.ascontiguousarray(np.asarray(inv_freq, dtype=np.float32).reshape(-1))
    if pos.shape[0] != n or inv.shape[0] != D // 2:
        raise ValueError("positions must have one entry per row and inv_freq D/2 entries")
    out = np.empty_like(xb)
    _load().oracle_rope_bf16(_ptr(xb), n, heads, D, _ptr(pos), _ptr(inv), _ptr(out))
    return out


def fp8_to_f64(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8 array) as fp64 (oracle_fp8_e4m3_to_f64)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    lib = _load()
    table = np.array([lib.oracle_fp8_e4m3_to_f64(i) for i in range(256)], dtype=np.float64)
    return table[c]


def f32_to_fp8(x) -> np.ndarray:
    """E4M3 codes of float32 values (oracle_f32_to_fp8_e4m3), elementwise."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    lib = _load()
    flat = np.array([lib.oracle_f32_to_fp8_e4m3(float(v)) for v in a.reshape(-1)],
                    dtype=np.uint8)
    return flat.reshape(a.shape)


def fp8_to_bf16_bits(codes) -> np.ndarray:
    """E4M3 codes -> bf16 bit patterns of the same values (exact)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    lib = _load()
    table = np.array([lib.oracle_fp8_e4m3_to_bf16(i) for i in range(256)], dtype=np.uint16)
    return table[c]


def kv_append_fp8(k_cache, v_cache, k_new, v_new, slot_mapping, k_ref=None) -> int:
    """In place on uint8 caches [S, Hkv, D]: k_cache[slot] = E4M3(k - k_ref),
    v_cache[slot] = E4M3(v) in row order (oracle_kv_append_fp8).  k_ref:
    float32 [Hkv, D] or None.  Returns skipped rows."""
    for c in (k_cache, v_cache):
        if c.dtype != np.uint8 or not c.flags.c_contiguous:
            raise TypeError("FP8 caches must be C-contiguous uint8 arrays")
    num_slots = k_cache.shape[0]
    row = int(np.prod(k_cache.shape[1:]))
    kn, vn = _u16(k_new), _u16(v_new)
    ref = None if k_ref is None else np.ascontiguousarray(k_ref, dtype=np.float32).reshape(-1)
    if ref is not None and ref.shape[0] != row:
        raise ValueError("k_ref must hold n_kv_heads * head_dim values")
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return int(_load().oracle_kv_append_fp8(_ptr(k_cache), _ptr(v_cache), num_slots, row,
                                            _ptr(kn), _ptr(vn), _ptr(ref), _ptr(sm),
                                            sm.shape[0]))


def kv_reference(k) -> np.ndarray:
    """Mean over rows of bf16 keys [n, Hkv, D] (uint16 bits), fp64 [Hkv, D]."""
    kb = _u16(k)
    n = kb.shape[0]
    row = int(np.prod(kb.shape[1:]))
    out = np.empty(row, dtype=np.float64)
    _load().oracle_kv_reference(_ptr(kb), n, row, _ptr(out))
    return out.reshape(kb.shape[1:])


def _cache_args(cache: dict):
    k, v = _u16(cache["k"]), _u16(cache["v"])
    bt = _i32(cache.get("block_table"))
    return (cache["kind"], k, v, k.shape[0], int(cache.get("slots_per_seq", 0)), bt,
            int(cache.get("block_size", 0)),
            int(bt.shape[1]) if bt is not None and bt.ndim == 2 else 0)


def decode(q, cache: dict, seq_lens, positions, window: int, scale: float, n_kv_heads: int):
    """Decode attention.  q: uint16 [B, R, Hq, D]; cache: dict with kind, k, v
    ([S, Hkv, D] uint16), slots_per_seq, block_table, block_size.
    Returns (status, out fp64 [B, R, Hq, D])."""
    q = _u16(q)
    B, R, Hq, D = q.shape
    kind, k, v, ns, sps, bt, bs, mb = _cache_args(cache)
    sl, pos = _i32(seq_lens), _i32(positions)
    out = np.empty((B, R, Hq, D), dtype=np.float64)
    rc = _load().oracle_decode(_ptr(q), B, R, Hq, n_kv_heads, D, kind, _ptr(k), _ptr(v), ns, sps,
                               _ptr(bt), bs, mb, _ptr(sl), _ptr(pos), window, scale, _ptr(out))
    return int(rc), out


def decode_weights(q, cache: dict, seq_lens, positions, window: int, scale: float,
                   n_kv_heads: int, b: int, r: int, h: int):
    """(absolute positions of the candidate keys, their attention weights) for
    one (request, row, head).  Masked candidates have weight 0."""
    q = _u16(q)
    B, R, Hq, D = q.shape
    kind, k, v, ns, sps, bt, bs, mb = _cache_args(cache)
    sl, pos = _i32(seq_lens), _i32(positions)
    cap = max(int(sps) if kind == RING else int(sl[b]), 1)
    tp = np.empty(cap, dtype=np.int64)
    w = np.empty(cap, dtype=np.float64)
    n = _load().oracle_decode_weights(_ptr(q), B, R, Hq, n_kv_heads, D, kind, _ptr(k), _ptr(v),
                                      ns, sps, _ptr(bt), bs, mb, _ptr(sl), _ptr(pos), window,
                                      scale, b, r, h, _ptr(tp), _ptr(w), cap)
    if n < 0:
        raise ValueError("oracle_decode_weights failed (bad args or empty key set)")
    return tp[:n].copy(), w[:n].copy()


def prefill(q, k, v, window: int, scale: float, rows=None):
    """Causal prefill.  q uint16 [B, T, Hq, D], k/v uint16 [B, T, Hkv, D].
    rows: optional query positions to compute (out then [B, len(rows), Hq, D]).
    Returns (status, out fp64)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    r = _i32(rows)
    nr = T if r is None else r.shape[0]
    out = np.empty((B, nr, Hq, D), dtype=np.float64)
    rc = _load().oracle_prefill(_ptr(q), _ptr(k), _ptr(v), B, T, window, Hq, Hkv, D, scale,
                                _ptr(r), 0 if r is None else nr, _ptr(out))
    return int(rc), out
