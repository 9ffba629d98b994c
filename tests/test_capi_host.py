"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/attn_kv.h declares, and refuses bad arguments with
the documented status before any launch."""
import ctypes
import os
import re

import pytest

import gqa_attention_kv_gb300 as gq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_kv.h")


@pytest.fixture(scope="module")
def lib():
    from gqa_attention_kv_gb300 import build

    build.build()
    return gq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("attn_kv_append", "attn_decode", "attn_decode_workspace_size", "attn_prefill",
                 "attn_decode_kernel_launches",
                 "attn_decode_append", "attn_kv_reference", "attn_status_string",
                 "attn_version"):
        assert want in names, names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for code in range(9):
        assert gq.attn_status_string(code) != "unknown status"
    assert gq.attn_status_string(99) == "unknown status"
    assert "sm_103a" in gq.attn_version()


class FakeTensor:
    """Pointer + shape stand-in: validation must refuse before touching it."""

    def __init__(self, ptr, shape):
        self._p, self.shape = ptr, shape

    def data_ptr(self):
        return self._p

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n

    def element_size(self):
        return 1


def cache(kind=gq.LINEAR, Hkv=8, D=128, slots=1024, sps=512, bt=None, bs=0, k=4096, v=8192,
          dtype=gq.ATTN_KV_BF16, k_ref=None):
    return gq.KVCache(kind, FakeTensor(k, (slots, Hkv, D)), FakeTensor(v, (slots, Hkv, D)),
                      slots_per_seq=sps, block_table=bt, block_size=bs, dtype=dtype,
                      k_ref=k_ref)


def decode_rc(lib, c, B=2, R=1, Hq=32, Hkv=8, D=128, L=512, W=0, q=16, out=32, ws=None,
              ws_bytes=0):
    cs = c.struct()
    return lib.attn_decode(q, ctypes.byref(cs), 64, 128, B, R, L, W, Hq, Hkv, D, 0.1, out,
                           ws, ws_bytes, None, None)


def test_decode_validation(lib):
    assert decode_rc(lib, cache(), Hq=30, Hkv=8) == gq.ATTN_ERR_SHAPE       # 30 % 8 != 0
    assert decode_rc(lib, cache(), D=96) == gq.ATTN_ERR_UNSUPPORTED
    assert decode_rc(lib, cache(), R=0) == gq.ATTN_ERR_SHAPE
    assert decode_rc(lib, cache(sps=600)) == gq.ATTN_ERR_SHAPE              # 2*600 > 1024 slots
    assert decode_rc(lib, cache(), q=None) == gq.ATTN_ERR_NULL
    assert decode_rc(lib, cache(), q=17) == gq.ATTN_ERR_ALIGN
    assert decode_rc(lib, cache(k=4100)) == gq.ATTN_ERR_ALIGN
    # ring: needs a window and ring >= window + q_rows - 1
    assert decode_rc(lib, cache(gq.RING, sps=512), W=0) == gq.ATTN_ERR_SHAPE
    assert decode_rc(lib, cache(gq.RING, sps=512), R=4, W=510) == gq.ATTN_ERR_SHAPE
    # paged: block table required, and the table must span max_seq_len
    assert decode_rc(lib, cache(gq.PAGED, sps=0, bs=16), L=512) in (gq.ATTN_ERR_SHAPE,
                                                                    gq.ATTN_ERR_NULL)
    bt = FakeTensor(1 << 20, (2, 8))
    assert decode_rc(lib, cache(gq.PAGED, sps=0, bt=bt, bs=16), L=512) == gq.ATTN_ERR_SHAPE
    # batch 0 is a no-op
    assert decode_rc(lib, cache(), B=0) == gq.ATTN_OK
    # the scale must be finite and positive
    cs = cache().struct()
    assert lib.attn_decode(16, ctypes.byref(cs), 64, 128, 2, 1, 512, 0, 32, 8, 128, -1.0, 32,
                           None, 0, None, None) == gq.ATTN_ERR_SHAPE


def test_decode_workspace_checks(lib):
    c = cache(slots=4096 * 4, sps=4096)
    cs = c.struct()
    need = lib.attn_decode_workspace_size(ctypes.byref(cs), 2, 1, 32, 8, 128, 4096, 0)
    assert need > 0 and need != ctypes.c_size_t(-1).value
    assert decode_rc(lib, c, L=4096, ws=None, ws_bytes=0) == gq.ATTN_ERR_NULL
    assert decode_rc(lib, c, L=4096, ws=1 << 20, ws_bytes=need - 1) == gq.ATTN_ERR_WORKSPACE
    bad = lib.attn_decode_workspace_size(ctypes.byref(cs), 2, 1, 30, 8, 128, 4096, 0)
    assert bad == ctypes.c_size_t(-1).value


def test_decode_kernel_launches(lib):
    """The plan query: -1 where attn_decode would refuse, 0 for no requests,
    otherwise split launches x (1 + merge kernel).  Without a GPU the library
    plans for 148 SMs (296 CTAs)."""
    f = lib.attn_decode_kernel_launches
    c = cache(slots=16384 * 40, sps=16384)
    cs = c.struct()
    assert f(ctypes.byref(cs), 2, 1, 30, 8, 128, 4096, 0, 0, 0, 0) == -1  # 30 q heads over 8
    assert f(None, 2, 1, 32, 8, 128, 4096, 0, 0, 0, 0) == -1
    assert f(ctypes.byref(cs), 0, 1, 32, 8, 128, 4096, 0, 0, 0, 0) == 0
    # short contexts: every unit spans at most 8 CTAs, merged in the split kernel
    assert f(ctypes.byref(cs), 2, 1, 32, 8, 128, 512, 0, 0, 0, 0) == 1
    # 16 units at 8,192 keys: few units over many CTAs -> merge kernel
    assert f(ctypes.byref(cs), 2, 1, 32, 8, 128, 8192, 0, 1, 0, 0) == 2
    # 320 units at 8,192 keys: too many units for the merge kernel's rule
    assert f(ctypes.byref(cs), 40, 1, 32, 8, 128, 8192, 0, 1, 0, 0) == 1
    # one unit that may span more than 128 CTAs: merge kernel
    assert f(ctypes.byref(cs), 40, 1, 8, 1, 128, 16384, 0, 0, 0, 0) == 2
    # more (request, row block) pairs than one launch's tables hold: 2 launches
    big = cache(slots=64 * 300, sps=64)
    bs = big.struct()
    assert f(ctypes.byref(bs), 300, 1, 8, 2, 128, 64, 0, 0, 0, 0) == 2
    # ATTN_DECODE_TABLES_EARLY plans the same kernels
    assert f(ctypes.byref(cs), 2, 1, 32, 8, 128, 8192, 0, 1, 0, 1) == 2
    assert f(ctypes.byref(bs), 300, 1, 8, 2, 128, 64, 0, 1, 0, 1) == 2
    assert f(ctypes.byref(cs), 2, 1, 32, 8, 128, 8192, 0, 1, 0, 3) == 2  # both early flags
    assert f(ctypes.byref(cs), 2, 1, 32, 8, 128, 8192, 0, 1, 0, 4) == -1  # unknown flag
    # a 29-row chunk of a 28/4 group (203 rows) over a linear cache: the chunk
    # kernel (+ its merge: 2 x 4 groups split over the key range; the append of
    # attn_decode_append is inside the chunk kernel); with a rotary embedding
    # the split kernel
    ch = cache(slots=14464 * 2, sps=14464, Hkv=4)
    hs = ch.struct()
    assert f(ctypes.byref(hs), 2, 29, 28, 4, 128, 14449, 0, 0, 0, 0) == 2
    assert f(ctypes.byref(hs), 2, 29, 28, 4, 128, 14449, 0, 1, 0, 0) == 2
    assert f(ctypes.byref(hs), 2, 29, 28, 4, 128, 14449, 0, 1, 1, 0) == 1


def test_prefill_validation(lib):
    f = lib.attn_prefill
    assert f(16, 32, 48, 1, 100, 0, 30, 8, 128, 0.1, 64, None, None) == gq.ATTN_ERR_SHAPE
    assert f(16, 32, 48, 1, 100, 0, 32, 8, 80, 0.1, 64, None, None) == gq.ATTN_ERR_UNSUPPORTED
    assert f(None, 32, 48, 1, 100, 0, 32, 8, 128, 0.1, 64, None, None) == gq.ATTN_ERR_NULL
    assert f(16, 40, 48, 1, 100, 0, 32, 8, 128, 0.1, 72, None, None) == gq.ATTN_ERR_ALIGN
    assert f(16, 32, 48, 0, 100, 0, 32, 8, 128, 0.1, 64, None, None) == gq.ATTN_OK
    assert f(16, 32, 48, 1, 0, 0, 32, 8, 128, 0.1, 64, None, None) == gq.ATTN_OK
    assert f(16, 32, 48, 1, 100, 0, 32, 8, 128, 0.0, 64, None, None) == gq.ATTN_ERR_SHAPE
    assert f(16, 32, 48, 1, 100, 0, 32, 8, 128, -0.1, 64, None, None) == gq.ATTN_ERR_SHAPE
    assert f(16, 32, 48, 1, 100, 0, 32, 8, 128, float("inf"), 64, None, None) == gq.ATTN_ERR_SHAPE


def test_append_validation(lib):
    c = cache()
    cs = c.struct()
    f = lib.attn_kv_append
    assert f(16, 32, 48, 0, ctypes.byref(cs), 8, 128, None, None) == gq.ATTN_OK   # n = 0
    assert f(16, 32, 48, -1, ctypes.byref(cs), 8, 128, None, None) == gq.ATTN_ERR_SHAPE
    assert f(None, 32, 48, 4, ctypes.byref(cs), 8, 128, None, None) == gq.ATTN_ERR_NULL
    assert f(16, 33, 48, 4, ctypes.byref(cs), 8, 128, None, None) == gq.ATTN_ERR_ALIGN
    assert f(16, 32, 48, 4, ctypes.byref(cs), 8, 100, None, None) == gq.ATTN_ERR_UNSUPPORTED


def test_product_path_does_not_reach_the_oracle():
    """The binding and the kernels never import the CPU checker."""
    pkg = os.path.join(ROOT, "gqa_attention_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "attn_oracle" not in text, f


def test_decode_append_validation(lib):
    """Host checks of attn_decode_append, made before any launch."""
    c = cache(slots=4096 * 4, sps=4096)
    cs = c.struct()
    f = lib.attn_decode_append
    need = lib.attn_decode_workspace_size(ctypes.byref(cs), 2, 1, 32, 8, 128, 4096, 0)
    args = lambda q=16, kn=32, vn=48, sm=64, ws=1 << 20, ws_bytes=need, scale=0.1, hq=32, \
        flags=0: (q, kn, vn, sm, None, ctypes.byref(cs), 80, 96, 2, 1, 4096, 0, hq, 8, 128, scale,
                  112, ws, ws_bytes, None, flags, None)
    assert f(*args(kn=None)) == gq.ATTN_ERR_NULL
    assert f(*args(sm=None)) == gq.ATTN_ERR_NULL
    assert f(*args(vn=40)) == gq.ATTN_ERR_ALIGN
    assert f(*args(ws_bytes=need - 1)) == gq.ATTN_ERR_WORKSPACE
    assert f(*args(hq=30)) == gq.ATTN_ERR_SHAPE
    assert f(*args(scale=0.0)) == gq.ATTN_ERR_SHAPE
    assert f(*args(flags=4)) == gq.ATTN_ERR_UNSUPPORTED


def test_fp8_cache_validation(lib):
    """FP8 caches: head_dim 128 only, no rotary embedding in the fused append,
    an aligned k_ref;
    an unknown dtype is refused."""
    fp8 = gq.ATTN_KV_FP8_E4M3
    assert decode_rc(lib, cache(dtype=fp8, D=64), D=64) == gq.ATTN_ERR_UNSUPPORTED
    assert decode_rc(lib, cache(dtype=7)) == gq.ATTN_ERR_UNSUPPORTED
    assert decode_rc(lib, cache(dtype=fp8), B=0) == gq.ATTN_OK
    c = cache(dtype=fp8)
    cs = c.struct()
    assert lib.attn_decode_workspace_size(ctypes.byref(cs), 2, 1, 32, 8, 128, 512, 0) > 0
    f = lib.attn_kv_append
    ref_bad = FakeTensor(4100, (8, 128))
    cs = cache(dtype=fp8, k_ref=ref_bad).struct()
    assert f(16, 32, 48, 4, ctypes.byref(cs), 8, 128, None, None) == gq.ATTN_ERR_ALIGN
    cs = cache(dtype=fp8, D=64).struct()
    assert f(16, 32, 48, 4, ctypes.byref(cs), 8, 64, None, None) == gq.ATTN_ERR_UNSUPPORTED
    cs = cache(dtype=fp8, slots=4096 * 4, sps=4096).struct()
    need = lib.attn_decode_workspace_size(ctypes.byref(cs), 2, 1, 32, 8, 128, 4096, 0)
    # the fused append takes FP8 caches, but not with the rotary embedding
    assert lib.attn_decode_append(16, 32, 48, 64, 128, ctypes.byref(cs), 80, 96, 2, 1, 4096,
                                  0, 32, 8, 128, 0.1, 112, 1 << 20, need, None, 0,
                                  None) == gq.ATTN_ERR_UNSUPPORTED


def test_kv_reference_validation(lib):
    f = lib.attn_kv_reference
    assert f(16, 0, 8, 128, 32, None) == gq.ATTN_ERR_SHAPE
    assert f(None, 4, 8, 128, 32, None) == gq.ATTN_ERR_NULL
    assert f(16, 4, 8, 128, None, None) == gq.ATTN_ERR_NULL
    assert f(18, 4, 8, 128, 32, None) == gq.ATTN_ERR_ALIGN


def test_layout_validation(lib):
    """Head-major caches need whole blocks; unknown layouts are refused."""
    c = cache()
    c.layout = 7
    assert decode_rc(lib, c) == gq.ATTN_ERR_UNSUPPORTED
    c = cache(slots=1000, sps=300)   # 1000 slots are not whole blocks of 300
    c.layout = gq.ATTN_LAYOUT_BHSD
    assert decode_rc(lib, c, B=2) == gq.ATTN_ERR_SHAPE
    cs = c.struct()
    assert lib.attn_kv_append(16, 32, 48, 4, ctypes.byref(cs), 8, 128, None,
                              None) == gq.ATTN_ERR_SHAPE
    c = cache(slots=1024, sps=512)
    c.layout = gq.ATTN_LAYOUT_BHSD
    assert decode_rc(lib, c, B=0) == gq.ATTN_OK
