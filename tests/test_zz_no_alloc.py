"""attn_decode_noalloc: the decode entry point for callers that cannot allocate.

Callers without a device allocator of their own, or that must not call
cudaMalloc inside their decode loop, use attn_decode_noalloc: it takes no
workspace and uses the library's fixed scratch array instead.  Its answers must
equal attn_decode's (which uses caller scratch) exactly, on two calls in a row
(the second call finds the first call's leftovers in the shared array), and
lie within the parity tolerance of the oracle.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import compare, oracle_decode

pytestmark = pytest.mark.gpu


def _noalloc_via_cabi(q, cache, seq, pos, max_seq, window, scale, out, err):
    """Call the C entry point directly, with ctypes, on the current stream."""
    f = gq.lib().attn_decode_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.POINTER(gq._Cache), ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    B, R, Hq, D = q.shape
    c = cache.struct()
    rc = f(q.data_ptr(), ctypes.byref(c), seq.data_ptr(), pos.data_ptr(), B, R, max_seq, window,
           Hq, cache.n_kv_heads, D, scale, out.data_ptr(), err.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    return rc


def _on_device(case, dev="cuda"):
    cache = gq.KVCache(case.kind, case.k_cache.to(dev), case.v_cache.to(dev),
                       slots_per_seq=case.slots_per_seq,
                       block_table=None if case.block_table is None else case.block_table.to(dev),
                       block_size=case.block_size)
    gq.attn_kv_append(case.k_new.to(dev), case.v_new.to(dev), case.slot_mapping.to(dev), cache)
    return cache, case.q.to(dev), case.seq_lens.to(dev), case.positions.to(dev)


def _two_calls_equal_attn_decode(case):
    """Two noalloc calls in a row give exactly attn_decode's output (both run
    the same plan and kernels, which are deterministic), and that output is
    within the parity tolerance of the oracle."""
    dev = "cuda"
    cache, q, seq, pos = _on_device(case)
    B, R, Hq, D = q.shape
    max_seq = case.max_seq_len()
    need = gq.attn_decode_workspace_size(cache, B, R, Hq, max_seq, case.window)
    assert 0 < need <= (32 << 20), "the case must use the scratch and fit in it"
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    want = gq.attn_decode(q, cache, seq, pos, max_seq, case.window, case.scale, err=err)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _noalloc_via_cabi(q, cache, seq, pos, max_seq, case.window, case.scale, out, err)
        assert rc == gq.ATTN_OK, gq.attn_status_string(rc)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out, want), f"call {call}: differs from attn_decode"
    ref, _, _ = oracle_decode(case)
    compare(out, ref, "noalloc vs oracle")


def test_noalloc_matches_attn_decode_twice():
    """Paged cache, 4 rows per request: split and merge kernels."""
    case = synth.decode_case(9101, synth.PAGED, 8, 4, 32, 8, 128,
                             [4096, 1500, 37, 2049, 700, 4, 3333, 128], block_size=16)
    _two_calls_equal_attn_decode(case)


def test_noalloc_chunk_kernel_twice():
    """A 29-row prefill chunk of 28/4 heads over a linear cache: the tcgen05
    chunk kernel, whose partial states sit after the split kernel's."""
    case = synth.decode_case(9102, synth.LINEAR, 2, 29, 28, 4, 128, [3000, 1700])
    _two_calls_equal_attn_decode(case)


def test_noalloc_batch_over_two_launches_twice():
    """300 requests: more than one launch's shared-memory tables hold, so the
    requests are split over two launches that share the scratch."""
    g = synth.generator(9103)
    sl = torch.randint(16, 200, (300,), generator=g, dtype=torch.int64).tolist()
    case = synth.decode_case(9103, synth.PAGED, 300, 1, 32, 8, 128, sl, block_size=16,
                             num_blocks=sum((n + 15) // 16 for n in sl) + 64)
    host = gq.KVCache(case.kind, case.k_cache, case.v_cache, block_table=case.block_table,
                      block_size=case.block_size)  # the plan is host-side only
    assert gq.attn_decode_kernel_launches(host, 300, 1, 32, case.max_seq_len()) >= 2
    _two_calls_equal_attn_decode(case)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    dev = "cuda"
    # 1024 requests x 16 KV heads x 32 query rows per head (8 rows x group 4)
    # over 32k keys needs more partial state than the fixed array holds:
    # refused before any launch.
    k = torch.zeros(16, 16, 128, dtype=torch.bfloat16, device=dev)
    cache = gq.KVCache(synth.LINEAR, k, k, slots_per_seq=16)
    big = gq.KVCache(synth.PAGED, k, k,
                     block_table=torch.zeros(1024, 2048, dtype=torch.int32, device=dev),
                     block_size=16)
    need = gq.attn_decode_workspace_size(big, 1024, 8, 64, 32768, 0)
    assert need > (32 << 20)
    q = torch.zeros(1024, 8, 64, 128, dtype=torch.bfloat16, device=dev)
    seq = torch.full((1024,), 16, dtype=torch.int32, device=dev)
    pos = torch.zeros(8192, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = _noalloc_via_cabi(q, big, seq, pos, 32768, 0, 0.1, out, err)
    assert rc == gq.ATTN_ERR_WORKSPACE
    del cache
