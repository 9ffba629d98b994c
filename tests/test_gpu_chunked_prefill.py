"""Chunked prefill against a KV cache, against the fp64 oracle.

A prompt arriving in chunks (the pages' streaming 7B backend feeds the decoder
29 rows at a time; talker_multiframe advances several rows per step) is a
K-row causal decode: the chunk's R rows sit at positions seq_len - R .. seq_len
- 1, each attends to every earlier key in the cache and causally to the rows
before it in the chunk.  The library runs it through attn_kv_append +
attn_decode with q_rows = R; the row blocks of a long GQA group (R x G rows)
split into several units.

A group of 64 or more rows over a linear slot-major bf16 cache runs on the
tcgen05 chunk kernel (the rows of a KV group packed into 128-row tiles, the
key range split over CTAs); the rest on the decode's split kernel.  Both are
checked against the oracle.
"""
import pytest
import torch

import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import compare, gpu_decode, oracle_decode, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def launches(case, **kw):
    return gq.attn_decode_kernel_launches(to_device(case, DEV), case.batch, case.q_rows,
                                          case.n_q_heads, case.max_seq_len(), case.window, **kw)


@pytest.mark.parametrize("R,Hq,Hkv", [(29, 28, 4), (29, 32, 8), (64, 32, 8), (16, 16, 16)])
@pytest.mark.parametrize("kind", [synth.LINEAR, synth.PAGED])
def test_chunk_against_cache(R, Hq, Hkv, kind):
    seq = [R + 1500, R, 3 * R + 7]  # a long context, a first chunk, a short one
    case = synth.decode_case(8000 + R * Hq + Hkv, kind, len(seq), R, Hq, Hkv, 128, seq,
                             block_size=16)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"{kind} chunk R={R} {Hq}/{Hkv}")


def test_chunk_in_sliding_window_ring():
    """A 29-row chunk over a 1500-slot ring with a 750-key window, past wrap
    (the streaming encoder's shape, Voxtral notes, "Encoder KV cache")."""
    R = 29
    seq = [4000, 1500 + R, 777]
    case = synth.decode_case(8100, synth.RING, len(seq), R, 32, 32, 64, seq, window=750,
                             ring=1500)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, "ring chunk R=29 W=750")


@pytest.mark.parametrize("R,Hq,Hkv,D", [(29, 28, 4, 128), (64, 32, 8, 128), (16, 16, 4, 64),
                                        (10, 56, 8, 128), (40, 12, 2, 64)])
def test_chunk_kernel_packings(R, Hq, Hkv, D):
    """Groups of 7 (18 rows a tile, two padding rows), 4 (32), 6 (21), and a
    chunk shorter than one tile's rows; requests of very different lengths, so
    some key splits are empty."""
    seq = [R + 5000, R, R + 300, 3 * R]
    case = synth.decode_case(8300 + R * Hq + D, synth.LINEAR, len(seq), R, Hq, Hkv, D, seq)
    assert launches(case) >= 1
    ref, _, _ = oracle_decode(case)
    a, _ = gpu_decode(case)
    b, _ = gpu_decode(case)
    assert torch.equal(a, b), "run-to-run results differ"
    compare(a, ref, f"chunk kernel R={R} {Hq}/{Hkv} D={D}")


def test_chunk_kernel_window():
    """A 29-row chunk with a 750-key window over a long linear cache."""
    R = 29
    case = synth.decode_case(8400, synth.LINEAR, 2, R, 28, 4, 128, [6000, 2000], window=750)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, "chunk kernel, window 750")


def test_chunk_kernel_fused_append_and_rope_fallback():
    """attn_decode_append on a chunk: the chunk kernel takes the step's rows
    from k_new / v_new and writes them to the cache (then its merge); with a
    rotary embedding the split kernel."""
    from test_gpu_decode_append import _run

    case = synth.decode_case(8500, synth.LINEAR, 2, 29, 28, 4, 128, [14449, 3000])
    assert launches(case, with_append=True) == 2
    assert launches(case, with_append=True, with_rope=True) == 1
    fused, _ = _run(case, fused=True)
    ref, _, _ = oracle_decode(case)
    compare(fused, ref, "fused chunk")


@pytest.mark.parametrize("R,Hq,Hkv,D,seq", [(29, 28, 4, 128, [14480, 1030]),
                                             (29, 28, 4, 128, [14449, 3000]),
                                             (29, 28, 4, 128, [200, 64]),
                                             (16, 32, 8, 64, [700, 136])])
def test_chunk_fused_append_equals_append_then_decode(R, Hq, Hkv, D, seq):
    """The chunk kernel with the step's rows fused in (taken from k_new / v_new,
    written to the cache by the same launch) equals the append kernel followed
    by the chunk kernel, output and cache bit for bit: new rows straddling a
    key-tile boundary (14,451..14,479 over 14,464; 1,001..1,029 over 1,024;
    120..135 over 128 at head_dim 64), inside one tile, and a short request."""
    from test_gpu_decode_append import _run

    case = synth.decode_case(8600 + seq[1] + D, synth.LINEAR, 2, R, Hq, Hkv, D, seq)
    assert launches(case, with_append=True) <= 2  # the chunk kernel (+ its merge)
    out_f, cache_f = _run(case, fused=True)
    out_u, cache_u = _run(case, fused=False)
    assert torch.equal(out_f, out_u), "fused chunk differs from append + chunk"
    assert torch.equal(cache_f.k, cache_u.k) and torch.equal(cache_f.v, cache_u.v)
    ref, _, _ = oracle_decode(case)
    compare(out_f, ref, f"fused chunk {seq}")
