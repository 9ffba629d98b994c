"""Chunked prefill against a KV cache, against the fp64 oracle.

A prompt arriving in chunks (the pages' streaming 7B backend feeds the decoder
29 rows at a time; talker_multiframe advances several rows per step) is a
K-row causal decode: the chunk's R rows sit at positions seq_len - R .. seq_len
- 1, each attends to every earlier key in the cache and causally to the rows
before it in the chunk.  The library runs it through attn_kv_append +
attn_decode with q_rows = R; the row blocks of a long GQA group (R x G rows)
split into several units.
"""
import pytest

from gqa_attention_kv_gb300 import synth
from helpers import compare, gpu_decode, oracle_decode

pytestmark = pytest.mark.gpu


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
