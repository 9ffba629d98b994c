"""The measured decode workloads at their full sizes, launched the way the
bench launches them, against the fp64 oracle.

Each case is the seeded synthetic input of one workload (Voxtral decoder
step, the Qwen2-7B two-slot decode at every context of the sweep, the ring
window decode, the paged K=4 decode, the streaming-encoder step, a 29-row
prefill chunk, and the FP8 ring and paged caches).  The library runs it as
one attn_decode_append call (the step's rows appended by the decode launch),
with the plan read before the previous kernel finishes (tables early) and a
workspace kept across calls, exactly as the bench does; the oracle appends
the rows and then attends, over every output element.
"""
import numpy as np
import pytest
import torch

import oracle
import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import bits, compare, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _device_cache(case, k, v, **kw):
    return gq.KVCache(case.kind, torch.as_tensor(k).to(DEV), torch.as_tensor(v).to(DEV),
                      slots_per_seq=case.slots_per_seq,
                      block_table=None if case.block_table is None else case.block_table.to(DEV),
                      block_size=case.block_size, **kw)


def _bench_launch(case, cache, max_seq_len, ws=None):
    """One decode step as the bench issues it."""
    if ws is None:
        ws = torch.zeros(gq.attn_decode_workspace_size(cache, case.batch, case.q_rows,
                                                       case.n_q_heads, max_seq_len, case.window),
                         dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gq.attn_decode_append(case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV),
                                case.slot_mapping.to(DEV), cache, case.seq_lens.to(DEV),
                                case.positions.to(DEV), max_seq_len, case.window, case.scale,
                                workspace=ws, err=err, tables_early=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item())}"
    return out


def _check_bf16(case, where, max_seq_len=None, ws=None):
    ref, kc, vc = oracle_decode(case)
    cache = _device_cache(case, case.k_cache, case.v_cache)
    out = _bench_launch(case, cache, max_seq_len or case.max_seq_len(), ws)
    assert np.array_equal(bits(cache.k), kc), f"{where}: K after the fused append"
    assert np.array_equal(bits(cache.v), vc), f"{where}: V after the fused append"
    compare(out, ref, where)
    return out


def test_voxtral_decode_step():
    _check_bf16(synth.voxtral_decode_step(), "voxtral decode, 512 keys")


def test_qwen_decode_sweep():
    """All five calls of the Qwen2-7B step, one workspace, the bench's grid
    bound (the longest context)."""
    cap = synth.QWEN_CONTEXTS[-1]
    ws = None
    for i, ctx in enumerate([(c, c) for c in synth.QWEN_CONTEXTS] +
                            [(synth.QWEN_PROMPT, cap)]):
        case = synth.qwen_decode(ctx, seed=20263 + 100 + i)
        if ws is None:  # sized from the host tensors' shapes (nothing is read)
            sizing = gq.KVCache(case.kind, case.k_cache, case.v_cache,
                                slots_per_seq=case.slots_per_seq)
            ws = torch.zeros(gq.attn_decode_workspace_size(sizing, 2, 1, 28, cap, 0),
                             dtype=torch.uint8, device=DEV)
        _check_bf16(case, f"qwen decode {ctx}", max_seq_len=cap, ws=ws)


def test_ring_window_decode():
    _check_bf16(synth.ring_window_decode(), "ring B=16, window 8192 of 16384")


def test_paged_multirow_decode():
    _check_bf16(synth.paged_multirow_decode(), "paged 64 x 4 rows, bs 16")


def test_streaming_encoder_step():
    _check_bf16(synth.streaming_encoder_step(), "streaming encoder step")


def test_chunked_prefill_step():
    _check_bf16(synth.chunked_prefill_step(), "29-row chunk at 14,449")


@pytest.mark.parametrize("make", [synth.ring_window_decode, synth.paged_multirow_decode],
                         ids=["ring-fp8", "paged-fp8"])
def test_fp8_workloads(make):
    """E4M3 caches with K relative to the mean of the first 512 keys, filled
    by the oracle's FP8 append; the step's rows encoded by the decode launch."""
    case = make()
    S, Hkv, D = case.k_cache.shape
    ref = oracle.kv_reference(bits(case.k_cache[:512])).astype(np.float32)
    kc = np.zeros((S, Hkv, D), dtype=np.uint8)
    vc = np.zeros((S, Hkv, D), dtype=np.uint8)
    oracle.kv_append_fp8(kc, vc, bits(case.k_cache), bits(case.v_cache), np.arange(S), k_ref=ref)
    cache = _device_cache(case, kc, vc, dtype=gq.ATTN_KV_FP8_E4M3,
                          k_ref=torch.from_numpy(ref).to(DEV))
    oracle.kv_append_fp8(kc, vc, bits(case.k_new), bits(case.v_new),
                         case.slot_mapping.cpu().numpy(), k_ref=ref)
    out = _bench_launch(case, cache, case.max_seq_len())
    assert np.array_equal(cache.k.cpu().numpy(), kc), "K codes after the fused append"
    assert np.array_equal(cache.v.cpu().numpy(), vc), "V codes after the fused append"
    cd = {"kind": case.kind, "k": oracle.fp8_to_bf16_bits(kc), "v": oracle.fp8_to_bf16_bits(vc),
          "slots_per_seq": case.slots_per_seq,
          "block_table": None if case.block_table is None else case.block_table.numpy(),
          "block_size": case.block_size}
    rc, want = oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(),
                             case.window, case.scale, Hkv)
    assert rc == 0
    compare(out, want, f"{make.__name__} fp8")
