"""attn_decode_append: the step's append fused into the decode launch.

It must give what attn_kv_append followed by attn_decode gives (vibevoice.c,
"The decode step is one submission": the new row lands at its device-side
slot, then attention reads it): the same output bits, the same cache bits
after the call, and the oracle's answer within the tolerance.
"""
import numpy as np
import pytest
import torch

import gqa_attention_kv_gb300 as gq
import oracle
from gqa_attention_kv_gb300 import synth
from helpers import compare, oracle_decode, to_device

pytestmark = pytest.mark.gpu

LINEAR, PAGED, RING = synth.LINEAR, synth.PAGED, synth.RING

CASES = [
    # kind, B, R, Hq, Hkv, D, seq_lens, extra
    (LINEAR, 3, 1, 32, 8, 128, [513, 1, 4097], {}),
    (LINEAR, 2, 4, 28, 4, 128, [2000, 37], {}),
    (PAGED, 4, 4, 32, 8, 128, [64, 100, 1030, 17], {"block_size": 16}),
    (PAGED, 3, 2, 16, 4, 64, [37, 300, 129], {"block_size": 5, "num_blocks": 200}),
    (RING, 4, 1, 32, 8, 128, [9000, 300, 16390, 8193], {"window": 8192, "ring": 16384}),
    (RING, 3, 4, 16, 4, 128, [1500 + 3, 4, 1501], {"window": 750, "ring": 1500}),
    # more requests than one launch takes: the batch is cut into launches
    (LINEAR, 260, 2, 8, 2, 128, [2 + (37 * i) % 150 for i in range(260)], {}),
]


def _run(case, fused):
    dev = "cuda"
    cache = to_device(case, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    q, kn, vn = case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev)
    sm, seq, pos = case.slot_mapping.to(dev), case.seq_lens.to(dev), case.positions.to(dev)
    if fused:
        out = gq.attn_decode_append(q, kn, vn, sm, cache, seq, pos, case.max_seq_len(),
                                    case.window, case.scale, err=err)
    else:
        gq.attn_kv_append(kn, vn, sm, cache, err=err)
        out = gq.attn_decode(q, cache, seq, pos, case.max_seq_len(), case.window, case.scale,
                             err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, cache


@pytest.mark.parametrize("kind,B,R,Hq,Hkv,D,seq,extra", CASES)
def test_fused_equals_append_then_decode(kind, B, R, Hq, Hkv, D, seq, extra):
    case = synth.decode_case(9200 + B * R + D + 10 * int(kind), kind, B, R, Hq, Hkv, D, seq, **extra)
    out_f, cache_f = _run(case, fused=True)
    out_u, cache_u = _run(case, fused=False)
    assert torch.equal(out_f, out_u), "fused decode differs from append + decode"
    assert torch.equal(cache_f.k, cache_u.k) and torch.equal(cache_f.v, cache_u.v)
    ref, kc, vc = oracle_decode(case)
    compare(out_f, ref, f"fused {kind} R={R}")
    assert np.array_equal(oracle.bf16_bits(cache_f.k), kc)
    assert np.array_equal(oracle.bf16_bits(cache_f.v), vc)


def test_fused_reports_out_of_range_slot():
    case = synth.decode_case(9300, LINEAR, 2, 1, 8, 2, 128, [40, 40])
    sm = case.slot_mapping.clone()
    sm[1] = 10_000_000
    case.slot_mapping = sm
    dev = "cuda"
    cache = to_device(case, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gq.attn_decode_append(case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev),
                                sm.to(dev), cache, case.seq_lens.to(dev), case.positions.to(dev),
                                40, 0, case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gq.ATTN_ERR_BOUNDS
    assert torch.isfinite(out.float()).all()


def _ulp_diff(a_bits, b_bits):
    """|a - b| in bf16 steps, for bit patterns of finite values."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(key(a_bits) - key(b_bits))


ROPE_CASES = [
    (LINEAR, 2, 1, 28, 4, 128, [14449, 900], {}),
    (PAGED, 3, 4, 32, 8, 128, [64, 1030, 17], {"block_size": 16}),
    (RING, 2, 4, 32, 32, 64, [6004, 777], {"window": 750, "ring": 1500}),
]


@pytest.mark.parametrize("kind,B,R,Hq,Hkv,D,seq,extra", ROPE_CASES)
def test_fused_rope(kind, B, R, Hq, Hkv, D, seq, extra):
    """q and the new keys rotated at their positions (interleaved pairs,
    float32 angle p * inv_freq[i]) before the append and the attention."""
    case = synth.decode_case(9400 + B * R + D + 10 * int(kind), kind, B, R, Hq, Hkv, D, seq,
                             **extra)
    inv = (1_000_000.0 ** (-np.arange(D // 2) / (D // 2))).astype(np.float32)
    dev = "cuda"
    cache = to_device(case, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gq.attn_decode_append(case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev),
                                case.slot_mapping.to(dev), cache, case.seq_lens.to(dev),
                                case.positions.to(dev), case.max_seq_len(), case.window,
                                case.scale, err=err, rope_inv_freq=torch.from_numpy(inv).to(dev))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle: rotate, append, attend
    qpos = case.positions.numpy()
    kpos = np.concatenate([np.arange(s - R, s) for s in case.seq_lens.tolist()])
    qb = oracle.bf16_bits(case.q).reshape(B * R, Hq, D)
    q_rot = oracle.rope(qb, qpos, inv).reshape(B, R, Hq, D)
    k_rot = oracle.rope(oracle.bf16_bits(case.k_new), kpos, inv)
    kc, vc = oracle.bf16_bits(case.k_cache).copy(), oracle.bf16_bits(case.v_cache).copy()
    oracle.kv_append(kc, vc, k_rot, oracle.bf16_bits(case.v_new), case.slot_mapping.numpy())
    cd = {"kind": case.kind, "k": kc, "v": vc, "slots_per_seq": case.slots_per_seq,
          "block_table": None if case.block_table is None else case.block_table.numpy(),
          "block_size": case.block_size}
    rc, ref = oracle.decode(q_rot, cd, case.seq_lens.numpy(), qpos, case.window, case.scale,
                            case.n_kv_heads)
    assert rc == 0
    compare(out, ref, f"fused rope {kind} R={R}")
    # the cache holds the rotated keys (float rounding: at most one bf16 step apart)
    assert np.array_equal(oracle.bf16_bits(cache.v), vc)
    d = _ulp_diff(oracle.bf16_bits(cache.k), kc)
    assert d.max() <= 1, f"rotated keys differ by {d.max()} bf16 steps"


def test_tables_early_same_result():
    """ATTN_DECODE_TABLES_EARLY changes when seq_lens and positions are read,
    not what is computed: back-to-back calls (each launched while the previous
    one finishes) give the same bits with and without it."""
    dev = "cuda"
    case = synth.decode_case(9500, PAGED, 4, 2, 32, 8, 128, [3000, 64, 1029, 2048],
                             block_size=16)
    outs = {}
    for early in (False, True):
        cache = to_device(case, dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        args = (case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev),
                case.slot_mapping.to(dev), cache, case.seq_lens.to(dev), case.positions.to(dev),
                case.max_seq_len(), 0, case.scale)
        res = [gq.attn_decode_append(*args, err=err, tables_early=early) for _ in range(4)]
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs[early] = res
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("kind,B,seq,window", [(LINEAR, 2, [8192, 5000], 0),
                                               (LINEAR, 1, [512], 0),
                                               (RING, 4, [9000, 20000, 4100, 16400], 4096),
                                               (PAGED, 4, [3000, 64, 1029, 2048], 0)])
def test_cache_early_same_result(kind, B, seq, window):
    """ATTN_DECODE_CACHE_EARLY lets the first cache tiles be loaded before the
    previous kernel completes; it changes when they are read, not what is
    computed: back-to-back calls give the bits of calls without it, and match
    the oracle."""
    dev = "cuda"
    case = synth.decode_case(9510 + B, kind, B, 1, 28 if kind == LINEAR else 32,
                             4 if kind == LINEAR else 8, 128, seq, window=window, block_size=16)
    outs = {}
    for early in (False, True):
        cache = to_device(case, dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        args = (case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev),
                case.slot_mapping.to(dev), cache, case.seq_lens.to(dev), case.positions.to(dev),
                case.max_seq_len(), window, case.scale)
        res = [gq.attn_decode_append(*args, err=err, tables_early=True, cache_early=early)
               for _ in range(4)]
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs[early] = res
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)
    ref, _, _ = oracle_decode(case)
    compare(outs[True][-1], ref, f"cache early {kind}")
