"""Prefill parity: the tcgen05 prefill kernel against the fp64 oracle.

Covers on and off every 128-row tile edge (vibevoice.c, "Attention
backends": prefill on and off every tile edge), head_dim 64 and 128, GQA
ratios 1, 4 and 7, sliding windows (Voxtral notes, "Offline Encoder"), and
batches of several sequences.
"""
import numpy as np
import pytest
import torch

import oracle
import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import bits, compare

pytestmark = pytest.mark.gpu


def run(p, rows=None):
    dev = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gq.attn_prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.window, p.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item())}"
    rc, ref = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), p.window, p.scale, rows=rows)
    assert rc == 0
    if rows is not None:
        out = out[:, rows]
    return out, ref


@pytest.mark.parametrize("T", [1, 2, 7, 127, 128, 129, 255, 256, 257, 300])
@pytest.mark.parametrize("D", [64, 128])
def test_tile_edges(T, D):
    p = synth.prefill_case(100 + T + D, 2, T, 8, 2, D)
    out, ref = run(p)
    compare(out, ref, f"T={T} D={D}")


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (28, 4), (12, 2), (32, 8)])
def test_gqa_ratios(Hq, Hkv):
    p = synth.prefill_case(200 + Hq, 1, 400, Hq, Hkv, 128)
    out, ref = run(p)
    compare(out, ref, f"{Hq}/{Hkv}")


@pytest.mark.parametrize("T,W", [(300, 1), (300, 17), (300, 128), (600, 200), (1000, 750),
                                 (257, 300)])
def test_window(T, W):
    p = synth.prefill_case(300 + W, 1, T, 8, 8, 64, window=W)
    out, ref = run(p)
    compare(out, ref, f"T={T} W={W}")


@pytest.mark.parametrize("T,W,Hq,Hkv,D", [(1100, 130, 28, 4, 128), (900, 64, 12, 2, 128),
                                          (1300, 257, 7, 1, 64), (520, 255, 4, 2, 64)])
def test_window_gqa(T, W, Hq, Hkv, D):
    """Windows with grouped heads, whose CTAs walk their key tiles from
    different starting tiles: key tiles that one query tile of a CTA sees and
    the other does not (before the window or after the diagonal), at any
    position of the walk."""
    p = synth.prefill_case(350 + W + Hq, 1, T, Hq, Hkv, D, window=W)
    out, ref = run(p)
    compare(out, ref, f"T={T} W={W} {Hq}/{Hkv} D={D}")


@pytest.mark.parametrize("B,T,Hq,Hkv,D,W", [(3, 1500, 16, 4, 128, 0), (2, 2333, 32, 8, 64, 700)])
def test_two_tile_ctas_batched(B, T, Hq, Hkv, D, W):
    """Launches large enough for two Q tiles per CTA (pairs x heads x batch at
    least the SM count) with several sequences, a ragged length and a window,
    checked on sampled rows: every tile edge of the first and last sequence's
    pairs, the first and last rows, and seeded random rows."""
    p = synth.prefill_case(700 + T + W, B, T, Hq, Hkv, D, window=W)
    edges = [r for t in range(128, T, 128) for r in (t - 1, t)]
    g = np.random.default_rng(T)
    rows = sorted(set(list(range(8)) + list(range(T - 8, T)) + edges[::3] +
                      g.integers(0, T, 24).tolist()))
    out, ref = run(p, rows=rows)
    compare(out, ref, f"B={B} T={T} {Hq}/{Hkv} D={D} W={W} (sampled rows)")


def test_encoder_prefill_full():
    """The speech-encoder shape at full size: T=750, 32 heads, D=64."""
    p = synth.encoder_prefill()
    out, ref = run(p)
    compare(out, ref, "encoder T=750")


def test_encoder_prefill_window_full():
    """The 1,500-frame variant with the 750-frame window."""
    p = synth.encoder_prefill(long=True)
    out, ref = run(p)
    compare(out, ref, "encoder T=1500 W=750")


def test_qwen_prompt_sampled_rows():
    """The 14,449-token Qwen2-7B prompt, checked on sampled rows: every tile
    edge, the first and last 64 rows and 64 seeded random rows."""
    p = synth.qwen_prefill()
    T = p.q.shape[1]
    edges = [r for t in range(128, T, 128) for r in (t - 1, t)]
    g = np.random.default_rng(20263)
    rows = sorted(set(list(range(64)) + list(range(T - 64, T)) + edges[::9] +
                      g.integers(0, T, 64).tolist()))
    out, ref = run(p, rows=rows)
    compare(out, ref, "qwen prompt (sampled rows)")


def test_deterministic():
    p = synth.prefill_case(400, 1, 700, 28, 4, 128)
    dev = "cuda"
    a = gq.attn_prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), 0, p.scale)
    b = gq.attn_prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), 0, p.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_large_values_within_f16_range():
    """V with magnitudes up to ~2^15 (N(0,1) x 2^12): converting V to f16 for
    P V is exact there and a power-of-two scale commutes with every rounding
    of the path, so each output is exactly 2^12 times the unscaled one, and
    the unscaled output meets the stated tolerance."""
    p = synth.prefill_case(410, 1, 300, 8, 2, 128)
    dev = "cuda"
    q, k, v = p.q.to(dev), p.k.to(dev), p.v.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    small = gq.attn_prefill(q, k, v, 0, p.scale, err=err)
    big = gq.attn_prefill(q, k, v * 4096.0, 0, p.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(big, small * 4096.0)
    rc, ref = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 0, p.scale)
    assert rc == 0
    compare(small, ref, "V unscaled")


def test_v_beyond_f16_is_reported():
    """A V element of magnitude 2^16 or more has no f16 value: the kernel
    saturates it, keeps every output finite and stores ATTN_ERR_UNSUPPORTED
    in the error word (it never faults)."""
    p = synth.prefill_case(411, 1, 200, 4, 4, 64)
    p.v[0, 150, 2, 7] = 1.0e5
    dev = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gq.attn_prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), 0, p.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gq.ATTN_ERR_UNSUPPORTED
    assert torch.isfinite(out.float()).all()
    # rows before position 150 never see the large value: unchanged parity
    rc, ref = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 0, p.scale, rows=list(range(150)))
    assert rc == 0
    compare(out[:, :150], ref, "rows before the large value")


@pytest.mark.parametrize("B,T,Hq,Hkv,D,W", [(2, 513, 8, 2, 128, 0), (1, 1100, 4, 4, 64, 300),
                                            (3, 900, 6, 3, 128, 0), (1, 640, 2, 1, 64, 129)])
def test_small_launches(B, T, Hq, Hkv, D, W):
    """Launches of fewer Q-tile pairs than SMs (one Q tile per CTA): batches,
    GQA, both head dims and windows."""
    p = synth.prefill_case(500 + T + D + W, B, T, Hq, Hkv, D, window=W)
    out, ref = run(p)
    compare(out, ref, f"B={B} T={T} {Hq}/{Hkv} D={D} W={W}")
