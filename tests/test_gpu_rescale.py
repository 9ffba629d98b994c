"""Parity under score profiles that move the running maximum late.

Every kernel keeps, per query row, a reference maximum for its online softmax
and rescales its running output only when a chunk's scores pass that
reference by more than 2^8 (the lazy rescale of the prefill, chunk and decode
kernels).  Seeded N(0, 1) inputs settle the maximum within the first tiles,
so these cases shape q and K instead: q of every head near a fixed +-1
direction u of its KV head, and the key at position t near a(t) u, so that
every row's scores follow a chosen level s(t) (log2 units, scaled by a factor
of the head within 10% of 1) plus small noise (pinned on the CPU in
`test_rescale_inputs.py`):

* ramp:   s rises by 0.5 per 16 keys: the reference moves every ~16 chunks,
          and P approaches 2^8 just before each move;
* stairs: jumps of 8.5 every 320 keys (a rescale by 2^-8.5 each time) with a
          7.5 step half way (no rescale: P near 2^7.5 on that half);
* saw:    alternates 0 / 7.5 every 160 keys: the reference never moves after
          the first chunk, and split partial states of comparable weight
          carry references below their true maxima into the merges;
* spike:  the last four keys of every 128-key tile 20 above the rest: a row
          maximum that missed a tile's last columns would leave P near 2^20,
          past f16's range (the prefill and chunk kernels).

The output is checked against the fp64 oracle at the stated tolerance, for
the decode split kernel (8-row and 16-row tilings, bf16 and E4M3 caches, one
unit split over many CTAs), the chunk kernel and the prefill kernel.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import bits, compare, gpu_decode, oracle_decode
from test_gpu_fp8 import check_case

pytestmark = pytest.mark.gpu

LINEAR, PAGED = synth.LINEAR, synth.PAGED


def level(profile, t):
    t = np.asarray(t, dtype=np.float64)
    if profile == "ramp":
        return t / 32.0
    if profile == "stairs":
        return 8.5 * np.floor(t / 320.0) + 7.5 * ((t % 320) >= 160)
    if profile == "saw":
        return 7.5 * (np.floor(t / 160.0) % 2)
    if profile == "spike":
        return 20.0 * ((t % 128) >= 124)
    raise ValueError(profile)


def directions(seed, n_kv_heads, D):
    g = np.random.default_rng(seed)
    return g.choice([-1.0, 1.0], size=(n_kv_heads, D))


def shaped(base, coef, u):
    """bf16 of coef * u + base / 4 (base: bf16 noise [..., Hkv, D])."""
    x = base.double().numpy() * 0.25 + coef[..., None, None] * u
    return torch.from_numpy(x).to(torch.bfloat16)


def per_unit(D, scale):
    """log2-score per unit of a(t): q.k ~ a * D for q ~ u, k ~ a u."""
    return D * scale * math.log2(math.e)


def shape_decode(case, profile, seed):
    """Shape q, the cache rows of every request's positions and the step's rows."""
    B, R, Hq, D = case.q.shape
    Hkv = case.n_kv_heads
    u = directions(seed, Hkv, D)
    ug = np.repeat(u, Hq // Hkv, axis=0)  # q head h -> u of its KV head
    q = case.q.double().numpy() * 0.25 + ug
    case.q = torch.from_numpy(q).to(torch.bfloat16)
    k = case.k_cache.clone()
    kn = case.k_new.clone()
    unit = per_unit(D, case.scale)
    seq = case.seq_lens.cpu().tolist()
    for b in range(B):
        t = np.arange(seq[b] - R)
        if case.kind == LINEAR:
            slots = b * case.slots_per_seq + t
        else:
            bt = case.block_table.cpu().numpy()
            slots = bt[b, t // case.block_size] * case.block_size + t % case.block_size
        slots = torch.from_numpy(slots.astype(np.int64))
        k[slots] = shaped(case.k_cache[slots], level(profile, t) / unit, u)
        tn = np.arange(seq[b] - R, seq[b])
        kn[b * R:(b + 1) * R] = shaped(case.k_new[b * R:(b + 1) * R], level(profile, tn) / unit, u)
    case.k_cache, case.k_new = k, kn
    return case


@pytest.mark.parametrize("profile", ["ramp", "stairs", "saw"])
@pytest.mark.parametrize("kind,R,Hq,Hkv,seq", [
    (LINEAR, 1, 28, 4, [4097, 2500]),        # 7 rows: the 8-row tiling
    (PAGED, 4, 32, 8, [4097, 1500, 700]),    # 16 rows: the 16-row tiling
])
def test_decode_bf16(profile, kind, R, Hq, Hkv, seq):
    case = synth.decode_case(9100 + R + len(seq), kind, len(seq), R, Hq, Hkv, 128, seq,
                             block_size=16)
    shape_decode(case, profile, 17)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"{profile} kind={kind} R={R} {Hq}/{Hkv}")


@pytest.mark.parametrize("profile", ["ramp", "stairs", "saw"])
@pytest.mark.parametrize("kind,R,Hq,Hkv,seq", [
    (LINEAR, 1, 28, 4, [4097, 2500]),
    (PAGED, 4, 32, 8, [4097, 1500, 700]),
])
def test_decode_fp8(profile, kind, R, Hq, Hkv, seq):
    case = synth.decode_case(9200 + R + len(seq), kind, len(seq), R, Hq, Hkv, 128, seq,
                             block_size=16)
    shape_decode(case, profile, 19)
    check_case(case, where=f"E4M3 {profile} kind={kind} R={R} {Hq}/{Hkv}")


@pytest.mark.parametrize("profile", ["stairs", "saw"])
def test_decode_one_unit_over_many_ctas(profile):
    """One request at 14,449 keys: its units split over many CTAs and merged."""
    case = synth.decode_case(9300, LINEAR, 1, 1, 28, 4, 128, [14449])
    shape_decode(case, profile, 23)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"{profile} one unit, 14,449 keys")


@pytest.mark.parametrize("profile", ["ramp", "stairs", "saw", "spike"])
def test_chunk_kernel(profile):
    """29-row chunks of 28/4 heads (203 rows a KV group: the tcgen05 chunk kernel)."""
    case = synth.decode_case(9400, LINEAR, 2, 29, 28, 4, 128, [3029, 1529])
    shape_decode(case, profile, 29)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"{profile} chunk")


@pytest.mark.parametrize("profile", ["ramp", "stairs", "saw", "spike"])
@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(1, 1500, 28, 4, 128), (2, 750, 32, 32, 64)])
def test_prefill(profile, B, T, Hq, Hkv, D):
    p = synth.prefill_case(9500 + T + D, B, T, Hq, Hkv, D)
    u = directions(31, Hkv, D)
    ug = np.repeat(u, Hq // Hkv, axis=0)
    p.q = torch.from_numpy(p.q.double().numpy() * 0.25 + ug).to(torch.bfloat16)
    a = level(profile, np.arange(T)) / per_unit(D, p.scale)
    p.k = shaped(p.k, np.broadcast_to(a, (B, T)), u)
    dev = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gq.attn_prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.window, p.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rc, ref = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), p.window, p.scale)
    assert rc == 0
    compare(out, ref, f"{profile} prefill B={B} T={T} {Hq}/{Hkv} D={D}")
