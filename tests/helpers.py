"""Shared helpers for the parity tests: run a case through the library and
through the oracle, and compare with the stated tolerance."""
import numpy as np
import torch

import oracle
import gqa_attention_kv_gb300 as gq

MAX_ABS = 1e-2   # bf16 output vs fp64 oracle, element-wise
REL_L2 = 2e-3    # ||out - ref|| / ||ref||
# The output is rounded once to bf16.  Below |o| = 4 every real lies within
# half a bf16 step (at most 1/128) of a bf16 value, so max-abs 1e-2 holds
# literally; from 4 up half a step is 1/64 or more, and no bf16 result can be
# within 1e-2 of every exact value.  There an element may differ from the
# exact value by half a bf16 step (the final rounding) plus ACCUM_SLACK * |o|:
# the kernels' own error before that rounding (P rounded once to f16, at most
# 2^-11 of the largest value a row attends, which in the few-key rows where
# |o| >= 4 occurs is about |o|; fp32 accumulation far less).
FAITHFUL_FROM = 4.0
ACCUM_SLACK = 2.0 ** -9


def bf16_step(x):
    """Spacing of bf16 values at |x| (|x| >= 2^-126): 2^(exponent - 7)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def element_bound(ref):
    big = 0.5 * bf16_step(ref) + ACCUM_SLACK * np.abs(ref)
    return np.where(np.abs(ref) >= FAITHFUL_FROM, big, MAX_ABS)


def bits(t):
    return oracle.bf16_bits(t)


def oracle_decode(case):
    """Oracle: append the step's rows, then decode.  Returns (out fp64, k, v bits)."""
    kc, vc = bits(case.k_cache).copy(), bits(case.v_cache).copy()
    oracle.kv_append(kc, vc, bits(case.k_new), bits(case.v_new), case.slot_mapping.cpu().numpy())
    cd = {"kind": case.kind, "k": kc, "v": vc, "slots_per_seq": case.slots_per_seq,
          "block_table": None if case.block_table is None else case.block_table.cpu().numpy(),
          "block_size": case.block_size}
    rc, out = oracle.decode(bits(case.q), cd, case.seq_lens.cpu().numpy(),
                            case.positions.cpu().numpy(), case.window, case.scale,
                            case.n_kv_heads)
    assert rc == 0, f"oracle status {rc}"
    return out, kc, vc


def to_device(case, dev="cuda"):
    cache = gq.KVCache(case.kind, case.k_cache.to(dev), case.v_cache.to(dev),
                       slots_per_seq=case.slots_per_seq,
                       block_table=None if case.block_table is None else case.block_table.to(dev),
                       block_size=case.block_size)
    return cache


def gpu_decode(case, dev="cuda", max_seq_len=None, err=None):
    """Library: append then decode on the device.  Returns (out, cache)."""
    cache = to_device(case, dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    gq.attn_kv_append(case.k_new.to(dev), case.v_new.to(dev), case.slot_mapping.to(dev), cache,
                      err=err)
    out = gq.attn_decode(case.q.to(dev), cache, case.seq_lens.to(dev), case.positions.to(dev),
                         max_seq_len or case.max_seq_len(), case.window, case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item())}"
    return out, cache


def compare(out, ref, where=""):
    got = out.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{where}: non-finite output"
    diff = np.abs(got - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got))
    over = diff / element_bound(ref) if diff.size else diff
    if diff.size:
        idx = np.unravel_index(int(over.argmax()), diff.shape)
        worst = (f"worst at {idx}: got {got[idx]:.5f} ref {ref[idx]:.5f} "
                 f"(bound {float(element_bound(ref[idx])):.4g})")
    else:
        worst = ""
    ok = bool((over <= 1.0).all()) if diff.size else True
    assert ok and rel <= REL_L2, \
        f"{where}: max-abs {max_abs:.3e} (<= {MAX_ABS} below |o| {FAITHFUL_FROM}, half a bf16 " \
        f"step + {ACCUM_SLACK:.3g} |o| above), rel-L2 {rel:.3e} (<= {REL_L2}); {worst}"
    return max_abs, rel
