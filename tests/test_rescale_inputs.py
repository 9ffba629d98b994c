"""The shaped inputs of the rescale parity tests have the score structure
those tests rely on (checked on the CPU, in fp64, from the bf16 inputs).

Every row's score against the key at position t must follow the profile's
level s(t) in log2 units: c s(t) plus noise, where c is a factor of the
query head near 1 (the head's own noise projected on its direction u); for
the spike profile the last four keys of each 128-key tile must stand far
enough above the rest that a row maximum missing any of them would push P
past f16's range (2^16).
"""
import math

import numpy as np
import pytest
import torch

from gqa_attention_kv_gb300 import synth
import test_gpu_rescale as R

NOISE = 2.0  # log2 units: |score - c level| for every key


def scores_log2(q_row, k_rows, scale):
    return (k_rows.double().numpy() @ q_row.double().numpy()) * scale * math.log2(math.e)


def check_follows(s, lv, profile, where):
    """s = c lv + noise with |c - 1| < 0.1 and |noise| < NOISE; spike gap > 16."""
    c = float(s @ lv / (lv @ lv)) if (lv @ lv) > 0 else 1.0
    assert abs(c - 1.0) < 0.1, (where, c)
    assert np.abs(s - c * lv).max() < NOISE, (where, np.abs(s - c * lv).max())
    if profile == "spike":
        top = lv > 0
        # a maximum that missed a spike column would leave P above 2^16
        assert s[top].min() - s[~top].max() > 16.0, where


@pytest.mark.parametrize("profile", ["ramp", "stairs", "saw", "spike"])
def test_decode_inputs_follow_the_level(profile):
    case = synth.decode_case(9100 + 4 + 3, R.PAGED, 3, 4, 32, 8, 128, [4097, 1500, 700],
                             block_size=16)
    R.shape_decode(case, profile, 17)
    bt = case.block_table.numpy()
    for b, L in enumerate([4097, 1500, 700]):
        t = np.arange(L - 4)
        slots = torch.from_numpy((bt[b, t // 16] * 16 + t % 16).astype(np.int64))
        for h in (0, 13, 31):  # q heads of KV heads 0, 3 and 7
            # the cache's rows and the step's own rows, in position order
            s = np.concatenate([
                scores_log2(case.q[b, 3, h], case.k_cache[slots, h // 4], case.scale),
                scores_log2(case.q[b, 3, h], case.k_new[b * 4:(b + 1) * 4, h // 4], case.scale)])
            check_follows(s, R.level(profile, np.arange(L)), profile, (profile, b, h))


@pytest.mark.parametrize("profile", ["ramp", "stairs", "saw", "spike"])
@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(1, 1500, 28, 4, 128), (2, 750, 32, 32, 64)])
def test_prefill_inputs_follow_the_level(profile, B, T, Hq, Hkv, D):
    p = synth.prefill_case(9500 + T + D, B, T, Hq, Hkv, D)
    u = R.directions(31, Hkv, D)
    ug = np.repeat(u, Hq // Hkv, axis=0)
    q = torch.from_numpy(p.q.double().numpy() * 0.25 + ug).to(torch.bfloat16)
    a = R.level(profile, np.arange(T)) / R.per_unit(D, p.scale)
    k = R.shaped(p.k, np.broadcast_to(a, (B, T)), u)
    t = np.arange(T)
    for b in range(B):
        for h in (0, Hq - 1):
            s = scores_log2(q[b, T - 1, h], k[b, :, h // (Hq // Hkv)], p.scale)
            check_follows(s, R.level(profile, t), profile, (profile, b, h))
