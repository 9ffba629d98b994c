"""Pins of the oracle's FP8 cache functions (vibevoice.c, "KV cache") to facts
fixed by the E4M3 format's definition and by arithmetic.

The FP8 format is E4M3 of the OCP 8-bit floating point specification: sign,
four exponent bits with bias 7, three mantissa bits, subnormals at exponent
field 0, S.1111.111 as NaN, no infinities, 448 the largest finite value.  The
pins below do not re-type the oracle's encoder: they check it against a
nearest-value search over the 127 non-negative codes, against values the
definition gives by hand, and against the error bound of round-to-nearest.
"""
import numpy as np
import torch

import oracle
from gqa_attention_kv_gb300 import synth


def test_fp8_values_from_the_definition():
    """Hand values (a wrong bias, a missing implicit bit or a subnormal read
    as normal fails one of them)."""
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5,
            0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x48: 4.0, 0x5D: 26.0, 0x62: 40.0, 0x77: 240.0, 0x7E: 448.0,
            0xB8: -1.0, 0xFE: -448.0}
    got = oracle.fp8_to_f64(np.array(list(want), dtype=np.uint8))
    assert got.tolist() == list(want.values())
    neg0 = oracle.fp8_to_f64(np.array([0x80], dtype=np.uint8))[0]
    assert neg0 == 0.0 and np.signbit(neg0)
    assert np.isnan(oracle.fp8_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_fp8_codes_ordered_and_symmetric():
    pos = oracle.fp8_to_f64(np.arange(0x7F, dtype=np.uint8))
    assert (np.diff(pos) > 0).all(), "non-negative codes 0x00..0x7E increase strictly"
    neg = oracle.fp8_to_f64(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)
    # spacing: 2^-9 below 2^-6, then 1/8 of the binade
    assert np.allclose(np.diff(pos[:9]), 2.0 ** -9)
    for e in range(1, 16):
        lo = 2.0 ** (e - 7)
        binade = pos[(pos >= lo) & (pos < 2 * lo)]
        assert np.allclose(np.diff(binade), lo / 8)


def test_fp8_encode_inverts_decode_on_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.fp8_to_f64(codes).astype(np.float32)
    assert np.array_equal(oracle.f32_to_fp8(vals), codes)


def _nearest_code(x):
    """Brute force: the finite code nearest to x, ties to the even code,
    magnitudes past 448 saturated."""
    if np.isnan(x):
        return 0x7F
    table = oracle.fp8_to_f64(np.arange(0x7F, dtype=np.uint8))
    a = min(abs(float(x)), 448.0)
    d = np.abs(table - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
    return code | (0x80 if np.signbit(x) else 0)


def test_fp8_encode_matches_nearest_search():
    g = np.random.default_rng(20260)
    table = oracle.fp8_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (table[1:] + table[:-1]) / 2  # every tie
    xs = np.concatenate([
        g.standard_normal(3000) * 10.0 ** g.uniform(-4, 3, 3000),
        mids, -mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(0)),
        [0.0, -0.0, 447.9, 448.0, 463.9, 464.0, 1e6, -1e6, np.inf, -np.inf, np.nan],
    ]).astype(np.float32)
    got = oracle.f32_to_fp8(xs)
    want = np.array([_nearest_code(x) for x in xs], dtype=np.uint8)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [(float(xs[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_fp8_ties_and_saturation_by_hand():
    cases = {2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02, 1 + 1 / 16: 0x38, 1 + 3 / 16: 0x3A,
             416.0: 0x7D, 432.0: 0x7E, 464.0: 0x7E, 1e30: 0x7E, float("inf"): 0x7E,
             float("-inf"): 0xFE, -2.0 ** -11: 0x80}
    got = oracle.f32_to_fp8(np.array(list(cases), dtype=np.float32))
    assert [int(c) for c in got] == list(cases.values())


def test_fp8_to_bf16_is_exact():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    bf = oracle.fp8_to_bf16_bits(codes)
    assert np.array_equal(oracle.bf16_to_f64(bf), oracle.fp8_to_f64(codes))


def test_fp8_append_within_rounding_bound_of_shifted_keys():
    """Each stored K code is the rounding of float32(k) - ref: the decoded
    value lies within half a step of it (2^-4 relative in the normal range,
    2^-10 absolute below it); V codes likewise without a shift.  Slot rules
    are the bf16 append's: out-of-range rows skipped, the last row wins."""
    g = synth.generator(77)
    S, Hkv, D, n = 40, 2, 16, 12
    k_new = synth.normal_bf16(g, (n, Hkv, D)) * 30
    v_new = synth.normal_bf16(g, (n, Hkv, D))
    ref = np.random.default_rng(1).standard_normal((Hkv, D)).astype(np.float32) * 25
    slots = np.array([3, 7, 7, 50, -1, 0, 11, 12, 13, 14, 15, 39], dtype=np.int64)
    kc = np.full((S, Hkv, D), 0x55, dtype=np.uint8)
    vc = np.full((S, Hkv, D), 0x55, dtype=np.uint8)
    skipped = oracle.kv_append_fp8(kc, vc, oracle.bf16_bits(k_new), oracle.bf16_bits(v_new),
                                   slots, k_ref=ref)
    assert skipped == 2
    kf = oracle.bf16_to_f64(oracle.bf16_bits(k_new))
    vf = oracle.bf16_to_f64(oracle.bf16_bits(v_new))
    for i, s in enumerate(slots):
        if s < 0 or s >= S or (s == 7 and i == 1):
            continue
        x = (kf[i].astype(np.float32) - ref).astype(np.float64)
        for want, got in ((x, oracle.fp8_to_f64(kc[s])), (vf[i], oracle.fp8_to_f64(vc[s]))):
            clipped = np.clip(want, -448, 448)
            bound = np.maximum(np.abs(clipped) * 2.0 ** -4, 2.0 ** -10)
            assert (np.abs(got - clipped) <= bound).all()
    untouched = [s for s in range(S) if s not in set(slots.tolist())]
    assert (kc[untouched] == 0x55).all() and (vc[untouched] == 0x55).all()


def test_kv_reference_is_the_row_mean():
    g = synth.generator(5)
    row = synth.normal_bf16(g, (1, 3, 8))
    same = row.expand(9, 3, 8).contiguous()
    assert np.array_equal(oracle.kv_reference(oracle.bf16_bits(same)),
                          oracle.bf16_to_f64(oracle.bf16_bits(row))[0])
    two = synth.normal_bf16(g, (2, 3, 8))
    t = oracle.bf16_to_f64(oracle.bf16_bits(two))
    assert np.allclose(oracle.kv_reference(oracle.bf16_bits(two)), (t[0] + t[1]) / 2,
                       rtol=0, atol=1e-15)
    many = synth.normal_bf16(g, (57, 3, 8))
    perm = many[np.random.default_rng(0).permutation(57)]
    assert np.allclose(oracle.kv_reference(oracle.bf16_bits(many)),
                       oracle.kv_reference(oracle.bf16_bits(perm)), rtol=0, atol=1e-13)


def _attention(q, k_bits, v_bits, seq, D, Hkv):
    B, R, Hq, _ = q.shape
    cache = {"kind": oracle.LINEAR, "k": k_bits, "v": v_bits, "slots_per_seq": seq}
    rc, out = oracle.decode(q, cache, np.array([seq], dtype=np.int32),
                            np.array([seq - 1], dtype=np.int32), 0, D ** -0.5, Hkv)
    assert rc == 0
    return out.reshape(-1)


def test_reference_shift_rescues_fp8_keys_with_a_common_component():
    """The page's finding, reproduced on synthetic keys shaped like the ones
    it describes (a common component of norm ~273 against ~11 for the rest):
    stored raw, FP8 keys lose the attention pattern; stored relative to the
    mean of the first chunk, the output stays close to the bf16 one."""
    g = synth.generator(2026)
    Hkv, D, seq, Hq = 2, 128, 512, 8
    common = synth.normal_bf16(g, (1, Hkv, D)).float() * (273 / D ** 0.5)
    k = (common + synth.normal_bf16(g, (seq, Hkv, D)).float()).to(torch.bfloat16)
    v = synth.normal_bf16(g, (seq, Hkv, D))
    q = oracle.bf16_bits(synth.normal_bf16(g, (1, 1, Hq, D)) * 3)
    kb, vb = oracle.bf16_bits(k), oracle.bf16_bits(v)
    exact = _attention(q, kb, vb, seq, D, Hkv)
    cos = {}
    for name, ref in (("raw", None),
                      ("shifted", oracle.kv_reference(kb[:128]).astype(np.float32))):
        kc = np.zeros((seq, Hkv, D), dtype=np.uint8)
        vc = np.zeros((seq, Hkv, D), dtype=np.uint8)
        oracle.kv_append_fp8(kc, vc, kb, vb, np.arange(seq), k_ref=ref)
        out = _attention(q, oracle.fp8_to_bf16_bits(kc), oracle.fp8_to_bf16_bits(vc), seq, D,
                         Hkv)
        cos[name] = float(out @ exact / np.linalg.norm(out) / np.linalg.norm(exact))
    assert cos["shifted"] > 0.995, cos
    assert cos["raw"] < cos["shifted"] - 0.02, cos
