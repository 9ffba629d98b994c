"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

Each test states which plausible mistake in the oracle it would catch.  None
of them re-types the oracle's loops: they use worked examples printed on the
pages (tests/golden), closed forms, invariants and an independent dense
(matrix) formulation on tiny shapes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_attention_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t):
    return oracle.bf16_bits(t)


def f64(t):
    return oracle.bf16_to_f64(bits(t))


def cache_dict(case, k=None, v=None):
    return {"kind": case.kind, "k": bits(case.k_cache if k is None else k),
            "v": bits(case.v_cache if v is None else v), "slots_per_seq": case.slots_per_seq,
            "block_table": None if case.block_table is None else case.block_table.numpy(),
            "block_size": case.block_size}


def run_case(case):
    """Append the step's rows, then decode, all in the oracle."""
    kc, vc = bits(case.k_cache).copy(), bits(case.v_cache).copy()
    skipped = oracle.kv_append(kc, vc, bits(case.k_new), bits(case.v_new),
                               case.slot_mapping.numpy())
    assert skipped == 0
    rc, out = oracle.decode(bits(case.q), cache_dict(case, None, None) | {"k": kc, "v": vc},
                            case.seq_lens.numpy(), case.positions.numpy(), case.window,
                            case.scale, case.n_kv_heads)
    return rc, out, kc, vc


# --------------------------------------------------------------------------
# exact widening and the pages' worked examples
# --------------------------------------------------------------------------

def test_bf16_widening_exact():
    # 1.0, -2.0, 0.15625, the smallest normal, and the largest finite bf16.
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3E20: 0.15625, 0x0080: 2.0 ** -126,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127}
    lib = oracle._load()
    for b, want in cases.items():
        assert lib.oracle_bf16_to_f64(b) == want
        assert oracle.bf16_to_f64(np.array([b], dtype=np.uint16))[0] == want


def test_ring_abs_pos_worked_example():
    """Catches a wrong sign or a truncating (not flooring) division."""
    g = json.load(open(os.path.join(GOLDEN, "ring_abs_pos.json")))
    for slot, want in g["slot_positions"].items():
        assert oracle.ring_abs_pos(int(slot), g["total_written"], g["buf_size"]) == want


def test_ring_abs_pos_unwritten_slots_negative():
    """Slots never written report a negative position (same section); a ring
    holds exactly the last `ring` positions written."""
    for ring in (1, 3, 8):
        for written in range(0, 3 * ring + 2):
            held = sorted(oracle.ring_abs_pos(j, written, ring) for j in range(ring))
            want = list(range(written - ring, written))
            assert held == want, (ring, written, held)


def _keyset_by_zero_query(kind, seq_len, q_rows, window, ring=None, D=16):
    """q = 0 makes every valid key weigh the same, so out = mean of the valid
    V rows.  V row of position t is the one-hot e_t, so out reveals the set."""
    B, Hq, Hkv = 1, 1, 1
    case = synth.decode_case(5, kind, B, q_rows, Hq, Hkv, D, [seq_len], window=window, ring=ring)
    # Overwrite values so that the V row at position t is e_t.
    k = torch.zeros_like(case.k_cache)
    v = torch.zeros_like(case.v_cache)
    kn = torch.zeros_like(case.k_new)
    vn = torch.zeros_like(case.v_new)
    # Fill history: write e_t at the slot holding position t, using the
    # caller's slot bookkeeping for every position 0..seq_len-1.
    all_pos = torch.arange(seq_len, dtype=torch.int32)
    if kind == synth.RING:
        slots = all_pos.to(torch.int64) % case.slots_per_seq
    elif kind == synth.LINEAR:
        slots = all_pos.to(torch.int64)
    else:
        bt = case.block_table[0].to(torch.int64)
        slots = bt[all_pos // case.block_size] * case.block_size + all_pos % case.block_size
    for t, s in zip(all_pos.tolist(), slots.tolist()):
        v[s] = 0
        v[s, 0, t % D] = 1.0
    for r in range(q_rows):
        t = int(case.positions[r])
        vn[r] = 0
        vn[r, 0, t % D] = 1.0
    case.k_cache, case.v_cache, case.k_new, case.v_new = k, v, kn, vn
    case.q = torch.zeros_like(case.q)
    rc, out, _, _ = run_case(case)
    assert rc == 0
    sets = []
    for r in range(q_rows):
        o = out[0, r, 0]
        n = round(1.0 / o.max())
        assert np.allclose(o[o > 0], 1.0 / n)
        sets.append(sorted(np.nonzero(o > 0)[0].tolist()))
    return case, sets


def test_ring_two_x_window_example():
    """The pages' reason for a 2x ring: window 4, 4 new rows at 5..8."""
    g = json.load(open(os.path.join(GOLDEN, "ring_two_x_window.json")))
    seq_len = g["start_pos"] + g["new_rows"]
    r = g["query_pos"] - g["start_pos"]
    _, s1 = _keyset_by_zero_query(synth.RING, seq_len, g["new_rows"], g["window"],
                                  ring=g["window"])
    _, s2 = _keyset_by_zero_query(synth.RING, seq_len, g["new_rows"], g["window"],
                                  ring=2 * g["window"])
    assert s1[r] == g["keys_1x"]
    assert s2[r] == g["keys_2x"]


@pytest.mark.parametrize("kind", [synth.LINEAR, synth.PAGED, synth.RING])
@pytest.mark.parametrize("window", [0, 1, 3, 5])
def test_zero_query_keyset(kind, window):
    """Catches off-by-one window bounds, a causal mask that lets a row see
    later rows of its own step, and ring slots read after being overwritten.
    The expected set is the pages' statement: the last `window` positions up
    to and including the row's own, among those the cache still holds."""
    D = 16
    for seq_len, q_rows in [(5, 1), (9, 3), (13, 4), (3, 3)]:
        ring = max(2 * window, window + q_rows - 1, 4) if kind == synth.RING else None
        if kind == synth.RING and window == 0:
            continue  # an unwindowed ring is the linear case
        case, sets = _keyset_by_zero_query(kind, seq_len, q_rows, window, ring=ring, D=D)
        for r in range(q_rows):
            pos = seq_len - q_rows + r
            lo = 0 if window <= 0 else pos - window + 1
            if kind == synth.RING:
                lo = max(lo, seq_len - ring)
            want = sorted({t % D for t in range(max(lo, 0), pos + 1)})
            assert sets[r] == want, (kind, window, seq_len, q_rows, r)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_single_key_returns_its_value():
    """A single valid key has weight exactly 1 (decode at 1 position)."""
    for kind in (synth.LINEAR, synth.PAGED):
        case = synth.decode_case(11, kind, 2, 1, 8, 2, 32, [1, 1])
        rc, out, kc, vc = run_case(case)
        assert rc == 0
        vn = f64(case.v_new)  # [B, Hkv, D]
        for b in range(2):
            for h in range(8):
                assert np.array_equal(out[b, 0, h], vn[b, h // 4])


def test_two_key_logistic_closed_form():
    """With two keys, weights are logistic(s1 - s0) with s = scale * q.k and a
    natural-base exponential.  Catches a missing scale, a base-2 exp, or a
    weight attached to the wrong key."""
    D = 8
    case = synth.decode_case(3, synth.LINEAR, 1, 1, 1, 1, D, [2], scale=0.37)
    q = torch.zeros_like(case.q)
    q[0, 0, 0, 0] = 1.5
    q[0, 0, 0, 1] = -0.5
    kc = torch.zeros_like(case.k_cache)
    kc[0, 0, 0] = 2.0   # key at position 0
    kc[0, 0, 1] = 1.0
    kn = torch.zeros_like(case.k_new)
    kn[0, 0, 0] = -1.0  # key at position 1 (the new row)
    kn[0, 0, 1] = 3.0
    case.q, case.k_cache, case.k_new = q, kc, kn
    rc, out, _, vc = run_case(case)
    assert rc == 0
    s0 = 0.37 * (1.5 * 2.0 - 0.5 * 1.0)
    s1 = 0.37 * (1.5 * -1.0 - 0.5 * 3.0)
    w1 = 1.0 / (1.0 + math.exp(-(s1 - s0)))
    v0 = f64(case.v_cache)[0, 0]
    v1 = f64(case.v_new)[0, 0]
    np.testing.assert_allclose(out[0, 0, 0], w1 * v1 + (1 - w1) * v0, rtol=1e-13, atol=1e-14)


def test_dominant_key_limit():
    """q aligned with one key and a large scale: out tends to that key's value."""
    D = 16
    case = synth.decode_case(4, synth.LINEAR, 1, 1, 1, 1, D, [6], scale=1.0)
    kc = torch.zeros_like(case.k_cache)
    for t in range(5):
        kc[t, 0, t] = 1.0
    q = torch.zeros_like(case.q)
    q[0, 0, 0, 2] = 60.0
    case.k_cache, case.q = kc, q
    case.k_new = torch.zeros_like(case.k_new)
    rc, out, _, _ = run_case(case)
    np.testing.assert_allclose(out[0, 0, 0], f64(case.v_cache)[2, 0], atol=1e-20, rtol=1e-20)


def test_softmax_weights_sum_to_one():
    for kind in (synth.LINEAR, synth.PAGED, synth.RING):
        case = synth.decode_case(21, kind, 2, 3, 4, 2, 16, [7, 12], window=5, ring=10)
        kc, vc = bits(case.k_cache).copy(), bits(case.v_cache).copy()
        oracle.kv_append(kc, vc, bits(case.k_new), bits(case.v_new), case.slot_mapping.numpy())
        cd = cache_dict(case) | {"k": kc, "v": vc}
        rc, out = oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(),
                                case.window, case.scale, case.n_kv_heads)
        assert rc == 0
        for b in range(2):
            for r in range(3):
                for h in range(4):
                    tp, w = oracle.decode_weights(bits(case.q), cd, case.seq_lens.numpy(),
                                                  case.positions.numpy(), case.window,
                                                  case.scale, 2, b, r, h)
                    assert abs(w.sum() - 1.0) < 1e-12
                    assert (w >= 0).all()
                    pos = int(case.positions[b * 3 + r])
                    masked = (tp < 0) | (tp > pos) | (pos - tp >= case.window)
                    assert (w[masked] == 0).all() and (w[~masked] > 0).all()


# --------------------------------------------------------------------------
# invariants the pages fix
# --------------------------------------------------------------------------

def test_gqa_equals_mha_with_replicated_kv():
    """GQA reads KV head h // G; with K/V heads replicated G times, MHA over the
    replicas must agree.  Catches h % Hkv in place of h // G."""
    case = synth.decode_case(31, synth.PAGED, 2, 2, 12, 2, 16, [9, 20])
    rc, out_gqa, kc, vc = run_case(case)
    assert rc == 0
    G = 6
    rep = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).repeat_interleave(G, 1)
    kc_m, vc_m = rep(kc), rep(vc)
    cd = cache_dict(case) | {"k": bits(kc_m), "v": bits(vc_m)}
    rc, out_mha = oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(),
                                0, case.scale, 12)
    assert rc == 0
    np.testing.assert_array_equal(out_gqa, out_mha)
    # and in prefill
    p = synth.prefill_case(32, 1, 11, 12, 2, 16)
    rc, o1 = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 0, p.scale)
    rc2, o2 = oracle.prefill(bits(p.q), bits(p.k.repeat_interleave(G, 2)),
                             bits(p.v.repeat_interleave(G, 2)), 0, p.scale)
    assert rc == rc2 == 0
    np.testing.assert_array_equal(o1, o2)


def test_window_at_least_sequence_is_full_causal():
    """Below the window length, windowed attention is full causal (Voxtral
    notes, 'Offline Encoder')."""
    p = synth.prefill_case(41, 2, 13, 4, 4, 8)
    _, full = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 0, p.scale)
    for w in (13, 14, 100):
        _, win = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), w, p.scale)
        np.testing.assert_array_equal(full, win)
    _, w12 = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 12, p.scale)
    assert not np.array_equal(full[:, 12], w12[:, 12])  # the last row loses key 0
    np.testing.assert_array_equal(full[:, :12], w12[:, :12])


def test_ring_past_wrap_equals_linear_last_window():
    """A ring past wrap holds the same keys as a linear cache of the last
    keys; with the window mask both give the same attention."""
    W, R, ring = 6, 2, 12
    for seq_len in (13, 20, 31, 37):
        rcase = synth.decode_case(51 + seq_len, synth.RING, 1, R, 4, 2, 16, [seq_len], window=W,
                                  ring=ring)
        rc, out_ring, kc, vc = run_case(rcase)
        assert rc == 0
        # linear cache holding positions 0..seq_len-1, filled from the ring
        # where the ring still holds them (others are masked anyway)
        lcase = synth.decode_case(7, synth.LINEAR, 1, R, 4, 2, 16, [seq_len], window=W,
                                  slots_per_seq=seq_len)
        lk = np.zeros_like(bits(lcase.k_cache))
        lv = np.zeros_like(lk)
        for t in range(max(0, seq_len - ring), seq_len):
            lk[t] = kc[t % ring]
            lv[t] = vc[t % ring]
        cd = {"kind": synth.LINEAR, "k": lk, "v": lv, "slots_per_seq": seq_len}
        rc, out_lin = oracle.decode(bits(rcase.q), cd, rcase.seq_lens.numpy(),
                                    rcase.positions.numpy(), W, rcase.scale, 2)
        assert rc == 0
        # the ring sums its keys in slot order, the linear cache in time
        # order: equal up to fp64 rounding
        np.testing.assert_allclose(out_ring, out_lin, rtol=1e-12, atol=1e-14)


def test_k_row_decode_equals_single_row_replays():
    """One K-row causal decode equals K one-row decodes where row k sees
    seq_len = its position + 1 (talker_multiframe, 'How a frame advances
    without the host').  Catches rows attending later rows of their step."""
    K = 4
    case = synth.decode_case(61, synth.PAGED, 3, K, 8, 2, 16, [5, 17, 33])
    rc, out, kc, vc = run_case(case)
    assert rc == 0
    cd = cache_dict(case) | {"k": kc, "v": vc}
    for r in range(K):
        q1 = bits(case.q)[:, r:r + 1].copy()
        pos = case.positions.numpy().reshape(3, K)[:, r].copy()
        rc, o1 = oracle.decode(q1, cd, pos + 1, pos, 0, case.scale, 2)
        assert rc == 0
        np.testing.assert_array_equal(out[:, r], o1[:, 0])


def test_shift_invariance_of_keys():
    """Adding one vector c to every key shifts each row's scores by q.c, which
    softmax ignores.  Integer-valued K and c keep bf16 exact."""
    g = torch.Generator().manual_seed(71)
    p = synth.prefill_case(71, 1, 10, 4, 2, 8)
    k = torch.randint(-3, 4, p.k.shape, generator=g).to(torch.bfloat16)
    c = torch.randint(-5, 6, (1, 1, 2, 8), generator=g).to(torch.bfloat16)
    _, o1 = oracle.prefill(bits(p.q), bits(k), bits(p.v), 0, p.scale)
    _, o2 = oracle.prefill(bits(p.q), bits(k + c), bits(p.v), 0, p.scale)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-12)


def test_paged_shuffled_table_equals_contiguous():
    """A shuffled page table with a partial last page equals a contiguous
    cache holding the same keys (vibevoice.c, 'Attention backends')."""
    case = synth.decode_case(81, synth.PAGED, 2, 2, 8, 4, 16, [37, 50], block_size=8,
                             num_blocks=20)
    rc, out_p, kc, vc = run_case(case)
    assert rc == 0
    S = 64
    lk = np.zeros((2 * S,) + kc.shape[1:], dtype=np.uint16)
    lv = np.zeros_like(lk)
    bt = case.block_table.numpy()
    for b, sl in enumerate(case.seq_lens.tolist()):
        for t in range(sl):
            s = bt[b, t // 8] * 8 + t % 8
            lk[b * S + t] = kc[s]
            lv[b * S + t] = vc[s]
    cd = {"kind": synth.LINEAR, "k": lk, "v": lv, "slots_per_seq": S}
    rc, out_l = oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(), 0,
                              case.scale, 4)
    assert rc == 0
    np.testing.assert_array_equal(out_p, out_l)


def test_prefill_row_equals_decode_row():
    """Prefill row i is decode of one row at position i over keys 0..i."""
    p = synth.prefill_case(91, 1, 12, 6, 2, 16)
    _, pre = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 5, p.scale)
    kc = bits(p.k)[0].copy()
    vc = bits(p.v)[0].copy()
    cd = {"kind": synth.LINEAR, "k": kc, "v": vc, "slots_per_seq": 12}
    for i in range(12):
        q1 = bits(p.q)[:, i:i + 1].copy()
        rc, d = oracle.decode(q1, cd, np.array([i + 1]), np.array([i]), 5, p.scale, 2)
        assert rc == 0
        np.testing.assert_array_equal(pre[0, i], d[0, 0])


def test_prefill_row_subset_matches_full():
    p = synth.prefill_case(92, 2, 20, 4, 1, 8)
    _, full = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 0, p.scale)
    rows = [0, 7, 19, 3]
    _, sub = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), 0, p.scale, rows=rows)
    np.testing.assert_array_equal(sub, full[:, rows])


# --------------------------------------------------------------------------
# brute force: a dense matrix formulation on tiny shapes
# --------------------------------------------------------------------------

def _dense_attention(Q, K, V, mask, scale):
    """Q [n, D], K/V [m, D], mask [n, m] bool: softmax(scale Q K^T + log mask) V."""
    from scipy.special import softmax

    S = scale * (Q @ K.T)
    S = np.where(mask, S, -np.inf)
    return softmax(S, axis=1) @ V


@pytest.mark.parametrize("D", [4, 8])
@pytest.mark.parametrize("window", [0, 3])
def test_brute_force_prefill(D, window):
    for B, T, Hq, Hkv in [(1, 1, 1, 1), (2, 5, 2, 1), (2, 9, 4, 2), (1, 7, 3, 3)]:
        p = synth.prefill_case(100 + T + D, B, T, Hq, Hkv, D, window=window)
        _, out = oracle.prefill(bits(p.q), bits(p.k), bits(p.v), window, p.scale)
        Q, K, V = f64(p.q), f64(p.k), f64(p.v)
        i = np.arange(T)[:, None]
        t = np.arange(T)[None, :]
        mask = (t <= i) & ((window <= 0) | (i - t < window))
        for b in range(B):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                want = _dense_attention(Q[b, :, h], K[b, :, g], V[b, :, g], mask, p.scale)
                np.testing.assert_allclose(out[b, :, h], want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind", [synth.LINEAR, synth.PAGED, synth.RING])
def test_brute_force_decode(kind):
    """Dense formulation: gather the keys a request's cache holds into a
    position-indexed matrix (ring: position t lives in ring slot t mod ring,
    the write rule), then mask by position."""
    D, Hq, Hkv, R, W = 8, 4, 2, 2, 4
    for seed, sl in [(1, [2, 9]), (2, [5, 3]), (3, [17, 25])]:
        ring = 6 if kind == synth.RING else None
        case = synth.decode_case(200 + seed, kind, 2, R, Hq, Hkv, D, sl,
                                 window=W if kind == synth.RING else 0, ring=ring, block_size=4)
        rc, out, kc, vc = run_case(case)
        assert rc == 0
        Kc, Vc = oracle.bf16_to_f64(kc), oracle.bf16_to_f64(vc)
        Q = f64(case.q)
        for b, seq_len in enumerate(sl):
            ts = np.arange(seq_len)
            if kind == synth.LINEAR:
                slots = b * case.slots_per_seq + ts
            elif kind == synth.PAGED:
                bt = case.block_table.numpy()[b]
                slots = bt[ts // 4] * 4 + ts % 4
            else:
                slots = b * ring + ts % ring
            held = ts >= (seq_len - ring if kind == synth.RING else 0)
            for r in range(R):
                pos = seq_len - R + r
                w = W if kind == synth.RING else 0
                mask = held & (ts <= pos) & ((w <= 0) | (pos - ts < w))
                for h in range(Hq):
                    g = h // (Hq // Hkv)
                    want = _dense_attention(Q[b, r, h][None], Kc[slots, g], Vc[slots, g],
                                            mask[None], case.scale)[0]
                    np.testing.assert_allclose(out[b, r, h], want, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# append semantics and error reporting
# --------------------------------------------------------------------------

def test_append_copies_bits_last_row_wins_and_skips_out_of_range():
    kc = np.zeros((6, 2, 4), dtype=np.uint16)
    vc = np.zeros_like(kc)
    kn = np.arange(4 * 8, dtype=np.uint16).reshape(4, 2, 4) + 1
    vn = kn + 1000
    skipped = oracle.kv_append(kc, vc, kn, vn, np.array([5, 1, 5, 6]))
    assert skipped == 1
    np.testing.assert_array_equal(kc[1], kn[1])
    np.testing.assert_array_equal(kc[5], kn[2])  # later row wins
    np.testing.assert_array_equal(vc[5], vn[2])
    assert (kc[[0, 2, 3, 4]] == 0).all()


def test_empty_keyset_is_reported():
    """A row whose position lies beyond the keys written has nothing to attend."""
    case = synth.decode_case(9, synth.LINEAR, 1, 1, 2, 1, 8, [4])
    cd = cache_dict(case)
    rc, out = oracle.decode(bits(case.q), cd, np.array([4]), np.array([4 + 10]), 3, case.scale, 1)
    assert rc == oracle.EMPTY_KEYSET
    assert np.isnan(out).all()


def test_slot_bookkeeping_matches_oracle_positions():
    """The caller's reserved slots (synth) hold, by the oracle's ring formula,
    the positions of the rows written there."""
    case = synth.decode_case(13, synth.RING, 3, 4, 4, 2, 8, [9, 30, 77], window=6, ring=10)
    for i, s in enumerate(case.slot_mapping.tolist()):
        b, j = divmod(s, 10)
        pos = int(case.positions[i])
        assert oracle.ring_abs_pos(j, int(case.seq_lens[b]), 10) == pos


# ---------------------------------------------------------------- RoPE (fused append)

def _bf16_of(values):
    """float values -> bf16 bits by round-to-nearest-even of their float32."""
    f = np.asarray(values, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def test_rope_position_zero_is_identity():
    g = np.random.default_rng(31)
    x = _bf16_of(g.standard_normal((5, 3, 16)))
    inv = (10000.0 ** (-np.arange(8) / 8)).astype(np.float32)
    assert np.array_equal(oracle.rope(x, np.zeros(5), inv), x)


def test_rope_quarter_turn_swaps_the_pair():
    """An angle of pi/2 maps (x0, x1) to (-x1, x0) (float32 pi/2 is off by
    4e-8, far below a bf16 step)."""
    g = np.random.default_rng(32)
    x = _bf16_of(g.standard_normal((4, 2, 8)))
    inv = np.full(4, np.float32(np.pi / 2), dtype=np.float32)
    out = oracle.rope(x, np.ones(4), inv).view(np.int16).astype(np.int32)
    xi = x.view(np.int16).astype(np.int32)
    neg = lambda b: (b ^ -0x8000)  # flip the bf16 sign bit
    assert np.array_equal(out[..., 0::2], neg(xi[..., 1::2]))
    assert np.array_equal(out[..., 1::2], xi[..., 0::2])


def test_rope_hand_value():
    """(1, 0) at position 1 with inv_freq 1 is (cos 1, sin 1), rounded to bf16."""
    x = _bf16_of([[[1.0, 0.0]]])
    out = oracle.rope(x, [1], np.ones(1, dtype=np.float32))
    assert np.array_equal(out.reshape(-1), _bf16_of([np.cos(1.0), np.sin(1.0)]))


def test_rope_preserves_pair_norms():
    g = np.random.default_rng(33)
    x = _bf16_of(g.standard_normal((6, 4, 32)))
    inv = (10000.0 ** (-np.arange(16) / 16)).astype(np.float32)
    pos = g.integers(0, 40000, size=6)
    y = oracle.bf16_to_f64(oracle.rope(x, pos, inv))
    x64 = oracle.bf16_to_f64(x)
    nx = np.hypot(x64[..., 0::2], x64[..., 1::2])
    ny = np.hypot(y[..., 0::2], y[..., 1::2])
    assert np.all(np.abs(ny - nx) <= 2.0 ** -7 * nx + 1e-30)


def test_rope_scores_depend_on_relative_position():
    """With power-of-two frequencies the float32 angles are exact, and
    <rope(q, m), rope(k, n)> depends on m - n only (up to the bf16 rounding of
    the rotated rows)."""
    g = np.random.default_rng(34)
    q = _bf16_of(g.standard_normal((1, 1, 64)))
    k = _bf16_of(g.standard_normal((1, 1, 64)))
    inv = (2.0 ** -np.arange(32)).astype(np.float32)
    dots = []
    for shift in (0, 7, 1000):
        qr = oracle.bf16_to_f64(oracle.rope(q, [50 + shift], inv))
        kr = oracle.bf16_to_f64(oracle.rope(k, [20 + shift], inv))
        dots.append(float((qr * kr).sum()))
    scale = float(np.linalg.norm(oracle.bf16_to_f64(q)) * np.linalg.norm(oracle.bf16_to_f64(k)))
    assert max(dots) - min(dots) <= 2.0 ** -6 * scale
