"""FP8 (E4M3) KV cache on the GPU against the oracle (vibevoice.c, "KV cache":
the cache stored as 8-bit floats, K relative to a per-layer reference vector
built from the first prefill chunk).

Append is compared bit for bit with the oracle's FP8 append (the rounding of
float32(k) - ref to E4M3 is taken in the same precision on both sides).
Decode is compared with the fp64 oracle run over the dequantized cache (every
E4M3 value is exact in bf16, so the oracle reads exactly what is stored), at
the tolerance of the bf16 path.
"""
import numpy as np
import pytest
import torch

import oracle
import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import bits, compare

pytestmark = pytest.mark.gpu

LINEAR, PAGED, RING = synth.LINEAR, synth.PAGED, synth.RING
FP8 = gq.ATTN_KV_FP8_E4M3
DEV = "cuda"


def fp8_codes(k, v, ref=None):
    """The oracle's FP8 append of every row of bf16 caches [S, Hkv, D]."""
    S, Hkv, D = k.shape
    kc = np.zeros((S, Hkv, D), dtype=np.uint8)
    vc = np.zeros((S, Hkv, D), dtype=np.uint8)
    oracle.kv_append_fp8(kc, vc, bits(k), bits(v), np.arange(S), k_ref=ref)
    return kc, vc


def oracle_fp8_step(case, kc, vc, ref=None):
    """Oracle: FP8 append of the step's rows, then decode over the values stored."""
    kc, vc = kc.copy(), vc.copy()
    oracle.kv_append_fp8(kc, vc, bits(case.k_new), bits(case.v_new),
                         case.slot_mapping.cpu().numpy(), k_ref=ref)
    cd = {"kind": case.kind, "k": oracle.fp8_to_bf16_bits(kc), "v": oracle.fp8_to_bf16_bits(vc),
          "slots_per_seq": case.slots_per_seq,
          "block_table": None if case.block_table is None else case.block_table.cpu().numpy(),
          "block_size": case.block_size}
    rc, out = oracle.decode(bits(case.q), cd, case.seq_lens.cpu().numpy(),
                            case.positions.cpu().numpy(), case.window, case.scale,
                            case.n_kv_heads)
    assert rc == 0
    return out, kc, vc


def gpu_fp8_step(case, kc, vc, ref=None, max_seq_len=None):
    cache = gq.KVCache(case.kind, torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
                       slots_per_seq=case.slots_per_seq,
                       block_table=None if case.block_table is None else case.block_table.to(DEV),
                       block_size=case.block_size, dtype=FP8,
                       k_ref=None if ref is None else torch.from_numpy(ref).to(DEV))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gq.attn_kv_append(case.k_new.to(DEV), case.v_new.to(DEV), case.slot_mapping.to(DEV), cache,
                      err=err)
    out = gq.attn_decode(case.q.to(DEV), cache, case.seq_lens.to(DEV), case.positions.to(DEV),
                         max_seq_len or case.max_seq_len(), case.window, case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item())}"
    return out, cache


def check_case(case, ref=None, where=""):
    kc, vc = fp8_codes(case.k_cache, case.v_cache, ref)
    want, kc2, vc2 = oracle_fp8_step(case, kc, vc, ref)
    out, cache = gpu_fp8_step(case, kc, vc, ref)
    assert np.array_equal(cache.k.cpu().numpy(), kc2), f"{where}: K codes after the append"
    assert np.array_equal(cache.v.cpu().numpy(), vc2), f"{where}: V codes after the append"
    compare(out, want, where)
    return out


# ---------------------------------------------------------------- append
@pytest.mark.parametrize("with_ref", [False, True])
@pytest.mark.parametrize("Hkv,n", [(8, 256), (4, 14449), (1, 1), (28, 3)])
def test_fp8_append_bit_exact(Hkv, n, with_ref):
    """Magnitudes from 1e-5 to 1e4: subnormal codes, every binade, and
    saturation at 448."""
    g = synth.generator(8100 + Hkv + n)
    D = 128
    S = max(2 * n, 64)
    scale = torch.pow(10.0, torch.empty(n, Hkv, D).uniform_(-5, 4, generator=g))
    k_new = (torch.randn(n, Hkv, D, generator=g) * scale).to(torch.bfloat16)
    v_new = (torch.randn(n, Hkv, D, generator=g) * scale.flip(0)).to(torch.bfloat16)
    ref = (np.random.default_rng(n).standard_normal((Hkv, D)) * 20).astype(np.float32) \
        if with_ref else None
    slots = torch.randperm(S, generator=g)[:n]
    kc = np.full((S, Hkv, D), 0x33, dtype=np.uint8)
    vc = np.full((S, Hkv, D), 0x33, dtype=np.uint8)
    kc_dev, vc_dev = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    oracle.kv_append_fp8(kc, vc, bits(k_new), bits(v_new), slots.numpy(), k_ref=ref)
    cache = gq.KVCache(LINEAR, kc_dev, vc_dev, slots_per_seq=S, dtype=FP8,
                       k_ref=None if ref is None else torch.from_numpy(ref).to(DEV))
    gq.attn_kv_append(k_new.to(DEV), v_new.to(DEV), slots.to(DEV), cache)
    torch.cuda.synchronize()
    assert np.array_equal(kc_dev.cpu().numpy(), kc)
    assert np.array_equal(vc_dev.cpu().numpy(), vc)


def test_fp8_append_special_values():
    """Zeros of both signs, infinities (saturate to +-448), NaN, the largest
    finite bf16, and values halfway between two codes."""
    D, Hkv = 128, 1
    vals = [0.0, -0.0, float("inf"), float("-inf"), float("nan"), 3.3895e38, -3.3895e38,
            2.0 ** -10, 3 * 2.0 ** -10, 1 + 1 / 16, 1 + 3 / 16, 432.0, 464.0, -2.0 ** -11,
            2.0 ** -6, 2.0 ** -9, 240.0, 0.1, -0.1]
    row = torch.tensor(vals + [1.0] * (D - len(vals)), dtype=torch.float32)
    k_new = row.view(1, Hkv, D).to(torch.bfloat16)
    kc = np.zeros((4, Hkv, D), dtype=np.uint8)
    vc = np.zeros((4, Hkv, D), dtype=np.uint8)
    kc_dev, vc_dev = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    oracle.kv_append_fp8(kc, vc, bits(k_new), bits(k_new), np.array([2]))
    cache = gq.KVCache(LINEAR, kc_dev, vc_dev, slots_per_seq=4, dtype=FP8)
    gq.attn_kv_append(k_new.to(DEV), k_new.to(DEV), torch.tensor([2], device=DEV), cache)
    torch.cuda.synchronize()
    got = kc_dev.cpu().numpy()
    assert np.array_equal(got, kc), [(v, hex(a), hex(b)) for v, a, b in
                                     zip(vals, got[2, 0], kc[2, 0]) if a != b]
    assert np.array_equal(vc_dev.cpu().numpy(), vc)


def test_fp8_append_out_of_range_slot_is_reported():
    kc = torch.zeros(8, 2, 128, dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    cache = gq.KVCache(LINEAR, kc, vc, slots_per_seq=8, dtype=FP8)
    kn = torch.ones(3, 2, 128, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gq.attn_kv_append(kn, kn, torch.tensor([5, 8, -1], device=DEV), cache, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gq.ATTN_ERR_BOUNDS
    assert (kc[5] == 0x38).all() and int(kc.sum()) == 0x38 * 256  # only row 0 landed


# ---------------------------------------------------------------- reference
@pytest.mark.parametrize("n,Hkv", [(1, 4), (29, 8), (14449, 4)])
def test_kv_reference_matches_oracle_mean(n, Hkv):
    g = synth.generator(8200 + n)
    k = (synth.normal_bf16(g, (n, Hkv, 128)).float() * 3 + 20).to(torch.bfloat16)
    want = oracle.kv_reference(bits(k))
    got = gq.attn_kv_reference(k.to(DEV)).cpu().numpy().astype(np.float64)
    # an fp64 sum in another order, rounded once to float32: within one float32 step
    assert (np.abs(got - want) <= np.spacing(np.abs(want).astype(np.float32))).all()
    again = gq.attn_kv_reference(k.to(DEV)).cpu().numpy()
    assert np.array_equal(again, got.astype(np.float32)), "run-to-run results differ"


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("seq_len", [1, 15, 16, 17, 63, 64, 65, 1025, 4097])
@pytest.mark.parametrize("heads", [(32, 8), (28, 4), (12, 2)])
def test_fp8_linear_positions(seq_len, heads):
    Hq, Hkv = heads
    case = synth.decode_case(8300 + seq_len, LINEAR, 2, 1, Hq, Hkv, 128,
                             [seq_len, max(1, seq_len // 2)])
    check_case(case, where=f"fp8 linear L={seq_len} {Hq}/{Hkv}")


@pytest.mark.parametrize("R,Hq,Hkv", [(4, 32, 8), (3, 12, 2), (8, 32, 4), (2, 7, 1),
                                       (4, 16, 16)])
def test_fp8_multirow_paged(R, Hq, Hkv):
    """rows x group of 8 or fewer, 16 and 32: the three tilings of the query rows."""
    case = synth.decode_case(8400 + R * Hq, PAGED, 5, R, Hq, Hkv, 128,
                             [64, 100, max(R, 4), 1030, 517], block_size=16)
    check_case(case, where=f"fp8 paged R={R} {Hq}/{Hkv}")


@pytest.mark.parametrize("block_size", [16, 32, 5, 24])
def test_fp8_paged_block_sizes(block_size):
    case = synth.decode_case(8500 + block_size, PAGED, 3, 2, 16, 4, 128, [37, 300, 129],
                             block_size=block_size, num_blocks=200)
    check_case(case, where=f"fp8 paged bs={block_size}")


@pytest.mark.parametrize("ring,window,R", [(64, 32, 1), (100, 37, 2), (1500, 750, 4),
                                           (16384, 8192, 1)])
def test_fp8_ring(ring, window, R):
    g = torch.Generator().manual_seed(ring + window + R)
    seq = torch.randint(window, 3 * ring + 50, (6,), generator=g).tolist()
    seq[0] = R
    seq[1] = ring + 3
    case = synth.decode_case(8600 + ring + R, RING, 6, R, 16, 4, 128, seq, window=window,
                             ring=ring)
    check_case(case, where=f"fp8 ring {ring}/{window} R={R}")


@pytest.mark.parametrize("window", [1, 100, 1000])
def test_fp8_linear_window(window):
    case = synth.decode_case(8700 + window, LINEAR, 3, 4, 32, 8, 128, [2000, 5, 700],
                             window=window)
    check_case(case, where=f"fp8 linear window={window}")


def test_fp8_long_context_and_determinism():
    """Qwen2-7B heads (28 / 4) at a long context: a unit spans many CTAs and
    the merge of their partial states runs; two runs give the same bits."""
    case = synth.decode_case(8800, LINEAR, 2, 1, 28, 4, 128, [14449, 23971])
    kc, vc = fp8_codes(case.k_cache, case.v_cache)
    want, _, _ = oracle_fp8_step(case, kc, vc)
    a, _ = gpu_fp8_step(case, kc, vc)
    b, _ = gpu_fp8_step(case, kc, vc)
    assert torch.equal(a, b), "run-to-run results differ"
    compare(a, want, "fp8 qwen 14449 / 23971")


def test_fp8_with_reference_and_shift_property():
    """Keys with a large common component (the page's Qwen2 observation): the
    library builds the reference from the first chunk, stores K relative to
    it, and decodes.  The output matches the oracle over the stored values,
    and stays close to bf16 attention over the original keys."""
    g = synth.generator(8900)
    Hq, Hkv, D, seq = 28, 4, 128, 2048
    case = synth.decode_case(8901, LINEAR, 1, 1, Hq, Hkv, D, [seq])
    common = synth.normal_bf16(g, (1, Hkv, D)).float() * (273 / D ** 0.5)
    case.k_cache = (case.k_cache.float() + common).to(torch.bfloat16)
    case.k_new = (case.k_new.float() + common).to(torch.bfloat16)
    ref = gq.attn_kv_reference(case.k_cache[:512].to(DEV)).cpu().numpy()
    out = check_case(case, ref=ref, where="fp8 with reference")
    from helpers import oracle_decode

    exact, _, _ = oracle_decode(case)
    got = out.float().cpu().numpy().reshape(-1).astype(np.float64)
    e = exact.reshape(-1)
    cos = float(got @ e / np.linalg.norm(got) / np.linalg.norm(e))
    assert cos > 0.995, cos


def test_fp8_noalloc_entry_point():
    case = synth.decode_case(9000, PAGED, 4, 4, 32, 8, 128, [300, 17, 1000, 64], block_size=16)
    kc, vc = fp8_codes(case.k_cache, case.v_cache)
    want, kc2, vc2 = oracle_fp8_step(case, kc, vc)
    cache = gq.KVCache(PAGED, torch.from_numpy(kc2).to(DEV), torch.from_numpy(vc2).to(DEV),
                       block_table=case.block_table.to(DEV), block_size=16, dtype=FP8)
    out = gq.attn_decode_noalloc(case.q.to(DEV), cache, case.seq_lens.to(DEV),
                                 case.positions.to(DEV), case.max_seq_len(), 0, case.scale)
    torch.cuda.synchronize()
    compare(out, want, "fp8 noalloc")


def test_fp8_batch_split_over_launches():
    g = torch.Generator().manual_seed(9100)
    seq = torch.randint(1, 200, (300,), generator=g).tolist()
    case = synth.decode_case(9101, LINEAR, 300, 1, 8, 2, 128, seq)
    check_case(case, where="fp8 batch 300")


def test_fp8_one_unit_over_many_ctas():
    case = synth.decode_case(9102, LINEAR, 1, 1, 8, 1, 128, [16000])
    check_case(case, where="fp8 one unit, 16000 keys")


@pytest.mark.parametrize("kind,B,R,Hq,Hkv,seq,extra", [
    (LINEAR, 3, 1, 28, 4, [513, 1, 4097], {}),
    (PAGED, 4, 4, 32, 8, [64, 100, 1030, 17], {"block_size": 16}),
    (PAGED, 3, 2, 16, 4, [37, 300, 129], {"block_size": 5, "num_blocks": 200}),
    (RING, 4, 1, 32, 8, [9000, 300, 16390, 8193], {"window": 8192, "ring": 16384}),
])
@pytest.mark.parametrize("with_ref", [False, True])
def test_fp8_fused_append_equals_append_then_decode(kind, B, R, Hq, Hkv, seq, extra, with_ref):
    """attn_decode_append over an FP8 cache encodes the step's rows on the way
    into the decode and into the cache: same codes and same output bits as
    the FP8 append followed by the decode, and the oracle's result."""
    case = synth.decode_case(9200 + B * R + int(kind), kind, B, R, Hq, Hkv, 128, seq, **extra)
    ref = (np.random.default_rng(B).standard_normal((Hkv, 128)) * 3).astype(np.float32) \
        if with_ref else None
    kc, vc = fp8_codes(case.k_cache, case.v_cache, ref)
    want, kc2, vc2 = oracle_fp8_step(case, kc, vc, ref)
    out_u, cache_u = gpu_fp8_step(case, kc, vc, ref)
    cache = gq.KVCache(case.kind, torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
                       slots_per_seq=case.slots_per_seq,
                       block_table=None if case.block_table is None else case.block_table.to(DEV),
                       block_size=case.block_size, dtype=FP8,
                       k_ref=None if ref is None else torch.from_numpy(ref).to(DEV))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_f = gq.attn_decode_append(case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV),
                                  case.slot_mapping.to(DEV), cache, case.seq_lens.to(DEV),
                                  case.positions.to(DEV), case.max_seq_len(), case.window,
                                  case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(cache.k.cpu().numpy(), kc2) and np.array_equal(cache.v.cpu().numpy(), vc2)
    assert torch.equal(out_f, out_u), "fused and two-launch FP8 results differ"
    compare(out_f, want, f"fp8 fused {kind}")


def test_fp8_fused_append_refuses_rope():
    case = synth.decode_case(9300, LINEAR, 1, 1, 8, 2, 128, [40])
    kc, vc = fp8_codes(case.k_cache, case.v_cache)
    cache = gq.KVCache(LINEAR, torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
                       slots_per_seq=case.slots_per_seq, dtype=FP8)
    inv = torch.ones(64, dtype=torch.float32, device=DEV)
    with pytest.raises(gq.AttnError) as e:
        gq.attn_decode_append(case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV),
                              case.slot_mapping.to(DEV), cache, case.seq_lens.to(DEV),
                              case.positions.to(DEV), 40, 0, case.scale, rope_inv_freq=inv)
    assert e.value.status == gq.ATTN_ERR_UNSUPPORTED
