"""Head-major caches (ATTN_LAYOUT_BHSD: the Voxtral notes' CUDA layout
[B, H, S, D], "KV cache"; pages as [page, H, rows, D]) against the oracle.

The oracle reads slot-major arrays; these tests build every case slot-major,
permute the cache into the head-major placement for the library (a pure
reordering of elements), and permute the library's cache back to compare the
append bit for bit.  Slot numbers, slot_mapping and block tables are the same
in both layouts.
"""
import numpy as np
import pytest
import torch

import oracle
import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import bits, compare, oracle_decode

pytestmark = pytest.mark.gpu

LINEAR, PAGED, RING = synth.LINEAR, synth.PAGED, synth.RING
BHSD = gq.ATTN_LAYOUT_BHSD
DEV = "cuda"


def rows_of(case):
    return case.block_size if case.kind == PAGED else case.slots_per_seq


def to_bhsd(t, rows):
    S, H, D = t.shape
    return t.reshape(S // rows, rows, H, D).permute(0, 2, 1, 3).contiguous()


def from_bhsd(t):
    nb, H, rows, D = t.shape
    return t.permute(0, 2, 1, 3).reshape(nb * rows, H, D)


def device_cache(case, k, v, **kw):
    r = rows_of(case)
    return gq.KVCache(case.kind, to_bhsd(k, r).to(DEV), to_bhsd(v, r).to(DEV),
                      slots_per_seq=case.slots_per_seq,
                      block_table=None if case.block_table is None else case.block_table.to(DEV),
                      block_size=case.block_size, layout=BHSD, **kw)


def run_bhsd(case, fused=False):
    cache = device_cache(case, case.k_cache, case.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (case.seq_lens.to(DEV), case.positions.to(DEV), case.max_seq_len(), case.window,
            case.scale)
    if fused:
        out = gq.attn_decode_append(case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV),
                                    case.slot_mapping.to(DEV), cache, *args, err=err)
    else:
        gq.attn_kv_append(case.k_new.to(DEV), case.v_new.to(DEV), case.slot_mapping.to(DEV),
                          cache, err=err)
        out = gq.attn_decode(case.q.to(DEV), cache, *args, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item())}"
    return out, cache


def check(case, where, fused=False):
    ref, kc, vc = oracle_decode(case)
    out, cache = run_bhsd(case, fused)
    assert np.array_equal(bits(from_bhsd(cache.k)), kc), f"{where}: K after the append"
    assert np.array_equal(bits(from_bhsd(cache.v)), vc), f"{where}: V after the append"
    compare(out, ref, where)


@pytest.mark.parametrize("seq", [[1, 16], [63, 64], [65, 1000], [4097, 3000]])
@pytest.mark.parametrize("heads", [(32, 8), (28, 4)])
def test_bhsd_linear(seq, heads):
    Hq, Hkv = heads
    case = synth.decode_case(11000 + seq[0] + Hq, LINEAR, 2, 1, Hq, Hkv, 128, seq)
    check(case, f"bhsd linear {seq} {Hq}/{Hkv}")


def test_bhsd_linear_block_not_a_multiple_of_16():
    """Per-request capacity 1,000: the last chunk of a request's block ends
    inside a 16-row box, so it is gathered row by row."""
    case = synth.decode_case(11100, LINEAR, 3, 2, 16, 4, 128, [1000, 999, 510],
                             slots_per_seq=1000)
    check(case, "bhsd linear capacity 1000")


@pytest.mark.parametrize("block_size", [16, 64, 5, 24])
@pytest.mark.parametrize("R", [1, 4])
def test_bhsd_paged(block_size, R):
    """16: one box per page; 64: whole 64-row tiles inside a page; 5, 24:
    gathered rows."""
    case = synth.decode_case(11200 + block_size + R, PAGED, 4, R, 32, 8, 128,
                             [37, 300, 1029, max(R, 4)], block_size=block_size)
    check(case, f"bhsd paged bs={block_size} R={R}")


@pytest.mark.parametrize("ring,window,R", [(64, 32, 1), (100, 37, 2), (1500, 750, 4),
                                           (16384, 8192, 1)])
def test_bhsd_ring(ring, window, R):
    g = torch.Generator().manual_seed(ring + R)
    seq = torch.randint(window, 3 * ring + 50, (5,), generator=g).tolist()
    seq[0] = R
    seq[1] = ring + 3
    case = synth.decode_case(11300 + ring + R, RING, 5, R, 16, 4, 128, seq, window=window,
                             ring=ring)
    check(case, f"bhsd ring {ring}/{window} R={R}")


@pytest.mark.parametrize("R,Hq,Hkv", [(8, 32, 4), (4, 28, 4), (2, 7, 1)])
def test_bhsd_row_tilings(R, Hq, Hkv):
    case = synth.decode_case(11400 + R * Hq, PAGED, 5, R, Hq, Hkv, 128,
                             [64, 100, max(R, 4), 1030, 517], block_size=16)
    check(case, f"bhsd paged R={R} {Hq}/{Hkv}")


def test_bhsd_head_dim_64():
    case = synth.streaming_encoder_step(batch=2)
    check(case, "bhsd streaming encoder D=64")


@pytest.mark.parametrize("kind", [LINEAR, PAGED, RING])
def test_bhsd_fused_append(kind):
    extra = {"block_size": 16} if kind == PAGED else (
        {"window": 750, "ring": 1500} if kind == RING else {})
    case = synth.decode_case(11500 + int(kind), kind, 3, 4, 32, 8, 128, [2000, 37, 1503], **extra)
    check(case, f"bhsd fused {kind}", fused=True)


def test_bhsd_fp8():
    """An FP8 cache in the head-major layout: codes placed by the library's
    append equal the oracle's, and decode matches the oracle over them."""
    case = synth.decode_case(11600, PAGED, 4, 1, 28, 4, 128, [3000, 64, 1029, 17],
                             block_size=16)
    S, Hkv, D = case.k_cache.shape
    kc = np.zeros((S, Hkv, D), dtype=np.uint8)
    vc = np.zeros((S, Hkv, D), dtype=np.uint8)
    oracle.kv_append_fp8(kc, vc, bits(case.k_cache), bits(case.v_cache), np.arange(S))
    want_k, want_v = kc.copy(), vc.copy()
    oracle.kv_append_fp8(want_k, want_v, bits(case.k_new), bits(case.v_new),
                         case.slot_mapping.numpy())
    cache = device_cache(case, torch.from_numpy(kc), torch.from_numpy(vc),
                         dtype=gq.ATTN_KV_FP8_E4M3)
    gq.attn_kv_append(case.k_new.to(DEV), case.v_new.to(DEV), case.slot_mapping.to(DEV), cache)
    out = gq.attn_decode(case.q.to(DEV), cache, case.seq_lens.to(DEV), case.positions.to(DEV),
                         case.max_seq_len(), 0, case.scale)
    torch.cuda.synchronize()
    assert np.array_equal(from_bhsd(cache.k).cpu().numpy(), want_k)
    assert np.array_equal(from_bhsd(cache.v).cpu().numpy(), want_v)
    cd = {"kind": PAGED, "k": oracle.fp8_to_bf16_bits(want_k), "v": oracle.fp8_to_bf16_bits(want_v),
          "block_table": case.block_table.numpy(), "block_size": 16}
    rc, ref = oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(), 0,
                            case.scale, Hkv)
    assert rc == 0
    compare(out, ref, "bhsd fp8 paged")


def test_bhsd_same_result_as_slot_major():
    """The layout moves bytes only: the same case gives bit-identical outputs
    in both layouts (same kernel, same order of arithmetic)."""
    from helpers import gpu_decode

    case = synth.decode_case(11700, LINEAR, 2, 4, 32, 8, 128, [5000, 129])
    a, _ = gpu_decode(case)
    b, _ = run_bhsd(case)
    assert torch.equal(a, b)


def test_bhsd_fused_append_with_rope():
    """Head-major cache, the step's rows rotated and appended by the decode
    launch: the same cache bits and output bits as the slot-major launch
    (the layout moves bytes only)."""
    from helpers import to_device

    case = synth.decode_case(11800, PAGED, 3, 4, 32, 8, 128, [2000, 37, 1503], block_size=16)
    inv = (10000.0 ** (-torch.arange(0, 64, dtype=torch.float32) / 64)).to(DEV)
    args = (case.seq_lens.to(DEV), case.positions.to(DEV), case.max_seq_len(), 0, case.scale)
    slot_major = to_device(case, DEV)
    a = gq.attn_decode_append(case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV),
                              case.slot_mapping.to(DEV), slot_major, *args, rope_inv_freq=inv)
    head_major = device_cache(case, case.k_cache, case.v_cache)
    b = gq.attn_decode_append(case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV),
                              case.slot_mapping.to(DEV), head_major, *args, rope_inv_freq=inv)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(from_bhsd(head_major.k).cpu(), slot_major.k.cpu())
    assert torch.equal(from_bhsd(head_major.v).cpu(), slot_major.v.cpu())


def test_bhsd_fp8_fused_append():
    case = synth.decode_case(11900, LINEAR, 3, 2, 28, 4, 128, [3000, 64, 1029])
    S, Hkv, D = case.k_cache.shape
    kc = np.zeros((S, Hkv, D), dtype=np.uint8)
    vc = np.zeros((S, Hkv, D), dtype=np.uint8)
    oracle.kv_append_fp8(kc, vc, bits(case.k_cache), bits(case.v_cache), np.arange(S))
    want_k, want_v = kc.copy(), vc.copy()
    oracle.kv_append_fp8(want_k, want_v, bits(case.k_new), bits(case.v_new),
                         case.slot_mapping.numpy())
    cache = device_cache(case, torch.from_numpy(kc), torch.from_numpy(vc),
                         dtype=gq.ATTN_KV_FP8_E4M3)
    out = gq.attn_decode_append(case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV),
                                case.slot_mapping.to(DEV), cache, case.seq_lens.to(DEV),
                                case.positions.to(DEV), case.max_seq_len(), 0, case.scale)
    torch.cuda.synchronize()
    assert np.array_equal(from_bhsd(cache.k).cpu().numpy(), want_k)
    assert np.array_equal(from_bhsd(cache.v).cpu().numpy(), want_v)
    cd = {"kind": LINEAR, "k": oracle.fp8_to_bf16_bits(want_k), "v": oracle.fp8_to_bf16_bits(want_v),
          "slots_per_seq": case.slots_per_seq}
    rc, ref = oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(), 0,
                            case.scale, Hkv)
    assert rc == 0
    compare(out, ref, "bhsd fp8 fused")
