"""Decode parity: the library (append + split-KV decode) against the fp64 oracle.

Shapes follow the pages' test list (vibevoice.c, "Attention backends"):
decode at 1, 1023, 1024, 1025, 4097, 16385 and 32767 positions, GQA 28/4 and
12/2, a paged cache with a shuffled table and a partial last page, K-row
decode (talker_multiframe), and ring buffers past their wrap point (Voxtral
notes, "Encoder KV cache").
"""
import numpy as np
import pytest
import torch

import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import compare, gpu_decode, oracle_decode, to_device

pytestmark = pytest.mark.gpu

LINEAR, PAGED, RING = synth.LINEAR, synth.PAGED, synth.RING


@pytest.mark.parametrize("seq_len", [1, 2, 15, 16, 17, 63, 64, 65, 1023, 1024, 1025, 4097])
@pytest.mark.parametrize("heads", [(32, 8), (28, 4), (12, 2)])
def test_linear_positions(seq_len, heads):
    Hq, Hkv = heads
    case = synth.decode_case(1000 + seq_len, LINEAR, 2, 1, Hq, Hkv, 128,
                             [seq_len, max(1, seq_len // 2)])
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"linear L={seq_len} {Hq}/{Hkv}")


@pytest.mark.parametrize("seq_len", [16385, 32767])
def test_linear_long(seq_len):
    case = synth.decode_case(2000 + seq_len, LINEAR, 1, 1, 28, 4, 128, [seq_len])
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"linear L={seq_len}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("block_size", [16, 32, 64, 5, 8, 24])
def test_paged_block_sizes(D, block_size):
    """block sizes that are multiples of 16 go through TMA boxes; the others
    are gathered row by row."""
    case = synth.decode_case(3000 + block_size + D, PAGED, 3, 2, 16, 4, D, [37, 300, 129],
                             block_size=block_size, num_blocks=200)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"paged bs={block_size} D={D}")


@pytest.mark.parametrize("R,Hq,Hkv", [(4, 32, 8), (4, 28, 4), (3, 12, 2), (8, 32, 4),
                                       (4, 16, 16), (2, 7, 1)])
def test_multirow_paged(R, Hq, Hkv):
    """K sequential query rows causal among themselves; rows x group spans
    one 16-row tile, two, or several row blocks."""
    case = synth.decode_case(4000 + R * Hq, PAGED, 5, R, Hq, Hkv, 128, [64, 100, max(R, 4), 1030, 517],
                             block_size=16)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"paged R={R} {Hq}/{Hkv}")


@pytest.mark.parametrize("ring,window,R", [(64, 32, 1), (48, 32, 4), (1500, 750, 4),
                                           (100, 37, 2), (16384, 8192, 1)])
def test_ring(ring, window, R):
    """Rings past wrap, including sizes that are not multiples of 16 (a chunk
    then straddles the wrap point and is gathered row by row)."""
    g = torch.Generator().manual_seed(ring + window + R)
    seq = torch.randint(window, 3 * ring + 50, (6,), generator=g).tolist()
    seq[0] = R  # a ring not yet full
    seq[1] = ring + 3  # just past the wrap
    case = synth.decode_case(5000 + ring + R, RING, 6, R, 16, 4, 128, seq, window=window,
                             ring=ring)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"ring {ring}/{window} R={R}")


@pytest.mark.parametrize("window", [1, 5, 100, 1000])
def test_linear_window(window):
    case = synth.decode_case(6000 + window, LINEAR, 3, 4, 32, 8, 128, [2000, 5, 700],
                             window=window)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"linear window={window}")


def test_split_count_independent_bound():
    """max_seq_len only sizes the grid: a larger bound (more splits) gives the
    same answer within tolerance, and each configuration is deterministic."""
    case = synth.decode_case(7001, LINEAR, 2, 1, 32, 8, 128, [3000, 2999], slots_per_seq=8192)
    ref, _, _ = oracle_decode(case)
    outs = []
    for bound in (3000, 8192):
        a, _ = gpu_decode(case, max_seq_len=bound)
        b, _ = gpu_decode(case, max_seq_len=bound)
        assert torch.equal(a, b), "run-to-run results differ"
        compare(a, ref, f"bound {bound}")
        outs.append(a)


def test_single_key_is_value():
    case = synth.decode_case(7002, PAGED, 4, 1, 32, 8, 128, [1, 1, 1, 1])
    out, _ = gpu_decode(case)
    want = case.v_new.view(4, 1, 8, 1, 128).expand(4, 1, 8, 4, 128).reshape(4, 1, 32, 128)
    assert torch.equal(out.cpu(), want), "one valid key must return its value exactly"


def test_graph_replay_follows_device_state():
    """A graph captured once replays for later steps whose seq_lens,
    positions and slot_mapping change only on the device (vibevoice.c, 'The
    decode step is one submission'): replays match direct launches."""
    dev = "cuda"
    Hq, Hkv, D, B = 32, 8, 128, 2
    cap = 2048
    case = synth.decode_case(7003, LINEAR, B, 1, Hq, Hkv, D, [1000, 1500], slots_per_seq=cap)
    cache = gq.KVCache(LINEAR, case.k_cache.to(dev), case.v_cache.to(dev), slots_per_seq=cap)
    q = case.q.to(dev)
    kn, vn = case.k_new.to(dev), case.v_new.to(dev)
    seq = case.seq_lens.to(dev)
    pos = case.positions.to(dev)
    slots = case.slot_mapping.to(dev)
    out = torch.empty_like(q)
    ws = torch.zeros(gq.attn_decode_workspace_size(cache, B, 1, Hq, cap, 0), dtype=torch.uint8,
                     device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        gq.attn_kv_append(kn, vn, slots, cache, err=err)  # warm-up outside capture
        gq.attn_decode(q, cache, seq, pos, cap, 0, case.scale, out=out, workspace=ws, err=err)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            gq.attn_kv_append(kn, vn, slots, cache, err=err)
            gq.attn_decode(q, cache, seq, pos, cap, 0, case.scale, out=out, workspace=ws,
                           err=err)
    torch.cuda.synchronize()
    for step in range(20):
        # next step: one more key per request, new row at the new position
        seq += 1
        pos += 1
        slots += 1
        kn.copy_(torch.randn(kn.shape, device=dev).to(torch.bfloat16))
        vn.copy_(torch.randn(vn.shape, device=dev).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        direct = gq.attn_decode(q, cache, seq, pos, cap, 0, case.scale, workspace=ws, err=err)
        torch.cuda.synchronize()
        assert torch.equal(got, direct), f"replay {step} differs from a direct launch"
    assert int(err.item()) == 0


def test_out_of_range_page_is_reported_not_faulted():
    case = synth.decode_case(7004, PAGED, 2, 1, 8, 2, 128, [40, 40], block_size=16)
    bt = case.block_table.clone()
    bt[1, 1] = 10_000_000  # a page id far outside the pool
    case.block_table = bt
    dev = "cuda"
    cache = gq.KVCache(PAGED, case.k_cache.to(dev), case.v_cache.to(dev),
                       block_table=bt.to(dev), block_size=16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gq.attn_decode(case.q.to(dev), cache, case.seq_lens.to(dev), case.positions.to(dev),
                         40, 0, case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gq.ATTN_ERR_BOUNDS
    assert torch.isfinite(out.float()).all()


def test_out_of_range_slot_mapping_is_reported():
    dev = "cuda"
    k = torch.zeros(64, 2, 128, dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    cache = gq.KVCache(LINEAR, k, v, slots_per_seq=64)
    kn = torch.ones(3, 2, 128, dtype=torch.bfloat16, device=dev)
    vn = 2 * kn
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    gq.attn_kv_append(kn, vn, torch.tensor([5, 64, -1], device=dev), cache, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == gq.ATTN_ERR_BOUNDS
    assert torch.equal(k[5].cpu(), kn[0].cpu()) and float(k.float().sum()) == 256.0


def test_append_bit_exact():
    dev = "cuda"
    g = torch.Generator().manual_seed(7005)
    for Hkv, D, n in [(8, 128, 256), (4, 128, 14449), (32, 64, 4), (1, 64, 1)]:
        S = max(4 * n, 64)
        k = synth.normal_bf16(g, (S, Hkv, D))
        v = synth.normal_bf16(g, (S, Hkv, D))
        kn = synth.normal_bf16(g, (n, Hkv, D))
        vn = synth.normal_bf16(g, (n, Hkv, D))
        slots = torch.randperm(S, generator=g)[:n]
        kc, vc = oracle_bits = (None, None)
        import oracle

        kc, vc = oracle.bf16_bits(k).copy(), oracle.bf16_bits(v).copy()
        oracle.kv_append(kc, vc, oracle.bf16_bits(kn), oracle.bf16_bits(vn), slots.numpy())
        cache = gq.KVCache(LINEAR, k.to(dev), v.to(dev), slots_per_seq=S)
        gq.attn_kv_append(kn.to(dev), vn.to(dev), slots.to(dev), cache)
        torch.cuda.synchronize()
        assert np.array_equal(oracle.bf16_bits(cache.k), kc)
        assert np.array_equal(oracle.bf16_bits(cache.v), vc)


@pytest.mark.parametrize("batch", [1, 3])
def test_streaming_encoder_step(batch):
    """4 new frames over a 1,500-slot ring with a 750-frame window, 32 = 32
    heads, D=64 (Voxtral notes, "Encoder KV cache"), long past the wrap."""
    case = synth.streaming_encoder_step(batch=batch)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"streaming encoder B={batch}")


@pytest.mark.parametrize("B,R,Hq,Hkv", [(300, 1, 8, 2), (150, 16, 8, 2), (260, 8, 16, 4)])
def test_batch_split_over_launches(B, R, Hq, Hkv):
    """More (request, row block) pairs than one launch's shared tables hold:
    the host cuts the batch into several launches (one of them ragged)."""
    g = torch.Generator().manual_seed(B * R)
    seq = torch.randint(R, 200, (B,), generator=g).tolist()
    case = synth.decode_case(7100 + B + R, LINEAR, B, R, Hq, Hkv, 128, seq)
    ref, _, _ = oracle_decode(case)
    out, _ = gpu_decode(case)
    compare(out, ref, f"batch {B} x {R} rows")


@pytest.mark.parametrize("L", [8192, 8200, 16000])
def test_one_unit_over_many_ctas(L):
    """One long (request, KV head) among 40 units (too many for the merge
    kernel), over 64-126 CTAs: its partial states are merged inside the
    split kernel in groups of eight (a ragged last group), then the groups;
    the largest of these bounds is the last one merged that way."""
    seq = [L] + [1 + (7 * i) % 40 for i in range(39)]
    case = synth.decode_case(7200 + L, LINEAR, 40, 1, 8, 1, 128, seq, slots_per_seq=L)
    cache = to_device(case)
    assert gq.attn_decode_kernel_launches(cache, 40, 1, 8, case.max_seq_len()) == 1
    ref, _, _ = oracle_decode(case)
    a, _ = gpu_decode(case)
    b, _ = gpu_decode(case)
    assert torch.equal(a, b), "run-to-run results differ"
    compare(a, ref, f"one unit of 40, {L} keys")


@pytest.mark.parametrize("L", [2000, 8192, 14449])
def test_few_units_merge_kernel(L):
    """Two requests x 4 KV heads (Qwen2-7B's grouping) at mid contexts: eight
    units over 304 CTAs, so their parts go to the merge kernel."""
    case = synth.decode_case(7250 + L, LINEAR, 2, 1, 28, 4, 128, [L, L - 77])
    cache = to_device(case)
    assert gq.attn_decode_kernel_launches(cache, 2, 1, 28, case.max_seq_len()) == 2
    ref, _, _ = oracle_decode(case)
    a, _ = gpu_decode(case)
    b, _ = gpu_decode(case)
    assert torch.equal(a, b), "run-to-run results differ"
    compare(a, ref, f"few units, {L} keys")


def test_merge_kernel_threshold():
    """Just past the bound where the library hands long units to its merge
    kernel: same answer within tolerance, deterministic."""
    case = synth.decode_case(7300, LINEAR, 1, 2, 16, 2, 128, [16400], slots_per_seq=16512)
    ref, _, _ = oracle_decode(case)
    a, _ = gpu_decode(case, max_seq_len=16512)
    b, _ = gpu_decode(case, max_seq_len=16512)
    assert torch.equal(a, b), "run-to-run results differ"
    compare(a, ref, "merge kernel threshold")


def test_one_workspace_serves_every_shape():
    """A serving loop keeps one workspace, sized for its largest shape, and
    calls the decode with whatever batch it has: the merge counters of every
    shape sit in one region at the start that every call leaves at zero, and
    the partial states after it, so a call that writes more partial states
    never leaves garbage where another shape counts."""
    g = torch.Generator().manual_seed(7500)
    small = synth.decode_case(7501, LINEAR, 40, 1, 32, 8, 128,
                              torch.randint(600, 1500, (40,), generator=g).tolist())
    large = synth.decode_case(7502, LINEAR, 64, 4, 32, 8, 128,
                              torch.randint(64, 2000, (64,), generator=g).tolist())
    sizes = []
    for c in (small, large):
        sizing = gq.KVCache(c.kind, c.k_cache, c.v_cache, slots_per_seq=c.slots_per_seq)
        sizes.append(gq.attn_decode_workspace_size(sizing, c.batch, c.q_rows, c.n_q_heads,
                                                   c.max_seq_len(), 0))
    ws = torch.zeros(max(sizes), dtype=torch.uint8, device="cuda")

    def run(case):
        cache = to_device(case)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gq.attn_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), cache,
                          err=err)
        out = gq.attn_decode(case.q.cuda(), cache, case.seq_lens.cuda(), case.positions.cuda(),
                             case.max_seq_len(), 0, case.scale, workspace=ws, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        return out

    first = run(small)
    run(large)
    again = run(small)
    assert torch.equal(first, again), "a call of another shape disturbed the workspace"
    ref, _, _ = oracle_decode(small)
    compare(again, ref, "small batch after a large one, one workspace")
