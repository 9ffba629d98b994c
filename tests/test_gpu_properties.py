"""Properties of the CUDA path that the pages test on their own kernels
(vibevoice.c, "Attention backends": the backend tests compare a paged cache
with a shuffled page table and a partial last page against the contiguous
cache bit for bit, and run decodes concurrently).

* A paged cache whose pages are dealt in a shuffled order, the last page of
  each request partly filled, gives exactly the bits of a linear cache that
  holds the same keys at the same positions: the split of the key range and
  the order of every sum depend on positions only.
* Two decodes issued on two streams with two workspaces, free to overlap on
  the GPU, each give exactly what they give alone and match the oracle.
"""
import numpy as np
import pytest
import torch

import gqa_attention_kv_gb300 as gq
from gqa_attention_kv_gb300 import synth
from helpers import compare, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _paged_and_linear(case):
    """Device caches of a paged case (after its append) and a linear cache
    holding the same keys: linear slot b * cap + t = page slot of (b, t)."""
    bs = case.block_size
    paged = gq.KVCache(synth.PAGED, case.k_cache.to(DEV), case.v_cache.to(DEV),
                       block_table=case.block_table.to(DEV), block_size=bs)
    gq.attn_kv_append(case.k_new.to(DEV), case.v_new.to(DEV), case.slot_mapping.to(DEV), paged)
    torch.cuda.synchronize()
    seq = case.seq_lens.cpu().tolist()
    cap = max(64, -(-max(seq) // 64) * 64)
    bt = case.block_table.cpu()
    idx = torch.zeros(case.batch * cap, dtype=torch.int64)
    for b, n in enumerate(seq):
        t = torch.arange(n)
        idx[b * cap: b * cap + n] = bt[b, t // bs].long() * bs + t % bs
    idx = idx.to(DEV)
    lin = gq.KVCache(synth.LINEAR, paged.k[idx].contiguous(), paged.v[idx].contiguous(),
                     slots_per_seq=cap)
    return paged, lin, cap


@pytest.mark.parametrize("block_size", [16, 64, 5])
@pytest.mark.parametrize("R,Hq,Hkv", [(1, 28, 4), (4, 32, 8)])
def test_paged_shuffled_equals_linear_bitwise(block_size, R, Hq, Hkv):
    seq = [3001, 17, 1024, 2050, 64 + R, 777]
    case = synth.decode_case(9600 + block_size + R, synth.PAGED, len(seq), R, Hq, Hkv, 128, seq,
                             block_size=block_size,
                             num_blocks=sum(-(-n // block_size) for n in seq) + 40)
    # the pages are dealt from a shuffled pool, and a last page is partial
    assert any(n % block_size for n in seq)
    paged, lin, cap = _paged_and_linear(case)
    q, sl, pos = case.q.to(DEV), case.seq_lens.to(DEV), case.positions.to(DEV)
    max_seq = max(seq)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_p = gq.attn_decode(q, paged, sl, pos, max_seq, 0, case.scale, err=err)
    out_l = gq.attn_decode(q, lin, sl, pos, max_seq, 0, case.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_p, out_l), "paged and linear caches of the same keys differ"
    ref, _, _ = oracle_decode(case)
    compare(out_p, ref, f"paged bs={block_size}")


def test_two_streams_two_workspaces_overlap():
    c1 = synth.decode_case(9701, synth.LINEAR, 2, 1, 28, 4, 128, [14449, 9000])
    c2 = synth.decode_case(9702, synth.PAGED, 16, 4, 32, 8, 128,
                           [int(x) for x in np.random.default_rng(9702).integers(64, 4096, 16)],
                           block_size=16)
    runs = []
    for c in (c1, c2):
        cache = gq.KVCache(c.kind, c.k_cache.to(DEV), c.v_cache.to(DEV),
                           slots_per_seq=c.slots_per_seq,
                           block_table=None if c.block_table is None else c.block_table.to(DEV),
                           block_size=c.block_size)
        gq.attn_kv_append(c.k_new.to(DEV), c.v_new.to(DEV), c.slot_mapping.to(DEV), cache)
        ws = torch.zeros(gq.attn_decode_workspace_size(cache, c.batch, c.q_rows, c.n_q_heads,
                                                       c.max_seq_len(), c.window),
                         dtype=torch.uint8, device=DEV)
        args = (c.q.to(DEV), cache, c.seq_lens.to(DEV), c.positions.to(DEV), c.max_seq_len(),
                c.window, c.scale)
        runs.append((c, args, ws))
    torch.cuda.synchronize()
    alone = [gq.attn_decode(*a, workspace=w) for _, a, w in runs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    errs = [torch.zeros(1, dtype=torch.int32, device=DEV) for _ in streams]
    outs = [torch.empty_like(a) for a in alone]
    for rep in range(3):
        # each stream issues its decode several times with nothing ordering
        # the two streams against each other
        for k in range(4):
            for (c, a, w), s, e, o in zip(runs, streams, errs, outs):
                with torch.cuda.stream(s):
                    gq.attn_decode(*a, out=o, workspace=w, err=e, stream=s)
        torch.cuda.synchronize()
        for e in errs:
            assert int(e.item()) == 0
        for o, want in zip(outs, alone):
            assert torch.equal(o, want), f"overlapping decodes differ (round {rep})"
    for (c, _, _), o in zip(runs, outs):
        ref, _, _ = oracle_decode(c)
        compare(o, ref, "two streams")
