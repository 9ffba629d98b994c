"""Seeded synthetic inputs shaped like the pages' models.

This module holds no attention arithmetic.  It draws the random tensors and
does the caller's bookkeeping that a serving engine would do before calling
the library: it picks sequence lengths and positions, deals pages of a pool
into block tables, and reserves the cache slot of every new K/V row
(``slot_mapping``).  Both the CUDA path and the fp64 oracle consume what it
returns; neither imports the other.

Random numbers are drawn with ``torch.Generator`` seeded per case, N(0, 1) in
fp32 and rounded to bf16.  ``device`` selects where they are drawn: the same
seed gives different (equally valid) numbers on CPU and CUDA generators.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

LINEAR, PAGED, RING = 0, 1, 2
KIND_NAMES = {LINEAR: "linear", PAGED: "paged", RING: "ring"}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(gen: torch.Generator, shape, device="cpu") -> torch.Tensor:
    """N(0, 1) drawn in fp32, rounded to bf16."""
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class DecodeCase:
    """One decode step: new rows are appended via slot_mapping, then attended.

    q        [B, R, Hq, D] bf16        query rows of the step
    k_cache  [S, Hkv, D] bf16          cache before the step's append
    v_cache  [S, Hkv, D] bf16
    k_new    [B*R, Hkv, D] bf16        the step's new K/V rows
    v_new    [B*R, Hkv, D] bf16
    slot_mapping [B*R] int64           slot reserved for each new row
    seq_lens [B] int32                 keys written after the append
    positions [B*R] int32              absolute position of each query row
    """
    kind: int
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    slot_mapping: torch.Tensor
    seq_lens: torch.Tensor
    positions: torch.Tensor
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    window: int
    scale: float
    slots_per_seq: int = 0
    block_table: Optional[torch.Tensor] = None
    block_size: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def q_rows(self) -> int:
        return self.q.shape[1]

    @property
    def num_slots(self) -> int:
        return self.k_cache.shape[0]

    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0


def positions_for(seq_lens: torch.Tensor, q_rows: int) -> torch.Tensor:
    """Rows of a step sit at the last q_rows positions: seq_len - R + r."""
    r = torch.arange(q_rows, dtype=torch.int64)
    pos = seq_lens.to(torch.int64)[:, None] - q_rows + r[None, :]
    return pos.reshape(-1).to(torch.int32)


def reserve_linear(seq_lens, q_rows, slots_per_seq):
    pos = positions_for(seq_lens, q_rows).to(torch.int64)
    b = torch.arange(seq_lens.shape[0], dtype=torch.int64).repeat_interleave(q_rows)
    return b * slots_per_seq + pos


def reserve_paged(seq_lens, q_rows, block_table, block_size):
    pos = positions_for(seq_lens, q_rows).to(torch.int64)
    b = torch.arange(seq_lens.shape[0], dtype=torch.int64).repeat_interleave(q_rows)
    page = block_table.to(torch.int64)[b, pos // block_size]
    return page * block_size + pos % block_size


def reserve_ring(seq_lens, q_rows, ring):
    pos = positions_for(seq_lens, q_rows).to(torch.int64)
    b = torch.arange(seq_lens.shape[0], dtype=torch.int64).repeat_interleave(q_rows)
    return b * ring + pos % ring


def deal_block_table(gen, seq_lens, block_size, num_blocks, max_blocks=None):
    """A seeded permutation of the pool's page ids dealt to requests in order."""
    need = [(int(s) + block_size - 1) // block_size for s in seq_lens.tolist()]
    total = sum(need)
    if total > num_blocks:
        raise ValueError(f"pool of {num_blocks} pages cannot hold {total}")
    mb = max_blocks or max(max(need), 1)
    perm = torch.randperm(num_blocks, generator=gen)
    table = torch.zeros((len(need), mb), dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n].to(torch.int32)
        at += n
    return table


def decode_case(seed, kind, batch, q_rows, n_q_heads, n_kv_heads, head_dim, seq_lens,
                window=0, slots_per_seq=None, block_size=16, num_blocks=None, ring=None,
                scale=None, device="cpu") -> DecodeCase:
    """Build one decode step of the given cache kind.

    seq_lens: list/tensor of keys written per request after the step's append.
    linear: slots_per_seq >= max(seq_lens) (default: max rounded up to 64).
    paged : block_size, num_blocks (default: exactly what the requests need + 3).
    ring  : ring size (default 2 * window, at least window + q_rows - 1).
    """
    gen = generator(seed, device)
    cpu_gen = generator(seed + 7919) if device != "cpu" else gen
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(-1)
    if seq_lens.shape[0] != batch:
        raise ValueError("seq_lens must have one entry per request")
    if int(seq_lens.min()) < q_rows:
        raise ValueError("every request must hold at least its q_rows new keys")
    D, Hkv = head_dim, n_kv_heads
    block_table = None
    meta = {}
    if kind == LINEAR:
        sps = slots_per_seq or max(64, int(math.ceil(int(seq_lens.max()) / 64.0)) * 64)
        num_slots = batch * sps
        slot_mapping = reserve_linear(seq_lens, q_rows, sps)
    elif kind == PAGED:
        need = sum((int(s) + block_size - 1) // block_size for s in seq_lens.tolist())
        nb = num_blocks or need + 3
        block_table = deal_block_table(cpu_gen, seq_lens, block_size, nb)
        num_slots = nb * block_size
        sps = 0
        slot_mapping = reserve_paged(seq_lens, q_rows, block_table, block_size)
    elif kind == RING:
        sps = ring or max(2 * window, window + q_rows - 1)
        num_slots = batch * sps
        slot_mapping = reserve_ring(seq_lens, q_rows, sps)
    else:
        raise ValueError(f"unknown cache kind {kind}")
    q = normal_bf16(gen, (batch, q_rows, n_q_heads, D), device)
    k_cache = normal_bf16(gen, (num_slots, Hkv, D), device)
    v_cache = normal_bf16(gen, (num_slots, Hkv, D), device)
    k_new = normal_bf16(gen, (batch * q_rows, Hkv, D), device)
    v_new = normal_bf16(gen, (batch * q_rows, Hkv, D), device)
    return DecodeCase(kind=kind, q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new,
                      v_new=v_new, slot_mapping=slot_mapping.to(device),
                      seq_lens=seq_lens.to(device),
                      positions=positions_for(seq_lens, q_rows).to(device),
                      n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=D, window=window,
                      scale=scale if scale is not None else 1.0 / math.sqrt(D),
                      slots_per_seq=sps,
                      block_table=None if block_table is None else block_table.to(device),
                      block_size=block_size if kind == PAGED else 0, meta=meta)


@dataclass
class PrefillCase:
    q: torch.Tensor  # [B, T, Hq, D]
    k: torch.Tensor  # [B, T, Hkv, D]
    v: torch.Tensor
    window: int
    scale: float

    @property
    def shape(self):
        B, T, Hq, D = self.q.shape
        return B, T, Hq, self.k.shape[2], D


def prefill_case(seed, batch, seq_len, n_q_heads, n_kv_heads, head_dim, window=0, scale=None,
                 device="cpu") -> PrefillCase:
    gen = generator(seed, device)
    q = normal_bf16(gen, (batch, seq_len, n_q_heads, head_dim), device)
    k = normal_bf16(gen, (batch, seq_len, n_kv_heads, head_dim), device)
    v = normal_bf16(gen, (batch, seq_len, n_kv_heads, head_dim), device)
    return PrefillCase(q=q, k=k, v=v, window=window,
                       scale=scale if scale is not None else 1.0 / math.sqrt(head_dim))


# ---------------------------------------------------------------------------
# The five workloads, shaped like the pages' models (seed = 20260 + number).
# ---------------------------------------------------------------------------

def voxtral_decode_step(device="cpu"):
    """Voxtral decoder, one step: B=1, R=1, 32 q / 8 kv heads, D=128, linear
    cache of 512 keys (the new row lands at position 511)."""
    return decode_case(20261, LINEAR, 1, 1, 32, 8, 128, [512], device=device)


def encoder_prefill(long: bool = False, device="cpu"):
    """Speech encoder causal prefill: T=750, 32 = 32 heads, D=64, scale 1/8;
    the long variant is T=1500 with a 750-frame window."""
    if long:
        return prefill_case(20262 + 100, 1, 1500, 32, 32, 64, window=750, scale=0.125,
                            device=device)
    return prefill_case(20262, 1, 750, 32, 32, 64, window=0, scale=0.125, device=device)


QWEN_PROMPT = 14449
QWEN_CONTEXTS = (14449, 17623, 20797, 23971)


def qwen_prefill(device="cpu"):
    """Qwen2-7B-shaped prompt prefill: T=14,449, 28 q / 4 kv heads, D=128."""
    return prefill_case(20263, 1, QWEN_PROMPT, 28, 4, 128, device=device)


def qwen_decode(contexts=(QWEN_PROMPT, QWEN_PROMPT), device="cpu", seed=20263):
    """Two slots decoding one row each at the given contexts (keys incl. the new row)."""
    return decode_case(seed + 1000, LINEAR, 2, 1, 28, 4, 128, list(contexts),
                       slots_per_seq=QWEN_CONTEXTS[-1] + 1, device=device)


def ring_window_decode(device="cpu", batch=16):
    """Streaming ring decode: ring 16,384, window 8,192, 16 sequences at
    positions uniform in [8,192, 40,000], one row each."""
    g = generator(20264)
    pos = torch.randint(8192, 40001, (batch,), generator=g, dtype=torch.int64)
    return decode_case(20264, RING, batch, 1, 32, 8, 128, (pos + 1).tolist(), window=8192,
                       ring=16384, device=device)


def streaming_encoder_step(device="cpu", batch=1):
    """Streaming speech encoder, one step of one layer: 4 new frames attend
    over a 1,500-slot ring with a 750-frame window, 32 = 32 heads, D=64, scale
    1/8, the stream long past the ring's wrap (Voxtral notes, "Encoder KV
    cache")."""
    return decode_case(20266, RING, batch, 4, 32, 32, 64, [6004] * batch, window=750,
                       ring=1500, scale=0.125, device=device)


def chunked_prefill_step(device="cpu", batch=2, chunk=29):
    """A prompt arriving in 29-row chunks (vibevoice.c's streaming 7B backend)
    on the Qwen2-7B decoder shape (28 q / 4 kv heads, D=128): the last chunk
    of each request's 14,449-token prompt, rows at positions 14,420 ..
    14,448, against a linear cache holding the earlier rows."""
    return decode_case(20267, LINEAR, batch, chunk, 28, 4, 128, [QWEN_PROMPT] * batch,
                       device=device)


def paged_multirow_decode(device="cpu", batch=64):
    """Paged K=4 uniform decode: 64 requests x 4 rows, bs 16, 200k-slot pool
    (12,500 pages dealt from a seeded permutation), seq_lens in [64, 4,096]."""
    g = generator(20265)
    sl = torch.randint(64, 4097, (batch,), generator=g, dtype=torch.int64)
    return decode_case(20265, PAGED, batch, 4, 32, 8, 128, sl.tolist(), block_size=16,
                       num_blocks=12500, device=device)
