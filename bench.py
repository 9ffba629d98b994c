#!/usr/bin/env python3
"""Throughput of the GQA attention hot path on one GB300 (or N replicas).

One step of the default workload is one pass of the whole path over the
Qwen2-7B-shaped decoder (28 q / 4 kv heads, head_dim 128, bf16):

  1. causal prefill of a 14,449-token prompt          (attn_prefill)
  2. KV append of those 14,449 prompt rows            (attn_kv_append)
  3. five decode steps of 2 slots x 1 row, at contexts 14,449 / 17,623 /
     20,797 / 23,971 and the mixed pair (14,449, 23,971), each appending its
     2 new rows in the same launch                     (attn_decode_append)

Printed metric (one JSON line): decode-attention KV GB/s over the step's
decode launches (``value``), prefill TFLOP/s over its prefill launch
(``prefill``), both as fractions of the measured HBM / dense-bf16 peaks.
Inputs are seeded synthetic tensors; decode caches rotate over copies that
total more than 4x the L2 so every decode reads DRAM; the prefill inputs and
output (236 MB) exceed the L2 by themselves.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload qwen|voxtral|encoder|encoder-long|ring|paged|
                              stream-encoder|ring-fp8|paged-fp8|voxtral-fp8|
                              qwen-prefill|prefill-8k|chunked] [--layout bshd|bhsd]

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (the oracle is the only reference implementation there is).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

NOMINAL_HBM_GBS = 7900.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------
# algorithmic work
# --------------------------------------------------------------------------

# DRAM bytes (read + write) of one full-size Qwen2-7B prompt prefill launch,
# T = 14,449, from ncu (profiles/prefill_kernel_qwen14449.md).  They
# describe the kernel built from these exact sources and are dropped (null)
# once either file changes.
PREFILL_TRAFFIC = {"T": 14449, "bytes": 198099200,
                   "sources": ("gqa_attention_kv_gb300/csrc/prefill.cu",
                               "gqa_attention_kv_gb300/csrc/ptx.cuh"),
                   "sha256": "115c6fa0c9008eea39e7d09d55a27d44c520a44b4e1242a749e24f57669c3c27"}


def prefill_traffic(T):
    import hashlib

    if T != PREFILL_TRAFFIC["T"]:
        return None
    h = hashlib.sha256()
    for f in PREFILL_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return PREFILL_TRAFFIC["bytes"] if h.hexdigest() == PREFILL_TRAFFIC["sha256"] else None


def prefill_flops(T, Hq, D, window=0):
    """4 * D * Hq * (unmasked query-key pairs): QK^T and PV, 2 flops per MAC."""
    if window and window > 0:
        pairs = sum(min(i + 1, window) for i in range(T))
    else:
        pairs = T * (T + 1) // 2
    return 4.0 * D * Hq * pairs


def decode_bytes(keys_per_request_head, Hkv, D, B, R, Hq, append_rows, kv_elem=2):
    """K+V bytes of the valid keys (each KV head read once) + q + out + the
    appended rows (bf16 read + cache write); kv_elem = bytes per cache element
    (2: bf16, 1: FP8)."""
    kv = 2 * kv_elem * D * Hkv * keys_per_request_head
    qo = 2 * 2 * B * R * Hq * D
    app = 2 * (2 + kv_elem) * append_rows * Hkv * D
    return kv + qo + app


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(gpu_index).uuid)
            self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.proc = None
        self.path = None

    def start(self):
        import tempfile

        try:
            fd, self.path = tempfile.mkstemp(prefix=f"gqa_clocks_{os.getpid()}_", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # nvidia-smi takes a moment to start: hold the timed region until the
        # first sample is on disk, so every sample falls inside it
        t_end = time.time() + 5.0
        while time.time() < t_end and self.proc.poll() is None:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[4]), parts[5:9]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        loaded = [r for r in rows if r[2] >= 50.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median([r[0] for r in loaded]) if loaded else None,
                "sm_max_mhz": max(r[1] for r in rows) if rows else None,
                "reasons": reasons, "samples": len(loaded)}


# --------------------------------------------------------------------------
# workloads (device side)
# --------------------------------------------------------------------------

class Workload:
    """A step = a fixed sequence of library calls.  Subclasses fill ``groups``:
    a list of (name, callable) that each issue launches on the current stream;
    events are recorded around every group."""

    name = ""
    describe = {}
    launches_per_step = 0

    def decode_bytes_per_step(self):
        return 0.0

    def prefill_flops_per_step(self):
        return 0.0


def _l2_bytes():
    import torch

    try:
        return int(torch.cuda.get_device_properties(0).L2_cache_size)
    except Exception:
        return 129 * 2 ** 20


class QwenWorkload(Workload):
    name = "qwen2-7b prompt prefill 14449 + decode 2x1 at 14449..23971"
    CONTEXTS = [(14449, 14449), (17623, 17623), (20797, 20797), (23971, 23971), (14449, 23971)]

    def __init__(self, dev, layout=0):
        import torch

        import gqa_attention_kv_gb300 as gq
        from gqa_attention_kv_gb300 import synth

        self.gq, self.torch = gq, torch
        Hq, Hkv, D = 28, 4, 128
        self.Hq, self.Hkv, self.D = Hq, Hkv, D
        self.T = synth.QWEN_PROMPT
        p = synth.qwen_prefill(device=dev)
        self.q, self.k, self.v, self.scale = p.q, p.k, p.v, p.scale
        self.out = torch.empty_like(self.q)
        self.cap = max(c for pair in self.CONTEXTS for c in pair)
        self.B = 2
        # decode caches: enough copies that consecutive decodes never share one
        # and the copies together exceed 4x the L2
        per_copy = 2 * self.B * self.cap * Hkv * D * 2
        self.ncopy = max(6, math.ceil(4 * _l2_bytes() / per_copy) + 1)
        g = synth.generator(20263 + 5000, dev)
        self.caches = []
        # slot-major [slot][head][D], or head-major [request][head][slot][D]
        shape = (self.B * self.cap, Hkv, D) if layout == 0 else (self.B, Hkv, self.cap, D)
        for _ in range(self.ncopy):
            kc = synth.normal_bf16(g, shape, dev)
            vc = synth.normal_bf16(g, shape, dev)
            self.caches.append(gq.KVCache(synth.LINEAR, kc, vc, slots_per_seq=self.cap,
                                          layout=layout))
        self.prompt_slots = torch.arange(self.T, dtype=torch.int64, device=dev)
        self.dec = []
        for i, ctx in enumerate(self.CONTEXTS):
            c = synth.decode_case(20263 + 100 + i, synth.LINEAR, self.B, 1, Hq, Hkv, D, list(ctx),
                                  slots_per_seq=self.cap, device=dev)
            self.dec.append({"q": c.q, "k_new": c.k_new, "v_new": c.v_new,
                             "slots": c.slot_mapping, "seq": c.seq_lens, "pos": c.positions,
                             "out": torch.empty_like(c.q), "ctx": ctx})
        self.max_seq = self.cap
        self.ws = torch.zeros(gq.attn_decode_workspace_size(self.caches[0], self.B, 1, Hq,
                                                            self.max_seq, 0),
                              dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.step_i = 0
        # prefill, prompt append, per decode the kernels the library plans
        # (split kernel + merge kernel at these long contexts)
        self.launches_per_step = 1 + 1 + len(self.CONTEXTS) * gq.attn_decode_kernel_launches(
            self.caches[0], self.B, 1, Hq, self.max_seq, 0, with_append=True, tables_early=True)
        self.describe = {"workload": self.name, "model": "Qwen2-7B-shaped decoder attention",
                         "n_q_heads": Hq, "n_kv_heads": Hkv, "head_dim": D,
                         "prefill_tokens": self.T, "decode_batch": self.B, "q_rows": 1,
                         "decode_contexts": [list(c) for c in self.CONTEXTS],
                         "cache": "linear", "decode_cache_copies": self.ncopy,
                         "kv_layout": "BHSD" if layout else "BSHD",
                         "l2_defeat": "decode caches rotate over copies > 4x L2; prefill "
                                      "inputs+output 236 MB > L2"}

    def prefill_flops_per_step(self):
        return prefill_flops(self.T, self.Hq, self.D)

    def decode_bytes_per_step(self):
        tot = 0.0
        for d in self.dec:
            keys = sum(d["ctx"])
            tot += decode_bytes(keys, self.Hkv, self.D, self.B, 1, self.Hq, self.B)
        return tot

    def prompt_append_bytes(self):
        return 2 * 2 * 2 * self.T * self.Hkv * self.D

    def _decode_part(self, s, e2e=False):
        gq = self.gq
        for i, d in enumerate(self.dec):
            if e2e:
                # this call's inputs, packed in one pinned buffer: one transfer
                pk = self.h["dec"][i]
                pk["dev"].copy_(pk["host"], non_blocking=True)
                d = pk["views"] | {"out": d["out"]}
            c = self.caches[(s * 6 + 1 + i) % self.ncopy]
            # seq_lens / positions are written before the step, never by the
            # kernel just before a decode, and the caches rotate, so no kernel
            # that may still run writes the cache a call reads: it may plan and
            # start its first cache tiles while that one finishes
            gq.attn_decode_append(d["q"], d["k_new"], d["v_new"], d["slots"], c, d["seq"],
                                  d["pos"], self.max_seq, 0, self.scale, out=d["out"],
                                  workspace=self.ws, err=self.err, tables_early=True,
                                  cache_early=True)
            if e2e:
                self.h["dec"][i]["out"].copy_(d["out"], non_blocking=True)

    def capture(self, stream, e2e=False):
        """One CUDA graph of the decode part per cache-rotation index (the
        launches are identical from step to step, as a serving engine replays
        them; vibevoice.c, 'The decode step is one submission')."""
        torch = self.torch
        graphs = []
        for r in range(self.ncopy):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self._decode_part(r, e2e)
            graphs.append(g)
        torch.cuda.synchronize()
        if e2e:
            self.graphs_e2e = graphs
        else:
            self.graphs = graphs

    def run_step(self, ev):
        """Issue one step; ev(name) records an event at a boundary."""
        gq = self.gq
        s = self.step_i
        self.step_i += 1
        ev("prefill")
        gq.attn_prefill(self.q, self.k, self.v, 0, self.scale, out=self.out, err=self.err)
        ev("prompt_append")
        c0 = self.caches[(s * 6) % self.ncopy]
        gq.attn_kv_append(self.k[0], self.v[0], self.prompt_slots, c0, err=self.err)
        ev("decode")
        if getattr(self, "graphs", None):
            self.graphs[s % self.ncopy].replay()
        else:
            self._decode_part(s)
        ev("end")

    # end to end through host buffers ---------------------------------------
    def _packed(self, d):
        """A decode call's inputs (q, k_new, v_new, slot_mapping, seq_lens,
        positions) at 256-byte offsets of one pinned host buffer, with views of
        the same offsets into one device buffer: the call copies them with one
        transfer, as a serving engine stages a step's inputs."""
        torch = self.torch
        keys = ("q", "k_new", "v_new", "slots", "seq", "pos")
        offs, n = [], 0
        for k in keys:
            offs.append(n)
            n += (d[k].numel() * d[k].element_size() + 255) // 256 * 256
        host = torch.empty(n, dtype=torch.uint8).pin_memory()
        dev = torch.empty(n, dtype=torch.uint8, device=d["q"].device)
        views = {}
        for k, o in zip(keys, offs):
            t = d[k]
            nb = t.numel() * t.element_size()
            host[o:o + nb].view(t.dtype).view(t.shape).copy_(t.detach().cpu())
            views[k] = dev[o:o + nb].view(t.dtype).view(t.shape)
        return {"host": host, "dev": dev, "views": views,
                "out": torch.empty(d["q"].shape, dtype=d["q"].dtype).pin_memory()}

    def setup_host(self):
        torch = self.torch
        pin = lambda t: t.detach().to("cpu").pin_memory()
        self.h = {"q": pin(self.q), "k": pin(self.k), "v": pin(self.v),
                  "out": torch.empty(self.q.shape, dtype=self.q.dtype).pin_memory(),
                  "dec": [self._packed(d) for d in self.dec]}
        self.h2d_prefill = sum(self.h[k].numel() * self.h[k].element_size() for k in "qkv")
        self.d2h_prefill = self.h["out"].numel() * self.h["out"].element_size()
        self.h2d_decode = sum(d["host"].numel() for d in self.h["dec"])
        self.d2h_decode = sum(d["out"].numel() * d["out"].element_size() for d in self.h["dec"])

    def run_step_e2e(self, ev):
        gq = self.gq
        h = self.h
        s = self.step_i
        self.step_i += 1
        ev("prefill")
        self.q.copy_(h["q"], non_blocking=True)
        self.k.copy_(h["k"], non_blocking=True)
        self.v.copy_(h["v"], non_blocking=True)
        gq.attn_prefill(self.q, self.k, self.v, 0, self.scale, out=self.out, err=self.err)
        h["out"].copy_(self.out, non_blocking=True)
        ev("prompt_append")
        c0 = self.caches[(s * 6) % self.ncopy]
        gq.attn_kv_append(self.k[0], self.v[0], self.prompt_slots, c0, err=self.err)
        ev("decode")
        if getattr(self, "graphs_e2e", None):
            self.graphs_e2e[s % self.ncopy].replay()
        else:
            self._decode_part(s, e2e=True)
        ev("end")


class DecodeOnlyWorkload(Workload):
    """A decode step (append + decode) over rotating cache copies."""

    def __init__(self, dev, which, layout=0):
        import torch

        import gqa_attention_kv_gb300 as gq
        from gqa_attention_kv_gb300 import synth

        self.gq, self.torch = gq, torch
        self.fp8 = which.endswith("-fp8")
        which = which[:-4] if self.fp8 else which
        make = {"voxtral": synth.voxtral_decode_step, "ring": synth.ring_window_decode,
                "stream-encoder": synth.streaming_encoder_step,
                "paged": synth.paged_multirow_decode,
                "chunked": synth.chunked_prefill_step}[which]
        base = make(device=dev)
        self.case = base
        self.kv_elem = 1 if self.fp8 else 2
        rows = base.block_size if base.kind == synth.PAGED else base.slots_per_seq

        def placed(t):  # [S, H, D] -> the layout's shape (a pure reordering)
            if layout == 0:
                return t
            S, H, D = t.shape
            return t.reshape(S // rows, rows, H, D).permute(0, 2, 1, 3).contiguous()
        per_copy = 2 * base.k_cache.numel() * self.kv_elem
        self.ncopy = max(2, min(256, math.ceil(4 * _l2_bytes() / per_copy) + 1))
        g = synth.generator(777, dev)
        if self.fp8:
            # E4M3 caches (keys relative to the reference of the first 512
            # rows), written by the library's own FP8 append
            S, Hkv, D = base.k_cache.shape
            all_slots = torch.arange(S, dtype=torch.int64, device=dev)
            self.k_ref = gq.attn_kv_reference(base.k_cache[:512])
            self.caches = []
            for i in range(self.ncopy):
                kb = base.k_cache if i == 0 else synth.normal_bf16(g, base.k_cache.shape, dev)
                vb = base.v_cache if i == 0 else synth.normal_bf16(g, base.v_cache.shape, dev)
                c = gq.KVCache(base.kind,
                               placed(torch.empty(S, Hkv, D, dtype=torch.uint8, device=dev)),
                               placed(torch.empty(S, Hkv, D, dtype=torch.uint8, device=dev)),
                               slots_per_seq=base.slots_per_seq, block_table=base.block_table,
                               block_size=base.block_size, dtype=gq.ATTN_KV_FP8_E4M3,
                               k_ref=self.k_ref, layout=layout)
                gq.attn_kv_append(kb, vb, all_slots, c)
                self.caches.append(c)
                del kb, vb
            torch.cuda.synchronize()
        else:
            self.caches = [gq.KVCache(base.kind, placed(base.k_cache if i == 0 else
                                      synth.normal_bf16(g, base.k_cache.shape, dev)),
                                      placed(base.v_cache if i == 0 else
                                      synth.normal_bf16(g, base.v_cache.shape, dev)),
                                      slots_per_seq=base.slots_per_seq,
                                      block_table=base.block_table, block_size=base.block_size,
                                      layout=layout)
                           for i in range(self.ncopy)]
        self.max_seq = base.max_seq_len()
        self.ws = torch.zeros(gq.attn_decode_workspace_size(
            self.caches[0], base.batch, base.q_rows, base.n_q_heads, self.max_seq, base.window),
            dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(base.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.step_i = 0
        # the step's append fused into the decode launch (bf16 and FP8)
        self.launches_per_step = gq.attn_decode_kernel_launches(
            self.caches[0], base.batch, base.q_rows, base.n_q_heads, self.max_seq, base.window,
            with_append=True, tables_early=True)
        # valid keys per (request, row) summed over rows' union per request
        seq = base.seq_lens.cpu().tolist()
        keys = 0
        pairs = 0  # (query row, key) pairs attended, per query head
        for b, L in enumerate(seq):
            lo = 0
            pos = base.positions.cpu().view(base.batch, base.q_rows)[b]
            if base.window > 0:
                lo = max(lo, int(pos.min()) - base.window + 1)
            if base.kind == synth.RING:
                lo = max(lo, L - base.slots_per_seq)
            keys += L - lo
            for p_ in pos.tolist():
                lo_r = 0 if base.window <= 0 else max(0, p_ - base.window + 1)
                if base.kind == synth.RING:
                    lo_r = max(lo_r, L - base.slots_per_seq)
                pairs += p_ + 1 - lo_r
        self.keys = keys
        # 4 D Hq flops per (row, key) pair: the score and P V contractions
        self.chunk_flops = 4.0 * base.head_dim * base.n_q_heads * pairs
        # one step = one decode per decoder layer, each layer its own cache
        # (Voxtral decoder: 26 layers); bigger workloads: one layer per step
        self.layers = {"voxtral": 26, "stream-encoder": 32}.get(which, 1)
        self.launches_per_step *= self.layers
        self.name = {"voxtral": "voxtral decode step B=1 R=1 32/8 D=128 linear 512 keys, "
                                "26 layers",
                     "ring": "ring window decode B=16 32/8 D=128 ring 16384 window 8192",
                     "stream-encoder": "streaming encoder step, 4 frames over a 1500-slot ring, "
                                       "window 750, 32/32 D=64, 32 layers",
                     "paged": "paged K=4 decode 64x4 rows 32/8 D=128 bs 16",
                     "chunked": "chunked prefill: 2 requests x a 29-row chunk at positions "
                                "14420..14448 of a linear cache, 28/4 D=128"}[which]
        if self.fp8:
            self.name += ", FP8 (E4M3) cache"
        self.describe = {"workload": self.name, "decode_cache_copies": self.ncopy,
                         "layers_per_step": self.layers, "kv_cache": "fp8_e4m3" if self.fp8
                         else "bf16", "kv_layout": "BHSD" if layout else "BSHD",
                         "l2_defeat": "caches rotate over copies > 4x L2"}

    def decode_bytes_per_step(self):
        c = self.case
        return self.layers * decode_bytes(self.keys, c.n_kv_heads, c.head_dim, c.batch,
                                          c.q_rows, c.n_q_heads, c.batch * c.q_rows,
                                          self.kv_elem)

    def _decode_part(self, s):
        c = self.case
        for layer in range(self.layers):
            cache = self.caches[(s * self.layers + layer) % self.ncopy]
            self.gq.attn_decode_append(c.q, c.k_new, c.v_new, c.slot_mapping, cache,
                                       c.seq_lens, c.positions, self.max_seq, c.window,
                                       c.scale, out=self.out, workspace=self.ws,
                                       err=self.err, tables_early=True, cache_early=True)

    def capture(self, stream, e2e=False):
        torch = self.torch
        period = self.ncopy // math.gcd(self.ncopy, self.layers)
        self.graphs = []
        for r in range(period):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self._decode_part(r)
            self.graphs.append(g)
        torch.cuda.synchronize()

    def run_step(self, ev):
        s = self.step_i
        self.step_i += 1
        ev("decode")
        if getattr(self, "graphs", None):
            self.graphs[s % len(self.graphs)].replay()
        else:
            self._decode_part(s)
        ev("end")


class PrefillOnlyWorkload(Workload):
    """Prefill launches.  The speech encoder runs as its 32 layers per step,
    each layer its own q/k/v (the Voxtral notes' "Offline Encoder": 32
    layers), replayed from one CUDA graph; the Qwen-shaped prompts are one
    launch per step (a single launch of that size has no launch gap to hide)."""

    def __init__(self, dev, which):
        import torch

        import gqa_attention_kv_gb300 as gq
        from gqa_attention_kv_gb300 import synth

        self.gq, self.torch = gq, torch
        if which == "encoder":
            base = synth.encoder_prefill(device=dev)
        elif which == "encoder-long":
            base = synth.encoder_prefill(long=True, device=dev)
        elif which == "qwen-prefill":
            base = synth.qwen_prefill(device=dev)
        else:  # prefill-8k: the Qwen shape at 8,192 tokens (inputs + output > L2)
            base = synth.prefill_case(20263, 1, 8192, 28, 4, 128, device=dev)
        self.layers = 32 if which.startswith("encoder") else 1
        # one input set per layer: together far larger than the L2
        g = synth.generator(99, dev)
        self.inputs = [(base.q, base.k, base.v)] + [
            tuple(synth.normal_bf16(g, t.shape, dev) for t in (base.q, base.k, base.v))
            for _ in range(self.layers - 1)]
        self.window, self.scale = base.window, base.scale
        self.outs = [torch.empty_like(base.q) for _ in range(self.layers)]
        B, T, Hq, Hkv, D = base.shape
        self.T, self.Hq, self.D = T, Hq, D
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches_per_step = self.layers
        self.name = {"encoder": "encoder prefill T=750 32 heads D=64, 32 layers",
                     "encoder-long": "encoder prefill T=1500 window 750 32 heads D=64, 32 layers",
                     "qwen-prefill": "qwen2-7b prompt prefill T=14449 28/4 D=128",
                     "prefill-8k": "qwen2-7b-shaped prefill T=8192 28/4 D=128"}[which]
        self.describe = {"workload": self.name, "layers_per_step": self.layers,
                         "l2_defeat": "per-layer inputs together > L2" if self.layers > 1
                         else "inputs + output > L2"}

    def prefill_flops_per_step(self):
        return self.layers * prefill_flops(self.T, self.Hq, self.D, self.window)

    def _prefill_part(self):
        for (q, k, v), out in zip(self.inputs, self.outs):
            self.gq.attn_prefill(q, k, v, self.window, self.scale, out=out, err=self.err)

    def capture(self, stream, e2e=False):
        if self.layers == 1:
            return
        torch = self.torch
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self._prefill_part()
        torch.cuda.synchronize()

    def run_step(self, ev):
        ev("prefill")
        if getattr(self, "graph", None) is not None:
            self.graph.replay()
        else:
            self._prefill_part()
        ev("end")


def make_workload(name, dev, layout=0):
    if name == "qwen":
        return QwenWorkload(dev, layout)
    if name in ("voxtral", "ring", "paged", "stream-encoder", "ring-fp8", "paged-fp8",
                "voxtral-fp8", "chunked"):
        return DecodeOnlyWorkload(dev, name, layout)
    if name in ("encoder", "encoder-long", "qwen-prefill", "prefill-8k"):
        return PrefillOnlyWorkload(dev, name)
    raise SystemExit(f"unknown workload {name}")


# --------------------------------------------------------------------------
# timing
# --------------------------------------------------------------------------

def timed_steps(wl, steps, warmup, stream, e2e=False):
    """Run warmup + steps; return per-group summed ms over the timed steps and
    the total ms (events bracketing the timed region)."""
    import torch

    run = wl.run_step_e2e if e2e else wl.run_step
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run(lambda name: None)
    torch.cuda.synchronize()
    if hasattr(wl, "capture"):
        wl.capture(stream, e2e=e2e)
        with torch.cuda.stream(stream):
            run(lambda name: None)  # one replay before timing
        torch.cuda.synchronize()
    marks = []  # per step: list of (name, event)

    def ev_factory(lst):
        def ev(name):
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            lst.append((name, e))
        return ev

    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            lst = []
            marks.append(lst)
            run(ev_factory(lst))
        stop.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(stop)
    groups = {}
    for lst in marks:
        for (name, e0), (_, e1) in zip(lst[:-1], lst[1:]):
            groups[name] = groups.get(name, 0.0) + e0.elapsed_time(e1)
    return groups, total


def cpu_sample(workload_name, steps=1, warmup=0, budget_s=None, max_rows=160):
    """The oracle on a bounded sample of the workload, on the host cores.
    With budget_s, the prefill rows per step shrink so that warmup + steps
    samples take about budget_s seconds."""
    import numpy as np

    import oracle
    from gqa_attention_kv_gb300 import synth

    oracle.build()
    bits = oracle.bf16_bits
    res = {"cores": oracle.threads()}
    if workload_name == "qwen":
        # decode: both slots at the first context, the whole computation
        case = synth.qwen_decode((14449, 14449))
        kc, vc = bits(case.k_cache).copy(), bits(case.v_cache).copy()
        cd = {"kind": case.kind, "k": kc, "v": vc, "slots_per_seq": case.slots_per_seq}
        # prefill: 24 seeded query rows of the prompt (all 28 heads)
        p = synth.qwen_prefill()
        all_rows = np.random.default_rng(7).integers(0, p.q.shape[1], max_rows).astype(np.int32)
        pq, pk, pv = bits(p.q), bits(p.k), bits(p.v)
        dbytes = decode_bytes(sum((14449, 14449)), 4, 128, 2, 1, 28, 2)
        n_rows = max_rows
        if budget_s is not None:
            # calibrate: one decode and a prefill of 8 rows
            t0 = time.perf_counter()
            oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(), 0,
                          case.scale, 4)
            t1 = time.perf_counter()
            oracle.prefill(pq, pk, pv, 0, p.scale, rows=all_rows[:8])
            t2 = time.perf_counter()
            per_step = budget_s / max(1, steps + warmup)
            per_row = (t2 - t1) / 8
            n_rows = int(max(1, min(max_rows, (per_step - (t1 - t0)) / max(per_row, 1e-9))))
        rows = np.sort(all_rows[:n_rows])
        pflops = 4.0 * 128 * 28 * float(np.sum(rows.astype(np.int64) + 1))

        def one():
            t0 = time.perf_counter()
            oracle.kv_append(kc, vc, bits(case.k_new), bits(case.v_new), case.slot_mapping.numpy())
            oracle.decode(bits(case.q), cd, case.seq_lens.numpy(), case.positions.numpy(), 0,
                          case.scale, 4)
            t1 = time.perf_counter()
            oracle.prefill(pq, pk, pv, 0, p.scale, rows=rows)
            t2 = time.perf_counter()
            return t1 - t0, t2 - t1

        sample = ("decode: 2 slots x 1 row at context 14,449 (all 28 heads, whole "
                  f"computation); prefill: {len(rows)} seeded query rows x 28 heads of the "
                  "14,449-token prompt")
    else:
        raise SystemExit("cpu sample defined for the qwen workload only")
    for _ in range(warmup):
        one()
    td = tp = 0.0
    for _ in range(max(1, steps)):
        a, b = one()
        td += a
        tp += b
    n = max(1, steps)
    res.update({"decode_gbs": dbytes * n / td / 1e9, "prefill_tflops": pflops * n / tp / 1e12,
                "decode_s": td / n, "prefill_s": tp / n, "sample": sample})
    return res


# The other configurations of the path, measured after the headline step by
# the default run (fixed step counts: each timed region a fraction of a
# second).  name -> (what it is, steps)
SWEEP = [
    ("voxtral", "Voxtral decoder step: B=1, 1 row, 32/8, D=128, linear cache of 512 keys; "
                "26 layers per step", 1000),
    ("encoder", "speech-encoder causal prefill T=750, 32/32, D=64; 32 layers per step", 300),
    ("encoder-long", "speech-encoder prefill T=1500, window 750; 32 layers per step", 200),
    ("ring", "ring decode: ring 16,384, window 8,192, B=16, 32/8, D=128", 2000),
    ("paged", "paged K=4 decode: 64 x 4 rows, 32/8, D=128, block size 16", 2000),
    ("chunked", "prefill chunk: 2 requests x 29 rows at 14,420..14,448, 28/4, D=128", 2000),
    ("ring-fp8", "ring decode over an E4M3 cache", 2000),
    ("paged-fp8", "paged K=4 decode over an E4M3 cache", 2000),
    ("stream-encoder", "streaming encoder: 4 frames over a 1,500-slot ring, window 750, "
                       "32/32, D=64; 32 layers per step", 1000),
]


def launch_floor_us(stream, n=26, reps=200):
    """Per-launch time of n back-to-back one-element torch kernels replayed
    from a CUDA graph: the floor any launch of this size pays."""
    import torch

    x = torch.zeros(1, device=stream.device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        x.add_(1.0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                x.add_(1.0)
        for _ in range(5):
            g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (reps * n)


def measure_config(name, dev, stream, reps, peaks, peak_src, steps, layout=0):
    """One configuration of SWEEP: its own workload object, warm-up, graph
    capture and timed steps; returns its sub-object for the JSON line."""
    import torch

    wl = make_workload(name, dev, layout)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    reps.barrier()
    clocks.start()
    groups, total_ms = timed_steps(wl, steps, 3, stream)
    reps.barrier()
    clk = clocks.stop()
    err = int(wl.err.item())
    if err != 0:
        raise SystemExit(f"{name}: device error word {err}")
    dec_ms = reps.reduce_max(groups.get("decode", 0.0))
    pre_ms = reps.reduce_max(groups.get("prefill", 0.0))
    total_ms = reps.reduce_max(total_ms)
    world = reps.world
    out = {"workload": wl.name, "steps": steps, "ms_per_step": round(total_ms / steps, 5),
           "launches_per_step": wl.launches_per_step, "clocks": clk}
    if pre_ms > 0:
        fl = wl.prefill_flops_per_step()
        tf = fl / (pre_ms / steps / 1e3) / 1e12
        out.update({"value": round(world * tf, 2), "unit": "TFLOP/s", "flops_per_step": fl,
                    "bound": "tensor", "peak": peaks["bf16_tflops"],
                    "frac_of_measured_peak": round(tf / peaks["bf16_tflops"], 4),
                    "peak_source": f"{peak_src} bf16_tflops (burst)"})
    else:
        by = wl.decode_bytes_per_step()
        gbs = by / (dec_ms / steps / 1e3) / 1e9
        out.update({"value": round(world * gbs, 2), "unit": "GB/s", "bytes_per_step": int(by),
                    "bound": "hbm", "peak": peaks["hbm_gbs"],
                    "frac_of_measured_peak": round(gbs / peaks["hbm_gbs"], 4),
                    "frac_of_nominal_hbm": round(gbs / NOMINAL_HBM_GBS, 4),
                    "peak_source": f"{peak_src} hbm_gbs",
                    "us_per_launch": round(1e3 * dec_ms / steps / wl.launches_per_step, 3)})
        cf = getattr(wl, "chunk_flops", 0.0) * getattr(wl, "layers", 1)
        if name == "chunked" and cf:
            ctf = cf / (dec_ms / steps / 1e3) / 1e12
            out["chunk"] = {"value": round(world * ctf, 2), "unit": "TFLOP/s",
                            "flops_per_step": cf, "bound": "tensor",
                            "frac_of_measured_bf16": round(ctf / peaks["bf16_tflops"], 4)}
    if name == "voxtral":
        out["launch_floor_us"] = round(launch_floor_us(stream), 3)
        out["launch_floor"] = ("per-launch time of 26 one-element torch kernels replayed "
                               "from one CUDA graph, CUDA events")
    del wl
    torch.cuda.empty_cache()
    return out


def dist_env():
    """(rank, local_rank, world_size) as torchrun exports them (1 process: 0, 0, 1)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


class Replicas:
    """The N-GPU run: one process per GPU, each running the whole workload on
    its own GPU with nothing crossing between them (the decode and prefill
    units are independent, so the library has no exchange step; this is the
    only multi-GPU form the path has).  It supplies the bench's barrier, the
    max over ranks of each time, and the whole-job value: the units all ranks
    processed over the slowest rank's time."""

    def __init__(self, world, backend="nccl", device=None):
        self.world, self.device = world, device
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend)

    def barrier(self):
        import torch

        if self.world > 1:
            import torch.distributed as dist

            dist.barrier()
        if self.device is not None and self.device.type == "cuda":
            torch.cuda.synchronize()

    def reduce_max(self, x):
        if self.world == 1:
            return x
        import torch
        import torch.distributed as dist

        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def whole_job_rate(self, units_per_rank, seconds):
        """Aggregate throughput: every rank processed units_per_rank in at
        most `seconds` (already the max over ranks)."""
        return self.world * units_per_rank / seconds

    def close(self):
        if self.world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layout", default="bshd", choices=["bshd", "bhsd"],
                    help="decode cache layout: slot-major [slot, head, D] (the configured "
                         "one) or head-major blocks [block, head, rows, D]")
    ap.add_argument("--workload", default="qwen",
                    choices=["qwen", "voxtral", "encoder", "encoder-long", "ring", "paged",
                             "stream-encoder", "ring-fp8", "paged-fp8", "voxtral-fp8",
                             "qwen-prefill", "prefill-8k", "chunked"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="default workload only: skip the other configurations")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    rank, local_rank, world = dist_env()
    peaks, peak_src = load_peaks()
    metric = "decode-attn KV GB/s (% of HBM peak); prefill-attn TFLOP/s (% bf16 peak)"

    if args.impl == "reference":
        if rank != 0:
            return 0
        r = cpu_sample(args.workload, steps=args.steps, warmup=warmup, budget_s=150.0)
        line = {"impl": "reference", "metric": metric, "value": round(r["decode_gbs"], 4),
                "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
                "ms_per_step": round(1e3 * (r["decode_s"] + r["prefill_s"]), 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": QwenWorkload.name, "sample": r["sample"]},
                "prefill": {"value": round(r["prefill_tflops"], 6), "unit": "TFLOP/s"},
                "cpu_baseline": {"value": round(r["decode_gbs"], 4), "unit": "GB/s",
                                 "cores": r["cores"], "kind": "oracle", "sample": r["sample"],
                                 "prefill_tflops": round(r["prefill_tflops"], 6)},
                "e2e": {"value": round(r["decode_gbs"], 4), "unit": "GB/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch

    import gqa_attention_kv_gb300 as gq
    from gqa_attention_kv_gb300 import build

    build.build()
    gq.lib()
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    reps = Replicas(world, "nccl", dev)
    wl = make_workload(args.workload, dev, 1 if args.layout == "bhsd" else 0)
    stream = torch.cuda.Stream(device=dev)

    barrier = reps.barrier
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier()
    clocks.start()
    groups, total_ms = timed_steps(wl, args.steps, warmup, stream)
    barrier()
    clk = clocks.stop()
    err = int(wl.err.item())
    if err != 0:
        raise SystemExit(f"device error word {err} ({gq.attn_status_string(err)})")

    reduce_max = reps.reduce_max
    K = args.steps
    total_ms = reduce_max(total_ms)
    dec_ms = reduce_max(groups.get("decode", 0.0))
    pre_ms = reduce_max(groups.get("prefill", 0.0))
    app_ms = reduce_max(groups.get("prompt_append", 0.0))
    dbytes = wl.decode_bytes_per_step()
    pflops = wl.prefill_flops_per_step()
    dec_gbs = reps.whole_job_rate(dbytes * K, dec_ms / 1e3) / 1e9 if dec_ms > 0 else None
    pre_tf = reps.whole_job_rate(pflops * K, pre_ms / 1e3) / 1e12 if pre_ms > 0 else None

    e2e = None
    if not args.no_e2e and hasattr(wl, "run_step_e2e"):
        wl.setup_host()
        barrier()
        eg, etot = timed_steps(wl, K, warmup, stream, e2e=True)
        barrier()
        edec = reduce_max(eg.get("decode", 0.0))
        epre = reduce_max(eg.get("prefill", 0.0))
        e2e = {"value": round(world * dbytes * K / (edec / 1e3) / 1e9, 2), "unit": "GB/s",
               "prefill_tflops": round(world * pflops * K / (epre / 1e3) / 1e12, 2),
               "h2d_bytes_per_step": wl.h2d_prefill + wl.h2d_decode,
               "d2h_bytes_per_step": wl.d2h_prefill + wl.d2h_decode,
               "ms_per_step": round(reduce_max(etot) / K, 4)}

    sweep = None
    if args.workload == "qwen" and not args.no_sweep:
        sweep = {}
        for name, what, steps in SWEEP:
            sweep[name] = {"config": what} | measure_config(
                name, dev, stream, reps, peaks, peak_src, steps,
                1 if args.layout == "bhsd" else 0)

    if rank != 0:
        reps.close()
        return 0

    if pre_tf is not None:
        dominant = "prefill"
        ach = pflops / (pre_ms / K / 1e3) / 1e12
        # The prefill launches of a timed region of a second or more run back
        # to back under the power cap: their denominator is the sustained
        # dense bf16 rate measured the same way; a short region takes the burst.
        long_region = total_ms >= 1000.0
        peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
        roof = {"kernel": f"gqa::pre::prefill_kernel<{getattr(wl, 'D', 128)}>",
                "bound": "tensor",
                "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "frac_of_burst": round(ach / peaks["bf16_tflops"], 4),
                "traffic": prefill_traffic(getattr(wl, "T", None)),
                "traffic_unit": "DRAM bytes per launch (ncu)",
                "peak_source": f"{peak_src} bf16_tflops_sustained (timed region "
                               f"{total_ms / 1e3:.1f} s, back to back)" if long_region
                else f"{peak_src} bf16_tflops (burst)"}
    else:
        dominant = "decode"
        ach = dbytes / (dec_ms / K / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": "gqa::dec::decode_split_kernel", "bound": "hbm",
                "achieved": round(ach, 2), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": None,
                "peak_source": f"{peak_src} hbm_gbs"}
    line = {"metric": metric,
            "value": round(dec_gbs, 2) if dec_gbs is not None else round(pre_tf, 2),
            "unit": "GB/s" if dec_gbs is not None else "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": warmup,
            "ms_per_step": round(total_ms / K, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 cache, f16 mma" if getattr(wl, "fp8", False) else "bf16",
            "data": "synthetic",
            "config": dict(wl.describe) | {"parallelism": f"replicas x{world}" if world > 1
                                            else "single GPU"},
            "step_ms": {"prefill": round(pre_ms / K, 4), "prompt_append": round(app_ms / K, 4),
                        "decode": round(dec_ms / K, 4)},
            "roofline": roof, "gpu_launches": wl.launches_per_step * K, "clocks": clk}
    if dec_gbs is not None:
        dach = dbytes / (dec_ms / K / 1e3) / 1e9
        line["decode"] = {"value": round(dec_gbs, 2), "unit": "GB/s",
                          "bytes_per_step": int(dbytes),
                          "frac_of_measured_hbm": round(dach / peaks["hbm_gbs"], 4),
                          "frac_of_nominal_hbm": round(dach / NOMINAL_HBM_GBS, 4)}
    if pre_tf is not None:
        line["prefill"] = {"value": round(pre_tf, 2), "unit": "TFLOP/s",
                           "flops_per_step": pflops,
                           "frac_of_measured_bf16": round(pre_tf / world / peaks["bf16_tflops"], 4),
                           "frac_of_measured_bf16_sustained":
                               round(pre_tf / world / peaks["bf16_tflops_sustained"], 4)}
    if app_ms > 0 and hasattr(wl, "prompt_append_bytes"):
        # the prompt's 14,449 rows appended (K and V read from the prefill
        # inputs, written to their slots): an HBM-bound copy
        ab = wl.prompt_append_bytes()
        agbs = ab / (app_ms / K / 1e3) / 1e9
        line["append"] = {"value": round(world * agbs, 2), "unit": "GB/s", "bytes_per_step": ab,
                          "kernel": "gqa::kv_append_kernel",
                          "frac_of_measured_hbm": round(agbs / peaks["hbm_gbs"], 4)}
    if dec_gbs is not None and pre_tf is not None:
        line["roofline_decode"] = {"bound": "hbm", "achieved": line["decode"]["value"] / world,
                                   "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": line["decode"]["frac_of_measured_hbm"]}
    cflops = getattr(wl, "chunk_flops", 0.0) * getattr(wl, "layers", 1)
    if getattr(wl, "name", "").startswith("chunked") and dec_ms > 0:
        # a prefill chunk is a dense contraction (the tcgen05 chunk kernel):
        # its rate against the measured dense bf16 peak is the roofline
        ctf = cflops / (dec_ms / K / 1e3) / 1e12
        line["chunk"] = {"value": round(ctf * world, 2), "unit": "TFLOP/s",
                         "flops_per_step": cflops,
                         "frac_of_measured_bf16": round(ctf / peaks["bf16_tflops"], 4)}
        line["roofline"] = {"kernel": "gqa::chk::chunk_kernel<128> (+ append, merge)",
                            "bound": "tensor", "achieved": round(ctf, 2),
                            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": round(ctf / peaks["bf16_tflops"], 4), "traffic": None,
                            "peak_source": f"{peak_src} bf16_tflops (burst)"}
    if e2e is not None:
        line["e2e"] = e2e
    if sweep is not None:
        line["configs"] = sweep
    if world == 1 and not args.no_cpu_baseline and args.workload == "qwen":
        r = cpu_sample(args.workload, steps=1, warmup=0)
        line["cpu_baseline"] = {"value": round(r["decode_gbs"], 4), "unit": "GB/s",
                                "cores": r["cores"], "kind": "oracle", "sample": r["sample"],
                                "prefill_tflops": round(r["prefill_tflops"], 6)}
    print(json.dumps(line))
    reps.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
