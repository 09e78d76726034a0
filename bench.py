"""Benchmark of the paged KV-cache hot path on GB300.

One step is one pass of every timed call of the five synthetic workloads
(kvgen), in this order:
  fused_write        kv_fill_slots x4, kv_write_fused_k_norm_rope_bf16 and
                     kv_write_v_only of 4 x 1024 tokens (8 KV heads, head_dim 128)
  bf16_prefill       kv_fill_slots x64 and kv_write_bf16 of ~278.5k tokens
  bf16_decode        paged_decode_attn_bf16, 64 sequences of 512..8192, GQA 32:8
  fp8k_prefill       kv_fill_slots x128 and kv_write_fp8k of 128 x 32768 tokens
                     (16 launches of 262144 tokens)
  fp8k_decode_w0     paged_decode_attn_fp8k, 128 x 32768, no window
  fp8k_decode_w4096  the same with sliding_window 4096
  fp8k_mixed_decode  paged_decode_attn_fp8k, 256 sequences of 128..65536
                     (log-uniform), GQA 64:8, block_size 64, split-KV
Beside the step, and not in it ("next_rows"), with L2 flushed before each
launch: the FP8-output and the MRoPE variants of the fused K write on the
fused_write tokens; the FP8 K+V cache (kv_write_fp8 of the fp8k_long tokens,
paged_decode_attn_fp8 of fp8k_long at W = 0 and of fp8k_mixed); and chunked
prefill attention (paged_prefill_attn_bf16 over the bf16_gqa4 cache and
paged_prefill_attn_fp8k over the first 32 fp8k_mixed sequences, the last
min(256, L) positions of each sequence as causal queries), reported in
TFLOP/s against the measured BF16 tensor peak.
The headline value is the step's algorithmic HBM bytes (what each call must
read and write, counted per call below) divided by the step time, in GB/s;
each call's GB/s, tokens/s and fraction of the measured HBM copy rate are
reported beside it. Inputs are synthetic (kvgen, seeded), resident in HBM
before the timed region; the step moves ~57 GB, far more than L2, so no
call finds its inputs in L2 from the previous step.

--impl reference runs the CPU oracle (the reference arm of this benchmark) on
a bounded sample of the same workloads on the host cores.
"""
from __future__ import annotations

import argparse
import itertools
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode KV-read GB/s & cache-write tokens/s, % of GB300 HBM peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_BF16_TFLOPS = 1900.0  # one earlier GB300 measurement (burst)
FALLBACK_HBM_GBS = 6800.0


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001 - the file is optional
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense BF16 tensor peak (burst: the prefill calls are timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:  # noqa: BLE001 - the file is optional
        return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_flops(seq_lens, q_lens, window, num_q_heads, head_dim):
    """4 * Hq * D per attended (query, key) pair: QK^T and PV, 2 flops per MAC."""
    pairs = 0
    for L, n in zip(seq_lens, q_lens):
        for j in range(int(n)):
            P = int(L) - int(n) + j
            if P < 0:
                continue
            pairs += min(P + 1, window) if window else P + 1
    return 4 * num_q_heads * head_dim * pairs


# ---------------------------------------------------------------------------
# algorithmic bytes (what a call must move through HBM, per call)
# ---------------------------------------------------------------------------
def decode_bytes(seq_lens, window, num_kv_heads, head_dim, k_bytes, num_seqs, num_q_heads,
                 max_blocks_per_seq, v_bytes=2):
    att = 0
    for L in seq_lens:
        L = int(L)
        att += min(L, window) if window else L
    kv = att * num_kv_heads * head_dim * (k_bytes + v_bytes)
    q = num_seqs * num_q_heads * head_dim * 2
    out = num_seqs * num_q_heads * head_dim * 4
    return kv + q + out + num_seqs * 4


def write_bytes_per_token(row, k_out_bytes, v_out_bytes=2):
    # K in (bf16) + K out + V in (bf16) + V out + the slot (int64)
    return row * 2 + row * k_out_bytes + row * 2 + row * v_out_bytes + 8


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi clock and throttle-reason samples during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.device_index = device_index

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:  # noqa: BLE001 - clocks are best effort
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


WORKLOAD_OF_PART = {"fused_write": "fused", "bf16_prefill": "bf16_gqa4", "bf16_decode": "bf16_gqa4",
                    "fp8k_prefill": "fp8k_long", "fp8k_decode_w0": "fp8k_long", "fp8k_decode_w4096": "fp8k_long",
                    "fp8k_mixed_decode": "fp8k_mixed",
                    # calls timed beside the step
                    "fused_k_write_fp8": "fused", "fused_k_write_mrope": "fused",
                    "fp8_kv_prefill": "fp8k_long", "fp8_kv_decode_w0": "fp8k_long",
                    "fp8_kv_mixed_decode": "fp8k_mixed", "bf16_chunked_prefill": "bf16_gqa4",
                    "fp8k_chunked_prefill": "fp8k_mixed", "fp8_kv_chunked_prefill": "fp8k_mixed",
                    "fused_write_65536": "fused_stream", "fused_k_write_65536": "fused_stream",
                    "fused_k_write_fp8_65536": "fused_stream", "fused_k_write_mrope_65536": "fused_stream"}


class GpuStep:
    # workload sizes for --small (profiling captures): fewer sequences, the
    # same shapes otherwise; every input still exceeds L2
    SMALL = {"bf16_gqa4": dict(num_seqs=16), "fp8k_long": dict(num_seqs=4), "fp8k_mixed": dict(num_seqs=32)}

    def __init__(self, dev, only_part=None, small=False):
        import torch

        import kvgen
        import paged_kv_cache_fill_gb300 as pk
        self.torch, self.kvgen, self.pk, self.dev = torch, kvgen, pk, dev
        self.parts = []          # (name, fn, bytes, tokens, launches)
        self.ws = None
        self.only_part = only_part
        self.small = small
        self._setup()

    # -- helpers
    def _slots_calls(self, w, tables, slots):
        """One kv_fill_slots per sequence into `slots`: returns a callable that
        runs them all, the launch count, and the per-sequence callables (the
        graph capture spreads these over parallel branches)."""
        pk = self.pk
        lens = w.seq_lens.tolist()
        offs = [0]
        for L in lens:
            offs.append(offs[-1] + L)

        def one(s):
            def f():
                pk.kv_fill_slots(slots[offs[s]:offs[s + 1]], tables[s], 0, lens[s], w.block_size)
            return f
        each = [one(s) for s, L in enumerate(lens) if L > 0]

        def run():
            for f in each:
                f()
        run.each = each
        # what the fills move: an int64 slot per token written, an int32
        # table entry per block read
        run.bytes = sum(8 * L + 4 * (-(-L // w.block_size)) for L in lens)
        run.tokens = sum(lens)
        return run, len(each)

    def _setup(self):
        torch, pk = self.torch, self.pk
        t0 = time.time()
        self.ws_bytes = 0  # the workspace must fit every decode of the step
        self.inputs_h2d, self.outputs_d2h = [], []
        self.extras = []  # calls timed beside the step, not in it
        # Each workload is set up in a method of its own, so every closure
        # binds its own shapes and buffers.
        want = WORKLOAD_OF_PART[self.only_part] if self.only_part else None
        for name, setup in (("fused", self._setup_fused), ("fused_stream", self._setup_fused_stream),
                            ("bf16_gqa4", self._setup_bf16_gqa4),
                            ("fp8k_long", self._setup_fp8k_long), ("fp8k_mixed", self._setup_fp8k_mixed)):
            if want in (None, name):
                setup()
        if self.only_part:
            # a call beside the step keeps its workload's parts (they fill the
            # slots and caches it reads)
            if any(x["name"] == self.only_part for x in self.extras):
                self.extras = [x for x in self.extras if x["name"] == self.only_part]
            else:
                self.parts = [p for p in self.parts if p["name"] == self.only_part]
                self.extras = []
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.dev)
        pk.kv_set_decode_workspace(self.ws)
        torch.cuda.synchronize()
        self.setup_s = time.time() - t0
        self.fill_bytes = sum(p["fill_fn"].bytes for p in self.parts if "fill_fn" in p)
        self.fill_tokens = sum(p["fill_fn"].tokens for p in self.parts if "fill_fn" in p)
        self.fill_launches = sum(len(p["fills"]) for p in self.parts if "fills" in p)
        self.total_bytes = sum(p["bytes"] for p in self.parts) + self.fill_bytes
        self.launches = sum(p["launches"] for p in self.parts)

    def _setup_fused(self):
        torch, kvgen, pk, dev = self.torch, self.kvgen, self.pk, self.dev
        w = kvgen.fused_write(device=dev)
        H, D, bs, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_tokens
        tables = w.block_tables.to(dev)
        slots = torch.empty(n, dtype=torch.int64, device=dev)
        kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        fill, nfill = self._slots_calls(w, tables, slots)
        wt, pos = w.extra["k_norm_weight"].to(dev), w.positions.to(dev)
        key, value = w.key.contiguous(), w.value.contiguous()

        def k_write():
            pk.kv_write_fused_k_norm_rope_bf16(key, wt, pos, kc, slots, n, H, D, 128, bs, 1e-6, 1e6)

        def v_write():
            pk.kv_write_v_only(value, vc, slots, n, H, D, bs, H * D)

        def run():
            fill()
            k_write()
            v_write()
        # the K and V writes touch different pools: the graph runs them side by side
        self.parts.append(dict(name="fused_write", fn=run, fills=fill.each, fill_fn=fill, mains=[k_write, v_write],
                               tokens=n,
                               launches=nfill + 2,
                               bytes=n * (2048 + 2048 + 4 + 8 + 2048 + 2048 + 8), kind="write"))
        self.inputs_h2d += [key, value, pos, tables]

        # the two siblings of the fused K write, timed on the same tokens
        # outside the step: the FP8-output write (E4M3 pool, inv_scale as the
        # FP8-K decode's 1/k_scale) and the MRoPE write (t/h/w position streams)
        kc8 = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", dev)
        g = torch.Generator().manual_seed(2024)
        pos_h = torch.randint(0, 1 << 17, (n,), generator=g).to(torch.int32).to(dev)
        pos_w = torch.randint(0, 512, (n,), generator=g).to(torch.int32).to(dev)

        def k_write_fp8():
            pk.kv_write_fused_k_norm_rope_fp8(key, wt, pos, kc8, slots, n, H, D, 128, bs, 1e-6, 1e6, 448.0 / 6.0)

        def k_write_mrope():
            pk.kv_write_fused_k_norm_rope_bf16_mrope(key, wt, pos, pos_h, pos_w, kc, slots, n, H, D, 128, bs,
                                                     1e-6, 1e6)
        # per token: K read 2048, K write (1024 as E4M3, 2048 as BF16),
        # positions (4, or 3 x 4) and the slot (8)
        self.extras += [dict(name="fused_k_write_fp8", fn=k_write_fp8, tokens=n, bytes=n * (2048 + 1024 + 4 + 8)),
                        dict(name="fused_k_write_mrope", fn=k_write_mrope, tokens=n,
                             bytes=n * (2048 + 2048 + 12 + 8))]

    def _setup_fused_stream(self):
        """The fused K write and its siblings at a streaming size, beside the
        step: 64 sequences x 1024 tokens (65,536 tokens; 134 MB of K and
        134 MB of V rows in, the same out), the fused_write recipe otherwise.
        The slots are filled once, untimed."""
        torch, kvgen, pk, dev = self.torch, self.kvgen, self.pk, self.dev
        w = kvgen.fused_write(device=dev, seqs=64, tokens_per_seq=1024)
        H, D, bs, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_tokens
        tables = w.block_tables.to(dev)
        slots = torch.empty(n, dtype=torch.int64, device=dev)
        fill, _ = self._slots_calls(w, tables, slots)
        fill()
        kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        kc8 = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", dev)
        wt, pos = w.extra["k_norm_weight"].to(dev), w.positions.to(dev)
        key, value = w.key.contiguous(), w.value.contiguous()
        g = torch.Generator().manual_seed(2024)
        pos_h = torch.randint(0, 1 << 17, (n,), generator=g).to(torch.int32).to(dev)
        pos_w = torch.randint(0, 512, (n,), generator=g).to(torch.int32).to(dev)

        def k_write():
            pk.kv_write_fused_k_norm_rope_bf16(key, wt, pos, kc, slots, n, H, D, 128, bs, 1e-6, 1e6)

        def k_and_v_write():
            k_write()
            pk.kv_write_v_only(value, vc, slots, n, H, D, bs, H * D)

        def k_write_fp8():
            pk.kv_write_fused_k_norm_rope_fp8(key, wt, pos, kc8, slots, n, H, D, 128, bs, 1e-6, 1e6, 448.0 / 6.0)

        def k_write_mrope():
            pk.kv_write_fused_k_norm_rope_bf16_mrope(key, wt, pos, pos_h, pos_w, kc, slots, n, H, D, 128, bs,
                                                     1e-6, 1e6)
        self.extras += [dict(name="fused_write_65536", fn=k_and_v_write, tokens=n,
                             bytes=n * (2048 + 2048 + 4 + 8 + 2048 + 2048 + 8)),
                        dict(name="fused_k_write_65536", fn=k_write, tokens=n, bytes=n * (2048 + 2048 + 4 + 8)),
                        dict(name="fused_k_write_fp8_65536", fn=k_write_fp8, tokens=n,
                             bytes=n * (2048 + 1024 + 4 + 8)),
                        dict(name="fused_k_write_mrope_65536", fn=k_write_mrope, tokens=n,
                             bytes=n * (2048 + 2048 + 12 + 8))]

    def _setup_bf16_gqa4(self):
        torch, kvgen, pk, dev = self.torch, self.kvgen, self.pk, self.dev
        w = kvgen.bf16_gqa4(device=dev, **(self.SMALL['bf16_gqa4'] if self.small else {}))
        H, D, bs, Hq, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_tokens
        tables = w.block_tables.to(dev)
        slots = torch.empty(n, dtype=torch.int64, device=dev)
        kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        fill, nfill = self._slots_calls(w, tables, slots)
        key, value, q, lens = w.key, w.value, w.q, w.seq_lens.to(dev)
        out = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=dev)

        def prefill_main():
            pk.kv_write_bf16(key, value, kc, vc, slots, n, H, D, bs, H * D, H * D)

        def prefill():
            fill()
            prefill_main()

        def decode():
            pk.paged_decode_attn_bf16(q, kc, vc, out, tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs,
                                      w.inv_sqrt_d, Hq * D, 0)
        self.parts.append(dict(name="bf16_prefill", fn=prefill, fills=fill.each, fill_fn=fill, main=prefill_main,
                               tokens=n,
                               launches=nfill + 1,
                               bytes=n * write_bytes_per_token(H * D, 2), kind="write"))
        self.parts.append(dict(name="bf16_decode", fn=decode, tokens=w.num_seqs,
                               launches=1 + self._combine(w), kind="decode",
                               bytes=decode_bytes(w.seq_lens.tolist(), 0, H, D, 2, w.num_seqs, Hq,
                                                  w.max_blocks_per_seq)))
        self._grow_ws(w)
        self.inputs_h2d += [key, value, q, tables, lens]
        self.outputs_d2h += [out]

        # chunked prefill over the same cache, timed beside the step: each
        # sequence's last min(256, L) positions are its query tokens (causal)
        q_lens = [min(256, int(L)) for L in w.seq_lens.tolist()]
        qsl = torch.tensor([0] + list(itertools.accumulate(q_lens)), dtype=torch.int32, device=dev)
        n_q = sum(q_lens)
        g = torch.Generator(device="cpu").manual_seed(2025)
        qp = torch.randn((n_q, Hq * D), generator=g).to(torch.bfloat16).to(dev)
        outp = torch.empty((n_q, Hq, D), dtype=torch.float32, device=dev)

        def prefill_attn():
            pk.paged_prefill_attn_bf16(qp, kc, vc, outp, tables, lens, qsl, w.max_blocks_per_seq, w.num_seqs, n_q,
                                       Hq, H, D, bs, w.inv_sqrt_d, Hq * D, 0)
        self.extras.append(dict(name="bf16_chunked_prefill", fn=prefill_attn, tokens=n_q,
                                flops=prefill_flops(w.seq_lens.tolist(), q_lens, 0, Hq, D),
                                bytes=sum(int(L) for L in w.seq_lens.tolist()) * H * D * 4 + n_q * Hq * D * (2 + 4)))

    def _setup_fp8k_long(self):
        torch, kvgen, pk, dev = self.torch, self.kvgen, self.pk, self.dev
        w = kvgen.fp8k_long(device=dev, **(self.SMALL['fp8k_long'] if self.small else {}))
        H, D, bs, Hq, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_tokens
        tables = w.block_tables.to(dev)
        slots = torch.empty(n, dtype=torch.int64, device=dev)
        kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", dev)
        vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        fill, nfill = self._slots_calls(w, tables, slots)
        key, value, q, lens, k_scale = w.key, w.value, w.q, w.seq_lens.to(dev), w.k_scale
        chunk = 262144
        chunks = [(c, min(n, c + chunk)) for c in range(0, n, chunk)]

        def write_chunk(c0, c1):
            pk.kv_write_fp8k(key[c0:c1], value[c0:c1], kc, vc, slots[c0:c1], c1 - c0, H, D, bs, H * D, H * D,
                             k_scale)

        def prefill_main():
            for c0, c1 in chunks:
                write_chunk(c0, c1)

        def prefill():
            fill()
            prefill_main()

        def make_decode(win, out):
            def decode():
                pk.paged_decode_attn_fp8k(q, kc, vc, out, tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D,
                                          bs, w.inv_sqrt_d, k_scale, Hq * D, win)
            return decode
        self.fp8_chunks, self.fp8_write_chunk, self.fp8_row = chunks, write_chunk, H * D
        self.parts.append(dict(name="fp8k_prefill", fn=prefill, fills=fill.each, fill_fn=fill, main=prefill_main,
                               tokens=n,
                               launches=nfill + len(chunks),
                               bytes=n * write_bytes_per_token(H * D, 1), kind="write"))
        outs = []
        for win in (0, 4096):
            out = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=dev)
            outs.append(out)
            self.parts.append(dict(name=f"fp8k_decode_w{win}", fn=make_decode(win, out), tokens=w.num_seqs,
                                   launches=1 + self._combine(w), kind="decode",
                                   bytes=decode_bytes(w.seq_lens.tolist(), win, H, D, 1, w.num_seqs, Hq,
                                                      w.max_blocks_per_seq)))
        self._grow_ws(w)
        self.inputs_h2d += [key, value, q, tables, lens]
        self.outputs_d2h += outs

        # FP8 K and V, timed beside the step: the same tokens written with
        # kv_write_fp8 (the K codes are the ones above), then decoded (W = 0)
        vc8 = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", dev)
        v_scale = w.v_scale

        def fp8kv_prefill():
            for c0, c1 in chunks:
                pk.kv_write_fp8(key[c0:c1], value[c0:c1], kc, vc8, slots[c0:c1], c1 - c0, H, D, bs, k_scale,
                                v_scale, H * D, H * D)
        out8 = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=dev)

        def fp8kv_decode():
            pk.paged_decode_attn_fp8(q, kc, vc8, out8, tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs,
                                     w.inv_sqrt_d, k_scale, v_scale, Hq * D, 0)
        self.extras += [dict(name="fp8_kv_prefill", fn=fp8kv_prefill, tokens=n,
                             bytes=n * write_bytes_per_token(H * D, 1, 1)),
                        dict(name="fp8_kv_decode_w0", fn=fp8kv_decode, tokens=w.num_seqs,
                             bytes=decode_bytes(w.seq_lens.tolist(), 0, H, D, 1, w.num_seqs, Hq,
                                                w.max_blocks_per_seq, v_bytes=1))]

    def _setup_fp8k_mixed(self):
        torch, kvgen, pk, dev = self.torch, self.kvgen, self.pk, self.dev
        w = kvgen.fp8k_mixed(device=dev, **(self.SMALL['fp8k_mixed'] if self.small else {}))
        H, D, bs, Hq, n = w.num_kv_heads, w.head_dim, w.block_size, w.num_q_heads, w.num_tokens
        tables = w.block_tables.to(dev)
        slots = torch.empty(n, dtype=torch.int64, device=dev)
        kc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", dev)
        vc = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "bf16", dev)
        vc8 = kvgen.poisoned_pool(w.num_blocks, bs, H, D, "fp8", dev)   # FP8 V, for the FP8 K+V decode
        fill, _ = self._slots_calls(w, tables, slots)
        fill()
        chunk = 262144
        for c0 in range(0, n, chunk):   # the caches are written once, untimed
            c1 = min(n, c0 + chunk)
            pk.kv_write_fp8k(w.key[c0:c1], w.value[c0:c1], kc, vc, slots[c0:c1], c1 - c0, H, D, bs, H * D, H * D,
                             w.k_scale)
            pk.kv_write_fp8(w.key[c0:c1], w.value[c0:c1], kc, vc8, slots[c0:c1], c1 - c0, H, D, bs, w.k_scale,
                            w.v_scale, H * D, H * D)
        torch.cuda.synchronize()
        w.key = w.value = None
        q, lens, k_scale = w.q, w.seq_lens.to(dev), w.k_scale
        out = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=dev)

        def decode():
            pk.paged_decode_attn_fp8k(q, kc, vc, out, tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs,
                                      w.inv_sqrt_d, k_scale, Hq * D, 0)
        self.parts.append(dict(name="fp8k_mixed_decode", fn=decode, tokens=w.num_seqs,
                               launches=1 + self._combine(w), kind="decode",
                               bytes=decode_bytes(w.seq_lens.tolist(), 0, H, D, 1, w.num_seqs, Hq,
                                                  w.max_blocks_per_seq)))
        self._grow_ws(w)
        self.inputs_h2d += [q, tables, lens]
        self.outputs_d2h += [out]
        out8 = torch.empty((w.num_seqs, Hq, D), dtype=torch.float32, device=dev)
        v_scale = w.v_scale

        def fp8kv_decode():
            pk.paged_decode_attn_fp8(q, kc, vc8, out8, tables, lens, w.max_blocks_per_seq, w.num_seqs, Hq, H, D, bs,
                                     w.inv_sqrt_d, k_scale, v_scale, Hq * D, 0)
        self.extras.append(dict(name="fp8_kv_mixed_decode", fn=fp8kv_decode, tokens=w.num_seqs,
                                bytes=decode_bytes(w.seq_lens.tolist(), 0, H, D, 1, w.num_seqs, Hq,
                                                   w.max_blocks_per_seq, v_bytes=1)))

        # chunked prefill over the FP8-K cache of the first 32 sequences: the
        # last min(256, L) positions of each are its query tokens (causal)
        ns = min(32, w.num_seqs)
        q_lens = [min(256, int(L)) for L in w.seq_lens[:ns].tolist()]
        qsl = torch.tensor([0] + list(itertools.accumulate(q_lens)), dtype=torch.int32, device=dev)
        n_q = sum(q_lens)
        g = torch.Generator(device="cpu").manual_seed(2026)
        qp = torch.randn((n_q, Hq * D), generator=g).to(torch.bfloat16).to(dev)
        outp = torch.empty((n_q, Hq, D), dtype=torch.float32, device=dev)
        lens_p = lens[:ns].contiguous()
        tables_p = tables[:ns].contiguous()

        def prefill_attn():
            pk.paged_prefill_attn_fp8k(qp, kc, vc, outp, tables_p, lens_p, qsl, w.max_blocks_per_seq, ns, n_q, Hq,
                                       H, D, bs, w.inv_sqrt_d, k_scale, Hq * D, 0)
        self.extras.append(dict(name="fp8k_chunked_prefill", fn=prefill_attn, tokens=n_q,
                                flops=prefill_flops(w.seq_lens[:ns].tolist(), q_lens, 0, Hq, D),
                                bytes=sum(int(L) for L in w.seq_lens[:ns].tolist()) * H * D * 3
                                + n_q * Hq * D * (2 + 4)))

        # the same queries over the FP8 K and V cache
        outpq = torch.empty((n_q, Hq, D), dtype=torch.float32, device=dev)

        def fp8kv_prefill_attn():
            pk.paged_prefill_attn_fp8(qp, kc, vc8, outpq, tables_p, lens_p, qsl, w.max_blocks_per_seq, ns, n_q, Hq,
                                      H, D, bs, w.inv_sqrt_d, k_scale, v_scale, Hq * D, 0)
        self.extras.append(dict(name="fp8_kv_chunked_prefill", fn=fp8kv_prefill_attn, tokens=n_q,
                                flops=prefill_flops(w.seq_lens[:ns].tolist(), q_lens, 0, Hq, D),
                                bytes=sum(int(L) for L in w.seq_lens[:ns].tolist()) * H * D * 2
                                + n_q * Hq * D * (2 + 4)))

    def _grow_ws(self, w):
        self.ws_bytes = max(self.ws_bytes, self.pk.kv_decode_workspace_bytes(
            w.max_blocks_per_seq, w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size))

    @staticmethod
    def _combine(w):
        # the split-KV combine kernel runs when a sequence can span more than 8 tiles of 16 positions
        return 1 if w.max_blocks_per_seq * w.block_size > 8 * 16 else 0

    def capture(self, branches: int = 8):
        """Capture one step into a CUDA graph. Each part's per-sequence slot
        fills run on `branches` parallel side streams (independent kernels),
        joined before the part's write; everything else is in stream order."""
        torch = self.torch
        self.graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        side = [torch.cuda.Stream() for _ in range(branches)]
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(self.graph, stream=cap):
            for p in self.parts:
                fills = p.get("fills")
                if fills:
                    for i, st in enumerate(side):
                        st.wait_stream(cap)
                        with torch.cuda.stream(st):
                            for f in fills[i::branches]:
                                f()
                    for st in side:
                        cap.wait_stream(st)
                    mains = p.get("mains") or [p["main"]]
                    for i, f in enumerate(mains):
                        st = side[i]
                        st.wait_stream(cap)
                        with torch.cuda.stream(st):
                            f()
                    for st in side[:len(mains)]:
                        cap.wait_stream(st)
                else:
                    p["fn"]()
        torch.cuda.current_stream().wait_stream(cap)
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()

    def capture_twin(self):
        """A second graph of the same step over a second set of input and
        output buffers, so that one step's inputs can be copied in while the
        other's kernels run. Every call reads its tensors when it is made, so
        giving the input and output tensors other storage during the capture
        re-points it; the originals are restored afterwards. Returns the
        graph and, per original tensor id, its twin."""
        torch = self.torch
        seen, tensors = set(), []
        for t in self.inputs_h2d + self.outputs_d2h:
            if id(t) not in seen:
                seen.add(id(t))
                tensors.append(t)
        twins = [torch.empty_like(t) for t in tensors]
        keep = [torch.empty(0, dtype=t.dtype, device=t.device).set_(t) for t in tensors]
        first = self.graph
        try:
            for t, a in zip(tensors, twins):
                t.set_(a)
            self.capture()
            twin_graph = self.graph
        finally:
            self.graph = first
            for t, k in zip(tensors, keep):
                t.set_(k)
        return twin_graph, {id(t): a for t, a in zip(tensors, twins)}

    def run_step(self):
        for p in self.parts:
            p["fn"]()

    def time_calls(self, reps: int) -> dict:
        """Each part as the step runs it, from CUDA graphs of its own (so that
        no host launch gap enters the time): its per-sequence slot fills
        (together "slot_fill"), then its main calls, side by side where the
        step runs them so. Before every timed replay (outside the events) L2
        is flushed by reading a 256 MiB buffer (flush_l2), so no part finds
        its inputs in L2."""
        torch = self.torch
        scrub = l2_flush_buffer(torch, self.dev)
        side = [torch.cuda.Stream() for _ in range(8)]
        cap = torch.cuda.Stream()

        def graph_of(fns, parallel):
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=cap):
                if parallel and len(fns) > 1:
                    for i, f in enumerate(fns):
                        st = side[i % len(side)]
                        st.wait_stream(cap)
                        with torch.cuda.stream(st):
                            f()
                    for st in side[:len(fns)]:
                        cap.wait_stream(st)
                else:
                    for f in fns:
                        f()
            torch.cuda.current_stream().wait_stream(cap)
            return g

        graphs = []
        for p in self.parts:
            if "fill_fn" in p:
                graphs.append(("slot_fill", graph_of(p["fills"], True)))
                mains = p.get("mains") or [p["main"]]
                graphs.append((p["name"], graph_of(mains, True)))
            else:
                graphs.append((p["name"], graph_of([p["fn"]], False)))
        torch.cuda.synchronize()
        rec = []
        for _ in range(reps):
            for name, g in graphs:
                flush_l2(scrub)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                rec.append((name, a, b))
        torch.cuda.synchronize()
        out = {}
        for name, a, b in rec:
            out[name] = out.get(name, 0.0) + a.elapsed_time(b) / reps
        del graphs
        return out

    def time_extras(self, reps: int) -> dict:
        """Eager launches of the calls outside the step, CUDA events around
        each; a call's first run is untimed. Their inputs fit in L2, so L2 is
        flushed (flush_l2) before every timed launch, outside the events."""
        torch = self.torch
        scrub = l2_flush_buffer(torch, self.dev)
        out = {}
        for x in self.extras:
            x["fn"]()
            evs = []
            for i in range(reps):
                flush_l2(scrub)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                x["fn"]()
                b.record()
                evs.append((a, b))
            torch.cuda.synchronize()
            out[x["name"]] = sum(a.elapsed_time(b) for a, b in evs) / reps
        return out


def l2_flush_buffer(torch, dev):
    """A 256 MiB device buffer (twice L2's 129 MB) for flush_l2, written once."""
    buf = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    return buf.view(torch.int64)


def flush_l2(buf):
    """Evict everything from L2 by reading a buffer twice its size. A read
    leaves L2 holding clean lines of this buffer: the dirty lines of earlier
    work are written back here, before the timed region, rather than by the
    next timed call (rewriting the buffer instead would leave ~129 MB of
    dirty lines for that call to write back)."""
    buf.sum()


class Ranks:
    """One process per GPU (torchrun sets RANK / WORLD_SIZE / LOCAL_RANK).
    Each rank runs its own replica of the step (weak scaling: the work per
    GPU is fixed); the only collectives are the barriers around the timed
    region and the max of the per-rank step times, never the data path."""

    def __init__(self, backend: str | None = None):
        import torch
        import torch.distributed as dist
        self.dist = dist
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1 and not dist.is_initialized():
            dist.init_process_group(backend or ("nccl" if torch.cuda.is_available() else "gloo"))
        self.device = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")

    def barrier(self):
        import torch
        if self.world > 1:
            self.dist.barrier()
        if torch.cuda.is_available():
            torch.cuda.synchronize()

    def max(self, value: float) -> float:
        """The largest of the ranks' values (every rank gets it)."""
        if self.world == 1:
            return float(value)
        import torch
        t = torch.tensor([float(value)], dtype=torch.float64,
                         device=self.device if self.device.type == "cuda" and
                         self.dist.get_backend() == "nccl" else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1 and self.dist.is_initialized():
            self.dist.destroy_process_group()


def run_gpu(args):
    import torch

    ranks = Ranks()
    rank, world, local = ranks.rank, ranks.world, ranks.local
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_fill_gb300 as pk

    step = GpuStep(dev, args.part, args.small)
    stream = torch.cuda.current_stream()
    if args.part:
        # one part only, for profiling: warm-up, then `steps` runs, no report.
        # A call beside the step runs after one pass of its workload's parts.
        runs = [step.run_step]
        if step.extras:
            step.run_step()
            runs = [x["fn"] for x in step.extras]
        times = []
        for it in range(args.warmup + args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for f in runs:
                f()
            b.record(stream)
            if it >= args.warmup:
                times.append((a, b))
        torch.cuda.synchronize()
        assert pk.kv_get_device_error() == 0
        ms = sorted(a.elapsed_time(b) for a, b in times)
        # back-to-back runs, L2 not flushed: a quick look, not a bench figure
        print(json.dumps({"part": args.part, "runs": args.warmup + args.steps, "ok": True,
                          "ms_median_unflushed": round(ms[len(ms) // 2], 4) if ms else None}))
        return

    barrier = ranks.barrier

    for _ in range(args.warmup):
        step.run_step()
    barrier()
    assert pk.kv_get_device_error() == 0, "kernel fault bits set during warm-up"
    step.capture()
    for _ in range(args.warmup):
        step.replay()
    barrier()

    with Clocks(local) as clk:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            step.replay()
        t_end.record(stream)
        barrier()
    assert pk.kv_get_device_error() == 0, "kernel fault bits set during the timed steps"
    # per-call times: the same calls launched eagerly, CUDA events around each
    clocks = clk.summary()
    elapsed_ms = t_start.elapsed_time(t_end)
    ms_per_step = elapsed_ms / args.steps
    call_ms = step.time_calls(args.steps)
    ms_per_step = ranks.max(ms_per_step)  # the job is as slow as its slowest rank

    peak, peak_kind = measured_peak()
    value = step.total_bytes * world / (ms_per_step * 1e-3) / 1e9

    # per-launch timing of the dominant kernel
    dom = max(step.parts, key=lambda p: call_ms[p["name"]])
    roofline = dominant_roofline(step, dom, stream, peak, peak_kind, args)

    entries = [(p["name"], p["bytes"], p["tokens"], p["launches"] - len(p.get("fills", ())))
               for p in step.parts]
    entries.insert(0, ("slot_fill", step.fill_bytes, step.fill_tokens, step.fill_launches))
    parts = {}
    for name, nbytes, tokens, launches in entries:
        ms = call_ms[name]
        gbs = nbytes / (ms * 1e-3) / 1e9
        parts[name] = {"ms": round(ms, 4), "GB_per_s": round(gbs, 1),
                       "tokens_per_s": round(tokens / (ms * 1e-3), 1),
                       "frac_measured_hbm": round(gbs / peak, 4),
                       "frac_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                       "algorithmic_bytes": int(nbytes), "launches": launches}

    extra_ms = step.time_extras(args.steps)
    next_rows = {}
    tf_peak, tf_kind = measured_bf16_tflops()
    for x in step.extras:
        ms = extra_ms[x["name"]]
        gbs = x["bytes"] / (ms * 1e-3) / 1e9
        next_rows[x["name"]] = {"ms": round(ms, 4), "GB_per_s": round(gbs, 1),
                                "tokens_per_s": round(x["tokens"] / (ms * 1e-3), 1),
                                "frac_measured_hbm": round(gbs / peak, 4), "algorithmic_bytes": int(x["bytes"])}
        if "flops" in x:
            # a contraction: its roofline is the tensor pipe, not HBM
            tfs = x["flops"] / (ms * 1e-3) / 1e12
            next_rows[x["name"]].update({"bound": "tensor", "TFLOP_per_s": round(tfs, 1),
                                         "frac_of_bf16_peak": round(tfs / tf_peak, 4),
                                         "bf16_peak": tf_peak, "peak_kind": tf_kind,
                                         "algorithmic_flops": int(x["flops"])})

    e2e = run_e2e(step, args, dev, world)
    cpu = cpu_baseline(args) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16/e4m3 storage, fp32 compute",
            "data": "synthetic (kvgen, seeded), inputs resident in HBM",
            "config": bench_config(world),
            "algorithmic_bytes_per_step": int(step.total_bytes),
            "step_mode": "one CUDA-graph replay per step (the per-sequence slot fills run as 8 parallel graph "
                         "branches, the fused K and V-only writes side by side); per-call 'parts' timed "
                         "from CUDA-graph replays of each part alone with CUDA events, L2 scrubbed before "
                         "each, the 196 per-sequence kv_fill_slots launches together as slot_fill",
            "parts": parts,
            "next_rows": next_rows,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": step.launches * args.steps,
            "clocks": clocks,
            "setup_s": round(step.setup_s, 1),
        }
        print(json.dumps(line))
    ranks.close()


def dominant_roofline(step, dom, stream, peak, peak_kind, args):
    """Average launch duration of the dominant part's main kernel: CUDA events
    on the launching stream around back-to-back launches, divided by the
    number of launches."""
    import torch
    torch.cuda.synchronize()
    reps = max(args.steps, 3)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dom["name"] == "fp8k_prefill":
        # the 16 kv_write_fp8k launches of 262144 tokens each
        a.record(stream)
        for _ in range(reps):
            for c0, c1 in step.fp8_chunks:
                step.fp8_write_chunk(c0, c1)
        b.record(stream)
        torch.cuda.synchronize()
        launches = reps * len(step.fp8_chunks)
        per_launch = statistics.mean((c1 - c0) * write_bytes_per_token(step.fp8_row, 1) for c0, c1 in step.fp8_chunks)
        kernel = "kv_write_fp8k (write_fp8_kernel<4, false, true>)"
    else:
        a.record(stream)
        for _ in range(reps):
            (dom.get("main") or dom["fn"])()
        b.record(stream)
        torch.cuda.synchronize()
        launches = reps
        per_launch = dom["bytes"]
        kernel = f"{dom['name']} (decode_kernel + combine_kernel)"
    avg_ms = a.elapsed_time(b) / launches
    achieved = per_launch / (avg_ms * 1e-3) / 1e9
    traffic = profiled_traffic(dom["name"])
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": int(per_launch), "avg_launch_ms": round(avg_ms, 4),
            "launches_timed": launches, "traffic": traffic}


def profiled_traffic(part_name):
    """DRAM bytes per launch from the committed ncu summary of the current
    kernels (profiles/traffic.json), or None when there is none."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            return json.load(f).get(part_name)
    except Exception:  # noqa: BLE001 - optional file
        return None


def run_e2e(step, args, dev, world):
    """The same step through the public API with host buffers: every step
    copies its inputs from pinned host memory to the device, runs the calls
    and reads the outputs back. Two sets of device buffers (and a graph for
    each) let the next step's inputs cross the host link while the current
    step's kernels run; every step's copies still lie inside the timed
    region."""
    import torch
    host_in = [t.to("cpu").pin_memory() for t in step.inputs_h2d]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in step.outputs_d2h] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    twin_graph, twins = step.capture_twin()
    graphs = [step.graph, twin_graph]
    dev_in = [step.inputs_h2d, [twins[id(t)] for t in step.inputs_h2d]]
    dev_out = [step.outputs_d2h, [twins[id(t)] for t in step.outputs_d2h]]
    compute = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    steps = max(1, min(args.steps, 5))
    copy_marks = []  # (start, end) of every step's host->device copies, during the run

    def copy_in(k):
        b = k % 2
        if k >= 2:
            h2d_s.wait_event(done[b])  # step k - 2's kernels have read this set
        a = torch.cuda.Event(enable_timing=True)
        a.record(h2d_s)
        with torch.cuda.stream(h2d_s):
            for h, d in zip(host_in, dev_in[b]):
                d.copy_(h, non_blocking=True)
        in_ready[b].record(h2d_s)
        e = torch.cuda.Event(enable_timing=True)
        e.record(h2d_s)
        copy_marks.append((a, e))

    def run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(compute)
        h2d_s.wait_event(start)
        d2h_s.wait_event(start)
        copy_in(0)
        for k in range(n):
            b = k % 2
            if k + 1 < n:
                copy_in(k + 1)
            compute.wait_event(in_ready[b])
            graphs[b].replay()
            done[b].record(compute)
            d2h_s.wait_event(done[b])
            with torch.cuda.stream(d2h_s):
                for h, d in zip(host_out[b], dev_out[b]):
                    h.copy_(d, non_blocking=True)
        compute.wait_stream(h2d_s)
        compute.wait_stream(d2h_s)
        end.record(compute)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    def copies_alone():
        # the step's own pinned buffers, copied with no kernel running: the
        # floor of a step's time on this host (placement of the pinned pages
        # and other traffic on the host included)
        t = []
        for src, dst in ((host_in, dev_in[0]), (dev_out[0], host_out[0])):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(h2d_s)
            with torch.cuda.stream(h2d_s):
                for x, y in zip(src, dst):
                    y.copy_(x, non_blocking=True)
            b.record(h2d_s)
            b.synchronize()
            t.append(a.elapsed_time(b))
        return t

    run(2)  # warm-up: both graphs and both buffer sets
    copy_marks.clear()
    ms = run(steps) / steps
    # the host->device copies of each step as they ran beside the kernels
    h2d_run_ms = statistics.mean(a.elapsed_time(e) for a, e in copy_marks)
    alone = [copies_alone() for _ in range(2)]
    h2d_ms, d2h_ms = min(t[0] for t in alone), min(t[1] for t in alone)
    del twin_graph, twins
    link = host_link_gbs(compute)
    link.update(step_h2d_gbs=round(h2d / (h2d_ms * 1e-3) / 1e9, 1), step_d2h_gbs=round(d2h / (d2h_ms * 1e-3) / 1e9, 1),
                step_h2d_ms_alone=round(h2d_ms, 3), step_d2h_ms_alone=round(d2h_ms, 3),
                step_h2d_ms_during_run=round(h2d_run_ms, 3),
                step_h2d_gbs_during_run=round(h2d / (h2d_run_ms * 1e-3) / 1e9, 1))
    # the step cannot end before its inputs have crossed the host link and
    # its outputs have come back: the step's own copies bound the end-to-end
    # rate, at the fastest they were seen to run in this process (alone, or
    # beside the kernels: on a shared host the link's speed drifts, and the
    # copies alone, timed after the run, have been the slower of the two)
    link_ms = min(h2d_ms, h2d_run_ms) + d2h_ms
    bound = step.total_bytes * world / (link_ms * 1e-3) / 1e9
    value = step.total_bytes * world / (ms * 1e-3) / 1e9
    return {"value": round(value, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "pipelined": "the next step's inputs are copied in while a step runs (2 buffer sets)",
            "host_link": dict(link, bound_value=round(bound, 1), frac_of_bound=round(value / bound, 4))}


def host_link_gbs(stream, nbytes=1 << 30, reps=3):
    """Pinned host <-> device copy rate of this machine, one 1 GiB copy each way
    (best of `reps`): the link every end-to-end step's inputs cross."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=torch.cuda.current_device())
    out = {}
    for name, dst, src in (("h2d_gbs", d, h), ("d2h_gbs", h, d)):
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
        out[name] = round(nbytes / (best * 1e-3) / 1e9, 1)
    del h, d
    return out


# ---------------------------------------------------------------------------
# CPU oracle: the cpu_baseline leg and the reference arm
# ---------------------------------------------------------------------------
def oracle_sample(budget_s: float):
    """Time the oracle on a bounded sample of the workloads: the fused write of
    the first 256 tokens, the BF16 write of a few sequences, and decode of
    sampled (sequence, query head) pairs from each decode workload, until
    about `budget_s` of CPU time. Returns (algorithmic bytes, seconds,
    description)."""
    import numpy as np
    import torch

    import kvgen
    import oracle
    oracle.build()

    def u16(t):
        return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))

    done_bytes, elapsed, pieces = 0, 0.0, []
    # fused write, 256 tokens
    w = kvgen.fused_write(seqs=1, tokens_per_seq=256)
    H, D, bs = w.num_kv_heads, w.head_dim, w.block_size
    slots = oracle.fill_slots(w.block_tables[0].numpy(), 0, 256, bs)
    kc = np.zeros((w.num_blocks, bs, H, D), np.uint16)
    t = time.perf_counter()
    oracle.write_fused_k_norm_rope_bf16(u16(w.key), u16(w.extra["k_norm_weight"]), w.positions.numpy(), kc, slots,
                                        256, H, D, 128, bs, 1e-6, 1e6)
    oracle.write_v_only(u16(w.value), kc.copy(), slots, 256, H, D, bs, H * D)
    elapsed += time.perf_counter() - t
    done_bytes += 256 * 8216
    pieces.append("fused+v_only 256 tokens")

    # decode: sequences of the decode workloads, one query head each, rotating
    rng = np.random.default_rng(0)
    specs = [("bf16_gqa4", False, 0), ("fp8k_long", True, 0), ("fp8k_long", True, 4096), ("fp8k_mixed", True, 0)]
    made = {}
    n_dec = 0
    while elapsed < budget_s and n_dec < 20000:  # the time budget ends it; the cap only bounds a runaway
        name, fp8, win = specs[n_dec % len(specs)]
        if name not in made:
            gen = {"bf16_gqa4": lambda: kvgen.custom(1003, seq_lens=[4352], num_q_heads=32, num_kv_heads=8,
                                                     head_dim=128, block_size=16),
                   "fp8k_long": lambda: kvgen.custom(1004, seq_lens=[32768], num_q_heads=32, num_kv_heads=8,
                                                     head_dim=128, block_size=16, fp8=True),
                   "fp8k_mixed": lambda: kvgen.custom(1005, seq_lens=[10500], num_q_heads=64, num_kv_heads=8,
                                                      head_dim=128, block_size=64, fp8=True)}[name]
            ww = gen()
            Hh, Dd, bsz = ww.num_kv_heads, ww.head_dim, ww.block_size
            sl = oracle.fill_slots(ww.block_tables[0].numpy(), 0, int(ww.seq_lens[0]), bsz)
            vr = np.zeros((ww.num_blocks, bsz, Hh, Dd), np.uint16)
            if fp8:
                kr = np.zeros((ww.num_blocks, bsz, Hh, Dd), np.uint8)
                oracle.write_fp8k(u16(ww.key), u16(ww.value), kr, vr, sl, len(sl), Hh, Dd, bsz, Hh * Dd, Hh * Dd,
                                  ww.k_scale)
            else:
                kr = np.zeros((ww.num_blocks, bsz, Hh, Dd), np.uint16)
                oracle.write_bf16(u16(ww.key), u16(ww.value), kr, vr, sl, len(sl), Hh, Dd, bsz, Hh * Dd, Hh * Dd)
            made[name] = (ww, kr, vr)
        ww, kr, vr = made[name]
        h = int(rng.integers(ww.num_q_heads))
        t = time.perf_counter()
        oracle.decode_one(u16(ww.q), None if fp8 else kr, kr if fp8 else None, vr, ww.block_tables.numpy(),
                          ww.seq_lens.numpy(), ww.max_blocks_per_seq, ww.num_q_heads, ww.num_kv_heads,
                          ww.head_dim, ww.block_size, ww.inv_sqrt_d, ww.k_scale, ww.num_q_heads * ww.head_dim,
                          win, 0, h)
        elapsed += time.perf_counter() - t
        L = int(ww.seq_lens[0])
        att = min(L, win) if win else L
        # one query head's share of the decode's KV bytes (the whole group's
        # bytes are read once per KV head on the GPU; per query head here)
        done_bytes += att * ww.head_dim * ((1 if fp8 else 2) + 2)
        n_dec += 1
    pieces.append(f"{n_dec} single-(sequence, query head) decodes over lengths 4352/32768/4096-window/10500")
    return done_bytes, elapsed, "; ".join(pieces)


def cpu_baseline(args):
    nbytes, secs, what = oracle_sample(args.cpu_budget)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": what, "seconds": round(secs, 2)}


def bench_config(world: int) -> dict:
    """The workload both arms report: the GPU arm times it whole, the
    reference arm (the oracle) a bounded sample of it, named in its
    cpu_baseline."""
    return {"workload": "one pass of every timed call of the five paged-KV workloads "
                        "(fused_write, bf16_gqa4 prefill+decode, fp8k_long prefill+decode W=0/4096, "
                        "fp8k_mixed decode)",
            "l2": "inputs larger than L2 (129 MB): the step moves ~57 GB and no call's inputs stay in L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    vals = []
    for _ in range(args.warmup):
        oracle_sample(min(args.cpu_budget, 5.0))
    per_step = max(2.0, args.cpu_budget / max(args.steps, 1))
    what = ""
    t_total, b_total = 0.0, 0
    for _ in range(args.steps):
        nbytes, secs, what = oracle_sample(per_step)
        vals.append(nbytes / secs / 1e9)
        t_total += secs
        b_total += nbytes
    value = b_total / t_total / 1e9
    world = int(os.environ.get("WORLD_SIZE", "1"))
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_total / args.steps * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 compute (oracle)", "data": "synthetic (kvgen)",
            "impl": "reference",
            "config": bench_config(world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"rank 0 only, 1 CPU thread, per step: {what}"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true", help="with --part: fewer sequences (profiling captures)")
    ap.add_argument("--part", choices=sorted(WORKLOAD_OF_PART), default=None,
                    help="set up one workload and run one part only (for ncu captures); prints no bench line")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
