"""Benchmark of the paged-KV attention hot path on one GB300 (or N replicas under torchrun).

Headline (the JSON line's metric/value): paged decode attention, KV-read GB/s, on the
decode-only Qwen3-235B-like layer: 256 sequences, context U[2000, 3000], 64 query / 4 KV
heads, head_dim 128, block size 16, shuffled blocks in a pool 1.2x the need. One step is one
pass of the hot path over that batch: batch_classify_reorder, kv_cache_write of the 256 new
tokens, paged_decode_attn. value = KV bytes the decode reads / step time.

Also reported on the same line: the mixed-batch step (Llama-3.1-70B-like: 192 decode, 8 extend
x 512 over 4k-32k cached, 4 prefill of 2k-8k, random arrival order) in tokens/s; prefill and
long-context extend TFLOP/s; KV write + per-layer pack GB/s over 80 layers of a 10k-token
prompt; the roofline of the dominant kernel; and the CPU oracle timed on a bounded sample.

--impl reference times the CPU oracle itself (the only reference implementation of this
method) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch
import torch.distributed

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from pkv_workloads import gen  # noqa: E402

L2_FLUSH_BYTES = 512 << 20


HEADLINE_WORKLOAD = "qwen3-235b-like decode layer: 256 seqs ctx U[2000,3000] Hq64/Hkv4 D128 bs16 bf16; reorder+write+decode"


def headline_config(kv_bytes: int, ws: int) -> dict:
    """The workload description both arms (GPU and --impl reference) print, key for key."""
    return {"workload": HEADLINE_WORKLOAD, "kv_bytes_per_step": kv_bytes,
            "l2": "inputs larger than L2 (1.3 GB KV per step); between timed steps the GPU arm writes 512 MiB, then reads it back",
            "parallelism": f"replicas x{ws}"}


def _r(x, n=4):
    """x rounded to n significant digits (keeps the JSON line short)."""
    if x is None or not isinstance(x, (int, float)) or x == 0 or not math.isfinite(x):
        return x
    return float(f"{x:.{n}g}")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device="cpu") -> float:
    """The largest of every rank's x (the slowest replica sets the job's time); x itself when
    running alone. `device` is where the process group's backend takes tensors (cuda for
    NCCL, cpu for gloo)."""
    if ws <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_rate(units_per_rank: float, ws: int, step_ms: float) -> float:
    """Whole-job rate of ws replicas that each process units_per_rank per step, timed by the
    slowest one (step_ms already maxed over ranks): units per second."""
    return ws * units_per_rank / (step_ms * 1e-3)


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout_s: float = 5.0):
        """Wait until the sampler has printed its first line (nvidia-smi takes a moment to start)."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.02)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sust": p["bf16_tflops_sustained"],
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sust": 1700.0, "source": "fallback"}


# The source files each profiled kernel is compiled from (its .cu and the headers it includes).
KERNEL_SOURCES = {
    "paged_decode": ["decode.cu", "decode_shares.cuh", "common.cuh", "launch.h"],
    "mla_decode": ["mla_decode.cu", "decode_shares.cuh", "common.cuh", "softmax.cuh", "launch.h"],
}


def kernel_source_hash(names) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_attention_reshape_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    source of the kernel; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[key]
        if e.get("source_sha") != kernel_source_hash(KERNEL_SOURCES[kernel]):
            return None
        return e["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


class Timer:
    """Per-step CUDA-event timing on a stream, with an L2 flush between steps (not timed).

    The timed steps run with no event inside them (an event between two kernels adds its own
    latency and stops the second from launching early). Per-call times, when asked for, come
    from a second pass of the same steps with events around each call."""

    def __init__(self, stream, flush_buf):
        self.stream = stream
        self.flush_buf = flush_buf
        self.flush_acc = torch.empty((), dtype=flush_buf.dtype, device=flush_buf.device)
        self.ms = []

    def flush(self):
        """Write the 512 MiB buffer (evicting whatever the last step left in L2), then read it
        back: the read makes L2 write back the dirty lines the write left, so the next timed
        step does not pay for the flush's own write-backs."""
        with torch.cuda.stream(self.stream):
            self.flush_buf.add_(1)
            torch.sum(self.flush_buf, dim=0, out=self.flush_acc)

    def _pass(self, fn, steps, marked):
        ms, sec = [], {}
        for _ in range(steps):
            self.flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            marks = [] if marked else None
            e0.record(self.stream)
            fn(marks)
            e1.record(self.stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
            for name, a, b in marks or []:
                sec.setdefault(name, []).append(a.elapsed_time(b))
        return ms, sec

    def run(self, fn, steps, warmup, sections=True):
        for _ in range(warmup):
            self.flush()
            fn(None)
        torch.cuda.synchronize()
        self.ms, _ = self._pass(fn, steps, False)
        sec = self._pass(fn, steps, True)[1] if sections else {}
        return self.ms, sec


def mark(marks, name, stream, fn):
    """Run fn, recording events around it on `stream` when marks is a list."""
    if marks is None:
        return fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    r = fn()
    b.record(stream)
    marks.append((name, a, b))
    return r


# ---- workloads ----------------------------------------------------------------------------------

def decode_workload(pkv, dev, seed_off=0):
    cfg = dict(gen.DECODE_QWEN3)
    cfg["seed"] += seed_off
    b = gen.decode_batch(**cfg, device=dev)
    R = b.R
    meta = dict(cu_q=b.cu_q.to(dev), seq_lens=b.seq_lens.to(dev), block_tables=b.block_tables.to(dev),
                slot_mapping=b.slot_mapping.to(dev))
    maxs = max(b.seq_lens_list)
    kv_bytes = sum(b.seq_lens_list) * b.Hkv * b.D * 2 * 2
    other = (b.q.numel() * 2 * 2 + R * b.Hq * 4 + sum((s + 15) // 16 for s in b.seq_lens_list) * 4)
    ws_n = pkv.paged_decode_workspace_size(R, b.Hq, b.Hkv, b.D, maxs)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    out = torch.empty_like(b.q)
    lse = torch.empty((R, b.Hq), dtype=torch.float32, device=dev)
    perm = torch.empty(R, dtype=torch.int32, device=dev)
    bounds = torch.empty(4, dtype=torch.int32, device=dev)
    cu_r = torch.empty(R + 1, dtype=torch.int32, device=dev)
    return dict(b=b, meta=meta, maxs=maxs, kv_bytes=kv_bytes, alg_bytes=kv_bytes + other, ws=ws, out=out,
                lse=lse, perm=perm, bounds=bounds, cu_r=cu_r)


def decode_step(pkv, w, stream, marks=None, q=None, meta=None, k_new=None, v_new=None, out=None, lse=None):
    b = w["b"]
    meta = meta or w["meta"]
    q = b.q if q is None else q
    k_new = b.k_new if k_new is None else k_new
    v_new = b.v_new if v_new is None else v_new
    out = w["out"] if out is None else out
    lse = w["lse"] if lse is None else lse
    R = b.R
    pkv.batch_classify_reorder(meta["cu_q"], meta["seq_lens"], perm=w["perm"], bounds=w["bounds"],
                               cu_q_reordered=w["cu_r"], stream=stream)
    pkv.kv_cache_write(k_new, v_new, meta["slot_mapping"], b.k_cache, b.v_cache, stream=stream)
    reqs = pkv.Reqs(max_reqs=R, batch_reqs=R, order=w["perm"], bounds=w["bounds"], cls=pkv.CLASS_DECODE)
    mark(marks, "decode", stream, lambda: pkv.paged_decode_attn(
        q, b.k_cache, b.v_cache, meta["block_tables"], meta["seq_lens"], w["maxs"], cu_q=meta["cu_q"],
        reqs=reqs, scale=1.0 / math.sqrt(b.D), out=out, lse=lse, workspace=w["ws"], stream=stream))


def bench_decode(pkv, dev, stream, timer, steps, warmup, seed_off=0, hold_s=0.0, on_ready=None):
    """The headline step, timed whole; then the decode call alone (L2 flushed before each
    launch, events right around it) for the kernel's launch duration. on_ready runs once the
    workload is built; hold_s more seconds of the same step follow the timing, untimed, so the
    clock sampler sees the GPU under this load for longer than the timed steps last."""
    w = decode_workload(pkv, dev, seed_off)
    if on_ready is not None:
        on_ready()
    n0 = pkv.launch_count()
    ms, _ = timer.run(lambda m: decode_step(pkv, w, stream, m), steps, warmup, sections=False)
    launches = (pkv.launch_count() - n0) // (warmup + steps)
    t_end = time.perf_counter() + hold_s
    while time.perf_counter() < t_end:
        for _ in range(20):
            timer.flush()
            decode_step(pkv, w, stream, None)
        torch.cuda.synchronize()
    b, meta, R = w["b"], w["meta"], w["b"].R
    reqs = pkv.Reqs(max_reqs=R, batch_reqs=R, order=w["perm"], bounds=w["bounds"], cls=pkv.CLASS_DECODE)
    launch_ms, _ = timer.run(lambda m: pkv.paged_decode_attn(
        b.q, b.k_cache, b.v_cache, meta["block_tables"], meta["seq_lens"], w["maxs"], cu_q=meta["cu_q"], reqs=reqs,
        scale=1.0 / math.sqrt(b.D), out=w["out"], lse=w["lse"], workspace=w["ws"], stream=stream),
        max(steps, 20), warmup, sections=False)
    return w, ms, {"decode": launch_ms}, launches


def bench_tiny_decode(pkv, dev, stream, timer, steps, warmup):
    """The tiny paged decode (4 sequences, context U[16,200], Hq 8 / Hkv 2, D 64, a 64-block
    pool): one decode call, L2 flushed before it. Latency-bound; its GB/s is informational."""
    b = gen.decode_batch(**gen.TINY_DECODE, device=dev)
    maxs = max(b.seq_lens_list)
    kv = sum(b.seq_lens_list) * b.Hkv * b.D * 2 * 2
    out = torch.empty_like(b.q)
    lse = torch.empty((b.R, b.Hq), dtype=torch.float32, device=dev)
    ws_n = pkv.paged_decode_workspace_size(b.R, b.Hq, b.Hkv, b.D, maxs)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    meta = dict(cu_q=b.cu_q.to(dev), seq_lens=b.seq_lens.to(dev), block_tables=b.block_tables.to(dev))
    ms, _ = timer.run(lambda m: pkv.paged_decode_attn(
        b.q, b.k_cache, b.v_cache, meta["block_tables"], meta["seq_lens"], maxs, cu_q=meta["cu_q"],
        scale=1.0 / math.sqrt(b.D), out=out, lse=lse, workspace=ws, stream=stream), steps, warmup, sections=False)
    t = sorted(ms)[len(ms) // 2]
    return {"kv_bytes": kv, "launch_ms": t, "kv_gbs": kv / (t * 1e-3) / 1e9}


def bench_decode_fp8(pkv, dev, stream, timer, steps, warmup):
    """The headline step over an FP8 (E4M3) cache: same batch, caches holding codes (synthesised
    from the bf16 values with per-tensor scales), new tokens quantised by kv_cache_write."""
    w = decode_workload(pkv, dev)
    b, meta, R = w["b"], w["meta"], w["b"].R
    ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
    kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
    del b.k_cache, b.v_cache
    torch.cuda.empty_cache()
    kv_bytes = sum(b.seq_lens_list) * b.Hkv * b.D * 2
    other = b.q.numel() * 2 * 2 + R * b.Hq * 4 + sum((x + 15) // 16 for x in b.seq_lens_list) * 4
    reqs = pkv.Reqs(max_reqs=R, batch_reqs=R, order=w["perm"], bounds=w["bounds"], cls=pkv.CLASS_DECODE)
    scale = 1.0 / math.sqrt(b.D)

    def decode():
        pkv.paged_decode_attn(b.q, kc, vc, meta["block_tables"], meta["seq_lens"], w["maxs"], cu_q=meta["cu_q"],
                              reqs=reqs, scale=scale, out=w["out"], lse=w["lse"], workspace=w["ws"], stream=stream,
                              k_scale=ks, v_scale=vs)

    def step(marks):
        pkv.batch_classify_reorder(meta["cu_q"], meta["seq_lens"], perm=w["perm"], bounds=w["bounds"],
                                   cu_q_reordered=w["cu_r"], stream=stream)
        pkv.kv_cache_write(b.k_new, b.v_new, meta["slot_mapping"], kc, vc, stream=stream, k_scale=ks, v_scale=vs)
        decode()

    ms, _ = timer.run(step, steps, warmup, sections=False)
    launch_ms, _ = timer.run(lambda m: decode(), max(steps, 20), warmup, sections=False)
    step_ms = sum(ms) / len(ms)
    dec_ms = sum(launch_ms) / len(launch_ms)
    return dict(step_ms=step_ms, launch_ms=dec_ms, kv_bytes=kv_bytes, alg_bytes=kv_bytes + other, R=R)


def bench_mla(pkv, dev, stream, timer, steps, warmup, Hq=None):
    """Absorbed MLA decode, DeepSeek-R1-like layer under tensor parallelism 8 (16 query heads
    over a 576-wide latent, 128 requests at 10K-11K tokens); Hq = 128 gives the same layer on one
    GPU without tensor parallelism. Step = kv_cache_write of the new tokens' latent rows +
    mla_decode_attn."""
    cfg = dict(gen.MLA_DEEPSEEK_TP8)
    if Hq is not None:
        cfg["Hq"] = Hq
    b = gen.mla_batch(**cfg, device=dev)
    R, maxs = b.R, max(b.seq_lens_list)
    bt64 = b.block_tables.to(torch.int64)
    pos = (b.seq_lens.to(torch.int64) - 1)
    slots = bt64[torch.arange(R, device=dev), pos // 16] * 16 + pos % 16
    new_rows = gen.randn_bf16((R, 1, gen.MLA_DEEPSEEK_TP8["Dk"]), torch.Generator(device=dev).manual_seed(7), dev)
    out = torch.empty((R, b.Hq, gen.MLA_DV), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, b.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, pkv.mla_decode_workspace_size(R, b.Hq, maxs)), dtype=torch.uint8, device=dev)
    lat_bytes = sum(b.seq_lens_list) * b.Dk * 2
    other = b.q.numel() * 2 + out.numel() * 2 + lse.numel() * 4 + sum((x + 15) // 16 for x in b.seq_lens_list) * 4

    def decode():
        pkv.mla_decode_attn(b.q, b.latent, b.block_tables, b.seq_lens, maxs, gen.MLA_SCALE, out=out, lse=lse,
                            workspace=ws, stream=stream)

    def step(marks):
        pkv.kv_cache_write(new_rows, new_rows, slots, b.latent, b.latent, stream=stream)
        decode()

    ms, _ = timer.run(step, steps, warmup, sections=False)
    launch_ms, _ = timer.run(lambda m: decode(), max(steps, 20), warmup, sections=False)
    errs = pkv.device_errors(clear=True)
    step_ms = sum(ms) / len(ms)
    dec_ms = sum(launch_ms) / len(launch_ms)
    flops = 2.0 * sum(b.seq_lens_list) * b.Hq * (b.Dk + gen.MLA_DV)
    return dict(step_ms=step_ms, launch_ms=dec_ms, lat_bytes=lat_bytes, alg_bytes=lat_bytes + other, R=R,
                flops=flops, errors=errs)


def bench_decode_e2e(pkv, w, dev, stream, steps, warmup, timer):
    """The same step through the public API with host buffers: every input of the step (q, the
    new K/V, slot mapping, lengths, block tables) is copied from pinned host memory and out/lse
    read back, inside the timed region. As a serving engine would, the step stages its inputs
    in one pinned buffer and one device buffer (one host-to-device copy) and its outputs in one
    device buffer (one device-to-host copy); the library calls take views into them. The KV
    cache stays resident (it is the state of the server)."""
    b = w["b"]
    parts = [("q", b.q), ("k_new", b.k_new), ("v_new", b.v_new)] + [(k, v) for k, v in w["meta"].items()]

    def layout(tensors):
        offs, off = {}, 0
        for name, t in tensors:
            off = (off + 255) // 256 * 256
            offs[name] = (off, t.numel() * t.element_size())
            off += offs[name][1]
        return offs, off

    in_offs, in_bytes = layout(parts)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    for name, t in parts:
        o, n = in_offs[name]
        h_in[o:o + n].copy_(t.detach().contiguous().view(-1).view(torch.uint8).cpu())

    def view(buf, offs, name, like):
        o, n = offs[name]
        return buf[o:o + n].view(like.dtype).view(like.shape)

    dq, dk, dv = (view(d_in, in_offs, n, t) for n, t in parts[:3])
    dmeta = {k: view(d_in, in_offs, k, v) for k, v in w["meta"].items()}
    out_parts = [("out", w["out"]), ("lse", w["lse"])]
    out_offs, out_bytes = layout(out_parts)
    d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    h_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    dout, dlse = view(d_out, out_offs, "out", w["out"]), view(d_out, out_offs, "lse", w["lse"])
    h2d, d2h = in_bytes, out_bytes

    def step():
        with torch.cuda.stream(stream):
            d_in.copy_(h_in, non_blocking=True)
        decode_step(pkv, w, stream, None, q=dq, meta=dmeta, k_new=dk, v_new=dv, out=dout, lse=dlse)
        with torch.cuda.stream(stream):
            h_out.copy_(d_out, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        timer.flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return ms, h2d, d2h


def bench_decode_e2e_pipelined(pkv, w, dev, stream, steps, warmup):
    """The end-to-end step as a serving engine with asynchronous scheduling runs it: every step
    still copies all of its inputs from pinned host memory and reads its out/lse back, but the
    copies run on their own streams into double buffers, so step i+1's inputs travel while step
    i computes and step i's results travel while step i+1 computes. Returns the device time of
    the whole run of `steps` steps (first host-to-device copy to last device-to-host copy)
    divided by `steps`. No L2 flush inside the run: each step reads 1.3 GB of KV, far more than
    L2."""
    b = w["b"]
    parts = [("q", b.q), ("k_new", b.k_new), ("v_new", b.v_new)] + [(k, v) for k, v in w["meta"].items()]
    out_parts = [("out", w["out"]), ("lse", w["lse"])]

    def layout(tensors):
        offs, off = {}, 0
        for name, t in tensors:
            off = (off + 255) // 256 * 256
            offs[name] = (off, t.numel() * t.element_size())
            off += offs[name][1]
        return offs, off

    def view(buf, offs, name, like):
        o, n = offs[name]
        return buf[o:o + n].view(like.dtype).view(like.shape)

    in_offs, in_bytes = layout(parts)
    out_offs, out_bytes = layout(out_parts)
    sets = []
    for _ in range(2):
        h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        for name, t in parts:
            o, n = in_offs[name]
            h_in[o:o + n].copy_(t.detach().contiguous().view(-1).view(torch.uint8).cpu())
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        h_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
        sets.append(dict(h_in=h_in, d_in=d_in, d_out=d_out, h_out=h_out,
                         q=view(d_in, in_offs, "q", b.q), k=view(d_in, in_offs, "k_new", b.k_new),
                         v=view(d_in, in_offs, "v_new", b.v_new),
                         meta={k: view(d_in, in_offs, k, v) for k, v in w["meta"].items()},
                         out=view(d_out, out_offs, "out", w["out"]), lse=view(d_out, out_offs, "lse", w["lse"])))
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def run(n):
        in_ready, computed, read_back = [], [], []
        for i in range(n):
            st = sets[i % 2]
            ev_in, ev_c, ev_out = (torch.cuda.Event() for _ in range(3))
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(computed[i - 2])  # step i-2 has finished reading this input buffer
                st["d_in"].copy_(st["h_in"], non_blocking=True)
                ev_in.record(h2d_s)
            stream.wait_event(ev_in)
            if i >= 2:
                stream.wait_event(read_back[i - 2])  # step i-2's results have left this output buffer
            decode_step(pkv, w, stream, None, q=st["q"], meta=st["meta"], k_new=st["k"], v_new=st["v"],
                        out=st["out"], lse=st["lse"])
            ev_c.record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_c)
                st["h_out"].copy_(st["d_out"], non_blocking=True)
                ev_out.record(d2h_s)
            in_ready.append(ev_in)
            computed.append(ev_c)
            read_back.append(ev_out)
        return read_back[-1]

    run(max(warmup, 2))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    stream.wait_event(e0)
    d2h_s.wait_event(e0)
    last = run(steps)
    d2h_s.wait_event(last)
    e1.record(d2h_s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, in_bytes, out_bytes


def mixed_workload(dev):
    b = gen.mixed_batch(**gen.MIXED_LLAMA70B, device=dev)
    return b


def bench_mixed(pkv, dev, stream, timer, steps, warmup):
    b = mixed_workload(dev)
    g = b
    R, T = b.R, b.T
    meta = dict(cu_q=b.cu_q.to(dev), seq_lens=b.seq_lens.to(dev), block_tables=b.block_tables.to(dev),
                slot_mapping=b.slot_mapping.to(dev))
    perm = torch.empty(R, dtype=torch.int32, device=dev)
    bounds = torch.empty(4, dtype=torch.int32, device=dev)
    cu_r = torch.empty(R + 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(b.q)
    lse = torch.empty((T, b.Hq), dtype=torch.float32, device=dev)
    kinds = b.kinds
    # host-side bounds the scheduler knows: class sizes and maxima per class
    n_dec = sum(k == gen.DECODE for k in kinds)
    n_ext = sum(k == gen.EXTEND for k in kinds)
    n_pre = sum(k == gen.PREFILL for k in kinds)
    max_dec = max(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.DECODE)
    max_ext_q = max(q for k, q in zip(kinds, b.q_lens) if k == gen.EXTEND)
    max_ext_s = max(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.EXTEND)
    max_pre = max(q for k, q in zip(kinds, b.q_lens) if k == gen.PREFILL)
    ws_n = pkv.paged_decode_workspace_size(n_dec, b.Hq, b.Hkv, b.D, max_dec)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(b.D)

    def step(marks):
        mark(marks, "reorder", stream, lambda: pkv.batch_classify_reorder(
            meta["cu_q"], meta["seq_lens"], perm=perm, bounds=bounds, cu_q_reordered=cu_r, stream=stream))
        mark(marks, "write", stream, lambda: pkv.kv_cache_write(
            g.k_new, g.v_new, meta["slot_mapping"], g.k_cache, g.v_cache, stream=stream))
        mark(marks, "decode", stream, lambda: pkv.paged_decode_attn(
            g.q, g.k_cache, g.v_cache, meta["block_tables"], meta["seq_lens"], max_dec, cu_q=meta["cu_q"],
            reqs=pkv.Reqs(n_dec, R, perm, bounds, pkv.CLASS_DECODE), scale=scale, out=out, lse=lse,
            workspace=ws, stream=stream))
        mark(marks, "extend", stream, lambda: pkv.extend_attn(
            g.q, g.k_new, g.v_new, meta["cu_q"], meta["seq_lens"], g.k_cache, g.v_cache,
            meta["block_tables"], max_ext_q, max_ext_s, reqs=pkv.Reqs(n_ext, R, perm, bounds, pkv.CLASS_EXTEND),
            chunk_budget_tokens=32768, scale=scale, out=out, lse=lse, stream=stream))
        mark(marks, "prefill", stream, lambda: pkv.varlen_prefill_attn(
            g.q, g.k_new, g.v_new, meta["cu_q"], max_pre, reqs=pkv.Reqs(n_pre, R, perm, bounds, pkv.CLASS_PREFILL),
            scale=scale, out=out, lse=lse, stream=stream))

    n0 = pkv.launch_count()
    ms, sec = timer.run(step, steps, warmup)
    launches = (pkv.launch_count() - n0) // (warmup + 2 * steps)  # warm-up, timed and marked passes

    # the unified variant for comparison: reorder-free, the whole batch in arrival order through
    # one extend_attn call (decode = one new token, prefill = no cached tokens)
    max_q, max_s = max(b.q_lens), max(b.seq_lens_list)

    def unified(marks):
        pkv.kv_cache_write(g.k_new, g.v_new, meta["slot_mapping"], g.k_cache, g.v_cache, stream=stream)
        pkv.extend_attn(g.q, g.k_new, g.v_new, meta["cu_q"], meta["seq_lens"], g.k_cache, g.v_cache,
                        meta["block_tables"], max_q, max_s, reqs=pkv.Reqs(R, R), chunk_budget_tokens=32768,
                        scale=scale, out=out, lse=lse, stream=stream)

    ums, _ = timer.run(unified, steps, warmup, sections=False)
    dec_bytes = sum(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.DECODE) * b.Hkv * b.D * 4
    ext_flops = sum(4 * b.Hq * b.D * (q * (s - q) + q * (q + 1) // 2)
                    for k, q, s in zip(kinds, b.q_lens, b.seq_lens_list) if k == gen.EXTEND)
    pre_flops = sum(4 * b.Hq * b.D * q * (q + 1) // 2 for k, q in zip(kinds, b.q_lens) if k == gen.PREFILL)
    return dict(b=b, ms=ms, sec=sec, launches=launches, tokens=T, dec_bytes=dec_bytes, unified_ms=ums,
                ext_flops=ext_flops, pre_flops=pre_flops)


def bench_mixed_fp8(pkv, dev, stream, timer, steps, warmup):
    """The mixed step over an FP8 (E4M3) cache: quantising write, decode dequantising as it
    reads, extend converting the context's codes in the kernel (head_dim 128: no workspace),
    prefill (no cache)."""
    b = mixed_workload(dev)
    R, T = b.R, b.T
    ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
    kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
    del b.k_cache, b.v_cache
    torch.cuda.empty_cache()
    meta = dict(cu_q=b.cu_q.to(dev), seq_lens=b.seq_lens.to(dev), block_tables=b.block_tables.to(dev),
                slot_mapping=b.slot_mapping.to(dev))
    perm = torch.empty(R, dtype=torch.int32, device=dev)
    bounds = torch.empty(4, dtype=torch.int32, device=dev)
    out = torch.empty_like(b.q)
    lse = torch.empty((T, b.Hq), dtype=torch.float32, device=dev)
    kinds = b.kinds
    n_dec = sum(k == gen.DECODE for k in kinds)
    n_ext = sum(k == gen.EXTEND for k in kinds)
    n_pre = sum(k == gen.PREFILL for k in kinds)
    max_dec = max(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.DECODE)
    max_ext_q = max(q for k, q in zip(kinds, b.q_lens) if k == gen.EXTEND)
    max_ext_s = max(s for k, s in zip(kinds, b.seq_lens_list) if k == gen.EXTEND)
    max_pre = max(q for k, q in zip(kinds, b.q_lens) if k == gen.PREFILL)
    ws = torch.empty(max(pkv.paged_decode_workspace_size(n_dec, b.Hq, b.Hkv, b.D, max_dec), 16), dtype=torch.uint8,
                     device=dev)
    ews = torch.empty(max(pkv.extend_fp8_workspace_size(n_ext, R, max_ext_s, b.block_tables.shape[1], b.Hkv, b.D), 16),
                      dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(b.D)

    def step(marks):
        mark(marks, "reorder", stream, lambda: pkv.batch_classify_reorder(
            meta["cu_q"], meta["seq_lens"], perm=perm, bounds=bounds, stream=stream))
        mark(marks, "write", stream, lambda: pkv.kv_cache_write(
            b.k_new, b.v_new, meta["slot_mapping"], kc, vc, stream=stream, k_scale=ks, v_scale=vs))
        mark(marks, "decode", stream, lambda: pkv.paged_decode_attn(
            b.q, kc, vc, meta["block_tables"], meta["seq_lens"], max_dec, cu_q=meta["cu_q"],
            reqs=pkv.Reqs(n_dec, R, perm, bounds, pkv.CLASS_DECODE), scale=scale, out=out, lse=lse,
            workspace=ws, stream=stream, k_scale=ks, v_scale=vs))
        mark(marks, "extend", stream, lambda: pkv.extend_attn(
            b.q, b.k_new, b.v_new, meta["cu_q"], meta["seq_lens"], kc, vc, meta["block_tables"], max_ext_q,
            max_ext_s, reqs=pkv.Reqs(n_ext, R, perm, bounds, pkv.CLASS_EXTEND), scale=scale, out=out, lse=lse,
            stream=stream, k_scale=ks, v_scale=vs, workspace=ews))
        mark(marks, "prefill", stream, lambda: pkv.varlen_prefill_attn(
            b.q, b.k_new, b.v_new, meta["cu_q"], max_pre, reqs=pkv.Reqs(n_pre, R, perm, bounds, pkv.CLASS_PREFILL),
            scale=scale, out=out, lse=lse, stream=stream))

    ms, sec = timer.run(step, steps, warmup)
    errs = pkv.device_errors(clear=True)
    return dict(ms=ms, sec=sec, tokens=T, errors=errs, ws_bytes=ews.numel())


def bench_attention_only(pkv, dev, stream, timer, steps, warmup, kind):
    """Prefill 4 x 8192 or the long-context extend (2 x (100k cached + 2048 new))."""
    if kind == "prefill":
        b = gen.prefill_batch([8192] * 4, Hq=64, Hkv=8, D=128, seed=5, device=dev)
        flops = sum(4 * b.Hq * b.D * q * (q + 1) // 2 for q in b.q_lens)
    else:
        b = gen.extend_batch(**gen.LONG_EXTEND, device=dev)
        flops = sum(4 * b.Hq * b.D * (q * (s - q) + q * (q + 1) // 2) for q, s in zip(b.q_lens, b.seq_lens_list))
    out = torch.empty_like(b.q)
    lse = torch.empty((b.T, b.Hq), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(b.D)
    meta = dict(cu_q=b.cu_q.to(dev), seq_lens=b.seq_lens.to(dev), block_tables=b.block_tables.to(dev))

    def step(marks):
        if kind == "prefill":
            mark(marks, kind, stream, lambda: pkv.varlen_prefill_attn(
                b.q, b.k_new, b.v_new, meta["cu_q"], max(b.q_lens), scale=scale, out=out, lse=lse, stream=stream))
        else:
            mark(marks, kind, stream, lambda: pkv.extend_attn(
                b.q, b.k_new, b.v_new, meta["cu_q"], meta["seq_lens"], b.k_cache, b.v_cache,
                meta["block_tables"], max(b.q_lens), max(b.seq_lens_list), chunk_budget_tokens=32768,
                scale=scale, out=out, lse=lse, stream=stream))

    ms, sec = timer.run(step, steps, warmup)
    return dict(ms=ms, sec=sec, flops=flops)


def bench_write_pack(pkv, dev, stream, timer, steps, warmup):
    """80 layers: write each layer's prompt K/V into its cache, pack each layer's blocks into
    its own staging buffer, and land each staging buffer in its own receiving pool at shuffled
    block ids. Every launch touches buffers of its own, so no layer's data is still in L2
    when a later launch reads it (the 80 layers hold about 16 GB)."""
    layers = gen.write_pack_layers(**gen.WRITE_PACK_LLAMA70B, device=dev)
    L0 = layers[0]
    nblk = L0.block_ids.numel()
    shape = (2, nblk) + tuple(L0.k_cache.shape[1:])
    dsts = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in layers]
    g = torch.Generator().manual_seed(10)
    recv_nb = L0.k_cache.shape[0]
    recv = [(torch.empty_like(L0.k_cache), torch.empty_like(L0.v_cache),
             torch.randperm(recv_nb, generator=g)[:nblk].to(torch.int32).to(dev)) for _ in layers]
    row_bytes = L0.key.numel() * 2
    write_bytes = len(layers) * (2 * row_bytes * 2 + L0.slot_mapping.numel() * 8)   # read + write, K and V
    pack_bytes = len(layers) * (2 * dsts[0].numel() * 2 + nblk * 4)   # read + write
    unpack_bytes = pack_bytes

    def step(marks):
        def w():
            for L in layers:
                pkv.kv_cache_write(L.key, L.value, L.slot_mapping, L.k_cache, L.v_cache, stream=stream)

        def p():
            for L, d in zip(layers, dsts):
                pkv.kv_block_pack(L.k_cache, L.v_cache, L.block_ids, dst=d, stream=stream)

        def u():
            for d, (rk, rv, ids) in zip(dsts, recv):
                pkv.kv_block_unpack(d, ids, rk, rv, stream=stream)
        mark(marks, "write", stream, w)
        mark(marks, "pack", stream, p)
        mark(marks, "unpack", stream, u)

    ms, sec = timer.run(step, steps, warmup)
    del layers, dsts, recv
    return dict(ms=ms, sec=sec, write_bytes=write_bytes, pack_bytes=pack_bytes, unpack_bytes=unpack_bytes)


def bench_handoff(pkv, dev, stream, timer, steps, warmup):
    """A prefill instance's layers with the per-layer KV handoff (vLLM blog "moriio-kv-connector",
    "Write mode"): for each of 80 Llama-3.1-70B-like layers, the 10,000-token prompt's K/V is
    written into the layer's cache and the layer's causal prefill attention (Hq 64 / Hkv 8) runs,
    on the bench stream; the layer's blocks are packed into a staging buffer of their own either
    on the same stream after the attention (serial) or staged on a copy stream beside it
    (pipelined, pkv_handoff_*). Both timed on the bench stream, which waits for the last pack."""
    layers = gen.write_pack_layers(**gen.WRITE_PACK_LLAMA70B, device=dev)
    L0 = layers[0]
    T, Hkv, D = L0.key.shape
    Hq = 64
    nblk = L0.block_ids.numel()
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    q = gen.randn_bf16((T, Hq, D), g, dev)
    out = torch.empty_like(q)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    dsts = [torch.empty((2, nblk) + tuple(L0.k_cache.shape[1:]), dtype=torch.bfloat16, device=dev) for _ in layers]
    ho = pkv.LayerHandoff(len(layers))
    flops = len(layers) * 4 * Hq * D * (T * (T + 1) // 2)

    def serial(marks):
        for L, d in zip(layers, dsts):
            pkv.kv_cache_write(L.key, L.value, L.slot_mapping, L.k_cache, L.v_cache, stream=stream)
            pkv.varlen_prefill_attn(q, L.key, L.value, cu, T, out=out, stream=stream)
            pkv.kv_block_pack(L.k_cache, L.v_cache, L.block_ids, dst=d, stream=stream)

    def pipelined(marks):
        for i, (L, d) in enumerate(zip(layers, dsts)):
            pkv.kv_cache_write(L.key, L.value, L.slot_mapping, L.k_cache, L.v_cache, stream=stream)
            ho.stage(i, L.k_cache, L.v_cache, L.block_ids, dst=d, compute_stream=stream)
            pkv.varlen_prefill_attn(q, L.key, L.value, cu, T, out=out, stream=stream)
        ho.ready(len(layers) - 1, stream)  # the copy stream is in order: the last pack ends it

    def alone(marks):
        for L, d in zip(layers, dsts):
            pkv.kv_cache_write(L.key, L.value, L.slot_mapping, L.k_cache, L.v_cache, stream=stream)
            pkv.varlen_prefill_attn(q, L.key, L.value, cu, T, out=out, stream=stream)

    # five rounds, the three modes interleaved in each, so that the spread between rounds shows
    # whether the difference between modes is above the noise
    rounds = {"serial": [], "pipelined": [], "no_pack": []}
    for _ in range(5):
        for name, fn in (("serial", serial), ("pipelined", pipelined), ("no_pack", alone)):
            ms, _ = timer.run(fn, steps, warmup if not rounds[name] else 1, sections=False)
            rounds[name].append(sorted(ms)[len(ms) // 2])
    torch.cuda.synchronize()
    med = {k: statistics.median(v) for k, v in rounds.items()}
    saved = [a - b for a, b in zip(rounds["serial"], rounds["pipelined"])]
    ok = True
    for L, d in zip(layers[:2], dsts[:2]):  # the staged buffers hold the layers' blocks
        ok &= bool(torch.equal(d[0], L.k_cache[L.block_ids.long()])) and bool(torch.equal(d[1], L.v_cache[L.block_ids.long()]))
    ho.close()
    del layers, dsts
    packs = [a - b for a, b in zip(rounds["serial"], rounds["no_pack"])]
    return {"serial_ms": med["serial"], "pipelined_ms": med["pipelined"], "without_pack_ms": med["no_pack"],
            "rounds_ms": {k: [_r(x) for x in v] for k, v in rounds.items()},
            "saved_ms_median": statistics.median(saved), "saved_ms_range": [_r(min(saved)), _r(max(saved))],
            "pack_cost_ms_median": statistics.median(packs),
            "pipelined_attn_tflops": flops / (med["pipelined"] * 1e-3) / 1e12, "staged_buffers_match": ok}


# ---- CPU oracle ---------------------------------------------------------------------------------

def oracle_decode_rate(b, budget_s=15.0, host=None):
    """KV GB/s of the fp64 oracle on the decode workload: whole requests in chunks, passes over
    the batch repeated until the time budget is spent (at least one chunk)."""
    import oracle
    threads = oracle.default_threads()
    if host is None:
        host = dict(q=gen.bf16_bits(b.q), kc=gen.bf16_bits(b.k_cache), vc=gen.bf16_bits(b.v_cache),
                    bt=b.block_tables.cpu().numpy(), sl=b.seq_lens.cpu().numpy(), cu=b.cu_q.cpu().numpy())
    R = b.R
    chunk = max(1, threads)
    done, t_total, kv = 0, 0.0, 0
    out = np.empty((b.T, b.Hq, b.D))
    lse = np.empty((b.T, b.Hq))
    while t_total < budget_s or done == 0:
        s0 = done % R
        ids = np.arange(s0, min(R, s0 + chunk), dtype=np.int32)
        t0 = time.perf_counter()
        oracle.paged_decode(host["q"], host["kc"], host["vc"], host["bt"], host["sl"], 1.0 / math.sqrt(b.D),
                            cu_q=host["cu"], req_ids=ids, nthreads=threads, out=out, lse=lse)
        t_total += time.perf_counter() - t0
        kv += int(host["sl"][ids].sum()) * b.Hkv * b.D * 4
        done += len(ids)
    return dict(value=kv / t_total / 1e9, unit="GB/s", cores=threads, kind="oracle",
                sample=f"{done} request-decodes ({done / R:.2f} passes over the {R}-request decode workload), "
                       f"whole requests, fp64 C++ oracle, {t_total:.1f} s")


# ---- reduced cases for ncu captures --------------------------------------------------------------

def profile_case(pkv, args):
    """A few launches of one kernel on a reduced case whose inputs still exceed L2 (129 MB), so
    DRAM counters mean something while the capture stays small (well under 1 GB on the device)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.current_stream()
    if args.profile == "decode":
        # 64 sequences of the decode workload's shape: ~330 MB of KV per launch
        b = gen.decode_batch(64, 2000, 3000, Hq=64, Hkv=4, D=128, seed=1, device=dev)
        maxs = max(b.seq_lens_list)
        ws = torch.empty(max(16, pkv.paged_decode_workspace_size(b.R, 64, 4, 128, maxs)), dtype=torch.uint8, device=dev)
        fn = lambda: pkv.paged_decode_attn(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, maxs,
                                           cu_q=b.cu_q, workspace=ws)
        what = f"decode B=64 kv_bytes={sum(b.seq_lens_list) * 4 * 128 * 4}"
    elif args.profile == "decode_fp8":
        # the same 64 sequences over an FP8 (E4M3) cache: ~164 MB of codes per launch
        b = gen.decode_batch(64, 2000, 3000, Hq=64, Hkv=4, D=128, seed=1, device=dev)
        ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
        kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
        maxs = max(b.seq_lens_list)
        ws = torch.empty(max(16, pkv.paged_decode_workspace_size(b.R, 64, 4, 128, maxs)), dtype=torch.uint8, device=dev)
        fn = lambda: pkv.paged_decode_attn(b.q, kc, vc, b.block_tables, b.seq_lens, maxs, cu_q=b.cu_q,
                                           workspace=ws, k_scale=ks, v_scale=vs)
        what = f"decode FP8 B=64 code_bytes={sum(b.seq_lens_list) * 4 * 128 * 2}"
    elif args.profile == "mla":
        # 32 requests of the MLA workload's shape: ~390 MB of latent rows per launch
        b = gen.mla_batch(32, 10000, 11000, Hq=16, seed=5, device=dev)
        maxs = max(b.seq_lens_list)
        ws = torch.empty(max(16, pkv.mla_decode_workspace_size(b.R, 16, maxs)), dtype=torch.uint8, device=dev)
        fn = lambda: pkv.mla_decode_attn(b.q, b.latent, b.block_tables, b.seq_lens, maxs, gen.MLA_SCALE,
                                         workspace=ws)
        what = f"mla B=32 latent_bytes={sum(b.seq_lens_list) * 1152}"
    elif args.profile == "mla128":
        # the same 32 requests with all 128 query heads (the tensor-core kernel on clusters of two)
        b = gen.mla_batch(32, 10000, 11000, Hq=128, seed=5, device=dev)
        maxs = max(b.seq_lens_list)
        ws = torch.empty(max(16, pkv.mla_decode_workspace_size(b.R, 128, maxs)), dtype=torch.uint8, device=dev)
        fn = lambda: pkv.mla_decode_attn(b.q, b.latent, b.block_tables, b.seq_lens, maxs, gen.MLA_SCALE,
                                         workspace=ws)
        what = f"mla 128 heads B=32 latent_bytes={sum(b.seq_lens_list) * 1152}"
    elif args.profile == "prefill":
        b = gen.prefill_batch([4096, 4096], Hq=64, Hkv=8, D=128, seed=5, device=dev)
        fn = lambda: pkv.varlen_prefill_attn(b.q, b.k_new, b.v_new, b.cu_q, 4096)
        what = "prefill 2 x 4096, Hq 64 / Hkv 8"
    elif args.profile == "extend":
        b = gen.extend_batch([512, 512], [16000, 16000], Hq=64, Hkv=8, D=128, seed=3, device=dev)
        fn = lambda: pkv.extend_attn(b.q, b.k_new, b.v_new, b.cu_q, b.seq_lens, b.k_cache, b.v_cache,
                                     b.block_tables, 512, max(b.seq_lens_list))
        what = "extend 2 x (16000 cached + 512 new)"
    elif args.profile == "extend_fp8":
        # the extend case over an FP8 (E4M3) cache: the tensor-core kernel reads the context's
        # codes (~131 MB a launch over both K and V) and converts them in shared memory
        b = gen.extend_batch([512, 512], [16000, 16000], Hq=64, Hkv=8, D=128, seed=3, device=dev)
        ks, vs = gen.fp8_scale(4.0), gen.fp8_scale(4.5)
        kc, vc = gen.fp8_codes(b.k_cache, ks), gen.fp8_codes(b.v_cache, vs)
        fn = lambda: pkv.extend_attn(b.q, b.k_new, b.v_new, b.cu_q, b.seq_lens, kc, vc, b.block_tables, 512,
                                     max(b.seq_lens_list), k_scale=ks, v_scale=vs)
        what = "extend over an FP8 cache, 2 x (16000 cached + 512 new)"
    else:
        layers = gen.write_pack_layers(4, 10000, Hkv=8, D=128, seed=4, device=dev)
        def fn():
            for L in layers:
                pkv.kv_cache_write(L.key, L.value, L.slot_mapping, L.k_cache, L.v_cache)
                pkv.kv_block_pack(L.k_cache, L.v_cache, L.block_ids)
        what = "write + pack, 4 layers x 10000 tokens"
    for _ in range(args.steps):
        fn()
    torch.cuda.synchronize()
    print(f"profile case done: {what}, {args.steps} launches, device errors {pkv.device_errors()}")


# ---- main ---------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="headline workload only")
    ap.add_argument("--oracle-seconds", type=float, default=10.0)
    ap.add_argument("--profile", choices=["decode", "decode_fp8", "mla", "mla128", "prefill", "extend", "extend_fp8", "write_pack"], default=None,
                    help="run a reduced case of one kernel --steps times for an ncu capture; prints "
                         "a one-line summary, no benchmark line")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    steps, warmup = args.steps, max(3, args.warmup)

    if args.impl == "reference":
        if rank != 0:
            return
        b = gen.decode_batch(**gen.DECODE_QWEN3, device="cpu")
        times, vals = [], []
        host = dict(q=gen.bf16_bits(b.q), kc=gen.bf16_bits(b.k_cache), vc=gen.bf16_bits(b.v_cache),
                    bt=b.block_tables.numpy(), sl=b.seq_lens.numpy(), cu=b.cu_q.numpy())
        budget = max(2.0, 120.0 / max(1, steps + warmup))
        for i in range(warmup + steps):
            r = oracle_decode_rate(b, budget_s=budget, host=host)
            if i >= warmup:
                vals.append(r["value"])
        v = statistics.median(vals)
        line = {"impl": "reference", "metric": "paged decode attn KV GB/s (frac of HBM peak); mixed-batch attn tokens/s",
                "value": v, "unit": "GB/s", "n_gpus": args.gpus, "steps": steps, "warmup": warmup,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": headline_config(sum(b.seq_lens_list) * b.Hkv * b.D * 2 * 2, args.gpus),
                "oracle_step": "the fp64 oracle's decode of whole requests of this batch (rank 0 only); the "
                               "reorder and the write are index copies it does not time",
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": r["cores"], "kind": "oracle", "sample": r["sample"]},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import paged_kv_attention_reshape_gb300 as pkv
    pkv.load()
    if args.profile:
        return profile_case(pkv, args)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    timer = Timer(stream, flush_buf)
    peaks = load_peaks()

    clocks = Clocks(local)
    with clocks:
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        w, ms, sec, launches = bench_decode(pkv, dev, stream, timer, steps, warmup, seed_off=rank, hold_s=1.0,
                                            on_ready=clocks.wait_first)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    step_ms = max_over_ranks(sum(ms) / len(ms), ws, dev)
    value = replica_rate(w["kv_bytes"], ws, step_ms) / 1e9
    dec_ms = sum(sec["decode"]) / len(sec["decode"])   # mean over the decode-alone launches
    achieved = w["alg_bytes"] / (dec_ms * 1e-3) / 1e9
    traffic = profiled_traffic("paged_decode", "paged_decode_qwen3")
    if ws > 1:
        torch.distributed.barrier()
    e2e_ms, h2d, d2h = bench_decode_e2e(pkv, w, dev, stream, steps, warmup, timer)
    serial_step = max_over_ranks(sum(e2e_ms) / len(e2e_ms), ws, dev)
    if ws > 1:
        torch.distributed.barrier()
    e2e_steps = max(steps, 8)
    pipe_ms, _, _ = bench_decode_e2e_pipelined(pkv, w, dev, stream, e2e_steps, warmup)
    e2e_step = max_over_ranks(pipe_ms, ws, dev)
    line = {
        "metric": "paged decode attn KV GB/s (frac of HBM peak); mixed-batch attn tokens/s",
        "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps, "warmup": warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": headline_config(w["kv_bytes"], ws),
        "roofline": {"kernel": "paged_decode_kernel", "bound": "hbm", "achieved": achieved,
                     "peak": peaks["hbm"], "unit": "GB/s", "frac": achieved / peaks["hbm"],
                     "traffic": traffic, "algorithmic_bytes_per_launch": w["alg_bytes"],
                     "peak_source": peaks["source"] + " (hbm copy, burst)", "launch_ms": dec_ms,
                     "launch_timing": f"mean of {len(sec['decode'])} lone decode calls, CUDA events, L2 flushed"},
        "e2e": {"value": replica_rate(w["kv_bytes"], ws, serial_step) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": serial_step,
                "steps": len(e2e_ms),
                "mode": "serial: copy in, step, copy out on one stream, each step alone after an L2 flush",
                "pipelined_value": replica_rate(w["kv_bytes"], ws, e2e_step) / 1e9,
                "pipelined_ms_per_step": e2e_step},
        "gpu_launches": launches * steps,
        "clocks": dict(clocks.summary(), window="nvidia-smi every 200 ms, first warm-up step to 1 s past the timed steps"),
    }
    summary = {"decode_frac_of_measured_hbm": _r(achieved / peaks["hbm"]),
               "decode_frac_of_nominal_8TBs": _r(w["kv_bytes"] / (dec_ms * 1e-3) / 8e12),
               "e2e_serial_gbs": _r(line["e2e"]["value"]), "e2e_pipelined_gbs": _r(line["e2e"]["pipelined_value"])}
    if not args.no_extras and rank == 0:
        extras = {}
        try:
            m = bench_mixed(pkv, dev, stream, timer, steps, warmup)
            mms = sum(m["ms"]) / len(m["ms"])
            per = {k: _r(sum(v) / len(v)) for k, v in m["sec"].items()}
            ums = sum(m["unified_ms"]) / len(m["unified_ms"])
            bound = (m["dec_bytes"] / (peaks["hbm"] * 1e9) + (m["ext_flops"] + m["pre_flops"]) /
                     (peaks["bf16_sust"] * 1e12)) * 1e3
            extras["mixed_batch"] = {
                "tokens_per_s": m["tokens"] / (mms * 1e-3), "ms_per_step": mms, "tokens": m["tokens"],
                "per_call_ms": per, "gpu_launches_per_step": m["launches"],
                "decode_kv_gbs": m["dec_bytes"] / (per["decode"] * 1e-3) / 1e9,
                "extend_tflops": m["ext_flops"] / (per["extend"] * 1e-3) / 1e12,
                "prefill_tflops": m["pre_flops"] / (per["prefill"] * 1e-3) / 1e12,
                "bound_ms": bound, "frac_of_bound": bound / mms,
                "unified_single_call": {"ms_per_step": ums, "tokens_per_s": m["tokens"] / (ums * 1e-3)}}
            summary.update(mixed_tokens_per_s=_r(m["tokens"] / (mms * 1e-3)), mixed_ms=_r(mms),
                           mixed_frac_of_bound=_r(bound / mms),
                           mixed_prefill_frac=_r(extras["mixed_batch"]["prefill_tflops"] / peaks["bf16"]),
                           mixed_extend_frac=_r(extras["mixed_batch"]["extend_tflops"] / peaks["bf16"]),
                           unified_tokens_per_s=_r(m["tokens"] / (ums * 1e-3)))
            del m
        except Exception as e:  # report, keep the headline
            extras["mixed_batch"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            m8 = bench_mixed_fp8(pkv, dev, stream, timer, steps, warmup)
            mms8 = sum(m8["ms"]) / len(m8["ms"])
            extras["mixed_batch_fp8"] = {
                "tokens_per_s": m8["tokens"] / (mms8 * 1e-3), "ms_per_step": mms8,
                "per_call_ms": {k: _r(sum(v) / len(v)) for k, v in m8["sec"].items()},
                "extend_workspace_bytes": m8["ws_bytes"], "device_errors": m8["errors"],
            }
            summary.update(fp8_mixed_tokens_per_s=_r(m8["tokens"] / (mms8 * 1e-3)))
        except Exception as e:
            extras["mixed_batch_fp8"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            r = bench_decode_fp8(pkv, dev, stream, timer, steps, warmup)
            fr = r["alg_bytes"] / (r["launch_ms"] * 1e-3) / 1e9 / peaks["hbm"]
            extras["decode_fp8"] = {
                "kv_bytes_per_step": r["kv_bytes"], "ms_per_step": r["step_ms"],
                "kv_gbs": r["kv_bytes"] / (r["step_ms"] * 1e-3) / 1e9,
                "decode_tokens_per_s": r["R"] / (r["step_ms"] * 1e-3),
                "bf16_decode_tokens_per_s": w["b"].R / (step_ms * 1e-3),
                "launch_ms": r["launch_ms"], "roofline_frac": fr,
            }
            summary.update(fp8_decode_frac=_r(fr), fp8_decode_tokens_per_s=_r(r["R"] / (r["step_ms"] * 1e-3)))
        except Exception as e:
            extras["decode_fp8"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            r = bench_mla(pkv, dev, stream, timer, steps, warmup)
            fr = r["alg_bytes"] / (r["launch_ms"] * 1e-3) / 1e9 / peaks["hbm"]
            extras["mla_decode"] = {
                "latent_bytes_per_step": r["lat_bytes"], "ms_per_step": r["step_ms"],
                "latent_gbs": r["lat_bytes"] / (r["step_ms"] * 1e-3) / 1e9,
                "decode_tokens_per_s": r["R"] / (r["step_ms"] * 1e-3),
                "launch_ms": r["launch_ms"], "roofline_frac": fr,
                "mma_tflops": r["flops"] / (r["launch_ms"] * 1e-3) / 1e12,
                "traffic": profiled_traffic("mla_decode", "mla_deepseek_tp8"),
                "algorithmic_bytes_per_launch": r["alg_bytes"], "device_errors": r["errors"],
            }
            summary.update(mla_decode_frac=_r(fr))
        except Exception as e:
            extras["mla_decode"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            # the same layer with all 128 heads on one GPU: compute-bound on the warp-level MMA
            # (informational; eight groups of 16 heads, L2 serving the groups' repeated reads)
            r = bench_mla(pkv, dev, stream, timer, max(3, steps // 2), warmup, Hq=128)
            extras["mla_decode_128"] = {
                "launch_ms": r["launch_ms"], "latent_gbs": r["lat_bytes"] / (r["launch_ms"] * 1e-3) / 1e9,
                "mma_tflops": r["flops"] / (r["launch_ms"] * 1e-3) / 1e12,
                "decode_tokens_per_s": r["R"] / (r["step_ms"] * 1e-3), "device_errors": r["errors"]}
            summary["mla128_latent_gbs"] = _r(extras["mla_decode_128"]["latent_gbs"])
        except Exception as e:
            extras["mla_decode_128"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        for kind in ("prefill", "extend_long"):
            try:
                r = bench_attention_only(pkv, dev, stream, timer, max(3, steps // 2), warmup,
                                         "prefill" if kind == "prefill" else "extend")
                k = "prefill" if kind == "prefill" else "extend"
                t = sum(r["sec"][k]) / len(r["sec"][k])
                tf = r["flops"] / (t * 1e-3) / 1e12
                extras[kind] = {"tflops": tf, "ms": t, "frac_of_bf16_peak": tf / peaks["bf16"],
                                "peak_tflops": peaks["bf16"], "peak_source": peaks["source"] + " (bf16 burst)"}
                summary[f"{kind}_tflops"] = _r(tf)
                summary[f"{kind}_frac"] = _r(tf / peaks["bf16"])
            except Exception as e:
                extras[kind] = {"error": repr(e)}
            torch.cuda.empty_cache()
        try:
            r = bench_write_pack(pkv, dev, stream, timer, max(3, steps // 2), warmup)
            res = {}
            for k in ("write", "pack", "unpack"):
                t = sum(r["sec"][k]) / len(r["sec"][k])
                res[f"{k}_gbs"] = r[f"{k}_bytes"] / (t * 1e-3) / 1e9
                res[f"{k}_ms_80_layers"] = t
                res[f"{k}_frac"] = res[f"{k}_gbs"] / peaks["hbm"]
                summary[f"{k}_frac"] = _r(res[f"{k}_frac"])
            extras["write_pack"] = res
        except Exception as e:
            extras["write_pack"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            r = bench_tiny_decode(pkv, dev, stream, timer, max(steps, 20), warmup)
            extras["tiny_decode"] = r
            summary["tiny_decode_gbs"] = _r(r["kv_gbs"])
        except Exception as e:
            extras["tiny_decode"] = {"error": repr(e)}
        try:
            r = bench_handoff(pkv, dev, stream, timer, max(3, steps // 4), warmup)
            extras["handoff_pipeline"] = r
            summary["handoff_saved_ms"] = _r(r["saved_ms_median"])
        except Exception as e:
            extras["handoff_pipeline"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        line["extras"] = extras
    if rank == 0:
        if ws == 1:
            line["cpu_baseline"] = oracle_decode_rate(w["b"], budget_s=args.oracle_seconds)
        line["summary"] = summary  # last: the key numbers of every row in the line's final characters
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
