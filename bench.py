#!/usr/bin/env python3
"""Benchmark of the fused attention backward on GB300.

One step = one full backward (preprocess, main kernel, dQ landing: every
launch of the path) over one batch of the causal MHA workload
B=2, S=2048, H=32, D=128, fp16 (the "llama-8b-long" row of the TileOPs MHA
backward page's performance table), inputs resident in HBM.  The metric is
TFLOP/s with the causal convention 2.5 x the causal forward = 5*B*H*S^2*D.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead, on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own copy of the workload (independent
batches, no collective in the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn-bwd TFLOP/s (dQ,dK,dV) & % of GB300 fp16/bf16 tensor peak; sparse: HBM GB/s"
MAIN_WORKLOAD = "mha_causal_2x2048x32x128_f16"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def dense_flops(w) -> float:
    """2.5 x forward; forward = 4*S_q*S_k*D per head, halved when causal; for
    packed varlen/window: 4*D per attended (query, key) pair."""
    if w.cu_seqlens is not None or w.window > 0:
        pairs = 0
        for a, e in zip(w.cu_seqlens[:-1], w.cu_seqlens[1:]):
            n = e - a
            for i in range(n):
                lo = max(0, i - w.window + 1) if w.window > 0 else 0
                pairs += i - lo + 1
        return 2.5 * 4.0 * w.D * pairs * w.HQ * w.B
    f = 4.0 * w.B * w.HQ * w.S * w.S * w.D
    return 2.5 * (f / 2 if w.causal else f)


def sparse_flops(w, idx) -> float:
    """Per valid (token, slot) pair and head: S (2*DQK), dP (2*DV), dV (2*DV),
    dK (2*DQK), dQ (2*DQK)."""
    valid = int(((idx >= 0) & (idx < w.S)).sum())
    return valid * w.HQ * 2.0 * (3 * w.D + 2 * w.Dv)


def sparse_valid_pairs(w, idx) -> int:
    return int(((idx >= 0) & (idx < w.S)).sum())


def sparse_hbm_bytes(w, idx):
    """Algorithmic DRAM bytes of each launch of the sparse path: every input and
    output crosses HBM once (the gathered latent rows come from L2: KV is read
    from DRAM once), the f32 dKV accumulator is read and written once by the
    scatter and read once by the landing pass."""
    B, S, H, HKV, DQK, DV, K = w.B, w.S, w.HQ, w.HKV, w.D, w.Dv, w.topk
    SKV = w.S
    pre = B * S * H * DV * 2 * 2 + B * H * S * 4 + B * S * H * 4 * 2 + B * SKV * HKV * DQK * 4
    main = (B * S * H * DQK * 2 * 2 + B * S * H * DV * 2 + B * S * H * 4 * 2 + B * S * HKV * K * 4
            + B * SKV * HKV * DQK * 2 + B * SKV * HKV * DQK * 4 * 2)
    land = B * SKV * HKV * DQK * (4 + 2)
    return {"preprocess": pre, "main": main, "land": land, "gathered_l2": sparse_valid_pairs(w, idx) * DQK * 2}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(kernel_src: str) -> str:
    """sha256 prefix over a kernel's .cu file and every header it includes,
    transitively (quoted includes found in the library's csrc/ and include/),
    in first-include order: a DRAM record stays valid only while none of them
    changed."""
    dirs = [os.path.dirname(kernel_src), os.path.join(ROOT, "include")]
    seen, order = set(), []

    def visit(path):
        if path in seen:
            return
        seen.add(path)
        order.append(path)
        with open(path) as f:
            for line in f:
                s = line.strip()
                if s.startswith("#include \""):
                    name = s.split('"')[1]
                    for d in dirs:
                        cand = os.path.join(d, name)
                        if os.path.exists(cand):
                            visit(cand)
                            break

    visit(kernel_src)
    h = hashlib.sha256()
    for path in order:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel_src: str, name: str):
    """DRAM bytes per launch of ``name`` from the committed ncu summary, only if
    it was taken on the current kernel sources (matching hash over the .cu file
    and its headers)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(name)
    if not rec:
        return None
    return rec.get("dram_bytes_per_launch") if rec.get("source_sha256_16") == source_hash(kernel_src) else None


# ------------------------------------------------------------------ inputs (GPU arm)

def gpu_dense_inputs(w, device):
    """Q, K, V, dO from the seeded generator; O and LSE from the library's own
    forward (attn_fwd_gqa) on the device (input preparation; it is timed
    separately, not as part of the backward's step)."""
    import torch

    import attention_backward_gb300 as ab
    from attention_backward_gb300 import inputs

    q, k, v, do = inputs.dense_inputs(w)
    tdt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    tq, tk, tv, tdo = (torch.from_numpy(a).to(device).to(tdt) for a in (q, k, v, do))
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=device) if w.cu_seqlens else None
    ws = torch.empty(256, dtype=torch.uint8, device=device)
    o, lse = ab.forward(tq, tk, tv, w.sm_scale, w.causal, w.window, cu, workspace=ws)
    ab.check_error(ws)
    return tq, tk, tv, o, tdo, lse


def time_forward(w, tensors, steps, warmup, device, flush_bytes=256 << 20):
    """The forward (attn_fwd_gqa) timed alone: events around each call, L2
    flushed before each."""
    import torch

    import attention_backward_gb300 as ab

    tq, tk, tv, to, tdo, lse, cu = tensors
    o, l_ = torch.empty_like(to), torch.empty_like(lse)
    ws = torch.empty(256, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(ev):
        ev[0].record(stream)
        ab.attn_fwd_gqa(tq, tk, tv, o, l_, ws, w.sm_scale, w.causal, w.window, cu, stream)
        ev[1].record(stream)

    per = _timed_steps(step, steps, warmup, device, stream, ws, 2, flush_bytes, 1)
    ts = [e[0].elapsed_time(e[1]) for e in per]
    return {"ms": float(np.mean(ts)), "ms_pct": _pct(ts)}


def time_sink_grad(w, ws, cu, steps, warmup, device, flush_bytes=256 << 20):
    """The attention-sink gradient (attn_bwd_sink_grad) timed alone on the rows
    a backward call left in ``ws``: events around each call, L2 flushed before
    each.  Seeded sink logits, one per query head."""
    import torch

    import attention_backward_gb300 as ab

    sink = torch.from_numpy(np.random.default_rng(w.seed).standard_normal(w.HQ).astype(np.float32)).to(device)
    stream = torch.cuda.current_stream(device)

    def step(ev):
        ev[0].record(stream)
        ab.sink_grad(sink, ws, w.B, w.S, cu, stream)
        ev[1].record(stream)

    per = _timed_steps(step, steps, warmup, device, stream, ws, 2, flush_bytes, 1)
    ts = [e[0].elapsed_time(e[1]) for e in per]
    return {"ms": float(np.mean(ts)), "ms_pct": _pct(ts)}


def gpu_sparse_inputs(w, device):
    """Q, KV, dO and the index lists from the seeded generator; O and LSE from a
    float32 torch forward over the listed rows on the device (not timed)."""
    import torch

    from attention_backward_gb300 import inputs

    q, kv, do, idx = inputs.sparse_inputs(w)
    tdt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    tq, tkv, tdo = (torch.from_numpy(a).to(device).to(tdt) for a in (q, kv, do))
    tidx = torch.from_numpy(idx).to(device)
    G = w.HQ // w.HKV
    o = torch.empty_like(tdo)
    lse = torch.empty(w.B, w.HQ, w.S, dtype=torch.float32, device=device)
    for b in range(w.B):
        for g in range(w.HKV):
            hs = slice(g * G, (g + 1) * G)
            for t0 in range(0, w.S, 128):
                t1 = min(w.S, t0 + 128)
                ix = tidx[b, t0:t1, g].long()
                ok = (ix >= 0) & (ix < w.S)
                rows = tkv[b, ix.clamp(0, w.S - 1), g].float()            # [T, topk, DQK]
                s_ = torch.einsum("thd,tkd->thk", tq[b, t0:t1, hs].float(), rows) * w.sm_scale
                s_ = s_.masked_fill(~ok[:, None, :], float("-inf"))
                l_ = torch.logsumexp(s_, dim=2)
                o[b, t0:t1, hs] = torch.einsum("thk,tkd->thd", torch.exp(s_ - l_[..., None]),
                                               rows[..., :w.Dv]).to(tdt)
                lse[b, hs, t0:t1] = l_.T
    return tq, tkv, o, tdo, lse, tidx, idx


# ------------------------------------------------------------------ GPU arm

def _timed_steps(step, steps, warmup, device, stream, ws, nev, flush_bytes, world):
    """W untimed steps, then K steps each bracketed by CUDA events on the
    launching stream, L2 flushed before each (a write larger than L2, read back
    so that no dirty line is left); a barrier and a device synchronisation on
    both sides of the timed region."""
    import torch

    import attention_backward_gb300 as ab

    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=device)

    def clear_l2():
        # a write larger than L2 evicts the previous step's lines; reading the
        # buffer back then writes the flush's own dirty lines back to HBM here,
        # outside the timed region, so every step starts from a cold L2 that
        # holds no dirty line
        flush.zero_()
        flush.sum()

    for _ in range(warmup):
        clear_l2()
        step([torch.cuda.Event(enable_timing=True) for _ in range(nev)])
    ab.check_error(ws, stream)
    torch.cuda.synchronize(device)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize(device)
    per = []
    for _ in range(steps):
        clear_l2()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
        step(ev)
        per.append(ev)
    torch.cuda.synchronize(device)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    ab.check_error(ws, stream)
    return per

def time_dense(w, steps, warmup, device, world=1, flush_bytes=256 << 20):
    """The dense backward timed through the one-call entry point attn_bwd_gqa
    (events around the call only), then, in a second pass, its launches one by
    one with events between them for the per-stage breakdown."""
    import torch

    import attention_backward_gb300 as ab

    tq, tk, tv, to, tdo, lse = gpu_dense_inputs(w, device)
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=device) if w.cu_seqlens else None
    ws = ab._binding.new_gqa_workspace(w.B, w.S, w.HQ, w.D, device=device)
    dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
    stream = torch.cuda.current_stream(device)

    def step(ev):
        ev[0].record(stream)
        ab.attn_bwd_gqa(tq, tk, tv, to, tdo, lse, dq, dk, dv, ws, w.sm_scale, w.causal, w.window, cu, stream)
        ev[1].record(stream)

    def staged(ev):
        ev[0].record(stream)
        ab.preprocess(to, tdo, lse, ws, Dq=w.D, stream=stream)
        ev[1].record(stream)
        ab.gqa_main(tq, tk, tv, tdo, dk, dv, ws, w.sm_scale, w.causal, w.window, cu, stream)
        ev[2].record(stream)
        ab.dq_land(dq, ws, w.sm_scale, stream)
        ev[3].record(stream)

    per = _timed_steps(step, steps, warmup, device, stream, ws, 2, flush_bytes, world)
    per_st = _timed_steps(staged, steps, warmup, device, stream, ws, 4, flush_bytes, world)
    tensors = (tq, tk, tv, to, tdo, lse, cu)
    sink = time_sink_grad(w, ws, cu, steps, warmup, device, flush_bytes)
    fwd = time_forward(w, tensors, steps, warmup, device, flush_bytes)
    return _stage_times(per, per_st) | {"tensors": tensors, "forward": fwd, "sink_grad": sink}


def time_sparse(w, steps, warmup, device, world=1, flush_bytes=256 << 20):
    """The sparse backward timed through the one-call entry point
    attn_bwd_sparse, then its launches one by one for the stage breakdown."""
    import torch

    import attention_backward_gb300 as ab

    tq, tkv, to, tdo, lse, tidx, idx = gpu_sparse_inputs(w, device)
    dkv_elems = tkv.numel()
    ws = ab._binding.new_workspace(w.B, w.S, w.HQ, 0, dkv_elems, device=device)
    dq, dkv = torch.empty_like(tq), torch.empty_like(tkv)
    stream = torch.cuda.current_stream(device)

    def step(ev):
        ev[0].record(stream)
        ab.attn_bwd_sparse(tq, tkv, to, tdo, lse, tidx, dq, dkv, ws, w.sm_scale, w.Dv, stream)
        ev[1].record(stream)

    def staged(ev):
        ev[0].record(stream)
        ab.preprocess(to, tdo, lse, ws, Dq=0, dkv_elems=dkv_elems, stream=stream)
        ev[1].record(stream)
        ab.sparse_main(tq, tkv, tdo, tidx, dq, ws, w.sm_scale, w.Dv, stream)
        ev[2].record(stream)
        ab.sparse_land(dkv, ws, w.B, w.S, w.HQ, stream)
        ev[3].record(stream)

    per = _timed_steps(step, steps, warmup, device, stream, ws, 2, flush_bytes, world)
    per_st = _timed_steps(staged, steps, warmup, device, stream, ws, 4, flush_bytes, world)
    return _stage_times(per, per_st) | {"tensors": (tq, tkv, to, tdo, lse, tidx), "idx": idx}


def _pct(xs):
    """Median and the 10th / 90th percentiles of a list of times (ms)."""
    return {"p10": float(np.percentile(xs, 10)), "median": float(np.median(xs)), "p90": float(np.percentile(xs, 90))}


def _stage_times(per, per_st):
    """Step times from the one-call pass (two events per step); stage times
    from the pass with events between the launches (they add a few
    microseconds of gaps there, which the step time does not carry)."""
    tot = [e[0].elapsed_time(e[1]) for e in per]
    main = [e[1].elapsed_time(e[2]) for e in per_st]
    return {"ms_step": float(np.mean(tot)), "ms_step_pct": _pct(tot),
            "ms_pre": float(np.mean([e[0].elapsed_time(e[1]) for e in per_st])),
            "ms_main": float(np.mean(main)), "ms_main_pct": _pct(main),
            "ms_land": float(np.mean([e[2].elapsed_time(e[3]) for e in per_st]))}


def time_e2e(w, tensors, steps, device, chunks=4):
    """The same backward through the public API with pinned host buffers:
    host->device copies of the inputs and device->host copies of the gradients
    inside the timed region.  Dense: attn_bwd_gqa_host, which pipelines the
    copies with the kernels chunk by chunk of KV heads.  Sparse: the copies,
    then the three launches."""
    import torch

    import attention_backward_gb300 as ab

    stream = torch.cuda.current_stream(device)
    if w.kind == "sparse":
        host_in = [t.cpu().pin_memory() for t in tensors]           # q, kv, o, do, lse, idx
        outs = (tensors[0], tensors[1])                             # dq like q, dkv like kv
        ws = ab._binding.new_workspace(w.B, w.S, w.HQ, 0, tensors[1].numel(), device=device)
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        dev_in = [torch.empty(t.shape, dtype=t.dtype, device=device) for t in host_in]

        def one():
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)
            grads = ab.sparse_backward(*dev_in, w.sm_scale, w.Dv, workspace=ws, stream=stream)
            for h, d in zip(host_out, grads):
                h.copy_(d, non_blocking=True)
    else:
        host_in = [t.cpu().contiguous().pin_memory() for t in tensors[:6]]  # q, k, v, o, do, lse
        cu = tensors[6]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in host_in[:3]]
        scratch = torch.empty(ab.host_scratch_size(w.B, w.S, w.HQ, w.HKV, w.D, chunks), dtype=torch.uint8,
                              device=device)
        streams = (stream, torch.cuda.Stream(device), torch.cuda.Stream(device))

        def one():
            ab.backward_host(*host_in, w.sm_scale, w.causal, w.window, cu, chunks=chunks, out=host_out,
                             scratch=scratch, streams=streams, device=device, sync=False)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    one()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / steps, h2d, d2h


def cpu_oracle_sample(w, budget_s=12.0):
    """The oracle timed on the host cores over a bounded sample of workload
    ``w``; inputs from the seeded generator and the oracle's own forward (not
    timed).  Returns (TFLOP/s of the workload's counted FLOPs, seconds timed,
    description of the sample).

    Short dense rows (S <= 4096, one sequence per batch row): whole query heads
    (a prefix, whole KV groups).  Long or packed rows: one KV group's query
    heads on seeded rows, dQ rows and dK/dV rows evaluated separately by the
    oracle (7 matrix products per row instead of the 5 of a whole-head
    evaluation), extrapolated linearly by rows and heads.  Sparse: the whole
    backward of a seeded sample of tokens, extrapolated by valid (token, slot)
    pairs."""
    import oracle
    from attention_backward_gb300 import inputs

    if w.kind == "sparse":
        return _cpu_sparse_sample(w, budget_s)
    q, k, v, do = inputs.dense_inputs(w)
    mask = dict(causal=w.causal, window=w.window, cu_seqlens=w.cu_seqlens)
    G = w.HQ // w.HKV
    if w.S <= 4096 and w.cu_seqlens is None:
        # calibrate on one head, then time as many whole KV groups as fit the budget
        o1, l1 = oracle.forward(q[:, :, :1], k[:, :, :1], v[:, :, :1], w.sm_scale, **mask)
        o1 = inputs.round_to_dtype(o1, w.dtype)
        t0 = time.perf_counter()
        oracle.backward(q[:, :, :1], k[:, :, :1], v[:, :, :1], o1, do[:, :, :1], l1, w.sm_scale, **mask)
        t1 = time.perf_counter() - t0
        nh = int(max(1, min(w.HQ, budget_s // max(t1, 1e-3))))
        nh = max(G, (nh // G) * G)
        qs, ks, vs, dos = q[:, :, :nh], k[:, :, :nh // G], v[:, :, :nh // G], do[:, :, :nh]
        o, lse = oracle.forward(qs, ks, vs, w.sm_scale, **mask)
        o = inputs.round_to_dtype(o, w.dtype)
        t0 = time.perf_counter()
        oracle.backward(qs, ks, vs, o, dos, lse, w.sm_scale, **mask)
        el = time.perf_counter() - t0
        frac = nh / w.HQ
        return (dense_flops(w) * frac / el / 1e12, el,
                f"{nh} of {w.HQ} query heads x {w.B} batch rows of {w.name}, whole heads, {el:.1f} s of float64 numpy")
    # long rows: the first KV group's heads on seeded rows
    qs, ks, vs, dos = q[:, :, :G], k[:, :, :1], v[:, :, :1], do[:, :, :G]
    o, lse = oracle.forward(qs, ks, vs, w.sm_scale, **mask)
    o = inputs.round_to_dtype(o, w.dtype)
    rng = np.random.default_rng(w.seed)
    if w.cu_seqlens is not None:  # rows inside sequences only
        inside = np.concatenate([np.arange(a, e) for a, e in zip(w.cu_seqlens[:-1], w.cu_seqlens[1:])])
    else:
        inside = np.arange(w.S)
    rows = np.sort(rng.choice(inside, size=min(64, inside.size), replace=False))
    t0 = time.perf_counter()
    oracle.backward(qs, ks, vs, o, dos, lse, w.sm_scale, q_rows=rows, k_rows=rows, **mask)
    t1 = time.perf_counter() - t0
    n = int(min(inside.size, max(64, rows.size * budget_s / max(t1, 1e-3))))
    rows = np.sort(rng.choice(inside, size=n, replace=False))
    t0 = time.perf_counter()
    oracle.backward(qs, ks, vs, o, dos, lse, w.sm_scale, q_rows=rows, k_rows=rows, **mask)
    el = time.perf_counter() - t0
    frac = (G / w.HQ) * (rows.size / inside.size) / w.B
    return (dense_flops(w) * frac / el / 1e12, el,
            f"{rows.size} seeded rows (dQ rows and dK/dV rows) of query heads 0-{G - 1} (one KV group) of "
            f"{w.name}, {el:.1f} s of float64 numpy, extrapolated linearly to every row and head")


def _cpu_sparse_sample(w, budget_s):
    """The oracle's whole sparse backward (dQ and the dKV contributions) over
    the tokens of a seeded sample, extrapolated by valid (token, slot) pairs."""
    import oracle
    from attention_backward_gb300 import inputs

    q, kv, do, idx = inputs.sparse_inputs(w)
    rng = np.random.default_rng(w.seed)
    valid = lambda ix: int(((ix >= 0) & (ix < kv.shape[1])).sum())  # noqa: E731

    def run(n):
        toks = np.sort(rng.choice(w.S, size=n, replace=False))
        qs, dos, ixs = q[:, toks], do[:, toks], idx[:, toks]
        o, lse = oracle.sparse_forward(qs, kv, ixs, w.sm_scale, w.Dv)
        o = inputs.round_to_dtype(o, w.dtype)
        t0 = time.perf_counter()
        oracle.sparse_backward(qs, kv, o, dos, lse, ixs, w.sm_scale, w.Dv)
        return time.perf_counter() - t0, valid(ixs), n

    el, pairs, n = run(16)
    n = int(min(w.S, max(16, n * budget_s / max(el, 1e-3))))
    el, pairs, n = run(n)
    frac = pairs / valid(idx)
    return (sparse_flops(w, idx) * frac / el / 1e12, el,
            f"the whole backward (dQ and dKV contributions) of {n} seeded tokens ({pairs} of {valid(idx)} valid "
            f"(token, slot) pairs) of {w.name}, {el:.1f} s of float64 numpy, extrapolated by pairs")


# ------------------------------------------------------------------ main

def dist_setup(n):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def reduce_max_over_ranks(vals, device=None):
    """Each value's maximum over all ranks: one all-reduce, outside the timed
    region.  With one process (or no process group) the values come back as is."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (weak scaling: each rank runs its own copy of the workload)."""
    return units_per_rank * world / (ms * 1e-3)


def run_reference(args):
    """CPU oracle arm: each step times the oracle on a bounded sample."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from attention_backward_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    vals, els = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        v_, el, desc = cpu_oracle_sample(w, budget_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)))
        if i >= args.warmup:
            vals.append(v_)
            els.append(el)
    value = float(np.mean(vals))
    cores = os.cpu_count()
    unit = "TFLOP/s"
    work = sparse_flops(w, inputs.sparse_inputs(w)[3]) if w.kind == "sparse" else dense_flops(w)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(els)) * 1e3,
            "ms_per_step_extrapolated": work / (value * 1e12) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": f"per step: {desc}"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def describe(w, r, pk, pk_kind, world=1):
    """Throughput, roofline and per-stage figures of one timed workload."""
    import os as _os

    ms, ms_main = r["ms_step"], r["ms_main"]
    csrc = _os.path.join(ROOT, "attention_backward_gb300", "csrc")
    if w.kind == "sparse":
        idx = r["idx"]
        flops = sparse_flops(w, idx)
        by = sparse_hbm_bytes(w, idx)
        step_bytes = by["preprocess"] + by["main"] + by["land"]
        kname = f"sparse_bwd_kernel<{w.dtype}>"
        t_tensor = flops / (float(pk["bf16_tflops"]) * 1e12)
        t_hbm = by["main"] / (float(pk["hbm_gbs"]) * 1e9)
        out = {"value": job_rate(step_bytes, world, ms) / 1e9, "unit": "GB/s",
               "TFLOP/s": job_rate(flops, world, ms) / 1e12,
               "valid_pairs": sparse_valid_pairs(w, idx), "algorithmic_bytes": by}
        achieved_t = flops / (ms_main * 1e-3) / 1e12
        achieved_b = by["main"] / (ms_main * 1e-3) / 1e9
        tensor_roof = {"bound": "tensor", "achieved": achieved_t, "peak": float(pk["bf16_tflops"]),
                       "unit": "TFLOP/s", "frac": achieved_t / float(pk["bf16_tflops"])}
        hbm_roof = {"bound": "hbm", "achieved": achieved_b, "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
                    "frac": achieved_b / float(pk["hbm_gbs"])}
        roof = dict(tensor_roof if t_tensor >= t_hbm else hbm_roof)
        roof["other_bound"] = hbm_roof if t_tensor >= t_hbm else tensor_roof
        roof["l2_gather_GB/s"] = by["gathered_l2"] / (ms_main * 1e-3) / 1e9
        src = _os.path.join(csrc, "sparse_bwd.cu")
    else:
        flops = dense_flops(w)
        out = {"value": job_rate(flops, world, ms) / 1e12, "unit": "TFLOP/s"}
        achieved = flops / (ms_main * 1e-3) / 1e12
        peak = float(pk["bf16_tflops"])  # fp16 and bf16 share the nominal dense rate
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak}
        if w.D == 128:  # head dim 128: 128-query steps
            kname, src = f"dense128_bwd_kernel<{w.dtype}>", _os.path.join(csrc, "dense128_bwd.cu")
        else:
            kname, src = f"dense_bwd_kernel<{w.D},{w.dtype}>", _os.path.join(csrc, "dense_bwd.cu")
        if "forward" in r:  # the forward that produced O and LSE, timed alone
            fflops = flops / 2.5
            fms = r["forward"]["ms"]
            fach = fflops / (fms * 1e-3) / 1e12
            fname = f"dense_fwd_kernel<{w.D},{w.dtype}>"
            out["forward"] = {
                "value": fach, "unit": "TFLOP/s", "ms": fms, "ms_pct": r["forward"]["ms_pct"], "flops": fflops,
                "roofline": {"bound": "tensor", "achieved": fach, "peak": peak, "unit": "TFLOP/s",
                             "frac": fach / peak, "kernel": fname, "kernel_ms": fms,
                             "peak_kind": f"bf16 burst, {pk_kind}",
                             "traffic": traffic_record(_os.path.join(csrc, "dense_fwd.cu"), fname + "@" + w.name)}}
        if "sink_grad" in r:  # dsink from the workspace rows: reads LSE2 and delta of every row once
            rows = w.B * w.HQ * (w.S if w.cu_seqlens is None else w.cu_seqlens[-1] - w.cu_seqlens[0])
            sbytes = rows * 8 + w.HQ * 8
            sms = r["sink_grad"]["ms"]
            hbm = float(pk["hbm_gbs"])
            out["sink_grad"] = {
                "ms": sms, "ms_pct": r["sink_grad"]["ms_pct"], "bytes": sbytes,
                "roofline": {"bound": "hbm", "achieved": sbytes / (sms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                             "frac": sbytes / (sms * 1e-3) / 1e9 / hbm, "kernel": "sink_grad_kernel",
                             "kernel_ms": sms, "peak_kind": f"copy, {pk_kind}", "traffic": None,
                             "note": "one block per query head over a few MB: launch- and latency-bound"}}
    roof["traffic"] = traffic_record(src, kname + "@" + w.name)
    roof["peak_kind"] = f"{'bf16 burst' if roof['bound'] == 'tensor' else 'copy'}, {pk_kind}"
    roof["kernel"] = kname
    roof["kernel_ms"] = ms_main
    out["roofline"] = roof
    out["stages_ms"] = {"preprocess": r["ms_pre"], "main": ms_main, "land": r["ms_land"]}
    out["ms_per_step"] = ms
    out["ms_per_step_pct"] = r["ms_step_pct"]
    out["main_ms_pct"] = r["ms_main_pct"]
    return out, flops


def workload_config(w):
    c = {"workload": w.name, "B": w.B, "S": w.S, "HQ": w.HQ, "HKV": w.HKV, "D": w.D, "causal": w.causal,
         "sm_scale": w.sm_scale}
    if w.kind == "sparse":
        c.update({"DV": w.Dv, "topk": w.topk})
    if w.window > 0:
        c["window"] = w.window
    if w.cu_seqlens is not None:
        c["cu_seqlens"] = list(w.cu_seqlens)
    c["l2"] = ("flushed before every step: a 256 MiB write, then a read of the same buffer, so the step starts "
               "from a cold L2 that holds no dirty line")
    c["timed"] = ("one call of the library's one-call entry point per step (its three launches: preprocess, main "
                  "kernel, landing); stages_ms comes from a second pass that launches them one by one")
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=MAIN_WORKLOAD, help="workload of the main line (profiling)")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch

    import __graft_entry__

    world, rank, local = dist_setup(args.gpus)
    __graft_entry__.build()
    from attention_backward_gb300 import inputs

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = inputs.WORKLOADS[args.workload]
    pk, pk_kind = peaks()
    timer = time_sparse if w.kind == "sparse" else time_dense

    clocks = ClockSampler(local)
    clocks.start()
    r = timer(w, args.steps, args.warmup, device, world)
    clk = clocks.stop()
    r["ms_step"], r["ms_main"] = reduce_max_over_ranks([r["ms_step"], r["ms_main"]], device)
    d, flops = describe(w, r, pk, pk_kind, world)
    line = {
        "metric": METRIC, "value": d["value"], "unit": d["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": workload_config(w),
        "ms_per_step_pct": r["ms_step_pct"], "roofline": d["roofline"], "stages_ms": d["stages_ms"],
    }
    if w.kind == "sparse":
        line["TFLOP/s"] = d["TFLOP/s"]
    else:
        line["forward"] = d.get("forward")
        line["sink_grad"] = d.get("sink_grad")
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(w, r["tensors"], max(3, args.steps // 4), device)
        per_step = d["value"] * r["ms_step"] / world  # this rank's units per step
        line["e2e"] = {"value": per_step * world / e2e_ms, "unit": d["unit"], "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
    else:
        line["e2e"] = None
    line["gpu_launches"] = 3 * args.steps
    line["clocks"] = clk
    del r
    torch.cuda.empty_cache()
    if not args.no_extra and world == 1:
        line["workloads"] = extra_workloads(w.name, max(5, args.steps // 2), args.warmup, device, pk, pk_kind,
                                            cpu=not args.no_cpu)
    if not args.no_cpu and world == 1 and rank == 0:
        line["cpu_baseline"] = cpu_baseline_entry(w)
    else:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()
    return 0


def cpu_baseline_entry(w):
    """The oracle timed on this host's cores on a bounded sample of ``w``."""
    cv, el, desc = cpu_oracle_sample(w)
    return {"value": cv, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
            "extrapolated": "whole heads" not in desc}


def extra_workloads(main_name, steps, warmup, device, pk, pk_kind, cpu=True):
    """The other workloads, same timing method, each with its own roofline and,
    with ``cpu``, the oracle timed beside it on a bounded sample."""
    import torch

    from attention_backward_gb300 import inputs

    out = {}
    for name, w in inputs.WORKLOADS.items():
        if name == main_name or name == "mha_causal_1x256x2x128_f16":  # the oracle-sized case is a parity case
            continue
        r = (time_sparse if w.kind == "sparse" else time_dense)(w, steps, warmup, device)
        d, _ = describe(w, r, pk, pk_kind)
        del r
        torch.cuda.empty_cache()
        d["config"] = workload_config(w)
        d["cpu_baseline"] = cpu_baseline_entry(w) if cpu else None
        out[name] = d
    return out


if __name__ == "__main__":
    sys.exit(main())
