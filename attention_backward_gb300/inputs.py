"""Seeded synthetic inputs for the attention backward.

This module is the only code shared by the CPU oracle and the CUDA path's
harnesses (tests, bench, smoke). It holds random number generation, 16-bit
rounding of the generated values and the workload shapes, and none of the
attention arithmetic: the forward that produces O and the log-sum-exp lives
with the oracle, and the gradients live in the kernels.

Generator: SplitMix64 over a counter, as published by Steele, Lea and Flood
("Fast splittable pseudorandom number generators", OOPSLA 2014), turned into
normal deviates with the Box-Muller transform in float64, then rounded to
float32 and from there, round-to-nearest-even, to fp16 or bf16.  Every tensor
draws from its own stream keyed by (seed, tensor id), so tensors are
independent of one another and of their generation order.

Workload shapes follow the five workloads these gradients are checked and
timed on: causal MHA 1x256x2x128 and 2x2048x32x128 fp16 (the TileOPs MHA
backward PR, test and "llama-8b-long" benchmark rows), dense GQA 1x16384
HQ32/Hkv4 D128 bf16 (the flash-linear-attention KV-head-owned dKV issue,
"Problem"), packed-varlen sliding-window GQA (same issue, "Frozen
correctness contract") and top-k sparse MLA (the tilelang sparse MLA
backward PR, "Benchmark").
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

_MASK64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def splitmix64(counter: np.ndarray) -> np.ndarray:
    """SplitMix64 output function applied to ``counter * golden + golden``."""
    with np.errstate(over="ignore"):
        z = (counter.astype(np.uint64) + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def _stream_base(seed: int, tensor_id: int) -> np.uint64:
    key = splitmix64(np.array([(seed & 0xFFFFFFFF) << 20 | (tensor_id & 0xFFFFF)], dtype=np.uint64))[0]
    return np.uint64(int(key) & 0xFFFFFFFF00000000)


def uniform_u64(seed: int, tensor_id: int, n: int) -> np.ndarray:
    """``n`` 64-bit words from stream (seed, tensor_id)."""
    base = _stream_base(seed, tensor_id)
    with np.errstate(over="ignore"):
        ctr = base + np.arange(n, dtype=np.uint64)
    return splitmix64(ctr)


def normal_f32(seed: int, tensor_id: int, shape: Sequence[int], chunk: int = 1 << 20) -> np.ndarray:
    """iid N(0, 1) as float32: Box-Muller in float64 on pairs of 53-bit uniforms.

    Value n of the stream depends only on (seed, tensor_id, n); chunks are
    filled by a thread pool.
    """
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)
    half = (n + 1) // 2
    base = _stream_base(seed, tensor_id)
    two_pi = 2.0 * math.pi

    def fill(start):
        m = min(chunk, half - start)
        with np.errstate(over="ignore"):
            ctr = base + np.uint64(2 * start) + np.arange(2 * m, dtype=np.uint64)
        words = splitmix64(ctr)
        u = ((words >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * m, dtype=np.float64)
        z[0::2] = r * np.cos(two_pi * u2)
        z[1::2] = r * np.sin(two_pi * u2)
        lo = 2 * start
        hi = min(n, lo + 2 * m)
        out[lo:hi] = z[: hi - lo].astype(np.float32)

    starts = list(range(0, half, chunk))
    if len(starts) <= 1:
        for s0 in starts:
            fill(s0)
    else:
        with ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
            list(ex.map(fill, starts))
    return out.reshape(shape)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16/bf16 (round-to-nearest-even) and return them
    widened back to float32, so every value is exactly representable in ``dtype``."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        # RNE on the bit pattern: add 0x7FFF plus the lowest kept bit, then
        # truncate.  For finite values the sum stays below 2^32; NaNs are kept.
        u = x.reshape(-1).view(np.uint32).copy()

        def rne(a, e):
            c = u[a:e]
            lsb = (c >> np.uint32(16)) & np.uint32(1)
            nan = (c & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
            keep = c[nan]
            c += np.uint32(0x7FFF)
            c += lsb
            c &= np.uint32(0xFFFF0000)
            c[nan] = keep

        step = 1 << 22
        with ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
            list(ex.map(lambda a: rne(a, min(a + step, u.size)), range(0, u.size, step)))
        return u.view(np.float32).reshape(x.shape)
    if dtype == "f32":
        return x
    raise ValueError(f"unknown dtype {dtype}")


def topk_index_sets(seed: int, tensor_id: int, s: int, topk: int) -> np.ndarray:
    """Top-k index lists, int32 [s, topk].

    Row t holds all of [0, t] followed by -1 when t < topk; otherwise ``topk``
    distinct indices drawn uniformly from [0, t] (the ``topk`` smallest of t+1
    seeded random keys), sorted ascending.
    """
    idx = np.full((s, topk), -1, dtype=np.int32)
    for t in range(s):
        n = t + 1
        if n <= topk:
            idx[t, :n] = np.arange(n, dtype=np.int32)
        else:
            keys = uniform_u64(seed, tensor_id * 65536 + t, n)
            pick = np.argpartition(keys, topk - 1)[:topk]
            idx[t] = np.sort(pick).astype(np.int32)
    return idx


@dataclasses.dataclass(frozen=True)
class Workload:
    """One backward problem: shapes, dtype, mask and the seed of its inputs."""

    name: str
    kind: str  # "dense" or "sparse"
    B: int
    S: int
    HQ: int
    HKV: int
    D: int  # head dim of Q and K (DQK for sparse)
    Dv: int  # head dim of V, O and dO
    dtype: str  # "f16" or "bf16"
    causal: bool
    window: int = -1  # -1: no window; W: i - W < j <= i
    cu_seqlens: Optional[tuple] = None  # packed varlen (B == 1)
    topk: int = 0  # sparse only
    seed: int = 0
    Sk: int = 0  # key/value length of a dense row when it differs from S (0: S)

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def G(self) -> int:
        return self.HQ // self.HKV

    @property
    def skv(self) -> int:
        """Key/value rows per batch row."""
        return self.Sk if self.Sk > 0 else self.S


# The five workloads.  Seeds follow "20260000 + k" for workload k.
WORKLOADS = {
    "mha_causal_1x256x2x128_f16": Workload(
        "mha_causal_1x256x2x128_f16", "dense", 1, 256, 2, 2, 128, 128, "f16", True, seed=20260000),
    "mha_causal_2x2048x32x128_f16": Workload(
        "mha_causal_2x2048x32x128_f16", "dense", 2, 2048, 32, 32, 128, 128, "f16", True, seed=20260001),
    "gqa_1x16384_hq32_hkv4_d128_bf16": Workload(
        "gqa_1x16384_hq32_hkv4_d128_bf16", "dense", 1, 16384, 32, 4, 128, 128, "bf16", False, seed=20260002),
    "gqa_varlen_window1024_hq32_hkv8_d64_bf16": Workload(
        "gqa_varlen_window1024_hq32_hkv8_d64_bf16", "dense", 1, 16384, 32, 8, 64, 64, "bf16", True,
        window=1024, cu_seqlens=(0, 3000, 8000, 9537, 16384), seed=20260003),
    "sparse_mla_s4096_h64_topk2048_bf16": Workload(
        "sparse_mla_s4096_h64_topk2048_bf16", "sparse", 1, 4096, 64, 1, 576, 512, "bf16", False,
        topk=2048, seed=20260004),
}

# tensor ids inside a workload's seed
T_Q, T_K, T_V, T_DO, T_IDX = 1, 2, 3, 4, 5


def dense_inputs(w: Workload):
    """Q [B,S,HQ,D], K [B,Sk,HKV,D], V [B,Sk,HKV,Dv], dO [B,S,HQ,Dv] as float32
    arrays holding values exactly representable in ``w.dtype`` (Sk = w.skv)."""
    q = round_to_dtype(normal_f32(w.seed, T_Q, (w.B, w.S, w.HQ, w.D)), w.dtype)
    k = round_to_dtype(normal_f32(w.seed, T_K, (w.B, w.skv, w.HKV, w.D)), w.dtype)
    v = round_to_dtype(normal_f32(w.seed, T_V, (w.B, w.skv, w.HKV, w.Dv)), w.dtype)
    do = round_to_dtype(normal_f32(w.seed, T_DO, (w.B, w.S, w.HQ, w.Dv)), w.dtype)
    return q, k, v, do


def sparse_inputs(w: Workload):
    """Q [B,S,H,DQK], KV [B,S,HKV,DQK], dO [B,S,H,DV] (float32 holding 16-bit
    values) and the index lists int32 [B,S,HKV,topk]."""
    q = round_to_dtype(normal_f32(w.seed, T_Q, (w.B, w.S, w.HQ, w.D)), w.dtype)
    kv = round_to_dtype(normal_f32(w.seed, T_K, (w.B, w.S, w.HKV, w.D)), w.dtype)
    do = round_to_dtype(normal_f32(w.seed, T_DO, (w.B, w.S, w.HQ, w.Dv)), w.dtype)
    idx = np.empty((w.B, w.S, w.HKV, w.topk), dtype=np.int32)
    for b in range(w.B):
        for g in range(w.HKV):
            idx[b, :, g, :] = topk_index_sets(w.seed, T_IDX + 16 * (b * w.HKV + g), w.S, w.topk)
    return q, kv, do, idx


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)
