"""Shared helpers of the GPU parity tests: seeded inputs, oracle references,
CUDA-path calls through the C ABI and the elementwise tolerance check.

Tolerance: |gpu - ref| <= atol + rtol * |ref| elementwise, ref the float64
oracle on the same 16-bit inputs; fp16 (5e-3, 1e-2), bf16 (1e-2, 2e-2).
"""
from __future__ import annotations

import functools

import numpy as np

import oracle
from attention_backward_gb300 import inputs

TOL = {"f16": (5e-3, 1e-2), "bf16": (1e-2, 2e-2)}


def torch_dtype(w):
    import torch

    return torch.float16 if w.dtype == "f16" else torch.bfloat16


def mask_of(w):
    return dict(causal=w.causal, window=w.window, cu_seqlens=w.cu_seqlens)


@functools.lru_cache(maxsize=4)
def dense_problem(w):
    """Inputs of workload ``w`` plus O and LSE from the oracle's float32 forward."""
    q, k, v, do = inputs.dense_inputs(w)
    o, lse = oracle.forward(q, k, v, w.sm_scale, **mask_of(w))
    o = inputs.round_to_dtype(o, w.dtype)
    return q, k, v, o, do, np.ascontiguousarray(lse, dtype=np.float32)


def sample_rows(S, n, seed, block=128, cu=None):
    """``n`` seeded positions plus every tile and sequence edge."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(S, size=min(n, S), replace=False).tolist())
    for e in range(0, S, block):
        rows.update({e, min(S - 1, e + block - 1), min(S - 1, e + 63), min(S - 1, e + 64)})
    if cu is not None:
        for x in cu:
            rows.update({max(0, x - 1), min(S - 1, x)})
    rows.update({0, S - 1})
    return np.array(sorted(rows))


def run_dense(w, problem, poison=True, workspace=None, stream=None, split=False):
    """The dense backward through the C ABI: the one-call attn_bwd_gqa, or with
    ``split`` its three launches one by one; outputs pre-filled with NaN so
    that any element the kernels fail to write shows up."""
    import torch

    import attention_backward_gb300 as ab

    q, k, v, o, do, lse = problem
    dt = torch_dtype(w)
    t = lambda a: torch.from_numpy(a).cuda().to(dt)  # noqa: E731
    tq, tk, tv, to, tdo = t(q), t(k), t(v), t(o), t(do)
    tl = torch.from_numpy(lse).cuda()
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda") if w.cu_seqlens else None
    fill = float("nan") if poison else 0.0
    dq = torch.full_like(tq, fill)
    dk = torch.full_like(tk, fill)
    dv = torch.full_like(tv, fill)
    ws = workspace if workspace is not None else ab._binding.new_gqa_workspace(w.B, w.S, w.HQ, w.D)
    if poison and workspace is None:
        ws.fill_(0xFF)
    if split:
        ab.preprocess(to, tdo, tl, ws, Dq=w.D, stream=stream)
        ab.gqa_main(tq, tk, tv, tdo, dk, dv, ws, w.sm_scale, w.causal, w.window, cu, stream)
        ab.dq_land(dq, ws, w.sm_scale, stream)
    else:
        ab.attn_bwd_gqa(tq, tk, tv, to, tdo, tl, dq, dk, dv, ws, w.sm_scale, w.causal, w.window, cu, stream)
    ab.check_error(ws, stream)
    return dq, dk, dv, ws


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, w, what):
    """Elementwise tolerance on every element the reference computed (NaN in
    ``ref`` marks rows the oracle skipped)."""
    atol, rtol = TOL[w.dtype]
    g = to_np(got) if not isinstance(got, np.ndarray) else got
    m = ~np.isnan(ref)
    assert m.any(), f"{what}: no reference elements"
    assert not np.isnan(g[m]).any(), f"{what}: {int(np.isnan(g[m]).sum())} unwritten/NaN elements"
    err = np.abs(g - np.where(m, ref, 0))
    bad = (err > atol + rtol * np.abs(np.where(m, ref, 0))) & m
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: gpu {g[tuple(i)]:.5g} ref {ref[tuple(i)]:.5g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {int(m.sum())} elements out of tolerance "
                             f"(max err {err[m].max():.3e}); e.g. {detail}")
    return float(err[m].max())


@functools.lru_cache(maxsize=2)
def sparse_problem(w, idx_override=None):
    """Inputs of a sparse workload plus O and LSE from the oracle's float32 forward."""
    q, kv, do, idx = inputs.sparse_inputs(w)
    if idx_override is not None:
        idx = np.array(idx_override, dtype=np.int32).reshape(idx.shape)
    o, lse = oracle.sparse_forward(q, kv, idx, w.sm_scale, w.Dv)
    o = inputs.round_to_dtype(o, w.dtype)
    return q, kv, do, idx, o, np.ascontiguousarray(lse, dtype=np.float32)


def run_sparse(w, problem, poison=True, split=False):
    """The sparse path through the C ABI (the one-call attn_bwd_sparse, or its
    three launches with ``split``), outputs NaN-poisoned."""
    import torch

    import attention_backward_gb300 as ab

    q, kv, do, idx, o, lse = problem
    dt = torch_dtype(w)
    t = lambda a: torch.from_numpy(a).cuda().to(dt)  # noqa: E731
    tq, tkv, tdo, to = t(q), t(kv), t(do), t(o)
    tidx = torch.from_numpy(idx).cuda()
    tl = torch.from_numpy(lse).cuda()
    B, S, H, DQK = q.shape
    SKV, HKV = kv.shape[1], kv.shape[2]
    dkv_elems = B * SKV * HKV * DQK
    ws = ab._binding.new_workspace(B, S, H, 0, dkv_elems)
    if poison:
        ws.fill_(0xFF)
    fill = float("nan") if poison else 0.0
    dq = torch.full_like(tq, fill)
    dkv = torch.full_like(tkv, fill)
    if split:
        ab.preprocess(to, tdo, tl, ws, Dq=0, dkv_elems=dkv_elems)
        ab.sparse_main(tq, tkv, tdo, tidx, dq, ws, w.sm_scale, w.Dv)
        ab.sparse_land(dkv, ws, B, S, H)
    else:
        ab.attn_bwd_sparse(tq, tkv, to, tdo, tl, tidx, dq, dkv, ws, w.sm_scale, w.Dv)
    ab.check_error(ws)
    return dq, dkv


def oracle_rows_chunked(problem, w, q_rows=None, k_rows=None, heads=None, chunk=1024):
    """The oracle's dQ rows ``q_rows`` and dK/dV rows ``k_rows`` (positions
    along S; None: none), evaluated ``chunk`` positions per call so that no
    call holds more than chunk x sequence-length score matrices; rows not
    asked for are NaN.  ``heads`` restricts the query heads as in
    oracle.backward (dK/dV rows of KV heads without a listed query head come
    back as zero)."""
    q, k, v, o, do, lse = problem
    out = None
    for which in ("q", "k"):
        rows = q_rows if which == "q" else k_rows
        if rows is None:
            continue
        rows = np.asarray(rows)
        for c0 in range(0, rows.size, chunk):
            r = rows[c0:c0 + chunk]
            part = oracle.backward(q, k, v, o, do, lse, w.sm_scale, heads=heads, **mask_of(w),
                                   **({"q_rows": r} if which == "q" else {"k_rows": r}))
            if out is None:
                out = [a.copy() for a in part]
            else:
                for a, b in zip(out, part):
                    m = ~np.isnan(b)
                    a[m] = b[m]
    return out
