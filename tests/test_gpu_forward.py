"""Parity of the dense CUDA forward (O and the natural-log LSE the backward
takes) with the CPU oracle's forward, element by element, through the C ABI.

Tolerance: O as the backward's outputs (|gpu - ref| <= atol + rtol |ref|, fp16
(5e-3, 1e-2), bf16 (1e-2, 2e-2)) against the float64 oracle; the LSE, an f32
sum of up to Sk exponentials per row on the GPU, within 2e-3 absolute (natural-
log units), -inf exactly where a query sees no key.
"""
import numpy as np
import pytest

import oracle
from attention_backward_gb300 import inputs

from _harness import TOL, assert_close, dense_problem, mask_of, torch_dtype
from test_gpu_dense import C1, C2, SMALL, UNEQUAL

pytestmark = pytest.mark.gpu

LSE_ATOL = 2e-3

CASES = SMALL + UNEQUAL


def _run_forward(w, q, k, v, poison=True):
    import torch

    import attention_backward_gb300 as ab

    dt = torch_dtype(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)  # noqa: E731
    tq, tk, tv = t(q), t(k), t(v)
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda") if w.cu_seqlens else None
    fill = float("nan") if poison else 0.0
    o = torch.full_like(tq, fill)
    lse = torch.full((w.B, w.HQ, w.S), fill, dtype=torch.float32, device="cuda")
    ws = torch.full((256,), 0xFF, dtype=torch.uint8, device="cuda")
    ab.attn_fwd_gqa(tq, tk, tv, o, lse, ws, w.sm_scale, w.causal, w.window, cu)
    ab.check_error(ws)
    return o, lse


def _check(w, o, lse, ro, rl, rows=None):
    """O within the dtype tolerance, LSE within LSE_ATOL, on the rows the
    oracle defines (all, or ``rows`` along S)."""
    go = o.float().cpu().numpy().astype(np.float64)
    gl = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        go, gl = go[:, rows], gl[:, :, rows]
        ro, rl = ro[:, rows], rl[:, :, rows]
    assert_close(go, np.asarray(ro, dtype=np.float64), w, "o")
    empty = np.isneginf(rl)
    assert (np.isneginf(gl) == empty).all(), "LSE -inf exactly where a query sees no key"
    assert not np.isnan(gl).any()
    err = np.abs(gl[~empty] - rl[~empty])
    assert err.max(initial=0.0) <= LSE_ATOL, f"lse max err {err.max():.3e}"
    assert (go[np.broadcast_to(empty.transpose(0, 2, 1)[..., None], go.shape)] == 0).all(), "O = 0 on empty rows"


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_matches_oracle(w):
    q, k, v, do = inputs.dense_inputs(w)
    ro, rl = oracle.forward(q, k, v, w.sm_scale, dtype=np.float64, **mask_of(w))
    o, lse = _run_forward(w, q, k, v)
    rows = None
    if w.cu_seqlens is not None:  # rows past the last sequence are not written
        rows = np.arange(w.cu_seqlens[-1])
    _check(w, o, lse, ro, rl, rows)


@pytest.mark.parametrize("tail", [37, 300])
def test_forward_rows_past_the_last_sequence_may_hold_nan(tail):
    """Q, K and V rows past the last packed sequence hold NaN: every row inside
    a sequence still matches the oracle, and the rows past the end are left as
    they were."""
    import torch

    w = inputs.scaled(W_VARLEN, name=f"fwd_tail{tail}", S=700 + tail, cu_seqlens=(0, 33, 161, 390, 700))
    q, k, v, do = inputs.dense_inputs(w)
    end = 700
    for a in (q, k, v):
        a[:, end:] = np.nan
    ro, rl = oracle.forward(q[:, :end], k[:, :end], v[:, :end], w.sm_scale, dtype=np.float64,
                            causal=w.causal, window=w.window, cu_seqlens=w.cu_seqlens)
    o, lse = _run_forward(w, q, k, v)
    _check(w, o[:, :end], lse[:, :, :end], ro, rl)
    assert torch.isnan(o[:, end:].float()).all() and torch.isnan(lse[:, :, end:]).all()


W_VARLEN = inputs.scaled(inputs.WORKLOADS["gqa_varlen_window1024_hq32_hkv8_d64_bf16"], HQ=4, HKV=2, window=100)


def test_forward_workload_mha_causal_2x2048x32x128_in_full():
    """The causal MHA workload at full size, every row, against the oracle's
    float32 forward (the one the backward's tests take O and LSE from)."""
    q, k, v, o_ref, do, lse_ref = dense_problem(C2)
    o, lse = _run_forward(C2, q, k, v)
    _check(C2, o, lse, o_ref, lse_ref)


def test_forward_output_feeds_the_backward():
    """The backward run on the GPU forward's O and LSE gives the oracle's
    gradients (the forward is what the backward's inputs come from)."""
    import torch

    import attention_backward_gb300 as ab
    from _harness import to_np

    w = inputs.scaled(C1, name="fwd_then_bwd", S=300, HQ=4, HKV=2)
    q, k, v, do = inputs.dense_inputs(w)
    o, lse = _run_forward(w, q, k, v)
    dt = torch_dtype(w)
    t = lambda a: torch.from_numpy(a).cuda().to(dt)  # noqa: E731
    dq, dk, dv = ab.backward(t(q), t(k), t(v), o, t(do), lse, w.sm_scale, causal=True)
    o64 = o.float().cpu().numpy().astype(np.float64)
    rq, rk, rv = oracle.backward(q, k, v, o64, do, lse.cpu().numpy(), w.sm_scale, causal=True)
    for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        assert_close(to_np(got), ref, w, name)
    assert TOL[w.dtype]
