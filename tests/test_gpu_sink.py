"""Attention sinks on the GPU: with O and LSE from a sink-aware forward, the
dense backward's dQ, dK, dV and attn_bwd_sink_grad's dsink match the oracle
(its sink gradient is pinned to finite differences in test_oracle_pins)."""
import numpy as np
import pytest

import oracle
from attention_backward_gb300 import inputs

from _harness import assert_close, mask_of, to_np, torch_dtype

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS
C1 = W["mha_causal_1x256x2x128_f16"]
C4 = W["gqa_varlen_window1024_hq32_hkv8_d64_bf16"]

CASES = [
    (inputs.scaled(C1, name="sink_causal_b2_s300_gqa_f16", B=2, S=300, HQ=4, HKV=2), 0),
    (inputs.scaled(C1, name="sink_noncausal_s200_bf16", S=200, HQ=2, HKV=1, causal=False, dtype="bf16"), 0),
    # packed, head dim 64, a window, 50 rows past the last sequence holding NaN
    (inputs.scaled(C4, name="sink_varlen_d64_w100_tail", S=700, HQ=4, HKV=2, window=100,
                   cu_seqlens=(0, 33, 161, 390, 650)), 50),
]


@pytest.mark.parametrize("w,tail", CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_sink_gradients_match_oracle(w, tail):
    import torch

    import attention_backward_gb300 as ab

    q, k, v, do = inputs.dense_inputs(w)
    sink = np.random.default_rng(w.seed).standard_normal(w.HQ).astype(np.float32) + 1.0
    o, lse = oracle.forward(q, k, v, w.sm_scale, sink=sink, **mask_of(w))
    o = inputs.round_to_dtype(o, w.dtype)
    lse = np.ascontiguousarray(lse, dtype=np.float32)
    dt = torch_dtype(w)
    t = lambda a: torch.from_numpy(a).cuda().to(dt)  # noqa: E731
    tq, tk, tv, to, tdo = t(q), t(k), t(v), t(o), t(do)
    tl = torch.from_numpy(lse).cuda()
    if tail:
        end = w.S - tail
        for x in (tq, tk, tv, to, tdo):
            x[:, end:] = float("nan")
        tl[:, :, end:] = float("nan")
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda") if w.cu_seqlens else None
    dq, dk, dv = (torch.full_like(x, float("nan")) for x in (tq, tk, tv))
    ws = ab._binding.new_gqa_workspace(w.B, w.S, w.HQ, w.D)
    ab.attn_bwd_gqa(tq, tk, tv, to, tdo, tl, dq, dk, dv, ws, w.sm_scale, w.causal, w.window, cu)
    tsink = torch.from_numpy(sink).cuda()
    dsink = ab.sink_grad(tsink, ws, w.B, w.S, cu)
    ab.check_error(ws)
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")
    want = oracle.sink_grad(o, do, lse, sink, w.cu_seqlens)
    got = to_np(dsink)
    # delta is formed in f32 from the same 16-bit O and dO on both sides; the
    # sum runs over at most a few thousand rows
    np.testing.assert_allclose(got, want, rtol=2e-4, atol=1e-4 * max(1.0, float(np.abs(want).max())))
    # the same workspace and inputs give the same dsink again (fixed order of additions)
    assert torch.equal(ab.sink_grad(tsink, ws, w.B, w.S, cu), dsink)
