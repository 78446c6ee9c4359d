"""attn_bwd_gqa_host: the dense backward from host buffers to host buffers,
chunk by chunk of batch rows and KV heads with the copies overlapped with the
kernels.  Every
chunk runs the same kernels on the same tiles as a single call, so dK and dV
(written once per tile) must be bit-identical to the device path; dQ (summed
from key tiles in a scheduling-dependent order) is checked against the oracle.
"""
import pytest

import oracle
from attention_backward_gb300 import inputs

from _harness import assert_close, dense_problem, run_dense, to_np, torch_dtype

pytestmark = pytest.mark.gpu

C1 = inputs.WORKLOADS["mha_causal_1x256x2x128_f16"]
C3 = inputs.WORKLOADS["gqa_1x16384_hq32_hkv4_d128_bf16"]
C4 = inputs.WORKLOADS["gqa_varlen_window1024_hq32_hkv8_d64_bf16"]

CASES = [
    (C1, 1),
    # 4 KV heads in chunks of 2 (asking for 3 chunks gives 2 chunks of 2 heads)
    (inputs.scaled(C3, name="gqa_g2_s384_bf16", S=384, HQ=8, HKV=4), 3),
    (inputs.scaled(C3, name="gqa_g4_causal_b2_f16", B=2, S=300, HQ=16, HKV=4, causal=True, dtype="f16"), 4),
    # more chunks than KV heads: one KV head per chunk
    (inputs.scaled(C4, name="varlen_window_d64", S=900, HQ=4, HKV=2, window=200, cu_seqlens=(0, 333, 900)), 8),
    # batch rows split first: 3 rows x 2 ranges of KV heads; and fewer chunks than rows (2 rows per chunk)
    (inputs.scaled(C3, name="gqa_b3_causal_f16", B=3, S=260, HQ=8, HKV=4, causal=True, dtype="f16"), 6),
    (inputs.scaled(C3, name="gqa_b3_rows_per_chunk_bf16", B=3, S=200, HQ=4, HKV=2), 2),
]


@pytest.mark.parametrize("w,chunks", CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_host_path_matches_device_path_and_oracle(w, chunks):
    import torch

    import attention_backward_gb300 as ab

    prob = dense_problem(w)
    _, rk, rv, _ = run_dense(w, prob)
    q, k, v, o, do, lse = prob
    dt = torch_dtype(w)
    h = lambda a: torch.from_numpy(a).to(dt).contiguous().pin_memory()  # noqa: E731
    hl = torch.from_numpy(lse).contiguous().pin_memory()
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda") if w.cu_seqlens else None
    dq, dk, dv = ab.backward_host(h(q), h(k), h(v), h(o), h(do), hl, w.sm_scale, w.causal, w.window, cu,
                                  chunks=chunks)
    assert not dq.is_cuda
    assert (dk.view(torch.int16) == rk.cpu().view(torch.int16)).all()
    assert (dv.view(torch.int16) == rv.cpu().view(torch.int16)).all()
    oq, _, _ = oracle.backward(q, k, v, o, do, lse, w.sm_scale, causal=w.causal, window=w.window,
                               cu_seqlens=w.cu_seqlens)
    assert_close(dq, oq, w, "dq")


def test_host_path_reuses_buffers_and_streams():
    """Two calls with caller-owned outputs, scratch and streams give the same
    dK/dV bits; the scratch starts with the workspace, so its error word reads
    clean."""
    import torch

    import attention_backward_gb300 as ab

    w = inputs.scaled(C3, name="gqa_reuse", S=256, HQ=8, HKV=2)
    q, k, v, o, do, lse = dense_problem(w)
    dt = torch_dtype(w)
    h = lambda a: torch.from_numpy(a).to(dt).contiguous().pin_memory()  # noqa: E731
    args = (h(q), h(k), h(v), h(o), h(do), torch.from_numpy(lse).contiguous().pin_memory())
    out = tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in args[:3])
    scratch = torch.empty(ab.host_scratch_size(w.B, w.S, w.HQ, w.HKV, w.D, 2), dtype=torch.uint8, device="cuda")
    streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
    first = [t.clone() for t in ab.backward_host(*args, w.sm_scale, chunks=2, out=out, scratch=scratch,
                                                 streams=streams)]
    second = ab.backward_host(*args, w.sm_scale, chunks=2, out=out, scratch=scratch, streams=streams)
    assert (first[1].view(torch.int16) == second[1].view(torch.int16)).all()
    assert (first[2].view(torch.int16) == second[2].view(torch.int16)).all()
    ab.check_error(scratch, streams[0])
    assert_close(second[0], to_np(first[0]), w, "dq (second call)")
