"""attn_bwd_gqa_noalloc: the backward for callers that cannot allocate device
memory (a plugin inside a framework that owns all device memory through its
own pool, or a latency-critical loop that cannot take cudaMalloc's implicit
synchronisation).  It must give the same gradients as the entry points that
take a caller-provided workspace, call after call, although every call reuses
the library's one scratch array.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes when run alone.
"""
import ctypes

import pytest

from attention_backward_gb300 import inputs

from _harness import assert_close, dense_problem, run_dense, to_np, torch_dtype

pytestmark = pytest.mark.gpu

CASES = [
    inputs.scaled(inputs.WORKLOADS["gqa_1x16384_hq32_hkv4_d128_bf16"], name="gqa_d128_causal_s640",
                  S=640, HQ=8, HKV=2, causal=True),
    inputs.scaled(inputs.WORKLOADS["gqa_varlen_window1024_hq32_hkv8_d64_bf16"], name="varlen_window_d64",
                  S=900, HQ=4, HKV=2, window=200, cu_seqlens=(0, 333, 900)),
    inputs.WORKLOADS["mha_causal_1x256x2x128_f16"],
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_workspace_entry_points_twice(w):
    import torch

    import attention_backward_gb300 as ab

    prob = dense_problem(w)
    # reference: the existing entry points with a caller-provided workspace
    rq, rk, rv, _ = run_dense(w, prob)
    rq, rk, rv = to_np(rq), to_np(rk), to_np(rv)
    q, k, v, o, do, lse = prob
    dt = torch_dtype(w)
    t = lambda a: torch.from_numpy(a).cuda().to(dt)  # noqa: E731
    tq, tk, tv, to, tdo = t(q), t(k), t(v), t(o), t(do)
    tl = torch.from_numpy(lse).cuda()
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda") if w.cu_seqlens else None
    for call in range(2):  # the second call reuses the scratch the first one left behind
        dq, dk, dv = ab._binding.backward_noalloc(tq, tk, tv, to, tdo, tl, w.sm_scale, w.causal, w.window, cu)
        torch.cuda.synchronize()
        assert_close(dq, rq, w, f"dq (call {call})")
        assert_close(dk, rk, w, f"dk (call {call})")
        assert_close(dv, rv, w, f"dv (call {call})")
        # dK and dV are written once by their owning CTA: the same bits as the reference
        assert (to_np(dk) == rk).all() and (to_np(dv) == rv).all()
    # no kernel recorded an error in the library-held workspace
    code = ctypes.c_int32(-1)
    assert ab.library().attn_bwd_noalloc_check_error(None, ctypes.byref(code)) == 0
    assert code.value == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    """A problem whose workspace exceeds the library's scratch array is refused
    with ATTN_ERR_WORKSPACE before anything is queued."""
    import torch

    import attention_backward_gb300 as ab

    lib = ab.library()
    S = ab._binding.Strides
    B, Sq, H, D = 1, 8192, 16, 128  # needs about 64 MiB of workspace
    assert ab.workspace_size(B, Sq, H, D) > (32 << 20)
    x = torch.zeros(16, dtype=torch.float16, device="cuda")  # never read: the size check comes first
    st = S(Sq * H * D, H * D, D)
    sl = S(H * Sq, 1, Sq)
    m = ab._binding.Mask(1, -1, None, 0)
    p = x.data_ptr()
    code = lib.attn_bwd_gqa_noalloc(p, st, p, st, p, st, p, st, p, st, p, sl, B, Sq, H, H, D, 0, 0.1,
                                    ctypes.byref(m), p, st, p, st, p, st, None)
    assert code == 3, lib.attn_bwd_status_string(code)
