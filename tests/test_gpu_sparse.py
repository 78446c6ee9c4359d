"""Parity of the top-k sparse CUDA path (preprocess, sparse kernel, dKV landing)
with the CPU oracle, through the C ABI on a GPU."""
import numpy as np
import pytest

import oracle
from attention_backward_gb300 import inputs

from _harness import assert_close, run_sparse, sample_rows, sparse_problem, to_np

pytestmark = pytest.mark.gpu

C5 = inputs.WORKLOADS["sparse_mla_s4096_h64_topk2048_bf16"]

SMALL = [
    inputs.scaled(C5, name="s300_topk128", S=300, topk=128),
    inputs.scaled(C5, name="s260_topk200_f16", S=260, topk=200, dtype="f16"),
    inputs.scaled(C5, name="s150_topk256_hkv2_b2", B=2, S=150, HQ=128, HKV=2, topk=256),
    # groups smaller than 64 heads (tensor-parallel splits), computed padded to 64:
    # padding past the last head (zero-filled), padding taken from the next group's
    # heads, and a group size that is not a power of two
    inputs.scaled(C5, name="s200_h32_topk128", S=200, HQ=32, HKV=1, topk=128),
    inputs.scaled(C5, name="s180_h64_hkv4_topk96_f16", S=180, HQ=64, HKV=4, topk=96, dtype="f16"),
    inputs.scaled(C5, name="s160_h48_hkv2_topk130", S=160, HQ=48, HKV=2, topk=130),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_sparse_cases_match_oracle(w):
    prob = sparse_problem(w)
    q, kv, do, idx, o, lse = prob
    rq, rkv = oracle.sparse_backward(q, kv, o, do, lse, idx, w.sm_scale, w.Dv)
    dq, dkv = run_sparse(w, prob)
    assert_close(dq, rq, w, "dq")
    assert_close(dkv, rkv, w, "dkv")


def test_sparse_split_launches_match_one_call():
    """attn_bwd_preprocess, attn_bwd_sparse_main and attn_bwd_sparse_land one
    by one give what the one-call attn_bwd_sparse gives (dQ is written once per
    token: the same bits; dKV within tolerance of the oracle)."""
    w = inputs.scaled(C5, name="split_s200", S=200, topk=128)
    prob = sparse_problem(w)
    q, kv, do, idx, o, lse = prob
    a = run_sparse(w, prob)
    b = run_sparse(w, prob, split=True)
    assert (to_np(a[0]) == to_np(b[0])).all()
    _, rkv = oracle.sparse_backward(q, kv, o, do, lse, idx, w.sm_scale, w.Dv)
    assert_close(b[1], rkv, w, "dkv (split launches)")


def test_sparse_edge_index_lists():
    """Repeated indices count as separate slots, out-of-range indices and -1
    are not visible, and a token with no visible slot gets dQ = 0."""
    w = inputs.scaled(C5, name="edges", S=140, topk=130)
    _, _, _, idx = inputs.sparse_inputs(w)
    idx = idx.copy()
    idx[0, 100, 0, 5] = idx[0, 100, 0, 4]      # a repeated row
    idx[0, 101, 0, 7] = w.S + 3                # out of range
    idx[0, 102, 0, :] = -1                     # nothing visible
    idx[0, 103, 0, 129] = 50                   # a valid slot in the partial last block
    prob = sparse_problem(w, tuple(idx.ravel().tolist()))
    q, kv, do, idx2, o, lse = prob
    rq, rkv = oracle.sparse_backward(q, kv, o, do, lse, idx2, w.sm_scale, w.Dv)
    rq = np.nan_to_num(rq)  # token 102 has no visible slot: its gradient is zero
    dq, dkv = run_sparse(w, prob)
    assert np.all(to_np(dq)[0, 102] == 0)
    assert_close(dq, rq, w, "dq")
    assert_close(dkv, rkv, w, "dkv")


def test_sparse_workload_4096_sampled():
    """The full sparse workload: dQ of 512 seeded tokens and dKV of 512 seeded
    latent rows (plus every 128-row tile edge and the rows 0, 1, 2047, 2048,
    4095, where the index lists change from full prefixes to sampled sets)
    against the oracle, and the column sums of dKV on every row."""
    w = C5
    prob = sparse_problem(w)
    q, kv, do, idx, o, lse = prob
    dq, dkv = run_sparse(w, prob)
    edge = [0, 1, 2047, 2048, w.S - 1]
    toks = np.union1d(sample_rows(w.S, 512, w.seed), edge)
    rows = np.union1d(sample_rows(w.S, 512, w.seed + 1), edge)
    rq, _ = oracle.sparse_backward(q, kv, o, do, lse, idx, w.sm_scale, w.Dv, tokens=toks)
    _, rkv = oracle.sparse_backward(q, kv, o, do, lse, idx, w.sm_scale, w.Dv, kv_rows=rows)
    assert_close(dq, rq, w, "dq (sampled tokens)")
    assert_close(dkv, rkv, w, "dkv (sampled rows)")
    # every token sees at least one row, so the V part of dKV sums to sum(dO)
    # and the K part (rows of dS sum to zero) to zero
    g = to_np(dkv)[0, :, 0]
    n = w.S * w.HQ
    np.testing.assert_allclose(g[:, :w.Dv].sum(0), do.astype(np.float64).sum(axis=(0, 1, 2)), atol=4e-3 * np.sqrt(n) * 4)
    np.testing.assert_allclose(g[:, w.Dv:].sum(0), 0.0, atol=4e-3 * np.sqrt(n) * 4)
