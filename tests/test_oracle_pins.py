"""Pins of the CPU oracle to facts other than itself.

The pages print no output values for any input, so every pin here is a
mathematical fact about the backward of softmax attention: finite differences
of L = sum(O * dO), closed forms on special cases, and invariants.  Each is
chosen so that a dropped term, a wrong sign, a swapped index or a transposed
operand in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from attention_backward_gb300 import inputs


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _loss_dense(q, k, v, do, scale, **mask):
    o, _ = oracle.forward(q, k, v, scale, dtype=np.float64, **mask)
    return float((o * do).sum())


def _fd_grad(f, x, h=1e-5):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = f()
        x[i] = old - h
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


DENSE_CASES = [
    dict(B=1, S=5, HQ=1, HKV=1, D=3, Dv=3, mask=dict(causal=False)),
    dict(B=2, S=4, HQ=1, HKV=1, D=3, Dv=2, mask=dict(causal=True)),
    dict(B=1, S=7, HQ=2, HKV=1, D=2, Dv=3, mask=dict(causal=True, window=2, cu_seqlens=(0, 3, 7))),
    dict(B=1, S=6, HQ=4, HKV=2, D=3, Dv=3, mask=dict(causal=False, cu_seqlens=(0, 1, 6))),
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: f"S{c['S']}H{c['HQ']}/{c['HKV']}{c['mask']}")
def test_dense_backward_matches_finite_differences(case):
    """dQ, dK, dV equal the central differences of L = sum(O * dO), O recomputed by the forward."""
    rng = np.random.default_rng(7)
    B, S, HQ, HKV, D, Dv = (case[x] for x in ("B", "S", "HQ", "HKV", "D", "Dv"))
    q, k = _rand(rng, B, S, HQ, D), _rand(rng, B, S, HKV, D)
    v, do = _rand(rng, B, S, HKV, Dv), _rand(rng, B, S, HQ, Dv)
    scale = 0.7
    mask = case["mask"]
    o, lse = oracle.forward(q, k, v, scale, dtype=np.float64, **mask)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, scale, **mask)
    f = lambda: _loss_dense(q, k, v, do, scale, **mask)  # noqa: E731
    for got, x in ((dq, q), (dk, k), (dv, v)):
        want = _fd_grad(f, x)
        np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-8)


# keys outnumbering the queries and the other way round (dense rows; the masks
# are aligned at the end of the row)
UNEQUAL_CASES = [
    dict(Sq=3, Sk=6, HQ=1, HKV=1, mask=dict(causal=True)),
    dict(Sq=6, Sk=4, HQ=2, HKV=1, mask=dict(causal=True)),
    dict(Sq=4, Sk=7, HQ=2, HKV=2, mask=dict(causal=True, window=3)),
    dict(Sq=5, Sk=3, HQ=1, HKV=1, mask=dict(causal=False)),
]


@pytest.mark.parametrize("case", UNEQUAL_CASES, ids=lambda c: f"Sq{c['Sq']}Sk{c['Sk']}{c['mask']}")
def test_unequal_lengths_backward_matches_finite_differences(case):
    """With Sk != Sq, dQ [Sq], dK and dV [Sk] equal the central differences of
    L = sum(O * dO), O recomputed by the forward under the end-aligned mask."""
    rng = np.random.default_rng(17)
    Sq, Sk, HQ, HKV, D, Dv = case["Sq"], case["Sk"], case["HQ"], case["HKV"], 3, 2
    q, k = _rand(rng, 2, Sq, HQ, D), _rand(rng, 2, Sk, HKV, D)
    v, do = _rand(rng, 2, Sk, HKV, Dv), _rand(rng, 2, Sq, HQ, Dv)
    scale, mask = 0.6, case["mask"]
    o, lse = oracle.forward(q, k, v, scale, dtype=np.float64, **mask)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, scale, **mask)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    f = lambda: _loss_dense(q, k, v, do, scale, **mask)  # noqa: E731
    for got, x in ((dq, q), (dk, k), (dv, v)):
        np.testing.assert_allclose(got, _fd_grad(f, x), rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("window", [-1, 3])
def test_fewer_queries_equal_the_last_rows_of_the_square_problem(window):
    """End alignment, checked against the square (Sq == Sk) causal evaluation:
    Sq < Sk queries are the last Sq rows of an Sk x Sk problem whose other rows
    carry dO = 0 (so they add nothing to dK, dV).  O, LSE, dQ of those rows and
    all of dK, dV must agree."""
    rng = np.random.default_rng(19)
    Sq, Sk, D = 4, 9, 3
    q_full, k, v = _rand(rng, 1, Sk, 2, D), _rand(rng, 1, Sk, 1, D), _rand(rng, 1, Sk, 1, D)
    do_full = _rand(rng, 1, Sk, 2, D)
    do_full[:, :Sk - Sq] = 0.0
    q, do = q_full[:, Sk - Sq:], do_full[:, Sk - Sq:]
    mask = dict(causal=True, window=window)
    o_full, lse_full = oracle.forward(q_full, k, v, 0.5, dtype=np.float64, **mask)
    o, lse = oracle.forward(q, k, v, 0.5, dtype=np.float64, **mask)
    np.testing.assert_allclose(o, o_full[:, Sk - Sq:], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_full[:, :, Sk - Sq:], rtol=1e-12, atol=1e-14)
    gq, gk, gv = oracle.backward(q_full, k, v, o_full, do_full, lse_full, 0.5, **mask)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, 0.5, **mask)
    np.testing.assert_allclose(dq, gq[:, Sk - Sq:], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, gk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, gv, rtol=1e-10, atol=1e-12)


def test_more_queries_than_keys_leave_the_first_rows_empty():
    """Sq > Sk under the end-aligned causal mask: the first Sq - Sk queries see
    no key (LSE = -inf, O = 0, dQ = 0, nothing added to dK, dV) and the last Sk
    queries behave as the square Sk x Sk causal problem."""
    rng = np.random.default_rng(29)
    Sq, Sk, D = 7, 4, 3
    q, k, v, do = _rand(rng, 1, Sq, 1, D), _rand(rng, 1, Sk, 1, D), _rand(rng, 1, Sk, 1, D), _rand(rng, 1, Sq, 1, D)
    o, lse = oracle.forward(q, k, v, 0.5, dtype=np.float64, causal=True)
    assert np.isneginf(lse[:, :, :Sq - Sk]).all() and (o[:, :Sq - Sk] == 0).all()
    o2, lse2 = oracle.forward(q[:, Sq - Sk:], k, v, 0.5, dtype=np.float64, causal=True)
    np.testing.assert_allclose(o[:, Sq - Sk:], o2, rtol=1e-12, atol=1e-14)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, 0.5, causal=True)
    gq, gk, gv = oracle.backward(q[:, Sq - Sk:], k, v, o2, do[:, Sq - Sk:], lse2, 0.5, causal=True)
    assert (dq[:, :Sq - Sk] == 0).all()
    np.testing.assert_allclose(dq[:, Sq - Sk:], gq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, gk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, gv, rtol=1e-10, atol=1e-12)


def test_one_query_sees_every_key():
    """A single query against Sk keys under the end-aligned causal mask sees all
    of them: the same O, LSE and gradients as the unmasked evaluation."""
    rng = np.random.default_rng(23)
    q, k, v, do = _rand(rng, 1, 1, 2, 4), _rand(rng, 1, 6, 1, 4), _rand(rng, 1, 6, 1, 3), _rand(rng, 1, 1, 2, 3)
    a = oracle.forward(q, k, v, 0.5, dtype=np.float64, causal=True)
    b = oracle.forward(q, k, v, 0.5, dtype=np.float64, causal=False)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12)
    ga = oracle.backward(q, k, v, a[0], do, a[1], 0.5, causal=True)
    gb = oracle.backward(q, k, v, b[0], do, b[1], 0.5, causal=False)
    for x, y in zip(ga, gb):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)


def test_sparse_backward_matches_finite_differences():
    """Sparse dQ and dKV (dK plus dV on the first DV columns) against finite differences,
    with -1 padding, an out-of-range index and a repeated index in the lists."""
    rng = np.random.default_rng(11)
    B, S, SKV, H, HKV, DQK, DV = 1, 4, 5, 2, 1, 4, 3
    q, kv, do = _rand(rng, B, S, H, DQK), _rand(rng, B, SKV, HKV, DQK), _rand(rng, B, S, H, DV)
    idx = np.array([[0, -1, -1], [1, 0, 7], [2, 2, 4], [3, 1, -1]], dtype=np.int32).reshape(B, S, HKV, 3)
    scale = 0.5

    def loss():
        o, _ = oracle.sparse_forward(q, kv, idx, scale, DV, dtype=np.float64)
        return float((o * do).sum())

    o, lse = oracle.sparse_forward(q, kv, idx, scale, DV, dtype=np.float64)
    dq, dkv = oracle.sparse_backward(q, kv, o, do, lse, idx, scale, DV)
    np.testing.assert_allclose(dq, _fd_grad(loss, q), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dkv, _fd_grad(loss, kv), rtol=1e-6, atol=1e-8)


def test_forward_rows_normalise_and_two_key_closed_form():
    """P rows sum to one; a causal first row copies v_0; the second row is the
    two-key logistic mix with LSE = log(e^a + e^b)."""
    rng = np.random.default_rng(3)
    q, k, v = _rand(rng, 1, 6, 1, 4), _rand(rng, 1, 6, 1, 4), _rand(rng, 1, 6, 1, 5)
    scale = 0.3
    o, lse = oracle.forward(q, k, v, scale, causal=True, dtype=np.float64)
    a = scale * q[0, 1, 0] @ k[0, 0, 0]
    b = scale * q[0, 1, 0] @ k[0, 1, 0]
    sig = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], scale * q[0, 0, 0] @ k[0, 0, 0], rtol=1e-14)
    np.testing.assert_allclose(o[0, 1, 0], sig * v[0, 0, 0] + (1 - sig) * v[0, 1, 0], rtol=1e-13)
    np.testing.assert_allclose(lse[0, 0, 1], math.log(math.exp(a) + math.exp(b)), rtol=1e-13)
    s = scale * np.einsum("id,jd->ij", q[0, :, 0], k[0, :, 0])
    m = np.tril(np.ones((6, 6), bool))
    rowsum = np.where(m, np.exp(s - lse[0, 0][:, None]), 0).sum(1)
    np.testing.assert_allclose(rowsum, 1.0, rtol=1e-13)


def test_forward_matches_explicit_loops_on_varlen_window():
    """The forward's per-sequence evaluation equals explicit loops over the
    brute-force visibility matrix."""
    rng = np.random.default_rng(5)
    S, cu, W = 9, (0, 4, 9), 3
    q, k, v = _rand(rng, 1, S, 2, 3), _rand(rng, 1, S, 1, 3), _rand(rng, 1, S, 1, 2)
    o, lse = oracle.forward(q, k, v, 0.9, causal=True, window=W, cu_seqlens=cu, dtype=np.float64)
    M = oracle.visible(S, True, W, cu)
    for h in range(2):
        for i in range(S):
            js = [j for j in range(S) if M[i, j]]
            w = [math.exp(0.9 * float(q[0, i, h] @ k[0, j, 0])) for j in js]
            z = sum(w)
            assert abs(lse[0, h, i] - math.log(z)) < 1e-12
            want = sum(wj / z * v[0, j, 0] for wj, j in zip(w, js))
            np.testing.assert_allclose(o[0, i, h], want, rtol=1e-12)


def test_visibility_window_and_sequence_bounds():
    """Query i sees exactly the keys i-W+1 .. i of its own sequence."""
    cu = (0, 33, 161, 390)  # the unequal packed lengths of the FLA issue's failing case
    W = 17
    M = oracle.visible(390, True, W, cu)
    for a, e in zip(cu[:-1], cu[1:]):
        for i in range(a, e):
            want = np.zeros(390, bool)
            want[max(a, i - W + 1):i + 1] = True
            assert (M[i] == want).all(), i
    Mc = oracle.visible(10, True, -1, None)
    assert (Mc == np.tril(np.ones((10, 10), bool))).all()
    assert oracle.visible(5, False, -1, None).all()


def test_single_position_closed_form():
    """S = 1: P = 1, so dV = dO, while dS = dP - delta = 0 gives dQ = dK = 0."""
    rng = np.random.default_rng(2)
    q, k, v, do = _rand(rng, 1, 1, 2, 4), _rand(rng, 1, 1, 1, 4), _rand(rng, 1, 1, 1, 4), _rand(rng, 1, 1, 2, 4)
    o, lse = oracle.forward(q, k, v, 0.5, causal=True, dtype=np.float64)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, 0.5, causal=True)
    np.testing.assert_allclose(dv[0, 0, 0], do[0, 0, 0] + do[0, 0, 1], rtol=1e-14)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14


def test_gradient_sums():
    """Rows of P sum to one, so sum_j dV_j = sum_i dO_i over a head group, and
    rows of dS sum to zero, so sum_j dK_j = 0."""
    rng = np.random.default_rng(9)
    B, S, HQ, HKV, D = 1, 12, 4, 2, 5
    q, k, v, do = _rand(rng, B, S, HQ, D), _rand(rng, B, S, HKV, D), _rand(rng, B, S, HKV, D), _rand(rng, B, S, HQ, D)
    mask = dict(causal=True, window=4, cu_seqlens=(0, 5, 12))
    o, lse = oracle.forward(q, k, v, 0.4, dtype=np.float64, **mask)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, 0.4, **mask)
    for g in range(HKV):
        np.testing.assert_allclose(dv[0, :, g].sum(0), do[0, :, 2 * g:2 * g + 2].sum((0, 1)), atol=1e-12)
        np.testing.assert_allclose(dk[0, :, g].sum(0), 0.0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(4)
    B, S, HQ, HKV, D = 2, 6, 6, 2, 3
    G = HQ // HKV
    q, k, v, do = _rand(rng, B, S, HQ, D), _rand(rng, B, S, HKV, D), _rand(rng, B, S, HKV, D), _rand(rng, B, S, HQ, D)
    o, lse = oracle.forward(q, k, v, 0.6, causal=True, dtype=np.float64)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, 0.6, causal=True)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    o2, lse2 = oracle.forward(q, kr, vr, 0.6, causal=True, dtype=np.float64)
    dq2, dk2, dv2 = oracle.backward(q, kr, vr, o2, do, lse2, 0.6, causal=True)
    np.testing.assert_allclose(o, o2, rtol=1e-13)
    np.testing.assert_allclose(dq, dq2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, S, HKV, G, D).sum(3), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, S, HKV, G, D).sum(3), rtol=1e-12, atol=1e-13)


def test_sparse_full_prefix_equals_dense_causal():
    """Index lists [0..t] (padded with -1) give dense causal MQA; dKV = dK + [dV, 0]."""
    rng = np.random.default_rng(8)
    S, H, DQK, DV, topk = 7, 3, 5, 3, 8
    q, kv, do = _rand(rng, 1, S, H, DQK), _rand(rng, 1, S, 1, DQK), _rand(rng, 1, S, H, DV)
    idx = np.full((1, S, 1, topk), -1, np.int32)
    for t in range(S):
        idx[0, t, 0, :t + 1] = np.arange(t + 1)
    o, lse = oracle.sparse_forward(q, kv, idx, 0.45, DV, dtype=np.float64)
    dq, dkv = oracle.sparse_backward(q, kv, o, do, lse, idx, 0.45, DV)
    od, lsed = oracle.forward(q, kv, kv[..., :DV], 0.45, causal=True, dtype=np.float64)
    dqd, dkd, dvd = oracle.backward(q, kv, kv[..., :DV], od, do, lsed, 0.45, causal=True)
    np.testing.assert_allclose(o, od, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lsed, rtol=1e-12)
    np.testing.assert_allclose(dq, dqd, rtol=1e-11, atol=1e-13)
    want = dkd.copy()
    want[..., :DV] += dvd
    np.testing.assert_allclose(dkv, want, rtol=1e-11, atol=1e-13)


def test_sparse_slot_order_is_irrelevant():
    rng = np.random.default_rng(12)
    S, H, DQK, DV, topk = 6, 2, 4, 3, 4
    q, kv, do = _rand(rng, 1, S, H, DQK), _rand(rng, 1, S, 1, DQK), _rand(rng, 1, S, H, DV)
    idx = inputs.topk_index_sets(1, 1, S, topk).reshape(1, S, 1, topk)
    perm = idx.copy()
    for t in range(S):
        perm[0, t, 0] = np.random.default_rng(t).permutation(perm[0, t, 0])
    o, lse = oracle.sparse_forward(q, kv, idx, 0.5, DV, dtype=np.float64)
    dq, dkv = oracle.sparse_backward(q, kv, o, do, lse, idx, 0.5, DV)
    o2, lse2 = oracle.sparse_forward(q, kv, perm, 0.5, DV, dtype=np.float64)
    dq2, dkv2 = oracle.sparse_backward(q, kv, o2, do, lse2, perm, 0.5, DV)
    np.testing.assert_allclose(dq, dq2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dkv, dkv2, rtol=1e-12, atol=1e-14)


def test_row_subsets_equal_full_evaluation():
    """Evaluating chosen dQ rows and dK/dV rows alone gives the rows of the full run."""
    rng = np.random.default_rng(13)
    B, S, HQ, HKV, D = 1, 20, 4, 2, 3
    q, k, v, do = _rand(rng, B, S, HQ, D), _rand(rng, B, S, HKV, D), _rand(rng, B, S, HKV, D), _rand(rng, B, S, HQ, D)
    mask = dict(causal=True, window=6, cu_seqlens=(0, 7, 20))
    o, lse = oracle.forward(q, k, v, 0.5, dtype=np.float64, **mask)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, 0.5, **mask)
    rows = np.array([0, 6, 7, 13, 19])
    dq2, dk2, dv2 = oracle.backward(q, k, v, o, do, lse, 0.5, q_rows=rows, k_rows=rows, **mask)
    np.testing.assert_allclose(dq2[:, rows], dq[:, rows], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dk2[:, rows], dk[:, rows], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dv2[:, rows], dv[:, rows], rtol=1e-12, atol=1e-14)
    # sparse: dKV rows alone equal the full scatter
    idx = inputs.topk_index_sets(3, 2, 10, 4).reshape(1, 10, 1, 4)
    qs, kvs, dos = _rand(rng, 1, 10, 2, 4), _rand(rng, 1, 10, 1, 4), _rand(rng, 1, 10, 2, 3)
    os_, ls = oracle.sparse_forward(qs, kvs, idx, 0.5, 3, dtype=np.float64)
    dqs, dkvs = oracle.sparse_backward(qs, kvs, os_, dos, ls, idx, 0.5, 3)
    _, dkv_rows = oracle.sparse_backward(qs, kvs, os_, dos, ls, idx, 0.5, 3, kv_rows=[0, 4, 9])
    np.testing.assert_allclose(dkv_rows[0, [0, 4, 9]], dkvs[0, [0, 4, 9]], rtol=1e-12, atol=1e-14)
    dq_t, _ = oracle.sparse_backward(qs, kvs, os_, dos, ls, idx, 0.5, 3, tokens=[2, 8])
    np.testing.assert_allclose(dq_t[0, [2, 8]], dqs[0, [2, 8]], rtol=1e-12, atol=1e-14)
    # two KV groups, a repeated index, an out-of-range index and -1 padding
    idx2 = np.stack([inputs.topk_index_sets(5, g, 10, 5) for g in range(2)], axis=1)[None]
    idx2[0, 6, 0, 1] = idx2[0, 6, 0, 0]
    idx2[0, 7, 1, 2] = 12
    idx2[0, 9, 1, :] = -1
    qs, kvs, dos = _rand(rng, 1, 10, 4, 4), _rand(rng, 1, 10, 2, 4), _rand(rng, 1, 10, 4, 3)
    os_, ls = oracle.sparse_forward(qs, kvs, idx2, 0.5, 3, dtype=np.float64)
    _, dkvs = oracle.sparse_backward(qs, kvs, os_, dos, ls, idx2, 0.5, 3)
    rows = [0, int(idx2[0, 6, 0, 0]), 5, 9]
    _, dkv_rows = oracle.sparse_backward(qs, kvs, os_, dos, ls, idx2, 0.5, 3, kv_rows=rows)
    np.testing.assert_allclose(dkv_rows[0, rows], dkvs[0, rows], rtol=1e-12, atol=1e-14)


def test_delta_is_rowwise_dot():
    o = np.arange(12, dtype=np.float64).reshape(1, 2, 2, 3)
    do = np.ones_like(o)
    d = oracle.delta(o, do)
    assert d.shape == (1, 2, 2)
    assert d[0, 0, 0] == 0 + 1 + 2 and d[0, 1, 1] == 9 + 10 + 11 and d[0, 1, 0] == 3 + 4 + 5


# attention sinks: one logit per query head in every row's normalisation, no value
SINK_CASES = [
    dict(B=1, S=5, HQ=2, HKV=1, mask=dict(causal=False)),
    dict(B=2, S=4, HQ=2, HKV=2, mask=dict(causal=True)),
    dict(B=1, S=7, HQ=4, HKV=2, mask=dict(causal=True, window=2, cu_seqlens=(0, 3, 7))),
]


@pytest.mark.parametrize("case", SINK_CASES, ids=lambda c: f"S{c['S']}H{c['HQ']}/{c['HKV']}{c['mask']}")
def test_sink_gradients_match_finite_differences(case):
    """With sinks in the forward, dsink and dQ, dK, dV (the backward given the
    sink-aware O and LSE) equal the central differences of L = sum(O * dO)."""
    rng = np.random.default_rng(11)
    B, S, HQ, HKV = (case[x] for x in ("B", "S", "HQ", "HKV"))
    D = 3
    q, k = _rand(rng, B, S, HQ, D), _rand(rng, B, S, HKV, D)
    v, do = _rand(rng, B, S, HKV, D), _rand(rng, B, S, HQ, D)
    sink = rng.standard_normal(HQ)
    scale = 0.8
    mask = case["mask"]
    o, lse = oracle.forward(q, k, v, scale, dtype=np.float64, sink=sink, **mask)

    def loss():
        o_, _ = oracle.forward(q, k, v, scale, dtype=np.float64, sink=sink, **mask)
        return float((o_ * do).sum())

    np.testing.assert_allclose(oracle.sink_grad(o, do, lse, sink, mask.get("cu_seqlens")), _fd_grad(loss, sink),
                               rtol=1e-6, atol=1e-9)
    dq, dk, dv = oracle.backward(q, k, v, o, do, lse, scale, **mask)
    for got, x in ((dq, q), (dk, k), (dv, v)):
        np.testing.assert_allclose(got, _fd_grad(loss, x), rtol=1e-6, atol=1e-8)


def test_sink_limits():
    """A sink at -inf is no sink; a row that sees no key puts all its mass on
    the sink (LSE = sink, O = 0); one key and a sink give the two-way softmax."""
    rng = np.random.default_rng(3)
    q, k, v = _rand(rng, 1, 4, 2, 3), _rand(rng, 1, 4, 1, 3), _rand(rng, 1, 4, 1, 3)
    o0, l0 = oracle.forward(q, k, v, 0.5, dtype=np.float64, causal=True)
    o1, l1 = oracle.forward(q, k, v, 0.5, dtype=np.float64, causal=True, sink=np.array([-np.inf, -np.inf]))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
    # fewer keys than queries, end-aligned causal: query 0 sees no key
    o2, l2 = oracle.forward(q, k[:, :2], v[:, :2], 0.5, dtype=np.float64, causal=True, sink=np.array([0.25, -1.0]))
    assert l2[0, 0, 0] == 0.25 and l2[0, 1, 0] == -1.0 and not o2[0, 0].any()
    # query 2 sees key 0 only: O = v0 * e^s / (e^s + e^sink)
    s = 0.5 * float(q[0, 2, 0] @ k[0, 0, 0])
    p = math.exp(s) / (math.exp(s) + math.exp(0.25))
    np.testing.assert_allclose(o2[0, 2, 0], p * v[0, 0, 0], rtol=1e-12)
    np.testing.assert_allclose(l2[0, 0, 2], math.log(math.exp(s) + math.exp(0.25)), rtol=1e-12)
