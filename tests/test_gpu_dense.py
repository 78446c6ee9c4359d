"""Parity of the dense CUDA path (preprocess, main kernel, dQ landing) with the
CPU oracle, element by element, through the C ABI on a GPU."""
import numpy as np
import pytest

import oracle
from attention_backward_gb300 import inputs

from _harness import assert_close, dense_problem, mask_of, oracle_rows_chunked, run_dense, sample_rows, to_np

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS
C1 = W["mha_causal_1x256x2x128_f16"]
C2 = W["mha_causal_2x2048x32x128_f16"]
C3 = W["gqa_1x16384_hq32_hkv4_d128_bf16"]
C4 = W["gqa_varlen_window1024_hq32_hkv8_d64_bf16"]

# Small cases the oracle checks in full: several tiles, ragged tails and the
# degenerate shapes of the method.
SMALL = [
    C1,
    inputs.scaled(C1, name="noncausal_f16", causal=False),
    inputs.scaled(C1, name="ragged_b2_s200", B=2, S=200),
    inputs.scaled(C1, name="s1", S=1),
    inputs.scaled(C1, name="s2_noncausal", S=2, causal=False),
    inputs.scaled(C1, name="s129_bf16", S=129, dtype="bf16"),
    inputs.scaled(C1, name="s127_b3", S=127, B=3, HQ=1, HKV=1),
    # group sizes in both dtypes, powers of two and not (every accepted G has a
    # case of its own in EVERY_G below).  bf16 groups of 8 and 16 on short causal
    # rows need the rounding residuals of P and dS that the kernels add on steps
    # with a large P: without them the 16-bit rounding of P before the dV
    # product (as the page's Tiled program does) exceeds the bf16 tolerance.
    inputs.scaled(C3, name="gqa_g4_s384", S=384, HQ=8, HKV=2),
    inputs.scaled(C3, name="gqa_g16_s300_causal_bf16", S=300, HQ=16, HKV=1, causal=True),
    inputs.scaled(C3, name="gqa_g16_s300_causal_f16", S=300, HQ=16, HKV=1, causal=True, dtype="f16"),
    inputs.scaled(C3, name="gqa_g8_s300_causal_bf16", S=300, HQ=8, HKV=1, causal=True),
    inputs.scaled(C3, name="gqa_g8_s300_causal_f16", S=300, HQ=16, HKV=2, causal=True, dtype="f16"),
    inputs.scaled(C3, name="gqa_g4_s260_causal_f16", S=260, HQ=8, HKV=2, causal=True, dtype="f16"),
    inputs.scaled(C3, name="gqa_g2_f16_s520", S=520, HQ=4, HKV=2, dtype="f16"),
    inputs.scaled(C3, name="gqa_g2_s330_causal_bf16", S=330, HQ=4, HKV=2, causal=True),
    inputs.scaled(C3, name="gqa_g3_s300_causal_bf16", S=300, HQ=6, HKV=2, causal=True),
    inputs.scaled(C3, name="gqa_g12_s280_causal_f16", S=280, HQ=12, HKV=1, causal=True, dtype="f16"),
    inputs.scaled(C4, name="gqa_g8_d64_s300_causal_bf16", S=300, HQ=16, HKV=2, window=-1, cu_seqlens=None),
    inputs.scaled(C4, name="varlen_d64_w100", S=700, HQ=4, HKV=2, window=100, cu_seqlens=(0, 33, 161, 390, 700)),
    inputs.scaled(C4, name="varlen_empty_and_single", S=300, HQ=2, HKV=1, window=64,
                  cu_seqlens=(0, 0, 1, 1, 130, 300)),
    inputs.scaled(C4, name="window1", S=200, HQ=2, HKV=2, window=1, cu_seqlens=(0, 200)),
    inputs.scaled(C4, name="varlen_causal_nowindow_d64", S=500, HQ=4, HKV=1, window=-1, cu_seqlens=(0, 250, 251, 500)),
    inputs.scaled(C4, name="d64_noncausal_b3_f16", B=3, S=190, HQ=2, HKV=2, causal=False, window=-1, cu_seqlens=None,
                  dtype="f16"),
    inputs.scaled(C4, name="varlen_d128_w300", D=128, Dv=128, S=900, HQ=4, HKV=2, window=300,
                  cu_seqlens=(0, 400, 900)),
    # head dim 128 without a mask runs the 128-query-step kernel: packed sequences
    # with a ragged last block
    inputs.scaled(C4, name="varlen_d128_noncausal", D=128, Dv=128, S=420, HQ=4, HKV=2, causal=False, window=-1,
                  cu_seqlens=(0, 150, 420)),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_cases_match_oracle(w):
    prob = dense_problem(w)
    q, k, v, o, do, lse = prob
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
    dq, dk, dv, _ = run_dense(w, prob)
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")


# Unmasked dense batches whose key tiles do not divide evenly over the SMs:
# at head dim 128 the one-call path draws the last round's tiles as units of
# fewer query heads and adds their dK/dV in f32 (160 tiles on 152 SMs: the
# last 8 tiles split into single-head units).  A ragged last key tile and the
# bf16 kernel with the rounding residuals are among them.
LAST_ROUND = [
    inputs.scaled(C3, name="split_g2_s1024_hkv20_f16", S=1024, HQ=40, HKV=20, dtype="f16"),
    inputs.scaled(C3, name="split_g2_s1000_hkv20_bf16", S=1000, HQ=40, HKV=20),
    inputs.scaled(C3, name="split_g8_b2_s512_hkv20_bf16", B=2, S=512, HQ=160, HKV=20),
]


@pytest.mark.parametrize("w", LAST_ROUND, ids=lambda w: w.name)
def test_last_round_split_matches_oracle(w):
    import torch

    import attention_backward_gb300 as ab

    tiles = w.B * w.HKV * ((w.S + 127) // 128)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = ab.tail_plan(tiles, min(tiles, sms), w.HQ // w.HKV)
    if plan[1] == 0:
        pytest.skip(f"{tiles} tiles on {sms} SMs: no last-round split")
    prob = dense_problem(w)
    q, k, v, o, do, lse = prob
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
    for split in (False, True):  # the one-call path, then the three launches one by one
        dq, dk, dv, _ = run_dense(w, prob, split=split)
        assert_close(dq, rq, w, "dq")
        assert_close(dk, rk, w, "dk")
        assert_close(dv, rv, w, "dv")


# Dense rows whose key length differs from the query length (kv_len in the C
# mask): the masks are aligned at the end of the row, query i at key position
# i + Sk - S.  Cases cover more and fewer keys than queries under every mask
# kind and both head dims, key tiles that no query sees (dK = dV = 0 written),
# queries that see no key (dQ = 0, LSE -inf from the forward), one query, one
# key, and ragged tiles on both sides.
UNEQUAL = [
    inputs.scaled(C1, name="sk520_sq200_causal_b2_f16", B=2, S=200, Sk=520),
    inputs.scaled(C1, name="sq520_sk200_causal_f16", S=520, Sk=200),
    inputs.scaled(C3, name="sk390_sq130_noncausal_g4_bf16", S=130, Sk=390, HQ=8, HKV=2),
    inputs.scaled(C3, name="sq300_sk170_causal_g2_bf16", S=300, Sk=170, HQ=4, HKV=2, causal=True),
    inputs.scaled(C4, name="sk700_sq300_w100_d64", S=300, Sk=700, HQ=4, HKV=2, window=100, cu_seqlens=None),
    inputs.scaled(C4, name="sq700_sk300_w64_d64_f16", S=700, Sk=300, HQ=2, HKV=1, window=64, cu_seqlens=None,
                  dtype="f16"),
    inputs.scaled(C4, name="sq390_sk130_noncausal_d64_b2", B=2, S=390, Sk=130, HQ=2, HKV=2, causal=False, window=-1,
                  cu_seqlens=None),
    inputs.scaled(C4, name="sk300_sq129_causal_d64_g4", S=129, Sk=300, HQ=8, HKV=2, window=-1, cu_seqlens=None),
    inputs.scaled(C1, name="sq1_sk700_causal", S=1, Sk=700),
    inputs.scaled(C1, name="sq1_sk700_noncausal", S=1, Sk=700, causal=False),
    inputs.scaled(C4, name="sq300_sk1_causal_d64", S=300, Sk=1, HQ=2, HKV=1, window=-1, cu_seqlens=None),
]


@pytest.mark.parametrize("w", UNEQUAL, ids=lambda w: w.name)
def test_unequal_query_and_key_lengths_match_oracle(w):
    prob = dense_problem(w)
    q, k, v, o, do, lse = prob
    assert k.shape[1] == w.Sk != w.S
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
    dq, dk, dv, _ = run_dense(w, prob)
    assert tuple(dk.shape) == k.shape and tuple(dv.shape) == v.shape
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")
    if w.S > w.Sk and w.causal:  # the first S - Sk queries see no key
        assert (to_np(dq)[:, : w.S - w.Sk] == 0).all()
    # the split launches take the key length from the same mask field
    b = run_dense(w, prob, split=True)
    assert (to_np(b[1]) == to_np(dk)).all() and (to_np(b[2]) == to_np(dv)).all()


# Every group size the ABI accepts, one small causal case each: G = 1..16 in
# both dtypes, alternating head dims 64 and 128, two KV heads.
EVERY_G = [
    inputs.scaled(C3, name=f"every_g{g}_{dt}_d{d}", S=200, HQ=2 * g, HKV=2, D=d, Dv=d, causal=True, dtype=dt,
                  seed=20260100 + g)
    for dt, gmax in (("f16", 16), ("bf16", 16)) for g in range(1, gmax + 1) for d in ((64, 128)[g % 2],)
]


@pytest.mark.parametrize("w", EVERY_G, ids=lambda w: w.name)
def test_every_accepted_group_size_matches_oracle(w):
    prob = dense_problem(w)
    q, k, v, o, do, lse = prob
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
    dq, dk, dv, _ = run_dense(w, prob)
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")


def test_split_launches_match_one_call():
    """The three launches called one by one (attn_bwd_preprocess,
    attn_bwd_gqa_main, attn_bwd_dq_land) give the one-call results: the same
    dK/dV bits, dQ within tolerance of the oracle."""
    for w in (inputs.scaled(C3, name="split_g4", S=384, HQ=8, HKV=2, causal=True),
              inputs.scaled(C4, name="split_d64", S=500, HQ=4, HKV=2, window=100, cu_seqlens=(0, 200, 500))):
        prob = dense_problem(w)
        a = run_dense(w, prob)
        b = run_dense(w, prob, split=True)
        assert (to_np(a[1]) == to_np(b[1])).all() and (to_np(a[2]) == to_np(b[2])).all()
        q, k, v, o, do, lse = prob
        rq, _, _ = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
        assert_close(b[0], rq, w, "dq (split launches)")


def test_group_size_limits_are_enforced():
    """Group sizes past the limit (16 query heads per KV head) are refused
    with ATTN_ERR_UNSUPPORTED before anything runs, in both dtypes."""
    import torch

    import attention_backward_gb300 as ab

    for dt, hq in ((torch.bfloat16, 32), (torch.float16, 32)):
        q = torch.zeros(1, 128, hq, 128, dtype=dt, device="cuda")
        kv = torch.zeros(1, 128, 1, 128, dtype=dt, device="cuda")
        lse = torch.zeros(1, hq, 128, dtype=torch.float32, device="cuda")
        with pytest.raises(ab.AttnBwdError, match="unsupported"):
            ab.backward(q, kv, kv, q, q, lse, 0.1, causal=True)


def _poisoned_tail_case(w, tail):
    """Packed sequences ending ``tail`` rows before S; every input row past the
    last sequence holds NaN (Q, K, V, O, dO and the LSE)."""
    import torch

    import attention_backward_gb300 as ab
    from _harness import torch_dtype

    q, k, v, o, do, lse = dense_problem(w)
    dt = torch_dtype(w)
    end = w.cu_seqlens[-1]
    assert end == w.S - tail
    t = lambda a: torch.from_numpy(a).cuda().to(dt)  # noqa: E731
    tq, tk, tv, to, tdo = t(q), t(k), t(v), t(o), t(do)
    tl = torch.from_numpy(lse).cuda()
    for x in (tq, tk, tv, to, tdo):
        x[:, end:] = float("nan")
    tl[:, :, end:] = float("nan")
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda")
    dq, dk, dv = ab.backward(tq, tk, tv, to, tdo, tl, w.sm_scale, w.causal, w.window, cu)
    torch.cuda.synchronize()
    return (q, k, v, o, do, lse), dq, dk, dv


@pytest.mark.parametrize("w,tail", [
    # head dim 128: the last sequence ends inside a key tile and a query block,
    # and a whole 128-row block lies past it
    (inputs.scaled(C4, name="tail_d128", D=128, Dv=128, S=700, HQ=4, HKV=2, window=-1,
                   cu_seqlens=(0, 250, 480)), 220),
    (inputs.scaled(C4, name="tail_d128_noncausal", D=128, Dv=128, S=400, HQ=2, HKV=2, causal=False, window=-1,
                   cu_seqlens=(0, 150, 301)), 99),
    # head dim 64 with a window
    (inputs.scaled(C4, name="tail_d64_w100", S=640, HQ=4, HKV=2, window=100, cu_seqlens=(0, 33, 161, 390)), 250),
], ids=lambda x: getattr(x, "name", str(x)))
def test_rows_past_the_last_sequence_may_hold_nan(w, tail):
    """Rows of a packed batch past cu_seqlens[num_seqs] belong to no sequence:
    NaN there must not reach any gradient of a row inside a sequence (a zero P
    or dS times NaN is NaN, so the kernels zero those rows after loading), and
    the dQ rows there are written as zero."""
    prob, dq, dk, dv = _poisoned_tail_case(w, tail)
    q, k, v, o, do, lse = prob
    end = w.cu_seqlens[-1]
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
    # the oracle leaves rows outside every sequence as NaN: they are skipped here
    assert np.isnan(rq[:, end:]).all() and not np.isnan(rq[:, :end]).any()
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")
    assert (to_np(dq)[:, end:] == 0).all()


def test_single_position_closed_form():
    """S = 1: P = 1, so dV = dO exactly (P rounds to 1 in 16 bits), and
    dS = dP - delta vanishes up to float32 summation order, so dQ, dK ~ 0."""
    w = inputs.scaled(C1, name="s1", S=1)
    prob = dense_problem(w)
    dq, dk, dv, _ = run_dense(w, prob)
    assert np.abs(to_np(dq)).max() < 1e-4 and np.abs(to_np(dk)).max() < 1e-4
    np.testing.assert_array_equal(to_np(dv), prob[4].astype(np.float64))


def test_preprocess_delta_and_lse2():
    """The workspace's delta and LSE*log2(e) after launch 1 (float32 against
    the float64 oracle delta)."""
    import torch

    w = inputs.scaled(C2, name="c2_half", B=1, S=1024, HQ=4, HKV=4)
    prob = dense_problem(w)
    _, _, _, ws = run_dense(w, prob)
    q, k, v, o, do, lse = prob
    rows = w.B * w.HQ * w.S
    raw = ws.cpu().numpy()
    lse2 = raw[256:256 + 4 * rows].view(np.float32).reshape(w.B, w.HQ, w.S)
    off = 256 + ((4 * rows + 255) // 256) * 256
    delta = raw[off:off + 4 * rows].view(np.float32).reshape(w.B, w.HQ, w.S)
    np.testing.assert_allclose(delta, oracle.delta(o, do), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(lse2, lse * np.log2(np.e), rtol=1e-6, atol=1e-6)
    del torch


def test_dk_dv_are_deterministic():
    """dK and dV are owned by one CTA and written once: bitwise identical
    across runs (dQ goes through f32 atomics and is compared with tolerance)."""
    w = inputs.scaled(C3, name="gqa_det", S=1024, HQ=8, HKV=2)
    prob = dense_problem(w)
    a = run_dense(w, prob)
    b = run_dense(w, prob)
    assert (to_np(a[1]) == to_np(b[1])).all()
    assert (to_np(a[2]) == to_np(b[2])).all()
    assert_close(a[0], to_np(b[0]), w, "dq run-to-run")


def test_strided_inputs():
    """Q, K, V taken as views of one packed [B, S, 3, H, D] tensor (non-dense
    strides) and dO a head-transposed view."""
    import torch

    import attention_backward_gb300 as ab
    from _harness import torch_dtype

    w = inputs.scaled(C1, name="strided", S=320, HQ=2, HKV=2)
    q, k, v, o, do, lse = dense_problem(w)
    dt = torch_dtype(w)
    qkv = torch.from_numpy(np.stack([q, k, v], axis=2)).cuda().to(dt)  # [B,S,3,H,D]
    tq, tk, tv = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    tdo = torch.from_numpy(np.ascontiguousarray(do.transpose(0, 2, 1, 3))).cuda().to(dt).transpose(1, 2)
    to = torch.from_numpy(o).cuda().to(dt)
    tl = torch.from_numpy(lse).cuda()
    dq, dk, dv = ab.backward(tq, tk, tv, to, tdo, tl, w.sm_scale, causal=True)
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, causal=True)
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")


def _sum_invariants(w, do, dk, dv):
    """Properties that hold on every row: rows of P sum to one and rows of dS
    to zero, so per KV head sum_j dV_j = sum_i dO_i and sum_j dK_j = 0."""
    G = w.HQ // w.HKV
    gv, gk = to_np(dv), to_np(dk)
    for b in range(w.B):
        for g in range(w.HKV):
            sum_do = do[b, :, g * G:(g + 1) * G].astype(np.float64).sum(axis=(0, 1))
            n = w.S * G
            np.testing.assert_allclose(gv[b, :, g].sum(0), sum_do, atol=2e-3 * np.sqrt(n) * 4)
            np.testing.assert_allclose(gk[b, :, g].sum(0), 0.0, atol=2e-3 * np.sqrt(n) * 4)


def test_workload_mha_causal_2x2048x32x128_in_full():
    """Causal MHA 2x2048x32x128 fp16, every element of dQ, dK and dV against
    the oracle."""
    w = C2
    prob = dense_problem(w)
    q, k, v, o, do, lse = prob
    dq, dk, dv, _ = run_dense(w, prob)
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, **mask_of(w))
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")
    _sum_invariants(w, do, dk, dv)


def test_workload_varlen_window_in_full():
    """Packed sliding-window GQA (4 sequences, 16384 tokens, window 1024, D 64
    bf16), every element against the oracle (evaluated 1024 rows at a time)."""
    w = C4
    prob = dense_problem(w)
    dq, dk, dv, _ = run_dense(w, prob)
    every = np.arange(w.S)
    rq, rk, rv = oracle_rows_chunked(prob, w, q_rows=every, k_rows=every)
    assert_close(dq, rq, w, "dq")
    assert_close(dk, rk, w, "dk")
    assert_close(dv, rv, w, "dv")
    _sum_invariants(w, prob[4], dk, dv)


def test_workload_gqa_16384():
    """Unmasked GQA 1x16384, HQ 32 / HKV 4, D 128 bf16: every dQ row of query
    heads 0 and 31, every dK/dV row of KV heads 0 and 3, and 512 seeded rows
    (plus every tile edge) of every head."""
    w = C3
    prob = dense_problem(w)
    q, k, v, o, do, lse = prob
    dq, dk, dv, _ = run_dense(w, prob)
    rows = sample_rows(w.S, 512, w.seed)
    rq, rk, rv = oracle_rows_chunked(prob, w, q_rows=rows, k_rows=rows)
    assert_close(dq, rq, w, "dq (seeded rows, every head)")
    assert_close(dk, rk, w, "dk (seeded rows, every KV head)")
    assert_close(dv, rv, w, "dv (seeded rows, every KV head)")
    G = w.HQ // w.HKV
    every = np.arange(w.S)
    for g, hq in ((0, 0), (w.HKV - 1, w.HQ - 1)):
        fq, _, _ = oracle_rows_chunked(prob, w, q_rows=every, heads=[hq], chunk=512)
        keep = np.full(w.HQ, False)
        keep[hq] = True
        fq[:, :, ~keep] = np.nan
        assert_close(dq, fq, w, f"dq (query head {hq}, every row)")
        _, fk, fv = oracle_rows_chunked(prob, w, k_rows=every, heads=list(range(g * G, (g + 1) * G)), chunk=512)
        kv_keep = np.full(w.HKV, False)
        kv_keep[g] = True
        fk[:, :, ~kv_keep] = np.nan
        fv[:, :, ~kv_keep] = np.nan
        assert_close(dk, fk, w, f"dk (KV head {g}, every row)")
        assert_close(dv, fv, w, f"dv (KV head {g}, every row)")
    _sum_invariants(w, do, dk, dv)


def test_workload_mha_causal_1x256_in_full():
    prob = dense_problem(C1)
    q, k, v, o, do, lse = prob
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, C1.sm_scale, causal=True)
    dq, dk, dv, _ = run_dense(C1, prob)
    for got, ref, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        assert_close(got, ref, C1, n)


def test_unsupported_head_dim_raises():
    import torch

    import attention_backward_gb300 as ab

    x = torch.zeros(1, 64, 2, 96, dtype=torch.float16, device="cuda")
    lse = torch.zeros(1, 2, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(ab.AttnBwdError, match="unsupported"):
        ab.backward(x, x, x, x, x, lse, 0.1, causal=True)


def test_bounded_wait_reports_timeout_and_context_survives():
    """A kernel waiting on a barrier nothing signals gives up after its limit,
    records the error and returns; the context keeps working afterwards."""
    import torch

    import attention_backward_gb300 as ab

    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    st, msg = ab.selftest_timeout(ws, timeout_us=20000)
    assert st == 5, msg
    w = inputs.scaled(C1, name="after_timeout", S=130)
    prob = dense_problem(w)
    dq, dk, dv, _ = run_dense(w, prob)
    q, k, v, o, do, lse = prob
    rq, rk, rv = oracle.backward(q, k, v, o, do, lse, w.sm_scale, causal=True)
    assert_close(dv, rv, w, "dv after a timed-out kernel")
