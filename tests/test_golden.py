"""Pins against stored values: numbers the pages print (tests/golden/page_values.txt,
each with its citation) and a stored float64 evaluation of the oracle on a tiny
causal GQA case (tests/golden/tiny_causal_gqa.txt, written by make_tiny.py from
the oracle alone), which guards the oracle against unintended changes."""
import os
import sys

import numpy as np
import pytest

import __graft_entry__

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")
sys.path.insert(0, GOLDEN)


def page_values():
    vals = {}
    for line in open(os.path.join(GOLDEN, "page_values.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("="))
            vals[k] = float(v)
    return vals


@pytest.fixture(scope="module")
def ab():
    __graft_entry__.build()
    import attention_backward_gb300 as ab

    return ab


def test_causal_step_counts_of_the_long_shape(ab):
    pv = page_values()
    S, BM, BN = 2048, 128, 64
    causal = sum(hi - lo for lo, hi in (ab.query_block_range(k0, BM, S, True, -1, BN) for k0 in range(0, S, BM)))
    full = sum(hi - lo for lo, hi in (ab.query_block_range(k0, BM, S, False, -1, BN) for k0 in range(0, S, BM)))
    assert causal == pv["causal_steps_long_shape"]
    assert full == pv["all_steps_long_shape"]


def test_dq_accumulator_of_the_short_shape(ab):
    """The f32 dQ accumulator is the part of the workspace that grows with D."""
    pv = page_values()
    B, S, H, D = 4, 512, 32, 128
    acc = ab.workspace_size(B, S, H, D) - ab.workspace_size(B, S, H, 0)
    assert acc == B * S * H * D * 4
    assert abs(acc / 1e6 - pv["dq_accumulator_short_shape_mb"]) < 0.1  # the page prints one decimal


def test_no_query_head_shaped_dk_dv(ab):
    """The page's two HQ-shaped f32 intermediates at T=16384, HQ=32, D=128 are
    512 MiB; the KV-head-owned path's workspace holds only LSE2, delta and the
    dQ accumulator."""
    pv = page_values()
    T, HQ, D = 16384, 32, 128
    assert 2 * T * HQ * D * 4 / 2**20 == pv["hq_shaped_f32_dkdv_mib"]
    rows = HQ * T
    assert ab.workspace_size(1, T, HQ, D) == 256 + 2 * rows * 4 + rows * D * 4


def test_oracle_matches_its_stored_tiny_evaluation():
    import make_tiny

    lines = [ln for ln in open(os.path.join(GOLDEN, "tiny_causal_gqa.txt")) if not ln.startswith("#")]
    stored = {}
    for head, data in zip(lines[0::2], lines[1::2]):
        name, *shape = head.split()
        stored[name] = np.array([float(x) for x in data.split()]).reshape([int(s) for s in shape])
    dq, dk, dv = make_tiny.evaluate()
    for name, arr in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(arr, stored[name], rtol=1e-12, atol=1e-14, err_msg=name)
