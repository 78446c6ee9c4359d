"""The seeded input generator: determinism, distribution, 16-bit rounding and
the top-k index-list structure of the sparse workload."""
import numpy as np
import torch

from attention_backward_gb300 import inputs


def test_streams_are_deterministic_and_independent():
    a = inputs.normal_f32(123, 1, (1000,))
    b = inputs.normal_f32(123, 1, (1000,))
    c = inputs.normal_f32(123, 2, (1000,))
    d = inputs.normal_f32(124, 1, (1000,))
    assert (a == b).all()
    assert not np.allclose(a, c) and not np.allclose(a, d)
    # a prefix of a longer draw is the shorter draw
    e = inputs.normal_f32(123, 1, (1001,))
    assert (e[:1000] == a).all()


def test_normal_moments():
    x = inputs.normal_f32(99, 3, (1 << 20,)).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 5e-3
    assert abs((x ** 4).mean() - 3.0) < 3e-2


def test_rounding_matches_torch_casts():
    x = inputs.normal_f32(5, 1, (4096,)) * np.float32(37.0)
    x = np.concatenate([x, np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 65504.0, 1e-8], np.float32)])
    for name, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        want = torch.from_numpy(x).to(tdt).float().numpy()
        got = inputs.round_to_dtype(x, name)
        assert (got == want).all(), name
    # ties go to even
    assert inputs.round_to_dtype(np.array([1 + 2 ** -8], np.float32), "bf16")[0] == 1.0
    assert inputs.round_to_dtype(np.array([1 + 3 * 2 ** -8], np.float32), "bf16")[0] == 1 + 2 ** -6


def test_topk_lists():
    s, k = 300, 128
    idx = inputs.topk_index_sets(7, 5, s, k)
    for t in range(s):
        row = idx[t]
        if t + 1 <= k:
            assert (row[:t + 1] == np.arange(t + 1)).all() and (row[t + 1:] == -1).all()
        else:
            assert (row >= 0).all() and (row <= t).all()
            assert len(np.unique(row)) == k and (np.diff(row) > 0).all()
    # the sets are spread over [0, t], not a prefix
    assert idx[s - 1].max() > k


def test_workload_table():
    w = inputs.WORKLOADS
    assert len(w) == 5
    c4 = w["gqa_varlen_window1024_hq32_hkv8_d64_bf16"]
    assert c4.cu_seqlens[-1] == c4.S == 16384 and c4.G == 4 and c4.window == 1024
    assert np.diff(c4.cu_seqlens).tolist() == [3000, 5000, 1537, 6847]
    c5 = w["sparse_mla_s4096_h64_topk2048_bf16"]
    assert (c5.D, c5.Dv, c5.topk, c5.HKV) == (576, 512, 2048, 1)
