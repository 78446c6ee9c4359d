"""The C-ABI library without a GPU: it loads, exports every declared entry
point, validates arguments before touching the device, and its tile schedule
matches a brute-force visibility mask."""
import ctypes
import os
import re

import numpy as np
import pytest

import __graft_entry__
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ab():
    __graft_entry__.build()
    import attention_backward_gb300 as ab

    return ab


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "attn_bwd.h")).read()
    return sorted(set(re.findall(r"ATTN_BWD_API\s+[\w\s\*]+?\b(attn_bwd\w*)\s*\(", src)))


def test_every_declared_symbol_is_exported(ab):
    names = declared_symbols()
    assert len(names) >= 11
    lib = ab.library()
    for n in names:
        assert hasattr(lib, n), n
    # and nothing else leaks out as a C symbol of ours
    assert "attn_bwd_gqa" in names and "attn_bwd_sparse" in names and "attn_bwd_preprocess" in names


def test_status_strings(ab):
    lib = ab.library()
    for code in range(7):
        s = lib.attn_bwd_status_string(code)
        assert s and s.decode()
    assert lib.attn_bwd_status_string(99).decode() == "unknown status"


def test_workspace_layout(ab):
    n = ab.workspace_size(2, 2048, 32, 128)
    rows = 2 * 32 * 2048
    assert n == 256 + 2 * rows * 4 + rows * 128 * 4
    assert n % 256 == 0
    s = ab.workspace_size(1, 4096, 64, 576, 4096 * 576)
    assert s == 256 + 2 * 4096 * 64 * 4 + 4096 * 64 * 576 * 4 + 4096 * 576 * 4
    assert ab.workspace_size(-1, 1, 1, 1) == 0


@pytest.mark.parametrize("cu", [(0, 33, 161, 390), (0, 3000, 8000, 9537, 16384)])
@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 1), (True, 100), (True, 1024)])
@pytest.mark.parametrize("bq", [64, 128])
def test_query_block_range_matches_brute_force(ab, cu, causal, window, bq):
    """Every query block holding a visible (query, key) pair is visited, and no
    other block is, for every key tile of every packed sequence."""
    for a, e in zip(cu[:-1], cu[1:]):
        n = e - a
        vis = oracle.visible(n, causal, window, None)
        for k0 in range(0, n, 128):
            lo, hi = ab.query_block_range(k0, 128, n, causal, window, bq)
            rows = np.nonzero(vis[:, k0:k0 + 128].any(axis=1))[0]
            assert set(range(lo, hi)) == set((rows // bq).tolist()), (a, e, k0, lo, hi)


def test_causal_step_count_matches_the_page(ab):
    """The causal kernel visits 272 of the 512 (key block, query block) steps of
    a 2048-row head at 128/64 blocks (TileOPs page, analysis bullets)."""
    steps = sum(np.subtract(*reversed(ab.query_block_range(k0, 128, 2048, True, -1, 64))) for k0 in range(0, 2048, 128))
    assert steps == 272


def test_argument_errors_return_before_any_launch(ab):
    lib = ab.library()
    S = ab._binding.Strides
    z = S(0, 0, 0)
    good = S(2048 * 32 * 128, 32 * 128, 128)
    m = ab._binding.Mask(1, -1, None, 0)
    # null pointers
    assert lib.attn_bwd_gqa(None, good, None, good, None, good, None, good, 2, 2048, 32, 32, 128, 0, 0.1,
                            ctypes.byref(m), None, good, None, good, None, 0, None) == 1
    fake = 1 << 20  # 16-byte aligned, never dereferenced: validation fails first
    # unsupported head dim
    assert lib.attn_bwd_gqa(fake, good, fake, good, fake, good, fake, good, 2, 2048, 32, 32, 96, 0, 0.1,
                            ctypes.byref(m), fake, good, fake, good, fake, 1 << 30, None) == 2
    # HQ not a multiple of HKV
    assert lib.attn_bwd_gqa(fake, good, fake, good, fake, good, fake, good, 2, 2048, 6, 4, 128, 0, 0.1,
                            ctypes.byref(m), fake, good, fake, good, fake, 1 << 30, None) == 1
    # misaligned pointer
    assert lib.attn_bwd_gqa(fake + 2, good, fake, good, fake, good, fake, good, 2, 2048, 32, 32, 128, 0, 0.1,
                            ctypes.byref(m), fake, good, fake, good, fake, 1 << 30, None) == 1
    # zero strides
    assert lib.attn_bwd_gqa(fake, z, fake, good, fake, good, fake, good, 2, 2048, 32, 32, 128, 0, 0.1,
                            ctypes.byref(m), fake, good, fake, good, fake, 1 << 30, None) == 1
    # workspace too small
    assert lib.attn_bwd_gqa(fake, good, fake, good, fake, good, fake, good, 2, 2048, 32, 32, 128, 0, 0.1,
                            ctypes.byref(m), fake, good, fake, good, fake, 1024, None) == 3
    # window of zero, varlen with B > 1
    m0 = ab._binding.Mask(1, 0, None, 0)
    assert lib.attn_bwd_gqa(fake, good, fake, good, fake, good, fake, good, 2, 2048, 32, 32, 128, 0, 0.1,
                            ctypes.byref(m0), fake, good, fake, good, fake, 1 << 30, None) == 1
    mv = ab._binding.Mask(1, -1, fake, 3)
    assert lib.attn_bwd_gqa(fake, good, fake, good, fake, good, fake, good, 2, 2048, 32, 32, 128, 0, 0.1,
                            ctypes.byref(mv), fake, good, fake, good, fake, 1 << 30, None) == 1
    # preprocess: bad head dim, workspace too small
    assert lib.attn_bwd_preprocess(fake, good, fake, good, fake, S(64, 1, 2048), 2, 2048, 32, 12, 128, 0, 0,
                                   fake, 1 << 30, None) == 1
    assert lib.attn_bwd_preprocess(fake, good, fake, good, fake, S(64, 1, 2048), 2, 2048, 32, 128, 128, 0, 0,
                                   fake, 4096, None) == 3
    # landing: unsupported dtype code
    assert lib.attn_bwd_dq_land(fake, good, 2, 2048, 32, 128, 7, 0.1, fake, 1 << 30, None) == 2
