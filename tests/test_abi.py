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


def _host_tile_bound(B, S, HKV, cu):
    """Tile draws the host sizes a launch for: 128-key tiles per (batch, KV
    head), one extra partial tile per packed sequence."""
    return ((S + 127) // 128 + (len(cu) - 1 if cu else 0)) * B * HKV


@pytest.mark.parametrize("B,S,HKV,causal,window,cu", [
    (2, 2048, 32, True, -1, None),                             # causal MHA 2x2048x32
    (1, 1000, 4, False, -1, None),                             # unmasked GQA, ragged last tile
    (3, 300, 5, True, -1, None),                               # pairs not a multiple of the group
    (1, 257, 20, True, 64, None),                              # window, 2.5 groups
    (1, 16384, 8, True, 1024, (0, 3000, 8000, 9537, 16384)),   # packed sequences with a window
    (1, 390, 3, False, -1, (0, 33, 161, 390)),                 # packed, unmasked, a 33-row sequence
])
def test_tile_schedule_draws_every_key_tile_once(ab, B, S, HKV, causal, window, cu):
    """The persistent dense kernels draw tiles from a counter and stop at the
    first invalid draw: every key tile of every (batch, KV head, sequence) must
    come exactly once before it, with the query-block range the mask needs,
    and, for dense batches, the longest tiles of each group of pairs first."""
    seqs = [(0, S)] if cu is None else list(zip(cu[:-1], cu[1:]))
    want = {(b, g, a, k0) for b in range(B) for g in range(HKV) for (a, e) in seqs for k0 in range(0, e - a, 128)}
    draws = [ab.tile_schedule(t, B, S, HKV, causal, window, cu) for t in range(_host_tile_bound(B, S, HKV, cu) + 4)]
    first_invalid = next(i for i, d in enumerate(draws) if not d[0])
    assert all(not d[0] for d in draws[first_invalid:])
    got = [d[1:5] for d in draws[:first_invalid]]
    assert len(got) == len(set(got)) == len(want)
    assert set(got) == want
    lens = {a: e - a for (a, e) in seqs}
    for valid, b, g, a, k0, qlo, nq in draws[:first_invalid]:
        lo, hi = ab.query_block_range(k0, 128, lens[a], causal, window, 128)
        assert (qlo, nq) == (lo, hi - lo)
    if cu is None:  # key block major inside each group of 8 (batch, KV head) pairs
        pairs = B * HKV
        for g0 in range(0, pairs, 8):
            k0s = [d[4] for d in draws[:first_invalid] if g0 <= d[1] * HKV + d[2] < g0 + 8]
            assert k0s == sorted(k0s)


def test_tile_schedule_rejects_bad_sizes(ab):
    assert ab.tile_schedule(0, 0, 128, 1, True, -1)[0] == 0
    assert ab.tile_schedule(0, 1, 0, 1, True, -1)[0] == 0
    assert ab.tile_schedule(-1, 1, 128, 1, True, -1)[0] == 0


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


def test_sparse_argument_errors_return_before_any_launch(ab):
    """attn_bwd_sparse and its landing pass reject bad calls with a status and
    queue nothing (the fake pointers below are never dereferenced)."""
    lib = ab.library()
    S = ab._binding.Strides
    fake = 1 << 20
    sq = S(4096 * 64 * 576, 64 * 576, 576)
    skv = S(4096 * 576, 576, 576)
    sdo = S(4096 * 64 * 512, 64 * 512, 512)
    sidx = S(4096 * 2048, 2048, 2048)

    def call(q=fake, kv=fake, do=fake, idx=fake, dq=fake, ws=fake, B=1, Sq=4096, SKV=4096, H=64, HKV=1, DQK=576,
             DV=512, topk=2048, dtype=1, scale=0.04, skv_=skv, ws_bytes=1 << 40):
        return lib.attn_bwd_sparse(q, sq, kv, skv_, do, sdo, idx, sidx, B, Sq, SKV, H, HKV, DQK, DV, topk, dtype,
                                   scale, dq, sq, ws, ws_bytes, None)

    assert call(q=None) == 1 and call(idx=None) == 1 and call(ws=None) == 1   # null pointers
    assert call(H=64, HKV=3) == 1                                              # H not a multiple of HKV
    assert call(topk=0) == 1
    assert call(scale=float("inf")) == 1
    assert call(DQK=512) == 2 and call(DV=448) == 2                            # only the 576 / 512 latent row
    assert call(H=128, HKV=1) == 2                                             # more than 64 heads per group
    assert call(dtype=7) == 2
    assert call(q=fake + 8) == 1                                               # misaligned
    assert call(skv_=S(4096 * 640, 640, 600)) == 2                             # latent rows not dense
    assert call(ws_bytes=4096) == 3                                            # workspace too small
    # landing of dKV: bad sizes, dtype, more than 2^31 rows
    assert lib.attn_bwd_sparse_land(fake, skv, 1, 4096, 4096, 64, 1, 570, 1, fake, 1 << 40, None) == 1
    assert lib.attn_bwd_sparse_land(fake, skv, 1, 4096, 4096, 64, 1, 576, 9, fake, 1 << 40, None) == 2
    assert lib.attn_bwd_sparse_land(fake, skv, 1 << 16, 4096, 1 << 16, 64, 1, 576, 1, fake, 1 << 62, None) == 2


def test_landing_and_noalloc_limits_return_before_any_launch(ab):
    lib = ab.library()
    S = ab._binding.Strides
    fake = 1 << 20
    good = S(2048 * 32 * 128, 32 * 128, 128)
    # dQ landing: more than 2^31 (b, s, h) rows is refused
    assert lib.attn_bwd_dq_land(fake, good, 1 << 12, 1 << 12, 1 << 8, 128, 0, 0.1, fake, 1 << 62, None) == 2
    # no-allocation entry point: sizes past its library-held scratch array, and
    # an unsupported head dim, are refused before it touches the device
    m = ab._binding.Mask(1, -1, None, 0)
    lse = S(32 * 65536, 1, 65536)
    big = S(65536 * 32 * 128, 32 * 128, 128)

    def noalloc(Sq=65536, D=128):
        return lib.attn_bwd_gqa_noalloc(fake, big, fake, big, fake, big, fake, big, fake, big, fake, lse, 1, Sq, 32,
                                        32, D, 0, 0.1, ctypes.byref(m), fake, big, fake, big, fake, big, None)

    assert noalloc() == 3
    assert noalloc(D=96) == 2
    # host-buffer entry point: null scratch, unsupported head dim, misaligned scratch
    def host(scratch=fake, D=128, chunks=4):
        return lib.attn_bwd_gqa_host(fake, fake, fake, fake, fake, fake, 2, 2048, 32, 32, D, 0, 0.1,
                                     ctypes.byref(m), fake, fake, fake, scratch, 1 << 40, chunks, None, None, None)

    assert host(scratch=None) == 1
    assert host(D=96) == 2
    assert host(scratch=fake + 16) == 1
    assert lib.attn_bwd_host_scratch_size(2, 2048, 32, 32, 96, 4) == 0
