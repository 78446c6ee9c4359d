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
    """Every entry point the public headers (include/*.h) declare."""
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    return sorted(set(re.findall(r"ATTN_BWD_API\s+[\w\s\*]+?\b(attn_(?:bwd|fwd)\w*)\s*\(", src)))


def test_every_declared_symbol_is_exported(ab):
    names = declared_symbols()
    assert len(names) >= 11
    lib = ab.library()
    for n in names:
        assert hasattr(lib, n), n
    # and nothing else leaks out as a C symbol of ours
    assert "attn_bwd_gqa" in names and "attn_bwd_sparse" in names and "attn_bwd_preprocess" in names
    assert "attn_fwd_gqa" in names


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


@pytest.mark.parametrize("sq,sk", [(100, 300), (300, 100), (257, 1000), (1000, 257), (128, 129), (129, 128),
                                   (1, 700), (700, 1)])
@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 1), (True, 100)])
@pytest.mark.parametrize("bq", [64, 128])
def test_query_block_range_of_unequal_rows_matches_brute_force(ab, sq, sk, causal, window, bq):
    """A dense row of sq queries and sk keys, masks aligned at the end of the
    row (the oracle's visibility with off = sk - sq): every query block with a
    visible pair is visited and no other block is."""
    from oracle.attention import _visible_block

    vis = _visible_block(np.arange(sq), np.arange(sk), causal, window, sk - sq)
    for k0 in range(0, sk, 128):
        lo, hi = ab.query_block_range_qk(k0, 128, sk, sq, causal, window, bq)
        rows = np.nonzero(vis[:, k0:k0 + 128].any(axis=1))[0]
        assert set(range(lo, hi)) == set((rows // bq).tolist()), (k0, lo, hi)
    for k0 in range(0, 1000, 128):  # equal lengths: the square helper
        assert ab.query_block_range_qk(k0, 128, 1000, 1000, causal, window, bq) == \
            ab.query_block_range(k0, 128, 1000, causal, window, bq)


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


@pytest.mark.parametrize("tiles,ctas,G,want", [
    (512, 152, 8, (456, 56, 1)),     # GQA 16384 with 4 KV heads: 3 rounds and 56 tiles, as 448 one-head units
    (160, 152, 2, (152, 8, 1)),      # 8 tiles left over, as 16 one-head units
    (304, 152, 8, (0, 0, 0)),        # tiles divide evenly
    (100, 152, 8, (0, 0, 0)),        # one round
    (160, 152, 1, (0, 0, 0)),        # one query head per KV head: nothing to split
    (303, 152, 2, (0, 0, 0)),        # 151 tiles left over: one-head units would take as long
    (200, 152, 4, (152, 48, 2)),     # 48 tiles as 96 two-head units: one unit round of half a tile
])
def test_tail_plan(ab, tiles, ctas, G, want):
    assert ab.tail_plan(tiles, ctas, G) == want


def test_tail_plan_is_the_best_split_by_brute_force(ab):
    """Over a grid of tile counts, CTA counts and group sizes: a plan is taken
    only when its makespan (in 1/G tiles) beats drawing whole tiles by the
    stated margin, and no other head count per unit does better."""
    for G in (1, 2, 3, 4, 6, 8, 12, 16):
        for ctas in (1, 5, 7, 148, 152):
            for T in list(range(1, 40)) + [151, 152, 153, 160, 200, 303, 304, 456, 512, 1000]:
                start, ntail, hpu = ab.tail_plan(T, ctas, G)
                full, R = divmod(T, ctas)
                whole = (full + (1 if R else 0)) * G
                options = {h: full * G + -(-(R * (G // h)) // ctas) * h for h in range(1, G) if G % h == 0}
                best = min(options.values()) if options and R and T > ctas else whole
                if ntail == 0:
                    assert G < 2 or T <= ctas or R == 0 or R > 256 or whole - best < max(1, G // 4), (T, ctas, G)
                else:
                    assert (start, ntail) == (T - R, R) and G % hpu == 0 and hpu < G
                    assert options[hpu] == best and whole - best >= max(1, G // 4)
                    assert hpu == max(h for h, v in options.items() if v == best)


@pytest.mark.parametrize("B,S,HKV,G,ctas", [(1, 16384, 4, 8, 152), (1, 1000, 20, 2, 152), (2, 512, 20, 8, 152),
                                            (3, 300, 5, 4, 7)])
def test_split_schedule_covers_every_head_of_every_tile_once(ab, B, S, HKV, G, ctas):
    """With the last-round split the draws cover every (batch, KV head, key
    tile, query head) exactly once: whole tiles take all G heads, the split
    tiles come as units of the planned head count with a partials slot per
    tile, and the draws end together."""
    tiles = B * HKV * ((S + 127) // 128)
    start, ntail, hpu = ab.tail_plan(tiles, ctas, G)
    assert ntail > 0
    want = {(b, g, k0, h) for b in range(B) for g in range(HKV) for k0 in range(0, S, 128) for h in range(G)}
    got, slot_tile = [], {}
    for t in range(start + ntail * (G // hpu) + 4):
        valid, b, g, s0, k0, qlo, nq, h0, hn, part = ab.tile_schedule_split(t, B, S, HKV, G, start, ntail, hpu)
        if t >= start + ntail * (G // hpu):
            assert not valid
            continue
        assert valid and s0 == 0 and (qlo, nq) == (0, (S + 127) // 128)
        if t < start:
            assert (h0, hn, part) == (0, G, -1)
            assert ab.tile_schedule(t, B, S, HKV, False, -1)[1:5] == (b, g, 0, k0)
        else:
            assert hn == hpu and 0 <= part < ntail and h0 % hpu == 0
            assert slot_tile.setdefault(part, (b, g, k0)) == (b, g, k0)
            assert ab.tile_schedule(start + part, B, S, HKV, False, -1)[1:5] == (b, g, 0, k0)
        got += [(b, g, k0, h) for h in range(h0, h0 + hn)]
    assert len(got) == len(set(got)) == len(want) and set(got) == want
    assert len(slot_tile) == ntail


def test_gqa_workspace_holds_the_last_round_partials(ab):
    base = ab.workspace_size(1, 16384, 32, 128)
    # 256 tiles of 2 x 128 x 128 f32 partials and 4 counters, behind the dQ accumulator
    assert ab.gqa_workspace_size(1, 16384, 32, 128) == base + 256 * 4 * 4 + 256 * 2 * 128 * 128 * 4
    # at most one tile per (query head, key block) of the batch: 2 here
    assert ab.gqa_workspace_size(1, 100, 2, 128) == ab.workspace_size(1, 100, 2, 128) + 256 + 2 * 2 * 128 * 128 * 4
    assert ab.gqa_workspace_size(1, 4096, 8, 64) == ab.workspace_size(1, 4096, 8, 64)  # head dim 64: no split


def test_tile_schedule_rejects_bad_sizes(ab):
    assert ab.tile_schedule(0, 0, 128, 1, True, -1)[0] == 0
    assert ab.tile_schedule(0, 1, 0, 1, True, -1)[0] == 0
    assert ab.tile_schedule(-1, 1, 128, 1, True, -1)[0] == 0


def test_sink_grad_rejects_bad_calls_before_any_launch(ab):
    lib = ab.library()
    fake = 1 << 20
    m = ab._binding.Mask(0, -1, None, 0)
    ws = ab.workspace_size(2, 100, 4, 0)

    def call(sink=fake, B=2, S=100, H=4, mask=m, ws_ptr=fake, ws_bytes=ws, dsink=fake):
        return lib.attn_bwd_sink_grad(sink, B, S, H, ctypes.byref(mask), ws_ptr, ws_bytes, dsink, None)

    assert call(sink=None) == 1 and call(dsink=None) == 1 and call(ws_ptr=None) == 1   # null pointers
    assert call(sink=fake + 2) == 1 and call(ws_ptr=fake + 4) == 1                      # misaligned
    assert call(B=0) == 1 and call(H=0) == 1
    assert call(ws_bytes=ws - 512) == 3                                                # no room for LSE2 / delta
    assert call(mask=ab._binding.Mask(0, -1, fake, 2)) == 1                            # packed rows with B > 1


def test_argument_errors_return_before_any_launch(ab):
    """The split-form launches reject bad calls with a status and queue nothing
    (the fake pointers are 16-byte aligned and never dereferenced)."""
    lib = ab.library()
    S = ab._binding.Strides
    z = S(0, 0, 0)
    good = S(2048 * 32 * 128, 32 * 128, 128)
    m = ab._binding.Mask(1, -1, None, 0)
    fake = 1 << 20

    def main(q=fake, sq=good, B=2, H=32, HKV=32, D=128, dtype=0, scale=0.1, mask=m, ws_bytes=1 << 30):
        return lib.attn_bwd_gqa_main(q, sq, fake, good, fake, good, fake, good, B, 2048, H, HKV, D, dtype, scale,
                                     ctypes.byref(mask), fake, good, fake, good, fake, ws_bytes, None)

    assert lib.attn_bwd_gqa_main(None, good, None, good, None, good, None, good, 2, 2048, 32, 32, 128, 0, 0.1,
                                 ctypes.byref(m), None, good, None, good, None, 0, None) == 1   # null pointers
    assert main(D=96) == 2                                 # unsupported head dim
    assert main(H=6, HKV=4) == 1                           # HQ not a multiple of HKV
    assert main(q=fake + 2) == 1                           # misaligned pointer
    assert main(sq=z) == 1                                 # zero strides
    assert main(ws_bytes=1024) == 3                        # workspace too small
    assert main(mask=ab._binding.Mask(1, 0, None, 0)) == 1            # window of zero
    assert main(mask=ab._binding.Mask(1, -1, fake, 3)) == 1           # varlen with B > 1
    assert main(scale=float("nan")) == 1
    # group sizes beyond the limit: 16 heads per KV head in either dtype
    assert main(H=32, HKV=1) == 2
    assert main(H=32, HKV=1, dtype=1) == 2
    # preprocess: bad head dim, workspace too small
    assert lib.attn_bwd_preprocess(fake, good, fake, good, fake, S(64, 1, 2048), 2, 2048, 32, 12, 128, 0, 0,
                                   fake, 1 << 30, None) == 1
    assert lib.attn_bwd_preprocess(fake, good, fake, good, fake, S(64, 1, 2048), 2, 2048, 32, 128, 128, 0, 0,
                                   fake, 4096, None) == 3
    # landing: unsupported dtype code, non-finite scale
    assert lib.attn_bwd_dq_land(fake, good, 2, 2048, 32, 128, 7, 0.1, fake, 1 << 30, None) == 2
    assert lib.attn_bwd_dq_land(fake, good, 2, 2048, 32, 128, 0, float("inf"), fake, 1 << 30, None) == 1


def _one_call_args(ab, **kw):
    """Arguments of attn_bwd_gqa / attn_bwd_gqa_noalloc for a 2x2048x32x128
    problem, with fake (never dereferenced) pointers; keywords override."""
    S = ab._binding.Strides
    fake = 1 << 20
    a = dict(q=fake, sq=S(2048 * 32 * 128, 32 * 128, 128), o=fake, lse=fake, slse=S(32 * 2048, 1, 2048),
             dq=fake, dk=fake, B=2, S=2048, HQ=32, HKV=32, D=128, dtype=0, scale=0.1,
             mask=ab._binding.Mask(1, -1, None, 0), ws=fake, ws_bytes=1 << 32)
    a.update(kw)
    return a


def _gqa(ab, **kw):
    a = _one_call_args(ab, **kw)
    f = 1 << 20
    sq = a["sq"]
    return ab.library().attn_bwd_gqa(a["q"], sq, f, sq, f, sq, a["o"], sq, f, sq, a["lse"], a["slse"], a["B"],
                                     a["S"], a["HQ"], a["HKV"], a["D"], a["dtype"], a["scale"],
                                     ctypes.byref(a["mask"]), a["dq"], sq, a["dk"], sq, f, sq, a["ws"],
                                     a["ws_bytes"], None)


def _noalloc(ab, **kw):
    a = _one_call_args(ab, **kw)
    f = 1 << 20
    sq = a["sq"]
    return ab.library().attn_bwd_gqa_noalloc(a["q"], sq, f, sq, f, sq, a["o"], sq, f, sq, a["lse"], a["slse"],
                                             a["B"], a["S"], a["HQ"], a["HKV"], a["D"], a["dtype"], a["scale"],
                                             ctypes.byref(a["mask"]), a["dq"], sq, a["dk"], sq, f, sq, None)


BAD_CALLS = [
    # (name, overrides, status): 1 invalid argument, 2 unsupported, 3 workspace
    ("null q", dict(q=None), 1),
    ("null o", dict(o=None), 1),
    ("null lse", dict(lse=None), 1),
    ("null dq", dict(dq=None), 1),
    ("misaligned q", dict(q=(1 << 20) + 2), 1),
    ("misaligned dq", dict(dq=(1 << 20) + 8), 1),
    ("misaligned lse", dict(lse=(1 << 20) + 2), 1),
    ("odd stride", dict(sq=None), 1),
    ("HQ % HKV", dict(HQ=6, HKV=4), 1),
    ("window 0", dict(mask=None), 1),
    ("window -2", dict(mask="w-2"), 1),
    ("varlen B > 1", dict(mask="varlen"), 1),
    ("varlen no sequences", dict(mask="varlen0", B=1), 1),
    ("negative kv_len", dict(mask="kvneg"), 1),
    ("kv_len with varlen", dict(mask="kvvarlen", B=1), 1),
    ("NaN scale", dict(scale=float("nan")), 1),
    ("infinite scale", dict(scale=float("inf")), 1),
    ("head dim 96", dict(D=96), 2),
    ("dtype 7", dict(dtype=7), 2),
    ("G = 32 fp16", dict(HQ=32, HKV=1), 2),
    ("G = 32 bf16", dict(HQ=32, HKV=1, dtype=1), 2),
]


def _resolve(ab, kw):
    S, M = ab._binding.Strides, ab._binding.Mask
    kw = dict(kw)
    if "sq" in kw and kw["sq"] is None:
        kw["sq"] = S(2048 * 32 * 128, 32 * 128 + 4, 128)  # 8-byte head stride: not a 16-byte multiple
    if "mask" in kw:
        kw["mask"] = {None: M(1, 0, None, 0), "w-2": M(1, -2, None, 0), "varlen": M(1, -1, 1 << 20, 3),
                      "varlen0": M(1, -1, 1 << 20, 0), "kvneg": M(1, -1, None, 0, -5),
                      "kvvarlen": M(1, -1, 1 << 20, 3, 100)}[kw["mask"]]
    return kw


@pytest.mark.parametrize("name,kw,status", BAD_CALLS, ids=[c[0] for c in BAD_CALLS])
def test_one_call_forms_reject_before_any_launch(ab, name, kw, status):
    """attn_bwd_gqa checks every argument of its three launches before it
    queues the first; attn_bwd_gqa_noalloc makes the same checks before it
    touches the device (no GPU here: a call that got further would fail
    differently)."""
    kw = _resolve(ab, kw)
    assert _gqa(ab, **kw) == status, name
    # a problem that fits the library-held 32 MiB workspace
    assert _noalloc(ab, **{"S": 256, **kw}) == status, name


def test_one_call_workspace_and_sparse_checks(ab):
    lib = ab.library()
    S = ab._binding.Strides
    assert _gqa(ab, ws_bytes=4096) == 3
    assert _gqa(ab, ws=None) == 1
    fake = 1 << 20
    sq = S(4096 * 64 * 576, 64 * 576, 576)
    skv = S(4096 * 576, 576, 576)
    sdo = S(4096 * 64 * 512, 64 * 512, 512)
    sidx = S(4096 * 2048, 2048, 2048)
    sl = S(64 * 4096, 1, 4096)

    def sparse(o=fake, lse=fake, dkv=fake, sdkv=skv, dtype=1, ws_bytes=1 << 40, topk=2048):
        return lib.attn_bwd_sparse(fake, sq, fake, skv, o, sdo, fake, sdo, lse, sl, fake, sidx, 1, 4096, 4096, 64, 1,
                                   576, 512, topk, dtype, 0.04, fake, sq, dkv, sdkv, fake, ws_bytes, None)

    assert sparse(o=None) == 1 and sparse(lse=None) == 1 and sparse(dkv=None) == 1
    assert sparse(dkv=fake + 4) == 1
    assert sparse(sdkv=S(0, 0, 0)) == 1
    assert sparse(ws_bytes=4096) == 3
    assert sparse(topk=0) == 1
    assert sparse(dtype=5) == 2


def test_sparse_argument_errors_return_before_any_launch(ab):
    """attn_bwd_sparse_main and its landing pass reject bad calls with a status
    and queue nothing (the fake pointers below are never dereferenced)."""
    lib = ab.library()
    S = ab._binding.Strides
    fake = 1 << 20
    sq = S(4096 * 64 * 576, 64 * 576, 576)
    skv = S(4096 * 576, 576, 576)
    sdo = S(4096 * 64 * 512, 64 * 512, 512)
    sidx = S(4096 * 2048, 2048, 2048)

    def call(q=fake, kv=fake, do=fake, idx=fake, dq=fake, ws=fake, B=1, Sq=4096, SKV=4096, H=64, HKV=1, DQK=576,
             DV=512, topk=2048, dtype=1, scale=0.04, skv_=skv, ws_bytes=1 << 40):
        return lib.attn_bwd_sparse_main(q, sq, kv, skv_, do, sdo, idx, sidx, B, Sq, SKV, H, HKV, DQK, DV, topk,
                                        dtype, scale, dq, sq, ws, ws_bytes, None)

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
    def host(scratch=fake, D=128, chunks=4, mask=m):
        return lib.attn_bwd_gqa_host(fake, fake, fake, fake, fake, fake, 2, 2048, 32, 32, D, 0, 0.1,
                                     ctypes.byref(mask), fake, fake, fake, scratch, 1 << 40, chunks, None, None, None)

    assert host(scratch=None) == 1
    assert host(D=96) == 2
    assert host(scratch=fake + 16) == 1
    assert host(mask=ab._binding.Mask(1, -1, None, 0, 4096)) == 1   # key rows of another length
    assert lib.attn_bwd_host_scratch_size(2, 2048, 32, 32, 96, 4) == 0


def test_forward_rejects_before_any_launch(ab):
    """attn_fwd_gqa checks every argument before it touches the device."""
    lib = ab.library()
    S, M = ab._binding.Strides, ab._binding.Mask
    fake = 1 << 20
    good = S(2048 * 32 * 128, 32 * 128, 128)
    lse = S(32 * 2048, 1, 2048)

    def fwd(q=fake, o=fake, lse_=fake, ws=fake, ws_bytes=256, D=128, HQ=32, HKV=32, B=2, dtype=0, scale=0.1,
            mask=M(1, -1, None, 0), sq=good):
        return lib.attn_fwd_gqa(q, sq, fake, good, fake, good, B, 2048, HQ, HKV, D, dtype, scale, ctypes.byref(mask),
                                o, good, lse_, lse, ws, ws_bytes, None)

    assert fwd(q=None) == 1 and fwd(o=None) == 1 and fwd(lse_=None) == 1 and fwd(ws=None) == 1
    assert fwd(q=fake + 2) == 1 and fwd(lse_=fake + 2) == 1
    assert fwd(sq=S(0, 0, 0)) == 1
    assert fwd(HQ=6, HKV=4) == 1
    assert fwd(scale=0.0) == 1 and fwd(scale=-0.1) == 1 and fwd(scale=float("nan")) == 1
    assert fwd(D=96) == 2 and fwd(dtype=7) == 2
    assert fwd(ws_bytes=128) == 3
    assert fwd(mask=M(1, 0, None, 0)) == 1
    assert fwd(mask=M(1, -1, fake, 3)) == 1                  # varlen with B > 1
    assert fwd(B=1, mask=M(1, -1, fake, 3, 100)) == 1         # a key length with packed sequences
    assert fwd(mask=M(1, -1, None, 0, -1)) == 1
