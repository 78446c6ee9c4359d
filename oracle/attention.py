"""CPU oracle for the fused softmax-attention backward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA library; the only module both sides use is the seeded input generator.

What it computes follows the unsplit f32 ``Reference`` program of the TileOPs
pull request "Serve MHA backward on a warp-specialized SM90 kernel and time
FA3's backward alone" (section "TileFoundry Description"), generalised in the
plainest way to the other cases these gradients are wanted for:

  * per (batch b, query head h) with key/value head g = h // G (contiguous
    query-head groups; GQA as in the flash-linear-attention issue "Evaluate
    KV-head-owned GQA dKV backward", section "Problem"),
  * scores      s_ij = scale * q_i . k_j
  * probability P_ij = exp(s_ij - LSE_i) where key j is visible to query i,
                       else 0   (natural-log LSE; the page's program uses a
                       base-2 LSE with exp2 and a log2(e) factor, which is the
                       same function)
  * row delta   delta_i = sum_d O_id dO_id   (O as given, widened)
  * dV_j = sum_i P_ij dO_i        dP_ij = dO_i . v_j
  * dS_ij = P_ij (dP_ij - delta_i) scale
  * dQ_i = sum_j dS_ij k_j        dK_j = sum_i dS_ij q_i
  * dK and dV of a key/value head are summed over the G query heads that
    read it.

Visibility ("mask"): within one sequence (packed varlen: ``cu_seqlens``
bounds; otherwise each batch row is one sequence), key position j is visible
to query position i iff
  * causal:           j <= i           (the page's ``cols <= rows``)
  * sliding window W: i - W < j <= i   (the pages name sliding-window cases
                                        without defining them; this is the
                                        plain reading: query i sees itself and
                                        the W-1 keys before it)
  * neither:          always.
When the keys of a (dense) batch row outnumber or fall short of its queries
(Sk != Sq; the pages define only Sq == Sk), the masks are aligned at the end
of the row: with off = Sk - Sq, query i stands at key position i + off, so
causal means j <= i + off and the window i + off - W < j <= i + off.  A query
with no visible key (i + off < 0) gets P = 0.

Sparse (top-k) attention follows the tilelang pull request "Adaptive threads
for sparse MLA backward" (sections "Motivation" and "Benchmark"): one latent
row per key holds both K (all DQK columns) and V (its first DV columns), and
query t attends exactly the key rows listed in ``idx[t]``; entries outside
[0, Skv) (the -1 padding) are not visible.  dKV_j = dK_j + [dV_j, 0].

Attention sink (named among the gradients of the flash-linear-attention
issue's "Frozen correctness contract" as dsink, without a formula; the plain
reading): one extra logit sink_h per query head joins every row's softmax
normalisation and carries no value, so LSE_i = log(sum_j exp(s_ij) +
exp(sink_h)) and O_i = sum_j exp(s_ij - LSE_i) v_j.  The sink's column has
dP = dO_i . 0 = 0, so dS_i,sink = -P_i,sink delta_i and
dsink_h = -sum_i exp(sink_h - LSE_i) delta_i; dQ, dK and dV keep the formulas
above with that O and LSE.

The forward that produces O and LSE runs in float32 (O is rounded to the input
dtype by the caller); the backward runs in float64.  The forward is exact
(two passes: max, then sum), not an online softmax.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


# --------------------------------------------------------------------------
# Visibility
# --------------------------------------------------------------------------

def sequences(S: int, cu_seqlens: Optional[Sequence[int]]):
    """(start, end) of every sequence along a batch row of length S."""
    if cu_seqlens is None:
        return [(0, S)]
    cu = [int(x) for x in cu_seqlens]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def visible(S: int, causal: bool, window: int, cu_seqlens=None) -> np.ndarray:
    """Brute-force visibility matrix M[i, j] (query i, key j) of one batch row."""
    seq_id = np.full(S, -1, dtype=np.int64)
    start = np.zeros(S, dtype=np.int64)
    for n, (a, b) in enumerate(sequences(S, cu_seqlens)):
        seq_id[a:b] = n
        start[a:b] = a
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    li = i - start[:, None]
    lj = j - start[None, :]
    m = (seq_id[:, None] == seq_id[None, :]) & (seq_id[:, None] >= 0)
    if causal or window > 0:
        m &= lj <= li
    if window > 0:
        m &= lj > li - window
    return m


def _visible_block(rows: np.ndarray, cols: np.ndarray, causal: bool, window: int, off: int = 0) -> np.ndarray:
    """Visibility of sequence-local query positions ``rows`` to key positions ``cols``
    (both inside the same sequence; query i stands at key position i + off)."""
    li = rows[:, None] + off
    lj = cols[None, :]
    m = np.ones((rows.size, cols.size), dtype=bool)
    if causal or window > 0:
        m &= lj <= li
    if window > 0:
        m &= lj > li - window
    return m


def _row_sequences(Sq: int, Sk: int, cu_seqlens):
    """(query start, query end, key start, key end, off) of every sequence of a
    batch row: packed sequences share their bounds; a dense row with Sk != Sq
    aligns its queries with the last Sq key positions."""
    if cu_seqlens is not None:
        if Sq != Sk:
            raise ValueError("packed sequences need equal query and key lengths")
        return [(a, e, a, e, 0) for (a, e) in sequences(Sq, cu_seqlens)]
    return [(0, Sq, 0, Sk, Sk - Sq)]


# --------------------------------------------------------------------------
# Dense forward (produces the O and LSE inputs of the backward)
# --------------------------------------------------------------------------

def forward(q, k, v, scale, causal=False, window=-1, cu_seqlens=None, dtype=np.float32,
            row_chunk=2048, sink=None):
    """O [B,S,HQ,Dv] and natural-log LSE [B,HQ,S] of softmax attention over
    keys k [B,Sk,HKV,D] and values v [B,Sk,HKV,Dv] (Sk = S unless the row is
    dense; see the module notes on Sk != S).

    Rows with no visible key get LSE = -inf and O = 0.  ``sink`` (one logit per
    query head) joins every row's normalisation (module notes): such a row then
    gets LSE = sink_h and O = 0.
    """
    B, S, HQ, _ = q.shape
    HKV = k.shape[2]
    G = HQ // HKV
    Dv = v.shape[3]
    o = np.zeros((B, S, HQ, Dv), dtype=dtype)
    lse = np.full((B, HQ, S), -np.inf, dtype=dtype)

    def unit(b, h):
        g = h // G
        for (a, e, ka, ke, off) in _row_sequences(S, k.shape[1], cu_seqlens):
            K = k[b, ka:ke, g, :].astype(dtype)
            V = v[b, ka:ke, g, :].astype(dtype)
            cols = np.arange(ke - ka)
            for r0 in range(0, e - a, row_chunk):
                r1 = min(e - a, r0 + row_chunk)
                Q = q[b, a + r0:a + r1, h, :].astype(dtype)
                s = (Q @ K.T) * dtype(scale)
                m = _visible_block(np.arange(r0, r1), cols, causal, window, off)
                s = np.where(m, s, -np.inf)
                mx = s.max(axis=1, keepdims=True)
                if sink is not None:
                    mx = np.maximum(mx, dtype(sink[h]))
                mx = np.where(np.isfinite(mx), mx, 0)
                e_ = np.exp(s - mx)
                tot = e_.sum(axis=1, keepdims=True)
                if sink is not None:
                    tot = tot + np.exp(dtype(sink[h]) - mx)
                with np.errstate(divide="ignore"):
                    lse[b, h, a + r0:a + r1] = (mx + np.log(tot))[:, 0]
                p = np.where(tot > 0, e_ / np.where(tot > 0, tot, 1), 0)
                o[b, a + r0:a + r1, h, :] = p @ V

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(lambda bh: unit(*bh), [(b, h) for b in range(B) for h in range(HQ)]))
    return o, lse


# --------------------------------------------------------------------------
# Dense backward
# --------------------------------------------------------------------------

def backward(q, k, v, o, do, lse, scale, causal=False, window=-1, cu_seqlens=None,
             q_rows=None, k_rows=None, heads=None):
    """dQ [B,S,HQ,D], dK [B,Sk,HKV,D], dV [B,Sk,HKV,Dv] in float64 (Sk = the key
    length of k, S unless the row is dense; see the module notes).

    ``q_rows`` / ``k_rows`` (positions along the query, respectively key,
    length) restrict which rows of dQ, respectively of dK and dV, are computed;
    the others are left as NaN.  ``heads`` restricts the query heads visited
    (dK/dV then sum only those).  With both row sets None every row is computed.
    """
    B, S, HQ, D = q.shape
    Sk = k.shape[1]
    HKV = k.shape[2]
    G = HQ // HKV
    Dv = v.shape[3]
    full = q_rows is None and k_rows is None
    dq = np.full((B, S, HQ, D), np.nan)
    dk = np.full((B, Sk, HKV, D), np.nan)
    dv = np.full((B, Sk, HKV, Dv), np.nan)
    head_list = list(range(HQ)) if heads is None else list(heads)
    qsel = np.zeros(S, bool) if q_rows is None else np.isin(np.arange(S), q_rows)
    ksel = np.zeros(Sk, bool) if k_rows is None else np.isin(np.arange(Sk), k_rows)
    if full:
        qsel[:] = True
        ksel[:] = True
    seqs = _row_sequences(S, Sk, cu_seqlens)

    def unit(b, h):
        g = h // G
        out = []
        for (a, e, ka, ke, off) in seqs:
            qpos = np.arange(e - a)
            kpos = np.arange(ke - ka)
            Qf = q[b, a:e, h, :].astype(np.float64)
            Kf = k[b, ka:ke, g, :].astype(np.float64)
            Vf = v[b, ka:ke, g, :].astype(np.float64)
            Of = o[b, a:e, h, :].astype(np.float64)
            dOf = do[b, a:e, h, :].astype(np.float64)
            L = lse[b, h, a:e].astype(np.float64)
            delta = (Of * dOf).sum(axis=1)
            qi = np.nonzero(qsel[a:e])[0]
            kj = np.nonzero(ksel[ka:ke])[0]
            if full:
                qi, kj = qpos, kpos
            res = {"a": a, "ka": ka, "qi": qi, "kj": kj}
            if qi.size:
                # rows of dQ: every key of the sequence
                s = scale * (Qf[qi] @ Kf.T)
                m = _visible_block(qi, kpos, causal, window, off)
                P = np.where(m, np.exp(np.where(m, s - L[qi, None], 0.0)), 0.0)
                dP = dOf[qi] @ Vf.T
                dS = P * (dP - delta[qi, None]) * scale
                res["dq"] = dS @ Kf
                if full:
                    res["dk"] = dS.T @ Qf
                    res["dv"] = P.T @ dOf
            if kj.size and not full:
                # rows of dK and dV: every query of the sequence
                s = scale * (Qf @ Kf[kj].T)
                m = _visible_block(qpos, kj, causal, window, off)
                P = np.where(m, np.exp(np.where(m, s - L[:, None], 0.0)), 0.0)
                dP = dOf @ Vf[kj].T
                dS = P * (dP - delta[:, None]) * scale
                res["dk"] = dS.T @ Qf
                res["dv"] = P.T @ dOf
            out.append(res)
        return b, h, g, out

    units = [(b, h) for b in range(B) for h in head_list]
    with ThreadPoolExecutor(_threads()) as ex:
        results = list(ex.map(lambda bh: unit(*bh), units))
    # dK/dV of a key/value head: sum over its query heads, in head order
    for b in range(B):
        for g in range(HKV):
            for (a, e, ka, ke, off) in seqs:
                kj = np.nonzero(ksel[ka:ke])[0] if not full else np.arange(ke - ka)
                dk[b, ka + kj, g, :] = 0.0
                dv[b, ka + kj, g, :] = 0.0
    for b, h, g, out in results:
        for res in out:
            if "dq" in res:
                dq[b, res["a"] + res["qi"], h, :] = res["dq"]
            if "dk" in res:
                dk[b, res["ka"] + res["kj"], g, :] += res["dk"]
                dv[b, res["ka"] + res["kj"], g, :] += res["dv"]
    return dq, dk, dv


def sink_grad(o, do, lse, sink, cu_seqlens=None):
    """dsink [HQ] in float64: -sum over the rows of every sequence (all batch
    rows) of exp(sink_h - LSE_i) delta_i (module notes); rows whose LSE is not
    finite add nothing."""
    B, S, HQ, _ = o.shape
    d = delta(o, do)
    rows = np.zeros(S, dtype=bool)
    for a, e in sequences(S, cu_seqlens):
        rows[a:e] = True
    out = np.zeros(HQ)
    for h in range(HQ):
        l = lse[:, h, :].astype(np.float64)[:, rows]
        ok = np.isfinite(l)
        w = np.where(ok, np.exp(float(sink[h]) - np.where(ok, l, 0.0)), 0.0)
        out[h] = -(w * d[:, h, rows]).sum()
    return out


def delta(o, do):
    """delta [B,H,S] = sum over the head dim of O * dO, in float64."""
    return np.einsum("bshd,bshd->bhs", o.astype(np.float64), do.astype(np.float64))


# --------------------------------------------------------------------------
# Sparse (top-k, shared latent K/V) forward and backward
# --------------------------------------------------------------------------

def _valid_slots(idx_row: np.ndarray, skv: int) -> np.ndarray:
    return idx_row[(idx_row >= 0) & (idx_row < skv)]


def sparse_forward(q, kv, idx, scale, dv_dim, dtype=np.float32, tokens=None):
    """O [B,S,H,DV] and LSE [B,H,S] of top-k attention over latent rows.

    q [B,S,H,DQK]; kv [B,SKV,HKV,DQK] (V = kv[..., :DV]); idx [B,S,HKV,topk].
    ``tokens`` restricts the query positions computed (others stay 0 / -inf).
    """
    B, S, H, DQK = q.shape
    SKV, HKV = kv.shape[1], kv.shape[2]
    G = H // HKV
    o = np.zeros((B, S, H, dv_dim), dtype=dtype)
    lse = np.full((B, H, S), -np.inf, dtype=dtype)
    toks = range(S) if tokens is None else tokens

    def unit(b, t):
        for g in range(HKV):
            sl = _valid_slots(idx[b, t, g], SKV)
            if sl.size == 0:
                continue
            Kt = kv[b, sl, g, :].astype(dtype)
            Qt = q[b, t, g * G:(g + 1) * G, :].astype(dtype)
            s = (Qt @ Kt.T) * dtype(scale)
            mx = s.max(axis=1, keepdims=True)
            e_ = np.exp(s - mx)
            tot = e_.sum(axis=1, keepdims=True)
            lse[b, g * G:(g + 1) * G, t] = (mx + np.log(tot))[:, 0]
            o[b, t, g * G:(g + 1) * G, :] = (e_ / tot) @ Kt[:, :dv_dim]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(lambda bt: unit(*bt), [(b, t) for b in range(B) for t in toks]))
    return o, lse


def sparse_backward(q, kv, o, do, lse, idx, scale, dv_dim, tokens=None, kv_rows=None):
    """dQ [B,S,H,DQK] and dKV [B,SKV,HKV,DQK] in float64.

    ``tokens`` restricts the dQ rows computed (others NaN).  ``kv_rows``
    restricts the dKV rows computed (others NaN); when it is given, every
    query token contributes to those rows.  With both None everything is
    computed.
    """
    B, S, H, DQK = q.shape
    SKV, HKV = kv.shape[1], kv.shape[2]
    G = H // HKV
    dq = np.full((B, S, H, DQK), np.nan)
    dkv = np.full((B, SKV, HKV, DQK), np.nan)
    full = tokens is None and kv_rows is None
    qtok = np.arange(S) if (tokens is None and kv_rows is None) else (
        np.asarray(tokens) if tokens is not None else np.zeros(0, np.int64))
    rows_wanted = None if kv_rows is None else np.asarray(kv_rows)

    def token_grads(b, t, g):
        """P, dS over the valid slots of token t, heads of group g."""
        sl = _valid_slots(idx[b, t, g], SKV)
        hs = slice(g * G, (g + 1) * G)
        Kt = kv[b, sl, g, :].astype(np.float64)
        Qt = q[b, t, hs, :].astype(np.float64)
        dOt = do[b, t, hs, :].astype(np.float64)
        Ot = o[b, t, hs, :].astype(np.float64)
        L = lse[b, hs, t].astype(np.float64)
        s = scale * (Qt @ Kt.T)
        P = np.exp(s - L[:, None])
        dP = dOt @ Kt[:, :dv_dim].T
        dlt = (Ot * dOt).sum(axis=1)
        dS = P * (dP - dlt[:, None]) * scale
        return sl, Kt, Qt, dOt, P, dS

    def unit(b, t):
        res = []
        for g in range(HKV):
            sl, Kt, Qt, dOt, P, dS = token_grads(b, t, g)
            r = {"g": g, "dq": dS @ Kt if sl.size else np.zeros((G, DQK))}
            if full:
                contrib = dS.T @ Qt
                contrib[:, :dv_dim] += P.T @ dOt
                r["sl"] = sl
                r["dkv"] = contrib
            res.append(r)
        return b, t, res

    if full or qtok.size:
        with ThreadPoolExecutor(_threads()) as ex:
            results = list(ex.map(lambda bt: unit(*bt), [(b, int(t)) for b in range(B) for t in qtok]))
        if full:
            dkv[:] = 0.0
        for b, t, res in results:
            for r in res:
                g = r["g"]
                dq[b, t, g * G:(g + 1) * G, :] = r["dq"]
                if full and r["sl"].size:
                    np.add.at(dkv[b, :, g, :], r["sl"], r["dkv"])

    if rows_wanted is not None:
        # dKV[j] = sum over the (token, slot) pairs that list row j of
        # dS[:, slot]^T Q_t (+ P[:, slot]^T dO_t on the value columns); P and dS
        # of such a slot need only row j itself and the token's LSE and delta.
        dlt_all = (o.astype(np.float64) * do.astype(np.float64)).sum(axis=-1)  # [B,S,H]

        def row_grad(b, g, j):
            hs = slice(g * G, (g + 1) * G)
            lists = idx[b, :, g, :]
            mult = (lists == j).sum(axis=1)          # a repeated index is a separate slot
            toks_j = np.nonzero(mult)[0]
            acc = np.zeros(DQK)
            if j < 0 or j >= SKV or toks_j.size == 0:
                return b, g, j, acc
            Kj = kv[b, j, g, :].astype(np.float64)
            for c0 in range(0, toks_j.size, 256):
                tt = toks_j[c0:c0 + 256]
                Qt = q[b, tt][:, hs, :].astype(np.float64)       # [n, G, DQK]
                dOt = do[b, tt][:, hs, :].astype(np.float64)     # [n, G, DV]
                L = lse[b, hs][:, tt].T.astype(np.float64)       # [n, G]
                P = np.exp(scale * (Qt @ Kj) - L)                # [n, G]
                dP = dOt @ Kj[:dv_dim]
                dS = P * (dP - dlt_all[b, tt][:, hs]) * scale
                m = mult[tt].astype(np.float64)[:, None]
                acc += np.einsum("ng,ngd->d", dS * m, Qt)
                acc[:dv_dim] += np.einsum("ng,ngd->d", P * m, dOt)
            return b, g, j, acc

        jobs = [(b, g, int(j)) for b in range(B) for g in range(HKV) for j in rows_wanted]
        with ThreadPoolExecutor(_threads()) as ex:
            for b, g, j, acc in ex.map(lambda a: row_grad(*a), jobs):
                dkv[b, j, g, :] = acc
    return dq, dkv
