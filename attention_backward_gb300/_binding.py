"""ctypes binding of the C ABI in ``include/attn_bwd.h``.

Argument marshalling only: torch tensors are turned into device pointers and
element strides, the current torch CUDA stream into a cudaStream_t, and
non-zero status codes into ``AttnBwdError``.  Every arithmetic step runs in
the library's kernels.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libattn_bwd.so")

c_i32, c_i64, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

DT_F16, DT_BF16 = 0, 1


class AttnBwdError(RuntimeError):
    pass


class Strides(ctypes.Structure):
    _fields_ = [("b", c_i64), ("s", c_i64), ("h", c_i64)]


class Mask(ctypes.Structure):
    _fields_ = [("causal", c_i32), ("window_left", c_i32), ("cu_seqlens", c_vp), ("num_seqs", c_i32),
                ("kv_len", c_i32)]


_SIGS = {
    "attn_bwd_workspace_size": (c_sz, [c_i64, c_i64, c_i64, c_i64, c_i64]),
    "attn_bwd_gqa_workspace_size": (c_sz, [c_i64, c_i64, c_i64, c_i64]),
    "attn_bwd_sink_grad": (c_i32, [c_vp, c_i64, c_i64, c_i64, ctypes.POINTER(Mask), c_vp, c_sz, c_vp, c_vp]),
    "attn_bwd_tail_plan": (None, [c_i64, c_i32, c_i32, ctypes.POINTER(c_i32)]),
    "attn_bwd_tile_schedule_split": (None, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                            ctypes.POINTER(c_i32)]),
    "attn_bwd_preprocess": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_i64, c_i64, c_i64, c_i64, c_i64,
                                    c_i64, c_i32, c_vp, c_sz, c_vp]),
    "attn_bwd_gqa": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp,
                             Strides, c_i64, c_i64, c_i64, c_i64, c_i64, c_i32, c_f32, ctypes.POINTER(Mask), c_vp,
                             Strides, c_vp, Strides, c_vp, Strides, c_vp, c_sz, c_vp]),
    "attn_bwd": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides,
                         c_i64, c_i64, c_i64, c_i64, c_i32, c_f32, ctypes.POINTER(Mask), c_vp, Strides, c_vp, Strides,
                         c_vp, Strides, c_vp, c_sz, c_vp]),
    "attn_bwd_gqa_main": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_i64, c_i64, c_i64,
                                  c_i64, c_i64, c_i32, c_f32, ctypes.POINTER(Mask), c_vp, Strides, c_vp, Strides, c_vp,
                                  c_sz, c_vp]),
    "attn_bwd_dq_land": (c_i32, [c_vp, Strides, c_i64, c_i64, c_i64, c_i64, c_i32, c_f32, c_vp, c_sz, c_vp]),
    "attn_bwd_sparse": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp,
                                Strides, c_i64, c_i64, c_i64, c_i64, c_i64, c_i64, c_i64, c_i64, c_i32, c_f32, c_vp,
                                Strides, c_vp, Strides, c_vp, c_sz, c_vp]),
    "attn_bwd_sparse_main": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_i64, c_i64, c_i64,
                                     c_i64, c_i64, c_i64, c_i64, c_i64, c_i32, c_f32, c_vp, Strides, c_vp, c_sz,
                                     c_vp]),
    "attn_bwd_sparse_land": (c_i32, [c_vp, Strides, c_i64, c_i64, c_i64, c_i64, c_i64, c_i64, c_i32, c_vp, c_sz,
                                     c_vp]),
    "attn_bwd_check_error": (c_i32, [c_vp, c_vp, ctypes.POINTER(c_i32)]),
    "attn_bwd_status_string": (ctypes.c_char_p, [c_i32]),
    "attn_bwd_query_block_range": (None, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_i32),
                                          ctypes.POINTER(c_i32)]),
    "attn_fwd_gqa": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_i64, c_i64, c_i64, c_i64, c_i64, c_i32,
                             c_f32, ctypes.POINTER(Mask), c_vp, Strides, c_vp, Strides, c_vp, c_sz, c_vp]),
    "attn_bwd_query_block_range_qk": (None, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_i32),
                                             ctypes.POINTER(c_i32)]),
    "attn_bwd_tile_schedule": (None, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_i32), c_i32,
                                      ctypes.POINTER(c_i32)]),
    "attn_bwd_selftest_timeout": (c_i32, [c_vp, c_sz, c_i32, c_vp]),
    "attn_bwd_gqa_noalloc": (c_i32, [c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp, Strides,
                                     c_vp, Strides, c_i64, c_i64, c_i64, c_i64, c_i64, c_i32, c_f32,
                                     ctypes.POINTER(Mask), c_vp, Strides, c_vp, Strides, c_vp, Strides, c_vp]),
    "attn_bwd_noalloc_check_error": (c_i32, [c_vp, ctypes.POINTER(c_i32)]),
    "attn_bwd_host_scratch_size": (c_sz, [c_i64, c_i64, c_i64, c_i64, c_i64, c_i64]),
    "attn_bwd_gqa_host": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_i64, c_i32, c_f32,
                                  ctypes.POINTER(Mask), c_vp, c_vp, c_vp, c_vp, c_sz, c_i64, c_vp, c_vp, c_vp]),
}

_lib: Optional[ctypes.CDLL] = None


def library() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise AttnBwdError(f"CUDA library missing at {LIB_PATH}: build it with attention_backward_gb300.build")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _status(code: int, what: str) -> None:
    if code != 0:
        msg = library().attn_bwd_status_string(code).decode()
        raise AttnBwdError(f"{what}: {msg} (status {code})")


def _dev(*ts: torch.Tensor) -> None:
    for t in ts:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise AttnBwdError("attention backward tensors must be CUDA tensors")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return DT_F16
    if t.dtype == torch.bfloat16:
        return DT_BF16
    raise AttnBwdError(f"unsupported dtype {t.dtype}: fp16 or bf16")


def _bshd(t: torch.Tensor) -> Strides:
    if t.dim() != 4 or t.stride(3) != 1:
        raise AttnBwdError("expected a BSHD tensor with a contiguous head dimension")
    return Strides(t.stride(0), t.stride(1), t.stride(2))


def _lse_strides(lse: torch.Tensor) -> Strides:
    if lse.dim() != 3 or lse.dtype != torch.float32:
        raise AttnBwdError("lse must be float32 [B, H, S]")
    return Strides(lse.stride(0), lse.stride(2), lse.stride(1))


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _mask(causal: bool, window: int, cu_seqlens: Optional[torch.Tensor], S: int = 0, Sk: int = 0) -> Mask:
    """The C mask; ``kv_len`` is set when the key length Sk differs from the
    query length S (masks then aligned at the end of each row)."""
    m = Mask(1 if causal else 0, int(window), None, 0, int(Sk) if Sk != S else 0)
    if cu_seqlens is not None:
        _dev(cu_seqlens)
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
            raise AttnBwdError("cu_seqlens must be a contiguous int32 vector")
        m.cu_seqlens = cu_seqlens.data_ptr()
        m.num_seqs = cu_seqlens.numel() - 1
    return m


def workspace_size(B: int, S: int, H: int, Dq: int, dkv_elems: int = 0) -> int:
    return int(library().attn_bwd_workspace_size(B, S, H, Dq, dkv_elems))


def new_workspace(B: int, S: int, H: int, Dq: int, dkv_elems: int = 0, device=None) -> torch.Tensor:
    n = workspace_size(B, S, H, Dq, dkv_elems)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def sink_grad(sink, workspace, B: int, S: int, cu_seqlens=None, stream=None):
    """dsink [HQ] f32 of per-head attention-sink logits ``sink`` (f32 [HQ],
    CUDA) from the LSE2 and delta that a dense backward call (with sink-aware
    O and LSE) left in ``workspace`` (see attn_bwd_sink_grad)."""
    _dev(sink, workspace)
    if sink.dtype != torch.float32 or sink.dim() != 1 or not sink.is_contiguous():
        raise AttnBwdError("sink must be a contiguous float32 vector")
    HQ = sink.numel()
    dsink = torch.empty_like(sink)
    m = _mask(False, -1, cu_seqlens, S, S)
    _status(library().attn_bwd_sink_grad(sink.data_ptr(), B, S, HQ, ctypes.byref(m), workspace.data_ptr(),
                                         workspace.numel(), dsink.data_ptr(), _stream(stream)), "attn_bwd_sink_grad")
    return dsink


def gqa_workspace_size(B: int, S: int, HQ: int, D: int) -> int:
    """Workspace bytes with room for the one-call dense path's last-round split."""
    return int(library().attn_bwd_gqa_workspace_size(B, S, HQ, D))


def new_gqa_workspace(B: int, S: int, HQ: int, D: int, device=None) -> torch.Tensor:
    return torch.empty(gqa_workspace_size(B, S, HQ, D), dtype=torch.uint8, device=device or "cuda")


def tail_plan(tiles: int, ctas: int, G: int) -> tuple:
    """(first split draw, split tiles, query heads per unit); zeros: no split."""
    out = (c_i32 * 3)()
    library().attn_bwd_tail_plan(tiles, ctas, G, out)
    return tuple(out)


def tile_schedule_split(t: int, B: int, S: int, HKV: int, G: int, tail_start: int, tail_tiles: int,
                        tail_hpu: int) -> tuple:
    """Draw t of an unmasked dense batch with a last-round split: the seven
    values of tile_schedule, then (first head, heads, partials slot)."""
    out = (c_i32 * 10)()
    library().attn_bwd_tile_schedule_split(t, B, S, HKV, G, tail_start, tail_tiles, tail_hpu, out)
    return tuple(out)


def preprocess(o, do, lse, workspace, Dq: Optional[int] = None, dkv_elems: int = 0, stream=None) -> None:
    """Launch 1: delta, LSE*log2(e), zeroed accumulators (see attn_bwd_preprocess)."""
    _dev(o, do, lse, workspace)
    B, S, H, Dv = o.shape
    Dq = Dv if Dq is None else Dq
    _status(library().attn_bwd_preprocess(o.data_ptr(), _bshd(o), do.data_ptr(), _bshd(do), lse.data_ptr(),
                                          _lse_strides(lse), B, S, H, Dv, Dq, dkv_elems, _dt(o),
                                          workspace.data_ptr(), workspace.numel(), _stream(stream)),
            "attn_bwd_preprocess")


def gqa_main(q, k, v, do, dk, dv, workspace, sm_scale: float, causal: bool = False, window: int = -1,
             cu_seqlens=None, stream=None) -> None:
    """Split form, launch 2: dK, dV written, dQ accumulated in the workspace
    (see attn_bwd_gqa_main)."""
    _dev(q, k, v, do, dk, dv, workspace)
    B, S, HQ, D = q.shape
    HKV = k.shape[2]
    m = _mask(causal, window, cu_seqlens, S, k.shape[1])
    _status(library().attn_bwd_gqa_main(q.data_ptr(), _bshd(q), k.data_ptr(), _bshd(k), v.data_ptr(), _bshd(v),
                                        do.data_ptr(), _bshd(do), B, S, HQ, HKV, D, _dt(q), float(sm_scale),
                                        ctypes.byref(m), dk.data_ptr(), _bshd(dk), dv.data_ptr(), _bshd(dv),
                                        workspace.data_ptr(), workspace.numel(), _stream(stream)),
            "attn_bwd_gqa_main")


def dq_land(dq, workspace, sm_scale: float, stream=None) -> None:
    """Split form, launch 3: dQ = cast(sm_scale * dQacc)."""
    _dev(dq, workspace)
    B, S, H, D = dq.shape
    _status(library().attn_bwd_dq_land(dq.data_ptr(), _bshd(dq), B, S, H, D, _dt(dq), float(sm_scale),
                                       workspace.data_ptr(), workspace.numel(), _stream(stream)),
            "attn_bwd_dq_land")


def attn_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, workspace, sm_scale: float, causal: bool = False,
                 window: int = -1, cu_seqlens=None, stream=None) -> None:
    """The whole dense backward in one call into caller-owned dq, dk, dv (see
    attn_bwd_gqa): preprocess, main kernel and dQ landing on ``stream``."""
    _dev(q, k, v, o, do, lse, dq, dk, dv, workspace)
    B, S, HQ, D = q.shape
    HKV = k.shape[2]
    m = _mask(causal, window, cu_seqlens, S, k.shape[1])
    _status(library().attn_bwd_gqa(q.data_ptr(), _bshd(q), k.data_ptr(), _bshd(k), v.data_ptr(), _bshd(v),
                                   o.data_ptr(), _bshd(o), do.data_ptr(), _bshd(do), lse.data_ptr(),
                                   _lse_strides(lse), B, S, HQ, HKV, D, _dt(q), float(sm_scale), ctypes.byref(m),
                                   dq.data_ptr(), _bshd(dq), dk.data_ptr(), _bshd(dk), dv.data_ptr(), _bshd(dv),
                                   workspace.data_ptr(), workspace.numel(), _stream(stream)), "attn_bwd_gqa")


def attn_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, sm_scale: float, causal: bool = False, window: int = -1,
             cu_seqlens=None, stream=None) -> None:
    """attn_bwd_gqa for multi-head attention (HQ == HKV), through the C entry
    point attn_bwd."""
    _dev(q, k, v, o, do, lse, dq, dk, dv, workspace)
    B, S, H, D = q.shape
    m = _mask(causal, window, cu_seqlens, S, k.shape[1])
    _status(library().attn_bwd(q.data_ptr(), _bshd(q), k.data_ptr(), _bshd(k), v.data_ptr(), _bshd(v),
                               o.data_ptr(), _bshd(o), do.data_ptr(), _bshd(do), lse.data_ptr(), _lse_strides(lse),
                               B, S, H, D, _dt(q), float(sm_scale), ctypes.byref(m), dq.data_ptr(), _bshd(dq),
                               dk.data_ptr(), _bshd(dk), dv.data_ptr(), _bshd(dv), workspace.data_ptr(),
                               workspace.numel(), _stream(stream)), "attn_bwd")


def attn_fwd_gqa(q, k, v, o, lse, workspace, sm_scale: float, causal: bool = False, window: int = -1,
                 cu_seqlens=None, stream=None) -> None:
    """The forward into caller-owned o (16-bit [B,S,HQ,D]) and lse (f32
    [B,HQ,S]) (see attn_fwd_gqa)."""
    _dev(q, k, v, o, lse, workspace)
    B, S, HQ, D = q.shape
    HKV = k.shape[2]
    m = _mask(causal, window, cu_seqlens, S, k.shape[1])
    _status(library().attn_fwd_gqa(q.data_ptr(), _bshd(q), k.data_ptr(), _bshd(k), v.data_ptr(), _bshd(v), B, S,
                                   HQ, HKV, D, _dt(q), float(sm_scale), ctypes.byref(m), o.data_ptr(), _bshd(o),
                                   lse.data_ptr(), _lse_strides(lse), workspace.data_ptr(), workspace.numel(),
                                   _stream(stream)), "attn_fwd_gqa")


def forward(q, k, v, sm_scale: Optional[float] = None, causal: bool = False, window: int = -1, cu_seqlens=None,
            workspace=None, stream=None):
    """O and the natural-log LSE [B,HQ,S] of softmax attention (new tensors)."""
    _dev(q, k, v)
    B, S, HQ, D = q.shape
    if sm_scale is None:
        sm_scale = D ** -0.5
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty(B, HQ, S, dtype=torch.float32, device=q.device)
    attn_fwd_gqa(q, k, v, o, lse, workspace, sm_scale, causal, window, cu_seqlens, stream)
    return o, lse


def _idx_strides(idx) -> Strides:
    if idx.dtype != torch.int32 or idx.dim() != 4 or idx.stride(3) != 1:
        raise AttnBwdError("idx must be int32 [B, S, HKV, topk] with unit slot stride")
    return Strides(idx.stride(0), idx.stride(1), idx.stride(2))


def sparse_main(q, kv, do, idx, dq, workspace, sm_scale: float, dv_dim: int, stream=None) -> None:
    """Split form, launch 2 of the top-k sparse path: writes dQ, accumulates
    dKV (see attn_bwd_sparse_main)."""
    _dev(q, kv, do, idx, dq, workspace)
    B, S, H, DQK = q.shape
    SKV, HKV = kv.shape[1], kv.shape[2]
    sidx = _idx_strides(idx)
    _status(library().attn_bwd_sparse_main(q.data_ptr(), _bshd(q), kv.data_ptr(), _bshd(kv), do.data_ptr(),
                                           _bshd(do), idx.data_ptr(), sidx, B, S, SKV, H, HKV, DQK, dv_dim,
                                           idx.shape[3], _dt(q), float(sm_scale), dq.data_ptr(), _bshd(dq),
                                           workspace.data_ptr(), workspace.numel(), _stream(stream)),
            "attn_bwd_sparse_main")


def sparse_land(dkv, workspace, B: int, S: int, H: int, stream=None) -> None:
    """Split form, launch 3 of the sparse path: dKV cast from its accumulator."""
    _dev(dkv, workspace)
    _, SKV, HKV, DQK = dkv.shape
    _status(library().attn_bwd_sparse_land(dkv.data_ptr(), _bshd(dkv), B, S, SKV, H, HKV, DQK, _dt(dkv),
                                           workspace.data_ptr(), workspace.numel(), _stream(stream)),
            "attn_bwd_sparse_land")


def attn_bwd_sparse(q, kv, o, do, lse, idx, dq, dkv, workspace, sm_scale: float, dv_dim: int,
                    stream=None) -> None:
    """The whole top-k sparse backward in one call into caller-owned dq, dkv
    (see attn_bwd_sparse)."""
    _dev(q, kv, o, do, lse, idx, dq, dkv, workspace)
    B, S, H, DQK = q.shape
    SKV, HKV = kv.shape[1], kv.shape[2]
    sidx = _idx_strides(idx)
    _status(library().attn_bwd_sparse(q.data_ptr(), _bshd(q), kv.data_ptr(), _bshd(kv), o.data_ptr(), _bshd(o),
                                      do.data_ptr(), _bshd(do), lse.data_ptr(), _lse_strides(lse), idx.data_ptr(),
                                      sidx, B, S, SKV, H, HKV, DQK, dv_dim, idx.shape[3], _dt(q), float(sm_scale),
                                      dq.data_ptr(), _bshd(dq), dkv.data_ptr(), _bshd(dkv), workspace.data_ptr(),
                                      workspace.numel(), _stream(stream)), "attn_bwd_sparse")


def check_error(workspace, stream=None) -> int:
    """Synchronises the stream; raises if a kernel recorded a device error."""
    code = c_i32(0)
    st = library().attn_bwd_check_error(workspace.data_ptr(), _stream(stream), ctypes.byref(code))
    if st != 0:
        msg = library().attn_bwd_status_string(st).decode()
        raise AttnBwdError(f"device error: {msg} (site 0x{code.value:x})")
    return 0


def selftest_timeout(workspace, timeout_us: int = 20000, stream=None) -> tuple:
    """Runs the bounded-wait self-test; returns (status, status string)."""
    st = library().attn_bwd_selftest_timeout(workspace.data_ptr(), workspace.numel(), int(timeout_us),
                                             _stream(stream))
    return st, library().attn_bwd_status_string(st).decode()


def query_block_range(k0: int, block_k: int, length: int, causal: bool, window: int, block_q: int) -> tuple:
    lo, hi = c_i32(0), c_i32(0)
    library().attn_bwd_query_block_range(k0, block_k, length, int(causal), int(window), block_q, ctypes.byref(lo),
                                         ctypes.byref(hi))
    return lo.value, hi.value


def query_block_range_qk(k0: int, block_k: int, kv_len: int, q_len: int, causal: bool, window: int,
                         block_q: int) -> tuple:
    lo, hi = c_i32(0), c_i32(0)
    library().attn_bwd_query_block_range_qk(k0, block_k, kv_len, q_len, int(causal), int(window), block_q,
                                            ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def tile_schedule(t: int, B: int, S: int, HKV: int, causal: bool, window: int, cu_seqlens=None) -> tuple:
    """The dense kernels' t-th tile draw: (valid, b, kv head, sequence start,
    first key, first query block, number of query blocks)."""
    out = (c_i32 * 7)()
    cu = None
    n = 0
    if cu_seqlens is not None:
        n = len(cu_seqlens) - 1
        cu = (c_i32 * len(cu_seqlens))(*[int(x) for x in cu_seqlens])
    library().attn_bwd_tile_schedule(t, B, S, HKV, int(causal), int(window), cu, n, out)
    return tuple(out)


def backward(q, k, v, o, do, lse, sm_scale: Optional[float] = None, causal: bool = False, window: int = -1,
             cu_seqlens=None, workspace=None, stream=None):
    """dQ, dK, dV of softmax attention through the one-call entry point.

    q, o, do: [B,S,HQ,D]; k, v: [B,Sk,HKV,D] (fp16/bf16, CUDA; Sk may differ
    from S in a dense batch, the masks then aligned at the end of each row);
    lse: f32 [B,HQ,S] (natural log).  Outputs are new tensors in the input
    dtype.
    """
    _dev(q, k, v, o, do, lse)
    B, S, HQ, D = q.shape
    if sm_scale is None:
        sm_scale = D ** -0.5
    if workspace is None:
        workspace = new_gqa_workspace(B, S, HQ, D, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    attn_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, workspace, sm_scale, causal, window, cu_seqlens, stream)
    return dq, dk, dv


def sparse_backward(q, kv, o, do, lse, idx, sm_scale: Optional[float] = None, dv_dim: Optional[int] = None,
                    workspace=None, stream=None):
    """dQ and dKV of top-k sparse attention over shared latent rows through
    the one-call entry point."""
    _dev(q, kv, o, do, lse, idx)
    B, S, H, DQK = q.shape
    SKV, HKV = kv.shape[1], kv.shape[2]
    dv_dim = do.shape[3] if dv_dim is None else dv_dim
    if sm_scale is None:
        sm_scale = DQK ** -0.5
    dkv_elems = B * SKV * HKV * DQK
    if workspace is None:
        workspace = new_workspace(B, S, H, 0, dkv_elems, device=q.device)
    dq = torch.empty_like(q)
    dkv = torch.empty_like(kv)
    attn_bwd_sparse(q, kv, o, do, lse, idx, dq, dkv, workspace, sm_scale, dv_dim, stream)
    return dq, dkv


def noalloc_check_error(stream=None) -> int:
    """Synchronises the stream; raises if a kernel recorded a device error in
    the no-allocation entry point's library-held workspace."""
    code = c_i32(0)
    st = library().attn_bwd_noalloc_check_error(_stream(stream), ctypes.byref(code))
    if st != 0:
        msg = library().attn_bwd_status_string(st).decode()
        raise AttnBwdError(f"device error: {msg} (site 0x{code.value:x})")
    return 0


def backward_noalloc(q, k, v, o, do, lse, sm_scale: Optional[float] = None, causal: bool = False, window: int = -1,
                     cu_seqlens=None, stream=None, check: bool = True):
    """dQ, dK, dV through attn_bwd_gqa_noalloc: the library's own device
    workspace instead of a caller-provided one (for callers that cannot
    allocate device memory).  Calls on one device must not overlap on the GPU.
    The output tensors here are allocated by torch for convenience; a caller
    without an allocator passes its own buffers to the C entry point.  With
    ``check`` the call synchronises and raises on an error the kernels
    recorded."""
    _dev(q, k, v, o, do, lse)
    B, S, HQ, D = q.shape
    HKV = k.shape[2]
    if sm_scale is None:
        sm_scale = D ** -0.5
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    m = _mask(causal, window, cu_seqlens, S, k.shape[1])
    _status(library().attn_bwd_gqa_noalloc(q.data_ptr(), _bshd(q), k.data_ptr(), _bshd(k), v.data_ptr(), _bshd(v),
                                           o.data_ptr(), _bshd(o), do.data_ptr(), _bshd(do), lse.data_ptr(),
                                           _lse_strides(lse), B, S, HQ, HKV, D, _dt(q), float(sm_scale),
                                           ctypes.byref(m), dq.data_ptr(), _bshd(dq), dk.data_ptr(), _bshd(dk),
                                           dv.data_ptr(), _bshd(dv), _stream(stream)), "attn_bwd_gqa_noalloc")
    if check:
        noalloc_check_error(stream)
    return dq, dk, dv


def host_scratch_size(B: int, S: int, HQ: int, HKV: int, D: int, chunks: int) -> int:
    """Device scratch bytes of attn_bwd_gqa_host."""
    return int(library().attn_bwd_host_scratch_size(B, S, HQ, HKV, D, chunks))


def backward_host(q, k, v, o, do, lse, sm_scale: Optional[float] = None, causal: bool = False, window: int = -1,
                  cu_seqlens=None, chunks: int = 4, out=None, scratch=None, streams=None, device=None,
                  sync: bool = True):
    """dQ, dK, dV from host tensors to host tensors through attn_bwd_gqa_host,
    the copies overlapped with the kernels chunk by chunk.

    q, k, v, o, do, lse: contiguous CPU tensors (page-locked for overlap);
    cu_seqlens: a CUDA int32 tensor or None.  ``out`` (dq, dk, dv), ``scratch``
    (a CUDA uint8 tensor) and ``streams`` (compute, copy-in, copy-out) may be
    passed to reuse them across calls.  Returns after the work completes, or,
    with ``sync=False``, once it is queued (``streams[0]`` then covers it)."""
    for t in (q, k, v, o, do, lse):
        if t.is_cuda or not t.is_contiguous():
            raise AttnBwdError("backward_host takes contiguous host tensors")
    B, S, HQ, D = q.shape
    HKV = k.shape[2]
    if sm_scale is None:
        sm_scale = D ** -0.5
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if out is None:
        out = tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q, k, v))
    need = host_scratch_size(B, S, HQ, HKV, D, chunks)
    if need == 0:
        raise AttnBwdError("attn_bwd_gqa_host: unsupported shape")
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=device)
    if streams is None:
        streams = (torch.cuda.current_stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device))
    m = _mask(causal, window, cu_seqlens, S, k.shape[1])
    dq, dk, dv = out
    _status(library().attn_bwd_gqa_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                        lse.data_ptr(), B, S, HQ, HKV, D, _dt(q), float(sm_scale), ctypes.byref(m),
                                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), scratch.data_ptr(),
                                        scratch.numel(), int(chunks), _stream(streams[0]), _stream(streams[1]),
                                        _stream(streams[2])), "attn_bwd_gqa_host")
    if sync:
        streams[0].synchronize()
    return dq, dk, dv
