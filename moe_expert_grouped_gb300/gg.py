"""ctypes binding of libgg.so (the C ABI in include/gg.h).

Argument marshalling only: every step of the expert path runs in the CUDA
kernels of libgg.so. torch tensors supply device pointers and the current
stream; outputs that the caller does not pass are allocated with torch (memory
plumbing, no compute). If libgg.so is missing the import fails loudly; there
is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgg.so")

GG_OK = 0
GG_EPI_NONE, GG_EPI_SWIGLU, GG_EPI_SWIGLU_BWD, GG_EPI_QGEGLU, GG_EPI_QGEGLU_BWD = 0, 1, 2, 3, 4
GG_ACT_SWIGLU, GG_ACT_QGEGLU = 0, 1
GG_PROB_COMBINE, GG_PROB_ACTIVATION, GG_PROB_PRE_FC1 = 0, 1, 2
_GATED_FWD = (GG_EPI_SWIGLU, GG_EPI_QGEGLU)
_GATED_BWD = (GG_EPI_SWIGLU_BWD, GG_EPI_QGEGLU_BWD)
STATUS_NAMES = {
    0: "GG_OK", 1: "GG_ERR_INVALID_ARG", 2: "GG_ERR_UNSUPPORTED_SHAPE", 3: "GG_ERR_MISALIGNED",
    4: "GG_ERR_WORKSPACE_TOO_SMALL", 5: "GG_ERR_UNSUPPORTED_DEVICE", 6: "GG_ERR_CUDA",
    16: "GG_ERR_DEVICE_BAD_EXPERT_ID", 17: "GG_ERR_DEVICE_BAD_OFFSETS", 18: "GG_ERR_DEVICE_BAD_ROW",
    19: "GG_ERR_DEVICE_TIMEOUT",
}

# (name, restype, argtypes) of every exported symbol in include/gg.h
_P, _I, _Z, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
SIGNATURES = [
    ("gg_status_string", ctypes.c_char_p, [_I]),
    ("gg_version", ctypes.c_char_p, []),
    ("gg_launch_count", _U64, []),
    ("gg_workspace_size", _Z, [_I, _I, _I]),
    ("gg_clear_status", _I, [_P, _P]),
    ("gg_read_status", _I, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    ("gg_permute", _I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    ("gg_permute_rows", _I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _Z, _P]),
    ("gg_grouped_fwd", _I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    ("gg_swiglu", _I, [_P, _P, _I, _I, _I, _P, _P]),
    ("gg_glu", _I, [_P, _P, _I, _I, _I, _I, _P, _P, _P]),
    ("gg_grouped_dgrad", _I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    ("gg_rowdot_blocks", _I, [_I]),
    ("gg_rowdot_stride", _I, [_I]),
    ("gg_unpermute_combine", _I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _Z, _P]),
    ("gg_unpermute_combine_dot", _I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    ("gg_ep_split_ids", _I, [_P, _I, _I, _I, _P, _P, _P, _Z, _P]),
    ("gg_gather_rows32", _I, [_P, _I, _I, _P, _I, _P, _P, _Z, _P]),
    ("gg_moe_buffers_size", _Z, [_I, _I, _I, _I, _I, _I]),
    ("gg_moe_buffers_bind", _I, [_P, _Z, _I, _I, _I, _I, _I, _I, _P]),
    ("gg_moe_mlp_fwd", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    ("gg_moe_mlp_bwd", _I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    ("gg_moe_mlp_fwd_ex", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    ("gg_moe_mlp_bwd_ex", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    ("gg_selftest_bounded_wait", _I, [_P, _Z, _U64, _P]),
    ("gg_permute_noalloc", _I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    ("gg_grouped_fwd_gather", _I,
     [_P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    ("gg_grouped_dgrad_gather", _I,
     [_P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    ("gg_mx_row_tiles", _I, [_I, _I, _I, _I]),
    ("gg_mx_weights_layout_of", _I, [_I, _I, _I, _P]),
    ("gg_mx_prepare_weights", _I, [_P, _P, _I, _I, _I, _P, _Z, _P]),
    ("gg_mx_quantize_rows", _I,
     [_P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    ("gg_mx_rowdot_blocks", _I, [_I]),
    ("gg_mx_rowdot_stride", _I, [_I]),
    ("gg_mx_grouped_gemm", _I,
     [_I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    ("gg_mx_buffers_size", _Z, [_I, _I, _I, _I, _I, _I]),
    ("gg_mx_buffers_bind", _I, [_P, _Z, _I, _I, _I, _I, _I, _I, _P]),
    ("gg_moe_mlp_fwd_mx", _I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    ("gg_moe_mlp_bwd_mx", _I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
]

GG_MX_FC1, GG_MX_FC2, GG_MX_DGRAD_FC2, GG_MX_DGRAD_FC1 = 0, 1, 2, 3


class GGBuffers(ctypes.Structure):
    """Mirror of struct gg_moe_buffers."""

    _fields_ = [(n, ctypes.c_void_p) for n in (
        "Xp", "H1", "A", "Yp", "dYp", "dH", "dXp", "offsets", "row_of_slot", "slot_of_row",
        "prob_of_row", "rowdot", "ws")] + [("ws_bytes", ctypes.c_size_t)]


class GGOptions(ctypes.Structure):
    """Mirror of struct gg_moe_options."""

    _fields_ = [("activation", ctypes.c_int), ("prob_mode", ctypes.c_int),
                ("recompute_h1", ctypes.c_int)]


class GGMxWeightsLayout(ctypes.Structure):
    """Mirror of struct gg_mx_weights_layout (byte offsets)."""

    _fields_ = [(n, ctypes.c_size_t) for n in (
        "w1", "w1_scales", "w2", "w2_scales", "w2t", "w2t_scales", "w1t", "w1t_scales", "bytes")]


class GGMxBuffers(ctypes.Structure):
    """Mirror of struct gg_mx_buffers."""

    _fields_ = [(n, ctypes.c_void_p) for n in (
        "Xq", "Xs", "H1", "Aq", "As", "Yp", "dYq", "dYs", "dHq", "dHs", "dXp", "offsets",
        "row_of_slot", "slot_of_row", "prob_of_row", "tiles_before", "rowdot")] + [
        ("n_tiles", ctypes.c_int), ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


class GGError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m moe_expert_grouped_gb300.build` "
            "(the expert path has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def _check(code: int, where: str) -> None:
    if code != GG_OK:
        raise GGError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, dtype: torch.dtype, shape, name: str) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def launch_count() -> int:
    return int(LIB.gg_launch_count())


def version() -> str:
    return LIB.gg_version().decode()


def status_string(code: int) -> str:
    return LIB.gg_status_string(int(code)).decode()


def workspace(T: int, k: int, E: int, device) -> torch.Tensor:
    """A zeroed workspace (status word first) for calls on a batch of T tokens."""
    n = int(LIB.gg_workspace_size(T, k, E))
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def read_status(ws: torch.Tensor) -> int:
    v = ctypes.c_int32(0)
    _check(LIB.gg_read_status(_ptr(ws), _stream(ws.device), ctypes.byref(v)), "gg_read_status")
    return int(v.value)


def clear_status(ws: torch.Tensor) -> None:
    _check(LIB.gg_clear_status(_ptr(ws), _stream(ws.device)), "gg_clear_status")


def r_cap(T: int, k: int, E: int, P: int) -> int:
    return T * k + E * (P - 1)


def permute(x, idx, prob, E: int, P: int = 1, ws=None, out=None):
    """gg_permute: returns dict(Xp, offsets, row_of_slot, slot_of_row, prob_of_row, ws)."""
    T, H = x.shape
    k = idx.shape[1]
    dev = x.device
    rc = r_cap(T, k, E, P)
    _need(x, torch.bfloat16, (T, H), "x")
    _need(idx, torch.int32, (T, k), "idx")
    _need(prob, torch.float32, (T, k), "prob")
    o = out or {}

    def buf(name, shape, dtype):
        t = o.get(name)
        return torch.empty(shape, dtype=dtype, device=dev) if t is None else t

    Xp = None if "Xp" in o and o["Xp"] is None else buf("Xp", (rc, H), torch.bfloat16)
    offsets = buf("offsets", (E + 1,), torch.int32)
    ros = buf("row_of_slot", (T * k,), torch.int32)
    sor = buf("slot_of_row", (rc,), torch.int32)
    por = buf("prob_of_row", (rc,), torch.float32)
    ws = workspace(T, k, E, dev) if ws is None else ws
    _check(LIB.gg_permute(_ptr(x), _ptr(idx), _ptr(prob), T, H, k, E, P, _ptr(Xp), _ptr(offsets),
                          _ptr(ros), _ptr(sor), _ptr(por), _ptr(ws), ws.numel(), _stream(dev)),
           "gg_permute")
    return dict(Xp=Xp, offsets=offsets, row_of_slot=ros, slot_of_row=sor, prob_of_row=por, ws=ws)


def permute_rows(src, row_of_slot, slot_of_row, offsets, k: int, E: int, P: int, R_cap: int, ws,
                 dst=None, prob=None):
    """gg_permute_rows: dst[row_of_slot[t*k+j]] = src[t] (times prob[t, j] when given;
    0 on padding rows)."""
    T, H = src.shape
    dst = torch.empty((R_cap, H), dtype=torch.bfloat16, device=src.device) if dst is None else dst
    _check(LIB.gg_permute_rows(_ptr(src), _ptr(row_of_slot), _ptr(slot_of_row), _ptr(offsets), T,
                               H, k, E, P, R_cap, _ptr(prob), _ptr(dst), _ptr(ws), ws.numel(),
                               _stream(src.device)),
           "gg_permute_rows")
    return dst


def grouped_fwd(A, B, offsets, epilogue: int = GG_EPI_NONE, ws=None, C=None, H1_save=None,
                prob_of_row=None):
    """gg_grouped_fwd. B is [E, N, K]; returns C ([R_cap, N] or, gated, [R_cap, N/2]);
    prob_of_row weights a gated activation."""
    R_cap, K = A.shape
    E, N, Kb = B.shape
    if Kb != K:
        raise ValueError("A and B disagree on K")
    dev = A.device
    ncols = N // 2 if epilogue in _GATED_FWD else N
    C = torch.empty((R_cap, ncols), dtype=torch.bfloat16, device=dev) if C is None else C
    ws = workspace(0, 1, E, dev) if ws is None else ws
    _check(LIB.gg_grouped_fwd(_ptr(A), _ptr(B), _ptr(offsets), E, R_cap, K, N, epilogue, _ptr(C),
                              _ptr(H1_save), _ptr(prob_of_row), _ptr(ws), ws.numel(),
                              _stream(dev)),
           "gg_grouped_fwd")
    return C


def grouped_fwd_gather(src, slot_of_row, k: int, B, offsets, epilogue: int = GG_EPI_NONE,
                       ws=None, C=None, H1_save=None, prob_of_row=None):
    """gg_grouped_fwd_gather: A rows gathered from token-major src [T, K]."""
    T, K = src.shape
    E, N, Kb = B.shape
    if Kb != K:
        raise ValueError("src and B disagree on K")
    R_cap = slot_of_row.shape[0]
    dev = src.device
    ncols = N // 2 if epilogue in _GATED_FWD else N
    C = torch.empty((R_cap, ncols), dtype=torch.bfloat16, device=dev) if C is None else C
    ws = workspace(0, 1, E, dev) if ws is None else ws
    _check(LIB.gg_grouped_fwd_gather(_ptr(src), T, _ptr(slot_of_row), k, _ptr(B), _ptr(offsets),
                                     E, R_cap, K, N, epilogue, _ptr(C), _ptr(H1_save),
                                     _ptr(prob_of_row), _ptr(ws), ws.numel(), _stream(dev)),
           "gg_grouped_fwd_gather")
    return C


def rowdot_blocks(F: int) -> int:
    """gg_rowdot_blocks: partial sums per row of the dprob epilogue output."""
    return int(LIB.gg_rowdot_blocks(int(F)))


def rowdot_stride(F: int) -> int:
    """gg_rowdot_stride: floats per row of the rowdot array [R_cap, stride]."""
    return int(LIB.gg_rowdot_stride(int(F)))


def grouped_dgrad_gather(src, slot_of_row, k: int, B, offsets, epilogue: int = GG_EPI_NONE,
                         H1=None, prob_of_row=None, ws=None, dA=None, rowdot=None):
    """gg_grouped_dgrad_gather: dC rows gathered from token-major src [T, N]."""
    T, N = src.shape
    E, Nb, K = B.shape
    if Nb != N:
        raise ValueError("src and B disagree on N")
    R_cap = slot_of_row.shape[0]
    dev = src.device
    ncols = 2 * K if epilogue in _GATED_BWD else K
    dA = torch.empty((R_cap, ncols), dtype=torch.bfloat16, device=dev) if dA is None else dA
    ws = workspace(0, 1, E, dev) if ws is None else ws
    _check(LIB.gg_grouped_dgrad_gather(_ptr(src), T, _ptr(slot_of_row), k, _ptr(B), _ptr(offsets),
                                       E, R_cap, K, N, epilogue, _ptr(H1), _ptr(prob_of_row),
                                       _ptr(dA), _ptr(rowdot), _ptr(ws), ws.numel(),
                                       _stream(dev)),
           "gg_grouped_dgrad_gather")
    return dA


def glu(H1, offsets, E: int, epilogue: int = GG_EPI_SWIGLU, prob_of_row=None, A=None):
    """gg_glu: the unfused gated activation (SwiGLU or QuickGeGLU), optionally weighted."""
    R_cap, F2 = H1.shape
    F = F2 // 2
    A = torch.empty((R_cap, F), dtype=torch.bfloat16, device=H1.device) if A is None else A
    _check(LIB.gg_glu(_ptr(H1), _ptr(offsets), E, R_cap, F, epilogue, _ptr(prob_of_row), _ptr(A),
                      _stream(H1.device)),
           "gg_glu")
    return A


def swiglu(H1, offsets, E: int, A=None):
    """gg_swiglu: A = silu(g) * u on a stored FC1 output."""
    R_cap, F2 = H1.shape
    F = F2 // 2
    A = torch.empty((R_cap, F), dtype=torch.bfloat16, device=H1.device) if A is None else A
    _check(LIB.gg_swiglu(_ptr(H1), _ptr(offsets), E, R_cap, F, _ptr(A), _stream(H1.device)),
           "gg_swiglu")
    return A


def grouped_dgrad(dC, B, offsets, epilogue: int = GG_EPI_NONE, H1=None, prob_of_row=None,
                  ws=None, dA=None, rowdot=None):
    """gg_grouped_dgrad. B is the forward weight [E, N, K]; dC is [R_cap, N]. With
    GG_EPI_SWIGLU_BWD, rowdot [R_cap, rowdot_stride(K)] fp32 receives the dprob
    partial sums (the first rowdot_blocks(K) of each row)."""
    R_cap, N = dC.shape
    E, Nb, K = B.shape
    if Nb != N:
        raise ValueError("dC and B disagree on N")
    dev = dC.device
    ncols = 2 * K if epilogue in _GATED_BWD else K
    dA = torch.empty((R_cap, ncols), dtype=torch.bfloat16, device=dev) if dA is None else dA
    ws = workspace(0, 1, E, dev) if ws is None else ws
    _check(LIB.gg_grouped_dgrad(_ptr(dC), _ptr(B), _ptr(offsets), E, R_cap, K, N, epilogue,
                                _ptr(H1), _ptr(prob_of_row), _ptr(dA), _ptr(rowdot), _ptr(ws),
                                ws.numel(), _stream(dev)),
           "gg_grouped_dgrad")
    return dA


def unpermute_combine(Yp, row_of_slot, prob, T: int, k: int, ws, out=None, rowdot=None,
                      dprob=None, n_rowdot=None, dot_src=None):
    """gg_unpermute_combine: probability-weighted (prob) or plain (None) sum of k rows;
    with rowdot [R_cap, stride] (and n_rowdot partials per row, default all but
    the padding of the last 8-group: pass n_rowdot when it differs) also
    dprob [T, k] = the sum of each pair's row partials."""
    R_cap, H = Yp.shape
    out = torch.empty((T, H), dtype=torch.bfloat16, device=Yp.device) if out is None else out
    if dot_src is not None and dprob is None:
        dprob = torch.empty((T, k), dtype=torch.float32, device=Yp.device)
    if rowdot is not None:
        if n_rowdot is None:
            raise ValueError("n_rowdot (rowdot_blocks(F)) is required with rowdot")
        if (n_rowdot + 7) // 8 * 8 != rowdot.shape[1]:
            raise ValueError("rowdot rows must hold n_rowdot rounded up to 8 floats")
        if dprob is None:
            dprob = torch.empty((T, k), dtype=torch.float32, device=Yp.device)
    _check(LIB.gg_unpermute_combine(_ptr(Yp), _ptr(row_of_slot), _ptr(prob), T, k, H, R_cap,
                                    _ptr(out), _ptr(rowdot), n_rowdot or 0, _ptr(dot_src),
                                    _ptr(dprob), _ptr(ws), ws.numel(), _stream(Yp.device)),
           "gg_unpermute_combine")
    return out if dprob is None else (out, dprob)


def unpermute_combine_dot(Sp, row_of_slot, prob, T: int, k: int, dot_src, dot_rows, ws,
                          out=None, dprob=None):
    """gg_unpermute_combine_dot: out [T, H] = the (probability-weighted when prob
    is given) sum of each token's k rows of Sp, and dprob [T, k] = <dot_src[t],
    dot_rows[row of (t, j)]>; returns (out, dprob)."""
    R_cap, H = Sp.shape
    out = torch.empty((T, H), dtype=torch.bfloat16, device=Sp.device) if out is None else out
    if dprob is None:
        dprob = torch.empty((T, k), dtype=torch.float32, device=Sp.device)
    _check(LIB.gg_unpermute_combine_dot(_ptr(Sp), _ptr(row_of_slot), _ptr(prob), T, k, H, R_cap,
                                        _ptr(out), _ptr(dot_src), _ptr(dot_rows), _ptr(dprob),
                                        _ptr(ws), ws.numel(), _stream(Sp.device)),
           "gg_unpermute_combine_dot")
    return out, dprob


def ep_split_ids(idx, El: int, n_ranks: int, ws, dest=None, local_eid=None):
    """gg_ep_split_ids: (dest, local_eid), each shaped like idx (int32): the rank
    owning each pair's expert and the expert's index on that rank."""
    _need(idx, torch.int32, tuple(idx.shape), "idx")
    if not idx.is_contiguous():
        raise ValueError("idx: contiguous tensor expected")
    n = idx.numel()
    dest = torch.empty_like(idx) if dest is None else dest
    local_eid = torch.empty_like(idx) if local_eid is None else local_eid
    _check(LIB.gg_ep_split_ids(_ptr(idx), n, El, n_ranks, _ptr(dest), _ptr(local_eid), _ptr(ws),
                               ws.numel(), _stream(idx.device)),
           "gg_ep_split_ids")
    return dest, local_eid


def gather_rows32(src, index, ws, out=None):
    """gg_gather_rows32: out[i] = src[index[i]] (zero where index is -1) for a
    1-D or 2-D int32 / float32 src; index int32 [n]."""
    if src.dtype not in (torch.int32, torch.float32) or not src.is_contiguous():
        raise ValueError("src: contiguous int32 or float32 expected")
    _need(index, torch.int32, (index.numel(),), "index")
    if not index.is_contiguous():
        raise ValueError("index: contiguous tensor expected")
    width = 1 if src.dim() == 1 else src.shape[1]
    n = index.numel()
    shape = (n,) if src.dim() == 1 else (n, width)
    out = torch.empty(shape, dtype=src.dtype, device=src.device) if out is None else out
    _check(LIB.gg_gather_rows32(_ptr(src), src.shape[0], width, _ptr(index), n, _ptr(out),
                                _ptr(ws), ws.numel(), _stream(src.device)),
           "gg_gather_rows32")
    return out


def selftest_bounded_wait(ws, limit_ns: int) -> None:
    _check(LIB.gg_selftest_bounded_wait(_ptr(ws), ws.numel(), int(limit_ns), _stream(ws.device)),
           "gg_selftest_bounded_wait")


class MoeLayer:
    """The whole expert layer (gg_moe_mlp_fwd / gg_moe_mlp_bwd) over one owned buffer.

    The buffer holds every intermediate (permuted rows, H1, A, Yp and their
    gradients, row maps, workspace); ``view(name)`` exposes each as a tensor.
    """

    _SHAPES = {
        "Xp": ("rc", "H"), "Yp": ("rc", "H"), "dYp": ("rc", "H"), "dXp": ("rc", "H"),
        "H1": ("rc", "2F"), "dH": ("rc", "2F"), "A": ("rc", "F"), "offsets": ("E1",),
        "row_of_slot": ("Tk",), "slot_of_row": ("rc",), "prob_of_row": ("rc",),
        "rowdot": ("rc", "nbs"), "ws": ("ws",),
    }

    def __init__(self, T: int, H: int, F: int, k: int, E: int, P: int = 1, device="cuda",
                 activation: int = GG_ACT_SWIGLU, prob_mode: int = GG_PROB_COMBINE,
                 recompute_h1: bool = False):
        self.T, self.H, self.F, self.k, self.E, self.P = T, H, F, k, E, P
        self.opt = GGOptions(activation, prob_mode, 1 if recompute_h1 else 0)
        self._saved = None  # the forward's (x, prob): the pre-FC1 backward needs them
        self._rows = None   # the forward's batch size
        self.R_cap = r_cap(T, k, E, P)
        self.device = torch.device(device)
        n = int(LIB.gg_moe_buffers_size(T, H, F, k, E, P))
        if n == 0:
            raise GGError(1, "gg_moe_buffers_size")
        self.storage = torch.zeros(n + 256, dtype=torch.uint8, device=self.device)
        base = self.storage.data_ptr()
        self._base = base + ((-base) % 256)
        self.buf = GGBuffers()
        _check(LIB.gg_moe_buffers_bind(ctypes.c_void_p(self._base), n, T, H, F, k, E, P,
                                       ctypes.byref(self.buf)), "gg_moe_buffers_bind")

    def view(self, name: str) -> torch.Tensor:
        """A torch view of one intermediate buffer of the struct."""
        dims = {"rc": self.R_cap, "H": self.H, "F": self.F, "2F": 2 * self.F, "E1": self.E + 1,
                "Tk": self.T * self.k, "ws": int(self.buf.ws_bytes),
                "nbs": rowdot_stride(self.F)}
        dtype = {"offsets": torch.int32, "row_of_slot": torch.int32, "slot_of_row": torch.int32,
                 "prob_of_row": torch.float32, "rowdot": torch.float32,
                 "ws": torch.uint8}.get(name, torch.bfloat16)
        shape = tuple(dims[d] for d in self._SHAPES[name])
        count = 1
        for s in shape:
            count *= s
        esize = torch.empty((), dtype=dtype).element_size()
        off = getattr(self.buf, name) - self.storage.data_ptr()
        return self.storage[off:off + count * esize].view(dtype).view(shape)

    def fits(self, T: int) -> bool:
        """Whether a batch of T tokens can run on this layer's buffer (T at
        most the bound size and its permute workspace no larger)."""
        return 0 <= T <= self.T and int(LIB.gg_workspace_size(T, self.k, self.E)) <= int(
            self.buf.ws_bytes)

    def forward(self, x, idx, prob, W1, W2, out=None):
        """out [T, H] for x [T, H]: T is the bound size or, for a buffer reused
        across batches, any smaller batch the buffer fits."""
        T = int(x.shape[0])
        H, F, k, E = self.H, self.F, self.k, self.E
        if not self.fits(T):
            raise GGError(4, f"{T} tokens do not fit a layer bound for {self.T}")
        _need(x, torch.bfloat16, (T, H), "x")
        _need(idx, torch.int32, (T, k), "idx")
        _need(prob, torch.float32, (T, k), "prob")
        _need(W1, torch.bfloat16, (E, 2 * F, H), "W1")
        _need(W2, torch.bfloat16, (E, H, F), "W2")
        out = torch.empty((T, H), dtype=torch.bfloat16, device=self.device) if out is None else out
        _check(LIB.gg_moe_mlp_fwd_ex(_ptr(x), _ptr(idx), _ptr(prob), _ptr(W1), _ptr(W2), T, H, F,
                                     k, E, self.P, ctypes.byref(self.opt), _ptr(out),
                                     ctypes.byref(self.buf), _stream(self.device)),
               "gg_moe_mlp_fwd_ex")
        self._saved = (x, prob)
        self._rows = T
        return out

    def backward(self, dOut, W1, W2, dX=None, dprob=None):
        """dX [T, H]; with dprob ([T, k] fp32 tensor, or True to allocate one) also
        the routing-probability gradient, returned as (dX, dprob). T is the
        last forward's batch."""
        T = self._rows if self._rows is not None else self.T
        H, F, k, E = self.H, self.F, self.k, self.E
        _need(dOut, torch.bfloat16, (T, H), "dOut")
        dX = torch.empty((T, H), dtype=torch.bfloat16, device=self.device) if dX is None else dX
        want = dprob is not None and dprob is not False
        if dprob is True:
            dprob = torch.empty((T, k), dtype=torch.float32, device=self.device)
        if want:
            _need(dprob, torch.float32, (T, k), "dprob")
        x, prob = self._saved if self._saved is not None else (None, None)
        _check(LIB.gg_moe_mlp_bwd_ex(_ptr(dOut), _ptr(x), _ptr(prob), _ptr(W1), _ptr(W2), T, H, F,
                                     k, E, self.P, ctypes.byref(self.opt), _ptr(dX),
                                     _ptr(dprob) if want else None, ctypes.byref(self.buf),
                                     _stream(self.device)),
               "gg_moe_mlp_bwd_ex")
        return (dX, dprob) if want else dX

    def status(self) -> int:
        return read_status(self.view("ws"))


def permute_noalloc(x, idx, prob, E: int, P: int = 1, out=None):
    """gg_permute_noalloc: the permute for callers that cannot allocate device
    memory; the library keeps its scratch in a fixed array of its own (batches
    with gg_workspace_size(T, k, E) > 256 KiB + 256 bytes are rejected). Only the outputs
    the caller does not pass are allocated here, by torch."""
    T, H = x.shape
    k = idx.shape[1]
    dev = x.device
    rc = r_cap(T, k, E, P)
    o = out or {}

    def buf(name, shape, dtype):
        t = o.get(name)
        return torch.empty(shape, dtype=dtype, device=dev) if t is None else t

    Xp = buf("Xp", (rc, H), torch.bfloat16)
    offsets = buf("offsets", (E + 1,), torch.int32)
    ros = buf("row_of_slot", (T * k,), torch.int32)
    sor = buf("slot_of_row", (rc,), torch.int32)
    por = buf("prob_of_row", (rc,), torch.float32)
    _check(LIB.gg_permute_noalloc(_ptr(x), _ptr(idx), _ptr(prob), T, H, k, E, P, _ptr(Xp),
                                  _ptr(offsets), _ptr(ros), _ptr(sor), _ptr(por), _stream(dev)),
           "gg_permute_noalloc")
    return dict(Xp=Xp, offsets=offsets, row_of_slot=ros, slot_of_row=sor, prob_of_row=por)


# ---------------------------------------------------------------- MXFP8 path

def mx_row_tiles(T: int, k: int, E: int, P: int = 1) -> int:
    return int(LIB.gg_mx_row_tiles(T, k, E, P))


def mx_rowdot_blocks(F: int) -> int:
    return int(LIB.gg_mx_rowdot_blocks(F))


def mx_rowdot_stride(F: int) -> int:
    return int(LIB.gg_mx_rowdot_stride(F))


def mx_weights_layout(E: int, H: int, F: int) -> dict:
    """gg_mx_weights_layout_of as a dict of byte offsets (and 'bytes')."""
    L = GGMxWeightsLayout()
    _check(LIB.gg_mx_weights_layout_of(E, H, F, ctypes.byref(L)), "gg_mx_weights_layout_of")
    return {n: int(getattr(L, n)) for n, _ in GGMxWeightsLayout._fields_}


def mx_prepare_weights(W1, W2):
    """gg_mx_prepare_weights: the four MXFP8 weight operands in one uint8
    device tensor (256-byte aligned start); returns (tensor, layout)."""
    E, F2, H = W1.shape
    F = F2 // 2
    _need(W1, torch.bfloat16, (E, 2 * F, H), "W1")
    _need(W2, torch.bfloat16, (E, H, F), "W2")
    L = mx_weights_layout(E, H, F)
    raw = torch.empty(L["bytes"] + 256, dtype=torch.uint8, device=W1.device)
    off = (-raw.data_ptr()) % 256
    mxw = raw[off:off + L["bytes"]]
    _check(LIB.gg_mx_prepare_weights(_ptr(W1), _ptr(W2), E, H, F, _ptr(mxw), L["bytes"],
                                     _stream(W1.device)), "gg_mx_prepare_weights")
    return mxw, L


def mx_quantize_rows(src, maps, k: int, E: int, P: int, ws, prob=None, n_tiles=None, out=None):
    """gg_mx_quantize_rows from the permute's maps (dict with row_of_slot,
    slot_of_row, offsets); prob [T, k] scales each pair's copy. Returns
    dict(Q [R_cap, K] uint8, S [n_tiles, K/128, 512] uint8, tiles_before [E+1])."""
    T, K = src.shape
    dev = src.device
    rc = r_cap(T, k, E, P)
    if n_tiles is None:
        n_tiles = (rc + 127) // 128 + E
    o = out or {}
    Q = o.get("Q")
    Q = torch.empty((rc, K), dtype=torch.uint8, device=dev) if Q is None else Q
    S = o.get("S")
    S = torch.empty((n_tiles, K // 128, 512), dtype=torch.uint8, device=dev) if S is None else S
    tb = o.get("tiles_before")
    tb = torch.empty((E + 1,), dtype=torch.int32, device=dev) if tb is None else tb
    _check(LIB.gg_mx_quantize_rows(_ptr(src), T, K, k, _ptr(maps["row_of_slot"]),
                                   _ptr(maps["slot_of_row"]), _ptr(maps["offsets"]), _ptr(prob),
                                   E, P, n_tiles, _ptr(tb), _ptr(Q), _ptr(S), _ptr(ws),
                                   ws.numel(), _stream(dev)), "gg_mx_quantize_rows")
    return dict(Q=Q, S=S, tiles_before=tb)


def mx_grouped_gemm(which: int, Aq, As, mxw, offsets, E: int, R_cap: int, H: int, F: int, ws,
                    activation: int = GG_ACT_SWIGLU, C=None, Cq=None, Cs=None, H1=None,
                    row_scale=None, rowdot=None):
    """gg_mx_grouped_gemm. Outputs the caller does not pass are allocated:
    FC1 -> (Cq [R_cap, F], Cs, H1 [R_cap, 2F]); FC2 / DGRAD_FC1 -> C [R_cap, H];
    DGRAD_FC2 -> (Cq [R_cap, 2F], Cs) (H1 is an input there)."""
    dev = Aq.device
    n_tiles = As.shape[0]
    if which == GG_MX_FC1:
        Cq = torch.empty((R_cap, F), dtype=torch.uint8, device=dev) if Cq is None else Cq
        Cs = torch.zeros((n_tiles, F // 128, 512), dtype=torch.uint8, device=dev) \
            if Cs is None else Cs
        H1 = torch.empty((R_cap, 2 * F), dtype=torch.bfloat16, device=dev) if H1 is None else H1
    elif which == GG_MX_DGRAD_FC2:
        Cq = torch.empty((R_cap, 2 * F), dtype=torch.uint8, device=dev) if Cq is None else Cq
        Cs = torch.zeros((n_tiles, 2 * F // 128, 512), dtype=torch.uint8, device=dev) \
            if Cs is None else Cs
    else:
        C = torch.empty((R_cap, H), dtype=torch.bfloat16, device=dev) if C is None else C
    _check(LIB.gg_mx_grouped_gemm(which, activation, _ptr(Aq), _ptr(As), _ptr(mxw),
                                  _ptr(offsets), E, R_cap, H, F, n_tiles, _ptr(C), _ptr(Cq),
                                  _ptr(Cs), _ptr(H1), _ptr(row_scale), _ptr(rowdot), _ptr(ws),
                                  ws.numel(), _stream(dev)), "gg_mx_grouped_gemm")
    if which == GG_MX_FC1:
        return Cq, Cs, H1
    if which == GG_MX_DGRAD_FC2:
        return Cq, Cs
    return C


class MxMoeLayer:
    """The MXFP8 expert layer (gg_moe_mlp_fwd_mx / gg_moe_mlp_bwd_mx) over one
    owned buffer, with weights prepared once by gg_mx_prepare_weights."""

    _SHAPES = {
        "Xq": ("rc", "H"), "dYq": ("rc", "H"), "Aq": ("rc", "F"), "dHq": ("rc", "2F"),
        "Xs": ("nt", "Hb", "512"), "dYs": ("nt", "Hb", "512"), "As": ("nt", "Fb", "512"),
        "dHs": ("nt", "F2b", "512"), "H1": ("rc", "2F"), "Yp": ("rc", "H"), "dXp": ("rc", "H"),
        "offsets": ("E1",), "tiles_before": ("E1",), "row_of_slot": ("Tk",),
        "slot_of_row": ("rc",), "prob_of_row": ("rc",), "rowdot": ("rc", "nbs"), "ws": ("ws",),
    }
    _DTYPES = {"H1": torch.bfloat16, "Yp": torch.bfloat16, "dXp": torch.bfloat16,
               "offsets": torch.int32, "tiles_before": torch.int32, "row_of_slot": torch.int32,
               "slot_of_row": torch.int32, "prob_of_row": torch.float32,
               "rowdot": torch.float32}

    def __init__(self, T: int, H: int, F: int, k: int, E: int, P: int = 1, device="cuda",
                 activation: int = GG_ACT_SWIGLU, prob_mode: int = GG_PROB_COMBINE):
        self.T, self.H, self.F, self.k, self.E, self.P = T, H, F, k, E, P
        self.opt = GGOptions(activation, prob_mode, 0)
        self._saved = None
        self.R_cap = r_cap(T, k, E, P)
        self.device = torch.device(device)
        n = int(LIB.gg_mx_buffers_size(T, H, F, k, E, P))
        if n == 0:
            raise GGError(2, "gg_mx_buffers_size")
        self.storage = torch.zeros(n + 256, dtype=torch.uint8, device=self.device)
        base = self.storage.data_ptr()
        self._base = base + ((-base) % 256)
        self.buf = GGMxBuffers()
        _check(LIB.gg_mx_buffers_bind(ctypes.c_void_p(self._base), n, T, H, F, k, E, P,
                                      ctypes.byref(self.buf)), "gg_mx_buffers_bind")

    def view(self, name: str) -> torch.Tensor:
        dims = {"rc": self.R_cap, "H": self.H, "F": self.F, "2F": 2 * self.F,
                "E1": self.E + 1, "Tk": self.T * self.k, "ws": int(self.buf.ws_bytes),
                "nbs": mx_rowdot_stride(self.F), "nt": int(self.buf.n_tiles),
                "Hb": self.H // 128, "Fb": self.F // 128, "F2b": 2 * self.F // 128, "512": 512}
        dtype = self._DTYPES.get(name, torch.uint8)
        shape = tuple(dims[d] for d in self._SHAPES[name])
        count = 1
        for s in shape:
            count *= s
        esize = torch.empty((), dtype=dtype).element_size()
        off = getattr(self.buf, name) - self.storage.data_ptr()
        return self.storage[off:off + count * esize].view(dtype).view(shape)

    def forward(self, x, idx, prob, mxw, out=None):
        T, H, F, k, E = self.T, self.H, self.F, self.k, self.E
        _need(x, torch.bfloat16, (T, H), "x")
        _need(idx, torch.int32, (T, k), "idx")
        _need(prob, torch.float32, (T, k), "prob")
        out = torch.empty((T, H), dtype=torch.bfloat16, device=self.device) if out is None else out
        _check(LIB.gg_moe_mlp_fwd_mx(_ptr(x), _ptr(idx), _ptr(prob), _ptr(mxw), T, H, F, k, E,
                                     self.P, ctypes.byref(self.opt), _ptr(out),
                                     ctypes.byref(self.buf), _stream(self.device)),
               "gg_moe_mlp_fwd_mx")
        self._saved = (x, prob)
        return out

    def backward(self, dOut, mxw, dX=None, dprob=None):
        T, H, F, k, E = self.T, self.H, self.F, self.k, self.E
        _need(dOut, torch.bfloat16, (T, H), "dOut")
        dX = torch.empty((T, H), dtype=torch.bfloat16, device=self.device) if dX is None else dX
        want = dprob is not None and dprob is not False
        if dprob is True:
            dprob = torch.empty((T, k), dtype=torch.float32, device=self.device)
        if want:
            _need(dprob, torch.float32, (T, k), "dprob")
        x, prob = self._saved if self._saved is not None else (None, None)
        _check(LIB.gg_moe_mlp_bwd_mx(_ptr(dOut), _ptr(x), _ptr(prob), _ptr(mxw), T, H, F, k, E,
                                     self.P, ctypes.byref(self.opt), _ptr(dX),
                                     _ptr(dprob) if want else None, ctypes.byref(self.buf),
                                     _stream(self.device)),
               "gg_moe_mlp_bwd_mx")
        return (dX, dprob) if want else dX

    def status(self) -> int:
        return read_status(self.view("ws"))
