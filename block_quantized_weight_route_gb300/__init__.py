"""Python binding of the block-quantised prefill GEMM / routed-MoE expert-stage
library (C ABI in include/qmm.h, CUDA kernels for sm_103a in csrc/).

Argument marshalling only: every step runs in the library's kernels, on the
current torch CUDA stream.  There is no CPU path; if the shared library is
missing or the device is not a GB300 the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB, build_library  # noqa: F401

QMM_WS_FIELDS = 19
WS_FIELD_NAMES = ("ids", "w", "counts", "offsets", "src", "row", "chunk_counts", "tiles", "tile_count",
                  "tiles256", "tile_count256", "X_perm", "Hq", "Hd", "Hs", "Hd32", "Yslot", "wrow", "total")
QMM_STAGE_SLOTS = 1

_STATUS = {0: "QMM_OK", 1: "QMM_ERR_INVALID_ARG", 2: "QMM_ERR_UNSUPPORTED_SHAPE",
           3: "QMM_ERR_UNSUPPORTED_DEVICE", 4: "QMM_ERR_WORKSPACE", 5: "QMM_ERR_CUDA", 6: "QMM_ERR_TIMEOUT"}


class QmmError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {_STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"CUDA library not built ({LIB}); run block_quantized_weight_route_gb300.build")
        L = ctypes.CDLL(LIB)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.qmm_last_error.restype = ctypes.c_char_p
        L.qmm_last_error.argtypes = []
        L.qmm_check_status.restype = i32
        L.qmm_check_status.argtypes = [P]
        L.qmm_w4a16.restype = i32
        L.qmm_w4a16.argtypes = [P, i32, i32, i32, P, P, ctypes.c_float, P, i32, P]
        L.qmm_fp8_blk128.restype = i32
        L.qmm_fp8_blk128.argtypes = [P, i32, i32, i32, P, P, P, P]
        L.qmm_dense_workspace_size.restype = sz
        L.qmm_dense_workspace_size.argtypes = [i32, i32, i32]
        L.qmm_w4a16_ws.restype = i32
        L.qmm_w4a16_ws.argtypes = [P, i32, i32, i32, P, P, ctypes.c_float, P, i32, P, sz, P]
        L.qmm_fp8_blk128_ws.restype = i32
        L.qmm_fp8_blk128_ws.argtypes = [P, i32, i32, i32, P, P, P, P, sz, P]
        L.moe_route_workspace_size.restype = sz
        L.moe_route_workspace_size.argtypes = [i32, i32, i32]
        L.moe_route_permute.restype = i32
        L.moe_route_permute.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
        L.moe_expert_stage_workspace_size.restype = sz
        L.moe_expert_stage_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.moe_expert_stage_workspace_layout.restype = i32
        L.moe_expert_stage_workspace_layout.argtypes = [i32, i32, i32, i32, i32, P]
        L.moe_route_permute_noalloc.restype = i32
        L.moe_route_permute_noalloc.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P]
        L.qmm_profile_enable.restype = i32
        L.qmm_profile_enable.argtypes = [i32]
        L.qmm_profile_read.restype = i32
        L.qmm_profile_read.argtypes = [P]
        L.qmm_profile_read_call.restype = i32
        L.qmm_profile_read_call.argtypes = [ctypes.c_long, P]
        L.moe_expert_stage_w4_iq4.restype = i32
        L.moe_expert_stage_w4_iq4.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
        L.moe_expert_stage_w4_iq4_ex.restype = i32
        L.moe_expert_stage_w4_iq4_ex.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, sz,
                                                 ctypes.c_uint, P]
        L.qmm_dbg_workspace_size.restype = sz
        L.qmm_dbg_workspace_size.argtypes = [i32, i32, i32, i32]
        L.qmm_dbg_gate_up_q8_1.restype = i32
        L.qmm_dbg_gate_up_q8_1.argtypes = [P, P, i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
        L.qmm_dbg_down_iq4.restype = i32
        L.qmm_dbg_down_iq4.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P, sz, P]
        L.qmm_dbg_combine.restype = i32
        L.qmm_dbg_combine.argtypes = [P, i32, P, P, i32, i32, i32, P, P]
        L.moe_expert_table_size.restype = sz
        L.moe_expert_table_size.argtypes = [i32]
        L.moe_expert_table_build.restype = i32
        L.moe_expert_table_build.argtypes = [i32, i32, i32, P, P, P, P, P, sz, P]
        L.moe_expert_stage_w4_iq4_table.restype = i32
        L.moe_expert_stage_w4_iq4_table.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, sz, ctypes.c_uint, P]
        L.qmm_q8_0_q8_1_workspace_size.restype = sz
        L.qmm_q8_0_q8_1_workspace_size.argtypes = [i32, i32, i32]
        L.qmm_q8_0_q8_1.restype = i32
        L.qmm_q8_0_q8_1.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
        L.qmm_dbg_wait_timeout.restype = i32
        L.qmm_dbg_wait_timeout.argtypes = [ctypes.c_uint, P]
        _lib = L
    return _lib


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise QmmError(fn, st, lib().qmm_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtypes, shape=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_F16 = (torch.float16, torch.int16, torch.uint16)
_U8 = (torch.uint8, torch.int8)


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def qmm_check_status(device=None) -> None:
    """Synchronise the current stream and raise if a kernel wait timed out."""
    _check("qmm_check_status", lib().qmm_check_status(_stream(device)))


def qmm_dense_workspace_size(M: int, K: int, N: int) -> int:
    return int(lib().qmm_dense_workspace_size(M, K, N))


def _dense_ws(ws, M: int, K: int, N: int, device):
    """The K-split workspace of a dense call: the caller's uint8 tensor, else one
    of qmm_dense_workspace_size bytes from torch's allocator (None if 0)."""
    if ws is None:
        n = qmm_dense_workspace_size(M, K, N)
        if n == 0:
            return None, 0
        ws = torch.empty(n, dtype=torch.uint8, device=device)
    _need(ws, "ws", _U8, (ws.numel(),))
    return ws, ws.numel()


def qmm_w4a16(X, Wc, Ws, scale2: float, out_dtype=torch.float32, Y=None, ws=None):
    """Y[M,N] = scale2 * X . dequant(Wc, Ws)^T  (e2m1 codes, E4M3 per-16 scales).
    ws: device workspace for K splits of the last wave (default: allocated)."""
    M, K = X.shape
    N = Wc.shape[0]
    _need(X, "X", _BF16, (M, K))
    _need(Wc, "Wc", _U8, (N, K // 2))
    _need(Ws, "Ws", _U8, (N, K // 16))
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out_dtype must be float32 or bfloat16")
    if Y is None:
        Y = torch.empty((M, N), dtype=out_dtype, device=X.device)
    _need(Y, "Y", (out_dtype,), (M, N))
    ws, nws = _dense_ws(ws, M, K, N, X.device)
    st = lib().qmm_w4a16_ws(_ptr(X), M, K, N, _ptr(Wc), _ptr(Ws), float(scale2), _ptr(Y),
                            0 if out_dtype == torch.float32 else 1, _ptr(ws) if ws is not None else None, nws,
                            _stream(X.device))
    _check("qmm_w4a16", st)
    return Y


def qmm_fp8_blk128(X, W, S, Y=None, ws=None):
    """Y[M,N] (bf16) = sum over 128x128 blocks of S[n/128, kb] * X . e4m3(W)^T.
    ws: device workspace for K splits of the last wave (default: allocated)."""
    M, K = X.shape
    N = W.shape[0]
    _need(X, "X", _BF16, (M, K))
    _need(W, "W", _U8 + (torch.float8_e4m3fn,), (N, K))
    _need(S, "S", (torch.float32,), (N // 128, K // 128))
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _need(Y, "Y", _BF16, (M, N))
    ws, nws = _dense_ws(ws, M, K, N, X.device)
    st = lib().qmm_fp8_blk128_ws(_ptr(X), M, K, N, _ptr(W), _ptr(S), _ptr(Y),
                                 _ptr(ws) if ws is not None else None, nws, _stream(X.device))
    _check("qmm_fp8_blk128", st)
    return Y


def qmm_q8_0_q8_1_workspace_size(M: int, K: int, N: int) -> int:
    return int(lib().qmm_q8_0_q8_1_workspace_size(M, K, N))


def qmm_q8_0_q8_1(Xq, Xd, Wq, Wd, ws=None, fp32_out: bool = False) -> dict:
    """Dense Q8_0 x q8_1 projection with its output rounded to q8_1 blocks.
    Xq int8 [M, K], Xd fp16 bits [M, K/32]; Wq int8 [N, K], Wd fp16 bits [N, K/32].
    Returns Yq int8 [M, N], Yd / Ys fp16 bits [M, N/32] and, with fp32_out, the
    fp32 rows Y [M, N] before the rounding."""
    M, K = Xq.shape
    N = Wq.shape[0]
    _need(Xq, "Xq", _U8, (M, K))
    _need(Xd, "Xd", _F16, (M, K // 32))
    _need(Wq, "Wq", _U8, (N, K))
    _need(Wd, "Wd", _F16, (N, K // 32))
    dev = Xq.device
    if ws is None:
        ws = torch.empty(max(qmm_q8_0_q8_1_workspace_size(M, K, N), 256), dtype=torch.uint8, device=dev)
    _need(ws, "ws", _U8)
    Yq = torch.empty((M, N), dtype=torch.int8, device=dev)
    Yd = torch.empty((M, N // 32), dtype=torch.int16, device=dev)
    Ys = torch.empty((M, N // 32), dtype=torch.int16, device=dev)
    Y = torch.empty((M, N), dtype=torch.float32, device=dev) if fp32_out else None
    _check("qmm_q8_0_q8_1", lib().qmm_q8_0_q8_1(_ptr(Xq), _ptr(Xd), M, K, N, _ptr(Wq), _ptr(Wd), _ptr(Yq), _ptr(Yd),
                                                _ptr(Ys), _ptr(Y), _ptr(ws), ws.numel(), _stream(dev)))
    return dict(Yq=Yq, Yd=Yd, Ys=Ys, Y=Y)


def moe_route_workspace_size(T: int, E: int, k: int) -> int:
    return int(lib().moe_route_workspace_size(T, E, k))


def moe_route_permute(logits, k: int, ws=None) -> dict:
    """Top-k routing and stable per-expert grouping; returns ids, w, counts,
    offsets, src, row as CUDA tensors."""
    T, E = logits.shape
    _need(logits, "logits", (torch.float32,), (T, E))
    dev = logits.device
    out = dict(ids=torch.empty((T, k), dtype=torch.int32, device=dev),
               w=torch.empty((T, k), dtype=torch.float32, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               src=torch.empty(T * k, dtype=torch.int32, device=dev),
               row=torch.empty((T, k), dtype=torch.int32, device=dev))
    need = moe_route_workspace_size(T, E, k)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(ws, "ws", _U8)
    st = lib().moe_route_permute(_ptr(logits), T, E, k, _ptr(out["ids"]), _ptr(out["w"]), _ptr(out["counts"]),
                                 _ptr(out["offsets"]), _ptr(out["src"]), _ptr(out["row"]), _ptr(ws), ws.numel(),
                                 _stream(dev))
    _check("moe_route_permute", st)
    return out


def moe_expert_stage_workspace_size(T: int, D: int, F: int, E: int, k: int) -> int:
    return int(lib().moe_expert_stage_workspace_size(T, D, F, E, k))


def moe_expert_stage_workspace_layout(T: int, D: int, F: int, E: int, k: int) -> dict:
    arr = (ctypes.c_size_t * QMM_WS_FIELDS)()
    _check("moe_expert_stage_workspace_layout",
           lib().moe_expert_stage_workspace_layout(T, D, F, E, k, ctypes.cast(arr, ctypes.c_void_p)))
    return dict(zip(WS_FIELD_NAMES, [int(v) for v in arr]))


def moe_expert_stage_w4_iq4(X, logits, Wgu_c, Wgu_s, gu_scale2, Wd_idx, Wd_s, k: int, ws=None, Y=None,
                            slots: bool = False):
    """The routed expert stage: route, W4 gate/up + SwiGLU + q8_1, IQ4_NL down,
    weighted combine.  Returns Y [T, D] fp32 (and leaves intermediates in ws).
    slots=False: the combine is fused into the down product (fp32 atomic adds,
    summation order not fixed); slots=True: per-row down outputs in the
    workspace's Yslot, then the j-ordered combine (moe_expert_stage_w4_iq4_ex
    with QMM_STAGE_SLOTS)."""
    T, D = X.shape
    E = logits.shape[1]
    F = Wgu_c.shape[1] // 2
    _need(X, "X", _BF16, (T, D))
    _need(logits, "logits", (torch.float32,), (T, E))
    _need(Wgu_c, "Wgu_c", _U8, (E, 2 * F, D // 2))
    _need(Wgu_s, "Wgu_s", _U8, (E, 2 * F, D // 16))
    _need(gu_scale2, "gu_scale2", (torch.float32,), (E,))
    _need(Wd_idx, "Wd_idx", _U8, (E, D, F // 2))
    _need(Wd_s, "Wd_s", _F16, (E, D, F // 32))
    dev = X.device
    if ws is None:
        ws = torch.empty(max(moe_expert_stage_workspace_size(T, D, F, E, k), 256), dtype=torch.uint8, device=dev)
    _need(ws, "ws", _U8)
    if Y is None:
        Y = torch.empty((T, D), dtype=torch.float32, device=dev)
    _need(Y, "Y", (torch.float32,), (T, D))
    if slots:
        st = lib().moe_expert_stage_w4_iq4_ex(_ptr(X), _ptr(logits), T, D, F, E, k, _ptr(Wgu_c), _ptr(Wgu_s),
                                              _ptr(gu_scale2), _ptr(Wd_idx), _ptr(Wd_s), _ptr(Y), _ptr(ws),
                                              ws.numel(), QMM_STAGE_SLOTS, _stream(dev))
    else:
        st = lib().moe_expert_stage_w4_iq4(_ptr(X), _ptr(logits), T, D, F, E, k, _ptr(Wgu_c), _ptr(Wgu_s),
                                           _ptr(gu_scale2), _ptr(Wd_idx), _ptr(Wd_s), _ptr(Y), _ptr(ws), ws.numel(),
                                           _stream(dev))
    _check("moe_expert_stage_w4_iq4", st)
    return Y


def moe_expert_table_build(Wgu_c, Wgu_s, Wd_idx, Wd_s) -> torch.Tensor:
    """A pointer table over per-expert weight tensors (lists of E CUDA tensors:
    [2F, D/2] and [2F, D/16] uint8, [D, F/2] uint8, [D, F/32] fp16 bits).  Returns
    the table (a uint8 device tensor); the weight tensors must outlive its use."""
    E = len(Wgu_c)
    if not (len(Wgu_s) == len(Wd_idx) == len(Wd_s) == E) or E < 1:
        raise ValueError("four lists of E per-expert tensors")
    F2, D2 = Wgu_c[0].shape
    F, D = F2 // 2, D2 * 2
    for e in range(E):
        _need(Wgu_c[e], "Wgu_c[e]", _U8, (2 * F, D // 2))
        _need(Wgu_s[e], "Wgu_s[e]", _U8, (2 * F, D // 16))
        _need(Wd_idx[e], "Wd_idx[e]", _U8, (D, F // 2))
        _need(Wd_s[e], "Wd_s[e]", _F16, (D, F // 32))
    dev = Wgu_c[0].device
    n = int(lib().moe_expert_table_size(E))
    table = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    arr = lambda ts: (ctypes.c_void_p * E)(*[t.data_ptr() for t in ts])  # noqa: E731
    _check("moe_expert_table_build",
           lib().moe_expert_table_build(D, F, E, arr(Wgu_c), arr(Wgu_s), arr(Wd_idx), arr(Wd_s), _ptr(table),
                                        table.numel(), _stream(dev)))
    return table


def moe_expert_stage_w4_iq4_table(X, logits, gu_scale2, table, F: int, k: int, ws=None, Y=None, slots: bool = False):
    """moe_expert_stage_w4_iq4 over a pointer table of per-expert weights
    (moe_expert_table_build)."""
    T, D = X.shape
    E = logits.shape[1]
    _need(X, "X", _BF16, (T, D))
    _need(logits, "logits", (torch.float32,), (T, E))
    _need(gu_scale2, "gu_scale2", (torch.float32,), (E,))
    _need(table, "table", _U8)
    dev = X.device
    if ws is None:
        ws = torch.empty(max(moe_expert_stage_workspace_size(T, D, F, E, k), 256), dtype=torch.uint8, device=dev)
    _need(ws, "ws", _U8)
    if Y is None:
        Y = torch.empty((T, D), dtype=torch.float32, device=dev)
    _need(Y, "Y", (torch.float32,), (T, D))
    _check("moe_expert_stage_w4_iq4_table",
           lib().moe_expert_stage_w4_iq4_table(_ptr(X), _ptr(logits), T, D, F, E, k, _ptr(gu_scale2), _ptr(table),
                                               _ptr(Y), _ptr(ws), ws.numel(), QMM_STAGE_SLOTS if slots else 0,
                                               _stream(dev)))
    return Y


def qmm_dbg_workspace_size(P: int, D: int, F: int, E: int) -> int:
    return int(lib().qmm_dbg_workspace_size(P, D, F, E))


def _dbg_ws(ws, P, D, F, E, dev):
    if ws is None:
        ws = torch.empty(max(qmm_dbg_workspace_size(P, D, F, E), 256), dtype=torch.uint8, device=dev)
    return _need(ws, "ws", _U8)


def qmm_dbg_gate_up_q8_1(X_perm, offsets, Wgu_c, Wgu_s, gu_scale2, ws=None):
    """Gate/up + SwiGLU + q8_1 of expert-grouped rows X_perm [P, D] (expert e owns
    rows offsets[e] .. offsets[e+1]-1).  Returns (Hq int8 [P, F], Hd, Hs fp16 bits
    as int16 [P, F/32])."""
    P, D = X_perm.shape
    E, F2 = Wgu_c.shape[0], Wgu_c.shape[1]
    F = F2 // 2
    _need(X_perm, "X_perm", _BF16, (P, D))
    _need(offsets, "offsets", (torch.int32,), (E + 1,))
    _need(Wgu_c, "Wgu_c", _U8, (E, F2, D // 2))
    _need(Wgu_s, "Wgu_s", _U8, (E, F2, D // 16))
    _need(gu_scale2, "gu_scale2", (torch.float32,), (E,))
    dev = X_perm.device
    ws = _dbg_ws(ws, P, D, F, E, dev)
    Hq = torch.empty((P, F), dtype=torch.int8, device=dev)
    Hd = torch.empty((P, F // 32), dtype=torch.int16, device=dev)
    Hs = torch.empty((P, F // 32), dtype=torch.int16, device=dev)
    st = lib().qmm_dbg_gate_up_q8_1(_ptr(X_perm), _ptr(offsets), P, D, F, E, _ptr(Wgu_c), _ptr(Wgu_s),
                                    _ptr(gu_scale2), _ptr(Hq), _ptr(Hd), _ptr(Hs), _ptr(ws), ws.numel(), _stream(dev))
    _check("qmm_dbg_gate_up_q8_1", st)
    return Hq, Hd, Hs


def qmm_dbg_down_iq4(Hq, Hd, offsets, Wd_idx, Wd_s, ws=None):
    """Down product of q8_1 rows (Hq int8 [P, F], Hd fp16 bits [P, F/32]) against
    IQ4_NL weights, grouped by offsets.  Returns Yslot fp32 [P, D]."""
    P, F = Hq.shape
    E, D = Wd_idx.shape[0], Wd_idx.shape[1]
    _need(Hq, "Hq", (torch.int8,), (P, F))
    _need(Hd, "Hd", _F16, (P, F // 32))
    _need(offsets, "offsets", (torch.int32,), (E + 1,))
    _need(Wd_idx, "Wd_idx", _U8, (E, D, F // 2))
    _need(Wd_s, "Wd_s", _F16, (E, D, F // 32))
    dev = Hq.device
    ws = _dbg_ws(ws, P, D, F, E, dev)
    Yslot = torch.empty((P, D), dtype=torch.float32, device=dev)
    st = lib().qmm_dbg_down_iq4(_ptr(Hq), _ptr(Hd), _ptr(offsets), P, D, F, E, _ptr(Wd_idx), _ptr(Wd_s),
                                _ptr(Yslot), _ptr(ws), ws.numel(), _stream(dev))
    _check("qmm_dbg_down_iq4", st)
    return Yslot


def qmm_dbg_combine(Yslot, row, w):
    """Y[t] = sum_j w[t, j] * Yslot[row[t, j]] (j ascending).  Returns Y fp32 [T, D]."""
    P, D = Yslot.shape
    T, k = row.shape
    _need(Yslot, "Yslot", (torch.float32,), (P, D))
    _need(row, "row", (torch.int32,), (T, k))
    _need(w, "w", (torch.float32,), (T, k))
    dev = Yslot.device
    Y = torch.empty((T, D), dtype=torch.float32, device=dev)
    st = lib().qmm_dbg_combine(_ptr(Yslot), P, _ptr(row), _ptr(w), T, k, D, _ptr(Y), _stream(dev))
    _check("qmm_dbg_combine", st)
    return Y


def qmm_dbg_wait_timeout(timeout_us: int, device=None) -> None:
    """Launch the wait-timeout probe (a bounded wait that nothing satisfies); the
    next qmm_check_status raises QmmError with status QMM_ERR_TIMEOUT."""
    _check("qmm_dbg_wait_timeout", lib().qmm_dbg_wait_timeout(int(timeout_us), _stream(device)))


PROFILE_PHASES = ("route", "gather", "gate_up", "down", "combine")


def qmm_profile_enable(on: bool) -> None:
    _check("qmm_profile_enable", lib().qmm_profile_enable(1 if on else 0))


def qmm_profile_read() -> dict:
    """Phase times (ms) of the last profiled expert-stage call (waits for it)."""
    arr = (ctypes.c_float * len(PROFILE_PHASES))()
    _check("qmm_profile_read", lib().qmm_profile_read(ctypes.cast(arr, ctypes.c_void_p)))
    return dict(zip(PROFILE_PHASES, [float(v) for v in arr]))


def qmm_profile_read_call(i: int) -> dict:
    """Phase times (ms) of the i-th profiled expert-stage call since profiling was
    switched on (one of the last 256; waits for that call only)."""
    arr = (ctypes.c_float * len(PROFILE_PHASES))()
    _check("qmm_profile_read_call", lib().qmm_profile_read_call(int(i), ctypes.cast(arr, ctypes.c_void_p)))
    return dict(zip(PROFILE_PHASES, [float(v) for v in arr]))


def workspace_view(ws: torch.Tensor, layout: dict, name: str, dtype, shape) -> torch.Tensor:
    """A typed view of one region of an expert-stage workspace."""
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    off = layout[name]
    return ws[off:off + nbytes].view(dtype).view(*shape)
