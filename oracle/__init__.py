"""CPU oracle for block-quantized prefill GEMMs and the routed-MoE expert stage.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
bench's CPU-baseline arm.  The library (block_quantized_weight_route_gb300)
never imports it.  The arithmetic lives in qmm_oracle.c (fp32 dequant, fp64
accumulation); this module only marshals numpy arrays through ctypes and
composes the C steps into the full expert stage.

Parity status per function: every function here is pinned by tests in
tests/test_oracle_pins.py (library special cases, closed forms, exhaustive
format tables, invariants and brute force on tiny inputs).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build_oracle()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        L.orc_e2m1.restype = ctypes.c_float
        L.orc_e2m1.argtypes = [ctypes.c_uint]
        L.orc_e4m3.restype = ctypes.c_float
        L.orc_e4m3.argtypes = [ctypes.c_uint]
        L.orc_f16.restype = ctypes.c_double
        L.orc_f16.argtypes = [ctypes.c_uint16]
        L.orc_bf16.restype = ctypes.c_float
        L.orc_bf16.argtypes = [ctypes.c_uint16]
        L.orc_f16_rne.restype = ctypes.c_uint16
        L.orc_f16_rne.argtypes = [ctypes.c_float]
        L.orc_swiglu.restype = ctypes.c_float
        L.orc_swiglu.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_iq4nl_value.restype = ctypes.c_int
        L.orc_iq4nl_value.argtypes = [ctypes.c_uint]
        L.orc_w4a16.restype = None
        L.orc_w4a16.argtypes = [P, i32, i32, i32, P, P, ctypes.c_float, P, i32, P, i32, P]
        L.orc_fp8_blk128.restype = None
        L.orc_fp8_blk128.argtypes = [P, i32, i32, i32, P, P, P, i32, P, i32, P]
        L.orc_route.restype = None
        L.orc_route.argtypes = [P, i32, i32, i32, P, P, P, P, P, P]
        L.orc_q8_1_block.restype = None
        L.orc_q8_1_block.argtypes = [P, P, P, P]
        L.orc_moe_gate_up_q8_1.restype = None
        L.orc_moe_gate_up_q8_1.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, i32, P, P, P, P]
        L.orc_moe_down_iq4.restype = None
        L.orc_moe_down_iq4.argtypes = [P, P, i32, i32, i32, P, P, P, P, i32, P]
        L.orc_q8_0_q8_1.restype = None
        L.orc_q8_0_q8_1.argtypes = [P, P, i32, i32, i32, P, P, P, i32, P, i32, P]
        L.orc_moe_combine.restype = None
        L.orc_moe_combine.argtypes = [P, P, P, i32, i32, i32, P]
        _lib = L
    return _lib


def set_threads(n: int | None) -> None:
    """Thread count of the oracle's OpenMP loops (None: leave the default)."""
    if n is not None:
        os.environ["OMP_NUM_THREADS"] = str(n)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _sel(idx):
    if idx is None:
        return None, None, 0
    a, p = _c(idx, np.int32)
    return a, p, int(a.size)


# -- scalar formats ----------------------------------------------------------

def e2m1(code: int) -> float:
    return float(lib().orc_e2m1(code))


def e4m3(byte: int) -> float:
    return float(lib().orc_e4m3(byte))


def f16(bits: int) -> float:
    return float(lib().orc_f16(bits))


def bf16(bits: int) -> float:
    return float(lib().orc_bf16(bits))


def f16_rne(x: float) -> int:
    return int(lib().orc_f16_rne(x))


def swiglu(g: float, u: float) -> float:
    return float(lib().orc_swiglu(g, u))


def iq4nl_value(idx: int) -> int:
    return int(lib().orc_iq4nl_value(idx))


# -- GEMMs -------------------------------------------------------------------

def w4a16(X, Wc, Ws, scale2, rows=None, cols=None) -> np.ndarray:
    """Y = scale2 * X . dequant(W)^T in fp64 (unrounded).  X: bf16 bits [M,K]."""
    Xa, Xp = _c(X, np.uint16)
    M, K = Xa.shape
    Wca, Wcp = _c(Wc, np.uint8)
    Wsa, Wsp = _c(Ws, np.uint8)
    N = Wca.shape[0]
    ra, rp, nr = _sel(rows)
    ca, cp, nc = _sel(cols)
    nr = nr if rows is not None else M
    nc = nc if cols is not None else N
    Y = np.zeros((nr, nc), dtype=np.float64)
    lib().orc_w4a16(Xp, M, K, N, Wcp, Wsp, float(scale2), rp, nr, cp, nc,
                    Y.ctypes.data_as(ctypes.c_void_p))
    return Y


def fp8_blk128(X, W, S, rows=None, cols=None) -> np.ndarray:
    """Y = sum_kb S[n/128,kb] * (X . e4m3(W)^T restricted to block kb), fp64."""
    Xa, Xp = _c(X, np.uint16)
    M, K = Xa.shape
    Wa, Wp = _c(W, np.uint8)
    N = Wa.shape[0]
    Sa, Sp = _c(S, np.float32)
    ra, rp, nr = _sel(rows)
    ca, cp, nc = _sel(cols)
    nr = nr if rows is not None else M
    nc = nc if cols is not None else N
    Y = np.zeros((nr, nc), dtype=np.float64)
    lib().orc_fp8_blk128(Xp, M, K, N, Wp, Sp, rp, nr, cp, nc, Y.ctypes.data_as(ctypes.c_void_p))
    return Y


# -- expert stage ------------------------------------------------------------

def route(logits, k: int) -> dict:
    La, Lp = _c(logits, np.float32)
    T, E = La.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    src = np.zeros(T * k, np.int32)
    row = np.zeros((T, k), np.int32)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    lib().orc_route(Lp, T, E, k, vp(ids), vp(w), vp(counts), vp(offsets), vp(src), vp(row))
    return dict(ids=ids, w=w, counts=counts, offsets=offsets, src=src, row=row)


def q8_1_block(h) -> tuple:
    ha, hp = _c(h, np.float32)
    assert ha.size == 32
    q = np.zeros(32, np.int8)
    d = np.zeros(1, np.uint16)
    s = np.zeros(1, np.uint16)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    lib().orc_q8_1_block(hp, vp(q), vp(d), vp(s))
    return q, int(d[0]), int(s[0])


def moe_gate_up_q8_1(X, Wgu_c, Wgu_s, gu_scale2, offsets, src, rows, want_h=False) -> dict:
    Xa, Xp = _c(X, np.uint16)
    T, D = Xa.shape
    Wca, Wcp = _c(Wgu_c, np.uint8)
    E, F2, _ = Wca.shape
    F = F2 // 2
    Wsa, Wsp = _c(Wgu_s, np.uint8)
    s2a, s2p = _c(gu_scale2, np.float32)
    oa, op = _c(offsets, np.int32)
    sa, sp = _c(src, np.int32)
    ra, rp = _c(rows, np.int32)
    n = ra.size
    Hq = np.zeros((n, F), np.int8)
    Hd = np.zeros((n, F // 32), np.uint16)
    Hs = np.zeros((n, F // 32), np.uint16)
    h = np.zeros((n, F), np.float32) if want_h else None
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p) if a is not None else None  # noqa: E731
    lib().orc_moe_gate_up_q8_1(Xp, D, F, E, op, sp, Wcp, Wsp, s2p, rp, n,
                               vp(Hq), vp(Hd), vp(Hs), vp(h))
    out = dict(Hq=Hq, Hd=Hd, Hs=Hs)
    if want_h:
        out["h"] = h
    return out


def moe_down_iq4(Hq, Hd, offsets, rows, Wd_idx, Wd_s) -> np.ndarray:
    Ha, Hp = _c(Hq, np.int8)
    n, F = Ha.shape
    Hda, Hdp = _c(Hd, np.uint16)
    Wia, Wip = _c(Wd_idx, np.uint8)
    E, D, _ = Wia.shape
    Wsa, Wsp = _c(Wd_s, np.uint16)
    oa, op = _c(offsets, np.int32)
    ra, rp = _c(rows, np.int32)
    Y = np.zeros((n, D), np.float64)
    lib().orc_moe_down_iq4(Hp, Hdp, F, D, E, op, Wip, Wsp, rp, n, Y.ctypes.data_as(ctypes.c_void_p))
    return Y


def moe_combine(w, slot, Ys) -> np.ndarray:
    wa, wp = _c(w, np.float32)
    ntok, k = wa.shape
    sa, sp = _c(slot, np.int32)
    Ya, Yp = _c(Ys, np.float64)
    D = Ya.shape[1]
    Y = np.zeros((ntok, D), np.float64)
    lib().orc_moe_combine(wp, sp, Yp, ntok, k, D, Y.ctypes.data_as(ctypes.c_void_p))
    return Y


def moe_expert_stage(X, logits, Wgu_c, Wgu_s, gu_scale2, Wd_idx, Wd_s, k, tokens=None) -> dict:
    """Full stage for the selected tokens (None: all): route every token, then
    gate/up -> SwiGLU -> q8_1 -> down -> combine for the selected tokens' pairs.
    Returns Y [ntok, D] fp64 plus the routing and the per-pair intermediates."""
    r = route(logits, k)
    T = r["ids"].shape[0]
    toks = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    pair_rows = r["row"][toks].reshape(-1).astype(np.int32)      # rows of (t, j), j ascending
    gu = moe_gate_up_q8_1(X, Wgu_c, Wgu_s, gu_scale2, r["offsets"], r["src"], pair_rows)
    Ys = moe_down_iq4(gu["Hq"], gu["Hd"], r["offsets"], pair_rows, Wd_idx, Wd_s)
    slot = np.arange(pair_rows.size, dtype=np.int32).reshape(len(toks), k)
    Y = moe_combine(r["w"][toks], slot, Ys)
    return dict(Y=Y, route=r, tokens=toks, pair_rows=pair_rows, Hq=gu["Hq"], Hd=gu["Hd"],
                Hs=gu["Hs"], Yslot=Ys)


def q8_0_q8_1(Xq, Xd, Wq, Wd, rows=None, cols=None) -> np.ndarray:
    """Dense Q8_0 weights x q8_1 activations (exact int block dots, fp64 fold),
    fp64 [rows][cols].  Xq int8 [M,K], Xd fp16 bits [M,K/32], Wq int8 [N,K],
    Wd fp16 bits [N,K/32]."""
    Xqa, Xqp = _c(Xq, np.int8)
    Xda, Xdp = _c(Xd, np.uint16)
    Wqa, Wqp = _c(Wq, np.int8)
    Wda, Wdp = _c(Wd, np.uint16)
    M, K = Xqa.shape
    N = Wqa.shape[0]
    ra, rp, nr = _sel(rows)
    ca, cp, nc = _sel(cols)
    nr = nr if rows is not None else M
    nc = nc if cols is not None else N
    Y = np.zeros((nr, nc), dtype=np.float64)
    lib().orc_q8_0_q8_1(Xqp, Xdp, M, K, N, Wqp, Wdp, rp, nr, cp, nc, Y.ctypes.data)
    return Y


def q8_0_q8_1_requant(Xq, Xd, Wq, Wd, rows=None) -> dict:
    """The projection followed by its re-quantisation to q8_1: each output row's
    fp32 values (the fp64 sum rounded once) in blocks of 32 columns, as the
    q8_1 rounding of H.  Returns Y (fp64), Yq int8, Yd / Ys fp16 bits."""
    Y = q8_0_q8_1(Xq, Xd, Wq, Wd, rows=rows)
    nr, N = Y.shape
    Yq = np.zeros((nr, N), np.int8)
    Yd = np.zeros((nr, N // 32), np.uint16)
    Ys = np.zeros((nr, N // 32), np.uint16)
    y32 = Y.astype(np.float32)
    for i in range(nr):
        for b in range(N // 32):
            q, d, s_ = q8_1_block(y32[i, b * 32:(b + 1) * 32])
            Yq[i, b * 32:(b + 1) * 32] = q
            Yd[i, b] = d
            Ys[i, b] = s_
    return {"Y": Y, "Yq": Yq, "Yd": Yd, "Ys": Ys}

