"""The C-ABI library builds, loads and exports every entry point declared in
include/*.h; host-side argument checks and workspace arithmetic (no GPU)."""
import ctypes
import glob
import os
import re

import pytest

from block_quantized_weight_route_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    path = qbuild.build_library()
    return ctypes.CDLL(path)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(", src, re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"qmm_w4a16", "qmm_fp8_blk128", "moe_route_permute", "moe_expert_stage_w4_iq4"} <= names
    for n in names:
        assert hasattr(L, n), n


def test_library_has_no_oracle_dependency():
    """The product library must not link or embed anything from oracle/."""
    data = open(qbuild.build_library(), "rb").read()
    assert b"orc_" not in data and b"liboracle" not in data


def _status(fn, *args):
    return fn(*args)


def test_argument_checks_return_before_any_device_work(L):
    P = ctypes.c_void_p
    L.qmm_w4a16.restype = ctypes.c_int
    L.qmm_w4a16.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_float, P, ctypes.c_int, P]
    # null pointers
    assert L.qmm_w4a16(None, 64, 512, 512, None, None, 1.0, None, 0, None) == 1
    # misaligned
    assert L.qmm_w4a16(P(16), 64, 512, 512, P(17), P(32), 1.0, P(48), 0, None) == 1
    # shapes: K not a multiple of 32, N not a multiple of 32
    assert L.qmm_w4a16(P(256), 64, 100, 512, P(256), P(256), 1.0, P(256), 0, None) == 2
    assert L.qmm_w4a16(P(256), 64, 16, 512, P(256), P(256), 1.0, P(256), 0, None) == 2
    assert L.qmm_w4a16(P(256), 64, 512, 500, P(256), P(256), 1.0, P(256), 0, None) == 2
    L.qmm_fp8_blk128.restype = ctypes.c_int
    L.qmm_fp8_blk128.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P]
    assert L.qmm_fp8_blk128(P(256), 64, 200, 256, P(256), P(256), P(256), None) == 2
    L.qmm_last_error.restype = ctypes.c_char_p
    assert b"qmm_fp8_blk128" in L.qmm_last_error()
    # the workspace variants: a workspace that is not 256-byte aligned
    sz = ctypes.c_size_t
    L.qmm_w4a16_ws.restype = ctypes.c_int
    L.qmm_w4a16_ws.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_float, P, ctypes.c_int,
                               P, sz, P]
    assert L.qmm_w4a16_ws(P(256), 64, 512, 512, P(256), P(256), 1.0, P(256), 0, P(4096 + 16), 1 << 20, None) == 1
    assert b"256-byte" in L.qmm_last_error()
    assert L.qmm_w4a16_ws(P(256), 64, 100, 512, P(256), P(256), 1.0, P(256), 0, P(4096), 1 << 20, None) == 2
    L.qmm_fp8_blk128_ws.restype = ctypes.c_int
    L.qmm_fp8_blk128_ws.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, sz, P]
    assert L.qmm_fp8_blk128_ws(P(256), 64, 256, 256, P(256), P(256), P(256), P(4096 + 128), 1 << 20, None) == 1
    # the workspace size: none for shapes that never split (K % 256 != 0)
    L.qmm_dense_workspace_size.restype = sz
    L.qmm_dense_workspace_size.argtypes = [ctypes.c_int] * 3
    assert L.qmm_dense_workspace_size(64, 384, 512) == 0
    assert L.qmm_dense_workspace_size(0, 512, 512) == 0
    L.moe_route_permute.restype = ctypes.c_int
    L.moe_route_permute.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int] + [P] * 7 + [ctypes.c_size_t, P]
    # k > 16, E > 512
    assert L.moe_route_permute(P(256), 10, 64, 17, *([P(256)] * 7), 1 << 20, None) == 2
    assert L.moe_route_permute(P(256), 10, 1024, 8, *([P(256)] * 7), 1 << 20, None) == 2
    # workspace too small
    L.moe_route_workspace_size.restype = ctypes.c_size_t
    need = L.moe_route_workspace_size(1000, 128, 8)
    assert need >= 4 * 128 * 4
    assert L.moe_route_permute(P(256), 1000, 128, 8, *([P(256)] * 7), need - 1, None) == 4
    # the dense Q8_0 x q8_1 projection: K not a multiple of 256, N not of 128, null pointers
    L.qmm_q8_0_q8_1.restype = ctypes.c_int
    L.qmm_q8_0_q8_1.argtypes = [P, P] + [ctypes.c_int] * 3 + [P] * 7 + [sz, P]
    assert L.qmm_q8_0_q8_1(*([P(256)] * 2), 64, 200, 128, *([P(256)] * 7), 1 << 30, None) == 2
    assert L.qmm_q8_0_q8_1(*([P(256)] * 2), 64, 256, 100, *([P(256)] * 7), 1 << 30, None) == 2
    assert L.qmm_q8_0_q8_1(None, None, 64, 256, 128, *([None] * 7), 1 << 30, None) == 1
    L.qmm_q8_0_q8_1_workspace_size.restype = sz
    L.qmm_q8_0_q8_1_workspace_size.argtypes = [ctypes.c_int] * 3
    assert L.qmm_q8_0_q8_1_workspace_size(2048, 5120, 8064) >= (2048 + 8064) * 5120 * 2   # both operands as f16
    assert L.qmm_q8_0_q8_1_workspace_size(2048, 100, 8064) == 0
    assert L.qmm_q8_0_q8_1_workspace_size(2048, 5120, 100) == 0
    # the stage with options: an unknown flag bit is rejected before any device work
    L.moe_expert_stage_w4_iq4_ex.restype = ctypes.c_int
    L.moe_expert_stage_w4_iq4_ex.argtypes = [P, P] + [ctypes.c_int] * 5 + [P] * 7 + [sz, ctypes.c_uint, P]
    assert L.moe_expert_stage_w4_iq4_ex(P(256), P(256), 10, 256, 256, 8, 2, *([P(256)] * 7), 1 << 30, 2, None) == 1
    assert b"flags" in L.qmm_last_error()


def test_expert_stage_workspace_layout_is_consistent(L):
    from block_quantized_weight_route_gb300 import QMM_WS_FIELDS
    L.moe_expert_stage_workspace_size.restype = ctypes.c_size_t
    L.moe_expert_stage_workspace_layout.restype = ctypes.c_int
    for (T, D, F, E, k) in [(5268, 2048, 768, 128, 8), (21504, 2560, 1024, 256, 8), (1, 128, 128, 2, 1)]:
        arr = (ctypes.c_size_t * QMM_WS_FIELDS)()
        assert L.moe_expert_stage_workspace_layout(T, D, F, E, k, arr) == 0
        off = list(arr)
        assert off[0] == 0 and all(o % 256 == 0 for o in off)
        assert all(b > a for a, b in zip(off, off[1:]))
        assert off[-1] == L.moe_expert_stage_workspace_size(T, D, F, E, k)
        P = T * k
        # the large regions have at least their nominal sizes
        assert off[12] - off[11] >= P * D * 2         # X_perm
        assert off[13] - off[12] >= P * F * 2         # Hq (f16 codes)
        assert off[17] - off[16] >= P * D * 4         # Yslot
        assert off[18] - off[17] >= P * 4             # wrow
    arr = (ctypes.c_size_t * QMM_WS_FIELDS)()
    assert L.moe_expert_stage_workspace_layout(10, 100, 128, 8, 2, arr) == 2     # D % 128
    assert L.moe_expert_stage_workspace_layout(10, 128, 2048, 8, 2, arr) == 2    # F > 1024


def test_dbg_substep_argument_checks(L):
    """The qmm_dbg_* sub-step calls reject bad arguments before any device work."""
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.qmm_dbg_workspace_size.restype = sz
    L.qmm_dbg_workspace_size.argtypes = [i32] * 4
    n = L.qmm_dbg_workspace_size(1000, 256, 256, 8)
    assert n >= 1000 * 256 * 2                        # f16 H codes
    assert L.qmm_dbg_workspace_size(2000, 256, 256, 8) > n
    L.qmm_dbg_down_iq4.restype = i32
    L.qmm_dbg_down_iq4.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P, sz, P]
    ok = [P(256)] * 3
    w = [P(256)] * 3
    assert L.qmm_dbg_down_iq4(None, P(256), P(256), 1000, 256, 256, 8, *w, P(256), n, None) == 1   # null
    assert L.qmm_dbg_down_iq4(*ok, 1000, 256, 256, 8, P(264), P(256), P(256), P(256), n, None) == 1  # misaligned
    assert L.qmm_dbg_down_iq4(*ok, 1000, 256, 256, 8, *w, P(256 + 16), n, None) == 1   # ws not 256-aligned
    assert L.qmm_dbg_down_iq4(*ok, 1000, 256, 2048, 8, *w, P(256), 1 << 40, None) == 2  # F > 1024
    assert L.qmm_dbg_down_iq4(*ok, 1000, 200, 256, 8, *w, P(256), 1 << 40, None) == 2   # D % 128
    assert L.qmm_dbg_down_iq4(*ok, 1000, 256, 256, 1024, *w, P(256), 1 << 40, None) == 2  # E > 512
    assert L.qmm_dbg_down_iq4(*ok, 1000, 256, 256, 8, *w, P(256), n - 1, None) == 4     # workspace
    L.qmm_dbg_gate_up_q8_1.restype = i32
    L.qmm_dbg_gate_up_q8_1.argtypes = [P, P, i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
    assert L.qmm_dbg_gate_up_q8_1(P(256), None, 1000, 256, 256, 8, *([P(256)] * 6), P(256), n, None) == 1
    assert L.qmm_dbg_gate_up_q8_1(*([P(256)] * 2), 1000, 256, 100, 8, *([P(256)] * 6), P(256), n, None) == 2
    L.qmm_dbg_combine.restype = i32
    L.qmm_dbg_combine.argtypes = [P, i32, P, P, i32, i32, i32, P, P]
    assert L.qmm_dbg_combine(P(256), 100, P(256), P(256), 50, 2, 66, P(256), None) == 2    # D % 4
    assert L.qmm_dbg_combine(P(256), 100, P(256), P(256), 50, 17, 64, P(256), None) == 2   # k > 16
    assert L.qmm_dbg_combine(None, 100, P(256), P(256), 50, 2, 64, P(256), None) == 1      # null
    L.qmm_last_error.restype = ctypes.c_char_p
    assert b"qmm_dbg_combine" in L.qmm_last_error()
    L.qmm_dbg_wait_timeout.restype = i32
    L.qmm_dbg_wait_timeout.argtypes = [ctypes.c_uint, P]
    assert L.qmm_dbg_wait_timeout(0, None) == 1
    assert L.qmm_dbg_wait_timeout(3000000, None) == 1
    L.qmm_profile_read_call.restype = i32
    L.qmm_profile_read_call.argtypes = [ctypes.c_long, P]
    assert L.qmm_profile_read_call(0, None) == 1
