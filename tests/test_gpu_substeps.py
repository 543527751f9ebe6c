"""Parity of each expert-stage sub-step (the qmm_dbg_* calls of the C ABI) with
the oracle, each step fed the oracle's own inputs for it, plus the check that
the three steps chained on the GPU reproduce the per-slot stage bit for bit.

Tolerances: q8_1 codes of H >= 99.9% equal and the rest off by one, d of H
within one fp16 ulp (the fp32 h feeding the block maximum is summed in another
order), s = d * sum(q) to fp16 rounding; the down product (exact integer block
dots, fp32 fold) within 1e-5 * max|oracle|; the combine (eight fp32 FMAs in j
order) within 1e-6 * max|oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def qlib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_weight_route_gb300 as q
    q.build_library()
    return q


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


def f16_of(bits):
    return np.asarray(bits).astype(np.uint16).view(np.float16).astype(np.float64)


CASES = [
    # T, D, F, E, k, zipf, seed: several tiles, ragged groups, empty experts
    (300, 256, 256, 8, 2, 0.0, 21),
    (333, 128, 384, 16, 4, 2.0, 22),
    (70, 384, 128, 64, 1, 0.0, 23),
]


@pytest.mark.parametrize("T,D,F,E,k,zipf,seed", CASES)
def test_dbg_gate_up_q8_1_matches_oracle(qlib, T, D, F, E, k, zipf, seed):
    g = wl.gen_moe(T, D, F, E, k, 1.0 / 128, zipf, seed=seed)
    r = oracle.route(g["logits"], k)
    P = T * k
    ref = oracle.moe_gate_up_q8_1(g["X"], g["Wgu_c"], g["Wgu_s"], g["gu_scale2"], r["offsets"], r["src"],
                                  np.arange(P))
    X_perm = g["X"][r["src"]]
    Hq, Hd, Hs = qlib.qmm_dbg_gate_up_q8_1(dev(X_perm.view(np.int16)).view(torch.bfloat16),
                                           dev(r["offsets"].astype(np.int32)), dev(g["Wgu_c"]), dev(g["Wgu_s"]),
                                           dev(g["gu_scale2"]))
    qlib.qmm_check_status()
    hq = Hq.cpu().numpy().astype(int)
    dq = hq - ref["Hq"].astype(int)
    assert np.max(np.abs(dq)) <= 1
    assert np.mean(dq == 0) >= 0.999
    hd = Hd.cpu().numpy().view(np.uint16)
    assert np.max(np.abs(hd.astype(int) - ref["Hd"].astype(int))) <= 1
    # s = d * sum(q) with the GPU's own codes and d
    hs = f16_of(Hs.cpu().numpy().view(np.uint16))
    ds = f16_of(hd) * hq.reshape(P, F // 32, 32).sum(axis=2)
    assert np.all(np.abs(hs - ds) <= 2.0 ** -10 * np.abs(ds) + 2.0 ** -24)


@pytest.mark.parametrize("T,D,F,E,k,zipf,seed", CASES)
def test_dbg_down_iq4_matches_oracle(qlib, T, D, F, E, k, zipf, seed):
    g = wl.gen_moe(T, D, F, E, k, 1.0 / 128, zipf, seed=seed)
    r = oracle.route(g["logits"], k)
    P = T * k
    # q8_1 inputs drawn directly: codes in [-127, 127], d in [2^-10, 2^-4]
    Hq = (wl.random_bytes(seed, 40, P * F).astype(np.int16) % 255 - 127).astype(np.int8).reshape(P, F)
    d = (2.0 ** -10 + wl.uniform(seed, 41, P * F // 32) * (2.0 ** -4 - 2.0 ** -10)).astype(np.float16)
    Hd = d.view(np.uint16).reshape(P, F // 32)
    ref = oracle.moe_down_iq4(Hq, Hd, r["offsets"], np.arange(P), g["Wd_idx"], g["Wd_s"])
    Ys = qlib.qmm_dbg_down_iq4(dev(Hq), dev(Hd.view(np.int16)), dev(r["offsets"].astype(np.int32)),
                               dev(g["Wd_idx"]), dev(g["Wd_s"].view(np.int16)))
    qlib.qmm_check_status()
    assert rel_err(Ys.cpu().numpy().astype(np.float64), ref) <= 1e-5


def test_dbg_down_iq4_extreme_codes_exact(qlib):
    """|q| = 127 against the codebook's extremes: every 32-block dot is the
    largest the format allows (32 * 127 * 127 < 2^24), with unit scales the
    fp32 fold of exact integers is exact."""
    T, D, F, E, k = 40, 128, 256, 2, 2
    g = wl.gen_moe(T, D, F, E, k, 1.0 / 128, 0.0, seed=24)
    r = oracle.route(g["logits"], k)
    P = T * k
    Hq = np.where(wl.random_bytes(24, 42, P * F).reshape(P, F) & 1, 127, -127).astype(np.int8)
    Hd = np.full((P, F // 32), 0x3C00, np.uint16)                 # d = 1
    Wd_idx = np.where(wl.random_bytes(24, 43, E * D * F // 2).reshape(E, D, F // 2) & 1, 0x00, 0xFF)
    Wd_idx = Wd_idx.astype(np.uint8)                                  # codebook -127 or 113
    Wd_s = np.full((E, D, F // 32), 0x3C00, np.uint16)              # d_W = 1
    ref = oracle.moe_down_iq4(Hq, Hd, r["offsets"], np.arange(P), Wd_idx, Wd_s)
    Ys = qlib.qmm_dbg_down_iq4(dev(Hq), dev(Hd.view(np.int16)), dev(r["offsets"].astype(np.int32)), dev(Wd_idx),
                               dev(Wd_s.view(np.int16)))
    qlib.qmm_check_status()
    assert np.array_equal(Ys.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("T,k,D", [(300, 2, 256), (1, 8, 128), (1000, 16, 64), (50, 8, 2560), (20, 4, 3072)])
def test_dbg_combine_matches_oracle(qlib, T, k, D):
    E = max(2 * k, 8)
    logits = (2.0 * wl.normal(31, 1, T * E)).astype(np.float32).reshape(T, E)
    r = oracle.route(logits, k)
    P = T * k
    Ys = wl.normal(31, 2, P * D).astype(np.float32).reshape(P, D)
    ref = oracle.moe_combine(r["w"], r["row"], Ys)
    Y = qlib.qmm_dbg_combine(dev(Ys), dev(r["row"].astype(np.int32)), dev(r["w"].astype(np.float32)))
    qlib.qmm_check_status()
    assert rel_err(Y.cpu().numpy().astype(np.float64), ref) <= 1e-6


def test_dbg_chain_reproduces_fused_stage(qlib):
    """route (from the stage's workspace) -> gate/up -> down -> combine through the
    sub-step calls gives the per-slot stage's Y (QMM_STAGE_SLOTS) bit for bit (same
    kernels), and the default stage, whose down product adds into Y with fp32
    atomics, agrees with it up to the order of the k terms."""
    T, D, F, E, k = 333, 256, 256, 16, 4
    g = wl.gen_moe(T, D, F, E, k, 1.0 / 128, 1.0, seed=25)
    size = qlib.moe_expert_stage_workspace_size(T, D, F, E, k)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    Xd = dev(g["X"].view(np.int16)).view(torch.bfloat16)
    args = (dev(g["Wgu_c"]), dev(g["Wgu_s"]), dev(g["gu_scale2"]), dev(g["Wd_idx"]), dev(g["Wd_s"].view(np.int16)))
    Yf = qlib.moe_expert_stage_w4_iq4(Xd, dev(g["logits"]), *args, k, ws=ws)
    Y = qlib.moe_expert_stage_w4_iq4(Xd, dev(g["logits"]), *args, k, ws=ws, slots=True)
    qlib.qmm_check_status()
    lay = qlib.moe_expert_stage_workspace_layout(T, D, F, E, k)
    P = T * k
    view = lambda name, dt, shape: qlib.workspace_view(ws, lay, name, dt, shape).clone()  # noqa: E731
    offsets, src = view("offsets", torch.int32, (E + 1,)), view("src", torch.int32, (P,))
    row, w = view("row", torch.int32, (T, k)), view("w", torch.float32, (T, k))
    Hq, Hd, _ = qlib.qmm_dbg_gate_up_q8_1(Xd[src.long()].contiguous(), offsets, *args[:3])
    Ys = qlib.qmm_dbg_down_iq4(Hq, Hd, offsets, *args[3:])
    Y2 = qlib.qmm_dbg_combine(Ys, row, w)
    qlib.qmm_check_status()
    assert torch.equal(Y, Y2)
    assert float((Yf - Y).abs().max()) <= 1e-6 * float(Y.abs().max())


def test_dbg_bad_offsets_are_reported(qlib):
    T, D, F, E, k = 50, 128, 128, 4, 2
    g = wl.gen_moe(T, D, F, E, k, 1.0 / 128, 0.0, seed=26)
    P = T * k
    Hq = torch.zeros((P, F), dtype=torch.int8, device="cuda")
    Hd = torch.zeros((P, F // 32), dtype=torch.int16, device="cuda")
    bad = dev(np.array([0, 60, 40, 90, P], np.int32))                 # not monotone
    qlib.qmm_dbg_down_iq4(Hq, Hd, bad, dev(g["Wd_idx"]), dev(g["Wd_s"].view(np.int16)))
    with pytest.raises(qlib.QmmError) as ei:
        qlib.qmm_check_status()
    assert ei.value.status == 1
    # the error word is cleared: a valid call afterwards is clean
    good = dev(np.array([0, 25, 50, 75, P], np.int32))
    qlib.qmm_dbg_down_iq4(Hq, Hd, good, dev(g["Wd_idx"]), dev(g["Wd_s"].view(np.int16)))
    qlib.qmm_check_status()


def test_dbg_combine_bad_row_is_reported(qlib):
    T, k, D = 10, 2, 64
    P = T * k
    Ys = torch.ones((P, D), dtype=torch.float32, device="cuda")
    row = torch.arange(P, dtype=torch.int32, device="cuda").view(T, k).contiguous()
    row[3, 1] = P                                                        # one past the end
    w = torch.full((T, k), 0.5, dtype=torch.float32, device="cuda")
    Y = qlib.qmm_dbg_combine(Ys, row, w)
    with pytest.raises(qlib.QmmError) as ei:
        qlib.qmm_check_status()
    assert ei.value.status == 1
    # the bad slot adds nothing; the others are summed
    assert float(Y[3, 0]) == 0.5 and float(Y[0, 0]) == 1.0


def test_bounded_wait_times_out_and_context_survives(qlib):
    """Failure detection without a fault: a bounded wait that nothing satisfies
    gives up after its limit, the host reads QMM_ERR_TIMEOUT through
    qmm_check_status, and the context keeps working (a GEMM right after is exact)."""
    qlib.qmm_dbg_wait_timeout(2000)                                   # 2 ms
    with pytest.raises(qlib.QmmError) as ei:
        qlib.qmm_check_status()
    assert ei.value.status == 6 and "device code 11" in str(ei.value)
    qlib.qmm_check_status()                                           # the word was cleared
    g = wl.gen_w4a16(64, 512, 512, 1.0 / 64, seed=27)
    Y = qlib.qmm_w4a16(dev(g["X"].view(np.int16)).view(torch.bfloat16), dev(g["Wc"]), dev(g["Ws"]),
                       float(g["scale2"]))
    qlib.qmm_check_status()
    ref = oracle.w4a16(g["X"], g["Wc"], g["Ws"], g["scale2"])
    assert rel_err(Y.cpu().numpy().astype(np.float64), ref) <= 1e-5
