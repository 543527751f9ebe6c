"""Parity of the dense Q8_0 x q8_1 projection re-quantised to q8_1 (qmm_q8_0_q8_1,
through the C ABI) with the CPU oracle ("Run Edge0-145B Q3_K on AMD HIP (Linux,
gfx1100)", commit 17c02cd: the latent layer's D and U projections as Q8_0 x q8_1
integer dots, D rounding its products to q8_1).

Tolerances: the fp32 rows before the rounding within 1e-5 * max|oracle| (exact
integer block dots, fp32 fold against the fp64 oracle); an exact match when
every block sum and fold is an exactly representable integer; q8_1 codes >= 99.9%
equal and the rest off by one (as the pages' own check of this kernel); the
block scales d equal wherever the two sides round the same block maximum, and
otherwise one fp16 ulp apart.
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


def run(qlib, g):
    out = qlib.qmm_q8_0_q8_1(dev(g["Xq"]), dev(g["Xd"].view(np.int16)), dev(g["Wq"]), dev(g["Wd"].view(np.int16)),
                             fp32_out=True)
    qlib.qmm_check_status()
    return {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}


def check(gpu, ref, rows):
    Y = gpu["Y"][rows].astype(np.float64)
    scale = max(np.max(np.abs(ref["Y"])), 1e-30)
    assert np.max(np.abs(Y - ref["Y"])) <= 1e-5 * scale
    dq = gpu["Yq"][rows].astype(int) - ref["Yq"].astype(int)
    assert np.max(np.abs(dq)) <= 1
    assert np.mean(dq == 0) >= 0.999
    # d: equal, or one fp16 ulp apart where the block maxima round differently
    d_gpu = gpu["Yd"][rows].view(np.uint16).astype(np.int64)
    d_ref = ref["Yd"].astype(np.int64)
    assert np.max(np.abs(d_gpu - d_ref)) <= 1
    assert np.mean(d_gpu == d_ref) >= 0.999
    # s = d * sum(q) of the GPU's own codes, within the fp16 rounding of s and of d
    d16 = gpu["Yd"][rows].view(np.float16).astype(np.float64)
    s16 = gpu["Ys"][rows].view(np.float16).astype(np.float64)
    qs = gpu["Yq"][rows].astype(np.int64).reshape(len(rows), -1, 32).sum(axis=2)
    assert np.all(np.abs(s16 - d16 * qs) <= 2.0 ** -10 * np.abs(d16 * qs) * 1.01 + 2.0 ** -24)


@pytest.mark.parametrize("M,K,N", [(64, 256, 128), (1, 256, 128), (130, 512, 256), (300, 1024, 384)])
def test_q8_0_q8_1_matches_oracle(qlib, M, K, N):
    g = wl.gen_q8_0_q8_1(M, K, N, seed=M + K + N)
    gpu = run(qlib, g)
    rows = np.arange(M)
    ref = oracle.q8_0_q8_1_requant(g["Xq"], g["Xd"], g["Wq"], g["Wd"], rows=rows)
    check(gpu, ref, rows)


def test_q8_0_q8_1_unit_scales_are_exact(qlib):
    """Scales 1.0 on both sides: y is the integer matmul of the codes, |y| <
    256 * 127 * 127 < 2^24, so the fp32 rows must equal the oracle exactly."""
    g = wl.gen_q8_0_q8_1(150, 256, 256, seed=7)
    g["Xd"] = np.full_like(g["Xd"], 0x3C00)
    g["Wd"] = np.full_like(g["Wd"], 0x3C00)
    gpu = run(qlib, g)
    ref = oracle.q8_0_q8_1(g["Xq"], g["Xd"], g["Wq"], g["Wd"])
    assert np.array_equal(gpu["Y"].astype(np.float64), ref)


def test_q8_0_q8_1_latent_d_shape_sampled(qlib):
    """M=2048 prompt rows at K=5120, N=8064: 41.3M multiply-adds per row, half of the
    82.6M the pages give for a latent layer's D and U projections together."""
    M, K, N = 2048, 5120, 8064
    g = wl.gen_q8_0_q8_1(M, K, N, seed=6)
    gpu = run(qlib, g)
    rows = np.array([0, 1, 127, 128, 129, 1000, 1919, 1920, 2046, 2047])
    ref = oracle.q8_0_q8_1_requant(g["Xq"], g["Xd"], g["Wq"], g["Wd"], rows=rows)
    check(gpu, ref, rows)


def test_q8_0_q8_1_rejects_bad_shapes(qlib):
    g = wl.gen_q8_0_q8_1(8, 256, 128, seed=1)
    with pytest.raises(qlib.QmmError):
        qlib.qmm_q8_0_q8_1(dev(g["Xq"][:, :160].copy()), dev(g["Xd"][:, :5].copy().view(np.int16)),
                           dev(g["Wq"][:, :160].copy()), dev(g["Wd"][:, :5].copy().view(np.int16)))
