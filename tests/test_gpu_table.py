"""The pointer-table form of the expert stage ("perf: strix-hip BF16 GEMMs via
hipBLASLt", routed-MoE twins: grouped MoE GEMMs over per-expert pointer tables):
each expert's weights in an allocation of its own, in shuffled order with unrelated
allocations in between, give the contiguous call's Y bit for bit (per-slot form)
and agree with it up to the order of the k terms (fused combine)."""
import numpy as np
import pytest
import torch

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


def scattered(arrays, order, rng):
    """One device tensor per expert, allocated in `order` with padding between."""
    out = [None] * len(arrays)
    keep = []
    for e in order:
        keep.append(torch.empty(int(rng.integers(1, 64)) * 256, dtype=torch.uint8, device="cuda"))
        out[e] = dev(arrays[e])
    return out, keep


@pytest.mark.parametrize("T,D,F,E,k,zipf", [(333, 256, 256, 16, 4, 1.0), (1500, 2048, 768, 128, 8, 0.0)])
def test_table_stage_equals_contiguous_stage(qlib, T, D, F, E, k, zipf):
    g = wl.gen_moe(T, D, F, E, k, 1.0 / 128, zipf, seed=T + E)
    X = dev(g["X"].view(np.int16)).view(torch.bfloat16)
    L, s2 = dev(g["logits"]), dev(g["gu_scale2"])
    args = (dev(g["Wgu_c"]), dev(g["Wgu_s"]), s2, dev(g["Wd_idx"]), dev(g["Wd_s"].view(np.int16)))
    Y_slots = qlib.moe_expert_stage_w4_iq4(X, L, *args, k, slots=True)
    Y_fused = qlib.moe_expert_stage_w4_iq4(X, L, *args, k)
    rng = np.random.default_rng(E)
    order = rng.permutation(E)
    gu_c, k1 = scattered([g["Wgu_c"][e] for e in range(E)], order, rng)
    gu_s, k2 = scattered([g["Wgu_s"][e] for e in range(E)], order[::-1], rng)
    dn_i, k3 = scattered([g["Wd_idx"][e] for e in range(E)], rng.permutation(E), rng)
    dn_s, k4 = scattered([g["Wd_s"][e].view(np.int16) for e in range(E)], rng.permutation(E), rng)
    table = qlib.moe_expert_table_build(gu_c, gu_s, dn_i, dn_s)
    Yt_slots = qlib.moe_expert_stage_w4_iq4_table(X, L, s2, table, F, k, slots=True)
    Yt_fused = qlib.moe_expert_stage_w4_iq4_table(X, L, s2, table, F, k)
    qlib.qmm_check_status()
    assert torch.equal(Yt_slots, Y_slots)
    scale = float(Y_slots.abs().max())
    assert float((Yt_fused - Y_slots).abs().max()) <= 1e-6 * scale
    assert float((Y_fused - Y_slots).abs().max()) <= 1e-6 * scale


def test_table_build_rejects_misaligned_expert_buffers(qlib):
    E, D, F = 2, 128, 128
    ok = [torch.zeros((2 * F, D // 2), dtype=torch.uint8, device="cuda") for _ in range(E)]
    s = [torch.zeros((2 * F, D // 16), dtype=torch.uint8, device="cuda") for _ in range(E)]
    di = [torch.zeros((D, F // 2), dtype=torch.uint8, device="cuda") for _ in range(E)]
    ds = [torch.zeros((D, F // 32), dtype=torch.int16, device="cuda") for _ in range(E)]
    big = torch.zeros(2 * F * (D // 2) + 8, dtype=torch.uint8, device="cuda")
    ok[1] = big[8:].view(2 * F, D // 2)          # 8 bytes past an aligned start
    with pytest.raises(qlib.QmmError):
        qlib.moe_expert_table_build(ok, s, di, ds)
