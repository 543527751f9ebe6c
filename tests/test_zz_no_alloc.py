"""moe_route_permute_noalloc: the routing entry point for callers that cannot
allocate device memory (for example code inside a CUDA stream capture, where
cudaMalloc is not allowed).  Its scratch is a fixed array inside the library.

Checked through the C ABI against moe_route_permute on the same inputs, on two
calls in a row with different inputs (the shared scratch keeps the previous
call's contents, which must not leak into the next result), directly against the
CPU oracle, and replayed from a CUDA graph captured in the global capture mode.
Integer outputs must be identical; routing weights identical to
moe_route_permute's (the same kernels run) and within 16 fp32 ulps of the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_weight_route_gb300 as q
    q.build_library()
    L = q.lib()
    P, i32 = ctypes.c_void_p, ctypes.c_int
    L.moe_route_permute_noalloc.restype = i32
    L.moe_route_permute_noalloc.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P]
    return q


def run_noalloc(q, logits, k):
    T, E = logits.shape
    dev = logits.device
    out = dict(ids=torch.full((T, k), -1, dtype=torch.int32, device=dev),
               w=torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
               counts=torch.full((E,), -1, dtype=torch.int32, device=dev),
               offsets=torch.full((E + 1,), -1, dtype=torch.int32, device=dev),
               src=torch.full((T * k,), -1, dtype=torch.int32, device=dev),
               row=torch.full((T, k), -1, dtype=torch.int32, device=dev))
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = q.lib().moe_route_permute_noalloc(p(logits), T, E, k, p(out["ids"]), p(out["w"]), p(out["counts"]),
                                           p(out["offsets"]), p(out["src"]), p(out["row"]),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, q.lib().qmm_last_error().decode()
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_moe_route_permute_on_two_calls_in_a_row(q):
    from synthetic import workloads as wl
    cases = [
        (wl.gen_moe(5268, 128, 128, 128, 8, 1.0, 0.0, seed=3)["logits"], 8),
        (wl.gen_moe(21504, 128, 128, 256, 8, 1.0, 1.1, seed=4)["logits"], 8),
    ]
    for logits_np, k in cases:
        logits = torch.from_numpy(logits_np).cuda()
        ref = q.moe_route_permute(logits, k)
        got = run_noalloc(q, logits, k)
        for key in ("ids", "counts", "offsets", "src", "row"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["w"], ref["w"])


def test_noalloc_matches_oracle(q):
    """The same routing checked directly against the CPU oracle: integer outputs
    identical, weights within 16 fp32 ulps (the bound of the other routing tests)."""
    import oracle
    from synthetic import workloads as wl
    for logits_np, k in [(wl.gen_moe(5268, 128, 128, 128, 8, 1.0, 0.0, seed=3)["logits"], 8),
                         (wl.gen_moe(700, 128, 128, 64, 4, 1.0, 2.0, seed=9)["logits"], 4)]:
        r = oracle.route(logits_np, k)
        got = run_noalloc(q, torch.from_numpy(logits_np).cuda(), k)
        for key in ("ids", "counts", "offsets", "src", "row"):
            assert np.array_equal(got[key].cpu().numpy().reshape(r[key].shape), r[key]), key
        w = got["w"].cpu().numpy().reshape(r["w"].shape).astype(np.float64)
        w32 = r["w"].astype(np.float32)
        assert np.max(np.abs(w - w32) / np.spacing(np.abs(w32))) <= 16


def test_noalloc_captured_in_cuda_graph(q):
    """Captured under the global capture mode (where an allocation would fail the
    capture) after one ordinary call, then replayed on new logits copied into the
    captured input: every output equals moe_route_permute's on those logits."""
    from synthetic import workloads as wl
    T, E, k = 3000, 128, 8
    L1 = torch.from_numpy(wl.gen_moe(T, 128, 128, E, k, 1.0, 0.0, seed=11)["logits"]).cuda()
    L2 = torch.from_numpy(wl.gen_moe(T, 128, 128, E, k, 1.0, 0.5, seed=12)["logits"]).cuda()
    static_in = L1.clone()
    run_noalloc(q, static_in, k)   # the first call on the device resolves the scratch address
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        out = dict(ids=torch.empty((T, k), dtype=torch.int32, device="cuda"),
                   w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
                   counts=torch.empty((E,), dtype=torch.int32, device="cuda"),
                   offsets=torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
                   src=torch.empty((T * k,), dtype=torch.int32, device="cuda"),
                   row=torch.empty((T, k), dtype=torch.int32, device="cuda"))
    torch.cuda.current_stream().wait_stream(side)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    with torch.cuda.graph(graph, capture_error_mode="global"):
        st = q.lib().moe_route_permute_noalloc(p(static_in), T, E, k, p(out["ids"]), p(out["w"]), p(out["counts"]),
                                               p(out["offsets"]), p(out["src"]), p(out["row"]),
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, q.lib().qmm_last_error().decode()
    for L in (L2, L1):
        static_in.copy_(L)
        graph.replay()
        torch.cuda.synchronize()
        ref = q.moe_route_permute(L, k)
        for key in ("ids", "w", "counts", "offsets", "src", "row"):
            assert torch.equal(out[key].reshape(ref[key].shape), ref[key]), key


def test_noalloc_rejects_shapes_beyond_its_scratch(q):
    L = q.lib()
    P = ctypes.c_void_p
    # ceil(200000 / 256) * 512 counters exceed the 1 MiB scratch: refused before any GPU work
    st = L.moe_route_permute_noalloc(P(256), 200000, 512, 8, *([P(256)] * 6), None)
    assert st == 2
    assert b"too large" in L.qmm_last_error()
