"""moe_route_permute_noalloc: the routing entry point for callers that cannot
allocate device memory (for example code inside a CUDA stream capture, where
cudaMalloc is not allowed).  Its scratch is a fixed array inside the library.

Checked through the C ABI against moe_route_permute on the same inputs, on two
calls in a row with different inputs (the shared scratch keeps the previous
call's contents, which must not leak into the next result).  Integer outputs
must be identical; routing weights within the tolerance of the other routing
tests (2^-21), and in practice identical since the same kernels run.
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
        assert torch.max(torch.abs(got["w"] - ref["w"])).item() <= 2 ** -21


def test_noalloc_rejects_shapes_beyond_its_scratch(q):
    L = q.lib()
    P = ctypes.c_void_p
    # ceil(200000 / 256) * 512 counters exceed the 1 MiB scratch: refused before any GPU work
    st = L.moe_route_permute_noalloc(P(256), 200000, 512, 8, *([P(256)] * 6), None)
    assert st == 2
    assert b"too large" in L.qmm_last_error()
