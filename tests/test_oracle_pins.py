"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties an oracle function to a library routine, an exhaustive format
table, a closed form, an invariant of the method, or brute force on tiny
inputs, chosen so that a plausible slip (a dropped term, a wrong sign or index,
a transposed operand, a swapped nibble) fails at least one of them.
"""
from fractions import Fraction
import os

import numpy as np
import pytest
import torch

import oracle
from synthetic import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers independent of the oracle: closed forms and library decoders
# ---------------------------------------------------------------------------

def e2m1_closed_form(code: int) -> Fraction:
    """e2m1 from its bit fields: sign bit 3, exponent bits 2..1 (bias 1),
    mantissa bit 0; exponent field 0 is subnormal (m/2)."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -v if s else v


def e4m3_torch(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_torch(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def w4_dequant_independent(Wc: np.ndarray, Ws: np.ndarray) -> np.ndarray:
    """[N, K] float64 weights: nibble order low-then-high, e2m1 from the closed
    form, E4M3 scales decoded by torch."""
    N, Kh = Wc.shape
    codes = np.empty((N, 2 * Kh), np.int64)
    codes[:, 0::2] = Wc & 15
    codes[:, 1::2] = Wc >> 4
    lut = np.array([float(e2m1_closed_form(c)) for c in range(16)])
    scales = np.repeat(e4m3_torch(Ws), 16, axis=1)
    return lut[codes] * scales


def iq4_codebook_golden() -> np.ndarray:
    with open(os.path.join(GOLDEN, "iq4nl_codebook.txt")) as f:
        vals = [int(v) for line in f if not line.startswith("#") for v in line.split()]
    return np.array(vals, np.int64)


# ---------------------------------------------------------------------------
# scalar formats
# ---------------------------------------------------------------------------

def test_e2m1_all_codes_match_bit_field_definition():
    for c in range(16):
        assert Fraction(oracle.e2m1(c)) == e2m1_closed_form(c), c


def test_e4m3_all_bytes_match_torch_float8():
    ref = e4m3_torch(np.arange(256, dtype=np.uint8))
    got = np.array([oracle.e4m3(b) for b in range(256)])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.all(np.isnan(got[nan]))
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x01) == 2.0 ** -9


def test_f16_decode_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.all(np.isnan(got[nan]))
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_all_bit_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_torch(bits)
    got = np.array([oracle.bf16(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.all(np.isnan(got[nan]))
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_rne_encoder_matches_numpy():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(5000) * 1e-6).astype(np.float32),           # fp16 subnormals
        (rng.standard_normal(2000) * 3e-8).astype(np.float32),           # around half the smallest
        (rng.standard_normal(2000) * 7e4).astype(np.float32),            # overflow region
        np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                  np.inf, -np.inf], dtype=np.float32),
    ])
    # exact ties between neighbouring fp16 values: k * 2^-11 + 2^-12 in [1, 2)
    ties = (1.0 + (np.arange(0, 1024, 7) * 2.0 + 1.0) * 2.0 ** -11).astype(np.float32)
    vals = np.concatenate([vals, ties, -ties])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_rne(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


def test_e2m1_times_e4m3_exact_in_bf16_and_f16_all_254_scale_bytes():
    """'perf: strix-hip BF16 GEMMs via hipBLASLt', commit 'f16a twins': e2m1 x E4M3
    is exact in f16 over all 254 non-NaN scale bytes x 16 codes.  The same holds
    in bf16 (at most 2 + 4 significant bits, exponents in range)."""
    n = 0
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        s = Fraction(oracle.e4m3(b))
        for c in range(16):
            exact = e2m1_closed_form(c) * s
            p = np.float32(oracle.e2m1(c)) * np.float32(oracle.e4m3(b))
            assert Fraction(float(p)) == exact
            t = torch.tensor([float(p)], dtype=torch.float64)
            assert Fraction(t.to(torch.bfloat16).to(torch.float64).item()) == exact
            assert Fraction(t.to(torch.float16).to(torch.float64).item()) == exact
            n += 1
    assert n == 254 * 16


def test_iq4nl_codebook_matches_fixture():
    cb = iq4_codebook_golden()
    assert cb.size == 16 and np.all(np.diff(cb) > 0)
    assert [oracle.iq4nl_value(i) for i in range(16)] == list(cb)


def test_swiglu_matches_torch_silu():
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(4000) * 6).astype(np.float32)
    u = (rng.standard_normal(4000) * 6).astype(np.float32)
    ref = (torch.nn.functional.silu(torch.from_numpy(g).double()) * torch.from_numpy(u).double()).float().numpy()
    got = np.array([oracle.swiglu(float(a), float(b)) for a, b in zip(g, u)], np.float32)
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)) <= 2 ** -23


# ---------------------------------------------------------------------------
# dense W4A16
# ---------------------------------------------------------------------------

def _bf16_bits_of(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_w4a16_unit_scales_equals_exact_integer_matmul():
    """All scale bytes 0x38 (= 1.0) and scale2 = 1: Y = X . e2m1(W)^T exactly;
    2*e2m1 is an integer, so int64 numpy matmul gives the exact result."""
    rng = np.random.default_rng(11)
    M, K, N = 7, 96, 13
    Xi = rng.integers(-20, 21, size=(M, K))
    X = _bf16_bits_of(Xi.astype(np.float32))
    Wc = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    Ws = np.full((N, K // 16), 0x38, np.uint8)
    codes = np.empty((N, K), np.int64)
    codes[:, 0::2] = Wc & 15
    codes[:, 1::2] = Wc >> 4
    twice = np.array([int(2 * e2m1_closed_form(c)) for c in range(16)], np.int64)
    exact2 = Xi @ twice[codes].T                          # 2 * Y, integers
    Y = oracle.w4a16(X, Wc, Ws, 1.0)
    assert np.array_equal(Y * 2, exact2.astype(np.float64))


def test_w4a16_single_code_selects_one_column_and_scale_block():
    rng = np.random.default_rng(12)
    M, K, N = 5, 64, 9
    X = _bf16_bits_of(rng.standard_normal((M, K)).astype(np.float32))
    xf = bf16_torch(X)
    for (n0, k0, code, sbyte) in [(0, 0, 0x3, 0x30), (8, 63, 0xF, 0x4D), (4, 17, 0x9, 0x01)]:
        Wc = np.zeros((N, K // 2), np.uint8)
        Wc[n0, k0 // 2] = code << 4 if (k0 & 1) else code
        Ws = np.full((N, K // 16), 0x38, np.uint8)
        Ws[n0, k0 // 16] = sbyte
        Y = oracle.w4a16(X, Wc, Ws, 0.25)
        expect = np.zeros((M, N))
        expect[:, n0] = xf[:, k0] * float(e2m1_closed_form(code)) * e4m3_torch(np.array([sbyte]))[0] * 0.25
        assert np.array_equal(Y, expect)


def test_w4a16_random_matches_torch_matmul_and_sampling():
    w = wl.gen_w4a16(33, 256, 40, 1.0 / 64, seed=5)
    Wf = w4_dequant_independent(w["Wc"], w["Ws"])
    ref = (torch.from_numpy(bf16_torch(w["X"])) @ torch.from_numpy(Wf).T).numpy() / 64
    Y = oracle.w4a16(w["X"], w["Wc"], w["Ws"], w["scale2"])
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))
    rows, cols = np.array([32, 0, 7]), np.array([39, 1])
    Ys = oracle.w4a16(w["X"], w["Wc"], w["Ws"], w["scale2"], rows=rows, cols=cols)
    assert np.array_equal(Ys, Y[np.ix_(rows, cols)])


# ---------------------------------------------------------------------------
# dense FP8 with 128x128 block scales
# ---------------------------------------------------------------------------

def test_fp8_blk128_matches_blockwise_torch_and_unit_scale_case():
    M, K, N = 9, 384, 256
    g = wl.gen_fp8_blk128(M, K, N, seed=9)
    X, W, S = g["X"], g["W"], g["S"]
    xf = torch.from_numpy(bf16_torch(X))
    wf = torch.from_numpy(e4m3_torch(W))
    ref = torch.zeros(M, N, dtype=torch.float64)
    for nb in range(N // 128):
        for kb in range(K // 128):
            blk = xf[:, kb * 128:(kb + 1) * 128] @ wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].T
            ref[:, nb * 128:(nb + 1) * 128] += float(S[nb, kb]) * blk
    Y = oracle.fp8_blk128(X, W, S)
    assert np.max(np.abs(Y - ref.numpy())) <= 1e-12 * ref.abs().max().item()
    # scale 1 everywhere: a plain matmul of the decoded codes
    Y1 = oracle.fp8_blk128(X, W, np.ones_like(S))
    ref1 = (xf @ wf.T).numpy()
    assert np.max(np.abs(Y1 - ref1)) <= 1e-12 * np.max(np.abs(ref1))
    # a block scale multiplies only its own 128x128 block
    S2 = S.copy()
    S2[1, 2] *= 2.0
    d = oracle.fp8_blk128(X, W, S2) - Y
    assert np.all(d[:, :128] == 0)
    blk = (xf[:, 256:384] @ wf[128:256, 256:384].T).numpy() * float(S[1, 2])
    assert np.max(np.abs(d[:, 128:] - blk)) <= 1e-12 * np.max(np.abs(blk))


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(37, 16, 4), (200, 128, 8), (64, 256, 8), (5, 8, 8), (23, 512, 16), (9, 3, 1)])
def test_route_matches_torch_topk_and_invariants(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    logits = (2 * rng.standard_normal((T, E))).astype(np.float32)
    r = oracle.route(logits, k)
    vals, ids = torch.topk(torch.from_numpy(logits).double(), k, dim=1)
    assert np.array_equal(r["ids"], ids.numpy())
    wref = torch.softmax(vals, dim=1).numpy()
    assert np.max(np.abs(r["w"] - wref)) <= 2 ** -23
    assert np.allclose(r["w"].astype(np.float64).sum(1), 1.0, atol=1e-6)
    # grouping invariants
    assert r["counts"].sum() == T * k
    assert np.array_equal(r["counts"], np.bincount(r["ids"].ravel(), minlength=E))
    assert r["offsets"][0] == 0 and r["offsets"][-1] == T * k
    assert np.all(np.diff(r["offsets"]) == r["counts"])
    row = r["row"].ravel()
    assert np.array_equal(np.sort(row), np.arange(T * k))             # bijection
    assert np.array_equal(r["src"][row], np.repeat(np.arange(T), k))   # src inverts row
    for e in range(E):                                                 # stable group order
        toks = r["src"][r["offsets"][e]:r["offsets"][e + 1]]
        assert np.all(np.diff(toks) > 0)
        assert np.all((r["ids"][toks] == e).any(1))


def test_route_ties_go_to_lower_expert_index():
    logits = np.zeros((3, 10), np.float32)
    logits[1, [2, 7]] = 1.0
    logits[2] = np.array([0, 1, 1, 1, 0, 0, 0, 0, 0, 1], np.float32)
    r = oracle.route(logits, 4)
    assert r["ids"][0].tolist() == [0, 1, 2, 3]
    assert r["ids"][1].tolist() == [2, 7, 0, 1]
    assert r["ids"][2].tolist() == [1, 2, 3, 9]
    assert np.allclose(r["w"][0], 0.25)


# ---------------------------------------------------------------------------
# q8_1
# ---------------------------------------------------------------------------

# Blocks whose d is exact (amax = 127 * 2^j), so the expected codes follow by
# hand from the q8_1 definition: d = max|h|/127, q = round-half-away(h/d).
Q8_1_HAND_CASES = [
    ([127.0, -63.5, 63.5, 0.5, -0.5, 1.5, -2.5, 2.25] + [0.0] * 24,
     [127, -64, 64, 1, -1, 2, -3, 2] + [0] * 24, 1.0),
    ([-254.0, 3.0, -1.0, 5.0, 1.0, 0.75, -0.75, 253.0] + [0.0] * 24,   # 253/2 = 126.5 -> 127
     [-127, 2, -1, 3, 1, 0, 0, 127] + [0] * 24, 2.0),
    ([2.0, -2.0, 6.0, -508.0, 10.0, -10.0] + [0.0] * 26,
     [1, -1, 2, -127, 3, -3] + [0] * 26, 4.0),
    ([0.0] * 32, [0] * 32, 0.0),
]


@pytest.mark.parametrize("h,q,d", Q8_1_HAND_CASES)
def test_q8_1_hand_derived_blocks(h, q, d):
    gq, gd, gs = oracle.q8_1_block(np.array(h, np.float32))
    assert gq.tolist() == q
    assert gd == int(np.float16(d).view(np.uint16))
    assert gs == int(np.float16(d * sum(q)).view(np.uint16))


def test_q8_1_invariants_on_random_blocks():
    rng = np.random.default_rng(5)
    for i in range(400):
        h = (rng.standard_normal(32) * 10 ** rng.uniform(-3, 3)).astype(np.float32)
        if i % 50 == 0:
            h[rng.integers(0, 32, 20)] = 0
        q, d16, s16 = oracle.q8_1_block(h)
        amax = np.max(np.abs(h))
        d = np.float32(amax) / np.float32(127.0)
        assert np.max(np.abs(q.astype(int))) == 127
        assert np.all(np.abs(h.astype(np.float64) - q * np.float64(d)) <= np.float64(d) / 2 * (1 + 2 ** -20))
        df = float(np.uint16(d16).view(np.float16))
        sf = float(np.uint16(s16).view(np.float16))
        tot = int(q.astype(int).sum())
        assert abs(sf - df * tot) <= 2 ** -10 * abs(df * tot) + 2 ** -24 + abs(float(d) - df) * abs(tot)
        assert abs(df - float(d)) <= 2 ** -11 * float(d) + 2 ** -25   # fp16 subnormal quantum is 2^-24


# ---------------------------------------------------------------------------
# expert stage steps
# ---------------------------------------------------------------------------

def _tiny_moe(T=24, D=64, F=64, E=6, k=2, seed=21, zipf=0.0):
    return wl.gen_moe(T, D, F, E, k, 1.0 / 128, zipf, seed=seed)


def test_gate_up_h_matches_torch_composition():
    g = _tiny_moe()
    r = oracle.route(g["logits"], 2)
    rows = np.arange(0, 48, 5, dtype=np.int32)
    out = oracle.moe_gate_up_q8_1(g["X"], g["Wgu_c"], g["Wgu_s"], g["gu_scale2"], r["offsets"], r["src"],
                                  rows, want_h=True)
    F = 64
    xf = torch.from_numpy(bf16_torch(g["X"]))
    for i, rr in enumerate(rows):
        e = int(np.searchsorted(r["offsets"], rr, side="right") - 1)
        Wf = torch.from_numpy(w4_dequant_independent(g["Wgu_c"][e], g["Wgu_s"][e]))
        y = (xf[r["src"][rr]] @ Wf.T) * float(g["gu_scale2"][e])
        g32, u32 = y[:F].float().double(), y[F:].float().double()
        h = (torch.nn.functional.silu(g32) * u32).float().numpy()
        assert np.array_equal(out["h"][i], h)
        for b in range(F // 32):
            q, d, s = oracle.q8_1_block(h[b * 32:(b + 1) * 32])
            assert np.array_equal(out["Hq"][i, b * 32:(b + 1) * 32], q)
            assert out["Hd"][i, b] == d and out["Hs"][i, b] == s


def test_down_iq4_matches_dequantised_torch_matmul():
    rng = np.random.default_rng(8)
    n, F, D, E = 11, 96, 40, 3
    Hq = rng.integers(-127, 128, size=(n, F)).astype(np.int8)
    Hd = (rng.uniform(2 ** -8, 2 ** -4, size=(n, F // 32))).astype(np.float16).view(np.uint16)
    idx = rng.integers(0, 256, size=(E, D, F // 2), dtype=np.uint8)
    Ws = rng.uniform(2 ** -12, 2 ** -10, size=(E, D, F // 32)).astype(np.float16).view(np.uint16)
    offsets = np.array([0, 4, 4, n], np.int32)                 # expert 1 empty
    rows = np.arange(n, dtype=np.int32)
    Y = oracle.moe_down_iq4(Hq, Hd, offsets, rows, idx, Ws)
    cb = iq4_codebook_golden()
    A = Hq.astype(np.float64) * np.repeat(Hd.view(np.float16).astype(np.float64), 32, axis=1)
    for i in range(n):
        e = 0 if i < 4 else 2
        codes = np.empty((D, F), np.int64)
        codes[:, 0::2] = idx[e] & 15
        codes[:, 1::2] = idx[e] >> 4
        B = cb[codes] * np.repeat(Ws[e].view(np.float16).astype(np.float64), 32, axis=1)
        ref = (torch.from_numpy(A[i:i + 1]) @ torch.from_numpy(B).T).numpy()[0]
        assert np.max(np.abs(Y[i] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_combine_matches_einsum():
    rng = np.random.default_rng(4)
    w = rng.random((6, 3)).astype(np.float32)
    Ys = rng.standard_normal((18, 10))
    slot = rng.permutation(18).reshape(6, 3).astype(np.int32)
    Y = oracle.moe_combine(w, slot, Ys)
    ref = np.einsum("tj,tjd->td", w.astype(np.float64), Ys[slot])
    assert np.max(np.abs(Y - ref)) <= 1e-14


def test_expert_stage_one_expert_k1_reduces_to_dense_chain():
    """E = 1, k = 1: every token routes to expert 0 with weight 1, so the stage
    is dense gate/up -> SwiGLU -> q8_1 -> down on X in token order."""
    g = wl.gen_moe(9, 64, 64, 1, 1, 1.0 / 128, 0.0, seed=2)
    st = oracle.moe_expert_stage(g["X"], g["logits"], g["Wgu_c"], g["Wgu_s"], g["gu_scale2"],
                                 g["Wd_idx"], g["Wd_s"], k=1)
    assert np.all(st["route"]["w"] == 1.0) and np.array_equal(st["route"]["src"], np.arange(9))
    Wg = w4_dequant_independent(g["Wgu_c"][0], g["Wgu_s"][0])
    y = (bf16_torch(g["X"]) @ Wg.T) * float(g["gu_scale2"][0])
    h = (torch.nn.functional.silu(torch.from_numpy(y[:, :64]).float().double())
         * torch.from_numpy(y[:, 64:]).float().double()).float().numpy()
    cb = iq4_codebook_golden()
    codes = np.empty((64, 64), np.int64)
    codes[:, 0::2] = g["Wd_idx"][0] & 15
    codes[:, 1::2] = g["Wd_idx"][0] >> 4
    B = cb[codes] * np.repeat(g["Wd_s"][0].view(np.float16).astype(np.float64), 32, axis=1)
    for t in range(9):
        qs, ds = [], []
        for b in range(2):
            q, d, _ = oracle.q8_1_block(h[t, b * 32:(b + 1) * 32])
            qs.append(q.astype(np.float64) * float(np.uint16(d).view(np.float16)))
        ref = np.concatenate(qs) @ B.T
        assert np.max(np.abs(st["Y"][t] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_expert_stage_invariant_under_expert_relabeling():
    g = _tiny_moe(T=16, E=5, k=2, seed=33)
    perm = np.array([3, 0, 4, 1, 2])                 # new expert i is old expert perm[i]
    st = oracle.moe_expert_stage(g["X"], g["logits"], g["Wgu_c"], g["Wgu_s"], g["gu_scale2"],
                                 g["Wd_idx"], g["Wd_s"], k=2)
    st2 = oracle.moe_expert_stage(g["X"], g["logits"][:, perm], g["Wgu_c"][perm], g["Wgu_s"][perm],
                                  g["gu_scale2"][perm], g["Wd_idx"][perm], g["Wd_s"][perm], k=2)
    # same experts chosen (up to relabelling), so every token sums the same terms;
    # only the combine order can differ where the slot order differs
    assert np.max(np.abs(st["Y"] - st2["Y"])) <= 1e-9 * np.max(np.abs(st["Y"]))


def test_expert_stage_token_sampling_matches_full_run():
    g = _tiny_moe(T=20, seed=44)
    full = oracle.moe_expert_stage(g["X"], g["logits"], g["Wgu_c"], g["Wgu_s"], g["gu_scale2"],
                                   g["Wd_idx"], g["Wd_s"], k=2)
    toks = np.array([19, 3, 0])
    part = oracle.moe_expert_stage(g["X"], g["logits"], g["Wgu_c"], g["Wgu_s"], g["gu_scale2"],
                                   g["Wd_idx"], g["Wd_s"], k=2, tokens=toks)
    assert np.array_equal(part["Y"], full["Y"][toks])


# ---------------------------------------------------------------------------
# synthetic inputs
# ---------------------------------------------------------------------------

def test_synthetic_inputs_are_seeded_and_follow_the_stated_distributions():
    a = wl.gen_w4a16(64, 512, 512, 1 / 64, seed=0)
    b = wl.gen_w4a16(64, 512, 512, 1 / 64, seed=0)
    for key in ("X", "Wc", "Ws"):
        assert np.array_equal(a[key], b[key])
    e = a["Ws"] >> 3
    m = a["Ws"] & 7
    assert e.min() == 4 and e.max() == 10 and m.min() == 0 and m.max() == 7
    codes = np.concatenate([(a["Wc"] & 15).ravel(), (a["Wc"] >> 4).ravel()])
    assert np.all(np.bincount(codes, minlength=16) > 0.8 * codes.size / 16)
    x = bf16_torch(a["X"])
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    f = wl.gen_fp8_blk128(8, 256, 128, seed=2)
    wv = e4m3_torch(f["W"])
    assert np.all(np.abs(wv) <= 448) and not np.any(np.isnan(wv))
    assert f["S"].min() >= 2 ** -8 and f["S"].max() <= 2 ** -6
    g = wl.gen_moe(64, 64, 64, 16, 8, 1 / 128, 1.1, seed=4)
    assert g["logits"].dtype == np.float32 and g["logits"].shape == (64, 16)
    ws = g["Wd_s"].view(np.float16).astype(np.float64)
    assert ws.min() >= 2 ** -12 and ws.max() <= 2 ** -10


# ------------------------------------------------ dense Q8_0 x q8_1 (next row)

def test_q8_0_q8_1_unit_scales_is_exact_integer_matmul():
    """d = 1 on both sides: the projection is the plain integer matrix product."""
    g = wl.gen_q8_0_q8_1(9, 96, 7, seed=41)
    one = np.float16(1.0).view(np.uint16)
    Xd = np.full_like(g["Xd"], one)
    Wd = np.full_like(g["Wd"], one)
    Y = oracle.q8_0_q8_1(g["Xq"], Xd, g["Wq"], Wd)
    ref = g["Xq"].astype(np.int64) @ g["Wq"].astype(np.int64).T
    assert np.array_equal(Y, ref.astype(np.float64))


def test_q8_0_q8_1_matches_dequantised_torch_matmul():
    g = wl.gen_q8_0_q8_1(13, 160, 21, seed=42)
    Y = oracle.q8_0_q8_1(g["Xq"], g["Xd"], g["Wq"], g["Wd"])
    A = g["Xq"].astype(np.float64) * np.repeat(g["Xd"].view(np.float16).astype(np.float64), 32, axis=1)
    B = g["Wq"].astype(np.float64) * np.repeat(g["Wd"].view(np.float16).astype(np.float64), 32, axis=1)
    ref = (torch.from_numpy(A) @ torch.from_numpy(B).T).numpy()
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_q8_0_q8_1_single_code_selects_one_block():
    """One non-zero weight code picks one column, scaled by its two block scales."""
    g = wl.gen_q8_0_q8_1(5, 128, 6, seed=43)
    Wq = np.zeros_like(g["Wq"])
    n0, k0 = 4, 77
    Wq[n0, k0] = -3
    Y = oracle.q8_0_q8_1(g["Xq"], g["Xd"], Wq, g["Wd"])
    f16 = lambda a: a.view(np.float16).astype(np.float64)  # noqa: E731
    want = f16(g["Xd"][:, k0 // 32]) * f16(g["Wd"][n0, k0 // 32]) * g["Xq"][:, k0].astype(np.float64) * -3
    assert np.array_equal(Y[:, n0], want)
    assert not np.any(np.delete(Y, n0, axis=1))


def test_q8_0_q8_1_sampling_and_requant_compose():
    """Row / column sampling equals the full run; the q8_1 output is the q8_1
    rounding of each row's fp32 values per 32 columns, with its invariants."""
    g = wl.gen_q8_0_q8_1(6, 96, 64, seed=44)
    full = oracle.q8_0_q8_1(g["Xq"], g["Xd"], g["Wq"], g["Wd"])
    rows, cols = np.array([5, 0, 3]), np.array([63, 1, 32, 31])
    part = oracle.q8_0_q8_1(g["Xq"], g["Xd"], g["Wq"], g["Wd"], rows=rows, cols=cols)
    assert np.array_equal(part, full[np.ix_(rows, cols)])
    r = oracle.q8_0_q8_1_requant(g["Xq"], g["Xd"], g["Wq"], g["Wd"])
    assert np.array_equal(r["Y"], full)
    for i in range(6):
        for b in range(2):
            q, d, s = oracle.q8_1_block(full[i, b * 32:(b + 1) * 32].astype(np.float32))
            assert np.array_equal(r["Yq"][i, b * 32:(b + 1) * 32], q)
            assert r["Yd"][i, b] == d and r["Ys"][i, b] == s
            assert np.max(np.abs(q.astype(int))) == 127
