"""Workload definitions and seeded input generators.

Random words come from a counter-based SplitMix64 stream (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): word i
of stream s under seed S is mix64(key(S, s) + (i + 1) * GOLDEN), where mix64 is
the SplitMix64 finaliser.  Uniform reals take the top 53 bits; normals use the
Box-Muller transform.  Everything is vectorised numpy, so the same seed gives
the same bytes on any host and any numpy version.

Float rounding of drawn values to the storage types (bf16, fp16, E4M3) is done
by library conversions (torch / numpy), never by code in this repository.

The workloads follow the prompt-length and projection shapes the pages measure
("Run Edge0-145B Q3_K on AMD HIP (Linux, gfx1100)", "Measured on Linux": 5.3K
and 21K-token prompts; "perf: strix-hip BF16 GEMMs via hipBLASLt", commit "f16a
twins": M=2048 prefill GEMMs).  Weights are random, not trained.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = _mix64(np.array([(seed * 0x100000001B3 + stream * 0x1F123BB5) & 0xFFFFFFFFFFFFFFFF],
                            dtype=np.uint64))
    return k[0]


def words(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n uint64 words of stream `stream` under `seed`, starting at counter `offset`."""
    key = _key(seed, stream)
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + i * _GOLDEN)


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n float64 uniforms in [0, 1)."""
    return (words(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """n float64 standard normals (Box-Muller on pairs of uniforms)."""
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    u1 = 1.0 - u[0::2]                      # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return z[:n]


def random_bytes(seed: int, stream: int, nbytes: int) -> np.ndarray:
    """nbytes uniformly random bytes (both nibbles of each byte uniform over 16 codes)."""
    nw = (nbytes + 7) // 8
    return words(seed, stream, nw).view(np.uint8)[:nbytes].copy()


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _scale_bytes(seed: int, stream: int, n: int) -> np.ndarray:
    """E4M3 scale bytes with exponent field uniform in 4..10 and mantissa uniform in 0..7."""
    w = words(seed, stream, n)
    e = np.uint64(4) + (((w >> np.uint64(32)) * np.uint64(7)) >> np.uint64(32))
    m = w & np.uint64(7)
    return ((e << np.uint64(3)) | m).astype(np.uint8)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "w4a16" | "fp8_blk128" | "moe"
    seed: int
    M: int = 0
    K: int = 0
    N: int = 0
    scale2: float = 1.0
    out: str = "f32"          # dense output type: "f32" | "bf16"
    T: int = 0
    D: int = 0
    F: int = 0
    E: int = 0
    k: int = 0
    gu_scale2: float = 1.0
    zipf_s: float = 0.0       # 0: uniform expert popularity

    def flops(self) -> float:
        if self.kind in ("w4a16", "fp8_blk128"):
            return 2.0 * self.M * self.N * self.K
        rows = self.T * self.k
        return 2.0 * rows * self.D * 2 * self.F + 2.0 * rows * self.F * self.D


# The workloads the path is measured and checked on.  Sizes and value
# distributions are the problem statement's; seeds are the workload's index.
WORKLOADS = {
    "w4a16_m64_k512_n512": Workload(
        name="w4a16_m64_k512_n512", kind="w4a16", seed=0, M=64, K=512, N=512,
        scale2=1.0 / 64, out="f32"),
    "w4a16_m2048_k5120_n17408": Workload(
        name="w4a16_m2048_k5120_n17408", kind="w4a16", seed=1, M=2048, K=5120, N=17408,
        scale2=1.0 / 256, out="bf16"),
    "fp8blk128_m2048_k5120_n5120": Workload(
        name="fp8blk128_m2048_k5120_n5120", kind="fp8_blk128", seed=2, M=2048, K=5120, N=5120,
        out="bf16"),
    "moe_t5268_d2048_f768_e128_k8": Workload(
        name="moe_t5268_d2048_f768_e128_k8", kind="moe", seed=3, T=5268, D=2048, F=768,
        E=128, k=8, gu_scale2=1.0 / 128),
    "moe_t21504_d2560_f1024_e256_k8_zipf": Workload(
        name="moe_t21504_d2560_f1024_e256_k8_zipf", kind="moe", seed=4, T=21504, D=2560,
        F=1024, E=256, k=8, gu_scale2=1.0 / 128, zipf_s=1.1),
    # the router projection in front of routing (logits = X . W_r^T, one row per
    # expert), at the router shape of the sources' W4A16 measurements; fp32 logits
    "w4a16_router_m2048_k2560_n512": Workload(
        name="w4a16_router_m2048_k2560_n512", kind="w4a16", seed=5, M=2048, K=2560, N=512,
        scale2=1.0 / 64, out="f32"),
}


def gen_w4a16(M: int, K: int, N: int, scale2: float, seed: int) -> dict:
    """X bf16 ~N(0,1) [M,K]; W codes [N, K/2] (element 2j in the low nibble of
    byte j); E4M3 scale bytes [N, K/16]; fp32 scale2."""
    X = _to_bf16_bits(normal(seed, 1, M * K).reshape(M, K))
    Wc = random_bytes(seed, 2, N * K // 2).reshape(N, K // 2)
    Ws = _scale_bytes(seed, 3, N * K // 16).reshape(N, K // 16)
    return dict(X=X, Wc=Wc, Ws=Ws, scale2=np.float32(scale2))


def gen_fp8_blk128(M: int, K: int, N: int, seed: int) -> dict:
    """X bf16 ~N(0,1) [M,K]; W = E4M3(RNE(8*N(0,1))) saturated at +-448, [N,K];
    one fp32 scale per 128x128 block, uniform in [2^-8, 2^-6]."""
    X = _to_bf16_bits(normal(seed, 1, M * K).reshape(M, K))
    w = np.clip(8.0 * normal(seed, 2, N * K), -448.0, 448.0).astype(np.float32)
    W = _to_e4m3_bits(w).reshape(N, K)
    u = uniform(seed, 3, (N // 128) * (K // 128))
    S = (2.0 ** -8 + u * (2.0 ** -6 - 2.0 ** -8)).astype(np.float32).reshape(N // 128, K // 128)
    return dict(X=X, W=W, S=S)


def gen_moe(T: int, D: int, F: int, E: int, k: int, gu_scale2: float, zipf_s: float,
            seed: int) -> dict:
    """Routed expert-stage inputs.

    logits fp32 [T,E] = 2*N(0,1) (+ ln p_e for Zipf popularity p_e ~ (e+1)^-s);
    X bf16 ~N(0,1) [T,D]; gate/up W4 codes [E, 2F, D/2] (rows 0..F-1 gate,
    F..2F-1 up) with E4M3 scale bytes [E, 2F, D/16] and fp32 scale2 per expert;
    down IQ4_NL indices [E, D, F/2] and fp16 scale bits [E, D, F/32] uniform in
    [2^-12, 2^-10]."""
    X = _to_bf16_bits(normal(seed, 1, T * D).reshape(T, D))
    logits = 2.0 * normal(seed, 2, T * E).reshape(T, E)
    if zipf_s:
        p = np.arange(1, E + 1, dtype=np.float64) ** (-zipf_s)
        logits = logits + np.log(p / p.sum())[None, :]
    logits = logits.astype(np.float32)
    Wgu_c = random_bytes(seed, 3, E * 2 * F * D // 2).reshape(E, 2 * F, D // 2)
    Wgu_s = _scale_bytes(seed, 4, E * 2 * F * D // 16).reshape(E, 2 * F, D // 16)
    gu_s2 = np.full(E, gu_scale2, dtype=np.float32)
    Wd_idx = random_bytes(seed, 5, E * D * F // 2).reshape(E, D, F // 2)
    u = uniform(seed, 6, E * D * F // 32)
    Wd_s = (2.0 ** -12 + u * (2.0 ** -10 - 2.0 ** -12)).astype(np.float16)
    Wd_s = Wd_s.view(np.uint16).reshape(E, D, F // 32)
    return dict(X=X, logits=logits, Wgu_c=Wgu_c, Wgu_s=Wgu_s, gu_scale2=gu_s2,
                Wd_idx=Wd_idx, Wd_s=Wd_s)


def gen_q8_0_q8_1(M: int, K: int, N: int, seed: int) -> dict:
    """Dense Q8_0 x q8_1 inputs, codes drawn directly: activation codes Xq int8
    uniform in [-127, 127] [M,K] with fp16 d bits [M,K/32] uniform in
    [2^-10, 2^-4]; weight codes Wq int8 uniform in [-127, 127] [N,K] with fp16
    scale bits [N,K/32] uniform in [2^-12, 2^-8]."""
    Xq = ((random_bytes(seed, 1, M * K).astype(np.int16) % 255) - 127).astype(np.int8).reshape(M, K)
    Xd = (2.0 ** -10 + uniform(seed, 2, M * K // 32) * (2.0 ** -4 - 2.0 ** -10)).astype(np.float16)
    Wq = ((random_bytes(seed, 3, N * K).astype(np.int16) % 255) - 127).astype(np.int8).reshape(N, K)
    Wd = (2.0 ** -12 + uniform(seed, 4, N * K // 32) * (2.0 ** -8 - 2.0 ** -12)).astype(np.float16)
    return dict(Xq=Xq, Xd=Xd.view(np.uint16).reshape(M, K // 32), Wq=Wq,
                Wd=Wd.view(np.uint16).reshape(N, K // 32))


def generate(w: Workload) -> dict:
    if w.kind == "w4a16":
        return gen_w4a16(w.M, w.K, w.N, w.scale2, w.seed)
    if w.kind == "fp8_blk128":
        return gen_fp8_blk128(w.M, w.K, w.N, w.seed)
    if w.kind == "moe":
        return gen_moe(w.T, w.D, w.F, w.E, w.k, w.gu_scale2, w.zipf_s, w.seed)
    raise ValueError(w.kind)
