"""The CUDA expansion tables checked against the formats they encode (CPU only).

The down product expands IQ4_NL indices to f16 with byte permutes into two
tables: the low and the high byte of the f16 value of each codebook entry, four
entries per 32-bit word (csrc/qgemm.cuh, kIq4L*/kIq4H*). This test reads those
constants from the source and checks that they reassemble, entry by entry, into
the f16 values of the IQ4_NL codebook fixture ("Run Edge0-145B Q3_K on AMD HIP
(Linux, gfx1100)", commit 4cb5224: the down weights are 4-bit indices into it),
and that the permute-based expansion, emulated here bit by bit, gives those
values for every combination of four indices.
"""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "block_quantized_weight_route_gb300", "csrc", "qgemm.cuh")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "iq4nl_codebook.txt")


def codebook():
    with open(GOLDEN) as f:
        vals = [int(t) for ln in f if not ln.startswith("#") for t in ln.split()]
    assert len(vals) == 16
    return vals


def table_words(prefix):
    src = open(SRC).read()
    words = []
    for i in range(4):
        m = re.search(r"%s%d\s*=\s*0x([0-9A-Fa-f]+)u" % (prefix, i), src)
        assert m, f"{prefix}{i} not found"
        words.append(int(m.group(1), 16))
    return words


def table_bytes(words):
    return [(words[e >> 2] >> (8 * (e & 3))) & 0xFF for e in range(16)]


def test_iq4_tables_are_the_codebook_in_f16():
    lo, hi = table_bytes(table_words("kIq4L")), table_bytes(table_words("kIq4H"))
    for e, v in enumerate(codebook()):
        bits = lo[e] | (hi[e] << 8)
        assert np.uint16(bits).view(np.float16) == np.float16(v), e
        assert float(np.float16(v)) == v          # every entry is exact in f16


def prmt(a, b, c):
    """PTX prmt.b32 (default mode): byte i of the result is byte (c_i & 7) of
    {b:a}, or that byte's sign replicated when c_i & 8."""
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    r = 0
    for i in range(4):
        sel = (c >> (4 * i)) & 0xF
        byte = src[sel & 7]
        if sel & 8:
            byte = 0xFF if byte & 0x80 else 0
        r |= byte << (8 * i)
    return r


def test_iq4_permute_expansion_every_index_quadruple():
    L, H = table_words("kIq4L"), table_words("kIq4H")
    f16 = [int(np.float16(v).view(np.uint16)) for v in codebook()]
    sel = lambda a, b, m: (a & ~m & 0xFFFFFFFF) | (b & m)    # lop3 0xD8: m ? b : a
    for x in range(1 << 16):                                  # four 4-bit indices
        m = prmt((x << 4) & 0xFFFFFFFF, x, 0xD9C8)
        lo = sel(prmt(L[0], L[1], x), prmt(L[2], L[3], x & 0x7777), m)
        hi = sel(prmt(H[0], H[1], x), prmt(H[2], H[3], x & 0x7777), m)
        n = [(x >> (4 * i)) & 15 for i in range(4)]
        assert prmt(lo, hi, 0x5140) == f16[n[0]] | (f16[n[1]] << 16)
        assert prmt(lo, hi, 0x7362) == f16[n[2]] | (f16[n[3]] << 16)
