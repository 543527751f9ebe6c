"""Toolchain facts the design rests on, checked with nvcc (no GPU needed).

The down product and the Q8_0 x q8_1 projection compute their exact per-32
integer block dots on the f16 tensor path (`tcgen05.mma kind::f16`, both
operands small integers exact in f16, fp32 sums below 2^24) because the int8
tensor path (`kind::i8`) is not available for sm_103a: ptxas rejects it there
while accepting it for sm_100a.
"""
import os
import shutil
import subprocess

import pytest

KIND_I8 = r'''
#include <cstdint>
__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::i8 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
'''


def _nvcc():
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    pytest.skip("nvcc not found")


def _compile(tmp_path, arch):
    src = tmp_path / "probe.cu"
    src.write_text(KIND_I8)
    r = subprocess.run([_nvcc(), "-gencode", f"arch=compute_{arch},code=sm_{arch}", "-c", str(src), "-o",
                        str(tmp_path / f"probe_{arch}.o")], capture_output=True, text=True)
    return r.returncode, r.stderr


def test_kind_i8_rejected_for_sm103a(tmp_path):
    rc, err = _compile(tmp_path, "103a")
    assert rc != 0
    assert "kind::i8" in err and "sm_103a" in err


def test_kind_i8_accepted_for_sm100a(tmp_path):
    rc, err = _compile(tmp_path, "100a")
    assert rc == 0, err
