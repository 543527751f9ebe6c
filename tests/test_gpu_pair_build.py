"""The CTA-pair (cta_group::2) form of the dense W4A16, FP8 block-128 and gate/up
GEMMs, a compile-time option (-DQMM_PAIR=1) that the default build leaves off:
built into a temporary directory and put through the parity tests of those
products and of the expert stage in a separate process (QMM_GB300_LIB points it
at the variant)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cta_pair_form_passes_the_parity_tests(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_weight_route_gb300.build import build_variant
    lib = build_variant(["-DQMM_PAIR=1"], str(tmp_path / "pair"))
    env = dict(os.environ, QMM_GB300_LIB=lib)
    sel = ("w4a16 or fp8 or router or expert_stage_small or ragged_groups or k_equals_e or t5268 or shape_limits "
           "or single_token")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert " passed" in r.stdout
