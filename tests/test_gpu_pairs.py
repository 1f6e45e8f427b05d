"""The grouped GEMMs with two-CTA clusters (one M = 256 MMA over two SMs) on
every grouped kind, and with none: the kernel-level emulation cases, the
layer parity cases and the fused forward's cases pass either way. The library reads MOE_GEMM_PAIRS once per
process, so each setting runs in a child pytest."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pairs", ["1", "0"])
def test_parity_with_and_without_cta_pairs(pairs):
    env = dict(os.environ, MOE_GEMM_PAIRS=pairs)
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         "tests/test_gpu_kernels_vs_emulation.py", "tests/test_gpu_parity.py",
         "tests/test_gpu_fused.py::test_fused_forward_parity"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
