"""GPU parity of every GEMM kernel variant.

The library picks a kernel per call: a persistent single-CTA kernel, a
persistent SM-pair kernel (tcgen05 cta_group::2) with two or three 64-wide
k-tiles per pipeline stage, and a split-K cluster kernel for either, depending
on the shape. The tuning overrides TPGQA_PAIR, TPGQA_KSUB and TPGQA_SPLIT force
one variant, so each variant here reruns the linear-layer and
MLP parity tests in a child process with the override set.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = ["tests/test_gpu_linear.py",
         "tests/test_gpu_blocks.py::test_gate_up_swiglu_matches_oracle_h",
         "tests/test_gpu_blocks.py::test_mlp_block_small_ragged"]


@pytest.mark.parametrize("pair,split,ksub", [("0", "1", "2"), ("1", "1", "2"), ("1", "1", "3"),
                                             ("0", "2", "2"), ("0", "4", "2"), ("1", "2", "2"),
                                             ("1", "4", "2")])
def test_kernel_variant_parity(pair, split, ksub):
    from gpu_util import need_gpu
    need_gpu()
    env = dict(os.environ, TPGQA_PAIR=pair, TPGQA_SPLIT=split, TPGQA_KSUB=ksub)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        *TESTS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
