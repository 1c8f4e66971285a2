"""GPU parity of every GEMM kernel variant.

The library picks a kernel per call: a persistent single-CTA kernel, a
persistent SM-pair kernel (tcgen05 cta_group::2) with two or three 64-wide
k-tiles per pipeline stage, and a split-K cluster kernel for either, depending
on the shape. The SM-pair kernels fetch each stage with one 3-D TMA copy per
operand when every K is a multiple of 64, else with one 2-D copy per k-tile.
Split-K reduces the splits' partials through the cluster's shared memory in a
fixed order. The persistent SM-pair kernel runs 256-, 224- or 128-column tiles
(and 448- and 512-column SwiGLU tiles: half gate, half up columns), the single-CTA
kernel 128- to 256-column ones. The tuning overrides TPGQA_PAIR,
TPGQA_KSUB, TPGQA_SPLIT, TPGQA_TMA3D, TPGQA_PAIR_BN and TPGQA_BN force one
variant, so each variant here reruns the linear-layer and MLP parity tests in a
child process with the override set.
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


@pytest.mark.parametrize("pair,split,ksub,tma3d,pair_bn,bn", [
    ("0", "1", "2", "1", "256", "256"), ("0", "1", "2", "1", "256", "224"), ("0", "1", "2", "1", "256", "192"),
    ("0", "1", "2", "1", "256", "128"), ("1", "1", "2", "1", "256", "256"), ("1", "1", "3", "1", "256", "256"),
    ("1", "1", "2", "0", "256", "256"), ("1", "1", "3", "0", "256", "256"), ("1", "1", "2", "1", "224", "256"),
    ("1", "1", "2", "0", "224", "256"), ("0", "2", "2", "1", "256", "256"), ("0", "4", "2", "1", "256", "256"),
    ("1", "2", "2", "1", "256", "256"), ("1", "4", "2", "1", "256", "256"), ("1", "2", "2", "0", "256", "256"),
    ("1", "1", "2", "1", "128", "256"), ("1", "1", "2", "0", "128", "256"), ("1", "1", "2", "1", "512", "256"),
    ("1", "1", "2", "1", "448", "256")])
def test_kernel_variant_parity(pair, split, ksub, tma3d, pair_bn, bn):
    from gpu_util import need_gpu
    need_gpu()
    env = dict(os.environ, TPGQA_PAIR=pair, TPGQA_SPLIT=split, TPGQA_KSUB=ksub, TPGQA_TMA3D=tma3d,
               TPGQA_PAIR_BN=pair_bn, TPGQA_BN=bn)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        *TESTS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


# Runs row-parallel GEMMs that split K three times each and checks that the
# fp32 outputs are the same bits every time: ragged shapes (partial last row and
# column tiles) on the SM-pair and the single-CTA kernels.
_REPEAT = r"""
import sys
sys.path.insert(0, "tests")
import numpy as np, torch
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import dev_bf16
for T, per, nout, n in [(200, 1024, 264, 2), (70, 2048, 520, 4), (512, 2048, 1024, 2)]:
    x = inputs.normal_bf16(61, 0, (T, n * per))
    w = inputs.normal_bf16(61, 1, (nout, n * per), 0.02)
    xs = [dev_bf16(x[:, r * per:(r + 1) * per]) for r in range(n)]
    ws = [dev_bf16(w[:, r * per:(r + 1) * per]) for r in range(n)]
    first = None
    for rep in range(3):
        ys = [torch.full((T, nout), float("nan"), device="cuda") for _ in range(n)]
        tp.tp_row_linear(n, xs, ws, ys, tp.TP_COMBINE_NONE)
        got = np.stack([y.cpu().numpy() for y in ys]).view(np.uint32)
        if first is None:
            first = got
        assert np.array_equal(got, first), (T, per, nout, n, rep)
assert tp.tp_device_status() == (tp.TP_OK, 0)
print("ok")
"""


@pytest.mark.parametrize("split", ["2", "4"])
def test_split_k_reduction_is_deterministic(split):
    """The splits' partials are added in split order 0..S-1 whatever order the
    CTAs finish in, so repeated runs give the same bits."""
    from gpu_util import need_gpu
    need_gpu()
    env = dict(os.environ, TPGQA_SPLIT=split)
    r = subprocess.run([sys.executable, "-c", _REPEAT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("pair_bn", ["448", "512"])
def test_wide_swiglu_tiles_with_block_tables(pair_bn):
    """The MoE block's gate/up GEMM takes each tile's expert weights through a
    block table; with the wide SwiGLU tiles forced, every gate and up row of a
    tile comes from its expert's slot. Reruns the MoE parity tests in a child
    process with TPGQA_PAIR_BN set."""
    from gpu_util import need_gpu
    need_gpu()
    env = dict(os.environ, TPGQA_PAIR_BN=pair_bn)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        "tests/test_gpu_moe.py::test_moe_block_matches_the_oracle"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
