"""The ring all-reduce folded into the row-parallel GEMM (mlxcel manual "텐서
병렬화", 통신 패턴: reduce-scatter then all-gather on the ring; chunk c is
reduced in the order c+1, c+2, ..., c).

Where every 256-row tile lies inside one ring chunk, tp_row_linear with
TP_COMBINE_RING_FUSED / RING_SHARED runs the ring-folding GEMM: each rank's
partial is computed from a zeroed accumulator exactly as the GEMM without a
combine computes it, and the partials are added in the chunk's ring order. The
result must therefore equal, bit for bit, the partials of TP_COMBINE_NONE
reduced by the one-pass ring (tp_allreduce_ring), and the step-by-step ring;
and it must match the fp64 oracle within the bf16 tolerance.
"""
import os

import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_bits_f32, host_f64, need_gpu

pytestmark = pytest.mark.gpu

# (tokens, ranks, output features, input features per rank): tiles inside one
# chunk (T/N a multiple of 256); ragged K (not a multiple of 64, odd k-tile
# counts), an output width that is not a multiple of the 256-column tile.
CASES = [
    (512, 2, 512, 256),
    (1024, 4, 768, 320),
    (2048, 8, 1000, 200),
    (2048, 4, 4096, 1024),   # the attention projection's o_proj shape
    # grids too small for one 256 x 256 tile per SM pair (the GEMM alone would
    # split K): the fold runs in the split-K pair kernel, one cluster split per
    # rank; with TPGQA_RANK_SPLIT=0 the GEMM splits K and the ring runs after it
    (512, 2, 2048, 4096),    # the T=512 MLP block's down projection
    (512, 2, 1000, 1000),
    (1024, 4, 264, 2048),
]
RANK_SPLIT = {(512, 2, 2048, 4096), (512, 2, 1000, 1000), (1024, 4, 264, 2048)}


@pytest.fixture(params=["0", "1"], ids=["rank_split_off", "rank_split"])
def rank_split(request, monkeypatch):
    monkeypatch.setenv("TPGQA_RANK_SPLIT", request.param)
    return request.param == "1"


def _torch():
    import torch
    return torch


def _layer(T, n, D, K, seed):
    x = [inputs.normal_bf16(seed, 40 + r, (T, K)) for r in range(n)]
    w = [inputs.normal_bf16(seed, 80 + r, (D, K), 0.05) for r in range(n)]
    return x, w


def _run(xd, wd, combine, env=None):
    torch = _torch()
    n = len(xd)
    T, D = xd[0].shape[0], wd[0].shape[0]
    ys = [torch.full((T, D), float("nan"), device="cuda") for _ in range(n)]
    old = os.environ.get("TPGQA_RING_EPILOGUE")
    try:
        if env is not None:
            os.environ["TPGQA_RING_EPILOGUE"] = env
        tp.tp_row_linear(n, xd, wd, ys, combine)
    finally:
        if env is not None:
            if old is None:
                del os.environ["TPGQA_RING_EPILOGUE"]
            else:
                os.environ["TPGQA_RING_EPILOGUE"] = old
    torch.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    return ys


@pytest.mark.parametrize("T,n,D,K", CASES)
def test_folded_ring_is_bit_identical_to_gemm_then_ring(T, n, D, K, rank_split):
    need_gpu()
    if rank_split and (T, n, D, K) not in RANK_SPLIT:
        pytest.skip("the rank-split setting changes nothing for this shape")
    x, w = _layer(T, n, D, K, seed=700 + T + n + D)
    xd = [dev_bf16(a) for a in x]
    wd = [dev_bf16(a) for a in w]
    # reference: partials of the GEMM without a combine, then the one-pass ring
    parts = _run(xd, wd, tp.TP_COMBINE_NONE)
    part_bits = [host_bits_f32(p) for p in parts]
    tp.tp_allreduce_ring(n, parts, tp.TP_RING_FUSED)
    _torch().cuda.synchronize()
    ref = host_bits_f32(parts[0])
    for p in parts[1:]:
        assert np.array_equal(host_bits_f32(p), ref)
    # the oracle's ring over the same f32 partials, in its own fold order
    oring = O.ring_all_reduce([b.view(np.float32).reshape(-1) for b in part_bits])
    assert np.array_equal(np.asarray(oring[0], dtype=np.float32).view(np.uint32).reshape(T, D), ref)
    # folded (default), and the same call with the fold turned off
    folded = _run(xd, wd, tp.TP_COMBINE_RING_FUSED)
    for r in range(n):
        assert np.array_equal(host_bits_f32(folded[r]), ref), f"rank {r}"
    unfolded = _run(xd, wd, tp.TP_COMBINE_RING_FUSED, env="0")
    for r in range(n):
        assert np.array_equal(host_bits_f32(unfolded[r]), ref), f"rank {r}, unfolded"
    shared = _run(xd, wd, tp.TP_COMBINE_RING_SHARED)
    assert np.array_equal(host_bits_f32(shared[0]), ref)
    steps = _run(xd, wd, tp.TP_COMBINE_RING)
    for r in range(n):
        assert np.array_equal(host_bits_f32(steps[r]), ref), f"rank {r}, step ring"
    # and the value against the fp64 definition: sum_r X_r W_r^T
    f = inputs.bf16_bits_to_f64
    exact = sum(O.linear(f(a), f(b)) for a, b in zip(x, w))
    assert_close(host_f64(folded[0]), exact, BF16_TOL, "folded sum")


def test_integer_inputs_give_the_exact_sum():
    """Small integers are exact in bf16 and every sum stays below 2^24, so the
    folded result equals the unsharded product exactly, whatever the order."""
    need_gpu()
    T, n, D, K = 1024, 4, 520, 192
    x = [inputs.small_int_bf16(77, 10 + r, (T, K), -3, 3) for r in range(n)]
    w = [inputs.small_int_bf16(77, 30 + r, (D, K), -3, 3) for r in range(n)]
    ys = _run([dev_bf16(a) for a in x], [dev_bf16(b) for b in w], tp.TP_COMBINE_RING_FUSED)
    f = inputs.bf16_bits_to_f64
    exact = O.linear(np.concatenate([f(a) for a in x], axis=1), np.concatenate([f(b) for b in w], axis=1))
    for y in ys:
        assert np.array_equal(host_f64(y), exact)


def test_consecutive_calls_and_other_buffers_unchanged():
    """Two calls in a row on new inputs give fresh results (no state carried in
    the kernel), and RING_SHARED writes y[0] only."""
    need_gpu()
    torch = _torch()
    T, n, D, K = 1024, 4, 512, 256
    for seed in (801, 802):
        x, w = _layer(T, n, D, K, seed)
        xd = [dev_bf16(a) for a in x]
        wd = [dev_bf16(a) for a in w]
        parts = _run(xd, wd, tp.TP_COMBINE_NONE)
        tp.tp_allreduce_ring(n, parts, tp.TP_RING_FUSED)
        ys = [torch.full((T, D), 7.0, device="cuda") for _ in range(n)]
        tp.tp_row_linear(n, xd, wd, ys, tp.TP_COMBINE_RING_SHARED)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits_f32(ys[0]), host_bits_f32(parts[0]))
        for y in ys[1:]:
            assert bool((y == 7.0).all())


@pytest.mark.parametrize("kind", ["decode", "decode_splitk", "pair", "fold"])
def test_early_weight_loads_change_no_bits(kind):
    """The GEMM kernels start their first weight (B) loads before the wait on the
    previous kernel; the arithmetic is unchanged, so every bit equals the run with
    TPGQA_EARLY_B=0 (all loads after the wait), for the single-CTA, split-K,
    SM-pair and ring-folding kernels."""
    need_gpu()
    torch = _torch()
    if kind == "decode":          # 64 tokens: single-CTA persistent kernel, 152 tiles
        T, n, D, K, combine = 64, 8, 4096, 512, tp.TP_COMBINE_NONE
    elif kind == "decode_splitk":  # few output tiles: split-K clusters
        T, n, D, K, combine = 64, 2, 512, 2048, tp.TP_COMBINE_NONE
    elif kind == "pair":
        T, n, D, K, combine = 640, 4, 1536, 384, tp.TP_COMBINE_NONE
    else:
        T, n, D, K, combine = 1024, 4, 768, 320, tp.TP_COMBINE_RING_FUSED
    x, w = _layer(T, n, D, K, seed=900 + T + D)
    xd = [dev_bf16(a) for a in x]
    wd = [dev_bf16(a) for a in w]
    outs = {}
    for env in ("0", "1"):
        old = os.environ.get("TPGQA_EARLY_B")
        os.environ["TPGQA_EARLY_B"] = env
        try:
            ys = [torch.full((T, D), float("nan"), device="cuda") for _ in range(n)]
            for _ in range(3):  # back to back, so the loads overlap the previous launch
                tp.tp_row_linear(n, xd, wd, ys, combine)
            torch.cuda.synchronize()
        finally:
            if old is None:
                del os.environ["TPGQA_EARLY_B"]
            else:
                os.environ["TPGQA_EARLY_B"] = old
        outs[env] = [host_bits_f32(y) for y in ys]
    for r in range(n):
        assert np.array_equal(outs["0"][r], outs["1"][r]), f"rank {r}"
    f = inputs.bf16_bits_to_f64
    assert_close(host_f64(ys[0]), O.linear(f(x[0]), f(w[0])) if combine == tp.TP_COMBINE_NONE else
                 sum(O.linear(f(a), f(b)) for a, b in zip(x, w)), BF16_TOL, "result")


@pytest.mark.parametrize("T,n,D,K", CASES)
def test_folded_ring_is_one_kernel_launch(T, n, D, K, rank_split):
    """With the fold the call is the GEMM alone; without it (TPGQA_RING_EPILOGUE=0,
    or a split-K shape with TPGQA_RANK_SPLIT=0) the GEMM and the one-pass ring."""
    need_gpu()
    folds = (T, n, D, K) not in RANK_SPLIT or rank_split
    if rank_split and (T, n, D, K) not in RANK_SPLIT:
        pytest.skip("the rank-split setting changes nothing for this shape")
    x, w = _layer(T, n, D, K, seed=900 + T + n + D)
    xd = [dev_bf16(a) for a in x]
    wd = [dev_bf16(a) for a in w]
    c0 = tp.tp_launch_count()
    _run(xd, wd, tp.TP_COMBINE_RING_FUSED)
    c1 = tp.tp_launch_count()
    _run(xd, wd, tp.TP_COMBINE_RING_FUSED, env="0")
    c2 = tp.tp_launch_count()
    assert c1 - c0 == (1 if folds else 2)
    assert c2 - c1 == 2
