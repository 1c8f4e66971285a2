"""GPU parity of the column- and row-parallel linear layers against the oracle.

bf16 inputs with fp32 accumulation: max|Y_gpu - Y_ref| <= 1e-2 * max|Y_ref|.
fp32 worked example: <= 1e-5 * max|Y_ref|. Small-integer inputs make every sum
exact, so there the GPU must equal the oracle exactly in every mode.
"""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import (BF16_TOL, F32_TOL, assert_close, dev_bf16, dev_f32, host_f64,
                      host_bits_f32, need_gpu)

pytestmark = pytest.mark.gpu
COMBINES = [tp.TP_COMBINE_NONE, tp.TP_COMBINE_FUSED, tp.TP_COMBINE_RING, tp.TP_COMBINE_RING_FUSED]


def torch():
    import torch as t
    return t


def _row_outputs(n, T, nout, combine):
    t = torch()
    k = 1 if combine == tp.TP_COMBINE_FUSED else n
    return [t.full((T, nout), float("nan"), device="cuda") for _ in range(k)]


def _check_row(ys, parts, combine, tol):
    ref = sum(parts)
    if combine == tp.TP_COMBINE_NONE:
        for y, p in zip(ys, parts):
            assert_close(host_f64(y), p, tol, "partial")
    else:
        for y in ys:
            assert_close(host_f64(y), ref, tol, "reduced")


# ---- fp32: the railscraft wiki's worked example ----------------------------------
def test_wiki_example_fp32_column_parallel():
    need_gpu()
    w = inputs.WORKLOADS["wiki_linear_fp32_tp2"]
    d = inputs.make_fp32_linear_inputs(w)
    n = w["tp"]
    x = dev_f32(d["x"])
    shards = O.split_rows(d["w"], n)
    wd = [dev_f32(s) for s in shards]
    t = torch()
    y = t.full((w["T"], w["d_out"]), float("nan"), device="cuda")
    tp.tp_column_linear(n, x, wd, [y], gather=True)
    ref = O.all_gather_columns(O.column_parallel(d["x"], shards))
    assert list(y.shape) == [32, 2048]
    assert_close(host_f64(y), ref, F32_TOL, "column gather")
    ys = [t.full((w["T"], w["d_out"] // n), float("nan"), device="cuda") for _ in range(n)]
    tp.tp_column_linear(n, x, wd, ys, gather=False)
    for r in range(n):
        assert_close(host_f64(ys[r]), ref[:, r * 1024:(r + 1) * 1024], F32_TOL, "column shard")


@pytest.mark.parametrize("combine", COMBINES)
def test_wiki_example_fp32_row_parallel(combine):
    need_gpu()
    w = inputs.WORKLOADS["wiki_linear_fp32_tp2"]
    d = inputs.make_fp32_linear_inputs(w)
    n = w["tp"]
    xs, ws = O.split_cols(d["x"], n), O.split_cols(d["w"], n)
    ys = _row_outputs(n, w["T"], w["d_out"], combine)
    tp.tp_row_linear(n, [dev_f32(a) for a in xs], [dev_f32(b) for b in ws], ys, combine)
    _check_row(ys, O.row_parallel(xs, ws), combine, F32_TOL)


# ---- bf16: exact small-integer cases (several tiles and a ragged tail) -------
@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [192, 200])
def test_column_exact_small_integers(n, out_dtype, K):
    need_gpu()
    t = torch()
    # 2 m-tiles (ragged), ragged n; K = 192 is 3 whole k-tiles (the last stage of
    # two k-tiles half past the end), K = 200 ends inside a k-tile
    T, per = 200, 136
    lo, hi = (-1, 1) if out_dtype == "bf16" else (-4, 4)   # bf16 holds integers <= 256 exactly
    x = inputs.small_int_bf16(21, 0, (T, K), lo, hi)
    wf = inputs.small_int_bf16(21, 1, (n * per, K), lo, hi)
    shards = O.split_rows(inputs.bf16_bits_to_f64(wf), n)
    dt = t.float32 if out_dtype == "f32" else t.bfloat16
    y = t.zeros((T, n * per), dtype=dt, device="cuda")
    tp.tp_column_linear(n, dev_bf16(x), [dev_bf16(wf[r * per:(r + 1) * per]) for r in range(n)],
                        [y], gather=True)
    ref = O.all_gather_columns(O.column_parallel(inputs.bf16_bits_to_f64(x), shards))
    assert np.array_equal(host_f64(y), ref)


@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("combine", COMBINES)
def test_row_exact_small_integers(n, combine):
    need_gpu()
    T, per, nout = 200, 64, 264       # K per rank 64, ragged T and n
    x = inputs.small_int_bf16(31, 0, (T, n * per))
    wf = inputs.small_int_bf16(31, 1, (nout, n * per))
    xs = O.split_cols(inputs.bf16_bits_to_f64(x), n)
    ws = O.split_cols(inputs.bf16_bits_to_f64(wf), n)
    ys = _row_outputs(n, T, nout, combine)
    tp.tp_row_linear(n, [dev_bf16(x[:, r * per:(r + 1) * per]) for r in range(n)],
                     [dev_bf16(wf[:, r * per:(r + 1) * per]) for r in range(n)], ys, combine)
    parts = O.row_parallel(xs, ws)
    if combine == tp.TP_COMBINE_NONE:
        for y, p in zip(ys, parts):
            assert np.array_equal(host_f64(y), p)
    else:
        for y in ys:
            assert np.array_equal(host_f64(y), sum(parts))


# ---- bf16: normal inputs against the fp64 oracle ----------------------------------
@pytest.mark.parametrize("T,K,per,n", [(1, 64, 16, 2), (130, 320, 264, 2), (257, 512, 128, 4),
                                       (512, 2048, 512, 8), (64, 4096, 512, 8)])
def test_column_bf16_normal(T, K, per, n):
    need_gpu()
    t = torch()
    x = inputs.normal_bf16(41, 0, (T, K))
    wf = inputs.normal_bf16(41, 1, (n * per, K), 0.02)
    ys = [t.full((T, per), float("nan"), dtype=t.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_column_linear(n, dev_bf16(x), [dev_bf16(wf[r * per:(r + 1) * per]) for r in range(n)],
                        ys, gather=False)
    ref = O.column_parallel(inputs.bf16_bits_to_f64(x), O.split_rows(inputs.bf16_bits_to_f64(wf), n))
    for r in range(n):
        assert_close(host_f64(ys[r]), ref[r], BF16_TOL, f"rank {r}")


@pytest.mark.parametrize("combine", COMBINES)
@pytest.mark.parametrize("T,per,nout,n", [(130, 192, 200, 2), (512, 1024, 2048, 4), (64, 512, 4096, 8)])
def test_row_bf16_normal(T, per, nout, n, combine):
    need_gpu()
    x = inputs.normal_bf16(51, 0, (T, n * per))
    wf = inputs.normal_bf16(51, 1, (nout, n * per), 0.02)
    ys = _row_outputs(n, T, nout, combine)
    tp.tp_row_linear(n, [dev_bf16(x[:, r * per:(r + 1) * per]) for r in range(n)],
                     [dev_bf16(wf[:, r * per:(r + 1) * per]) for r in range(n)], ys, combine)
    parts = O.row_parallel(O.split_cols(inputs.bf16_bits_to_f64(x), n),
                           O.split_cols(inputs.bf16_bits_to_f64(wf), n))
    _check_row(ys, parts, combine, BF16_TOL)


def test_row_ring_modes_bitwise_equal():
    need_gpu()
    n, T, per, nout = 4, 256, 256, 512
    x = inputs.normal_bf16(61, 0, (T, n * per))
    wf = inputs.normal_bf16(61, 1, (nout, n * per), 0.02)
    xs = [dev_bf16(x[:, r * per:(r + 1) * per]) for r in range(n)]
    ws = [dev_bf16(wf[:, r * per:(r + 1) * per]) for r in range(n)]
    a = _row_outputs(n, T, nout, tp.TP_COMBINE_RING)
    b = _row_outputs(n, T, nout, tp.TP_COMBINE_RING_FUSED)
    tp.tp_row_linear(n, xs, ws, a, tp.TP_COMBINE_RING)
    tp.tp_row_linear(n, xs, ws, b, tp.TP_COMBINE_RING_FUSED)
    for r in range(n):
        assert np.array_equal(host_bits_f32(a[r]), host_bits_f32(b[r]))
        assert np.array_equal(host_bits_f32(a[r]), host_bits_f32(a[0]))


@pytest.mark.parametrize("n,T,per,nout", [(2, 512, 4096, 2048), (4, 200, 2048, 264), (8, 64, 2048, 1000)])
def test_row_ring_modes_bitwise_equal_split_k(n, T, per, nout):
    """Shapes small enough in T for the split-K GEMM (pair and single-CTA,
    ragged rows and columns): the one-pass ring all-reduce must give the step
    ring's bits on every rank, on repeated calls, and the oracle's value."""
    need_gpu()
    x = inputs.normal_bf16(62, 0, (T, n * per))
    wf = inputs.normal_bf16(62, 1, (nout, n * per), 0.02)
    xs = [dev_bf16(x[:, r * per:(r + 1) * per]) for r in range(n)]
    ws = [dev_bf16(wf[:, r * per:(r + 1) * per]) for r in range(n)]
    a = _row_outputs(n, T, nout, tp.TP_COMBINE_RING)
    tp.tp_row_linear(n, xs, ws, a, tp.TP_COMBINE_RING)
    for rep in range(2):
        b = _row_outputs(n, T, nout, tp.TP_COMBINE_RING_FUSED)
        tp.tp_row_linear(n, xs, ws, b, tp.TP_COMBINE_RING_FUSED)
        for r in range(n):
            assert np.array_equal(host_bits_f32(a[r]), host_bits_f32(b[r])), (rep, r)
    parts = O.row_parallel(O.split_cols(inputs.bf16_bits_to_f64(x), n),
                           O.split_cols(inputs.bf16_bits_to_f64(wf), n))
    assert_close(host_f64(b[0]), sum(parts), BF16_TOL, "ring fold vs oracle")
    assert tp.tp_device_status() == (tp.TP_OK, 0)


def test_column_gather_into_strided_output():
    need_gpu()
    t = torch()
    n, T, K, per = 2, 70, 128, 64
    x = inputs.normal_bf16(71, 0, (T, K))
    wf = inputs.normal_bf16(71, 1, (n * per, K), 0.02)
    big = t.full((T, n * per + 64), 3.0, device="cuda")
    y = big[:, 32:32 + n * per]
    tp.tp_column_linear(n, dev_bf16(x), [dev_bf16(wf[r * per:(r + 1) * per]) for r in range(n)],
                        [y], gather=True)
    ref = O.linear(inputs.bf16_bits_to_f64(x), inputs.bf16_bits_to_f64(wf))
    assert_close(host_f64(y), ref, BF16_TOL, "strided gather")
    assert t.all(big[:, :32] == 3.0) and t.all(big[:, 32 + n * per:] == 3.0)


def test_empty_and_zero_k():
    need_gpu()
    t = torch()
    n = 2
    x0 = t.zeros((0, 64), dtype=t.bfloat16, device="cuda")
    w = [t.zeros((32, 64), dtype=t.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_column_linear(n, x0, w, [t.zeros((0, 64), dtype=t.bfloat16, device="cuda")], gather=True)
    xk = t.zeros((5, 0), dtype=t.bfloat16, device="cuda")
    wk = [t.zeros((32, 0), dtype=t.bfloat16, device="cuda") for _ in range(n)]
    y = t.full((5, 64), 9.0, device="cuda")
    tp.tp_column_linear(n, xk, wk, [y], gather=True)
    assert t.all(y == 0.0)
