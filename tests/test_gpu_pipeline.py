"""GPU parity of the row-parallel -> reduce-scatter -> column-parallel pipeline
([MLX] 통신 패턴, Reduce-scatter: a row-parallel result going straight into a
column-parallel op, without the all-gather step), through the C ABI.

tp_reduce_scatter_bf16 folds each chunk over the ranks in the ring's order in
fp32 and rounds once to bf16; the oracle's fp32 ring followed by its bf16
rounding gives the same bits. tp_column_linear_chunks reads the input rows from
the N chunk buffers; on small-integer inputs (exact under any summation order)
it equals the oracle exactly, on normal inputs within the bf16 tolerance.
"""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_f64, need_gpu

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _bits(t):
    """uint16 bit patterns of a CUDA bf16 tensor."""
    return t.view(_torch().int16).cpu().numpy().view(np.uint16)


def _bf16_bits_of(x64):
    """bf16 bit patterns of values that are exactly bfloat16 (float64 in)."""
    return (np.asarray(x64, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("n,t,cols,ld", [(2, 16, 64, 64), (4, 10, 6, 8), (8, 33, 20, 24), (2, 5, 7, 8),
                                         (8, 64, 4096, 4096), (4, 7, 12, 16)])
def test_reduce_scatter_bf16_matches_the_oracle_ring(n, t, cols, ld):
    need_gpu()
    torch = _torch()
    g = inputs.rng(301, n * 100 + t)
    parts = [g.standard_normal((t, cols)).astype(np.float32) for _ in range(n)]
    dev = [torch.from_numpy(p).cuda() for p in parts]
    sentinel = 0x7FC1  # a NaN pattern no sum produces
    outs = [torch.full((t, ld), 0, dtype=torch.int16, device="cuda").fill_(sentinel).view(torch.bfloat16)
            for _ in range(n)]
    tp.tp_reduce_scatter_bf16(n, dev, [o[:, :cols] for o in outs])
    torch.cuda.synchronize()
    want = O.reduce_scatter_then_column(parts, [np.ones((1, cols))] * n, round_bf16=True)["chunks"]
    size = t * cols
    for c in range(n):
        lo, hi = O.chunk_bounds(size, n, c)
        got = _bits(outs[c])
        flat = got[:, :cols].reshape(-1)
        assert np.array_equal(flat[lo:hi], _bf16_bits_of(want[c])), f"chunk {c}"
        # nothing outside chunk c of out[c] (nor past cols) is written
        rest = np.ones(size, dtype=bool)
        rest[lo:hi] = False
        assert np.all(flat[rest] == sentinel)
        assert np.all(got[:, cols:] == sentinel)
    assert tp.tp_device_status() == (tp.TP_OK, 0)


def _chunk_buffers(x_bits, n):
    """Rank c's buffer: rows of chunk c hold X, every other row holds NaN bits."""
    torch = _torch()
    t = x_bits.shape[0]
    tc = t // n
    bufs = []
    for c in range(n):
        b = np.full(x_bits.shape, 0x7FC1, dtype=np.uint16)
        b[c * tc:(c + 1) * tc] = x_bits[c * tc:(c + 1) * tc]
        bufs.append(dev_bf16(b))
    return bufs


@pytest.mark.parametrize("n,t,k,per", [(2, 512, 256, 136), (4, 200, 192, 64), (8, 64, 128, 40),
                                       (2, 8, 64, 16), (4, 1024, 512, 256)])
@pytest.mark.parametrize("gather", [0, 1])
def test_column_linear_chunks_exact_small_integers(n, t, k, per, gather):
    need_gpu()
    torch = _torch()
    x = inputs.small_int_bf16(311, n, (t, k))
    w = inputs.small_int_bf16(311, 100 + n, (n * per, k))
    ws = [dev_bf16(w[r * per:(r + 1) * per]) for r in range(n)]
    ys = ([torch.full((t, n * per), float("nan"), device="cuda")] if gather else
          [torch.full((t, per), float("nan"), device="cuda") for _ in range(n)])
    tp.tp_column_linear_chunks(n, _chunk_buffers(x, n), ws, ys, gather=bool(gather))
    torch.cuda.synchronize()
    xf = inputs.bf16_bits_to_f64(x)
    ref = O.column_parallel(xf, O.split_rows(inputs.bf16_bits_to_f64(w), n))
    if gather:
        assert np.array_equal(host_f64(ys[0]), O.all_gather_columns(ref))
    else:
        for r in range(n):
            assert np.array_equal(host_f64(ys[r]), ref[r])


@pytest.mark.parametrize("n,t,k,per", [(2, 512, 2048, 512), (8, 64, 512, 128), (4, 256, 1024, 320)])
def test_column_linear_chunks_bf16_normal(n, t, k, per):
    need_gpu()
    torch = _torch()
    x = inputs.normal_bf16(321, n, (t, k))
    w = inputs.normal_bf16(321, 100 + n, (n * per, k), 0.02)
    ys = [torch.full((t, per), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_column_linear_chunks(n, _chunk_buffers(x, n), [dev_bf16(w[r * per:(r + 1) * per]) for r in range(n)],
                               ys, gather=False)
    ref = O.column_parallel(inputs.bf16_bits_to_f64(x), O.split_rows(inputs.bf16_bits_to_f64(w), n))
    for r in range(n):
        assert_close(host_f64(ys[r]), ref[r], BF16_TOL, f"rank {r}")


@pytest.mark.parametrize("n,t,k_row,d,per", [(2, 512, 1024, 512, 256), (4, 128, 512, 256, 96),
                                             (8, 64, 256, 512, 64)])
def test_row_reduce_scatter_column_pipeline(n, t, k_row, d, per):
    """Row-parallel partials -> ring reduce-scatter into bf16 -> column-parallel
    GEMM over the chunks, against the oracle's pipeline."""
    need_gpu()
    torch = _torch()
    a = inputs.normal_bf16(331, n, (t, n * k_row))
    wo = inputs.normal_bf16(331, 100 + n, (d, n * k_row), 0.02)
    wq = inputs.normal_bf16(331, 200 + n, (n * per, d), 0.02)
    parts = [torch.empty((t, d), device="cuda") for _ in range(n)]
    tp.tp_row_linear(n, [dev_bf16(a[:, r * k_row:(r + 1) * k_row]) for r in range(n)],
                     [dev_bf16(wo[:, r * k_row:(r + 1) * k_row]) for r in range(n)], parts, tp.TP_COMBINE_NONE)
    chunks = [torch.empty((t, d), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_reduce_scatter_bf16(n, parts, chunks)
    ys = [torch.empty((t, per), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_column_linear_chunks(n, chunks, [dev_bf16(wq[r * per:(r + 1) * per]) for r in range(n)], ys,
                               gather=False)
    torch.cuda.synchronize()
    part_ref = O.row_parallel(O.split_cols(inputs.bf16_bits_to_f64(a), n), O.split_cols(inputs.bf16_bits_to_f64(wo), n))
    ref = O.reduce_scatter_then_column(part_ref, O.split_rows(inputs.bf16_bits_to_f64(wq), n))
    for r in range(n):
        assert_close(host_f64(ys[r]), ref["y"][r], BF16_TOL, f"rank {r}")
    assert tp.tp_device_status() == (tp.TP_OK, 0)


def test_rs_column_tp8_t4096_sampled_rows():
    """The full-size pipeline in the launch configuration the benchmark times (TP=8,
    T=4096, down projection 28672 -> 8192 feeding the fused q/k/v projection of
    1280 columns per rank), checked on a seeded sample of token rows: every output
    row depends only on its own input row. The all-gathered variant is run on the
    same partials and must agree with the deferred one bit for bit."""
    need_gpu()
    torch = _torch()
    w = inputs.WORKLOADS["rs_column_tp8_t4096"]
    n, t, d, f = w["tp"], w["T"], w["hidden"], w["ffn"]
    data = inputs.make_bf16_inputs(w)
    fr = f // n
    h, wd, wqkv = dev_bf16(data["h"]), dev_bf16(data["wd"]), dev_bf16(data["wqkv"])
    per = wqkv.shape[0] // n
    parts = [torch.empty((t, d), device="cuda") for _ in range(n)]
    tp.tp_row_linear(n, [h[:, r * fr:(r + 1) * fr] for r in range(n)],
                     [wd[:, r * fr:(r + 1) * fr] for r in range(n)], parts, tp.TP_COMBINE_NONE)
    chunks = [torch.empty((t, d), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_reduce_scatter_bf16(n, parts, chunks)
    del parts
    wc = [wqkv[r * per:(r + 1) * per] for r in range(n)]
    ys = [torch.full((t, per), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_column_linear_chunks(n, chunks, wc, ys, gather=False)
    xfull = torch.empty((t, d), dtype=torch.bfloat16, device="cuda")
    tp.tp_all_gather(n, [chunks[r][r * t // n:(r + 1) * t // n] for r in range(n)], [xfull], axis=0)
    yg = [torch.empty((t, per), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    tp.tp_column_linear(n, xfull, wc, yg, gather=False)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    for r in range(n):
        assert torch.equal(ys[r].view(torch.int16), yg[r].view(torch.int16)), f"rank {r}"
    rows = np.sort(inputs.rng(w["seed"], 99).choice(t, size=48, replace=False))
    hf = inputs.bf16_bits_to_f64(data["h"][rows])
    part_ref = O.row_parallel(O.split_cols(hf, n), O.split_cols(inputs.bf16_bits_to_f64(data["wd"]), n))
    ref = O.reduce_scatter_then_column(part_ref, O.split_rows(inputs.bf16_bits_to_f64(data["wqkv"]), n),
                                       round_bf16=True)
    for r in range(n):
        assert_close(host_f64(ys[r])[rows], ref["y"][r], BF16_TOL, f"rank {r}")
