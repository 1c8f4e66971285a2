"""GPU parity of the ring collectives and the concatenating all-gather.

The ring kernels add in fp32 in the ring's fold order, so they must equal the
oracle's ring run on the same fp32 buffers bit for bit (the oracle computes in
the buffers' dtype). Step and fused modes must therefore agree bitwise too.
"""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import dev_bf16, dev_f32, host_bits_f32, host_f64, need_gpu

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (1, 7), (3, 5), (16, 64), (37, 101), (512, 2048), (1024, 1027)]
NS = [1, 2, 4, 8]
MODES = [tp.TP_RING_STEPS, tp.TP_RING_FUSED]


def _host_bufs(n, shape, seed):
    return [inputs.normal_f32(seed, 200 + r, shape) for r in range(n)]


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).reshape(-1)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("shape", SHAPES)
def test_allreduce_bit_exact(n, shape, mode):
    need_gpu()
    host = _host_bufs(n, shape, seed=7 + n)
    dev = [dev_f32(h) for h in host]
    tp.tp_allreduce_ring(n, dev, mode)
    ref = O.ring_all_reduce([h.reshape(-1) for h in host])
    for r in range(n):
        assert np.array_equal(host_bits_f32(dev[r]).reshape(-1), _bits(ref[r])), (n, shape, mode, r)


@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("shape", SHAPES)
def test_allreduce_shared_result_bit_exact(n, shape):
    """The one-pass ring all-reduce with its result stored once: buf[0] holds the
    oracle ring's sum bit for bit, buf[1..N-1] keep their partials."""
    need_gpu()
    host = _host_bufs(n, shape, seed=17 + n)
    dev = [dev_f32(h) for h in host]
    tp.tp_allreduce_ring(n, dev, tp.TP_RING_FUSED_SHARED)
    ref = O.ring_all_reduce([h.reshape(-1) for h in host])
    assert np.array_equal(host_bits_f32(dev[0]).reshape(-1), _bits(ref[0])), (n, shape)
    for r in range(1, n):
        assert np.array_equal(host_bits_f32(dev[r]).reshape(-1), _bits(host[r])), (n, shape, r)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [2, 4, 8])
@pytest.mark.parametrize("shape", [(1, 7), (37, 101), (512, 2048)])
def test_reduce_scatter_owned_chunk_bit_exact(n, shape, mode):
    need_gpu()
    host = _host_bufs(n, shape, seed=11 + n)
    dev = [dev_f32(h) for h in host]
    tp.tp_reduce_scatter(n, dev, mode)
    ref = O.ring_reduce_scatter([h.reshape(-1) for h in host])
    size = shape[0] * shape[1]
    for r in range(n):
        lo, hi = O.chunk_bounds(size, n, r)
        got = host_bits_f32(dev[r]).reshape(-1)[lo:hi]
        assert np.array_equal(got, _bits(ref[r])[lo:hi]), (n, shape, mode, r)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [2, 4, 8])
@pytest.mark.parametrize("shape", [(1, 7), (37, 101), (512, 2048)])
def test_ring_all_gather_bit_exact(n, shape, mode):
    need_gpu()
    host = _host_bufs(n, shape, seed=13 + n)
    dev = [dev_f32(h) for h in host]
    tp.tp_ring_all_gather(n, dev, mode)
    ref = O.ring_all_gather([h.reshape(-1) for h in host])
    for r in range(n):
        assert np.array_equal(host_bits_f32(dev[r]).reshape(-1), _bits(ref[r]))


def test_allreduce_large_partials_steps_equal_fused():
    # a combine of four 32 MiB partials (the attention-projection output size)
    need_gpu()
    n, shape = 4, (2048, 4096)
    host = _host_bufs(n, shape, seed=5)
    a = [dev_f32(h) for h in host]
    b = [dev_f32(h) for h in host]
    tp.tp_allreduce_ring(n, a, tp.TP_RING_STEPS)
    tp.tp_allreduce_ring(n, b, tp.TP_RING_FUSED)
    ref = O.ring_all_reduce([h.reshape(-1) for h in host])
    for r in range(n):
        ga, gb = host_bits_f32(a[r]).reshape(-1), host_bits_f32(b[r]).reshape(-1)
        assert np.array_equal(ga, gb)
        assert np.array_equal(ga, _bits(ref[r]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("n_out", ["one", "all"])
def test_all_gather_columns(dtype, n, n_out):
    need_gpu()
    rows = 37
    cols = [8 * (r + 1) for r in range(n)]
    if dtype == "f32":
        host = [inputs.normal_f32(3, 300 + r, (rows, c)) for r, c in enumerate(cols)]
        shards = [dev_f32(h) for h in host]
        import torch
        outs = [torch.full((rows, sum(cols)), -7.0, device="cuda") for _ in range(1 if n_out == "one" else n)]
        ref = O.all_gather_columns([h.astype(np.float64) for h in host])
    else:
        host = [inputs.normal_bf16(3, 300 + r, (rows, c)) for r, c in enumerate(cols)]
        shards = [dev_bf16(h) for h in host]
        import torch
        outs = [torch.zeros((rows, sum(cols)), dtype=torch.bfloat16, device="cuda")
                for _ in range(1 if n_out == "one" else n)]
        ref = O.all_gather_columns([inputs.bf16_bits_to_f64(h) for h in host])
    tp.tp_all_gather(n, shards, outs, axis=1)
    for o in outs:
        assert np.array_equal(host_f64(o), ref)


@pytest.mark.parametrize("n", [2, 4])
def test_all_gather_rows_into_strided_output(n):
    need_gpu()
    import torch
    cols = 13
    rows = [3 * r + 1 for r in range(n)]
    host = [inputs.normal_f32(4, 400 + r, (rr, cols)) for r, rr in enumerate(rows)]
    shards = [dev_f32(h) for h in host]
    big = torch.full((sum(rows), 32), 5.0, device="cuda")
    out = big[:, 4:4 + cols]                       # ld 32, offset 4 elements
    tp.tp_all_gather(n, shards, [out], axis=0)
    ref = O.gather_flat_shards(host).reshape(sum(rows), cols).astype(np.float64)
    assert np.array_equal(host_f64(out), ref)
    assert torch.all(big[:, :4] == 5.0) and torch.all(big[:, 4 + cols:] == 5.0)
