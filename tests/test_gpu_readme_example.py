"""The README's MLP example (TP=2, T=512, D=2048, F=8192: plan, slicing the
weights by the plan's ranges, tp_mlp_block with the ring all-reduce) run as
written, on seeded inputs, and checked against the fp64 oracle's unsharded
MLP within the bf16 tolerance on every rank."""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_f64, need_gpu

pytestmark = pytest.mark.gpu


def test_readme_mlp_example():
    need_gpu()
    import torch
    n, T, D, F = 2, 512, 2048, 8192
    plan = tp.tp_plan_create(n, D, 16, 4, 128, F)
    xb = inputs.normal_bf16(701, 1, (T, D))
    gb, ub = inputs.normal_bf16(701, 2, (F, D), 0.02), inputs.normal_bf16(701, 3, (F, D), 0.02)
    db = inputs.normal_bf16(701, 4, (D, F), 0.02)
    x, wg, wu, wd = dev_bf16(xb), dev_bf16(gb), dev_bf16(ub), dev_bf16(db)
    shard = [tp.tp_plan_query_rank(plan, r)["ranges"] for r in range(n)]
    w_gate = [wg[slice(*s["gate_proj"])] for s in shard]
    w_up = [wu[slice(*s["up_proj"])] for s in shard]
    w_down = [wd[:, slice(*s["down_proj"])] for s in shard]
    y = [torch.empty(T, D, device="cuda") for _ in range(n)]
    ws = torch.empty(tp.tp_mlp_block_workspace_size(plan, T), dtype=torch.uint8, device="cuda")
    tp.tp_mlp_block(plan, x, w_gate, w_up, w_down, y, tp.TP_COMBINE_RING_FUSED, ws)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    f = inputs.bf16_bits_to_f64
    ref = O.mlp_unsharded(f(xb), f(gb), f(ub), f(db))
    for r in range(n):
        assert_close(host_f64(y[r]), ref, BF16_TOL, f"rank {r}")
    assert torch.equal(y[0], y[1])
