"""Failure detection on the GPU without a GPU fault: a bounded device wait that
runs out reports TP_ERR_TIMEOUT and leaves the context usable; a rank marked
failed stops a block call before anything is enqueued."""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import dev_f32, host_bits_f32, need_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    need_gpu()
    import torch
    tp.tp_set_wait_budget(20_000_000)          # 20 ms
    try:
        tp.tp_debug_wait_timeout()
        st, word = tp.tp_device_status()
    finally:
        tp.tp_set_wait_budget(0)
    assert st == tp.TP_ERR_TIMEOUT and word == 0x1FF
    assert tp.tp_device_status() == (tp.TP_OK, 0)    # cleared
    host = [inputs.normal_f32(1, r, (16, 16)) for r in range(2)]
    dev = [dev_f32(h) for h in host]
    tp.tp_allreduce_ring(2, dev)
    torch.cuda.synchronize()
    ref = O.ring_all_reduce([h.reshape(-1) for h in host])
    assert np.array_equal(host_bits_f32(dev[0]).reshape(-1), ref[0].view(np.uint32))


def test_failed_rank_stops_block_before_launch():
    need_gpu()
    import torch
    plan = tp.tp_plan_create(2, 256, 4, 2, 64, 512)
    x = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    g = [torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    d = [torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ys = [torch.full((8, 256), 4.0, device="cuda") for _ in range(2)]
    ws = torch.empty(tp.tp_mlp_block_workspace_size(plan, 8), dtype=torch.uint8, device="cuda")
    tp.tp_set_rank_health(1, False)
    try:
        with pytest.raises(tp.TPError) as e:
            tp.tp_mlp_block(plan, x, g, g, d, ys, tp.TP_COMBINE_RING, ws)
        assert e.value.status == tp.TP_ERR_RANK_FAILED
        torch.cuda.synchronize()
        assert all(torch.all(y == 4.0) for y in ys)
    finally:
        tp.tp_set_rank_health(1, True)
    tp.tp_mlp_block(plan, x, g, g, d, ys, tp.TP_COMBINE_RING, ws)
    torch.cuda.synchronize()
    assert all(torch.all(y == 0.0) for y in ys)
    assert tp.tp_device_status() == (tp.TP_OK, 0)
