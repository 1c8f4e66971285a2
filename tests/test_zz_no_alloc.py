"""tp_mlp_block_static: the MLP block for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: a plug-in whose host framework
owns all device memory and lends none of it, or a server that reserved all free
HBM at start-up and must not call cudaMalloc while serving. For them the block
keeps its intermediate H in a fixed 16 MiB array inside the library. These tests
check, through the C ABI, that two calls in a row give what tp_mlp_block gives
with a caller-provided workspace, and that a request too large for the array is
refused before anything runs.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest

import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_f64, need_gpu


def _problem(seed):
    w = dict(kind="mlp", T=300, hidden=1024, ffn=4096, tp=4, seed=seed, w_std=0.05)
    return w, inputs.make_bf16_inputs(w)


def _run(w, data, static):
    import torch
    n, T, D = w["tp"], w["T"], w["hidden"]
    plan = tp.tp_plan_create(n, D, 8, 8, 128, w["ffn"])
    sh = [tp.tp_plan_query_rank(plan, r) for r in range(n)]
    x, wg, wu, wd = (dev_bf16(data[k]) for k in ("x", "wg", "wu", "wd"))
    g = [wg[slice(*sh[r]["ranges"]["gate_proj"])] for r in range(n)]
    u = [wu[slice(*sh[r]["ranges"]["up_proj"])] for r in range(n)]
    d = [wd[:, slice(*sh[r]["ranges"]["down_proj"])] for r in range(n)]
    ys = [torch.full((T, D), float("nan"), device="cuda") for _ in range(n)]
    if static:
        tp.tp_mlp_block_static(plan, x, g, u, d, ys, tp.TP_COMBINE_RING)
    else:
        ws = torch.empty(tp.tp_mlp_block_workspace_size(plan, T), dtype=torch.uint8, device="cuda")
        tp.tp_mlp_block(plan, x, g, u, d, ys, tp.TP_COMBINE_RING, ws)
    torch.cuda.synchronize()
    return [host_f64(y) for y in ys]


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice():
    need_gpu()
    # Two calls in a row on different inputs: the second call must not see the
    # first call's H left in the shared array.
    for seed in (201, 202):
        w, data = _problem(seed)
        got = _run(w, data, static=True)
        ref = _run(w, data, static=False)
        for g, r in zip(got, ref):
            assert_close(g, r, BF16_TOL, f"static vs workspace (seed {seed})")
    assert tp.tp_device_status() == (tp.TP_OK, 0)


def test_static_scratch_refuses_oversized_requests():
    # 16 MiB holds tokens * ffn <= 8 Mi bf16 values; 1025 * 8192 is one row too many.
    assert tp.tp_mlp_block_static_max_bytes() == 16 << 20
    plan = tp.tp_plan_create(2, 2048, 16, 8, 128, 8192)
    x = tp.TpTensor(1 << 40, tp.TP_BF16, 0, 1025, 2048, 2048)   # never dereferenced
    dummy = (tp.TpTensor * 2)()
    st = tp.raw_status("tp_mlp_block_static", plan.handle, ctypes.byref(x), dummy, dummy, dummy,
                       dummy, tp.TP_COMBINE_RING, None)
    assert st == tp.TP_ERR_WORKSPACE
