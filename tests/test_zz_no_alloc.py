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

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_f64, need_gpu


def _problem(seed):
    w = dict(kind="mlp", T=300, hidden=1024, ffn=4096, tp=4, seed=seed, w_std=0.05)
    return w, inputs.make_bf16_inputs(w)


class _Block:
    """Device copies of one MLP problem, sharded per the plan, with its outputs."""

    def __init__(self, w, data):
        import torch
        n, T, D = w["tp"], w["T"], w["hidden"]
        self.plan = tp.tp_plan_create(n, D, 8, 8, 128, w["ffn"])
        sh = [tp.tp_plan_query_rank(self.plan, r) for r in range(n)]
        self.x, wg, wu, wd = (dev_bf16(data[k]) for k in ("x", "wg", "wu", "wd"))
        self.g = [wg[slice(*sh[r]["ranges"]["gate_proj"])] for r in range(n)]
        self.u = [wu[slice(*sh[r]["ranges"]["up_proj"])] for r in range(n)]
        self.d = [wd[:, slice(*sh[r]["ranges"]["down_proj"])] for r in range(n)]
        self.keep = (wg, wu, wd)
        self.ys = [torch.full((T, D), float("nan"), device="cuda") for _ in range(n)]
        self.ws = torch.empty(tp.tp_mlp_block_workspace_size(self.plan, T), dtype=torch.uint8, device="cuda")

    def run(self, static):
        import torch
        for y in self.ys:
            y.fill_(float("nan"))
        if static:
            tp.tp_mlp_block_static(self.plan, self.x, self.g, self.u, self.d, self.ys, tp.TP_COMBINE_RING)
        else:
            tp.tp_mlp_block(self.plan, self.x, self.g, self.u, self.d, self.ys, tp.TP_COMBINE_RING, self.ws)
        torch.cuda.synchronize()
        return [host_f64(y) for y in self.ys]


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice():
    need_gpu()
    # Two calls in a row on different inputs: the second call must not see the
    # first call's H left in the shared array. Each result is checked against the
    # workspace entry point and against the oracle's sharded MLP block.
    for seed in (201, 202):
        w, data = _problem(seed)
        b = _Block(w, data)
        got = b.run(static=True)
        ref = b.run(static=False)
        f = {k: inputs.bf16_bits_to_f64(data[k]) for k in ("x", "wg", "wu", "wd")}
        exact = O.mlp_sharded(f["x"], f["wg"], f["wu"], f["wd"], w["tp"])["y"][0]
        for g, r in zip(got, ref):
            assert_close(g, r, BF16_TOL, f"static vs workspace (seed {seed})")
            assert_close(g, exact, BF16_TOL, f"static vs oracle (seed {seed})")
    assert tp.tp_device_status() == (tp.TP_OK, 0)


@pytest.mark.gpu
def test_static_calls_leave_free_device_memory_unchanged():
    """After one call (the first call of a process may load the library's device
    code, which brings the scratch array with it), further calls change the
    device's free memory by nothing: the entry point allocates no device memory."""
    import torch
    need_gpu()
    w, data = _problem(203)
    b = _Block(w, data)
    b.run(static=True)
    free0, _total = torch.cuda.mem_get_info()
    for _ in range(3):
        tp.tp_mlp_block_static(b.plan, b.x, b.g, b.u, b.d, b.ys, tp.TP_COMBINE_RING)
    torch.cuda.synchronize()
    free1, _total = torch.cuda.mem_get_info()
    assert free1 == free0


def test_static_scratch_refuses_oversized_requests():
    # 16 MiB holds tokens * ffn <= 8 Mi bf16 values; 1025 * 8192 is one row too many.
    assert tp.tp_mlp_block_static_max_bytes() == 16 << 20
    plan = tp.tp_plan_create(2, 2048, 16, 8, 128, 8192)
    x = tp.TpTensor(1 << 40, tp.TP_BF16, 0, 1025, 2048, 2048)   # never dereferenced
    dummy = (tp.TpTensor * 2)()
    st = tp.raw_status("tp_mlp_block_static", plan.handle, ctypes.byref(x), dummy, dummy, dummy,
                       dummy, tp.TP_COMBINE_RING, None)
    assert st == tp.TP_ERR_WORKSPACE
