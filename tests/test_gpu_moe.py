"""GPU parity of the mixture-of-experts block ([MLX] MoE 전문가 병렬화: Expert
Parallel and Within-Expert Parallel), through the C ABI, against the fp64 oracle.

The GPU rounds H to bf16 and sums in f32, so outputs are compared within the
bf16 tolerance (max|Y_gpu - Y_ref| <= 1e-2 * max|Y_ref|). The two ring modes
fold in the same order and must agree bit for bit, and repeated calls must give
the same bits (the routing sort is stable, the combine sums slots in order).
"""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_f64, need_gpu

pytestmark = pytest.mark.gpu
MODES = {O.MOE_EXPERT_PARALLEL: tp.TP_MOE_EXPERT_PARALLEL, O.MOE_WITHIN_EXPERT: tp.TP_MOE_WITHIN_EXPERT}


def _torch():
    import torch
    return torch


def stacked_weights(eg, eu, ed, n, mode):
    """Per-rank stacked weight bits in the layout tp_moe_block takes (host side,
    plain slicing): within-expert, rank r holds every expert's F/N slice;
    expert parallel, rank r holds experts r, r+N, ... whole."""
    E, F, _D = eg.shape
    if mode == O.MOE_WITHIN_EXPERT:
        fs = F // n
        g = [np.concatenate([eg[e, r * fs:(r + 1) * fs] for e in range(E)]) for r in range(n)]
        u = [np.concatenate([eu[e, r * fs:(r + 1) * fs] for e in range(E)]) for r in range(n)]
        d = [np.concatenate([ed[e][:, r * fs:(r + 1) * fs] for e in range(E)]) for r in range(n)]
    else:
        g = [np.concatenate([eg[e] for e in range(r, E, n)]) for r in range(n)]
        u = [np.concatenate([eu[e] for e in range(r, E, n)]) for r in range(n)]
        d = [np.concatenate([ed[e] for e in range(r, E, n)]) for r in range(n)]
    return g, u, d


class Moe:
    def __init__(self, n, mode, E, k, T, D, F, seed, ids=None, wts=None):
        torch = _torch()
        self.n, self.mode, self.E, self.k, self.T, self.D, self.F = n, mode, E, k, T, D, F
        self.x = inputs.normal_bf16(seed, 1, (T, D))
        self.eg = inputs.normal_bf16(seed, 2, (E, F, D), 0.05)
        self.eu = inputs.normal_bf16(seed, 3, (E, F, D), 0.05)
        self.ed = inputs.normal_bf16(seed, 4, (E, D, F), 0.05)
        if ids is None:
            ids, wts = inputs.routing(seed, 5, T, E, k)
        self.ids, self.wts = ids.astype(np.int32), wts.astype(np.float32)
        g, u, d = stacked_weights(self.eg, self.eu, self.ed, n, mode)
        self.dev = dict(x=dev_bf16(self.x), g=[dev_bf16(t) for t in g], u=[dev_bf16(t) for t in u],
                        d=[dev_bf16(t) for t in d], ids=torch.from_numpy(self.ids).cuda(),
                        w=torch.from_numpy(self.wts).cuda())
        self.dims = tp.moe_dims(n, MODES[mode], E, k, D, F)
        self.ws = torch.empty(tp.tp_moe_workspace_size(self.dims, T), dtype=torch.uint8, device="cuda")

    def run(self, combine):
        torch = _torch()
        ys = [torch.full((self.T, self.D), float("nan"), device="cuda")
              for _ in range(1 if combine == tp.TP_COMBINE_FUSED else self.n)]
        dv = self.dev
        tp.tp_moe_block(self.dims, dv["x"], dv["ids"], dv["w"], dv["g"], dv["u"], dv["d"], ys, combine, self.ws)
        torch.cuda.synchronize()
        return ys

    def oracle(self, rows=None):
        f = inputs.bf16_bits_to_f64
        sel = slice(None) if rows is None else rows
        E = self.E
        return O.moe_sharded(f(self.x[sel]), self.ids[sel], self.wts[sel].astype(np.float64),
                             [f(self.eg[e]) for e in range(E)], [f(self.eu[e]) for e in range(E)],
                             [f(self.ed[e]) for e in range(E)], self.n, self.mode)


CASES = [  # n, E, k, T, D, F
    (2, 4, 2, 300, 256, 512),    # pair GEMMs (T*k > 128), ragged expert loads
    (4, 8, 2, 64, 128, 256),     # single-CTA GEMMs (T*k = 128)
    (8, 8, 2, 200, 256, 1024),
    (4, 4, 1, 33, 192, 384),     # top-1, K not a multiple of 64 in the down GEMM
    (1, 2, 2, 96, 128, 256),
]


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("n,E,k,T,D,F", CASES)
def test_moe_block_matches_the_oracle(mode, n, E, k, T, D, F):
    need_gpu()
    if mode == O.MOE_EXPERT_PARALLEL and E % n:
        pytest.skip("expert parallel needs E divisible by N")
    m = Moe(n, mode, E, k, T, D, F, seed=500 + n * 10 + E)
    ref = m.oracle()
    parts = m.run(tp.TP_COMBINE_NONE)
    for r in range(n):
        assert_close(host_f64(parts[r]), ref["partials"][r], BF16_TOL, f"partial {r}")
    fused = m.run(tp.TP_COMBINE_FUSED)
    assert_close(host_f64(fused[0]), ref["y"][0], BF16_TOL, "fused")
    ring = m.run(tp.TP_COMBINE_RING)
    ring_fused = m.run(tp.TP_COMBINE_RING_FUSED)
    for r in range(n):
        assert_close(host_f64(ring_fused[r]), ref["y"][r], BF16_TOL, f"ring_fused {r}")
        assert _torch().equal(ring[r], ring_fused[r]), f"ring modes differ on rank {r}"
    again = m.run(tp.TP_COMBINE_RING_FUSED)
    for r in range(n):
        assert _torch().equal(again[r], ring_fused[r]), "not deterministic"
    assert tp.tp_device_status() == (tp.TP_OK, 0)


@pytest.mark.parametrize("mode", list(MODES))
def test_skewed_routing(mode):
    """Every token picks expert 1 first; expert 3 gets no token at all."""
    need_gpu()
    n, E, k, T = 2, 4, 2, 260
    ids = np.stack([np.ones(T, dtype=np.int32), np.where(np.arange(T) % 3 == 0, 0, 2).astype(np.int32)], axis=1)
    wts = np.tile(np.array([0.75, 0.25], dtype=np.float32), (T, 1))
    m = Moe(n, mode, E, k, T, 128, 256, seed=531, ids=ids, wts=wts)
    ref = m.oracle()
    ys = m.run(tp.TP_COMBINE_RING_FUSED)
    assert_close(host_f64(ys[0]), ref["y"][0], BF16_TOL, "y")
    parts = m.run(tp.TP_COMBINE_NONE)
    for r in range(n):
        assert_close(host_f64(parts[r]), ref["partials"][r], BF16_TOL, f"partial {r}")
    if mode == O.MOE_EXPERT_PARALLEL:
        # rank 1 holds experts 1 and 3: every token's first slot lands there
        assert np.all(host_f64(parts[1]) != 0.0)


def test_bad_expert_id_drops_the_slot():
    need_gpu()
    n, E, k, T = 2, 4, 2, 40
    ids, wts = inputs.routing(541, 5, T, E, k)
    ids[3, 1] = E      # out of range
    ids[7, 0] = -2
    m = Moe(n, O.MOE_WITHIN_EXPERT, E, k, T, 128, 256, seed=541, ids=ids, wts=wts)
    ys = m.run(tp.TP_COMBINE_FUSED)
    st, word = tp.tp_device_status()
    assert st == tp.TP_ERR_BAD_TOKEN and word != 0
    keep = wts.copy()
    keep[3, 1] = 0.0
    keep[7, 0] = 0.0
    ids_ok = np.clip(ids, 0, E - 1)
    f = inputs.bf16_bits_to_f64
    ref = O.moe_unsharded(f(m.x), ids_ok, keep.astype(np.float64), [f(m.eg[e]) for e in range(E)],
                          [f(m.eu[e]) for e in range(E)], [f(m.ed[e]) for e in range(E)])
    assert_close(host_f64(ys[0]), ref, BF16_TOL, "y")
    assert tp.tp_device_status() == (tp.TP_OK, 0)


def test_moe_mixtral_tp8_t4096_sampled_rows():
    """The benchmarked configuration (within-expert, TP=8, 8 experts of
    4096 x 14336, top-2, 4096 tokens, ring all-reduce in one pass), checked on a
    seeded sample of token rows: each output row depends only on its own token."""
    need_gpu()
    torch = _torch()
    w = inputs.WORKLOADS["moe_mixtral_tp8_t4096"]
    n, T, D, F, E, k = w["tp"], w["T"], w["hidden"], w["ffn"], w["experts"], w["top_k"]
    data = inputs.make_bf16_inputs(w)
    g, u, d = stacked_weights(data["eg"], data["eu"], data["ed"], n, O.MOE_WITHIN_EXPERT)
    dims = tp.moe_dims(n, tp.TP_MOE_WITHIN_EXPERT, E, k, D, F)
    ws = torch.empty(tp.tp_moe_workspace_size(dims, T), dtype=torch.uint8, device="cuda")
    ys = [torch.empty((T, D), device="cuda") for _ in range(n)]
    tp.tp_moe_block(dims, dev_bf16(data["x"]), torch.from_numpy(data["topk_ids"]).cuda(),
                    torch.from_numpy(data["topk_w"]).cuda(), [dev_bf16(t) for t in g], [dev_bf16(t) for t in u],
                    [dev_bf16(t) for t in d], ys, tp.TP_COMBINE_RING_FUSED, ws)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    rows = np.sort(inputs.rng(w["seed"], 99).choice(T, size=16, replace=False))
    f = inputs.bf16_bits_to_f64
    xs, ids_s, w_s = f(data["x"][rows]), data["topk_ids"][rows], data["topk_w"][rows].astype(np.float64)
    # The mixture is linear in the routing weights: sum it expert by expert (the
    # other slots weighted 0), so that one expert's fp64 weights are held at a time.
    ref = np.zeros((rows.size, D))
    for e in range(E):
        w_e = np.where(ids_s == e, w_s, 0.0)
        ref += O.moe_unsharded(xs, np.zeros_like(ids_s), w_e, [f(data["eg"][e])], [f(data["eu"][e])],
                               [f(data["ed"][e])])
    for r in (0, n - 1):
        assert_close(host_f64(ys[r])[rows], ref, BF16_TOL, f"rank {r}")


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("n,E,k,T,D,F", [(4, 4, 2, 31, 200, 256), (8, 8, 2, 31, 200, 512), (2, 4, 2, 300, 256, 512)])
def test_ring_folded_into_the_combine(mode, n, E, k, T, D, F, monkeypatch):
    """RING_FUSED and RING_SHARED fold the ranks' partials inside the weighted
    combine, each element in its ring chunk's order (31 x 200 outputs put chunk
    boundaries inside float4 units). The bits equal the combine followed by the
    one-pass ring (TPGQA_MOE_RING_FOLD=0) and the step ring, on every rank."""
    need_gpu()
    if mode == O.MOE_EXPERT_PARALLEL and E % n:
        pytest.skip("expert parallel needs E divisible by N")
    m = Moe(n, mode, E, k, T, D, F, seed=530 + n * 10 + E)
    folded = m.run(tp.TP_COMBINE_RING_FUSED)
    shared = m.run(tp.TP_COMBINE_RING_SHARED)
    steps = m.run(tp.TP_COMBINE_RING)
    monkeypatch.setenv("TPGQA_MOE_RING_FOLD", "0")
    unfolded = m.run(tp.TP_COMBINE_RING_FUSED)
    torch = _torch()
    for r in range(n):
        assert torch.equal(folded[r], unfolded[r]), f"rank {r}"
        assert torch.equal(folded[r], steps[r]), f"rank {r}, step ring"
    assert torch.equal(shared[0], folded[0])
    ref = m.oracle()
    assert_close(host_f64(folded[0]), ref["y"][0], BF16_TOL, "folded")
    assert tp.tp_device_status() == (tp.TP_OK, 0)
