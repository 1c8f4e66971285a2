"""Pins of the oracle's mixture-of-experts block ([MLX] MoE 전문가 병렬화: Expert
Parallel puts expert i whole on rank i % tp_size; Within-Expert Parallel shards
every expert's FFN over all ranks like the dense FFN).

Each pin checks the oracle against something other than its own formula: the
placement against the pages' flowchart; the block against explicit loops with
math.exp, against the dense MLP (one expert, or identical experts whose routing
weights sum to one), against linearity in the routing weights; the sharded modes
against the plain mixture, against where each mode's work may land, and the
all-reduce against its message log.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "moe_expert_parallel.json")
MODES = [O.MOE_EXPERT_PARALLEL, O.MOE_WITHIN_EXPERT]


def _experts(e, d, f, seed, ints=False):
    g = np.random.default_rng(seed)
    if ints:
        mk = lambda shp: g.integers(-2, 3, shp).astype(np.float64)  # noqa: E731
    else:
        mk = lambda shp: g.standard_normal(shp) * 0.3  # noqa: E731
    return [mk((f, d)) for _ in range(e)], [mk((f, d)) for _ in range(e)], [mk((d, f)) for _ in range(e)]


def _routing(t, e, k, seed):
    """k distinct experts per token and softmax weights over the k slots."""
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(e)[:k] for _ in range(t)]).astype(np.int64)
    logits = g.standard_normal((t, k))
    w = np.exp(logits) / np.exp(logits).sum(axis=1, keepdims=True)
    return ids, w


def test_expert_placement_matches_the_flowchart():
    with open(GOLDEN) as fh:
        case = json.load(fh)["cases"][0]
    n = case["tp_size"]
    got = [[i for i in range(case["num_experts"]) if O.expert_rank(i, n) == r] for r in range(n)]
    assert got == case["experts_per_rank"]


def _loops_moe(x, ids, w, wg, wu, wd):
    """The mixture by explicit loops, silu written with math.exp."""
    t_, d_ = x.shape
    y = np.zeros((t_, wd[0].shape[0]))
    for t in range(t_):
        for j in range(ids.shape[1]):
            e = ids[t, j]
            f_ = wg[e].shape[0]
            h = np.zeros(f_)
            for f in range(f_):
                g = sum(x[t, i] * wg[e][f, i] for i in range(d_))
                u = sum(x[t, i] * wu[e][f, i] for i in range(d_))
                h[f] = g / (1.0 + math.exp(-g)) * u
            for o in range(wd[e].shape[0]):
                y[t, o] += w[t, j] * sum(h[f] * wd[e][o, f] for f in range(f_))
    return y


@pytest.mark.parametrize("t,e,k,d,f", [(3, 4, 2, 3, 4), (5, 2, 1, 2, 6), (4, 8, 3, 2, 2)])
def test_moe_unsharded_by_loops(t, e, k, d, f):
    wg, wu, wd = _experts(e, d, f, t * e)
    x = np.random.default_rng(t).standard_normal((t, d))
    ids, w = _routing(t, e, k, e + k)
    assert np.allclose(O.moe_unsharded(x, ids, w, wg, wu, wd), _loops_moe(x, ids, w, wg, wu, wd),
                       rtol=1e-12, atol=1e-12)


def test_one_expert_top1_is_the_dense_mlp():
    wg, wu, wd = _experts(1, 6, 8, 3)
    x = np.random.default_rng(4).standard_normal((7, 6))
    y = O.moe_unsharded(x, np.zeros((7, 1), dtype=np.int64), np.ones((7, 1)), wg, wu, wd)
    assert np.allclose(y, O.mlp_unsharded(x, wg[0], wu[0], wd[0]), rtol=1e-13, atol=1e-13)


def test_identical_experts_with_unit_weights_are_the_dense_mlp():
    wg, wu, wd = _experts(1, 5, 6, 8)
    e = 4
    x = np.random.default_rng(2).standard_normal((6, 5))
    ids, w = _routing(6, e, 3, 1)
    y = O.moe_unsharded(x, ids, w, wg * e, wu * e, wd * e)
    assert np.allclose(y, O.mlp_unsharded(x, wg[0], wu[0], wd[0]), rtol=1e-12, atol=1e-12)


def test_linear_in_the_routing_weights():
    wg, wu, wd = _experts(4, 3, 4, 5)
    x = np.random.default_rng(6).standard_normal((5, 3))
    ids, w = _routing(5, 4, 2, 7)
    y1 = O.moe_unsharded(x, ids, w, wg, wu, wd)
    y2 = O.moe_unsharded(x, ids, 2.5 * w, wg, wu, wd)
    assert np.allclose(y2, 2.5 * y1, rtol=1e-13, atol=1e-13)
    # slot j's term alone: zero the other slot's weight
    w0 = w.copy()
    w0[:, 1] = 0.0
    y0 = O.moe_unsharded(x, ids, w0, wg, wu, wd)
    for t in range(5):
        e = ids[t, 0]
        assert np.allclose(y0[t], w[t, 0] * O.mlp_unsharded(x[t:t + 1], wg[e], wu[e], wd[e])[0])


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,e,k", [(1, 4, 2), (2, 4, 2), (4, 8, 2), (4, 2, 1), (8, 8, 3)])
def test_sharded_modes_equal_the_plain_mixture(mode, n, e, k):
    if mode == O.MOE_WITHIN_EXPERT and 8 % n:
        pytest.skip("F must split over the ranks")
    wg, wu, wd = _experts(e, 4, 8, n * e + k)
    x = np.random.default_rng(n).standard_normal((6, 4))
    ids, w = _routing(6, e, k, 3 * n)
    ref = O.moe_unsharded(x, ids, w, wg, wu, wd)
    out = O.moe_sharded(x, ids, w, wg, wu, wd, n, mode)
    for r in range(n):
        assert np.allclose(out["y"][r], ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(sum(out["partials"]), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_integer_inputs_are_exact(mode):
    """Small-integer weights and inputs with gate sums that are large and
    positive (silu(g) = g up to e^-g) keep every product exact; each rank's
    partial is then compared with loops over the work that mode gives it."""
    n, e, k, d, f = 2, 4, 2, 2, 4
    wg, wu, wd = _experts(e, d, f, 11, ints=True)
    wg = [np.abs(g) + 20.0 for g in wg]  # gate sums >= 40: silu(g) == g in float64
    x = np.ones((3, d))
    ids = np.array([[0, 1], [2, 3], [1, 2]])
    w = np.array([[1.0, 2.0], [0.5, 0.25], [3.0, 1.0]])
    out = O.moe_sharded(x, ids, w, wg, wu, wd, n, mode)
    for r in range(n):
        want = np.zeros((3, d))
        for t, j in itertools.product(range(3), range(k)):
            ex = ids[t, j]
            if mode == O.MOE_EXPERT_PARALLEL and ex % n != r:
                continue
            fs = range(f) if mode == O.MOE_EXPERT_PARALLEL else range(r * f // n, (r + 1) * f // n)
            for o in range(d):
                want[t, o] += w[t, j] * sum((x[t] @ wg[ex][ff]) * (x[t] @ wu[ex][ff]) * wd[ex][o, ff] for ff in fs)
        assert np.array_equal(out["partials"][r], want), f"rank {r}"


def test_expert_parallel_partials_only_hold_local_experts():
    n, e = 4, 8
    wg, wu, wd = _experts(e, 3, 4, 9)
    x = np.random.default_rng(1).standard_normal((5, 3))
    ids = np.array([[0, 4], [1, 5], [0, 1], [4, 0], [6, 2]])  # rank 3 (experts 3, 7) gets nothing
    w = np.full((5, 2), 0.5)
    out = O.moe_sharded(x, ids, w, wg, wu, wd, n, O.MOE_EXPERT_PARALLEL)
    assert np.all(out["partials"][3] == 0.0)
    assert np.all(out["partials"][0][[1, 4]] == 0.0)  # tokens 1 and 4 route to no expert of rank 0
    assert np.all(out["partials"][2][:4] == 0.0)


@pytest.mark.parametrize("n", [2, 4, 8])
def test_moe_all_reduce_messages(n):
    wg, wu, wd = _experts(n, 2, 8, n)
    x = np.random.default_rng(n).standard_normal((4, 2))
    ids, w = _routing(4, n, 2, n)
    log = O.RingLog(n)
    O.moe_sharded(x, ids, w, wg, wu, wd, n, O.MOE_WITHIN_EXPERT, log=log)
    size = 4 * 2 * 8
    for r in range(n):
        assert log.bytes_sent(r) == 2 * (n - 1) * size // n


# ---- planted mistakes must trip the pins above ----------------------------------
import oracle.tp_oracle as T  # noqa: E402


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(T, name, fn)
    monkeypatch.setattr(O, name, fn)


def _fails(check, *args):
    with pytest.raises(AssertionError):
        check(*args)


def test_mutation_contiguous_expert_blocks_are_caught(monkeypatch):
    _patch(monkeypatch, "expert_rank", lambda i, n: i * n // 4)  # blocks of E/N experts
    _fails(test_expert_placement_matches_the_flowchart)


def test_mutation_unweighted_slots_are_caught(monkeypatch):
    def unweighted(x, topk_ids, topk_w, wg, wu, wd):
        x = np.asarray(x, dtype=np.float64)
        ids = np.asarray(topk_ids)
        y = np.zeros((x.shape[0], np.asarray(wd[0]).shape[0]))
        for t in range(x.shape[0]):
            for j in range(ids.shape[1]):
                e = ids[t, j]
                y[t] += T.mlp_unsharded(x[t:t + 1], wg[e], wu[e], wd[e])[0]
        return y
    _patch(monkeypatch, "moe_unsharded", unweighted)
    _fails(test_linear_in_the_routing_weights)


def test_mutation_wrong_slot_weight_is_caught(monkeypatch):
    orig = T.moe_unsharded

    def swapped(x, topk_ids, topk_w, wg, wu, wd):
        return orig(x, topk_ids, np.asarray(topk_w)[:, ::-1], wg, wu, wd)
    _patch(monkeypatch, "moe_unsharded", swapped)
    _fails(test_moe_unsharded_by_loops, 3, 4, 2, 3, 4)
