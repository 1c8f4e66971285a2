"""Pins of the oracle's SwiGLU and of the sharded MLP / attention-projection blocks.

The pages name no activation; the MLP block uses SwiGLU silu(g)*u with
silu(x) = x*sigmoid(x). Closed forms: sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4,
silu(x) - silu(-x) = x. The blocks are pinned by 'sharded equals unsharded'
(railscraft wiki '텐서 병렬 처리', 상세 1, last paragraph: the column/row pattern
applies to QKV / output projections and the MLP) and by brute force.
"""
import math

import numpy as np
import pytest

import oracle as O


def check_silu_closed_forms():
    assert O.silu(np.array([0.0]))[0] == 0.0
    ln3 = math.log(3.0)
    assert abs(O.silu(np.array([ln3]))[0] - 0.75 * ln3) < 1e-15
    assert abs(O.silu(np.array([-ln3]))[0] + 0.25 * ln3) < 1e-15
    x = np.linspace(-30, 30, 601)
    assert np.max(np.abs(O.silu(x) - O.silu(-x) - x)) < 1e-12
    h = 1e-6
    d0 = (O.silu(np.array([h]))[0] - O.silu(np.array([-h]))[0]) / (2 * h)
    assert abs(d0 - 0.5) < 1e-9


def test_silu_closed_forms():
    check_silu_closed_forms()


def test_silu_limits():
    assert O.silu(np.array([60.0]))[0] == pytest.approx(60.0, rel=1e-15)
    big_neg = O.silu(np.array([-1000.0]))[0]
    assert big_neg == 0.0 and not math.isnan(big_neg)
    assert abs(O.silu(np.array([-40.0]))[0]) < 1e-15


def test_swiglu_special_cases():
    g = np.array([0.0, 2.0, -3.0, 50.0])
    assert np.array_equal(O.swiglu(g, np.zeros(4)), np.zeros(4))
    assert O.swiglu(np.array([0.0]), np.array([7.0]))[0] == 0.0
    assert O.swiglu(np.array([50.0]), np.array([2.0]))[0] == pytest.approx(100.0, rel=1e-15)


def _rand(seed, shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


@pytest.mark.parametrize("tp", [1, 2, 4])
def test_mlp_sharded_equals_unsharded(tp):
    T, D, F = 7, 16, 32
    x, wg, wu, wd = _rand(1, (T, D)), _rand(2, (F, D)), _rand(3, (F, D)), _rand(4, (D, F))
    out = O.mlp_sharded(x, wg, wu, wd, tp)
    ref = O.mlp_unsharded(x, wg, wu, wd)
    for y in out["y"]:
        assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))
        assert np.array_equal(y, out["y"][0])
    h_full = O.swiglu(O.linear(x, wg), O.linear(x, wu))
    hcat = np.concatenate(out["h"], axis=1)
    assert np.max(np.abs(hcat - h_full)) <= 1e-12 * np.max(np.abs(h_full))


def test_mlp_brute_force_tiny():
    T, D, F, tp = 2, 3, 4, 2
    x, wg, wu, wd = _rand(5, (T, D)), _rand(6, (F, D)), _rand(7, (F, D)), _rand(8, (D, F))
    y = O.mlp_sharded(x, wg, wu, wd, tp)["y"][0]
    for i in range(T):
        h = []
        for f in range(F):
            g = sum(x[i, k] * wg[f, k] for k in range(D))
            u = sum(x[i, k] * wu[f, k] for k in range(D))
            h.append(g / (1.0 + math.exp(-g)) * u)
        for j in range(D):
            assert abs(y[i, j] - sum(h[f] * wd[j, f] for f in range(F))) < 1e-12


@pytest.mark.parametrize("tp,hq,hkv", [(4, 8, 4), (8, 8, 4), (2, 4, 1), (1, 4, 2)])
def test_attn_proj_sharded_equals_unsharded(tp, hq, hkv):
    T, D, hd = 5, 16, 4
    x, a = _rand(9, (T, D)), _rand(10, (T, hq * hd))
    wq, wk, wv = _rand(11, (hq * hd, D)), _rand(12, (hkv * hd, D)), _rand(13, (hkv * hd, D))
    wo = _rand(14, (D, hq * hd))
    plan = O.shard_plan(tp, D, hq, hkv, hd, 8 * tp)
    out = O.attn_proj_sharded(x, wq, wk, wv, a, wo, plan, hd)
    ref = O.attn_proj_unsharded(x, wq, wk, wv, a, wo)
    assert np.max(np.abs(np.concatenate(out["q"], 1) - ref["q"])) < 1e-12
    if hkv < tp:
        for r in range(tp):
            assert np.max(np.abs(out["k"][r] - ref["k"])) < 1e-12
            assert np.max(np.abs(out["v"][r] - ref["v"])) < 1e-12
    else:
        assert np.max(np.abs(np.concatenate(out["k"], 1) - ref["k"])) < 1e-12
        assert np.max(np.abs(np.concatenate(out["v"], 1) - ref["v"])) < 1e-12
    for y in out["y"]:
        assert np.max(np.abs(y - ref["y"])) <= 1e-12 * np.max(np.abs(ref["y"]))
