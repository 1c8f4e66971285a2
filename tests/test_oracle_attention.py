"""Pins of the oracle's attention core (the step between the q/k/v and o_proj
projections; [MLX] GQA 인식 어텐션 샤딩: every local q head attends with the kv
head the plan maps it to, K/V sharded or replicated).

Each pin checks the oracle against something other than its own formula:
closed forms (the first causal row sees only key 0; equal scores average the
visible values; two keys give a logistic weight with the 1/sqrt(d) scale),
explicit loops with math.exp, invariance to a shift shared by all keys, a key
that dominates, and the q -> kv grouping read off values that are constant per
kv head.
"""
import itertools
import math

import numpy as np
import pytest

import oracle as O


def _loops(q, k, v, causal):
    t, d = q.shape
    out = np.zeros((t, v.shape[1]))
    for i in range(t):
        js = [j for j in range(t) if (j <= i or not causal)]
        s = [sum(q[i, c] * k[j, c] for c in range(d)) / math.sqrt(d) for j in js]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        for j, w in zip(js, e):
            out[i] += w / z * v[j]
    return out


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("t,d", [(5, 3), (4, 8), (1, 2)])
def test_attention_head_by_loops(t, d, causal):
    g = np.random.default_rng(t * d)
    q, k, v = g.standard_normal((t, d)), g.standard_normal((t, d)), g.standard_normal((t, d))
    assert np.allclose(O.attention_head(q, k, v, causal), _loops(q, k, v, causal), rtol=1e-12, atol=1e-12)


def test_first_causal_row_is_the_first_value():
    g = np.random.default_rng(1)
    q, k, v = g.standard_normal((6, 4)), g.standard_normal((6, 4)), g.standard_normal((6, 4))
    assert np.array_equal(O.attention_head(q, k, v, True)[0], v[0])


@pytest.mark.parametrize("causal", [True, False])
def test_equal_scores_average_the_visible_values(causal):
    g = np.random.default_rng(2)
    t = 7
    v = g.standard_normal((t, 3))
    a = O.attention_head(np.zeros((t, 3)), g.standard_normal((t, 3)), v, causal)
    want = np.cumsum(v, axis=0) / np.arange(1, t + 1)[:, None] if causal else np.tile(v.mean(axis=0), (t, 1))
    assert np.allclose(a, want, rtol=1e-13, atol=1e-13)


def test_two_keys_give_the_logistic_weight_with_the_scale():
    d = 4
    q = np.array([[1.0, 0, 0, 0], [3.0, 0, 0, 0]])
    k = np.array([[0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    v = np.array([[0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    a = O.attention_head(q, k, v, causal=True)
    # query 1 sees both keys: scores 0 and 3/sqrt(4) = 1.5, weight of key 1 = 1/(1+e^-1.5)
    assert abs(a[1, 0] - 1.0 / (1.0 + math.exp(-1.5))) < 1e-15
    assert a[0, 0] == 0.0


def test_a_shift_shared_by_all_keys_changes_nothing():
    g = np.random.default_rng(3)
    q, k, v = g.standard_normal((5, 4)), g.standard_normal((5, 4)), g.standard_normal((5, 4))
    shifted = k + g.standard_normal((1, 4))
    for causal in (True, False):
        assert np.allclose(O.attention_head(q, shifted, v, causal), O.attention_head(q, k, v, causal),
                           rtol=1e-12, atol=1e-12)


def test_a_dominant_visible_key_is_picked():
    t, d = 6, 8
    k = 40.0 * np.eye(t, d)          # key j points along axis j
    v = np.arange(t * 2, dtype=np.float64).reshape(t, 2)
    q = 40.0 * np.eye(t, d)[[3, 3, 3, 3, 3, 3]]   # every query points at key 3
    a = O.attention_head(q, k, v, causal=True)
    assert np.allclose(a[3:], np.tile(v[3], (3, 1)), atol=1e-12)
    # queries before key 3 cannot see it: equal scores over their visible keys
    assert np.allclose(a[1], v[:2].mean(axis=0), atol=1e-12)


@pytest.mark.parametrize("tp_size,hq,hkv", [(2, 8, 2), (4, 8, 2), (4, 32, 8), (8, 32, 4), (1, 4, 4)])
def test_each_q_head_uses_its_gqa_kv_head(tp_size, hq, hkv):
    """Values constant per kv head (head g holds g + 1) make every output column
    of q head h equal 1 + its kv head, which the GQA grouping fixes: global q head
    h reads global kv head h // (hq / hkv)."""
    d, t = 4, 5
    plan = O.shard_plan(tp_size, 64, hq, hkv, d, 8 * tp_size)
    g = np.random.default_rng(tp_size + hq)
    rep = plan[0].kv_replicated
    nkv_src = 1 if rep else tp_size
    q, k, v = [], [], []
    for r, s in enumerate(plan):
        q.append(g.standard_normal((t, (s.q_heads[1] - s.q_heads[0]) * d)))
    for r in range(nkv_src):
        s = plan[r]
        heads = range(s.kv_heads[0], s.kv_heads[1])
        k.append(g.standard_normal((t, len(heads) * d)))
        v.append(np.concatenate([np.full((t, d), float(h + 1)) for h in heads], axis=1))
    a = O.attention_core_sharded(q, k, v, plan, d, causal=True)
    for r, s in enumerate(plan):
        for j, hglob in enumerate(range(s.q_heads[0], s.q_heads[1])):
            want = hglob // (hq // hkv) + 1
            assert np.allclose(a[r][:, j * d:(j + 1) * d], want, rtol=1e-13), (r, hglob)


# ---- planted mistakes must trip the pins above ----------------------------------
import oracle.tp_oracle as T  # noqa: E402


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(T, name, fn)
    monkeypatch.setattr(O, name, fn)


def _fails(check, *args):
    with pytest.raises(AssertionError):
        check(*args)


def test_mutation_missing_scale_is_caught(monkeypatch):
    def unscaled(q, k, v, causal):
        q = np.asarray(q, dtype=np.float64)
        s = q @ np.asarray(k, dtype=np.float64).T
        if causal:
            n = s.shape[0]
            s = np.where(np.arange(n)[None, :] <= np.arange(n)[:, None], s, -np.inf)
        return T.softmax_rows(s) @ np.asarray(v, dtype=np.float64)
    _patch(monkeypatch, "attention_head", unscaled)
    _fails(test_two_keys_give_the_logistic_weight_with_the_scale)


def test_mutation_strict_causal_mask_is_caught(monkeypatch):
    def strict(q, k, v, causal):
        q = np.asarray(q, dtype=np.float64)
        s = q @ np.asarray(k, dtype=np.float64).T / np.sqrt(q.shape[1])
        n = s.shape[0]
        s = np.where(np.arange(n)[None, :] < np.arange(n)[:, None] + 0 * causal, s, -np.inf)
        s[0, 0] = 0.0  # keep row 0 finite; it then attends to key 0 with score 0
        return T.softmax_rows(s) @ np.asarray(v, dtype=np.float64)
    _patch(monkeypatch, "attention_head", strict)
    _fails(test_attention_head_by_loops, 5, 3, True)


def test_mutation_round_robin_kv_heads_are_caught(monkeypatch):
    orig = T.attention_core_sharded

    def round_robin(q, k, v, plan, head_dim, causal=True):
        for s in plan:
            n_kv = s.kv_heads[1] - s.kv_heads[0]
            s.q_to_kv = [h % n_kv for h in range(len(s.q_to_kv))]
        return orig(q, k, v, plan, head_dim, causal)
    _patch(monkeypatch, "attention_core_sharded", round_robin)
    _fails(test_each_q_head_uses_its_gqa_kv_head, 4, 32, 8)
