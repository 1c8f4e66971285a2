"""Pins of the oracle's linear algebra (column / row parallel, concatenation).

Sources: railscraft wiki '텐서 병렬 처리', 상세 1 (Y_i = X W_i, Y = [Y_1..Y_n];
Y_i = X_i W_i, Y = sum Y_i) and 예시 1 (weights stored [out x in], Y_i = X W_i^T,
printed shapes); mlxcel manual '텐서 병렬화', Column Parallel / Row Parallel.
"""
import json
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ints(seed, shape, lo=-4, hi=4):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=shape).astype(np.float64)


# --- the Y = X W^T convention, against special cases and brute force --------
def check_identity_weight():
    x = _ints(1, (5, 7))
    assert np.array_equal(O.linear(x, np.eye(7)), x)


def check_permutation_weight():
    # W[j, perm[j]] = 1 selects input feature perm[j] into output j.
    x = _ints(2, (4, 6))
    perm = np.array([3, 0, 5, 1, 4, 2, 3, 0])            # 8 outputs, 6 inputs
    w = np.zeros((8, 6))
    w[np.arange(8), perm] = 1.0
    y = O.linear(x, w)
    assert y.shape == (4, 8)
    assert np.array_equal(y, x[:, perm])


def check_brute_force(seed=3, T=3, K=5, N=4):
    x, w = _ints(seed, (T, K)), _ints(seed + 1, (N, K))
    y = O.linear(x, w)
    for i in range(T):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += x[i, k] * w[j, k]
            assert y[i, j] == acc


def check_column_concat_exact(tp, seed=11, T=6, K=16, out=32):
    x, w = _ints(seed, (T, K)), _ints(seed + 1, (out, K))
    shards = O.split_rows(w, tp)
    ys = O.column_parallel(x, shards)
    assert len(ys) == tp
    for y in ys:
        assert y.shape == (T, out // tp)
    assert np.array_equal(O.all_gather_columns(ys), O.linear(x, w))


def check_row_sum_exact(tp, seed=21, T=5, K=32, out=12):
    x, w = _ints(seed, (T, K)), _ints(seed + 1, (out, K))
    parts = O.row_parallel(O.split_cols(x, tp), O.split_cols(w, tp))
    assert len(parts) == tp
    assert np.array_equal(sum(parts), O.linear(x, w))


def test_identity_weight():
    check_identity_weight()


def test_permutation_weight_catches_transpose():
    check_permutation_weight()


def test_brute_force_tiny():
    for s in range(5):
        check_brute_force(seed=10 * s, T=1 + s, K=2 + s, N=3 + s)


def test_closed_form_ones():
    # X = 1, W = 1: every output equals K.
    assert np.array_equal(O.linear(np.ones((3, 9)), np.ones((4, 9))), np.full((3, 4), 9.0))


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_column_parallel_concat_equals_unsharded(tp):
    check_column_concat_exact(tp)


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_row_parallel_sum_equals_unsharded(tp):
    check_row_sum_exact(tp)


def test_row_parallel_partial_depends_only_on_own_slice():
    tp, T, K, out = 4, 3, 16, 5
    x, w = _ints(5, (T, K)), _ints(6, (out, K))
    base = O.row_parallel(O.split_cols(x, tp), O.split_cols(w, tp))
    x2 = x.copy()
    x2[:, 4:8] += 1.0                 # disturb rank 1's slice only
    moved = O.row_parallel(O.split_cols(x2, tp), O.split_cols(w, tp))
    for r in range(tp):
        assert np.array_equal(base[r], moved[r]) == (r != 1)


def test_float_inputs_sharded_matches_unsharded():
    rng = np.random.default_rng(7)
    x, w = rng.standard_normal((9, 64)), rng.standard_normal((24, 64))
    for tp in (2, 4, 8):
        yc = O.all_gather_columns(O.column_parallel(x, O.split_rows(w, tp)))
        yr = sum(O.row_parallel(O.split_cols(x, tp), O.split_cols(w, tp)))
        ref = O.linear(x, w)
        assert np.max(np.abs(yc - ref)) <= 1e-12 * np.max(np.abs(ref))
        assert np.max(np.abs(yr - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_wiki_worked_example_shapes():
    g = json.load(open(os.path.join(GOLDEN, "wiki_column_example.json")))
    rng = np.random.default_rng(0)
    x = rng.standard_normal(tuple(g["input_shape"]))
    w = rng.standard_normal((g["out_features"], g["in_features"]))
    shards = O.split_rows(w, g["num_gpus"])
    assert [list(s.shape) for s in shards] == [g["shard_shape"]] * g["num_gpus"]
    y = O.all_gather_columns(O.column_parallel(x, shards))
    assert list(y.shape) == g["output_shape"]
    ref = O.linear(x, w)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))
