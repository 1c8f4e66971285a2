"""Pins of the oracle's vocab-parallel embedding lookup and LM head ([MLX] 가중치
샤딩 전략, Vocab Parallel: every rank owns one contiguous slice of the token
vocabulary, used for the embedding lookup and the LM-head logits; 임베딩 및 LM
Head 샤딩, vocab_parallel: the vocabulary dimension is sharded and the lookup and
the logits need an all-gather).

Each pin checks the oracle against something other than its own formula: the
lookup against a one-hot matrix product and against explicit loops; the pieces
against the slice rule; the all-gather against its message log; the logits
against loops, against a weight whose rows expose the column order, and against
a tied table whose argmax must return the token ids.
"""
import itertools

import numpy as np
import pytest

import oracle as O


def _table(v, d, seed):
    return np.random.default_rng(seed).integers(-9, 10, (v, d)).astype(np.float64)


def _boundary_ids(v, n, extra, seed):
    """Every slice's first and last id, plus random ids (repeats included)."""
    per = v // n
    ids = [b for r in range(n) for b in (r * per, (r + 1) * per - 1)]
    ids += list(np.random.default_rng(seed).integers(0, v, extra))
    return np.array(ids, dtype=np.int64)


def test_embedding_is_the_one_hot_product():
    v, d = 24, 5
    t = _table(v, d, 1)
    ids = _boundary_ids(v, 4, 30, 2)
    one_hot = np.zeros((ids.size, v))
    one_hot[np.arange(ids.size), ids] = 1.0
    assert np.array_equal(O.embedding(ids, t), one_hot @ t)


@pytest.mark.parametrize("v,n", [(8, 1), (16, 2), (24, 4), (64, 8)])
def test_vocab_ranges_are_contiguous_equal_slices(v, n):
    r = O.vocab_ranges(v, n)
    assert r[0][0] == 0 and r[-1][1] == v
    assert all(r[i][1] == r[i + 1][0] for i in range(n - 1))
    assert len({hi - lo for lo, hi in r}) == 1


@pytest.mark.parametrize("v,n,kind", [(10, 4, "not_divisible"), (12, 3, "tp_size"), (0, 2, "not_divisible")])
def test_vocab_ranges_reject(v, n, kind):
    with pytest.raises(O.PlanError) as e:
        O.vocab_ranges(v, n)
    assert e.value.kind == kind


@pytest.mark.parametrize("v,n,d", [(8, 2, 3), (24, 4, 5), (64, 8, 2), (16, 1, 4)])
def test_vocab_parallel_embedding_brute_force(v, n, d):
    t = _table(v, d, v + n)
    ids = _boundary_ids(v, n, 20, v * n)
    out = O.vocab_parallel_embedding(ids, O.split_rows(t, n))
    want = np.zeros((ids.size, d))
    for i, j in itertools.product(range(ids.size), range(d)):
        want[i, j] = t[ids[i], j]
    for r in range(n):
        assert np.array_equal(out["y"][r], want), f"rank {r}"


@pytest.mark.parametrize("n", [2, 4, 8])
def test_pieces_partition_the_tokens_by_slice(n):
    v, d = 8 * n, 3
    ids = _boundary_ids(v, n, 25, n)
    out = O.vocab_parallel_embedding(ids, O.split_rows(_table(v, d, n), n))
    seen = []
    for r, (pos, rows) in enumerate(out["pieces"]):
        lo, hi = r * (v // n), (r + 1) * (v // n)
        assert all(lo <= ids[i] < hi for i in pos)
        assert rows.shape == (len(pos), d)
        seen += pos
    assert sorted(seen) == list(range(ids.size))


@pytest.mark.parametrize("n", [2, 4, 8])
def test_embedding_all_gather_messages(n):
    v, d = 4 * n, 2
    ids = _boundary_ids(v, n, 11, 3 * n)
    log = O.RingLog(n)
    out = O.vocab_parallel_embedding(ids, O.split_rows(_table(v, d, 7), n), log=log)
    assert log.steps("all_gather") == n - 1
    assert {m[0] for m in log.sends} == {"all_gather"}
    assert all(dst == (src + 1) % n for (_p, _s, src, dst, _c, _b) in log.sends)
    sizes = [rows.nbytes for (_pos, rows) in out["pieces"]]
    for r in range(n):
        # every piece but the one of the rank it sends to passes through rank r once
        assert log.bytes_sent(r) == sum(sizes) - sizes[(r + 1) % n]


def test_skewed_ids_all_in_one_slice():
    n, v, d = 4, 32, 3
    t = _table(v, d, 9)
    ids = np.array([8, 9, 15, 8, 12])  # all in rank 1's slice
    out = O.vocab_parallel_embedding(ids, O.split_rows(t, n))
    assert [len(p[0]) for p in out["pieces"]] == [0, 5, 0, 0]
    assert np.array_equal(out["y"][3], t[ids])


def test_empty_ids():
    out = O.vocab_parallel_embedding(np.zeros(0, dtype=np.int64), O.split_rows(_table(8, 2, 1), 2))
    assert all(y.shape == (0, 2) for y in out["y"])


@pytest.mark.parametrize("bad", [-1, 16])
def test_out_of_range_ids_raise(bad):
    with pytest.raises(ValueError):
        O.vocab_parallel_embedding([0, bad], O.split_rows(_table(16, 2, 1), 2))
    with pytest.raises(ValueError):
        O.embedding([bad], _table(16, 2, 1))


@pytest.mark.parametrize("n,t,d,v", [(2, 3, 4, 8), (4, 2, 3, 16), (8, 2, 2, 16)])
def test_lm_head_brute_force(n, t, d, v):
    g = np.random.default_rng(n * v)
    x = g.integers(-4, 5, (t, d)).astype(np.float64)
    w = g.integers(-4, 5, (v, d)).astype(np.float64)
    out = O.vocab_parallel_lm_head(x, O.split_rows(w, n))
    want = np.zeros((t, v))
    for i, o, j in itertools.product(range(t), range(v), range(d)):
        want[i, o] += x[i, j] * w[o, j]
    assert np.array_equal(out["logits"], want)
    per = v // n
    for r in range(n):
        assert np.array_equal(out["parts"][r], want[:, r * per:(r + 1) * per])


def test_lm_head_column_order():
    """Row v of the weight picks input feature v mod D, scaled by v + 1: logit
    column v must then equal (v + 1) * x[:, v mod D], so any misplaced shard shows."""
    n, d, v = 4, 3, 16
    x = np.random.default_rng(4).standard_normal((5, d))
    w = np.zeros((v, d))
    for o in range(v):
        w[o, o % d] = o + 1
    logits = O.vocab_parallel_lm_head(x, O.split_rows(w, n))["logits"]
    for o in range(v):
        assert np.array_equal(logits[:, o], (o + 1) * x[:, o % d])


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_tied_table_argmax_recovers_the_ids(n):
    """With the table c*I (V = D) used both to embed and as the LM head, the
    logits of token t are c^2 at column t and 0 elsewhere: the argmax is t."""
    v = 16
    table = 3.0 * np.eye(v)
    ids = _boundary_ids(v, n, 10, 5)
    x = O.vocab_parallel_embedding(ids, O.split_rows(table, n))["y"][0]
    logits = O.vocab_parallel_lm_head(x, O.split_rows(table, n))["logits"]
    assert np.array_equal(np.argmax(logits, axis=1), ids)


# ---- planted mistakes must trip the pins above ----------------------------------
import oracle.tp_oracle as T  # noqa: E402


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(T, name, fn)
    monkeypatch.setattr(O, name, fn)


def _fails(check, *args):
    with pytest.raises(AssertionError):
        check(*args)


def _embedding_with(local_row, owns):
    """A vocab-parallel lookup whose ownership rule owns(t, r, per, n) and local
    row local_row(t, r, per, n) are replaced."""
    def emb(ids, table_shards, log=None):
        ids = np.asarray(ids, dtype=np.int64).reshape(-1)
        n = len(table_shards)
        per = np.asarray(table_shards[0]).shape[0]
        d = np.asarray(table_shards[0]).shape[1]
        pieces = []
        for r in range(n):
            pos = [i for i in range(ids.size) if owns(ids[i], r, per, n)]
            shard = np.asarray(table_shards[r], dtype=np.float64)
            rows = np.array([shard[local_row(ids[i], r, per, n)] for i in pos]).reshape(len(pos), d)
            pieces.append((pos, rows))
        y = np.full((ids.size, d), np.nan)
        for pos, rows in pieces:
            for j, i in enumerate(pos):
                y[i] = rows[j]
        return {"pieces": pieces, "y": [y.copy() for _ in range(n)]}
    return emb


def test_mutation_round_robin_slices_are_caught(monkeypatch):
    # ids dealt to ranks cyclically (t mod N) instead of in contiguous slices
    _patch(monkeypatch, "vocab_parallel_embedding",
           _embedding_with(lambda t, r, per, n: t // n, lambda t, r, per, n: t % n == r))
    _fails(test_vocab_parallel_embedding_brute_force, 24, 4, 5)


def test_mutation_slice_boundary_off_by_one_is_caught(monkeypatch):
    _patch(monkeypatch, "vocab_parallel_embedding",
           _embedding_with(lambda t, r, per, n: (t - r * per) % per,
                           lambda t, r, per, n: r * per < t <= (r + 1) * per))
    _fails(test_pieces_partition_the_tokens_by_slice, 4)


def test_mutation_reversed_logit_shards_are_caught(monkeypatch):
    def reversed_head(x, w_shards):
        parts = T.column_parallel(x, w_shards)
        return {"parts": parts, "logits": T.all_gather_columns(parts[::-1])}
    _patch(monkeypatch, "vocab_parallel_lm_head", reversed_head)
    _fails(test_lm_head_column_order)
