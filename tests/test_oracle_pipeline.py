"""Pins of the oracle's row-parallel -> reduce-scatter -> column-parallel pipeline
and of its bfloat16 rounding ([MLX] 통신 패턴, Reduce-scatter: used when a
row-parallel result goes straight into a column-parallel op, so that the
all-gather step is avoided).

Each pin checks the oracle against something other than its own formula:
the bf16 rounding against a brute-force choice of the nearest bfloat16 (ties to
even); the pipeline against explicit loops on tiny integer inputs, against the
ring's message log (no all-gather message, (N-1)/N of the tensor sent per
rank), and against the all-reduce's result chunk by chunk.
"""
import itertools

import numpy as np
import pytest

import oracle as O


def _nearest_bf16_brute(x32: np.ndarray) -> np.ndarray:
    """The bfloat16 nearest to each float32, chosen by comparing the two
    candidates that bracket it (ties go to the candidate with an even last
    mantissa bit)."""
    out = np.empty(x32.shape, dtype=np.float64)
    for i, v in enumerate(x32.reshape(-1)):
        bits = int(np.float32(v).view(np.uint32))
        lo_bits = bits & 0xFFFF0000
        hi_bits = (lo_bits + 0x10000) & 0xFFFFFFFF
        lo = float(np.uint32(lo_bits).view(np.float32))
        hi = float(np.uint32(hi_bits).view(np.float32))
        dv = float(v)
        d_lo, d_hi = abs(dv - lo), abs(hi - dv)
        if d_lo < d_hi:
            out.reshape(-1)[i] = lo
        elif d_hi < d_lo:
            out.reshape(-1)[i] = hi
        else:
            out.reshape(-1)[i] = lo if ((lo_bits >> 16) & 1) == 0 else hi
    return out


def test_round_to_bf16_special_values():
    one = 1.0
    cases = {
        1.0: 1.0, -2.5: -2.5, 0.15625: 0.15625, 0.0: 0.0,
        one + 2.0 ** -8: 1.0,                      # halfway, ties to the even 1.0
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,      # halfway, ties to the even neighbour above
        one + 2.0 ** -8 + 2.0 ** -20: one + 2.0 ** -7,  # just above halfway
        -(one + 2.0 ** -8 + 2.0 ** -20): -(one + 2.0 ** -7),
        3.0 * 2.0 ** -130: 3.0 * 2.0 ** -130,      # subnormal, exactly representable
    }
    for x, want in cases.items():
        got = O.round_to_bf16(np.array([x], dtype=np.float32))[0]
        assert got == want, (x, got, want)


def test_round_to_bf16_is_the_nearest_bfloat16():
    g = np.random.default_rng(7)
    x = np.concatenate([g.standard_normal(3000) * 10.0 ** g.integers(-6, 6, 3000),
                        g.uniform(-1, 1, 1000)]).astype(np.float32)
    assert np.array_equal(O.round_to_bf16(x), _nearest_bf16_brute(x))


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_pipeline_sends_only_reduce_scatter_messages(n):
    t, k = 8, 6
    g = np.random.default_rng(11 + n)
    parts = [g.integers(-5, 6, (t, k)).astype(np.float64) for _ in range(n)]
    log = O.RingLog(n)
    O.reduce_scatter_then_column(parts, [np.ones((2, k))] * n, log=log)
    kinds = {m[0] for m in log.sends}
    assert kinds <= {"reduce_scatter"}
    assert len(log.sends) == n * (n - 1)
    assert log.steps("all_gather") == 0 and log.steps("reduce_scatter") == n - 1
    # (N-1) of N chunks leave every rank once: half the all-reduce's 2(N-1)/N
    for r in range(n):
        assert log.bytes_sent(r) == (n - 1) * (t * k // n) * 8  # t*k = 48 splits evenly


@pytest.mark.parametrize("n,t,k", [(2, 4, 3), (4, 6, 5), (8, 8, 2), (4, 7, 3)])
def test_pipeline_brute_force_integers(n, t, k):
    g = np.random.default_rng(100 + n * t + k)
    parts = [g.integers(-4, 5, (t, k)).astype(np.float64) for _ in range(n)]
    ws = [g.integers(-3, 4, (int(g.integers(1, 4)), k)).astype(np.float64) for _ in range(n)]
    out = O.reduce_scatter_then_column(parts, ws)
    # the input assembled from the reduced chunks is the sum of the partials
    full = np.zeros((t, k))
    for p in parts:
        for i, j in itertools.product(range(t), range(k)):
            full[i, j] += p[i, j]
    assert np.array_equal(out["x"], full)
    # each rank's output is the plain product with its weight shard, by loops
    for r, w in enumerate(ws):
        want = np.zeros((t, w.shape[0]))
        for i, o, j in itertools.product(range(t), range(w.shape[0]), range(k)):
            want[i, o] += full[i, j] * w[o, j]
        assert np.array_equal(out["y"][r], want)


@pytest.mark.parametrize("n,t,k", [(2, 16, 8), (4, 10, 6), (8, 16, 3)])
def test_pipeline_chunks_match_the_all_reduce(n, t, k):
    g = np.random.default_rng(5 * n + t)
    parts = [g.standard_normal((t, k)).astype(np.float32) for _ in range(n)]
    out = O.reduce_scatter_then_column(parts, [g.standard_normal((3, k))] * n, round_bf16=True)
    ar = O.ring_all_reduce(parts)
    for c in range(n):
        lo, hi = O.chunk_bounds(t * k, n, c)
        # the ring's fp32 fold, then one rounding to bfloat16
        assert np.array_equal(out["chunks"][c], _nearest_bf16_brute(ar[0][lo:hi]))
        assert np.array_equal(ar[c][lo:hi], ar[0][lo:hi])


# ---- planted mistakes must trip the pins above ----------------------------------
import oracle.tp_oracle as T  # noqa: E402


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(T, name, fn)
    monkeypatch.setattr(O, name, fn)


def _fails(check, *args):
    with pytest.raises(AssertionError):
        check(*args)


def test_mutation_truncating_bf16_is_caught(monkeypatch):
    def trunc(x):
        b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)
        return (b & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    _patch(monkeypatch, "round_to_bf16", trunc)
    _fails(test_round_to_bf16_special_values)


def test_mutation_ties_away_from_zero_is_caught(monkeypatch):
    def away(x):
        b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
        return ((b + 0x8000) & 0xFFFF0000).astype(np.uint32).view(np.float32).astype(np.float64)
    _patch(monkeypatch, "round_to_bf16", away)
    _fails(test_round_to_bf16_special_values)


def test_mutation_wrong_chunk_owner_is_caught(monkeypatch):
    orig = T.reduce_scatter_then_column

    def shifted(partials, w_shards, round_bf16=False, log=None):
        n = len(partials)
        t, k = np.asarray(partials[0]).shape
        rs = T.ring_reduce_scatter(partials, log)
        chunks = []
        for c in range(n):
            lo, hi = T.chunk_bounds(t * k, n, c)
            chunks.append(rs[(c + 1) % n][lo:hi])  # reads a rank that does not own chunk c
        x = T.gather_flat_shards(chunks).reshape(t, k)
        return {"chunks": chunks, "x": x, "y": T.column_parallel(x, w_shards)}
    _patch(monkeypatch, "reduce_scatter_then_column", shifted)
    _fails(test_pipeline_brute_force_integers, 4, 6, 5)
    assert orig is not shifted


def test_mutation_unreduced_chunks_are_caught(monkeypatch):
    def unreduced(partials, w_shards, round_bf16=False, log=None):
        n = len(partials)
        t, k = np.asarray(partials[0]).shape
        chunks = []
        for c in range(n):
            lo, hi = T.chunk_bounds(t * k, n, c)
            chunks.append(np.asarray(partials[c], dtype=np.float64).reshape(-1)[lo:hi])  # no reduction
        x = T.gather_flat_shards(chunks).reshape(t, k)
        return {"chunks": chunks, "x": x, "y": T.column_parallel(x, w_shards)}
    _patch(monkeypatch, "reduce_scatter_then_column", unreduced)
    _fails(test_pipeline_brute_force_integers, 2, 4, 3)
