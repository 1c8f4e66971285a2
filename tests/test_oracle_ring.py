"""Pins of the oracle's ring collectives.

Source: mlxcel manual '텐서 병렬화', 통신 패턴 (Communication patterns): ring
all-reduce = reduce-scatter + all-gather, 2*(N-1)/N*tensor_size per rank; rank r
sends to (r+1)%N and receives from (r+N-1)%N; N-1 steps. Fixture:
tests/golden/ring_rule.json.
"""
import numpy as np
import pytest

import oracle as O

SIZES = [0, 1, 3, 7, 64, 1000, 4099]
NS = [1, 2, 4, 8]


def _bufs(n, size, seed=0):
    rng = np.random.default_rng(seed)
    return [rng.integers(-50, 51, size=size).astype(np.float64) for _ in range(n)]


def check_rs_owns_reduced_chunk(n, size):
    bufs = _bufs(n, size, seed=n * 1000 + size)
    total = sum(bufs) if n else None
    out = O.ring_reduce_scatter(bufs)
    for r in range(n):
        lo, hi = O.chunk_bounds(size, n, r)
        assert np.array_equal(out[r][lo:hi], total[lo:hi]), (n, size, r)


def check_allreduce_everywhere(n, size):
    bufs = _bufs(n, size, seed=7 + n + size)
    total = sum(bufs)
    out = O.ring_all_reduce(bufs)
    for r in range(n):
        assert np.array_equal(out[r], total)


def check_each_contribution_once(n, size):
    # Rank r contributes (n+1)^r everywhere. A sum of these with multiplicities
    # m_r <= n equals sum_r (n+1)^r only when every m_r is exactly 1.
    base = float(n + 1)
    bufs = [np.full(size, base ** r) for r in range(n)]
    expect = sum(base ** r for r in range(n))
    for y in O.ring_all_reduce(bufs):
        assert np.all(y == expect)


def check_neighbour_and_steps(n, size):
    log = O.RingLog(n)
    O.ring_all_reduce(_bufs(n, size), log)
    for phase in ("reduce_scatter", "all_gather"):
        sends = [s for s in log.sends if s[0] == phase]
        assert log.steps(phase) == (n - 1 if n > 1 else 0)
        for (_p, step, src, dst, _c, _b) in sends:
            assert dst == (src + 1) % n
            assert 0 <= step < n - 1
        # every rank sends exactly once per step and receives from (r+N-1)%N
        for step in range(n - 1):
            srcs = sorted(s[2] for s in sends if s[1] == step)
            assert srcs == list(range(n))
            for s in sends:
                if s[1] == step:
                    assert s[2] == (s[3] + n - 1) % n


def check_volume_formula(n, size, elem_bytes=8):
    # tensor_size divisible by N: per rank exactly (N-1)/N*S per phase, 2(N-1)/N*S total.
    log = O.RingLog(n)
    O.ring_all_reduce(_bufs(n, size), log)
    S = size * elem_bytes
    for r in range(n):
        assert log.bytes_sent(r, "reduce_scatter") * n == (n - 1) * S
        assert log.bytes_sent(r, "all_gather") * n == (n - 1) * S
        assert log.bytes_sent(r) * n == 2 * (n - 1) * S


def check_step_order(n):
    # Non-commutative "+" (tuple concatenation) records the order in which the
    # contributions entered each element: chunk c must fold c+1, c+2, ..., c.
    size = 2 * n
    bufs = []
    for r in range(n):
        b = np.empty(size, dtype=object)
        for i in range(size):
            b[i] = (r,)
        bufs.append(b)
    out = O.ring_all_reduce(bufs)
    for c in range(n):
        lo, hi = O.chunk_bounds(size, n, c)
        expect = tuple((c + 1 + j) % n for j in range(n))
        for r in range(n):
            for i in range(lo, hi):
                assert out[r][i] == expect, (n, c, r, out[r][i])


@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("size", SIZES)
def test_reduce_scatter_rank_r_owns_chunk_r(n, size):
    check_rs_owns_reduced_chunk(n, size)


@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("size", SIZES)
def test_allreduce_gives_sum_on_every_rank(n, size):
    check_allreduce_everywhere(n, size)


@pytest.mark.parametrize("n", NS)
def test_each_contribution_exactly_once(n):
    check_each_contribution_once(n, 37)


@pytest.mark.parametrize("n", NS)
def test_ring_neighbour_rule_and_step_count(n):
    check_neighbour_and_steps(n, 40)


@pytest.mark.parametrize("n", [2, 4, 8])
@pytest.mark.parametrize("size", [8, 64, 4096])
def test_volume_is_2_nm1_over_n_times_size(n, size):
    check_volume_formula(n, size)


def test_volume_ragged_counts_all_but_own_chunk():
    n, size = 4, 10
    log = O.RingLog(n)
    O.ring_all_reduce(_bufs(n, size), log)
    for r in range(n):
        lo, hi = O.chunk_bounds(size, n, r)
        lo1, hi1 = O.chunk_bounds(size, n, (r + 1) % n)
        assert log.bytes_sent(r, "reduce_scatter") == (size - (hi - lo)) * 8
        assert log.bytes_sent(r, "all_gather") == (size - (hi1 - lo1)) * 8


@pytest.mark.parametrize("n", [2, 3, 4, 8])
def test_fold_order_follows_step_rule(n):
    check_step_order(n)


def test_all_gather_from_owned_chunks():
    n, size = 4, 13
    full = np.arange(size, dtype=np.float64) + 1
    bufs = []
    for r in range(n):
        b = np.zeros(size)
        lo, hi = O.chunk_bounds(size, n, r)
        b[lo:hi] = full[lo:hi]
        bufs.append(b)
    for y in O.ring_all_gather(bufs):
        assert np.array_equal(y, full)


def test_fp32_buffers_compute_in_fp32():
    rng = np.random.default_rng(3)
    bufs = [rng.standard_normal(100).astype(np.float32) for _ in range(4)]
    out = O.ring_all_reduce(bufs)
    assert all(o.dtype == np.float32 for o in out)
    for o in out[1:]:
        assert np.array_equal(o.view(np.uint32), out[0].view(np.uint32))
    ref = sum(b.astype(np.float64) for b in bufs)
    assert np.max(np.abs(out[0] - ref)) < 1e-5


def test_inputs_untouched():
    bufs = _bufs(4, 20)
    keep = [b.copy() for b in bufs]
    O.ring_all_reduce(bufs)
    for a, b in zip(bufs, keep):
        assert np.array_equal(a, b)
