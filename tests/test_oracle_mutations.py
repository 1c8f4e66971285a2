"""Planted mistakes in the oracle must trip its pins.

Each test swaps one oracle function for a copy carrying a plausible mistake (a
wrong chunk index, a wrong neighbour, a dropped term, a transposed operand, an
off-by-one in the plan rule, a wrong activation) and checks that at least one
pin fails. Everything runs on the CPU and touches only the oracle.
"""
import numpy as np
import pytest

import oracle as O
import oracle.tp_oracle as T
import test_oracle_blocks as PB
import test_oracle_linear as PL
import test_oracle_plan as PP
import test_oracle_ring as PR


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(T, name, fn)
    monkeypatch.setattr(O, name, fn)


def _fails(check, *args):
    with pytest.raises(AssertionError):
        check(*args)


def _rs_with(chunk_of, dst_of):
    def rs(bufs, log=None):
        n = len(bufs)
        out = [np.array(b, copy=True).reshape(-1) for b in bufs]
        size = out[0].size
        for s in range(n - 1):
            msgs = []
            for r in range(n):
                c = chunk_of(r, s, n)
                lo, hi = T.chunk_bounds(size, n, c)
                msgs.append((dst_of(r, n), c, out[r][lo:hi].copy(), r))
            for dst, c, data, src in msgs:
                lo, hi = T.chunk_bounds(size, n, c)
                out[dst][lo:hi] = data + out[dst][lo:hi]
                if log is not None:
                    log.sends.append(("reduce_scatter", s, src, dst, c, data.nbytes))
        return out
    return rs


def test_rs_wrong_chunk_index(monkeypatch):
    _patch(monkeypatch, "ring_reduce_scatter", _rs_with(lambda r, s, n: (r - s) % n,
                                                        lambda r, n: (r + 1) % n))
    _fails(PR.check_rs_owns_reduced_chunk, 4, 64)


def test_rs_wrong_neighbour(monkeypatch):
    _patch(monkeypatch, "ring_reduce_scatter", _rs_with(lambda r, s, n: (r - 1 - s) % n,
                                                        lambda r, n: (r + 2) % n))
    _fails(PR.check_neighbour_and_steps, 4, 40)


def test_rs_one_step_short(monkeypatch):
    good = T.ring_reduce_scatter

    def short(bufs, log=None):
        n = len(bufs)
        if n <= 2:
            return good(bufs, log)
        # run the real ring on n-1 ranks' worth of steps: drop the last step
        out = [np.array(b, copy=True).reshape(-1) for b in bufs]
        size = out[0].size
        for s in range(n - 2):
            msgs = []
            for r in range(n):
                c = (r - 1 - s) % n
                lo, hi = T.chunk_bounds(size, n, c)
                msgs.append(((r + 1) % n, c, out[r][lo:hi].copy()))
            for dst, c, data in msgs:
                lo, hi = T.chunk_bounds(size, n, c)
                out[dst][lo:hi] = data + out[dst][lo:hi]
        return out
    _patch(monkeypatch, "ring_reduce_scatter", short)
    _fails(PR.check_each_contribution_once, 4, 37)


def test_ag_wrong_chunk(monkeypatch):
    def ag(bufs, log=None):
        n = len(bufs)
        out = [np.array(b, copy=True).reshape(-1) for b in bufs]
        size = out[0].size
        for s in range(n - 1):
            msgs = []
            for r in range(n):
                c = (r - 1 - s) % n          # mistake: the reduce-scatter index
                lo, hi = T.chunk_bounds(size, n, c)
                msgs.append(((r + 1) % n, c, out[r][lo:hi].copy()))
            for dst, c, data in msgs:
                lo, hi = T.chunk_bounds(size, n, c)
                out[dst][lo:hi] = data
        return out
    _patch(monkeypatch, "ring_all_gather", ag)
    _fails(PR.check_allreduce_everywhere, 4, 64)


def test_linear_transposed_operand(monkeypatch):
    _patch(monkeypatch, "linear", lambda x, w: np.asarray(x, float) @ np.asarray(w, float))
    with pytest.raises((AssertionError, ValueError)):
        PL.check_permutation_weight()


def test_row_parallel_drops_last_rank(monkeypatch):
    good = T.row_parallel
    _patch(monkeypatch, "row_parallel", lambda xs, ws: good(xs, ws)[:-1] + [0 * good(xs, ws)[-1]])
    _fails(PL.check_row_sum_exact, 4)


def test_column_split_off_by_one(monkeypatch):
    def bad_split(w, n):
        k = w.shape[0] // n
        return [w[max(r * k - 1, 0):max(r * k - 1, 0) + k, :] for r in range(n)]
    _patch(monkeypatch, "split_rows", bad_split)
    _fails(PL.check_column_concat_exact, 4)


def test_plan_replicates_when_equal(monkeypatch):
    good = T.shard_plan

    def bad(tp, hidden, hq, hkv, hd, ffn):
        # mistake: '<=' instead of '<' (replicates when num_kv_heads == tp_size)
        if hkv == tp and tp > 1:
            p = good(tp, hidden, hq, hkv // 2 if hkv % 2 == 0 else hkv, hd, ffn)
            for s in p:
                s.kv_replicated = True
                s.kv_heads = (0, hkv)
            return p
        return good(tp, hidden, hq, hkv, hd, ffn)
    _patch(monkeypatch, "shard_plan", bad)
    _fails(PP.check_rule_text, 8, 64, 8)


def test_plan_q_to_kv_off_by_group(monkeypatch):
    good = T.shard_plan

    def bad(*a):
        p = good(*a)
        for s in p:
            s.q_to_kv = [min(j, s.kv_heads[1] - s.kv_heads[0] - 1) for j in range(len(s.q_to_kv))]
        return p
    _patch(monkeypatch, "shard_plan", bad)
    _fails(PP.check_q_to_kv, 4, 32, 8)


def test_gqa_example_q_heads_miscount(monkeypatch):
    good = T.shard_plan

    def bad(tp, hidden, hq, hkv, hd, ffn):
        # mistake: q heads split by kv grouping instead of by tp_size
        p = good(tp, hidden, hq, hkv, hd, ffn)
        for s in p:
            s.q_heads = (s.kv_heads[0], s.kv_heads[1])
        return p
    _patch(monkeypatch, "shard_plan", bad)
    _fails(PP.check_gqa_examples)


def test_silu_wrong_activation(monkeypatch):
    _patch(monkeypatch, "silu", lambda x: 1.0 / (1.0 + np.exp(-np.asarray(x, float))))
    _fails(PB.check_silu_closed_forms)
