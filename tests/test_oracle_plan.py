"""Pins of the oracle's shard plan.

Sources: mlxcel manual '텐서 병렬화' - 아키텍처 인식 샤드 플랜 (plan table; GQA-aware
attention sharding and its two diagram cases), 가중치 샤딩 전략 (Column / Row /
Replicated ranges), 설정 (--tp-size power of two). Fixtures:
tests/golden/gqa_examples.json, tests/golden/plan_table.json.
"""
import json
import os

import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _plan(tp, hq, hkv, hd=8, hidden=64, ffn=None):
    return O.shard_plan(tp, hidden, hq, hkv, hd, ffn if ffn is not None else 16 * tp)


def check_gqa_examples():
    g = json.load(open(os.path.join(GOLDEN, "gqa_examples.json")))
    for case in g["cases"]:
        plan = _plan(case["tp_size"], case["num_q_heads"], case["num_kv_heads"], hd=128)
        assert len(plan) == case["tp_size"]
        for s in plan:
            assert s.kv_replicated == case["kv_replicated"]
            assert s.kv_heads[1] - s.kv_heads[0] == case["kv_heads_per_rank"]
            assert s.q_heads[1] - s.q_heads[0] == case["q_heads_per_rank"]


def check_rule_text(tp, hq, hkv):
    """'num_kv_heads >= tp_size: sharded; < tp_size: replicated on every rank.'"""
    plan = _plan(tp, hq, hkv)
    for s in plan:
        assert s.kv_replicated == (hkv < tp)
        if hkv < tp:
            assert s.kv_heads == (0, hkv)
            assert s.strategy["k_proj"] == O.REPLICATED
    if hkv >= tp:
        # sharded: kv heads partition [0, hkv), no rank holds a fraction of a head
        covered = []
        for s in plan:
            covered.extend(range(*s.kv_heads))
            assert s.kv_heads[1] - s.kv_heads[0] >= 1
        assert covered == list(range(hkv))


def check_partitions(tp, hq, hkv, hd=8, ffn=None):
    ffn = ffn if ffn is not None else 16 * tp
    plan = _plan(tp, hq, hkv, hd=hd, ffn=ffn)
    q = []
    for s in plan:
        q.extend(range(*s.q_heads))
    assert q == list(range(hq))
    for wname, total in (("q_proj", hq * hd), ("o_proj", hq * hd), ("gate_proj", ffn),
                         ("up_proj", ffn), ("down_proj", ffn)):
        feats = []
        for s in plan:
            feats.extend(range(*s.ranges[wname]))
        assert feats == list(range(total)), wname
    sizes = {s.ranges["q_proj"][1] - s.ranges["q_proj"][0] for s in plan}
    assert len(sizes) == 1


def check_q_to_kv(tp, hq, hkv):
    """The local map reproduces GQA grouping: q heads sharing a kv head are
    contiguous groups of hq/hkv heads, in order, each group on one kv head."""
    plan = _plan(tp, hq, hkv)
    globals_ = []
    for s in plan:
        nkv = s.kv_heads[1] - s.kv_heads[0]
        assert len(s.q_to_kv) == s.q_heads[1] - s.q_heads[0]
        for j in s.q_to_kv:
            assert 0 <= j < nkv
        assert list(s.q_to_kv) == sorted(s.q_to_kv)
        globals_.extend(s.kv_heads[0] + j for j in s.q_to_kv)
    group = hq // hkv
    assert len(globals_) == hq
    for kv in range(hkv):
        assert globals_[kv * group:(kv + 1) * group] == [kv] * group


def test_gqa_worked_examples():
    check_gqa_examples()


def test_plan_table_matches_page():
    t = json.load(open(os.path.join(GOLDEN, "plan_table.json")))
    for s in _plan(4, 32, 8):
        for row in t["rows"]:
            assert s.strategy[row["weight"]] == row["strategy"]
            assert s.comm[row["weight"]] == row["comm"]
    for s in _plan(8, 32, 4):
        assert s.strategy["k_proj"] == t["replicated_kv_strategy"]
        assert s.strategy["v_proj"] == t["replicated_kv_strategy"]


SWEEP = [(tp, hkv * g, hkv) for tp in (1, 2, 4, 8, 16) for hkv in range(1, 17)
         for g in (1, 2, 4, 8) if (hkv * g) % tp == 0 and (hkv < tp or hkv % tp == 0)]


@pytest.mark.parametrize("tp,hq,hkv", SWEEP)
def test_exhaustive_small_sweep(tp, hq, hkv):
    check_rule_text(tp, hq, hkv)
    check_partitions(tp, hq, hkv)
    check_q_to_kv(tp, hq, hkv)


@pytest.mark.parametrize("tp", [0, 3, 5, 6, 12, -2])
def test_tp_size_must_be_power_of_two(tp):
    with pytest.raises(O.PlanError) as e:
        _plan(tp, 32, 8)
    assert e.value.kind in ("tp_size_not_pow2",)


@pytest.mark.parametrize("tp,hq,hkv,kind", [
    (8, 48, 12, "gqa_shape"),    # 12 kv heads >= 8 but not divisible
    (4, 30, 6, "gqa_shape"),     # q heads not divisible by tp
    (2, 12, 5, "gqa_shape"),     # q heads not a multiple of kv heads
])
def test_bad_gqa_shapes_rejected(tp, hq, hkv, kind):
    with pytest.raises(O.PlanError) as e:
        _plan(tp, hq, hkv)
    assert e.value.kind == kind


def test_ffn_not_divisible_rejected():
    with pytest.raises(O.PlanError) as e:
        O.shard_plan(4, 64, 8, 4, 8, 30)
    assert e.value.kind == "not_divisible"


def test_tp1_is_identity_plan():
    (s,) = _plan(1, 16, 4, hd=8, ffn=40)
    assert s.q_heads == (0, 16) and s.kv_heads == (0, 4) and not s.kv_replicated
    assert s.ranges["gate_proj"] == (0, 40) and s.ranges["o_proj"] == (0, 128)


def test_kv_equal_tp_is_sharded_one_per_rank():
    for s in _plan(8, 64, 8):
        assert not s.kv_replicated and s.kv_heads[1] - s.kv_heads[0] == 1
