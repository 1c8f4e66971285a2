"""CPU tests of bench.py's timed oracle arm (the CPU baseline and `--impl
reference`): on small workloads of every kind, a pass over the first R token rows
gives the first R rows of the pass over all T rows (every output row depends only
on its own token, and a causal query only on the keys before it), so a row
sample times the same computation the GPU step runs."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from tensor_sharded_linear_gqa_gb300 import inputs  # noqa: E402

SMALL = {
    "mlp": dict(kind="mlp", T=24, hidden=64, ffn=128, tp=2, seed=901, w_std=0.02),
    "attn": dict(kind="attn", T=24, hidden=256, q_heads=4, kv_heads=2, head_dim=64, tp=2, seed=902, w_std=0.02),
    "layer_replicated_kv": dict(kind="layer", T=24, hidden=256, q_heads=8, kv_heads=2, head_dim=32, ffn=128, tp=4,
                                seed=903, w_std=0.02),
    "decoder_layer": dict(kind="layer", attention=True, T=24, hidden=256, q_heads=4, kv_heads=2, head_dim=64,
                          ffn=128, tp=2, seed=904, w_std=0.02),
    "rs_column": dict(kind="rs_column", T=24, hidden=64, q_heads=4, kv_heads=2, head_dim=16, ffn=128, tp=2,
                      seed=905, w_std=0.02),
    "vocab": dict(kind="vocab", T=24, hidden=32, vocab=64, tp=2, seed=906, w_std=0.02),
    "attn_core": dict(kind="attn_core", T=24, hidden=256, q_heads=4, kv_heads=2, head_dim=64, tp=2, seed=907),
    "moe": dict(kind="moe", T=24, hidden=32, ffn=64, experts=4, top_k=2, tp=2, seed=908, w_std=0.02),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("moe_mode", ["within_expert", "expert_parallel"])
def test_row_sample_is_a_prefix_of_the_full_pass(name, moe_mode):
    w = SMALL[name]
    if moe_mode == "expert_parallel" and w["kind"] != "moe":
        pytest.skip("the MoE mode applies to the MoE workload only")
    one_pass, power = bench.oracle_pass(w, moe_mode)
    assert power == (2 if w["kind"] == "attn_core" else 1)
    full = one_pass(w["T"])
    for rows in (1, 7):
        part = one_pass(rows)
        assert len(part) == len(full)
        for got, ref in zip(part, full):
            assert got.shape[0] == rows
            np.testing.assert_allclose(got, ref[:rows], rtol=1e-12, atol=1e-12 * float(np.max(np.abs(ref))))


def test_vocab_sample_looks_up_exactly():
    w = SMALL["vocab"]
    one_pass, _ = bench.oracle_pass(w, "within_expert")
    emb_rows = one_pass(5)[0]
    d = inputs.make_bf16_inputs(w)
    table = inputs.bf16_bits_to_f64(d["emb"])
    assert np.array_equal(emb_rows, table[d["ids"][:5]])


def test_sample_flops_scale_with_the_rows():
    for w in SMALL.values():
        full = bench.sample_flops(w, w["T"])
        assert full == sum(f for f, _ in bench.phase_costs(w, "ring_fused").values()) > 0
        if w.get("attention"):
            continue  # linear projections plus a causal core: neither law alone
        if w["kind"] == "attn_core":
            # causal: the first R queries meet R(R+1)/2 keys in all
            assert bench.sample_flops(w, 6) == pytest.approx(full * (6 * 7) / (24 * 25))
        else:
            assert bench.sample_flops(w, 6) == pytest.approx(full * 6 / 24)


def test_every_workload_fits_the_host_cap():
    for name, w in inputs.WORKLOADS.items():
        if w["kind"] != "linear_fp32":
            assert bench.cpu_too_large(w) is None, name
    huge = dict(SMALL["vocab"], vocab=1 << 24, hidden=8192)
    assert "GiB" in bench.cpu_too_large(huge)
