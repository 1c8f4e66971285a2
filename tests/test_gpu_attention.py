"""GPU parity of the attention core (between the q/k/v projections and o_proj;
[MLX] GQA 인식 어텐션 샤딩: each rank's q heads attend with the kv heads the plan
gives it), through the C ABI, against the fp64 oracle.

The kernel computes S and the running output in f32 and rounds P to bf16 for
the P V product and A to bf16, so outputs are compared within the bf16
tolerance (max|A_gpu - A_ref| <= 1e-2 * max|A_ref|).
"""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_f64, need_gpu

pytestmark = pytest.mark.gpu
HD = 128


def _torch():
    import torch
    return torch


class Attn:
    def __init__(self, n, hq, hkv, t, seed, scale=1.0, key_ramp=0.0):
        self.plan = tp.tp_plan_create(n, 64 * n, hq, hkv, HD, 8 * n)
        self.oplan = O.shard_plan(n, 64 * n, hq, hkv, HD, 8 * n)
        sh = [tp.tp_plan_query_rank(self.plan, r) for r in range(n)]
        rep = sh[0]["kv_replicated"]
        nkv = 1 if rep else n
        self.n, self.t = n, t
        self.q = [inputs.normal_bf16(seed, 10 + r, (t, (sh[r]["q_heads"][1] - sh[r]["q_heads"][0]) * HD), scale)
                  for r in range(n)]
        kvc = (sh[0]["kv_heads"][1] - sh[0]["kv_heads"][0]) * HD
        self.k, self.v = [], []
        for r in range(nkv):
            kb = inputs.normal_f32(seed, 100 + r, (t, kvc), scale)
            if key_ramp:
                # key magnitudes grow with position: later key blocks raise the row maxima
                kb = kb * (1.0 + key_ramp * np.arange(t, dtype=np.float32)[:, None] / t)
            self.k.append(inputs.f32_to_bf16_bits(kb))
            self.v.append(inputs.normal_bf16(seed, 200 + r, (t, kvc)))

    def run(self, causal):
        torch = _torch()
        a = [torch.full((self.t, q.shape[1]), float("nan"), dtype=torch.bfloat16, device="cuda") for q in self.q]
        ws = torch.empty(max(1, tp.tp_attn_core_workspace_size(self.plan, self.t)), dtype=torch.uint8,
                         device="cuda")
        tp.tp_attn_core(self.plan, [dev_bf16(q) for q in self.q], [dev_bf16(k) for k in self.k],
                        [dev_bf16(v) for v in self.v], a, causal, ws)
        torch.cuda.synchronize()
        assert tp.tp_device_status() == (tp.TP_OK, 0)
        return a

    def oracle(self, causal):
        f = inputs.bf16_bits_to_f64
        return O.attention_core_sharded([f(q) for q in self.q], [f(k) for k in self.k], [f(v) for v in self.v],
                                        self.oplan, HD, causal)


CASES = [  # n, hq, hkv, T
    (1, 2, 1, 128),
    (2, 8, 2, 300),     # sharded kv, ragged last tile
    (4, 8, 2, 257),     # replicated kv (Hkv < N)
    (4, 32, 8, 640),
    (8, 32, 4, 200),    # replicated
    (2, 4, 4, 33),      # a single partial tile
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("n,hq,hkv,t", CASES)
def test_attention_core_matches_the_oracle(n, hq, hkv, t, causal):
    need_gpu()
    m = Attn(n, hq, hkv, t, seed=600 + n * 7 + t)
    got = m.run(causal)
    ref = m.oracle(causal)
    for r in range(n):
        assert_close(host_f64(got[r]), ref[r], BF16_TOL, f"rank {r}")


@pytest.mark.parametrize("causal", [True, False])
def test_peaked_scores_and_growing_maxima(causal):
    """Scores of standard deviation ~16 with key magnitudes growing along the
    sequence: the row maxima move block after block, exercising the rescale of O."""
    need_gpu()
    m = Attn(2, 4, 2, 700, seed=611, scale=4.0, key_ramp=3.0)
    got = m.run(causal)
    ref = m.oracle(causal)
    for r in range(2):
        assert_close(host_f64(got[r]), ref[r], BF16_TOL, f"rank {r}")


def test_first_row_is_the_first_value_row():
    """Causal query 0 sees key 0 only: A row 0 is V row 0 of its kv head, rounded to bf16 exactly."""
    need_gpu()
    m = Attn(2, 8, 2, 150, seed=612)
    got = m.run(True)
    g = m.oplan[0].q_to_kv
    v0 = inputs.bf16_bits_to_f64(m.v[0])
    for h, kvh in enumerate(g):
        assert np.array_equal(host_f64(got[0])[0, h * HD:(h + 1) * HD], v0[0, kvh * HD:(kvh + 1) * HD])


@pytest.mark.parametrize("kernel", ["2", "4"])
def test_attn_core_tp8_t4096_sampled_rows(kernel, monkeypatch):
    """The benchmarked configuration (TP=8, 64 q heads, 8 kv heads, 4096 tokens,
    causal), checked on a seeded sample of query rows of two heads per rank:
    causal row i is the full softmax over keys 0..i. Run with the default
    two-tile kernel and with the SM-pair kernel (TPGQA_ATTN=4)."""
    need_gpu()
    monkeypatch.setenv("TPGQA_ATTN", kernel)
    torch = _torch()
    w = inputs.WORKLOADS["attn_core_tp8_t4096"]
    n, t = w["tp"], w["T"]
    data = inputs.make_bf16_inputs(w)
    plan = tp.tp_plan_create(n, w["hidden"], w["q_heads"], w["kv_heads"], HD, 8 * n)
    oplan = O.shard_plan(n, w["hidden"], w["q_heads"], w["kv_heads"], HD, 8 * n)
    # per-rank slices by the plan: q heads of each rank, kv heads of each rank (sharded here)
    qs = [data["q"][:, s.q_heads[0] * HD:s.q_heads[1] * HD] for s in oplan]
    ks = [data["k"][:, s.kv_heads[0] * HD:s.kv_heads[1] * HD] for s in oplan]
    vs = [data["v"][:, s.kv_heads[0] * HD:s.kv_heads[1] * HD] for s in oplan]
    a = [torch.empty((t, q.shape[1]), dtype=torch.bfloat16, device="cuda") for q in qs]
    ws = torch.empty(tp.tp_attn_core_workspace_size(plan, t), dtype=torch.uint8, device="cuda")
    tp.tp_attn_core(plan, [dev_bf16(q) for q in qs], [dev_bf16(k) for k in ks], [dev_bf16(v) for v in vs], a,
                    True, ws)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    data = {"q": qs, "k": ks, "v": vs}
    rows = np.sort(inputs.rng(w["seed"], 99).choice(t, size=12, replace=False))
    f = inputs.bf16_bits_to_f64
    for r in (0, n - 1):
        got = host_f64(a[r])
        for h in (0, len(oplan[r].q_to_kv) - 1):
            g = oplan[r].q_to_kv[h]
            q = f(data["q"][r][:, h * HD:(h + 1) * HD])
            k = f(data["k"][r][:, g * HD:(g + 1) * HD])
            v = f(data["v"][r][:, g * HD:(g + 1) * HD])
            ref = np.stack([O.attention_head(q[i:i + 1], k[:i + 1], v[:i + 1], causal=False)[0] for i in rows])
            assert_close(got[rows, h * HD:(h + 1) * HD], ref, BF16_TOL, f"rank {r} head {h}")


@pytest.mark.parametrize("tp_size,hq,hkv", [(4, 8, 2), (2, 4, 4)])
def test_projection_attention_o_proj_chain(tp_size, hq, hkv):
    """x -> q/k/v projections (column-parallel) -> causal attention core per rank ->
    o_proj (row-parallel) with the ring all-reduce, against the oracle's chain of
    the same three steps."""
    need_gpu()
    torch = _torch()
    t, d = 200, 512
    w = dict(kind="attn", T=t, hidden=d, q_heads=hq, kv_heads=hkv, head_dim=HD, tp=tp_size, seed=613,
             w_std=0.05)
    data = inputs.make_bf16_inputs(w)
    plan = tp.tp_plan_create(tp_size, d, hq, hkv, HD, 8 * tp_size)
    oplan = O.shard_plan(tp_size, d, hq, hkv, HD, 8 * tp_size)
    sh = [tp.tp_plan_query_rank(plan, r) for r in range(tp_size)]
    rep = sh[0]["kv_replicated"]
    nkv = 1 if rep else tp_size
    dev = {k: dev_bf16(data[k]) for k in ("x", "wq", "wk", "wv", "wo")}
    wq = [dev["wq"][slice(*sh[r]["ranges"]["q_proj"])] for r in range(tp_size)]
    wk = [dev["wk"][slice(*sh[r]["ranges"]["k_proj"])] for r in range(nkv)]
    wv = [dev["wv"][slice(*sh[r]["ranges"]["v_proj"])] for r in range(nkv)]
    wo = [dev["wo"][:, slice(*sh[r]["ranges"]["o_proj"])] for r in range(tp_size)]
    q = [torch.empty((t, x.shape[0]), dtype=torch.bfloat16, device="cuda") for x in wq]
    k = [torch.empty((t, x.shape[0]), dtype=torch.bfloat16, device="cuda") for x in wk]
    v = [torch.empty((t, x.shape[0]), dtype=torch.bfloat16, device="cuda") for x in wv]
    a = torch.empty((t, hq * HD), dtype=torch.bfloat16, device="cuda")
    a_r = [a[:, slice(*sh[r]["ranges"]["o_proj"])] for r in range(tp_size)]
    ys = [torch.empty((t, d), device="cuda") for _ in range(tp_size)]
    ws = torch.empty(tp.tp_attn_core_workspace_size(plan, t), dtype=torch.uint8, device="cuda")
    tp.tp_qkv_proj(plan, dev["x"], wq, wk, wv, q, k, v)
    tp.tp_attn_core(plan, q, k, v, a_r, True, ws)
    tp.tp_row_linear(tp_size, a_r, wo, ys, tp.TP_COMBINE_RING_FUSED)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    f = {k: inputs.bf16_bits_to_f64(data[k]) for k in ("x", "wq", "wk", "wv", "wo")}
    proj = O.attn_proj_sharded(f["x"], f["wq"], f["wk"], f["wv"], np.zeros((t, hq * HD)), f["wo"], oplan, HD)
    att = O.attention_core_sharded(proj["q"], proj["k"], proj["v"], oplan, HD, True)
    ref = sum(O.linear(att[r], f["wo"][:, slice(*oplan[r].ranges["o_proj"])]) for r in range(tp_size))
    for r in range(tp_size):
        assert_close(host_f64(ys[r]), ref, BF16_TOL, f"rank {r}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kernel", ["2", "4"])
def test_running_maximum_lags_then_moves(kernel, causal, monkeypatch):
    """The kernels take p against the row's running maximum and look for a block's
    own maximum only when the block's sum of p passes 2^64. Keys of the second
    128-key block scaled by 8 put each row's maximum 15 to 30 (log2 units, for
    the first head of rank 0) above the first block's, so p reaches 2^15 to 2^30
    with the maximum left where it is; keys of the third block scaled by 30 put
    it 70 to 110 above, so the maximum moves, p is taken again and O is rescaled;
    the fourth block is back to ordinary scores. The result must still be the
    softmax of the oracle."""
    need_gpu()
    monkeypatch.setenv("TPGQA_ATTN", kernel)
    m = Attn(2, 4, 2, 512, seed=622)
    factor = np.ones((512, 1), dtype=np.float32)
    factor[128:256] = 8.0
    factor[256:384] = 30.0
    for r in range(len(m.k)):
        kb = inputs.normal_f32(622, 300 + r, m.k[r].shape) * factor
        m.k[r] = inputs.f32_to_bf16_bits(kb)
    got = m.run(causal)
    ref = m.oracle(causal)
    for r in range(m.n):
        assert_close(host_f64(got[r]), ref[r], BF16_TOL, f"kernel {kernel} rank {r}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kernel", ["1", "2", "3", "4"])
def test_every_attention_kernel_matches_the_oracle(kernel, causal, monkeypatch):
    """The four attention kernels (TPGQA_ATTN=1: one 128-query tile per work item;
    2, the default: two tiles over 128-key blocks; 3: two tiles over 64-key
    blocks; 4: a 256-query tile on an SM pair), each against the oracle, on a
    ragged sharded case and on peaked scores whose row maxima move block after
    block."""
    need_gpu()
    monkeypatch.setenv("TPGQA_ATTN", kernel)
    for m in (Attn(2, 8, 2, 300, seed=620), Attn(2, 4, 2, 700, seed=621, scale=4.0, key_ramp=3.0)):
        got = m.run(causal)
        ref = m.oracle(causal)
        for r in range(m.n):
            assert_close(host_f64(got[r]), ref[r], BF16_TOL, f"kernel {kernel} rank {r}")
