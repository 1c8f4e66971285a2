"""GPU parity of the MLP and attention-projection blocks at the workload sizes,
against the fp64 oracle (bf16 inputs: max|Y_gpu - Y_ref| <= 1e-2 * max|Y_ref|).

The prefill layer is checked on a seeded sample of 64 token rows: every output
row depends only on its own input row, so the oracle evaluates just those rows.
"""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, host_bits_f32, host_f64, need_gpu

pytestmark = pytest.mark.gpu
COMBINES = [tp.TP_COMBINE_FUSED, tp.TP_COMBINE_RING, tp.TP_COMBINE_RING_FUSED]


def torch():
    import torch as t
    return t


class Layer:
    """Device copies of a workload's bf16 inputs, sharded per the library's plan."""

    def __init__(self, w, data):
        t = torch()
        self.w, self.n, self.T = w, w["tp"], w["T"]
        self.plan = tp.tp_plan_create(w["tp"], w["hidden"], w.get("q_heads", 8), w.get("kv_heads", 8),
                                      w.get("head_dim", 128), w.get("ffn", 8 * w["tp"]))
        self.shards = [tp.tp_plan_query_rank(self.plan, r) for r in range(self.n)]
        self.x = dev_bf16(data["x"])
        self.dev = {}
        for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "a"):
            if name in data:
                self.dev[name] = dev_bf16(data[name])
        self.t = t

    def rng(self, r, wname):
        return self.shards[r]["ranges"][wname]

    def mlp(self, combine):
        t, n, T = self.t, self.n, self.T
        D = self.w["hidden"]
        g = [self.dev["wg"][slice(*self.rng(r, "gate_proj"))] for r in range(n)]
        u = [self.dev["wu"][slice(*self.rng(r, "up_proj"))] for r in range(n)]
        d = [self.dev["wd"][:, slice(*self.rng(r, "down_proj"))] for r in range(n)]
        ys = [t.full((T, D), float("nan"), device="cuda")
              for _ in range(1 if combine == tp.TP_COMBINE_FUSED else n)]
        ws = t.empty(tp.tp_mlp_block_workspace_size(self.plan, T), dtype=t.uint8, device="cuda")
        tp.tp_mlp_block(self.plan, self.x, g, u, d, ys, combine, ws)
        h = ws.view(t.bfloat16).view(T, self.w["ffn"])
        return ys, h

    def attn(self, combine):
        t, n, T = self.t, self.n, self.T
        D = self.w["hidden"]
        rep = self.shards[0]["kv_replicated"]
        wq = [self.dev["wq"][slice(*self.rng(r, "q_proj"))] for r in range(n)]
        kv_ranks = 1 if rep else n
        wk = [self.dev["wk"][slice(*self.rng(r, "k_proj"))] for r in range(kv_ranks)]
        wv = [self.dev["wv"][slice(*self.rng(r, "v_proj"))] for r in range(kv_ranks)]
        a = [self.dev["a"][:, slice(*self.rng(r, "o_proj"))] for r in range(n)]
        wo = [self.dev["wo"][:, slice(*self.rng(r, "o_proj"))] for r in range(n)]
        q = [t.empty((T, x.shape[0]), dtype=t.bfloat16, device="cuda") for x in wq]
        k = [t.empty((T, x.shape[0]), dtype=t.bfloat16, device="cuda") for x in wk]
        v = [t.empty((T, x.shape[0]), dtype=t.bfloat16, device="cuda") for x in wv]
        ys = [t.full((T, D), float("nan"), device="cuda")
              for _ in range(1 if combine == tp.TP_COMBINE_FUSED else n)]
        tp.tp_attn_proj(self.plan, self.x, wq, wk, wv, q, k, v, a, wo, ys, combine)
        return q, k, v, ys


_cache = {}


def layer(name):
    if name not in _cache:
        w = inputs.WORKLOADS[name]
        data = inputs.make_bf16_inputs(w)
        _cache.clear()
        _cache[name] = (Layer(w, data), {k: inputs.bf16_bits_to_f64(v) for k, v in data.items()})
    return _cache[name]


def _oracle_plan(w):
    return O.shard_plan(w["tp"], w["hidden"], w["q_heads"], w["kv_heads"], w["head_dim"],
                        w.get("ffn", 8 * w["tp"]))


# ---- MLP block ------------------------------------------------------------------------
@pytest.mark.parametrize("combine", COMBINES)
def test_mlp_block_tp2_t512(combine):
    need_gpu()
    L, f = layer("mlp_tp2_t512")
    ys, h = L.mlp(combine)
    ref = O.mlp_sharded(f["x"], f["wg"], f["wu"], f["wd"], L.n)
    assert_close(host_f64(h), np.concatenate(ref["h"], axis=1), BF16_TOL, "H (SwiGLU)")
    for y in ys:
        assert_close(host_f64(y), ref["y"][0], BF16_TOL, "Y")
    if combine != tp.TP_COMBINE_FUSED:
        for y in ys[1:]:
            assert np.array_equal(host_bits_f32(y), host_bits_f32(ys[0]))


def test_gate_up_swiglu_matches_oracle_h():
    need_gpu()
    t = torch()
    w = dict(kind="mlp", T=333, hidden=512, ffn=2048, tp=4, seed=12, w_std=0.05)
    data = inputs.make_bf16_inputs(w)
    L = Layer(w, data)
    f = {k: inputs.bf16_bits_to_f64(v) for k, v in data.items()}
    g = [L.dev["wg"][slice(*L.rng(r, "gate_proj"))] for r in range(4)]
    u = [L.dev["wu"][slice(*L.rng(r, "up_proj"))] for r in range(4)]
    h = [t.full((333, 512), float("nan"), dtype=t.bfloat16, device="cuda") for _ in range(4)]
    tp.tp_gate_up_swiglu(L.plan, L.x, g, u, h)
    ref = O.mlp_sharded(f["x"], f["wg"], f["wu"], f["wd"], 4)["h"]
    for r in range(4):
        assert_close(host_f64(h[r]), ref[r], BF16_TOL, f"H[{r}]")


@pytest.mark.parametrize("combine", [tp.TP_COMBINE_NONE] + COMBINES)
def test_mlp_block_small_ragged(combine):
    need_gpu()
    w = dict(kind="mlp", T=200, hidden=256, ffn=1024, tp=4, seed=9, w_std=0.05)
    data = inputs.make_bf16_inputs(w)
    L = Layer(w, data)
    f = {k: inputs.bf16_bits_to_f64(v) for k, v in data.items()}
    ys, h = L.mlp(combine)
    ref = O.mlp_sharded(f["x"], f["wg"], f["wu"], f["wd"], 4)
    assert_close(host_f64(h), np.concatenate(ref["h"], axis=1), BF16_TOL, "H")
    if combine == tp.TP_COMBINE_NONE:
        for y, p in zip(ys, ref["partials"]):
            assert_close(host_f64(y), p, BF16_TOL, "partial")
    else:
        for y in ys:
            assert_close(host_f64(y), ref["y"][0], BF16_TOL, "Y")


@pytest.mark.parametrize("name", ["mlp_tp2_t512", "decode_gqa_rep_tp8_t64"])
def test_ring_shared_result_is_the_ring_fused_result(name):
    """TP_COMBINE_RING_SHARED folds in the ring's order like RING_FUSED and stores
    the result once, in y[0]: bit-identical to RING_FUSED's y[0] (y[1..N-1] are
    scratch)."""
    need_gpu()
    L, _f = layer(name)
    fused, _ = L.mlp(tp.TP_COMBINE_RING_FUSED)
    ref0 = host_bits_f32(fused[0])
    del fused
    shared, _ = L.mlp(tp.TP_COMBINE_RING_SHARED)
    assert np.array_equal(host_bits_f32(shared[0]), ref0)
    if "wq" not in L.dev:  # an MLP-only workload
        return
    _q, _k, _v, ya = L.attn(tp.TP_COMBINE_RING_FUSED)
    refa = host_bits_f32(ya[0])
    del ya
    _q, _k, _v, yb = L.attn(tp.TP_COMBINE_RING_SHARED)
    assert np.array_equal(host_bits_f32(yb[0]), refa)


# ---- attention projections ----------------------------------------------------------
def _check_attn(L, f, q, k, v, ys):
    w = L.w
    ref = O.attn_proj_sharded(f["x"], f["wq"], f["wk"], f["wv"], f["a"], f["wo"], _oracle_plan(w),
                              w["head_dim"])
    for r in range(L.n):
        assert_close(host_f64(q[r]), ref["q"][r], BF16_TOL, f"q[{r}]")
    for r in range(len(k)):
        assert_close(host_f64(k[r]), ref["k"][r], BF16_TOL, f"k[{r}]")
        assert_close(host_f64(v[r]), ref["v"][r], BF16_TOL, f"v[{r}]")
    for y in ys:
        assert_close(host_f64(y), ref["y"][0], BF16_TOL, "Y")


@pytest.mark.parametrize("combine", COMBINES)
def test_attn_proj_gqa_tp4_t2048(combine):
    need_gpu()
    L, f = layer("attn_gqa_tp4_t2048")
    assert [s["kv_heads"] for s in L.shards] == [(0, 2), (2, 4), (4, 6), (6, 8)]
    q, k, v, ys = L.attn(combine)
    assert len(k) == 4
    _check_attn(L, f, q, k, v, ys)


@pytest.mark.parametrize("combine", COMBINES)
def test_decode_replicated_kv_tp8_t64(combine):
    need_gpu()
    L, f = layer("decode_gqa_rep_tp8_t64")
    assert all(s["kv_replicated"] and s["kv_heads"] == (0, 4) for s in L.shards)
    q, k, v, ys = L.attn(combine)
    assert len(k) == 1                     # replicated K/V computed once
    _check_attn(L, f, q, k, v, ys)
    ys, h = L.mlp(combine)
    ref = O.mlp_sharded(f["x"], f["wg"], f["wu"], f["wd"], L.n)
    for y in ys:
        assert_close(host_f64(y), ref["y"][0], BF16_TOL, "MLP Y")


def _attn_then_core(L, combine):
    """tp_attn_proj into NaN-filled q/k/v, then, on the same stream and with no
    synchronisation between, the attention core over those q/k/v."""
    t, n, T = L.t, L.n, L.T
    D = L.w["hidden"]
    rep = L.shards[0]["kv_replicated"]
    kv_ranks = 1 if rep else n
    wq = [L.dev["wq"][slice(*L.rng(r, "q_proj"))] for r in range(n)]
    wk = [L.dev["wk"][slice(*L.rng(r, "k_proj"))] for r in range(kv_ranks)]
    wv = [L.dev["wv"][slice(*L.rng(r, "v_proj"))] for r in range(kv_ranks)]
    a = [L.dev["a"][:, slice(*L.rng(r, "o_proj"))] for r in range(n)]
    wo = [L.dev["wo"][:, slice(*L.rng(r, "o_proj"))] for r in range(n)]
    nan = float("nan")
    q = [t.full((T, x.shape[0]), nan, dtype=t.bfloat16, device="cuda") for x in wq]
    k = [t.full((T, x.shape[0]), nan, dtype=t.bfloat16, device="cuda") for x in wk]
    v = [t.full((T, x.shape[0]), nan, dtype=t.bfloat16, device="cuda") for x in wv]
    ys = [t.full((T, D), nan, device="cuda") for _ in range(1 if combine == tp.TP_COMBINE_FUSED else n)]
    att = [t.full((T, x.shape[0]), nan, dtype=t.bfloat16, device="cuda") for x in wq]
    ws = t.empty(max(1, tp.tp_attn_core_workspace_size(L.plan, T)), dtype=t.uint8, device="cuda")
    t.cuda.synchronize()
    tp.tp_attn_proj(L.plan, L.x, wq, wk, wv, q, k, v, a, wo, ys, combine)
    tp.tp_attn_core(L.plan, q, k, v, att, True, ws)
    t.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    return [host_bits_f32(y) for y in ys], [host_f64(x) for x in q + k + v], [host_f64(x) for x in att]


@pytest.mark.parametrize("combine", [tp.TP_COMBINE_RING_FUSED, tp.TP_COMBINE_RING, tp.TP_COMBINE_FUSED])
def test_decode_oproj_beside_qkv(combine, monkeypatch):
    """At decode sizes o_proj runs beside the q/k/v GEMM on the SMs it leaves
    free and waits for it only before exiting (not with the FUSED combine, whose
    single problem splits K). The results equal, bit for bit, those of the
    serial order (TPGQA_CONCURRENT_OPROJ=0), and a kernel launched after the call
    on the same stream (the attention core, reading q/k/v) sees q/k/v complete:
    NaN-filled q/k/v read too early would spread into its output."""
    need_gpu()
    L, _f = layer("decode_gqa_rep_tp8_t64")
    monkeypatch.setenv("TPGQA_CONCURRENT_OPROJ", "0")
    y0, qkv0, att0 = _attn_then_core(L, combine)
    monkeypatch.setenv("TPGQA_CONCURRENT_OPROJ", "1")
    for _ in range(3):
        y1, qkv1, att1 = _attn_then_core(L, combine)
        for a_, b_ in zip(y0, y1):
            assert np.array_equal(a_, b_)
        for a_, b_ in zip(qkv0 + att0, qkv1 + att1):
            assert np.isfinite(b_).all()
            assert np.array_equal(a_, b_)


@pytest.mark.parametrize("tp_size,hq,hkv", [(4, 8, 4), (8, 16, 2)])
def test_qkv_proj_matches_oracle(tp_size, hq, hkv):
    need_gpu()
    t = torch()
    w = dict(kind="attn", T=150, hidden=256, q_heads=hq, kv_heads=hkv, head_dim=64, tp=tp_size, seed=31,
             w_std=0.05)
    data = inputs.make_bf16_inputs(w)
    L = Layer(w, data)
    f = {k: inputs.bf16_bits_to_f64(v) for k, v in data.items()}
    rep = L.shards[0]["kv_replicated"]
    nkv = 1 if rep else tp_size
    wq = [L.dev["wq"][slice(*L.rng(r, "q_proj"))] for r in range(tp_size)]
    wk = [L.dev["wk"][slice(*L.rng(r, "k_proj"))] for r in range(nkv)]
    wv = [L.dev["wv"][slice(*L.rng(r, "v_proj"))] for r in range(nkv)]
    q = [t.full((150, x.shape[0]), float("nan"), dtype=t.bfloat16, device="cuda") for x in wq]
    k = [t.full((150, x.shape[0]), float("nan"), dtype=t.bfloat16, device="cuda") for x in wk]
    v = [t.full((150, x.shape[0]), float("nan"), dtype=t.bfloat16, device="cuda") for x in wv]
    tp.tp_qkv_proj(L.plan, L.x, wq, wk, wv, q, k, v)
    ref = O.attn_proj_sharded(f["x"], f["wq"], f["wk"], f["wv"], f["a"], f["wo"], _oracle_plan(w), 64)
    for r in range(tp_size):
        assert_close(host_f64(q[r]), ref["q"][r], BF16_TOL, f"q[{r}]")
    for r in range(nkv):
        assert_close(host_f64(k[r]), ref["k"][r], BF16_TOL, f"k[{r}]")
        assert_close(host_f64(v[r]), ref["v"][r], BF16_TOL, f"v[{r}]")


def test_prefill_layer_tp8_t4096_sampled_rows():
    need_gpu()
    L, f = layer("prefill_layer_tp8_t4096")
    rows = np.sort(inputs.rng(L.w["seed"], 99).choice(L.T, size=L.w["oracle_rows"], replace=False))
    q, k, v, ys = L.attn(tp.TP_COMBINE_RING_FUSED)
    plan = _oracle_plan(L.w)
    ref = O.attn_proj_sharded(f["x"][rows], f["wq"], f["wk"], f["wv"], f["a"][rows], f["wo"], plan,
                              L.w["head_dim"])
    for r in range(L.n):
        assert_close(host_f64(q[r])[rows], ref["q"][r], BF16_TOL, f"q[{r}]")
        assert_close(host_f64(k[r])[rows], ref["k"][r], BF16_TOL, f"k[{r}]")
    for y in ys:
        assert_close(host_f64(y)[rows], ref["y"][0], BF16_TOL, "attn Y")
    del q, k, v
    ys, h = L.mlp(tp.TP_COMBINE_FUSED)
    ref = O.mlp_sharded(f["x"][rows], f["wg"], f["wu"], f["wd"], L.n)
    assert_close(host_f64(ys[0])[rows], ref["y"][0], BF16_TOL, "MLP Y")


# ---- the benchmarked layers at their full size ----------------------------------------
def _sampled_rows(w, count=64):
    return np.sort(inputs.rng(w["seed"], 99).choice(w["T"], size=count, replace=False))


_ring_fused_bits = {}


@pytest.mark.parametrize("combine", [tp.TP_COMBINE_RING, tp.TP_COMBINE_RING_SHARED])
def test_prefill_layer_tp8_t4096_ring_modes(combine):
    """The step-by-step ring (N-1 reduce-scatter and N-1 all-gather launches) and the
    ring whose result is stored once, on the benchmarked prefill layer (8 ranks, 128 MiB
    f32 partials per rank): both blocks against the oracle on 64 sampled rows, and bit
    for bit against TP_COMBINE_RING_FUSED, which folds every chunk in the same ring
    order (mlxcel manual "텐서 병렬화", 통신 패턴: reduce-scatter then all-gather,
    rank r sending to (r+1) % N)."""
    need_gpu()
    L, f = layer("prefill_layer_tp8_t4096")
    rows = _sampled_rows(L.w, L.w["oracle_rows"])
    if not _ring_fused_bits:
        _q, _k, _v, ya = L.attn(tp.TP_COMBINE_RING_FUSED)
        _ring_fused_bits["attn"] = host_bits_f32(ya[0])
        del ya
        ym, _h = L.mlp(tp.TP_COMBINE_RING_FUSED)
        _ring_fused_bits["mlp"] = host_bits_f32(ym[0])
        del ym
    copies = L.n if combine == tp.TP_COMBINE_RING else 1
    plan = _oracle_plan(L.w)
    _q, _k, _v, ya = L.attn(combine)
    ref = O.attn_proj_sharded(f["x"][rows], f["wq"], f["wk"], f["wv"], f["a"][rows], f["wo"], plan,
                              L.w["head_dim"])
    for r in range(copies):
        assert np.array_equal(host_bits_f32(ya[r]), _ring_fused_bits["attn"]), f"attention rank {r}"
    assert_close(host_f64(ya[0])[rows], ref["y"][0], BF16_TOL, "attn Y")
    del ya, _q, _k, _v
    ym, _h = L.mlp(combine)
    for r in range(copies):
        assert np.array_equal(host_bits_f32(ym[r]), _ring_fused_bits["mlp"]), f"MLP rank {r}"
    ref = O.mlp_sharded(f["x"][rows], f["wg"], f["wu"], f["wd"], L.n)
    assert_close(host_f64(ym[0])[rows], ref["y"][0], BF16_TOL, "MLP Y")


_decoder_ref = {}


def _decoder_oracle(w, f, rows):
    """The decoder layer on the sampled rows, in the oracle: q/k/v column-parallel
    per rank, causal attention of each sampled query over the keys of every earlier
    token (keys and values of all T rows), o_proj row-parallel with the ring
    all-reduce, then the MLP block on the same input rows."""
    hd, n = w["head_dim"], w["tp"]
    plan = _oracle_plan(w)
    q, k, v, att = [], [], [], []
    for s in plan:
        q.append(O.linear(f["x"][rows], f["wq"][slice(*s.ranges["q_proj"])]))
        k.append(O.linear(f["x"], f["wk"][slice(*s.ranges["k_proj"])]))
        v.append(O.linear(f["x"], f["wv"][slice(*s.ranges["v_proj"])]))
        a = np.empty_like(q[-1])
        for h, g in enumerate(s.q_to_kv):
            kh, vh = k[-1][:, g * hd:(g + 1) * hd], v[-1][:, g * hd:(g + 1) * hd]
            for j, i in enumerate(rows):
                a[j, h * hd:(h + 1) * hd] = O.attention_head(q[-1][j:j + 1, h * hd:(h + 1) * hd], kh[:i + 1],
                                                             vh[:i + 1], causal=False)[0]
        att.append(a)
    parts = [O.linear(att[r], f["wo"][:, slice(*plan[r].ranges["o_proj"])]) for r in range(n)]
    y_o = O.ring_all_reduce([p.reshape(-1) for p in parts])[0].reshape(len(rows), -1)
    y_mlp = O.mlp_sharded(f["x"][rows], f["wg"], f["wu"], f["wd"], n)["y"][0]
    return {"q": q, "k": [t[rows] for t in k], "v": [t[rows] for t in v], "a": att, "y_o": y_o, "y_mlp": y_mlp}


@pytest.mark.parametrize("combine", [tp.TP_COMBINE_RING_FUSED, tp.TP_COMBINE_FUSED, tp.TP_COMBINE_RING_SHARED])
def test_decoder_layer_tp8_t4096_sampled_rows(combine):
    """The whole benchmarked decoder layer (T=4096, D=8192, 64 q / 8 kv heads, F=28672,
    TP=8) through the public calls, as the benchmark chains them: tp_qkv_proj, the causal
    tp_attn_core into the o_proj input, tp_row_linear with the combine, tp_mlp_block.
    Checked on 64 seeded rows: q/k/v, the attention output, the o_proj result and the
    MLP result against the oracle's chain of the same steps (mlxcel manual "텐서 병렬화",
    아키텍처 인식 샤드 플랜 and GQA 인식 어텐션 샤딩)."""
    need_gpu()
    t = torch()
    w = inputs.WORKLOADS["decoder_layer_tp8_t4096"]
    L, f = layer("decoder_layer_tp8_t4096")
    n, T, D, hd = L.n, L.T, w["hidden"], w["head_dim"]
    rows = _sampled_rows(w)
    if not _decoder_ref:
        _decoder_ref.update(_decoder_oracle(w, f, rows))
    ref = _decoder_ref
    rep = L.shards[0]["kv_replicated"]
    nkv = 1 if rep else n
    wq = [L.dev["wq"][slice(*L.rng(r, "q_proj"))] for r in range(n)]
    wk = [L.dev["wk"][slice(*L.rng(r, "k_proj"))] for r in range(nkv)]
    wv = [L.dev["wv"][slice(*L.rng(r, "v_proj"))] for r in range(nkv)]
    wo = [L.dev["wo"][:, slice(*L.rng(r, "o_proj"))] for r in range(n)]
    q = [t.empty((T, x.shape[0]), dtype=t.bfloat16, device="cuda") for x in wq]
    k = [t.empty((T, x.shape[0]), dtype=t.bfloat16, device="cuda") for x in wk]
    v = [t.empty((T, x.shape[0]), dtype=t.bfloat16, device="cuda") for x in wv]
    a = t.full((T, w["q_heads"] * hd), float("nan"), dtype=t.bfloat16, device="cuda")
    a_r = [a[:, slice(*L.rng(r, "o_proj"))] for r in range(n)]
    yo = [t.full((T, D), float("nan"), device="cuda") for _ in range(1 if combine == tp.TP_COMBINE_FUSED else n)]
    ws = t.empty(tp.tp_attn_core_workspace_size(L.plan, T), dtype=t.uint8, device="cuda")
    tp.tp_qkv_proj(L.plan, L.x, wq, wk, wv, q, k, v)
    tp.tp_attn_core(L.plan, q, k, v, a_r, True, ws)
    tp.tp_row_linear(n, a_r, wo, yo, combine)
    t.cuda.synchronize()
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    for r in range(n):
        assert_close(host_f64(q[r])[rows], ref["q"][r], BF16_TOL, f"q[{r}]")
        assert_close(host_f64(a_r[r])[rows], ref["a"][r], BF16_TOL, f"attention output of rank {r}")
    for r in range(nkv):
        assert_close(host_f64(k[r])[rows], ref["k"][r], BF16_TOL, f"k[{r}]")
        assert_close(host_f64(v[r])[rows], ref["v"][r], BF16_TOL, f"v[{r}]")
    copies = 1 if combine in (tp.TP_COMBINE_FUSED, tp.TP_COMBINE_RING_SHARED) else n
    for r in range(copies):
        assert_close(host_f64(yo[r])[rows], ref["y_o"], BF16_TOL, f"o_proj Y, rank {r}")
    del q, k, v, a, a_r, yo, ws
    ym, _h = L.mlp(combine)
    for r in range(copies):
        assert_close(host_f64(ym[r])[rows], ref["y_mlp"], BF16_TOL, f"MLP Y, rank {r}")


@pytest.mark.parametrize("tp_size,hq,hkv,hd,T", [(8, 64, 8, 128, 600), (4, 16, 4, 64, 300), (8, 16, 2, 64, 257)])
def test_qkv_paired_kv_tiles_equal_separate_problems(tp_size, hq, hkv, hd, T):
    """Where each rank's k and v projections are at most 128 columns wide, the
    SM-pair kernel computes them in one 256-column tile (k's weight rows in one
    CTA, v's in the other). Each output element is the same MMA sequence as with
    separate problems, so the bits agree with TPGQA_QKV_PAIRED=0; and q/k/v match
    the oracle."""
    import os
    need_gpu()
    t = torch()
    w = dict(kind="attn", T=T, hidden=256, q_heads=hq, kv_heads=hkv, head_dim=hd, tp=tp_size, seed=41,
             w_std=0.05)
    data = inputs.make_bf16_inputs(w)
    L = Layer(w, data)
    f = {k: inputs.bf16_bits_to_f64(v) for k, v in data.items()}
    nkv = 1 if L.shards[0]["kv_replicated"] else tp_size
    wq = [L.dev["wq"][slice(*L.rng(r, "q_proj"))] for r in range(tp_size)]
    wk = [L.dev["wk"][slice(*L.rng(r, "k_proj"))] for r in range(nkv)]
    wv = [L.dev["wv"][slice(*L.rng(r, "v_proj"))] for r in range(nkv)]

    def run(paired):
        q = [t.full((T, x.shape[0]), float("nan"), dtype=t.bfloat16, device="cuda") for x in wq]
        k = [t.full((T, x.shape[0]), float("nan"), dtype=t.bfloat16, device="cuda") for x in wk]
        v = [t.full((T, x.shape[0]), float("nan"), dtype=t.bfloat16, device="cuda") for x in wv]
        old = os.environ.get("TPGQA_QKV_PAIRED")
        os.environ["TPGQA_QKV_PAIRED"] = "1" if paired else "0"
        try:
            tp.tp_qkv_proj(L.plan, L.x, wq, wk, wv, q, k, v)
        finally:
            if old is None:
                del os.environ["TPGQA_QKV_PAIRED"]
            else:
                os.environ["TPGQA_QKV_PAIRED"] = old
        t.cuda.synchronize()
        return [host_bits_f32(a.view(t.int16).to(t.int32)) for a in q + k + v], (q, k, v)

    bits_p, (q, k, v) = run(True)
    bits_s, _ = run(False)
    for i, (a, b) in enumerate(zip(bits_p, bits_s)):
        assert np.array_equal(a, b), f"output {i}"
    ref = O.attn_proj_sharded(f["x"], f["wq"], f["wk"], f["wv"], f["a"], f["wo"], _oracle_plan(w), hd)
    for r in range(tp_size):
        assert_close(host_f64(q[r]), ref["q"][r], BF16_TOL, f"q[{r}]")
    for r in range(nkv):
        assert_close(host_f64(k[r]), ref["k"][r], BF16_TOL, f"k[{r}]")
        assert_close(host_f64(v[r]), ref["v"][r], BF16_TOL, f"v[{r}]")
