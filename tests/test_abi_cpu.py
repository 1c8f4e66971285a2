"""CPU tests of the C ABI: the library loads, exports every declared symbol, its
plan is bit-exact against the oracle's, and argument / health checks return
their status before any CUDA call (so they run without a GPU)."""
import ctypes
import os
import re

import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tpgqa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(tp_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tp_plan_create", "tp_column_linear", "tp_row_linear", "tp_reduce_scatter",
                     "tp_all_gather", "tp_allreduce_ring", "tp_mlp_block", "tp_attn_proj"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = tp.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in tp.EXPORTED, name


def test_status_strings():
    for i, name in enumerate(tp.STATUS_NAMES):
        assert tp.tp_status_str(i) == name
    assert tp.tp_version().startswith("tpgqa")


STRAT = {O.COLUMN: tp.TP_SHARD_COLUMN, O.ROW: tp.TP_SHARD_ROW, O.VOCAB: tp.TP_SHARD_VOCAB,
         O.REPLICATED: tp.TP_SHARD_REPLICATED}
COMM = {O.NO_COMM: tp.TP_COMM_NONE, O.ALL_REDUCE: tp.TP_COMM_ALL_REDUCE,
        O.ALL_GATHER: tp.TP_COMM_ALL_GATHER, O.REDUCE_SCATTER: tp.TP_COMM_REDUCE_SCATTER}

PLAN_CASES = [(tp_, hkv * g, hkv, hd, ffn)
              for tp_ in (1, 2, 4, 8, 16) for hkv in (1, 2, 3, 4, 8, 16) for g in (1, 2, 4)
              for hd, ffn in ((64, 256), (128, 14336))
              if (hkv * g) % tp_ == 0 and (hkv < tp_ or hkv % tp_ == 0) and ffn % tp_ == 0]
PLAN_CASES += [(4, 32, 8, 128, 14336), (8, 32, 4, 128, 14336), (8, 64, 8, 128, 28672),
               (2, 16, 8, 128, 8192)]


@pytest.mark.parametrize("tp_size,hq,hkv,hd,ffn", PLAN_CASES)
def test_plan_bit_exact_vs_oracle(tp_size, hq, hkv, hd, ffn):
    hidden = 512
    ref = O.shard_plan(tp_size, hidden, hq, hkv, hd, ffn)
    plan = tp.tp_plan_create(tp_size, hidden, hq, hkv, hd, ffn)
    for s in ref:
        got = tp.tp_plan_query_rank(plan, s.rank)
        assert got["q_heads"] == s.q_heads
        assert got["kv_heads"] == s.kv_heads
        assert got["kv_replicated"] == s.kv_replicated
        for w in O.WEIGHTS:
            assert got["strategy"][w] == STRAT[s.strategy[w]], w
            assert got["comm"][w] == COMM[s.comm[w]], w
            assert got["ranges"][w] == tuple(s.ranges[w]), w
        assert tp.tp_plan_q_to_kv(plan, s.rank) == list(s.q_to_kv)


ERR = {"tp_size_not_pow2": tp.TP_ERR_TP_SIZE_NOT_POW2, "gqa_shape": tp.TP_ERR_GQA_SHAPE,
       "not_divisible": tp.TP_ERR_NOT_DIVISIBLE, "invalid": tp.TP_ERR_INVALID_ARG}


@pytest.mark.parametrize("args", [(3, 64, 32, 8, 128, 1024), (0, 64, 32, 8, 128, 1024),
                                  (8, 64, 48, 12, 128, 1024), (4, 64, 30, 6, 128, 1024),
                                  (2, 64, 12, 5, 128, 1024), (4, 64, 8, 4, 8, 30),
                                  (4, 0, 8, 4, 8, 32), (4, 64, 8, 4, 0, 32)])
def test_plan_errors_match_oracle(args):
    with pytest.raises(O.PlanError) as e:
        O.shard_plan(*args)
    with pytest.raises(tp.TPError) as g:
        tp.tp_plan_create(*args)
    assert g.value.status == ERR[e.value.kind]


def test_query_rank_out_of_range():
    plan = tp.tp_plan_create(4, 64, 8, 4, 8, 32)
    s = tp.TpRankShard()
    assert tp.raw_status("tp_plan_query_rank", plan.handle, 4, ctypes.byref(s)) == tp.TP_ERR_INVALID_ARG
    assert tp.raw_status("tp_plan_query_rank", plan.handle, -1, ctypes.byref(s)) == tp.TP_ERR_INVALID_ARG
    small = (ctypes.c_int32 * 1)()
    assert tp.raw_status("tp_plan_q_to_kv", plan.handle, 0, small, 1) == tp.TP_ERR_INVALID_ARG


def test_workspace_size():
    plan = tp.tp_plan_create(2, 2048, 16, 8, 128, 8192)
    assert tp.tp_mlp_block_workspace_size(plan, 512) == 512 * 8192 * 2
    assert tp.tp_mlp_block_workspace_size(plan, 0) == 0


# ---- argument checks that return before any CUDA call -------------------------
FAKE = 1 << 40  # never dereferenced: every case below fails validation first


def T(ptr, dtype, rows, cols, ld=None):
    return tp.TpTensor(ptr, dtype, 0, rows, cols, ld if ld is not None else cols)


def arr(*ts):
    a = (tp.TpTensor * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t
    return a


BF, F32 = tp.TP_BF16, tp.TP_F32


def col_status(n, x, ws, ys, gather=1):
    return tp.raw_status("tp_column_linear", n, ctypes.byref(x), arr(*ws), arr(*ys), gather, None)


def test_column_linear_rejects_bad_arguments():
    x = T(FAKE, BF, 64, 128)
    w = [T(FAKE, BF, 32, 128), T(FAKE, BF, 32, 128)]
    y = [T(FAKE, BF, 64, 64)]
    assert col_status(3, x, w + [w[0]], y) == tp.TP_ERR_TP_SIZE_NOT_POW2
    assert col_status(2, x, [w[0], T(FAKE, BF, 32, 100)], y) == tp.TP_ERR_INVALID_ARG
    assert col_status(2, x, [w[0], T(FAKE, F32, 32, 128)], y) == tp.TP_ERR_DTYPE
    assert col_status(2, x, w, [T(FAKE, BF, 64, 65)]) == tp.TP_ERR_INVALID_ARG
    assert col_status(2, T(FAKE + 2, BF, 64, 128), w, y) == tp.TP_ERR_ALIGNMENT
    assert col_status(2, T(FAKE, BF, 64, 100, 100), [T(FAKE, BF, 32, 100)] * 2, y) == \
        tp.TP_ERR_ALIGNMENT  # row pitch of 200 bytes
    assert col_status(2, T(None, BF, 64, 128), w, y) == tp.TP_ERR_INVALID_ARG
    assert col_status(2, x, w, y, gather=2) == tp.TP_ERR_INVALID_ARG


def test_row_linear_rejects_bad_arguments():
    xs = [T(FAKE, BF, 64, 64), T(FAKE, BF, 64, 64)]
    ws = [T(FAKE, BF, 128, 64), T(FAKE, BF, 128, 64)]
    ys = [T(FAKE, F32, 64, 128), T(FAKE + 4096, F32, 64, 128)]

    def st(xs_, ws_, ys_, combine):
        return tp.raw_status("tp_row_linear", 2, arr(*xs_), arr(*ws_), arr(*ys_), combine, None)
    assert st(xs, ws, ys, 7) == tp.TP_ERR_INVALID_ARG
    assert st(xs, ws, [T(FAKE, BF, 64, 128)] * 2, tp.TP_COMBINE_NONE) == tp.TP_ERR_DTYPE
    assert st(xs, [ws[0], T(FAKE, BF, 128, 32)], ys, tp.TP_COMBINE_NONE) == tp.TP_ERR_INVALID_ARG
    # ring combine needs distinct, contiguous buffers
    assert st(xs, ws, [ys[0], ys[0]], tp.TP_COMBINE_RING) == tp.TP_ERR_INVALID_ARG
    assert st(xs, ws, [T(FAKE, F32, 64, 128, 256), ys[1]], tp.TP_COMBINE_RING) == tp.TP_ERR_INVALID_ARG
    # ranges that share elements would race in the ring: a second buffer four
    # floats into the first (aligned, distinct base) is rejected as well
    far = [T(FAKE, F32, 64, 128), T(FAKE + 64 * 128 * 4, F32, 64, 128)]
    for combine in (tp.TP_COMBINE_RING, tp.TP_COMBINE_RING_FUSED, tp.TP_COMBINE_RING_SHARED):
        assert st(xs, ws, [far[0], T(FAKE + 16, F32, 64, 128)], combine) == tp.TP_ERR_INVALID_ARG
        assert st(xs, ws, [T(FAKE + 64 * 128 * 4 - 16, F32, 64, 128), far[0]], combine) == tp.TP_ERR_INVALID_ARG


def test_collectives_reject_overlapping_rank_buffers():
    def st(fn, bufs, mode=0, n=2):
        return tp.raw_status(fn, n, arr(*bufs), mode, None)
    a = T(FAKE, F32, 8, 8)                   # 256 bytes
    for fn in ("tp_reduce_scatter", "tp_ring_all_gather", "tp_allreduce_ring"):
        assert st(fn, [a, T(FAKE + 16, F32, 8, 8)]) == tp.TP_ERR_INVALID_ARG
        assert st(fn, [T(FAKE + 240, F32, 8, 8), a]) == tp.TP_ERR_INVALID_ARG
        four = [a, T(FAKE + 256, F32, 8, 8), T(FAKE + 512, F32, 8, 8), T(FAKE + 752, F32, 8, 8)]
        assert st(fn, four, n=4) == tp.TP_ERR_INVALID_ARG   # the last two share one float4


def test_collectives_reject_bad_arguments():
    good = [T(FAKE, F32, 8, 8), T(FAKE + 1024, F32, 8, 8)]

    def st(fn, bufs, mode=0, n=2):
        return tp.raw_status(fn, n, arr(*bufs), mode, None)
    for fn in ("tp_reduce_scatter", "tp_ring_all_gather", "tp_allreduce_ring"):
        assert st(fn, good, mode=5) == tp.TP_ERR_INVALID_ARG
        assert st(fn, [good[0], T(FAKE + 1024, BF, 8, 8)]) == tp.TP_ERR_DTYPE
        assert st(fn, [good[0], T(FAKE + 1028, F32, 8, 8)]) == tp.TP_ERR_ALIGNMENT
        assert st(fn, [good[0], T(FAKE + 1024, F32, 8, 9)]) == tp.TP_ERR_INVALID_ARG
        assert st(fn, good + [good[0]], n=3) == tp.TP_ERR_TP_SIZE_NOT_POW2
    # the shared-result mode exists for the all-reduce only
    assert st("tp_reduce_scatter", good, mode=tp.TP_RING_FUSED_SHARED) == tp.TP_ERR_INVALID_ARG
    assert st("tp_ring_all_gather", good, mode=tp.TP_RING_FUSED_SHARED) == tp.TP_ERR_INVALID_ARG


def test_reduce_scatter_bf16_rejects_bad_arguments():
    parts = [T(FAKE, F32, 8, 8), T(FAKE + 1024, F32, 8, 8)]
    outs = [T(FAKE + 4096, BF, 8, 8), T(FAKE + 8192, BF, 8, 8)]

    def st(p_, o_, n=2):
        return tp.raw_status("tp_reduce_scatter_bf16", n, arr(*p_), arr(*o_), None)
    assert st(parts, [outs[0], T(FAKE + 8192, F32, 8, 8)]) == tp.TP_ERR_DTYPE
    assert st(parts, [outs[0], T(FAKE + 8192, BF, 8, 16)]) == tp.TP_ERR_INVALID_ARG
    assert st(parts, [outs[0], T(FAKE + 8194, BF, 8, 8)]) == tp.TP_ERR_ALIGNMENT
    assert st([parts[0], T(FAKE + 1024, BF, 8, 8)], outs) == tp.TP_ERR_DTYPE
    assert st(parts + [parts[0]], outs + [outs[0]], n=3) == tp.TP_ERR_TP_SIZE_NOT_POW2


def test_column_linear_chunks_rejects_bad_arguments():
    xs = [T(FAKE, BF, 64, 128), T(FAKE + (1 << 20), BF, 64, 128)]
    w = [T(FAKE, BF, 32, 128), T(FAKE, BF, 32, 128)]
    y = [T(FAKE, BF, 64, 64)]

    def st(x_, w_, y_, gather=1, n=2):
        return tp.raw_status("tp_column_linear_chunks", n, arr(*x_), arr(*w_), arr(*y_), gather, None)
    # the chunk boundary of 63 rows over 2 ranks falls inside a row of the flat buffer
    assert st([T(FAKE, BF, 63, 128)] * 2, w, [T(FAKE, BF, 63, 64)]) == tp.TP_ERR_NOT_DIVISIBLE
    assert st([xs[0], T(FAKE, BF, 64, 120)], w, y) == tp.TP_ERR_INVALID_ARG
    assert st([xs[0], T(FAKE, F32, 64, 128)], w, y) == tp.TP_ERR_DTYPE
    assert st(xs, [w[0], T(FAKE, F32, 32, 128)], y) == tp.TP_ERR_DTYPE
    assert st(xs, w, [T(FAKE, BF, 64, 65)]) == tp.TP_ERR_INVALID_ARG
    assert st([xs[0], T(FAKE + 2, BF, 64, 128)], w, y) == tp.TP_ERR_ALIGNMENT
    assert st(xs, w, y, gather=2) == tp.TP_ERR_INVALID_ARG
    assert st(xs + [xs[0]], w + [w[0]], y, n=3) == tp.TP_ERR_TP_SIZE_NOT_POW2


def test_all_gather_rejects_bad_arguments():
    sh = [T(FAKE, F32, 8, 4), T(FAKE + 512, F32, 8, 4)]
    out = [T(FAKE + 4096, F32, 8, 8)]

    def st(shards, outs, axis, n_out=None):
        return tp.raw_status("tp_all_gather", 2, arr(*shards), arr(*outs),
                             n_out if n_out is not None else len(outs), axis, None)
    assert st(sh, out, 2) == tp.TP_ERR_INVALID_ARG
    assert st(sh, out, 0) == tp.TP_ERR_INVALID_ARG          # rows would be 16
    assert st(sh, [T(FAKE + 4096, BF, 8, 8)], 1) == tp.TP_ERR_DTYPE
    assert st(sh, out * 3, 1, 3) == tp.TP_ERR_INVALID_ARG    # n_out must be 1 or tp_size


def test_vocab_embedding_rejects_bad_arguments():
    tab = [T(FAKE, BF, 16, 64), T(FAKE + 4096, BF, 16, 64)]
    out = [T(FAKE + 8192, BF, 5, 64)]
    ids = FAKE + (1 << 16)

    def st(t_, o_, n_tok=5, n=2, ids_=ids, n_out=None):
        return tp.raw_status("tp_vocab_embedding", n, ids_, n_tok, arr(*t_), arr(*o_),
                             n_out if n_out is not None else len(o_), None)
    assert st(tab, out, ids_=0) == tp.TP_ERR_INVALID_ARG          # no ids
    assert st(tab, out, n_tok=-1) == tp.TP_ERR_INVALID_ARG
    assert st([tab[0], T(FAKE + 4096, BF, 15, 64)], out) == tp.TP_ERR_INVALID_ARG  # slices differ
    assert st([tab[0], T(FAKE + 4096, F32, 16, 64)], out) == tp.TP_ERR_DTYPE
    assert st(tab, [T(FAKE + 8192, F32, 5, 64)]) == tp.TP_ERR_DTYPE
    assert st(tab, [T(FAKE + 8192, BF, 4, 64)]) == tp.TP_ERR_INVALID_ARG  # rows != n_tokens
    assert st(tab, [T(FAKE + 8192, BF, 5, 32)]) == tp.TP_ERR_INVALID_ARG  # cols != D
    assert st(tab, out * 3, n_out=3) == tp.TP_ERR_INVALID_ARG          # n_out must be 1 or tp_size
    assert st(tab + [tab[0]], out, n=3) == tp.TP_ERR_TP_SIZE_NOT_POW2
    assert st(tab, out, ids_=ids + 2) == tp.TP_ERR_ALIGNMENT
    assert st([tab[0], T(FAKE + 4097, BF, 16, 64)], out) == tp.TP_ERR_ALIGNMENT
    f32tab = [T(FAKE, F32, 16, 64), T(FAKE + 4096, F32, 16, 64)]
    assert st(f32tab, [T(FAKE + 8194, F32, 5, 64)]) == tp.TP_ERR_ALIGNMENT
    assert st(tab, [T(FAKE + 8192, BF, 0, 64)], n_tok=0, ids_=0) == tp.TP_OK  # nothing to look up
    tp.tp_set_rank_health(1, False)
    try:
        assert st(tab, out) == tp.TP_ERR_RANK_FAILED
    finally:
        tp.tp_set_rank_health(1, True)


def test_vocab_lm_head_rejects_bad_arguments():
    x = T(FAKE, BF, 64, 128)
    w = [T(FAKE, BF, 32, 128), T(FAKE + 8192, BF, 32, 128)]
    logits = [T(FAKE, F32, 64, 64)]

    def st(w_, y_, gather=1, n=2):
        return tp.raw_status("tp_vocab_lm_head", n, ctypes.byref(x), arr(*w_), arr(*y_), gather, None)
    assert st([w[0], T(FAKE + 8192, BF, 24, 128)], [T(FAKE, F32, 64, 56)]) == tp.TP_ERR_INVALID_ARG
    assert st(w, [T(FAKE, F32, 64, 60)]) == tp.TP_ERR_INVALID_ARG
    assert st(w, [T(FAKE + 4, F32, 64, 64)]) == tp.TP_ERR_ALIGNMENT
    assert st(w, logits, gather=3) == tp.TP_ERR_INVALID_ARG


def test_moe_rejects_bad_arguments():
    n, E, k, D, F, Tt = 2, 4, 2, 64, 128, 16
    within = tp.moe_dims(n, tp.TP_MOE_WITHIN_EXPERT, E, k, D, F)
    x = T(FAKE, BF, Tt, D)
    g = [T(FAKE, BF, E * F // n, D)] * n
    d = [T(FAKE, BF, E * D, F // n)] * n
    y = [T(FAKE, F32, Tt, D)] * n
    ws_need = tp.tp_moe_workspace_size(within, Tt)
    assert ws_need > 0

    def st(dims, x_=x, g_=g, u_=g, d_=d, y_=y, combine=tp.TP_COMBINE_RING_FUSED, ws=FAKE, wsb=None, ids=FAKE,
           wts=FAKE):
        return tp.raw_status("tp_moe_block", ctypes.byref(dims), ctypes.byref(x_), ids, wts, arr(*g_), arr(*u_),
                             arr(*d_), arr(*y_), combine, ws, ws_need if wsb is None else wsb, None)
    assert st(tp.moe_dims(3, 1, E, k, D, F)) == tp.TP_ERR_TP_SIZE_NOT_POW2
    assert st(tp.moe_dims(n, 2, E, k, D, F)) == tp.TP_ERR_INVALID_ARG          # mode
    assert st(tp.moe_dims(n, 1, 0, k, D, F)) == tp.TP_ERR_INVALID_ARG          # no experts
    assert st(tp.moe_dims(n, 1, 257, k, D, F)) == tp.TP_ERR_INVALID_ARG        # over 256 experts
    assert st(tp.moe_dims(n, 0, 3, k, D, F)) == tp.TP_ERR_NOT_DIVISIBLE        # E % N (expert parallel)
    assert st(tp.moe_dims(n, 1, E, k, D, 129)) == tp.TP_ERR_NOT_DIVISIBLE      # F % N (within expert)
    assert st(tp.moe_dims(n, 1, E, k, 60, F)) == tp.TP_ERR_ALIGNMENT           # D not a multiple of 8
    assert st(within, g_=[T(FAKE, BF, E * F // n - 8, D)] * n) == tp.TP_ERR_INVALID_ARG
    assert st(within, d_=[T(FAKE, F32, E * D, F // n)] * n) == tp.TP_ERR_DTYPE
    assert st(within, y_=[T(FAKE, BF, Tt, D)] * n) == tp.TP_ERR_DTYPE
    assert st(within, ws=FAKE + 16) == tp.TP_ERR_ALIGNMENT
    assert st(within, wsb=ws_need - 1) == tp.TP_ERR_WORKSPACE
    assert st(within, ids=0) == tp.TP_ERR_INVALID_ARG
    assert st(within, ids=FAKE + 2) == tp.TP_ERR_ALIGNMENT
    assert st(within, combine=7) == tp.TP_ERR_INVALID_ARG
    assert st(within, y_=[T(FAKE, F32, Tt, D, ld=D + 8)] * n) == tp.TP_ERR_INVALID_ARG  # ring needs ld == D
    # expert parallel takes [(E/N)*F x D] gate/up and [(E/N)*D x F] down per rank
    ep = tp.moe_dims(n, tp.TP_MOE_EXPERT_PARALLEL, E, k, D, F)
    ws_need = tp.tp_moe_workspace_size(ep, Tt)
    assert st(ep, g_=[T(FAKE, BF, E // n * F, D)] * n, d_=[T(FAKE, BF, E // n * D, F)] * n,
              ids=FAKE + 2) == tp.TP_ERR_ALIGNMENT  # shapes accepted, then the ids pointer is checked
    assert tp.tp_moe_workspace_size(tp.moe_dims(n, 0, 3, k, D, F), Tt) == 0
    tp.tp_set_rank_health(1, False)
    try:
        assert st(within, wsb=tp.tp_moe_workspace_size(within, Tt)) == tp.TP_ERR_RANK_FAILED
    finally:
        tp.tp_set_rank_health(1, True)


def test_attn_core_rejects_bad_arguments():
    plan = tp.tp_plan_create(2, 256, 8, 2, 128, 16)   # 4 q heads and 1 kv head per rank
    Tt = 64
    q = [T(FAKE, BF, Tt, 512), T(FAKE + 65536, BF, Tt, 512)]
    kv = [T(FAKE, BF, Tt, 128), T(FAKE + 65536, BF, Tt, 128)]
    need = tp.tp_attn_core_workspace_size(plan, Tt)
    assert need == 2 * 128 * 64 * 2

    def st(q_=q, k_=kv, v_=kv, a_=q, causal=1, ws=FAKE, wsb=need, pl=plan):
        return tp.raw_status("tp_attn_core", pl.handle, arr(*q_), arr(*k_), arr(*v_), arr(*a_), causal, ws, wsb,
                             None)
    assert st(causal=2) == tp.TP_ERR_INVALID_ARG
    assert st(q_=[q[0], T(FAKE, BF, Tt, 384)]) == tp.TP_ERR_INVALID_ARG        # rank 1 holds 4 heads
    assert st(k_=[kv[0], T(FAKE, F32, Tt, 128)]) == tp.TP_ERR_DTYPE
    assert st(a_=[q[0], T(FAKE + 2, BF, Tt, 512)]) == tp.TP_ERR_ALIGNMENT
    assert st(wsb=need - 1) == tp.TP_ERR_WORKSPACE
    assert st(ws=FAKE + 8) == tp.TP_ERR_ALIGNMENT
    p64 = tp.tp_plan_create(2, 256, 8, 2, 64, 16)                     # head_dim 64 is not built
    assert st(pl=p64) == tp.TP_ERR_UNSUPPORTED
    tp.tp_set_rank_health(1, False)
    try:
        assert st() == tp.TP_ERR_RANK_FAILED
    finally:
        tp.tp_set_rank_health(1, True)


def test_failed_rank_stops_the_group_before_any_launch():
    # Host-side fault injection: rank 1 reports unhealthy; every call that involves
    # it returns TP_ERR_RANK_FAILED before enqueuing work (no GPU needed).
    x = T(FAKE, BF, 64, 128)
    w = [T(FAKE, BF, 32, 128), T(FAKE, BF, 32, 128)]
    y = [T(FAKE, BF, 64, 64)]
    bufs = [T(FAKE, F32, 8, 8), T(FAKE + 1024, F32, 8, 8)]
    tp.tp_set_rank_health(1, False)
    try:
        assert col_status(2, x, w, y) == tp.TP_ERR_RANK_FAILED
        assert tp.raw_status("tp_allreduce_ring", 2, arr(*bufs), 0, None) == tp.TP_ERR_RANK_FAILED
        # a single-rank call does not involve rank 1
        assert tp.raw_status("tp_allreduce_ring", 1, arr(bufs[0]), 0, None) == tp.TP_OK
    finally:
        tp.tp_set_rank_health(1, True)
    assert tp.raw_status("tp_set_rank_health", 64, 0) == tp.TP_ERR_INVALID_ARG


def test_empty_inputs_enqueue_nothing():
    # zero tokens: valid, returns TP_OK without touching CUDA
    x = T(None, BF, 0, 128)
    w = [T(FAKE, BF, 32, 128), T(FAKE, BF, 32, 128)]
    y = [T(None, BF, 0, 64)]
    assert col_status(2, x, w, y) == tp.TP_OK
    empty = [T(None, F32, 0, 0, 1), T(None, F32, 0, 0, 1)]
    assert tp.raw_status("tp_allreduce_ring", 2, arr(*empty), 0, None) == tp.TP_OK


def test_every_call_takes_zero_tokens():
    # Valid shapes with T = 0 return TP_OK before any CUDA call: on this machine
    # (no device) any CUDA call would return an error instead.
    n, D, F = 2, 256, 512
    plan = tp.tp_plan_create(n, D, 4, 2, 128, F)   # 2 q heads and 1 kv head of 128 per rank
    x0 = T(None, BF, 0, D)
    wcol, wrow = [T(FAKE, BF, F // n, D)] * n, [T(FAKE, BF, D, F // n)] * n
    y0 = arr(*[T(None, F32, 0, D)] * n)
    q0, kv0 = [T(None, BF, 0, 256)] * n, [T(None, BF, 0, 128)] * n
    wq, wkv, wo = [T(FAKE, BF, 256, D)] * n, [T(FAKE, BF, 128, D)] * n, [T(FAKE, BF, D, 256)] * n
    flat0 = arr(*[T(None, F32, 0, 0, 1)] * n)
    ring = tp.TP_COMBINE_RING_FUSED
    moe = tp.moe_dims(n, tp.TP_MOE_WITHIN_EXPERT, 4, 2, D, F)
    calls = {
        "tp_row_linear": (n, arr(*[T(None, BF, 0, F // n)] * n), arr(*wrow), y0, ring, None),
        "tp_reduce_scatter": (n, flat0, 0, None),
        "tp_ring_all_gather": (n, flat0, 0, None),
        "tp_all_gather": (n, arr(*[T(None, BF, 0, 64)] * n), arr(T(None, BF, 0, 128)), 1, 1, None),
        "tp_reduce_scatter_bf16": (n, y0, arr(*[T(None, BF, 0, D)] * n), None),
        "tp_column_linear_chunks": (n, arr(*[T(None, BF, 0, D)] * n), arr(*wcol), arr(T(None, BF, 0, F)), 1, None),
        "tp_vocab_embedding": (n, None, 0, arr(*[T(FAKE, BF, 64, D)] * n), arr(T(None, BF, 0, D)), 1, None),
        "tp_vocab_lm_head": (n, ctypes.byref(x0), arr(*[T(FAKE, BF, 64, D)] * n), arr(T(None, F32, 0, 128)), 1,
                             None),
        "tp_attn_core": (plan.handle, arr(*q0), arr(*kv0), arr(*kv0), arr(*q0), 1, None, 0, None),
        "tp_moe_block": (ctypes.byref(moe), ctypes.byref(x0), None, None, arr(*[T(FAKE, BF, 4 * F // n, D)] * n),
                         arr(*[T(FAKE, BF, 4 * F // n, D)] * n), arr(*[T(FAKE, BF, 4 * D, F // n)] * n), y0, ring,
                         None, 0, None),
        "tp_gate_up_swiglu": (plan.handle, ctypes.byref(x0), arr(*wcol), arr(*wcol),
                              arr(*[T(None, BF, 0, F // n)] * n), None),
        "tp_mlp_block": (plan.handle, ctypes.byref(x0), arr(*wcol), arr(*wcol), arr(*wrow), y0, ring, None, 0, None),
        "tp_mlp_block_static": (plan.handle, ctypes.byref(x0), arr(*wcol), arr(*wcol), arr(*wrow), y0, ring, None),
        "tp_qkv_proj": (plan.handle, ctypes.byref(x0), arr(*wq), arr(*wkv), arr(*wkv), arr(*q0), arr(*kv0),
                        arr(*kv0), None),
        "tp_attn_proj": (plan.handle, ctypes.byref(x0), arr(*wq), arr(*wkv), arr(*wkv), arr(*q0), arr(*kv0),
                         arr(*kv0), arr(*q0), arr(*wo), y0, ring, None),
    }
    for name, args in calls.items():
        assert tp.raw_status(name, *args) == tp.TP_OK, name
    assert tp.tp_attn_core_workspace_size(plan, 0) == 0
    assert tp.tp_mlp_block_workspace_size(plan, 0) == 0
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except ImportError:
        has_gpu = False
    if not has_gpu:
        # control: the same call with one token passes validation and then fails at its first CUDA call
        m = 1 << 24
        xs = [T(FAKE + i * m, BF, 1, F // n) for i in range(n)]
        ws = [T(FAKE + (2 + i) * m, BF, D, F // n) for i in range(n)]
        ys = [T(FAKE + (4 + i) * m, F32, 1, D) for i in range(n)]
        assert tp.raw_status("tp_row_linear", n, arr(*xs), arr(*ws), arr(*ys), ring, None) == tp.TP_ERR_CUDA


def test_dimensions_fit_32_bit_indices():
    # rows and cols each below 2^31 (GEMM and TMA coordinates are 32-bit)
    big = 1 << 31
    w = [T(FAKE, BF, 32, 128), T(FAKE + (1 << 24), BF, 32, 128)]
    assert col_status(2, T(FAKE, BF, big, 128), w, [T(FAKE, BF, big, 64)] * 2, gather=0) == tp.TP_ERR_INVALID_ARG
    assert col_status(2, T(FAKE, BF, 64, big), [T(FAKE, BF, 32, big)] * 2, [T(FAKE, BF, 64, 64)]) == \
        tp.TP_ERR_INVALID_ARG
    flat = [T(FAKE, F32, big, 1), T(FAKE + (1 << 36), F32, big, 1)]
    assert tp.raw_status("tp_allreduce_ring", 2, arr(*flat), 0, None) == tp.TP_ERR_INVALID_ARG


def test_wait_budget_argument():
    assert tp.raw_status("tp_set_wait_budget", -1) == tp.TP_ERR_INVALID_ARG
    assert tp.raw_status("tp_set_wait_budget", 0) == tp.TP_OK
