"""GPU parity of the vocab-parallel embedding lookup and LM head ([MLX] 가중치
샤딩 전략, Vocab Parallel; 임베딩 및 LM Head 샤딩, vocab_parallel), through the C ABI.

The lookup moves bits, so it must equal the oracle's lookup exactly, with no
byte written outside the outputs' rows. A bad token id leaves zero rows and is
reported by tp_device_status as TP_ERR_BAD_TOKEN, after which the context works
on. The LM head equals the oracle exactly on small-integer inputs and within
the bf16 tolerance on normal ones.
"""
import numpy as np
import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp
from tensor_sharded_linear_gqa_gb300 import inputs
from gpu_util import BF16_TOL, assert_close, dev_bf16, dev_f32, host_f64, need_gpu

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _ids(v, n, extra, seed):
    """Every slice's first and last id, then uniform ids (repeats included)."""
    per = v // n
    b = [x for r in range(n) for x in (r * per, (r + 1) * per - 1)]
    return np.concatenate([np.array(b, dtype=np.int32), inputs.token_ids(seed, 0, extra, v)])


def _dev_ids(ids):
    return _torch().from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()


def _nan_like(rows, cols, dtype, ld=None):
    torch = _torch()
    buf = torch.full((rows, ld or cols), float("nan"), dtype=dtype, device="cuda")
    return buf, buf[:, :cols]


@pytest.mark.parametrize("n,v,d", [(1, 64, 64), (2, 256, 128), (4, 512, 8192), (8, 1024, 96),
                                   (8, 128, 100), (2, 64, 7)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("per_rank_out", [False, True])
def test_embedding_matches_the_oracle_exactly(n, v, d, dtype, per_rank_out):
    torch = _torch()
    need_gpu()
    ids = _ids(v, n, 77, n * v + d)
    if dtype == "bf16":
        bits = inputs.normal_bf16(401, d, (v, d))
        table_f64, table_dev, tdt = inputs.bf16_bits_to_f64(bits), dev_bf16(bits), torch.bfloat16
    else:
        a = inputs.normal_f32(401, d, (v, d))
        table_f64, table_dev, tdt = a.astype(np.float64), dev_f32(a), torch.float32
    per = v // n
    shards = [table_dev[r * per:(r + 1) * per] for r in range(n)]
    bufs = [_nan_like(ids.size, d, tdt, ld=d + 8) for _ in range(n if per_rank_out else 1)]
    tp.tp_vocab_embedding(n, _dev_ids(ids), shards, [b[1] for b in bufs])
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    ref = O.vocab_parallel_embedding(ids, O.split_rows(table_f64, n))["y"]
    for o, (buf, view) in enumerate(bufs):
        assert np.array_equal(host_f64(view), ref[o]), f"output {o}"
        assert torch.isnan(buf[:, d:]).all()  # the padding past D is untouched


def test_embedding_strided_and_unaligned_views():
    """Shards that are column views of a wider buffer (row pitch > D) and outputs
    that start one element past a 16-byte boundary take the element path."""
    torch = _torch()
    need_gpu()
    n, v, d = 4, 256, 64
    bits = inputs.normal_bf16(402, 1, (v, d + 24))
    wide = dev_bf16(bits)
    per = v // n
    shards = [wide[r * per:(r + 1) * per, 3:3 + d] for r in range(n)]  # base 6 bytes in
    ids = _ids(v, n, 40, 9)
    buf = torch.full((ids.size, d + 9), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[:, 1:1 + d]
    tp.tp_vocab_embedding(n, _dev_ids(ids), shards, [out])
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    table = inputs.bf16_bits_to_f64(bits)[:, 3:3 + d]
    assert np.array_equal(host_f64(out), O.embedding(ids, table))
    assert torch.isnan(buf[:, 0]).all() and torch.isnan(buf[:, 1 + d:]).all()


def test_embedding_skewed_and_single_token():
    torch = _torch()
    need_gpu()
    n, v, d = 8, 1024, 256
    bits = inputs.normal_bf16(403, 1, (v, d))
    table = dev_bf16(bits)
    shards = [table[r * (v // n):(r + 1) * (v // n)] for r in range(n)]
    for ids in (np.full(300, 5, dtype=np.int32), np.array([v - 1], dtype=np.int32)):
        out = torch.empty((ids.size, d), dtype=torch.bfloat16, device="cuda")
        tp.tp_vocab_embedding(n, _dev_ids(ids), shards, [out])
        assert np.array_equal(host_f64(out), O.embedding(ids, inputs.bf16_bits_to_f64(bits)))
    assert tp.tp_device_status() == (tp.TP_OK, 0)


def test_bad_token_ids_give_zero_rows_and_a_status():
    torch = _torch()
    need_gpu()
    n, v, d = 2, 64, 64
    bits = inputs.normal_bf16(404, 1, (v, d))
    table = dev_bf16(bits)
    shards = [table[:32], table[32:]]
    ids = np.array([3, -1, 40, v, 63], dtype=np.int32)
    out = torch.full((ids.size, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    tp.tp_vocab_embedding(n, _dev_ids(ids), shards, [out])
    st, word = tp.tp_device_status()
    assert st == tp.TP_ERR_BAD_TOKEN and word != 0
    got = host_f64(out)
    assert np.all(got[[1, 3]] == 0.0)
    good = [0, 2, 4]
    assert np.array_equal(got[good], O.embedding(ids[good], inputs.bf16_bits_to_f64(bits)))
    # the status word was cleared and the context still works
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    tp.tp_vocab_embedding(n, _dev_ids(ids[good]), shards, [out[:3]])
    assert tp.tp_device_status() == (tp.TP_OK, 0)


@pytest.mark.parametrize("n,t,d,v", [(2, 64, 128, 512), (4, 200, 192, 1024), (8, 300, 256, 2048),
                                     (8, 8, 64, 128)])
@pytest.mark.parametrize("gather", [0, 1])
def test_lm_head_exact_small_integers(n, t, d, v, gather):
    torch = _torch()
    need_gpu()
    x = inputs.small_int_bf16(405, n, (t, d))
    w = inputs.small_int_bf16(405, 100 + n, (v, d))
    wd = dev_bf16(w)
    per = v // n
    shards = [wd[r * per:(r + 1) * per] for r in range(n)]
    logits = ([torch.full((t, v), float("nan"), device="cuda")] if gather else
              [torch.full((t, per), float("nan"), device="cuda") for _ in range(n)])
    tp.tp_vocab_lm_head(n, dev_bf16(x), shards, logits, gather=bool(gather))
    ref = O.vocab_parallel_lm_head(inputs.bf16_bits_to_f64(x), O.split_rows(inputs.bf16_bits_to_f64(w), n))
    if gather:
        assert np.array_equal(host_f64(logits[0]), ref["logits"])
    else:
        for r in range(n):
            assert np.array_equal(host_f64(logits[r]), ref["parts"][r])


def test_lm_head_bf16_normal_and_bf16_logits():
    torch = _torch()
    need_gpu()
    n, t, d, v = 4, 384, 1024, 4096
    x = inputs.normal_bf16(406, 1, (t, d))
    w = inputs.normal_bf16(406, 2, (v, d), 0.02)
    wd = dev_bf16(w)
    shards = [wd[r * (v // n):(r + 1) * (v // n)] for r in range(n)]
    ref = O.vocab_parallel_lm_head(inputs.bf16_bits_to_f64(x), O.split_rows(inputs.bf16_bits_to_f64(w), n))
    for dt in (torch.float32, torch.bfloat16):
        logits = torch.full((t, v), float("nan"), dtype=dt, device="cuda")
        tp.tp_vocab_lm_head(n, dev_bf16(x), shards, [logits], gather=True)
        assert_close(host_f64(logits), ref["logits"], BF16_TOL, str(dt))


@pytest.mark.parametrize("n", [1, 2, 8])
def test_tied_table_argmax_recovers_the_ids(n):
    """Embedding and LM head share the table 2*I (V = D = 256): the logits of each
    looked-up token are 4 at its id and 0 elsewhere."""
    torch = _torch()
    need_gpu()
    v = 256
    table = (2.0 * torch.eye(v, device="cuda")).to(torch.bfloat16)
    shards = [table[r * (v // n):(r + 1) * (v // n)] for r in range(n)]
    ids = _ids(v, n, 120, n)
    x = torch.empty((ids.size, v), dtype=torch.bfloat16, device="cuda")
    tp.tp_vocab_embedding(n, _dev_ids(ids), shards, [x])
    logits = torch.empty((ids.size, v), device="cuda")
    tp.tp_vocab_lm_head(n, x, shards, [logits], gather=True)
    assert np.array_equal(torch.argmax(logits, dim=1).cpu().numpy(), ids)
    assert tp.tp_device_status() == (tp.TP_OK, 0)


def test_vocab_tp8_t4096_in_the_benchmark_configuration():
    """The benchmarked workload: 4096 ids looked up in the 128256 x 8192 table
    sharded over 8 ranks (checked exactly for every row), and the LM-head logits
    of 4096 hidden states over the whole vocabulary, gathered into one f32
    [4096 x 128256] tensor (checked on a seeded sample of rows)."""
    torch = _torch()
    need_gpu()
    w = inputs.WORKLOADS["vocab_tp8_t4096"]
    n, t, d, v = w["tp"], w["T"], w["hidden"], w["vocab"]
    data = inputs.make_bf16_inputs(w)
    per = v // n
    emb = dev_bf16(data["emb"])
    out = torch.empty((t, d), dtype=torch.bfloat16, device="cuda")
    tp.tp_vocab_embedding(n, _dev_ids(data["ids"]), [emb[r * per:(r + 1) * per] for r in range(n)], [out])
    assert tp.tp_device_status() == (tp.TP_OK, 0)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, data["emb"][data["ids"]])  # bits of the looked-up rows
    del emb, out
    wlm = dev_bf16(data["wlm"])
    logits = torch.empty((t, v), device="cuda")
    tp.tp_vocab_lm_head(n, dev_bf16(data["x"]), [wlm[r * per:(r + 1) * per] for r in range(n)], [logits],
                        gather=True)
    torch.cuda.synchronize()
    rows = np.sort(inputs.rng(w["seed"], 99).choice(t, size=24, replace=False))
    ref = O.vocab_parallel_lm_head(inputs.bf16_bits_to_f64(data["x"][rows]),
                                   O.split_rows(inputs.bf16_bits_to_f64(data["wlm"]), n))["logits"]
    assert_close(host_f64(logits[torch.from_numpy(rows).cuda()]), ref, BF16_TOL, "logits")
    assert tp.tp_device_status() == (tp.TP_OK, 0)
