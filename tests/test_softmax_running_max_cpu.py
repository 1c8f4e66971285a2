"""The reading behind the attention kernels' softmax, checked on the CPU.

The kernels take p = 2^(s*c - m) against a running row maximum m (c = log2(e) /
sqrt(d)). A row's maximum is found only on its first 128-key block, or on a later
block whose sum of p passes 2^64. Then m moves to that block's maximum if it
exceeds m by more than 8 (log2 units), p is taken again, and the row's output is
rescaled by 2^(m_old - m_new). Softmax does not change with the constant taken off
a row's scores. So the rule, carried out in f32 with p rounded to bf16 for the P V
product as the kernels do, must give the oracle's softmax(Q K^T / sqrt(d)) V
within the bf16 tolerance. This holds even when a row's later blocks score far
above its first. The blockwise rule is written out here in numpy, independently of
the GPU; inputs built the same way run through the kernels in the GPU attention
test of the lagging and moving maximum.
"""
import numpy as np
import pytest

import oracle as O
from tensor_sharded_linear_gqa_gb300 import inputs

BLOCK = 128
SUM_LIMIT = 2.0 ** 64
TOL = 1e-2  # max|A - A_ref| <= TOL * max|A_ref|, the bf16 tolerance of the GPU tests


def blockwise_attention(q, k, v, causal, rescale=True):
    """One head, row by row, block by block, in f32: the kernels' rule."""
    f32 = np.float32
    t, d = q.shape
    c = f32(np.log2(np.e) / np.sqrt(d))
    s_all = q.astype(f32) @ k.astype(f32).T
    out = np.zeros((t, d))
    stats = {"lagging": 0, "moved_late": 0}
    for i in range(t):
        m, l = f32(-np.inf), f32(0.0)
        o = np.zeros(d, dtype=f32)
        nkeys = i + 1 if causal else k.shape[0]
        for j0 in range(0, nkeys, BLOCK):
            s = s_all[i, j0:j0 + BLOCK].copy()
            s[max(0, nkeys - j0):] = -np.inf  # masked keys
            find = j0 == 0
            while True:
                move, m_new = False, m
                if find:
                    m_blk = f32(s.max() * c)
                    move = bool(m_blk > m + f32(8.0))
                    m_new = m_blk if move else m
                with np.errstate(over="ignore"):  # p = inf sends the block to the fallback, as on the GPU
                    p = np.exp2((s * c - m_new).astype(f32)).astype(f32)
                    total = p.sum(dtype=f32)
                if find or total <= SUM_LIMIT:
                    break
                find = True  # the sum passed the limit: find the maximum, take p again
            if j0 > 0 and find:
                stats["moved_late"] += 1
            elif j0 > 0 and p.max() > 1.0:
                stats["lagging"] += 1
            alpha = np.exp2(f32(m - m_new)).astype(f32) if move else f32(1.0)
            l = f32(l * alpha + total)
            if move and j0 > 0 and rescale:
                o = (o * alpha).astype(f32)
            pb = O.round_to_bf16(p.astype(np.float64)).astype(f32)
            o = (o + pb @ v[j0:j0 + BLOCK].astype(f32)).astype(f32)
            m = m_new
        out[i] = o / l
    return out, stats


def _inputs(t, d, seed):
    """bf16 q, k, v; the keys of the second and third 128-key blocks scaled by 8
    and by 30, so that (at seed 630, over the 512 rows) the block maxima lie 15 to
    47 and 61 to 180 (log2 units) above the first block's, and the fourth block
    is back to ordinary scores."""
    q = inputs.bf16_bits_to_f64(inputs.normal_bf16(seed, 1, (t, d)))
    factor = np.ones((t, 1), dtype=np.float32)
    factor[128:256] = 8.0
    factor[256:384] = 30.0
    k = inputs.bf16_bits_to_f64(inputs.f32_to_bf16_bits(inputs.normal_f32(seed, 2, (t, d)) * factor))
    v = inputs.bf16_bits_to_f64(inputs.normal_bf16(seed, 3, (t, d)))
    return q, k, v


def _rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))


@pytest.mark.parametrize("causal", [False, True])
def test_running_maximum_rule_gives_the_softmax(causal):
    q, k, v = _inputs(512, 128, seed=630)
    got, stats = blockwise_attention(q, k, v, causal)
    ref = O.attention_head(q, k, v, causal)
    assert _rel_err(got, ref) <= TOL
    # both departures from a per-block maximum occur: p above 1 against a lagging
    # maximum, and a later block whose sum passed the limit and moved the maximum
    assert stats["lagging"] > 0 and stats["moved_late"] > 0


def test_a_missing_rescale_is_caught():
    """A planted mistake: moving the maximum without rescaling the row's output
    must fail the same comparison."""
    q, k, v = _inputs(512, 128, seed=630)
    got, _ = blockwise_attention(q, k, v, False, rescale=False)
    assert _rel_err(got, O.attention_head(q, k, v, False)) > TOL
