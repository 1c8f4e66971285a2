"""Seeded synthetic inputs and workload shapes for the tensor-parallel linear block.

This module is shared by the tests, the benchmark and ``smoke()``. It draws
random numbers, rounds them to bf16 bit patterns and describes the shapes of
the workloads. It holds none of the block's arithmetic (no products, sums,
activations, shard plans or collectives), so both the CUDA path and the fp64
oracle can take their inputs from it without sharing any of the method.

Generator: numpy PCG64 through ``SeedSequence(seed, spawn_key=(stream,))``; one
independent stream per tensor (see ``STREAM``). Values are drawn as float64
normals, narrowed to float32 and rounded to bf16 by round-to-nearest-even on
the bit pattern. The oracle widens the same bits exactly to float64.
"""
from __future__ import annotations

import numpy as np

# One independent random stream per tensor role.
STREAM = {
    "x": 0,      # activations X [T x hidden]
    "a": 1,      # attention context A [T x q_heads*head_dim] (input of o_proj)
    "wq": 2, "wk": 3, "wv": 4, "wo": 5,
    "wg": 6, "wu": 7, "wd": 8,
    "w": 9,      # plain linear weight of the fp32 worked example
    "buf": 10,   # raw collective buffers
    "h": 11,     # row-parallel input H [T x ffn] of the reduce-scatter pipeline
    "wqkv": 12,  # fused per-rank q/k/v weight of the reduce-scatter pipeline
    "ids": 13,   # token ids of the vocab-parallel lookup
    "emb": 14,   # embedding table [V x D]
    "wlm": 15,   # LM-head weight [V x D]
    "route": 16,  # MoE routing: expert ids and weights per token
    "eg": 17, "eu": 18, "ed": 19,  # MoE expert weights [E x F x D], [E x F x D], [E x D x F]
    "aq": 20, "ak": 21, "av": 22,  # attention core inputs Q [T x Hq*d], K and V [T x Hkv*d]
}

# Workloads, named by what they are. Weight tensors are stored [out x in]
# row-major (K-major). ``w_std`` is the standard deviation of the weights,
# activations are N(0, 1).
WORKLOADS = {
    # Column-parallel simulation worked example of the railscraft wiki page
    # (in 1024, out 2048, two virtual GPUs, batch 32), run in fp32 both as a
    # column-parallel and as a row-parallel layer.
    "wiki_linear_fp32_tp2": dict(kind="linear_fp32", T=32, d_in=1024, d_out=2048,
                                 tp=2, seed=101, w_std=1.0),
    # Llama-style MLP block, TP=2, bf16.
    "mlp_tp2_t512": dict(kind="mlp", T=512, hidden=2048, ffn=8192, tp=2,
                         seed=102, w_std=0.02),
    # Attention projections with GQA sharding, TP=4, bf16.
    "attn_gqa_tp4_t2048": dict(kind="attn", T=2048, hidden=4096, q_heads=32,
                               kv_heads=8, head_dim=128, tp=4, seed=103,
                               w_std=0.02),
    # Decode-shaped step: 4 KV heads replicated over 8 ranks, bf16.
    "decode_gqa_rep_tp8_t64": dict(kind="layer", T=64, hidden=4096, q_heads=32,
                                   kv_heads=4, head_dim=128, ffn=14336, tp=8,
                                   seed=104, w_std=0.02),
    # Large decoder-layer projections + MLP prefill, TP=8, bf16.
    "prefill_layer_tp8_t4096": dict(kind="layer", T=4096, hidden=8192, q_heads=64,
                                    kv_heads=8, head_dim=128, ffn=28672, tp=8,
                                    seed=105, w_std=0.02, oracle_rows=64),
    # The prefill layer with its attention: q/k/v projections, causal attention
    # core, o_proj + all-reduce, then the MLP block (no explicit A input).
    "decoder_layer_tp8_t4096": dict(kind="layer", attention=True, T=4096, hidden=8192, q_heads=64,
                                    kv_heads=8, head_dim=128, ffn=28672, tp=8, seed=110, w_std=0.02),
    # Row-parallel down projection whose result feeds the next layer's q/k/v
    # projection (column-parallel) through a reduce-scatter, TP=8, bf16. The
    # q/k/v weights are stored fused per rank: rank r's rows are its q heads,
    # then its k head, then its v head.
    "rs_column_tp8_t4096": dict(kind="rs_column", T=4096, hidden=8192, q_heads=64,
                                kv_heads=8, head_dim=128, ffn=28672, tp=8,
                                seed=106, w_std=0.02),
    # Vocab-parallel embedding lookup and LM head of a 128256-token vocabulary
    # (above the 100k tokens where vocab sharding pays), hidden 8192, TP=8, bf16
    # with f32 logits: 4096 uniformly drawn token ids are looked up, and the
    # logits of 4096 hidden states are computed over the whole vocabulary.
    "vocab_tp8_t4096": dict(kind="vocab", T=4096, hidden=8192, vocab=128256, tp=8,
                            seed=107, w_std=0.02),
    # Attention core of the prefill layer: causal attention of 4096 tokens,
    # 64 q heads and 8 kv heads of 128 over 8 ranks (8 q heads and 1 kv head
    # each); Q, K, V drawn N(0,1).
    "attn_core_tp8_t4096": dict(kind="attn_core", T=4096, hidden=8192, q_heads=64, kv_heads=8,
                                head_dim=128, tp=8, seed=109),
    # Mixtral-8x7B-shaped MoE layer: 8 experts of hidden 4096 and FFN 14336, top-2
    # routing drawn uniformly (two distinct experts a token, softmax weights over
    # the two), 4096 tokens, TP=8; within-expert sharding (F/N = 1792 per rank).
    "moe_mixtral_tp8_t4096": dict(kind="moe", T=4096, hidden=4096, ffn=14336, experts=8, top_k=2,
                                  tp=8, seed=108, w_std=0.02),
}


def rng(seed: int, stream: int) -> np.random.Generator:
    """Independent PCG64 generator for (seed, stream)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(stream,))))


def normal_f32(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) samples as float32."""
    g = rng(seed, stream)
    out = g.standard_normal(size=shape, dtype=np.float64)
    if std != 1.0:
        out *= std
    return out.astype(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 exactly."""
    return bf16_bits_to_f32(b).astype(np.float64)


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16, as uint16 bit patterns.

    Large tensors are drawn in blocks of leading rows from one generator: the
    values are the same as from one draw of the whole shape (the generator is
    consumed in order), with a bounded peak of host memory."""
    shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
    total = int(np.prod(shape))
    if total <= _BLOCK or len(shape) < 2:
        return f32_to_bf16_bits(normal_f32(seed, stream, shape, std))
    g = rng(seed, stream)
    out = np.empty(shape, dtype=np.uint16)
    step = max(1, _BLOCK // int(np.prod(shape[1:])))
    for r0 in range(0, shape[0], step):
        blk = g.standard_normal(size=(min(step, shape[0] - r0),) + shape[1:], dtype=np.float64)
        if std != 1.0:
            blk *= std
        out[r0:r0 + blk.shape[0]] = f32_to_bf16_bits(blk.astype(np.float32))
    return out


_BLOCK = 1 << 24  # elements per block of normal_bf16


def token_ids(seed: int, stream: int, n: int, vocab: int) -> np.ndarray:
    """n token ids drawn uniformly from [0, vocab), as int32."""
    return rng(seed, stream).integers(0, vocab, size=n).astype(np.int32)


def routing(seed: int, stream: int, tokens: int, experts: int, k: int) -> tuple:
    """Synthetic top-k routing: k distinct experts per token drawn uniformly
    (int32 [T x k]) and weights that are the softmax of k N(0,1) draws (float32)."""
    g = rng(seed, stream)
    keys = g.random((tokens, experts))
    ids = np.argsort(keys, axis=1)[:, :k].astype(np.int32)  # a uniform k-subset, in random order
    z = g.standard_normal((tokens, k))
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return ids, (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def small_int_bf16(seed: int, stream: int, shape, lo: int = -4, hi: int = 4) -> np.ndarray:
    """Uniform integers in [lo, hi] as bf16 bits (exact in bf16; used for bit-exact cases)."""
    g = rng(seed, stream)
    v = g.integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(v)


def small_int_f32(seed: int, stream: int, shape, lo: int = -4, hi: int = 4) -> np.ndarray:
    """Uniform integers in [lo, hi] as float32."""
    g = rng(seed, stream)
    return g.integers(lo, hi + 1, size=shape).astype(np.float32)


def weight_shapes(w: dict) -> dict:
    """Full (unsharded) weight shapes [out x in] of a workload."""
    kind = w["kind"]
    if kind == "linear_fp32":
        return {"w": (w["d_out"], w["d_in"])}
    D = w["hidden"]
    out = {}
    if kind in ("attn", "layer"):
        hd = w["head_dim"]
        out.update(wq=(w["q_heads"] * hd, D), wk=(w["kv_heads"] * hd, D),
                   wv=(w["kv_heads"] * hd, D), wo=(D, w["q_heads"] * hd))
    if kind in ("mlp", "layer"):
        F = w["ffn"]
        out.update(wg=(F, D), wu=(F, D), wd=(D, F))
    if kind == "vocab":
        out.update(emb=(w["vocab"], D), wlm=(w["vocab"], D))
    if kind == "moe":
        E, F = w["experts"], w["ffn"]
        out.update(eg=(E, F, D), eu=(E, F, D), ed=(E, D, F))
    if kind == "rs_column":
        n, hd = w["tp"], w["head_dim"]
        per = (w["q_heads"] // n + 2 * max(1, w["kv_heads"] // n)) * hd
        out.update(wd=(D, w["ffn"]), wqkv=(n * per, D))
    return out


def make_bf16_inputs(w: dict, rows: int | None = None) -> dict:
    """Full bf16 inputs (uint16 bits) of a bf16 workload.

    ``x`` and ``a`` are [T x .] N(0,1); weights are N(0, w_std^2). ``rows`` limits
    nothing here: activations are always drawn whole so that a row sample of them
    is the same bits the GPU sees.
    """
    seed, T = w["seed"], w["T"]
    out = {"x": normal_bf16(seed, STREAM["x"], (T, w["hidden"]))}
    if w["kind"] == "rs_column":
        out["h"] = normal_bf16(seed, STREAM["h"], (T, w["ffn"]))
    if w["kind"] == "vocab":
        out["ids"] = token_ids(seed, STREAM["ids"], T, w["vocab"])
    if w["kind"] == "moe":
        out["topk_ids"], out["topk_w"] = routing(seed, STREAM["route"], T, w["experts"], w["top_k"])
    if w["kind"] == "attn_core":
        hd = w["head_dim"]
        out["q"] = normal_bf16(seed, STREAM["aq"], (T, w["q_heads"] * hd))
        out["k"] = normal_bf16(seed, STREAM["ak"], (T, w["kv_heads"] * hd))
        out["v"] = normal_bf16(seed, STREAM["av"], (T, w["kv_heads"] * hd))
    if w["kind"] in ("attn", "layer") and not w.get("attention"):
        out["a"] = normal_bf16(seed, STREAM["a"], (T, w["q_heads"] * w["head_dim"]))
    for name, shp in weight_shapes(w).items():
        out[name] = normal_bf16(seed, STREAM[name], shp, w["w_std"])
    return out


def make_fp32_linear_inputs(w: dict) -> dict:
    """fp32 inputs of the worked fp32 linear example: X [T x d_in], W [d_out x d_in]."""
    seed = w["seed"]
    return {"x": normal_f32(seed, STREAM["x"], (w["T"], w["d_in"])),
            "w": normal_f32(seed, STREAM["w"], (w["d_out"], w["d_in"]), w["w_std"])}
