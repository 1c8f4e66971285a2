"""fp64 CPU oracle of the tensor-parallel sharded linear block (GQA-aware).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this module. The library
(``tensor_sharded_linear_gqa_gb300``) never imports it and has no CPU fallback;
the two share no code. Inputs come from the seeded generators in
``tensor_sharded_linear_gqa_gb300.inputs``, which hold none of the method.

It is a plain, slow, obviously correct restatement of what the pages define:

[MLX]  mlxcel manual, "텐서 병렬화" (Tensor parallelism)
       - 개념 (Concept): every rank sees the same input, holds one shard of W.
       - 가중치 샤딩 전략 (Weight-sharding strategies): Column Parallel splits the
         output dimension, rank r holds W[:, r*D_out/N:(r+1)*D_out/N]; Row
         Parallel splits the input dimension, rank r holds W[r*D_in/N:(r+1)*D_in/N, :];
         Replicated keeps a full copy on every rank.
       - 통신 패턴 (Communication patterns): ring all-reduce = reduce-scatter then
         all-gather, 2*(N-1)/N*tensor_size sent per rank; in every step rank r
         sends to (r+1)%N and receives from (r+N-1)%N, N-1 steps.
       - 아키텍처 인식 샤드 플랜 (Architecture-aware shard plan): the standard
         transformer table (q/k/v/gate/up ColumnParallel, o/down RowParallel +
         AllReduce, q AllGather) and the GQA rule (shard K/V when
         num_kv_heads >= tp_size, replicate otherwise), with its two examples.
       - 설정 (Configuration): --tp-size is a power of two, default 1.
       - MoE 전문가 병렬화 (MoE expert parallelism): Expert Parallel puts
         expert i whole on rank i % tp_size; Within-Expert Parallel shards every
         expert's FFN over all ranks with the dense FFN's column-parallel
         gate/up and row-parallel down projections.
       - Vocab Parallel (a weight-sharding strategy) and 임베딩 및 LM Head 샤딩
         (Embedding and LM-head sharding): the vocabulary dimension of the
         embedding table and the LM head is split into contiguous per-rank
         slices; in vocab_parallel mode the lookup and the logits need an
         all-gather.
[WIKI] railscraft wiki, "텐서 병렬 처리" (Tensor parallel processing)
       - 상세 1 (Details 1, column & row parallel): Y_i = X W_i, Y = [Y_1..Y_n];
         Y_i = X_i W_i, Y = sum_i Y_i.
       - 예시 1 (Example 1): single-process column-parallel simulation; weights
         are stored [out x in] and each shard computes X * W_i^T.

Conventions (readings of the pages, each listed in the design notes):
  * Weights are stored [out x in] (the simulation's layout), Y = X * W^T. A
    "column shard" of the manual's W[D_in x D_out] is therefore a contiguous
    block of stored rows, a "row shard" a block of stored columns.
  * Ring chunks are contiguous flat ranges, chunk c = [floor(c*S/N), floor((c+1)*S/N)).
  * Reduce-scatter step s: rank r sends chunk (r-1-s) mod N to rank (r+1)%N, which
    adds it to its own copy; afterwards rank r holds the reduced chunk r.
    All-gather step s: rank r sends chunk (r-s) mod N, the receiver overwrites.
    A chunk received in step s is the one sent in step s+1.
  * The collectives compute in the dtype of the buffers they are given: float64
    by default, float32 when a caller wants the bit pattern of an fp32 ring
    (each add is one IEEE add in that precision, in the order above).
  * Activation of the MLP block: SwiGLU, silu(g) * u with silu(x) = x / (1 + e^-x)
    (the pages name no activation).
  * The o_proj input (attention context A) is an explicit input of the
    projection block. The attention core that produces it (attention_core_sharded)
    is scaled dot-product attention, causal for prefill, 1/sqrt(d) scale, no
    position encoding (the pages name none); each local q head uses the kv head
    the plan's q->kv map gives it.
  * MoE: the routing (top-k expert ids and weights per token) is an input; a
    rank's partial output sums, in slot order, the weighted contributions of the
    slots it runs, and the partials are all-reduced on the ring.
  * Vocab slices are equal (V divisible by N). The embedding all-gather moves
    each rank's looked-up rows ("piece") around the ring like any all-gather;
    every token's row comes from the one rank whose slice holds its id.

Parity status: every public function is pinned by a CPU test against facts the
pages and the mathematics fix (closed forms, worked examples, invariants,
brute force on tiny inputs); see tests/test_oracle_*.py. None is unpinned.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# Plan vocabulary ([MLX] 가중치 샤딩 전략 / 통신 패턴 / 아키텍처 인식 샤드 플랜)
# ---------------------------------------------------------------------------
COLUMN, ROW, VOCAB, REPLICATED = "ColumnParallel", "RowParallel", "VocabParallel", "Replicated"
NO_COMM, ALL_REDUCE, ALL_GATHER, REDUCE_SCATTER = "None", "AllReduce", "AllGather", "ReduceScatter"

WEIGHTS = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")


class PlanError(ValueError):
    """Raised for a configuration the plan rule does not accept. ``kind`` names why."""

    def __init__(self, kind: str, msg: str):
        super().__init__(msg)
        self.kind = kind


@dataclass
class RankShard:
    rank: int
    q_heads: tuple            # [begin, end) of global q heads on this rank
    kv_heads: tuple           # [begin, end) of global kv heads on this rank
    kv_replicated: bool
    strategy: dict = field(default_factory=dict)   # weight -> strategy
    comm: dict = field(default_factory=dict)       # weight -> comm pattern after it
    # weight -> [begin, end): output features (column weights) or input features
    # (row weights) of the manual's W[D_in x D_out] that this rank holds.
    ranges: dict = field(default_factory=dict)
    q_to_kv: list = field(default_factory=list)    # local q head -> local kv head


def _is_pow2(n: int) -> bool:
    return n >= 1 and (n & (n - 1)) == 0


def shard_plan(tp_size: int, hidden: int, num_q_heads: int, num_kv_heads: int,
               head_dim: int, ffn: int) -> list:
    """Per-rank shard plan of one decoder layer.

    [MLX] 설정: tp_size must be a power of two (default 1).
    [MLX] 아키텍처 인식 샤드 플랜, standard-transformer table: q/k/v ColumnParallel
    (q followed by AllGather), o RowParallel + AllReduce, gate/up ColumnParallel
    with no communication, down RowParallel + AllReduce.
    [MLX] GQA-aware attention sharding: num_kv_heads >= tp_size -> K/V sharded;
    num_kv_heads < tp_size -> K/V replicated on every rank (no rank gets a
    fraction of a KV head).
    Divisibility the pages leave open is required: q heads and ffn split evenly,
    q heads group evenly over kv heads, sharded kv heads split evenly.
    """
    N = tp_size
    if not _is_pow2(N):
        raise PlanError("tp_size_not_pow2", f"tp_size {N} is not a power of two")
    for name, v in (("hidden", hidden), ("num_q_heads", num_q_heads),
                    ("num_kv_heads", num_kv_heads), ("head_dim", head_dim), ("ffn", ffn)):
        if v < 1:
            raise PlanError("invalid", f"{name} must be >= 1")
    if num_q_heads % num_kv_heads != 0:
        raise PlanError("gqa_shape", "num_q_heads must be a multiple of num_kv_heads")
    if num_q_heads % N != 0:
        raise PlanError("gqa_shape", "num_q_heads must divide evenly over tp_size")
    replicated = num_kv_heads < N
    if not replicated and num_kv_heads % N != 0:
        raise PlanError("gqa_shape", "sharded num_kv_heads must divide evenly over tp_size")
    if ffn % N != 0:
        raise PlanError("not_divisible", "ffn must divide evenly over tp_size")

    q_per = num_q_heads // N
    group = num_q_heads // num_kv_heads          # q heads sharing one kv head
    plan = []
    for r in range(N):
        qb, qe = r * q_per, (r + 1) * q_per
        if replicated:
            kb, ke = 0, num_kv_heads
        else:
            kv_per = num_kv_heads // N
            kb, ke = r * kv_per, (r + 1) * kv_per
        fb, fe = r * (ffn // N), (r + 1) * (ffn // N)
        kv_strategy = REPLICATED if replicated else COLUMN
        s = RankShard(rank=r, q_heads=(qb, qe), kv_heads=(kb, ke), kv_replicated=replicated)
        s.strategy = {"q_proj": COLUMN, "k_proj": kv_strategy, "v_proj": kv_strategy,
                      "o_proj": ROW, "gate_proj": COLUMN, "up_proj": COLUMN,
                      "down_proj": ROW}
        s.comm = {"q_proj": ALL_GATHER, "k_proj": NO_COMM, "v_proj": NO_COMM,
                  "o_proj": ALL_REDUCE, "gate_proj": NO_COMM, "up_proj": NO_COMM,
                  "down_proj": ALL_REDUCE}
        s.ranges = {"q_proj": (qb * head_dim, qe * head_dim),
                    "k_proj": (kb * head_dim, ke * head_dim),
                    "v_proj": (kb * head_dim, ke * head_dim),
                    "o_proj": (qb * head_dim, qe * head_dim),
                    "gate_proj": (fb, fe), "up_proj": (fb, fe), "down_proj": (fb, fe)}
        # Local q head j is global head qb+j; it reads global kv head (qb+j)//group,
        # which sits at local index (that - kb) on this rank.
        s.q_to_kv = [(qb + j) // group - kb for j in range(q_per)]
        plan.append(s)
    return plan


# ---------------------------------------------------------------------------
# Linear algebra ([WIKI] 상세 1, 예시 1; [MLX] Column Parallel / Row Parallel)
# ---------------------------------------------------------------------------
def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Unsharded Y = X * W^T with W stored [out x in] ([WIKI] 예시 1)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    return x @ w.T


def split_rows(w: np.ndarray, n: int) -> list:
    """Column-parallel shards: contiguous blocks of stored rows (output features)."""
    out = w.shape[0]
    assert out % n == 0
    k = out // n
    return [w[r * k:(r + 1) * k, :] for r in range(n)]


def split_cols(a: np.ndarray, n: int) -> list:
    """Row-parallel shards: contiguous blocks of stored columns (input features)."""
    inn = a.shape[1]
    assert inn % n == 0
    k = inn // n
    return [a[:, r * k:(r + 1) * k] for r in range(n)]


def column_parallel(x: np.ndarray, w_shards: list) -> list:
    """Per-rank Y_r = X * W_r^T, X replicated ([MLX] Column Parallel; [WIKI] 상세 1)."""
    return [linear(x, w) for w in w_shards]


def all_gather_columns(ys: list) -> np.ndarray:
    """All-gather as concatenation along features, Y = [Y_1, ..., Y_N] ([WIKI] 상세 1)."""
    return np.concatenate([np.asarray(y, dtype=np.float64) for y in ys], axis=1)


def row_parallel(x_shards: list, w_shards: list) -> list:
    """Per-rank partial P_r = X_r * W_r^T ([MLX] Row Parallel; [WIKI] 상세 1)."""
    assert len(x_shards) == len(w_shards)
    return [linear(x, w) for x, w in zip(x_shards, w_shards)]


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + e^-x), in float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """SwiGLU gating of the MLP block: silu(g) * u."""
    return silu(g) * np.asarray(u, dtype=np.float64)


# ---------------------------------------------------------------------------
# Ring collectives ([MLX] 통신 패턴)
# ---------------------------------------------------------------------------
@dataclass
class RingLog:
    """What a simulated ring did: every send with its step, ends, chunk and bytes."""
    n: int
    sends: list = field(default_factory=list)  # (phase, step, src, dst, chunk, nbytes)

    def bytes_sent(self, rank: int, phase: str | None = None) -> int:
        return sum(b for (p, _s, src, _d, _c, b) in self.sends
                   if src == rank and (phase is None or p == phase))

    def steps(self, phase: str) -> int:
        st = {s for (p, s, *_rest) in self.sends if p == phase}
        return len(st)


def chunk_bounds(size: int, n: int, c: int) -> tuple:
    """Flat element range of ring chunk c of a buffer of ``size`` elements."""
    return (c * size) // n, ((c + 1) * size) // n


def ring_reduce_scatter(bufs: list, log: RingLog | None = None) -> list:
    """Ring reduce-scatter, in place on copies of ``bufs`` (flat per-rank buffers).

    N-1 steps; in step s every rank r sends chunk (r-1-s) mod N to (r+1)%N, which
    adds what it receives to its own copy of that chunk. All sends of a step are
    taken from the buffers as they stand before the step. Afterwards rank r holds
    the fully reduced chunk r ([MLX] 통신 패턴: All-reduce (ring), Reduce-scatter,
    ring topology).
    """
    n = len(bufs)
    out = [np.array(b, copy=True).reshape(-1) for b in bufs]
    size = out[0].size
    for s in range(n - 1):
        msgs = []
        for r in range(n):
            c = (r - 1 - s) % n
            lo, hi = chunk_bounds(size, n, c)
            msgs.append(((r + 1) % n, c, out[r][lo:hi].copy(), r))
        for dst, c, data, src in msgs:
            lo, hi = chunk_bounds(size, n, c)
            out[dst][lo:hi] = data + out[dst][lo:hi]
            if log is not None:
                log.sends.append(("reduce_scatter", s, src, dst, c, data.nbytes))
    return out


def ring_all_gather(bufs: list, log: RingLog | None = None) -> list:
    """Ring all-gather of chunk-owned buffers: rank r starts owning chunk r.

    N-1 steps; in step s rank r sends chunk (r-s) mod N to (r+1)%N, which
    overwrites its copy. Afterwards every rank holds every chunk
    ([MLX] 통신 패턴: All-gather, ring forwarding).
    """
    n = len(bufs)
    out = [np.array(b, copy=True).reshape(-1) for b in bufs]
    size = out[0].size
    for s in range(n - 1):
        msgs = []
        for r in range(n):
            c = (r - s) % n
            lo, hi = chunk_bounds(size, n, c)
            msgs.append(((r + 1) % n, c, out[r][lo:hi].copy(), r))
        for dst, c, data, src in msgs:
            lo, hi = chunk_bounds(size, n, c)
            out[dst][lo:hi] = data
            if log is not None:
                log.sends.append(("all_gather", s, src, dst, c, data.nbytes))
    return out


def ring_all_reduce(bufs: list, log: RingLog | None = None) -> list:
    """Ring all-reduce = reduce-scatter followed by all-gather ([MLX] 통신 패턴)."""
    return ring_all_gather(ring_reduce_scatter(bufs, log), log)


def gather_flat_shards(shards: list) -> np.ndarray:
    """Full tensor assembled from per-rank flat shards (rank r contributes chunk r)."""
    return np.concatenate([np.asarray(s).reshape(-1) for s in shards])


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16 (ties to even), returned as
    float64. bfloat16 keeps the top 16 bits of an IEEE float32 (8 exponent bits,
    7 stored mantissa bits); rounding adds half an ulp of the kept part, plus the
    kept part's lowest bit for ties, then truncates."""
    b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def reduce_scatter_then_column(partials: list, w_shards: list, round_bf16: bool = False,
                               log: RingLog | None = None) -> dict:
    """A row-parallel result feeding a column-parallel op directly ([MLX] 통신 패턴,
    Reduce-scatter: used when a row-parallel result goes straight into a
    column-parallel op; the all-gather step is avoided).

    The per-rank partials [T x K] are reduce-scattered on the ring (rank c ends
    holding reduced chunk c); optionally the reduced values are rounded to
    bfloat16, the operand type of the next GEMM. The column-parallel op then
    multiplies the input made of the N reduced chunks, taken where they lie, by
    each rank's weight shard. Returns the chunks, that input and the outputs.
    """
    n = len(partials)
    t, k = np.asarray(partials[0]).shape
    rs = ring_reduce_scatter(partials, log)
    chunks = []
    for c in range(n):
        lo, hi = chunk_bounds(t * k, n, c)
        v = rs[c][lo:hi]
        chunks.append(round_to_bf16(v) if round_bf16 else v)
    x = gather_flat_shards(chunks).reshape(t, k)
    return {"chunks": chunks, "x": x, "y": column_parallel(x.astype(np.float64), w_shards)}


# ---------------------------------------------------------------------------
# Vocab parallel ([MLX] 가중치 샤딩 전략, Vocab Parallel; 임베딩 및 LM Head 샤딩)
# ---------------------------------------------------------------------------
def vocab_ranges(vocab: int, n: int) -> list:
    """[begin, end) of the token ids each rank holds: the vocabulary dimension
    is split into N contiguous slices of V/N ids ([MLX] Vocab Parallel: every
    rank owns one contiguous slice of the token vocabulary). V must divide by N,
    as every other split dimension must."""
    if not _is_pow2(n):
        raise PlanError("tp_size", f"tp_size {n} is not a power of two")
    if vocab <= 0 or vocab % n:
        raise PlanError("not_divisible", f"vocab {vocab} does not split over {n} ranks")
    per = vocab // n
    return [(r * per, (r + 1) * per) for r in range(n)]


def embedding(ids, table) -> np.ndarray:
    """The plain lookup: row i of the result is row ids[i] of the table [V x D]."""
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    table = np.asarray(table, dtype=np.float64)
    if ids.size and (ids.min() < 0 or ids.max() >= table.shape[0]):
        raise ValueError("token id outside the vocabulary")
    out = np.empty((ids.size, table.shape[1]))
    for i, t in enumerate(ids):
        out[i] = table[t]
    return out


def vocab_parallel_embedding(ids, table_shards: list, log: RingLog | None = None) -> dict:
    """Embedding lookup over a vocab-sharded table ([MLX] 임베딩 및 LM Head 샤딩,
    vocab_parallel: the vocabulary dimension is sharded and the lookup needs an
    all-gather).

    Rank r holds table rows [r*V/N, (r+1)*V/N) as its shard. It looks up the
    tokens whose ids fall in its slice, at local row id - r*V/N, and contributes
    those rows (its "piece", keyed by token position). The pieces are all-gathered
    on the ring (step s: rank r forwards piece (r-s) mod N to (r+1)%N), after
    which every rank holds every token's row, taken from the one rank owning it.
    """
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    n = len(table_shards)
    per = np.asarray(table_shards[0]).shape[0]
    d = np.asarray(table_shards[0]).shape[1]
    rng_ = vocab_ranges(per * n, n)
    if ids.size and (ids.min() < 0 or ids.max() >= per * n):
        raise ValueError("token id outside the vocabulary")
    pieces = []
    for r, (lo, hi) in enumerate(rng_):
        shard = np.asarray(table_shards[r], dtype=np.float64)
        pos = [i for i in range(ids.size) if lo <= ids[i] < hi]
        rows = np.array([shard[ids[i] - lo] for i in pos]).reshape(len(pos), d)
        pieces.append((pos, rows))
    # ring all-gather of the pieces: held[r] = {owner: piece} that rank r has
    held = [{r: pieces[r]} for r in range(n)]
    for s in range(n - 1):
        msgs = []
        for r in range(n):
            owner = (r - s) % n
            msgs.append(((r + 1) % n, owner, held[r][owner], r))
        for dst, owner, piece, src in msgs:
            held[dst][owner] = piece
            if log is not None:
                log.sends.append(("all_gather", s, src, dst, owner, piece[1].nbytes))
    outs = []
    for r in range(n):
        y = np.full((ids.size, d), np.nan)
        for owner in range(n):
            pos, rows = held[r][owner]
            for j, i in enumerate(pos):
                y[i] = rows[j]
        outs.append(y)
    return {"pieces": pieces, "y": outs}


def vocab_parallel_lm_head(x, w_shards: list) -> dict:
    """LM-head logits over a vocab-sharded weight ([MLX] 임베딩 및 LM Head 샤딩,
    vocab_parallel: the logits need an all-gather). Weights are stored [V x D];
    rank r's shard is rows [r*V/N, (r+1)*V/N), so its logits X W_r^T are the
    columns of its vocabulary slice, and the all-gather concatenates them in
    rank order into the full [T x V] logits."""
    parts = column_parallel(x, w_shards)
    return {"parts": parts, "logits": all_gather_columns(parts)}


# ---------------------------------------------------------------------------
# Blocks ([MLX] 아키텍처 인식 샤드 플랜; [WIKI] 상세 1, last paragraph)
# ---------------------------------------------------------------------------
def mlp_unsharded(x, wg, wu, wd) -> np.ndarray:
    """Y = (silu(X Wg^T) * (X Wu^T)) Wd^T, the plain definition."""
    return linear(swiglu(linear(x, wg), linear(x, wu)), wd)


def mlp_sharded(x, wg, wu, wd, tp_size: int, log: RingLog | None = None) -> dict:
    """MLP block sharded per the plan table: gate/up ColumnParallel (no comm),
    down RowParallel + ring AllReduce. Returns per-rank H_r, partials P_r and
    the all-reduced per-rank outputs (each [T x D])."""
    T = x.shape[0]
    D = wd.shape[0]
    g = column_parallel(x, split_rows(wg, tp_size))
    u = column_parallel(x, split_rows(wu, tp_size))
    h = [swiglu(gr, ur) for gr, ur in zip(g, u)]
    p = row_parallel(h, split_cols(wd, tp_size))
    y = ring_all_reduce([pr.reshape(-1) for pr in p], log)
    return {"h": h, "partials": p, "y": [yr.reshape(T, D) for yr in y]}


# ---------------------------------------------------------------------------
# Attention core between q/k/v and o_proj ([MLX] GQA 인식 어텐션 샤딩: each rank
# attends with its own q heads over the kv heads the plan gives it)
# ---------------------------------------------------------------------------
def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row-wise softmax exp(s - max) / sum exp(s - max); -inf entries get 0."""
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=1, keepdims=True)


def attention_head(q, k, v, causal: bool) -> np.ndarray:
    """Scaled dot-product attention of one head: softmax(q k^T / sqrt(d)) v,
    with query i seeing keys j <= i when causal. q [T x d], k and v [T x d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (q @ k.T) / np.sqrt(q.shape[1])
    if causal:
        t = s.shape[0]
        s = np.where(np.arange(t)[None, :] <= np.arange(t)[:, None], s, -np.inf)
    return softmax_rows(s) @ v


def attention_core_sharded(q, k, v, plan: list, head_dim: int, causal: bool = True) -> list:
    """Rank r's attention output A_r [T x Hq_r*d]: for each of its local q heads h,
    attention_head of q head h with the kv head q_to_kv[h] of the rank's K/V
    (its own kv heads when sharded, all of them when replicated). q[r] is
    [T x Hq_r*d]; k[r], v[r] are [T x Hkv_r*d] (one shared entry when the plan
    replicates K/V). A_r's columns are the rank's slice of the o_proj input."""
    out = []
    d = head_dim
    for r, s in enumerate(plan):
        kr = k[0] if s.kv_replicated else k[r]
        vr = v[0] if s.kv_replicated else v[r]
        heads = []
        for h, g in enumerate(s.q_to_kv):
            heads.append(attention_head(q[r][:, h * d:(h + 1) * d], kr[:, g * d:(g + 1) * d],
                                        vr[:, g * d:(g + 1) * d], causal))
        out.append(np.concatenate(heads, axis=1))
    return out


# ---------------------------------------------------------------------------
# Mixture of experts ([MLX] MoE 전문가 병렬화: Expert Parallel, Within-Expert Parallel)
# ---------------------------------------------------------------------------
MOE_EXPERT_PARALLEL, MOE_WITHIN_EXPERT = "expert_parallel", "within_expert"


def expert_rank(expert: int, tp_size: int) -> int:
    """Rank holding expert i whole in expert-parallel mode: experts are dealt to
    the ranks round-robin, expert i on rank i % tp_size ([MLX] Expert Parallel)."""
    return expert % tp_size


def moe_unsharded(x, topk_ids, topk_w, wg, wu, wd) -> np.ndarray:
    """The plain top-k mixture: token t's output is the sum over its k routing
    slots j of topk_w[t, j] times expert topk_ids[t, j]'s FFN (the dense MLP's
    SwiGLU definition with that expert's weights) applied to x[t]. The routing
    (ids and weights) is an input; the router itself is not part of the block."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    y = np.zeros((x.shape[0], np.asarray(wd[0]).shape[0]))
    for t in range(x.shape[0]):
        for j in range(ids.shape[1]):
            e = ids[t, j]
            y[t] += w[t, j] * mlp_unsharded(x[t:t + 1], wg[e], wu[e], wd[e])[0]
    return y


def moe_sharded(x, topk_ids, topk_w, wg, wu, wd, tp_size: int, mode: str,
                log: RingLog | None = None) -> dict:
    """MoE block over tp_size ranks ([MLX] MoE 전문가 병렬화).

    expert_parallel: rank r runs, whole, the experts i with i % tp_size == r and
    only the routing slots that chose them; no communication inside an expert.
    within_expert: every expert's FFN is sharded over all ranks like the dense
    FFN (gate/up column-parallel, down row-parallel), so rank r runs every slot
    with its slice of every expert.
    Either way rank r's partial output sums its slots' weighted contributions,
    and the partials are combined by the ring all-reduce (the row-parallel
    down projection's all-reduce, as in the dense FFN; the router runs on every
    rank, so every rank sees the same routing).
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    n, T = tp_size, x.shape[0]
    D = np.asarray(wd[0]).shape[0]
    if mode not in (MOE_EXPERT_PARALLEL, MOE_WITHIN_EXPERT):
        raise ValueError(f"unknown MoE mode {mode}")
    partials = [np.zeros((T, D)) for _ in range(n)]
    for r in range(n):
        for t in range(T):
            for j in range(ids.shape[1]):
                e = ids[t, j]
                if mode == MOE_EXPERT_PARALLEL:
                    if expert_rank(e, n) != r:
                        continue
                    contrib = mlp_unsharded(x[t:t + 1], wg[e], wu[e], wd[e])[0]
                else:
                    g_r = split_rows(np.asarray(wg[e], dtype=np.float64), n)[r]
                    u_r = split_rows(np.asarray(wu[e], dtype=np.float64), n)[r]
                    d_r = split_cols(np.asarray(wd[e], dtype=np.float64), n)[r]
                    contrib = linear(swiglu(linear(x[t:t + 1], g_r), linear(x[t:t + 1], u_r)), d_r)[0]
                partials[r][t] += w[t, j] * contrib
    y = ring_all_reduce([p.reshape(-1) for p in partials], log)
    return {"partials": partials, "y": [yr.reshape(T, D) for yr in y]}


def attn_proj_unsharded(x, wq, wk, wv, a, wo) -> dict:
    """q/k/v = X W^T for each projection; Y = A Wo^T."""
    return {"q": linear(x, wq), "k": linear(x, wk), "v": linear(x, wv), "y": linear(a, wo)}


def attn_proj_sharded(x, wq, wk, wv, a, wo, plan: list, head_dim: int,
                      log: RingLog | None = None) -> dict:
    """Attention projections sharded per the plan: q/k/v column-parallel on the
    rank's heads (K/V whole on every rank when replicated), o_proj row-parallel on
    the rank's slice of A + ring all-reduce."""
    q, k, v, parts = [], [], [], []
    for s in plan:
        qb, qe = s.ranges["q_proj"]
        kb, ke = s.ranges["k_proj"]
        q.append(linear(x, wq[qb:qe, :]))
        k.append(linear(x, wk[kb:ke, :]))
        v.append(linear(x, wv[kb:ke, :]))
        ob, oe = s.ranges["o_proj"]
        parts.append(linear(a[:, ob:oe], wo[:, ob:oe]))
    T, D = a.shape[0], wo.shape[0]
    y = ring_all_reduce([p.reshape(-1) for p in parts], log)
    return {"q": q, "k": k, "v": v, "partials": parts, "y": [yr.reshape(T, D) for yr in y]}
