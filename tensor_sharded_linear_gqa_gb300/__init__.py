"""Python binding of libtpgqa, the tensor-parallel sharded linear block on GB300.

Argument marshalling only: every function forwards to the C entry point of the
same name (declared in include/tpgqa.h); every step of the computation runs in
the library's CUDA kernels. There is no CPU fallback: the first call loads
``libtpgqa.so`` and raises ImportError when it is missing (build it with
``python -m tensor_sharded_linear_gqa_gb300.build``).

Tensors are passed either as ``TpTensor`` or as 2-D CUDA ``torch.Tensor`` views
with unit column stride (float32 or bfloat16). Per-rank arguments are Python
sequences. ``stream`` is a ``torch.cuda.Stream``, a raw ``cudaStream_t`` int, or
None for the current torch stream.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtpgqa.so")


# ---- constants (mirror include/tpgqa.h) ------------------------------------
TP_OK = 0
STATUS_NAMES = ["TP_OK", "TP_ERR_INVALID_ARG", "TP_ERR_TP_SIZE_NOT_POW2", "TP_ERR_NOT_DIVISIBLE",
                "TP_ERR_GQA_SHAPE", "TP_ERR_DTYPE", "TP_ERR_ALIGNMENT", "TP_ERR_RANK_FAILED",
                "TP_ERR_TIMEOUT", "TP_ERR_CUDA", "TP_ERR_WORKSPACE", "TP_ERR_UNSUPPORTED",
                "TP_ERR_BAD_TOKEN"]
for _i, _n in enumerate(STATUS_NAMES):
    globals()[_n] = _i
TP_F32, TP_BF16 = 0, 1
TP_SHARD_COLUMN, TP_SHARD_ROW, TP_SHARD_VOCAB, TP_SHARD_REPLICATED = 0, 1, 2, 3
TP_COMM_NONE, TP_COMM_ALL_REDUCE, TP_COMM_ALL_GATHER, TP_COMM_REDUCE_SCATTER = 0, 1, 2, 3
TP_W_Q, TP_W_K, TP_W_V, TP_W_O, TP_W_GATE, TP_W_UP, TP_W_DOWN, TP_W_COUNT = range(8)
WEIGHT_NAMES = ["q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj"]
TP_COMBINE_NONE, TP_COMBINE_FUSED, TP_COMBINE_RING, TP_COMBINE_RING_FUSED, TP_COMBINE_RING_SHARED = 0, 1, 2, 3, 4
TP_RING_STEPS, TP_RING_FUSED, TP_RING_FUSED_SHARED = 0, 1, 2
TP_MOE_EXPERT_PARALLEL, TP_MOE_WITHIN_EXPERT = 0, 1


class TpTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld", ctypes.c_int64)]


class TpDims(ctypes.Structure):
    _fields_ = [("tp_size", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32)]


class TpRankShard(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("q_head_begin", ctypes.c_int32),
                ("q_head_end", ctypes.c_int32), ("kv_head_begin", ctypes.c_int32),
                ("kv_head_end", ctypes.c_int32), ("kv_replicated", ctypes.c_int32),
                ("strategy", ctypes.c_int32 * TP_W_COUNT), ("comm", ctypes.c_int32 * TP_W_COUNT),
                ("range_begin", ctypes.c_int64 * TP_W_COUNT),
                ("range_end", ctypes.c_int64 * TP_W_COUNT)]


class TpMoeDims(ctypes.Structure):
    _fields_ = [("tp_size", ctypes.c_int32), ("mode", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64)]


class TPError(RuntimeError):
    def __init__(self, status: int, where: str):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else f"status {status}"
        extra = ""
        if status == 9:  # TP_ERR_CUDA
            extra = f" (cudaError {int(_lib.tp_last_cuda_error())})"
        super().__init__(f"{where}: {name}{extra}")
        self.status = status
        self.name = name


_P = ctypes.POINTER
_T = _P(TpTensor)
_S = ctypes.c_void_p  # cudaStream_t
_SIGS = {
    "tp_plan_create": ([_P(TpDims), _P(ctypes.c_void_p)], ctypes.c_int),
    "tp_plan_destroy": ([ctypes.c_void_p], ctypes.c_int),
    "tp_plan_dims": ([ctypes.c_void_p, _P(TpDims)], ctypes.c_int),
    "tp_plan_query_rank": ([ctypes.c_void_p, ctypes.c_int32, _P(TpRankShard)], ctypes.c_int),
    "tp_plan_q_to_kv": ([ctypes.c_void_p, ctypes.c_int32, _P(ctypes.c_int32), ctypes.c_int32],
                        ctypes.c_int),
    "tp_column_linear": ([ctypes.c_int32, _T, _T, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_row_linear": ([ctypes.c_int32, _T, _T, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_reduce_scatter": ([ctypes.c_int32, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_reduce_scatter_bf16": ([ctypes.c_int32, _T, _T, _S], ctypes.c_int),
    "tp_column_linear_chunks": ([ctypes.c_int32, _T, _T, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_ring_all_gather": ([ctypes.c_int32, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_allreduce_ring": ([ctypes.c_int32, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_all_gather": ([ctypes.c_int32, _T, _T, ctypes.c_int32, ctypes.c_int32, _S], ctypes.c_int),
    "tp_vocab_embedding": ([ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, _T, _T, ctypes.c_int32, _S],
                           ctypes.c_int),
    "tp_vocab_lm_head": ([ctypes.c_int32, _T, _T, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_attn_core_workspace_size": ([ctypes.c_void_p, ctypes.c_int64], ctypes.c_size_t),
    "tp_attn_core": ([ctypes.c_void_p, _T, _T, _T, _T, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, _S],
                     ctypes.c_int),
    "tp_moe_workspace_size": ([_P(TpMoeDims), ctypes.c_int64], ctypes.c_size_t),
    "tp_moe_block": ([_P(TpMoeDims), _T, ctypes.c_void_p, ctypes.c_void_p, _T, _T, _T, _T, ctypes.c_int32,
                      ctypes.c_void_p, ctypes.c_size_t, _S], ctypes.c_int),
    "tp_gate_up_swiglu": ([ctypes.c_void_p, _T, _T, _T, _T, _S], ctypes.c_int),
    "tp_mlp_block_workspace_size": ([ctypes.c_void_p, ctypes.c_int64], ctypes.c_size_t),
    "tp_mlp_block": ([ctypes.c_void_p, _T, _T, _T, _T, _T, ctypes.c_int32, ctypes.c_void_p,
                      ctypes.c_size_t, _S], ctypes.c_int),
    "tp_mlp_block_static": ([ctypes.c_void_p, _T, _T, _T, _T, _T, ctypes.c_int32, _S], ctypes.c_int),
    "tp_mlp_block_static_max_bytes": ([], ctypes.c_size_t),
    "tp_qkv_proj": ([ctypes.c_void_p, _T, _T, _T, _T, _T, _T, _T, _S], ctypes.c_int),
    "tp_attn_proj": ([ctypes.c_void_p, _T, _T, _T, _T, _T, _T, _T, _T, _T, _T, ctypes.c_int32,
                      _S], ctypes.c_int),
    "tp_status_str": ([ctypes.c_int], ctypes.c_char_p),
    "tp_last_cuda_error": ([], ctypes.c_int32),
    "tp_set_rank_health": ([ctypes.c_int32, ctypes.c_int32], ctypes.c_int),
    "tp_device_status": ([_S, _P(ctypes.c_int32)], ctypes.c_int),
    "tp_set_wait_budget": ([ctypes.c_int64], ctypes.c_int),
    "tp_debug_wait_timeout": ([_S], ctypes.c_int),
    "tp_launch_count": ([], ctypes.c_uint64),
    "tp_version": ([], ctypes.c_char_p),
}
EXPORTED = tuple(_SIGS)


class _Lib:
    """The loaded libtpgqa.so; loading fails loudly when the library is missing."""

    def __init__(self):
        self._cdll = None

    def __getattr__(self, name):
        if self._cdll is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -m tensor_sharded_linear_gqa_gb300.build); there is no CPU fallback")
            cdll = ctypes.CDLL(LIB_PATH)
            for n, (args, res) in _SIGS.items():
                f = getattr(cdll, n)
                f.argtypes = args
                f.restype = res
            self._cdll = cdll
        return getattr(self._cdll, name)


_lib = _Lib()


def load() -> ctypes.CDLL:
    """Loads the library now (raises ImportError if it is missing) and returns it."""
    _lib.tp_version  # noqa: B018
    return _lib._cdll


def _check(status: int, where: str) -> None:
    if status != TP_OK:
        raise TPError(status, where)


# ---- marshalling ------------------------------------------------------------
def tensor(t) -> TpTensor:
    """TpTensor view of a 2-D CUDA torch tensor with unit column stride (or a TpTensor)."""
    if isinstance(t, TpTensor):
        return t
    import torch
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.numel() > 0 and t.stride(1) != 1:
        raise ValueError("expected unit stride along columns")
    if t.dtype == torch.float32:
        dt = TP_F32
    elif t.dtype == torch.bfloat16:
        dt = TP_BF16
    else:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.numel() > 0 and not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    ld = t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1], 1)
    return TpTensor(t.data_ptr() if t.numel() > 0 else None, dt, 0, t.shape[0], t.shape[1], ld)


def _arr(seq):
    seq = list(seq)
    a = (TpTensor * max(len(seq), 1))()
    for i, t in enumerate(seq):
        a[i] = tensor(t)
    return a


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- plan -----------------------------------------------------------------------
class Plan:
    """Owner of a tp_plan*; freed with tp_plan_destroy."""

    def __init__(self, handle: int, dims: TpDims):
        self.handle = handle
        self.dims = dims

    @property
    def tp_size(self) -> int:
        return self.dims.tp_size

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            _lib.tp_plan_destroy(h)
            self.handle = None


def tp_plan_create(tp_size: int, hidden: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   ffn: int) -> Plan:
    d = TpDims(tp_size, hidden, num_q_heads, num_kv_heads, head_dim, ffn)
    h = ctypes.c_void_p()
    _check(_lib.tp_plan_create(ctypes.byref(d), ctypes.byref(h)), "tp_plan_create")
    return Plan(h.value, d)


def tp_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        _check(_lib.tp_plan_destroy(plan.handle), "tp_plan_destroy")
        plan.handle = None


def tp_plan_query_rank(plan: Plan, rank: int) -> dict:
    s = TpRankShard()
    _check(_lib.tp_plan_query_rank(plan.handle, rank, ctypes.byref(s)), "tp_plan_query_rank")
    return {
        "rank": s.rank,
        "q_heads": (s.q_head_begin, s.q_head_end),
        "kv_heads": (s.kv_head_begin, s.kv_head_end),
        "kv_replicated": bool(s.kv_replicated),
        "strategy": {WEIGHT_NAMES[i]: s.strategy[i] for i in range(TP_W_COUNT)},
        "comm": {WEIGHT_NAMES[i]: s.comm[i] for i in range(TP_W_COUNT)},
        "ranges": {WEIGHT_NAMES[i]: (s.range_begin[i], s.range_end[i]) for i in range(TP_W_COUNT)},
    }


def tp_plan_q_to_kv(plan: Plan, rank: int) -> list:
    cap = max(plan.dims.num_q_heads, 1)
    out = (ctypes.c_int32 * cap)()
    _check(_lib.tp_plan_q_to_kv(plan.handle, rank, out, cap), "tp_plan_q_to_kv")
    s = tp_plan_query_rank(plan, rank)
    return [out[j] for j in range(s["q_heads"][1] - s["q_heads"][0])]


# ---- linear layers and collectives ---------------------------------------------
def tp_column_linear(tp_size: int, x, w, y, gather: bool, stream=None) -> None:
    xs = tensor(x)
    _check(_lib.tp_column_linear(tp_size, ctypes.byref(xs), _arr(w), _arr(y), int(gather),
                                 _stream(stream)), "tp_column_linear")


def tp_row_linear(tp_size: int, x, w, y, combine: int, stream=None) -> None:
    _check(_lib.tp_row_linear(tp_size, _arr(x), _arr(w), _arr(y), combine, _stream(stream)),
           "tp_row_linear")


def tp_reduce_scatter(tp_size: int, bufs, mode: int = TP_RING_STEPS, stream=None) -> None:
    _check(_lib.tp_reduce_scatter(tp_size, _arr(bufs), mode, _stream(stream)), "tp_reduce_scatter")


def tp_reduce_scatter_bf16(tp_size: int, partials, out, stream=None) -> None:
    """Ring reduce-scatter of f32 partials; chunk r of out[r] receives the bf16 sum."""
    _check(_lib.tp_reduce_scatter_bf16(tp_size, _arr(partials), _arr(out), _stream(stream)),
           "tp_reduce_scatter_bf16")


def tp_column_linear_chunks(tp_size: int, x_chunks, w, y, gather: bool, stream=None) -> None:
    """Column-parallel linear whose input rows [c*T/N, (c+1)*T/N) are read from x_chunks[c]."""
    _check(_lib.tp_column_linear_chunks(tp_size, _arr(x_chunks), _arr(w), _arr(y), int(gather),
                                        _stream(stream)), "tp_column_linear_chunks")


def tp_ring_all_gather(tp_size: int, bufs, mode: int = TP_RING_STEPS, stream=None) -> None:
    _check(_lib.tp_ring_all_gather(tp_size, _arr(bufs), mode, _stream(stream)),
           "tp_ring_all_gather")


def tp_allreduce_ring(tp_size: int, bufs, mode: int = TP_RING_STEPS, stream=None) -> None:
    _check(_lib.tp_allreduce_ring(tp_size, _arr(bufs), mode, _stream(stream)), "tp_allreduce_ring")


def tp_all_gather(tp_size: int, shards, outs, axis: int, stream=None) -> None:
    outs = list(outs)
    _check(_lib.tp_all_gather(tp_size, _arr(shards), _arr(outs), len(outs), axis, _stream(stream)),
           "tp_all_gather")


def ids_ptr(ids) -> int:
    """Device address of a contiguous int32 CUDA tensor of token ids (0 when empty)."""
    if str(ids.dtype) != "torch.int32" or not ids.is_contiguous():
        raise TypeError("token ids must be a contiguous int32 tensor")
    return ids.data_ptr() if ids.numel() else 0


def tp_vocab_embedding(tp_size: int, ids, table, outs, stream=None) -> None:
    """Rows ids[i] of the vocab-sharded table (table[r] = rank r's slice) into
    every output (1 shared copy or tp_size copies)."""
    outs = list(outs)
    _check(_lib.tp_vocab_embedding(tp_size, ids_ptr(ids), ids.numel(), _arr(table), _arr(outs), len(outs),
                                   _stream(stream)), "tp_vocab_embedding")


def tp_vocab_lm_head(tp_size: int, x, w, logits, gather: bool, stream=None) -> None:
    xs = tensor(x)
    _check(_lib.tp_vocab_lm_head(tp_size, ctypes.byref(xs), _arr(w), _arr(logits), int(gather),
                                 _stream(stream)), "tp_vocab_lm_head")


def tp_attn_core_workspace_size(plan: Plan, tokens: int) -> int:
    return int(_lib.tp_attn_core_workspace_size(plan.handle, tokens))


def tp_attn_core(plan: Plan, q, k, v, a, causal: bool, workspace, stream=None) -> None:
    """q[r], a[r]: rank r's [T x Hq_r*d] bf16; k, v: one entry per rank, or one
    shared entry when the plan replicates K/V; workspace: a CUDA byte tensor."""
    _check(_lib.tp_attn_core(plan.handle, _arr(q), _arr(k), _arr(v), _arr(a), int(causal),
                             workspace.data_ptr(), workspace.numel(), _stream(stream)), "tp_attn_core")


def moe_dims(tp_size: int, mode: int, num_experts: int, top_k: int, hidden: int, ffn: int) -> TpMoeDims:
    return TpMoeDims(tp_size, mode, num_experts, top_k, hidden, ffn)


def tp_moe_workspace_size(dims: TpMoeDims, tokens: int) -> int:
    return int(_lib.tp_moe_workspace_size(ctypes.byref(dims), tokens))


def _dev_ptr(t, dtype: str) -> int:
    if str(t.dtype) != dtype or not t.is_contiguous():
        raise TypeError(f"expected a contiguous {dtype} tensor")
    return t.data_ptr() if t.numel() else 0


def tp_moe_block(dims: TpMoeDims, x, topk_ids, topk_w, w_gate, w_up, w_down, y, combine: int, workspace,
                 stream=None) -> None:
    """topk_ids: int32 [T x k] CUDA tensor; topk_w: float32 [T x k]; workspace: a
    CUDA byte tensor of at least tp_moe_workspace_size bytes."""
    xs = tensor(x)
    _check(_lib.tp_moe_block(ctypes.byref(dims), ctypes.byref(xs), _dev_ptr(topk_ids, "torch.int32"),
                             _dev_ptr(topk_w, "torch.float32"), _arr(w_gate), _arr(w_up), _arr(w_down),
                             _arr(y), combine, workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "tp_moe_block")


def tp_gate_up_swiglu(plan: Plan, x, w_gate, w_up, h, stream=None) -> None:
    xs = tensor(x)
    _check(_lib.tp_gate_up_swiglu(plan.handle, ctypes.byref(xs), _arr(w_gate), _arr(w_up), _arr(h),
                                  _stream(stream)), "tp_gate_up_swiglu")


def tp_mlp_block_workspace_size(plan: Plan, tokens: int) -> int:
    return int(_lib.tp_mlp_block_workspace_size(plan.handle, tokens))


def tp_mlp_block(plan: Plan, x, w_gate, w_up, w_down, y, combine: int, workspace,
                 workspace_bytes: int | None = None, stream=None) -> None:
    """``workspace`` is a CUDA torch tensor (any dtype) or a raw device pointer int."""
    if isinstance(workspace, int) or workspace is None:
        wptr, wbytes = workspace, workspace_bytes or 0
    else:
        wptr = workspace.data_ptr()
        wbytes = workspace.numel() * workspace.element_size()
    xs = tensor(x)
    _check(_lib.tp_mlp_block(plan.handle, ctypes.byref(xs), _arr(w_gate), _arr(w_up),
                             _arr(w_down), _arr(y), combine, wptr, wbytes, _stream(stream)),
           "tp_mlp_block")


def tp_mlp_block_static(plan: Plan, x, w_gate, w_up, w_down, y, combine: int, stream=None) -> None:
    """tp_mlp_block without a workspace argument, for callers that cannot allocate
    device memory: H lives in the library's fixed 16 MiB scratch array. Calls on
    one device share that array, so calls that overlap on the GPU race."""
    xs = tensor(x)
    _check(_lib.tp_mlp_block_static(plan.handle, ctypes.byref(xs), _arr(w_gate), _arr(w_up),
                                    _arr(w_down), _arr(y), combine, _stream(stream)),
           "tp_mlp_block_static")


def tp_mlp_block_static_max_bytes() -> int:
    return int(_lib.tp_mlp_block_static_max_bytes())


def tp_qkv_proj(plan: Plan, x, w_q, w_k, w_v, q, k, v, stream=None) -> None:
    xs = tensor(x)
    _check(_lib.tp_qkv_proj(plan.handle, ctypes.byref(xs), _arr(w_q), _arr(w_k), _arr(w_v), _arr(q),
                            _arr(k), _arr(v), _stream(stream)), "tp_qkv_proj")


def tp_attn_proj(plan: Plan, x, w_q, w_k, w_v, q, k, v, a, w_o, y, combine: int,
                 stream=None) -> None:
    xs = tensor(x)
    _check(_lib.tp_attn_proj(plan.handle, ctypes.byref(xs), _arr(w_q), _arr(w_k), _arr(w_v),
                             _arr(q), _arr(k), _arr(v), _arr(a), _arr(w_o), _arr(y), combine,
                             _stream(stream)), "tp_attn_proj")


# ---- status and diagnostics ---------------------------------------------------
def tp_status_str(status: int) -> str:
    return _lib.tp_status_str(status).decode()


def tp_last_cuda_error() -> int:
    return int(_lib.tp_last_cuda_error())


def tp_set_rank_health(rank: int, healthy: bool) -> None:
    _check(_lib.tp_set_rank_health(rank, int(healthy)), "tp_set_rank_health")


def tp_device_status(stream=None) -> tuple:
    """(status, raw word): synchronises the stream and reads/clears the device status word."""
    word = ctypes.c_int32(0)
    st = _lib.tp_device_status(_stream(stream), ctypes.byref(word))
    return st, word.value


def tp_set_wait_budget(nanoseconds: int) -> None:
    _check(_lib.tp_set_wait_budget(nanoseconds), "tp_set_wait_budget")


def tp_debug_wait_timeout(stream=None) -> None:
    _check(_lib.tp_debug_wait_timeout(_stream(stream)), "tp_debug_wait_timeout")


def tp_launch_count() -> int:
    """Kernel launches the library has enqueued in this process so far."""
    return int(_lib.tp_launch_count())


def tp_version() -> str:
    return _lib.tp_version().decode()


def arr(seq):
    """ctypes array of TpTensor for a per-rank argument (kept alive by the caller)."""
    return _arr(seq)


class Prepared:
    """A C entry point with its arguments marshalled once, for tight loops: calling
    it makes only the ctypes call. Raises TPError on a non-OK status."""

    def __init__(self, fn_name: str, *args):
        self.fn = getattr(_lib, fn_name)
        self.name = fn_name
        self.args = args  # keeps the ctypes objects alive

    def __call__(self) -> None:
        st = self.fn(*self.args)
        if st != TP_OK:
            raise TPError(st, self.name)


def raw_status(fn_name: str, *args) -> int:
    """Calls a C entry point with ready-made ctypes arguments and returns its status
    (for tests of the error paths)."""
    return getattr(_lib, fn_name)(*args)
