/*
 * tpgqa.h - C ABI of the tensor-parallel sharded linear block (GQA-aware) on
 * one GB300 (sm_103a).
 *
 * Execution model. All N logical tensor-parallel ranks live in one GPU's HBM
 * and run in lockstep in one process (mlxcel manual "텐서 병렬화", section
 * 현재 런타임 지원 범위 / Current runtime support: in-process multi-rank). A
 * rank's shard is a tp_tensor; a "collective" is a kernel that moves or reduces
 * shard buffers on this one device. No peer-to-peer or network traffic exists.
 *
 * Weights are stored [out x in], row-major (K-major), and every linear
 * computes Y = X * W^T (railscraft wiki "텐서 병렬 처리", 예시 1 / Example 1). A
 * column shard of the manual's W[D_in x D_out] is therefore a contiguous block
 * of stored rows; a row shard is a block of stored columns.
 *
 * Conventions shared by every call:
 *  - Ownership: the caller owns every tensor buffer and every workspace; the
 *    library allocates no device memory in these calls. The only object the
 *    library owns is tp_plan (host memory, freed by tp_plan_destroy).
 *  - Streams: every call that touches device memory only enqueues work on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream) and returns
 *    without synchronising. Buffers must stay valid until that work is done.
 *  - Overlap: kernels are launched with programmatic dependent launch, so a
 *    call's kernels may start while the previous kernel on the stream is still
 *    running; they wait for it before touching activations, outputs or
 *    workspaces. Weights (the w arguments of the GEMM calls, which no earlier
 *    kernel of a step writes) are read from the start, so the first weight
 *    tiles stream in during the previous kernel's tail. A weight buffer must
 *    therefore not be written by the kernel that immediately precedes its use
 *    on the same stream (put an event wait, a host synchronisation or other
 *    work in between), or set the environment variable TPGQA_EARLY_B=0 (read at
 *    every launch) to make weight loads wait as well. Block-table (MoE) GEMMs
 *    never read weights early.
 *  - Pointers: tp_tensor.ptr is a device pointer. Arrays of tp_tensor
 *    (per-rank arguments) are host arrays, read during the call only.
 *  - Errors: every call returns a tp_status and never aborts. Arguments are
 *    checked before any launch; on an error nothing is enqueued. TP_ERR_CUDA
 *    means a CUDA runtime call failed; tp_last_cuda_error() gives its code.
 *    Device-side errors (a bounded wait that ran out) are recorded in a device
 *    status word and reported by tp_device_status().
 *  - Alignment: tensors handed to the tensor-core (bf16) path need a 16-byte
 *    aligned base and a row pitch (ld * element size) that is a multiple of 16
 *    bytes, else TP_ERR_ALIGNMENT. Collective buffers need a 16-byte aligned
 *    base.
 *  - Empty inputs: zero rows (tokens) or zero elements is valid and enqueues
 *    nothing.
 *  - Thread safety: calls on different streams may run concurrently; a plan
 *    is immutable after creation and may be shared.
 */
#ifndef TPGQA_H
#define TPGQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *tp_stream_t;

typedef enum tp_status {
  TP_OK = 0,
  TP_ERR_INVALID_ARG = 1,      /* null pointer, bad shape, bad mode, ...            */
  TP_ERR_TP_SIZE_NOT_POW2 = 2, /* tp_size is not a power of two (설정 / --tp-size)   */
  TP_ERR_NOT_DIVISIBLE = 3,    /* ffn (or another split dimension) not divisible by N */
  TP_ERR_GQA_SHAPE = 4,        /* head counts the GQA rule cannot shard             */
  TP_ERR_DTYPE = 5,            /* dtype combination not supported                    */
  TP_ERR_ALIGNMENT = 6,        /* base or pitch not 16-byte aligned                  */
  TP_ERR_RANK_FAILED = 7,      /* a rank is marked unhealthy (tp_set_rank_health)    */
  TP_ERR_TIMEOUT = 8,          /* a bounded device-side wait ran out                 */
  TP_ERR_CUDA = 9,             /* a CUDA runtime call failed; see tp_last_cuda_error */
  TP_ERR_WORKSPACE = 10,       /* workspace missing or too small                     */
  TP_ERR_UNSUPPORTED = 11,     /* valid request the library does not implement       */
  TP_ERR_BAD_TOKEN = 12        /* an embedding lookup met a token id outside [0, V)  */
} tp_status;

typedef enum tp_dtype { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;

/* A 2-D row-major view: element (i, j) lives at ptr + (i * ld + j) * size(dtype).
 * ld >= cols. rows or cols may be 0 (empty); each is below 2^31 (their product,
 * and ld, are not limited). */
typedef struct tp_tensor {
  void *ptr;
  int32_t dtype; /* tp_dtype */
  int32_t reserved;
  int64_t rows;
  int64_t cols;
  int64_t ld;
} tp_tensor;

/* ---------------------------------------------------------------------------
 * Shard plan (mlxcel manual "텐서 병렬화": 가중치 샤딩 전략 / Weight-sharding
 * strategies; 아키텍처 인식 샤드 플랜 / Architecture-aware shard plan, its
 * standard-transformer table and the GQA-aware attention sharding rule).
 * ------------------------------------------------------------------------- */
typedef struct tp_dims {
  int32_t tp_size;      /* N, a power of two >= 1                      */
  int32_t hidden;       /* D                                           */
  int32_t num_q_heads;  /* Hq                                          */
  int32_t num_kv_heads; /* Hkv; Hq must be a multiple of Hkv           */
  int32_t head_dim;     /* hd                                          */
  int32_t ffn;          /* F, divisible by N                           */
} tp_dims;

typedef enum tp_shard_strategy {
  TP_SHARD_COLUMN = 0,
  TP_SHARD_ROW = 1,
  TP_SHARD_VOCAB = 2,
  TP_SHARD_REPLICATED = 3
} tp_shard_strategy;

typedef enum tp_comm_pattern {
  TP_COMM_NONE = 0,
  TP_COMM_ALL_REDUCE = 1,
  TP_COMM_ALL_GATHER = 2,
  TP_COMM_REDUCE_SCATTER = 3
} tp_comm_pattern;

typedef enum tp_weight {
  TP_W_Q = 0, TP_W_K = 1, TP_W_V = 2, TP_W_O = 3,
  TP_W_GATE = 4, TP_W_UP = 5, TP_W_DOWN = 6,
  TP_W_COUNT = 7
} tp_weight;

typedef struct tp_rank_shard {
  int32_t rank;
  int32_t q_head_begin, q_head_end;   /* global q heads [begin, end) on this rank        */
  int32_t kv_head_begin, kv_head_end; /* global kv heads on this rank (all when replicated) */
  int32_t kv_replicated;              /* 1 when num_kv_heads < tp_size                   */
  int32_t strategy[TP_W_COUNT];       /* tp_shard_strategy per weight                    */
  int32_t comm[TP_W_COUNT];           /* tp_comm_pattern that follows the weight         */
  /* Feature range [begin, end) this rank holds: output features for column
   * weights (q, k, v, gate, up), input features for row weights (o, down),
   * in the manual's W[D_in x D_out] terms (rows of the [out x in] storage for
   * column weights, columns of it for row weights). */
  int64_t range_begin[TP_W_COUNT];
  int64_t range_end[TP_W_COUNT];
} tp_rank_shard;

typedef struct tp_plan tp_plan;

/* Builds the plan of one decoder layer. Rule: q heads split evenly; K/V sharded
 * when num_kv_heads >= tp_size (num_kv_heads % tp_size must be 0), replicated
 * on every rank otherwise; q/k/v/gate/up ColumnParallel, o/down RowParallel +
 * AllReduce, q followed by AllGather (the manual's table). On success *out owns
 * a new plan. Errors: TP_ERR_INVALID_ARG (null, non-positive dims),
 * TP_ERR_TP_SIZE_NOT_POW2, TP_ERR_GQA_SHAPE, TP_ERR_NOT_DIVISIBLE. Host only. */
tp_status tp_plan_create(const tp_dims *dims, tp_plan **out);

/* Frees a plan created by tp_plan_create. NULL is accepted. */
tp_status tp_plan_destroy(tp_plan *plan);

/* Copies the dims the plan was built from. */
tp_status tp_plan_dims(const tp_plan *plan, tp_dims *out);

/* Fills *out with rank `rank`'s shard description. TP_ERR_INVALID_ARG for a
 * rank outside [0, tp_size). Host only. */
tp_status tp_plan_query_rank(const tp_plan *plan, int32_t rank, tp_rank_shard *out);

/* Local GQA map of rank `rank`: out[j] = local kv head read by local q head j,
 * j in [0, q_head_end - q_head_begin). `capacity` is the length of `out`;
 * TP_ERR_INVALID_ARG when it is too small. Host only. */
tp_status tp_plan_q_to_kv(const tp_plan *plan, int32_t rank, int32_t *out, int32_t capacity);

/* ---------------------------------------------------------------------------
 * Linear layers (mlxcel manual: Column Parallel / Row Parallel; railscraft
 * wiki 상세 1: Y_i = X W_i with Y = [Y_1..Y_n], and Y_i = X_i W_i with Y = sum Y_i).
 * ------------------------------------------------------------------------- */

/* Column-parallel linear: Y_r = X * W_r^T for r in [0, tp_size), X replicated.
 *  x       : [T x K]. bf16 (tensor cores, fp32 accumulation) or f32 (exact fp32 FMA).
 *  w[r]    : [n_r x K], same dtype as x.
 *  gather=1: y[0] is one [T x sum_r n_r] tensor; shard r is written straight into
 *            columns [sum_{q<r} n_q, ...) (the all-gather is the concatenation
 *            and moves no extra bytes).
 *  gather=0: y[r] is rank r's own [T x n_r] output.
 *  y dtype : f32 or bf16 for bf16 inputs (rounded to nearest even); f32 for f32.
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_CUDA. */
tp_status tp_column_linear(int32_t tp_size, const tp_tensor *x, const tp_tensor *w,
                           tp_tensor *y, int32_t gather, tp_stream_t stream);

typedef enum tp_combine {
  TP_COMBINE_NONE = 0,       /* y[r] = partial P_r (no reduction)                           */
  TP_COMBINE_FUSED = 1,      /* y[0] = sum_r P_r, summed in the tensor-core accumulator over
                                shards 0..N-1 in order; no partial is written              */
  TP_COMBINE_RING = 2,       /* y[r] = P_r, then the ring all-reduce as N-1 reduce-scatter and
                                N-1 all-gather step launches; every y[r] ends equal to the sum */
  TP_COMBINE_RING_FUSED = 3, /* as TP_COMBINE_RING, the partials folded in one pass in the
                                ring's order (bit-identical to TP_COMBINE_RING)            */
  TP_COMBINE_RING_SHARED = 4 /* as TP_COMBINE_RING_FUSED, with the result stored once, in
                                y[0] (bit-identical to it): for ranks that share one output
                                on this device; y[1..N-1] are scratch, unspecified after   */
} tp_combine;
/* With bf16 inputs, RING_FUSED and RING_SHARED fold the ring into the GEMM when
 * every 256-row tile lies inside one ring chunk (T % N == 0, T/N a multiple of
 * 256, more than 128 tokens, an output width n that is a multiple of 4 with
 * y[r].ld == n, N <= 16, and a shape that the
 * GEMM without a combine runs without split-K): each rank's partial is computed
 * exactly as TP_COMBINE_NONE computes it, then added in its chunk's ring order
 * in the epilogue, so no partial is written and no second pass runs. The bits
 * are those of the GEMM followed by the one-pass ring. Other shapes run the GEMM
 * and then the one-pass ring. The environment variable TPGQA_RING_EPILOGUE=0
 * (read on every call) turns the fold off. */

/* Row-parallel linear: P_r = X_r * W_r^T, then the combine above.
 *  x[r] : [T x k_r] (rank r's slice of the input features), bf16 or f32.
 *  w[r] : [n x k_r] (rank r's block of stored columns), same dtype as x[r].
 *  y    : f32; y[0] alone for TP_COMBINE_FUSED, y[0..N-1] otherwise, each [T x n].
 * The partials are the f32 accumulators. f32 inputs support NONE, RING and
 * RING_FUSED. Errors: as tp_column_linear. */
tp_status tp_row_linear(int32_t tp_size, const tp_tensor *x, const tp_tensor *w,
                        tp_tensor *y, int32_t combine, tp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Ring collectives (mlxcel manual, 통신 패턴 / Communication patterns).
 * buf[r] is rank r's f32 buffer; all N have the same rows x cols and are viewed
 * flat in row-major order (S elements). Chunk c is the flat element range
 * [floor(c*S/N), floor((c+1)*S/N)). Reduce-scatter step s: rank r sends chunk
 * (r-1-s) mod N to rank (r+1) % N, which adds it to its copy; after N-1 steps
 * rank r holds the reduced chunk r, summed in the order c+1, c+2, ..., c.
 * All-gather step s: rank r sends chunk (r-s) mod N to (r+1) % N, which
 * overwrites its copy. Buffers must be contiguous (ld == cols) and 16-byte
 * aligned.
 * ------------------------------------------------------------------------- */
typedef enum tp_ring_mode {
  TP_RING_STEPS = 0, /* one launch per ring step, N-1 per phase                       */
  TP_RING_FUSED = 1, /* one launch per phase; same fold order, bit-identical results   */
  TP_RING_FUSED_SHARED = 2 /* tp_allreduce_ring only: one pass, the sum written to buf[0]
                              alone (the N equal results stored once); buf[1..N-1] keep
                              their partials                                            */
} tp_ring_mode;

/* In-place reduce-scatter; afterwards chunk r of buf[r] is reduced. The other
 * chunks of every buffer are unspecified afterwards (the step mode leaves
 * intermediate sums there, the fused mode the original partials). */
tp_status tp_reduce_scatter(int32_t tp_size, tp_tensor *buf, int32_t mode, tp_stream_t stream);

/* In-place ring all-gather: on entry chunk r of buf[r] is rank r's chunk; on
 * return every buffer holds every chunk. */
tp_status tp_ring_all_gather(int32_t tp_size, tp_tensor *buf, int32_t mode, tp_stream_t stream);

/* In-place all-reduce = reduce-scatter + all-gather; every buf[r] ends equal. */
tp_status tp_allreduce_ring(int32_t tp_size, tp_tensor *buf, int32_t mode, tp_stream_t stream);

/* Concatenating all-gather of separate shards (all-gather as concatenation).
 *  shard[r] : [rows_r x cols_r], one dtype for all, f32 or bf16.
 *  axis = 1 : columns; every shard has the same rows, out is [rows x sum cols_r].
 *  axis = 0 : rows; every shard has the same cols, out is [sum rows_r x cols].
 *  out[0..n_out-1]: n_out = 1 (one copy shared by all ranks) or tp_size (a copy
 *  per rank). */
tp_status tp_all_gather(int32_t tp_size, const tp_tensor *shard, tp_tensor *out, int32_t n_out,
                        int32_t axis, tp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Row-parallel -> column-parallel pipeline without the all-gather (mlxcel
 * manual, 통신 패턴 / Communication patterns, Reduce-scatter: used when the
 * result of a row-parallel op goes straight into a column-parallel op; the
 * all-gather step is avoided).
 * ------------------------------------------------------------------------- */

/* One-pass ring reduce-scatter of f32 partials into bf16 chunks.
 *  partial[r] : rank r's f32 [T x n] partial, contiguous (ld == cols), 16-byte
 *               aligned; read only.
 *  out[r]     : rank r's bf16 [T x n] buffer (any ld, a multiple of 8); only
 *               chunk r (flat range [floor(r*S/N), floor((r+1)*S/N)) of the
 *               row-major [T x n] view) is written, with the sum of chunk r
 *               over the ranks in the ring's order r+1, r+2, ..., r, in f32,
 *               rounded once to bf16 (nearest even). The rest of out[r] is
 *               left as it was.
 * The f32 sums are bit-identical to tp_reduce_scatter's. bf16 is the operand
 * type of the column-parallel GEMM that reads the chunks next.
 * Errors: TP_ERR_INVALID_ARG (sizes differ, N not a power of two), TP_ERR_DTYPE,
 * TP_ERR_ALIGNMENT, TP_ERR_RANK_FAILED, TP_ERR_CUDA. */
tp_status tp_reduce_scatter_bf16(int32_t tp_size, const tp_tensor *partial, tp_tensor *out,
                                 tp_stream_t stream);

/* Column-parallel linear whose input is the N reduced chunks where they lie:
 * rank c's buffer holds rows [c*T/N, (c+1)*T/N) of X (chunk c of a reduce-
 * scatter), and the GEMM reads each block of rows from its chunk's buffer, so
 * no all-gather runs. Y_r = X * W_r^T as in tp_column_linear.
 *  x_chunks[c] : bf16 [T x K] buffer of rank c; rows [c*T/N, (c+1)*T/N) are
 *                read, the rest is ignored. T must be a multiple of N (chunk
 *                boundaries on rows), else TP_ERR_NOT_DIVISIBLE.
 *  w[r], y, gather : as tp_column_linear (bf16 weights).
 * Results are bit-identical to tp_column_linear on the assembled X.
 * Errors: as tp_column_linear, plus TP_ERR_NOT_DIVISIBLE. */
tp_status tp_column_linear_chunks(int32_t tp_size, const tp_tensor *x_chunks, const tp_tensor *w,
                                  tp_tensor *y, int32_t gather, tp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Vocab parallel (mlxcel manual, 가중치 샤딩 전략 / Weight-sharding strategies,
 * Vocab Parallel: the vocabulary dimension of the embedding table and of the
 * LM head is split into contiguous per-rank slices; 임베딩 및 LM Head 샤딩 /
 * Embedding and LM-head sharding, vocab_parallel: the lookup and the logits
 * need an all-gather).
 * ------------------------------------------------------------------------- */

/* Embedding lookup over a vocab-sharded table, with the all-gather of the rows
 * looked up: row i of every output is row ids[i] of the full table [V x D],
 * V = tp_size * table[0].rows. Rank r holds ids [r*V/N, (r+1)*V/N) as table[r]
 * (id at local row id - r*V/N). Each token's row is read once, from the rank
 * owning its id, and written to every output.
 *  ids      : device pointer to n_tokens int32 token ids (n_tokens >= 0).
 *  table[r] : [V/N x D] f32 or bf16; every shard has the same shape and dtype.
 *  out[o]   : [n_tokens x D] in the table's dtype; n_out = 1 (one copy shared
 *             by all ranks) or tp_size (a copy per rank).
 * An id outside [0, V) is not looked up: its rows are written as zeros and the
 * device status word records it (tp_device_status then returns
 * TP_ERR_BAD_TOKEN). 16-byte aligned bases, pitches and rows take a vector
 * path; anything else is copied element by element. Bases must be aligned to
 * the element size and ids to 4 bytes, else TP_ERR_ALIGNMENT.
 * Errors: TP_ERR_INVALID_ARG (null, shapes differ, n_out), TP_ERR_TP_SIZE_NOT_POW2,
 * TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_RANK_FAILED, TP_ERR_CUDA. */
tp_status tp_vocab_embedding(int32_t tp_size, const int32_t *ids, int64_t n_tokens,
                             const tp_tensor *table, tp_tensor *out, int32_t n_out,
                             tp_stream_t stream);

/* LM-head logits over a vocab-sharded weight, with their all-gather: rank r's
 * logits are X W_r^T for its vocabulary slice W_r = rows [r*V/N, (r+1)*V/N) of
 * the LM-head weight [V x D]. gather = 1 writes them as column blocks, in rank
 * order, of one [T x V] logits tensor (the all-gather as concatenation, no
 * copy); gather = 0 leaves logits[r] = [T x V/N] per rank.
 *  x      : [T x D] bf16 (f32 with f32 weights, as tp_column_linear).
 *  w[r]   : [V/N x D]; every shard has the same number of rows.
 *  logits : f32 or bf16 (f32 for f32 inputs).
 * Errors: as tp_column_linear; TP_ERR_INVALID_ARG when the shards differ in rows. */
tp_status tp_vocab_lm_head(int32_t tp_size, const tp_tensor *x, const tp_tensor *w,
                           tp_tensor *logits, int32_t gather, tp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Attention core between q/k/v and o_proj (mlxcel manual, GQA 인식 어텐션 샤딩 /
 * GQA-aware attention sharding: each rank's q heads attend with the kv heads
 * the plan gives it, its own when K/V are sharded, all of them when replicated).
 * ------------------------------------------------------------------------- */

/* Workspace bytes tp_attn_core needs for `tokens` tokens (the transposed V of
 * every kv source, bf16). 0 for a null plan or negative tokens. */
size_t tp_attn_core_workspace_size(const tp_plan *plan, int64_t tokens);

/* A_r = per local q head h of rank r: softmax(Q_h K_g^T / sqrt(d)) V_g with g
 * the plan's q->kv map (tp_plan_q_to_kv), query i seeing keys j <= i when
 * causal = 1, every key when causal = 0. No position encoding is applied.
 * S and the running output are f32 (tensor cores, TMEM); P is rounded to bf16
 * for the P V product; A is written as bf16.
 *  q[r]  : [T x Hq_r*d] bf16 (tp_qkv_proj's q output of rank r).
 *  k[r], v[r] : [T x Hkv_r*d] bf16; one shared entry (k[0], v[0], all kv heads)
 *          when the plan replicates K/V, else one per rank.
 *  a[r]  : [T x Hq_r*d] bf16 output, rank r's slice of the o_proj input.
 *  workspace : at least tp_attn_core_workspace_size bytes, 16-byte aligned.
 * d must be 128 and tp_size at most 32, with at most 256 q heads in all,
 * else TP_ERR_UNSUPPORTED.
 * The kernel is chosen on every call by the environment variable TPGQA_ATTN:
 * unset (or any other value), two 128-query tiles per CTA; 1, one tile per
 * CTA; 3, two tiles over 64-key blocks; 4, a 256-query tile on an SM pair. All
 * compute the same result within rounding (P and A are rounded to bf16).
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_WORKSPACE,
 * TP_ERR_UNSUPPORTED, TP_ERR_RANK_FAILED, TP_ERR_CUDA. */
tp_status tp_attn_core(const tp_plan *plan, const tp_tensor *q, const tp_tensor *k, const tp_tensor *v,
                       tp_tensor *a, int32_t causal, void *workspace, size_t workspace_bytes,
                       tp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Mixture of experts (mlxcel manual, MoE 전문가 병렬화 / MoE expert parallelism:
 * Expert Parallel puts expert i whole on rank i % tp_size, with no
 * communication inside an expert; Within-Expert Parallel shards every expert's
 * FFN over all ranks with the dense FFN's column-parallel gate/up and
 * row-parallel down projections).
 * ------------------------------------------------------------------------- */
typedef enum tp_moe_mode {
  TP_MOE_EXPERT_PARALLEL = 0,
  TP_MOE_WITHIN_EXPERT = 1
} tp_moe_mode;

typedef struct tp_moe_dims {
  int32_t tp_size;      /* N, a power of two                                       */
  int32_t mode;         /* tp_moe_mode                                             */
  int32_t num_experts;  /* E, 1..256; a multiple of N for expert parallel          */
  int32_t top_k;        /* k routing slots per token, >= 1                         */
  int64_t hidden;       /* D, a multiple of 8                                      */
  int64_t ffn;          /* F per expert; F/N a multiple of 8 for within-expert      */
} tp_moe_dims;

/* Workspace bytes tp_moe_block needs for `tokens` tokens: the routed layout of
 * T*k rows (each expert's rows padded to whole GEMM tiles), the gathered
 * inputs, H and the f32 down-projection rows of every rank. 0 for bad dims. */
size_t tp_moe_workspace_size(const tp_moe_dims *dims, int64_t tokens);

/* MoE block: Y = sum_r Y_r, where rank r's partial output is, per token t, the
 * sum over its slots j (in slot order) of topk_w[t,j] times the FFN (SwiGLU,
 * silu(X G^T) * (X U^T) then D^T, H rounded to bf16) of expert topk_ids[t,j]
 * restricted to what rank r holds of it:
 *  - expert parallel: the whole expert when expert % N == r, else nothing;
 *  - within-expert: rows [r*F/N, (r+1)*F/N) of its gate and up weights and the
 *    same columns of its down weight.
 * The routing is an input (the router runs on every rank, so all ranks share
 * it); the block routes, gathers, runs the expert GEMMs and combines on the
 * device, with no host synchronisation.
 *  x         : [T x D] bf16.
 *  topk_ids  : device int32 [T x k], row-major. An id outside [0, E) drops that
 *              slot and is reported by tp_device_status as TP_ERR_BAD_TOKEN.
 *  topk_w    : device f32 [T x k], row-major.
 *  w_gate[r], w_up[r] : rank r's expert weights stacked by slot, bf16:
 *              within-expert [E*F/N x D], expert e's slice at rows [e*F/N, ...);
 *              expert parallel [(E/N)*F x D], slot s = expert r + s*N at rows [s*F, ...).
 *  w_down[r] : within-expert [E*D x F/N], expert e at rows [e*D, (e+1)*D);
 *              expert parallel [(E/N)*D x F], slot s at rows [s*D, (s+1)*D).
 *  y         : f32 [T x D]; y[0] for TP_COMBINE_FUSED (the sum over ranks),
 *              y[0..N-1] otherwise (TP_COMBINE_NONE leaves the partials, RING
 *              and RING_FUSED all-reduce them on the ring).
 *  workspace : device memory of at least tp_moe_workspace_size bytes, 256-byte
 *              aligned; its contents on entry do not matter.
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_TP_SIZE_NOT_POW2, TP_ERR_NOT_DIVISIBLE,
 * TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_WORKSPACE, TP_ERR_RANK_FAILED, TP_ERR_CUDA. */
tp_status tp_moe_block(const tp_moe_dims *dims, const tp_tensor *x, const int32_t *topk_ids,
                       const float *topk_w, const tp_tensor *w_gate, const tp_tensor *w_up,
                       const tp_tensor *w_down, tp_tensor *y, int32_t combine, void *workspace,
                       size_t workspace_bytes, tp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Blocks (mlxcel manual, 아키텍처 인식 샤드 플랜: gate/up ColumnParallel with no
 * communication, down RowParallel + AllReduce; q/k/v ColumnParallel, o
 * RowParallel + AllReduce).
 * ------------------------------------------------------------------------- */

/* Workspace bytes tp_mlp_block needs for `tokens` tokens (H_r of every rank,
 * bf16, T x F in total). */
size_t tp_mlp_block_workspace_size(const tp_plan *plan, int64_t tokens);

/* Column-parallel gate/up projection of the MLP with SwiGLU fused into the
 * GEMM epilogue: H_r = silu(X G_r^T) * (X U_r^T), rounded to bf16, for every
 * rank in one launch (the first half of tp_mlp_block; the manual's table lists
 * no communication after gate/up).
 *  x         : [T x D] bf16.
 *  w_gate[r] : [F/N x D] bf16; w_up[r] likewise.
 *  h[r]      : [T x F/N] bf16 output of rank r.
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_RANK_FAILED,
 * TP_ERR_CUDA. */
tp_status tp_gate_up_swiglu(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_gate,
                            const tp_tensor *w_up, tp_tensor *h, tp_stream_t stream);

/* MLP block: H_r = silu(X G_r^T) * (X U_r^T) (SwiGLU fused into the gate/up
 * GEMM's epilogue, H_r rounded to bf16), then Y = sum_r H_r D_r^T.
 *  x         : [T x D] bf16.
 *  w_gate[r] : [F/N x D] bf16; w_up[r] likewise (rows plan.range(GATE/UP) of G, U).
 *  w_down[r] : [D x F/N] bf16 (columns plan.range(DOWN) of Down [D x F]).
 *  y         : f32 [T x D]; y[0] for TP_COMBINE_FUSED, y[0..N-1] otherwise
 *              (TP_COMBINE_NONE leaves the partials).
 *  workspace : device memory of at least tp_mlp_block_workspace_size bytes,
 *              16-byte aligned; its contents on entry do not matter.
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_WORKSPACE,
 * TP_ERR_RANK_FAILED, TP_ERR_CUDA. */
tp_status tp_mlp_block(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_gate,
                       const tp_tensor *w_up, const tp_tensor *w_down, tp_tensor *y,
                       int32_t combine, void *workspace, size_t workspace_bytes,
                       tp_stream_t stream);

/* tp_mlp_block without a caller-provided workspace. The pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory: for example a plug-in inside a framework that owns all device
 * memory through its own allocator and lends none of it, or a serving process
 * that reserved all free HBM at start-up and must not call cudaMalloc (which
 * can fail, or stall other streams) while requests are in flight.
 *
 * It computes exactly what tp_mlp_block computes, with the same arguments
 * except the workspace: H (tokens x ffn bf16 values) is kept in one fixed
 * scratch array inside the library, tp_mlp_block_static_max_bytes() = 16 MiB
 * long. Every GPU that loads the library reserves that array when the library's
 * device code is loaded and keeps it until the process exits.
 *  - Size limit: x->rows * ffn * 2 bytes must not exceed the maximum, else
 *    TP_ERR_WORKSPACE is returned and nothing is enqueued.
 *  - Allocation: the call allocates nothing (no cudaMalloc / cudaFree, no
 *    allocating library routine).
 *  - Set-up: the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make that
 *    first call before any stream capture. The cached address belongs to the
 *    device's context at that time: do not use the library across a
 *    cudaDeviceReset of that device (see tp_device_status).
 *  - Sharing: every call on a device uses the same array, which keeps the last
 *    call's H. Each call overwrites H in full before reading it, so nothing has
 *    to be cleared; but calls that can overlap on the GPU (different streams
 *    without ordering between them) race on the array and give wrong results.
 * The caller still passes and owns x, the weights and y. Other errors: as
 * tp_mlp_block. */
tp_status tp_mlp_block_static(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_gate,
                              const tp_tensor *w_up, const tp_tensor *w_down, tp_tensor *y,
                              int32_t combine, tp_stream_t stream);

/* Size in bytes of tp_mlp_block_static's fixed scratch array (16 MiB). */
size_t tp_mlp_block_static_max_bytes(void);

/* Column-parallel q/k/v projections with the GQA rule, as one grouped launch
 * (the first half of tp_attn_proj; the manual's table puts q/k/v in
 * ColumnParallel, with K/V replicated when num_kv_heads < tp_size).
 *  x        : [T x D] bf16.
 *  w_q[r]   : [(q heads of r) * hd x D] bf16;  q[r]: [T x same] bf16 out.
 *  w_k, w_v : N tensors when sharded, ONE shared tensor when replicated (computed
 *             once); k, v outputs likewise (bf16).
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_RANK_FAILED,
 * TP_ERR_CUDA. */
tp_status tp_qkv_proj(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_q,
                      const tp_tensor *w_k, const tp_tensor *w_v, tp_tensor *q, tp_tensor *k,
                      tp_tensor *v, tp_stream_t stream);

/* Attention projections with GQA sharding.
 *  x        : [T x D] bf16.
 *  w_q[r]   : [(q heads of r) * hd x D] bf16;  q[r]: [T x same] bf16 out.
 *  w_k, w_v : sharded -> N tensors [(kv heads of r) * hd x D];
 *             replicated -> ONE tensor [Hkv * hd x D] shared by every rank (it is
 *             computed once); k, v outputs likewise (N or 1 tensors, bf16).
 *  a[r]     : [T x (q heads of r) * hd] bf16, rank r's slice of the attention
 *             context that feeds o_proj (attention itself is not part of this call).
 *  w_o[r]   : [D x (q heads of r) * hd] bf16 (columns plan.range(O) of Wo).
 *  y        : f32 [T x D]; y[0] for TP_COMBINE_FUSED, y[0..N-1] otherwise.
 * Ordering: the call's results are complete for every kernel enqueued after it
 * on the stream. At decode sizes (T <= 128) o_proj runs on the device beside
 * the q/k/v GEMM, when a and y share no byte with q, k, v (nor y with x and the
 * q/k/v weights); overlapping buffers are allowed and run the two in order.
 * Errors: as tp_mlp_block (no workspace). */
tp_status tp_attn_proj(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_q,
                       const tp_tensor *w_k, const tp_tensor *w_v, tp_tensor *q, tp_tensor *k,
                       tp_tensor *v, const tp_tensor *a, const tp_tensor *w_o, tp_tensor *y,
                       int32_t combine, tp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Status, health and diagnostics.
 * ------------------------------------------------------------------------- */

/* Static string naming a status. */
const char *tp_status_str(tp_status s);

/* cudaError_t of the last failed CUDA runtime call made by this library in the
 * calling thread (0 if none). */
int32_t tp_last_cuda_error(void);

/* Marks logical rank `rank` healthy (1) or failed (0), process-wide. While any
 * rank that a call involves is failed, the call returns TP_ERR_RANK_FAILED
 * before enqueuing anything, so the whole TP group stops together (mlxcel
 * manual, TP 실행기 / TP executor: health reporting and error propagation). */
tp_status tp_set_rank_health(int32_t rank, int32_t healthy);

/* Synchronises `stream`, then reads and clears the device status word that
 * kernels set when a bounded wait runs out or an embedding lookup meets a bad
 * token id (the first such event is kept). Returns TP_OK, TP_ERR_TIMEOUT,
 * TP_ERR_BAD_TOKEN or TP_ERR_CUDA. *detail (optional) receives the raw word
 * (0 = none).
 * The library looks up the device addresses of its own device variables (this
 * status word, the scratch array of tp_mlp_block_static) once per device and
 * keeps them for the life of the process. A cudaDeviceReset destroys the
 * context they belong to, so the library must not be used on a device after
 * that device has been reset. */
tp_status tp_device_status(tp_stream_t stream, int32_t *detail);

/* Sets the time budget, in nanoseconds, of every bounded device-side wait of
 * kernels enqueued afterwards (0 restores the default of 2 s). Process-wide;
 * meant for tests of the timeout path. */
tp_status tp_set_wait_budget(int64_t nanoseconds);

/* Enqueues one kernel whose bounded wait is on an mbarrier that no thread
 * completes, so it always runs out; the kernel records TP_ERR_TIMEOUT in the
 * device status word and returns. Used to test the timeout path without a
 * GPU fault or hang. */
tp_status tp_debug_wait_timeout(tp_stream_t stream);

/* Kernel launches this library has enqueued in this process so far, on every
 * stream and device (each successful kernel launch of every call counts one;
 * memsets and copies do not count). A caller reads it before and after a region
 * of work to count that region's launches. Never fails. */
uint64_t tp_launch_count(void);

/* Library version string. */
const char *tp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TPGQA_H */
