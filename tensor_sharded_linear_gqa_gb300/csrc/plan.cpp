// Shard plan of one decoder layer (mlxcel manual "텐서 병렬화":
//  - 설정 / Configuration: --tp-size is a power of two, default 1;
//  - 가중치 샤딩 전략 / Weight-sharding strategies: Column Parallel gives rank r
//    output features [r*D_out/N, (r+1)*D_out/N), Row Parallel input features
//    [r*D_in/N, (r+1)*D_in/N), Replicated a full copy;
//  - 아키텍처 인식 샤드 플랜 / Architecture-aware shard plan: q/k/v/gate/up
//    ColumnParallel, o/down RowParallel followed by AllReduce, q followed by
//    AllGather; GQA rule: K/V sharded when num_kv_heads >= tp_size, replicated
//    on every rank when num_kv_heads < tp_size).
// Host-only C++; no CUDA calls.
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "tpgqa.h"

struct tp_plan {
  tp_dims dims;
  std::vector<tp_rank_shard> ranks;
  std::vector<std::vector<int32_t>> q_to_kv;
};

namespace {

bool is_pow2(int32_t n) { return n >= 1 && (n & (n - 1)) == 0; }

}  // namespace

extern "C" tp_status tp_plan_create(const tp_dims *dims, tp_plan **out) {
  if (!dims || !out) return TP_ERR_INVALID_ARG;
  *out = nullptr;
  const tp_dims d = *dims;
  if (!is_pow2(d.tp_size)) return TP_ERR_TP_SIZE_NOT_POW2;
  if (d.hidden < 1 || d.num_q_heads < 1 || d.num_kv_heads < 1 || d.head_dim < 1 || d.ffn < 1)
    return TP_ERR_INVALID_ARG;
  const int32_t N = d.tp_size;
  // A query group (q heads sharing one kv head) must be whole.
  if (d.num_q_heads % d.num_kv_heads != 0) return TP_ERR_GQA_SHAPE;
  if (d.num_q_heads % N != 0) return TP_ERR_GQA_SHAPE;
  const bool replicate_kv = d.num_kv_heads < N;
  if (!replicate_kv && d.num_kv_heads % N != 0) return TP_ERR_GQA_SHAPE;
  if (d.ffn % N != 0) return TP_ERR_NOT_DIVISIBLE;

  tp_plan *p = new (std::nothrow) tp_plan;
  if (!p) return TP_ERR_INVALID_ARG;
  p->dims = d;
  p->ranks.resize(N);
  p->q_to_kv.resize(N);
  const int32_t q_per_rank = d.num_q_heads / N;
  const int32_t group = d.num_q_heads / d.num_kv_heads;
  const int64_t hd = d.head_dim;
  const int64_t f_per_rank = d.ffn / N;
  for (int32_t r = 0; r < N; ++r) {
    tp_rank_shard &s = p->ranks[r];
    std::memset(&s, 0, sizeof(s));
    s.rank = r;
    s.q_head_begin = r * q_per_rank;
    s.q_head_end = (r + 1) * q_per_rank;
    if (replicate_kv) {
      s.kv_head_begin = 0;
      s.kv_head_end = d.num_kv_heads;
      s.kv_replicated = 1;
    } else {
      const int32_t kv_per_rank = d.num_kv_heads / N;
      s.kv_head_begin = r * kv_per_rank;
      s.kv_head_end = (r + 1) * kv_per_rank;
      s.kv_replicated = 0;
    }
    const int32_t kv_strategy = replicate_kv ? TP_SHARD_REPLICATED : TP_SHARD_COLUMN;
    s.strategy[TP_W_Q] = TP_SHARD_COLUMN;
    s.strategy[TP_W_K] = kv_strategy;
    s.strategy[TP_W_V] = kv_strategy;
    s.strategy[TP_W_O] = TP_SHARD_ROW;
    s.strategy[TP_W_GATE] = TP_SHARD_COLUMN;
    s.strategy[TP_W_UP] = TP_SHARD_COLUMN;
    s.strategy[TP_W_DOWN] = TP_SHARD_ROW;
    s.comm[TP_W_Q] = TP_COMM_ALL_GATHER;
    s.comm[TP_W_K] = TP_COMM_NONE;
    s.comm[TP_W_V] = TP_COMM_NONE;
    s.comm[TP_W_O] = TP_COMM_ALL_REDUCE;
    s.comm[TP_W_GATE] = TP_COMM_NONE;
    s.comm[TP_W_UP] = TP_COMM_NONE;
    s.comm[TP_W_DOWN] = TP_COMM_ALL_REDUCE;
    s.range_begin[TP_W_Q] = s.q_head_begin * hd;
    s.range_end[TP_W_Q] = s.q_head_end * hd;
    s.range_begin[TP_W_K] = s.range_begin[TP_W_V] = s.kv_head_begin * hd;
    s.range_end[TP_W_K] = s.range_end[TP_W_V] = s.kv_head_end * hd;
    // o_proj's input features are the attention heads this rank computes.
    s.range_begin[TP_W_O] = s.q_head_begin * hd;
    s.range_end[TP_W_O] = s.q_head_end * hd;
    s.range_begin[TP_W_GATE] = s.range_begin[TP_W_UP] = s.range_begin[TP_W_DOWN] = r * f_per_rank;
    s.range_end[TP_W_GATE] = s.range_end[TP_W_UP] = s.range_end[TP_W_DOWN] = (r + 1) * f_per_rank;
    std::vector<int32_t> &m = p->q_to_kv[r];
    m.resize(q_per_rank);
    for (int32_t j = 0; j < q_per_rank; ++j) {
      const int32_t global_q = s.q_head_begin + j;
      const int32_t global_kv = global_q / group;  // q heads [g*group, (g+1)*group) read kv head g
      m[j] = global_kv - s.kv_head_begin;
    }
  }
  *out = p;
  return TP_OK;
}

extern "C" tp_status tp_plan_destroy(tp_plan *plan) {
  delete plan;
  return TP_OK;
}

extern "C" tp_status tp_plan_dims(const tp_plan *plan, tp_dims *out) {
  if (!plan || !out) return TP_ERR_INVALID_ARG;
  *out = plan->dims;
  return TP_OK;
}

extern "C" tp_status tp_plan_query_rank(const tp_plan *plan, int32_t rank, tp_rank_shard *out) {
  if (!plan || !out) return TP_ERR_INVALID_ARG;
  if (rank < 0 || rank >= plan->dims.tp_size) return TP_ERR_INVALID_ARG;
  *out = plan->ranks[rank];
  return TP_OK;
}

extern "C" tp_status tp_plan_q_to_kv(const tp_plan *plan, int32_t rank, int32_t *out,
                                     int32_t capacity) {
  if (!plan || !out) return TP_ERR_INVALID_ARG;
  if (rank < 0 || rank >= plan->dims.tp_size) return TP_ERR_INVALID_ARG;
  const std::vector<int32_t> &m = plan->q_to_kv[rank];
  if (capacity < static_cast<int32_t>(m.size())) return TP_ERR_INVALID_ARG;
  for (size_t j = 0; j < m.size(); ++j) out[j] = m[j];
  return TP_OK;
}
