// Vocab-parallel embedding lookup (mlxcel manual "텐서 병렬화", 가중치 샤딩 전략 /
// Weight-sharding strategies, Vocab Parallel: the vocabulary dimension of the
// embedding table is split into contiguous per-rank slices; 임베딩 및 LM Head
// 샤딩 / Embedding and LM-head sharding, vocab_parallel: the lookup needs an
// all-gather).
//
// All ranks' shards live in this GPU's memory, so the lookup and its all-gather
// are one kernel: token i's row is read once, from the shard of the rank whose
// slice holds its id (local row id - r*V/N), and stored to every output copy.
// One CTA handles one token row at a time (grid-stride over tokens); its threads
// move the row in 16-byte units, four loads in flight per thread before the
// stores, or in element units when an address or pitch is not 16-byte aligned.
// The copy is dtype-agnostic (bytes), so f32 and bf16 tables take the same path.
#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

tp_status launch_checked(cudaError_t e) {
  if (e != cudaSuccess) return cuda_fail(e);
  const cudaError_t l = cudaGetLastError();
  return l == cudaSuccess ? TP_OK : cuda_fail(l);
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_vocab_embed(EmbedArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const long long vocab = a.rows_per_rank * a.n;
  for (long long i = blockIdx.x; i < a.n_tokens; i += gridDim.x) {
    const long long id = __ldg(a.ids + i);
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0) atomicCAS(a.status, 0, kDevBadToken);
    const int r = ok ? static_cast<int>(id / a.rows_per_rank) : 0;
    const char *src = a.tab[r] + (ok ? id - r * a.rows_per_rank : 0) * a.tab_pitch[r];
    if constexpr (VEC) {
      const long long nv = a.row_bytes >> 4;
      const uint4 zero = make_uint4(0, 0, 0, 0);
      long long v = threadIdx.x;
      for (; v + 3 * kThreads < nv; v += 4 * kThreads) {
        uint4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          x[u] = ok ? __ldg(reinterpret_cast<const uint4 *>(src) + v + u * kThreads) : zero;
        for (int o = 0; o < a.n_outs; ++o) {
          uint4 *dst = reinterpret_cast<uint4 *>(a.out[o] + i * a.out_pitch[o]);
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[v + u * kThreads] = x[u];
        }
      }
      for (; v < nv; v += kThreads) {
        const uint4 x = ok ? __ldg(reinterpret_cast<const uint4 *>(src) + v) : zero;
        for (int o = 0; o < a.n_outs; ++o) reinterpret_cast<uint4 *>(a.out[o] + i * a.out_pitch[o])[v] = x;
      }
    } else if (a.esize == 4) {
      const long long ne = a.row_bytes >> 2;
      for (long long e = threadIdx.x; e < ne; e += kThreads) {
        const unsigned int x = ok ? __ldg(reinterpret_cast<const unsigned int *>(src) + e) : 0u;
        for (int o = 0; o < a.n_outs; ++o)
          reinterpret_cast<unsigned int *>(a.out[o] + i * a.out_pitch[o])[e] = x;
      }
    } else {
      const long long ne = a.row_bytes >> 1;
      for (long long e = threadIdx.x; e < ne; e += kThreads) {
        const unsigned short x = ok ? __ldg(reinterpret_cast<const unsigned short *>(src) + e) : 0;
        for (int o = 0; o < a.n_outs; ++o)
          reinterpret_cast<unsigned short *>(a.out[o] + i * a.out_pitch[o])[e] = x;
      }
    }
  }
}

}  // namespace

tp_status launch_vocab_embed(const EmbedArgs &args, bool vec16, cudaStream_t s) {
  if (args.n_tokens == 0 || args.row_bytes == 0) return TP_OK;
  DevCtx ctx;
  const cudaError_t e = get_dev_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e);
  EmbedArgs a = args;
  a.status = ctx.status;
  // Enough CTAs for every SM's thread slots (8 x 256); each loops over tokens.
  long long grid = static_cast<long long>(num_sms()) * 8;
  if (grid > a.n_tokens) grid = a.n_tokens;
  void (*k)(EmbedArgs) = vec16 ? k_vocab_embed<true> : k_vocab_embed<false>;
  return launch_checked(launch_kernel(k, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s, 1, a));
}

}  // namespace tpgqa
