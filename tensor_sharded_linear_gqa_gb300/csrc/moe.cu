// Mixture-of-experts block over N logical ranks in this GPU's memory (mlxcel
// manual "텐서 병렬화", MoE 전문가 병렬화 / MoE expert parallelism):
//  - expert parallel: expert i lives whole on rank i % N;
//  - within-expert parallel: every expert's FFN is sharded over all ranks like
//    the dense FFN (gate/up column-parallel, down row-parallel).
// The routing (top-k expert ids and weights per token) is an input.
//
// Steps, all on the device:
//  1. k_moe_route sorts the T*k (token, slot) assignments by expert, stably, into
//     a row layout where each expert's rows start on a tile boundary (BM rows:
//     256 for the SM-pair GEMM, 128 for the single-CTA one). It writes each
//     assignment's row (pos), each row's assignment (inv, -1 for padding) and a
//     block table with one entry per tile of rows: the expert's weight slot and
//     map offset, or -1 past the last expert.
//  2. k_moe_gather copies token rows of X into that layout (zeros in padding).
//  3. The gate/up GEMM with the SwiGLU epilogue and the down GEMM run on the
//     persistent tcgen05 kernels; the block table picks each tile's expert
//     weights and skips the tiles past the last expert. Within-expert: one
//     problem per rank over all tiles, with that rank's slice of every expert
//     (or, for the fused combine, one down problem whose K segments are the
//     ranks, summed in the accumulator). Expert parallel: one problem over all
//     tiles, each tile taking the weights of the rank its expert lives on (every
//     tile belongs to exactly one rank).
//  4. k_moe_combine gives rank r's partial output: per token, the sum over its
//     slots in slot order of weight * the slot's down-projection row, for the
//     slots rank r ran. The caller's ring all-reduce then combines the ranks;
//     for the one-pass ring (every rank's output, or the shared one) the same
//     kernel folds the ranks' partials in the ring's order instead (mlxcel
//     manual "텐서 병렬화", 통신 패턴: chunk c of the flat output reduced as
//     x_{c+1} + ... + x_c), so the partials are never written.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
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

struct RouteArgs {
  const int *ids;       // [A] expert of each assignment (token-major, slot-minor)
  int *pos;             // [A] row of each assignment, -1 for a bad expert id
  int *inv;             // [rows] assignment of each row, -1 for padding
  int *blk;             // [nblk] block table
  long long assignments, rows;
  int nblk, bm, experts, n, mode;
  int *status;
};

// One CTA. Warp w owns the contiguous assignments [w*chunk, (w+1)*chunk): pass 1
// counts them per expert, the per-warp counts are turned into starting rows
// (expert by expert, warps in order), and pass 2 places every assignment at
// its expert's next row in order, so the layout is the stable sort by expert.
__global__ void __launch_bounds__(kRouteThreads) k_moe_route(RouteArgs a) {
  __shared__ int cnt[kRouteWarps][kMaxExperts];
  __shared__ int off[kMaxExperts + 1];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.experts;
  for (int i = tid; i < kRouteWarps * kMaxExperts; i += kRouteThreads) (&cnt[0][0])[i] = 0;
  __syncthreads();
  const long long chunk = ((a.assignments + kRouteWarps - 1) / kRouteWarps + 31) / 32 * 32;
  const long long lo = static_cast<long long>(warp) * chunk;
  const long long hi = lo + chunk < a.assignments ? lo + chunk : a.assignments;
  for (long long i = lo + lane; i < hi; i += 32) {
    const int e = __ldg(a.ids + i);
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[warp][e], 1);
    } else {
      a.pos[i] = -1;
      atomicCAS(a.status, 0, kDevBadToken);
    }
  }
  __syncthreads();
  // expert totals, padded to whole tiles, and their prefix (one warp, 8 experts a lane)
  if (warp == 0) {
    int local[kMaxExperts / 32];
    int sum = 0;
#pragma unroll
    for (int q = 0; q < kMaxExperts / 32; ++q) {
      const int e = lane * (kMaxExperts / 32) + q;
      int tot = 0;
      if (e < E)
        for (int w = 0; w < kRouteWarps; ++w) tot += cnt[w][e];
      local[q] = (tot + a.bm - 1) / a.bm * a.bm;
      sum += local[q];
    }
    int incl = sum;
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int q = 0; q < kMaxExperts / 32; ++q) {
      off[lane * (kMaxExperts / 32) + q] = run;
      run += local[q];
    }
    if (lane == 31) off[kMaxExperts] = run;
  }
  __syncthreads();
  // starting row of every (warp, expert) run
  if (tid < E) {
    int run = off[tid];
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = cnt[w][tid];
      cnt[w][tid] = run;
      run += c;
    }
  }
  for (long long r = tid; r < a.rows; r += kRouteThreads) a.inv[r] = -1;
  const int used = off[E];
  for (int b = tid; b < a.nblk; b += kRouteThreads) {
    const int row = b * a.bm;
    int v = -1;
    if (row < used) {
      int l = 0, h = E - 1;  // last expert whose rows start at or before `row`
      while (l < h) {
        const int mid = (l + h + 1) >> 1;
        if (off[mid] <= row) l = mid;
        else h = mid - 1;
      }
      v = a.mode == TP_MOE_EXPERT_PARALLEL ? ((l % a.n) << 16) | (l / a.n) : l;
    }
    a.blk[b] = v;
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (long long base = lo; base < hi; base += 32) {
    const long long i = base + lane;
    const int e = i < hi ? __ldg(a.ids + i) : -1;
    const bool ok = e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : E + lane);
    const int rank = __popc(peers & lt);
    if (ok) {
      const int p = cnt[warp][e] + rank;
      a.pos[i] = p;
      a.inv[p] = static_cast<int>(i);
    }
    __syncwarp();
    if (ok && rank == 0) cnt[warp][e] += __popc(peers);
    __syncwarp();
  }
}

struct GatherArgs {
  const char *x;          // [T x D] bf16 rows
  long long x_pitch;      // bytes
  char *xp;               // [rows x D] bf16, contiguous
  const int *inv;
  long long rows, row_vecs;  // 16-byte units per row
  int k;
};

__global__ void __launch_bounds__(kThreads) k_moe_gather(GatherArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (long long row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const int asg = __ldg(a.inv + row);
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (asg >= 0 ? asg / a.k : 0) * a.x_pitch);
    uint4 *dst = reinterpret_cast<uint4 *>(a.xp + row * a.row_vecs * 16);
    for (long long v = threadIdx.x; v < a.row_vecs; v += kThreads) dst[v] = asg >= 0 ? __ldg(src + v) : zero;
  }
}

struct CombineArgs {
  const int *pos, *ids;
  const float *w;
  const float *yp[kMaxRanks];  // down-projection rows [rows x D] f32
  float *y[kMaxRanks];         // outputs [T x D] f32
  long long y_ld[kMaxRanks];   // their row pitches (elements)
  long long tokens, d4;        // d4: float4 units per row
  int k, n, per_rank_src, ep_filter;
  // 0: output o gets rank o's partial; 1: every output gets the ring all-reduce
  // of the partials; 2: output 0 alone gets it. Outputs are contiguous ([T x D])
  // when ring != 0.
  int ring;
};

// Rank r's partial of token t, float4 unit v: the sum over the token's slots in
// order of weight * the slot's down-projection row, over the slots rank r ran.
__device__ __forceinline__ float4 moe_partial(const CombineArgs &a, int r, long long t, long long v) {
  const float4 *src = reinterpret_cast<const float4 *>(a.yp[a.per_rank_src ? r : 0]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < a.k; ++j) {
    const long long s = t * a.k + j;
    const int p = __ldg(a.pos + s);
    if (p < 0) continue;
    if (a.ep_filter && __ldg(a.ids + s) % a.n != r) continue;
    const float wt = __ldg(a.w + s);
    const float4 x = src[p * a.d4 + v];
    acc.x = fmaf(wt, x.x, acc.x);
    acc.y = fmaf(wt, x.y, acc.y);
    acc.z = fmaf(wt, x.z, acc.z);
    acc.w = fmaf(wt, x.w, acc.w);
  }
  return acc;
}

// Ring chunk of flat element e of S: chunk c holds [floor(cS/N), floor((c+1)S/N)).
__device__ __forceinline__ int ring_chunk(long long e, long long S, int n) {
  return static_cast<int>(((e + 1) * n + S - 1) / S - 1);
}

__device__ __forceinline__ float lane_of(const float4 &x, int i) {
  return i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w;
}

// Grid (token CTAs, outputs). Output o sums, for each token, its slots in order
// (weight * row pos of the slot) over the slots rank o ran. With a.ring, one
// grid row computes every rank's partial of an element and folds them in the
// order of the element's ring chunk, rank c+1 first, as the one-pass ring adds
// the stored partials.
__global__ void __launch_bounds__(kThreads) k_moe_combine(CombineArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  if (a.ring) {
    const int n = a.n;
    const long long S = a.tokens * a.d4 * 4;
    for (long long t = blockIdx.x; t < a.tokens; t += gridDim.x) {
      for (long long v = threadIdx.x; v < a.d4; v += kThreads) {
        const long long e = (t * a.d4 + v) * 4;
        const int c = ring_chunk(e, S, n);
        float4 sum;
        if (c == ring_chunk(e + 3, S, n)) {
          for (int j = 0; j < n; ++j) {
            const float4 x = moe_partial(a, (c + 1 + j) % n, t, v);
            if (j == 0) {
              sum = x;
            } else {
              sum.x = sum.x + x.x;
              sum.y = sum.y + x.y;
              sum.z = sum.z + x.z;
              sum.w = sum.w + x.w;
            }
          }
        } else {  // the unit straddles two chunks: fold each element in its own order
          float f[4];
          for (int i = 0; i < 4; ++i) {
            const int ci = ring_chunk(e + i, S, n);
            for (int j = 0; j < n; ++j) {
              const float x = lane_of(moe_partial(a, (ci + 1 + j) % n, t, v), i);
              f[i] = j == 0 ? x : f[i] + x;
            }
          }
          sum = make_float4(f[0], f[1], f[2], f[3]);
        }
        for (int o = 0; o < (a.ring == 1 ? n : 1); ++o)
          reinterpret_cast<float4 *>(a.y[o] + t * a.y_ld[o])[v] = sum;
      }
    }
    return;
  }
  const int o = blockIdx.y;
  const float4 *src = reinterpret_cast<const float4 *>(a.yp[a.per_rank_src ? o : 0]);
  for (long long t = blockIdx.x; t < a.tokens; t += gridDim.x) {
    float4 *dst = reinterpret_cast<float4 *>(a.y[o] + t * a.y_ld[o]);
    for (long long v = threadIdx.x; v < a.d4; v += kThreads) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < a.k; ++j) {
        const long long s = t * a.k + j;
        const int p = __ldg(a.pos + s);
        if (p < 0) continue;
        if (a.ep_filter && __ldg(a.ids + s) % a.n != o) continue;
        const float wt = __ldg(a.w + s);
        const float4 r = src[p * a.d4 + v];
        acc.x = fmaf(wt, r.x, acc.x);
        acc.y = fmaf(wt, r.y, acc.y);
        acc.z = fmaf(wt, r.z, acc.z);
        acc.w = fmaf(wt, r.w, acc.w);
      }
      dst[v] = acc;
    }
  }
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

MoeLayout moe_layout(int n, int mode, int experts, int k, long long tokens, long long hidden, long long ffn) {
  MoeLayout L;
  const long long a = tokens * k;
  L.pair = choose_pair(a);
  L.bm = L.pair ? 256 : 128;
  L.rows = (a + static_cast<long long>(experts) * (L.bm - 1) + L.bm - 1) / L.bm * L.bm;
  L.nblk = L.rows / L.bm;
  const long long ypart_copies = mode == TP_MOE_WITHIN_EXPERT ? n : 1;
  size_t o = 0;
  L.off_pos = o;
  o += align256(static_cast<size_t>(a) * 4);
  L.off_inv = o;
  o += align256(static_cast<size_t>(L.rows) * 4);
  L.off_blk = o;
  o += align256(static_cast<size_t>(L.nblk) * 4);
  L.off_xp = o;
  o += align256(static_cast<size_t>(L.rows * hidden) * 2);
  L.off_h = o;  // within-expert: rank r's [rows x F/N] at r * rows * F/N; else [rows x F]
  o += align256(static_cast<size_t>(L.rows * ffn) * 2);
  L.off_yp = o;  // within-expert: rank r's [rows x D] f32 at r * rows * D; else one
  o += align256(static_cast<size_t>(ypart_copies * L.rows * hidden) * 4);
  L.total = o;
  return L;
}

bool moe_ring_folded(int32_t combine, int n) {
  if (n < 2 || (combine != TP_COMBINE_RING_FUSED && combine != TP_COMBINE_RING_SHARED)) return false;
  const char *env = getenv("TPGQA_MOE_RING_FOLD");
  return !(env && env[0] == '0');
}

tp_status moe_forward(const MoeCall &c, cudaStream_t s) {
  const int n = c.n, E = c.experts, k = c.k;
  const long long T = c.x->rows, D = c.hidden, F = c.ffn;
  const bool within = c.mode == TP_MOE_WITHIN_EXPERT;
  const bool fused = c.combine == TP_COMBINE_FUSED;
  const MoeLayout L = moe_layout(n, c.mode, E, k, T, D, F);
  char *ws = static_cast<char *>(c.workspace);
  int *pos = reinterpret_cast<int *>(ws + L.off_pos);
  int *inv = reinterpret_cast<int *>(ws + L.off_inv);
  int *blk = reinterpret_cast<int *>(ws + L.off_blk);
  char *xp = ws + L.off_xp;
  char *hbuf = ws + L.off_h;
  char *yp = ws + L.off_yp;
  DevCtx ctx;
  cudaError_t e = get_dev_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e);

  RouteArgs ra;
  ra.ids = c.ids;
  ra.pos = pos;
  ra.inv = inv;
  ra.blk = blk;
  ra.assignments = T * k;
  ra.rows = L.rows;
  ra.nblk = static_cast<int>(L.nblk);
  ra.bm = L.bm;
  ra.experts = E;
  ra.n = n;
  ra.mode = c.mode;
  ra.status = ctx.status;
  tp_status st = launch_checked(launch_kernel(k_moe_route, dim3(1), dim3(kRouteThreads), 0, s, 1, ra));
  if (st != TP_OK) return st;

  GatherArgs ga;
  ga.x = static_cast<const char *>(c.x->ptr);
  ga.x_pitch = c.x->ld * 2;
  ga.xp = xp;
  ga.inv = inv;
  ga.rows = L.rows;
  ga.row_vecs = D * 2 / 16;
  ga.k = k;
  long long g = static_cast<long long>(num_sms()) * 8;
  if (g > L.rows) g = L.rows;
  st = launch_checked(launch_kernel(k_moe_gather, dim3(static_cast<unsigned>(g)), dim3(kThreads), 0, s, 1, ga));
  if (st != TP_OK) return st;

  // ---- gate/up with SwiGLU: H rows of the routed layout ----
  const long long Fs = within ? F / n : F;  // columns of H per problem
  const int nprob = within ? n : 1;
  // Tiles in groups of about one expert's m-tiles, each group n-tile by n-tile:
  // with the m-tile fastest over all routed rows, every wave of tiles read all
  // of them and a slice of every expert's weights, about 3.6 times the operand
  // bytes from DRAM on the Mixtral shape.
  const int m_group = static_cast<int>(std::max<long long>(1, (T * k / E + L.bm - 1) / L.bm));
  {
    GemmBuilder b;
    b.epi = kEpiSwiGLU;
    b.m_group = m_group;
    b.pair = L.pair;
    std::vector<long long> nc(nprob, Fs);
    int b_rows = 0;
    if (b.pair) {
      b.bn = choose_pair_bn(L.rows, nc.data(), nprob, true, &b_rows);
    } else {
      b.bn = choose_bn(L.rows, nc.data(), nprob, true);
      b_rows = b.bn / 2;
    }
    b.a_rows = b.pair ? 128 : a_box_rows(L.rows);
    b.split = 1;
    tp_status err = TP_OK;
    const int am = b.add_map(xp, L.rows, D, D, b.a_rows, &err);
    if (am < 0) return err;
    // map blocks: gate maps of every rank, then up maps of every rank
    int g0 = -1, u0 = -1;
    for (int r = 0; r < n; ++r) {
      const int m = b.add_map(c.w_gate[r].ptr, c.w_gate[r].rows, D, c.w_gate[r].ld, b_rows, &err);
      if (m < 0) return err;
      if (r == 0) g0 = m;
    }
    for (int r = 0; r < n; ++r) {
      const int m = b.add_map(c.w_up[r].ptr, c.w_up[r].rows, D, c.w_up[r].ld, b_rows, &err);
      if (m < 0) return err;
      if (r == 0) u0 = m;
    }
    const long long ks = D;
    for (int r = 0; r < nprob; ++r) {
      const int gm = g0 + r, um = u0 + r;
      void *out = hbuf + static_cast<size_t>(r) * L.rows * Fs * 2;
      if (!b.add_problem(static_cast<int>(L.rows), static_cast<int>(Fs), out, Fs, &am, &gm, &um, &ks, 1, blk,
                         static_cast<int>(Fs), within ? 1 : n))
        return TP_ERR_UNSUPPORTED;
    }
    if ((st = b.launch(s)) != TP_OK) return st;
  }

  // ---- down projection: f32 rows of the routed layout ----
  {
    GemmBuilder b;
    b.epi = kEpiF32;
    b.m_group = m_group;
    b.pair = L.pair;
    const int dprob = within && !fused ? n : 1;
    std::vector<long long> nc(dprob, D);
    int b_rows = 0;
    if (b.pair) {
      b.bn = choose_pair_bn(L.rows, nc.data(), dprob, false, &b_rows);
    } else {
      b.bn = choose_bn(L.rows, nc.data(), dprob, false);
      b_rows = b.bn;
    }
    b.a_rows = b.pair ? 128 : a_box_rows(L.rows);
    b.split = 1;
    tp_status err = TP_OK;
    std::vector<int> am(nprob), bm(n);
    for (int r = 0; r < nprob; ++r) {
      am[r] = b.add_map(hbuf + static_cast<size_t>(r) * L.rows * Fs * 2, L.rows, Fs, Fs, b.a_rows, &err);
      if (am[r] < 0) return err;
    }
    for (int r = 0; r < n; ++r) {
      bm[r] = b.add_map(c.w_down[r].ptr, c.w_down[r].rows, Fs, c.w_down[r].ld, b_rows, &err);
      if (bm[r] < 0) return err;
    }
    const int brows = static_cast<int>(D);
    if (within && fused) {
      // K segments over the ranks: the accumulator sums every rank's slice
      std::vector<long long> ks(n, Fs);
      if (!b.add_problem(static_cast<int>(L.rows), static_cast<int>(D), yp, D, am.data(), bm.data(), nullptr,
                         ks.data(), n, blk, brows, 1))
        return TP_ERR_UNSUPPORTED;
    } else if (within) {
      const long long ks = Fs;
      for (int r = 0; r < n; ++r)
        if (!b.add_problem(static_cast<int>(L.rows), static_cast<int>(D),
                           yp + static_cast<size_t>(r) * L.rows * D * 4, D, &am[r], &bm[r], nullptr, &ks, 1, blk,
                           brows, 1))
          return TP_ERR_UNSUPPORTED;
    } else {
      const long long ks = F;
      if (!b.add_problem(static_cast<int>(L.rows), static_cast<int>(D), yp, D, &am[0], &bm[0], nullptr, &ks, 1, blk,
                         brows, n))
        return TP_ERR_UNSUPPORTED;
    }
    if ((st = b.launch(s)) != TP_OK) return st;
  }

  // ---- weighted combine of every token's slots, per output rank ----
  CombineArgs ca;
  std::memset(&ca, 0, sizeof(ca));
  ca.pos = pos;
  ca.ids = c.ids;
  ca.w = c.weights;
  const int n_out = fused ? 1 : n;
  for (int r = 0; r < (within && !fused ? n : 1); ++r)
    ca.yp[r] = reinterpret_cast<const float *>(yp + static_cast<size_t>(r) * L.rows * D * 4);
  for (int o = 0; o < n_out; ++o) {
    ca.y[o] = static_cast<float *>(c.y[o].ptr);
    ca.y_ld[o] = c.y[o].ld;
  }
  ca.tokens = T;
  ca.d4 = D / 4;
  ca.k = k;
  ca.n = n;
  ca.per_rank_src = within && !fused;
  ca.ep_filter = !within && !fused;
  // the one-pass ring folded into the combine (TPGQA_MOE_RING_FOLD=0 leaves it
  // to the caller's all-reduce; read on every call)
  ca.ring = moe_ring_folded(c.combine, n) ? (c.combine == TP_COMBINE_RING_FUSED ? 1 : 2) : 0;
  if (ca.ring) {
    long long gx = static_cast<long long>(num_sms()) * 8;
    if (gx > T) gx = T;
    return launch_checked(launch_kernel(k_moe_combine, dim3(static_cast<unsigned>(gx), 1), dim3(kThreads), 0, s, 1,
                                        ca));
  }
  long long gx = static_cast<long long>(num_sms()) * 8 / n_out;
  if (gx < 1) gx = 1;
  if (gx > T) gx = T;
  return launch_checked(launch_kernel(k_moe_combine, dim3(static_cast<unsigned>(gx), n_out), dim3(kThreads), 0, s,
                                      1, ca));
}

}  // namespace tpgqa
