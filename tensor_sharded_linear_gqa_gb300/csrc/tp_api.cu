// C ABI of the library: argument checks, launch sequencing and status codes.
// Every entry point validates everything before it enqueues anything; on an
// error nothing is launched. No entry point allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "tp_internal.h"

namespace tpgqa {

// moe.cu: whether moe_forward folds the one-pass ring (RING_FUSED or RING_SHARED)
// into the MoE block's weighted combine, leaving no all-reduce to the caller.
bool moe_ring_folded(int32_t combine, int n);
// attention.cu: rows of the V^T boxes the attention kernel of this variant loads.
int attention_v_box_rows(int variant);
namespace {

__device__ int g_dev_status = 0;

constexpr long long kDefaultWaitNs = 2000000000LL;  // 2 s
std::atomic<long long> g_wait_ns{kDefaultWaitNs};
std::atomic<unsigned long long> g_failed_ranks{0};
thread_local int t_last_cuda_error = 0;

std::mutex g_dev_mu;
int *g_status_addr[64] = {nullptr};
int g_sm_count[64] = {0};

size_t esize(int32_t dt) { return dt == TP_F32 ? 4 : (dt == TP_BF16 ? 2 : 0); }

// Rows and columns each fit a 32-bit signed index (GEMM tile coordinates and TMA
// box coordinates are 32-bit); element counts and offsets are 64-bit throughout.
constexpr long long kMaxDim = 0x7fffffffLL;

bool shape_ok(const tp_tensor &t) {
  if (esize(t.dtype) == 0) return false;
  if (t.rows < 0 || t.cols < 0 || t.ld < t.cols || t.ld < 1) return false;
  if (t.rows > kMaxDim || t.cols > kMaxDim) return false;
  if (t.rows > 0 && t.cols > 0 && t.ptr == nullptr) return false;
  return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Base and row pitch on 16-byte boundaries (tensor maps, vector stores).
bool pitch_ok(const tp_tensor &t) {
  return aligned16(t.ptr) && ((t.ld * static_cast<long long>(esize(t.dtype))) % 16) == 0;
}

bool pow2_in_range(int32_t n) { return n >= 1 && n <= kMaxRanks && (n & (n - 1)) == 0; }

tp_status check_health(int32_t n) {
  const unsigned long long mask = g_failed_ranks.load();
  if (!mask) return TP_OK;
  for (int32_t r = 0; r < n && r < 64; ++r)
    if (mask & (1ULL << r)) return TP_ERR_RANK_FAILED;
  return TP_OK;
}

char *byte_ptr(void *p, long long elems, int32_t dt) {
  return static_cast<char *>(p) + elems * static_cast<long long>(esize(dt));
}

tp_status zero_fill(const tp_tensor &t, long long col0, long long cols, cudaStream_t s) {
  if (t.rows == 0 || cols == 0) return TP_OK;
  const size_t es = esize(t.dtype);
  const cudaError_t e = cudaMemset2DAsync(byte_ptr(t.ptr, col0, t.dtype), t.ld * es, 0, cols * es,
                                          t.rows, s);
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

// ---- ring collectives over y[0..n-1] ----
tp_status check_ring_bufs(int32_t n, const tp_tensor *buf) {
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (!buf) return TP_ERR_INVALID_ARG;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(buf[r])) return TP_ERR_INVALID_ARG;
    if (buf[r].dtype != TP_F32) return TP_ERR_DTYPE;
    if (buf[r].rows != buf[0].rows || buf[r].cols != buf[0].cols) return TP_ERR_INVALID_ARG;
    if (buf[r].rows > 1 && buf[r].ld != buf[r].cols) return TP_ERR_INVALID_ARG;
    if (buf[r].rows * buf[r].cols > 0 && !aligned16(buf[r].ptr)) return TP_ERR_ALIGNMENT;
  }
  // Every rank's buffer is written by the ring: byte ranges that share even one
  // element would race, so any overlap of two ranks' ranges is rejected.
  const uintptr_t bytes = static_cast<uintptr_t>(buf[0].rows * buf[0].cols) * 4u;
  if (bytes == 0) return TP_OK;
  for (int32_t r = 0; r < n; ++r)
    for (int32_t q = 0; q < r; ++q) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(buf[q].ptr), b = reinterpret_cast<uintptr_t>(buf[r].ptr);
      if (a < b + bytes && b < a + bytes) return TP_ERR_INVALID_ARG;
    }
  return TP_OK;
}

RankPtrs rank_ptrs(int32_t n, const tp_tensor *buf) {
  RankPtrs p;
  std::memset(&p, 0, sizeof(p));
  for (int32_t r = 0; r < n; ++r) p.p[r] = static_cast<float *>(buf[r].ptr);
  return p;
}

tp_status run_reduce_scatter(int32_t n, const tp_tensor *buf, int32_t mode, cudaStream_t s) {
  const long long size = buf[0].rows * buf[0].cols;
  if (n == 1 || size == 0) return TP_OK;
  const RankPtrs p = rank_ptrs(n, buf);
  if (mode == TP_RING_FUSED) return launch_ring_fused(p, n, size, 0, s);
  for (int step = 0; step < n - 1; ++step) {
    const tp_status st = launch_ring_rs_step(p, n, size, step, s);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}

tp_status run_all_gather_ring(int32_t n, const tp_tensor *buf, int32_t mode, cudaStream_t s) {
  const long long size = buf[0].rows * buf[0].cols;
  if (n == 1 || size == 0) return TP_OK;
  const RankPtrs p = rank_ptrs(n, buf);
  if (mode == TP_RING_FUSED) return launch_ring_ag_fused(p, n, size, s);
  for (int step = 0; step < n - 1; ++step) {
    const tp_status st = launch_ring_ag_step(p, n, size, step, s);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}

tp_status run_allreduce(int32_t n, const tp_tensor *buf, int32_t mode, cudaStream_t s) {
  const long long size = buf[0].rows * buf[0].cols;
  if (n == 1 || size == 0) return TP_OK;
  if (mode == TP_RING_FUSED) return launch_ring_fused(rank_ptrs(n, buf), n, size, 1, s);
  if (mode == TP_RING_FUSED_SHARED) return launch_ring_fused(rank_ptrs(n, buf), n, size, 2, s);
  tp_status st = run_reduce_scatter(n, buf, TP_RING_STEPS, s);
  if (st != TP_OK) return st;
  return run_all_gather_ring(n, buf, TP_RING_STEPS, s);
}

// ---- GEMM sequencing ----
// Column-parallel problems: one per rank, A = x, B = w[r], output to outs[r].
struct ColOut {
  void *ptr;
  long long ld;
};

tp_status gemm_bf16_column(const tp_tensor &x, int32_t nb, const tp_tensor *w, const ColOut *outs,
                           int epi, cudaStream_t s, int *ctas_out = nullptr) {
  const long long T = x.rows, K = x.cols;
  long long t256 = 0, t128 = 0;
  for (int32_t r = 0; r < nb; ++r) {
    t256 += ((T + 127) / 128) * ((w[r].rows + 255) / 256);
    t128 += ((T + 127) / 128) * ((w[r].rows + 127) / 128);
  }
  GemmBuilder b;
  b.epi = epi;
  (void)t256;
  (void)t128;
  b.pair = choose_pair(T);
  int b_rows = 0;
  {
    std::vector<long long> nc(nb);
    for (int32_t r = 0; r < nb; ++r) nc[r] = w[r].rows;
    if (b.pair) {
      b.bn = choose_pair_bn(T, nc.data(), nb, false, &b_rows);
    } else {
      b.bn = choose_bn(T, nc.data(), nb, false);
      b_rows = b.bn;
    }
  }
  b.a_rows = b.pair ? 128 : a_box_rows(T);
  tp_status err = TP_OK;
  const int am = b.add_map(x.ptr, T, K, x.ld, b.a_rows, &err);
  if (am < 0) return err;
  for (int32_t r = 0; r < nb; ++r) {
    if (w[r].rows == 0) continue;
    const int bm = b.add_map(w[r].ptr, w[r].rows, K, w[r].ld, b_rows, &err);
    if (bm < 0) return err;
    const long long ks = K;
    if (!b.add_problem(static_cast<int>(T), static_cast<int>(w[r].rows), outs[r].ptr, outs[r].ld,
                       &am, &bm, nullptr, &ks, 1))
      return TP_ERR_UNSUPPORTED;
  }
  const tp_status st = b.launch(s);
  if (ctas_out) *ctas_out = b.ctas;
  return st;
}

// Column-parallel GEMM whose input rows come from N chunk buffers: rows
// [c*T/N, (c+1)*T/N) live in x_chunks[c]. Every (chunk, rank) pair is one problem
// of the grouped GEMM: T/N rows read from chunk c's buffer times rank r's
// weights, written at row offset c*T/N of rank r's output.
tp_status gemm_bf16_column_chunks(int32_t n, const tp_tensor *x_chunks, const tp_tensor *w, const ColOut *outs,
                                  int32_t ydt, int epi, cudaStream_t s) {
  const long long T = x_chunks[0].rows, K = x_chunks[0].cols, Tc = T / n;
  GemmBuilder b;
  b.epi = epi;
  b.pair = choose_pair(Tc);
  int b_rows = 0;
  {
    std::vector<long long> nc;
    for (int32_t c = 0; c < n; ++c)
      for (int32_t r = 0; r < n; ++r) nc.push_back(w[r].rows);
    if (b.pair) {
      b.bn = choose_pair_bn(Tc, nc.data(), static_cast<int>(nc.size()), false, &b_rows);
    } else {
      b.bn = choose_bn(Tc, nc.data(), static_cast<int>(nc.size()), false);
      b_rows = b.bn;
    }
  }
  b.a_rows = b.pair ? 128 : a_box_rows(Tc);
  tp_status err = TP_OK;
  std::vector<int> am(n), bm(n, -1);
  for (int32_t c = 0; c < n; ++c) {
    am[c] = b.add_map(byte_ptr(x_chunks[c].ptr, c * Tc * x_chunks[c].ld, TP_BF16), Tc, K, x_chunks[c].ld,
                      b.a_rows, &err);
    if (am[c] < 0) return err;
  }
  for (int32_t r = 0; r < n; ++r) {
    if (w[r].rows == 0) continue;
    bm[r] = b.add_map(w[r].ptr, w[r].rows, K, w[r].ld, b_rows, &err);
    if (bm[r] < 0) return err;
  }
  // Rank-major: the tiles that run together (consecutive tile indices) share one
  // rank's weight block over all chunks, as one problem over the gathered X would.
  // Chunk-major order has every wave touch all N weight blocks.
  for (int32_t r = 0; r < n; ++r)
    for (int32_t c = 0; c < n; ++c) {
      if (w[r].rows == 0) continue;
      const long long ks = K;
      if (!b.add_problem(static_cast<int>(Tc), static_cast<int>(w[r].rows),
                         byte_ptr(outs[r].ptr, c * Tc * outs[r].ld, ydt), outs[r].ld, &am[c], &bm[r], nullptr,
                         &ks, 1))
        return TP_ERR_UNSUPPORTED;
    }
  return b.launch(s);
}

// Row-parallel shapes whose per-rank GEMM would split K over SM-pair clusters
// (too few 256 x 256 tiles for every pair) while the per-rank partials fit one
// wave of 256 x 128 pair tiles in clusters of 2N CTAs (N = 2 or 4, every
// 256-row tile inside one ring chunk). These layers compute each rank's partial
// on 256 x 128 pair tiles without split-K, whatever the combine, so that the
// ring fold with one cluster split per rank gives the bits of the GEMM followed
// by the ring. At T = 512, N = 2 (the MLP block's down projection) the step
// takes 49.0 us against 50.6 us for the split-K GEMM and the one-pass ring,
// although a 256 x 128 tile loads 1.5 MB of operands per CTA there against
// 1.0 MB for a split-K 256 x 256 tile. TPGQA_RANK_SPLIT=0 turns it off (read
// on every call).
bool rank_split_shape(int32_t n, const tp_tensor *x, const tp_tensor *w) {
  const char *env = getenv("TPGQA_RANK_SPLIT");
  if (env && env[0] == '0') return false;
  const long long T = x[0].rows, nout = w[0].rows;
  if ((n != 2 && n != 4) || !choose_pair(T) || T % n != 0 || (T / n) % 256 != 0 || T > (1LL << 30)) return false;
  if (nout < 1 || nout > (1LL << 30)) return false;
  int b_rows = 0;
  const std::vector<long long> nc(static_cast<size_t>(n), nout);
  if (choose_pair_bn(T, nc.data(), n, false, &b_rows) != 256) return false;
  long long min_stages = -1;
  for (int32_t r = 0; r < n; ++r) {
    const long long st = ((x[r].cols + 63) / 64 + 1) / 2;
    if (min_stages < 0 || st < min_stages) min_stages = st;
  }
  const long long tiles256 = static_cast<long long>(n) * (T / 256) * ((nout + 255) / 256);
  if (choose_split(tiles256, true, min_stages) == 1) return false;
  const long long tiles128 = (T / 256) * ((nout + 127) / 128);
  const int resident = max_active_clusters(2 * n);
  return resident > 0 && tiles128 <= resident;
}

// Row-parallel: fused = one problem whose segments are the ranks; else one problem per rank.
// max_ctas and defer_dep_wait: see GemmParams (single-CTA kernel, T <= 128).
tp_status gemm_bf16_row(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y,
                        bool fused, cudaStream_t s, int max_ctas = 0, bool defer_dep_wait = false) {
  const long long T = x[0].rows, nout = w[0].rows;
  const long long mt = (T + 127) / 128;
  const long long probs = fused ? 1 : n;
  GemmBuilder b;
  b.epi = kEpiF32;
  (void)probs;
  (void)mt;
  b.pair = choose_pair(T);
  int b_rows = 0;
  {
    const std::vector<long long> nc(static_cast<size_t>(probs), nout);
    if (b.pair) {
      b.bn = choose_pair_bn(T, nc.data(), static_cast<int>(probs), false, &b_rows);
    } else {
      b.bn = choose_bn(T, nc.data(), static_cast<int>(probs), false, max_ctas);
      b_rows = b.bn;
      b.max_ctas = max_ctas;
      b.defer_dep_wait = defer_dep_wait;
    }
  }
  if (!fused && rank_split_shape(n, x, w)) {
    b.pair = true;
    b.bn = 128;
    b_rows = 64;
    b.split = 1;
  }
  b.a_rows = b.pair ? 128 : a_box_rows(T);
  tp_status err = TP_OK;
  std::vector<int> am(n), bm(n);
  std::vector<long long> ks(n);
  for (int32_t r = 0; r < n; ++r) {
    am[r] = b.add_map(x[r].ptr, T, x[r].cols, x[r].ld, b.a_rows, &err);
    if (am[r] < 0) return err;
    bm[r] = b.add_map(w[r].ptr, nout, w[r].cols, w[r].ld, b_rows, &err);
    if (bm[r] < 0) return err;
    ks[r] = x[r].cols;
  }
  if (fused) {
    if (!b.add_problem(static_cast<int>(T), static_cast<int>(nout), y[0].ptr, y[0].ld, am.data(),
                       bm.data(), nullptr, ks.data(), n))
      return TP_ERR_UNSUPPORTED;
  } else {
    for (int32_t r = 0; r < n; ++r)
      if (!b.add_problem(static_cast<int>(T), static_cast<int>(nout), y[r].ptr, y[r].ld, &am[r],
                         &bm[r], nullptr, &ks[r], 1))
        return TP_ERR_UNSUPPORTED;
  }
  return b.launch(s);
}

// Whether the ring all-reduce of a bf16 row-parallel layer can be folded into
// its GEMM (the ring-folding pair kernel) with results bit-identical to the
// GEMM followed by the one-pass ring: the layer runs on the SM-pair kernel
// without split-K, every 256-row tile lies inside one ring chunk (T % N == 0,
// T/N a multiple of 256; the chunks are then whole rows), and the outputs can
// be written by 2-D TMA stores. TPGQA_RING_EPILOGUE=0 turns it off (read on
// every call).
bool ring_fold_ok(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y, int copies) {
  const char *env = getenv("TPGQA_RING_EPILOGUE");
  if (env && env[0] == '0') return false;
  const long long T = x[0].rows, nout = w[0].rows;
  if (n < 2 || n > kMaxSegs || 2 * n + copies > kMaxMaps) return false;
  if (!choose_pair(T) || T % n != 0 || (T / n) % 256 != 0 || T > (1LL << 30)) return false;
  if (nout % 4 != 0 || nout > (1LL << 30)) return false;
  for (int r = 0; r < copies; ++r)
    if (y[r].ld != nout) return false;
  // the GEMM without a combine must also run the persistent pair kernel (no split-K)
  int b_rows = 0;
  const std::vector<long long> nc(static_cast<size_t>(n), nout);
  const int bn = choose_pair_bn(T, nc.data(), n, false, &b_rows);
  if (bn == 256) {
    long long min_stages = -1;
    for (int32_t r = 0; r < n; ++r) {
      const long long st = ((x[r].cols + 63) / 64 + 1) / 2;
      if (min_stages < 0 || st < min_stages) min_stages = st;
    }
    const long long tiles = static_cast<long long>(n) * (T / 256) * ((nout + 255) / 256);
    if (choose_split(tiles, true, min_stages) != 1) return false;
  }
  return true;
}

// Row-parallel GEMM with the ring all-reduce folded in: one problem whose
// segments are the ranks, the sum written to y[0..copies-1].
tp_status gemm_bf16_row_ring(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y, int copies,
                             cudaStream_t s) {
  const long long T = x[0].rows, nout = w[0].rows;
  GemmBuilder b;
  b.epi = kEpiF32;
  b.pair = true;
  b.ring = true;
  b.split = 1;
  int b_rows = 0;
  {
    const std::vector<long long> nc(static_cast<size_t>(n), nout);
    b.bn = choose_pair_bn(T, nc.data(), n, false, &b_rows);  // the width the unfolded GEMM takes
  }
  b.a_rows = 128;
  // Tiles in groups of two ring chunks' row tiles: the tiles of one chunk fold
  // the ranks in the same order, so with few chunks in flight fewer ranks' K
  // slices are live in L2 at once. On the prefill layer's down projection
  // (T = 4096, N = 8, K = 3584 per rank) DRAM reads drop from 4.64 to 3.77 GB
  // and the launch from 1.297 to 1.264 ms; one or four chunks per group did less.
  const long long chunk_tiles = (T / n) / 256;
  b.m_group = chunk_tiles > 0 && chunk_tiles <= (1 << 20) ? static_cast<int>(2 * chunk_tiles) : 0;
  tp_status err = TP_OK;
  std::vector<int> am(n), bm(n);
  std::vector<long long> ks(n);
  for (int32_t r = 0; r < n; ++r) {
    am[r] = b.add_map(x[r].ptr, T, x[r].cols, x[r].ld, b.a_rows, &err);
    if (am[r] < 0) return err;
    bm[r] = b.add_map(w[r].ptr, nout, w[r].cols, w[r].ld, b_rows, &err);
    if (bm[r] < 0) return err;
    ks[r] = x[r].cols;
  }
  if (!b.add_problem(static_cast<int>(T), static_cast<int>(nout), y[0].ptr, y[0].ld, am.data(), bm.data(), nullptr,
                     ks.data(), n))
    return TP_ERR_UNSUPPORTED;
  int first = -1;
  for (int r = 0; r < copies; ++r) {
    const int m = b.add_out_map_f32(y[r].ptr, T, nout, y[r].ld, &err);
    if (m < 0) return err;
    if (r == 0) first = m;
  }
  b.p.ring_rows = static_cast<int>(T / n);
  b.p.ring_out = first;
  b.p.ring_copies = copies;
  return b.launch(s);
}

// Row-parallel GEMM with the ring all-reduce folded into the split-K SM-pair
// kernel: one cluster per 256 x 128 tile, split s computing rank s's partial,
// the owned rows summed in their chunk's ring order and written to
// y[0..copies-1]. For the shapes of rank_split_shape; every output shares y[0]'s
// row pitch.
bool ring_split_ok(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y, int copies) {
  const char *env = getenv("TPGQA_RING_EPILOGUE");
  if (env && env[0] == '0') return false;
  if (copies < 1 || copies > kMaxRingCopies) return false;
  for (int r = 1; r < copies; ++r)
    if (y[r].ld != y[0].ld) return false;
  return rank_split_shape(n, x, w);
}

tp_status gemm_bf16_row_ring_split(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y,
                                   int copies, cudaStream_t s) {
  const long long T = x[0].rows, nout = w[0].rows;
  GemmBuilder b;
  b.epi = kEpiF32;
  b.pair = true;
  b.bn = 128;
  b.ring_split = true;
  b.a_rows = 128;
  tp_status err = TP_OK;
  std::vector<int> am(n), bm(n);
  std::vector<long long> ks(n);
  for (int32_t r = 0; r < n; ++r) {
    am[r] = b.add_map(x[r].ptr, T, x[r].cols, x[r].ld, b.a_rows, &err);
    if (am[r] < 0) return err;
    bm[r] = b.add_map(w[r].ptr, nout, w[r].cols, w[r].ld, 64, &err);
    if (bm[r] < 0) return err;
    ks[r] = x[r].cols;
  }
  if (!b.add_problem(static_cast<int>(T), static_cast<int>(nout), y[0].ptr, y[0].ld, am.data(), bm.data(), nullptr,
                     ks.data(), n))
    return TP_ERR_UNSUPPORTED;
  b.p.ring_rows = static_cast<int>(T / n);
  b.p.ring_copies = copies;
  for (int r = 0; r < copies; ++r) b.p.ring_dst[r] = y[r].ptr;
  return b.launch(s);
}

tp_status gemm_f32_column(const tp_tensor &x, int32_t n, const tp_tensor *w, const ColOut *outs,
                          cudaStream_t s) {
  F32Params p;
  std::memset(&p, 0, sizeof(p));
  int np = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (w[r].rows == 0) continue;
    if (np >= kMaxF32Problems) return TP_ERR_UNSUPPORTED;
    F32Problem &pr = p.prob[np];
    pr.m = static_cast<int>(x.rows);
    pr.n = static_cast<int>(w[r].rows);
    pr.m_tiles = (pr.m + 31) / 32;
    pr.n_tiles = (pr.n + 63) / 64;
    pr.tile_begin = p.total_tiles;
    pr.seg_begin = np;
    pr.seg_count = 1;
    pr.out = static_cast<float *>(outs[r].ptr);
    pr.ldc = outs[r].ld;
    p.seg[np] = F32Seg{static_cast<const float *>(x.ptr), x.ld, static_cast<const float *>(w[r].ptr),
                       w[r].ld, static_cast<int>(x.cols)};
    p.total_tiles += pr.m_tiles * pr.n_tiles;
    ++np;
  }
  p.num_problems = np;
  return launch_gemm_f32(p, s);
}

tp_status gemm_f32_row(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y,
                       bool fused, cudaStream_t s) {
  F32Params p;
  std::memset(&p, 0, sizeof(p));
  const int T = static_cast<int>(x[0].rows), nout = static_cast<int>(w[0].rows);
  const int probs = fused ? 1 : n;
  for (int q = 0; q < probs; ++q) {
    F32Problem &pr = p.prob[q];
    pr.m = T;
    pr.n = nout;
    pr.m_tiles = (T + 31) / 32;
    pr.n_tiles = (nout + 63) / 64;
    pr.tile_begin = p.total_tiles;
    pr.seg_begin = fused ? 0 : q;
    pr.seg_count = fused ? n : 1;
    pr.out = static_cast<float *>(y[q].ptr);
    pr.ldc = y[q].ld;
    p.total_tiles += pr.m_tiles * pr.n_tiles;
  }
  for (int32_t r = 0; r < n; ++r)
    p.seg[r] = F32Seg{static_cast<const float *>(x[r].ptr), x[r].ld,
                      static_cast<const float *>(w[r].ptr), w[r].ld, static_cast<int>(x[r].cols)};
  p.num_problems = probs;
  return launch_gemm_f32(p, s);
}

// Validates a row-parallel argument set; on success fills T, n.
tp_status check_row_args(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y,
                         int32_t combine, int32_t *in_dtype) {
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (!x || !w || !y) return TP_ERR_INVALID_ARG;
  if (combine < TP_COMBINE_NONE || combine > TP_COMBINE_RING_SHARED) return TP_ERR_INVALID_ARG;
  const int32_t dt = x[0].dtype;
  const long long T = x[0].rows, nout = w[0].rows;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(x[r]) || !shape_ok(w[r])) return TP_ERR_INVALID_ARG;
    if (x[r].dtype != dt || w[r].dtype != dt) return TP_ERR_DTYPE;
    if (x[r].rows != T || w[r].rows != nout || w[r].cols != x[r].cols) return TP_ERR_INVALID_ARG;
    if (dt == TP_BF16 && T > 0 && (!pitch_ok(x[r]) || !pitch_ok(w[r]))) return TP_ERR_ALIGNMENT;
  }
  const int32_t ny = combine == TP_COMBINE_FUSED ? 1 : n;
  for (int32_t q = 0; q < ny; ++q) {
    if (!shape_ok(y[q])) return TP_ERR_INVALID_ARG;
    if (y[q].dtype != TP_F32) return TP_ERR_DTYPE;
    if (y[q].rows != T || y[q].cols != nout) return TP_ERR_INVALID_ARG;
    if (T > 0 && nout > 0 && !pitch_ok(y[q])) return TP_ERR_ALIGNMENT;
  }
  if (combine == TP_COMBINE_RING || combine == TP_COMBINE_RING_FUSED || combine == TP_COMBINE_RING_SHARED) {
    const tp_status st = check_ring_bufs(n, y);
    if (st != TP_OK) return st;
  }
  *in_dtype = dt;
  return TP_OK;
}

tp_status row_linear_impl(int32_t n, const tp_tensor *x, const tp_tensor *w, const tp_tensor *y,
                          int32_t combine, int32_t dt, cudaStream_t s, int max_ctas = 0,
                          bool defer_dep_wait = false) {
  const long long T = x[0].rows, nout = w[0].rows;
  if (T == 0 || nout == 0) return TP_OK;
  const bool fused = combine == TP_COMBINE_FUSED;
  bool all_k_zero = true;
  for (int32_t r = 0; r < n; ++r) all_k_zero = all_k_zero && x[r].cols == 0;
  tp_status st = TP_OK;
  if (all_k_zero) {
    for (int32_t q = 0; q < (fused ? 1 : n) && st == TP_OK; ++q) st = zero_fill(y[q], 0, nout, s);
    return st;
  }
  for (int32_t r = 0; r < n; ++r)
    if (x[r].cols == 0) return TP_ERR_UNSUPPORTED;  // a rank with an empty K slice
  if (dt == TP_BF16 && (combine == TP_COMBINE_RING_FUSED || combine == TP_COMBINE_RING_SHARED)) {
    const int copies = combine == TP_COMBINE_RING_FUSED ? n : 1;
    if (ring_fold_ok(n, x, w, y, copies)) return gemm_bf16_row_ring(n, x, w, y, copies, s);
    if (ring_split_ok(n, x, w, y, copies)) return gemm_bf16_row_ring_split(n, x, w, y, copies, s);
  }
  if (dt == TP_BF16)
    st = gemm_bf16_row(n, x, w, y, fused, s, max_ctas, defer_dep_wait);
  else
    st = gemm_f32_row(n, x, w, y, fused, s);
  if (st != TP_OK) return st;
  if (combine == TP_COMBINE_RING) return run_allreduce(n, y, TP_RING_STEPS, s);
  if (combine == TP_COMBINE_RING_FUSED) return run_allreduce(n, y, TP_RING_FUSED, s);
  if (combine == TP_COMBINE_RING_SHARED) return run_allreduce(n, y, TP_RING_FUSED_SHARED, s);
  return TP_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Shared helpers declared in tp_internal.h
// ---------------------------------------------------------------------------
cudaError_t get_dev_ctx(DevCtx *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_dev_mu);
  if (!g_status_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dev_status);
    if (e != cudaSuccess) return e;
    g_status_addr[dev] = static_cast<int *>(p);
  }
  out->status = g_status_addr[dev];
  out->wait_ns = g_wait_ns.load();
  return cudaSuccess;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> g(g_dev_mu);
  if (!g_sm_count[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
      v = 148;
    g_sm_count[dev] = v;
  }
  return g_sm_count[dev];
}

bool pdl_enabled() {
  static const bool on = [] {
    const char *e = getenv("TPGQA_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

tp_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return TP_ERR_CUDA;
}

}  // namespace tpgqa

using namespace tpgqa;

// ---------------------------------------------------------------------------
// Linear layers
// ---------------------------------------------------------------------------
extern "C" tp_status tp_column_linear(int32_t n, const tp_tensor *x, const tp_tensor *w,
                                      tp_tensor *y, int32_t gather, tp_stream_t stream) {
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (!x || !w || !y || (gather != 0 && gather != 1)) return TP_ERR_INVALID_ARG;
  if (!shape_ok(*x)) return TP_ERR_INVALID_ARG;
  const int32_t dt = x->dtype;
  const long long T = x->rows, K = x->cols;
  long long total = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(w[r])) return TP_ERR_INVALID_ARG;
    if (w[r].dtype != dt) return TP_ERR_DTYPE;
    if (w[r].cols != K) return TP_ERR_INVALID_ARG;
    total += w[r].rows;
  }
  const int32_t ny = gather ? 1 : n;
  for (int32_t q = 0; q < ny; ++q) {
    if (!shape_ok(y[q])) return TP_ERR_INVALID_ARG;
    if (y[q].rows != T || y[q].cols != (gather ? total : w[q].rows)) return TP_ERR_INVALID_ARG;
    if (dt == TP_F32 && y[q].dtype != TP_F32) return TP_ERR_DTYPE;
  }
  const int32_t ydt = y[0].dtype;
  for (int32_t q = 1; q < ny; ++q)
    if (y[q].dtype != ydt) return TP_ERR_DTYPE;
  if (dt == TP_BF16 && T > 0 && K > 0) {
    if (!pitch_ok(*x)) return TP_ERR_ALIGNMENT;
    for (int32_t r = 0; r < n; ++r)
      if (w[r].rows > 0 && !pitch_ok(w[r])) return TP_ERR_ALIGNMENT;
  }
  if (T > 0) {
    for (int32_t q = 0; q < ny; ++q)
      if (y[q].cols > 0 && !pitch_ok(y[q])) return TP_ERR_ALIGNMENT;
    if (gather)
      for (int32_t r = 0; r < n; ++r)
        if ((w[r].rows * static_cast<long long>(esize(ydt))) % 16) return TP_ERR_ALIGNMENT;
  }
  tp_status st = check_health(n);
  if (st != TP_OK) return st;
  if (T == 0 || total == 0) return TP_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  std::vector<ColOut> outs(n);
  long long off = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (gather)
      outs[r] = ColOut{byte_ptr(y[0].ptr, off, ydt), y[0].ld};
    else
      outs[r] = ColOut{y[r].ptr, y[r].ld};
    off += w[r].rows;
  }
  if (K == 0) {
    off = 0;
    for (int32_t r = 0; r < n && st == TP_OK; ++r) {
      st = gather ? zero_fill(y[0], off, w[r].rows, s) : zero_fill(y[r], 0, w[r].rows, s);
      off += w[r].rows;
    }
    return st;
  }
  if (dt == TP_F32) return gemm_f32_column(*x, n, w, outs.data(), s);
  return gemm_bf16_column(*x, n, w, outs.data(), ydt == TP_F32 ? kEpiF32 : kEpiBF16, s);
}

extern "C" tp_status tp_row_linear(int32_t n, const tp_tensor *x, const tp_tensor *w, tp_tensor *y,
                                   int32_t combine, tp_stream_t stream) {
  int32_t dt = 0;
  tp_status st = check_row_args(n, x, w, y, combine, &dt);
  if (st != TP_OK) return st;
  st = check_health(n);
  if (st != TP_OK) return st;
  return row_linear_impl(n, x, w, y, combine, dt, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Collectives
// ---------------------------------------------------------------------------
extern "C" tp_status tp_reduce_scatter(int32_t n, tp_tensor *buf, int32_t mode, tp_stream_t stream) {
  tp_status st = check_ring_bufs(n, buf);
  if (st != TP_OK) return st;
  if (mode != TP_RING_STEPS && mode != TP_RING_FUSED) return TP_ERR_INVALID_ARG;
  if ((st = check_health(n)) != TP_OK) return st;
  return run_reduce_scatter(n, buf, mode, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_reduce_scatter_bf16(int32_t n, const tp_tensor *partial, tp_tensor *out,
                                            tp_stream_t stream) {
  tp_status st = check_ring_bufs(n, partial);
  if (st != TP_OK) return st;
  if (!out) return TP_ERR_INVALID_ARG;
  const long long rows = partial[0].rows, cols = partial[0].cols;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(out[r])) return TP_ERR_INVALID_ARG;
    if (out[r].dtype != TP_BF16) return TP_ERR_DTYPE;
    if (out[r].rows != rows || out[r].cols != cols || out[r].ld != out[0].ld) return TP_ERR_INVALID_ARG;
    if (rows * cols > 0 && !pitch_ok(out[r])) return TP_ERR_ALIGNMENT;
  }
  if ((st = check_health(n)) != TP_OK) return st;
  const long long size = rows * cols;
  if (size == 0) return TP_OK;
  Bf16Outs o;
  std::memset(&o, 0, sizeof(o));
  for (int32_t r = 0; r < n; ++r) o.p[r] = out[r].ptr;
  o.ld = out[0].ld;
  o.cols = cols;
  return launch_ring_rs_bf16(rank_ptrs(n, partial), o, n, size, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_column_linear_chunks(int32_t n, const tp_tensor *x_chunks, const tp_tensor *w,
                                             tp_tensor *y, int32_t gather, tp_stream_t stream) {
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (!x_chunks || !w || !y || (gather != 0 && gather != 1)) return TP_ERR_INVALID_ARG;
  const long long T = x_chunks[0].rows, K = x_chunks[0].cols;
  for (int32_t c = 0; c < n; ++c) {
    if (!shape_ok(x_chunks[c])) return TP_ERR_INVALID_ARG;
    if (x_chunks[c].dtype != TP_BF16) return TP_ERR_DTYPE;
    if (x_chunks[c].rows != T || x_chunks[c].cols != K) return TP_ERR_INVALID_ARG;
  }
  if (T % n != 0) return TP_ERR_NOT_DIVISIBLE;
  long long total = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(w[r])) return TP_ERR_INVALID_ARG;
    if (w[r].dtype != TP_BF16) return TP_ERR_DTYPE;
    if (w[r].cols != K) return TP_ERR_INVALID_ARG;
    total += w[r].rows;
  }
  const int32_t ny = gather ? 1 : n;
  for (int32_t q = 0; q < ny; ++q) {
    if (!shape_ok(y[q])) return TP_ERR_INVALID_ARG;
    if (y[q].rows != T || y[q].cols != (gather ? total : w[q].rows)) return TP_ERR_INVALID_ARG;
  }
  const int32_t ydt = y[0].dtype;
  for (int32_t q = 1; q < ny; ++q)
    if (y[q].dtype != ydt) return TP_ERR_DTYPE;
  if (T > 0 && K > 0) {
    for (int32_t c = 0; c < n; ++c)
      if (!pitch_ok(x_chunks[c])) return TP_ERR_ALIGNMENT;
    for (int32_t r = 0; r < n; ++r)
      if (w[r].rows > 0 && !pitch_ok(w[r])) return TP_ERR_ALIGNMENT;
  }
  if (T > 0) {
    for (int32_t q = 0; q < ny; ++q)
      if (y[q].cols > 0 && !pitch_ok(y[q])) return TP_ERR_ALIGNMENT;
    if (gather)
      for (int32_t r = 0; r < n; ++r)
        if ((w[r].rows * static_cast<long long>(esize(ydt))) % 16) return TP_ERR_ALIGNMENT;
  }
  tp_status st = check_health(n);
  if (st != TP_OK) return st;
  if (T == 0 || total == 0) return TP_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<ColOut> outs(n);
  long long off = 0;
  for (int32_t r = 0; r < n; ++r) {
    outs[r] = gather ? ColOut{byte_ptr(y[0].ptr, off, ydt), y[0].ld} : ColOut{y[r].ptr, y[r].ld};
    off += w[r].rows;
  }
  if (K == 0) {
    off = 0;
    for (int32_t r = 0; r < n && st == TP_OK; ++r) {
      st = gather ? zero_fill(y[0], off, w[r].rows, s) : zero_fill(y[r], 0, w[r].rows, s);
      off += w[r].rows;
    }
    return st;
  }
  return gemm_bf16_column_chunks(n, x_chunks, w, outs.data(), ydt, ydt == TP_F32 ? kEpiF32 : kEpiBF16, s);
}

extern "C" tp_status tp_vocab_embedding(int32_t n, const int32_t *ids, int64_t n_tokens, const tp_tensor *table,
                                        tp_tensor *out, int32_t n_out, tp_stream_t stream) {
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (!table || !out || (n_out != 1 && n_out != n) || n_tokens < 0 || (n_tokens > 0 && !ids))
    return TP_ERR_INVALID_ARG;
  const int32_t dt = table[0].dtype;
  const long long rows = table[0].rows, D = table[0].cols;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(table[r])) return TP_ERR_INVALID_ARG;
    if (table[r].dtype != dt) return TP_ERR_DTYPE;
    if (table[r].rows != rows || table[r].cols != D) return TP_ERR_INVALID_ARG;
  }
  if (rows == 0 && n_tokens > 0) return TP_ERR_INVALID_ARG;  // no id can be valid
  for (int32_t o = 0; o < n_out; ++o) {
    if (!shape_ok(out[o])) return TP_ERR_INVALID_ARG;
    if (out[o].dtype != dt) return TP_ERR_DTYPE;
    if (out[o].rows != n_tokens || out[o].cols != D) return TP_ERR_INVALID_ARG;
  }
  // element-aligned bases and pitches (the element path), 4-byte aligned ids
  const long long es = static_cast<long long>(esize(dt));
  auto elem_ok = [&](const tp_tensor &t) { return (reinterpret_cast<uintptr_t>(t.ptr) % es) == 0; };
  if (n_tokens > 0 && (reinterpret_cast<uintptr_t>(ids) & 3) != 0) return TP_ERR_ALIGNMENT;
  for (int32_t r = 0; r < n; ++r)
    if (!elem_ok(table[r])) return TP_ERR_ALIGNMENT;
  for (int32_t o = 0; o < n_out; ++o)
    if (!elem_ok(out[o])) return TP_ERR_ALIGNMENT;
  tp_status st = check_health(n);
  if (st != TP_OK) return st;
  if (n_tokens == 0 || D == 0) return TP_OK;
  EmbedArgs a;
  std::memset(&a, 0, sizeof(a));
  bool vec16 = (D * es) % 16 == 0;  // ids are read one int at a time
  for (int32_t r = 0; r < n; ++r) {
    a.tab[r] = static_cast<const char *>(table[r].ptr);
    a.tab_pitch[r] = table[r].ld * es;
    vec16 = vec16 && pitch_ok(table[r]);
  }
  for (int32_t o = 0; o < n_out; ++o) {
    a.out[o] = static_cast<char *>(out[o].ptr);
    a.out_pitch[o] = out[o].ld * es;
    vec16 = vec16 && pitch_ok(out[o]);
  }
  a.ids = ids;
  a.n_tokens = n_tokens;
  a.rows_per_rank = rows;
  a.row_bytes = D * es;
  a.n = n;
  a.n_outs = n_out;
  a.esize = static_cast<int>(es);
  return launch_vocab_embed(a, vec16, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_vocab_lm_head(int32_t n, const tp_tensor *x, const tp_tensor *w, tp_tensor *logits,
                                      int32_t gather, tp_stream_t stream) {
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (!w) return TP_ERR_INVALID_ARG;
  for (int32_t r = 1; r < n; ++r)
    if (w[r].rows != w[0].rows) return TP_ERR_INVALID_ARG;  // slices of V/N ids each
  return tp_column_linear(n, x, w, logits, gather, stream);
}

namespace {

size_t attn_vt_bytes(long long cols, long long tokens) {
  const long long tp8 = (tokens + 7) / 8 * 8;  // V^T row pitch: 16-byte multiple
  return static_cast<size_t>((cols * tp8 * 2 + 255) / 256 * 256);
}

}  // namespace

extern "C" size_t tp_attn_core_workspace_size(const tp_plan *plan, int64_t tokens) {
  tp_dims d;
  tp_rank_shard s0;
  if (!plan || tokens < 0 || tp_plan_dims(plan, &d) != TP_OK || tp_plan_query_rank(plan, 0, &s0) != TP_OK)
    return 0;
  const int nkv = s0.kv_replicated ? 1 : d.tp_size;
  return nkv * attn_vt_bytes((s0.kv_head_end - s0.kv_head_begin) * static_cast<long long>(d.head_dim), tokens);
}

extern "C" tp_status tp_attn_core(const tp_plan *plan, const tp_tensor *q, const tp_tensor *k, const tp_tensor *v,
                                  tp_tensor *a, int32_t causal, void *workspace, size_t workspace_bytes,
                                  tp_stream_t stream) {
  tp_dims d;
  if (!plan || tp_plan_dims(plan, &d) != TP_OK) return TP_ERR_INVALID_ARG;
  if (!q || !k || !v || !a || (causal != 0 && causal != 1)) return TP_ERR_INVALID_ARG;
  const int32_t n = d.tp_size;
  const long long hd = d.head_dim;
  if (hd != 128 || n > kMaxAttnRanks) return TP_ERR_UNSUPPORTED;
  std::vector<tp_rank_shard> sh(n);
  for (int32_t r = 0; r < n; ++r)
    if (tp_plan_query_rank(plan, r, &sh[r]) != TP_OK) return TP_ERR_INVALID_ARG;
  const bool rep = sh[0].kv_replicated != 0;
  const int32_t nkv = rep ? 1 : n;
  const long long T = q[0].rows;
  auto check = [&](const tp_tensor &t, long long cols) -> tp_status {
    if (!shape_ok(t)) return TP_ERR_INVALID_ARG;
    if (t.dtype != TP_BF16) return TP_ERR_DTYPE;
    if (t.rows != T || t.cols != cols) return TP_ERR_INVALID_ARG;
    if (T > 0 && !pitch_ok(t)) return TP_ERR_ALIGNMENT;
    return TP_OK;
  };
  tp_status st;
  int total_heads = 0;
  for (int32_t r = 0; r < n; ++r) {
    const long long qc = (sh[r].q_head_end - sh[r].q_head_begin) * hd;
    if ((st = check(q[r], qc)) != TP_OK) return st;
    if ((st = check(a[r], qc)) != TP_OK) return st;
    total_heads += sh[r].q_head_end - sh[r].q_head_begin;
  }
  const long long kvc = (sh[0].kv_head_end - sh[0].kv_head_begin) * hd;
  for (int32_t r = 0; r < nkv; ++r) {
    if ((st = check(k[r], kvc)) != TP_OK) return st;
    if ((st = check(v[r], kvc)) != TP_OK) return st;
  }
  if (total_heads > kMaxAttnHeads || T > 0x7fffffffLL - 256) return TP_ERR_UNSUPPORTED;
  const size_t vt = attn_vt_bytes(kvc, T);
  if (T > 0) {
    if (!workspace || workspace_bytes < nkv * vt) return TP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TP_ERR_ALIGNMENT;
  }
  if ((st = check_health(n)) != TP_OK) return st;
  if (T == 0 || total_heads == 0) return TP_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long tp8 = (T + 7) / 8 * 8;
  // V -> V^T for every kv source in one launch, so that P V reads K-major tiles
  TransposeArgs ta;
  std::memset(&ta, 0, sizeof(ta));
  for (int32_t r = 0; r < nkv; ++r) {
    ta.in[r] = v[r].ptr;
    ta.ld_in[r] = v[r].ld;
    ta.out[r] = static_cast<char *>(workspace) + r * vt;
  }
  ta.ld_out = tp8;
  ta.rows = static_cast<int>(T);
  ta.cols = static_cast<int>(kvc);
  if ((st = launch_transpose_bf16(ta, nkv, s)) != TP_OK) return st;
  static thread_local AttnParams prm;  // ~22 KB: kept off the stack
  std::memset(&prm, 0, sizeof(prm));
  prm.variant = attention_variant();
  const int k_box = attention_k_box_rows(prm.variant);
  for (int32_t r = 0; r < n; ++r)
    if (!encode_bf16_map_2d(&prm.maps[r], q[r].ptr, T, q[r].cols, q[r].ld, 128)) return TP_ERR_INVALID_ARG;
  for (int32_t r = 0; r < nkv; ++r) {
    if (!encode_bf16_map_2d(&prm.maps[n + r], k[r].ptr, T, kvc, k[r].ld, k_box)) return TP_ERR_INVALID_ARG;
    if (!encode_bf16_map_2d(&prm.maps[n + nkv + r], static_cast<char *>(workspace) + r * vt, kvc, T, tp8,
                            attention_v_box_rows(prm.variant)))
      return TP_ERR_INVALID_ARG;
  }
  int h = 0;
  std::vector<int32_t> q2kv;
  for (int32_t r = 0; r < n; ++r) {
    const int nq = sh[r].q_head_end - sh[r].q_head_begin;
    q2kv.assign(nq, 0);
    if (nq > 0 && tp_plan_q_to_kv(plan, r, q2kv.data(), nq) != TP_OK) return TP_ERR_INVALID_ARG;
    const int src = rep ? 0 : r;
    for (int j = 0; j < nq; ++j, ++h) {
      AttnHead &e = prm.heads[h];
      e.q_map = r;
      e.k_map = n + src;
      e.v_map = n + nkv + src;
      e.q_col = static_cast<int>(j * hd);
      e.kv_col = static_cast<int>(q2kv[j] * hd);
      e.out = byte_ptr(a[r].ptr, j * hd, TP_BF16);
      e.out_ld = a[r].ld;
    }
  }
  prm.tokens = static_cast<int>(T);
  prm.q_tiles = static_cast<int>((T + 127) / 128);
  prm.causal = causal;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(hd)));
  return launch_attention(prm, total_heads, s);
}

namespace {

tp_status moe_check_dims(const tp_moe_dims *d) {
  if (!d) return TP_ERR_INVALID_ARG;
  const int32_t n = d->tp_size;
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (d->mode != TP_MOE_EXPERT_PARALLEL && d->mode != TP_MOE_WITHIN_EXPERT) return TP_ERR_INVALID_ARG;
  if (d->num_experts < 1 || d->num_experts > kMaxExperts || d->top_k < 1 || d->hidden < 1 || d->ffn < 1)
    return TP_ERR_INVALID_ARG;
  const bool within = d->mode == TP_MOE_WITHIN_EXPERT;
  if (!within && d->num_experts % n) return TP_ERR_NOT_DIVISIBLE;
  if (within && d->ffn % n) return TP_ERR_NOT_DIVISIBLE;
  if (d->hidden % 8 || (within ? d->ffn / n : d->ffn) % 8) return TP_ERR_ALIGNMENT;  // 16-byte rows
  return TP_OK;
}

bool moe_tokens_ok(const tp_moe_dims *d, int64_t tokens) {
  // assignments and rows of the routed layout are indexed with 32-bit ints
  return tokens >= 0 && tokens <= (0x7fffffffLL - 256LL * kMaxExperts) / d->top_k;
}

}  // namespace

extern "C" size_t tp_moe_workspace_size(const tp_moe_dims *d, int64_t tokens) {
  if (moe_check_dims(d) != TP_OK || !moe_tokens_ok(d, tokens)) return 0;
  return moe_layout(d->tp_size, d->mode, d->num_experts, d->top_k, tokens, d->hidden, d->ffn).total;
}

extern "C" tp_status tp_moe_block(const tp_moe_dims *d, const tp_tensor *x, const int32_t *topk_ids,
                                  const float *topk_w, const tp_tensor *w_gate, const tp_tensor *w_up,
                                  const tp_tensor *w_down, tp_tensor *y, int32_t combine, void *workspace,
                                  size_t workspace_bytes, tp_stream_t stream) {
  tp_status st = moe_check_dims(d);
  if (st != TP_OK) return st;
  if (!x || !w_gate || !w_up || !w_down || !y) return TP_ERR_INVALID_ARG;
  if (combine < TP_COMBINE_NONE || combine > TP_COMBINE_RING_SHARED) return TP_ERR_INVALID_ARG;
  const int32_t n = d->tp_size, E = d->num_experts;
  const bool within = d->mode == TP_MOE_WITHIN_EXPERT;
  const long long D = d->hidden, F = d->ffn, T = x->rows;
  const long long e_loc = within ? E : E / n, Fs = within ? F / n : F;
  if (!shape_ok(*x) || x->cols != D) return TP_ERR_INVALID_ARG;
  if (x->dtype != TP_BF16) return TP_ERR_DTYPE;
  if (!moe_tokens_ok(d, T)) return TP_ERR_INVALID_ARG;
  auto check_w = [&](const tp_tensor &t, long long rows, long long cols) -> tp_status {
    if (!shape_ok(t)) return TP_ERR_INVALID_ARG;
    if (t.dtype != TP_BF16) return TP_ERR_DTYPE;
    if (t.rows != rows || t.cols != cols) return TP_ERR_INVALID_ARG;
    if (!pitch_ok(t)) return TP_ERR_ALIGNMENT;
    return TP_OK;
  };
  for (int32_t r = 0; r < n; ++r) {
    if ((st = check_w(w_gate[r], e_loc * Fs, D)) != TP_OK) return st;
    if ((st = check_w(w_up[r], e_loc * Fs, D)) != TP_OK) return st;
    if ((st = check_w(w_down[r], e_loc * D, Fs)) != TP_OK) return st;
  }
  const int32_t ny = combine == TP_COMBINE_FUSED ? 1 : n;
  for (int32_t q = 0; q < ny; ++q) {
    if (!shape_ok(y[q])) return TP_ERR_INVALID_ARG;
    if (y[q].dtype != TP_F32) return TP_ERR_DTYPE;
    if (y[q].rows != T || y[q].cols != D) return TP_ERR_INVALID_ARG;
    if (T > 0 && !pitch_ok(y[q])) return TP_ERR_ALIGNMENT;
  }
  if ((combine == TP_COMBINE_RING || combine == TP_COMBINE_RING_FUSED || combine == TP_COMBINE_RING_SHARED) && n > 1)
    for (int32_t q = 0; q < n; ++q)
      if (y[q].ld != D) return TP_ERR_INVALID_ARG;  // the ring reduces contiguous buffers
  if (T > 0) {
    if (!pitch_ok(*x)) return TP_ERR_ALIGNMENT;
    if (!topk_ids || !topk_w) return TP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(topk_ids) & 3) || (reinterpret_cast<uintptr_t>(topk_w) & 3))
      return TP_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < tp_moe_workspace_size(d, T)) return TP_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return TP_ERR_ALIGNMENT;
  }
  if ((st = check_health(n)) != TP_OK) return st;
  if (T == 0) return TP_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MoeCall c;
  c.n = n;
  c.mode = d->mode;
  c.experts = E;
  c.k = d->top_k;
  c.combine = combine;
  c.hidden = D;
  c.ffn = F;
  c.x = x;
  c.ids = topk_ids;
  c.weights = topk_w;
  c.w_gate = w_gate;
  c.w_up = w_up;
  c.w_down = w_down;
  c.y = y;
  c.workspace = workspace;
  if ((st = moe_forward(c, s)) != TP_OK) return st;
  if (moe_ring_folded(combine, n)) return TP_OK;  // the combine kernel ran the one-pass ring
  if (combine == TP_COMBINE_RING) return run_allreduce(n, y, TP_RING_STEPS, s);
  if (combine == TP_COMBINE_RING_FUSED) return run_allreduce(n, y, TP_RING_FUSED, s);
  if (combine == TP_COMBINE_RING_SHARED) return run_allreduce(n, y, TP_RING_FUSED_SHARED, s);
  return TP_OK;
}

extern "C" tp_status tp_ring_all_gather(int32_t n, tp_tensor *buf, int32_t mode, tp_stream_t stream) {
  tp_status st = check_ring_bufs(n, buf);
  if (st != TP_OK) return st;
  if (mode != TP_RING_STEPS && mode != TP_RING_FUSED) return TP_ERR_INVALID_ARG;
  if ((st = check_health(n)) != TP_OK) return st;
  return run_all_gather_ring(n, buf, mode, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_allreduce_ring(int32_t n, tp_tensor *buf, int32_t mode, tp_stream_t stream) {
  tp_status st = check_ring_bufs(n, buf);
  if (st != TP_OK) return st;
  if (mode != TP_RING_STEPS && mode != TP_RING_FUSED && mode != TP_RING_FUSED_SHARED) return TP_ERR_INVALID_ARG;
  if ((st = check_health(n)) != TP_OK) return st;
  return run_allreduce(n, buf, mode, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_all_gather(int32_t n, const tp_tensor *shard, tp_tensor *out, int32_t n_out,
                                   int32_t axis, tp_stream_t stream) {
  if (!pow2_in_range(n)) return n >= 1 && n <= kMaxRanks ? TP_ERR_TP_SIZE_NOT_POW2 : TP_ERR_INVALID_ARG;
  if (!shard || !out || (n_out != 1 && n_out != n) || (axis != 0 && axis != 1))
    return TP_ERR_INVALID_ARG;
  const int32_t dt = shard[0].dtype;
  long long sum = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(shard[r])) return TP_ERR_INVALID_ARG;
    if (shard[r].dtype != dt) return TP_ERR_DTYPE;
    if (axis == 1 && shard[r].rows != shard[0].rows) return TP_ERR_INVALID_ARG;
    if (axis == 0 && shard[r].cols != shard[0].cols) return TP_ERR_INVALID_ARG;
    sum += axis == 1 ? shard[r].cols : shard[r].rows;
  }
  const long long orows = axis == 1 ? shard[0].rows : sum;
  const long long ocols = axis == 1 ? sum : shard[0].cols;
  for (int32_t o = 0; o < n_out; ++o) {
    if (!shape_ok(out[o])) return TP_ERR_INVALID_ARG;
    if (out[o].dtype != dt) return TP_ERR_DTYPE;
    if (out[o].rows != orows || out[o].cols != ocols) return TP_ERR_INVALID_ARG;
  }
  tp_status st = check_health(n);
  if (st != TP_OK) return st;
  const long long es = static_cast<long long>(esize(dt));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CopyBatch b;
  std::memset(&b, 0, sizeof(b));
  for (int32_t o = 0; o < n_out; ++o) {
    long long off = 0;
    for (int32_t r = 0; r < n; ++r) {
      const tp_tensor &sh = shard[r];
      Copy2D c;
      c.src = static_cast<const char *>(sh.ptr);
      c.src_pitch = sh.ld * es;
      c.dst_pitch = out[o].ld * es;
      c.rows = sh.rows;
      c.row_bytes = sh.cols * es;
      c.dst = axis == 1 ? byte_ptr(out[o].ptr, off, dt) : byte_ptr(out[o].ptr, off * out[o].ld, dt);
      off += axis == 1 ? sh.cols : sh.rows;
      if (c.rows == 0 || c.row_bytes == 0) continue;
      b.c[b.n++] = c;
      if (b.n == kMaxCopies) {
        if ((st = launch_copy_batch(b, s)) != TP_OK) return st;
        b.n = 0;
      }
    }
  }
  return launch_copy_batch(b, s);
}

// ---------------------------------------------------------------------------
// Blocks
// ---------------------------------------------------------------------------
extern "C" size_t tp_mlp_block_workspace_size(const tp_plan *plan, int64_t tokens) {
  tp_dims d;
  if (tp_plan_dims(plan, &d) != TP_OK || tokens < 0) return 0;
  return static_cast<size_t>(tokens) * static_cast<size_t>(d.ffn) * 2;
}

namespace {

// Checks the gate/up weights against the plan; Fr = ffn / tp_size.
tp_status check_gate_up(const tp_dims &d, const tp_tensor *x, const tp_tensor *w_gate,
                        const tp_tensor *w_up) {
  const int32_t n = d.tp_size;
  const long long D = d.hidden, Fr = d.ffn / n, T = x->rows;
  if (!shape_ok(*x) || x->cols != D) return TP_ERR_INVALID_ARG;
  if (x->dtype != TP_BF16) return TP_ERR_DTYPE;
  if (T > 0 && !pitch_ok(*x)) return TP_ERR_ALIGNMENT;
  for (int32_t r = 0; r < n; ++r) {
    const tp_tensor *ws[2] = {&w_gate[r], &w_up[r]};
    for (const tp_tensor *t : ws) {
      if (!shape_ok(*t)) return TP_ERR_INVALID_ARG;
      if (t->dtype != TP_BF16) return TP_ERR_DTYPE;
      if (t->rows != Fr || t->cols != D) return TP_ERR_INVALID_ARG;
      if (!pitch_ok(*t)) return TP_ERR_ALIGNMENT;
    }
  }
  return TP_OK;
}

// One grouped launch: problem r = (X, G_r | U_r) -> h[r] with the SwiGLU epilogue.
tp_status launch_gate_up(const tp_dims &d, const tp_tensor *x, const tp_tensor *w_gate,
                         const tp_tensor *w_up, const tp_tensor *h, cudaStream_t s) {
  const int32_t n = d.tp_size;
  const long long D = d.hidden, Fr = d.ffn / n, T = x->rows;
  GemmBuilder b;
  b.epi = kEpiSwiGLU;
  const long long mt = (T + 127) / 128;
  (void)mt;
  b.pair = choose_pair(T);
  int b_rows = 0;
  {
    const std::vector<long long> nc(static_cast<size_t>(n), Fr);
    if (b.pair) {
      b.bn = choose_pair_bn(T, nc.data(), n, true, &b_rows);
    } else {
      b.bn = choose_bn(T, nc.data(), n, true);
      b_rows = b.bn / 2;
    }
  }
  b.a_rows = b.pair ? 128 : a_box_rows(T);
  tp_status err = TP_OK;
  const int am = b.add_map(x->ptr, T, D, x->ld, b.a_rows, &err);
  if (am < 0) return err;
  for (int32_t r = 0; r < n; ++r) {
    // gate and up each fill half of a tile's accumulator columns
    const int gm = b.add_map(w_gate[r].ptr, Fr, D, w_gate[r].ld, b_rows, &err);
    if (gm < 0) return err;
    const int um = b.add_map(w_up[r].ptr, Fr, D, w_up[r].ld, b_rows, &err);
    if (um < 0) return err;
    const long long ks = D;
    if (!b.add_problem(static_cast<int>(T), static_cast<int>(Fr), h[r].ptr, h[r].ld, &am, &gm, &um,
                       &ks, 1))
      return TP_ERR_UNSUPPORTED;
  }
  return b.launch(s);
}

}  // namespace

extern "C" tp_status tp_gate_up_swiglu(const tp_plan *plan, const tp_tensor *x,
                                       const tp_tensor *w_gate, const tp_tensor *w_up, tp_tensor *h,
                                       tp_stream_t stream) {
  tp_dims d;
  if (!plan || tp_plan_dims(plan, &d) != TP_OK) return TP_ERR_INVALID_ARG;
  if (!x || !w_gate || !w_up || !h) return TP_ERR_INVALID_ARG;
  tp_status st = check_gate_up(d, x, w_gate, w_up);
  if (st != TP_OK) return st;
  const int32_t n = d.tp_size;
  const long long Fr = d.ffn / n, T = x->rows;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(h[r])) return TP_ERR_INVALID_ARG;
    if (h[r].dtype != TP_BF16) return TP_ERR_DTYPE;
    if (h[r].rows != T || h[r].cols != Fr) return TP_ERR_INVALID_ARG;
    if (T > 0 && !pitch_ok(h[r])) return TP_ERR_ALIGNMENT;
  }
  if ((st = check_health(n)) != TP_OK) return st;
  if (T == 0) return TP_OK;
  return launch_gate_up(d, x, w_gate, w_up, h, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_mlp_block(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_gate,
                                  const tp_tensor *w_up, const tp_tensor *w_down, tp_tensor *y,
                                  int32_t combine, void *workspace, size_t workspace_bytes,
                                  tp_stream_t stream) {
  tp_dims d;
  if (!plan || tp_plan_dims(plan, &d) != TP_OK) return TP_ERR_INVALID_ARG;
  if (!x || !w_gate || !w_up || !w_down || !y) return TP_ERR_INVALID_ARG;
  if (combine < TP_COMBINE_NONE || combine > TP_COMBINE_RING_SHARED) return TP_ERR_INVALID_ARG;
  tp_status st = check_gate_up(d, x, w_gate, w_up);
  if (st != TP_OK) return st;
  const int32_t n = d.tp_size;
  const long long D = d.hidden, Fr = d.ffn / n, T = x->rows;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(w_down[r])) return TP_ERR_INVALID_ARG;
    if (w_down[r].dtype != TP_BF16) return TP_ERR_DTYPE;
    if (w_down[r].rows != D || w_down[r].cols != Fr) return TP_ERR_INVALID_ARG;
    if (!pitch_ok(w_down[r])) return TP_ERR_ALIGNMENT;
  }
  // H_r is rank r's column block of one [T x F] bf16 buffer in the workspace.
  if ((Fr * 2) % 16) return TP_ERR_ALIGNMENT;
  std::vector<tp_tensor> h(n);
  for (int32_t r = 0; r < n; ++r)
    h[r] = tp_tensor{byte_ptr(workspace, r * Fr, TP_BF16), TP_BF16, 0, T, Fr,
                     static_cast<int64_t>(d.ffn)};
  if (T > 0) {
    if (!workspace || workspace_bytes < tp_mlp_block_workspace_size(plan, T)) return TP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TP_ERR_ALIGNMENT;
  } else {
    for (int32_t r = 0; r < n; ++r) h[r].ptr = nullptr;
  }
  int32_t dt = 0;
  if ((st = check_row_args(n, h.data(), w_down, y, combine, &dt)) != TP_OK) return st;
  if ((st = check_health(n)) != TP_OK) return st;
  if (T == 0) return TP_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launch_gate_up(d, x, w_gate, w_up, h.data(), s)) != TP_OK) return st;
  // down row-parallel GEMM + combine.
  return row_linear_impl(n, h.data(), w_down, y, combine, TP_BF16, s);
}

namespace {

// Checks x, the q/k/v weights and outputs against the plan; sets T.
tp_status check_qkv(const tp_dims &d, const tp_rank_shard &s0, const tp_tensor *x, const tp_tensor *w_q,
                    const tp_tensor *w_k, const tp_tensor *w_v, const tp_tensor *q, const tp_tensor *k,
                    const tp_tensor *v) {
  const int32_t n = d.tp_size;
  const long long D = d.hidden, hd = d.head_dim, T = x->rows;
  if (!shape_ok(*x) || x->cols != D) return TP_ERR_INVALID_ARG;
  if (x->dtype != TP_BF16) return TP_ERR_DTYPE;
  if (T > 0 && !pitch_ok(*x)) return TP_ERR_ALIGNMENT;
  const int32_t nkv = s0.kv_replicated ? 1 : n;
  const long long qcols = (s0.q_head_end - s0.q_head_begin) * hd;
  const long long kvcols = (s0.kv_head_end - s0.kv_head_begin) * hd;
  auto check_w = [&](const tp_tensor &t, long long rows, long long cols) -> tp_status {
    if (!shape_ok(t)) return TP_ERR_INVALID_ARG;
    if (t.dtype != TP_BF16) return TP_ERR_DTYPE;
    if (t.rows != rows || t.cols != cols) return TP_ERR_INVALID_ARG;
    if (!pitch_ok(t)) return TP_ERR_ALIGNMENT;
    return TP_OK;
  };
  auto check_out = [&](const tp_tensor &t, long long cols) -> tp_status {
    if (!shape_ok(t)) return TP_ERR_INVALID_ARG;
    if (t.dtype != TP_BF16) return TP_ERR_DTYPE;
    if (t.rows != T || t.cols != cols) return TP_ERR_INVALID_ARG;
    if (T > 0 && !pitch_ok(t)) return TP_ERR_ALIGNMENT;
    return TP_OK;
  };
  tp_status st;
  for (int32_t r = 0; r < n; ++r) {
    if ((st = check_w(w_q[r], qcols, D)) != TP_OK) return st;
    if ((st = check_out(q[r], qcols)) != TP_OK) return st;
  }
  for (int32_t r = 0; r < nkv; ++r) {
    if ((st = check_w(w_k[r], kvcols, D)) != TP_OK) return st;
    if ((st = check_w(w_v[r], kvcols, D)) != TP_OK) return st;
    if ((st = check_out(k[r], kvcols)) != TP_OK) return st;
    if ((st = check_out(v[r], kvcols)) != TP_OK) return st;
  }
  return TP_OK;
}

// q/k/v column-parallel as one grouped launch (K/V once when replicated).
// q/k/v on the SM-pair kernel with each rank's k and v (at most 128 columns each)
// sharing one 256-column tile: k's rows feed one CTA of the pair, v's the other,
// and the two halves of the accumulator are stored to k and v. Separate k and v
// problems of 128 columns would each fill only half of a 256-column tile.
tp_status gemm_bf16_qkv_paired(int32_t n, int32_t nkv, const tp_tensor &x, const tp_tensor *w_q,
                               const tp_tensor *w_k, const tp_tensor *w_v, const tp_tensor *q, const tp_tensor *k,
                               const tp_tensor *v, cudaStream_t s) {
  const long long T = x.rows, K = x.cols;
  GemmBuilder b;
  b.epi = kEpiBF16;
  b.pair = true;
  b.bn = 256;
  b.split = 1;
  b.a_rows = 128;
  tp_status err = TP_OK;
  const int am = b.add_map(x.ptr, T, K, x.ld, 128, &err);
  if (am < 0) return err;
  for (int32_t r = 0; r < n; ++r) {
    if (w_q[r].rows == 0) continue;
    const int bm = b.add_map(w_q[r].ptr, w_q[r].rows, K, w_q[r].ld, 128, &err);
    if (bm < 0) return err;
    if (!b.add_problem(static_cast<int>(T), static_cast<int>(w_q[r].rows), q[r].ptr, q[r].ld, &am, &bm, nullptr,
                       &K, 1))
      return TP_ERR_UNSUPPORTED;
  }
  for (int32_t r = 0; r < nkv; ++r) {
    const int bk = b.add_map(w_k[r].ptr, w_k[r].rows, K, w_k[r].ld, 128, &err);
    if (bk < 0) return err;
    const int bv = b.add_map(w_v[r].ptr, w_v[r].rows, K, w_v[r].ld, 128, &err);
    if (bv < 0) return err;
    if (!b.add_dual_problem(static_cast<int>(T), static_cast<int>(w_k[r].rows), k[r].ptr, k[r].ld, v[r].ptr,
                            v[r].ld, am, bk, bv, K))
      return TP_ERR_UNSUPPORTED;
  }
  return b.launch(s);
}

tp_status launch_qkv(const tp_dims &d, const tp_rank_shard &s0, const tp_tensor *x, const tp_tensor *w_q,
                     const tp_tensor *w_k, const tp_tensor *w_v, const tp_tensor *q, const tp_tensor *k,
                     const tp_tensor *v, cudaStream_t s, int *ctas_out = nullptr) {
  const int32_t n = d.tp_size;
  const int32_t nkv = s0.kv_replicated ? 1 : n;
  {
    // TPGQA_QKV_PAIRED=0 keeps k and v as separate problems (read on every call).
    const char *env = getenv("TPGQA_QKV_PAIRED");
    bool paired = !(env && env[0] == '0') && choose_pair(x->rows) && 1 + n + 2 * nkv <= kMaxMaps &&
                  n + nkv <= kMaxProblems;
    for (int32_t r = 0; paired && r < nkv; ++r)
      paired = w_k[r].rows == w_v[r].rows && w_k[r].rows > 0 && w_k[r].rows <= 128;
    if (paired) return gemm_bf16_qkv_paired(n, nkv, *x, w_q, w_k, w_v, q, k, v, s);
  }
  std::vector<tp_tensor> ws;
  std::vector<ColOut> outs;
  for (int32_t r = 0; r < n; ++r) {
    ws.push_back(w_q[r]);
    outs.push_back(ColOut{q[r].ptr, q[r].ld});
  }
  for (int32_t r = 0; r < nkv; ++r) {
    ws.push_back(w_k[r]);
    outs.push_back(ColOut{k[r].ptr, k[r].ld});
    ws.push_back(w_v[r]);
    outs.push_back(ColOut{v[r].ptr, v[r].ld});
  }
  return gemm_bf16_column(*x, static_cast<int32_t>(ws.size()), ws.data(), outs.data(), kEpiBF16, s, ctas_out);
}

// Bytes [begin, end) a tensor's elements span.
struct Span {
  uintptr_t begin, end;
};
Span tensor_span(const tp_tensor &t) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(t.ptr);
  if (t.rows <= 0 || t.cols <= 0) return Span{b, b};
  const long long es = t.dtype == TP_F32 ? 4 : 2;
  return Span{b, b + static_cast<uintptr_t>(((t.rows - 1) * t.ld + t.cols) * es)};
}
bool spans_overlap(const tp_tensor *a, int na, const tp_tensor *b, int nb) {
  for (int i = 0; i < na; ++i) {
    const Span x = tensor_span(a[i]);
    for (int j = 0; j < nb; ++j) {
      const Span y = tensor_span(b[j]);
      if (x.begin < y.end && y.begin < x.end) return true;
    }
  }
  return false;
}

}  // namespace

extern "C" tp_status tp_qkv_proj(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_q,
                                 const tp_tensor *w_k, const tp_tensor *w_v, tp_tensor *q, tp_tensor *k,
                                 tp_tensor *v, tp_stream_t stream) {
  tp_dims d;
  if (!plan || tp_plan_dims(plan, &d) != TP_OK) return TP_ERR_INVALID_ARG;
  if (!x || !w_q || !w_k || !w_v || !q || !k || !v) return TP_ERR_INVALID_ARG;
  tp_rank_shard s0;
  tp_plan_query_rank(plan, 0, &s0);
  tp_status st = check_qkv(d, s0, x, w_q, w_k, w_v, q, k, v);
  if (st != TP_OK) return st;
  if ((st = check_health(d.tp_size)) != TP_OK) return st;
  if (x->rows == 0) return TP_OK;
  return launch_qkv(d, s0, x, w_q, w_k, w_v, q, k, v, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tp_status tp_attn_proj(const tp_plan *plan, const tp_tensor *x, const tp_tensor *w_q,
                                  const tp_tensor *w_k, const tp_tensor *w_v, tp_tensor *q,
                                  tp_tensor *k, tp_tensor *v, const tp_tensor *a,
                                  const tp_tensor *w_o, tp_tensor *y, int32_t combine,
                                  tp_stream_t stream) {
  tp_dims d;
  if (!plan || tp_plan_dims(plan, &d) != TP_OK) return TP_ERR_INVALID_ARG;
  if (!x || !w_q || !w_k || !w_v || !q || !k || !v || !a || !w_o || !y) return TP_ERR_INVALID_ARG;
  if (combine < TP_COMBINE_NONE || combine > TP_COMBINE_RING_SHARED) return TP_ERR_INVALID_ARG;
  const int32_t n = d.tp_size;
  const long long D = d.hidden, hd = d.head_dim, T = x->rows;
  tp_rank_shard s0;
  tp_plan_query_rank(plan, 0, &s0);
  tp_status st = check_qkv(d, s0, x, w_q, w_k, w_v, q, k, v);
  if (st != TP_OK) return st;
  const long long qcols = (s0.q_head_end - s0.q_head_begin) * hd;
  for (int32_t r = 0; r < n; ++r) {
    if (!shape_ok(w_o[r])) return TP_ERR_INVALID_ARG;
    if (w_o[r].dtype != TP_BF16) return TP_ERR_DTYPE;
    if (w_o[r].rows != D || w_o[r].cols != qcols) return TP_ERR_INVALID_ARG;
    if (!pitch_ok(w_o[r])) return TP_ERR_ALIGNMENT;
  }
  int32_t dt = 0;
  if ((st = check_row_args(n, a, w_o, y, combine, &dt)) != TP_OK) return st;
  if (dt != TP_BF16) return TP_ERR_DTYPE;
  if (a[0].rows != T) return TP_ERR_INVALID_ARG;
  if ((st = check_health(n)) != TP_OK) return st;
  if (T == 0) return TP_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int qkv_ctas = 0;
  if ((st = launch_qkv(d, s0, x, w_q, w_k, w_v, q, k, v, s, &qkv_ctas)) != TP_OK) return st;
  // o_proj row-parallel + combine. o_proj does not read what q/k/v write, so at
  // decode sizes (T <= 128, where neither GEMM fills the GPU's HBM stream alone)
  // it runs beside q/k/v on the SMs q/k/v leaves free, and waits for q/k/v only
  // before it exits. Only where the GEMM alone would run one problem per rank
  // without split-K (its partials then have the same bits on fewer CTAs), and
  // not when its buffers overlap q/k/v's; TPGQA_CONCURRENT_OPROJ=0 turns it off
  // (read on every call).
  bool beside = false;
  {
    const char *env = getenv("TPGQA_CONCURRENT_OPROJ");
    const int32_t nkv = s0.kv_replicated ? 1 : n;
    const int32_t ny = combine == TP_COMBINE_FUSED ? 1 : n;
    bool unsplit = false;
    if (combine != TP_COMBINE_FUSED && T <= 128 && !choose_pair(T)) {
      const std::vector<long long> nc(static_cast<size_t>(n), D);
      const int bn = choose_bn(T, nc.data(), n, false);
      const long long tiles = static_cast<long long>(n) * ((T + 127) / 128) * ((D + bn - 1) / bn);
      unsplit = !(bn == 256 && tiles * 2 <= num_sms());
    }
    beside = !(env && env[0] == '0') && unsplit && qkv_ctas > 0 && qkv_ctas + 16 <= num_sms() &&
             !spans_overlap(a, n, q, n) && !spans_overlap(a, n, k, nkv) && !spans_overlap(a, n, v, nkv) &&
             !spans_overlap(y, ny, q, n) && !spans_overlap(y, ny, k, nkv) && !spans_overlap(y, ny, v, nkv) &&
             !spans_overlap(y, ny, x, 1) && !spans_overlap(y, ny, w_q, n) && !spans_overlap(y, ny, w_k, nkv) &&
             !spans_overlap(y, ny, w_v, nkv);
  }
  if (beside) return row_linear_impl(n, a, w_o, y, combine, TP_BF16, s, num_sms() - qkv_ctas, true);
  return row_linear_impl(n, a, w_o, y, combine, TP_BF16, s);
}

// ---------------------------------------------------------------------------
// Status, health, diagnostics
// ---------------------------------------------------------------------------
extern "C" const char *tp_status_str(tp_status s) {
  switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG";
    case TP_ERR_TP_SIZE_NOT_POW2: return "TP_ERR_TP_SIZE_NOT_POW2";
    case TP_ERR_NOT_DIVISIBLE: return "TP_ERR_NOT_DIVISIBLE";
    case TP_ERR_GQA_SHAPE: return "TP_ERR_GQA_SHAPE";
    case TP_ERR_DTYPE: return "TP_ERR_DTYPE";
    case TP_ERR_ALIGNMENT: return "TP_ERR_ALIGNMENT";
    case TP_ERR_RANK_FAILED: return "TP_ERR_RANK_FAILED";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
    case TP_ERR_CUDA: return "TP_ERR_CUDA";
    case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
    case TP_ERR_BAD_TOKEN: return "TP_ERR_BAD_TOKEN";
  }
  return "TP_ERR_UNKNOWN";
}

extern "C" int32_t tp_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" tp_status tp_set_rank_health(int32_t rank, int32_t healthy) {
  if (rank < 0 || rank >= 64) return TP_ERR_INVALID_ARG;
  const unsigned long long bit = 1ULL << rank;
  if (healthy)
    g_failed_ranks.fetch_and(~bit);
  else
    g_failed_ranks.fetch_or(bit);
  return TP_OK;
}

extern "C" tp_status tp_device_status(tp_stream_t stream, int32_t *detail) {
  if (detail) *detail = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_dev_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (detail) *detail = word;
  return word == 0 ? TP_OK : (word == kDevBadToken ? TP_ERR_BAD_TOKEN : TP_ERR_TIMEOUT);
}

extern "C" tp_status tp_set_wait_budget(int64_t nanoseconds) {
  if (nanoseconds < 0) return TP_ERR_INVALID_ARG;
  g_wait_ns.store(nanoseconds == 0 ? kDefaultWaitNs : nanoseconds);
  return TP_OK;
}

extern "C" tp_status tp_debug_wait_timeout(tp_stream_t stream) {
  return launch_debug_wait(reinterpret_cast<cudaStream_t>(stream));
}

namespace tpgqa {
namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace tpgqa

extern "C" uint64_t tp_launch_count(void) { return tpgqa::g_launches.load(std::memory_order_relaxed); }

extern "C" const char *tp_version(void) { return "tpgqa 0.1 (sm_103a)"; }
