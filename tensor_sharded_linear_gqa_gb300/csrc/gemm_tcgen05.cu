// bf16 grouped GEMM on the 5th-generation tensor cores: C = A * B^T with A
// [M x K] and B [N x K] both K-major (weights stored [out x in]), fp32
// accumulation in tensor memory.
//
// Three kernels share one problem/segment model and one warp layout:
//   k_gemm_bf16        persistent, one CTA per SM, 128 x BN tiles (BN 128..256),
//                      used for at most 128 rows (decode);
//   k_gemm_bf16_pair   persistent over 2-CTA clusters, 256 x BN tiles with
//                      tcgen05.mma.cta_group::2 (BN 256 or 224);
//   k_gemm_bf16_splitk one tile per cluster, K split over the cluster's CTAs and
//                      reduced through distributed shared memory in fixed order.
// Warp roles:
//   warp 0      TMA producer: one thread streams A and B k-tiles into a ring of
//               shared-memory stages (128-byte swizzle), one copy per operand
//               per k-tile, or per stage with 3-D tensor maps.
//   warp 1      owns TMEM (two fp32 accumulators; alloc / dealloc); one thread
//               issues tcgen05.mma (K=16, four per 64-wide k-tile), frees each
//               stage with tcgen05.commit and hands each finished accumulator
//               to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (each warp reads its
//               32-lane quarter), fused output transform, global stores; the
//               accumulator is released as soon as it has been read.
// A problem's K loop runs over its segments in order, so a row-parallel layer
// can sum every rank's shard in the same accumulator (segments = ranks).
// Every mbarrier wait is bounded; a wait that runs out records a code in the
// device status word, the CTA drains its in-flight copies, frees TMEM and exits.
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "sm100_ptx.cuh"
#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // bf16 elements in one 128-byte swizzled row
constexpr int UMMA_K = 16;
constexpr int kThreads = 192;

// Single-CTA tiles: 128 x BN, one 64-wide k-tile per pipeline stage. A stage
// holds a_rows x 128 bytes of A (the rows loaded) followed by BN x 128 bytes of
// B, so the number of stages, and with it the bytes in flight per SM, follows
// a_rows: at T = 64, five 40 KB stages instead of four 48 KB ones. The host
// computes the count (one_stages_for) and the kernel reads it from its params.
template <int BN>
struct TileCfg {
  static constexpr int kBBytes = BN * BK * 2;
};
constexpr int kMaxOneStages = 8;
constexpr int kSmemLimit = 227 * 1024;  // dynamic shared memory per CTA on sm_100-class GPUs

// Stages of the single-CTA kernels for A boxes of a_rows rows and BN-column tiles.
inline int one_stages_for(int a_rows, int bn) {
  const int stage = a_rows * BK * 2 + bn * BK * 2;
  int s = (kSmemLimit - 1024 - 256) / stage;
  return s > kMaxOneStages ? kMaxOneStages : s;
}
inline int one_smem_bytes(int a_rows, int bn, int stages) {
  return 1024 + stages * (a_rows * BK * 2 + bn * BK * 2) + 256;
}

__device__ __forceinline__ void record(int *status, int code) { atomicCAS(status, 0, code); }

// silu(g) = g * sigmoid(g); for g < -87 the denominator exceeds 2^126 and the
// fast division returns 0, the correctly signed limit to within 1e-36.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ void store_f32_row32(float *out, long long ldc, int row, int col0, int n,
                                                const float (&f)[32]) {
  float *dst = out + static_cast<long long>(row) * ldc + col0;
  if (col0 + 32 <= n) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      *reinterpret_cast<float4 *>(dst + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
  } else {
    for (int j = 0; j < 32; ++j)
      if (col0 + j < n) dst[j] = f[j];
  }
}

__device__ __forceinline__ void store_bf16_row32(__nv_bfloat16 *out, long long ldc, int row, int col0,
                                                 int n, const float (&f)[32]) {
  __nv_bfloat16 *dst = out + static_cast<long long>(row) * ldc + col0;
  if (col0 + 32 <= n) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      uint4 w;
      __nv_bfloat162 h0 = __floats2bfloat162_rn(f[j + 0], f[j + 1]);
      __nv_bfloat162 h1 = __floats2bfloat162_rn(f[j + 2], f[j + 3]);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(f[j + 4], f[j + 5]);
      __nv_bfloat162 h3 = __floats2bfloat162_rn(f[j + 6], f[j + 7]);
      memcpy(&w.x, &h0, 4);
      memcpy(&w.y, &h1, 4);
      memcpy(&w.z, &h2, 4);
      memcpy(&w.w, &h3, 4);
      *reinterpret_cast<uint4 *>(dst + j) = w;
    }
  } else {
    for (int j = 0; j < 32; ++j)
      if (col0 + j < n) dst[j] = __float2bfloat16_rn(f[j]);
  }
}

__device__ __forceinline__ void store_bf16_row16(__nv_bfloat16 *out, long long ldc, int row, int col0,
                                                 int n, const float (&f)[16]) {
  __nv_bfloat16 *dst = out + static_cast<long long>(row) * ldc + col0;
  if (col0 + 16 <= n) {
#pragma unroll
    for (int j = 0; j < 16; j += 8) {
      uint4 w;
      __nv_bfloat162 h0 = __floats2bfloat162_rn(f[j + 0], f[j + 1]);
      __nv_bfloat162 h1 = __floats2bfloat162_rn(f[j + 2], f[j + 3]);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(f[j + 4], f[j + 5]);
      __nv_bfloat162 h3 = __floats2bfloat162_rn(f[j + 6], f[j + 7]);
      memcpy(&w.x, &h0, 4);
      memcpy(&w.y, &h1, 4);
      memcpy(&w.z, &h2, 4);
      memcpy(&w.w, &h3, 4);
      *reinterpret_cast<uint4 *>(dst + j) = w;
    }
  } else {
    for (int j = 0; j < 16; ++j)
      if (col0 + j < n) dst[j] = __float2bfloat16_rn(f[j]);
  }
}

// Walks this CTA's (tile, segment, k-tile) sequence: tiles blockIdx.x,
// blockIdx.x + gridDim.x, ...; within a tile every segment of its problem in
// order, within a segment its k-tiles.
struct Cursor {
  int tile, prob, mt, nt, seg, kt, kt_in_tile;
  int moff, brow;  // B map offset and first B row of the tile (block tables)
  bool valid;
};

// The problem holding a tile: the last one whose tile_begin is <= tile (problems
// are laid out in tile order), by binary search over up to kMaxProblems.
__device__ __forceinline__ int find_problem(const GemmParams &p, int tile) {
  int lo = 0, hi = p.num_problems - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile >= p.prob[mid].tile_begin) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// (m-tile, n-tile) of a problem's tile `local`: m fastest over the problem, or
// with GROUPED over groups of m_group m-tiles (the last group may be shorter).
// Only the kernels that take grouped problems compile the grouped form: its
// mere presence in the other kernels cost 1.5-3 us per step of back-to-back
// small GEMMs (the T=512 MLP block, decode), with m_group = 0 at run time.
template <bool GROUPED>
__device__ __forceinline__ void tile_coords(const GemmProblem &pr, int local, int &mt, int &nt) {
  if constexpr (GROUPED) {
    const int g = pr.m_group;
    if (g > 0 && g < pr.m_tiles) {
      const int per_group = g * pr.n_tiles;
      const int grp = local / per_group, r = local - grp * per_group;
      const int rows = min(g, pr.m_tiles - grp * g);
      mt = grp * g + r % rows;
      nt = r / rows;
      return;
    }
  }
  mt = local % pr.m_tiles;
  nt = local / pr.m_tiles;
}

// First tile at or after `tile`, stepping by `stride`, that its problem's block
// table does not skip (every tile when there is no table). The producer, the
// MMA issuer and the epilogue all step with it, so they see the same tiles.
template <bool GROUPED = false>
__device__ __forceinline__ int live_tile(const GemmParams &p, int tile, int stride) {
  for (; tile < p.total_tiles; tile += stride) {
    const GemmProblem &pr = p.prob[find_problem(p, tile)];
    if (!pr.blk) break;
    int mt, nt;
    tile_coords<GROUPED>(pr, tile - pr.tile_begin, mt, nt);
    const int v = __ldg(pr.blk + mt);
    if (v >= 0 && (v >> 16) < pr.n_moff) break;
  }
  return tile;
}

// B map offset and first B row of m-tile mt of a problem.
__device__ __forceinline__ void tile_b_origin(const GemmProblem &pr, int mt, int &moff, int &brow) {
  const int v = pr.blk ? __ldg(pr.blk + mt) : 0;
  moff = v >> 16;
  brow = (v & 0xFFFF) * pr.b_rows_per_blk;
}

__device__ __forceinline__ void cursor_tile(const GemmParams &p, Cursor &c, int tile) {
  tile = live_tile(p, tile, gridDim.x);
  c.tile = tile;
  c.valid = tile < p.total_tiles;
  if (!c.valid) return;
  c.prob = find_problem(p, tile);
  const GemmProblem &pr = p.prob[c.prob];
  tile_coords<false>(pr, tile - pr.tile_begin, c.mt, c.nt);
  tile_b_origin(pr, c.mt, c.moff, c.brow);
  c.seg = 0;
  c.kt = 0;
  c.kt_in_tile = 0;
}

__device__ __forceinline__ void cursor_next(const GemmParams &p, Cursor &c) {
  const GemmProblem &pr = p.prob[c.prob];
  ++c.kt;
  ++c.kt_in_tile;
  if (c.kt < p.seg[pr.seg_begin + c.seg].k_tiles) return;
  c.kt = 0;
  if (++c.seg < pr.seg_count) return;
  cursor_tile(p, c, c.tile + gridDim.x);
}

__device__ __forceinline__ int tile_k_tiles(const GemmParams &p, int prob) {
  const GemmProblem &pr = p.prob[prob];
  int n = 0;
  for (int s = 0; s < pr.seg_count; ++s) n += p.seg[pr.seg_begin + s].k_tiles;
  return n;
}

// Persistent kernel: one CTA per SM walks tiles blockIdx.x + j * gridDim.x.
// TMEM holds two accumulators, so the epilogue of tile j overlaps the MMAs of
// tile j+1. The producer can also prefetch B tiles kPrefetch k-blocks ahead into
// L2 (off by default: it slowed every measured shape).
template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1) k_gemm_bf16(const __grid_constant__ GemmParams p) {
  using C = TileCfg<BN>;
  constexpr int kBRows = (EPI == kEpiSwiGLU) ? BN / 2 : BN;  // rows per B map box
  constexpr int kOutCols = (EPI == kEpiSwiGLU) ? BN / 2 : BN;
  const int kPrefetch = p.prefetch;
  // Two accumulators; TMEM is allocated in powers of two, so BN in (128, 256]
  // takes 512 columns with the accumulators at columns 0 and 256.
  constexpr uint32_t kAccStride = BN <= 128 ? 128 : 256;
  constexpr uint32_t kTmemCols = 2 * kAccStride;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  // stage st: A (a_rows x 128 B) at sbase + st*kStage, B right after it
  const int kStagesRt = p.one_stages;
  const uint32_t kAT = static_cast<uint32_t>(p.a_rows) * 128u;
  const uint32_t kStage = kAT + C::kBBytes;
  const uint32_t sbase = ptx::smem_addr(smem);
  auto a_slot = [&](int st) { return sbase + static_cast<uint32_t>(st) * kStage; };
  auto b_slot = [&](int st) { return sbase + static_cast<uint32_t>(st) * kStage + kAT; };
  uint8_t *bar_area = smem + static_cast<uint32_t>(kStagesRt) * kStage;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  // layout: full[S], empty[S], tmem_full[2], tmem_empty[2], drain, then slot / flag words
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (kStagesRt + i); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStagesRt + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStagesRt + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStagesRt + 4);
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 8 * (2 * kStagesRt + 5));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 8 * (2 * kStagesRt + 5) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesRt; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.n_maps_used; ++i) ptx::prefetch_tensormap(&p.maps[i]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Weights do not come from the previous kernel: the producer starts the B
  // loads of its first stages before the grid-dependency wait (each stage's
  // barrier expects the A bytes too, which follow the wait).
  int pre = 0;  // leading k-blocks whose B loads were issued early (thread 0 only)
  if (warp == 0 && lane == 0 && p.early_b) {
    Cursor c;
    cursor_tile(p, c, blockIdx.x);
    for (; pre < kStagesRt && c.valid; ++pre) {
      const GemmSeg &sg = p.seg[p.prob[c.prob].seg_begin + c.seg];
      ptx::mbar_arrive_expect_tx(full_bar(pre), static_cast<uint32_t>(p.a_rows * 128 + C::kBBytes));
      ptx::tma_load_2d(b_slot(pre), &p.maps[sg.b_map + c.moff], c.kt * BK, c.brow + c.nt * kBRows, full_bar(pre));
      if (EPI == kEpiSwiGLU)
        ptx::tma_load_2d(b_slot(pre) + kBRows * 128, &p.maps[sg.b2_map + c.moff], c.kt * BK,
                         c.brow + c.nt * kBRows, full_bar(pre));
      cursor_next(p, c);
    }
  }
  // Prologue done: wait for the previous kernel in the stream, then let the next
  // one launch. With defer_dep_wait the kernel shares no buffer with the previous
  // kernel and waits for it only before exiting (below).
  if (!p.defer_dep_wait) ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  int issued = 0;  // k-blocks whose loads the producer started (thread 0 only)
  if (warp == 0) {
    if (lane == 0) {
      Cursor ld, pf;
      cursor_tile(p, ld, blockIdx.x);
      cursor_tile(p, pf, blockIdx.x);
      auto prefetch = [&](const Cursor &c) {
        const GemmSeg &sg = p.seg[p.prob[c.prob].seg_begin + c.seg];
        ptx::tma_prefetch_l2_2d(&p.maps[sg.b_map + c.moff], c.kt * BK, c.brow + c.nt * kBRows);
        if (EPI == kEpiSwiGLU)
          ptx::tma_prefetch_l2_2d(&p.maps[sg.b2_map + c.moff], c.kt * BK, c.brow + c.nt * kBRows);
      };
      for (int i = 0; i < kPrefetch && pf.valid; ++i) {
        prefetch(pf);
        cursor_next(p, pf);
      }
      int kb = 0;
      while (ld.valid) {
        if (kPrefetch > 0 && pf.valid) {
          prefetch(pf);
          cursor_next(p, pf);
        }
        const int st = kb % kStagesRt;
        const uint32_t ph = (kb / kStagesRt) & 1;
        if (*abort_flag) break;
        const GemmSeg &sg = p.seg[p.prob[ld.prob].seg_begin + ld.seg];
        if (kb < pre) {  // B already in flight, the stage's barrier already armed: A only
          ptx::tma_load_2d(a_slot(st), &p.maps[sg.a_map], ld.kt * BK, ld.mt * BM, full_bar(st));
          issued = ++kb;
          cursor_next(p, ld);
          continue;
        }
        if (!ptx::mbar_wait(empty_bar(st), ph ^ 1, p.wait_ns)) {
          record(p.status, kDevTimeoutProducer);
          *abort_flag = 1;
          break;
        }
        ptx::mbar_arrive_expect_tx(full_bar(st), static_cast<uint32_t>(p.a_rows * 128 + C::kBBytes));
        ptx::tma_load_2d(a_slot(st), &p.maps[sg.a_map], ld.kt * BK, ld.mt * BM, full_bar(st));
        ptx::tma_load_2d(b_slot(st), &p.maps[sg.b_map + ld.moff], ld.kt * BK, ld.brow + ld.nt * kBRows,
                         full_bar(st));
        if (EPI == kEpiSwiGLU)
          ptx::tma_load_2d(b_slot(st) + kBRows * 128, &p.maps[sg.b2_map + ld.moff], ld.kt * BK,
                           ld.brow + ld.nt * kBRows, full_bar(st));
        issued = ++kb;
        cursor_next(p, ld);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      int kb = 0;
      bool ok = true;
      for (int tile = live_tile(p, blockIdx.x, gridDim.x), j = 0; ok && tile < p.total_tiles;
           tile = live_tile(p, tile + gridDim.x, gridDim.x), ++j) {
        const int a = j & 1;
        const uint32_t use = static_cast<uint32_t>(j >> 1);
        if (*abort_flag || !ptx::mbar_wait(tempty_bar(a), (use & 1) ^ 1, p.wait_ns)) {
          if (!*abort_flag) record(p.status, kDevTimeoutMma);
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(a) * kAccStride;
        const int nk = tile_k_tiles(p, find_problem(p, tile));
        for (int k0 = 0; k0 < nk; ++k0, ++kb) {
          const int st = kb % kStagesRt;
          const uint32_t ph = (kb / kStagesRt) & 1;
          if (*abort_flag) { ok = false; break; }
          if (!ptx::mbar_wait(full_bar(st), ph, p.wait_ns)) {
            record(p.status, kDevTimeoutMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          // A rows past a_rows read the next bytes of the stage (B): their
          // accumulator rows are never stored
          const uint64_t ad = ptx::smem_desc_sw128(a_slot(st));
          const uint64_t bd = ptx::smem_desc_sw128(b_slot(st));
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            ptx::mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (k0 | k) != 0 ? 1u : 0u);
          ptx::mma_commit(empty_bar(st));
        }
        ptx::mma_commit(tfull_bar(a));
      }
      // Every MMA this thread issued has completed once the drain barrier fires.
      ptx::mma_commit(drain_bar);
      if (!ptx::mbar_wait(drain_bar, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    // ---- epilogue: warps 2..5, warp w reads TMEM lanes [32*(w%4), 32*(w%4)+32) ----
    const int q = warp & 3;
    for (int tile = live_tile(p, blockIdx.x, gridDim.x), j = 0; tile < p.total_tiles;
         tile = live_tile(p, tile + gridDim.x, gridDim.x), ++j) {
      const int a = j & 1;
      const uint32_t use = static_cast<uint32_t>(j >> 1);
      const bool ready = ptx::mbar_wait(tfull_bar(a), use & 1, p.wait_ns);
      if (!ready && lane == 0) record(p.status, kDevTimeoutEpilogue);
      ptx::tc_fence_after();
      if (!__all_sync(0xffffffffu, ready && (*abort_flag == 0))) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      const GemmProblem &pr = p.prob[find_problem(p, tile)];
      int mt, nt;
      tile_coords<false>(pr, tile - pr.tile_begin, mt, nt);
      const int row = mt * BM + q * 32 + lane;
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(a) * kAccStride +
                             (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (EPI == kEpiSwiGLU) {
        // gate sums in accumulator columns [0, BN/2), up sums in [BN/2, BN)
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(pr.out);
        constexpr int kFull = (BN / 2) / 32 * 32;  // columns handled 32 at a time
#pragma unroll 1
        for (int c = 0; c < kFull; c += 32) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32cols(tbase + c, g);
          ptx::tmem_ld_32cols(tbase + BN / 2 + c, u);
          ptx::tmem_ld_wait();
          if (c + 32 == BN / 2) {  // accumulator fully read: hand it back to the MMA warp
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty_bar(a));
          }
          float h[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) h[jj] = silu(__uint_as_float(g[jj])) * __uint_as_float(u[jj]);
          if (row < pr.m) store_bf16_row32(out, pr.ldc, row, nt * kOutCols + c, pr.n, h);
        }
        if constexpr (BN / 2 > kFull) {
          static_assert(BN / 2 - kFull == 16, "a 16-column tail");
          uint32_t g[16], u[16];
          ptx::tmem_ld_16cols(tbase + kFull, g);
          ptx::tmem_ld_16cols(tbase + BN / 2 + kFull, u);
          ptx::tmem_ld_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(tempty_bar(a));
          float h[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) h[jj] = silu(__uint_as_float(g[jj])) * __uint_as_float(u[jj]);
          if (row < pr.m) store_bf16_row16(out, pr.ldc, row, nt * kOutCols + kFull, pr.n, h);
        }
      } else {
        static_assert(BN % 32 == 0, "32-column epilogue chunks");
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32cols(tbase + c, v);
          ptx::tmem_ld_wait();
          if (c + 32 == BN) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty_bar(a));
          }
          float f[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) f[jj] = __uint_as_float(v[jj]);
          if (row < pr.m) {
            if constexpr (EPI == kEpiF32)
              store_f32_row32(static_cast<float *>(pr.out), pr.ldc, row, nt * kOutCols + c, pr.n, f);
            else
              store_bf16_row32(static_cast<__nv_bfloat16 *>(pr.out), pr.ldc, row, nt * kOutCols + c,
                               pr.n, f);
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // Loads the producer started must land before the CTA's shared memory goes away.
    const int first = issued > kStagesRt ? issued - kStagesRt : 0;
    for (int kb = first; kb < issued; ++kb)
      if (!ptx::mbar_wait(full_bar(kb % kStagesRt), (kb / kStagesRt) & 1, p.wait_ns))
        record(p.status, kDevTimeoutDrain);
    if (pre > issued) {
      // early B loads whose stage never received its A: their barrier cannot
      // complete, so give the copies time to land
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ptx::globaltimer_ns() - t0 < 2000000ull) {
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
  // The grid completes only after the previous kernel has: kernels after this one
  // that wait for it also see the previous kernel's writes.
  if (p.defer_dep_wait && threadIdx.x == 0) ptx::griddep_wait();
}

// ---------------------------------------------------------------------------
// Pair kernel: two CTAs of a cluster (an SM pair) compute one 256 x BN tile
// with tcgen05.mma.cta_group::2 (M=256, N=BN, K=16). CTA r of the pair loads
// A rows [128r, 128r+128) of the tile and BN/2 rows of B (for SwiGLU: the gate
// rows in CTA 0, the up rows in CTA 1), so each SM streams half the B bytes of
// the single-CTA kernel per MMA flop. Only CTA 0 issues MMAs; its commits arrive
// on the stage and accumulator barriers of both CTAs. Each CTA holds its own 128
// accumulator rows in TMEM (two buffers, at columns 0 and 256) and runs its own
// epilogue; the epilogue warps of both CTAs release an accumulator on CTA 0's
// barrier.
// ---------------------------------------------------------------------------
// A stage holds KSUB consecutive 64-wide k-tiles (KSUB boxes of A and of B per
// CTA under one barrier): the TMA unit of an SM delivers more bytes per clock
// with more boxes in flight per barrier phase, so 128-wide stages (KSUB = 2)
// keep the tensor pipe fed better than 64-wide ones.
constexpr int kPairABytes = 128 * BK * 2;  // one 64-wide k-tile of this CTA's 128 A rows
// BN accumulator columns per tile: each CTA holds BN/2 rows of B (for SwiGLU,
// BN/2 gate rows in CTA 0 and BN/2 up rows in CTA 1). BN is 256, or 224 when
// narrower tiles fill the last wave better. BN = 512 or 448 (SwiGLU only, one
// 64-wide k-tile per stage): BN/2 gate and BN/2 up columns per tile, computed by
// two N = BN/2 MMAs per k-step into accumulators at TMEM columns 0 and 256; each
// CTA holds BN/4 gate rows and BN/4 up rows of B (its half of each MMA's N).
template <int KSUB, int BN>
struct PairCfg {
  static constexpr int kBRows = BN / 2;
  static constexpr int kBBytes = kBRows * BK * 2;  // one 64-wide k-tile of this CTA's B rows
  static constexpr int kStageBytes = KSUB * (kPairABytes + kBBytes);
  // as many stages as fit beside the barriers: 3 for 256- and 224-column tiles
  // of 128-deep stages, 4 for 128-column tiles
  static constexpr int kMaxStages = KSUB == 1 ? 5 : 4;
  static constexpr int kStages =
      (kSmemLimit - 1280) / kStageBytes > kMaxStages ? kMaxStages : (kSmemLimit - 1280) / kStageBytes;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 256;
  static_assert(kBBytes % 1024 == 0, "B k-tiles must keep the 1024-byte swizzle alignment");
};

template <int KSUB>
__device__ __forceinline__ int seg_stages(const GemmSeg &sg) { return (sg.k_tiles + KSUB - 1) / KSUB; }

template <int KSUB>
__device__ __forceinline__ int tile_stages(const GemmParams &p, int prob) {
  const GemmProblem &pr = p.prob[prob];
  int n = 0;
  for (int s = 0; s < pr.seg_count; ++s) n += seg_stages<KSUB>(p.seg[pr.seg_begin + s]);
  return n;
}

// GROUPED: the problems may order their tiles in groups of m-tiles (m_group).
template <int EPI, int KSUB, int BN, bool GROUPED = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm_bf16_pair(const __grid_constant__ GemmParams p) {
  using PC = PairCfg<KSUB, BN>;
  constexpr int kPairSub = KSUB;
  constexpr int kPairStages = PC::kStages;
  constexpr int kPairStageBytes = PC::kStageBytes;
  constexpr int kPairBBytes = PC::kBBytes;
  constexpr int kHalfB = PC::kBRows;  // B rows per CTA
  constexpr int kOutCols = (EPI == kEpiSwiGLU) ? BN / 2 : BN;
  const int kPrefetch = p.prefetch;
  constexpr uint32_t kTmemCols = 512;  // two accumulators, at columns 0 and 256 (one of 512 columns at BN 512)
  constexpr int S = kPairStages;
  constexpr bool kWide = BN == 512 || BN == 448;
  static_assert(!kWide || (EPI == kEpiSwiGLU && KSUB == 1), "wide tiles: SwiGLU, 64-wide stages");
  constexpr int kAcc = kWide ? 1 : 2;          // accumulators in TMEM
  constexpr int kMmaN = kWide ? BN / 2 : BN;   // N of one MMA
  constexpr int kWideRows = BN / 4;            // wide tiles: gate (and up) rows of B per CTA
  constexpr uint32_t kWideUp = static_cast<uint32_t>(kWideRows) * 128u;  // up rows after the gate rows
  constexpr int kUpCol = kWide ? 256 : BN / 2;  // TMEM column of the up sums (SwiGLU)
  static_assert(kWideUp % 1024 == 0, "up rows keep the 1024-byte swizzle alignment");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  // stage st: A k-tiles at sA0 + (st*KSUB + j)*kPairABytes, B at sB0 + (st*KSUB + j)*kPairBBytes
  const uint32_t sA0 = ptx::smem_addr(smem);
  const uint32_t sB0 = sA0 + S * kPairSub * kPairABytes;
  uint8_t *bar_area = smem + S * kPairStageBytes;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (S + i); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 8 * (2 * S + 5));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 8 * (2 * S + 5) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0 or 1 within the pair
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 8);  // 4 epilogue warps in each CTA of the pair
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.n_maps_used; ++i) ptx::prefetch_tensormap(&p.maps[i]);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Weights do not come from the previous kernel: the B loads of the first
  // tile's first stages start before the grid-dependency wait, their A loads
  // after it (block tables, written by an earlier kernel, never load early).
  int pre = 0;
  if (warp == 0 && lane == 0 && p.early_b && pair < p.total_tiles) {
    const GemmProblem &pr = p.prob[find_problem(p, pair)];
    int mt0, nt;
    tile_coords<GROUPED>(pr, pair - pr.tile_begin, mt0, nt);
    for (int sgi = 0; sgi < pr.seg_count && pre < S; ++sgi) {
      const GemmSeg &sg = p.seg[pr.seg_begin + sgi];
      const bool two_b = EPI == kEpiSwiGLU || sg.b2_map >= 0;
      const int map = two_b ? (leader ? sg.b_map : sg.b2_map) : sg.b_map;
      const int row = two_b ? nt * kHalfB : nt * BN + static_cast<int>(rank) * kHalfB;
      for (int kt = 0; kt < seg_stages<KSUB>(sg) && pre < S; ++kt, ++pre) {
        const uint32_t lead_full = ptx::mapa_shared(full_bar(pre), 0);
        if (leader) ptx::mbar_arrive_expect_tx(full_bar(pre), 2 * kPairStageBytes);
        if constexpr (kWide) {
          const int wrow = nt * (BN / 2) + static_cast<int>(rank) * kWideRows;
          ptx::tma_load_2d_pair(sB0 + pre * kPairBBytes, &p.maps[sg.b_map], kt * BK, wrow, lead_full);
          ptx::tma_load_2d_pair(sB0 + pre * kPairBBytes + kWideUp, &p.maps[sg.b2_map], kt * BK, wrow, lead_full);
        } else if (p.box_kt > 1) {
          ptx::tma_load_3d_pair(sB0 + pre * kPairSub * kPairBBytes, &p.maps[map], 0, row, kt * kPairSub, lead_full);
        } else {
#pragma unroll
          for (int j = 0; j < kPairSub; ++j)
            ptx::tma_load_2d_pair(sB0 + (pre * kPairSub + j) * kPairBBytes, &p.maps[map], (kt * kPairSub + j) * BK,
                                  row, lead_full);
        }
      }
    }
  }
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // Cursor over this pair's tiles: tiles pair, pair + npairs, ...
      auto first = [&](Cursor &c) {
        const int t = live_tile<GROUPED>(p, pair, npairs);
        c.tile = t;
        c.valid = t < p.total_tiles;
        if (!c.valid) return;
        c.prob = find_problem(p, t);
        const GemmProblem &pr = p.prob[c.prob];
        tile_coords<GROUPED>(pr, t - pr.tile_begin, c.mt, c.nt);
        tile_b_origin(pr, c.mt, c.moff, c.brow);
        c.seg = c.kt = c.kt_in_tile = 0;
      };
      auto next = [&](Cursor &c) {
        const GemmProblem &pr = p.prob[c.prob];
        ++c.kt;
        ++c.kt_in_tile;
        if (c.kt < seg_stages<KSUB>(p.seg[pr.seg_begin + c.seg])) return;
        c.kt = 0;
        if (++c.seg < pr.seg_count) return;
        const int t = live_tile<GROUPED>(p, c.tile + npairs, npairs);
        c.tile = t;
        c.valid = t < p.total_tiles;
        if (!c.valid) return;
        c.prob = find_problem(p, t);
        const GemmProblem &q = p.prob[c.prob];
        tile_coords<GROUPED>(q, t - q.tile_begin, c.mt, c.nt);
        tile_b_origin(q, c.mt, c.moff, c.brow);
        c.seg = c.kt = c.kt_in_tile = 0;
      };
      // This CTA's half of B: rows of its own map and offset.
      auto b_src = [&](const Cursor &c, int &map, int &row) {
        const GemmSeg &sg = p.seg[p.prob[c.prob].seg_begin + c.seg];
        if (kWide) {  // both B matrices in each CTA (the gate map is named here)
          map = sg.b_map + c.moff;
          row = c.brow + c.nt * (BN / 2) + static_cast<int>(rank) * kWideRows;
        } else if (EPI == kEpiSwiGLU || sg.b2_map >= 0) {  // two B matrices, one half of the tile each
          map = (leader ? sg.b_map : sg.b2_map) + c.moff;
          row = c.brow + c.nt * kHalfB;
        } else {
          map = sg.b_map + c.moff;
          row = c.brow + c.nt * BN + static_cast<int>(rank) * kHalfB;
        }
      };
      Cursor ld, pf;
      first(ld);
      first(pf);
      for (int i = 0; i < kPrefetch && pf.valid; ++i) {
        int m, r;
        b_src(pf, m, r);
        if (p.box_kt > 1)
          ptx::tma_prefetch_l2_3d(&p.maps[m], 0, r, pf.kt * kPairSub);
        else
          ptx::tma_prefetch_l2_2d(&p.maps[m], pf.kt * kPairSub * BK, r);
        next(pf);
      }
      int kb = 0;
      while (ld.valid) {
        if (kPrefetch > 0 && pf.valid) {
          int m, r;
          b_src(pf, m, r);
          if (p.box_kt > 1)
            ptx::tma_prefetch_l2_3d(&p.maps[m], 0, r, pf.kt * kPairSub);
          else
            ptx::tma_prefetch_l2_2d(&p.maps[m], pf.kt * kPairSub * BK, r);
          next(pf);
        }
        const int st = kb % S;
        const uint32_t ph = (kb / S) & 1;
        if (*abort_flag) break;
        const bool early = kb < pre;  // B already in flight and the stage's barrier armed
        if (!early && !ptx::mbar_wait(empty_bar(st), ph ^ 1, p.wait_ns)) {
          record(p.status, kDevTimeoutProducer);
          *abort_flag = 1;
          break;
        }
        const uint32_t lead_full = ptx::mapa_shared(full_bar(st), 0);
        if (leader && !early) ptx::mbar_arrive_expect_tx(full_bar(st), 2 * kPairStageBytes);
        const GemmSeg &sg = p.seg[p.prob[ld.prob].seg_begin + ld.seg];
        int m, r;
        b_src(ld, m, r);
        const int a_row = ld.mt * 256 + static_cast<int>(rank) * 128;
        if constexpr (kWide) {
          const int x = ld.kt * BK;
          ptx::tma_load_2d_pair(sA0 + st * kPairABytes, &p.maps[sg.a_map], x, a_row, lead_full);
          if (!early) {
            ptx::tma_load_2d_pair(sB0 + st * kPairBBytes, &p.maps[m], x, r, lead_full);
            ptx::tma_load_2d_pair(sB0 + st * kPairBBytes + kWideUp, &p.maps[sg.b2_map + ld.moff], x, r, lead_full);
          }
        } else if (p.box_kt > 1) {
          // one copy per operand brings the stage's KSUB k-tiles (3-D maps)
          ptx::tma_load_3d_pair(sA0 + st * kPairSub * kPairABytes, &p.maps[sg.a_map], 0, a_row,
                                ld.kt * kPairSub, lead_full);
          if (!early)
            ptx::tma_load_3d_pair(sB0 + st * kPairSub * kPairBBytes, &p.maps[m], 0, r, ld.kt * kPairSub,
                                  lead_full);
        } else {
#pragma unroll
          for (int j = 0; j < kPairSub; ++j) {
            // a k-tile past the segment's end reads zeros (out-of-range TMA fill)
            const int x = (ld.kt * kPairSub + j) * BK;
            ptx::tma_load_2d_pair(sA0 + (st * kPairSub + j) * kPairABytes, &p.maps[sg.a_map], x, a_row,
                                  lead_full);
            if (!early)
              ptx::tma_load_2d_pair(sB0 + (st * kPairSub + j) * kPairBBytes, &p.maps[m], x, r, lead_full);
          }
        }
        ++kb;
        next(ld);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(256, kMmaN);
      int kb = 0;
      bool ok = true;
      for (int tile = live_tile<GROUPED>(p, pair, npairs), j = 0; ok && tile < p.total_tiles;
           tile = live_tile<GROUPED>(p, tile + npairs, npairs), ++j) {
        const int a = j % kAcc;
        const uint32_t use = static_cast<uint32_t>(j / kAcc);
        if (*abort_flag || !ptx::mbar_wait(tempty_bar(a), (use & 1) ^ 1, p.wait_ns)) {
          if (!*abort_flag) record(p.status, kDevTimeoutMma);
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(a * 256);
        const int nk = tile_stages<KSUB>(p, find_problem(p, tile));
        for (int k0 = 0; k0 < nk; ++k0, ++kb) {
          const int st = kb % S;
          const uint32_t ph = (kb / S) & 1;
          if (*abort_flag) { ok = false; break; }
          if (!ptx::mbar_wait(full_bar(st), ph, p.wait_ns)) {
            record(p.status, kDevTimeoutMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int j = 0; j < kPairSub; ++j) {
            const uint64_t ad = ptx::smem_desc_sw128(sA0 + (st * kPairSub + j) * kPairABytes);
            const uint64_t bd = ptx::smem_desc_sw128(sB0 + (st * kPairSub + j) * kPairBBytes);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              ptx::mma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc, (k0 | j | k) != 0 ? 1u : 0u);
              if constexpr (kWide) {
                const uint64_t ud = ptx::smem_desc_sw128(sB0 + (st * kPairSub + j) * kPairBBytes + kWideUp);
                ptx::mma_bf16_pair(d + static_cast<uint32_t>(kUpCol), ad + 2 * k, ud + 2 * k, idesc,
                                   (k0 | j | k) != 0 ? 1u : 0u);
              }
            }
          }
          ptx::mma_commit_pair_multicast(empty_bar(st), 0x3);
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(tfull_bar(a), 0x3);
      }
      ptx::mma_commit_pair_multicast(drain_bar, 0x1);
      if (!ptx::mbar_wait(drain_bar, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    const int q = warp & 3;
    for (int tile = live_tile<GROUPED>(p, pair, npairs), j = 0; tile < p.total_tiles;
         tile = live_tile<GROUPED>(p, tile + npairs, npairs), ++j) {
      const int a = j % kAcc;
      const uint32_t use = static_cast<uint32_t>(j / kAcc);
      const bool ready = ptx::mbar_wait(tfull_bar(a), use & 1, p.wait_ns);
      if (!ready && lane == 0) record(p.status, kDevTimeoutEpilogue);
      ptx::tc_fence_after();
      if (!__all_sync(0xffffffffu, ready && (*abort_flag == 0))) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      const GemmProblem &pr = p.prob[find_problem(p, tile)];
      int mt, nt;
      tile_coords<GROUPED>(pr, tile - pr.tile_begin, mt, nt);
      const int row = mt * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(a * 256) +
                             (static_cast<uint32_t>(q * 32) << 16);
      const uint32_t lead_tempty = ptx::mapa_shared(tempty_bar(a), 0);
      if constexpr (EPI == kEpiSwiGLU) {
        // gate sums in accumulator columns [0, BN/2), up sums in [BN/2, BN)
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(pr.out);
        constexpr int kFull = (BN / 2) / 32 * 32;  // columns handled 32 at a time
#pragma unroll 1
        for (int c = 0; c < kFull; c += 32) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32cols(tbase + c, g);
          ptx::tmem_ld_32cols(tbase + kUpCol + c, u);
          ptx::tmem_ld_wait();
          ptx::tmem_regs_ready(g);
          ptx::tmem_regs_ready(u);
          if (c + 32 == BN / 2) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_remote(lead_tempty);
          }
          float h[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) h[jj] = silu(__uint_as_float(g[jj])) * __uint_as_float(u[jj]);
          if (row < pr.m) store_bf16_row32(out, pr.ldc, row, nt * kOutCols + c, pr.n, h);
        }
        if constexpr (BN / 2 > kFull) {
          static_assert(BN / 2 - kFull == 16, "a 16-column tail");
          uint32_t g[16], u[16];
          ptx::tmem_ld_16cols(tbase + kFull, g);
          ptx::tmem_ld_16cols(tbase + kUpCol + kFull, u);
          ptx::tmem_ld_wait();
          ptx::tmem_regs_ready(g);
          ptx::tmem_regs_ready(u);
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_remote(lead_tempty);
          float h[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) h[jj] = silu(__uint_as_float(g[jj])) * __uint_as_float(u[jj]);
          if (row < pr.m) store_bf16_row16(out, pr.ldc, row, nt * kOutCols + kFull, pr.n, h);
        }
      } else {
        static_assert(BN % 32 == 0, "32-column epilogue chunks");
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32cols(tbase + c, v);
          ptx::tmem_ld_wait();
          if (c + 32 == BN) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_remote(lead_tempty);
          }
          float f[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) f[jj] = __uint_as_float(v[jj]);
          if (row < pr.m) {
            if constexpr (EPI == kEpiF32) {
              store_f32_row32(static_cast<float *>(pr.out), pr.ldc, row, nt * kOutCols + c, pr.n, f);
            } else if (EPI == kEpiBF16 && BN == 256 && pr.out2 != nullptr) {
              // two outputs: accumulator columns [0, 128) to out, [128, 256) to out2
              const bool second = c >= BN / 2;
              store_bf16_row32(static_cast<__nv_bfloat16 *>(second ? pr.out2 : pr.out), second ? pr.ldc2 : pr.ldc,
                               row, nt * (BN / 2) + (second ? c - BN / 2 : c), pr.n, f);
            } else {
              store_bf16_row32(static_cast<__nv_bfloat16 *>(pr.out), pr.ldc, row, nt * kOutCols + c,
                               pr.n, f);
            }
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // A wait ran out somewhere in the pair: give copies already in flight (into
    // either CTA) time to land before the pair's shared memory goes away.
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  ptx::cluster_sync();  // neither CTA leaves while the other may still touch its smem
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Ring-folding row-parallel pair kernel: the row-parallel GEMM and the ring
// all-reduce of its partials in one pass (mlxcel manual "텐서 병렬화", 통신 패턴:
// the reduced chunk c is the fold x_{c+1} + x_{c+2} + ... + x_c of the ranks'
// partials, indices mod N). One problem holds the N ranks' K slices as
// segments. Each 256 x BN tile lies inside one ring chunk c; its SM pair runs
// the segments in that chunk's fold order, rank c+1 first, each from a zeroed
// accumulator, so every per-rank partial has exactly the bits the GEMM without
// a combine writes (same tile width, same k-stage sequence). The epilogue adds
// each partial to the running sum in TMEM in the same order as the one-pass
// ring kernel adds them, then stores the sum to every rank's output (or to
// y[0] alone) with TMA stores. The result is bit-identical to the GEMM
// followed by the ring, and no partial ever reaches global memory.
//
// TMEM holds two 256-column regions. Tile jt of this pair keeps its running
// sum in region jt & 1 (the first partial lands there directly) and receives
// the later partials in the other region; after the last add the sum is
// written back to its region, the partial's region goes back to the MMA warp
// (it becomes the next tile's sum region) and the stores drain from the sum
// region while the next tile's first partial is computed.
// ---------------------------------------------------------------------------
constexpr int kRingStagingBytes = 4 * 2 * 32 * 128;  // 4 epilogue warps x 2 buffers x [32 rows x 128 B]

template <int KSUB, int BN>
struct PairRingCfg {
  using PC = PairCfg<KSUB, BN>;
  static constexpr int kSmem = 1024 + PC::kStages * PC::kStageBytes + kRingStagingBytes + 256;
  static_assert(kSmem <= kSmemLimit, "stages, staging buffers and barriers fit in shared memory");
  static_assert(PC::kStageBytes % 1024 == 0, "staging buffers keep the 1024-byte swizzle alignment");
};

template <int KSUB, int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm_bf16_pair_ring(const __grid_constant__ GemmParams p) {
  using PC = PairCfg<KSUB, BN>;
  constexpr int S = PC::kStages;
  constexpr int kHalfB = PC::kBRows;  // B rows per CTA
  constexpr int kPairBBytes = PC::kBBytes;
  constexpr uint32_t kTmemCols = 512;  // two regions, at columns 0 and 256
  constexpr int kChunks = BN / 32;
  static_assert(BN % 32 == 0, "32-column epilogue chunks");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sA0 = ptx::smem_addr(smem);
  const uint32_t sB0 = sA0 + S * KSUB * kPairABytes;
  uint8_t *staging = smem + S * PC::kStageBytes;
  uint8_t *bar_area = staging + kRingStagingBytes;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (S + i); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 8 * (2 * S + 5));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 8 * (2 * S + 5) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = ptx::cluster_ctarank();  // 0 or 1 within the SM pair
  const bool leader = crank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const GemmProblem &pr = p.prob[0];
  const int nrank = pr.seg_count;
  // The tile's ring chunk, and with it the rank whose partial comes s-th.
  auto fold_rank = [&](int mt, int s) { return ((mt * 256) / p.ring_rows + 1 + s) % nrank; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 8);  // 4 epilogue warps in each CTA of the pair
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.n_maps_used; ++i) ptx::prefetch_tensormap(&p.maps[i]);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Weights do not come from the previous kernel: the B loads of the first
  // tile's first stages start before the grid-dependency wait.
  int pre = 0;
  if (warp == 0 && lane == 0 && p.early_b && pair < p.total_tiles) {
    int mt, nt;
    tile_coords<true>(pr, pair, mt, nt);
    const int b_row = nt * BN + static_cast<int>(crank) * kHalfB;
    for (int s = 0; s < nrank && pre < S; ++s) {
      const GemmSeg &sg = p.seg[pr.seg_begin + fold_rank(mt, s)];
      for (int kt = 0; kt < seg_stages<KSUB>(sg) && pre < S; ++kt, ++pre) {
        const uint32_t lead_full = ptx::mapa_shared(full_bar(pre), 0);
        if (leader) ptx::mbar_arrive_expect_tx(full_bar(pre), 2 * PC::kStageBytes);
        if (p.box_kt > 1) {
          ptx::tma_load_3d_pair(sB0 + pre * KSUB * kPairBBytes, &p.maps[sg.b_map], 0, b_row, kt * KSUB, lead_full);
        } else {
#pragma unroll
          for (int j = 0; j < KSUB; ++j)
            ptx::tma_load_2d_pair(sB0 + (pre * KSUB + j) * kPairBBytes, &p.maps[sg.b_map], (kt * KSUB + j) * BK,
                                  b_row, lead_full);
        }
      }
    }
  }
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      int kb = 0;
      bool go = true;
      for (int t = pair; go && t < p.total_tiles; t += npairs) {
        int mt, nt;
        tile_coords<true>(pr, t, mt, nt);
        const int a_row = mt * 256 + static_cast<int>(crank) * 128;
        const int b_row = nt * BN + static_cast<int>(crank) * kHalfB;
        for (int s = 0; go && s < nrank; ++s) {
          const GemmSeg &sg = p.seg[pr.seg_begin + fold_rank(mt, s)];
          const int nst = seg_stages<KSUB>(sg);
          for (int kt = 0; kt < nst; ++kt, ++kb) {
            const int st = kb % S;
            const uint32_t ph = (kb / S) & 1;
            if (*abort_flag) { go = false; break; }
            const bool early = kb < pre;  // B already in flight and the stage's barrier armed
            if (!early && !ptx::mbar_wait(empty_bar(st), ph ^ 1, p.wait_ns)) {
              record(p.status, kDevTimeoutProducer);
              *abort_flag = 1;
              go = false;
              break;
            }
            const uint32_t lead_full = ptx::mapa_shared(full_bar(st), 0);
            if (leader && !early) ptx::mbar_arrive_expect_tx(full_bar(st), 2 * PC::kStageBytes);
            if (p.box_kt > 1) {
              ptx::tma_load_3d_pair(sA0 + st * KSUB * kPairABytes, &p.maps[sg.a_map], 0, a_row, kt * KSUB,
                                    lead_full);
              if (!early)
                ptx::tma_load_3d_pair(sB0 + st * KSUB * kPairBBytes, &p.maps[sg.b_map], 0, b_row, kt * KSUB,
                                      lead_full);
            } else {
#pragma unroll
              for (int j = 0; j < KSUB; ++j) {
                const int x = (kt * KSUB + j) * BK;  // past the segment's K: zero fill
                ptx::tma_load_2d_pair(sA0 + (st * KSUB + j) * kPairABytes, &p.maps[sg.a_map], x, a_row,
                                      lead_full);
                if (!early)
                  ptx::tma_load_2d_pair(sB0 + (st * KSUB + j) * kPairBBytes, &p.maps[sg.b_map], x, b_row,
                                        lead_full);
              }
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(256, BN);
      int kb = 0;
      uint32_t taken0 = 0, taken1 = 0;  // acquisitions of each TMEM region so far
      bool ok = true;
      for (int t = pair, jt = 0; ok && t < p.total_tiles; t += npairs, ++jt) {
        int mt, nt;
        tile_coords<true>(pr, t, mt, nt);
        for (int s = 0; ok && s < nrank; ++s) {
          const int reg = s == 0 ? (jt & 1) : ((jt & 1) ^ 1);
          uint32_t &taken = reg ? taken1 : taken0;
          if (*abort_flag || !ptx::mbar_wait(tempty_bar(reg), (taken & 1) ^ 1, p.wait_ns)) {
            if (!*abort_flag) record(p.status, kDevTimeoutMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          ++taken;
          ptx::tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(reg * 256);
          const int nst = seg_stages<KSUB>(p.seg[pr.seg_begin + fold_rank(mt, s)]);
          for (int k0 = 0; k0 < nst; ++k0, ++kb) {
            const int st = kb % S;
            const uint32_t ph = (kb / S) & 1;
            if (*abort_flag) { ok = false; break; }
            if (!ptx::mbar_wait(full_bar(st), ph, p.wait_ns)) {
              record(p.status, kDevTimeoutMma);
              *abort_flag = 1;
              ok = false;
              break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
              const uint64_t ad = ptx::smem_desc_sw128(sA0 + (st * KSUB + j) * kPairABytes);
              const uint64_t bd = ptx::smem_desc_sw128(sB0 + (st * KSUB + j) * kPairBBytes);
#pragma unroll
              for (int k = 0; k < BK / UMMA_K; ++k)
                ptx::mma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc, (k0 | j | k) != 0 ? 1u : 0u);
            }
            ptx::mma_commit_pair_multicast(empty_bar(st), 0x3);
          }
          if (!ok) break;
          ptx::mma_commit_pair_multicast(tfull_bar(reg), 0x3);
        }
      }
      ptx::mma_commit_pair_multicast(drain_bar, 0x1);
      if (!ptx::mbar_wait(drain_bar, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    // ---- epilogue: warp w reads TMEM lanes [32*(w%4), 32*(w%4)+32): rows of this CTA ----
    const int q = warp & 3;
    uint8_t *mine = staging + q * (2 * 32 * 128);  // this warp's two [32 x 128 B] buffers
    uint32_t seen0 = 0, seen1 = 0;  // completions of each region consumed so far
    const uint32_t lead_tempty0 = ptx::mapa_shared(tempty_bar(0), 0);
    const uint32_t lead_tempty1 = ptx::mapa_shared(tempty_bar(1), 0);
    int groups = 0;  // bulk store groups this warp has committed (lane 0 issues them)
    bool alive = true;
    auto await = [&](int reg) {
      uint32_t &seen = reg ? seen1 : seen0;
      const bool ready = ptx::mbar_wait(tfull_bar(reg), seen & 1, p.wait_ns);
      ++seen;
      if (!ready && lane == 0) record(p.status, kDevTimeoutEpilogue);
      ptx::tc_fence_after();
      if (!__all_sync(0xffffffffu, ready && (*abort_flag == 0))) {
        if (lane == 0) *abort_flag = 1;
        alive = false;
      }
      return alive;
    };
    for (int t = pair, jt = 0; alive && t < p.total_tiles; t += npairs, ++jt) {
      int mt, nt;
      tile_coords<true>(pr, t, mt, nt);
      const int rs = jt & 1, ra = rs ^ 1;
      const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
      const uint32_t tsum = tmem_base + static_cast<uint32_t>(rs * 256) + lane_off;
      const uint32_t tacc = tmem_base + static_cast<uint32_t>(ra * 256) + lane_off;
      if (!await(rs)) break;  // the first partial of the fold, in the sum region
      for (int s = 1; s < nrank; ++s) {
        if (!await(ra)) break;
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          uint32_t a[32], b[32];
          ptx::tmem_ld_32cols(tsum + c * 32, a);
          ptx::tmem_ld_32cols(tacc + c * 32, b);
          ptx::tmem_ld_wait();
          ptx::tmem_regs_ready(a);
          ptx::tmem_regs_ready(b);
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = __float_as_uint(__uint_as_float(a[j]) + __uint_as_float(b[j]));
          ptx::tmem_st_32cols(tsum + c * 32, a);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_remote(ra ? lead_tempty1 : lead_tempty0);
      }
      if (!alive) break;
      // The reduced rows [y0, y0 + 32) x columns [nt*BN, nt*BN + BN): staged 32
      // columns at a time (128-byte swizzle) and stored to every output.
      const int y0 = mt * 256 + static_cast<int>(crank) * 128 + q * 32;
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32cols(tsum + c * 32, v);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        if (c + 1 == kChunks) {  // the sum region is read: hand it back to the MMA warp
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_remote(rs ? lead_tempty1 : lead_tempty0);
        }
        uint8_t *buf = mine + (groups & 1) * (32 * 128);
        if (groups >= 2) {  // the stores that read this buffer two chunks ago are done reading
          if (lane == 0) ptx::bulk_wait_group_read<1>();
          __syncwarp();
        }
        float4 *row = reinterpret_cast<float4 *>(buf + lane * 128);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          row[u ^ (lane & 7)] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                            __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int r = 0; r < p.ring_copies; ++r)
            ptx::tma_store_2d(&p.maps[p.ring_out + r], ptx::smem_addr(buf), nt * BN + c * 32, y0);
          ptx::bulk_commit_group();
        }
        ++groups;
      }
    }
    if (lane == 0) ptx::bulk_wait_group_all();  // every store has landed before the CTA leaves
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  ptx::cluster_sync();  // neither CTA leaves while the other may still touch its smem
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Split-K cluster kernel for problems with too few output tiles to fill the
// GPU (small-token row-parallel layers, decode). A cluster computes one tile:
// CTA ranks are (split, member), member = the M-half for SM pairs. Split s
// accumulates k-stages [s*ns/S, (s+1)*ns/S) of the tile in TMEM. After a
// cluster barrier each split owns a slice of the tile's rows: every CTA stages
// its fp32 accumulator in its own shared memory and sends each owner that
// owner's rows with one bulk copy into the owner's shared memory (DSMEM). The
// owner adds the partials in split order 0, 1, ..., S-1 and stores. The sum
// order is fixed, so the result does not depend on timing; no global workspace
// is used. When the shared memory cannot hold the staged tile and the received
// rows together, rows are pushed from registers with st.async instead.
// ---------------------------------------------------------------------------
// Stores one 16-byte unit (4 fp32 sums g, and for SwiGLU the matching up sums u)
// of output row `grow` at unit c4 of tile column block nt, with the epilogue
// transform of EPI; columns past the problem's n are dropped.
struct OutDesc {
  void *out;
  long long ldc;
  int n;
};

template <int EPI, int BN>
__device__ __forceinline__ void store_unit(const OutDesc &pr, int grow, int nt, int c4, float4 g, float4 u) {
  const float f[4] = {g.x, g.y, g.z, g.w};
  if (EPI == kEpiF32) {
    const int col = nt * BN + c4 * 4;
    float *dst = static_cast<float *>(pr.out) + static_cast<long long>(grow) * pr.ldc + col;
    if (col + 4 <= pr.n) {
      *reinterpret_cast<float4 *>(dst) = g;
    } else {
      for (int e = 0; e < 4; ++e)
        if (col + e < pr.n) dst[e] = f[e];
    }
    return;
  }
  float o[4];
  int col;
  if (EPI == kEpiSwiGLU) {
    const float uu[4] = {u.x, u.y, u.z, u.w};
    for (int e = 0; e < 4; ++e) o[e] = silu(f[e]) * uu[e];
    col = nt * (BN / 2) + c4 * 4;
  } else {
    for (int e = 0; e < 4; ++e) o[e] = f[e];
    col = nt * BN + c4 * 4;
  }
  __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(pr.out) + static_cast<long long>(grow) * pr.ldc + col;
  if (col + 4 <= pr.n) {
    __nv_bfloat162 h0 = __floats2bfloat162_rn(o[0], o[1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(o[2], o[3]);
    uint2 w;
    memcpy(&w.x, &h0, 4);
    memcpy(&w.y, &h1, 4);
    *reinterpret_cast<uint2 *>(dst) = w;
  } else {
    for (int e = 0; e < 4; ++e)
      if (col + e < pr.n) dst[e] = __float2bfloat16_rn(o[e]);
  }
}

template <bool PAIR, int BN>
struct SplitCfg {
  static constexpr int kSub = PAIR ? 2 : 1;  // 64-wide k-tiles per stage
  static constexpr int kABytes = 128 * BK * 2;
  static constexpr int kBRows = PAIR ? BN / 2 : BN;  // B rows per CTA per k-tile
  static constexpr int kBBytes = kBRows * BK * 2;
  static constexpr int kStageBytes = kSub * (kABytes + kBBytes);
  static constexpr int kStages = (6 * 32768) / kStageBytes;  // 192 KB of stages
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 256;
};

template <bool PAIR, int EPI, int BN>
__global__ void __launch_bounds__(kThreads, 1) k_gemm_bf16_splitk(const __grid_constant__ GemmParams p) {
  using C = SplitCfg<PAIR, BN>;
  static_assert(!PAIR || BN == 256 || BN == 128, "SM pairs run 256- or 128-column tiles");
  constexpr int KS = C::kSub;
  // SM pairs: fixed stages of 128-row A k-tiles. Single CTAs: an A k-tile holds
  // the a_rows rows loaded and the stage count comes from the host.
  const int S = PAIR ? C::kStages : p.one_stages;
  const uint32_t kAT = PAIR ? static_cast<uint32_t>(C::kABytes) : static_cast<uint32_t>(p.a_rows) * 128u;
  const uint32_t kStageArea = static_cast<uint32_t>(S * KS) * (kAT + C::kBBytes);
  constexpr uint32_t kTmemCols = BN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sA0 = ptx::smem_addr(smem);
  const uint32_t sB0 = sA0 + static_cast<uint32_t>(S * KS) * kAT;
  uint8_t *bar_area = smem + kStageArea;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (S + i); };
  const uint32_t accum_bar = bar0 + 8u * (2 * S);
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 1);
  const uint32_t recv_bar = bar0 + 8u * (2 * S + 2);
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 8 * (2 * S + 3));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 8 * (2 * S + 3) + 4);
  // Receive buffer, reusing the stage ring once every CTA of the cluster has
  // finished its main loop: recv[t][rl] holds split t's partial of owned row rl
  // (BN fp32, kRowBytes). Unit c4 of a row sits at ((c4 ^ (rl & 7)) * 16) so that
  // the row-wise writes and the column-wise reads are free of bank conflicts.
  const uint32_t red0 = sA0;
  constexpr int kRowBytes = BN * 4;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = ptx::cluster_ctarank();
  const int csize = static_cast<int>(ptx::cluster_nctarank());
  const int member = PAIR ? static_cast<int>(crank & 1) : 0;
  const int split = PAIR ? static_cast<int>(crank >> 1) : static_cast<int>(crank);
  const int nsplit = PAIR ? csize / 2 : csize;
  const uint32_t lead = PAIR ? (crank & ~1u) : crank;  // CTA that issues this pair's MMAs
  const bool issuer = !PAIR || member == 0;
  const int tile = blockIdx.x / csize;

  const int pi = find_problem(p, tile);
  const GemmProblem &pr = p.prob[pi];
  int mt, nt;
  tile_coords<false>(pr, tile - pr.tile_begin, mt, nt);
  // Ring folding (ring_rows > 0): split s is segment (rank) s, whole. Otherwise
  // the problem's stages are cut into nsplit near-equal ranges.
  const bool ring = p.ring_rows > 0;
  int k_begin = 0, k_end = 0;
  {
    int ns = 0;
    for (int q = 0; q < pr.seg_count; ++q) {
      const int n = (p.seg[pr.seg_begin + q].k_tiles + KS - 1) / KS;
      if (ring && q == split) {
        k_begin = ns;
        k_end = ns + n;
      }
      ns += n;
    }
    if (!ring) {
      k_begin = (split * ns) / nsplit;
      k_end = ((split + 1) * ns) / nsplit;
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), 1);
    }
    ptx::mbar_init(accum_bar, 1);
    ptx::mbar_init(drain_bar, 1);
    ptx::mbar_init(recv_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int q = 0; q < pr.seg_count; ++q) {
      const GemmSeg &sg = p.seg[pr.seg_begin + q];
      ptx::prefetch_tensormap(&p.maps[sg.a_map]);
      ptx::prefetch_tensormap(&p.maps[sg.b_map]);
      if (EPI == kEpiSwiGLU) ptx::prefetch_tensormap(&p.maps[sg.b2_map]);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR)
      ptx::tmem_alloc_pair(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    else
      ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    if constexpr (PAIR)
      ptx::tmem_relinquish_pair();
    else
      ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  // The producer's loads of one stage: A (activations, which may come from the
  // previous kernel) and B (weights, which do not).
  const uint32_t stage_tx = PAIR ? 2 * C::kStageBytes : static_cast<uint32_t>(KS * (p.a_rows * 128 + C::kBBytes));
  const int a_row = PAIR ? mt * 256 + member * 128 : mt * 128;
  auto load_a = [&](int st, const GemmSeg &sg, int kt, uint32_t fb) {
    if (PAIR && p.box_kt > 1) {
      ptx::tma_load_3d_pair(sA0 + st * KS * kAT, &p.maps[sg.a_map], 0, a_row, kt * KS, fb);  // past K: zero fill
      return;
    }
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      const int x = (kt * KS + j) * BK;  // past the segment's K: zero fill
      const uint32_t da = sA0 + (st * KS + j) * kAT;
      if constexpr (PAIR)
        ptx::tma_load_2d_pair(da, &p.maps[sg.a_map], x, a_row, fb);
      else
        ptx::tma_load_2d(da, &p.maps[sg.a_map], x, a_row, fb);
    }
  };
  auto load_b = [&](int st, const GemmSeg &sg, int kt, uint32_t fb) {
    if (PAIR && p.box_kt > 1) {
      const int z = kt * KS;
      if (EPI == kEpiSwiGLU)
        ptx::tma_load_3d_pair(sB0 + st * KS * C::kBBytes, &p.maps[member == 0 ? sg.b_map : sg.b2_map], 0,
                              nt * (BN / 2), z, fb);
      else
        ptx::tma_load_3d_pair(sB0 + st * KS * C::kBBytes, &p.maps[sg.b_map], 0, nt * BN + member * (BN / 2), z,
                              fb);
      return;
    }
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      const int x = (kt * KS + j) * BK;
      const uint32_t db = sB0 + (st * KS + j) * C::kBBytes;
      if constexpr (PAIR) {
        if (EPI == kEpiSwiGLU)
          ptx::tma_load_2d_pair(db, &p.maps[member == 0 ? sg.b_map : sg.b2_map], x, nt * (BN / 2), fb);
        else
          ptx::tma_load_2d_pair(db, &p.maps[sg.b_map], x, nt * BN + member * (BN / 2), fb);
      } else {
        if (EPI == kEpiSwiGLU) {
          ptx::tma_load_2d(db, &p.maps[sg.b_map], x, nt * (BN / 2), fb);
          ptx::tma_load_2d(db + (BN / 2) * 128, &p.maps[sg.b2_map], x, nt * (BN / 2), fb);
        } else {
          ptx::tma_load_2d(db, &p.maps[sg.b_map], x, nt * BN, fb);
        }
      }
    }
  };
  // (segment, stage within the segment) of this split's first stage
  int seg0 = 0, kt0 = k_begin;
  while (seg0 < pr.seg_count) {
    const int n = (p.seg[pr.seg_begin + seg0].k_tiles + KS - 1) / KS;
    if (kt0 < n) break;
    kt0 -= n;
    ++seg0;
  }
  // Weights do not come from the previous kernel: the B loads of the first
  // stages start before the grid-dependency wait, their A loads after it.
  int pre = 0;
  if (warp == 0 && lane == 0 && p.early_b) {
    int seg = seg0, kt = kt0;
    for (; pre < S && pre < k_end - k_begin; ++pre) {
      const GemmSeg &sg = p.seg[pr.seg_begin + seg];
      if (issuer) ptx::mbar_arrive_expect_tx(full_bar(pre), stage_tx);
      load_b(pre, sg, kt, PAIR ? ptx::mapa_shared(full_bar(pre), lead) : full_bar(pre));
      if (++kt == (sg.k_tiles + KS - 1) / KS) {
        kt = 0;
        ++seg;
      }
    }
  }
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      int seg = seg0, kt = kt0;
      for (int kb = 0; kb < k_end - k_begin; ++kb) {
        const int st = kb % S;
        const uint32_t ph = (kb / S) & 1;
        if (*abort_flag) break;
        const GemmSeg &sg = p.seg[pr.seg_begin + seg];
        const uint32_t fb = PAIR ? ptx::mapa_shared(full_bar(st), lead) : full_bar(st);
        if (kb >= pre) {
          if (!ptx::mbar_wait(empty_bar(st), ph ^ 1, p.wait_ns)) {
            record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            break;
          }
          if (issuer) ptx::mbar_arrive_expect_tx(full_bar(st), stage_tx);
          load_b(st, sg, kt, fb);
        }
        load_a(st, sg, kt, fb);
        if (++kt == (sg.k_tiles + KS - 1) / KS) {
          kt = 0;
          ++seg;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && issuer) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(PAIR ? 256 : 128, BN);
      const uint16_t mask = static_cast<uint16_t>(3u << lead);
      for (int kb = 0; kb < k_end - k_begin; ++kb) {
        const int st = kb % S;
        const uint32_t ph = (kb / S) & 1;
        if (*abort_flag) break;
        if (!ptx::mbar_wait(full_bar(st), ph, p.wait_ns)) {
          record(p.status, kDevTimeoutMma);
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          const uint64_t ad = ptx::smem_desc_sw128(sA0 + (st * KS + j) * kAT);
          const uint64_t bd = ptx::smem_desc_sw128(sB0 + (st * KS + j) * C::kBBytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint32_t acc = (kb | j | k) != 0 ? 1u : 0u;
            if constexpr (PAIR)
              ptx::mma_bf16_pair(tmem_d, ad + 2 * k, bd + 2 * k, idesc, acc);
            else
              ptx::mma_bf16(tmem_d, ad + 2 * k, bd + 2 * k, idesc, acc);
          }
        }
        if constexpr (PAIR)
          ptx::mma_commit_pair_multicast(empty_bar(st), mask);
        else
          ptx::mma_commit(empty_bar(st));
      }
      if constexpr (PAIR) {
        ptx::mma_commit_pair_multicast(accum_bar, mask);
        ptx::mma_commit_pair_multicast(drain_bar, static_cast<uint16_t>(1u << lead));
      } else {
        ptx::mma_commit(accum_bar);
        ptx::mma_commit(drain_bar);
      }
      if (!ptx::mbar_wait(drain_bar, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    const bool ready = ptx::mbar_wait(accum_bar, 0, p.wait_ns);
    if (!ready && lane == 0) record(p.status, kDevTimeoutEpilogue);
    if (!__all_sync(0xffffffffu, ready)) {
      if (lane == 0) *abort_flag = 1;
    }
  }

  // Every CTA of the cluster has finished its main loop (and its stage ring is
  // idle) before any partial is pushed into another CTA's shared memory.
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();

  const int rows_per = 128 / nsplit;  // rows of this member's half owned by each split
  // Bulk path: stage the whole accumulator in own shared memory, then send each
  // owner its contiguous block of rows with one bulk copy; the owner receives the
  // other splits' blocks after its own staging area. Needs room for both.
  const bool bulk = static_cast<uint32_t>((128 + (nsplit - 1) * rows_per) * kRowBytes) <= kStageArea;
  if (bulk) {
    const uint32_t recv0 = red0 + 128u * kRowBytes;  // slot j: rows_per rows of split (j < split ? j : j + 1)
    if (warp >= 2) {
      const int q = warp & 3;
      const int tid = threadIdx.x - 64;
      if (tid == 0)
        ptx::mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((nsplit - 1) * rows_per * kRowBytes));
      if (*abort_flag == 0) {
        const int r = q * 32 + lane;
        const uint32_t tbase = tmem_d + (static_cast<uint32_t>(q * 32) << 16);
        const bool has_work = k_end > k_begin;
        float4 *row = reinterpret_cast<float4 *>(smem + r * kRowBytes);
        // 128 columns per wait: four TMEM loads in flight instead of one
#pragma unroll 1
        for (int c = 0; c < BN; c += 128) {
          uint32_t v[4][32];
#pragma unroll
          for (int h = 0; h < 4; ++h) ptx::tmem_ld_32cols(tbase + c + 32 * h, v[h]);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 4; ++h) ptx::tmem_regs_ready(v[h]);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int c4 = (c + 32 * h) / 4 + j;
              row[c4 ^ (r & 7)] =
                  has_work ? make_float4(__uint_as_float(v[h][4 * j]), __uint_as_float(v[h][4 * j + 1]),
                                         __uint_as_float(v[h][4 * j + 2]), __uint_as_float(v[h][4 * j + 3]))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
      }
      ptx::fence_proxy_async_smem();  // staged rows visible to the bulk-copy engine
      ptx::named_barrier(1, 128);
      if (tid < nsplit && tid != split && *abort_flag == 0) {
        const int o = tid;  // destination split
        const uint32_t dst_rank = PAIR ? static_cast<uint32_t>(2 * o + member) : static_cast<uint32_t>(o);
        const int slot = split < o ? split : split - 1;
        ptx::bulk_copy_to_cluster(
            ptx::mapa_shared(recv0 + static_cast<uint32_t>(slot * rows_per * kRowBytes), dst_rank),
            red0 + static_cast<uint32_t>(o * rows_per * kRowBytes),
            static_cast<uint32_t>(rows_per * kRowBytes), ptx::mapa_shared(recv_bar, dst_rank));
      }
    }
    // All six warps (the producer and MMA warps are idle by now) wait for the
    // other splits' rows and share the summation and the stores.
    {
      const int tid = threadIdx.x;
      const bool got = ptx::mbar_wait(recv_bar, 0, p.wait_ns);
      if (!got && tid == 0) record(p.status, kDevTimeoutEpilogue);
      if (got && *abort_flag == 0) {
        // Sum the owned rows over splits in order 0..S-1. Problem fields live in
        // registers; each thread takes kBatch units and issues every shared load
        // of a split before adding, so loads overlap.
        const int lo = split * rows_per;
        const int row0 = PAIR ? mt * 256 + member * 128 : mt * 128;
        const OutDesc od{pr.out, pr.ldc, pr.n};
        // ring folding: the tile's chunk c = row / ring_rows is summed in the ring's
        // order c+1, c+2, ..., c (split t = rank t); otherwise splits 0..S-1
        const int first = ring ? ((row0 + lo) / p.ring_rows + 1) % nsplit : 0;
        const int m_rows = pr.m;
        constexpr int kUnits = (EPI == kEpiSwiGLU) ? BN / 8 : BN / 4;
        constexpr int kBatch = (EPI == kEpiSwiGLU) ? 4 : 8;
        constexpr int kMaxSplit = PAIR ? 4 : 8;
        const int total = rows_per * kUnits;
        for (int base = tid; base < total; base += kThreads * kBatch) {
          float4 g[kBatch], u[kBatch];
#pragma unroll
          for (int t = 0; t < kMaxSplit; ++t) {
            if (t >= nsplit) break;
            float4 vg[kBatch], vu[kBatch];
            const int ts = ring ? (first + t) % nsplit : t;
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
              const int idx = base + b * kThreads < total ? base + b * kThreads : base;
              const int rl = idx / kUnits;
              const int c4 = idx % kUnits;
              const int prow = (ts == split) ? lo + rl : 128 + (ts < split ? ts : ts - 1) * rows_per + rl;
              const uint32_t rowa = red0 + static_cast<uint32_t>(prow * kRowBytes);
              vg[b] = ptx::ld_shared_f4(rowa + static_cast<uint32_t>(((c4 ^ (rl & 7)) * 16)));
              if (EPI == kEpiSwiGLU)
                vu[b] = ptx::ld_shared_f4(rowa + static_cast<uint32_t>((((c4 + BN / 8) ^ (rl & 7)) * 16)));
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
              if (t == 0) {
                g[b] = vg[b];
                if (EPI == kEpiSwiGLU) u[b] = vu[b];
              } else {
                g[b].x += vg[b].x; g[b].y += vg[b].y; g[b].z += vg[b].z; g[b].w += vg[b].w;
                if (EPI == kEpiSwiGLU) {
                  u[b].x += vu[b].x; u[b].y += vu[b].y; u[b].z += vu[b].z; u[b].w += vu[b].w;
                }
              }
            }
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int idx = base + b * kThreads;
            if (idx >= total) break;
            const int rl = idx / kUnits;
            const int grow = row0 + lo + rl;
            if (grow >= m_rows) continue;
            if (ring) {
              for (int c = 0; c < p.ring_copies; ++c)
                store_unit<EPI, BN>(OutDesc{p.ring_dst[c], pr.ldc, pr.n}, grow, nt, idx % kUnits, g[b], u[b]);
            } else {
              store_unit<EPI, BN>(od, grow, nt, idx % kUnits, g[b], u[b]);
            }
          }
        }
      }
    }
    // Outgoing bulk copies read this CTA's staging area until the owner's barrier
    // has seen their bytes: nobody leaves before every owner has received.
    ptx::cluster_sync();
  } else {
    if (warp >= 2) {
      const int q = warp & 3;
      const int tid = threadIdx.x - 64;
      if (tid == 0)
        ptx::mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((nsplit - 1) * rows_per * kRowBytes));
      // push: row r of this CTA's accumulator goes to the split that owns it
      if (*abort_flag == 0) {
        const int r = q * 32 + lane;
        const int owner = r / rows_per;
        const int rl = r - owner * rows_per;
        const uint32_t dst_rank = PAIR ? static_cast<uint32_t>(2 * owner + member) : static_cast<uint32_t>(owner);
        const uint32_t row_off = red0 + static_cast<uint32_t>((split * rows_per + rl) * kRowBytes);
        const bool local_row = owner == split;
        const uint32_t rbar = ptx::mapa_shared(recv_bar, dst_rank);
        const uint32_t tbase = tmem_d + (static_cast<uint32_t>(q * 32) << 16);
        const bool has_work = k_end > k_begin;
  #pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32cols(tbase + c, v);
          ptx::tmem_ld_wait();
  #pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c4 = c / 4 + j;
            const float4 f = has_work ? make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                    __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            const uint32_t a = row_off + static_cast<uint32_t>((c4 ^ (rl & 7)) * 16);
            if (local_row)
              *reinterpret_cast<float4 *>(smem + (a - red0)) = f;
            else
              ptx::st_async_f4(ptx::mapa_shared(a, dst_rank), f, rbar);
          }
        }
      }
      // wait for the other splits' partials of the rows this CTA owns
      const bool got = ptx::mbar_wait(recv_bar, 0, p.wait_ns);
      if (!got && lane == 0) record(p.status, kDevTimeoutEpilogue);
      ptx::named_barrier(1, 128);  // local partial writes of all four epilogue warps
      if (got && *abort_flag == 0) {
        // rows [lo, lo + rows_per) of this member's half, summed over splits in order
        // 0..S-1, or in the ring order of the tile's chunk when folding
        const int lo = split * rows_per;
        const int row0 = PAIR ? mt * 256 + member * 128 : mt * 128;
        const int first = ring ? ((row0 + lo) / p.ring_rows + 1) % nsplit : 0;
        constexpr int kUnits = (EPI == kEpiSwiGLU) ? BN / 8 : BN / 4;  // output 16-byte units per row
        const int total = rows_per * kUnits;
        for (int idx = tid; idx < total; idx += 128) {
          const int rl = idx / kUnits;
          const int c4 = idx % kUnits;
          const int grow = row0 + lo + rl;
          float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
          for (int t = 0; t < nsplit; ++t) {
            const int ts = ring ? (first + t) % nsplit : t;
            const uint8_t *rowp = smem + (ts * rows_per + rl) * kRowBytes;
            const float4 vg = *reinterpret_cast<const float4 *>(rowp + ((c4 ^ (rl & 7)) * 16));
            if (t == 0) {
              g = vg;
            } else {
              g.x += vg.x; g.y += vg.y; g.z += vg.z; g.w += vg.w;
            }
            if (EPI == kEpiSwiGLU) {
              const float4 vu = *reinterpret_cast<const float4 *>(rowp + (((c4 + BN / 8) ^ (rl & 7)) * 16));
              if (t == 0) {
                u = vu;
              } else {
                u.x += vu.x; u.y += vu.y; u.z += vu.z; u.w += vu.w;
              }
            }
          }
          if (grow >= pr.m) continue;
          if (ring) {
            for (int c = 0; c < p.ring_copies; ++c)
              store_unit<EPI, BN>(OutDesc{p.ring_dst[c], pr.ldc, pr.n}, grow, nt, c4, g, u);
          } else {
            store_unit<EPI, BN>(OutDesc{pr.out, pr.ldc, pr.n}, grow, nt, c4, g, u);
          }
        }
      }
    }
  }


  if (*abort_flag && threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem_d, kTmemCols);
    else
      ptx::tmem_dealloc(tmem_d, kTmemCols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

template <int BN, int EPI>
tp_status launch_one(const GemmParams &p, cudaStream_t stream) {
  static int configured_mask = 0;  // one bit per device ordinal (< 32)
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 32 || !(configured_mask & (1 << dev))) {
      e = cudaFuncSetAttribute(k_gemm_bf16<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
      if (e != cudaSuccess) return cuda_fail(e);
      if (dev < 32) configured_mask |= (1 << dev);
    }
  }
  const int cap = p.max_ctas > 0 && p.max_ctas < num_sms() ? p.max_ctas : num_sms();
  const int grid = p.total_tiles < cap ? p.total_tiles : cap;
  e = launch_kernel(k_gemm_bf16<BN, EPI>, dim3(grid), dim3(kThreads), one_smem_bytes(p.a_rows, BN, p.one_stages),
                    stream, 1, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

template <int EPI, int KSUB, int BN, bool GROUPED = false>
tp_status launch_pair_ks(const GemmParams &p, cudaStream_t stream) {
  static int configured_mask = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 32 || !(configured_mask & (1 << dev))) {
      e = cudaFuncSetAttribute(k_gemm_bf16_pair<EPI, KSUB, BN, GROUPED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairCfg<KSUB, BN>::kSmem);
      if (e != cudaSuccess) return cuda_fail(e);
      if (dev < 32) configured_mask |= (1 << dev);
    }
  }
  const int pairs_max = num_sms() / 2;
  const int pairs = p.total_tiles < pairs_max ? p.total_tiles : pairs_max;
  e = launch_kernel(k_gemm_bf16_pair<EPI, KSUB, BN, GROUPED>, dim3(2 * pairs), dim3(kThreads),
                    PairCfg<KSUB, BN>::kSmem, stream, 1, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

// 64-wide k-tiles per pipeline stage of the pair kernel (TPGQA_KSUB=2|3 overrides).
// Two (three 64 KB stages) measured faster than three (two 96 KB stages): the
// TMA unit delivers more bytes per clock with more boxes per barrier phase, but
// two stages leave the loads and the MMAs too little overlap.
int pair_ksub() {
  static const int k = [] {
    const char *e = getenv("TPGQA_KSUB");
    const int v = e ? atoi(e) : 2;
    return (v == 2 || v == 3) ? v : 2;
  }();
  return k;
}

template <int EPI>
tp_status launch_pair(const GemmParams &p, int bn, cudaStream_t stream) {
  if (bn == 512 || bn == 448) {
    if constexpr (EPI == kEpiSwiGLU)
      return bn == 512 ? launch_pair_ks<EPI, 1, 512>(p, stream) : launch_pair_ks<EPI, 1, 448>(p, stream);
    else
      return TP_ERR_UNSUPPORTED;
  }
  if (bn == 224) return launch_pair_ks<EPI, 2, 224>(p, stream);
  if (bn == 128) return launch_pair_ks<EPI, 2, 128>(p, stream);
  if (bn != 256) return TP_ERR_UNSUPPORTED;
  if (pair_ksub() != 2) return launch_pair_ks<EPI, 3, 256>(p, stream);
  // The grouped tile order (MoE problems) has its own instantiation; other
  // widths run every problem m-tile first, which changes no result.
  bool grouped = false;
  for (int i = 0; i < p.num_problems; ++i) grouped = grouped || p.prob[i].m_group > 0;
  return grouped ? launch_pair_ks<EPI, 2, 256, true>(p, stream) : launch_pair_ks<EPI, 2, 256>(p, stream);
}

template <int KSUB, int BN>
tp_status launch_pair_ring_ks(const GemmParams &p, cudaStream_t stream) {
  static int configured_mask = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 32 || !(configured_mask & (1 << dev))) {
      e = cudaFuncSetAttribute(k_gemm_bf16_pair_ring<KSUB, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairRingCfg<KSUB, BN>::kSmem);
      if (e != cudaSuccess) return cuda_fail(e);
      if (dev < 32) configured_mask |= (1 << dev);
    }
  }
  const int pairs_max = num_sms() / 2;
  const int pairs = p.total_tiles < pairs_max ? p.total_tiles : pairs_max;
  e = launch_kernel(k_gemm_bf16_pair_ring<KSUB, BN>, dim3(2 * pairs), dim3(kThreads), PairRingCfg<KSUB, BN>::kSmem,
                    stream, 1, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

// Same tile width and k-stage grouping as launch_pair, so the partials match
// the GEMM without a combine bit for bit.
tp_status launch_pair_ring(const GemmParams &p, int bn, cudaStream_t stream) {
  if (bn == 224) return launch_pair_ring_ks<2, 224>(p, stream);
  if (bn == 128) return launch_pair_ring_ks<2, 128>(p, stream);
  if (bn != 256) return TP_ERR_UNSUPPORTED;
  return pair_ksub() == 2 ? launch_pair_ring_ks<2, 256>(p, stream) : launch_pair_ring_ks<3, 256>(p, stream);
}

template <bool PAIR, int EPI, int BN>
tp_status launch_splitk(const GemmParams &p, cudaStream_t stream) {
  using C = SplitCfg<PAIR, BN>;
  static int configured_mask = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 32 || !(configured_mask & (1 << dev))) {
      e = cudaFuncSetAttribute(k_gemm_bf16_splitk<PAIR, EPI, BN>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, PAIR ? C::kSmem : kSmemLimit);
      if (e != cudaSuccess) return cuda_fail(e);
      if (dev < 32) configured_mask |= (1 << dev);
    }
  }
  const int csize = (PAIR ? 2 : 1) * p.split;
  const int smem = PAIR ? C::kSmem : one_smem_bytes(p.a_rows, BN, p.one_stages);
  e = launch_kernel(k_gemm_bf16_splitk<PAIR, EPI, BN>, dim3(static_cast<unsigned>(p.total_tiles * csize)),
                    dim3(kThreads), smem, stream, static_cast<unsigned>(csize), p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

}  // namespace

// Clusters of `csize` split-K CTAs that can be resident at once, or -1 if the
// runtime cannot say. A cluster has to fit inside one GPC, so this can be well
// below SMs / csize (on GB300: 36 clusters of 4 and 15 of 8 for 152 SMs). All
// split-K instantiations use the same shared memory and block size, so one of
// them stands for all.
int max_active_clusters(int csize) {
  static std::mutex mu;
  static int cache[32][17] = {};  // [device][cluster size], 0 = not queried yet
  int dev = 0;
  if (csize < 1 || csize > 16 || cudaGetDevice(&dev) != cudaSuccess || dev >= 32) return -1;
  std::lock_guard<std::mutex> g(mu);
  if (cache[dev][csize] == 0) {
    using C = SplitCfg<true, 256>;
    auto kern = k_gemm_bf16_splitk<true, kEpiF32, 256>;
    int n = -1;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(csize));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = C::kSmem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = static_cast<unsigned>(csize);
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = -1;
    }
    cudaGetLastError();  // a failed query leaves no sticky error behind
    cache[dev][csize] = n;
  }
  return cache[dev][csize];
}

bool encode_bf16_map_2d(CUtensorMap *map, const void *base, long long rows, long long cols, long long ld,
                        int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

GemmBuilder::GemmBuilder() { std::memset(&p, 0, sizeof(p)); }

int GemmBuilder::add_map(const void *base, long long rows, long long k, long long ld, int box_rows,
                         tp_status *err) {
  if (n_maps >= kMaxMaps) {
    *err = TP_ERR_UNSUPPORTED;
    return -1;
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    *err = cuda_fail(cudaErrorNotSupported);
    return -1;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(&p.maps[n_maps], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = TP_ERR_INVALID_ARG;
    return -1;
  }
  margs[n_maps] = MapArgs{base, rows, k, ld, box_rows};
  return n_maps++;
}

int GemmBuilder::add_out_map_f32(void *base, long long rows, long long cols, long long ld, tp_status *err) {
  if (n_maps >= kMaxMaps) {
    *err = TP_ERR_UNSUPPORTED;
    return -1;
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    *err = cuda_fail(cudaErrorNotSupported);
    return -1;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&p.maps[n_maps], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    *err = TP_ERR_INVALID_ARG;
    return -1;
  }
  margs[n_maps] = MapArgs{base, rows, cols, ld, 32};
  out_map[n_maps] = true;
  return n_maps++;
}

int GemmBuilder::use_3d_boxes(int kt) {
  // TPGQA_TMA3D=0 keeps the 2-D maps (tuning override).
  static const int enabled = [] {
    const char *e = getenv("TPGQA_TMA3D");
    return e ? atoi(e) : 1;
  }();
  if (kt <= 1 || !enabled) return 1;
  for (int i = 0; i < n_maps; ++i)
    if (!out_map[i] && (margs[i].k % BK != 0 || margs[i].k / BK < kt)) return 1;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return 1;
  // View a [rows x k] matrix as [k/64][rows][64]: element (x, y, z) is column
  // z*64 + x of row y, so dim 2 steps by 128 bytes inside a row. A box of
  // {64, box_rows, kt} lands as kt swizzled [box_rows x 128 B] k-tiles back to
  // back, the same shared-memory layout that kt 2-D copies produce.
  CUtensorMap tmp[kMaxMaps];
  for (int i = 0; i < n_maps; ++i) {
    if (out_map[i]) continue;
    const MapArgs &m = margs[i];
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(m.rows),
                                static_cast<cuuint64_t>(m.k / BK)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(m.ld) * 2, static_cast<cuuint64_t>(BK) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(m.box_rows),
                               static_cast<cuuint32_t>(kt)};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tmp[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(m.base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return 1;  // keep the 2-D maps, all of them
  }
  for (int i = 0; i < n_maps; ++i)
    if (!out_map[i]) p.maps[i] = tmp[i];
  return kt;
}

bool GemmBuilder::add_problem(int m, int n, void *out, long long ldc, const int *a_maps,
                              const int *b_maps, const int *b2_maps, const long long *ks, int nseg,
                              const int *blk, int b_rows_per_blk, int n_moff) {
  if (n_probs >= kMaxProblems || n_segs + nseg > kMaxSegs) return false;
  const int out_cols = (epi == kEpiSwiGLU) ? bn / 2 : bn;
  const int tile_m = pair ? 2 * BM : BM;
  GemmProblem &pr = p.prob[n_probs];
  pr.m = m;
  pr.n = n;
  pr.m_tiles = (m + tile_m - 1) / tile_m;
  pr.n_tiles = (n + out_cols - 1) / out_cols;
  pr.tile_begin = p.total_tiles;
  pr.seg_begin = n_segs;
  pr.seg_count = nseg;
  pr.out = out;
  pr.ldc = ldc;
  pr.blk = blk;
  pr.b_rows_per_blk = b_rows_per_blk;
  pr.n_moff = n_moff;
  pr.m_group = m_group;
  if (blk) split = 1;  // block tables run on the persistent kernels only
  for (int s = 0; s < nseg; ++s) {
    GemmSeg &sg = p.seg[n_segs + s];
    sg.a_map = a_maps[s];
    sg.b_map = b_maps[s];
    sg.b2_map = b2_maps ? b2_maps[s] : -1;
    sg.k_tiles = static_cast<int>((ks[s] + BK - 1) / BK);
  }
  n_segs += nseg;
  p.total_tiles += pr.m_tiles * pr.n_tiles;
  ++n_probs;
  return true;
}

bool GemmBuilder::add_dual_problem(int m, int n, void *out, long long ldc, void *out2, long long ldc2, int a_map,
                                   int b_map, int b2_map, long long k) {
  if (!pair || bn != 256 || epi != kEpiBF16 || n > 128) return false;
  const long long ks = k;
  const int saved_epi = epi;
  epi = kEpiSwiGLU;  // tile count: 128 output columns per 256-column tile
  const bool ok = add_problem(m, n, out, ldc, &a_map, &b_map, &b2_map, &ks, 1);
  epi = saved_epi;
  if (!ok) return false;
  p.prob[n_probs - 1].out2 = out2;
  p.prob[n_probs - 1].ldc2 = ldc2;
  dual = true;
  return true;
}

tp_status GemmBuilder::launch(cudaStream_t stream) {
  p.num_problems = n_probs;
  p.n_maps_used = n_maps;
  ctas = 0;
  if (p.total_tiles == 0) return TP_OK;
  DevCtx ctx;
  cudaError_t e = get_dev_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e);
  p.status = ctx.status;
  p.wait_ns = ctx.wait_ns;
  // L2 prefetch depth of B tiles in k-blocks, issued by the TMA producer
  // (TPGQA_PREFETCH overrides). Off by default: every prefetch costs the single
  // producer thread about as much as a load, and the T=512 MLP block ran 4%
  // slower with a depth of 8 and 10% slower with 32.
  static const int prefetch = [] {
    const char *e = getenv("TPGQA_PREFETCH");
    return e ? atoi(e) : 0;
  }();
  p.prefetch = prefetch;
  p.a_rows = pair ? 128 : a_rows;
  p.one_stages = one_stages_for(p.a_rows, bn);
  {
    // TPGQA_EARLY_B=0 keeps every load behind the grid-dependency wait (read on
    // every launch). Block tables are written by an earlier kernel and decide
    // which weights a tile reads, so their problems never load early.
    const char *env = getenv("TPGQA_EARLY_B");
    bool early = !(env && env[0] == '0');
    for (int i = 0; i < n_probs; ++i)
      if (p.prob[i].blk) early = false;
    p.early_b = early ? 1 : 0;
  }
  if (split == 0) {
    // fewest k-stages of any problem decides how far K can be split
    const int ksub = pair ? 2 : 1;
    long long min_stages = -1;
    for (int i = 0; i < n_probs; ++i) {
      long long st = 0;
      for (int q = 0; q < p.prob[i].seg_count; ++q)
        st += (p.seg[p.prob[i].seg_begin + q].k_tiles + ksub - 1) / ksub;
      if (min_stages < 0 || st < min_stages) min_stages = st;
    }
    split = choose_split(p.total_tiles, pair, min_stages < 0 ? 0 : min_stages);
  }
  if (ring_split) {
    // one split per segment (rank) on 256 x 128 pair tiles, f32 sums in ring order
    if (!pair || bn != 128 || epi != kEpiF32 || n_probs != 1 || p.prob[0].seg_count < 2 ||
        p.prob[0].seg_count > 4 || p.ring_rows <= 0 || p.ring_rows % 256 != 0 || p.ring_copies < 1 ||
        p.ring_copies > kMaxRingCopies)
      return TP_ERR_UNSUPPORTED;
    p.split = p.prob[0].seg_count;
    p.box_kt = use_3d_boxes(SplitCfg<true, 128>::kSub);
    return launch_splitk<true, kEpiF32, 128>(p, stream);
  }
  if (split < 1 || (pair && bn != 256) || (!pair && bn != 256 && bn != 128) || ring || dual)
    split = 1;  // split-K runs 256-column pair tiles and 128/256-column single-CTA tiles
  if (defer_dep_wait || max_ctas > 0) split = 1;
  p.split = split;
  // the deferred wait and the CTA cap are built into the persistent single-CTA kernel only
  const bool one = !pair && split == 1;
  p.defer_dep_wait = defer_dep_wait && one ? 1 : 0;
  p.max_ctas = one ? max_ctas : 0;
  {
    const int sms = num_sms();
    if (split > 1)
      ctas = p.total_tiles * (pair ? 2 : 1) * split;
    else if (pair)
      ctas = 2 * (p.total_tiles < sms / 2 ? p.total_tiles : sms / 2);
    else {
      const int cap = p.max_ctas > 0 && p.max_ctas < sms ? p.max_ctas : sms;
      ctas = p.total_tiles < cap ? p.total_tiles : cap;
    }
  }
  // The SM-pair kernels load KSUB k-tiles per stage; one 3-D copy per operand
  // and stage replaces KSUB 2-D copies. The single-CTA kernels load one k-tile
  // per stage and keep the 2-D maps.
  p.box_kt = !pair || bn == 512 || bn == 448 ? 1 : use_3d_boxes(split > 1 || bn != 256 ? SplitCfg<true, 256>::kSub : pair_ksub());
  if (ring) return launch_pair_ring(p, bn, stream);
  if (split > 1) {
    if (pair) {
      if (epi == kEpiF32) return launch_splitk<true, kEpiF32, 256>(p, stream);
      if (epi == kEpiBF16) return launch_splitk<true, kEpiBF16, 256>(p, stream);
      return launch_splitk<true, kEpiSwiGLU, 256>(p, stream);
    }
    if (bn == 128) {
      if (epi == kEpiF32) return launch_splitk<false, kEpiF32, 128>(p, stream);
      if (epi == kEpiBF16) return launch_splitk<false, kEpiBF16, 128>(p, stream);
      return launch_splitk<false, kEpiSwiGLU, 128>(p, stream);
    }
    if (epi == kEpiF32) return launch_splitk<false, kEpiF32, 256>(p, stream);
    if (epi == kEpiBF16) return launch_splitk<false, kEpiBF16, 256>(p, stream);
    return launch_splitk<false, kEpiSwiGLU, 256>(p, stream);
  }
  if (pair) {
    if (epi == kEpiF32) return launch_pair<kEpiF32>(p, bn, stream);
    if (epi == kEpiBF16) return launch_pair<kEpiBF16>(p, bn, stream);
    return launch_pair<kEpiSwiGLU>(p, bn, stream);
  }
  if (bn == 256) {
    if (epi == kEpiF32) return launch_one<256, kEpiF32>(p, stream);
    if (epi == kEpiBF16) return launch_one<256, kEpiBF16>(p, stream);
    return launch_one<256, kEpiSwiGLU>(p, stream);
  }
  if (bn == 224) {
    if (epi == kEpiF32) return launch_one<224, kEpiF32>(p, stream);
    if (epi == kEpiBF16) return launch_one<224, kEpiBF16>(p, stream);
    return launch_one<224, kEpiSwiGLU>(p, stream);
  }
  if (bn == 192) {
    if (epi == kEpiF32) return launch_one<192, kEpiF32>(p, stream);
    if (epi == kEpiBF16) return launch_one<192, kEpiBF16>(p, stream);
    return launch_one<192, kEpiSwiGLU>(p, stream);
  }
  if (epi == kEpiF32) return launch_one<128, kEpiF32>(p, stream);
  if (epi == kEpiBF16) return launch_one<128, kEpiBF16>(p, stream);
  return launch_one<128, kEpiSwiGLU>(p, stream);
}

bool choose_pair(long long rows) {
  // TPGQA_PAIR=0|1 forces the single-CTA / SM-pair kernel (tuning override).
  static const int forced = [] {
    const char *e = getenv("TPGQA_PAIR");
    return e ? atoi(e) : -1;
  }();
  if (forced == 0 || forced == 1) return forced == 1;
  // Pairs compute 256-row tiles; at 128 rows or fewer half of every pair MMA
  // would be padding, so the single-CTA kernel runs those.
  return rows > 128;
}

int choose_split(long long tiles, bool pair, long long stages_per_tile) {
  // TPGQA_SPLIT=n forces the split factor (tuning override; 1 disables).
  static const int forced = [] {
    const char *e = getenv("TPGQA_SPLIT");
    return e ? atoi(e) : 0;
  }();
  const int per_tile = pair ? 2 : 1;
  const int max_split = 8 / per_tile;  // portable cluster size limit
  if (forced >= 1) return forced <= max_split ? forced : max_split;
  const long long sms = num_sms();
  int s = 1;
  // Double the split while the grid still fits in one wave and each split keeps
  // at least four k-stages to pipeline.
  while (2 * s <= max_split && tiles * per_tile * 2 * s <= sms && stages_per_tile >= 8LL * s) s *= 2;
  // One wave also needs every cluster (one tile's splits) resident at once.
  while (s > 1) {
    const int m = max_active_clusters(per_tile * s);
    if (m < 0 || tiles <= m) break;
    s /= 2;
  }
  return s;
}

int choose_bn(long long rows, const long long *ncols, int nprob, bool swiglu, long long max_ctas) {
  // TPGQA_BN=128|192|224|256 forces the tile width (tuning override).
  static const int forced = [] {
    const char *e = getenv("TPGQA_BN");
    return e ? atoi(e) : 0;
  }();
  if (forced == 128 || forced == 192 || forced == 224 || forced == 256) return forced;
  // Single-CTA tiles stream the weights (few rows of activations): a tile's time
  // goes with its width, the kernel's with the waves of tiles over the SMs.
  // 128-column tiles need twice the operand bytes per MMA flop; grids small
  // enough for split-K keep 256 columns. max_ctas > 0: the CTAs the launch may use.
  const long long sms = max_ctas > 0 && max_ctas < num_sms() ? max_ctas : num_sms();
  const long long mt = (rows + 127) / 128;
  int best = 256;
  long long best_cost = -1;
  for (int bn : {256, 224, 192}) {
    const int out_cols = swiglu ? bn / 2 : bn;
    long long tiles = 0;
    for (int i = 0; i < nprob; ++i) tiles += mt * ((ncols[i] + out_cols - 1) / out_cols);
    if (bn == 256 && tiles * 2 <= sms) return 256;  // split-K territory
    const long long cost = ((tiles + sms - 1) / sms) * bn;
    if (best_cost < 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

int choose_pair_bn(long long m, const long long *ncols, int nprob, bool swiglu, int *b_rows) {
  // TPGQA_PAIR_BN=128|224|256|448|512 forces the SM-pair tile width (tuning
  // override; 448 and 512 apply to SwiGLU problems only).
  static const int forced = [] {
    const char *e = getenv("TPGQA_PAIR_BN");
    return e ? atoi(e) : 0;
  }();
  int best = 256;
  if (forced == 128 || forced == 224 || forced == 256 || ((forced == 448 || forced == 512) && swiglu)) {
    best = forced;
  } else {
    // A tile's time goes with its stage bytes (the loads bound the pair's
    // k-loop), the kernel's with the number of waves of tiles over the SM
    // pairs. Narrower tiles win when they save a wave. Grids small enough for
    // split-K keep 256 columns (the split-K pair kernel runs only those).
    const long long pairs = num_sms() / 2;
    const long long mt = (m + 255) / 256;
    long long cost256 = 0;
    for (int bn : {256, 224}) {
      const int out_cols = swiglu ? bn / 2 : bn;
      long long tiles = 0;
      for (int i = 0; i < nprob; ++i) tiles += mt * ((ncols[i] + out_cols - 1) / out_cols);
      const long long waves = (tiles + pairs - 1) / pairs;
      const long long cost = waves * (2 * (16384 + (bn / 2) * 128));
      if (bn == 256) {
        cost256 = cost;
        if (tiles * 4 <= num_sms()) break;  // split-K territory
      } else if (cost < cost256) {
        best = bn;
      }
    }
    // SwiGLU grids of more than one wave of 256-column tiles that fit one wave
    // of wide tiles (BN/2 gate and BN/2 up columns): one tile per SM pair, half
    // the A bytes per MMA flop. A single wave's time goes with the tile width,
    // so the narrower of 448 and 512 that fits wins. The single accumulator
    // leaves no epilogue overlap, which a single wave does not need.
    if (swiglu && forced == 0) {
      long long t256 = 0, t448 = 0, t512 = 0;
      for (int i = 0; i < nprob; ++i) {
        t256 += mt * ((ncols[i] + 127) / 128);
        t448 += mt * ((ncols[i] + 223) / 224);
        t512 += mt * ((ncols[i] + 255) / 256);
      }
      if (t256 > pairs && t448 <= pairs)
        best = 448;
      else if (t256 > pairs && t512 <= pairs)
        best = 512;
    }
  }
  *b_rows = best == 512 || best == 448 ? best / 4 : best / 2;
  return best;
}

int a_box_rows(long long rows) {
  const long long r = ((rows + 7) / 8) * 8;
  return static_cast<int>(r < 128 ? (r < 8 ? 8 : r) : 128);
}

}  // namespace tpgqa
