// bf16 grouped GEMM on the 5th-generation tensor cores: C = A * B^T with A
// [M x K] and B [N x K] both K-major (weights stored [out x in]), fp32
// accumulation in tensor memory.
//
// One CTA computes one 128 x BN output tile of one problem. Warp roles:
//   warp 0      TMA producer: one thread streams 128x64 A and BNx64 B tiles
//               into a ring of shared-memory stages (128-byte swizzle).
//   warp 1      owns the TMEM accumulator (alloc / dealloc); one thread issues
//               tcgen05.mma (M=128, N=BN, K=16, four per 64-wide stage) and
//               frees each stage with tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (each warp reads its
//               32-lane quarter), fused output transform, global stores.
// A problem's K loop runs over its segments in order, so a row-parallel layer
// can sum every rank's shard in the same accumulator (segments = ranks).
// Every mbarrier wait is bounded; a wait that runs out records a code in the
// device status word, the CTA drains its in-flight copies, frees TMEM and exits.
#include <cuda_bf16.h>

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

template <int BN>
struct TileCfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;
};

__device__ __forceinline__ void record(int *status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

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

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1) k_gemm_bf16(const __grid_constant__ GemmParams p) {
  using C = TileCfg<BN>;
  constexpr int kBRows = (EPI == kEpiSwiGLU) ? BN / 2 : BN;  // rows per B map box
  constexpr int kOutCols = (EPI == kEpiSwiGLU) ? BN / 2 : BN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sA0 = ptx::smem_addr(smem);
  const uint32_t sB0 = sA0 + C::kStages * C::kABytes;
  uint8_t *bar_area = smem + C::kStages * C::kStageBytes;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  const uint32_t accum_bar = bar0 + 16 * C::kStages;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 16 * C::kStages + 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 16 * C::kStages + 16);
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (C::kStages + i); };

  // ---- which tile of which problem ----
  const int tile = blockIdx.x;
  int pi = 0;
  for (int i = 1; i < p.num_problems; ++i)
    if (tile >= p.prob[i].tile_begin) pi = i;
  const GemmProblem &pr = p.prob[pi];
  const int local = tile - pr.tile_begin;
  const int mt = local % pr.m_tiles;
  const int nt = local / pr.m_tiles;
  int total_kt = 0;
  for (int s = 0; s < pr.seg_count; ++s) total_kt += p.seg[pr.seg_begin + s].k_tiles;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      ptx::mbar_init(full_bar(i), 1);
      ptx::mbar_init(empty_bar(i), 1);
    }
    ptx::mbar_init(accum_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < pr.seg_count; ++s) {
      const GemmSeg &sg = p.seg[pr.seg_begin + s];
      ptx::prefetch_tensormap(&p.maps[sg.a_map]);
      ptx::prefetch_tensormap(&p.maps[sg.b_map]);
      if (EPI == kEpiSwiGLU) ptx::prefetch_tensormap(&p.maps[sg.b2_map]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), BN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  int issued = 0;  // k-blocks whose loads the producer started (thread 0 only)
  if (warp == 0) {
    if (lane == 0) {
      const int a_row = mt * BM;
      const int b_row = nt * kBRows;
      bool ok = true;
      int kb = 0;
      for (int s = 0; ok && s < pr.seg_count; ++s) {
        const GemmSeg sg = p.seg[pr.seg_begin + s];
        for (int kt = 0; kt < sg.k_tiles; ++kt, ++kb) {
          const int st = kb % C::kStages;
          const uint32_t ph = (kb / C::kStages) & 1;
          if (*abort_flag) { ok = false; break; }
          if (!ptx::mbar_wait(empty_bar(st), ph ^ 1, p.wait_ns)) {
            record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full_bar(st), C::kStageBytes);
          ptx::tma_load_2d(sA0 + st * C::kABytes, &p.maps[sg.a_map], kt * BK, a_row, full_bar(st));
          ptx::tma_load_2d(sB0 + st * C::kBBytes, &p.maps[sg.b_map], kt * BK, b_row, full_bar(st));
          if (EPI == kEpiSwiGLU)
            ptx::tma_load_2d(sB0 + st * C::kBBytes + kBRows * 128, &p.maps[sg.b2_map], kt * BK,
                             b_row, full_bar(st));
          issued = kb + 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      for (int kb = 0; kb < total_kt; ++kb) {
        const int st = kb % C::kStages;
        const uint32_t ph = (kb / C::kStages) & 1;
        if (*abort_flag) break;
        if (!ptx::mbar_wait(full_bar(st), ph, p.wait_ns)) {
          record(p.status, kDevTimeoutMma);
          *abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint64_t ad = ptx::smem_desc_sw128(sA0 + st * C::kABytes);
        const uint64_t bd = ptx::smem_desc_sw128(sB0 + st * C::kBBytes);
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k)
          ptx::mma_bf16(tmem_d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
        ptx::mma_commit(empty_bar(st));
      }
      ptx::mma_commit(accum_bar);
    }
  } else {
    // ---- epilogue: warps 2..5, warp w reads TMEM lanes [32*(w%4), 32*(w%4)+32) ----
    const int q = warp & 3;
    const bool ready = ptx::mbar_wait(accum_bar, 0, p.wait_ns);
    if (!ready && lane == 0) record(p.status, kDevTimeoutEpilogue);
    ptx::tc_fence_after();
    const bool go = __all_sync(0xffffffffu, ready && (*abort_flag == 0));
    if (go) {
      const int row = mt * BM + q * 32 + lane;
      const uint32_t tbase = tmem_d + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (EPI == kEpiSwiGLU) {
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(pr.out);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32cols(tbase + c, g);
          ptx::tmem_ld_32cols(tbase + BN / 2 + c, u);
          ptx::tmem_ld_wait();
          float h[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) h[j] = silu(__uint_as_float(g[j])) * __uint_as_float(u[j]);
          if (row < pr.m) store_bf16_row32(out, pr.ldc, row, nt * kOutCols + c, pr.n, h);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32cols(tbase + c, v);
          ptx::tmem_ld_wait();
          float f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
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
    const int first = issued > C::kStages ? issued - C::kStages : 0;
    for (int kb = first; kb < issued; ++kb)
      if (!ptx::mbar_wait(full_bar(kb % C::kStages), (kb / C::kStages) & 1, p.wait_ns))
        record(p.status, kDevTimeoutDrain);
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_d, BN);
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
      e = cudaFuncSetAttribute(k_gemm_bf16<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               TileCfg<BN>::kSmem);
      if (e != cudaSuccess) return cuda_fail(e);
      if (dev < 32) configured_mask |= (1 << dev);
    }
  }
  k_gemm_bf16<BN, EPI><<<p.total_tiles, kThreads, TileCfg<BN>::kSmem, stream>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

}  // namespace

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
  return n_maps++;
}

bool GemmBuilder::add_problem(int m, int n, void *out, long long ldc, const int *a_maps,
                              const int *b_maps, const int *b2_maps, const long long *ks, int nseg) {
  if (n_probs >= kMaxProblems || n_segs + nseg > kMaxSegs) return false;
  const int out_cols = (epi == kEpiSwiGLU) ? bn / 2 : bn;
  GemmProblem &pr = p.prob[n_probs];
  pr.m = m;
  pr.n = n;
  pr.m_tiles = (m + BM - 1) / BM;
  pr.n_tiles = (n + out_cols - 1) / out_cols;
  pr.tile_begin = p.total_tiles;
  pr.seg_begin = n_segs;
  pr.seg_count = nseg;
  pr.out = out;
  pr.ldc = ldc;
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

tp_status GemmBuilder::launch(cudaStream_t stream) {
  p.num_problems = n_probs;
  if (p.total_tiles == 0) return TP_OK;
  DevCtx ctx;
  cudaError_t e = get_dev_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e);
  p.status = ctx.status;
  p.wait_ns = ctx.wait_ns;
  if (bn == 256) {
    if (epi == kEpiF32) return launch_one<256, kEpiF32>(p, stream);
    if (epi == kEpiBF16) return launch_one<256, kEpiBF16>(p, stream);
    return launch_one<256, kEpiSwiGLU>(p, stream);
  }
  if (epi == kEpiF32) return launch_one<128, kEpiF32>(p, stream);
  if (epi == kEpiBF16) return launch_one<128, kEpiBF16>(p, stream);
  return launch_one<128, kEpiSwiGLU>(p, stream);
}

int choose_bn(long long tiles_256, long long tiles_128, int epi) {
  (void)tiles_128;
  (void)epi;
  // Wide tiles halve the A re-reads; fall back to narrow ones when the wide
  // grid would leave most SMs idle.
  return tiles_256 >= num_sms() ? 256 : 128;
}

}  // namespace tpgqa
