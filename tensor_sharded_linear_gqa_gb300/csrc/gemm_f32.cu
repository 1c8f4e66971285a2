// Exact fp32 grouped GEMM on the CUDA cores: C = A * B^T, A [M x K] and B [N x K]
// row-major, one fused multiply-add per product in increasing k order (no TF32).
// A problem's K loop runs over its segments in order. Used for the fp32 layer
// (the railscraft wiki's worked example) where TF32 rounding would exceed the
// 1e-5 relative bound.
#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr int FBM = 32, FBN = 64, FBK = 32, FTHREADS = 256;

__global__ void __launch_bounds__(FTHREADS) k_gemm_f32(const __grid_constant__ F32Params p) {
  __shared__ float As[FBK][FBM + 1];
  __shared__ float Bs[FBK][FBN + 1];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tile = blockIdx.x;
  int pi = 0;
  for (int i = 1; i < p.num_problems; ++i)
    if (tile >= p.prob[i].tile_begin) pi = i;
  const F32Problem &pr = p.prob[pi];
  const int local = tile - pr.tile_begin;
  const int m0 = (local % pr.m_tiles) * FBM;
  const int n0 = (local / pr.m_tiles) * FBN;

  const int tid = threadIdx.x;
  const int tx = tid % 16;  // 4 output columns each
  const int ty = tid / 16;  // 2 output rows each
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};

  for (int s = 0; s < pr.seg_count; ++s) {
    const F32Seg sg = p.seg[pr.seg_begin + s];
    for (int k0 = 0; k0 < sg.k; k0 += FBK) {
#pragma unroll
      for (int i = 0; i < (FBM * FBK) / FTHREADS; ++i) {
        const int idx = tid + i * FTHREADS;
        const int r = idx / FBK, k = idx % FBK;
        const int gr = m0 + r, gk = k0 + k;
        As[k][r] = (gr < pr.m && gk < sg.k) ? sg.a[static_cast<long long>(gr) * sg.lda + gk] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < (FBN * FBK) / FTHREADS; ++i) {
        const int idx = tid + i * FTHREADS;
        const int r = idx / FBK, k = idx % FBK;
        const int gr = n0 + r, gk = k0 + k;
        Bs[k][r] = (gr < pr.n && gk < sg.k) ? sg.b[static_cast<long long>(gr) * sg.ldb + gk] : 0.f;
      }
      __syncthreads();
      const int kmax = min(FBK, sg.k - k0);
      for (int kk = 0; kk < kmax; ++kk) {
        const float a0 = As[kk][ty * 2], a1 = As[kk][ty * 2 + 1];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float b = Bs[kk][tx * 4 + j];
          acc[0][j] = __fmaf_rn(a0, b, acc[0][j]);
          acc[1][j] = __fmaf_rn(a1, b, acc[1][j]);
        }
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = m0 + ty * 2 + i;
    if (r >= pr.m) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c < pr.n) pr.out[static_cast<long long>(r) * pr.ldc + c] = acc[i][j];
    }
  }
}

}  // namespace

tp_status launch_gemm_f32(const F32Params &p, cudaStream_t stream) {
  if (p.total_tiles == 0) return TP_OK;
  cudaError_t e = launch_kernel(k_gemm_f32, dim3(p.total_tiles), dim3(FTHREADS), 0, stream, 1, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

}  // namespace tpgqa
