// Collectives over the shard buffers of the N logical ranks, all in this GPU's
// memory (mlxcel manual "텐서 병렬화", 통신 패턴 / Communication patterns: ring
// all-reduce = reduce-scatter + all-gather; rank r sends to (r+1) % N in each of
// N-1 steps).
//
// Buffers are flat fp32 arrays of `size` elements; chunk c is the element range
// [floor(c*size/N), floor((c+1)*size/N)). Each kernel walks one chunk per
// (rank or chunk) row of the grid: a scalar head up to the first 16-byte
// boundary, a float4 body (four independent 16-byte loads in flight per thread
// per iteration), a scalar tail. All buffers share one base alignment (16 bytes),
// so a chunk's element offsets have the same alignment in every buffer.
//
// Reduce-scatter step s: rank r sends chunk (r-1-s) mod N to rank (r+1) % N,
// which stores (received + own). All-gather step s: rank r sends chunk
// (r-s) mod N, which the receiver stores. The fused kernels fold chunk c in the
// same order, c+1, c+2, ..., c (mod N), in registers, so their results are
// bit-identical to the step kernels (IEEE addition is commutative; the
// association is the ring's left fold).
#include <cuda_bf16.h>

#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void chunk_range(long long size, int n, int c, long long &lo,
                                            long long &hi) {
  lo = (static_cast<long long>(c) * size) / n;
  hi = (static_cast<long long>(c + 1) * size) / n;
}

// Splits [lo, hi) into a scalar head [lo, vlo), a float4 body [vlo, vhi), a tail [vhi, hi).
__device__ __forceinline__ void split_vec(long long lo, long long hi, long long &vlo,
                                          long long &vhi) {
  vlo = (lo + 3) & ~3LL;
  if (vlo > hi) vlo = hi;
  vhi = hi & ~3LL;
  if (vhi < vlo) vhi = vlo;
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// One reduce-scatter step; grid.y = sending rank.
__global__ void __launch_bounds__(kThreads) k_ring_rs_step(RankPtrs b, int n, long long size,
                                                           int step) {
  griddep_wait();
  griddep_launch_dependents();
  const int r = blockIdx.y;
  const int c = ((r - 1 - step) % n + n) % n;
  const float *__restrict__ src = b.p[r];
  float *__restrict__ dst = b.p[(r + 1) % n];
  long long lo, hi, vlo, vhi;
  chunk_range(size, n, c, lo, hi);
  split_vec(lo, hi, vlo, vhi);
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if (t < vlo - lo) dst[lo + t] = src[lo + t] + dst[lo + t];
  if (t < hi - vhi) dst[vhi + t] = src[vhi + t] + dst[vhi + t];
  const float4 *__restrict__ s4 = reinterpret_cast<const float4 *>(src + vlo);
  float4 *__restrict__ d4 = reinterpret_cast<float4 *>(dst + vlo);
  const long long nv = (vhi - vlo) >> 2;
  long long i = t;
  for (; i + 3 * stride < nv; i += 4 * stride) {
    const float4 a0 = s4[i], a1 = s4[i + stride], a2 = s4[i + 2 * stride], a3 = s4[i + 3 * stride];
    const float4 b0 = d4[i], b1 = d4[i + stride], b2 = d4[i + 2 * stride], b3 = d4[i + 3 * stride];
    d4[i] = add4(a0, b0);
    d4[i + stride] = add4(a1, b1);
    d4[i + 2 * stride] = add4(a2, b2);
    d4[i + 3 * stride] = add4(a3, b3);
  }
  for (; i < nv; i += stride) d4[i] = add4(s4[i], d4[i]);
}

// One all-gather step; grid.y = sending rank.
__global__ void __launch_bounds__(kThreads) k_ring_ag_step(RankPtrs b, int n, long long size,
                                                           int step) {
  griddep_wait();
  griddep_launch_dependents();
  const int r = blockIdx.y;
  const int c = ((r - step) % n + n) % n;
  const float *__restrict__ src = b.p[r];
  float *__restrict__ dst = b.p[(r + 1) % n];
  long long lo, hi, vlo, vhi;
  chunk_range(size, n, c, lo, hi);
  split_vec(lo, hi, vlo, vhi);
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if (t < vlo - lo) dst[lo + t] = src[lo + t];
  if (t < hi - vhi) dst[vhi + t] = src[vhi + t];
  const float4 *__restrict__ s4 = reinterpret_cast<const float4 *>(src + vlo);
  float4 *__restrict__ d4 = reinterpret_cast<float4 *>(dst + vlo);
  const long long nv = (vhi - vlo) >> 2;
  long long i = t;
  for (; i + 3 * stride < nv; i += 4 * stride) {
    const float4 a0 = s4[i], a1 = s4[i + stride], a2 = s4[i + 2 * stride], a3 = s4[i + 3 * stride];
    d4[i] = a0;
    d4[i + stride] = a1;
    d4[i + 2 * stride] = a2;
    d4[i + 3 * stride] = a3;
  }
  for (; i < nv; i += stride) d4[i] = s4[i];
}

// Folds chunk c (grid.y) over all ranks in ring order; writes every buffer
// (write_all = 1: all-reduce), buffer 0 only (2: the all-reduce's result stored
// once, for ranks that share one output on this device; every element is read
// and written by one thread, so buffer 0 can hold a partial on entry) or
// buffer c only (0: reduce-scatter). NT = N when N is 2, 4 or 8
// (fully unrolled, two float4 per thread per pass with every load issued before
// the first add); NT = 0 handles any N.
template <int NT>
__global__ void __launch_bounds__(kThreads) k_ring_fused(RankPtrs b, int n_rt, long long size,
                                                         int write_all) {
  griddep_wait();
  griddep_launch_dependents();
  const int n = NT ? NT : n_rt;
  const int c = blockIdx.y;
  long long lo, hi, vlo, vhi;
  chunk_range(size, n, c, lo, hi);
  split_vec(lo, hi, vlo, vhi);
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  auto scalar = [&](long long e) {
    float acc = b.p[(c + 1) % n][e];
    for (int j = 2; j <= n; ++j) acc = acc + b.p[(c + j) % n][e];
    if (write_all == 1) {
      for (int r = 0; r < n; ++r) b.p[r][e] = acc;
    } else {
      b.p[write_all == 2 ? 0 : c][e] = acc;
    }
  };
  if (t < vlo - lo) scalar(lo + t);
  if (t < hi - vhi) scalar(vhi + t);
  const long long v0 = vlo >> 2, nv = (vhi - vlo) >> 2;
  if constexpr (NT > 0) {
    const float4 *src[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) src[j] = reinterpret_cast<const float4 *>(b.p[(c + 1 + j) % NT]) + v0;
    long long i = t;
    for (; i + stride < nv; i += 2 * stride) {
      float4 x0[NT], x1[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        x0[j] = src[j][i];
        x1[j] = src[j][i + stride];
      }
      float4 a0 = x0[0], a1 = x1[0];
#pragma unroll
      for (int j = 1; j < NT; ++j) {
        a0 = add4(a0, x0[j]);
        a1 = add4(a1, x1[j]);
      }
      if (write_all == 1) {
#pragma unroll
        for (int r = 0; r < NT; ++r) {
          reinterpret_cast<float4 *>(b.p[r])[v0 + i] = a0;
          reinterpret_cast<float4 *>(b.p[r])[v0 + i + stride] = a1;
        }
      } else {
        float4 *dst = reinterpret_cast<float4 *>(b.p[write_all == 2 ? 0 : c]);
        dst[v0 + i] = a0;
        dst[v0 + i + stride] = a1;
      }
    }
    for (; i < nv; i += stride) {
      float4 x[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) x[j] = src[j][i];
      float4 a = x[0];
#pragma unroll
      for (int j = 1; j < NT; ++j) a = add4(a, x[j]);
      if (write_all == 1) {
#pragma unroll
        for (int r = 0; r < NT; ++r) reinterpret_cast<float4 *>(b.p[r])[v0 + i] = a;
      } else {
        reinterpret_cast<float4 *>(b.p[write_all == 2 ? 0 : c])[v0 + i] = a;
      }
    }
  } else {
    for (long long i = t; i < nv; i += stride) {
      float4 acc = reinterpret_cast<const float4 *>(b.p[(c + 1) % n])[v0 + i];
      for (int j = 2; j <= n; ++j)
        acc = add4(acc, reinterpret_cast<const float4 *>(b.p[(c + j) % n])[v0 + i]);
      if (write_all == 1) {
        for (int r = 0; r < n; ++r) reinterpret_cast<float4 *>(b.p[r])[v0 + i] = acc;
      } else {
        reinterpret_cast<float4 *>(b.p[write_all == 2 ? 0 : c])[v0 + i] = acc;
      }
    }
  }
}

// In-place all-gather in one pass: chunk c (grid.y) of buffer c to every other buffer.
__global__ void __launch_bounds__(kThreads) k_ring_ag_fused(RankPtrs b, int n, long long size) {
  griddep_wait();
  griddep_launch_dependents();
  const int c = blockIdx.y;
  long long lo, hi, vlo, vhi;
  chunk_range(size, n, c, lo, hi);
  split_vec(lo, hi, vlo, vhi);
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const float *src = b.p[c];
  if (t < vlo - lo)
    for (int r = 0; r < n; ++r)
      if (r != c) b.p[r][lo + t] = src[lo + t];
  if (t < hi - vhi)
    for (int r = 0; r < n; ++r)
      if (r != c) b.p[r][vhi + t] = src[vhi + t];
  const long long v0 = vlo >> 2, nv = (vhi - vlo) >> 2;
  for (long long i = t; i < nv; i += stride) {
    const float4 v = reinterpret_cast<const float4 *>(src)[v0 + i];
    for (int r = 0; r < n; ++r)
      if (r != c) reinterpret_cast<float4 *>(b.p[r])[v0 + i] = v;
  }
}

template <typename U>
__device__ __forceinline__ void copy_rows(const Copy2D &cp) {
  const long long upr = cp.row_bytes / static_cast<long long>(sizeof(U));
  for (long long row = blockIdx.x; row < cp.rows; row += gridDim.x) {
    const U *s = reinterpret_cast<const U *>(cp.src + row * cp.src_pitch);
    U *d = reinterpret_cast<U *>(cp.dst + row * cp.dst_pitch);
    for (long long u = threadIdx.x; u < upr; u += blockDim.x) d[u] = s[u];
  }
}

// grid.y = copy index; each copy moves `rows` rows of `row_bytes` bytes in the
// widest unit that divides every address, pitch and row length.
__global__ void __launch_bounds__(kThreads) k_copy_batch(const __grid_constant__ CopyBatch b) {
  griddep_wait();
  griddep_launch_dependents();
  const Copy2D &cp = b.c[blockIdx.y];
  const unsigned long long bits = reinterpret_cast<unsigned long long>(cp.src) |
                                  reinterpret_cast<unsigned long long>(cp.dst) |
                                  static_cast<unsigned long long>(cp.src_pitch) |
                                  static_cast<unsigned long long>(cp.dst_pitch) |
                                  static_cast<unsigned long long>(cp.row_bytes);
  if ((bits & 15) == 0)
    copy_rows<uint4>(cp);
  else if ((bits & 7) == 0)
    copy_rows<uint2>(cp);
  else if ((bits & 3) == 0)
    copy_rows<uint32_t>(cp);
  else if ((bits & 1) == 0)
    copy_rows<uint16_t>(cp);
  else
    copy_rows<uint8_t>(cp);
}

// An mbarrier that expects one arrival nobody makes: the bounded wait always
// runs out and records a timeout.
__global__ void k_debug_wait(int *status, long long wait_ns) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(1) : "memory");
    bool done = false;
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (!done) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(a), "r"(0)
          : "memory");
      if (ok) break;
      unsigned long long t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
      if (static_cast<long long>(t1 - t0) > wait_ns) done = true;
    }
    if (done) atomicCAS(status, 0, kDevTimeoutDebug);
  }
}

// Blocks per grid row: about four float4 per thread when the buffers are large
// (several loads in flight per thread), one per thread when that would leave SMs
// idle, at most four blocks per SM in total.
int blocks_for(long long elems, int ranks_in_grid) {
  const long long rows = ranks_in_grid > 0 ? ranks_in_grid : 1;
  long long vec_threads = (elems / 4 + 4 * kThreads - 1) / (4 * kThreads);
  if (vec_threads * rows < 2LL * num_sms()) vec_threads = (elems / 4 + kThreads - 1) / kThreads;
  long long cap = static_cast<long long>(num_sms()) * 4 / rows;
  if (cap < 1) cap = 1;
  long long g = vec_threads < cap ? vec_threads : cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

tp_status check_launch() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_fail(e);
}

tp_status launch_checked(cudaError_t e) {
  if (e != cudaSuccess) return cuda_fail(e);
  return check_launch();
}


// One-pass reduce-scatter into bf16 (grid.y = chunk): every element of chunk c
// is folded over the ranks in the ring's order c+1, c+2, ..., c in f32, exactly
// as k_ring_fused does, then rounded once to bf16 (nearest even) and stored in
// buffer c's row-major [rows x cols] matrix with row pitch ld. Flat element e
// sits at row e / cols, column e % cols. The partials are read once, with
// streaming (evict-first) loads, so that they do not push the bf16 chunks just
// written out of L2: the next kernel, a GEMM over the chunks, reads them there.
template <int NT>
__global__ void __launch_bounds__(kThreads) k_ring_rs_bf16(RankPtrs b, Bf16Outs o, int n_rt, long long size) {
  griddep_wait();
  griddep_launch_dependents();
  const int n = NT ? NT : n_rt;
  const int c = blockIdx.y;
  long long lo, hi;
  chunk_range(size, n, c, lo, hi);
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(o.p[c]);
  const bool small = size < (1LL << 31);
  auto at = [&](long long e) {
    long long row, col;
    if (small) {
      const unsigned int ue = static_cast<unsigned int>(e), uc = static_cast<unsigned int>(o.cols);
      row = ue / uc;
      col = ue - static_cast<unsigned int>(row) * uc;
    } else {
      row = e / o.cols;
      col = e - row * o.cols;
    }
    return out + row * o.ld + col;
  };
  auto fold1 = [&](long long e) {
    float acc = b.p[(c + 1) % n][e];
    for (int j = 2; j <= n; ++j) acc = acc + b.p[(c + j) % n][e];
    return acc;
  };
  if ((o.cols & 3) != 0) {  // rows not in whole float4 units: scalar throughout
    for (long long e = lo + t; e < hi; e += stride) *at(e) = __float2bfloat16_rn(fold1(e));
    return;
  }
  long long vlo, vhi;
  split_vec(lo, hi, vlo, vhi);
  if (t < vlo - lo) *at(lo + t) = __float2bfloat16_rn(fold1(lo + t));
  if (t < hi - vhi) *at(vhi + t) = __float2bfloat16_rn(fold1(vhi + t));
  const long long v0 = vlo >> 2, v1 = vhi >> 2;
  for (long long i = v0 + t; i < v1; i += stride) {
    float4 a;
    if constexpr (NT > 0) {
      float4 x[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) x[j] = __ldcs(reinterpret_cast<const float4 *>(b.p[(c + 1 + j) % NT]) + i);
      a = x[0];
#pragma unroll
      for (int j = 1; j < NT; ++j) a = add4(a, x[j]);
    } else {
      a = __ldcs(reinterpret_cast<const float4 *>(b.p[(c + 1) % n]) + i);
      for (int j = 2; j <= n; ++j) a = add4(a, __ldcs(reinterpret_cast<const float4 *>(b.p[(c + j) % n]) + i));
    }
    // four elements of one row (cols is a multiple of 4): one 8-byte store
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y), h1 = __floats2bfloat162_rn(a.z, a.w);
    uint2 w;
    w.x = *reinterpret_cast<const unsigned int *>(&h0);
    w.y = *reinterpret_cast<const unsigned int *>(&h1);
    *reinterpret_cast<uint2 *>(at(i * 4)) = w;
  }
}

}  // namespace

tp_status launch_ring_rs_step(const RankPtrs &b, int n, long long size, int step, cudaStream_t s) {
  const dim3 grid(blocks_for(size / n + 4, n), n);
  return launch_checked(launch_kernel(k_ring_rs_step, grid, dim3(kThreads), 0, s, 1, b, n, size, step));
}

tp_status launch_ring_ag_step(const RankPtrs &b, int n, long long size, int step, cudaStream_t s) {
  const dim3 grid(blocks_for(size / n + 4, n), n);
  return launch_checked(launch_kernel(k_ring_ag_step, grid, dim3(kThreads), 0, s, 1, b, n, size, step));
}

tp_status launch_ring_fused(const RankPtrs &b, int n, long long size, int write_all,
                            cudaStream_t s) {
  const dim3 grid(blocks_for(size / n + 4, n), n);
  void (*k)(RankPtrs, int, long long, int) = n == 2   ? k_ring_fused<2>
                                            : n == 4 ? k_ring_fused<4>
                                            : n == 8 ? k_ring_fused<8>
                                                     : k_ring_fused<0>;
  return launch_checked(launch_kernel(k, grid, dim3(kThreads), 0, s, 1, b, n, size, write_all));
}

tp_status launch_ring_rs_bf16(const RankPtrs &b, const Bf16Outs &o, int n, long long size, cudaStream_t s) {
  const dim3 grid(blocks_for(size / n + 4, n), n);
  void (*k)(RankPtrs, Bf16Outs, int, long long) = n == 2   ? k_ring_rs_bf16<2>
                                                  : n == 4 ? k_ring_rs_bf16<4>
                                                  : n == 8 ? k_ring_rs_bf16<8>
                                                           : k_ring_rs_bf16<0>;
  return launch_checked(launch_kernel(k, grid, dim3(kThreads), 0, s, 1, b, o, n, size));
}

tp_status launch_ring_ag_fused(const RankPtrs &b, int n, long long size, cudaStream_t s) {
  const dim3 grid(blocks_for(size / n + 4, n), n);
  return launch_checked(launch_kernel(k_ring_ag_fused, grid, dim3(kThreads), 0, s, 1, b, n, size));
}

tp_status launch_copy_batch(const CopyBatch &b, cudaStream_t s) {
  if (b.n == 0) return TP_OK;
  long long rows = 1;
  for (int i = 0; i < b.n; ++i) rows = b.c[i].rows > rows ? b.c[i].rows : rows;
  long long gx = static_cast<long long>(num_sms()) * 4 / b.n;
  if (gx < 1) gx = 1;
  if (gx > rows) gx = rows;
  return launch_checked(
      launch_kernel(k_copy_batch, dim3(static_cast<unsigned>(gx), b.n), dim3(kThreads), 0, s, 1, b));
}

tp_status launch_debug_wait(cudaStream_t s) {
  DevCtx ctx;
  const cudaError_t e = get_dev_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e);
  k_debug_wait<<<1, 32, 0, s>>>(ctx.status, ctx.wait_ns);
  note_launch();
  return check_launch();
}

}  // namespace tpgqa
