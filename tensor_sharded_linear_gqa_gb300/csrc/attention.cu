// Attention core between the q/k/v projections and o_proj, per rank on its own
// q heads (mlxcel manual "텐서 병렬화", GQA 인식 어텐션 샤딩 / GQA-aware attention
// sharding: each rank's q heads attend with the kv heads the shard plan maps
// them to, its own kv heads when K/V are sharded, all of them when replicated).
// A_h = softmax(Q_h K_g^T / sqrt(d)) V_g, causal (query i sees keys j <= i) or
// full, d = 128.
//
// k_attention: one CTA per (128-query tile, q head); causal grids run the
// longest query tiles first. Warp roles:
//   warp 0     TMA producer: the Q tile once, then K and V^T tiles of 128 keys
//              through a 2-stage ring (V is transposed beforehand, so every MMA
//              operand is a K-major, 128-byte-swizzled tile);
//   warp 1     MMA issuer: S_j = Q K_j^T (M=128, N=128 keys, K=128) into one of
//              two TMEM buffers, then O += P_j V_j (N=128, K=128 keys) into a
//              third that accumulates over the key blocks; S_{j+1} is issued
//              before P_j V_j so it overlaps the softmax;
//   warps 2-5  softmax: one thread per query row (TMEM lane). Pass 1 takes the
//              row maximum of S_j; the row's reference maximum m moves only when
//              the block's maximum exceeds it by more than 8 (in log2 units),
//              and then the row of O is rescaled in TMEM by 2^(m_old - m_new)
//              after the previous P V has landed; so p = exp2(s*c - m) <= 2^8.
//              Pass 2 writes p as bf16 into the shared-memory P tile (K-major,
//              swizzled) and sums it into the row sum l. At the end O / l.
// Every wait is bounded; on a timeout the kernel records it, stops issuing,
// drains its TMA loads, frees TMEM and returns.
//
// k_transpose_bf16: V [T x C] -> V^T [C x T] through 64 x 64 shared tiles.
#include <cuda_bf16.h>

#include <cstring>

#include "sm100_ptx.cuh"
#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr int kAttnThreads = 192;
constexpr int kTileQ = 128, kTileK = 128, kHd = 128;
constexpr uint32_t kSub = 128u * 128u;            // one [128 rows x 64 bf16] swizzled k-tile
constexpr uint32_t kTile = 2 * kSub;              // a [128 x 128] bf16 operand tile
constexpr uint32_t kSmemQ = 0, kSmemK = kTile, kSmemV = 3 * kTile, kSmemP = 5 * kTile;
constexpr uint32_t kSmemBar = 6 * kTile;          // barriers after the six tiles
constexpr size_t kAttnSmem = 6 * kTile + 1024 + 256;  // + alignment slack + barriers
constexpr uint32_t kTmemCols = 512;               // S0, S1, O at columns 0, 128, 256

__device__ __forceinline__ void record(int *status, int code) { atomicCAS(status, 0, code); }

tp_status launch_checked(cudaError_t e) {
  if (e != cudaSuccess) return cuda_fail(e);
  const cudaError_t l = cudaGetLastError();
  return l == cudaSuccess ? TP_OK : cuda_fail(l);
}

__global__ void __launch_bounds__(kAttnThreads, 1) k_attention(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t sQ = sbase + kSmemQ, sK0 = sbase + kSmemK, sV0 = sbase + kSmemV, sP = sbase + kSmemP;
  uint8_t *bar_area = smem + kSmemBar;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  const uint32_t q_full = bar0, kv_full0 = bar0 + 8, kv_empty0 = bar0 + 24, s_full0 = bar0 + 40,
                 p_full = bar0 + 56, o_full = bar0 + 64, drain = bar0 + 72;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 96);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 100);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work item: causal grids start with the last (longest) query tiles
  const int qt = p.causal ? p.q_tiles - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  const int head = blockIdx.y;
  const AttnHead hd = p.heads[head];
  const int q0 = qt * kTileQ;
  const int nb = p.causal ? qt + 1 : (p.tokens + kTileK - 1) / kTileK;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(kv_full0 + 8 * s, 1);
      ptx::mbar_init(kv_empty0 + 8 * s, 1);
      ptx::mbar_init(s_full0 + 8 * s, 1);
    }
    ptx::mbar_init(p_full, 128);
    ptx::mbar_init(o_full, 1);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&p.maps[hd.q_map]);
    ptx::prefetch_tensormap(&p.maps[hd.k_map]);
    ptx::prefetch_tensormap(&p.maps[hd.v_map]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  int issued[2] = {0, 0};  // loads started per KV stage (producer thread)
  bool q_issued = false;
  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(q_full, kTile);
      for (int c = 0; c < 2; ++c)
        ptx::tma_load_2d(sQ + c * kSub, &p.maps[hd.q_map], hd.q_col + c * 64, q0, q_full);
      q_issued = true;
      for (int j = 0; j < nb; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (*abort_flag) break;
        if (!ptx::mbar_wait(kv_empty0 + 8 * s, ph ^ 1, p.wait_ns)) {
          record(p.status, kDevTimeoutProducer);
          *abort_flag = 1;
          break;
        }
        ptx::mbar_arrive_expect_tx(kv_full0 + 8 * s, 2 * kTile);
        for (int c = 0; c < 2; ++c) {
          ptx::tma_load_2d(sK0 + s * kTile + c * kSub, &p.maps[hd.k_map], hd.kv_col + c * 64, j * kTileK,
                           kv_full0 + 8 * s);
          ptx::tma_load_2d(sV0 + s * kTile + c * kSub, &p.maps[hd.v_map], j * kTileK + c * 64, hd.kv_col,
                           kv_full0 + 8 * s);
        }
        ++issued[s];
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileQ, 128);
      bool ok = ptx::mbar_wait(q_full, 0, p.wait_ns);
      if (!ok) record(p.status, kDevTimeoutMma);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (*abort_flag || !ptx::mbar_wait(kv_full0 + 8 * s, (j >> 1) & 1, p.wait_ns)) {
          if (!*abort_flag) record(p.status, kDevTimeoutMma);
          return false;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(s * 128);
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(sQ + (kk >> 2) * kSub) + 2 * (kk & 3);
          const uint64_t bd = ptx::smem_desc_sw128(sK0 + s * kTile + (kk >> 2) * kSub) + 2 * (kk & 3);
          ptx::mma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full0 + 8 * s);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nb; ++j) {
        if (j + 1 < nb && !issue_s(j + 1)) { ok = false; break; }
        // O += P_j V_j once the softmax has written P_j (and rescaled O if needed)
        if (*abort_flag || !ptx::mbar_wait(p_full, j & 1, p.wait_ns)) {
          if (!*abort_flag) record(p.status, kDevTimeoutMma);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const int s = j & 1;
        const uint32_t d = tmem + 256u;
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(sP + (kk >> 2) * kSub) + 2 * (kk & 3);
          const uint64_t bd = ptx::smem_desc_sw128(sV0 + s * kTile + (kk >> 2) * kSub) + 2 * (kk & 3);
          ptx::mma_bf16(d, ad, bd, idesc, (j | kk) > 0 ? 1u : 0u);
        }
        ptx::mma_commit(o_full);
        ptx::mma_commit(kv_empty0 + 8 * s);
      }
      if (!ok) *abort_flag = 1;
      ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    // ---- softmax: warp w reads TMEM lanes [32*(w%4), +32); one query row per thread ----
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    const int qrow = q0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t ob = tmem + lane_off + 256u;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // waits for O += P_{j} V_{j} to land (the P tile is free again, O is current)
    auto wait_o = [&](int j) -> bool {
      const bool ready = ptx::mbar_wait(o_full, j & 1, p.wait_ns);
      if (!__all_sync(0xffffffffu, ready && *abort_flag == 0)) {
        if (lane == 0) {
          if (!ready) record(p.status, kDevTimeoutEpilogue);
          *abort_flag = 1;
        }
        return false;
      }
      ptx::tc_fence_after();
      return true;
    };
    for (int j = 0; j < nb; ++j) {
      const int s = j & 1;
      const bool ready = ptx::mbar_wait(s_full0 + 8 * s, (j >> 1) & 1, p.wait_ns);
      if (!__all_sync(0xffffffffu, ready && *abort_flag == 0)) {
        if (lane == 0) {
          if (!ready) record(p.status, kDevTimeoutEpilogue);
          *abort_flag = 1;
        }
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t sb = tmem + lane_off + static_cast<uint32_t>(s * 128);
      const int k0 = j * kTileK;
      // keys past the query (causal) or past the sequence are masked
      const int lim = min(p.causal ? qrow - k0 + 1 : kTileK, p.tokens - k0);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32cols(sb + c * 32, v);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c * 32 + i < lim) mx = fmaxf(mx, __uint_as_float(v[i]));
      }
      const float m_blk = mx * p.scale_log2;
      const bool move = m_blk > m + 8.f;  // always on the first block (m = -inf)
      const float m_new = move ? m_blk : m;
      const float alpha = move ? exp2f(m - m_new) : 1.f;  // 0 on the first block
      if (j > 0) {
        if (!wait_o(j - 1)) { ok = false; break; }
        if (__any_sync(0xffffffffu, move)) {
          // rescale this warp's rows of O (lanes that keep their maximum scale by 1)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            ptx::tmem_ld_32cols(ob + c * 32, v);
            ptx::tmem_ld_wait();
            ptx::tmem_regs_ready(v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            ptx::tmem_st_32cols(ob + c * 32, v);
          }
          ptx::tmem_st_wait();
        }
      }
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32cols(sb + c * 32, v);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float a0 = c * 32 + i < lim ? exp2f(__uint_as_float(v[i]) * p.scale_log2 - m_new) : 0.f;
          const float a1 = c * 32 + i + 1 < lim ? exp2f(__uint_as_float(v[i + 1]) * p.scale_log2 - m_new) : 0.f;
          lsum += a0 + a1;
          const __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
          memcpy(&packed[i >> 1], &h, 4);
        }
        // keys [32c, 32c+32) of this row: k-tile c/2, 16-byte chunks (c%2)*4 .. +3, swizzled by row
        const uint32_t rbase = sP + (c >> 1) * kSub + row * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t chunk = static_cast<uint32_t>(((c & 1) * 4 + u) ^ (row & 7));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rbase + chunk * 16),
                       "r"(packed[4 * u]), "r"(packed[4 * u + 1]), "r"(packed[4 * u + 2]), "r"(packed[4 * u + 3])
                       : "memory");
        }
      }
      l = l * alpha + lsum;
      m = m_new;
      ptx::fence_proxy_async_smem();  // P visible to the tensor core
      ptx::tc_fence_before();
      ptx::mbar_arrive(p_full);
    }
    if (ok && wait_o(nb - 1)) {
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32cols(ob + c * 32, v);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        if (qrow < p.tokens) {
          __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(hd.out) + static_cast<long long>(qrow) * hd.out_ld + c * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[i + 4]) * inv, __uint_as_float(v[i + 5]) * inv);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(__uint_as_float(v[i + 6]) * inv, __uint_as_float(v[i + 7]) * inv);
            memcpy(&w.x, &h0, 4);
            memcpy(&w.y, &h1, 4);
            memcpy(&w.z, &h2, 4);
            memcpy(&w.w, &h3, 4);
            *reinterpret_cast<uint4 *>(dst + i) = w;
          }
        }
      }
    }
  }

  // ---- teardown: every TMA load this CTA started has landed before it exits ----
  __syncthreads();
  if (warp == 0 && lane == 0) {
    if (q_issued && !ptx::mbar_wait(q_full, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    for (int s = 0; s < 2; ++s)
      if (issued[s] > 0 && !ptx::mbar_wait(kv_full0 + 8 * s, (issued[s] - 1) & 1, p.wait_ns))
        record(p.status, kDevTimeoutDrain);
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// V [T x C] (row pitch ld_in) -> V^T [C x T] (row pitch ld_out), 64 x 64 tiles.
__global__ void __launch_bounds__(256) k_transpose_bf16(const __nv_bfloat16 *in, long long ld_in,
                                                        __nv_bfloat16 *out, long long ld_out, int rows,
                                                        int cols) {
  __shared__ __nv_bfloat16 tile[64][66];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int r0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int r = i / 64, c = i % 64;
    if (r0 + r < rows && c0 + c < cols) tile[r][c] = in[static_cast<long long>(r0 + r) * ld_in + c0 + c];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int c = i / 64, r = i % 64;
    if (r0 + r < rows && c0 + c < cols) out[static_cast<long long>(c0 + c) * ld_out + r0 + r] = tile[r][c];
  }
}

}  // namespace

tp_status launch_transpose_bf16(const void *in, long long ld_in, void *out, long long ld_out, int rows, int cols,
                                cudaStream_t s) {
  if (rows == 0 || cols == 0) return TP_OK;
  const dim3 grid((rows + 63) / 64, (cols + 63) / 64);
  return launch_checked(launch_kernel(k_transpose_bf16, grid, dim3(256), 0, s, 1,
                                      static_cast<const __nv_bfloat16 *>(in), ld_in,
                                      static_cast<__nv_bfloat16 *>(out), ld_out, rows, cols));
}

tp_status launch_attention(AttnParams &p, int total_heads, cudaStream_t s) {
  DevCtx ctx;
  cudaError_t e = get_dev_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e);
  p.status = ctx.status;
  p.wait_ns = ctx.wait_ns;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(k_attention, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kAttnSmem));
    if (e != cudaSuccess) return cuda_fail(e);
    attr_set = true;
  }
  const dim3 grid(static_cast<unsigned>(p.q_tiles), static_cast<unsigned>(total_heads));
  return launch_checked(launch_kernel(k_attention, grid, dim3(kAttnThreads), kAttnSmem, s, 1, p));
}

}  // namespace tpgqa
