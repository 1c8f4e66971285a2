// Attention core between the q/k/v projections and o_proj, per rank on its own
// q heads (mlxcel manual "텐서 병렬화", GQA 인식 어텐션 샤딩 / GQA-aware attention
// sharding: each rank's q heads attend with the kv heads the shard plan maps
// them to, its own kv heads when K/V are sharded, all of them when replicated).
// A_h = softmax(Q_h K_g^T / sqrt(d)) V_g, causal (query i sees keys j <= i) or
// full, d = 128.
//
// k_attention: persistent, one CTA per SM walking (128-query tile, q head) work
// items, the longest causal query tiles first; TMEM, barriers and the pipeline
// phases carry over from item to item. Warp roles:
//   warp 0     TMA producers: lane 0 loads each item's Q tile (as soon as the
//              previous item's last S = Q K^T has read the last one) and K tiles of 128
//              keys through a 2-stage ring, lane 1 V^T tiles through another (V
//              is transposed beforehand, so every MMA operand is a K-major,
//              128-byte-swizzled tile). A K stage frees when its S = Q K^T is
//              done, two blocks before the V stage beside it;
//   warp 1     MMA issuer: S_j = Q K_j^T (M=128, N=128 keys, K=128) into one of
//              two TMEM buffers, then O += P_j V_j (N=128, K=128 keys) into a
//              third that accumulates over the key blocks; S_{j+1} is issued
//              before P_j V_j so it overlaps the softmax;
//   warps 2-9  softmax: two threads per query row (TMEM lane), warps w and w+4
//              taking keys and output columns [0, 64) and [64, 128). They take the
//              row maximum of S_j and combine it through shared memory (a bounded
//              mbarrier handshake per warp pair); the row's reference maximum m moves only when
//              the block's maximum exceeds it by more than 8 (in log2 units),
//              and then the row of O is rescaled in TMEM by 2^(m_old - m_new)
//              after the previous P V has landed; so p = exp2(s*c - m) <= 2^8.
//              Pass 2 writes p as bf16 into the shared-memory P tile (K-major,
//              swizzled) and sums it into the row sum l. At the end of an item
//              O / l is stored and the MMA warp is told O is free again.
// Every wait is bounded; on a timeout the kernel records it, stops issuing,
// drains its TMA loads, frees TMEM and returns.
//
// k_transpose_bf16: V [T x C] -> V^T [C x T] through 64 x 64 shared tiles.
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "sm100_ptx.cuh"
#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr int kAttnThreads = 320;  // producer warp, MMA warp, 8 softmax warps
constexpr int kTileQ = 128, kTileK = 128, kHd = 128;
constexpr uint32_t kSub = 128u * 128u;            // one [128 rows x 64 bf16] swizzled k-tile
constexpr uint32_t kTile = 2 * kSub;              // a [128 x 128] bf16 operand tile
constexpr uint32_t kSmemQ = 0, kSmemK = kTile, kSmemV = 3 * kTile, kSmemP = 5 * kTile;  // P: 2 tiles
constexpr uint32_t kSmemBar = 7 * kTile;          // barriers after the seven tiles (176 bytes)
constexpr uint32_t kSmemRed = kSmemBar + 192;      // row-maximum / row-sum exchange, [2][128] f32
constexpr size_t kAttnSmem = kSmemRed + 1024 + 1024;  // + the exchange + alignment slack (226.1 KB)
constexpr uint32_t kTmemCols = 512;               // S0, S1, O at columns 0, 128, 256

__device__ __forceinline__ void record(int *status, int code) { atomicCAS(status, 0, code); }

// max(a, b, c) in one instruction (three-input max.f32).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two f32 lanes in one 64-bit register, and the packed (f32x2) add and fma.
__device__ __forceinline__ uint64_t pack2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 2^x by the SFU's approximate base-2 exponential (PTX ex2.approx.ftz.f32):
// relative error of order 2^-22, far below the bf16 rounding P goes through next.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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
  const uint32_t q_full = bar0, q_empty = bar0 + 8, k_full0 = bar0 + 16, k_empty0 = bar0 + 32,
                 v_full0 = bar0 + 48, v_empty0 = bar0 + 64, s_full0 = bar0 + 80, p_full = bar0 + 96,
                 p_empty0 = bar0 + 104, o_free = bar0 + 120, drain = bar0 + 128;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 136);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 140);
  const uint32_t xbar0 = bar0 + 144;  // one exchange barrier per softmax warp pair

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = p.q_tiles * p.heads_total;
  // work item -> (query tile, head); causal runs the longest query tiles first
  auto item = [&](int it, int &qt, int &nb) -> const AttnHead & {
    const int r = it / p.heads_total;
    qt = p.causal ? p.q_tiles - 1 - r : r;
    nb = p.causal ? qt + 1 : (p.tokens + kTileK - 1) / kTileK;
    return p.heads[it % p.heads_total];
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(k_full0 + 8 * s, 1);
      ptx::mbar_init(k_empty0 + 8 * s, 1);
      ptx::mbar_init(v_full0 + 8 * s, 1);
      ptx::mbar_init(v_empty0 + 8 * s, 1);
      ptx::mbar_init(s_full0 + 8 * s, 1);
      ptx::mbar_init(p_empty0 + 8 * s, 1);
    }
    ptx::mbar_init(p_full, 256);
    ptx::mbar_init(o_free, 256);
    ptx::mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) ptx::mbar_init(xbar0 + 8 * q, 64);
    *abort_flag = 0;
    ptx::fence_barrier_init();
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

  // Pipeline phases run on counters over this CTA's whole sequence of items:
  // ic (items started) and g (key blocks, over all items).
  int issued[2] = {0, 0};  // loads started per stage of this producer lane's ring
  int q_loads = 0;
  if (warp == 0) {
    if (lane < 2) {
      // lane 0: Q of each item, then the K ring; lane 1: the V^T ring
      const uint32_t full0 = lane == 0 ? k_full0 : v_full0, empty0 = lane == 0 ? k_empty0 : v_empty0;
      const uint32_t dst0 = lane == 0 ? sK0 : sV0;
      bool run = true;
      int g = 0;
      for (int it = blockIdx.x, ic = 0; run && it < items; it += gridDim.x, ++ic) {
        int qt, nb;
        const AttnHead &hd = item(it, qt, nb);
        if (lane == 0) {
          // the previous item's last S = Q K^T has read Q
          if (*abort_flag || !ptx::mbar_wait(q_empty, (ic & 1) ^ 1, p.wait_ns)) {
            if (!*abort_flag) record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            break;
          }
          ptx::mbar_arrive_expect_tx(q_full, kTile);
          for (int c = 0; c < 2; ++c)
            ptx::tma_load_2d(sQ + c * kSub, &p.maps[hd.q_map], hd.q_col + c * 64, qt * kTileQ, q_full);
          ++q_loads;
        }
        const CUtensorMap *map = &p.maps[lane == 0 ? hd.k_map : hd.v_map];
        for (int j = 0; j < nb; ++j, ++g) {
          const int s = g & 1;
          if (*abort_flag || !ptx::mbar_wait(empty0 + 8 * s, ((g >> 1) & 1) ^ 1, p.wait_ns)) {
            if (!*abort_flag) record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            run = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full0 + 8 * s, kTile);
          for (int c = 0; c < 2; ++c) {
            if (lane == 0)
              ptx::tma_load_2d(dst0 + s * kTile + c * kSub, map, hd.kv_col + c * 64, j * kTileK, full0 + 8 * s);
            else
              ptx::tma_load_2d(dst0 + s * kTile + c * kSub, map, j * kTileK + c * 64, hd.kv_col, full0 + 8 * s);
          }
          ++issued[s];
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileQ, 128);
      bool ok = true;
      auto fail = [&]() {
        if (!*abort_flag) record(p.status, kDevTimeoutMma);
        ok = false;
      };
      // S_g = Q K_g^T into TMEM buffer g % 2 (free: its previous S was read before
      // the softmax signalled p_full for that block, which this thread waited on)
      auto issue_s = [&](int g) {
        const int s = g & 1;
        if (*abort_flag || !ptx::mbar_wait(k_full0 + 8 * s, (g >> 1) & 1, p.wait_ns)) return fail();
        ptx::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(s * 128);
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(sQ + (kk >> 2) * kSub) + 2 * (kk & 3);
          const uint64_t bd = ptx::smem_desc_sw128(sK0 + s * kTile + (kk >> 2) * kSub) + 2 * (kk & 3);
          ptx::mma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full0 + 8 * s);
        ptx::mma_commit(k_empty0 + 8 * s);
      };
      int g = 0;
      for (int it = blockIdx.x, ic = 0; ok && it < items; it += gridDim.x, ++ic) {
        int qt, nb;
        item(it, qt, nb);
        // this item's Q has landed
        if (*abort_flag || !ptx::mbar_wait(q_full, ic & 1, p.wait_ns)) {
          fail();
          break;
        }
        issue_s(g);
        if (ok && nb == 1) ptx::mma_commit(q_empty);
        for (int j = 0; ok && j < nb; ++j, ++g) {
          if (j + 1 < nb) {
            issue_s(g + 1);
            if (!ok) break;
            if (j + 2 == nb) ptx::mma_commit(q_empty);  // the item's last S is issued
          }
          // O += P_g V_g once the softmax has written P_g (and rescaled O if needed);
          // the item's first one overwrites O, so the previous item's output must
          // have been read from it
          if (*abort_flag || !ptx::mbar_wait(p_full, g & 1, p.wait_ns) ||
              !ptx::mbar_wait(v_full0 + 8 * (g & 1), (g >> 1) & 1, p.wait_ns) ||
              (j == 0 && !ptx::mbar_wait(o_free, (ic & 1) ^ 1, p.wait_ns))) {
            fail();
            break;
          }
          ptx::tc_fence_after();
          const int s = g & 1;
          const uint32_t d = tmem + 256u;
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {
            const uint64_t ad = ptx::smem_desc_sw128(sP + s * kTile + (kk >> 2) * kSub) + 2 * (kk & 3);
            const uint64_t bd = ptx::smem_desc_sw128(sV0 + s * kTile + (kk >> 2) * kSub) + 2 * (kk & 3);
            ptx::mma_bf16(d, ad, bd, idesc, (j | kk) > 0 ? 1u : 0u);
          }
          ptx::mma_commit(p_empty0 + 8 * s);  // P_g read, O current up to block g
          ptx::mma_commit(v_empty0 + 8 * s);
        }
      }
      if (!ok) *abort_flag = 1;
      ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    // ---- softmax: warps w and w+4 read TMEM lanes [32*(w%4), +32); a thread pair per row ----
    const int qw = warp & 3;
    const int half = (warp - 2) >> 2;  // 0: keys / output columns [0, 64), 1: [64, 128)
    const int row = qw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t ob = tmem + lane_off + 256u + 64u * half;
    const uint32_t xbar = xbar0 + 8 * qw;  // the two warps sharing these rows
    volatile float *red = reinterpret_cast<volatile float *>(smem + kSmemRed);
    bool ok = true;
    // A bounded warp-wide wait; on a timeout (or another role's abort) the warp gives up.
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool ready = ptx::mbar_wait(bar, parity, p.wait_ns);
      if (!__all_sync(0xffffffffu, ready && *abort_flag == 0)) {
        if (lane == 0) {
          if (!ready) record(p.status, kDevTimeoutEpilogue);
          *abort_flag = 1;
        }
        return false;
      }
      return true;
    };
    // The partner's value of this row through shared memory. Each exchange takes
    // two phases of the pair's barrier: both values written, then both read (so
    // the next exchange cannot overwrite a value not yet read).
    auto exchange = [&](float x, float &y) -> bool {
      red[half * 128 + row] = x;
      ptx::mbar_arrive(xbar);
      if (!wait_all(xbar, 0)) return false;
      y = red[(half ^ 1) * 128 + row];
      ptx::mbar_arrive(xbar);
      return wait_all(xbar, 1);
    };
    // O += P_i V_i has landed: P tile i % 2 is free and O is current up to block i
    // (tcgen05 operations complete in issue order)
    auto wait_pv = [&](int i) -> bool {
      if (!wait_all(p_empty0 + 8 * (i & 1), (i >> 1) & 1)) return false;
      ptx::tc_fence_after();
      return true;
    };
    const int c0 = 64 * half;  // first key of this thread's half
    int g = 0;
    for (int it = blockIdx.x; ok && it < items; it += gridDim.x) {
      int qt, nb;
      const AttnHead &hd = item(it, qt, nb);
      const int qrow = qt * kTileQ + row;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nb; ++j, ++g) {
        const int s = g & 1;
        if (!wait_all(s_full0 + 8 * s, (g >> 1) & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t sb = tmem + lane_off + static_cast<uint32_t>(s * 128 + c0);
        const int k0 = j * kTileK;
        // keys past the query (causal) or past the sequence are masked
        const int lim = min(p.causal ? qrow - k0 + 1 : kTileK, p.tokens - k0) - c0;
        uint32_t v[64];
        {
          uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
          uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
          ptx::tmem_ld_32cols(sb, v0);
          ptx::tmem_ld_32cols(sb + 32, v1);
          ptx::tmem_ld_wait();
          ptx::tmem_regs_ready(v);
        }
        if (!__all_sync(0xffffffffu, lim >= 64)) {  // a masked key in this warp's half
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i >= lim) v[i] = __float_as_uint(-INFINITY);
        }
        float mx = __uint_as_float(v[63]);
#pragma unroll
        for (int i = 0; i < 62; i += 2) mx = max3f(mx, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        mx = fmaxf(mx, __uint_as_float(v[62]));
        float mx2;
        if (!exchange(mx, mx2)) { ok = false; break; }
        mx = fmaxf(mx, mx2);
        const float m_blk = mx * p.scale_log2;
        const bool move = m_blk > m + 8.f;  // always on the item's first block (m = -inf)
        const float m_new = move ? m_blk : m;
        const float alpha = move ? exp2f(m - m_new) : 1.f;  // 0 on the first block
        bool pv1_done = false;
        if (j > 0 && __any_sync(0xffffffffu, move)) {
          if (!wait_pv(g - 1)) { ok = false; break; }
          pv1_done = true;
          // rescale this thread's half of the row of O (rows keeping their maximum scale by 1)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            ptx::tmem_ld_32cols(ob + c * 32, o);
            ptx::tmem_ld_wait();
            ptx::tmem_regs_ready(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            ptx::tmem_st_32cols(ob + c * 32, o);
          }
          ptx::tmem_st_wait();
        }
        // P tile s was last read by P_{g-2} V_{g-2}
        if (g >= 2 && !pv1_done && !wait_pv(g - 2)) { ok = false; break; }
        // p = 2^(s*c - m) two lanes at a time (packed f32x2 fma and sum)
        const uint64_t c2 = pack2(p.scale_log2, p.scale_log2), nm2 = pack2(-m_new, -m_new);
        uint64_t sum2 = pack2(0.f, 0.f);
        // k-tile `half` of the P tile holds this thread's 64 keys
        const uint32_t pbase = sP + s * kTile + half * kSub + row * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // keys [8q, 8q+8) of the half: one 16-byte chunk
          uint32_t packed[4];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            float y0, y1;
            unpack2(fma2(pack2(__uint_as_float(v[8 * q + i]), __uint_as_float(v[8 * q + i + 1])), c2, nm2), y0, y1);
            const float a0 = ex2_approx(y0), a1 = ex2_approx(y1);
            sum2 = add2(sum2, pack2(a0, a1));
            const __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
            memcpy(&packed[i >> 1], &h, 4);
          }
          const uint32_t addr = pbase + static_cast<uint32_t>((q ^ (row & 7)) * 16);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[0]), "r"(packed[1]),
                       "r"(packed[2]), "r"(packed[3])
                       : "memory");
        }
        float s0, s1;
        unpack2(sum2, s0, s1);
        l = l * alpha + (s0 + s1);
        m = m_new;
        ptx::fence_proxy_async_smem();  // P visible to the tensor core
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full);
      }
      if (!ok) break;
      // the item's output: O / l once its last P V has landed
      float l2 = 0.f;
      if (!wait_pv(g - 1) || !exchange(l, l2)) { ok = false; break; }
      const float inv = 1.f / (l + l2);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32cols(ob + c * 32, v);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        if (qrow < p.tokens) {
          __nv_bfloat16 *dst =
              static_cast<__nv_bfloat16 *>(hd.out) + static_cast<long long>(qrow) * hd.out_ld + c0 + c * 32;
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
      ptx::tc_fence_before();
      ptx::mbar_arrive(o_free);  // O may be overwritten by the next item's first P V
    }
  }

  // ---- teardown: every TMA load this CTA started has landed before it exits ----
  __syncthreads();
  if (warp == 0 && lane < 2) {
    if (q_loads > 0 && !ptx::mbar_wait(q_full, (q_loads - 1) & 1, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    const uint32_t full0 = lane == 0 ? k_full0 : v_full0;
    for (int s = 0; s < 2; ++s)
      if (issued[s] > 0 && !ptx::mbar_wait(full0 + 8 * s, (issued[s] - 1) & 1, p.wait_ns))
        record(p.status, kDevTimeoutDrain);
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// k_attention2: two query tiles per work item. An item is a pair of adjacent
// 128-query tiles (2i, 2i+1) of one q head, so the causal work of the two is
// nearly equal and every K / V^T tile loaded serves both. Warp roles:
//   warp 0     TMA producers: lane 0 loads the item's two Q tiles and the K
//              ring (2 stages), lane 1 the V^T ring (2 stages);
//   warp 1     MMA issuer, in the order S_A(0), S_B(0), P_A(0)V, S_A(1),
//              P_B(0)V, S_B(1), ...: while one tile's softmax runs, the
//              tensor core works on the other tile;
//   warps 2-5  softmax of tile A, warps 6-9 of tile B: one thread per query
//              row (its TMEM lane) over all 128 keys of a block, so no row
//              value is exchanged between threads.
// TMEM: S of tile A at columns 0-127, of tile B at 128-255, O of A at 256-383,
// of B at 384-511. The softmax writes P as bf16 over the first 64 columns of its
// S (two values per 32-bit column), and P V reads it from there as the A
// operand (the tensor-memory form of tcgen05.mma), so P never goes through
// shared memory. S of the next block is issued after P V of this one, which has
// read P by then (the tensor core runs one issuer's MMAs in order). The
// reference maximum moves only when a block's maximum exceeds it by more than
// 8 (log2 units); then that row of O is rescaled in TMEM: O is current up to the
// previous block whenever S of a block is complete, so no extra wait is needed.
// Every wait is bounded, as in k_attention.
// ---------------------------------------------------------------------------
constexpr uint32_t k2SmemQ = 0, k2SmemK = 2 * kTile, k2SmemV = 4 * kTile;  // Q_A, Q_B; K ring; V^T ring
constexpr uint32_t k2SmemBar = 6 * kTile;
constexpr size_t kAttn2Smem = k2SmemBar + 256 + 1024;  // + barriers + alignment slack (193.3 KB)

__global__ void __launch_bounds__(kAttnThreads, 1) k_attention2(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t sQ = sbase + k2SmemQ, sK0 = sbase + k2SmemK, sV0 = sbase + k2SmemV;
  uint8_t *bar_area = smem + k2SmemBar;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  // barriers (8 bytes each): per tile X in {0 = A, 1 = B}: s_full, p_full, o_full, o_free
  const uint32_t q_full = bar0, q_empty = bar0 + 8, k_full0 = bar0 + 16, k_empty0 = bar0 + 32,
                 v_full0 = bar0 + 48, v_empty0 = bar0 + 64, s_full0 = bar0 + 80, p_full0 = bar0 + 96,
                 o_full0 = bar0 + 112, o_free0 = bar0 + 128, drain = bar0 + 144;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 152);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 156);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kv_blocks = (p.tokens + kTileK - 1) / kTileK;
  const int pairs = (p.q_tiles + 1) / 2;
  const int items = pairs * p.heads_total;
  // This CTA's r-th item: ranks in snake order over the CTAs (r-th round forward
  // when r is even, backward when odd), so with the longest items ranked first
  // every CTA's total stays close to the mean. -1 past the last item.
  auto rank_of = [&](int r) {
    const int pos = (r & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                            : static_cast<int>(blockIdx.x);
    const int k = r * static_cast<int>(gridDim.x) + pos;
    return k < items ? k : -1;
  };
  // work item -> (first query tile, blocks of tile A, blocks of tile B, head);
  // causal ranks the longest pairs first; a tile past the sequence has no blocks
  auto item = [&](int it, int &qt0, int &nba, int &nbb) -> const AttnHead & {
    const int r = it / p.heads_total;
    const int pi = p.causal ? pairs - 1 - r : r;
    qt0 = 2 * pi;
    nba = p.causal ? qt0 + 1 : kv_blocks;
    nbb = qt0 + 1 < p.q_tiles ? (p.causal ? qt0 + 2 : kv_blocks) : 0;
    return p.heads[it % p.heads_total];
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(k_full0 + 8 * s, 1);
      ptx::mbar_init(k_empty0 + 8 * s, 1);
      ptx::mbar_init(v_full0 + 8 * s, 1);
      ptx::mbar_init(v_empty0 + 8 * s, 1);
      ptx::mbar_init(s_full0 + 8 * s, 1);
      ptx::mbar_init(p_full0 + 8 * s, 128);
      ptx::mbar_init(o_full0 + 8 * s, 1);
      ptx::mbar_init(o_free0 + 8 * s, 128);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
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

  int issued[2] = {0, 0};  // loads started per stage of this producer lane's ring
  int q_loads = 0;
  if (warp == 0) {
    if (lane < 2) {
      // lane 0: the Q tiles of each item, then the K ring; lane 1: the V^T ring
      const uint32_t full0 = lane == 0 ? k_full0 : v_full0, empty0 = lane == 0 ? k_empty0 : v_empty0;
      const uint32_t dst0 = lane == 0 ? sK0 : sV0;
      bool run = true;
      int g = 0;
      for (int ic = 0, it = rank_of(0); run && it >= 0; it = rank_of(++ic)) {
        int qt0, nba, nbb;
        const AttnHead &hd = item(it, qt0, nba, nbb);
        const int nbm = nba > nbb ? nba : nbb;
        if (lane == 0) {
          // the previous item's last S has read both Q tiles
          if (*abort_flag || !ptx::mbar_wait(q_empty, (ic & 1) ^ 1, p.wait_ns)) {
            if (!*abort_flag) record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            break;
          }
          ptx::mbar_arrive_expect_tx(q_full, nbb > 0 ? 2 * kTile : kTile);
          for (int t = 0; t < (nbb > 0 ? 2 : 1); ++t)
            for (int c = 0; c < 2; ++c)
              ptx::tma_load_2d(sQ + t * kTile + c * kSub, &p.maps[hd.q_map], hd.q_col + c * 64,
                               (qt0 + t) * kTileQ, q_full);
          ++q_loads;
        }
        const CUtensorMap *map = &p.maps[lane == 0 ? hd.k_map : hd.v_map];
        for (int j = 0; j < nbm; ++j, ++g) {
          const int s = g & 1;
          if (*abort_flag || !ptx::mbar_wait(empty0 + 8 * s, ((g >> 1) & 1) ^ 1, p.wait_ns)) {
            if (!*abort_flag) record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            run = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full0 + 8 * s, kTile);
          for (int c = 0; c < 2; ++c) {
            if (lane == 0)
              ptx::tma_load_2d(dst0 + s * kTile + c * kSub, map, hd.kv_col + c * 64, j * kTileK, full0 + 8 * s);
            else
              ptx::tma_load_2d(dst0 + s * kTile + c * kSub, map, j * kTileK + c * 64, hd.kv_col, full0 + 8 * s);
          }
          ++issued[s];
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileQ, 128);
      bool ok = true;
      auto fail = [&]() {
        if (!*abort_flag) record(p.status, kDevTimeoutMma);
        ok = false;
      };
      auto wait = [&](uint32_t bar, uint32_t parity) {
        if (*abort_flag || !ptx::mbar_wait(bar, parity, p.wait_ns)) {
          fail();
          return false;
        }
        return true;
      };
      // S_X = Q_X K^T for the K stage of block g, into tile X's S columns
      auto issue_s = [&](int x, int g) {
        const uint32_t d = tmem + static_cast<uint32_t>(x * 128);
        const uint32_t kq = sQ + static_cast<uint32_t>(x) * kTile, kk0 = sK0 + static_cast<uint32_t>(g & 1) * kTile;
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(kq + (kk >> 2) * kSub) + 2 * (kk & 3);
          const uint64_t bd = ptx::smem_desc_sw128(kk0 + (kk >> 2) * kSub) + 2 * (kk & 3);
          ptx::mma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full0 + 8 * x);
      };
      // O_X += P_X V^T_g, P_X read from tile X's S columns in tensor memory
      auto issue_pv = [&](int x, int g, bool first) {
        const uint32_t d = tmem + 256u + static_cast<uint32_t>(x * 128);
        const uint32_t a = tmem + static_cast<uint32_t>(x * 128);
        const uint32_t vv = sV0 + static_cast<uint32_t>(g & 1) * kTile;
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk) {
          const uint64_t bd = ptx::smem_desc_sw128(vv + (kk >> 2) * kSub) + 2 * (kk & 3);
          ptx::mma_bf16_ts(d, a + 8u * kk, bd, idesc, (!first || kk > 0) ? 1u : 0u);
        }
      };
      int g = 0;                    // K / V blocks over all items
      uint32_t np[2] = {0, 0};      // softmax hand-offs consumed per tile
      uint32_t nact[2] = {0, 0};    // items in which the tile was active
      for (int ic = 0, it = rank_of(0); ok && it >= 0; it = rank_of(++ic)) {
        int qt0, nba, nbb;
        item(it, qt0, nba, nbb);
        const int nb[2] = {nba, nbb};
        const int nbm = nba > nbb ? nba : nbb;
        if (!wait(q_full, ic & 1)) break;
        // S of block 0 of both tiles
        if (!wait(k_full0 + 8 * (g & 1), (g >> 1) & 1)) break;
        ptx::tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if (nb[x] > 0) issue_s(x, g);
        ptx::mma_commit(k_empty0 + 8 * (g & 1));
        if (nbm == 1) ptx::mma_commit(q_empty);
        for (int j = 0; ok && j < nbm; ++j) {
          const int gj = g + j;
          if (!wait(v_full0 + 8 * (gj & 1), (gj >> 1) & 1)) break;
          bool next_k = false;  // K of block j+1 waited for
          for (int x = 0; ok && x < 2; ++x) {
            if (j >= nb[x]) continue;
            // P_X(j) is in TMEM; the item's first P V overwrites O_X, so its previous
            // item's output must have been read
            if (!wait(p_full0 + 8 * x, np[x] & 1)) break;
            ++np[x];
            if (j == 0 && !wait(o_free0 + 8 * x, (nact[x] & 1) ^ 1)) break;
            ptx::tc_fence_after();
            issue_pv(x, gj, j == 0);
            if (j + 1 == nb[x]) {
              ptx::mma_commit(o_full0 + 8 * x);  // O_X complete for this item
            } else {
              if (!next_k) {
                if (!wait(k_full0 + 8 * ((gj + 1) & 1), ((gj + 1) >> 1) & 1)) break;
                ptx::tc_fence_after();
                next_k = true;
              }
              issue_s(x, gj + 1);
            }
          }
          if (!ok) break;
          ptx::mma_commit(v_empty0 + 8 * (gj & 1));  // V of block j read by every P V of it
          if (next_k) {
            ptx::mma_commit(k_empty0 + 8 * ((gj + 1) & 1));  // K of block j+1 read by every S of it
            if (j + 2 == nbm) ptx::mma_commit(q_empty);        // the item's last S is issued
          }
        }
        for (int x = 0; x < 2; ++x)
          if (nb[x] > 0) ++nact[x];
        g += nbm;
      }
      if (!ok) *abort_flag = 1;
      ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    // ---- softmax: warps 2-5 tile A, 6-9 tile B; warp w reads TMEM lanes [32*(w%4), +32) ----
    const int x = (warp - 2) >> 2;  // 0 = tile A, 1 = tile B
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t sb = tmem + lane_off + static_cast<uint32_t>(x * 128);   // S, then P over its first half
    const uint32_t ob = tmem + lane_off + 256u + static_cast<uint32_t>(x * 128);
    const uint32_t s_full = s_full0 + 8 * x, p_full = p_full0 + 8 * x, o_full = o_full0 + 8 * x,
                   o_free = o_free0 + 8 * x;
    bool ok = true;
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool ready = ptx::mbar_wait(bar, parity, p.wait_ns);
      if (!__all_sync(0xffffffffu, ready && *abort_flag == 0)) {
        if (lane == 0) {
          if (!ready) record(p.status, kDevTimeoutEpilogue);
          *abort_flag = 1;
        }
        return false;
      }
      return true;
    };
    uint32_t gs = 0, nact = 0;  // S blocks of this tile consumed; items it was active in
    for (int ic = 0, it = rank_of(0); ok && it >= 0; it = rank_of(++ic)) {
      int qt0, nba, nbb;
      const AttnHead &hd = item(it, qt0, nba, nbb);
      const int nb = x == 0 ? nba : nbb;
      if (nb == 0) continue;
      const int qrow = (qt0 + x) * kTileQ + row;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nb; ++j, ++gs) {
        if (!wait_all(s_full, gs & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const int k0 = j * kTileK;
        // keys past the query (causal) or past the sequence are masked
        const int lim = min(p.causal ? qrow - k0 + 1 : kTileK, p.tokens - k0);
        uint32_t v[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t (&vc)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]);
          ptx::tmem_ld_32cols(sb + 32 * c, vc);
        }
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        if (!__all_sync(0xffffffffu, lim >= kTileK)) {  // a masked key in this warp's rows
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) v[i] = __float_as_uint(-INFINITY);
        }
        // the row maximum as four independent chains over the key quarters
        float mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mq[q] = __uint_as_float(v[32 * q + 31]);
#pragma unroll
          for (int i = 0; i < 30; i += 2)
            mq[q] = max3f(mq[q], __uint_as_float(v[32 * q + i]), __uint_as_float(v[32 * q + i + 1]));
          mq[q] = fmaxf(mq[q], __uint_as_float(v[32 * q + 30]));
        }
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        const float m_blk = mx * p.scale_log2;
        const bool move = m_blk > m + 8.f;  // always on the item's first block (m = -inf)
        const float m_new = move ? m_blk : m;
        const float alpha = move ? exp2f(m - m_new) : 1.f;  // 0 on the first block
        // p = 2^(s*c - m), two keys at a time (packed f32x2 fma and sum), packed as
        // bf16 pairs into the first 64 columns of S, 16 columns at a time
        const uint64_t c2 = pack2(p.scale_log2, p.scale_log2), nm2 = pack2(-m_new, -m_new);
        uint64_t sumh[4];  // one running pair of sums per 32-key quarter
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint64_t &sum2 = sumh[h];
          sum2 = pack2(0.f, 0.f);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float y0, y1;
            unpack2(fma2(pack2(__uint_as_float(v[32 * h + i]), __uint_as_float(v[32 * h + i + 1])), c2, nm2), y0,
                    y1);
            const float a0 = ex2_approx(y0), a1 = ex2_approx(y1);
            sum2 = add2(sum2, pack2(a0, a1));
            const __nv_bfloat162 hb = __floats2bfloat162_rn(a0, a1);
            memcpy(&pk[i >> 1], &hb, 4);
          }
          ptx::tmem_st_16cols(sb + 16 * h, pk);
        }
        float s0, s1;
        unpack2(add2(add2(sumh[0], sumh[1]), add2(sumh[2], sumh[3])), s0, s1);
        l = l * alpha + (s0 + s1);
        m = m_new;
        if (j > 0 && __any_sync(0xffffffffu, move)) {
          // O holds P V up to block j-1 (S_j completes after that P V) and block j's
          // P V waits for this thread's hand-off; rows keeping their maximum scale by 1
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            ptx::tmem_ld_32cols(ob + c * 32, o);
            ptx::tmem_ld_wait();
            ptx::tmem_regs_ready(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            ptx::tmem_st_32cols(ob + c * 32, o);
          }
        }
        ptx::tmem_st_wait();   // P (and a rescaled O) in tensor memory before the hand-off
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full);
      }
      if (!ok) break;
      // the item's output: O / l once its last P V has landed
      if (!wait_all(o_full, nact & 1)) { ok = false; break; }
      ++nact;
      ptx::tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32cols(ob + c * 32, v);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        if (qrow < p.tokens) {
          __nv_bfloat16 *dst =
              static_cast<__nv_bfloat16 *>(hd.out) + static_cast<long long>(qrow) * hd.out_ld + c * 32;
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
      ptx::tc_fence_before();
      ptx::mbar_arrive(o_free);  // O_X may be overwritten by the next item's first P V
    }
  }

  // ---- teardown: every TMA load this CTA started has landed before it exits ----
  __syncthreads();
  if (warp == 0 && lane < 2) {
    if (q_loads > 0 && !ptx::mbar_wait(q_full, (q_loads - 1) & 1, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    const uint32_t full0 = lane == 0 ? k_full0 : v_full0;
    for (int s = 0; s < 2; ++s)
      if (issued[s] > 0 && !ptx::mbar_wait(full0 + 8 * s, (issued[s] - 1) & 1, p.wait_ns))
        record(p.status, kDevTimeoutDrain);
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// k_attention3: as k_attention2 (two query tiles of one head per work item, one
// softmax thread per row, P in tensor memory), with blocks of 64 keys, so that
// S, P and O of both tiles lie apart in TMEM: tile x has S at 256x, P at
// 256x + 64 (64 bf16 keys, two per 32-bit column) and O at 256x + 128. The
// softmax releases S as soon as it has loaded it, and the MMA warp issues the
// tile's next S right away, so that S is ready when this block's softmax ends
// and the softmax of consecutive blocks runs back to back; the next P is written
// once the previous P V has read P (and updated O). Every barrier phase is
// waited for exactly once, in order, by one side:
//   s_full (MMA -> softmax: S ready), s_free (softmax -> MMA: S read),
//   p_full (softmax -> MMA: P written), pv_done (MMA -> softmax: P V done, so P
//   is free and O current), o_free (softmax -> MMA: O of the item read).
// K tiles are 64 keys x 128 dims (two swizzled 8 KB k-tiles), V^T tiles 128 dims
// x 64 keys (one 16 KB k-tile), in four-stage rings shared by both query tiles.
// On causal attention over 4096 tokens (64 q heads) it takes 0.41 ms against
// k_attention2's 0.25 ms, its tensor pipe active 30 % of the time (52 % for
// k_attention2): k_attention2 stays the default, this kernel runs with
// TPGQA_ATTN=3.
// ---------------------------------------------------------------------------
constexpr int kKb = 64;                        // keys per block
constexpr uint32_t kKSub = 64u * 128u;         // one [64 keys x 64 dims] swizzled k-tile of K
constexpr uint32_t kKTile = 2 * kKSub;         // a K block (all 128 dims)
constexpr uint32_t kVTile = 128u * 128u;       // a V^T block: [128 dims x 64 keys]
constexpr int k3Stages = 4;
constexpr uint32_t k3SmemQ = 0, k3SmemK = 2 * kTile, k3SmemV = k3SmemK + k3Stages * kKTile;
constexpr uint32_t k3SmemBar = k3SmemV + k3Stages * kVTile;  // 192 KB
constexpr size_t kAttn3Smem = k3SmemBar + 256 + 1024;

__global__ void __launch_bounds__(kAttnThreads, 1) k_attention3(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t sQ = sbase + k3SmemQ, sK0 = sbase + k3SmemK, sV0 = sbase + k3SmemV;
  uint8_t *bar_area = smem + k3SmemBar;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  // ring barriers: k_full[4], k_empty[4], v_full[4], v_empty[4]; then per tile x:
  // s_full, s_free, p_full, pv_done, o_free; q_full, q_empty, drain
  auto k_full = [&](int s) { return bar0 + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 8u * (4 + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (8 + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (12 + s); };
  auto tbar = [&](int x, int which) { return bar0 + 8u * (16 + 5 * x + which); };
  constexpr int S_FULL = 0, S_FREE = 1, P_FULL = 2, PV_DONE = 3, O_FREE = 4;
  const uint32_t q_full = bar0 + 8u * 26, q_empty = bar0 + 8u * 27, drain = bar0 + 8u * 28;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 8 * 29);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 8 * 29 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kv_blocks = (p.tokens + kKb - 1) / kKb;
  const int pairs = (p.q_tiles + 1) / 2;
  const int items = pairs * p.heads_total;
  auto rank_of = [&](int r) {
    const int pos = (r & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                            : static_cast<int>(blockIdx.x);
    const int k = r * static_cast<int>(gridDim.x) + pos;
    return k < items ? k : -1;
  };
  // work item -> (first query tile, 64-key blocks of tile A and of tile B, head);
  // causal ranks the longest pairs first; a tile past the sequence has no blocks
  auto item = [&](int it, int &qt0, int &nba, int &nbb) -> const AttnHead & {
    const int r = it / p.heads_total;
    const int pi = p.causal ? pairs - 1 - r : r;
    qt0 = 2 * pi;
    const int nb_causal_a = ((qt0 + 1) * kTileQ < p.tokens ? (qt0 + 1) * kTileQ : p.tokens);
    nba = p.causal ? (nb_causal_a + kKb - 1) / kKb : kv_blocks;
    const int nb_causal_b = ((qt0 + 2) * kTileQ < p.tokens ? (qt0 + 2) * kTileQ : p.tokens);
    nbb = qt0 + 1 < p.q_tiles ? (p.causal ? (nb_causal_b + kKb - 1) / kKb : kv_blocks) : 0;
    return p.heads[it % p.heads_total];
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < k3Stages; ++s) {
      ptx::mbar_init(k_full(s), 1);
      ptx::mbar_init(k_empty(s), 1);
      ptx::mbar_init(v_full(s), 1);
      ptx::mbar_init(v_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(tbar(x, S_FULL), 1);
      ptx::mbar_init(tbar(x, S_FREE), 128);
      ptx::mbar_init(tbar(x, P_FULL), 128);
      ptx::mbar_init(tbar(x, PV_DONE), 1);
      ptx::mbar_init(tbar(x, O_FREE), 128);
    }
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
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

  int issued[k3Stages] = {0, 0, 0, 0};  // loads started per stage of this producer lane's ring
  int q_loads = 0;
  if (warp == 0) {
    if (lane < 2) {
      // lane 0: the Q tiles of each item, then the K ring; lane 1: the V^T ring
      bool run = true;
      int g = 0;
      for (int ic = 0, it = rank_of(0); run && it >= 0; it = rank_of(++ic)) {
        int qt0, nba, nbb;
        const AttnHead &hd = item(it, qt0, nba, nbb);
        const int nbm = nba > nbb ? nba : nbb;
        if (lane == 0) {
          if (*abort_flag || !ptx::mbar_wait(q_empty, (ic & 1) ^ 1, p.wait_ns)) {
            if (!*abort_flag) record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            break;
          }
          ptx::mbar_arrive_expect_tx(q_full, nbb > 0 ? 2 * kTile : kTile);
          for (int t = 0; t < (nbb > 0 ? 2 : 1); ++t)
            for (int c = 0; c < 2; ++c)
              ptx::tma_load_2d(sQ + t * kTile + c * kSub, &p.maps[hd.q_map], hd.q_col + c * 64,
                               (qt0 + t) * kTileQ, q_full);
          ++q_loads;
        }
        for (int j = 0; j < nbm; ++j, ++g) {
          const int s = g % k3Stages;
          const uint32_t ph = (g / k3Stages) & 1;
          const uint32_t full = lane == 0 ? k_full(s) : v_full(s), empty = lane == 0 ? k_empty(s) : v_empty(s);
          if (*abort_flag || !ptx::mbar_wait(empty, ph ^ 1, p.wait_ns)) {
            if (!*abort_flag) record(p.status, kDevTimeoutProducer);
            *abort_flag = 1;
            run = false;
            break;
          }
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(full, kKTile);
            for (int c = 0; c < 2; ++c)
              ptx::tma_load_2d(sK0 + s * kKTile + c * kKSub, &p.maps[hd.k_map], hd.kv_col + c * 64, j * kKb, full);
          } else {
            ptx::mbar_arrive_expect_tx(full, kVTile);
            ptx::tma_load_2d(sV0 + s * kVTile, &p.maps[hd.v_map], j * kKb, hd.kv_col, full);
          }
          ++issued[s];
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kTileQ, kKb);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(kTileQ, kHd);
      bool ok = true;
      auto wait = [&](uint32_t bar, uint32_t parity) {
        if (*abort_flag || !ptx::mbar_wait(bar, parity, p.wait_ns)) {
          if (!*abort_flag) record(p.status, kDevTimeoutMma);
          ok = false;
          return false;
        }
        return true;
      };
      // S_x = Q_x K^T of the K stage holding block g (64 keys), into tile x's S
      auto issue_s = [&](int x, int g) {
        const uint32_t d = tmem + static_cast<uint32_t>(256 * x);
        const uint32_t kq = sQ + static_cast<uint32_t>(x) * kTile, kk0 = sK0 + static_cast<uint32_t>(g % k3Stages) * kKTile;
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(kq + (kk >> 2) * kSub) + 2 * (kk & 3);
          const uint64_t bd = ptx::smem_desc_sw128(kk0 + (kk >> 2) * kKSub) + 2 * (kk & 3);
          ptx::mma_bf16(d, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(tbar(x, S_FULL));
      };
      // O_x += P_x V^T_g, P_x from tensor memory
      auto issue_pv = [&](int x, int g, bool first) {
        const uint32_t d = tmem + static_cast<uint32_t>(256 * x + 128);
        const uint32_t a = tmem + static_cast<uint32_t>(256 * x + 64);
        const uint32_t vv = sV0 + static_cast<uint32_t>(g % k3Stages) * kVTile;
#pragma unroll
        for (int kk = 0; kk < kKb / 16; ++kk) {
          const uint64_t bd = ptx::smem_desc_sw128(vv) + 2 * kk;
          ptx::mma_bf16_ts(d, a + 8u * kk, bd, idesc_pv, (!first || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(tbar(x, PV_DONE));
      };
      int g = 0;                          // K / V blocks over all items
      uint32_t ns[2] = {0, 0};            // S issued per tile (all items)
      uint32_t np[2] = {0, 0};            // P hand-offs consumed per tile
      uint32_t nact[2] = {0, 0};          // items in which the tile was active
      for (int ic = 0, it = rank_of(0); ok && it >= 0; it = rank_of(++ic)) {
        int qt0, nba, nbb;
        item(it, qt0, nba, nbb);
        const int nb[2] = {nba, nbb};
        const int nbm = nba > nbb ? nba : nbb;
        if (!wait(q_full, ic & 1)) break;
        // S of block j of every active tile: after the softmax has read the tile's
        // previous S (the first S of this CTA has none)
        auto issue_block_s = [&](int j) {
          const int gj = g + j;
          if (!wait(k_full(gj % k3Stages), (gj / k3Stages) & 1)) return;
          for (int x = 0; x < 2 && ok; ++x) {
            if (j >= nb[x]) continue;
            if (ns[x] > 0 && !wait(tbar(x, S_FREE), (ns[x] - 1) & 1)) return;
            ptx::tc_fence_after();
            issue_s(x, gj);
            ++ns[x];
          }
          ptx::mma_commit(k_empty(gj % k3Stages));  // K of block j read by every S of it
          if (j + 1 == nbm) ptx::mma_commit(q_empty);  // the item's last S is issued
        };
        issue_block_s(0);
        for (int j = 0; ok && j < nbm; ++j) {
          if (j + 1 < nbm) {
            issue_block_s(j + 1);
            if (!ok) break;
          }
          const int gj = g + j;
          if (!wait(v_full(gj % k3Stages), (gj / k3Stages) & 1)) break;
          for (int x = 0; x < 2 && ok; ++x) {
            if (j >= nb[x]) continue;
            if (!wait(tbar(x, P_FULL), np[x] & 1)) break;
            ++np[x];
            if (j == 0 && !wait(tbar(x, O_FREE), (nact[x] & 1) ^ 1)) break;
            ptx::tc_fence_after();
            issue_pv(x, gj, j == 0);
          }
          if (!ok) break;
          ptx::mma_commit(v_empty(gj % k3Stages));  // V of block j read by every P V of it
        }
        for (int x = 0; x < 2; ++x)
          if (nb[x] > 0) ++nact[x];
        g += nbm;
      }
      if (!ok) *abort_flag = 1;
      ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else {
    // ---- softmax: warps 2-5 tile A, 6-9 tile B; warp w reads TMEM lanes [32*(w%4), +32) ----
    const int x = (warp - 2) >> 2;
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t sb = tmem + lane_off + static_cast<uint32_t>(256 * x);
    const uint32_t pb = sb + 64u, ob = sb + 128u;
    bool ok = true;
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool ready = ptx::mbar_wait(bar, parity, p.wait_ns);
      if (!__all_sync(0xffffffffu, ready && *abort_flag == 0)) {
        if (lane == 0) {
          if (!ready) record(p.status, kDevTimeoutEpilogue);
          *abort_flag = 1;
        }
        return false;
      }
      return true;
    };
    uint32_t gs = 0;  // S blocks of this tile consumed (all items); P V done waits follow the same count
    for (int ic = 0, it = rank_of(0); ok && it >= 0; it = rank_of(++ic)) {
      int qt0, nba, nbb;
      const AttnHead &hd = item(it, qt0, nba, nbb);
      const int nb = x == 0 ? nba : nbb;
      if (nb == 0) continue;
      const int qrow = (qt0 + x) * kTileQ + row;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nb; ++j, ++gs) {
        if (!wait_all(tbar(x, S_FULL), gs & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const int k0 = j * kKb;
        const int lim = min(p.causal ? qrow - k0 + 1 : kKb, p.tokens - k0);
        uint32_t v[64];
        {
          uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
          uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
          ptx::tmem_ld_32cols(sb, v0);
          ptx::tmem_ld_32cols(sb + 32, v1);
          ptx::tmem_ld_wait();
          ptx::tmem_regs_ready(v);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(tbar(x, S_FREE));  // S read: the tile's next S may be computed
        if (!__all_sync(0xffffffffu, lim >= kKb)) {  // a masked key in this warp's rows
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i >= lim) v[i] = __float_as_uint(-INFINITY);
        }
        float mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mq[q] = __uint_as_float(v[16 * q + 15]);
#pragma unroll
          for (int i = 0; i < 14; i += 2)
            mq[q] = max3f(mq[q], __uint_as_float(v[16 * q + i]), __uint_as_float(v[16 * q + i + 1]));
          mq[q] = fmaxf(mq[q], __uint_as_float(v[16 * q + 14]));
        }
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        const float m_blk = mx * p.scale_log2;
        const bool move = m_blk > m + 8.f;  // always on the item's first block (m = -inf)
        const float m_new = move ? m_blk : m;
        const float alpha = move ? exp2f(m - m_new) : 1.f;  // 0 on the first block
        const uint64_t c2 = pack2(p.scale_log2, p.scale_log2), nm2 = pack2(-m_new, -m_new);
        uint64_t sumh[2];
        uint32_t pk[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          sumh[h] = pack2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float y0, y1;
            unpack2(fma2(pack2(__uint_as_float(v[32 * h + i]), __uint_as_float(v[32 * h + i + 1])), c2, nm2), y0,
                    y1);
            const float a0 = ex2_approx(y0), a1 = ex2_approx(y1);
            sumh[h] = add2(sumh[h], pack2(a0, a1));
            const __nv_bfloat162 hb = __floats2bfloat162_rn(a0, a1);
            memcpy(&pk[h][i >> 1], &hb, 4);
          }
        }
        float s0, s1;
        unpack2(add2(sumh[0], sumh[1]), s0, s1);
        l = l * alpha + (s0 + s1);
        m = m_new;
        // the previous P V has read P and brought O up to date
        if (j > 0) {
          if (!wait_all(tbar(x, PV_DONE), (gs - 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
          if (__any_sync(0xffffffffu, move)) {  // rows keeping their maximum scale by 1
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              ptx::tmem_ld_32cols(ob + c * 32, o);
              ptx::tmem_ld_wait();
              ptx::tmem_regs_ready(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              ptx::tmem_st_32cols(ob + c * 32, o);
            }
          }
        }
        ptx::tmem_st_16cols(pb, pk[0]);
        ptx::tmem_st_16cols(pb + 16, pk[1]);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(tbar(x, P_FULL));
      }
      if (!ok) break;
      // the item's output: O / l once its last P V has landed
      if (!wait_all(tbar(x, PV_DONE), (gs - 1) & 1)) { ok = false; break; }
      ptx::tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32cols(ob + c * 32, v);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        if (qrow < p.tokens) {
          __nv_bfloat16 *dst =
              static_cast<__nv_bfloat16 *>(hd.out) + static_cast<long long>(qrow) * hd.out_ld + c * 32;
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
      ptx::tc_fence_before();
      ptx::mbar_arrive(tbar(x, O_FREE));  // O_x may be overwritten by the next item's first P V
    }
  }

  // ---- teardown: every TMA load this CTA started has landed before it exits ----
  __syncthreads();
  if (warp == 0 && lane < 2) {
    if (lane == 0 && q_loads > 0 && !ptx::mbar_wait(q_full, (q_loads - 1) & 1, p.wait_ns))
      record(p.status, kDevTimeoutDrain);
    for (int s = 0; s < k3Stages; ++s)
      if (issued[s] > 0 && !ptx::mbar_wait(lane == 0 ? k_full(s) : v_full(s), (issued[s] - 1) & 1, p.wait_ns))
        record(p.status, kDevTimeoutDrain);
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// V [T x C] (row pitch ld_in) -> V^T [C x T] (row pitch ld_out) for every kv
// source in one launch (grid z = source), 64 x 64 tiles through shared memory.
__global__ void __launch_bounds__(256) k_transpose_bf16(TransposeArgs a) {
  __shared__ __nv_bfloat16 tile[64][66];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const __nv_bfloat16 *in = static_cast<const __nv_bfloat16 *>(a.in[blockIdx.z]);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out[blockIdx.z]);
  const long long ld_in = a.ld_in[blockIdx.z];
  const int r0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int r = i / 64, c = i % 64;
    if (r0 + r < a.rows && c0 + c < a.cols) tile[r][c] = in[static_cast<long long>(r0 + r) * ld_in + c0 + c];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int c = i / 64, r = i % 64;
    if (r0 + r < a.rows && c0 + c < a.cols) out[static_cast<long long>(c0 + c) * a.ld_out + r0 + r] = tile[r][c];
  }
}

}  // namespace

tp_status launch_transpose_bf16(const TransposeArgs &a, int sources, cudaStream_t s) {
  if (a.rows == 0 || a.cols == 0 || sources == 0) return TP_OK;
  const dim3 grid((a.rows + 63) / 64, (a.cols + 63) / 64, sources);
  return launch_checked(launch_kernel(k_transpose_bf16, grid, dim3(256), 0, s, 1, a));
}

int attention_variant() {
  const char *env = getenv("TPGQA_ATTN");
  if (env && (env[0] == '1' || env[0] == '3') && env[1] == 0) return env[0] - '0';
  return 2;
}

int attention_k_box_rows(int variant) { return variant == 3 ? kKb : kTileK; }

tp_status launch_attention(AttnParams &p, int total_heads, cudaStream_t s) {
  DevCtx ctx;
  cudaError_t e = get_dev_ctx(&ctx);
  if (e != cudaSuccess) return cuda_fail(e);
  p.status = ctx.status;
  p.wait_ns = ctx.wait_ns;
  // the shared-memory opt-in is per device: set it once on each
  static std::mutex mu;
  static unsigned long long configured = 0;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 64 || !(configured & (1ULL << dev))) {
      e = cudaFuncSetAttribute(k_attention, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kAttnSmem));
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attention2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kAttn2Smem));
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attention3, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kAttn3Smem));
      if (e != cudaSuccess) return cuda_fail(e);
      if (dev < 64) configured |= 1ULL << dev;
    }
  }
  p.heads_total = total_heads;
  if (p.variant == 1) {
    const long long items = static_cast<long long>(p.q_tiles) * total_heads;
    const dim3 grid(static_cast<unsigned>(items < num_sms() ? items : num_sms()));
    return launch_checked(launch_kernel(k_attention, grid, dim3(kAttnThreads), kAttnSmem, s, 1, p));
  }
  const long long items = static_cast<long long>((p.q_tiles + 1) / 2) * total_heads;
  const dim3 grid(static_cast<unsigned>(items < num_sms() ? items : num_sms()));
  if (p.variant == 2)
    return launch_checked(launch_kernel(k_attention2, grid, dim3(kAttnThreads), kAttn2Smem, s, 1, p));
  return launch_checked(launch_kernel(k_attention3, grid, dim3(kAttnThreads), kAttn3Smem, s, 1, p));
}

}  // namespace tpgqa
