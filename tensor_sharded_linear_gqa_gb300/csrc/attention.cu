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

// The two-tile and SM-pair kernels take p = 2^(s*c - m) against the row's running
// maximum m without first finding the maximum of each key block: softmax does not
// change with the constant taken off a row's scores, so m only has to keep p and
// the sums far inside the f32 range. p above 1 keeps the same relative precision
// in bf16 P and in the f32 sums. The block's maximum is found (find_max) on an
// item's first block, and on a later block only when the block's sum of p
// passes kSumLimit or is not finite; then m moves to that maximum when it
// exceeds m by more than 8 (log2 units), p is taken again, and the row of O is
// rescaled by 2^(m_old - m_new). So p <= 2^64 always, and a row of O sums at
// most 2^64 * T * max|v|, far inside the f32 range (2^128) for values of
// ordinary size.
constexpr float kSumLimit = 0x1p64f;

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
// read P by then (the tensor core runs one issuer's MMAs in order). p is taken
// against the row's running maximum, which moves only as kSumLimit describes;
// then that row of O is rescaled in TMEM: O is current up to the previous block
// whenever S of a block is complete, so no extra wait is needed.
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
        // p = 2^(s*c - m) against the row's running maximum m (see find_max)
        const uint64_t c2 = pack2(p.scale_log2, p.scale_log2);
        bool find_max = j == 0, move = false;
        float m_new = m, s0, s1;
#pragma unroll 1
        for (;;) {
          if (find_max) {
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
            const float m_blk = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
            move = m_blk > m + 8.f;  // always on the item's first block (m = -inf)
            m_new = move ? m_blk : m;
          }
          // two keys at a time (packed f32x2 fma and sum), packed as bf16 pairs
          // into the first 64 columns of S, 16 columns at a time
          const uint64_t nm2 = pack2(-m_new, -m_new);
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
          unpack2(add2(add2(sumh[0], sumh[1]), add2(sumh[2], sumh[3])), s0, s1);
          if (find_max || !__any_sync(0xffffffffu, !(s0 + s1 <= kSumLimit))) break;
          find_max = true;
          ptx::tmem_st_wait();  // this pass's P is written over before the next pass's
        }
        const float alpha = move ? exp2f(m - m_new) : 1.f;  // 0 on the first block
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

// ---------------------------------------------------------------------------
// k_attention4: one 256-query tile of one q head per work item, on an SM pair
// (a cluster of two CTAs whose MMAs are cta_group::2). CTA c of the pair holds
// query rows [128c, 128c + 128) of the tile, keys [64c, 64c + 64) of every
// 128-key K block and head dims [64c, 64c + 64) of every V^T block, so each K
// and V^T block is loaded once for 256 queries. In the leader CTA one thread
// issues S = Q K^T (M = 256, N = 128 keys, K = 128 dims) and another O += P V
// (M = 256, N = 128 dims, K = 128 keys, P read from tensor memory): the tensor
// core queues little more than the MMA it runs, so a lone issuer leaves it idle
// while it waits and commits; with two, one thread's bookkeeping overlaps the
// other's MMAs.
// TMEM of each CTA: O at columns 0-127, S buffers at 128 and 256, P buffers
// (bf16, two keys per column) at 384 and 448; block g uses S and P buffers
// g % 2. S of block g + 2 is issued as soon as the softmax of both CTAs has
// loaded S of block g; the S barrier of block g takes two arrivals, S of block g
// done and P V of block g - 2 done (so P buffer g % 2 is free again).
// Warp roles in each CTA:
//   warp 0     TMA: lane 0 the item's Q rows (two buffers, so the next item's
//              Q lands while this one's last S are issued) and the K ring, lane 1
//              the V^T ring (four stages each). Every copy completes on the
//              leader CTA's barrier, which the leader arms with both CTAs' bytes;
//   warp 1     TMEM allocation; in the leader, the S thread;
//   warps 2-5  softmax: one thread per query row (its TMEM lane) over all 128
//              keys of a block. The hand-offs ("S loaded", "P written") of both
//              CTAs arrive on the leader's barriers with relaxed cluster-scope
//              arrives: each follows the thread's own wait for its tcgen05 loads
//              or stores, and the release form costs a thousand cycles on a busy
//              SM. p is taken against the row's running maximum, which moves
//              only as kSumLimit describes; then the row of O is rescaled in
//              TMEM once the previous P V has landed. At the end of
//              an item O / l is stored; the next item's first P V, which
//              overwrites O, waits for the same threads' next P hand-off;
//   warp 6     in the leader, the P V thread.
// Every wait is bounded; on a timeout the CTA records it, stops issuing, gives
// copies in flight time to land, frees TMEM and returns.
// ---------------------------------------------------------------------------
constexpr int kAttn4Threads = 224;  // producer, S issuer, 4 softmax warps, P V issuer
constexpr int k4Stages = 4;
constexpr uint32_t k4KVSub = 64u * 128u;     // one [64 rows x 64 bf16] swizzled k-tile (8 KB)
constexpr uint32_t k4KVStage = 2 * k4KVSub;  // this CTA's half of a K block or of a V^T block
constexpr uint32_t k4SmemQ = 0, k4SmemK = 2 * kTile, k4SmemV = k4SmemK + k4Stages * k4KVStage;
constexpr uint32_t k4SmemBar = k4SmemV + k4Stages * k4KVStage;  // 192 KB
constexpr size_t kAttn4Smem = k4SmemBar + 384 + 1024;            // + barriers + alignment slack
constexpr uint32_t k4ColS = 128, k4ColP = 384;  // TMEM columns of S buffer 0 and P buffer 0 (O at 0)
// barrier slots (8 bytes each) from k4SmemBar
enum : int {
  k4QFull = 0, k4QEmpty = 2, k4KFull = 4, k4KEmpty = 8, k4VFull = 12, k4VEmpty = 16,
  k4SFull = 20, k4SFree = 22, k4PFull = 24, k4PvDone = 26, k4DrainS = 30, k4DrainPv = 31, k4NumBars = 32
};
static_assert(8 * k4NumBars + 8 <= 384, "barriers, TMEM slot and abort flag fit before the exchange");

// D (TMEM) (+)= A * B^T on the SM pair, A read from tensor memory: each CTA's
// 128 rows of A on its own TMEM lanes, K bf16 values two per 32-bit column; B
// halves from both CTAs' shared memory at the same offset.
__device__ __forceinline__ void mma_bf16_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrival on an mbarrier of another CTA of the cluster (shared::cluster
// address), without release semantics: the caller has already waited for what
// the arrival announces (tcgen05 loads or stores completed, then a CTA-scope
// barrier acquired), so it carries no data of its own and skips the
// cluster-wide release, which costs a thousand cycles on a busy SM.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Bounded wait for an mbarrier phase whose common case, a phase already
// complete, costs one try_wait: the timed retry loop is out of line.
__device__ __noinline__ bool mbar_wait_retry(uint32_t bar, uint32_t parity, long long budget_ns) {
  return ptx::mbar_wait(bar, parity, budget_ns);
}
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity, long long budget_ns) {
  if (__builtin_expect(ptx::mbar_try_wait(bar, parity), 1)) return true;
  return mbar_wait_retry(bar, parity, budget_ns);
}

// Non-blocking test of an mbarrier phase (mbarrier.test_wait: never suspends
// the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait that polls with test_wait, for the threads whose reaction time
// is on the critical path (a suspended try_wait took about 500 cycles to see a
// phase complete); the clock is read every 64 polls.
__device__ __noinline__ bool mbar_spin_retry(uint32_t bar, uint32_t parity, long long budget_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (static_cast<long long>(ptx::globaltimer_ns() - t0) > budget_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, long long budget_ns) {
  if (__builtin_expect(mbar_test_wait(bar, parity), 1)) return true;
  return mbar_spin_retry(bar, parity, budget_ns);
}

// A position in a CTA pair's sequence of work items and their key blocks.
struct Attn4Cursor {
  int ic;                // items started
  int j, nb, qt;         // key block in the item, blocks of the item, 256-query tile
  const AttnHead *hd;    // null past the last item
};

__global__ void __launch_bounds__(kAttn4Threads, 1) k_attention4(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t sQ = sbase + k4SmemQ, sK = sbase + k4SmemK, sV = sbase + k4SmemV;
  uint8_t *bar_area = smem + k4SmemBar;
  const uint32_t bar0 = ptx::smem_addr(bar_area);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bar_area + 8 * k4NumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 8 * k4NumBars + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 1), nclusters = static_cast<int>(gridDim.x >> 1);
  const int kv_blocks = (p.tokens + kTileK - 1) / kTileK;
  const int tiles = (p.tokens + 255) / 256;
  const int items = tiles * p.heads_total;
  // The pair's r-th item, in snake order over the pairs (longest items first
  // when causal); -1 past the last.
  auto rank_of = [&](int r) {
    const int pos = (r & 1) ? nclusters - 1 - cluster : cluster;
    const int k = r * nclusters + pos;
    return k < items ? k : -1;
  };
  auto load = [&](Attn4Cursor &c) {
    const int it = rank_of(c.ic);
    c.j = 0;
    if (it < 0) {
      c.hd = nullptr;
      c.nb = c.qt = 0;
      return;
    }
    const int r = it / p.heads_total;
    c.qt = p.causal ? tiles - 1 - r : r;
    c.nb = p.causal ? min(2 * c.qt + 2, kv_blocks) : kv_blocks;
    c.hd = &p.heads[it % p.heads_total];
  };
  auto advance = [&](Attn4Cursor &c) {
    if (++c.j == c.nb) {
      ++c.ic;
      load(c);
    }
  };
  // A bounded single-thread wait; on a timeout the thread records it and gives up.
  auto wait1 = [&](int b, uint32_t parity, int code) {
    if (mbar_wait_fast(bar(b), parity, p.wait_ns)) return true;
    if (!*abort_flag) record(p.status, code);
    *abort_flag = 1;
    return false;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(k4QFull + i), 1);
      ptx::mbar_init(bar(k4QEmpty + i), 1);
      // S of block g done, and P V of block g - 2 done (so P buffer g % 2 is free)
      ptx::mbar_init(bar(k4SFull + i), 2);
      // the 4 softmax warps of both CTAs (used in the leader only)
      ptx::mbar_init(bar(k4SFree + i), 8);
      ptx::mbar_init(bar(k4PFull + i), 8);
    }
    for (int s = 0; s < k4Stages; ++s) {
      ptx::mbar_init(bar(k4KFull + s), 1);
      ptx::mbar_init(bar(k4KEmpty + s), 1);
      ptx::mbar_init(bar(k4VFull + s), 1);
      ptx::mbar_init(bar(k4VEmpty + s), 1);
    }
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(bar(k4PvDone + i), 1);
    }
    ptx::mbar_init(bar(k4DrainS), 1);
    ptx::mbar_init(bar(k4DrainPv), 1);
    // blocks 0 and 1 have no P V two blocks back
    ptx::mbar_arrive(bar(k4SFull));
    ptx::mbar_arrive(bar(k4SFull + 1));
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(256, 128);

  if (warp == 0) {
    if (lane < 2) {
      // lane 0: each item's Q rows, then the K ring; lane 1: the V^T ring
      Attn4Cursor c{0, 0, 0, 0, nullptr};
      load(c);
      uint32_t st = 0, ph = 0;  // ring stage and phase of block g
      for (int g = 0; c.hd; ++g, advance(c)) {
        const AttnHead &hd = *c.hd;
        if (lane == 0 && c.j == 0) {
          // Q buffer ic % 2: the last S of the item that used it before has read it
          const int qb = c.ic & 1;
          if (*abort_flag || !wait1(k4QEmpty + qb, ((c.ic >> 1) & 1) ^ 1, kDevTimeoutProducer)) break;
          if (leader) ptx::mbar_arrive_expect_tx(bar(k4QFull + qb), 2 * kTile);
          const uint32_t lead_full = ptx::mapa_shared(bar(k4QFull + qb), 0);
          for (int sub = 0; sub < 2; ++sub)
            ptx::tma_load_2d_pair(sQ + static_cast<uint32_t>(qb) * kTile + sub * kSub, &p.maps[hd.q_map],
                                  hd.q_col + 64 * sub, c.qt * 256 + 128 * static_cast<int>(rank), lead_full);
        }
        const int full = (lane == 0 ? k4KFull : k4VFull) + static_cast<int>(st);
        const int empty = (lane == 0 ? k4KEmpty : k4VEmpty) + static_cast<int>(st);
        if (*abort_flag || !wait1(empty, ph ^ 1, kDevTimeoutProducer)) break;
        if (leader) ptx::mbar_arrive_expect_tx(bar(full), 2 * k4KVStage);
        const uint32_t lead_full = ptx::mapa_shared(bar(full), 0);
        const uint32_t dst = (lane == 0 ? sK : sV) + st * k4KVStage;
        for (int sub = 0; sub < 2; ++sub) {
          if (lane == 0)  // keys [64 rank, +64) of the block, head dims [64 sub, +64)
            ptx::tma_load_2d_pair(dst + sub * k4KVSub, &p.maps[hd.k_map], hd.kv_col + 64 * sub,
                                  c.j * kTileK + 64 * static_cast<int>(rank), lead_full);
          else  // head dims [64 rank, +64) of V^T, keys [64 sub, +64) of the block
            ptx::tma_load_2d_pair(dst + sub * k4KVSub, &p.maps[hd.v_map], c.j * kTileK + 64 * sub,
                                  hd.kv_col + 64 * static_cast<int>(rank), lead_full);
        }
        if (++st == k4Stages) {
          st = 0;
          ph ^= 1;
        }
      }
    }
  } else if ((warp == 1 || warp == 6) && lane == 0) {
    if (leader && warp == 1) {
      // ---- S thread: S(g) = Q K^T into S buffer g % 2 ----
      const uint64_t q_desc = ptx::smem_desc_sw128(sQ), k_desc = ptx::smem_desc_sw128(sK);
      Attn4Cursor c{0, 0, 0, 0, nullptr};
      load(c);
      uint32_t b = 0, bph = 0, st = 0, kph = 0;  // S buffer and phase, K stage and phase
      bool ok = true;
      for (; c.hd; advance(c)) {
        const int qb = c.ic & 1;
        // the softmax has loaded S of block g - 2 out of this buffer (both CTAs)
        if (!wait1(k4SFree + static_cast<int>(b), bph ^ 1, kDevTimeoutMma) ||
            (c.j == 0 && !wait1(k4QFull + qb, (c.ic >> 1) & 1, kDevTimeoutMma)) ||
            !wait1(k4KFull + static_cast<int>(st), kph, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + k4ColS + 128u * b;
        const uint64_t ad = q_desc + ((static_cast<uint32_t>(qb) * kTile) >> 4);
        const uint64_t bd = k_desc + ((st * k4KVStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk)
          ptx::mma_bf16_pair(d, ad + (((kk >> 2) * kSub) >> 4) + 2 * (kk & 3),
                             bd + (((kk >> 2) * k4KVSub) >> 4) + 2 * (kk & 3), idesc, kk > 0 ? 1u : 0u);
        ptx::mma_commit_pair_multicast(bar(k4SFull + static_cast<int>(b)), 0x3);
        ptx::mma_commit_pair_multicast(bar(k4KEmpty + static_cast<int>(st)), 0x3);
        if (c.j + 1 == c.nb) ptx::mma_commit_pair_multicast(bar(k4QEmpty + qb), 0x3);  // the item's last S
        if (++b == 2) {
          b = 0;
          bph ^= 1;
        }
        if (++st == k4Stages) {
          st = 0;
          kph ^= 1;
        }
      }
      if (!ok) *abort_flag = 1;
      ptx::mma_commit_pair_multicast(bar(k4DrainS), 0x1);
      if (!ptx::mbar_wait(bar(k4DrainS), 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    } else if (leader) {
      // ---- P V thread: O += P(g) V(g), P from P buffer g % 2 ----
      const uint64_t v_desc = ptx::smem_desc_sw128(sV);
      Attn4Cursor c{0, 0, 0, 0, nullptr};
      load(c);
      uint32_t b = 0, bph = 0, st = 0, vph = 0, n = 0;  // P buffer and phase, V stage and phase, P V issued
      bool ok = true;
      for (; c.hd; advance(c), ++n) {
        // P(g) in both CTAs (their O rescaled where it had to be) and V^T of block g
        if (!wait1(k4PFull + static_cast<int>(b), bph, kDevTimeoutMma) ||
            !wait1(k4VFull + static_cast<int>(st), vph, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a = tmem + k4ColP + 64u * b;
        const uint64_t bd = v_desc + ((st * k4KVStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk)
          mma_bf16_pair_ts(tmem, a + 8u * static_cast<uint32_t>(kk), bd + (((kk >> 2) * k4KVSub) >> 4) + 2 * (kk & 3),
                           idesc, (c.j > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit_pair_multicast(bar(k4PvDone + static_cast<int>(n & 3)), 0x3);
        // the second arrival on the S barrier of block g + 2: P buffer g % 2 is free
        ptx::mma_commit_pair_multicast(bar(k4SFull + static_cast<int>(b)), 0x3);
        ptx::mma_commit_pair_multicast(bar(k4VEmpty + static_cast<int>(st)), 0x3);
        if (++b == 2) {
          b = 0;
          bph ^= 1;
        }
        if (++st == k4Stages) {
          st = 0;
          vph ^= 1;
        }
      }
      if (!ok) *abort_flag = 1;
      ptx::mma_commit_pair_multicast(bar(k4DrainPv), 0x1);
      if (!ptx::mbar_wait(bar(k4DrainPv), 0, p.wait_ns)) record(p.status, kDevTimeoutDrain);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---- softmax: warp w reads TMEM lanes [32*(w%4), +32), one thread per query row ----
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t ob = tmem + lane_off;
    // hand-offs go to the leader CTA's barriers (the MMA threads live there)
    const uint32_t lead_sfree = ptx::mapa_shared(bar(k4SFree), 0), lead_pfull = ptx::mapa_shared(bar(k4PFull), 0);
    bool ok = true;
    // A bounded warp-wide wait: lane 0 polls and the warp converges on its answer;
    // on a timeout (or another role's abort) the warp gives up.
    auto wait_all = [&](uint32_t bb, uint32_t parity) -> bool {
      int go = 0;
      if (lane == 0) {
        const bool ready = mbar_spin(bb, parity, p.wait_ns);
        if (!ready) record(p.status, kDevTimeoutEpilogue);
        if (!ready || *abort_flag) *abort_flag = 1;
        else go = 1;
      }
      return __shfl_sync(0xffffffffu, go, 0) != 0;
    };
    // P V of block gq has landed: O is current up to it (four barriers in turn,
    // so a phase waited for is never two behind the barrier's current one)
    auto wait_pv = [&](int gq) -> bool {
      if (!wait_all(bar(k4PvDone + (gq & 3)), (gq >> 2) & 1)) return false;
      ptx::tc_fence_after();
      return true;
    };
    Attn4Cursor c{0, 0, 0, 0, nullptr};
    load(c);
    int g = 0;                // key blocks over all items
    uint32_t b = 0, bph = 0;  // S / P buffer of block g and the S phase
    while (ok && c.hd) {
      const AttnHead &hd = *c.hd;
      const int qrow = c.qt * 256 + 128 * static_cast<int>(rank) + row;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < c.nb; ++j, ++g) {
        // S of block g, and P V of block g - 2 done (P buffer b free)
        if (!wait_all(bar(k4SFull + static_cast<int>(b)), bph)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t sb = tmem + lane_off + k4ColS + 128u * b;
        uint32_t v[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t (&vq)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32 * q]);
          ptx::tmem_ld_32cols(sb + 32u * static_cast<uint32_t>(q), vq);
        }
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(v);
        // S of this block is in registers: the S buffer may take block g + 2
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(lead_sfree + 8u * b);
        const int k0 = j * kTileK;
        // keys past the query (causal) or past the sequence are masked
        const int lim = min(p.causal ? qrow - k0 + 1 : kTileK, p.tokens - k0);
        if (!__all_sync(0xffffffffu, lim >= kTileK)) {  // a masked key in this warp's rows
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) v[i] = __float_as_uint(-INFINITY);
        }
        // p = 2^(s*c - m) against the row's running maximum m (see find_max)
        const uint64_t c2 = pack2(p.scale_log2, p.scale_log2);
        const uint32_t pb = tmem + lane_off + k4ColP + 64u * b;
        bool find_max = j == 0, move = false;
        float m_new = m, s0, s1;
#pragma unroll 1
        for (;;) {
          if (find_max) {
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
            const float m_blk = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
            move = m_blk > m + 8.f;  // always on the item's first block (m = -inf)
            m_new = move ? m_blk : m;
          }
          // two keys at a time, packed as bf16 pairs into P buffer b, 16 columns
          // (32 keys) at a time
          const uint64_t nm2 = pack2(-m_new, -m_new);
          uint64_t sumh[4];
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
            ptx::tmem_st_16cols(pb + 16u * static_cast<uint32_t>(h), pk);
          }
          unpack2(add2(add2(sumh[0], sumh[1]), add2(sumh[2], sumh[3])), s0, s1);
          if (find_max || !__any_sync(0xffffffffu, !(s0 + s1 <= kSumLimit))) break;
          find_max = true;
          ptx::tmem_st_wait();  // this pass's P is written over before the next pass's
        }
        const float alpha = move ? exp2f(m - m_new) : 1.f;  // 0 on the first block
        l = l * alpha + (s0 + s1);
        m = m_new;
        if (j > 0 && __any_sync(0xffffffffu, move)) {
          // O must hold P V up to block j - 1 before it is rescaled (rows keeping
          // their maximum scale by 1)
          if (!wait_pv(g - 1)) { ok = false; break; }
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            ptx::tmem_ld_32cols(ob + 32u * static_cast<uint32_t>(cc), o);
            ptx::tmem_ld_wait();
            ptx::tmem_regs_ready(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            ptx::tmem_st_32cols(ob + 32u * static_cast<uint32_t>(cc), o);
          }
        }
        ptx::tmem_st_wait();  // P (and a rescaled O) in tensor memory before the hand-off
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(lead_pfull + 8u * b);
        if (++b == 2) {
          b = 0;
          bph ^= 1;
        }
      }
      if (!ok) break;
      // the item's output: O / l once its last P V has landed
      if (!wait_pv(g - 1)) { ok = false; break; }
      const float inv = 1.f / l;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        ptx::tmem_ld_32cols(ob + 32u * static_cast<uint32_t>(cc), o);
        ptx::tmem_ld_wait();
        ptx::tmem_regs_ready(o);
        if (qrow < p.tokens) {
          __nv_bfloat16 *dst =
              static_cast<__nv_bfloat16 *>(hd.out) + static_cast<long long>(qrow) * hd.out_ld + 32 * cc;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
            memcpy(&w.x, &h0, 4);
            memcpy(&w.y, &h1, 4);
            memcpy(&w.z, &h2, 4);
            memcpy(&w.w, &h3, 4);
            *reinterpret_cast<uint4 *>(dst + i) = w;
          }
        }
      }
      // O has been read before this thread's next P hand-off, after which the
      // next item's first P V overwrites it
      ptx::tc_fence_before();
      ++c.ic;
      load(c);
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
  ptx::cluster_sync();  // neither CTA leaves while the other may still touch its smem or TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
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
  if (env && (env[0] == '1' || env[0] == '3' || env[0] == '4') && env[1] == 0) return env[0] - '0';
  return 2;
}

int attention_k_box_rows(int variant) { return variant == 3 || variant == 4 ? kKb : kTileK; }

// Rows of the V^T boxes: the SM-pair kernel loads half of the head dims per CTA.
int attention_v_box_rows(int variant) { return variant == 4 ? 64 : kTileK; }

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
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attention4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kAttn4Smem));
      if (e != cudaSuccess) return cuda_fail(e);
      if (dev < 64) configured |= 1ULL << dev;
    }
  }
  p.heads_total = total_heads;
  if (p.variant == 4) {
    // one pair per 256-query item, at most as many pairs as are resident at once
    static int resident[64] = {};
    std::lock_guard<std::mutex> g(mu);
    int pairs = dev < 64 ? resident[dev] : 0;
    if (pairs <= 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(kAttn4Threads);
      cfg.dynamicSmemBytes = kAttn4Smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&pairs, k_attention4, &cfg) != cudaSuccess || pairs <= 0)
        pairs = num_sms() / 2;
      cudaGetLastError();  // a failed query leaves no sticky error behind
      if (dev < 64) resident[dev] = pairs;
    }
    const long long items = static_cast<long long>((p.tokens + 255) / 256) * total_heads;
    const dim3 grid(static_cast<unsigned>(2 * (items < pairs ? items : pairs)));
    return launch_checked(launch_kernel(k_attention4, grid, dim3(kAttn4Threads), kAttn4Smem, s, 2, p));
  }
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
