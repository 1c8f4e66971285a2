// Internal declarations shared by the library's translation units (not part of
// the public ABI). Kernels of different translation units reach the device
// status word through a pointer argument, so no relocatable device code is
// needed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "tpgqa.h"

namespace tpgqa {

// ---------------------------------------------------------------------------
// Device status word and bounded waits
// ---------------------------------------------------------------------------
// Codes written to the device status word (first writer wins).
enum : int {
  kDevOk = 0,
  kDevTimeoutProducer = 0x101,  // TMA producer gave up waiting for a free stage
  kDevTimeoutMma = 0x102,       // MMA issuer gave up waiting for a full stage
  kDevTimeoutEpilogue = 0x103,  // epilogue gave up waiting for the accumulator
  kDevTimeoutDrain = 0x104,     // teardown gave up waiting for in-flight copies
  kDevTimeoutDebug = 0x1FF,     // tp_debug_wait_timeout's wait
  kDevBadToken = 0x201,         // an embedding lookup met a token id outside [0, V)
};

struct DevCtx {
  int *status;           // device status word
  long long wait_ns;     // budget of every bounded wait, nanoseconds
};

// Returns the context for kernels launched now (status word address is
// resolved once per device). Returns cudaSuccess or the failing error.
cudaError_t get_dev_ctx(DevCtx *out);

int num_sms();

// Records a failed CUDA call for tp_last_cuda_error() and returns TP_ERR_CUDA.
tp_status cuda_fail(cudaError_t e);

// Whether kernels are launched with programmatic stream serialization (PDL):
// every kernel of the library waits (griddepcontrol.wait) before it touches
// global memory, so the next kernel in a stream may launch and run its prologue
// while the previous one finishes. TPGQA_PDL=0 turns it off.
bool pdl_enabled();

// Counts one kernel launch issued by the library (tp_launch_count).
void note_launch();

// Launches `kernel` on `stream`, with PDL when enabled and with a cluster of
// `cluster_x` CTAs when cluster_x > 1 (kernels whose cluster shape is fixed at
// compile time pass 1).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, unsigned cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster_x > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) note_launch();
  return e;
}

// ---------------------------------------------------------------------------
// bf16 tensor-core grouped GEMM (tcgen05 + TMA), C = A * B^T, both K-major.
// ---------------------------------------------------------------------------
constexpr int kMaxMaps = 48;
constexpr int kMaxRingCopies = 8;  // outputs of the split-K ring fold
constexpr int kMaxProblems = 72;  // a column GEMM over reduce-scatter chunks has N*N problems
constexpr int kMaxSegs = 80;

enum Epilogue : int {
  kEpiF32 = 0,     // store fp32 accumulators
  kEpiBF16 = 1,    // store bf16 (round to nearest even)
  kEpiSwiGLU = 2,  // B tile = [gate rows ; up rows]; store bf16 silu(g) * u
};

// One K segment of a problem: the accumulator runs over every segment of its
// problem in order (a row-parallel fused sum runs one segment per rank).
struct GemmSeg {
  int a_map;    // tensor map of A (rows = output rows)
  int b_map;    // tensor map of B (rows = output cols; gate rows for SwiGLU)
  int b2_map;   // up rows for SwiGLU, else -1
  int k_tiles;  // ceil(K / 64)
};

struct GemmProblem {
  int m, n;              // output rows / cols of this problem (n counts outputs)
  int m_tiles, n_tiles;
  int tile_begin;        // first linear tile id of this problem
  int seg_begin, seg_count;
  int b_rows_per_blk;    // with a block table: B rows per block slot
  int n_moff;            // with a block table: B maps per segment (entries whose
                         // map offset is not below it are skipped like -1)
  int m_group;           // tile order: 0 = m-tile fastest over the whole problem;
                         // g > 0 = groups of g m-tiles, each group's tiles n-tile by
                         // n-tile (keeps a group's A and B rows in L2 together)
  void *out;             // output base (row-major)
  long long ldc;         // elements
  // Two-output problem (SM-pair kernel, bf16 epilogue, 256-column tiles only):
  // B comes from b_map (first 128 tile columns, stored to out) and b2_map (last
  // 128, stored to out2), n columns each. Null: one output.
  void *out2;
  long long ldc2;
  // Optional device table, one entry per m-tile, written by an earlier kernel
  // (the MoE routing): -1 skips the tile; otherwise (map_offset << 16) | slot
  // takes B from map b_map + map_offset (b2_map + map_offset for SwiGLU), rows
  // from slot * b_rows_per_blk on. Null: every tile, B rows from 0.
  const int *blk;
};

struct GemmParams {
  CUtensorMap maps[kMaxMaps];
  GemmProblem prob[kMaxProblems];
  GemmSeg seg[kMaxSegs];
  int num_problems;
  int total_tiles;
  int n_maps_used;
  int prefetch;  // L2 prefetch distance of B tiles, in k-blocks (0 = none)
  int split;     // split-K factor of the cluster kernel (1 = persistent kernels)
  int a_rows;    // rows of every A box (128, or the token count rounded up to 8 when
                 // it is smaller: accumulator rows past it are never stored)
  int box_kt;    // 64-wide k-tiles per TMA copy: 1 = 2-D maps (one copy per k-tile),
                 // >1 = 3-D maps whose box spans that many k-tiles (a whole stage)
  int one_stages;  // pipeline stages of the single-CTA kernels (sized from a_rows)
  // 1: the producer issues the weight (B) loads of its first stages before the
  // grid-dependency wait, so they overlap the previous kernel's tail; the A
  // loads follow the wait. Only when no problem has a block table (which an
  // earlier kernel writes).
  int early_b;
  // Ring-folding row-parallel kernel (0 rows = not folding): one problem whose
  // segments are the N ranks' K slices; every tile lies inside one ring chunk of
  // ring_rows rows, and its per-rank partials are added in that chunk's ring
  // order. The sum goes to ring_copies f32 outputs through the tensor maps
  // ring_out .. ring_out + ring_copies - 1 (32 x 32 boxes, 128-byte swizzle).
  int ring_rows;
  int ring_out;
  int ring_copies;
  // The same fold in the split-K SM-pair kernel (GemmBuilder::ring_split): split s
  // of a cluster computes rank s's partial; the owned rows are summed in the
  // chunk's ring order and stored to ring_dst[0 .. ring_copies - 1] (row pitch of
  // the problem's output).
  void *ring_dst[kMaxRingCopies];
  // Persistent single-CTA kernel only. max_ctas > 0 caps its grid (the other SMs
  // are left to a kernel running beside it). defer_dep_wait = 1: the kernel
  // reads nothing the previous kernel on its stream writes and writes nothing
  // that kernel touches, so it starts at once, and waits for that kernel only
  // before it exits (its completion still implies the previous kernel's).
  int max_ctas;
  int defer_dep_wait;
  int *status;
  long long wait_ns;
};

// Host-side builder of a GemmParams.
struct GemmBuilder {
  GemmParams p;
  int n_maps = 0, n_probs = 0, n_segs = 0;
  int bn = 256;       // tile width in accumulator columns (single CTA: 128, 192,
                      // 224 or 256; SM pair: 256 or 224)
  int epi = kEpiF32;
  bool pair = false;  // SM-pair kernel: 256 x bn tiles, cta_group::2
  int a_rows = 128;   // A box rows of the single-CTA kernels (see a_box_rows)
  int split = 0;      // 0: chosen at launch; >1: split-K over a cluster, reduced in fixed
                      // order through DSMEM; 1: the persistent kernels
  int m_group = 0;    // tile order of the problems added after it is set (GemmProblem::m_group)
  // What each map was made from, so launch() can re-encode them as 3-D maps.
  struct MapArgs {
    const void *base;
    long long rows, k, ld;
    int box_rows;
  };
  MapArgs margs[kMaxMaps];
  bool out_map[kMaxMaps] = {};  // maps made by add_out_map_f32 (kept 2-D)
  GemmBuilder();
  // Tensor map of a bf16 [rows x k] matrix with row pitch ld (elements), boxes
  // of 64 x box_rows, 128-byte swizzle. Returns the map index or -1.
  int add_map(const void *base, long long rows, long long k, long long ld, int box_rows,
              tp_status *err);
  // Tensor map of an f32 [rows x cols] output with row pitch ld (elements), for
  // stores of 32 x 32 boxes from 128-byte-swizzled shared memory. Returns the
  // map index or -1. Not re-encoded by use_3d_boxes.
  int add_out_map_f32(void *base, long long rows, long long cols, long long ld, tp_status *err);
  bool ring = false;  // launch the ring-folding pair kernel (see GemmParams::ring_rows)
  // launch the split-K SM-pair kernel with one split per segment (rank) and the
  // ring fold in its reduction (see GemmParams::ring_dst); 128-column tiles
  bool ring_split = false;
  // Re-encodes every map as a 3-D map whose box spans kt k-tiles, if every
  // map's K is a multiple of 64 with at least kt k-tiles; returns kt, or 1 (the
  // 2-D maps kept) otherwise.
  int use_3d_boxes(int kt);
  // Adds a problem with segments [(a_map, b_map, b2_map, k)...]; returns false
  // if the tables are full.
  bool add_problem(int m, int n, void *out, long long ldc, const int *a_maps, const int *b_maps,
                   const int *b2_maps, const long long *ks, int nseg, const int *blk = nullptr,
                   int b_rows_per_blk = 0, int n_moff = 1);
  // A two-output problem (see GemmProblem::out2): C1 = A * B1^T to out, C2 =
  // A * B2^T to out2, both [m x n], in shared 256-column pair tiles.
  bool add_dual_problem(int m, int n, void *out, long long ldc, void *out2, long long ldc2, int a_map,
                        int b_map, int b2_map, long long k);
  bool dual = false;  // some problem has two outputs (forces the SM-pair kernel, no split)
  int max_ctas = 0;             // see GemmParams::max_ctas (forces no split)
  bool defer_dep_wait = false;  // see GemmParams::defer_dep_wait (forces no split)
  int ctas = 0;                 // after launch(): the CTAs the launch started
  tp_status launch(cudaStream_t stream);
};

// Tile width of the single-CTA kernels (256, 224 or 192 accumulator columns)
// for problems of `rows` rows and ncols[i] output columns.
// max_ctas > 0: the CTAs the launch may use (default: every SM).
int choose_bn(long long rows, const long long *ncols, int nprob, bool swiglu, long long max_ctas = 0);
// Rows of an A box for problems of `rows` rows on the single-CTA kernels.
int a_box_rows(long long rows);
// Tile width of the SM-pair kernel (256 or 224 accumulator columns) for
// problems of m rows and ncols[i] output columns; *b_rows receives the rows of
// a B box (bn / 2: each CTA of the pair loads half of B).
int choose_pair_bn(long long m, const long long *ncols, int nprob, bool swiglu, int *b_rows);
// Whether to run the SM-pair kernel for problems of this many rows.
bool choose_pair(long long rows);
// Split-K factor for `tiles` output tiles of `stages_per_tile` k-stages each
// (1 = no split).
int choose_split(long long tiles, bool pair, long long stages_per_tile);
// Clusters of csize split-K CTAs that can be resident at once on the current
// device, or -1 if the runtime cannot say.
int max_active_clusters(int csize);

// ---------------------------------------------------------------------------
// Exact fp32 SIMT grouped GEMM, C = A * B^T with per-problem K segments.
// ---------------------------------------------------------------------------
constexpr int kMaxF32Problems = 16;
constexpr int kMaxF32Segs = 32;

struct F32Seg {
  const float *a; long long lda;
  const float *b; long long ldb;
  int k;
};
struct F32Problem {
  int m, n, m_tiles, n_tiles, tile_begin, seg_begin, seg_count;
  float *out; long long ldc;
};
struct F32Params {
  F32Problem prob[kMaxF32Problems];
  F32Seg seg[kMaxF32Segs];
  int num_problems, total_tiles;
};
tp_status launch_gemm_f32(const F32Params &p, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Collectives on shard buffers of one device.
// ---------------------------------------------------------------------------
constexpr int kMaxRanks = 64;
struct RankPtrs {
  float *p[kMaxRanks];
};
// One reduce-scatter / all-gather ring step over every rank.
tp_status launch_ring_rs_step(const RankPtrs &b, int n, long long size, int step, cudaStream_t s);
tp_status launch_ring_ag_step(const RankPtrs &b, int n, long long size, int step, cudaStream_t s);
// One pass that folds each chunk in the ring's order; write_all = 1 gives the
// all-reduce, 0 the reduce-scatter (only chunk c of buffer c is written).
tp_status launch_ring_fused(const RankPtrs &b, int n, long long size, int write_all, cudaStream_t s);
// In-place all-gather in one pass: chunk c of buffer c is copied to every other buffer.
tp_status launch_ring_ag_fused(const RankPtrs &b, int n, long long size, cudaStream_t s);
// bf16 destinations of a reduce-scatter: buffer r is a [rows x cols] bf16 matrix
// with row pitch ld (elements) at p[r].
struct Bf16Outs {
  void *p[kMaxRanks];
  long long ld, cols;
};
// One-pass reduce-scatter of the f32 buffers b into bf16: chunk c, folded in the
// ring's order in f32, is rounded to bf16 and written to o.p[c] only.
tp_status launch_ring_rs_bf16(const RankPtrs &b, const Bf16Outs &o, int n, long long size, cudaStream_t s);

// Strided 2-D copy of a shard into an output (all-gather as concatenation).
struct Copy2D {
  const char *src; long long src_pitch;   // bytes
  char *dst; long long dst_pitch;         // bytes
  long long rows, row_bytes;
};
constexpr int kMaxCopies = 128;
struct CopyBatch {
  Copy2D c[kMaxCopies];
  int n;
};
tp_status launch_copy_batch(const CopyBatch &b, cudaStream_t s);

// Vocab-parallel embedding lookup with its all-gather: token i's row comes from
// shard r = ids[i] / rows_per_rank (its row ids[i] - r * rows_per_rank) and is
// stored to every output. Bad ids give zero rows and kDevBadToken.
struct EmbedArgs {
  const char *tab[kMaxRanks];
  long long tab_pitch[kMaxRanks];   // bytes between rows of shard r
  char *out[kMaxRanks];
  long long out_pitch[kMaxRanks];   // bytes between rows of output o
  const int *ids;
  long long n_tokens, rows_per_rank, row_bytes;
  int n, n_outs, esize;
  int *status;
};
// vec16: every base, pitch and the row length are multiples of 16 bytes.
tp_status launch_vocab_embed(const EmbedArgs &a, bool vec16, cudaStream_t s);

// Tensor map of a bf16 [rows x cols] matrix with row pitch ld (elements):
// boxes of 64 columns x box_rows rows, 128-byte swizzle, zero fill out of range.
bool encode_bf16_map_2d(CUtensorMap *map, const void *base, long long rows, long long cols, long long ld,
                        int box_rows);

// ---------------------------------------------------------------------------
// Attention core (attention.cu): one CTA per (128-query tile, q head).
// ---------------------------------------------------------------------------
constexpr int kMaxAttnRanks = 32;
constexpr int kMaxAttnMaps = 3 * kMaxAttnRanks;
constexpr int kMaxAttnHeads = 256;
struct AttnHead {
  int q_map, k_map, v_map;  // map indices: Q of the rank, K and V^T of its kv source
  int q_col;                // first column of this q head in Q (= local head * d)
  int kv_col;               // first column of its kv head in K (= first row in V^T)
  int pad;
  void *out;                // bf16 A_r + q_col: this head's output columns
  long long out_ld;
};
struct AttnParams {
  CUtensorMap maps[kMaxAttnMaps];
  AttnHead heads[kMaxAttnHeads];
  int tokens, q_tiles, causal, heads_total;
  int variant;              // kernel: 1 one query tile per item, 2 two tiles, 3 two tiles in 64-key blocks
  float scale_log2;         // log2(e) / sqrt(d)
  int *status;
  long long wait_ns;
};
tp_status launch_attention(AttnParams &p, int total_heads, cudaStream_t s);
// The attention kernel a call runs (2 by default; TPGQA_ATTN=1 or 3 selects
// another, read on every call) and the rows of its K boxes (keys per block).
int attention_variant();
int attention_k_box_rows(int variant);
// V [rows x cols] (pitch ld_in[z]) -> V^T [cols x rows] (pitch ld_out), bf16,
// for sources z = 0..sources-1 in one launch.
struct TransposeArgs {
  const void *in[kMaxAttnRanks];
  long long ld_in[kMaxAttnRanks];
  void *out[kMaxAttnRanks];
  long long ld_out;
  int rows, cols;
};
tp_status launch_transpose_bf16(const TransposeArgs &a, int sources, cudaStream_t s);

// ---------------------------------------------------------------------------
// Mixture-of-experts block (moe.cu).
// ---------------------------------------------------------------------------
constexpr int kMaxExperts = 256;
// Rows of the routed layout and the workspace regions of tp_moe_block.
struct MoeLayout {
  bool pair;         // SM-pair GEMMs (256-row tiles) or single-CTA (128)
  int bm;            // rows per tile; every expert's rows start on a tile
  long long rows;    // capacity of the layout: T*k + E*(bm-1), rounded up to bm
  long long nblk;    // tiles of rows (entries of the block table)
  size_t off_pos, off_inv, off_blk, off_xp, off_h, off_yp, total;
};
MoeLayout moe_layout(int n, int mode, int experts, int k, long long tokens, long long hidden, long long ffn);
// A validated tp_moe_block call (the combine's all-reduce is left to the caller).
struct MoeCall {
  int n, mode, experts, k, combine;
  long long hidden, ffn;
  const tp_tensor *x;
  const int *ids;
  const float *weights;
  const tp_tensor *w_gate, *w_up, *w_down, *y;
  void *workspace;
};
tp_status moe_forward(const MoeCall &c, cudaStream_t s);

// Kernel that always times out its bounded wait (tests of the timeout path).
tp_status launch_debug_wait(cudaStream_t s);

}  // namespace tpgqa
