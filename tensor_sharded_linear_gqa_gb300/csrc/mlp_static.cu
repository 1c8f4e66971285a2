// tp_mlp_block_static: the MLP block with its intermediate H kept in a fixed
// scratch array that is part of the library image, for callers that cannot
// allocate device memory or hand the library a workspace.
//
// Who needs this: a plug-in loaded into a host framework that owns every byte
// of device memory through its own allocator and gives plug-ins no way to
// borrow any; a serving process that reserved all free HBM for weights and KV
// cache at start-up, where a later cudaMalloc would fail, or would stall every
// stream while requests are in flight. Such callers still own their inputs and
// outputs, but cannot provide the [tokens x ffn] bf16 buffer that tp_mlp_block
// takes as `workspace`.
//
// The scratch is a file-scope __device__ array of kStaticScratchBytes (16 MiB).
// Every GPU that loads this library reserves it when the module is loaded and
// keeps it until the process exits. Host code cannot use the array's name as a
// device address (on the host it names a shadow variable), so the device
// address is looked up once per device with cudaGetSymbolAddress, with that
// device current, and handed to the kernels.
#include <mutex>

#include "tp_internal.h"

namespace tpgqa {
namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // holds H for tokens * ffn <= 8 Mi elements

static __device__ __align__(256) unsigned char g_mlp_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {nullptr};

// Device address of the scratch on the current device; the first call on a
// device performs the lookup (with that device current) and caches it.
tp_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return TP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mlp_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TP_OK;
}

}  // namespace
}  // namespace tpgqa

extern "C" size_t tp_mlp_block_static_max_bytes(void) { return tpgqa::kStaticScratchBytes; }

extern "C" tp_status tp_mlp_block_static(const tp_plan *plan, const tp_tensor *x,
                                         const tp_tensor *w_gate, const tp_tensor *w_up,
                                         const tp_tensor *w_down, tp_tensor *y, int32_t combine,
                                         tp_stream_t stream) {
  if (!plan || !x) return TP_ERR_INVALID_ARG;
  if (x->rows < 0) return TP_ERR_INVALID_ARG;
  // H needs tokens * ffn bf16 values; refuse anything the fixed scratch cannot hold.
  const size_t need = tp_mlp_block_workspace_size(plan, x->rows);
  if (need > tpgqa::kStaticScratchBytes) return TP_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (x->rows > 0) {
    const tp_status st = tpgqa::scratch_address(&scratch);
    if (st != TP_OK) return st;
  }
  // H is written in full by the gate/up GEMM before the down GEMM reads it, so
  // the scratch needs no clearing between calls.
  return tp_mlp_block(plan, x, w_gate, w_up, w_down, y, combine, scratch,
                      tpgqa::kStaticScratchBytes, stream);
}
