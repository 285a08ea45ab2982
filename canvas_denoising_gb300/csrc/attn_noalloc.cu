// dg_canvas_attn_noalloc: canvas attention without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they run attention:
// hosts whose memory manager owns every device allocation and forbids side
// allocations, plugins that are handed tensors but no scratch buffer, and
// latency-critical loops where a cudaMalloc could synchronise the device. For
// them this entry point keeps its split-KV scratch in a fixed array in device
// memory that is part of the library image itself.
//
// The array is kAttnScratchBytes (32 MiB). Every GPU that loads the library
// keeps that memory reserved until the process exits. All calls share the one
// array: calls that can overlap on the GPU (different streams without
// ordering between them) race on it and must not be issued. The contents left
// by the previous call do not matter: the call zeroes the per-group arrival
// counters it needs, stream-ordered, before the attention kernel reads them
// (the same reset the workspace entry point issues), and every partial result
// is written before it is read.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side shadow). The device address is looked up with
// cudaGetSymbolAddress once per device, on the first call made while that
// device is current; that first call should therefore come before any stream
// capture begins on the device.
#include <mutex>

#include "dg_common.cuh"

namespace dg {
namespace {

constexpr size_t kAttnScratchBytes = 32u << 20;

static __device__ __align__(256) unsigned char g_attn_scratch[kAttnScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set-up on first use).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_attn_scratch) != cudaSuccess || !ptr) return DG_ERR_CUDA;
    g_addr[dev] = ptr;
  }
  *out = g_addr[dev];
  return DG_OK;
}

}  // namespace
}  // namespace dg

extern "C" size_t dg_canvas_attn_noalloc_max_scratch(void) { return dg::kAttnScratchBytes; }

extern "C" int dg_canvas_attn_noalloc(const void* q, const void* k_cache, const void* v_cache, int64_t cap,
                                      int64_t prefix_len, const void* k_canvas, const void* v_canvas, void* out,
                                      float* lse, int C, int Hq, int Hkv, int hd, float scale, int dtype, int mask,
                                      void* stream) {
  const size_t need = dg_canvas_attn_workspace_size(C, Hq, Hkv, hd, prefix_len, dtype);
  if (need > dg::kAttnScratchBytes) return DG_ERR_WORKSPACE;  // beyond this entry point's fixed scratch
  void* scratch = nullptr;
  const int rc = dg::scratch_address(&scratch);
  if (rc != DG_OK) return rc;
  return dg_canvas_attn(q, k_cache, v_cache, cap, prefix_len, k_canvas, v_canvas, out, lse, C, Hq, Hkv, hd, scale,
                        dtype, mask, scratch, dg::kAttnScratchBytes, stream);
}
