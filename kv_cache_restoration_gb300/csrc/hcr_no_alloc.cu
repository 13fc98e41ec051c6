// hcr_restore_no_alloc: hcr_restore for callers that cannot allocate device
// memory.
//
// A restore needs a small device scratch area (per-token slot and position,
// per-row norm statistics).  hcr_restore takes it from the caller.  Some
// callers have no way to provide it: a serving engine that handed all of
// its free HBM to the paged KV pool when it started has nothing left to
// allocate from, and cudaMalloc/cudaFree can synchronise the device, which
// would stall the decode work the engine keeps running on other streams.
// For them the scratch lives here, in one fixed array in device global
// memory that is part of the library image: every GPU that loads the
// library holds it until the process exits.
//
// Host code may not use the array's name as a device address (on the host it
// names a stand-in object), so the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and then passed to the
// kernels like any caller-provided workspace.
#include <mutex>

#include "hcr_host.h"

namespace hcr {
namespace {

static __device__ __align__(256) uint8_t g_restore_scratch[HCR_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace
}  // namespace hcr

extern "C" hcr_status hcr_restore_no_alloc(hcr_handle* h, const void* hidden, int32_t layer_begin,
                                           int32_t layer_end, int32_t n_req, int32_t n_tokens,
                                           const int32_t* cu_seqlens, const int32_t* start_pos,
                                           const int32_t* block_table,
                                           int32_t max_blocks_per_req, void* k_cache,
                                           void* v_cache, const hcr_cache_layout* layout,
                                           void* stream) {
  using namespace hcr;
  if (!h) return set_last_error(HCR_ERR_INVALID_ARG, "handle is NULL");
  const size_t need = hcr_workspace_bytes(h, n_tokens, layer_end - layer_begin);
  if (need > size_t(HCR_NO_ALLOC_SCRATCH_BYTES))
    return set_last_error(HCR_ERR_WORKSPACE,
                          "restore needs %zu bytes of scratch; hcr_restore_no_alloc has %u "
                          "(restore fewer tokens or layers per call, or use hcr_restore)",
                          need, unsigned(HCR_NO_ALLOC_SCRATCH_BYTES));
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_last_error(HCR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  }
  if (dev != h->impl.device)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "device %d is current but the handle was created on device %d", dev,
                          h->impl.device);
  if (dev < 0 || dev >= kMaxDevices)
    return set_last_error(HCR_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_restore_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return set_last_error(HCR_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                              cudaGetErrorString(e));
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return hcr_restore(h, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                     block_table, max_blocks_per_req, k_cache, v_cache, layout, scratch,
                     HCR_NO_ALLOC_SCRATCH_BYTES, stream);
}
