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
// names a stand-in object), so the address is looked up with
// cudaGetSymbolAddress, with the handle's device current, and then passed to
// the kernels like any caller-provided workspace.  The lookup is done once
// per device and CUDA context: a context that is torn down and created again
// (cudaDeviceReset, or a released primary context) loads the library's device
// code again, possibly at another address, so the cached address is keyed on
// the context's unique id and looked up again when that id changes.
#include <mutex>

#include "hcr_host.h"

namespace hcr {
namespace {

static __device__ __align__(256) uint8_t g_restore_scratch[HCR_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id = 0;   // 0: not looked up yet
  void* addr = nullptr;
};
std::mutex g_scratch_mutex;
ScratchAddr g_scratch[kMaxDevices];

// The unique id of the calling thread's current CUDA context (0 if none is
// current yet), through the runtime's driver entry points, so the library
// needs no link-time dependency on libcuda.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

hcr_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  *id = 0;
  if (!get_current || !get_id)
    return set_last_error(HCR_ERR_CUDA, "driver entry points cuCtxGetCurrent/cuCtxGetId missing");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS)
    return set_last_error(HCR_ERR_CUDA, "cuCtxGetCurrent failed");
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS)
    return set_last_error(HCR_ERR_CUDA, "cuCtxGetId failed");
  return HCR_OK;
}

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
  const size_t need = workspace_min_bytes(h, n_tokens, layer_end - layer_begin);
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
  unsigned long long ctx = 0;
  hcr_status st = current_context_id(&ctx);
  if (st != HCR_OK) return st;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddr& c = g_scratch[dev];
    if (ctx == 0 || c.ctx_id != ctx) {
      // first call in this context (or no context current on this thread yet:
      // the lookup makes the device's primary context current)
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_restore_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return set_last_error(HCR_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                              cudaGetErrorString(e));
      }
      if (ctx == 0 && (st = current_context_id(&ctx)) != HCR_OK) return st;
      c.ctx_id = ctx;
      c.addr = p;
    }
    scratch = c.addr;
  }
  return hcr_restore(h, hidden, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos,
                     block_table, max_blocks_per_req, k_cache, v_cache, layout, scratch,
                     HCR_NO_ALLOC_SCRATCH_BYTES, stream);
}
