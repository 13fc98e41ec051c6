// The save side of hidden-state restoration: scatter layer inputs into
// fixed-size chunks laid out token-before-layer.
//
// HCache episode ("Fast State Restoration for Evicted LLM KV Caches"):
// generation produces hidden states layer-before-token (cue 16: each step
// yields every layer's input for its one new token), while a restore wants
// one layer's tokens together; they are stored in fixed 64-token chunks
// (cue 22).  Here a chunk holds positions [C*k, C*k + C) of one request for
// all layers, element (l, p, i) at chunk[id][l][p % C][i], with the
// physical id from a per-request chunk table.  Within one chunk each layer's
// tokens are contiguous, so a restore of one layer reads 64-token runs.
//
// save_kernel: one warp per (layer, token) row; grid.y runs over layers.  Lane 0 maps the token to
// (request, position, chunk id, offset) by binary search on cu_seqlens and
// broadcasts it; the warp then copies the row's d_model 16-bit values with
// 16-byte vector loads and stores (four in flight per lane).  Rows whose
// chunk id or logical chunk is out of range are skipped and flagged in the
// handle's device error word.  The chunk store may be device memory or
// pinned host memory the device can address: then these stores cross the
// host link directly and no separate snapshot copy is needed.
#include "hcr_host.h"

namespace hcr {
namespace {

constexpr int kSaveThreads = 256;

struct SaveParams {
  const uint16_t* hidden;      // [Lr][T][d]
  const int32_t* cu_seqlens;
  const int32_t* start_pos;
  const int32_t* chunk_table;  // [R][max_chunks]
  uint16_t* store;             // [num_chunks][n_layers][C][d]
  uint32_t* err;
  int32_t n_req, n_tokens, max_chunks, chunk_tokens, num_chunks, n_layers_total, layer_begin,
      n_layers, d_model;
};

// grid.y = layer within the range; warps of grid.x stride over tokens.
__global__ void __launch_bounds__(kSaveThreads) save_kernel(const SaveParams p) {
  const int lane = threadIdx.x & 31;
  const int li = blockIdx.y;
  const int warp0 = int((blockIdx.x * kSaveThreads + threadIdx.x) >> 5);
  const int nwarps = int((gridDim.x * kSaveThreads) >> 5);
  const int nvec = p.d_model >> 3;   // 16-byte vectors per row
  for (int t = warp0; t < p.n_tokens; t += nwarps) {
    const int64_t row = int64_t(li) * p.n_tokens + t;
    int cid_sel = -1, off_sel = 0;   // chunk id and offset (lane 0), -1: skip the row
    if (lane == 0) {
      uint32_t bad = 0;
      int lo = 0, hi = p.n_req - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu_seqlens + mid) <= t) lo = mid; else hi = mid - 1;
      }
      const int c0 = __ldg(p.cu_seqlens + lo), c1 = __ldg(p.cu_seqlens + lo + 1);
      if (!(c0 <= t && t < c1)) {
        bad = HCR_DEVERR_SEQLENS;
      } else {
        const int start = __ldg(p.start_pos + lo);
        const int pos = start + (t - c0);
        if (start < 0 || pos < start) {
          bad = HCR_DEVERR_POSITION;
        } else if (pos / p.chunk_tokens >= p.max_chunks) {
          bad = HCR_DEVERR_LOGICAL_BLOCK;
        } else {
          const int cid = __ldg(p.chunk_table + int64_t(lo) * p.max_chunks + pos / p.chunk_tokens);
          if (cid < 0 || cid >= p.num_chunks) {
            bad = HCR_DEVERR_BLOCK_ID;
          } else {
            cid_sel = cid;
            off_sel = pos % p.chunk_tokens;
          }
        }
      }
      if (bad && li == 0) atomicOr(p.err, bad);   // report once per token
    }
    cid_sel = __shfl_sync(0xffffffffu, cid_sel, 0);
    off_sel = __shfl_sync(0xffffffffu, off_sel, 0);
    if (cid_sel < 0) continue;
    const int64_t dst_row =
        (int64_t(cid_sel) * p.n_layers_total + p.layer_begin + li) * p.chunk_tokens + off_sel;
    const uint4* src = reinterpret_cast<const uint4*>(p.hidden + row * p.d_model);
    uint4* dst = reinterpret_cast<uint4*>(p.store + dst_row * p.d_model);
    int v = lane;
    for (; v + 96 < nvec; v += 128) {
      const uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64),
                  e = __ldg(src + v + 96);
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = e;
    }
    for (; v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

}  // namespace

// Host memory is used through its device address; memory the device cannot
// reach (unregistered pageable memory without pageable-memory access) is
// refused instead of letting a kernel fault on it.
hcr_status device_view(const Handle& H, void* ptr, const char* what, void** out) {
  *out = ptr;
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_last_error(HCR_ERR_CUDA, "cudaPointerGetAttributes(%s): %s", what,
                          cudaGetErrorString(e));
  }
  if (attr.type == cudaMemoryTypeHost) {
    if (!attr.devicePointer)
      return set_last_error(HCR_ERR_INVALID_ARG, "%s host memory is not mapped", what);
    *out = attr.devicePointer;
  } else if (attr.type == cudaMemoryTypeUnregistered) {
    int pageable = 0;
    cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, H.device);
    if (!pageable)
      return set_last_error(HCR_ERR_INVALID_ARG,
                            "%s is unregistered host memory the device cannot access", what);
  }
  return HCR_OK;
}

}  // namespace hcr

using namespace hcr;

extern "C" hcr_status hcr_save_hidden(hcr_handle* h, const void* hidden, int32_t layer_begin,
                                      int32_t layer_end, int32_t n_req, int32_t n_tokens,
                                      const int32_t* cu_seqlens, const int32_t* start_pos,
                                      const int32_t* chunk_table, int32_t max_chunks_per_req,
                                      int32_t chunk_tokens, void* chunk_store,
                                      int32_t num_chunks, void* stream) {
  NvtxRange range("hcr_save_hidden");
  if (!h) return set_last_error(HCR_ERR_INVALID_ARG, "handle is NULL");
  const hcr_model_dims& d = h->impl.dims;
  if (layer_begin < 0 || layer_end < layer_begin || layer_end > d.n_layers)
    return set_last_error(HCR_ERR_INVALID_ARG, "layer range [%d, %d) outside [0, %d)",
                          layer_begin, layer_end, d.n_layers);
  if (n_tokens < 0 || n_req < 0)
    return set_last_error(HCR_ERR_INVALID_ARG, "n_tokens and n_req must be >= 0");
  if (n_tokens == 0 || layer_end == layer_begin) return HCR_OK;
  if (n_req < 1) return set_last_error(HCR_ERR_INVALID_ARG, "n_tokens > 0 needs n_req >= 1");
  if (!hidden || !chunk_store || reinterpret_cast<uintptr_t>(hidden) % 16 ||
      reinterpret_cast<uintptr_t>(chunk_store) % 16)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "hidden and chunk_store must be non-NULL and 16-byte aligned");
  if (!cu_seqlens || !start_pos || !chunk_table)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "cu_seqlens, start_pos and chunk_table must be non-NULL");
  if (max_chunks_per_req < 1 || chunk_tokens < 1 || num_chunks < 1)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "max_chunks_per_req, chunk_tokens and num_chunks must be >= 1");
  void* store = nullptr;
  hcr_status st = device_view(h->impl, chunk_store, "chunk_store", &store);
  if (st != HCR_OK) return st;
  SaveParams p{};
  p.hidden = static_cast<const uint16_t*>(hidden);
  p.cu_seqlens = cu_seqlens;
  p.start_pos = start_pos;
  p.chunk_table = chunk_table;
  p.store = static_cast<uint16_t*>(store);
  p.err = h->impl.err;
  p.n_req = n_req;
  p.n_tokens = n_tokens;
  p.max_chunks = max_chunks_per_req;
  p.chunk_tokens = chunk_tokens;
  p.num_chunks = num_chunks;
  p.n_layers_total = d.n_layers;
  p.layer_begin = layer_begin;
  p.n_layers = layer_end - layer_begin;
  p.d_model = d.d_model;
  // enough warps per layer to keep ~16 resident 256-thread blocks per SM busy
  const int64_t want_x = (int64_t(n_tokens) * 32 + kSaveThreads - 1) / kSaveThreads;
  const int64_t cap_x = std::max<int64_t>(1, int64_t(h->impl.num_sms) * 16 / p.n_layers);
  const dim3 grid(unsigned(std::min(want_x, cap_x)), unsigned(p.n_layers));
  save_kernel<<<grid, kSaveThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_last_error(HCR_ERR_CUDA, "save launch: %s", cudaGetErrorString(e));
  return HCR_OK;
}
