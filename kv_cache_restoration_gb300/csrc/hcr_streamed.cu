// hcr_restore_streamed: the layer-pipelined restore.
//
// The HCache episode ("Fast State Restoration for Evicted LLM KV Caches",
// cue 15) overlaps the two resources a restore needs: while layer N's hidden
// states are projected into K and V on the GPU, layer N+1's are already
// being transferred.  Here the hidden states sit in pinned host memory and
// reach HBM over the host link (NVLink-C2C on GB300) by the copy engines on
// a copy stream owned by the handle, one chunk of layers at a time, into a
// ring of staging slots in device memory; each chunk is restored on the
// caller's stream as soon as its copy lands, and a slot is refilled only
// after the restore that read it has finished.
//
//   copy stream:   [copy c0][copy c1][copy c2]....          (waits done[slot])
//   caller stream:          [restore c0][restore c1][....   (waits copied[slot])
#include <mutex>

#include "hcr_internal.h"

namespace hcr {

struct StreamedRes {
  std::mutex mutex;                 // one streamed restore enqueued at a time per handle
  cudaStream_t copy = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t copied[kMaxStagingSlots] = {};
  cudaEvent_t done[kMaxStagingSlots] = {};
};

void release_streamed(Handle& H) {
  StreamedRes* r = H.streamed;
  if (!r) return;
  if (r->copy) cudaStreamDestroy(r->copy);
  if (r->start) cudaEventDestroy(r->start);
  for (int i = 0; i < kMaxStagingSlots; ++i) {
    if (r->copied[i]) cudaEventDestroy(r->copied[i]);
    if (r->done[i]) cudaEventDestroy(r->done[i]);
  }
  delete r;
  H.streamed = nullptr;
}

namespace {

std::mutex g_create_mutex;

hcr_status ensure_resources(Handle& H, StreamedRes** out) {
  std::lock_guard<std::mutex> lock(g_create_mutex);
  if (!H.streamed) {
    auto* r = new (std::nothrow) StreamedRes();
    if (!r) return set_last_error(HCR_ERR_OOM, "host allocation failed");
    cudaError_t e = cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->start, cudaEventDisableTiming);
    for (int i = 0; e == cudaSuccess && i < kMaxStagingSlots; ++i) {
      e = cudaEventCreateWithFlags(&r->copied[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->done[i], cudaEventDisableTiming);
    }
    H.streamed = r;
    if (e != cudaSuccess) {
      release_streamed(H);
      cudaGetLastError();
      return set_last_error(HCR_ERR_CUDA, "creating the copy stream/events: %s",
                            cudaGetErrorString(e));
    }
  }
  *out = H.streamed;
  return HCR_OK;
}

}  // namespace
}  // namespace hcr

using namespace hcr;

extern "C" hcr_status hcr_restore_streamed(
    hcr_handle* h, const void* hidden_host, int32_t layer_begin, int32_t layer_end,
    int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens, const int32_t* start_pos,
    const int32_t* block_table, int32_t max_blocks_per_req, void* k_cache, void* v_cache,
    const hcr_cache_layout* layout, void* staging, size_t staging_bytes,
    int32_t layers_per_chunk, void* workspace, size_t workspace_bytes, void* stream) {
  if (!h) return set_last_error(HCR_ERR_INVALID_ARG, "handle is NULL");
  const hcr_model_dims& d = h->impl.dims;
  if (layer_begin < 0 || layer_end < layer_begin || layer_end > d.n_layers)
    return set_last_error(HCR_ERR_INVALID_ARG, "layer range [%d, %d) outside [0, %d)",
                          layer_begin, layer_end, d.n_layers);
  if (n_tokens < 0) return set_last_error(HCR_ERR_INVALID_ARG, "n_tokens must be >= 0");
  if (n_tokens == 0 || layer_end == layer_begin) return HCR_OK;
  if (!hidden_host) return set_last_error(HCR_ERR_INVALID_ARG, "hidden_host is NULL");
  if (!layout) return set_last_error(HCR_ERR_INVALID_ARG, "layout is NULL");
  if (layers_per_chunk < 1)
    return set_last_error(HCR_ERR_INVALID_ARG, "layers_per_chunk must be >= 1");
  const int32_t n_layers = layer_end - layer_begin;
  const int32_t chunk = std::min(layers_per_chunk, n_layers);
  const size_t layer_bytes = size_t(n_tokens) * size_t(d.d_model) * 2;
  const size_t chunk_bytes = layer_bytes * size_t(chunk);
  if (!staging || reinterpret_cast<uintptr_t>(staging) % 256)
    return set_last_error(HCR_ERR_WORKSPACE, "staging must be non-NULL and 256-byte aligned");
  const int slots = int(std::min<size_t>(staging_bytes / chunk_bytes, kMaxStagingSlots));
  if (slots < 1)
    return set_last_error(HCR_ERR_WORKSPACE, "staging has %zu bytes; one chunk of %d layers "
                          "needs %zu", staging_bytes, chunk, chunk_bytes);
  if (workspace_bytes < hcr_workspace_bytes(h, n_tokens, chunk))
    return set_last_error(HCR_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu for a chunk",
                          workspace_bytes, hcr_workspace_bytes(h, n_tokens, chunk));
  const int64_t row = int64_t(d.n_kv_heads) * d.head_dim;
  const int64_t stride = layout->layer_stride_elems
                             ? layout->layer_stride_elems
                             : int64_t(layout->num_blocks) * layout->block_size * row;

  StreamedRes* r = nullptr;
  hcr_status st = ensure_resources(h->impl, &r);
  if (st != HCR_OK) return st;
  std::lock_guard<std::mutex> lock(r->mutex);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto cuda_err = [](cudaError_t e, const char* what) {
    cudaGetLastError();
    return set_last_error(HCR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  };
  cudaError_t e;
  // Work already queued on the caller's stream (an earlier user of the
  // staging ring, say) comes before the first copy.
  if ((e = cudaEventRecord(r->start, s)) != cudaSuccess) return cuda_err(e, "event record");
  if ((e = cudaStreamWaitEvent(r->copy, r->start, 0)) != cudaSuccess)
    return cuda_err(e, "stream wait");
  const uint8_t* src = static_cast<const uint8_t*>(hidden_host);
  uint8_t* ring = static_cast<uint8_t*>(staging);
  int c = 0;
  for (int32_t l0 = 0; l0 < n_layers; l0 += chunk, ++c) {
    const int32_t nl = std::min(chunk, n_layers - l0);
    const int slot = c % slots;
    void* dst = ring + size_t(slot) * chunk_bytes;
    if (c >= slots && (e = cudaStreamWaitEvent(r->copy, r->done[slot], 0)) != cudaSuccess)
      return cuda_err(e, "stream wait");
    if ((e = cudaMemcpyAsync(dst, src + size_t(l0) * layer_bytes, size_t(nl) * layer_bytes,
                             cudaMemcpyHostToDevice, r->copy)) != cudaSuccess)
      return cuda_err(e, "hidden-state copy");
    if ((e = cudaEventRecord(r->copied[slot], r->copy)) != cudaSuccess)
      return cuda_err(e, "event record");
    if ((e = cudaStreamWaitEvent(s, r->copied[slot], 0)) != cudaSuccess)
      return cuda_err(e, "stream wait");
    st = hcr_restore(h, dst, layer_begin + l0, layer_begin + l0 + nl, n_req, n_tokens,
                     cu_seqlens, start_pos, block_table, max_blocks_per_req,
                     static_cast<uint16_t*>(k_cache) + int64_t(l0) * stride,
                     static_cast<uint16_t*>(v_cache) + int64_t(l0) * stride, layout, workspace,
                     workspace_bytes, stream);
    if (st != HCR_OK) return st;
    if ((e = cudaEventRecord(r->done[slot], s)) != cudaSuccess)
      return cuda_err(e, "event record");
  }
  return HCR_OK;
}
