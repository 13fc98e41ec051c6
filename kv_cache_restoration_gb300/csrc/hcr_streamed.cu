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
//
// The host copy is either [layer][token][d] hidden states (one linear copy
// per chunk of layers) or a store of fixed-size chunks as hcr_save_hidden
// writes them ([chunk][layer][row][d]): then every run of one request's
// tokens inside one chunk becomes one 2-D copy that gathers its rows for all
// layers of the chunk of layers at once, so the copy engines do the
// chunk-to-layer transpose on the way.
#include <functional>
#include <mutex>
#include <vector>

#include "hcr_host.h"

namespace hcr {

struct StreamedRes {
  std::mutex mutex;                 // one streamed restore enqueued at a time per handle
  cudaStream_t copy = nullptr;
  cudaStream_t side = nullptr;      // work between a copy and its restore (the codec's decode)
  cudaEvent_t start = nullptr;
  cudaEvent_t copied[kMaxStagingSlots] = {};
  cudaEvent_t landed[kMaxStagingSlots] = {};   // copy done, before the side work
  cudaEvent_t done[kMaxStagingSlots] = {};
};

void release_streamed(Handle& H) {
  StreamedRes* r = H.streamed;
  if (!r) return;
  if (r->copy) cudaStreamDestroy(r->copy);
  if (r->side) cudaStreamDestroy(r->side);
  if (r->start) cudaEventDestroy(r->start);
  for (int i = 0; i < kMaxStagingSlots; ++i) {
    if (r->copied[i]) cudaEventDestroy(r->copied[i]);
    if (r->landed[i]) cudaEventDestroy(r->landed[i]);
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
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&r->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->start, cudaEventDisableTiming);
    for (int i = 0; e == cudaSuccess && i < kMaxStagingSlots; ++i) {
      e = cudaEventCreateWithFlags(&r->copied[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->landed[i], cudaEventDisableTiming);
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

// One unit of the pipeline: layers [l0, l0 + nl) (relative to the call's
// first layer), restored from hidden states or, for kv, placed from saved K/V.
struct Item {
  bool kv;
  int32_t l0, nl;
};

// Copies an item's host data into `dst` on `copy`: hidden states laid out
// [nl][n_tokens][d_model], or K/V laid out [nl][2][n_tokens][d_kv].
using CopyFn = std::function<hcr_status(const Item& it, void* dst, cudaStream_t copy)>;

// Optional GPU work between an item's copy and its processing (the codec's
// decode), enqueued on the handle's side stream after the copy has landed, so
// that the next copies do not queue behind it.
using SideFn = std::function<hcr_status(const Item& it, void* dst, cudaStream_t side)>;

hcr_status copy_status(cudaError_t e) {
  if (e == cudaSuccess) return HCR_OK;
  cudaGetLastError();
  return set_last_error(HCR_ERR_CUDA, "host copy: %s", cudaGetErrorString(e));
}

hcr_status run_pipeline(hcr_handle* h, const std::vector<Item>& items, size_t slot_bytes,
                        int32_t layer_begin, int32_t n_req, int32_t n_tokens,
                        const int32_t* cu_seqlens, const int32_t* start_pos,
                        const int32_t* block_table, int32_t max_blocks_per_req, void* k_cache,
                        void* v_cache, const hcr_cache_layout* layout, void* staging,
                        size_t staging_bytes, size_t workspace_need, void* workspace,
                        size_t workspace_bytes, void* stream, const CopyFn& copy_item,
                        const SideFn* side = nullptr, size_t hidden_offset = 0) {
  NvtxRange range("hcr.streamed_pipeline");
  const hcr_model_dims& d = h->impl.dims;
  if (!layout) return set_last_error(HCR_ERR_INVALID_ARG, "layout is NULL");
  if (!staging || reinterpret_cast<uintptr_t>(staging) % 256)
    return set_last_error(HCR_ERR_WORKSPACE, "staging must be non-NULL and 256-byte aligned");
  const int slots = int(std::min<size_t>(staging_bytes / slot_bytes, kMaxStagingSlots));
  if (slots < 1)
    return set_last_error(HCR_ERR_WORKSPACE, "staging has %zu bytes; one slot needs %zu",
                          staging_bytes, slot_bytes);
  if (workspace_bytes < workspace_need)
    return set_last_error(HCR_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu for a chunk",
                          workspace_bytes, workspace_need);
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
  // Overlapped statistics: when the workspace has room for one group's norm
  // statistics per staging slot, the slot map is computed once here, each
  // hidden-state group's statistics on the side stream as soon as the group
  // has landed (and been decoded), and the caller's stream only projects.
  // The statistics' read of the group's rows then runs under the previous
  // group's projection instead of before its own.  Otherwise every group is
  // restored with hcr_restore.
  int32_t max_nl = 0, extent = 0;
  for (const Item& it : items) {
    if (!it.kv) max_nl = std::max(max_nl, it.nl);
    extent = std::max(extent, it.l0 + it.nl);
  }
  bool overlap = false;
  if (max_nl > 0 &&
      (st = pipeline_placement(h, staging, layer_begin, layer_begin + extent, n_req, n_tokens,
                               cu_seqlens, start_pos, block_table, max_blocks_per_req, k_cache,
                               v_cache, layout, workspace, workspace_bytes, slots * max_nl,
                               stream, &overlap)) != HCR_OK)
    return st;
  const WorkspaceLayout wl =
      workspace_layout(n_tokens, int64_t(slots) * max_nl, d.norm == HCR_NORM_LAYER);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t slot_stats = size_t(max_nl) * size_t(n_tokens);   // floats per slot
  uint8_t* ring = static_cast<uint8_t*>(staging);
  for (size_t c = 0; c < items.size(); ++c) {
    const Item& it = items[c];
    const int slot = int(c % size_t(slots));
    void* dst = ring + size_t(slot) * slot_bytes;
    if (c >= size_t(slots) &&
        (e = cudaStreamWaitEvent(r->copy, r->done[slot], 0)) != cudaSuccess)
      return cuda_err(e, "stream wait");
    {
      NvtxRange copy_range(it.kv ? "hcr.copy_kv_group" : "hcr.copy_hidden_group");
      if ((st = copy_item(it, dst, r->copy)) != HCR_OK) return st;
    }
    const int32_t lb = layer_begin + it.l0;
    uint8_t* rows = static_cast<uint8_t*>(dst) + hidden_offset;   // the group's hidden rows
    const bool own_stats = overlap && !it.kv;
    float* rstd = own_stats
                      ? reinterpret_cast<float*>(ws + wl.rstd_off) + size_t(slot) * slot_stats
                      : nullptr;
    float* mean = own_stats && d.norm == HCR_NORM_LAYER
                      ? reinterpret_cast<float*>(ws + wl.mean_off) + size_t(slot) * slot_stats
                      : nullptr;
    cudaStream_t ready = r->copy;   // where the item is ready for processing
    if ((side && !it.kv) || own_stats) {
      if ((e = cudaEventRecord(r->landed[slot], r->copy)) != cudaSuccess)
        return cuda_err(e, "event record");
      if ((e = cudaStreamWaitEvent(r->side, r->landed[slot], 0)) != cudaSuccess)
        return cuda_err(e, "stream wait");
      if (side && !it.kv && (st = (*side)(it, dst, r->side)) != HCR_OK) return st;
      if (own_stats &&
          (st = pipeline_stats(h, rows, lb, lb + it.nl, n_req, n_tokens, cu_seqlens, start_pos,
                               block_table, max_blocks_per_req, k_cache, v_cache, layout,
                               workspace, workspace_bytes, rstd, mean, r->side)) != HCR_OK)
        return st;
      ready = r->side;
    }
    if ((e = cudaEventRecord(r->copied[slot], ready)) != cudaSuccess)
      return cuda_err(e, "event record");
    if ((e = cudaStreamWaitEvent(s, r->copied[slot], 0)) != cudaSuccess)
      return cuda_err(e, "stream wait");
    auto* kc = static_cast<uint16_t*>(k_cache) + int64_t(it.l0) * stride;
    auto* vc = static_cast<uint16_t*>(v_cache) + int64_t(it.l0) * stride;
    if (it.kv)
      st = hcr_load_kv(h, dst, lb, lb + it.nl, n_req, n_tokens, cu_seqlens, start_pos,
                       block_table, max_blocks_per_req, kc, vc, layout, workspace,
                       workspace_bytes, stream);
    else if (own_stats)
      st = pipeline_project(h, rows, lb, lb + it.nl, n_req, n_tokens, cu_seqlens, start_pos,
                            block_table, max_blocks_per_req, kc, vc, layout, workspace,
                            workspace_bytes, rstd, mean, stream);
    else
      st = hcr_restore(h, rows, lb, lb + it.nl, n_req, n_tokens, cu_seqlens, start_pos,
                       block_table, max_blocks_per_req, kc, vc, layout, workspace,
                       workspace_bytes, stream);
    if (st != HCR_OK) return st;
    if ((e = cudaEventRecord(r->done[slot], s)) != cudaSuccess)
      return cuda_err(e, "event record");
  }
  return HCR_OK;
}

// Hidden-state groups of `layers_per_chunk` layers over [layer_begin, layer_end).
hcr_status hidden_pipeline(hcr_handle* h, int32_t layer_begin, int32_t layer_end, int32_t n_req,
                           int32_t n_tokens, const int32_t* cu_seqlens, const int32_t* start_pos,
                           const int32_t* block_table, int32_t max_blocks_per_req,
                           void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                           void* staging, size_t staging_bytes, int32_t layers_per_chunk,
                           void* workspace, size_t workspace_bytes, void* stream,
                           const CopyFn& copy_item) {
  if (layers_per_chunk < 1)
    return set_last_error(HCR_ERR_INVALID_ARG, "layers_per_chunk must be >= 1");
  const int32_t n_layers = layer_end - layer_begin;
  const int32_t chunk = std::min(layers_per_chunk, n_layers);
  std::vector<Item> items;
  for (int32_t l0 = 0; l0 < n_layers; l0 += chunk)
    items.push_back({false, l0, std::min(chunk, n_layers - l0)});
  const size_t slot_bytes = size_t(chunk) * size_t(n_tokens) * size_t(h->impl.dims.d_model) * 2;
  return run_pipeline(h, items, slot_bytes, layer_begin, n_req, n_tokens, cu_seqlens, start_pos,
                      block_table, max_blocks_per_req, k_cache, v_cache, layout, staging,
                      staging_bytes, workspace_min_bytes(h, n_tokens, chunk), workspace,
                      workspace_bytes, stream, copy_item);
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
  const uint8_t* src = static_cast<const uint8_t*>(hidden_host);
  const size_t layer_bytes = size_t(n_tokens) * size_t(d.d_model) * 2;
  return hidden_pipeline(
      h, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos, block_table,
      max_blocks_per_req, k_cache, v_cache, layout, staging, staging_bytes, layers_per_chunk,
      workspace, workspace_bytes, stream, [&](const Item& it, void* dst, cudaStream_t copy) {
        return copy_status(cudaMemcpyAsync(dst, src + size_t(it.l0) * layer_bytes,
                                           size_t(it.nl) * layer_bytes, cudaMemcpyHostToDevice,
                                           copy));
      });
}

extern "C" hcr_status hcr_restore_streamed_chunks(
    hcr_handle* h, const hcr_chunk_source* source, int32_t layer_begin, int32_t layer_end,
    int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens, const int32_t* start_pos,
    const int32_t* block_table, int32_t max_blocks_per_req, void* k_cache, void* v_cache,
    const hcr_cache_layout* layout, void* staging, size_t staging_bytes,
    int32_t layers_per_chunk, void* workspace, size_t workspace_bytes, void* stream) {
  if (!h) return set_last_error(HCR_ERR_INVALID_ARG, "handle is NULL");
  const hcr_model_dims& d = h->impl.dims;
  if (layer_begin < 0 || layer_end < layer_begin || layer_end > d.n_layers)
    return set_last_error(HCR_ERR_INVALID_ARG, "layer range [%d, %d) outside [0, %d)",
                          layer_begin, layer_end, d.n_layers);
  if (n_tokens < 0 || n_req < 0)
    return set_last_error(HCR_ERR_INVALID_ARG, "n_tokens and n_req must be >= 0");
  if (n_tokens == 0 || layer_end == layer_begin) return HCR_OK;
  if (!source || !source->store || !source->chunk_table || !source->cu_seqlens ||
      !source->start_pos)
    return set_last_error(HCR_ERR_INVALID_ARG, "source and its host arrays must be non-NULL");
  const hcr_chunk_source& src = *source;
  if (src.chunk_tokens < 1 || src.num_chunks < 1 || src.max_chunks < 1)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "chunk_tokens, num_chunks and max_chunks must be >= 1");
  if (src.cu_seqlens[0] != 0 || src.cu_seqlens[n_req] != n_tokens)
    return set_last_error(HCR_ERR_INVALID_ARG, "host cu_seqlens must run from 0 to n_tokens");

  // Plan the gathers once.  A run is one request's tokens inside one chunk;
  // its rows for nl consecutive layers sit C*d elements apart in the chunk and
  // n_tokens*d apart in the staging slot, so one 2-D copy moves them all.  A
  // span is a run of whole chunks with consecutive ids: for one layer its
  // chunks sit n_layers*C*d apart in the store and land C*d apart, so one 2-D
  // copy per layer moves the whole span -- fewer copies when the span holds
  // more chunks than the group has layers.
  struct Run {
    size_t src_off;     // bytes into the store: (first chunk, layer_begin, first row)
    size_t dst_off;     // bytes into a staging slot: (layer 0, first token)
    size_t width;       // bytes per chunk: rows x d_model x 2
    int64_t n_chunks;   // whole consecutive chunks in a span; 0 for a partial run
  };
  std::vector<Run> runs;
  const int64_t C = src.chunk_tokens;
  const size_t row_bytes = size_t(d.d_model) * 2;
  const size_t chunk_stride = size_t(d.n_layers) * size_t(C) * row_bytes;   // next chunk id
  int32_t prev_cid = -1;
  for (int32_t r = 0; r < n_req; ++r) {
    const int32_t a = src.cu_seqlens[r], b = src.cu_seqlens[r + 1];
    if (b < a) return set_last_error(HCR_ERR_INVALID_ARG, "host cu_seqlens must not decrease");
    const int64_t p0 = src.start_pos[r];
    if (p0 < 0) return set_last_error(HCR_ERR_INVALID_ARG, "request %d: negative start", r);
    bool span_open = false;
    for (int64_t p = p0; p < p0 + (b - a);) {
      const int64_t k = p / C, off = p % C;
      const int64_t rows = std::min<int64_t>(C - off, p0 + (b - a) - p);
      if (k >= src.max_chunks)
        return set_last_error(HCR_ERR_INVALID_ARG, "request %d: position %lld has no chunk", r,
                              (long long)p);
      const int32_t cid = src.chunk_table[int64_t(r) * src.max_chunks + k];
      if (cid < 0 || cid >= src.num_chunks)
        return set_last_error(HCR_ERR_INVALID_ARG, "request %d: chunk id %d out of range", r,
                              cid);
      const int64_t t = a + (p - p0);
      const bool whole = rows == C;
      if (whole && span_open && cid == prev_cid + 1) {
        ++runs.back().n_chunks;
      } else {
        runs.push_back({((size_t(cid) * d.n_layers + layer_begin) * C + off) * row_bytes,
                        size_t(t) * row_bytes, size_t(rows) * row_bytes, whole ? 1 : 0});
      }
      span_open = whole;
      prev_cid = cid;
      p += rows;
    }
  }
  const uint8_t* store = static_cast<const uint8_t*>(src.store);
  const size_t layer_in_chunk = size_t(C) * row_bytes;       // next layer inside a chunk
  const size_t layer_in_slot = size_t(n_tokens) * row_bytes;  // next layer in the slot
  return hidden_pipeline(
      h, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, start_pos, block_table,
      max_blocks_per_req, k_cache, v_cache, layout, staging, staging_bytes, layers_per_chunk,
      workspace, workspace_bytes, stream, [&](const Item& it, void* dst, cudaStream_t copy) {
        const int32_t l0 = it.l0, nl = it.nl;
        uint8_t* slot = static_cast<uint8_t*>(dst);
        cudaError_t e = cudaSuccess;
        for (const Run& run : runs) {
          const uint8_t* base = store + run.src_off + size_t(l0) * layer_in_chunk;
          if (run.n_chunks > nl) {
            for (int32_t l = 0; l < nl && e == cudaSuccess; ++l)
              e = cudaMemcpy2DAsync(slot + size_t(l) * layer_in_slot + run.dst_off,
                                    layer_in_chunk, base + size_t(l) * layer_in_chunk,
                                    chunk_stride, run.width, size_t(run.n_chunks),
                                    cudaMemcpyHostToDevice, copy);
          } else {
            for (int64_t j = 0; j < std::max<int64_t>(run.n_chunks, 1) && e == cudaSuccess; ++j)
              e = cudaMemcpy2DAsync(slot + run.dst_off + size_t(j) * layer_in_chunk,
                                    layer_in_slot, base + size_t(j) * chunk_stride,
                                    layer_in_chunk, run.width, size_t(nl),
                                    cudaMemcpyHostToDevice, copy);
          }
          if (e != cudaSuccess) return copy_status(e);
        }
        return HCR_OK;
      });
}

extern "C" hcr_status hcr_restore_streamed_split(
    hcr_handle* h, const void* hidden_host, const void* kv_host, int32_t layer_begin,
    int32_t split_layer, int32_t layer_end, int32_t n_req, int32_t n_tokens,
    const int32_t* cu_seqlens, const int32_t* start_pos, const int32_t* block_table,
    int32_t max_blocks_per_req, void* k_cache, void* v_cache, const hcr_cache_layout* layout,
    void* staging, size_t staging_bytes, int32_t layers_per_chunk, void* workspace,
    size_t workspace_bytes, void* stream) {
  if (!h) return set_last_error(HCR_ERR_INVALID_ARG, "handle is NULL");
  const hcr_model_dims& d = h->impl.dims;
  if (layer_begin < 0 || split_layer < layer_begin || layer_end < split_layer ||
      layer_end > d.n_layers)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "need 0 <= layer_begin <= split_layer <= layer_end <= %d, got %d, %d, %d",
                          d.n_layers, layer_begin, split_layer, layer_end);
  if (n_tokens < 0) return set_last_error(HCR_ERR_INVALID_ARG, "n_tokens must be >= 0");
  if (n_tokens == 0 || layer_end == layer_begin) return HCR_OK;
  if (layers_per_chunk < 1)
    return set_last_error(HCR_ERR_INVALID_ARG, "layers_per_chunk must be >= 1");
  const int32_t n_hid = split_layer - layer_begin, n_kv = layer_end - split_layer;
  if ((n_hid > 0 && !hidden_host) || (n_kv > 0 && !kv_host))
    return set_last_error(HCR_ERR_INVALID_ARG, "hidden_host/kv_host is NULL");
  const size_t hid_layer = size_t(n_tokens) * size_t(d.d_model) * 2;
  const size_t kv_layer = size_t(n_tokens) * 2 * size_t(d.n_kv_heads) * d.head_dim * 2;
  // A slot holds one hidden-state group, or as many whole K/V layers as fit
  // (at least one).
  const int32_t ch = std::min(layers_per_chunk, n_hid);
  const size_t slot_bytes = std::max(size_t(ch) * hid_layer, n_kv > 0 ? kv_layer : size_t(0));
  const int32_t ck = n_kv > 0 ? int32_t(std::min<size_t>(size_t(n_kv), slot_bytes / kv_layer)) : 0;
  std::vector<Item> hid_items, kv_items, items;
  for (int32_t l0 = 0; l0 < n_hid; l0 += ch) hid_items.push_back({false, l0, std::min(ch, n_hid - l0)});
  for (int32_t l0 = 0; l0 < n_kv; l0 += ck)
    kv_items.push_back({true, n_hid + l0, std::min(ck, n_kv - l0)});
  // Spread the K/V groups evenly among the hidden-state groups so both the
  // copy stream and the compute stream stay busy: item i of a list of n sits
  // at (i + 1/2) / n, and the hidden-state group goes first on a tie.
  const size_t a = hid_items.size(), b = kv_items.size();
  for (size_t i = 0, j = 0; i < a || j < b;) {
    if (j == b || (i < a && (2 * i + 1) * b <= (2 * j + 1) * a))
      items.push_back(hid_items[i++]);
    else
      items.push_back(kv_items[j++]);
  }
  const uint8_t* hid = static_cast<const uint8_t*>(hidden_host);
  const uint8_t* kv = static_cast<const uint8_t*>(kv_host);
  return run_pipeline(
      h, items, slot_bytes, layer_begin, n_req, n_tokens, cu_seqlens, start_pos, block_table,
      max_blocks_per_req, k_cache, v_cache, layout, staging, staging_bytes,
      workspace_min_bytes(h, n_tokens, std::max(ch, 1)), workspace, workspace_bytes, stream,
      [&](const Item& it, void* dst, cudaStream_t copy) {
        if (it.kv)
          return copy_status(cudaMemcpyAsync(dst, kv + size_t(it.l0 - n_hid) * kv_layer,
                                             size_t(it.nl) * kv_layer, cudaMemcpyHostToDevice,
                                             copy));
        return copy_status(cudaMemcpyAsync(dst, hid + size_t(it.l0) * hid_layer,
                                           size_t(it.nl) * hid_layer, cudaMemcpyHostToDevice,
                                           copy));
      });
}

extern "C" hcr_status hcr_restore_streamed_encoded(
    hcr_handle* h, const hcr_codec_params* params, const void* codes_host,
    const void* scales_host, int32_t layer_begin, int32_t layer_end, int32_t n_req,
    int32_t n_tokens, const int32_t* cu_seqlens, const int32_t* start_pos,
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
  if (!params || !codes_host || !scales_host)
    return set_last_error(HCR_ERR_INVALID_ARG, "params, codes_host and scales_host are needed");
  bool empty = false;
  hcr_status st = check_codec(h, params, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                              &empty);
  if (st != HCR_OK || empty) return st;
  if (layers_per_chunk < 1)
    return set_last_error(HCR_ERR_INVALID_ARG, "layers_per_chunk must be >= 1");
  if (!staging || reinterpret_cast<uintptr_t>(staging) % 256)
    return set_last_error(HCR_ERR_WORKSPACE, "staging must be non-NULL and 256-byte aligned");
  const int32_t n_layers = layer_end - layer_begin;
  const int32_t chunk = std::min(layers_per_chunk, n_layers);
  const size_t T = size_t(n_tokens), dm = size_t(d.d_model);
  // a slot: [codes][scales][decoded hidden states], each 256-byte aligned
  const size_t codes_bytes = align_up(size_t(chunk) * T * dm, 256);
  const size_t scales_bytes = align_up(size_t(chunk) * T * 4, 256);
  const size_t slot_bytes = codes_bytes + scales_bytes + align_up(size_t(chunk) * T * dm * 2, 256);
  // The codes are half the hidden states' bytes, so a group's copy takes
  // about half as long as its restore: groups of 1, 2, 4 ... layers up to
  // `chunk` start the first restore early without the restores ever waiting
  // on a copy.
  std::vector<Item> items;
  for (int32_t l0 = 0, nl = 1; l0 < n_layers; l0 += nl, nl = std::min(2 * nl, chunk))
    items.push_back({false, l0, std::min(nl, n_layers - l0)});
  const uint8_t* codes = static_cast<const uint8_t*>(codes_host);
  const uint8_t* scales = static_cast<const uint8_t*>(scales_host);
  // The decode runs on the side stream once the group's codes have landed, so
  // the copies of the next groups go on meanwhile; the restore reads the
  // slot's decoded part.
  const SideFn decode = [&](const Item& it, void* dst, cudaStream_t side) {
    uint8_t* slot = static_cast<uint8_t*>(dst);
    const int32_t lb = layer_begin + it.l0;
    return hcr_decode_hidden(h, params, slot, slot + codes_bytes, lb, lb + it.nl, n_req,
                             n_tokens, cu_seqlens, slot + codes_bytes + scales_bytes, side);
  };
  return run_pipeline(
      h, items, slot_bytes, layer_begin, n_req, n_tokens, cu_seqlens, start_pos, block_table,
      max_blocks_per_req, k_cache, v_cache, layout, staging, staging_bytes,
      workspace_min_bytes(h, n_tokens, chunk), workspace, workspace_bytes, stream,
      [&](const Item& it, void* dst, cudaStream_t copy) {
        uint8_t* slot = static_cast<uint8_t*>(dst);
        cudaError_t e = cudaMemcpyAsync(slot, codes + size_t(it.l0) * T * dm,
                                        size_t(it.nl) * T * dm, cudaMemcpyHostToDevice, copy);
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(slot + codes_bytes, scales + size_t(it.l0) * T * 4,
                              size_t(it.nl) * T * 4, cudaMemcpyHostToDevice, copy);
        return copy_status(e);
      },
      &decode, codes_bytes + scales_bytes);
}
