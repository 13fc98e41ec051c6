// Host-side declarations shared by the library's entry points: the handle,
// error recording, NVTX ranges, and launchers of the kernels outside the
// restore itself.  Not part of the public ABI.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include "hcr_internal.h"

namespace hcr {

constexpr int kMaxStagingSlots = 8;    // staging ring of the layer-pipelined restore

struct StreamedRes;  // copy stream + events of hcr_restore_streamed (hcr_streamed.cu)

// ---------------------------------------------------------------------------
// Handle
// ---------------------------------------------------------------------------
struct Handle {
  hcr_model_dims dims;
  int device = 0;
  int num_sms = 0;
  void* w_packed = nullptr;    // [L][2*d_kv][d] storage dtype, gamma folded in
  float* col_sum = nullptr;    // [L][2*d_kv] sum_i W'[j][i] (LayerNorm only)
  float* col_bias = nullptr;   // [L][2*d_kv] folded bias (LN: W beta + b; RMS: b), or null
  float2* rope_tab = nullptr;  // [max_position][head_dim/2] (cos, sin), or null
  uint32_t* err = nullptr;     // device error word (HCR_DEVERR_* bits)
  CUtensorMap tmap_w;          // 3-D map over w_packed: (d, 2*d_kv, L), box (64, 256, 1)
  CUtensorMap tmap_w_half;     // same tensor, box (64, 128, 1): half a tile per CTA of a pair
  int pair_clusters = 0;       // co-resident CTA pairs of the pair variant (0: unavailable)
  // Weight-row tiles (head_dim 128 only): 5-D view of w_packed, dims (d, 8, 2,
  // 8, L * 2 * n_kv_heads) with row strides (1, 64, 8, 128), box (64, 8, 2, 8, 1)
  CUtensorMap tmap_w5;
  int swap_clusters = 0;       // co-resident CTA pairs of that kernel (0: unavailable)
  int enc_clusters = 0;        // co-resident CTA pairs decoding the codec's form (0: unavailable)
  uint32_t debug_stall = 0;    // test hook: see hcr_debug_set_stall
  int32_t variant = 0;         // test hook: 0 auto, 1 single CTAs, 2 CTA pairs, 3/4 weight rows
  StreamedRes* streamed = nullptr;  // created on the first hcr_restore_streamed call
};

void release_streamed(Handle& H);

// Records a message for hcr_last_error() on this host thread; returns s.
hcr_status set_last_error(hcr_status s, const char* fmt, ...);

// An NVTX range on the calling host thread for the scope's lifetime: the
// library's entry points and stages show up by name in a timeline profiler
// (nothing is recorded when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Rows of K and V between the paged cache and a dense [layer][K|V][token][row]
// store (hcr_kv.cu).  Pointers to host memory are the device's mapped view.
struct KvRowsParams {
  const int64_t* slot;     // [T] from the prepare kernel; -1 rows are skipped
  uint4* dense;            // [n_layers][2][T][row_vecs]
  void* k_cache;           // base of the first layer
  void* v_cache;
  int64_t layer_stride_vecs;
  int32_t row_vecs;        // n_kv_heads * head_dim / 8
  int32_t n_tokens, n_layers;
};

cudaError_t launch_kv_rows(const KvRowsParams& p, bool to_cache, int num_sms, cudaStream_t s);
// The device address of caller memory that may live on the host (mapped pinned
// memory, or pageable memory when the device can reach it); an error status
// names `what` when the device cannot address it.
hcr_status device_view(const Handle& H, void* ptr, const char* what, void** out);

// The smallest workspace a restore of n_tokens tokens over n_layers layers
// accepts (hcr_workspace_bytes adds the fused statistics' flags to it).
size_t workspace_min_bytes(const hcr_handle* h, int32_t n_tokens, int32_t n_layers);

// Pieces of hcr_restore for the layer-pipelined restores (hcr_streamed.cu);
// arguments as in hcr_restore.
//   pipeline_placement: checks a whole call's arguments (`staging` stands for
//     the hidden rows) and, when the workspace also holds statistics for
//     stats_layers layers (*ok), enqueues the slot map on `stream`.
//   pipeline_stats: the norm statistics of hidden rows [layer_begin,
//     layer_end) into rstd / mean ([layer][token]) on `stream` (the slot map
//     is not touched).
//   pipeline_project: the projection of those rows with the given statistics
//     and the slot map already in the workspace.
hcr_status pipeline_placement(hcr_handle* h, const void* staging, int32_t layer_begin,
                              int32_t layer_end, int32_t n_req, int32_t n_tokens,
                              const int32_t* cu_seqlens, const int32_t* start_pos,
                              const int32_t* block_table, int32_t max_blocks_per_req,
                              void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                              void* workspace, size_t workspace_bytes, int32_t stats_layers,
                              void* stream, bool* ok);
hcr_status pipeline_stats(hcr_handle* h, const void* hidden, int32_t layer_begin,
                          int32_t layer_end, int32_t n_req, int32_t n_tokens,
                          const int32_t* cu_seqlens, const int32_t* start_pos,
                          const int32_t* block_table, int32_t max_blocks_per_req,
                          void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                          void* workspace, size_t workspace_bytes, float* rstd, float* mean,
                          void* stream);
hcr_status pipeline_project(hcr_handle* h, const void* hidden, int32_t layer_begin,
                            int32_t layer_end, int32_t n_req, int32_t n_tokens,
                            const int32_t* cu_seqlens, const int32_t* start_pos,
                            const int32_t* block_table, int32_t max_blocks_per_req,
                            void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                            void* workspace, size_t workspace_bytes, const float* rstd,
                            const float* mean, void* stream);

// Host checks of a codec call (hcr_encode_hidden / hcr_decode_hidden); sets
// *empty for a call with no work.
hcr_status check_codec(const hcr_handle* h, const hcr_codec_params* cp, int32_t layer_begin,
                       int32_t layer_end, int32_t n_req, int32_t n_tokens,
                       const int32_t* cu_seqlens, bool* empty);

}  // namespace hcr

struct hcr_handle {
  hcr::Handle impl;
};
