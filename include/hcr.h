/*
 * hcr.h -- restore an attention KV cache from saved per-layer hidden states.
 *
 * The operation (HCache episode, "Fast State Restoration for Evicted LLM KV
 * Caches", cue 14): instead of keeping an evicted request's K and V, keep
 * each layer's input hidden state H (cue 3: the layer input, the embedding
 * output for the first layer) and rebuild the cache by running only the
 * key/value projections, K = W_k H and V = W_v H; attention and the FFN are
 * skipped.  A restore reads every token of one layer together (cue 16) and
 * many requests' tokens are projected together so the GEMM shape stays
 * regular (cue 20).
 *
 * This library adds what a pre-norm transformer needs around that
 * projection: the layer's input norm (RMSNorm with gamma, or LayerNorm with
 * gamma/beta), optional K/V biases, rotate-half RoPE on K at each token's
 * absolute position, and a paged cache addressed through a block table.
 *
 * For each layer l in [layer_begin, layer_end) and each restored token t of
 * request r at position p:
 *     x      = norm_l(H_l[t])                         (RMSNorm or LayerNorm)
 *     k      = x W_k[l]^T (+ b_k[l]),   v = x W_v[l]^T (+ b_v[l])
 *     k      = RoPE(k, p)  per head: pairs (i, i+dh/2) turn by p*theta^(-2i/dh)
 *     slot   = block_table[r][p / B] * B + p % B
 *     k_cache[l][slot] = k,   v_cache[l][slot] = v      (rounded to nearest even)
 *
 * Numbers: inputs and outputs are bf16 or fp16 (one type per handle); the
 * projection accumulates in fp32 on the tensor cores; norm statistics, bias,
 * RoPE and the cast run in fp32.  gamma is folded into the packed weights
 * (W' = [W_k; W_v] diag(gamma), rounded once to the storage type), so the
 * norm is applied as a per-row scale after the GEMM.
 *
 * Threading and streams: a handle is immutable after hcr_create (apart from
 * the hcr_debug_* testing hooks) and may be used from several host threads
 * and streams at once, provided each concurrent restore has its own
 * workspace.  The handle's device error word is shared: bits raised by any
 * of its restores are reported (and cleared) by the next
 * hcr_check_device_error.  Every call that takes a stream only enqueues work
 * on it; it does not synchronise unless stated.
 *
 * All entry points return hcr_status.  Host-side argument errors are
 * reported before any work is enqueued, and hcr_last_error() then returns a
 * message naming the offending argument.
 */
#ifndef HCR_H_
#define HCR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HCR_OK = 0,
  HCR_ERR_INVALID_ARG = 1,   /* a host argument is null, out of range or inconsistent      */
  HCR_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim not 64/128/256)   */
  HCR_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (no device, launch, ...) */
  HCR_ERR_OOM = 4,           /* device allocation inside hcr_create failed                  */
  HCR_ERR_WORKSPACE = 5,     /* workspace pointer null/misaligned or smaller than needed    */
  HCR_ERR_DEVICE_BOUNDS = 6, /* (device) a block id, logical block or position was out of
                                range; the affected rows were skipped, nothing else written */
  HCR_ERR_TIMEOUT = 7        /* (device) a pipeline wait exceeded its time limit; the kernel
                                stopped early and released its resources                   */
} hcr_status;

enum { HCR_NORM_RMS = 0, HCR_NORM_LAYER = 1 };
enum { HCR_ROPE_NONE = 0, HCR_ROPE_ROTATE_HALF = 1 };
enum { HCR_DTYPE_BF16 = 0, HCR_DTYPE_FP16 = 1 };

/* Device error bits accumulated by the kernels (see hcr_check_device_error). */
enum {
  HCR_DEVERR_BLOCK_ID = 1u << 0,     /* block_table entry < 0 or >= num_blocks           */
  HCR_DEVERR_LOGICAL_BLOCK = 1u << 1,/* position / B >= max_blocks_per_req               */
  HCR_DEVERR_POSITION = 1u << 2,     /* start_pos < 0, or position >= max_position (RoPE) */
  HCR_DEVERR_SEQLENS = 1u << 3,      /* cu_seqlens not non-decreasing from 0 to n_tokens */
  HCR_DEVERR_TIMEOUT = 1u << 4       /* a bounded pipeline wait gave up                  */
};

/* Model dimensions, fixed at hcr_create. */
typedef struct {
  int32_t n_layers;      /* layers whose parameters the handle holds                       */
  int32_t d_model;       /* width of the hidden state; multiple of 8                       */
  int32_t n_heads;       /* query heads (only checked: multiple of n_kv_heads)             */
  int32_t n_kv_heads;    /* key/value heads; n_kv_heads < n_heads is grouped-query attn.   */
  int32_t head_dim;      /* 64, 128 or 256                                                 */
  int32_t norm;          /* HCR_NORM_RMS or HCR_NORM_LAYER                                 */
  float norm_eps;        /* added to the mean square (RMS) or variance (LN) inside the sqrt */
  int32_t rope;          /* HCR_ROPE_NONE or HCR_ROPE_ROTATE_HALF                          */
  float rope_theta;      /* RoPE base, e.g. 10000                                          */
  int32_t max_position;  /* RoPE positions supported: 0 .. max_position-1 (table size)     */
  int32_t dtype;         /* HCR_DTYPE_BF16 or HCR_DTYPE_FP16: weights, hidden and cache    */
  int32_t has_kv_bias;   /* nonzero: b_k and b_v are given                                 */
} hcr_model_dims;

/* Paged cache geometry.  k_cache and v_cache are each laid out as
 *   [layer][num_blocks][block_size][n_kv_heads][head_dim]
 * with layer_stride_elems elements between consecutive layers (0 means the
 * dense stride num_blocks*block_size*n_kv_heads*head_dim). */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int64_t layer_stride_elems;
} hcr_cache_layout;

typedef struct hcr_handle hcr_handle;

/*
 * hcr_create -- pack one model's restore parameters on the current device.
 *
 * gamma, w_k, w_v: host arrays of n_layers DEVICE pointers, in the dims'
 * dtype: gamma[l] [d_model]; w_k[l], w_v[l] [n_kv_heads*head_dim][d_model]
 * row-major (PyTorch Linear layout, K = X W_k^T).  beta: same, [d_model],
 * required for HCR_NORM_LAYER, must be NULL for RMS.  b_k, b_v: [n_kv*dh],
 * required iff has_kv_bias, else NULL.
 *
 * The caller keeps ownership of its parameters and may free them once this
 * returns; the handle owns packed copies: W' = [W_k; W_v] diag(gamma) in the
 * storage dtype, per-column fp32 constants (LayerNorm column sums and the
 * folded bias W beta + b), an fp32 RoPE cos/sin table built in fp64 on the
 * host, and a device error word.  Synchronises the device before returning.
 * Errors: HCR_ERR_INVALID_ARG, HCR_ERR_UNSUPPORTED, HCR_ERR_CUDA, HCR_ERR_OOM;
 * *out is set to NULL on error.
 */
hcr_status hcr_create(const hcr_model_dims* dims, const void* const* gamma,
                      const void* const* beta, const void* const* w_k,
                      const void* const* w_v, const void* const* b_k,
                      const void* const* b_v, hcr_handle** out);

/* Releases everything the handle owns.  Synchronises the device.  NULL is a no-op. */
void hcr_destroy(hcr_handle* h);

/*
 * hcr_workspace_bytes -- device scratch for a restore of n_tokens tokens over
 * n_layers_in_range layers: per-token slot and position, per-row norm
 * statistics, and one int32 flag per 16 tokens and layer.  With the flags'
 * room the projection computes most layers' norm statistics itself
 * (hcr_debug_fused_stats); a restore also accepts the smaller workspace
 * without them (this size minus the flags, rounded to 256 bytes) and then
 * computes every layer's statistics in its prepare kernel.  Returns 0 for
 * invalid arguments or an empty restore.
 */
size_t hcr_workspace_bytes(const hcr_handle* h, int32_t n_tokens, int32_t n_layers_in_range);

/*
 * hcr_restore -- restore layers [layer_begin, layer_end) of n_req requests.
 *
 * hidden:      DEVICE [layer_end-layer_begin][n_tokens][d_model], dtype of the
 *              handle, 16-byte aligned.  Row t is the t-th token of the
 *              requests concatenated in order (HCache episode, cue 16: one
 *              layer's tokens are read together).
 * n_req, n_tokens: host values; n_tokens must equal cu_seqlens[n_req].
 * cu_seqlens:  DEVICE int32 [n_req+1], cu_seqlens[0] = 0, non-decreasing;
 *              request r owns rows cu_seqlens[r] .. cu_seqlens[r+1]-1.
 * start_pos:   DEVICE int32 [n_req]; row cu_seqlens[r]+i sits at absolute
 *              position start_pos[r]+i.  Positions below start_pos[r] are a
 *              resident prefix and are never written.
 * block_table: DEVICE int32 [n_req][max_blocks_per_req]; entry [r][b] is the
 *              physical block holding positions b*B .. b*B+B-1 of request r.
 * k_cache, v_cache: DEVICE, base of layer layer_begin, laid out as
 *              hcr_cache_layout says, 16-byte aligned.  Only the slots of the
 *              restored positions are written; every other byte is untouched.
 * workspace:   DEVICE, >= hcr_workspace_bytes(h, n_tokens, layers), 256-byte
 *              aligned, owned by the caller, not shared with a concurrent call.
 * stream:      a cudaStream_t (NULL = legacy default stream).
 *
 * Enqueues two kernels (hcr_restore_prepare, then hcr_restore_project) and
 * returns.  n_tokens == 0 or an empty layer range enqueues nothing.
 * Distinct requests must not share physical blocks (the result is then
 * undefined).  Out-of-range block ids or positions found on the device skip
 * the affected rows and set error bits; read them with
 * hcr_check_device_error.
 */
hcr_status hcr_restore(hcr_handle* h, const void* hidden, int32_t layer_begin,
                       int32_t layer_end, int32_t n_req, int32_t n_tokens,
                       const int32_t* cu_seqlens, const int32_t* start_pos,
                       const int32_t* block_table, int32_t max_blocks_per_req,
                       void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * hcr_restore_prepare / hcr_restore_project -- the two stages of hcr_restore,
 * with identical arguments (workspace and workspace_bytes included).  prepare
 * maps every token to its (position, slot) and computes the (layer, token)
 * rows' norm statistics into the workspace; project runs the fused K||V GEMM
 * with the norm, bias, RoPE, cast and paged scatter in its epilogue, reading
 * that workspace.  When the call fuses the statistics (hcr_debug_fused_stats)
 * prepare computes only the first layers' and clears the flags, and project
 * computes the rest; both stages decide that from the same arguments, so they
 * must be the same.  Calling prepare then project on one stream with the same
 * arguments is exactly hcr_restore; splitting them lets a caller time or
 * overlap the stages.
 */
hcr_status hcr_restore_prepare(hcr_handle* h, const void* hidden, int32_t layer_begin,
                               int32_t layer_end, int32_t n_req, int32_t n_tokens,
                               const int32_t* cu_seqlens, const int32_t* start_pos,
                               const int32_t* block_table, int32_t max_blocks_per_req,
                               void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                               void* workspace, size_t workspace_bytes, void* stream);
hcr_status hcr_restore_project(hcr_handle* h, const void* hidden, int32_t layer_begin,
                               int32_t layer_end, int32_t n_req, int32_t n_tokens,
                               const int32_t* cu_seqlens, const int32_t* start_pos,
                               const int32_t* block_table, int32_t max_blocks_per_req,
                               void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * hcr_restore_streamed -- the layer-pipelined restore from host memory.
 *
 * The HCache episode (cue 15) overlaps the transfer of layer N+1's hidden
 * states with the projection of layer N.  This call does that for hidden
 * states held in host memory: it copies them to the device one chunk of
 * layers_per_chunk layers at a time, on a copy stream owned by the handle,
 * into a ring of chunk-sized slots carved from `staging`, and restores each
 * chunk on `stream` (exactly as hcr_restore would) as soon as its copy has
 * landed; a slot is refilled only after the restore that read it finished.
 *
 * hidden_host: HOST [layer_end-layer_begin][n_tokens][d_model]; pinned
 *              (page-locked) memory lets the copies overlap the restores.
 * staging:     DEVICE, 256-byte aligned, owned by the caller; its size
 *              decides the ring: min(8, staging_bytes / chunk bytes) slots,
 *              at least one (one slot restores correctly but serialises).
 * workspace:   as hcr_restore, sized for one chunk:
 *              hcr_workspace_bytes(h, n_tokens, layers_per_chunk).  Given
 *              statistics room for every slot's chunk,
 *              hcr_workspace_bytes(h, n_tokens, slots * layers_per_chunk),
 *              the slot map is computed once and each chunk's norm
 *              statistics on a second stream the handle owns as soon as
 *              the chunk lands, so `stream` runs only the projections; the
 *              caches are the same bits either way.  The same holds for
 *              hcr_restore_streamed_chunks, hcr_restore_streamed_split
 *              (hidden-state groups) and hcr_restore_streamed_encoded.
 * Every other argument is as in hcr_restore (k_cache and v_cache are the
 * base of layer layer_begin).  Returns after enqueueing; the restore is
 * complete when `stream` reaches this point.  Calls through one handle are
 * serialised on the host while they enqueue.
 */
hcr_status hcr_restore_streamed(hcr_handle* h, const void* hidden_host, int32_t layer_begin,
                                int32_t layer_end, int32_t n_req, int32_t n_tokens,
                                const int32_t* cu_seqlens, const int32_t* start_pos,
                                const int32_t* block_table, int32_t max_blocks_per_req,
                                void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                                void* staging, size_t staging_bytes, int32_t layers_per_chunk,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * hcr_save_hidden -- the save side: store layer inputs in fixed-size chunks.
 *
 * HCache episode, cue 16: generation produces hidden states layer before
 * token (each decode step yields every layer's input for its new token),
 * while a restore reads all tokens of one layer together; cue 22: they are
 * kept in fixed 64-token chunks.  A chunk holds positions [C*k, C*k + C) of
 * one request (logical chunk k = position / C) for ALL layers, laid out
 *     chunk_store[id][layer][position % C][d_model]
 * so inside a chunk each layer's tokens are contiguous (token before layer).
 *
 * hidden:       DEVICE [layer_end-layer_begin][n_tokens][d_model], 16-byte
 *               aligned: row t of layer layer_begin+i.  A decode step is one
 *               token per request; a prefill saves a whole prompt.
 * n_req, n_tokens, cu_seqlens, start_pos: as in hcr_restore.
 * chunk_table:  DEVICE int32 [n_req][max_chunks_per_req]; entry [r][k] is the
 *               physical chunk of request r's positions [C*k, C*k + C).
 * chunk_tokens: C, tokens per chunk (64 on the page).
 * chunk_store:  [num_chunks][n_layers][C][d_model] in the handle's dtype,
 *               16-byte aligned; device memory, or pinned (mapped) host
 *               memory -- the stores then cross the host link directly,
 *               with no separate snapshot copy.  Host memory the device
 *               cannot address is rejected with HCR_ERR_INVALID_ARG.
 * Only the slots of the given rows are written.  Rows whose chunk id or
 * logical chunk is out of range are skipped and flagged
 * (HCR_DEVERR_BLOCK_ID / HCR_DEVERR_LOGICAL_BLOCK; read them with
 * hcr_check_device_error).  Enqueues one kernel on `stream`.
 */
hcr_status hcr_save_hidden(hcr_handle* h, const void* hidden, int32_t layer_begin,
                           int32_t layer_end, int32_t n_req, int32_t n_tokens,
                           const int32_t* cu_seqlens, const int32_t* start_pos,
                           const int32_t* chunk_table, int32_t max_chunks_per_req,
                           int32_t chunk_tokens, void* chunk_store, int32_t num_chunks,
                           void* stream);

/*
 * hcr_restore_streamed_chunks -- hcr_restore_streamed from a host store of
 * fixed-size chunks, in the layout hcr_save_hidden writes:
 *     store[chunk][layer][row][d_model],  chunk = chunk_table[r][pos / C],
 *     row = pos % C.
 * This is the restore half of the HCache episode's storage scheme (cue 22:
 * 64-token chunks).  The copy engines gather each request's rows straight
 * from the chunks into the staging ring with 2-D copies (one per run of a
 * request's tokens inside one chunk, per chunk of layers), so no host-side
 * transpose is needed.  The host needs the request layout to plan those
 * copies, so it is given in host memory here (the device copies in the
 * argument list are still used by the kernels).  Every other argument and
 * all behaviour are as in hcr_restore_streamed.  Host-side checks reject a
 * position without a chunk or a chunk id outside [0, num_chunks).
 */
typedef struct {
  const void* store;           /* HOST (pinned) [num_chunks][n_layers][chunk_tokens][d_model] */
  int32_t chunk_tokens;        /* C: tokens per chunk (64 on the page)                         */
  int32_t num_chunks;
  const int32_t* chunk_table;  /* HOST [n_req][max_chunks]                                     */
  int32_t max_chunks;
  const int32_t* cu_seqlens;   /* HOST [n_req+1], same values as the device copy              */
  const int32_t* start_pos;    /* HOST [n_req], same values as the device copy                */
} hcr_chunk_source;

hcr_status hcr_restore_streamed_chunks(hcr_handle* h, const hcr_chunk_source* source,
                                       int32_t layer_begin, int32_t layer_end, int32_t n_req,
                                       int32_t n_tokens, const int32_t* cu_seqlens,
                                       const int32_t* start_pos, const int32_t* block_table,
                                       int32_t max_blocks_per_req, void* k_cache,
                                       void* v_cache, const hcr_cache_layout* layout,
                                       void* staging, size_t staging_bytes,
                                       int32_t layers_per_chunk, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * hcr_save_kv / hcr_load_kv -- the KV-offload side of a layer-split restore
 * (HCache episode, cue 18: layers not restored from hidden states are handed
 * to a complementary method; the one provided here is KV offload).
 *
 * A dense K/V store holds, for layers [layer_begin, layer_end) and the
 * n_tokens tokens of the request layout (cu_seqlens order):
 *     kv[layer - layer_begin][0][t][:] = K row of token t (position-embedded)
 *     kv[layer - layer_begin][1][t][:] = V row of token t
 * each row n_kv_heads * head_dim elements of the storage dtype.
 * hcr_save_kv copies those rows out of the paged cache (e.g. when a
 * request's cache is evicted); hcr_load_kv places them back, at the slots the
 * block table gives -- the same placement hcr_restore uses.  `kv` may be
 * device memory or pinned (mapped) host memory; it must be 16-byte aligned.
 * Other arguments are as in hcr_restore; the workspace needs
 * hcr_workspace_bytes(h, n_tokens, 1) bytes (only the slot map is built).
 * Rows whose placement is invalid are skipped and flagged as in hcr_restore.
 * Each call enqueues two kernels on `stream`.
 */
hcr_status hcr_load_kv(hcr_handle* h, const void* kv, int32_t layer_begin, int32_t layer_end,
                       int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                       const int32_t* start_pos, const int32_t* block_table,
                       int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                       const hcr_cache_layout* layout, void* workspace, size_t workspace_bytes,
                       void* stream);
hcr_status hcr_save_kv(hcr_handle* h, void* kv, int32_t layer_begin, int32_t layer_end,
                       int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                       const int32_t* start_pos, const int32_t* block_table,
                       int32_t max_blocks_per_req, const void* k_cache, const void* v_cache,
                       const hcr_cache_layout* layout, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * The bubble-free layer split (HCache episode, cue 18; cue 20 on splitting by
 * layer rather than by token).  A restore of L layers pipelines host-to-device
 * transfer against GPU work; whichever is slower sets the pace.  Restoring a
 * layer from hidden states costs hidden_copy_s of transfer and restore_s of
 * GPU time; loading it as saved K/V costs kv_copy_s and kv_place_s.
 * hcr_plan_layer_split returns the split with the smallest
 *     max(transfer, compute),  transfer = (L-k)*hidden_copy_s + k*kv_copy_s,
 *                              compute  = (L-k)*restore_s     + k*kv_place_s
 * over k = 0..L layers loaded as K/V (ties: the smaller k).  Host-only; all
 * costs in seconds per layer, finite and >= 0.
 *
 * hcr_profile_layer_costs measures the four costs on the current GPU for
 * n_tokens tokens, restoring groups of layers_per_chunk layers as the
 * streamed restore does, with CUDA events on `stream`.  The GPU costs come
 * from restores and placements run back to back -- half a second of warm-up
 * (at least `reps` rounds), then the mean of `reps` rounds -- so they are
 * those of a GPU under sustained load (a power-capped GPU clocks down under
 * sustained tensor work); the copy costs from `reps` copies of each kind.  It allocates device and pinned host buffers
 * for one group (freed before it returns) and synchronises `stream`.
 */
typedef struct {
  double restore_s;       /* GPU time to restore one layer from hidden states  */
  double hidden_copy_s;   /* host-to-device time for one layer's hidden states */
  double kv_copy_s;       /* host-to-device time for one layer's K and V       */
  double kv_place_s;      /* GPU time to place one layer's K and V             */
} hcr_layer_costs;

typedef struct {
  int32_t hidden_layers;  /* restored from hidden states (the first group) */
  int32_t kv_layers;      /* loaded as saved K and V (the last group)     */
  double transfer_s, compute_s, predicted_s;   /* predicted = max of the two */
} hcr_layer_split;

hcr_status hcr_plan_layer_split(const hcr_layer_costs* costs, int32_t n_layers,
                                hcr_layer_split* out);
hcr_status hcr_profile_layer_costs(hcr_handle* h, int32_t n_tokens, int32_t layers_per_chunk,
                                   int32_t reps, void* stream, hcr_layer_costs* out);

/*
 * hcr_restore_streamed_split -- the layer-split restore from host memory.
 * Layers [layer_begin, split_layer) are restored from hidden states
 *     hidden_host: HOST (pinned) [split_layer - layer_begin][n_tokens][d_model]
 * and layers [split_layer, layer_end) are placed from saved K/V
 *     kv_host:     HOST (pinned) [layer_end - split_layer][2][n_tokens][d_kv]
 * (the hcr_load_kv layout).  Both go through the staging ring of
 * hcr_restore_streamed on the handle's copy stream: one slot holds a group of
 * layers_per_chunk hidden-state layers, or as many K/V layers as fit (at
 * least one; the slot size is the larger of the two).  The K/V groups are
 * spread evenly among the hidden-state groups so that transfer and compute
 * overlap throughout.  The caches are bit-identical to hcr_restore over the
 * hidden-state layers and to hcr_load_kv over the K/V layers.  The workspace
 * needs hcr_workspace_bytes(h, n_tokens, min(layers_per_chunk, hidden
 * layers)) bytes (at least one layer's).  Other arguments are as in
 * hcr_restore_streamed; split_layer = layer_end is a plain streamed restore.
 */
hcr_status hcr_restore_streamed_split(hcr_handle* h, const void* hidden_host,
                                      const void* kv_host, int32_t layer_begin,
                                      int32_t split_layer, int32_t layer_end, int32_t n_req,
                                      int32_t n_tokens, const int32_t* cu_seqlens,
                                      const int32_t* start_pos, const int32_t* block_table,
                                      int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                                      const hcr_cache_layout* layout, void* staging,
                                      size_t staging_bytes, int32_t layers_per_chunk,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Hidden-state codec (HCache episode, cues 30 and 32: quantise hidden states
 * the way CacheGen quantises KV; CacheGen review, section 核心方法: groups of
 * 10 tokens with an 8-bit anchor and deltas from it, quantised with bins of
 * 0.5 / 1 / 1.5 for the first / middle / last third of the layers).  The
 * page's lossless arithmetic-coding stage is not part of this library.
 *
 *   groups:  token i of a request belongs to the group whose anchor is token
 *            group_tokens * (i / group_tokens) of the same request;
 *   anchor:  s = max|h| / 127 (float32), q = rint(h * (1 / s)) in
 *            [-127, 127]; s = 0 and all codes 0 when s < 2^-126; decoded q * s;
 *   others:  c = rint((h - q s) * (1 / b)) in [-127, 127]; decoded q s + c b,
 *            with b = bins[min(2, 3 l / n_layers)] for model layer l;
 *   1 / s and 1 / b are single binary32 divisions;
 *   every step one IEEE binary32 operation rounded to nearest even; the
 *   decoded value rounded once to the storage dtype.
 *
 * Encoded form: codes int8 [layer_end - layer_begin][n_tokens][d_model] and
 * scales float32 [layer_end - layer_begin][n_tokens] (anchor rows only; other
 * entries are not written).  Codes and scales may be device memory or pinned
 * (mapped) host memory; hidden must be device memory, 16-byte aligned;
 * codes 8-byte and scales 4-byte aligned.  cu_seqlens is a device array as
 * in hcr_restore.  Each call enqueues one kernel on `stream`; a token in no
 * request (cu_seqlens inconsistent with n_tokens) is skipped and flagged
 * HCR_DEVERR_SEQLENS.  Bins must be finite and > 0, group_tokens >= 1.
 */
typedef struct {
  float bins[3];          /* delta bins for the first, middle, last third of the layers */
  int32_t group_tokens;   /* tokens per anchor group (10 on the page)                     */
} hcr_codec_params;

hcr_status hcr_encode_hidden(hcr_handle* h, const hcr_codec_params* params, const void* hidden,
                             int32_t layer_begin, int32_t layer_end, int32_t n_req,
                             int32_t n_tokens, const int32_t* cu_seqlens, void* codes,
                             void* scales, void* stream);
hcr_status hcr_decode_hidden(hcr_handle* h, const hcr_codec_params* params, const void* codes,
                             const void* scales, int32_t layer_begin, int32_t layer_end,
                             int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                             void* hidden, void* stream);

/*
 * hcr_restore_encoded -- hcr_restore straight from the codec's encoded form
 * in device memory, decoded inside the restore kernels (HCache episode, cues
 * 30 and 32: restore from compressed hidden states; CacheGen review, section
 * 核心方法: the anchor + delta groups):
 *     codes  [layer_end - layer_begin][n_tokens][d_model] int8
 *     scales [layer_end - layer_begin][n_tokens] float32
 * as hcr_encode_hidden writes them with the same params.  The prepare kernel
 * computes the norm statistics of the decoded rows and each token's group
 * anchor; the projection (CTA pairs) loads the int8 codes with TMA and its
 * converter warps decode each k-block into the MMA's operand in shared
 * memory, so no decoded copy is written.  The caches are bit-identical to
 * hcr_decode_hidden followed by hcr_restore with the same arguments.
 *
 * codes and scales must be device memory (codes 16-byte, scales 4-byte
 * aligned); d_model must be a multiple of 16.  The workspace needs
 * hcr_encoded_workspace_bytes(h, n_tokens, layer_end - layer_begin) bytes
 * (the statistics plus 4 bytes per token).  Codec parameters are checked as
 * in hcr_decode_hidden and the rest as in hcr_restore before anything is
 * enqueued; HCR_ERR_UNSUPPORTED when the device fits no CTA pair of this
 * kernel.  A token in no request is decoded as zeros and flagged
 * HCR_DEVERR_SEQLENS; the other device-side checks are hcr_restore's.
 */
size_t hcr_encoded_workspace_bytes(const hcr_handle* h, int32_t n_tokens,
                                   int32_t n_layers_in_range);
hcr_status hcr_restore_encoded(hcr_handle* h, const hcr_codec_params* params, const void* codes,
                               const void* scales, int32_t layer_begin, int32_t layer_end,
                               int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                               const int32_t* start_pos, const int32_t* block_table,
                               int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                               const hcr_cache_layout* layout, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * hcr_restore_streamed_encoded -- hcr_restore_streamed from the codec's
 * encoded form in pinned host memory:
 *     codes_host  [layer_end - layer_begin][n_tokens][d_model] int8
 *     scales_host [layer_end - layer_begin][n_tokens] float32
 * as hcr_encode_hidden writes them (with the same params).  Each group of
 * layers is copied (about half the bytes of the hidden states) on the
 * handle's copy stream, decoded into its staging slot on a second stream the
 * handle owns (so later copies never wait for a decode), then restored on
 * `stream`.  Groups grow 1, 2, 4 ... layers up to layers_per_chunk (the copy of
 * the codes is about twice as fast as a restore, so small first groups start
 * the restores early without stalling them later).  The caches are
 * bit-identical to hcr_restore of hcr_decode_hidden's output.
 * staging (256-byte aligned) holds the slots, each align256(chunk * n_tokens
 * * d_model) + align256(chunk * n_tokens * 4) + align256(chunk * n_tokens *
 * d_model * 2) bytes (codes, scales, decoded hidden states; up to 8 slots are
 * used), chunk = min(layers_per_chunk, layer_end - layer_begin).  Codec
 * parameters are checked as in hcr_decode_hidden before anything is
 * enqueued.  Other arguments and behaviour are as in hcr_restore_streamed.
 */
hcr_status hcr_restore_streamed_encoded(hcr_handle* h, const hcr_codec_params* params,
                                        const void* codes_host, const void* scales_host,
                                        int32_t layer_begin, int32_t layer_end, int32_t n_req,
                                        int32_t n_tokens, const int32_t* cu_seqlens,
                                        const int32_t* start_pos, const int32_t* block_table,
                                        int32_t max_blocks_per_req, void* k_cache,
                                        void* v_cache, const hcr_cache_layout* layout,
                                        void* staging, size_t staging_bytes,
                                        int32_t layers_per_chunk, void* workspace,
                                        size_t workspace_bytes, void* stream);

/*
 * hcr_restore_no_alloc -- hcr_restore without a caller-provided workspace.
 *
 * The paper has no counterpart to this call; it exists for callers of this
 * library that cannot allocate device memory when they need a restore, for
 * example a serving engine that gave all free HBM to its paged KV pool at
 * start-up, or one that must not call cudaMalloc/cudaFree (which can
 * synchronise the device) while decode kernels run on its other streams.
 *
 * Same arguments and results as hcr_restore, minus workspace and
 * workspace_bytes.  The scratch is one fixed array of
 * HCR_NO_ALLOC_SCRATCH_BYTES in device global memory, part of the library
 * image: every GPU that loads the library holds it until the process exits.
 * A restore whose hcr_workspace_bytes() exceeds that size is rejected with
 * HCR_ERR_WORKSPACE before anything is enqueued (restore fewer tokens or
 * layers per call).  The handle's device must be current.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and looks it up again
 * whenever the current CUDA context differs from the one of the last lookup
 * (after cudaDeviceReset, say, the array may sit elsewhere); make the first
 * call in each context before any stream capture.  Every call on a device shares the one array,
 * which keeps the last call's contents; nothing in it needs to start at
 * zero (each restore writes every scratch word it later reads).  Calls
 * whose GPU work can overlap -- on different streams, or from different
 * handles, without ordering between them -- race on the array and give
 * undefined results.  This call allocates nothing: no cudaMalloc, cudaFree
 * or allocating library routine.
 */
#define HCR_NO_ALLOC_SCRATCH_BYTES (16u << 20)
hcr_status hcr_restore_no_alloc(hcr_handle* h, const void* hidden, int32_t layer_begin,
                                int32_t layer_end, int32_t n_req, int32_t n_tokens,
                                const int32_t* cu_seqlens, const int32_t* start_pos,
                                const int32_t* block_table, int32_t max_blocks_per_req,
                                void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                                void* stream);

/*
 * hcr_project_variant -- the tile variant the projection of n_tokens tokens
 * over n_layers layers uses: 1 for single CTAs (128x256 tiles), 2 for CTA
 * pairs (256x256 tiles, cta_group::2), 3 for CTA pairs with the weight rows
 * as the MMA's M side (two 128-wide heads) and a chunk of tokens as its N side
 * (tokens padded to a multiple of 16 instead of 128 rows; 128-wide heads
 * only).  Host-only; 0 for a NULL handle or empty sizes.  The choice, made
 * from measurements on GB300: 3 for 257..320 tokens; otherwise pairs when
 * there is more than one 128-row tile of tokens, d_model <= 4096 (or, for
 * wider models, a call of at most 6.5 TFLOP that leaves the pairs no half
 * tail tile), padding to
 * 128-row tiles saves less than 10% of the rows that 256-row tiles pad, and
 * the call is at most 32 TFLOP (4 d_model d_kv n_tokens n_layers); single
 * CTAs otherwise.  hcr_debug_set_variant overrides it.
 */
int32_t hcr_project_variant(const hcr_handle* h, int32_t n_tokens, int32_t n_layers);

/*
 * hcr_check_device_error -- synchronise `stream`, then read and clear the
 * handle's device error word.  Returns HCR_OK, HCR_ERR_DEVICE_BOUNDS or
 * HCR_ERR_TIMEOUT (timeout wins), or HCR_ERR_CUDA if the synchronisation
 * failed.  The raw HCR_DEVERR_* bits go to *flags when flags is not NULL.
 */
hcr_status hcr_check_device_error(hcr_handle* h, void* stream, uint32_t* flags);

/*
 * hcr_debug_set_stall -- testing hook for the bounded pipeline waits.
 *
 * With enable != 0, later restores through this handle arm the first
 * shared-memory stage of each CTA without issuing its loads, so the tensor
 * core's wait for that stage can never complete.  The wait gives up after
 * its time limit (2 s), the kernel sets HCR_DEVERR_TIMEOUT, stops every
 * role, drains its in-flight copies and MMAs with bounded waits, frees its
 * tensor memory and returns; hcr_check_device_error then reports
 * HCR_ERR_TIMEOUT and the CUDA context stays usable.  enable = 0 restores
 * normal operation.  Not for production use; do not change it while a
 * restore through the handle may be enqueued.
 */
hcr_status hcr_debug_set_stall(hcr_handle* h, int32_t enable);

/*
 * hcr_debug_set_variant -- testing hook: which project-kernel variant later
 * restores through this handle use.  0 (default): automatic -- the choice
 * hcr_project_variant reports for the call's token and layer counts; 1:
 * always single CTAs (128-token tiles); 2: always CTA pairs (cta_group::2,
 * 256-token tiles; HCR_ERR_UNSUPPORTED if the device cannot co-schedule them);
 * 3: always CTA pairs with weight rows as M (HCR_ERR_UNSUPPORTED unless
 * head_dim is 128 and the pairs can be co-scheduled).
 * All variants compute the same values bit for bit.  Do not change it while
 * a restore through the handle may be enqueued.
 */
hcr_status hcr_debug_set_variant(hcr_handle* h, int32_t variant);

/*
 * hcr_debug_fused_stats -- testing hook (host-only): whether a restore of
 * n_tokens tokens over n_layers layers with a workspace of workspace_bytes
 * computes most of its norm statistics inside the projection kernel.
 * Returns 0 when it does not (the prepare kernel computes every layer's);
 * otherwise L0 >= 1: the prepare kernel computes layers [0, L0) of the call
 * and the projection's statistics warps the rest, each tile's epilogue
 * waiting (bounded) for its rows.  The results are the same bits either way.
 * It does when the projection runs token-row tiles (variants 1 and 2) of at
 * most 8 m-tiles per layer (2048 tokens for CTA pairs, 1024 for single
 * CTAs; above that the projection runs at its per-SM ingress limit and the
 * statistics' reads would cost it what the prepare pass does), the call has
 * more layers than the projection's first three rounds of tiles reach, and
 * workspace_bytes >= hcr_workspace_bytes (which includes room for the
 * per-16-token flags; the smaller minimum workspace disables it).
 */
int32_t hcr_debug_fused_stats(const hcr_handle* h, int32_t n_tokens, int32_t n_layers,
                              size_t workspace_bytes);

/*
 * hcr_debug_plan -- testing hook (host-only: no handle, no CUDA call): the
 * choices a restore of n_tokens tokens over n_layers layers of a model with
 * dims *d makes on a device with num_sms SMs, pair_clusters co-resident CTA
 * pairs of the token-row kernel and swap_clusters of the weight-row kernel
 * (0: unavailable), with a workspace of workspace_bytes bytes.  Writes
 * out[2] = {the tile variant hcr_project_variant would report, the layers the
 * prepare kernel keeps when the statistics are fused (hcr_debug_fused_stats),
 * else 0}.  HCR_ERR_INVALID_ARG if d or out is NULL.
 */
hcr_status hcr_debug_plan(const hcr_model_dims* d, int32_t n_tokens, int32_t n_layers,
                          int32_t num_sms, int32_t pair_clusters, int32_t swap_clusters,
                          size_t workspace_bytes, int32_t* out);

/*
 * hcr_debug_swap_plan -- testing hook (host-only, no handle, no CUDA call):
 * the token chunks and TMEM accumulator slots the weight-row tiles (variant
 * 3) would use for a projection of n_tokens tokens.  Writes out[6] = {chunk,
 * n_chunks, last_n, slot_cols, n_slots, ok}: n_chunks - 1 chunks of `chunk`
 * tokens and a last one of last_n (both multiples of 16); n_slots == 2: two
 * slots of slot_cols (256) TMEM columns, one per tile; n_slots == 3 (one
 * chunk of 257..320 tokens): two big slots of slot_cols columns taken in turn
 * and a small slot at column 2 * slot_cols for each tile's first
 * chunk - slot_cols columns.  ok is 0 when the variant cannot take the count.
 * HCR_ERR_INVALID_ARG if out is NULL.
 */
hcr_status hcr_debug_swap_plan(int32_t n_tokens, int32_t* out);

/*
 * hcr_debug_timeout_record -- diagnostics for HCR_ERR_TIMEOUT: synchronise
 * `stream`, copy the record of the first pipeline wait that gave up since the
 * last call into out[6] = {which wait (0: none), CTA, thread, a, b, parity}
 * and clear it.  Which wait: 1 producer (stage free), 3 MMA (accumulator
 * free), 4 MMA (stage full), 7 epilogue (accumulator full); a and b are the
 * tile index and the k-block or accumulator.
 */
hcr_status hcr_debug_timeout_record(hcr_handle* h, void* stream, uint32_t out[6]);

/* Static description of a status code. */
const char* hcr_status_string(hcr_status s);

/* Message for the most recent error returned on the calling host thread. */
const char* hcr_last_error(void);

/* Number of SMs the handle's persistent kernel is sized for (diagnostics). */
int32_t hcr_num_sms(const hcr_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* HCR_H_ */
