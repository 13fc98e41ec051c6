// Host side of the C ABI declared in include/hcr.h: argument validation,
// handle construction (weight packing, RoPE table), workspace planning,
// TMA tensor-map encoding and kernel launches.  No host code here touches
// restore data; every step of the computation runs in the CUDA kernels.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "hcr_host.h"

namespace hcr {
namespace {

thread_local std::string g_last_error;

hcr_status vrecord(hcr_status s, const char* fmt, va_list ap) {
  char buf[512];
  vsnprintf(buf, sizeof buf, fmt, ap);
  g_last_error = buf;
  return s;
}

hcr_status fail(hcr_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vrecord(s, fmt, ap);
  va_end(ap);
  return s;
}

hcr_status cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();  // clear a sticky-free error so later calls start clean
  return fail(e == cudaErrorMemoryAllocation ? HCR_ERR_OOM : HCR_ERR_CUDA, "%s: %s (%s)", what,
              cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library needs no link-time dependency on libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D K-major operand map: dims (inner, rows, layers), box (64, box_rows, 1),
// 128-byte swizzle, zero fill outside the tensor.
hcr_status encode_3d(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t rows,
                     uint64_t layers, uint32_t box_rows, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(HCR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {inner, rows, layers};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {uint32_t(kBlockK), box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map,
                  dtype == HCR_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HCR_ERR_CUDA, "tensor map for %s: CUresult %d", what, int(r));
  return HCR_OK;
}

// 5-D view of the packed weights [L][2 d_kv][d] for the weight-row tiles: dims
// (d, 8, 2, 8, heads) with row strides (1, 64, 8, 128) inside a 128-row head,
// box (64, 8, 2, 8, 1).  The box lands in shared memory as 128 rows in the
// order (k fastest) 8 * half + 16 * g + k for head row 64 * half + 8 * g + k,
// which puts each rotate-half pair (i, i + 64) eight TMEM lanes apart.
hcr_status encode_w5(CUtensorMap* map, const void* base, int dtype, uint64_t d, uint64_t heads) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(HCR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const uint64_t row = d * 2;   // bytes
  const cuuint64_t dims[5] = {d, 8, 2, 8, heads};
  const cuuint64_t strides[4] = {row, 64 * row, 8 * row, 128 * row};
  const cuuint32_t box[5] = {uint32_t(kBlockK), 8, 2, 8, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map,
                  dtype == HCR_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  5, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(HCR_ERR_CUDA, "tensor map for packed weights (weight rows): CUresult %d", int(r));
  return HCR_OK;
}

hcr_status validate_dims(const hcr_model_dims* d) {
  if (!d) return fail(HCR_ERR_INVALID_ARG, "dims is NULL");
  if (d->n_layers < 1) return fail(HCR_ERR_INVALID_ARG, "n_layers must be >= 1");
  if (d->d_model < 8 || d->d_model % 8)
    return fail(HCR_ERR_INVALID_ARG, "d_model must be a positive multiple of 8");
  if (d->n_kv_heads < 1 || d->n_heads < d->n_kv_heads || d->n_heads % d->n_kv_heads)
    return fail(HCR_ERR_INVALID_ARG, "n_heads must be a positive multiple of n_kv_heads");
  if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
    return fail(HCR_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (int64_t(d->n_kv_heads) * d->head_dim > (1 << 20))
    return fail(HCR_ERR_UNSUPPORTED, "n_kv_heads * head_dim too large");
  if (d->norm != HCR_NORM_RMS && d->norm != HCR_NORM_LAYER)
    return fail(HCR_ERR_INVALID_ARG, "norm must be HCR_NORM_RMS or HCR_NORM_LAYER");
  if (!(d->norm_eps >= 0.f) || !std::isfinite(d->norm_eps))
    return fail(HCR_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
  if (d->rope != HCR_ROPE_NONE && d->rope != HCR_ROPE_ROTATE_HALF)
    return fail(HCR_ERR_INVALID_ARG, "rope must be HCR_ROPE_NONE or HCR_ROPE_ROTATE_HALF");
  if (d->rope) {
    if (!(d->rope_theta > 0.f) || !std::isfinite(d->rope_theta))
      return fail(HCR_ERR_INVALID_ARG, "rope_theta must be finite and > 0");
    if (d->max_position < 1 || d->max_position > (1 << 24))
      return fail(HCR_ERR_INVALID_ARG, "max_position must be in [1, 2^24]");
  }
  if (d->dtype != HCR_DTYPE_BF16 && d->dtype != HCR_DTYPE_FP16)
    return fail(HCR_ERR_INVALID_ARG, "dtype must be HCR_DTYPE_BF16 or HCR_DTYPE_FP16");
  return HCR_OK;
}

#define HCR_RESTORE_ARGS_IN                                                                      \
  RestoreArgs a{hidden,     layer_begin, layer_end,          n_req,   n_tokens,                  \
                cu_seqlens, start_pos,   block_table,        max_blocks_per_req,                 \
                k_cache,    v_cache,     layout,             workspace, workspace_bytes,         \
                static_cast<cudaStream_t>(stream)}

struct RestoreArgs {
  const void* hidden;
  int32_t layer_begin, layer_end, n_req, n_tokens;
  const int32_t *cu_seqlens, *start_pos, *block_table;
  int32_t max_blocks;
  void *k_cache, *v_cache;
  const hcr_cache_layout* layout;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  // Statistics of the call's rows, [layer][token], when they do not live in
  // the workspace (the layer-pipelined restores keep one set per staging slot)
  const float* rstd = nullptr;
  const float* mean = nullptr;
};

// Returns HCR_OK with *empty set when there is nothing to do.  `stats` says
// whether the workspace must hold norm statistics for the layer range, not
// only the slot map.
hcr_status validate_restore(const hcr_handle* h, const RestoreArgs& a, bool* empty,
                            bool stats = true, const char* input = "hidden",
                            bool encoded = false) {
  *empty = false;
  if (!h) return fail(HCR_ERR_INVALID_ARG, "handle is NULL");
  const hcr_model_dims& d = h->impl.dims;
  if (a.layer_begin < 0 || a.layer_end < a.layer_begin || a.layer_end > d.n_layers)
    return fail(HCR_ERR_INVALID_ARG, "layer range [%d, %d) outside [0, %d)", a.layer_begin,
                a.layer_end, d.n_layers);
  if (a.n_tokens < 0) return fail(HCR_ERR_INVALID_ARG, "n_tokens must be >= 0");
  if (a.n_req < 0) return fail(HCR_ERR_INVALID_ARG, "n_req must be >= 0");
  if (a.n_tokens == 0 || a.layer_end == a.layer_begin) {
    *empty = true;
    return HCR_OK;
  }
  if (a.n_req < 1) return fail(HCR_ERR_INVALID_ARG, "n_tokens > 0 needs n_req >= 1");
  if (!a.hidden) return fail(HCR_ERR_INVALID_ARG, "%s is NULL", input);
  if (!aligned(a.hidden, 16))
    return fail(HCR_ERR_INVALID_ARG, "%s must be 16-byte aligned", input);
  if (!a.cu_seqlens || !a.start_pos || !a.block_table)
    return fail(HCR_ERR_INVALID_ARG, "cu_seqlens, start_pos and block_table must be non-NULL");
  if (a.max_blocks < 1) return fail(HCR_ERR_INVALID_ARG, "max_blocks_per_req must be >= 1");
  if (!a.k_cache || !a.v_cache) return fail(HCR_ERR_INVALID_ARG, "k_cache/v_cache is NULL");
  if (!aligned(a.k_cache, 16) || !aligned(a.v_cache, 16))
    return fail(HCR_ERR_INVALID_ARG, "k_cache and v_cache must be 16-byte aligned");
  if (!a.layout) return fail(HCR_ERR_INVALID_ARG, "layout is NULL");
  if (a.layout->num_blocks < 1 || a.layout->block_size < 1)
    return fail(HCR_ERR_INVALID_ARG, "num_blocks and block_size must be >= 1");
  const int64_t row = int64_t(d.n_kv_heads) * d.head_dim;
  const int64_t dense = int64_t(a.layout->num_blocks) * a.layout->block_size * row;
  if (a.layout->layer_stride_elems != 0 && a.layout->layer_stride_elems < dense)
    return fail(HCR_ERR_INVALID_ARG, "layer_stride_elems %lld smaller than one layer (%lld)",
                (long long)a.layout->layer_stride_elems, (long long)dense);
  if (a.layout->layer_stride_elems % 8)
    return fail(HCR_ERR_INVALID_ARG, "layer_stride_elems must be a multiple of 8");
  const size_t need = workspace_layout(a.n_tokens, stats ? a.layer_end - a.layer_begin : 0,
                                       d.norm == HCR_NORM_LAYER, encoded).total;
  if (!a.workspace) return fail(HCR_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(a.workspace, 256))
    return fail(HCR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (a.workspace_bytes < need)
    return fail(HCR_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", a.workspace_bytes, need);
  return HCR_OK;
}

// Norm statistics fused into the token-row projection: the prepare kernel
// computes the first layer0 layers of the call (those the projection's first
// three rounds of tiles reach) and the projection's statistics warps the rest,
// items of kStatsItemRows tokens per layer.  On when the projection runs
// token-row tiles, the call covers more layers than that, its statistics live
// in the workspace and the workspace has room for the flags.
struct FusedStats {
  bool on = false;
  int32_t layer0 = 0, items = 0;
};
constexpr int64_t kFusedStatsMaxMTiles = 8;   // token m-tiles per layer
FusedStats fused_stats(const Handle& H, const RestoreArgs& a);

// stats = false: the slot map only (the K/V row copies need no statistics).
// enc: the statistics of the rows decoded from the codec's form, and each
// token's group anchor for the projection (a.hidden is then unused).
hcr_status do_prepare(hcr_handle* h, const RestoreArgs& a, bool stats = true,
                      const CodecInput* enc = nullptr, float* stats_rstd = nullptr,
                      float* stats_mean = nullptr) {
  NvtxRange range("hcr.prepare");
  const Handle& H = h->impl;
  const hcr_model_dims& d = H.dims;
  const int32_t nl = stats ? a.layer_end - a.layer_begin : 0;
  const WorkspaceLayout w =
      workspace_layout(a.n_tokens, nl, d.norm == HCR_NORM_LAYER, enc != nullptr);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  PrepareParams p{};
  p.cu_seqlens = a.cu_seqlens;
  p.start_pos = a.start_pos;
  p.block_table = a.block_table;
  p.n_req = a.n_req;
  p.n_tokens = a.n_tokens;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.layout->num_blocks;
  p.block_size = a.layout->block_size;
  p.max_position = d.max_position;
  p.check_position = d.rope != HCR_ROPE_NONE;
  p.slot = reinterpret_cast<int64_t*>(ws + w.slot_off);
  p.pos = reinterpret_cast<int32_t*>(ws + w.pos_off);
  p.hidden = a.hidden;
  p.n_layers = nl;
  p.d_model = d.d_model;
  p.layer_norm = d.norm == HCR_NORM_LAYER;
  p.dtype = d.dtype;
  p.eps = d.norm_eps;
  p.rstd = reinterpret_cast<float*>(ws + w.rstd_off);
  p.mean = p.layer_norm ? reinterpret_cast<float*>(ws + w.mean_off) : nullptr;
  p.err = H.err;
  p.layer_begin = a.layer_begin;
  if (stats_rstd) {   // statistics only, into the given arrays
    p.skip_placement = 1;
    p.rstd = stats_rstd;
    p.mean = p.layer_norm ? stats_mean : nullptr;
  }
  if (enc) {
    p.enc = *enc;
    p.enc.anchor = reinterpret_cast<int32_t*>(ws + w.anchor_off);
  }
  if (stats && !enc && !stats_rstd) {
    const FusedStats fs = fused_stats(H, a);
    if (fs.on) {
      p.n_layers = fs.layer0;
      p.zero_flags = reinterpret_cast<int32_t*>(ws + w.flags_off);
      p.n_zero_flags = int64_t(nl) * fs.items;
    }
  }
  cudaError_t e = launch_prepare(p, a.stream);
  if (e != cudaSuccess) return cuda_fail(e, "prepare launch");
  return HCR_OK;
}

// The automatic tile-variant choice, one table.  Every threshold comes from a
// measurement on GB300 (project kernel time, CUDA events); for a new shape,
// re-derive it with `bench.py --workload <shape>-T<n> --variant 1|2|3` at the
// token counts around it.
struct VariantPolicy {
  // CTA pairs need more than one 128-row tile of tokens: at 64 and 128 tokens
  // single CTAs ran 0.337 / 0.348 ms, and pairs only pad their second half.
  int32_t pair_min_tokens = kBlockM + 1;
  // Widths above 4096: single CTAs ran 4-5% faster on the 13B (5120) and
  // OPT-30B (7168) shapes in long power-capped restores and no slower at
  // 2-4K tokens; at 4096 the pairs win by 5-7%.  In calls of at most
  // pair_wide_max_call_flops, when the pairs need no half tail tile, the pairs
  // win at those widths too (project ms, single against pairs: 13B 256 tokens
  // 0.855/0.749, 512 1.524/1.387, 768 2.147/2.000, 1024 2.865/2.708, 1280
  // 3.452/3.358, 1536 4.080/3.988; OPT-30B 256 tokens 2.064/1.884, 512
  // 3.666/3.506).  Above that the power cap makes them tie or lose (13B 2048
  // tokens, 8.6 TFLOP: 5.386/5.378; OPT-30B 768, 7.6 TFLOP: 5.40/5.41; 1024
  // 7.02/7.14; 1536 10.18/10.71), and with a half tail they lose at OPT-30B's
  // width (384 tokens 2.888/3.136, 640 4.511/4.951, 794 5.993/6.510).
  int32_t pair_max_d_model = 4096;
  double pair_wide_max_call_flops = 6.5e12;
  // Calls above 32 TFLOP (4 d_model d_kv tokens layers): pairs draw more power
  // per clock and the cap pulls their clock down (629K tokens in 8-layer calls
  // of 338 TFLOP: single CTAs 10% faster; 35 TFLOP: a tie; 8.8: pairs 5.5%).
  double pair_max_call_flops = 32e12;
  // Single CTAs where their 128-row tiles pad at least 10% fewer rows than
  // the pairs' 256-row tiles (counting the pairs' half tail tile as 128 rows).
  double pair_pad_ratio = 0.9;
  // Weight rows as M for 257..320 tokens (one chunk of up to 320 on the
  // three-slot TMEM layout): 7B 0.526 against 0.576 ms (pairs), 13B 0.974
  // against 1.080 (single CTAs), OPT-30B 2.33 against 2.54 ms (single CTAs);
  // from 384 tokens the token-row pairs were faster (7B, one session: 384
  // tokens 0.632 against 0.659 ms, 512 0.703/0.742, 794 1.272/1.299, 1024
  // 1.366/1.445, 1536 2.034/2.137).
  int32_t rows_min_tokens = kBlockN + 1;
  int32_t rows_max_tokens = kSwapMaxChunk;
};
constexpr VariantPolicy kPolicy{};

// A pair projection can end each layer with an M=128 "half tail" tile (64
// rows per CTA) when the last 256-row tile holds at most 128 rows; its
// epilogue splits a row's 256 columns in two 128-column halves, so heads must
// fit in 128 columns.
bool half_tail_fits(const hcr_model_dims& d, int32_t n_tokens) {
  const int32_t rem = n_tokens % (2 * kBlockM);
  return d.head_dim <= kBlockN / 2 && rem > 0 && rem <= kBlockM;
}

bool use_pairs(const Handle& H, int32_t n_tokens, int32_t n_layers) {
  const hcr_model_dims& d = H.dims;
  const int64_t d_kv = int64_t(d.n_kv_heads) * d.head_dim;
  // rows each variant computes: 128-row tiles, or 256-row tiles whose last
  // tile may be a 128-row half tail
  const int64_t pad128 = (int64_t(n_tokens) + kBlockM - 1) / kBlockM * kBlockM;
  const int64_t pad_pair = (int64_t(n_tokens) + 2 * kBlockM - 1) / (2 * kBlockM) * (2 * kBlockM) -
                           (half_tail_fits(d, n_tokens) ? kBlockM : 0);
  const double call_flops = 4.0 * d.d_model * double(d_kv) * double(n_tokens) * n_layers;
  bool pair = H.pair_clusters > 0 && n_tokens >= kPolicy.pair_min_tokens &&
              (d.d_model <= kPolicy.pair_max_d_model ||
               (call_flops <= kPolicy.pair_wide_max_call_flops &&
                !half_tail_fits(d, n_tokens))) &&
              double(pad128) > kPolicy.pair_pad_ratio * double(pad_pair) &&
              call_flops <= kPolicy.pair_max_call_flops;
  if (H.variant == 1) pair = false;
  if (H.variant == 2) pair = H.pair_clusters > 0;
  return pair;
}

// Token chunks of the weight-row tiles: n_chunks chunks of `chunk` tokens (a
// multiple of 16) and a last chunk of last_n (a multiple of 16), balanced so
// padding stays below 16 tokens per chunk, on TMEM accumulator slots of
// slot_cols columns: everything up to 256 tokens per chunk on two 256-column
// slots, and 257..320 tokens as one chunk on two big slots of the largest
// multiple of 32 columns that leaves room for the chunk's remaining columns in
// a third, small slot after them (192 + 192 + 112 columns for 304 tokens).
struct SwapPlan {
  int32_t chunk = 0, n_chunks = 0, last_n = 0, slot_cols = 0, n_slots = 0;
  bool ok = false;
};

SwapPlan swap_plan(int32_t n_tokens) {
  SwapPlan s;
  if (n_tokens <= 0) return s;
  const int64_t T = n_tokens;
  const bool ring3 = T > kBlockN && T <= kSwapMaxChunk;
  s.n_slots = ring3 ? 3 : 2;
  const int64_t max_chunk = ring3 ? kSwapMaxChunk : kBlockN;
  s.n_chunks = int32_t((T + max_chunk - 1) / max_chunk);
  const int64_t per = (T + s.n_chunks - 1) / s.n_chunks;
  s.chunk = int32_t((per + 15) / 16 * 16);
  const int64_t rest = T - int64_t(s.n_chunks - 1) * s.chunk;
  s.last_n = int32_t((rest + 15) / 16 * 16);
  s.slot_cols = ring3 ? (kSwapTmemCols - s.chunk) / 32 * 32 : kBlockN;
  s.ok = s.chunk >= 16 && s.chunk <= max_chunk && rest > 0 && s.last_n <= s.chunk &&
         (!ring3 || (s.chunk - s.slot_cols >= 16 && 2 * s.slot_cols + (s.chunk - s.slot_cols) <=
                                                        kSwapTmemCols));
  return s;
}

bool swap_available(const Handle& H) { return H.swap_clusters > 0; }

// Tile variant of a projection (kPolicy): 1 single CTAs, 2 CTA pairs (token
// rows as M), 3 CTA pairs with weight rows as M and chunks of tokens as N.
int32_t choose_variant(const Handle& H, int32_t n_tokens, int32_t n_layers) {
  const bool swap_ok = swap_available(H) && swap_plan(n_tokens).ok;
  int32_t v = use_pairs(H, n_tokens, n_layers) ? 2 : 1;
  if (swap_ok && n_tokens >= kPolicy.rows_min_tokens && n_tokens <= kPolicy.rows_max_tokens)
    v = 3;
  if (H.variant == 1) v = 1;
  if (H.variant == 2) v = H.pair_clusters > 0 ? 2 : 1;
  if (H.variant == 3 && swap_ok) v = 3;
  return v;
}

FusedStats fused_stats(const Handle& H, const RestoreArgs& a) {
  FusedStats f;
  const hcr_model_dims& d = H.dims;
  const int32_t nl = a.layer_end - a.layer_begin;
  if (nl < 2 || a.rstd || a.n_tokens <= 0) return f;
  const int32_t v = choose_variant(H, a.n_tokens, nl);
  if (v != 1 && v != 2) return f;
  if (a.workspace_bytes < workspace_layout(a.n_tokens, nl, d.norm == HCR_NORM_LAYER).total_fused)
    return f;
  const int64_t tile_m = v == 2 ? 2 * kBlockM : kBlockM;
  const int64_t m_tiles = (a.n_tokens + tile_m - 1) / tile_m;
  // With more m-tiles per layer the projection runs at its per-SM ingress
  // limit and the statistics warps' reads cost it what the prepare pass would
  // (7B, CTA pairs, alternating builds: 1100 tokens 1.548/1.561 against
  // 1.589/1.601 ms per step, 2048 tokens 2.695/2.707 against 2.703/2.747,
  // 4096 tokens 5.555/5.526 against 5.489/5.518).
  if (m_tiles > kFusedStatsMaxMTiles) return f;
  const int64_t n_tiles = (2 * int64_t(d.n_kv_heads) * d.head_dim + kBlockN - 1) / kBlockN;
  const int64_t per_layer = m_tiles * n_tiles;
  const int64_t units = std::min<int64_t>(per_layer * nl, v == 2 ? H.pair_clusters : H.num_sms);
  const int64_t layer0 = std::max<int64_t>(1, (3 * units + per_layer - 1) / per_layer);
  if (layer0 >= nl) return f;
  f.on = true;
  f.layer0 = int32_t(layer0);
  f.items = (a.n_tokens + kStatsItemRows - 1) / kStatsItemRows;
  return f;
}

hcr_status do_project_swap(hcr_handle* h, const RestoreArgs& a) {
  const Handle& H = h->impl;
  const hcr_model_dims& d = H.dims;
  const int32_t nl = a.layer_end - a.layer_begin;
  const WorkspaceLayout w = workspace_layout(a.n_tokens, nl, d.norm == HCR_NORM_LAYER);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int32_t d_kv = d.n_kv_heads * d.head_dim;
  const SwapPlan sp = swap_plan(a.n_tokens);

  CUtensorMap tmap_h;
  hcr_status st = encode_3d(&tmap_h, a.hidden, d.dtype, uint64_t(d.d_model),
                            uint64_t(a.n_tokens), uint64_t(nl), uint32_t(sp.chunk / 2),
                            "hidden (token chunks)");
  if (st != HCR_OK) return st;

  ProjectParams p{};
  p.n_tokens = a.n_tokens;
  p.d_model = d.d_model;
  p.n_cols = 2 * d_kv;
  p.d_kv = d_kv;
  p.head_dim = d.head_dim;
  p.n_layers = nl;
  p.layer_begin = a.layer_begin;
  p.k_blocks = (d.d_model + kBlockK - 1) / kBlockK;
  p.chunk = sp.chunk;
  p.n_chunks = sp.n_chunks;
  p.last_n = sp.last_n;
  p.head_pairs = d.n_kv_heads;
  p.stages = swap_stages(sp.chunk);
  p.slot_cols = sp.slot_cols;
  p.n_slots = sp.n_slots;
  p.num_tiles = int64_t(nl) * p.head_pairs * p.n_chunks;
  p.layer_norm = d.norm == HCR_NORM_LAYER;
  p.has_bias = H.col_bias != nullptr;
  p.rope = d.rope != HCR_ROPE_NONE;
  p.dtype = d.dtype;
  p.slot = reinterpret_cast<const int64_t*>(ws + w.slot_off);
  p.pos = reinterpret_cast<const int32_t*>(ws + w.pos_off);
  p.rstd = a.rstd ? a.rstd : reinterpret_cast<const float*>(ws + w.rstd_off);
  p.mean = !p.layer_norm ? nullptr
                         : (a.mean ? a.mean : reinterpret_cast<const float*>(ws + w.mean_off));
  p.col_sum = H.col_sum ? H.col_sum + int64_t(a.layer_begin) * 2 * d_kv : nullptr;
  p.col_bias = H.col_bias ? H.col_bias + int64_t(a.layer_begin) * 2 * d_kv : nullptr;
  p.rope_tab = H.rope_tab;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.layer_stride = a.layout->layer_stride_elems
                       ? a.layout->layer_stride_elems
                       : int64_t(a.layout->num_blocks) * a.layout->block_size * d_kv;
  p.row_elems = d_kv;
  p.err = H.err;
  p.debug_stall = H.debug_stall;
  const int64_t units = std::min<int64_t>(p.num_tiles, H.swap_clusters);
  // Tiles past the last whole round run as two half-chunk units each when
  // that round then fits in half a tile's time on the pairs.
  const int64_t rest = p.num_tiles % units;
  p.split_tail =
      (rest > 0 && 2 * rest <= units && p.chunk >= 32 && p.last_n >= 32) ? int32_t(rest) : 0;
  const int grid = 2 * int(units);
  cudaError_t e = launch_project_swap(tmap_h, H.tmap_w5, p, grid, a.stream);
  if (e != cudaSuccess) return cuda_fail(e, "project launch (weight rows)");
  return HCR_OK;
}

// Parameters of a token-row projection (single CTAs, CTA pairs, and the
// pairs that decode the codec's form); `encoded` places the workspace's
// statistics as the encoded restore lays them out.
ProjectParams token_row_params(const Handle& H, const RestoreArgs& a, bool pair, bool encoded) {
  const hcr_model_dims& d = H.dims;
  const int32_t nl = a.layer_end - a.layer_begin;
  const WorkspaceLayout w = workspace_layout(a.n_tokens, nl, d.norm == HCR_NORM_LAYER, encoded);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int32_t d_kv = d.n_kv_heads * d.head_dim;
  ProjectParams p{};
  p.n_tokens = a.n_tokens;
  p.d_model = d.d_model;
  p.n_cols = 2 * d_kv;
  p.d_kv = d_kv;
  p.head_dim = d.head_dim;
  p.n_layers = nl;
  p.layer_begin = a.layer_begin;
  const int tile_m = pair ? 2 * kBlockM : kBlockM;
  p.half_tail = pair && half_tail_fits(d, a.n_tokens);
  p.m_tiles = (a.n_tokens + tile_m - 1) / tile_m;
  p.n_tiles = (2 * d_kv + kBlockN - 1) / kBlockN;
  p.k_blocks = (d.d_model + kBlockK - 1) / kBlockK;
  p.num_tiles = int64_t(nl) * p.m_tiles * p.n_tiles;
  p.layer_norm = d.norm == HCR_NORM_LAYER;
  p.has_bias = H.col_bias != nullptr;
  p.rope = d.rope != HCR_ROPE_NONE;
  p.dtype = d.dtype;
  p.slot = reinterpret_cast<const int64_t*>(ws + w.slot_off);
  p.pos = reinterpret_cast<const int32_t*>(ws + w.pos_off);
  p.rstd = a.rstd ? a.rstd : reinterpret_cast<const float*>(ws + w.rstd_off);
  p.mean = !p.layer_norm ? nullptr
                         : (a.mean ? a.mean : reinterpret_cast<const float*>(ws + w.mean_off));
  p.col_sum = H.col_sum ? H.col_sum + int64_t(a.layer_begin) * 2 * d_kv : nullptr;
  p.col_bias = H.col_bias ? H.col_bias + int64_t(a.layer_begin) * 2 * d_kv : nullptr;
  p.rope_tab = H.rope_tab;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  const int64_t row = int64_t(d_kv);
  p.layer_stride = a.layout->layer_stride_elems
                       ? a.layout->layer_stride_elems
                       : int64_t(a.layout->num_blocks) * a.layout->block_size * row;
  p.row_elems = d_kv;
  p.err = H.err;
  p.debug_stall = H.debug_stall;
  return p;
}

hcr_status do_project(hcr_handle* h, const RestoreArgs& a) {
  NvtxRange range("hcr.project");
  const Handle& H = h->impl;
  const hcr_model_dims& d = H.dims;
  const int32_t nl = a.layer_end - a.layer_begin;
  const int32_t variant = choose_variant(H, a.n_tokens, nl);
  if (variant == 3) return do_project_swap(h, a);

  CUtensorMap tmap_h;
  hcr_status st = encode_3d(&tmap_h, a.hidden, d.dtype, uint64_t(d.d_model),
                            uint64_t(a.n_tokens), uint64_t(nl), kBlockM, "hidden");
  if (st != HCR_OK) return st;

  const bool pair = variant == 2;
  ProjectParams p = token_row_params(H, a, pair, false);
  const FusedStats fs = fused_stats(H, a);
  if (fs.on) {
    const WorkspaceLayout w = workspace_layout(a.n_tokens, nl, d.norm == HCR_NORM_LAYER);
    p.stats_flags = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.workspace) + w.flags_off);
    p.stats_layer0 = fs.layer0;
    p.stats_items = fs.items;
    p.hidden_rows = a.hidden;
    p.eps = d.norm_eps;
  }
  const int grid = pair ? 2 * int(std::min<int64_t>(p.num_tiles, H.pair_clusters))
                        : int(std::min<int64_t>(p.num_tiles, H.num_sms));
  CUtensorMap tmap_h64 = tmap_h;
  if (p.half_tail) {
    st = encode_3d(&tmap_h64, a.hidden, d.dtype, uint64_t(d.d_model), uint64_t(a.n_tokens),
                   uint64_t(nl), kBlockM / 2, "hidden (64-row boxes)");
    if (st != HCR_OK) return st;
  }
  cudaError_t e = launch_project(tmap_h, tmap_h64, pair ? H.tmap_w_half : H.tmap_w, p, grid,
                                 pair, a.stream);
  if (e != cudaSuccess) return cuda_fail(e, "project launch");
  return HCR_OK;
}

// 4-D map of the codec's int8 codes [Lr][T][d] viewed as (16 codes, T rows,
// d/16 column chunks, Lr layers): a box (16, kEncCodeRows, 4, 1) lands one
// k-block's 64 codes of kEncCodeRows rows chunk-major in shared memory, each
// 16-code chunk of the rows kEncCodeRows x 16 bytes after the previous one.
// No swizzle; zero fill outside the tensor (the first tile's box starts at row
// -kEncCodeHalo, a ragged last k-block's box ends past d/16).
hcr_status encode_codes(CUtensorMap* map, const void* codes, uint64_t d, uint64_t rows,
                        uint64_t layers) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(HCR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[4] = {16, rows, d / 16, layers};
  const cuuint64_t strides[3] = {d, 16, d * rows};
  const cuuint32_t box[4] = {16, uint32_t(kEncCodeRows), uint32_t(kBlockK / 16), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(codes), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HCR_ERR_CUDA, "tensor map for codes: CUresult %d", int(r));
  return HCR_OK;
}

// The projection of a restore from the codec's form (CTA pairs whose
// converter warps decode the A operand); enc.anchor is set from the workspace.
hcr_status do_project_enc(hcr_handle* h, const RestoreArgs& a, const CodecInput& enc) {
  NvtxRange range("hcr.project_encoded");
  const Handle& H = h->impl;
  const hcr_model_dims& d = H.dims;
  const int32_t nl = a.layer_end - a.layer_begin;
  CUtensorMap tmap_c;
  hcr_status st = encode_codes(&tmap_c, enc.codes, uint64_t(d.d_model), uint64_t(a.n_tokens),
                               uint64_t(nl));
  if (st != HCR_OK) return st;
  const ProjectParams p = token_row_params(H, a, true, true);
  CodecInput e = enc;
  const WorkspaceLayout w = workspace_layout(a.n_tokens, nl, d.norm == HCR_NORM_LAYER, true);
  e.anchor = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.workspace) + w.anchor_off);
  const int grid = 2 * int(std::min<int64_t>(p.num_tiles, H.enc_clusters));
  cudaError_t err = launch_project_enc(tmap_c, H.tmap_w_half, p, e, grid, a.stream);
  if (err != cudaSuccess) return cuda_fail(err, "project launch (encoded input)");
  return HCR_OK;
}

}  // namespace

size_t workspace_min_bytes(const hcr_handle* h, int32_t n_tokens, int32_t n_layers) {
  if (!h || n_tokens <= 0 || n_layers <= 0) return 0;
  return workspace_layout(n_tokens, n_layers, h->impl.dims.norm == HCR_NORM_LAYER).total;
}

// Pieces of hcr_restore for the layer-pipelined restores (hcr_streamed.cu).
hcr_status pipeline_placement(hcr_handle* h, const void* staging, int32_t layer_begin,
                              int32_t layer_end, int32_t n_req, int32_t n_tokens,
                              const int32_t* cu_seqlens, const int32_t* start_pos,
                              const int32_t* block_table, int32_t max_blocks_per_req,
                              void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                              void* workspace, size_t workspace_bytes, int32_t stats_layers,
                              void* stream, bool* ok) {
  *ok = false;
  const void* hidden = staging;
  HCR_RESTORE_ARGS_IN;
  bool empty = false;
  hcr_status st = validate_restore(h, a, &empty, /*stats=*/false, "staging");
  if (st != HCR_OK || empty) return st;
  const WorkspaceLayout w = workspace_layout(n_tokens, stats_layers,
                                             h->impl.dims.norm == HCR_NORM_LAYER);
  if (workspace_bytes < w.total) return HCR_OK;   // no room: the caller restores group by group
  *ok = true;
  return do_prepare(h, a, /*stats=*/false);
}

hcr_status pipeline_stats(hcr_handle* h, const void* hidden, int32_t layer_begin,
                          int32_t layer_end, int32_t n_req, int32_t n_tokens,
                          const int32_t* cu_seqlens, const int32_t* start_pos,
                          const int32_t* block_table, int32_t max_blocks_per_req,
                          void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                          void* workspace, size_t workspace_bytes, float* rstd, float* mean,
                          void* stream) {
  HCR_RESTORE_ARGS_IN;
  return do_prepare(h, a, true, nullptr, rstd, mean);
}

hcr_status pipeline_project(hcr_handle* h, const void* hidden, int32_t layer_begin,
                            int32_t layer_end, int32_t n_req, int32_t n_tokens,
                            const int32_t* cu_seqlens, const int32_t* start_pos,
                            const int32_t* block_table, int32_t max_blocks_per_req,
                            void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                            void* workspace, size_t workspace_bytes, const float* rstd,
                            const float* mean, void* stream) {
  HCR_RESTORE_ARGS_IN;
  a.rstd = rstd;
  a.mean = mean;
  return do_project(h, a);
}

namespace {

void free_handle(Handle& H) {
  release_streamed(H);
  cudaFree(H.w_packed);
  cudaFree(H.col_sum);
  cudaFree(H.col_bias);
  cudaFree(H.rope_tab);
  cudaFree(H.err);
  H.w_packed = nullptr;
  H.col_sum = H.col_bias = nullptr;
  H.rope_tab = nullptr;
  H.err = nullptr;
}

}  // namespace

hcr_status set_last_error(hcr_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vrecord(s, fmt, ap);
  va_end(ap);
  return s;
}

}  // namespace hcr

using namespace hcr;

extern "C" {

const char* hcr_status_string(hcr_status s) {
  switch (s) {
    case HCR_OK: return "HCR_OK";
    case HCR_ERR_INVALID_ARG: return "HCR_ERR_INVALID_ARG: invalid argument";
    case HCR_ERR_UNSUPPORTED: return "HCR_ERR_UNSUPPORTED: unsupported configuration";
    case HCR_ERR_CUDA: return "HCR_ERR_CUDA: CUDA call failed";
    case HCR_ERR_OOM: return "HCR_ERR_OOM: device allocation failed";
    case HCR_ERR_WORKSPACE: return "HCR_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case HCR_ERR_DEVICE_BOUNDS:
      return "HCR_ERR_DEVICE_BOUNDS: out-of-range block id or position; rows skipped";
    case HCR_ERR_TIMEOUT: return "HCR_ERR_TIMEOUT: device pipeline wait timed out";
  }
  return "unknown hcr_status";
}

const char* hcr_last_error(void) { return g_last_error.c_str(); }

hcr_status hcr_create(const hcr_model_dims* dims, const void* const* gamma,
                      const void* const* beta, const void* const* w_k, const void* const* w_v,
                      const void* const* b_k, const void* const* b_v, hcr_handle** out) {
  if (!out) return fail(HCR_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  hcr_status st = validate_dims(dims);
  if (st != HCR_OK) return st;
  const hcr_model_dims& d = *dims;
  const bool ln = d.norm == HCR_NORM_LAYER;
  if (!gamma || !w_k || !w_v) return fail(HCR_ERR_INVALID_ARG, "gamma, w_k, w_v must be given");
  if (ln && !beta) return fail(HCR_ERR_INVALID_ARG, "LayerNorm needs beta");
  if (!ln && beta) return fail(HCR_ERR_INVALID_ARG, "RMSNorm takes no beta (pass NULL)");
  if (d.has_kv_bias && (!b_k || !b_v))
    return fail(HCR_ERR_INVALID_ARG, "has_kv_bias needs b_k and b_v");
  if (!d.has_kv_bias && (b_k || b_v))
    return fail(HCR_ERR_INVALID_ARG, "b_k/b_v given but has_kv_bias is 0");
  for (int l = 0; l < d.n_layers; ++l) {
    if (!gamma[l] || !w_k[l] || !w_v[l] || (ln && !beta[l]) ||
        (d.has_kv_bias && (!b_k[l] || !b_v[l])))
      return fail(HCR_ERR_INVALID_ARG, "layer %d: a parameter pointer is NULL", l);
  }

  auto* h = new (std::nothrow) hcr_handle();
  if (!h) return fail(HCR_ERR_OOM, "host allocation of the handle failed");
  Handle& H = h->impl;
  H.dims = d;
  const int32_t d_kv = d.n_kv_heads * d.head_dim;
  const int64_t per_layer = int64_t(2) * d_kv * d.d_model;
  cudaError_t e;
  auto bail = [&](cudaError_t err, const char* what) {
    hcr_status s = cuda_fail(err, what);
    free_handle(H);
    delete h;
    return s;
  };
  if ((e = cudaGetDevice(&H.device)) != cudaSuccess) return bail(e, "cudaGetDevice");
  if ((e = cudaDeviceGetAttribute(&H.num_sms, cudaDevAttrMultiProcessorCount, H.device)) !=
      cudaSuccess)
    return bail(e, "cudaDeviceGetAttribute");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, H.device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, H.device);
  if (major != 10 || minor != 3) {
    free_handle(H);
    delete h;
    return fail(HCR_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a",
                major, minor);
  }

  if ((e = cudaMalloc(&H.w_packed, size_t(per_layer) * d.n_layers * 2)) != cudaSuccess)
    return bail(e, "cudaMalloc(packed weights)");
  if (ln && (e = cudaMalloc(&H.col_sum, sizeof(float) * 2 * d_kv * d.n_layers)) != cudaSuccess)
    return bail(e, "cudaMalloc(column sums)");
  if ((ln || d.has_kv_bias) &&
      (e = cudaMalloc(&H.col_bias, sizeof(float) * 2 * d_kv * d.n_layers)) != cudaSuccess)
    return bail(e, "cudaMalloc(column bias)");
  if ((e = cudaMalloc(&H.err, sizeof(uint32_t) * kErrWords)) != cudaSuccess)
    return bail(e, "cudaMalloc(err)");
  if ((e = cudaMemset(H.err, 0, sizeof(uint32_t) * kErrWords)) != cudaSuccess)
    return bail(e, "cudaMemset");

  for (int l = 0; l < d.n_layers; ++l) {
    void* dst = static_cast<uint8_t*>(H.w_packed) + size_t(per_layer) * 2 * l;
    if ((e = launch_pack_weights(w_k[l], w_v[l], gamma[l], dst, d_kv, d.d_model, d.dtype, 0)) !=
        cudaSuccess)
      return bail(e, "pack launch");
    if (H.col_sum || H.col_bias) {
      if ((e = launch_column_constants(dst, w_k[l], w_v[l], ln ? beta[l] : nullptr,
                                       d.has_kv_bias ? b_k[l] : nullptr,
                                       d.has_kv_bias ? b_v[l] : nullptr,
                                       H.col_sum ? H.col_sum + int64_t(l) * 2 * d_kv : nullptr,
                                       H.col_bias ? H.col_bias + int64_t(l) * 2 * d_kv : nullptr,
                                       d_kv, d.d_model, d.dtype, ln, d.has_kv_bias, 0)) !=
          cudaSuccess)
        return bail(e, "column-constant launch");
    }
  }

  if (d.rope) {
    // cos/sin of pos * theta^(-2i/dh), evaluated in double precision and
    // rounded once to float.
    const int half = d.head_dim / 2;
    std::vector<float> tab(size_t(d.max_position) * half * 2);
    std::vector<double> omega(half);
    for (int i = 0; i < half; ++i)
      omega[i] = std::pow(double(d.rope_theta), -2.0 * i / double(d.head_dim));
    for (int64_t p = 0; p < d.max_position; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = double(p) * omega[i];
        tab[(size_t(p) * half + i) * 2 + 0] = float(std::cos(ang));
        tab[(size_t(p) * half + i) * 2 + 1] = float(std::sin(ang));
      }
    if ((e = cudaMalloc(&H.rope_tab, tab.size() * sizeof(float))) != cudaSuccess)
      return bail(e, "cudaMalloc(rope table)");
    if ((e = cudaMemcpy(H.rope_tab, tab.data(), tab.size() * sizeof(float),
                        cudaMemcpyHostToDevice)) != cudaSuccess)
      return bail(e, "cudaMemcpy(rope table)");
  }
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return bail(e, "create synchronize");

  st = encode_3d(&H.tmap_w, H.w_packed, d.dtype, uint64_t(d.d_model), uint64_t(2) * d_kv,
                 uint64_t(d.n_layers), kBlockN, "packed weights");
  if (st == HCR_OK)
    st = encode_3d(&H.tmap_w_half, H.w_packed, d.dtype, uint64_t(d.d_model), uint64_t(2) * d_kv,
                   uint64_t(d.n_layers), kBlockN / 2, "packed weights (pair)");
  if (st != HCR_OK) {
    free_handle(H);
    delete h;
    return st;
  }
  // How many CTA pairs fit at once; without any, restores use single CTAs.
  H.pair_clusters = std::max(0, project_pair_clusters(d.dtype));
  cudaGetLastError();
  // The same for the pairs that decode the codec's form (hcr_restore_encoded).
  H.enc_clusters = std::max(0, project_enc_clusters(d.dtype));
  cudaGetLastError();
  // Weight-row tiles need 128-wide heads (one head per CTA of a pair).
  if (d.head_dim == 128 && H.pair_clusters > 0 &&
      encode_w5(&H.tmap_w5, H.w_packed, d.dtype, uint64_t(d.d_model),
                uint64_t(d.n_layers) * 2 * d.n_kv_heads) == HCR_OK) {
    H.swap_clusters = std::max(0, project_swap_clusters(d.dtype));
    cudaGetLastError();
  }
  g_last_error.clear();
  *out = h;
  return HCR_OK;
}

void hcr_destroy(hcr_handle* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_handle(h->impl);
  delete h;
}

size_t hcr_workspace_bytes(const hcr_handle* h, int32_t n_tokens, int32_t n_layers_in_range) {
  if (!h || n_tokens <= 0 || n_layers_in_range <= 0) return 0;
  return workspace_layout(n_tokens, n_layers_in_range, h->impl.dims.norm == HCR_NORM_LAYER)
      .total_fused;
}

#define HCR_RESTORE_ARGS                                                                         \
  RestoreArgs a{hidden,     layer_begin, layer_end,          n_req,   n_tokens,                  \
                cu_seqlens, start_pos,   block_table,        max_blocks_per_req,                 \
                k_cache,    v_cache,     layout,             workspace, workspace_bytes,         \
                static_cast<cudaStream_t>(stream)}

hcr_status hcr_restore_prepare(hcr_handle* h, const void* hidden, int32_t layer_begin,
                               int32_t layer_end, int32_t n_req, int32_t n_tokens,
                               const int32_t* cu_seqlens, const int32_t* start_pos,
                               const int32_t* block_table, int32_t max_blocks_per_req,
                               void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                               void* workspace, size_t workspace_bytes, void* stream) {
  HCR_RESTORE_ARGS;
  bool empty = false;
  hcr_status st = validate_restore(h, a, &empty);
  if (st != HCR_OK || empty) return st;
  return do_prepare(h, a);
}

hcr_status hcr_restore_project(hcr_handle* h, const void* hidden, int32_t layer_begin,
                               int32_t layer_end, int32_t n_req, int32_t n_tokens,
                               const int32_t* cu_seqlens, const int32_t* start_pos,
                               const int32_t* block_table, int32_t max_blocks_per_req,
                               void* k_cache, void* v_cache, const hcr_cache_layout* layout,
                               void* workspace, size_t workspace_bytes, void* stream) {
  HCR_RESTORE_ARGS;
  bool empty = false;
  hcr_status st = validate_restore(h, a, &empty);
  if (st != HCR_OK || empty) return st;
  return do_project(h, a);
}

hcr_status hcr_restore(hcr_handle* h, const void* hidden, int32_t layer_begin, int32_t layer_end,
                       int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                       const int32_t* start_pos, const int32_t* block_table,
                       int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                       const hcr_cache_layout* layout, void* workspace, size_t workspace_bytes,
                       void* stream) {
  NvtxRange range("hcr_restore");
  HCR_RESTORE_ARGS;
  bool empty = false;
  hcr_status st = validate_restore(h, a, &empty);
  if (st != HCR_OK || empty) return st;
  st = do_prepare(h, a);
  if (st != HCR_OK) return st;
  return do_project(h, a);
}

size_t hcr_encoded_workspace_bytes(const hcr_handle* h, int32_t n_tokens,
                                   int32_t n_layers_in_range) {
  if (!h || n_tokens <= 0 || n_layers_in_range <= 0) return 0;
  return workspace_layout(n_tokens, n_layers_in_range, h->impl.dims.norm == HCR_NORM_LAYER, true)
      .total;
}

static bool device_memory(const void* ptr) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
}

hcr_status hcr_restore_encoded(hcr_handle* h, const hcr_codec_params* params, const void* codes,
                               const void* scales, int32_t layer_begin, int32_t layer_end,
                               int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                               const int32_t* start_pos, const int32_t* block_table,
                               int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                               const hcr_cache_layout* layout, void* workspace,
                               size_t workspace_bytes, void* stream) {
  NvtxRange range("hcr_restore_encoded");
  const void* hidden = codes;
  HCR_RESTORE_ARGS;
  bool empty = false;
  hcr_status st = validate_restore(h, a, &empty, true, "codes", true);
  if (st != HCR_OK || empty) return st;
  if ((st = check_codec(h, params, layer_begin, layer_end, n_req, n_tokens, cu_seqlens,
                        &empty)) != HCR_OK)
    return st;
  if (!scales || !aligned(scales, 4))
    return fail(HCR_ERR_INVALID_ARG, "scales must be non-NULL and 4-byte aligned");
  const Handle& H = h->impl;
  if (H.dims.d_model % 16)
    return fail(HCR_ERR_UNSUPPORTED,
                "the encoded restore needs d_model a multiple of 16 (the codes' row pitch "
                "for TMA), got %d", H.dims.d_model);
  if (H.enc_clusters <= 0)
    return fail(HCR_ERR_UNSUPPORTED, "no CTA pair of the encoded projection fits on this device");
  if (!device_memory(codes) || !device_memory(scales))
    return fail(HCR_ERR_INVALID_ARG, "codes and scales must be device memory");
  CodecInput enc{};
  enc.codes = static_cast<const int8_t*>(codes);
  enc.scales = static_cast<const float*>(scales);
  enc.cu_seqlens = cu_seqlens;
  enc.n_req = n_req;
  enc.group_tokens = params->group_tokens;
  enc.n_layers_total = H.dims.n_layers;
  for (int i = 0; i < 3; ++i) enc.bins[i] = params->bins[i];
  // c * b exact for every code c in [-127, 127] and every bin: the projection
  // may then add it with one fused multiply-add
  enc.exact_products = 1;
  for (float b : params->bins)
    for (int c = -127; c <= 127; ++c)
      if (const float prod = float(c) * b; double(prod) != double(c) * double(b))
        enc.exact_products = 0;
  st = do_prepare(h, a, true, &enc);
  if (st != HCR_OK) return st;
  return do_project_enc(h, a, enc);
}

static hcr_status kv_rows(hcr_handle* h, const RestoreArgs& a, bool to_cache, const char* what) {
  NvtxRange range(to_cache ? "hcr_load_kv" : "hcr_save_kv");
  bool empty = false;
  hcr_status st = validate_restore(h, a, &empty, /*stats=*/false, what);
  if (st != HCR_OK || empty) return st;
  void* dense = nullptr;
  st = device_view(h->impl, const_cast<void*>(a.hidden), what, &dense);
  if (st != HCR_OK) return st;
  st = do_prepare(h, a, /*stats=*/false);
  if (st != HCR_OK) return st;
  const hcr_model_dims& d = h->impl.dims;
  const int64_t row = int64_t(d.n_kv_heads) * d.head_dim;
  const int64_t stride = a.layout->layer_stride_elems
                             ? a.layout->layer_stride_elems
                             : int64_t(a.layout->num_blocks) * a.layout->block_size * row;
  const WorkspaceLayout w = workspace_layout(a.n_tokens, 0, false);
  KvRowsParams p{};
  p.slot = reinterpret_cast<const int64_t*>(static_cast<uint8_t*>(a.workspace) + w.slot_off);
  p.dense = static_cast<uint4*>(dense);
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.layer_stride_vecs = stride / 8;
  p.row_vecs = int32_t(row / 8);
  p.n_tokens = a.n_tokens;
  p.n_layers = a.layer_end - a.layer_begin;
  cudaError_t e = launch_kv_rows(p, to_cache, h->impl.num_sms, a.stream);
  if (e != cudaSuccess) return cuda_fail(e, "K/V row copy launch");
  return HCR_OK;
}

hcr_status hcr_load_kv(hcr_handle* h, const void* kv, int32_t layer_begin, int32_t layer_end,
                       int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                       const int32_t* start_pos, const int32_t* block_table,
                       int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                       const hcr_cache_layout* layout, void* workspace, size_t workspace_bytes,
                       void* stream) {
  RestoreArgs a{kv,         layer_begin, layer_end,   n_req,   n_tokens,  cu_seqlens,
                start_pos,  block_table, max_blocks_per_req, k_cache, v_cache,   layout,
                workspace,  workspace_bytes, static_cast<cudaStream_t>(stream)};
  return kv_rows(h, a, /*to_cache=*/true, "kv");
}

hcr_status hcr_save_kv(hcr_handle* h, void* kv, int32_t layer_begin, int32_t layer_end,
                       int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens,
                       const int32_t* start_pos, const int32_t* block_table,
                       int32_t max_blocks_per_req, const void* k_cache, const void* v_cache,
                       const hcr_cache_layout* layout, void* workspace, size_t workspace_bytes,
                       void* stream) {
  RestoreArgs a{kv,         layer_begin, layer_end,   n_req,   n_tokens,  cu_seqlens,
                start_pos,  block_table, max_blocks_per_req, const_cast<void*>(k_cache),
                const_cast<void*>(v_cache), layout, workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream)};
  return kv_rows(h, a, /*to_cache=*/false, "kv");
}

hcr_status hcr_debug_swap_plan(int32_t n_tokens, int32_t* out) {
  if (!out) return fail(HCR_ERR_INVALID_ARG, "out is NULL");
  const SwapPlan sp = swap_plan(n_tokens);
  out[0] = sp.chunk;
  out[1] = sp.n_chunks;
  out[2] = sp.last_n;
  out[3] = sp.slot_cols;
  out[4] = sp.n_slots;
  out[5] = sp.ok ? 1 : 0;
  return HCR_OK;
}

hcr_status hcr_debug_plan(const hcr_model_dims* d, int32_t n_tokens, int32_t n_layers,
                          int32_t num_sms, int32_t pair_clusters, int32_t swap_clusters,
                          size_t workspace_bytes, int32_t* out) {
  if (!d || !out) return fail(HCR_ERR_INVALID_ARG, "dims and out must be non-NULL");
  out[0] = out[1] = 0;
  if (n_tokens <= 0 || n_layers <= 0) return HCR_OK;
  Handle H{};
  H.dims = *d;
  H.num_sms = num_sms;
  H.pair_clusters = pair_clusters;
  // as hcr_create: the weight-row tiles take 128-wide heads and need the pairs
  H.swap_clusters = (d->head_dim == 128 && pair_clusters > 0) ? swap_clusters : 0;
  out[0] = choose_variant(H, n_tokens, n_layers);
  RestoreArgs a{};
  a.layer_begin = 0;
  a.layer_end = n_layers;
  a.n_tokens = n_tokens;
  a.workspace_bytes = workspace_bytes;
  const FusedStats fs = fused_stats(H, a);
  out[1] = fs.on ? fs.layer0 : 0;
  return HCR_OK;
}

int32_t hcr_debug_fused_stats(const hcr_handle* h, int32_t n_tokens, int32_t n_layers,
                              size_t workspace_bytes) {
  if (!h || n_tokens <= 0 || n_layers <= 0) return 0;
  RestoreArgs a{};
  a.layer_begin = 0;
  a.layer_end = n_layers;
  a.n_tokens = n_tokens;
  a.workspace_bytes = workspace_bytes;
  const FusedStats fs = fused_stats(h->impl, a);
  return fs.on ? fs.layer0 : 0;
}

int32_t hcr_project_variant(const hcr_handle* h, int32_t n_tokens, int32_t n_layers) {
  if (!h || n_tokens <= 0 || n_layers <= 0) return 0;
  return choose_variant(h->impl, n_tokens, n_layers);
}

hcr_status hcr_check_device_error(hcr_handle* h, void* stream, uint32_t* flags) {
  if (flags) *flags = 0;
  if (!h) return fail(HCR_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t bits = 0;
  if ((e = cudaMemcpyAsync(&bits, h->impl.err, sizeof bits, cudaMemcpyDeviceToHost, s)) !=
      cudaSuccess)
    return cuda_fail(e, "read device error word");
  if ((e = cudaMemsetAsync(h->impl.err, 0, sizeof(uint32_t), s)) != cudaSuccess)
    return cuda_fail(e, "clear device error word");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
  if (flags) *flags = bits;
  if (bits & HCR_DEVERR_TIMEOUT) return fail(HCR_ERR_TIMEOUT, "device error bits 0x%x", bits);
  if (bits) return fail(HCR_ERR_DEVICE_BOUNDS, "device error bits 0x%x", bits);
  return HCR_OK;
}

int32_t hcr_num_sms(const hcr_handle* h) { return h ? h->impl.num_sms : 0; }

hcr_status hcr_debug_timeout_record(hcr_handle* h, void* stream, uint32_t out[6]) {
  if (!h || !out) return fail(HCR_ERR_INVALID_ARG, "handle and out must be non-NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaMemcpy(out, h->impl.err + kDiagOffset, 6 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->impl.err + kDiagOffset, 0, 6 * sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(e, "reading the timeout record");
  return HCR_OK;
}

hcr_status hcr_debug_set_variant(hcr_handle* h, int32_t variant) {
  if (!h) return fail(HCR_ERR_INVALID_ARG, "handle is NULL");
  if (variant < 0 || variant > 3)
    return fail(HCR_ERR_INVALID_ARG, "variant must be 0, 1, 2 or 3");
  if (variant == 2 && h->impl.pair_clusters <= 0)
    return fail(HCR_ERR_UNSUPPORTED, "CTA pairs cannot be co-scheduled on this device");
  if (variant == 3 && !swap_available(h->impl))
    return fail(HCR_ERR_UNSUPPORTED,
                "weight-row tiles need head_dim 128 and co-schedulable CTA pairs");
  h->impl.variant = variant;
  return HCR_OK;
}

hcr_status hcr_debug_set_stall(hcr_handle* h, int32_t enable) {
  if (!h) return fail(HCR_ERR_INVALID_ARG, "handle is NULL");
  h->impl.debug_stall = enable ? 1u : 0u;
  return HCR_OK;
}

}  // extern "C"
