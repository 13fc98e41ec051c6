// Internal declarations the restore kernels (hcr_prepare.cu, hcr_project*.cu)
// are compiled from: tiling constants, the instruction descriptor, the
// workspace layout, kernel parameters and their launchers.  Host-only
// declarations live in hcr_host.h.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/hcr.h"

namespace hcr {

// ---------------------------------------------------------------------------
// Tiling of the fused K||V projection
// ---------------------------------------------------------------------------
constexpr int kBlockM = 128;           // tokens per tile (TMEM lanes)
constexpr int kBlockN = 256;           // K||V columns per tile (TMEM columns per accumulator)
constexpr int kBlockK = 64;            // 64 x 2 bytes = one 128-byte swizzle row
constexpr int kUmmaK = 16;             // K of one tcgen05.mma kind::f16
constexpr int kStages = 4;             // TMA -> MMA ring depth, single-CTA variant (48 KB stages)
constexpr int kStagesPair = 7;         // ring depth per CTA, CTA-pair variant (32 KB stages)
constexpr int kStagesMax = 10;         // barrier slots in the pipeline state (any variant)
constexpr int kAccums = 2;             // TMEM accumulators (epilogue overlaps next mainloop)
constexpr int kTileBytesA = kBlockM * kBlockK * 2;
constexpr int kTileBytesB = kBlockN * kBlockK * 2;
constexpr int kStageBytes = kTileBytesA + kTileBytesB;
constexpr int kEpilogueWarps = 4;
constexpr int kStatsWarps = 4;         // fused norm statistics
// warp 0 TMA, warp 1 MMA, warps 2..5 epilogue, warps 6..9 statistics
constexpr int kProjectThreads = 32 * (2 + kEpilogueWarps + kStatsWarps);
constexpr int kStatsItemRows = 16;     // tokens per statistics item (one flag)
constexpr int kGroupM = 16;            // m-tiles per raster group (L2 reuse of hidden rows)
// dynamic shared memory of each variant's ring + slack to align it to 1024 bytes
constexpr size_t kSmemSingle = size_t(kStages) * kStageBytes + 1024;
constexpr size_t kSmemPair = size_t(kStagesPair) * (kTileBytesA + kTileBytesB / 2) + 1024;
static_assert(kSmemSingle <= 232448 - 512 && kSmemPair <= 232448 - 512,
              "ring does not fit the 227 KB of shared memory a CTA can use");
// Weight-row tiles (tokens as the MMA's N side, CTA pairs): a ring of stages
// of 16 KB of weights plus chunk/2 token rows (128 B each) per CTA, as many as
// fit (at most kStagesMax), 8 epilogue warps, and a 1 KB transpose buffer
// (two blocks) per epilogue warp.  Short chunks get deeper rings: in the weight-streaming
// regime the ring depth sets how many weight bytes are in flight from HBM.
constexpr int kSwapEpilogueWarps = 8;
constexpr int kSwapThreads = 64 + 32 * kSwapEpilogueWarps;
// TMEM holds accumulator slots, one MMA's N each: two slots of 256 columns (a
// tile of up to 256 tokens takes one), or for tiles of 257..320 tokens two big
// slots taken in turn plus a small slot after them (a tile takes its big slot
// and the small one).
constexpr int kSwapSlotsMax = 3;
constexpr int kSwapTmemCols = 512;     // allocated (a power of two >= the ring)
constexpr int kSwapMaxChunk = 320;     // tokens per tile (three-slot ring)
constexpr size_t kSmemSwap = 232448 - 1024;   // dynamic shared memory of the kernel
constexpr size_t kSwapStaging = size_t(kSwapEpilogueWarps) * 1024;
// per-token table of a tile for the epilogue: rstd, mean, position (4 B each)
// and slot (8 B) of up to 512 tokens
constexpr size_t kSwapTokenTable = 512 * (4 + 4 + 4 + 8);
inline int swap_stages(int chunk) {
  const size_t stage = size_t(kTileBytesA) + size_t(chunk / 2) * kBlockK * 2;
  const size_t n = (kSmemSwap - 1024 - kSwapStaging - kSwapTokenTable) / stage;
  return int(n < size_t(kStagesMax) ? n : size_t(kStagesMax));
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded pipeline waits: 2 s
// The device error word is followed, at this word offset, by a record of the
// first bounded wait that gave up: {which wait, CTA, thread, a, b, parity}.
constexpr int kDiagOffset = 8;
constexpr int kErrWords = 16;
enum : uint32_t {
  kWaitProducerEmpty = 1,   // a, b = tile, k-block
  kWaitMmaAccum = 3,        // a, b = tile, accumulator
  kWaitMmaFull = 4,         // a, b = tile, k-block
  kWaitEpilogueAccum = 7,   // a, b = tile, accumulator
  kWaitCodesEmpty = 8,      // encoded input: code producer, a, b = tile, k-block
  kWaitConvCodes = 9,       // encoded input: converter waits for codes, a, b = tile, k-block
  kWaitConvStage = 10,      // encoded input: converter waits for a free A stage
  kWaitStats = 11,          // epilogue waits for fused statistics, a, b = tile, item
};

// tcgen05 instruction descriptor for kind::f16, fp32 accumulate, both
// operands K-major: D format F32 (1) in bits [4,6), A and B format in
// [7,10) and [10,13) (F16 = 0, BF16 = 1), N >> 3 in [17,23), M >> 4 in [24,29).
constexpr uint32_t make_idesc_f16(int dtype, int m, int n) {
  return (1u << 4) | (uint32_t(dtype == HCR_DTYPE_BF16 ? 1 : 0) << 7) |
         (uint32_t(dtype == HCR_DTYPE_BF16 ? 1 : 0) << 10) | (uint32_t(n >> 3) << 17) |
         (uint32_t(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned)
// ---------------------------------------------------------------------------
struct WorkspaceLayout {
  size_t slot_off, pos_off, rstd_off, mean_off, anchor_off, total;
  // After `total` (the minimum), room for the fused statistics' flags, one
  // int32 per kStatsItemRows tokens per layer: a workspace of total_fused
  // bytes lets the token-row projection compute most layers' statistics.
  size_t flags_off, total_fused;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// encoded: a restore from the codec's form also keeps each token's group
// anchor (int32 [T]) after the statistics.
inline WorkspaceLayout workspace_layout(int64_t n_tokens, int64_t n_layers, bool layer_norm,
                                        bool encoded = false) {
  WorkspaceLayout w{};
  size_t off = 0;
  w.slot_off = off;
  off = align_up(off + size_t(n_tokens) * 8, 256);
  w.pos_off = off;
  off = align_up(off + size_t(n_tokens) * 4, 256);
  w.rstd_off = off;
  off = align_up(off + size_t(n_tokens) * size_t(n_layers) * 4, 256);
  w.mean_off = off;
  if (layer_norm) off = align_up(off + size_t(n_tokens) * size_t(n_layers) * 4, 256);
  w.anchor_off = off;
  if (encoded) off = align_up(off + size_t(n_tokens) * 4, 256);
  w.total = off;
  w.flags_off = off;
  if (!encoded && n_layers > 0)
    off = align_up(off + size_t(n_layers) *
                             size_t((n_tokens + kStatsItemRows - 1) / kStatsItemRows) * 4,
                   256);
  w.total_fused = off;
  return w;
}

// ---------------------------------------------------------------------------
// Kernel parameters
// ---------------------------------------------------------------------------
// The codec's encoded hidden states as the restore kernels read them
// directly (hcr_restore_encoded): int8 codes and per-anchor-row scales of the
// call's first layer, the request table that forms the anchor groups, the
// group anchor of every token, and the layer-third bins.
// Rows of codes a k-block's code stage holds before the tile's own rows (the
// group anchors of the tile's first rows), and the rows it holds in all: the
// tile's 128, the halo, and one more so that the stage's four 16-code column
// chunks lie 145 rows of 16 bytes apart (an odd pitch, so that rows four apart
// fall in different bank groups).
constexpr int kEncCodeHalo = 16;
constexpr int kEncCodeRows = 128 + kEncCodeHalo + 1;

struct CodecInput {
  const int8_t* codes;       // [Lr][T][d]
  const float* scales;       // [Lr][T]
  const int32_t* cu_seqlens;   // [n_req + 1]
  int32_t* anchor;           // [T] workspace: token of each token's group anchor, -1 for a
                             // token in no request (written by the prepare kernel)
  int32_t n_req, group_tokens, n_layers_total;
  float bins[3];
  int32_t exact_products;    // every code times every bin is exact in binary32
};

struct PrepareParams {
  // A0: placement
  const int32_t* cu_seqlens;
  const int32_t* start_pos;
  const int32_t* block_table;
  int32_t n_req, n_tokens, max_blocks, num_blocks, block_size, max_position, check_position;
  int64_t* slot;   // [T]; -1 marks a row that must not be written
  int32_t* pos;    // [T]
  // A1: norm statistics of rows (layer, token)
  const void* hidden;  // [Lr][T][d]
  int32_t n_layers, d_model, layer_norm, dtype;
  float eps;
  float* rstd;   // [Lr][T]
  float* mean;   // [Lr][T] (LayerNorm only)
  uint32_t* err;
  int32_t slot_blocks;  // leading blocks of the grid that do placement
  int32_t skip_placement;   // statistics only (the slot map is written elsewhere)
  int32_t layer_begin;  // model layer of hidden layer 0 (codec bins)
  CodecInput enc;       // codes != nullptr: statistics of the decoded rows
  int32_t* zero_flags;  // the placement blocks set these n_zero_flags words to 0
  int64_t n_zero_flags;
};

struct ProjectParams {
  int32_t n_tokens, d_model, n_cols, d_kv, head_dim, n_layers, layer_begin;
  int32_t m_tiles, n_tiles, k_blocks;
  // CTA pairs only: the last m-tile of each layer holds at most 128 rows and
  // runs as an M=128 pair tile (64 rows per CTA) instead of a 256-row one.
  int32_t half_tail;
  int64_t num_tiles;
  int32_t layer_norm, has_bias, rope, dtype;
  const int64_t* slot;
  const int32_t* pos;
  const float* rstd;
  const float* mean;
  const float* col_sum;   // base of layer layer_begin
  const float* col_bias;  // base of layer layer_begin
  const float2* rope_tab;
  void* k_cache;          // base of layer layer_begin
  void* v_cache;
  int64_t layer_stride;   // elements
  int32_t row_elems;      // n_kv_heads * head_dim
  uint32_t* err;
  uint32_t debug_stall;
  // Weight-row tiles only: tiles are (layer, head pair, token chunk); chunks
  // hold `chunk` tokens (a multiple of 16, at most kSwapMaxChunk) except the
  // last, which holds last_n (a multiple of 16, at most chunk).
  int32_t chunk, n_chunks, last_n, head_pairs;
  int32_t split_tail;   // the launch's last split_tail tiles run as two half-chunk units
  int32_t stages;   // ring depth (swap_stages(chunk))
  int32_t slot_cols, n_slots;   // TMEM slots: 2 x 256, or 2 big of slot_cols + 1 small
  // Token-row kernels only, fused norm statistics (stats_flags != nullptr):
  // the kernel's statistics warps write rstd (and mean) of layers
  // [stats_layer0, n_layers) from hidden_rows, kStatsItemRows tokens per item,
  // and set stats_flags[l * stats_items + j] to 1 once item j of layer l is
  // written; an epilogue waits for the items of its rows first.  Layers below
  // stats_layer0 come from the prepare kernel.
  const void* hidden_rows;   // [n_layers][n_tokens][d_model]
  float eps;
  int32_t stats_layer0, stats_items;
  int32_t* stats_flags;
};

// Launchers (return cudaGetLastError() of the launch).
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t s);
// tmap_h64: the hidden states with 64-row boxes, read by half tail tiles.
cudaError_t launch_project(const CUtensorMap& tmap_h, const CUtensorMap& tmap_h64,
                           const CUtensorMap& tmap_w, const ProjectParams& p, int grid, bool pair,
                           cudaStream_t s);
// Co-resident clusters of the CTA-pair variant on the current device (< 0 on error).
int project_pair_clusters(int dtype);
// Weight-row tiles: tmap_h has boxes of chunk/2 token rows; tmap_w5 is the 5-D
// view of the packed weights (box = one head's 128 rows, reordered so that
// each rotate-half pair shares a thread in the epilogue).  grid is even.
cudaError_t launch_project_swap(const CUtensorMap& tmap_h, const CUtensorMap& tmap_w5,
                                const ProjectParams& p, int grid, cudaStream_t s);
int project_swap_clusters(int dtype);
// Token-row CTA pairs whose A operand is decoded from the codec's int8 codes
// in shared memory: tmap_c is the codes' 3-D map (d, T, Lr) with 128-row
// boxes, tmap_w the pair's half-tile weight map.  grid is even.
cudaError_t launch_project_enc(const CUtensorMap& tmap_c, const CUtensorMap& tmap_w,
                               const ProjectParams& p, const CodecInput& e, int grid,
                               cudaStream_t s);
int project_enc_clusters(int dtype);
cudaError_t launch_pack_weights(const void* w_k, const void* w_v, const void* gamma, void* dst,
                                int d_kv, int d, int dtype, cudaStream_t s);
cudaError_t launch_column_constants(const void* w_packed, const void* w_k, const void* w_v,
                                    const void* beta, const void* b_k, const void* b_v,
                                    float* col_sum, float* col_bias, int d_kv, int d, int dtype,
                                    int layer_norm, int has_bias, cudaStream_t s);

}  // namespace hcr

