// Tile order and epilogue of the token-row projection tiles, shared by the
// kernel that stages hidden states with TMA (hcr_project.cu) and the one that
// decodes them from the codec's int8 form in shared memory
// (hcr_project_enc.cu).  Both produce the same accumulator for a tile, so
// the same epilogue finishes it:
//     RMS:  x = rstd_t * acc                        (+ b_j if the model has K/V bias)
//     LN:   x = rstd_t * (acc - mean_t * colsum_j) + (W beta + b)_j
//     K columns: rotate-half RoPE at the token's absolute position
//     cast to the storage type and 16-byte stores into the token's cache slot.
#pragma once

#include "hcr_internal.h"
#include "hcr_pipe.cuh"
#include "ptx.cuh"

namespace hcr {
namespace pipe {

struct TileCoord {
  int l, m, n;
};

// Tile order: layer-major; inside a layer, groups of kGroupM m-tiles sweep
// all n-tiles with m fastest, so the concurrently running CTAs share a few
// weight tiles and a bounded set of hidden rows in L2.
__device__ __forceinline__ TileCoord tile_coord(int64_t tile, const ProjectParams& p) {
  const int64_t per_layer = int64_t(p.m_tiles) * p.n_tiles;
  TileCoord c;
  c.l = int(tile / per_layer);
  const int r = int(tile - int64_t(c.l) * per_layer);
  const int group_tiles = kGroupM * p.n_tiles;
  const int g = r / group_tiles;
  const int within = r - g * group_tiles;
  const int rows = min(kGroupM, p.m_tiles - g * kGroupM);
  c.m = g * kGroupM + within % rows;
  c.n = within / rows;
  return c;
}

// Tile of round k for scheduling unit `unit` of `units` (a CTA or a CTA
// pair of the persistent grid): round k covers the tiles [k units,
// (k + 1) units), the set a plain stride would give it, with the unit's place
// in it rotated by k.  With a plain stride a unit keeps its place in every
// round, so when units is a multiple of the layer's m-tiles (76 pairs and 4
// m-tiles at 794 tokens) every tile a unit gets has the same m: the units
// that get the cheap half tail tiles idle while the others run only full
// tiles.  Rotating gives each unit every place in turn.
__device__ __forceinline__ int64_t round_tile(int64_t k, int64_t unit, int64_t units) {
  return k * units + (unit + k) % units;
}

// Token of TMEM lane `row` (0..127) of this CTA in tile c: a full tile's
// lane is the CTA's token row; a half tail tile's CTA holds 64 rows, each in
// two lanes (row % 64).
template <bool PAIR, bool HT>
__device__ __forceinline__ int tile_token(const ProjectParams& p, const TileCoord& c,
                                          uint32_t rank, int row) {
  constexpr int kTileM = PAIR ? 2 * kBlockM : kBlockM;
  const bool half_tile = HT && c.m == p.m_tiles - 1;
  return c.m * kTileM +
         (half_tile ? int(rank) * (kBlockM / 2) + (row & 63) : int(rank) * kBlockM + row);
}

// Epilogue of one finished tile, run by each of the four epilogue warps of a
// CTA on its 32-lane TMEM quadrant `quad` (tacc: the accumulator's TMEM
// address with the quadrant's lane offset).
//
// Full tile: TMEM lane `row` holds this CTA's token row `row`, all 256
// columns.  Half tail tile (pairs, M=128): lane L holds row L % 64 of this
// CTA's 64 rows, for the tile's columns 128 * (L / 64) .. +127, stored at
// TMEM columns 0..127 (the tcgen05 layout of a cta_group::2 M=128 MMA).
template <int DT, bool PAIR, bool HT>
__device__ __forceinline__ void token_tile_epilogue(const ProjectParams& p, const TileCoord& c,
                                                    uint32_t rank, int quad, int lane,
                                                    uint32_t tacc) {
  const int row = quad * 32 + lane;   // token row within this CTA's 128 rows
  const int half = p.head_dim >> 1;
  const bool half_tile = HT && c.m == p.m_tiles - 1;
  const int col_lo = half_tile ? (row >> 6) * (kBlockN / 2) : 0;
  const int col_hi = half_tile ? col_lo + kBlockN / 2 : kBlockN;
  const int t = tile_token<PAIR, HT>(p, c, rank, row);
  bool valid = t < p.n_tokens;
  int64_t slot = -1;
  int pos = 0;
  float rstd = 0.f, mean = 0.f;
  if (valid) {
    slot = __ldg(p.slot + t);
    pos = __ldg(p.pos + t);
    const int64_t srow = int64_t(c.l) * p.n_tokens + t;
    // written in this kernel by other CTAs when the statistics are fused:
    // read through L2, after the wait for their flag
    rstd = __ldcg(p.rstd + srow);
    if (p.layer_norm) mean = __ldcg(p.mean + srow);
  }
  valid = valid && slot >= 0;
  const float* csum = p.layer_norm ? p.col_sum + int64_t(c.l) * p.n_cols : nullptr;
  const float* cbias = p.has_bias ? p.col_bias + int64_t(c.l) * p.n_cols : nullptr;

  for (int h0 = col_lo; h0 < col_hi; h0 += p.head_dim) {   // warp-uniform bounds
    const int col0 = c.n * kBlockN + h0;
    if (col0 >= p.n_cols) break;   // ragged last n-tile (warp-uniform)
    const bool is_k = col0 < p.d_kv;
    const int head = (is_k ? col0 : col0 - p.d_kv) / p.head_dim;
    uint16_t* dst = nullptr;
    if (valid) {
      uint16_t* base = reinterpret_cast<uint16_t*>(is_k ? p.k_cache : p.v_cache);
      dst = base + int64_t(c.l) * p.layer_stride + slot * int64_t(p.row_elems) +
            int64_t(head) * p.head_dim;
    }
    const bool do_rope = is_k && p.rope;
    for (int j = 0; j < half; j += 16) {
      uint32_t ra[16], rb[16];
      ptx::tmem_ld16(tacc + uint32_t(h0 - col_lo + j), ra);
      ptx::tmem_ld16(tacc + uint32_t(h0 - col_lo + half + j), rb);
      ptx::tmem_ld_wait();
      float a[16], b[16];
      const int ca = col0 + j, cb = col0 + half + j;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool ln = p.layer_norm;
        float xa = norm_scale(__uint_as_float(ra[i]), rstd, mean,
                              ln ? __ldg(csum + ca + i) : 0.f, ln);
        float xb = norm_scale(__uint_as_float(rb[i]), rstd, mean,
                              ln ? __ldg(csum + cb + i) : 0.f, ln);
        if (cbias) {
          xa = __fadd_rn(xa, __ldg(cbias + ca + i));
          xb = __fadd_rn(xb, __ldg(cbias + cb + i));
        }
        a[i] = xa;
        b[i] = xb;
      }
      if (do_rope && valid) {
        const float4* tab =
            reinterpret_cast<const float4*>(p.rope_tab + int64_t(pos) * half + j);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 cs = __ldg(tab + i);   // (cos, sin) of pairs j+2i, j+2i+1
          rope_pair(a[2 * i], b[2 * i], cs.x, cs.y);
          rope_pair(a[2 * i + 1], b[2 * i + 1], cs.z, cs.w);
        }
      }
      if (valid) {
        store16<DT>(dst + j, a);
        store16<DT>(dst + half + j, b);
      }
    }
  }
}

}  // namespace pipe
}  // namespace hcr
