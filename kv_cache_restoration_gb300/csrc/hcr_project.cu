// The fused K||V projection of a restore (HCache episode, "Fast State
// Restoration for Evicted LLM KV Caches", cue 14: K = W_k H, V = W_v H).
//
// One persistent kernel per restore call covers every (layer, m-tile,
// n-tile) of
//     acc[t][j] = sum_i H_l[t][i] * W'_l[j][i],   W'_l = [W_k; W_v] diag(gamma)
// on the 5th-generation tensor cores, and finishes each tile in registers:
//     RMS:  x = rstd_t * acc                        (+ b_j if the model has K/V bias)
//     LN:   x = rstd_t * (acc - mean_t * colsum_j) + (W beta + b)_j
//     K columns: rotate-half RoPE at the token's absolute position
//     cast to bf16/fp16 (round to nearest even) and 16-byte stores straight
//     into the paged cache slot of the token; no intermediate K/V tensor.
//
// Ragged multi-request batches (cue 20: project all tokens of a layer
// together so the GEMM shape stays regular) are handled by concatenating
// every request's tokens along M: tiles are full except the very last one,
// whatever the request lengths.
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0      one lane issues TMA loads of hidden and weight tiles into a
//               shared-memory ring;
//   warp 1      allocates TMEM (2 accumulators x 256 fp32 columns) and one
//               lane issues tcgen05.mma (K=16) for each stage;
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator (each warp
//               owns one 32-lane TMEM quadrant = 32 tokens), overlapping the
//               MMA of the next tile into the other accumulator;
//   warps 6..9  when the host fuses the norm statistics into the call: the
//               statistics of layers the prepare kernel left out, 16 tokens
//               per item, each item's flag set once written; an epilogue
//               waits (bounded) for its rows' flags.  Otherwise idle.
// Two variants: single CTAs with 128x256 tiles (cta_group::1, 4 stages of
// 48 KB), and CTA pairs with 256x256 tiles (cta_group::2, 7 stages of 32 KB
// per CTA).  The pair halves each SM's share of the weight tile, which cuts
// shared-memory traffic per MMA by a third; the host picks the variant by
// token count, width and call size.  A pair launch whose layers end in at most
// 128 rows runs that last m-tile as an M=128 pair tile (64 rows per CTA), so
// the pair pads no more rows than single CTAs do.
// Every pipeline wait is bounded (kWaitLimitNs); on expiry the kernel sets
// HCR_DEVERR_TIMEOUT, stops all roles, drains in-flight copies and MMAs with
// a bounded wait, frees TMEM and returns.  The tile order and the epilogue
// are in hcr_epilogue.cuh, shared with the kernel that decodes the codec's
// int8 form into its A operand (hcr_project_enc.cu).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hcr_epilogue.cuh"
#include "hcr_stats.cuh"
#include "hcr_internal.h"
#include "hcr_pipe.cuh"
#include "ptx.cuh"

namespace hcr {
namespace {

using namespace pipe;

// Per-variant tiling.  Single: one CTA computes a 128x256 tile with
// cta_group::1.  Pair: a cluster of two CTAs computes a 256x256 tile with one
// cta_group::2 MMA stream; each CTA stages its own 128 rows of A and half of
// B (128 rows), so a stage is 32 KB instead of 48 KB and seven fit.
template <bool PAIR>
struct Tiling {
  static constexpr int kStages = PAIR ? ::hcr::kStagesPair : ::hcr::kStages;
  static constexpr int kRowsB = PAIR ? kBlockN / 2 : kBlockN;   // B rows staged per CTA
  static constexpr int kTileM = PAIR ? 2 * kBlockM : kBlockM;   // token rows per tile
  static constexpr int kBytesB = kRowsB * kBlockK * 2;
  static constexpr int kStageBytes = kTileBytesA + kBytesB;
};

// HT (pairs only): each layer's last m-tile is a half tail tile (M=128 across
// the pair).  A separate instantiation, so the common kernel carries none of
// its checks.
template <int DT, bool PAIR, bool HT>
__global__ void __launch_bounds__(kProjectThreads, 1)
    project_kernel(const __grid_constant__ CUtensorMap tmap_h,
                   const __grid_constant__ CUtensorMap tmap_h64,
                   const __grid_constant__ CUtensorMap tmap_w, const ProjectParams p) {
  using Tl = Tiling<PAIR>;
  constexpr int S = Tl::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ PipeState ps;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;                                   // S x [128][64]
  uint8_t* smem_b = smem + size_t(S) * kTileBytesA;         // S x [kRowsB][64]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int32_t* abort = &ps.abort;
  // In a pair, CTA rank 0 (the leader) issues every MMA for both CTAs.
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int64_t unit = PAIR ? int64_t(blockIdx.x >> 1) : int64_t(blockIdx.x);
  const int64_t units = PAIR ? int64_t(gridDim.x >> 1) : int64_t(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_u32(&ps.full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&ps.empty[s]), 1);
    }
    for (int a = 0; a < kAccums; ++a) {
      ptx::mbar_init(ptx::smem_u32(&ps.tfull[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&ps.tempty[a]), PAIR ? 2 * kEpilogueWarps : kEpilogueWarps);
    }
    ptx::mbar_init(ptx::smem_u32(&ps.drain), 1);
    ps.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(ptx::smem_u32(&ps.tmem_base), kAccums * kBlockN);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(&ps.tmem_base), kAccums * kBlockN);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();   // peer barriers initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = ps.tmem_base;

  int64_t issued = 0;   // TMA stages armed by the producer (warp 0, lane 0)
  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_h);
      ptx::tma_prefetch_desc(&tmap_w);
      if (HT) ptx::tma_prefetch_desc(&tmap_h64);
      // A weight tile is read by every m-tile of its raster group: with several
      // m-tiles keep it in L2 ahead of other data (with one it is streamed
      // once and loaded without a hint).
      const bool reuse_w = p.m_tiles > 1;
      const uint64_t keep = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t rnd = 0, tile; ok && (tile = round_tile(rnd, unit, units)) < p.num_tiles; ++rnd) {
        const TileCoord c = tile_coord(tile, p);
        // a half tail tile stages 64 rows of A per CTA (M=128 across the pair)
        const bool half_tile = HT && c.m == p.m_tiles - 1;
        const int row_a = c.m * Tl::kTileM + int(rank) * (half_tile ? kBlockM / 2 : kBlockM);
        const int row_b = c.n * kBlockN + int(rank) * Tl::kRowsB;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(ptx::smem_u32(&ps.empty[stage]), phase ^ 1u, abort, p, kWaitProducerEmpty,
                          uint32_t(tile), uint32_t(kb))) {
            ok = false;
            break;
          }
          const uint32_t full = ptx::smem_u32(&ps.full[stage]);
          const uint32_t dst_a = ptx::smem_u32(smem_a + size_t(stage) * kTileBytesA);
          const uint32_t dst_b = ptx::smem_u32(smem_b + size_t(stage) * Tl::kBytesB);
          if constexpr (PAIR) {
            // both CTAs' bytes complete on the leader's barrier; only the
            // leader arrives (with the pair's total byte count)
            if (leader)
              ptx::mbar_arrive_expect_tx(
                  full, half_tile ? 2 * (kTileBytesA / 2 + Tl::kBytesB) : 2 * Tl::kStageBytes);
            const uint32_t full_leader = ptx::mapa_shared(full, 0);
            if (!(p.debug_stall && issued == 0)) {
              ptx::tma_load_3d_pair(dst_a, half_tile ? &tmap_h64 : &tmap_h, full_leader,
                                    kb * kBlockK, row_a, c.l);
              if (reuse_w)
                ptx::tma_load_3d_pair_hint(dst_b, &tmap_w, full_leader, kb * kBlockK, row_b,
                                           p.layer_begin + c.l, keep);
              else
                ptx::tma_load_3d_pair(dst_b, &tmap_w, full_leader, kb * kBlockK, row_b,
                                      p.layer_begin + c.l);
            }
          } else {
            ptx::mbar_arrive_expect_tx(full, Tl::kStageBytes);
            if (!(p.debug_stall && issued == 0)) {
              ptx::tma_load_3d(dst_a, &tmap_h, full, kb * kBlockK, row_a, c.l);
              if (reuse_w)
                ptx::tma_load_3d_hint(dst_b, &tmap_w, full, kb * kBlockK, row_b,
                                      p.layer_begin + c.l, keep);
              else
                ptx::tma_load_3d(dst_b, &tmap_w, full, kb * kBlockK, row_b, p.layer_begin + c.l);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = make_idesc_f16(DT, Tl::kTileM, kBlockN);
      constexpr uint32_t idesc_half = make_idesc_f16(DT, kBlockM, kBlockN);   // pairs, M=128
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t rnd = 0, tile; ok && (tile = round_tile(rnd, unit, units)) < p.num_tiles; ++rnd) {
        if (!wait_phase(ptx::smem_u32(&ps.tempty[acc]), acc_phase ^ 1u, abort, p, kWaitMmaAccum,
                        uint32_t(tile), uint32_t(acc)))
          break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * kBlockN);
        const uint32_t id =
            (HT && tile_coord(tile, p).m == p.m_tiles - 1) ? idesc_half : idesc;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(ptx::smem_u32(&ps.full[stage]), phase, abort, p, kWaitMmaFull,
                          uint32_t(tile), uint32_t(kb))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smem_a + size_t(stage) * kTileBytesA);
          const uint32_t b0 = ptx::smem_u32(smem_b + size_t(stage) * Tl::kBytesB);
#pragma unroll
          for (int k = 0; k < kBlockK / kUmmaK; ++k) {
            const uint64_t da = ptx::sw128_kmajor_desc(a0 + k * kUmmaK * 2);
            const uint64_t db = ptx::sw128_kmajor_desc(b0 + k * kUmmaK * 2);
            if constexpr (PAIR)
              ptx::mma_f16_pair(d_tmem, da, db, id, (kb | k) != 0 ? 1u : 0u);
            else
              ptx::mma_f16(d_tmem, da, db, id, (kb | k) != 0 ? 1u : 0u);
          }
          if constexpr (PAIR)
            ptx::mma_commit_pair_multicast(ptx::smem_u32(&ps.empty[stage]), 0x3);
          else
            ptx::mma_commit(ptx::smem_u32(&ps.empty[stage]));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&ps.tfull[acc]), 0x3);
        else
          ptx::mma_commit(ptx::smem_u32(&ps.tfull[acc]));
        if (++acc == kAccums) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA this thread issued has completed once `drain` flips.
      if constexpr (PAIR)
        ptx::mma_commit_pair_multicast(ptx::smem_u32(&ps.drain), 0x1);
      else
        ptx::mma_commit(ptx::smem_u32(&ps.drain));
      drain_wait(ptx::smem_u32(&ps.drain), 0);
    }
  } else if (warp < 2 + kEpilogueWarps) {
    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;               // TMEM lanes [32*quad, 32*quad+32)
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t rnd = 0, tile; (tile = round_tile(rnd, unit, units)) < p.num_tiles; ++rnd) {
      const TileCoord c = tile_coord(tile, p);
      int ok = 0;
      if (lane == 0)
        ok = wait_phase(ptx::smem_u32(&ps.tfull[acc]), acc_phase, abort, p, kWaitEpilogueAccum,
                        uint32_t(tile), uint32_t(acc));
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (p.stats_flags && c.l >= p.stats_layer0) {
        // this lane's row statistics come from a statistics item of this
        // kernel: wait (bounded) until its flag is set
        const int t = tile_token<PAIR, HT>(p, c, rank, quad * 32 + lane);
        const int item = t / kStatsItemRows;
        const bool got = t >= p.n_tokens ||
                         wait_flag(p.stats_flags + int64_t(c.l) * p.stats_items + item, abort, p,
                                   kWaitStats, uint32_t(tile), uint32_t(item));
        if (!__all_sync(0xffffffffu, got)) break;
      }
      ptx::tc_fence_after();

      token_tile_epilogue<DT, PAIR, HT>(
          p, c, rank, quad, lane,
          tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * kBlockN));
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)   // the leader's MMA reuses the accumulator in both CTAs
          ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&ps.tempty[acc]), 0));
        else
          ptx::mbar_arrive(ptx::smem_u32(&ps.tempty[acc]));
      }
      if (++acc == kAccums) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (p.stats_flags) {
    // ------------------------------------------------------------- statistics
    // Norm statistics of layers [stats_layer0, n_layers), kStatsItemRows
    // tokens per item, items in layer order over every statistics warp of the
    // grid; each item's flag is set once its rows are written.  These warps
    // wait for nothing.
    PrepareParams sp{};
    sp.hidden = p.hidden_rows;
    sp.n_tokens = p.n_tokens;
    sp.d_model = p.d_model;
    sp.layer_norm = p.layer_norm;
    sp.dtype = p.dtype;
    sp.eps = p.eps;
    sp.rstd = const_cast<float*>(p.rstd);
    sp.mean = const_cast<float*>(p.mean);
    const int64_t gw = int64_t(blockIdx.x) * kStatsWarps + (warp - 2 - kEpilogueWarps);
    const int64_t nw = int64_t(gridDim.x) * kStatsWarps;
    const int64_t items = int64_t(p.n_layers - p.stats_layer0) * p.stats_items;
    for (int64_t it = gw; it < items && !*abort; it += nw) {
      const int l = p.stats_layer0 + int(it / p.stats_items);
      const int j = int(it - int64_t(l - p.stats_layer0) * p.stats_items);
      const int t1 = min((j + 1) * kStatsItemRows, p.n_tokens);
      for (int t = j * kStatsItemRows; t < t1; ++t)
        stats::row_stats<DT, false>(sp, int64_t(l) * p.n_tokens + t, lane);
      __syncwarp();
      if (lane == 0)   // after lane 0's own writes of the item's statistics
        ptx::st_release_gpu(p.stats_flags + int64_t(l) * p.stats_items + j, 1);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // Both CTAs have left their roles.  The leader's full barriers count both
    // CTAs' loads, so the leader waits (bounded; immediate unless a role gave
    // up) for its last S stages before either CTA releases its memory.
    ptx::cluster_sync();
    if (leader && warp == 0 && lane == 0) {
      const int64_t first = issued > S ? issued - S : 0;
      for (int64_t i = first; i < issued; ++i)
        drain_wait(ptx::smem_u32(&ps.full[i % S]), uint32_t((i / S) & 1));
    }
    ptx::cluster_sync();
    if (warp == 1) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc_pair(tmem_base, kAccums * kBlockN);
    }
  } else {
    if (*abort) {
      // Some role gave up: loads the producer armed may still be landing in
      // shared memory.  They are among its last S; wait for each (bounded)
      // before the CTA releases its memory.
      if (warp == 0 && lane == 0) {
        const int64_t first = issued > S ? issued - S : 0;
        for (int64_t i = first; i < issued; ++i)
          drain_wait(ptx::smem_u32(&ps.full[i % S]), uint32_t((i / S) & 1));
      }
      __syncthreads();
    }
    if (warp == 1) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc(tmem_base, kAccums * kBlockN);
    }
  }
}

template <int DT, bool PAIR, bool HT = false>
cudaError_t launch_variant(const CUtensorMap& tmap_h, const CUtensorMap& tmap_h64,
                           const CUtensorMap& tmap_w, const ProjectParams& p, int grid,
                           cudaStream_t s) {
  auto kernel = project_kernel<DT, PAIR, HT>;
  constexpr size_t smem = PAIR ? kSmemPair : kSmemSingle;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kProjectThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, tmap_h, tmap_h64, tmap_w, p);
}

template <int DT>
int max_pair_clusters() {
  auto kernel = project_kernel<DT, true, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemPair)) != cudaSuccess)
    return -1;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(sms & ~1));
  cfg.blockDim = dim3(kProjectThreads);
  cfg.dynamicSmemBytes = kSmemPair;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return -1;
  return n;
}

}  // namespace

cudaError_t launch_project(const CUtensorMap& tmap_h, const CUtensorMap& tmap_h64,
                           const CUtensorMap& tmap_w, const ProjectParams& p, int grid, bool pair,
                           cudaStream_t s) {
  const bool ht = pair && p.half_tail;
  if (p.dtype == HCR_DTYPE_BF16) {
    if (ht) return launch_variant<HCR_DTYPE_BF16, true, true>(tmap_h, tmap_h64, tmap_w, p, grid, s);
    return pair ? launch_variant<HCR_DTYPE_BF16, true>(tmap_h, tmap_h64, tmap_w, p, grid, s)
                : launch_variant<HCR_DTYPE_BF16, false>(tmap_h, tmap_h64, tmap_w, p, grid, s);
  }
  if (ht) return launch_variant<HCR_DTYPE_FP16, true, true>(tmap_h, tmap_h64, tmap_w, p, grid, s);
  return pair ? launch_variant<HCR_DTYPE_FP16, true>(tmap_h, tmap_h64, tmap_w, p, grid, s)
              : launch_variant<HCR_DTYPE_FP16, false>(tmap_h, tmap_h64, tmap_w, p, grid, s);
}

int project_pair_clusters(int dtype) {
  return dtype == HCR_DTYPE_BF16 ? max_pair_clusters<HCR_DTYPE_BF16>()
                                 : max_pair_clusters<HCR_DTYPE_FP16>();
}

}  // namespace hcr
