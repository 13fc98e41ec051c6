// The fused K||V projection from the codec's encoded hidden states: the
// token-row CTA-pair kernel (256x256 tiles, cta_group::2) whose A operand is
// decoded in the kernel instead of loaded.
//
// The HCache episode ("Fast State Restoration for Evicted LLM KV Caches",
// cues 30 and 32) proposes compressing the saved hidden states the way
// CacheGen compresses KV caches (CacheGen review, section 核心方法: groups of
// 10 tokens, an 8-bit anchor per group, the other tokens as quantised deltas
// from it).  Here the restore reads that form directly: TMA brings each
// k-block's int8 codes (half the bytes of the hidden states) into shared
// memory, and converter warps write the bf16/fp16 A stage the MMA reads, in
// the 128-byte-swizzled K-major layout a TMA load would have produced:
//     anchor row:  q * s                     (its codes, its scale)
//     other rows:  q_anchor * s + c * b       (its codes c, the layer's bin b)
// each one binary32 operation, then one rounding to the storage type, so the
// operand, and therefore every cache element, is bit-identical to restoring
// from hcr_decode_hidden's output.  The norm statistics come from the prepare
// kernel decoding the same rows; the epilogue is the token-row kernel's.
//
// On GB300 this restore is slower than the decode kernel followed by the
// token-row kernel (8.3 against 5.8 ms for the Llama2-7B-shaped step): every A
// tile is decoded again for each of the 32 n-tiles, and the k-block's period
// follows the converter warps' latency on it.  The layer-pipelined encoded
// restore therefore decodes first.
//
// Warp roles (480 threads, one CTA per SM, clusters of two):
//   warp 0       one lane loads the pair's weight half-tiles (TMA, completion
//                on the leader's stage barrier, as in the token-row kernel);
//   warp 1       TMEM (2 x 256 columns) and, in the leader, the MMA issuer;
//   warps 2..5   epilogue (one 32-lane TMEM quadrant each);
//   warp 6       one lane loads the codes of each k-block (TMA, 145 rows x 64
//                codes, stored as four 16-code column chunks);
//   warps 7..14  converters, in two groups that take alternate k-blocks;
//                each warp decodes 32 rows, a lane 16 elements (two 16-byte
//                chunks of the A row) of a run of 4 consecutive rows,
//                carrying the group anchor's decoded value from row to row.
// A stage (decoded A and weights) is full when the leader's barrier has
// counted both CTAs' weight bytes and an arrival from every converter warp of
// the group that decoded it, in both CTAs (each after a proxy fence that makes
// its shared-memory writes visible to the tensor core).  A code stage also
// holds the 16 rows before the tile, where the group anchors of its first rows
// lie; an anchor further back (groups of more than 17 tokens) is read from
// global memory.  Every wait is bounded as in the other projection kernels.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hcr_decode.cuh"
#include "hcr_epilogue.cuh"
#include "hcr_internal.h"
#include "hcr_pipe.cuh"
#include "ptx.cuh"

namespace hcr {
namespace {

using namespace pipe;

constexpr int kEncStages = 5;        // stages of decoded A + weights, 32 KB per CTA
constexpr int kEncCodeStages = 5;    // code stages, 9 KB
constexpr int kEncCodeWarp = 6;
constexpr int kEncConvWarp0 = 7;
constexpr int kEncConvWarps = 8;
constexpr uint32_t kSleepNs = 100000;   // longest sleep of one barrier probe (100 us)
constexpr int kConvGroups = 2;       // k-blocks converted at once
constexpr int kGroupWarps = kEncConvWarps / kConvGroups;
constexpr int kGroupRows = kBlockM / kGroupWarps;   // tile rows per converter warp
constexpr int kRunRows = 4;          // consecutive rows of a converter lane's run
constexpr int kEncThreads = 32 * (kEncConvWarp0 + kEncConvWarps);
// A code stage holds the tile's rows and the kCodeHalo rows before them, so a
// group anchor up to kCodeHalo rows before the tile is in shared memory too.
constexpr int kCodeHalo = kEncCodeHalo;
constexpr int kCodeChunkBytes = kEncCodeRows * 16;   // one 16-code column chunk of the rows
constexpr int kCodeBytes = 4 * kCodeChunkBytes;      // the box: 4 chunks x 145 rows x 16 codes
constexpr int kCodeStageBytes = (kCodeBytes + 127) / 128 * 128;   // stage stride
constexpr int kPairBytesB = kTileBytesB / 2;       // a CTA's half of the weight tile
constexpr size_t kSmemEnc = size_t(kEncStages) * (kTileBytesA + kPairBytesB) +
                            size_t(kEncCodeStages) * kCodeStageBytes + 1024;
static_assert(kSmemEnc <= 232448 - 1024, "ring does not fit the shared memory of a CTA");
static_assert(kEncStages <= kStagesMax, "stage barriers");
static_assert(kGroupRows == 8 * kRunRows, "converter lanes: 8 runs of 4 lanes per warp");
static_assert(kConvGroups < kEncStages && kConvGroups < kEncCodeStages, "converter groups");

struct __align__(8) EncState {
  uint64_t full[kEncStages];         // leader: weights of both CTAs + the converter warps
  uint64_t empty[kEncStages];        // MMA commit (both CTAs): A and weights consumed
  uint64_t cfull[kEncCodeStages];    // codes landed
  uint64_t cempty[kEncCodeStages];   // every converter warp of the CTA is done with them
  uint64_t tfull[kAccums];
  uint64_t tempty[kAccums];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
};

// A converter lane's run of kRunRows consecutive rows within one tile, with
// the per-row factors of the decode (see decode_run) built once per tile.
struct Run {
  float2 keep[kRunRows];   // (0, 0) where the row starts a group, else (1, 1)
  float2 s[kRunRows];      // its scale where it starts one (0 for a row with no token)
  float2 b[kRunRows];      // the layer's bin, or 0 where the row starts a group
  int32_t a0;              // group anchor of row 0 (token index; row 0 itself if it is one)
  float s0;                // that anchor's scale (0 when row 0 is an anchor itself)
};

// Rows t0 .. t0+kRunRows-1 of layer li, from the group anchor of each token
// (the prepare kernel's table) and the scales: two rounds of independent
// loads.  A row past n_tokens or outside every request decodes as zeros (the
// epilogue stores no such row).
__device__ __forceinline__ Run make_run(const ProjectParams& p, const CodecInput& e, int li,
                                        int t0, float bin) {
  const float* sc = e.scales + int64_t(li) * p.n_tokens;
  int32_t a[kRunRows];
  float s[kRunRows];
#pragma unroll
  for (int i = 0; i < kRunRows; ++i) {
    const int t = t0 + i;
    a[i] = t < p.n_tokens ? __ldg(e.anchor + t) : -1;
    s[i] = t < p.n_tokens ? __ldg(sc + t) : 0.f;
  }
  Run run;
#pragma unroll
  for (int i = 0; i < kRunRows; ++i) {
    const bool own = a[i] == t0 + i;
    const bool starts = own || a[i] < 0;
    const float si = own ? s[i] : 0.f;
    run.keep[i] = starts ? make_float2(0.f, 0.f) : make_float2(1.f, 1.f);
    run.s[i] = make_float2(si, si);
    run.b[i] = starts ? make_float2(0.f, 0.f) : make_float2(bin, bin);
  }
  const bool first_starts = a[0] == t0 || a[0] < 0;
  run.a0 = first_starts ? t0 : a[0];
  run.s0 = first_starts ? 0.f : __ldg(sc + a[0]);
  return run;
}

// Decodes elements 16p .. 16p+15 of k-block kb of the run's rows r0 ..
// r0+kRunRows-1 of this CTA's tile from the code stage (column chunk p of its
// rows; its row 0 is token win0, kCodeHalo rows before the tile) into the A
// stage (16-byte chunks 2p and 2p+1 of each row).
//
// Bank conflicts: at each step the 8 runs of a warp sit at rows four apart.
// In the chunk-major code stage (an odd pitch of 145 rows) the 8 lanes of a
// quarter warp read 8 different 16-byte bank groups; for the 128-byte-swizzled
// A stage, lanes of odd runs (swap) store their odd chunk first, so that the
// two runs of a quarter warp write chunks of opposite parity.
//
// Branch-free, so that the rows' arithmetic interleaves: the running anchor
// value a (16 elements) is updated on every row as a = a * keep + x * s, with
// keep = 0 and s = the row's scale on a row that starts a group, and keep = 1,
// s = 0 on the others; both forms are exact (a * 1 + 0 = a, a * 0 + t = t for
// the finite values decoding produces).  The row's value is then a + x * b
// with b = 0 on a group's first row, i.e. exactly q * s or q_anchor * s + c * b.
// EXACT: every c * b is exact in binary32 (the host checked all 255 codes
// against the bins), so a + c * b rounds once either way and one fused
// multiply-add replaces the multiply and the add.
template <int DT, bool EXACT>
__device__ __forceinline__ void decode_run(uint32_t a_stage, uint32_t c_stage, const Run& run,
                                           const int8_t* codes_l, int d, int win0, int r0,
                                           int kb, int p16, bool swap) {
  const uint32_t chunk = c_stage + uint32_t(p16 * kCodeChunkBytes);
  // the lane's 16 codes of a row, elements 8..15 first when swapping
  auto load = [&](uint32_t addr) {
    const uint4 v = ptx::lds128(addr);
    return swap ? make_uint4(v.z, v.w, v.x, v.y) : v;
  };
  uint4 w[kRunRows];
#pragma unroll
  for (int i = 0; i < kRunRows; ++i) w[i] = load(chunk + uint32_t((kCodeHalo + r0 + i) * 16));
  // row 0's group anchor: in the code stage, or (group_tokens > kCodeHalo + 1)
  // further back, in global memory
  const int ar = run.a0 - win0;
  const int col = kb * kBlockK + 16 * p16;
  uint4 aw = make_uint4(0u, 0u, 0u, 0u);
  if (ar >= 0) {
    aw = load(chunk + uint32_t(ar * 16));
  } else if (col < d) {   // d is a multiple of 16: all 16 codes or none are in the row
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(codes_l + int64_t(run.a0) * d + col));
    aw = swap ? make_uint4(v.z, v.w, v.x, v.y) : v;
  }
  float2 a[8];
  {
    float2 q[8];
    dec::codes_to_float(make_uint2(aw.x, aw.y), *reinterpret_cast<float2(*)[4]>(q));
    dec::codes_to_float(make_uint2(aw.z, aw.w), *reinterpret_cast<float2(*)[4]>(q + 4));
    const float2 s0 = make_float2(run.s0, run.s0);
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = __fmul2_rn(q[k], s0);
  }
  const uint32_t c_first = uint32_t(2 * p16 + (swap ? 1 : 0));
  const uint32_t c_second = c_first ^ 1u;
#pragma unroll
  for (int i = 0; i < kRunRows; ++i) {
    float2 x[8], y[8];
    dec::codes_to_float(make_uint2(w[i].x, w[i].y), *reinterpret_cast<float2(*)[4]>(x));
    dec::codes_to_float(make_uint2(w[i].z, w[i].w), *reinterpret_cast<float2(*)[4]>(x + 4));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      a[k] = __ffma2_rn(a[k], run.keep[i], __fmul2_rn(x[k], run.s[i]));
      y[k] = EXACT ? __ffma2_rn(x[k], run.b[i], a[k])
                   : __fadd2_rn(a[k], __fmul2_rn(x[k], run.b[i]));
    }
    const int r = r0 + i;
    const uint4 first = dec::narrow8<DT>(*reinterpret_cast<const float2(*)[4]>(y));
    const uint4 second = dec::narrow8<DT>(*reinterpret_cast<const float2(*)[4]>(y + 4));
    // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
    const uint32_t row = a_stage + uint32_t(r * (kBlockK * 2));
    ptx::sts128(row + ((c_first ^ uint32_t(r & 7)) << 4), first.x, first.y, first.z, first.w);
    ptx::sts128(row + ((c_second ^ uint32_t(r & 7)) << 4), second.x, second.y, second.z,
                second.w);
  }
}

template <int DT, bool HT>
__global__ void __launch_bounds__(kEncThreads, 1)
    project_enc_kernel(const __grid_constant__ CUtensorMap tmap_c,
                       const __grid_constant__ CUtensorMap tmap_w, const ProjectParams p,
                       const CodecInput e) {
  constexpr int S = kEncStages;
  constexpr int C = kEncCodeStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ EncState es;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;                                      // S x [128][64], decoded here
  uint8_t* smem_b = smem_a + size_t(S) * kTileBytesA;          // S x [128][64], TMA
  uint8_t* smem_c = smem_b + size_t(S) * kPairBytesB;          // C x [4][145][16] int8, TMA

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int32_t* abort = &es.abort;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t unit = int64_t(blockIdx.x >> 1);
  const int64_t units = int64_t(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_u32(&es.full[s]), 1 + 2 * kGroupWarps);
      ptx::mbar_init(ptx::smem_u32(&es.empty[s]), 1);
    }
    for (int c = 0; c < C; ++c) {
      ptx::mbar_init(ptx::smem_u32(&es.cfull[c]), 1);
      ptx::mbar_init(ptx::smem_u32(&es.cempty[c]), kGroupWarps);
    }
    for (int a = 0; a < kAccums; ++a) {
      ptx::mbar_init(ptx::smem_u32(&es.tfull[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&es.tempty[a]), 2 * kEpilogueWarps);
    }
    ptx::mbar_init(ptx::smem_u32(&es.drain), 1);
    es.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&es.tmem_base), kAccums * kBlockN);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // peer barriers initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = es.tmem_base;

  int64_t issued = 0;    // weight stages armed (warp 0, lane 0)
  int64_t cissued = 0;   // code stages armed (warp 6, lane 0)
  if (warp == 0) {
    // --------------------------------------------------------- weight producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_w);
      const bool reuse_w = p.m_tiles > 1;
      const uint64_t keep = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t rnd = 0, tile; ok && (tile = round_tile(rnd, unit, units)) < p.num_tiles; ++rnd) {
        const TileCoord c = tile_coord(tile, p);
        const int row_b = c.n * kBlockN + int(rank) * (kBlockN / 2);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase_sleep(ptx::smem_u32(&es.empty[stage]), phase ^ 1u, abort, p,
                                kWaitProducerEmpty, uint32_t(tile), uint32_t(kb), kSleepNs)) {
            ok = false;
            break;
          }
          const uint32_t full = ptx::smem_u32(&es.full[stage]);
          const uint32_t dst_b = ptx::smem_u32(smem_b + size_t(stage) * kPairBytesB);
          if (leader) ptx::mbar_arrive_expect_tx(full, 2 * kPairBytesB);
          const uint32_t full_leader = ptx::mapa_shared(full, 0);
          if (reuse_w)
            ptx::tma_load_3d_pair_hint(dst_b, &tmap_w, full_leader, kb * kBlockK, row_b,
                                       p.layer_begin + c.l, keep);
          else
            ptx::tma_load_3d_pair(dst_b, &tmap_w, full_leader, kb * kBlockK, row_b,
                                  p.layer_begin + c.l);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == kEncCodeWarp) {
    // ----------------------------------------------------------- code producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_c);
      int cs = 0;
      uint32_t cphase = 0;
      bool ok = true;
      for (int64_t rnd = 0, tile; ok && (tile = round_tile(rnd, unit, units)) < p.num_tiles; ++rnd) {
        const TileCoord c = tile_coord(tile, p);
        const bool half_tile = HT && c.m == p.m_tiles - 1;
        const int row_a = c.m * 2 * kBlockM + int(rank) * (half_tile ? kBlockM / 2 : kBlockM);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase_sleep(ptx::smem_u32(&es.cempty[cs]), cphase ^ 1u, abort, p,
                                kWaitCodesEmpty, uint32_t(tile), uint32_t(kb), kSleepNs)) {
            ok = false;
            break;
          }
          const uint32_t cfull = ptx::smem_u32(&es.cfull[cs]);
          ptx::mbar_arrive_expect_tx(cfull, kCodeBytes);
          if (!(p.debug_stall && cissued == 0))
            ptx::tma_load_4d(ptx::smem_u32(smem_c + size_t(cs) * kCodeStageBytes), &tmap_c,
                             cfull, 0, row_a - kCodeHalo, kb * (kBlockK / 16), c.l);
          ++cissued;
          if (++cs == C) {
            cs = 0;
            cphase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = make_idesc_f16(DT, 2 * kBlockM, kBlockN);
      constexpr uint32_t idesc_half = make_idesc_f16(DT, kBlockM, kBlockN);   // M=128
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t rnd = 0, tile; ok && (tile = round_tile(rnd, unit, units)) < p.num_tiles; ++rnd) {
        if (!wait_phase_sleep(ptx::smem_u32(&es.tempty[acc]), acc_phase ^ 1u, abort, p,
                              kWaitMmaAccum, uint32_t(tile), uint32_t(acc), kSleepNs))
          break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * kBlockN);
        const uint32_t id = (HT && tile_coord(tile, p).m == p.m_tiles - 1) ? idesc_half : idesc;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase_sleep(ptx::smem_u32(&es.full[stage]), phase, abort, p, kWaitMmaFull,
                                uint32_t(tile), uint32_t(kb), kSleepNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smem_a + size_t(stage) * kTileBytesA);
          const uint32_t b0 = ptx::smem_u32(smem_b + size_t(stage) * kPairBytesB);
#pragma unroll
          for (int k = 0; k < kBlockK / kUmmaK; ++k) {
            const uint64_t da = ptx::sw128_kmajor_desc(a0 + k * kUmmaK * 2);
            const uint64_t db = ptx::sw128_kmajor_desc(b0 + k * kUmmaK * 2);
            ptx::mma_f16_pair(d_tmem, da, db, id, (kb | k) != 0 ? 1u : 0u);
          }
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&es.empty[stage]), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(ptx::smem_u32(&es.tfull[acc]), 0x3);
        if (++acc == kAccums) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      ptx::mma_commit_pair_multicast(ptx::smem_u32(&es.drain), 0x1);
      drain_wait(ptx::smem_u32(&es.drain), 0);
    }
  } else if (warp < kEncCodeWarp) {
    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t rnd = 0, tile; (tile = round_tile(rnd, unit, units)) < p.num_tiles; ++rnd) {
      const TileCoord c = tile_coord(tile, p);
      int ok = 0;
      if (lane == 0)
        ok = wait_phase_sleep(ptx::smem_u32(&es.tfull[acc]), acc_phase, abort, p,
                              kWaitEpilogueAccum, uint32_t(tile), uint32_t(acc), kSleepNs);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      token_tile_epilogue<DT, true, HT>(
          p, c, rank, quad, lane,
          tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * kBlockN));
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0)
        ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&es.tempty[acc]), 0));
      if (++acc == kAccums) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ converters
    // Group g of kConvGroups converts the k-blocks g, g + kConvGroups, ... of
    // this CTA's sequence (tiles in order, k-blocks in order), so the groups'
    // waits, proxy fences and arrivals overlap instead of adding up per
    // k-block; each of a group's warps decodes 32 rows of the tile.
    const int cw = warp - kEncConvWarp0;
    const int grp = cw / kGroupWarps;
    const int p16 = lane & 3;                      // 16 codes = 2 chunks of the A row
    const bool swap = (lane >> 2) & 1;             // odd run: store the odd chunk first
    // this lane's run: rows r0 .. r0+kRunRows-1 of the tile
    const int r0 = kGroupRows * (cw % kGroupWarps) + kRunRows * (lane >> 2);
    int kb = grp, stage = grp, cs = grp;
    uint32_t phase = 0, cphase = 0;
    int64_t rnd = 0;               // the unit's tiles in the other roles' order
    while (kb >= p.k_blocks) {   // fewer k-blocks per tile than groups
      kb -= p.k_blocks;
      ++rnd;
    }
    int64_t tile = round_tile(rnd, unit, units);
    int64_t run_tile = -1;
    Run run;
    TileCoord c{};
    int rows = 0, row_a = 0;
    const int8_t* codes_l = nullptr;
    while (tile < p.num_tiles) {
      if (tile != run_tile) {
        run_tile = tile;
        c = tile_coord(tile, p);
        const bool half_tile = HT && c.m == p.m_tiles - 1;
        rows = half_tile ? kBlockM / 2 : kBlockM;
        row_a = c.m * 2 * kBlockM + int(rank) * rows;
        codes_l = e.codes + int64_t(c.l) * p.n_tokens * p.d_model;
        if (r0 < rows)
          run = make_run(p, e, c.l, row_a + r0, dec::layer_bin(e, p.layer_begin + c.l));
      }
      // every lane observes both phases itself: it reads the codes TMA wrote
      // and overwrites the A stage the tensor core read
      const bool got =
          wait_phase_sleep(ptx::smem_u32(&es.cfull[cs]), cphase, abort, p, kWaitConvCodes,
                           uint32_t(tile), uint32_t(kb), kSleepNs) &&
          wait_phase_sleep(ptx::smem_u32(&es.empty[stage]), phase ^ 1u, abort, p,
                           kWaitConvStage, uint32_t(tile), uint32_t(kb), kSleepNs);
      if (!__all_sync(0xffffffffu, got)) break;
      if (r0 < rows) {   // warp-uniform
        const uint32_t a_st = ptx::smem_u32(smem_a + size_t(stage) * kTileBytesA);
        const uint32_t c_st = ptx::smem_u32(smem_c + size_t(cs) * kCodeStageBytes);
        if (e.exact_products)
          decode_run<DT, true>(a_st, c_st, run, codes_l, p.d_model, row_a - kCodeHalo, r0, kb,
                               p16, swap);
        else
          decode_run<DT, false>(a_st, c_st, run, codes_l, p.d_model, row_a - kCodeHalo, r0, kb,
                                p16, swap);
      }
      ptx::fence_proxy_async_smem();   // generic writes -> the tensor core's reads
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&es.full[stage]), 0));
        ptx::mbar_arrive(ptx::smem_u32(&es.cempty[cs]));
      }
      // this group's next k-block
      kb += kConvGroups;
      while (kb >= p.k_blocks) {
        kb -= p.k_blocks;
        ++rnd;
      }
      tile = round_tile(rnd, unit, units);
      stage += kConvGroups;
      while (stage >= S) {
        stage -= S;
        phase ^= 1u;
      }
      cs += kConvGroups;
      while (cs >= C) {
        cs -= C;
        cphase ^= 1u;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // Both CTAs have left their roles.  Loads still in flight after an abort
  // are among the last S weight stages (counted on the leader's barriers) and
  // the last C code stages of each CTA; wait for them (bounded) before either
  // CTA releases its memory.
  ptx::cluster_sync();
  if (lane == 0) {
    if (leader && warp == 0) {
      const int64_t first = issued > S ? issued - S : 0;
      for (int64_t i = first; i < issued; ++i)
        drain_wait(ptx::smem_u32(&es.full[i % S]), uint32_t((i / S) & 1));
    }
    if (warp == kEncCodeWarp && *abort) {
      const int64_t first = cissued > C ? cissued - C : 0;
      for (int64_t i = first; i < cissued; ++i)
        drain_wait(ptx::smem_u32(&es.cfull[i % C]), uint32_t((i / C) & 1));
    }
  }
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kAccums * kBlockN);
  }
}

template <int DT, bool HT>
cudaError_t launch_enc(const CUtensorMap& tmap_c, const CUtensorMap& tmap_w,
                       const ProjectParams& p, const CodecInput& e, int grid, cudaStream_t s) {
  auto kernel = project_enc_kernel<DT, HT>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemEnc));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kEncThreads);
  cfg.dynamicSmemBytes = kSmemEnc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tmap_c, tmap_w, p, e);
}

template <int DT>
int max_enc_clusters() {
  auto kernel = project_enc_kernel<DT, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemEnc)) != cudaSuccess)
    return -1;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(sms & ~1));
  cfg.blockDim = dim3(kEncThreads);
  cfg.dynamicSmemBytes = kSmemEnc;
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

cudaError_t launch_project_enc(const CUtensorMap& tmap_c, const CUtensorMap& tmap_w,
                               const ProjectParams& p, const CodecInput& e, int grid,
                               cudaStream_t s) {
  const bool ht = p.half_tail != 0;
  if (p.dtype == HCR_DTYPE_BF16)
    return ht ? launch_enc<HCR_DTYPE_BF16, true>(tmap_c, tmap_w, p, e, grid, s)
              : launch_enc<HCR_DTYPE_BF16, false>(tmap_c, tmap_w, p, e, grid, s);
  return ht ? launch_enc<HCR_DTYPE_FP16, true>(tmap_c, tmap_w, p, e, grid, s)
            : launch_enc<HCR_DTYPE_FP16, false>(tmap_c, tmap_w, p, e, grid, s);
}

int project_enc_clusters(int dtype) {
  return dtype == HCR_DTYPE_BF16 ? max_enc_clusters<HCR_DTYPE_BF16>()
                                 : max_enc_clusters<HCR_DTYPE_FP16>();
}

}  // namespace hcr
