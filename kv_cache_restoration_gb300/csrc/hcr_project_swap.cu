// The fused K||V projection with weight-row tiles: the same restore as
// hcr_project.cu (HCache episode, "Fast State Restoration for Evicted LLM KV
// Caches", cue 14: K = W_k H, V = W_v H), with the operands of the tensor-core
// MMA swapped.  The packed weight rows are the MMA's M side and the tokens its
// N side:
//     acc[j][t] = sum_i W'_l[j][i] * H_l[t][i].
// M is two heads of 128 rows across a CTA pair (cta_group::2, one head per
// CTA), and N is a chunk of tokens padded only to a multiple of 16.  Token-row
// tiles pad a restore to 128 rows per CTA; at a few hundred tokens that
// padding is a large share of the work (300 tokens run as 384 or 512 rows),
// and cue 20 of the same episode singles out such awkward token counts (794).
// With weight rows as M, 300 tokens run as one chunk of 304 columns, 794 as
// 800.
//
// Tile space: (layer, head pair, token chunk), chunk fastest, so the chunks
// that share a pair of heads' weights run at the same time and read them from
// HBM once.  Warp roles as in the token-row pair kernel: warp 0 issues TMA
// loads, warp 1 allocates TMEM and issues the MMAs, and warps 2..9 run the
// epilogue, two warps per TMEM lane quadrant, each taking every other block
// of 8 tokens, two blocks at a time (a block's chain of loads, conversions
// and stores is latency-bound; two independent chains overlap).
//
// Epilogue.  A CTA's 128 TMEM lanes are one head's 128 dims, its columns the
// chunk's tokens.  The weights arrive through a 5-D view of the packed
// weights whose box reorders a head's rows: TMEM lane 16g + 8h + k holds dim
// 64h + 8g + k (g < 8, h < 2, k < 8).  A tcgen05.ld of shape 16x256b gives a
// thread lanes L and L + 8 of a 16-lane group -- dims i and i + 64, one
// rotate-half pair -- for two adjacent tokens, so RoPE needs no exchange
// between threads.  The thread then holds, per 8x8 block of (8 dims, 8 tokens),
// the fragment that stmatrix.trans writes to shared memory transposed: one
// 16-byte row of 8 consecutive dims per token, which goes to the token's
// paged cache slot as one 16-byte store.  The arithmetic is the token-row
// kernels' (shared helpers), so both compute every element bit for bit the
// same.
//
// Chunk size and TMEM.  Each CTA stages, per k-block, 16 KB of weights and
// 128 B per token of its half of the chunk, and moves those bytes from L2
// into shared memory at a rate that has a ceiling per SM (about 46 B per
// clock, measured on every tile shape here: the token-row pair tiles at 4096
// tokens sit right at it).  The flops per staged byte grow with the chunk, so
// short chunks are ingress-bound: 160 tokens need about 60 B per clock at
// full tensor rate, 256 about 46, 304 about 42.  The accumulators come from a
// ring of TMEM slots, taken in order by the MMA issuer and drained in the
// same order by the epilogue:
//   * two slots of 256 columns, one per tile of up to 256 tokens: the
//     epilogue of a tile overlaps the whole mainloop of the next;
//   * for tiles of 257..320 tokens, two "big" slots of b columns (b the
//     largest multiple of 32 with b + n <= 512: 192 for 304 tokens) taken in
//     turn, and one "small" slot after them: a tile puts its first n - b
//     columns (the first MMA) in the small slot and the other b (the second
//     MMA) in its big slot, and the epilogue drains the small part first.
//     The next tile's big slot is free while the epilogue drains the
//     previous tile, and its small slot is the part the epilogue drains
//     first -- the MMA waits for the drain of n - b columns (112 of 304),
//     about a third of one tile's epilogue.  It is the ring for restores of
//     257..320 tokens, which otherwise run as two ingress-bound chunks of
//     160 or less.
//
// With two MMAs, CTA r of the pair stages the chunk's tokens
// [r n/2, (r+1) n/2) as rows 0 .. n/2-1; the first MMA reads rows [0, n1/2) of
// both CTAs (tile columns [0, n1/2) from CTA 0, [n1/2, n1) from CTA 1), the
// second rows [n1/2, n/2) (tile columns [n1, n1 + n2/2) and [n1 + n2/2, n)).
// The epilogue maps each 8-column block back to its 8 consecutive tokens.
//
// Every pipeline wait is bounded as in hcr_project.cu.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hcr_internal.h"
#include "hcr_pipe.cuh"
#include "ptx.cuh"

namespace hcr {
namespace {

using namespace pipe;

struct SwapCoord {
  int l, hp, c;
};

__device__ __forceinline__ SwapCoord swap_coord(int64_t tile, const ProjectParams& p) {
  const int64_t per_layer = int64_t(p.head_pairs) * p.n_chunks;
  SwapCoord s;
  s.l = int(tile / per_layer);
  const int r = int(tile - int64_t(s.l) * per_layer);
  s.hp = r / p.n_chunks;
  s.c = r - s.hp * p.n_chunks;
  return s;
}

__device__ __forceinline__ int chunk_tokens(const ProjectParams& p, int c) {
  return c == p.n_chunks - 1 ? p.last_n : p.chunk;
}

// A unit of work of a CTA pair: a tile, or half of one.  The last
// p.split_tail tiles of the launch run as two units each, halves of their
// token chunk (N rounded to multiples of 16), so that the pairs' last round
// takes half a tile where it would leave most pairs idle for a whole one.
// Units number num_tiles + split_tail.
struct SwapUnit {
  int l, hp;
  int start, n;   // first token and token count
};

__device__ __forceinline__ SwapUnit swap_unit(int64_t u, const ProjectParams& p) {
  const int64_t whole = p.num_tiles - p.split_tail;
  const int64_t tile = u < whole ? u : whole + (u - whole) / 2;
  const SwapCoord c = swap_coord(tile, p);
  SwapUnit s{c.l, c.hp, c.c * p.chunk, chunk_tokens(p, c.c)};
  if (u >= whole) {
    const int n1 = (s.n / 2 + 15) & ~15;
    if ((u - whole) & 1) {
      s.start += n1;
      s.n -= n1;
    } else {
      s.n = n1;
    }
  }
  return s;
}

// N of the first MMA of a unit of n tokens on slots of slot_cols columns
// (the second has n - n1; none when n1 == n): a unit wider than one slot puts
// its first n - slot_cols columns in the small slot.
__device__ __forceinline__ int first_mma_n(int n, int slot_cols) {
  return n <= slot_cols ? n : n - slot_cols;
}

// TMEM column of accumulator slot s: big slots 0 and 1 at s * slot_cols, the
// small slot (2) after them.
__device__ __forceinline__ uint32_t slot_col(int s, const ProjectParams& p) {
  return uint32_t(s * p.slot_cols);
}

// The MMAs of one k-block: four K = 16 steps, each one MMA (TWO = false) or
// two (the second into accumulator columns n1.., reading token rows from
// b_off2 bytes into the stage).  The branch between the two forms is taken
// once per tile, outside the k-block loop.
template <bool TWO>
__device__ __forceinline__ void kblock_mmas(uint32_t d1, uint32_t d2, uint32_t a0, uint32_t b0,
                                            uint32_t id1, uint32_t id2, uint32_t b_off2,
                                            bool first) {
#pragma unroll
  for (int k = 0; k < kBlockK / kUmmaK; ++k) {
    const uint32_t accumulate = (first && k == 0) ? 0u : 1u;
    const uint64_t da = ptx::sw128_kmajor_desc(a0 + k * kUmmaK * 2);
    ptx::mma_f16_pair(d1, da, ptx::sw128_kmajor_desc(b0 + k * kUmmaK * 2), id1, accumulate);
    if constexpr (TWO)
      ptx::mma_f16_pair(d2, da, ptx::sw128_kmajor_desc(b0 + b_off2 + k * kUmmaK * 2), id2,
                        accumulate);
  }
}

// First token of tile columns [c0, c0 + 8) of a chunk of n tokens starting at
// `start` (see the staging order above).
__device__ __forceinline__ int block_token(int c0, int n, int n1, int start) {
  const int half = n >> 1;
  if (c0 < n1) {
    const int h1 = n1 >> 1;
    return c0 < h1 ? start + c0 : start + half + (c0 - h1);
  }
  const int local = c0 - n1, h1 = n1 >> 1, h2 = (n - n1) >> 1;
  return local < h2 ? start + h1 + local : start + half + h1 + (local - h2);
}

template <int DT>
__global__ void __launch_bounds__(kSwapThreads, 1)
    project_swap_kernel(const __grid_constant__ CUtensorMap tmap_h,
                        const __grid_constant__ CUtensorMap tmap_w5, const ProjectParams p) {
  const int S = p.stages;
  constexpr int kHead = 128;                        // head_dim of this variant
  extern __shared__ uint8_t smem_raw[];
  __shared__ PipeState ps;

  // stage s: [128 weight rows][64] then [chunk/2 token rows][64], 1024-aligned
  // (chunk is a multiple of 16, so chunk/2 rows of 128 B are whole 1 KB atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t bytes_b = uint32_t(p.chunk / 2) * kBlockK * 2;   // token box per CTA
  const size_t stage_bytes = size_t(kTileBytesA) + bytes_b;
  uint8_t* smem_a = smem;                                    // + s * stage_bytes
  uint8_t* smem_b = smem + kTileBytesA;                      // + s * stage_bytes
  uint8_t* staging = smem + size_t(S) * stage_bytes;         // 512 B per epilogue warp
  // token table of the tile in the epilogue: rstd, mean, position, slot
  float* tab_rstd = reinterpret_cast<float*>(staging + kSwapStaging);
  float* tab_mean = tab_rstd + 512;
  int32_t* tab_pos = reinterpret_cast<int32_t*>(tab_mean + 512);
  int64_t* tab_slot = reinterpret_cast<int64_t*>(tab_pos + 512);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int32_t* abort = &ps.abort;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t unit = int64_t(blockIdx.x >> 1);
  const int64_t units = int64_t(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_u32(&ps.full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&ps.empty[s]), 1);
    }
    for (int a = 0; a < p.n_slots; ++a) {
      ptx::mbar_init(ptx::smem_u32(&ps.slot_full[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&ps.slot_empty[a]), 2 * kSwapEpilogueWarps);
    }
    ptx::mbar_init(ptx::smem_u32(&ps.drain), 1);
    ptx::mbar_init(ptx::smem_u32(&ps.tab_full), kSwapEpilogueWarps);
    ptx::mbar_init(ptx::smem_u32(&ps.tab_free), kSwapEpilogueWarps);
    ps.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&ps.tmem_base), kSwapTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // peer barriers initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = ps.tmem_base;

  int64_t issued = 0;   // TMA stages armed by the producer (warp 0, lane 0)
  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_h);
      ptx::tma_prefetch_desc(&tmap_w5);
      // A head pair's weights are read by every chunk of the layer; with
      // several chunks keep them in L2 ahead of other data.
      const bool reuse_w = p.n_chunks > 1;
      const uint64_t keep = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int64_t n_units = p.num_tiles + p.split_tail;
      for (int64_t tile = unit; ok && tile < n_units; tile += units) {
        const SwapUnit c = swap_unit(tile, p);
        const int n = c.n;
        // each CTA stages n/2 of the unit's tokens (its box holds chunk/2 rows;
        // the MMAs read the first n/2)
        const int row_b = c.start + int(rank) * (n >> 1);
        const int head = (p.layer_begin + c.l) * 2 * p.head_pairs + 2 * c.hp + int(rank);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(ptx::smem_u32(&ps.empty[stage]), phase ^ 1u, abort, p,
                          kWaitProducerEmpty, uint32_t(tile), uint32_t(kb))) {
            ok = false;
            break;
          }
          const uint32_t full = ptx::smem_u32(&ps.full[stage]);
          const uint32_t dst_a = ptx::smem_u32(smem_a + size_t(stage) * stage_bytes);
          const uint32_t dst_b = ptx::smem_u32(smem_b + size_t(stage) * stage_bytes);
          // both CTAs' bytes complete on the leader's barrier
          if (leader) ptx::mbar_arrive_expect_tx(full, 2 * (uint32_t(kTileBytesA) + bytes_b));
          const uint32_t full_leader = ptx::mapa_shared(full, 0);
          if (!(p.debug_stall && issued == 0)) {
            if (reuse_w)
              ptx::tma_load_5d_pair_hint(dst_a, &tmap_w5, full_leader, kb * kBlockK, 0, 0, 0,
                                         head, keep);
            else
              ptx::tma_load_5d_pair(dst_a, &tmap_w5, full_leader, kb * kBlockK, 0, 0, 0, head);
            ptx::tma_load_3d_pair(dst_b, &tmap_h, full_leader, kb * kBlockK, row_b, c.l);
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
      constexpr uint32_t idesc_m256 = make_idesc_f16(DT, 2 * kBlockM, 0);   // N filled per tile
      int stage = 0;
      uint32_t phase = 0;
      int big = 0;             // this unit's big slot (0, 1 in turn)
      uint32_t uses = 0;       // bit s: parity of slot s's uses so far
      bool ok = true;
      const int64_t n_units = p.num_tiles + p.split_tail;
      for (int64_t tile = unit; ok && tile < n_units; tile += units) {
        const int n = swap_unit(tile, p).n;
        const int n1 = first_mma_n(n, p.slot_cols), n2 = n - n1;
        const bool two = n2 > 0;
        const int s1 = two ? 2 : big, s2 = big;   // first MMA: the small slot if two
        // the slots must be drained of their previous tiles (free on first use)
        if (!wait_phase(ptx::smem_u32(&ps.slot_empty[s1]), ((uses >> s1) & 1u) ^ 1u, abort, p,
                        kWaitMmaAccum, uint32_t(tile), uint32_t(s1)))
          break;
        if (two && !wait_phase(ptx::smem_u32(&ps.slot_empty[s2]), ((uses >> s2) & 1u) ^ 1u,
                               abort, p, kWaitMmaAccum, uint32_t(tile), uint32_t(s2)))
          break;
        ptx::tc_fence_after();
        const uint32_t d1 = tmem_base + slot_col(s1, p);
        const uint32_t d2 = tmem_base + slot_col(s2, p);
        const uint32_t id1 = idesc_m256 | (uint32_t(n1 >> 3) << 17);
        const uint32_t id2 = idesc_m256 | (uint32_t(n2 >> 3) << 17);
        const uint32_t b_off2 = uint32_t(n1 / 2) * kBlockK * 2;   // second MMA's token rows
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(ptx::smem_u32(&ps.full[stage]), phase, abort, p, kWaitMmaFull,
                          uint32_t(tile), uint32_t(kb))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smem_a + size_t(stage) * stage_bytes);
          const uint32_t b0 = ptx::smem_u32(smem_b + size_t(stage) * stage_bytes);
          if (two)
            kblock_mmas<true>(d1, d2, a0, b0, id1, id2, b_off2, kb == 0);
          else
            kblock_mmas<false>(d1, d2, a0, b0, id1, id2, b_off2, kb == 0);
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&ps.empty[stage]), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(ptx::smem_u32(&ps.slot_full[s1]), 0x3);
        uses ^= 1u << s1;
        if (two) {
          ptx::mma_commit_pair_multicast(ptx::smem_u32(&ps.slot_full[s2]), 0x3);
          uses ^= 1u << s2;
        }
        big ^= 1;
      }
      // Every MMA this thread issued has completed once `drain` flips.
      ptx::mma_commit_pair_multicast(ptx::smem_u32(&ps.drain), 0x1);
      drain_wait(ptx::smem_u32(&ps.drain), 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int e = warp - 2;                  // 0 .. kSwapEpilogueWarps-1
    const int quad = warp & 3;               // TMEM lanes [32*quad, 32*quad+32)
    constexpr int kPerQuad = kSwapEpilogueWarps / 4;   // warps sharing a lane quadrant
    const int sub = e >> 2;                  // which of the kPerQuad interleaved block sets
    const int q = lane >> 2;                 // fragment row: dims 8g+q and 64+8g+q
    const int r2 = (lane & 3) * 2;           // fragment columns: tokens r2, r2+1 of a block
    const uint32_t stg = ptx::smem_u32(staging + e * 1024);   // two 512-byte halves
    // stmatrix: this thread gives the address of row (lane & 7) of matrix (lane >> 3);
    // a staged row is one token's 4 x 16 bytes
    const uint32_t st_addr = stg + uint32_t((lane & 7) * 64 + (lane >> 3) * 16);
    // after the transpose this thread stores token (lane >> 2), 16-byte piece (lane & 3)
    const uint32_t ld_addr = stg + uint32_t((lane >> 2) * 64 + (lane & 3) * 16);
    const int piece = lane & 3;              // matrix: (lane group piece>>1, dims hi if piece&1)
    const int dim0 = 64 * (piece & 1) + 8 * (2 * quad + (piece >> 1));
    const bool ln = p.layer_norm != 0;
    int big = 0;             // the unit's big slot, in the MMA issuer's order
    uint32_t uses = 0;
    uint32_t tab_phase = 0;
    bool ok_all = true;
    const int64_t n_units = p.num_tiles + p.split_tail;
    for (int64_t tile = unit; ok_all && tile < n_units; tile += units) {
      const SwapUnit c = swap_unit(tile, p);
      const int n = c.n;
      const int n1 = first_mma_n(n, p.slot_cols);
      const bool two = n > n1;
      const int start = c.start;
      const int64_t srow = int64_t(c.l) * p.n_tokens;
      // The tile's per-token table, written while the MMA still works on the
      // tile: one coalesced round of loads instead of dependent loads per block.
      // Wait until every epilogue warp is done with the previous tile's table.
      int ok = 0;
      if (lane == 0)
        ok = wait_phase(ptx::smem_u32(&ps.tab_free), tab_phase ^ 1u, abort, p, kWaitEpilogueAccum,
                        uint32_t(tile), 8u);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      for (int i = e * 32 + lane; i < n; i += 32 * kSwapEpilogueWarps) {
        const int t = start + i;
        const bool valid = t < p.n_tokens;
        tab_rstd[i] = valid ? __ldg(p.rstd + srow + t) : 0.f;
        tab_mean[i] = (valid && p.layer_norm) ? __ldg(p.mean + srow + t) : 0.f;
        tab_pos[i] = (valid && p.rope) ? __ldg(p.pos + t) : 0;
        tab_slot[i] = valid ? __ldg(p.slot + t) : int64_t(-1);
      }
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(ptx::smem_u32(&ps.tab_full));
        ok = wait_phase(ptx::smem_u32(&ps.tab_full), tab_phase, abort, p, kWaitEpilogueAccum,
                        uint32_t(tile), 9u);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();   // the table lane 0 saw complete is read by every lane

      const int hg = 2 * c.hp + int(rank);           // head in the K||V list
      const bool is_k = hg < p.head_pairs;            // head_pairs == n_kv_heads
      const int kvh = is_k ? hg : hg - p.head_pairs;
      const bool do_rope = is_k && p.rope;
      // per-dim constants of this thread's four dims (lane groups j = 0, 1; lo, hi)
      float csum[2][2], cbias[2][2];
      const int64_t colb = int64_t(c.l) * p.n_cols + int64_t(hg) * kHead;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int lo = 8 * (2 * quad + j) + q;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          csum[j][h] = ln ? __ldg(p.col_sum + colb + lo + 64 * h) : 0.f;
          cbias[j][h] = p.has_bias ? __ldg(p.col_bias + colb + lo + 64 * h) : 0.f;
        }
      }
      uint16_t* base = reinterpret_cast<uint16_t*>(is_k ? p.k_cache : p.v_cache) +
                       int64_t(c.l) * p.layer_stride + int64_t(kvh) * kHead + dim0;

      // the unit's one or two slots, drained in the order the next units need
      // them: the small slot (the first MMA's columns) before the big one
      for (int part = 0; part < (two ? 2 : 1); ++part) {
        const int sl = (two && part == 0) ? 2 : big;
        const int c_lo = part == 0 ? 0 : n1, c_hi = part == 0 ? n1 : n;
        // RoPE (cos, sin) of this thread's two tokens and two frequencies in
        // block bb, loaded two blocks ahead of their use (the loads miss L1;
        // the first two blocks' before the slot is waited for)
        auto rope_load = [&](int bb, float2 (&cs)[2][2]) {
          const int ib = block_token(8 * bb, n, n1, start) - start + r2;
          const int pa = tab_pos[ib], pb = tab_pos[ib + 1];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int i = 8 * (2 * quad + j) + q;   // frequency index of the pair
            cs[j][0] = __ldg(p.rope_tab + int64_t(pa) * (kHead / 2) + i);
            cs[j][1] = __ldg(p.rope_tab + int64_t(pb) * (kHead / 2) + i);
          }
        };
        // This warp's blocks b0, b0 + kPerQuad, ..., two per iteration: their
        // chains of loads, conversions and stores are independent and overlap.
        const int b_end = c_hi / 8, b0 = c_lo / 8 + sub, step = kPerQuad;
        float2 cs_cur[2][2][2] = {}, cs_nxt[2][2][2] = {};   // [block][j][token]
        if (do_rope) {
          if (b0 < b_end) rope_load(b0, cs_cur[0]);
          if (b0 + step < b_end) rope_load(b0 + step, cs_cur[1]);
        }
        if (lane == 0)
          ok = wait_phase(ptx::smem_u32(&ps.slot_full[sl]), (uses >> sl) & 1u, abort, p,
                          kWaitEpilogueAccum, uint32_t(tile), uint32_t(sl));
        uses ^= 1u << sl;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          ok_all = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tslot =
            tmem_base + (uint32_t(quad * 32) << 16) + slot_col(sl, p);
        for (int b = b0; b < b_end; b += 2 * step) {
          const int nw = b + step < b_end ? 2 : 1;   // blocks this iteration (warp-uniform)
          if (do_rope) {
            if (b + 2 * step < b_end) rope_load(b + 2 * step, cs_nxt[0]);
            if (b + 3 * step < b_end) rope_load(b + 3 * step, cs_nxt[1]);
          }
          int t0[2];
          uint32_t R[2][2][4];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            if (w < nw) {
              const int bb = b + w * step;
              t0[w] = block_token(8 * bb, n, n1, start);
              const uint32_t col = uint32_t(8 * bb - c_lo);
              ptx::tmem_ld_16x256b(tslot + col, R[w][0]);
              ptx::tmem_ld_16x256b(tslot + (16u << 16) + col, R[w][1]);
            }
          }
          float rs[2][2], mu[2][2];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            // the two tokens of this thread's fragment columns (table rows ia, ia+1)
            const int ia = (w < nw ? t0[w] : t0[0]) - start + r2;
            rs[w][0] = tab_rstd[ia];
            rs[w][1] = tab_rstd[ia + 1];
            mu[w][0] = tab_mean[ia];
            mu[w][1] = tab_mean[ia + 1];
          }
          ptx::tmem_ld_wait();
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            if (w < nw) {
              uint32_t P[4];
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                float x[2][2];   // [token a/b][dim lo/hi]
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    float v = norm_scale(__uint_as_float(R[w][j][2 * h + u]), rs[w][u], mu[w][u],
                                         csum[j][h], ln);
                    if (p.has_bias) v = __fadd_rn(v, cbias[j][h]);
                    x[u][h] = v;
                  }
                if (do_rope) {
#pragma unroll
                  for (int u = 0; u < 2; ++u)
                    rope_pair(x[u][0], x[u][1], cs_cur[w][j][u].x, cs_cur[w][j][u].y);
                }
                P[2 * j] = pack2<DT>(x[0][0], x[1][0]);       // dims 8g+q, tokens r2, r2+1
                P[2 * j + 1] = pack2<DT>(x[0][1], x[1][1]);   // dims 64+8g+q
              }
              ptx::stmatrix_x4_trans(st_addr + uint32_t(w * 512), P[0], P[1], P[2], P[3]);
            }
          }
          __syncwarp();
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            if (w < nw) {
              const uint4 v = ptx::lds128(ld_addr + uint32_t(w * 512));
              const int64_t slot_t = tab_slot[t0[w] - start + (lane >> 2)];   // -1: skip
              if (slot_t >= 0) *reinterpret_cast<uint4*>(base + slot_t * int64_t(p.row_elems)) = v;
            }
          }
          __syncwarp();
#pragma unroll
          for (int w = 0; w < 2; ++w)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              cs_cur[w][j][0] = cs_nxt[w][j][0];
              cs_cur[w][j][1] = cs_nxt[w][j][1];
            }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)   // the leader's MMA reuses the slot in both CTAs
          ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&ps.slot_empty[sl]), 0));
      }
      if (!ok_all) break;
      big ^= 1;
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ps.tab_free));
      tab_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // Both CTAs have left their roles.  The leader's full barriers count both
  // CTAs' loads, so the leader waits (bounded; immediate unless a role gave up)
  // for its last S stages before either CTA releases its memory.
  ptx::cluster_sync();
  if (leader && warp == 0 && lane == 0) {
    const int64_t first = issued > S ? issued - S : 0;
    for (int64_t i = first; i < issued; ++i)
      drain_wait(ptx::smem_u32(&ps.full[i % S]), uint32_t((i / S) & 1));
  }
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kSwapTmemCols);
  }
}

template <int DT>
cudaError_t launch_swap(const CUtensorMap& tmap_h, const CUtensorMap& tmap_w5,
                        const ProjectParams& p, int grid, cudaStream_t s) {
  auto kernel = project_swap_kernel<DT>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kSmemSwap));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kSwapThreads);
  cfg.dynamicSmemBytes = kSmemSwap;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tmap_h, tmap_w5, p);
}

template <int DT>
int max_swap_clusters() {
  auto kernel = project_swap_kernel<DT>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemSwap)) != cudaSuccess)
    return -1;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(sms & ~1));
  cfg.blockDim = dim3(kSwapThreads);
  cfg.dynamicSmemBytes = kSmemSwap;
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

cudaError_t launch_project_swap(const CUtensorMap& tmap_h, const CUtensorMap& tmap_w5,
                                const ProjectParams& p, int grid, cudaStream_t s) {
  return p.dtype == HCR_DTYPE_BF16 ? launch_swap<HCR_DTYPE_BF16>(tmap_h, tmap_w5, p, grid, s)
                                   : launch_swap<HCR_DTYPE_FP16>(tmap_h, tmap_w5, p, grid, s);
}

int project_swap_clusters(int dtype) {
  return dtype == HCR_DTYPE_BF16 ? max_swap_clusters<HCR_DTYPE_BF16>()
                                 : max_swap_clusters<HCR_DTYPE_FP16>();
}

}  // namespace hcr
