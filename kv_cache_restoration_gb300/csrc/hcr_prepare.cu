// Restore prologue and create-time packing.
//
// prepare_kernel (one launch, two block ranges):
//   * placement -- token t of the concatenated requests belongs to request r
//     with cu_seqlens[r] <= t < cu_seqlens[r+1] (binary search), sits at
//     position p = start_pos[r] + t - cu_seqlens[r], and goes to cache slot
//     block_table[r][p / B] * B + p % B.  Rows whose block id, logical
//     block or position is out of range get slot -1 (never written) and set
//     a device error bit.
//   * norm statistics -- one warp per (layer, token) row of the saved hidden
//     states: RMSNorm rstd = 1/sqrt(mean(h^2) + eps); LayerNorm mean, then
//     rstd = 1/sqrt(biased var + eps) from a second pass of squared
//     deviations from that mean.  The hidden states are the layer inputs the
//     HCache episode ("Fast State Restoration for Evicted LLM KV Caches",
//     cue 14) restores from; applying the input norm is this library's
//     reading of its K = W_k H shorthand for pre-norm models.  With the
//     codec's encoded form as input the warp decodes the row (its codes, its
//     group anchor's codes and scale) into the values hcr_decode_hidden would
//     store and reduces those, and placement also records each token's group
//     anchor for the projection.
//
// pack_kernel and column_constants_kernel run once in hcr_create: the packed
// weight W'[j][i] = W[j][i] * gamma[i] (W = [W_k; W_v]) rounded once to the
// storage type, and the per-column fp32 constants the GEMM epilogue needs
// (LayerNorm: colsum_j = sum_i W'[j][i], bias_j = sum_i W[j][i] beta_i + b_j).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hcr_decode.cuh"
#include "hcr_internal.h"
#include "hcr_stats.cuh"

namespace hcr {
namespace {

using namespace stats;

constexpr int kPrepareThreads = 256;

template <int DT>
__device__ __forceinline__ float to_float(uint16_t v) {
  if constexpr (DT == HCR_DTYPE_BF16) {
    return __bfloat162float(*reinterpret_cast<__nv_bfloat16*>(&v));
  } else {
    return __half2float(*reinterpret_cast<__half*>(&v));
  }
}

template <int DT>
__device__ __forceinline__ uint16_t from_float(float x) {
  if constexpr (DT == HCR_DTYPE_BF16) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
  } else {
    __half h = __float2half_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
  }
}

__device__ void place_token(const PrepareParams& p, int t) {
  const int32_t* cu = p.cu_seqlens;
  uint32_t bad = 0;
  // last r in [0, n_req) with cu[r] <= t
  int lo = 0, hi = p.n_req - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const int c0 = __ldg(cu + r), c1 = __ldg(cu + r + 1);
  int64_t slot = -1;
  int pos = 0;
  if (!(c0 <= t && t < c1)) {
    bad |= HCR_DEVERR_SEQLENS;
  } else {
    const int start = __ldg(p.start_pos + r);
    const int64_t p64 = int64_t(start) + (t - c0);
    if (start < 0 || p64 > INT32_MAX || (p.check_position && p64 >= p.max_position)) {
      bad |= HCR_DEVERR_POSITION;
    } else {
      pos = int(p64);
      const int lb = pos / p.block_size;
      if (lb >= p.max_blocks) {
        bad |= HCR_DEVERR_LOGICAL_BLOCK;
      } else {
        const int blk = __ldg(p.block_table + int64_t(r) * p.max_blocks + lb);
        if (blk < 0 || blk >= p.num_blocks) {
          bad |= HCR_DEVERR_BLOCK_ID;
        } else {
          slot = int64_t(blk) * p.block_size + pos % p.block_size;
        }
      }
    }
  }
  if (bad) atomicOr(p.err, bad);
  p.slot[t] = slot;
  p.pos[t] = pos;
  if (p.enc.anchor) {
    const int g = p.enc.group_tokens;
    p.enc.anchor[t] = (c0 >= 0 && c0 <= t && t < c1) ? c0 + (t - c0) / g * g : -1;
  }
}

template <int DT, bool ENC>
__global__ void __launch_bounds__(kPrepareThreads) prepare_kernel(const PrepareParams p) {
  if (int(blockIdx.x) < p.slot_blocks) {
    const int t = blockIdx.x * kPrepareThreads + threadIdx.x;
    if (t < p.n_tokens) place_token(p, t);
    // the projection's statistics flags of this call start cleared
    for (int64_t i = t; i < p.n_zero_flags; i += int64_t(p.slot_blocks) * kPrepareThreads)
      p.zero_flags[i] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      // the host sized the grid from n_tokens; the table must agree
      if (__ldg(p.cu_seqlens) != 0 || __ldg(p.cu_seqlens + p.n_req) != p.n_tokens)
        atomicOr(p.err, uint32_t(HCR_DEVERR_SEQLENS));
    }
    return;
  }
  const int warps = kPrepareThreads / 32;
  const int64_t row =
      int64_t(blockIdx.x - p.slot_blocks) * warps + (threadIdx.x >> 5);
  if (row >= int64_t(p.n_layers) * p.n_tokens) return;
  row_stats<DT, ENC>(p, row, threadIdx.x & 31);
}

// W'[j][i] = round(W[j][i] * gamma[i]); rows j < d_kv from w_k, the rest from w_v.
template <int DT>
__global__ void pack_kernel(const uint16_t* __restrict__ w_k, const uint16_t* __restrict__ w_v,
                            const uint16_t* __restrict__ gamma, uint16_t* __restrict__ dst,
                            int d_kv, int d) {
  const int64_t n = int64_t(2) * d_kv * d;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t j = e / d;
    const int i = int(e - j * d);
    const uint16_t w = j < d_kv ? w_k[e] : w_v[e - int64_t(d_kv) * d];
    dst[e] = from_float<DT>(to_float<DT>(w) * to_float<DT>(gamma[i]));
  }
}

// One warp per output column j of the packed weight.
template <int DT>
__global__ void column_constants_kernel(const uint16_t* __restrict__ w_packed,
                                        const uint16_t* __restrict__ w_k,
                                        const uint16_t* __restrict__ w_v,
                                        const uint16_t* __restrict__ beta,
                                        const uint16_t* __restrict__ b_k,
                                        const uint16_t* __restrict__ b_v, float* col_sum,
                                        float* col_bias, int d_kv, int d, int layer_norm,
                                        int has_bias) {
  const int j = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= 2 * d_kv) return;
  const uint16_t* wp = w_packed + int64_t(j) * d;
  const uint16_t* w = j < d_kv ? w_k + int64_t(j) * d : w_v + int64_t(j - d_kv) * d;
  float s = 0.f, sb = 0.f;
  for (int i = lane; i < d; i += 32) {
    if (layer_norm) {
      s += to_float<DT>(wp[i]);
      sb = fmaf(to_float<DT>(w[i]), to_float<DT>(beta[i]), sb);
    }
  }
  s = warp_sum(s);
  sb = warp_sum(sb);
  if (lane == 0) {
    if (layer_norm) col_sum[j] = s;
    if (col_bias) {
      float b = layer_norm ? sb : 0.f;
      if (has_bias) b += to_float<DT>(j < d_kv ? b_k[j] : b_v[j - d_kv]);
      col_bias[j] = b;
    }
  }
}

}  // namespace

cudaError_t launch_prepare(const PrepareParams& p0, cudaStream_t s) {
  PrepareParams p = p0;
  p.slot_blocks = p.skip_placement ? 0 : (p.n_tokens + kPrepareThreads - 1) / kPrepareThreads;
  const int64_t rows = int64_t(p.n_layers) * p.n_tokens;
  const int64_t stat_blocks = (rows + kPrepareThreads / 32 - 1) / (kPrepareThreads / 32);
  const int64_t grid = p.slot_blocks + stat_blocks;
  if (grid <= 0) return cudaSuccess;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  const bool enc = p.enc.codes != nullptr;
  if (p.dtype == HCR_DTYPE_BF16) {
    if (enc)
      prepare_kernel<HCR_DTYPE_BF16, true><<<unsigned(grid), kPrepareThreads, 0, s>>>(p);
    else
      prepare_kernel<HCR_DTYPE_BF16, false><<<unsigned(grid), kPrepareThreads, 0, s>>>(p);
  } else {
    if (enc)
      prepare_kernel<HCR_DTYPE_FP16, true><<<unsigned(grid), kPrepareThreads, 0, s>>>(p);
    else
      prepare_kernel<HCR_DTYPE_FP16, false><<<unsigned(grid), kPrepareThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const void* w_k, const void* w_v, const void* gamma, void* dst,
                                int d_kv, int d, int dtype, cudaStream_t s) {
  const int threads = 256;
  const int64_t n = int64_t(2) * d_kv * d;
  const int blocks = int(std::min<int64_t>((n + threads - 1) / threads, 65536));
  auto* k = static_cast<const uint16_t*>(w_k);
  auto* v = static_cast<const uint16_t*>(w_v);
  auto* g = static_cast<const uint16_t*>(gamma);
  auto* o = static_cast<uint16_t*>(dst);
  if (dtype == HCR_DTYPE_BF16)
    pack_kernel<HCR_DTYPE_BF16><<<blocks, threads, 0, s>>>(k, v, g, o, d_kv, d);
  else
    pack_kernel<HCR_DTYPE_FP16><<<blocks, threads, 0, s>>>(k, v, g, o, d_kv, d);
  return cudaGetLastError();
}

cudaError_t launch_column_constants(const void* w_packed, const void* w_k, const void* w_v,
                                    const void* beta, const void* b_k, const void* b_v,
                                    float* col_sum, float* col_bias, int d_kv, int d, int dtype,
                                    int layer_norm, int has_bias, cudaStream_t s) {
  const int threads = 256;
  const int blocks = (2 * d_kv + threads / 32 - 1) / (threads / 32);
  auto cast = [](const void* x) { return static_cast<const uint16_t*>(x); };
  if (dtype == HCR_DTYPE_BF16)
    column_constants_kernel<HCR_DTYPE_BF16><<<blocks, threads, 0, s>>>(
        cast(w_packed), cast(w_k), cast(w_v), cast(beta), cast(b_k), cast(b_v), col_sum,
        col_bias, d_kv, d, layer_norm, has_bias);
  else
    column_constants_kernel<HCR_DTYPE_FP16><<<blocks, threads, 0, s>>>(
        cast(w_packed), cast(w_k), cast(w_v), cast(beta), cast(b_k), cast(b_v), col_sum,
        col_bias, d_kv, d, layer_norm, has_bias);
  return cudaGetLastError();
}

}  // namespace hcr
