// Norm statistics of one hidden row, computed by one warp: RMSNorm rstd =
// 1/sqrt(mean(h^2) + eps); LayerNorm mean, then rstd = 1/sqrt(biased var +
// eps) from a second pass of squared deviations from that mean.  Shared by
// the prepare kernel (hcr_prepare.cu) and the statistics warps of the
// token-row projection kernel (hcr_project.cu), so both write the same bits
// for a row.  The hidden states are the layer inputs the HCache episode
// ("Fast State Restoration for Evicted LLM KV Caches", cue 14) restores from;
// applying the input norm is this library's reading of its K = W_k H
// shorthand for pre-norm models.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hcr_decode.cuh"
#include "hcr_internal.h"

namespace hcr {
namespace stats {

template <int DT>
__device__ __forceinline__ float2 to_float2(uint32_t v) {
  if constexpr (DT == HCR_DTYPE_BF16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
    return __bfloat1622float2(h);
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// The storage-type values of one hidden row, 8 at a time (vector v holds
// elements 8v .. 8v+7): read as stored, or decoded from the codec's codes
// exactly as hcr_decode_hidden writes them.
template <int DT, bool ENC>
struct RowSource {
  const uint4* hv;        // stored row
  const uint2* own;       // encoded: the row's codes
  const uint2* anchor;    // encoded: its group anchor's codes
  float s, b;             // encoded: anchor scale, layer bin
  bool is_anchor;

  __device__ __forceinline__ uint4 operator()(int v) const {
    if constexpr (!ENC) {
      return __ldg(hv + v);
    } else {
      float2 q[4], a[4];
      dec::codes_to_float(__ldg(anchor + v), q);
      dec::anchor8(q, s, a);
      if (is_anchor) return dec::narrow8<DT>(a);
      float2 c[4], y[4];
      dec::codes_to_float(__ldg(own + v), c);
      dec::delta8(a, c, b, y);
      return dec::narrow8<DT>(y);
    }
  }
};

template <int DT, bool ENC>
__device__ RowSource<DT, ENC> row_source(const PrepareParams& p, int64_t row) {
  RowSource<DT, ENC> src{};
  const int d = p.d_model;
  if constexpr (!ENC) {
    src.hv = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.hidden) +
                                            row * int64_t(d));
  } else {
    const CodecInput& e = p.enc;
    const int li = int(row / p.n_tokens);
    const int t = int(row - int64_t(li) * p.n_tokens);
    int r, c0, c1;
    int64_t arow = row;   // a token in no request decodes as zeros (and is flagged by placement)
    src.s = 0.f;
    src.is_anchor = true;
    if (dec::request_of(e.cu_seqlens, e.n_req, t, &r, &c0, &c1)) {
      const int a = c0 + (t - c0) / e.group_tokens * e.group_tokens;
      arow = int64_t(li) * p.n_tokens + a;
      src.s = __ldg(e.scales + arow);
      src.is_anchor = a == t;
    }
    src.own = reinterpret_cast<const uint2*>(e.codes + row * int64_t(d));
    src.anchor = reinterpret_cast<const uint2*>(e.codes + arow * int64_t(d));
    src.b = dec::layer_bin(e, p.layer_begin + li);
  }
  return src;
}

template <int DT, bool ENC>
__device__ void row_stats(const PrepareParams& p, int64_t row, int lane) {
  const RowSource<DT, ENC> src = row_source<DT, ENC>(p, row);
  const int d = p.d_model;
  const int nvec = d >> 3;
  const float inv_d = 1.0f / float(d);
  if (!p.layer_norm) {
    float s2 = 0.f;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      const uint4 q = src(v);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = to_float2<DT>(w[k]);
        s2 = fmaf(f.x, f.x, s2);
        s2 = fmaf(f.y, f.y, s2);
      }
    }
    s2 = warp_sum(s2);
    if (lane == 0) p.rstd[row] = 1.0f / sqrtf(s2 * inv_d + p.eps);
    return;
  }
  // LayerNorm in two passes over the row: the mean (summed around the row's
  // first element, which keeps the partial sums small when |mean| >> spread),
  // then the sum of squared deviations from that mean.  The second pass reads
  // the row again from L1/L2.  A one-pass sum(x^2) - mean^2 cancels when
  // |mean| or an outlier channel is large against the spread.
  const float shift = to_float2<DT>(src(0).x).x;
  float s1 = 0.f;
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) {
    const uint4 q = src(v);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = to_float2<DT>(w[k]);
      s1 += (f.x - shift) + (f.y - shift);
    }
  }
  s1 = warp_sum(s1);
  const float mean = shift + s1 * inv_d;
  float s2 = 0.f;
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) {
    const uint4 q = src(v);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = to_float2<DT>(w[k]);
      const float x0 = f.x - mean, x1 = f.y - mean;
      s2 = fmaf(x0, x0, s2);
      s2 = fmaf(x1, x1, s2);
    }
  }
  s2 = warp_sum(s2);
  if (lane == 0) {
    p.mean[row] = mean;
    p.rstd[row] = 1.0f / sqrtf(s2 * inv_d + p.eps);
  }
}

}  // namespace stats
}  // namespace hcr
