// Decoding the hidden-state codec's int8 form inside the restore kernels
// (hcr_prepare.cu: norm statistics of the decoded rows; hcr_project_enc.cu:
// the GEMM's A operand), bit for bit what hcr_decode_hidden writes.
//
// The codec (HCache episode, "Fast State Restoration for Evicted LLM KV
// Caches", cues 30 and 32; CacheGen review, section 核心方法) groups 10
// tokens of a request behind an anchor: the anchor row decodes as q * s (its
// codes q, its scale s), every other row of the group as q_anchor * s + c * b
// (its codes c, the bin b of the layer's third).  Each step is one binary32
// operation rounded to nearest even, then one rounding to the storage type.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hcr_internal.h"

namespace hcr {
namespace dec {

// Eight int8 codes (two little-endian words) as exact floats.  A code byte b
// placed in the low mantissa byte of 2^23, after flipping its sign bit, is the
// binary32 value 2^23 + (b + 128); subtracting 2^23 + 128 leaves b exactly.
// One byte permute per code and one packed add per pair of codes, instead of
// an integer-to-float conversion per code.
__device__ __forceinline__ void codes_to_float(uint2 w, float2 (&x)[4]) {
  const uint32_t u0 = w.x ^ 0x80808080u, u1 = w.y ^ 0x80808080u;
  constexpr uint32_t kHi = 0x4B000000u;   // 2^23: bytes 1..3 of the result
  const float2 bias = make_float2(-8388736.f, -8388736.f);   // -(2^23 + 128)
  x[0] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u0, kHi, 0x7540)),
                                __uint_as_float(__byte_perm(u0, kHi, 0x7541))), bias);
  x[1] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u0, kHi, 0x7542)),
                                __uint_as_float(__byte_perm(u0, kHi, 0x7543))), bias);
  x[2] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u1, kHi, 0x7540)),
                                __uint_as_float(__byte_perm(u1, kHi, 0x7541))), bias);
  x[3] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u1, kHi, 0x7542)),
                                __uint_as_float(__byte_perm(u1, kHi, 0x7543))), bias);
}

// Anchor row: a = q * s.
__device__ __forceinline__ void anchor8(const float2 (&q)[4], float s, float2 (&a)[4]) {
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int k = 0; k < 4; ++k) a[k] = __fmul2_rn(q[k], s2);
}

// Other rows: y = a + c * b.
__device__ __forceinline__ void delta8(const float2 (&a)[4], const float2 (&c)[4], float b,
                                       float2 (&y)[4]) {
  const float2 b2 = make_float2(b, b);
#pragma unroll
  for (int k = 0; k < 4; ++k) y[k] = __fadd2_rn(a[k], __fmul2_rn(c[k], b2));
}

// Storage-type bits of a float pair, round to nearest even.
template <int DT>
__device__ __forceinline__ uint32_t narrow2(float2 v) {
  if constexpr (DT == HCR_DTYPE_BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(v.x, v.y);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int DT>
__device__ __forceinline__ uint4 narrow8(const float2 (&y)[4]) {
  return make_uint4(narrow2<DT>(y[0]), narrow2<DT>(y[1]), narrow2<DT>(y[2]), narrow2<DT>(y[3]));
}

// Bin of model layer l: bins[min(2, 3 l / n_layers_total)].
__device__ __forceinline__ float layer_bin(const CodecInput& e, int model_layer) {
  const int g = min(2, (3 * model_layer) / e.n_layers_total);
  return g == 0 ? e.bins[0] : (g == 1 ? e.bins[1] : e.bins[2]);   // no indexed param array
}

// Request of token t: the last r with cu[r] <= t, with its bounds [*c0, *c1).
// False when t lies in no request (an inconsistent table).
__device__ __forceinline__ bool request_of(const int32_t* cu, int n_req, int t, int* r, int* c0,
                                           int* c1) {
  int lo = 0, hi = n_req - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  *r = lo;
  *c0 = __ldg(cu + lo);
  *c1 = __ldg(cu + lo + 1);
  return *c0 >= 0 && *c0 <= t && t < *c1;
}

}  // namespace dec
}  // namespace hcr
