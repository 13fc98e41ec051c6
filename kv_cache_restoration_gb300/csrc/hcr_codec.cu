// Hidden-state codec: anchor + delta groups with layer-wise bins.
//
// The HCache episode ("Fast State Restoration for Evicted LLM KV Caches",
// cues 30 and 32) proposes quantising hidden states the way CacheGen
// quantises KV caches.  CacheGen's encoder (CacheGen review, section 核心方法)
// cuts tokens into groups of 10 consecutive tokens; the first token of a
// group, its anchor, is kept with 8-bit quantisation and every other token as
// its difference from the anchor, quantised with a bin that grows with depth
// (0.5, 1, 1.5 for the first, middle and last third of the layers).  The
// lossless arithmetic-coding stage that follows on the page is not part of
// this library.
//
// This library's reading, fixed here and in the oracle alike:
//   * groups are formed per request (token i of a request belongs to the group
//     whose anchor is token G * (i / G) of that request);
//   * anchor row: scale s = max|h| / 127, code q = rint(h * (1 / s)) in
//     [-127, 127]; a row with s below 2^-126 codes as all zero (s = 0);
//   * other rows: code c = rint((h - q s) * (1 / b)) in [-127, 127] -- the
//     delta from the anchor as the decoder sees it; decoded value q s + c b;
//   * the reciprocals 1 / s (per anchor row) and 1 / b (per layer) are one
//     binary32 division each, so the per-element work is multiplications;
//   * layer l of L uses bin bins[min(2, 3 l / L)];
//   * every step is one IEEE binary32 operation rounded to nearest even (the
//     _rn intrinsics keep the compiler from contracting them), so the codes
//     and the decoded values are bit-identical to a binary32 reference.
//
// Encoded form: codes int8 [layer][token][d_model] and scales float32
// [layer][token] (entries of non-anchor rows are left untouched).
//
// encode_kernel: four warps per group (groups numbered request by request; a
// warp finds its group by a scan over the requests); grid.y runs over layers.
// Each warp reduces the anchor's max|h| over the whole row, then streams its
// quarter of the 16-byte vectors (8 elements per lane) of every row of the
// group, the decoded anchor recomputed per vector and four rows loaded before
// their codes are stored.  decode_kernel: one warp per token
// row, grid.y over layers; a row reads its anchor's codes and scale and its
// own codes and writes the storage type.  Both are HBM-bound; a row with no
// request (cu_seqlens inconsistent with n_tokens) is skipped and flagged.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "hcr_host.h"

namespace hcr {
namespace {

constexpr int kCodecThreads = 256;
constexpr int kWarpsPerGroup = 4;   // encode: warps sharing one group's rows (the max is
                                    // reduced by each over the whole anchor row)

struct CodecParams {
  const uint16_t* hidden;   // encode: input [Lr][T][d]
  uint16_t* out;            // decode: output [Lr][T][d]
  int8_t* codes;            // [Lr][T][d]
  float* scales;            // [Lr][T]
  const int32_t* cu_seqlens;
  uint32_t* err;
  int32_t n_req, n_tokens, d_model, layer_begin, n_layers_total, group_tokens, dtype;
  float bins[3];
};

template <int DT>
__device__ __forceinline__ float2 widen2(uint32_t v) {
  if constexpr (DT == HCR_DTYPE_BF16)
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
  else
    return __half22float2(*reinterpret_cast<__half2*>(&v));
}

template <int DT>
__device__ __forceinline__ uint32_t narrow2(float a, float b) {
  if constexpr (DT == HCR_DTYPE_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int DT>
__device__ __forceinline__ void widen8(const uint4& q, float (&x)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = widen2<DT>(w[k]);
    x[2 * k] = f.x;
    x[2 * k + 1] = f.y;
  }
}

__device__ __forceinline__ int8_t code_of(float x) {
  return int8_t(fminf(fmaxf(rintf(x), -127.f), 127.f));
}

__device__ __forceinline__ uint2 pack_codes(const int8_t (&c)[8]) {
  uint2 r;
  r.x = uint32_t(uint8_t(c[0])) | uint32_t(uint8_t(c[1])) << 8 | uint32_t(uint8_t(c[2])) << 16 |
        uint32_t(uint8_t(c[3])) << 24;
  r.y = uint32_t(uint8_t(c[4])) | uint32_t(uint8_t(c[5])) << 8 | uint32_t(uint8_t(c[6])) << 16 |
        uint32_t(uint8_t(c[7])) << 24;
  return r;
}

__device__ __forceinline__ void unpack_codes(uint2 r, float (&c)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    c[k] = float(int8_t(r.x >> (8 * k)));
    c[4 + k] = float(int8_t(r.y >> (8 * k)));
  }
}

// Request of token t (last r with cu[r] <= t), or -1 when t lies in no request.
__device__ __forceinline__ int request_of(const CodecParams& p, int t, int* c0, int* c1) {
  int lo = 0, hi = p.n_req - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens + mid) <= t) lo = mid; else hi = mid - 1;
  }
  *c0 = __ldg(p.cu_seqlens + lo);
  *c1 = __ldg(p.cu_seqlens + lo + 1);
  return (*c0 <= t && t < *c1) ? lo : -1;
}

__device__ __forceinline__ float layer_bin(const CodecParams& p, int li) {
  const int g = min(2, (3 * (p.layer_begin + li)) / p.n_layers_total);
  return g == 0 ? p.bins[0] : (g == 1 ? p.bins[1] : p.bins[2]);   // no indexed param array
}

// Group k of a layer (groups numbered request by request): its anchor token
// and row count, or n = 0 past the last group.  A linear scan over the
// requests; rows past n_tokens are never addressed (flagged instead).
__device__ __forceinline__ void group_of(const CodecParams& p, int k, int* t, int* n) {
  int base = 0;
  *n = 0;
  for (int r = 0; r < p.n_req; ++r) {
    const int c0 = __ldg(p.cu_seqlens + r), c1 = __ldg(p.cu_seqlens + r + 1);
    const int len = max(0, c1 - c0);
    const int g = (len + p.group_tokens - 1) / p.group_tokens;
    if (k < base + g) {
      *t = c0 + (k - base) * p.group_tokens;
      *n = min(p.group_tokens, c1 - *t);
      if (*t < 0 || *t + *n > p.n_tokens) {
        atomicOr(p.err, uint32_t(HCR_DEVERR_SEQLENS));
        *n = 0;
      }
      return;
    }
    base += g;
  }
}

template <int DT>
__global__ void __launch_bounds__(kCodecThreads) encode_kernel(const CodecParams p) {
  constexpr int kBatch = 4;   // group rows loaded together before their codes are stored
  const int lane = threadIdx.x & 31;
  const int li = blockIdx.y;
  const int wid = int((blockIdx.x * kCodecThreads + threadIdx.x) >> 5);
  const int k = wid / kWarpsPerGroup;       // the group
  const int part = wid % kWarpsPerGroup;    // this warp's share of each row's vectors
  const int nvec = p.d_model >> 3;
  const float b = layer_bin(p, li);
  if (wid == 0 && li == 0 && lane == 0 &&
      (__ldg(p.cu_seqlens) != 0 || __ldg(p.cu_seqlens + p.n_req) != p.n_tokens))
    atomicOr(p.err, uint32_t(HCR_DEVERR_SEQLENS));
  int t = 0, n = 0;
  group_of(p, k, &t, &n);
  if (n == 0) return;
  const int64_t row0 = int64_t(li) * p.n_tokens + t;
  const uint4* __restrict__ src = reinterpret_cast<const uint4*>(p.hidden + row0 * p.d_model);
  uint2* __restrict__ dst = reinterpret_cast<uint2*>(p.codes + row0 * p.d_model);
  float m = 0.f;
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) {
    float x[8];
    widen8<DT>(__ldg(src + v), x);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // a row below 127 * 2^-126 codes as all zero, so 1 / s stays finite
  const float s_raw = __fdiv_rn(m, 127.f);
  const float s = s_raw < 1.17549435e-38f ? 0.f : s_raw;
  const float inv_s = s == 0.f ? 0.f : __fdiv_rn(1.f, s);
  const float inv_b = __fdiv_rn(1.f, b);
  if (lane == 0 && part == 0) p.scales[row0] = s;
  for (int v = part * 32 + lane; v < nvec; v += 32 * kWarpsPerGroup) {
    float x[8], a_hat[8];
    int8_t q[8];
    widen8<DT>(__ldg(src + v), x);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      q[i] = s == 0.f ? int8_t(0) : code_of(__fmul_rn(x[i], inv_s));
      a_hat[i] = __fmul_rn(float(q[i]), s);
    }
    dst[v] = pack_codes(q);
    for (int j0 = 1; j0 < n; j0 += kBatch) {
      uint4 raw[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (j0 + u < n) raw[u] = __ldg(src + int64_t(j0 + u) * nvec + v);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (j0 + u >= n) break;
        float y[8];
        int8_t c[8];
        widen8<DT>(raw[u], y);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = code_of(__fmul_rn(__fsub_rn(y[i], a_hat[i]), inv_b));
        dst[int64_t(j0 + u) * nvec + v] = pack_codes(c);
      }
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kCodecThreads) decode_kernel(const CodecParams p) {
  const int lane = threadIdx.x & 31;
  const int li = blockIdx.y;
  const int warp0 = int((blockIdx.x * kCodecThreads + threadIdx.x) >> 5);
  const int nwarps = int((gridDim.x * kCodecThreads) >> 5);
  const int nvec = p.d_model >> 3;
  const float b = layer_bin(p, li);
  for (int t = warp0; t < p.n_tokens; t += nwarps) {
    int c0, c1;
    if (request_of(p, t, &c0, &c1) < 0) {
      if (lane == 0) atomicOr(p.err, uint32_t(HCR_DEVERR_SEQLENS));
      continue;
    }
    const int a = c0 + (t - c0) / p.group_tokens * p.group_tokens;
    const int64_t row = int64_t(li) * p.n_tokens + t;
    const int64_t arow = int64_t(li) * p.n_tokens + a;
    const float s = __ldg(p.scales + arow);
    const uint2* a_codes = reinterpret_cast<const uint2*>(p.codes + arow * p.d_model);
    const uint2* r_codes = reinterpret_cast<const uint2*>(p.codes + row * p.d_model);
    uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.d_model);
    for (int v = lane; v < nvec; v += 32) {
      float q[8], y[8];
      unpack_codes(__ldg(a_codes + v), q);
#pragma unroll
      for (int k = 0; k < 8; ++k) y[k] = __fmul_rn(q[k], s);
      if (a != t) {
        float c[8];
        unpack_codes(__ldg(r_codes + v), c);
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = __fadd_rn(y[k], __fmul_rn(c[k], b));
      }
      uint4 o;
      o.x = narrow2<DT>(y[0], y[1]);
      o.y = narrow2<DT>(y[2], y[3]);
      o.z = narrow2<DT>(y[4], y[5]);
      o.w = narrow2<DT>(y[6], y[7]);
      dst[v] = o;
    }
  }
}

}  // namespace

hcr_status check_codec(const hcr_handle* h, const hcr_codec_params* cp, int32_t layer_begin,
                       int32_t layer_end, int32_t n_req, int32_t n_tokens,
                       const int32_t* cu_seqlens, bool* empty) {
  *empty = false;
  if (!h || !cp) return set_last_error(HCR_ERR_INVALID_ARG, "handle and params must be non-NULL");
  const hcr_model_dims& d = h->impl.dims;
  if (layer_begin < 0 || layer_end < layer_begin || layer_end > d.n_layers)
    return set_last_error(HCR_ERR_INVALID_ARG, "layer range [%d, %d) outside [0, %d)",
                          layer_begin, layer_end, d.n_layers);
  if (n_tokens < 0 || n_req < 0)
    return set_last_error(HCR_ERR_INVALID_ARG, "n_tokens and n_req must be >= 0");
  if (cp->group_tokens < 1)
    return set_last_error(HCR_ERR_INVALID_ARG, "group_tokens must be >= 1");
  for (float b : cp->bins)
    if (!(b > 0.f) || !std::isfinite(b))
      return set_last_error(HCR_ERR_INVALID_ARG, "bins must be finite and > 0");
  if (n_tokens == 0 || layer_end == layer_begin) {
    *empty = true;
    return HCR_OK;
  }
  if (n_req < 1) return set_last_error(HCR_ERR_INVALID_ARG, "n_tokens > 0 needs n_req >= 1");
  if (!cu_seqlens) return set_last_error(HCR_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (d.dtype != HCR_DTYPE_BF16 && d.dtype != HCR_DTYPE_FP16)
    return set_last_error(HCR_ERR_UNSUPPORTED, "codec supports bf16 and fp16 hidden states");
  return HCR_OK;
}

namespace {

CodecParams make_params(const hcr_handle* h, const hcr_codec_params* cp, int32_t layer_begin,
                        int32_t n_req, int32_t n_tokens, const int32_t* cu_seqlens) {
  const hcr_model_dims& d = h->impl.dims;
  CodecParams p{};
  p.cu_seqlens = cu_seqlens;
  p.err = h->impl.err;
  p.n_req = n_req;
  p.n_tokens = n_tokens;
  p.d_model = d.d_model;
  p.layer_begin = layer_begin;
  p.n_layers_total = d.n_layers;
  p.group_tokens = cp->group_tokens;
  p.dtype = d.dtype;
  for (int i = 0; i < 3; ++i) p.bins[i] = cp->bins[i];
  return p;
}

dim3 codec_grid(const hcr_handle* h, int32_t n_tokens, int32_t n_layers, int rows_per_warp) {
  // enough warps per layer to keep ~16 resident 256-thread blocks per SM busy
  const int64_t warps = (int64_t(n_tokens) + rows_per_warp - 1) / rows_per_warp * rows_per_warp;
  const int64_t want_x = (warps * 32 + kCodecThreads - 1) / kCodecThreads;
  const int64_t cap_x = std::max<int64_t>(1, int64_t(h->impl.num_sms) * 16 / n_layers);
  return dim3(unsigned(std::max<int64_t>(1, std::min(want_x, cap_x))), unsigned(n_layers));
}

}  // namespace
}  // namespace hcr

using namespace hcr;

extern "C" hcr_status hcr_encode_hidden(hcr_handle* h, const hcr_codec_params* cp,
                                        const void* hidden, int32_t layer_begin,
                                        int32_t layer_end, int32_t n_req, int32_t n_tokens,
                                        const int32_t* cu_seqlens, void* codes, void* scales,
                                        void* stream) {
  NvtxRange range("hcr_encode_hidden");
  bool empty = false;
  hcr_status st = check_codec(h, cp, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, &empty);
  if (st != HCR_OK || empty) return st;
  if (!hidden || !codes || !scales || reinterpret_cast<uintptr_t>(hidden) % 16 ||
      reinterpret_cast<uintptr_t>(codes) % 8 || reinterpret_cast<uintptr_t>(scales) % 4)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "hidden (16-byte), codes (8-byte) and scales (4-byte) must be "
                          "non-NULL and aligned");
  void *dcodes = nullptr, *dscales = nullptr;
  if ((st = device_view(h->impl, codes, "codes", &dcodes)) != HCR_OK) return st;
  if ((st = device_view(h->impl, scales, "scales", &dscales)) != HCR_OK) return st;
  CodecParams p = make_params(h, cp, layer_begin, n_req, n_tokens, cu_seqlens);
  p.hidden = static_cast<const uint16_t*>(hidden);
  p.codes = static_cast<int8_t*>(dcodes);
  p.scales = static_cast<float*>(dscales);
  const int32_t nl = layer_end - layer_begin;
  // one warp per group: at most one group per request plus one per
  // group_tokens tokens
  const int64_t groups = int64_t(n_req) + (int64_t(n_tokens) + cp->group_tokens - 1) /
                                              cp->group_tokens;
  const int64_t blocks = (groups * kWarpsPerGroup * 32 + kCodecThreads - 1) / kCodecThreads;
  if (blocks > INT32_MAX) return set_last_error(HCR_ERR_UNSUPPORTED, "too many groups");
  const dim3 grid{unsigned(blocks), unsigned(nl)};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == HCR_DTYPE_BF16)
    encode_kernel<HCR_DTYPE_BF16><<<grid, kCodecThreads, 0, s>>>(p);
  else
    encode_kernel<HCR_DTYPE_FP16><<<grid, kCodecThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_last_error(HCR_ERR_CUDA, "encode launch: %s", cudaGetErrorString(e));
  return HCR_OK;
}

extern "C" hcr_status hcr_decode_hidden(hcr_handle* h, const hcr_codec_params* cp,
                                        const void* codes, const void* scales,
                                        int32_t layer_begin, int32_t layer_end, int32_t n_req,
                                        int32_t n_tokens, const int32_t* cu_seqlens,
                                        void* hidden, void* stream) {
  NvtxRange range("hcr_decode_hidden");
  bool empty = false;
  hcr_status st = check_codec(h, cp, layer_begin, layer_end, n_req, n_tokens, cu_seqlens, &empty);
  if (st != HCR_OK || empty) return st;
  if (!hidden || !codes || !scales || reinterpret_cast<uintptr_t>(hidden) % 16 ||
      reinterpret_cast<uintptr_t>(codes) % 8 || reinterpret_cast<uintptr_t>(scales) % 4)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "hidden (16-byte), codes (8-byte) and scales (4-byte) must be "
                          "non-NULL and aligned");
  void *dcodes = nullptr, *dscales = nullptr;
  if ((st = device_view(h->impl, const_cast<void*>(codes), "codes", &dcodes)) != HCR_OK)
    return st;
  if ((st = device_view(h->impl, const_cast<void*>(scales), "scales", &dscales)) != HCR_OK)
    return st;
  CodecParams p = make_params(h, cp, layer_begin, n_req, n_tokens, cu_seqlens);
  p.out = static_cast<uint16_t*>(hidden);
  p.codes = static_cast<int8_t*>(dcodes);
  p.scales = static_cast<float*>(dscales);
  const dim3 grid = codec_grid(h, n_tokens, layer_end - layer_begin, 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == HCR_DTYPE_BF16)
    decode_kernel<HCR_DTYPE_BF16><<<grid, kCodecThreads, 0, s>>>(p);
  else
    decode_kernel<HCR_DTYPE_FP16><<<grid, kCodecThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_last_error(HCR_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return HCR_OK;
}
