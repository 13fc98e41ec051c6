// The bubble-free layer split: how many layers to hand to KV offload.
//
// HCache episode ("Fast State Restoration for Evicted LLM KV Caches", cue
// 18): transfer and computation of a restore run in a pipeline, and whichever
// is slower sets the pace while the other idles.  The scheduler splits the
// model's layers into two groups -- most restored from hidden states (a
// hidden-state transfer plus a projection per layer), the rest by a
// complementary method (here KV offload: a K/V transfer plus a placement per
// layer) -- and picks the sizes by a min-max over per-layer costs measured
// offline on the hardware (cue 18, and cue 20 on why the split is by layer,
// not by token).
//
// hcr_plan_layer_split enumerates every split k = 0..L (k layers loaded as
// K/V) and keeps the one with the smallest max(transfer(k), compute(k)),
// where transfer(k) = (L-k)*hidden_copy + k*kv_copy and
// compute(k) = (L-k)*restore + k*kv_place; ties keep the smaller k (K/V take
// more host memory).  It reads no device state.
//
// hcr_profile_layer_costs measures those four per-layer costs on this GPU
// for a token count: it restores one group of layers from device-resident
// hidden states, places the same layers' K/V, and times host-to-device copies
// of both, with CUDA events on the caller's stream, averaged over `reps`
// runs after as many warm-up runs.  It allocates (and frees) its own buffers
// and fills the hidden states with a counter-based pseudo-random pattern so
// that the tensor cores see realistic operand switching.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>
#include <vector>

#include "hcr_internal.h"

namespace hcr {
namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

// Values uniform in [-2, 2), rounded to the storage type.
__global__ void fill_kernel(uint16_t* x, int64_t n, uint64_t seed, int dtype) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const float u = float(splitmix64(seed + uint64_t(i)) >> 40) * (1.0f / 16777216.0f);
    const float v = 4.0f * u - 2.0f;
    if (dtype == HCR_DTYPE_BF16) {
      __nv_bfloat16 b = __float2bfloat16_rn(v);
      x[i] = *reinterpret_cast<uint16_t*>(&b);
    } else {
      __half b = __float2half_rn(v);
      x[i] = *reinterpret_cast<uint16_t*>(&b);
    }
  }
}

bool finite_nonneg(double x) { return std::isfinite(x) && x >= 0.0; }

// Device and pinned host buffers of one profiling run, freed on every path.
struct Buffers {
  std::vector<void*> dev, host;
  ~Buffers() {
    for (void* p : dev) cudaFree(p);
    for (void* p : host) cudaFreeHost(p);
  }
  cudaError_t dalloc(void** p, size_t n) {
    cudaError_t e = cudaMalloc(p, std::max<size_t>(n, 256));
    if (e == cudaSuccess) dev.push_back(*p);
    return e;
  }
  cudaError_t halloc(void** p, size_t n) {
    cudaError_t e = cudaHostAlloc(p, std::max<size_t>(n, 256), cudaHostAllocDefault);
    if (e == cudaSuccess) host.push_back(*p);
    return e;
  }
};

struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
};

}  // namespace
}  // namespace hcr

using namespace hcr;

extern "C" hcr_status hcr_plan_layer_split(const hcr_layer_costs* c, int32_t n_layers,
                                           hcr_layer_split* out) {
  if (!c || !out) return set_last_error(HCR_ERR_INVALID_ARG, "costs and out must be non-NULL");
  if (n_layers < 0) return set_last_error(HCR_ERR_INVALID_ARG, "n_layers must be >= 0");
  if (!finite_nonneg(c->restore_s) || !finite_nonneg(c->hidden_copy_s) ||
      !finite_nonneg(c->kv_copy_s) || !finite_nonneg(c->kv_place_s))
    return set_last_error(HCR_ERR_INVALID_ARG, "costs must be finite and >= 0");
  hcr_layer_split best{};
  best.predicted_s = INFINITY;
  for (int32_t k = 0; k <= n_layers; ++k) {
    const double hidden = double(n_layers - k);
    const double transfer = hidden * c->hidden_copy_s + double(k) * c->kv_copy_s;
    const double compute = hidden * c->restore_s + double(k) * c->kv_place_s;
    const double t = std::max(transfer, compute);
    if (t < best.predicted_s) {
      best.hidden_layers = n_layers - k;
      best.kv_layers = k;
      best.transfer_s = transfer;
      best.compute_s = compute;
      best.predicted_s = t;
    }
  }
  *out = best;
  return HCR_OK;
}

extern "C" hcr_status hcr_profile_layer_costs(hcr_handle* h, int32_t n_tokens,
                                              int32_t layers_per_chunk, int32_t reps,
                                              void* stream, hcr_layer_costs* out) {
  if (!h || !out) return set_last_error(HCR_ERR_INVALID_ARG, "handle and out must be non-NULL");
  if (n_tokens < 1 || layers_per_chunk < 1 || reps < 1)
    return set_last_error(HCR_ERR_INVALID_ARG,
                          "n_tokens, layers_per_chunk and reps must be >= 1");
  const hcr_model_dims& d = h->impl.dims;
  const int32_t nl = std::min(layers_per_chunk, d.n_layers);
  const int64_t T = n_tokens;
  const int64_t d_kv = int64_t(d.n_kv_heads) * d.head_dim;
  // Requests of at most max_position tokens from position 0, contiguous blocks.
  const int32_t kB = 16;
  const int64_t per_req = d.rope != HCR_ROPE_NONE ? std::min<int64_t>(T, d.max_position) : T;
  const int32_t n_req = int32_t((T + per_req - 1) / per_req);
  const int32_t max_blocks = int32_t((per_req + kB - 1) / kB);
  const int32_t num_blocks = n_req * max_blocks;
  std::vector<int32_t> cu(n_req + 1), start(n_req, 0), table(size_t(n_req) * max_blocks);
  for (int32_t r = 0; r <= n_req; ++r) cu[r] = int32_t(std::min<int64_t>(T, r * per_req));
  for (size_t i = 0; i < table.size(); ++i) table[i] = int32_t(i);

  const size_t hid_bytes = size_t(nl) * T * d.d_model * 2;
  const size_t kv_bytes = size_t(nl) * 2 * T * d_kv * 2;
  const size_t cache_bytes = size_t(nl) * num_blocks * kB * d_kv * 2;
  const size_t ws_bytes = hcr_workspace_bytes(h, n_tokens, nl);
  Buffers b;
  void *hidden, *kv, *kc, *vc, *ws, *scratch, *dcu, *dstart, *dtable, *hh, *hkv;
  cudaError_t e = cudaSuccess;
  for (auto [p, n] : {std::pair<void**, size_t>{&hidden, hid_bytes}, {&kv, kv_bytes},
                      {&kc, cache_bytes}, {&vc, cache_bytes}, {&ws, ws_bytes},
                      {&scratch, std::max(hid_bytes, kv_bytes)},
                      {&dcu, cu.size() * 4}, {&dstart, start.size() * 4},
                      {&dtable, table.size() * 4}}) {
    if (e == cudaSuccess) e = b.dalloc(p, n);
  }
  if (e == cudaSuccess) e = b.halloc(&hh, hid_bytes);
  if (e == cudaSuccess) e = b.halloc(&hkv, kv_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_last_error(e == cudaErrorMemoryAllocation ? HCR_ERR_OOM : HCR_ERR_CUDA,
                          "profiling buffers: %s", cudaGetErrorString(e));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::memset(hh, 0x3c, hid_bytes);
  std::memset(hkv, 0x3c, kv_bytes);
  e = cudaMemcpyAsync(dcu, cu.data(), cu.size() * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dstart, start.data(), start.size() * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dtable, table.data(), table.size() * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) {
    const int grid = h->impl.num_sms * 4;
    fill_kernel<<<grid, 256, 0, s>>>(static_cast<uint16_t*>(hidden), int64_t(hid_bytes / 2),
                                     0x5EED, d.dtype);
    fill_kernel<<<grid, 256, 0, s>>>(static_cast<uint16_t*>(kv), int64_t(kv_bytes / 2),
                                     0xC0FFEE, d.dtype);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_last_error(HCR_ERR_CUDA, "profiling setup: %s", cudaGetErrorString(e));
  }
  const hcr_cache_layout layout{num_blocks, kB, 0};
  Events ev;
  const int kOps = 4;   // restore, place, hidden copy, K/V copy
  for (int i = 0; i < 2 * kOps * reps && e == cudaSuccess; ++i) {
    cudaEvent_t x;
    e = cudaEventCreate(&x);
    if (e == cudaSuccess) ev.ev.push_back(x);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_last_error(HCR_ERR_CUDA, "profiling events: %s", cudaGetErrorString(e));
  }
  auto run = [&](int rep, bool timed) -> hcr_status {
    for (int op = 0; op < kOps; ++op) {
      cudaEvent_t* pair = timed ? &ev.ev[size_t(2) * (rep * kOps + op)] : nullptr;
      if (pair && (e = cudaEventRecord(pair[0], s)) != cudaSuccess) break;
      hcr_status st = HCR_OK;
      if (op == 0)
        st = hcr_restore(h, hidden, 0, nl, n_req, n_tokens, static_cast<int32_t*>(dcu),
                         static_cast<int32_t*>(dstart), static_cast<int32_t*>(dtable),
                         max_blocks, kc, vc, &layout, ws, ws_bytes, stream);
      else if (op == 1)
        st = hcr_load_kv(h, kv, 0, nl, n_req, n_tokens, static_cast<int32_t*>(dcu),
                         static_cast<int32_t*>(dstart), static_cast<int32_t*>(dtable),
                         max_blocks, kc, vc, &layout, ws, ws_bytes, stream);
      else if (op == 2)
        e = cudaMemcpyAsync(scratch, hh, hid_bytes, cudaMemcpyHostToDevice, s);
      else
        e = cudaMemcpyAsync(scratch, hkv, kv_bytes, cudaMemcpyHostToDevice, s);
      if (st != HCR_OK) return st;
      if (e != cudaSuccess) break;
      if (pair && (e = cudaEventRecord(pair[1], s)) != cudaSuccess) break;
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return set_last_error(HCR_ERR_CUDA, "profiling run: %s", cudaGetErrorString(e));
    }
    return HCR_OK;
  };
  for (int r = 0; r < reps; ++r) {
    hcr_status st = run(r, false);
    if (st != HCR_OK) return st;
  }
  for (int r = 0; r < reps; ++r) {
    hcr_status st = run(r, true);
    if (st != HCR_OK) return st;
  }
  uint32_t flags = 0;
  hcr_status st = hcr_check_device_error(h, stream, &flags);   // synchronises the stream
  if (st != HCR_OK) return st;
  double sum[kOps] = {0, 0, 0, 0};
  for (int r = 0; r < reps; ++r)
    for (int op = 0; op < kOps; ++op) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, ev.ev[size_t(2) * (r * kOps + op)],
                               ev.ev[size_t(2) * (r * kOps + op) + 1]);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return set_last_error(HCR_ERR_CUDA, "profiling timing: %s", cudaGetErrorString(e));
      }
      sum[op] += ms;
    }
  const double per = 1e-3 / (double(reps) * nl);   // ms over reps and layers -> s per layer
  out->restore_s = sum[0] * per;
  out->kv_place_s = sum[1] * per;
  out->hidden_copy_s = sum[2] * per;
  out->kv_copy_s = sum[3] * per;
  return HCR_OK;
}
