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
// for a token count, with CUDA events on the caller's stream.  GPU phase: it
// restores one group of layers from device-resident hidden states and places
// the same layers' K/V, alternately and back to back -- half a second of
// warm-up (at least `reps` rounds), then `reps` timed rounds -- so the costs
// are those of a GPU under sustained load, at the clocks a long restore runs
// at.  Copy phase: `reps` timed host-to-device copies of both kinds.  It allocates (and frees) its own buffers
// and fills the hidden states with a counter-based pseudo-random pattern so
// that the tensor cores see realistic operand switching.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>
#include <vector>

#include "hcr_host.h"

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
  NvtxRange range("hcr_profile_layer_costs");
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
  auto cuda_err = [&](const char* what) {
    cudaGetLastError();
    return set_last_error(HCR_ERR_CUDA, "profiling %s: %s", what, cudaGetErrorString(e));
  };
  // Two ops per phase: GPU work (restore, place) back to back, then copies.
  auto gpu_op = [&](int op) -> hcr_status {
    const int32_t* c = static_cast<int32_t*>(dcu);
    const int32_t* st = static_cast<int32_t*>(dstart);
    const int32_t* tb = static_cast<int32_t*>(dtable);
    return op == 0 ? hcr_restore(h, hidden, 0, nl, n_req, n_tokens, c, st, tb, max_blocks, kc,
                                 vc, &layout, ws, ws_bytes, stream)
                   : hcr_load_kv(h, kv, 0, nl, n_req, n_tokens, c, st, tb, max_blocks, kc, vc,
                                 &layout, ws, ws_bytes, stream);
  };
  auto copy_op = [&](int op) -> cudaError_t {
    return op == 0 ? cudaMemcpyAsync(scratch, hh, hid_bytes, cudaMemcpyHostToDevice, s)
                   : cudaMemcpyAsync(scratch, hkv, kv_bytes, cudaMemcpyHostToDevice, s);
  };
  Events ev;
  for (int i = 0; i < 4 * reps + 2 && e == cudaSuccess; ++i) {
    cudaEvent_t x;
    e = cudaEventCreate(&x);
    if (e == cudaSuccess) ev.ev.push_back(x);
  }
  if (e != cudaSuccess) return cuda_err("events");
  // events: [0, 2*reps) GPU ops (restore, place per rep), [2*reps, 4*reps)
  // copies, and the last two bracket the first GPU round for the warm-up.
  auto elapsed = [&](size_t i0, size_t i1, double* ms) -> bool {
    float f = 0.f;
    e = cudaEventElapsedTime(&f, ev.ev[i0], ev.ev[i1]);
    *ms = f;
    return e == cudaSuccess;
  };
  const size_t w0 = size_t(4) * reps, w1 = w0 + 1;
  hcr_status st = HCR_OK;
  // GPU phase.  Warm up for at least kWarmSeconds of uninterrupted work so
  // the clocks settle where a long restore runs them (a power-capped GPU
  // clocks down under sustained tensor work), then time `reps` rounds with
  // nothing else in between.
  constexpr double kWarmSeconds = 0.5;
  if ((e = cudaEventRecord(ev.ev[w0], s)) != cudaSuccess) return cuda_err("event record");
  if ((st = gpu_op(0)) != HCR_OK || (st = gpu_op(1)) != HCR_OK) return st;
  if ((e = cudaEventRecord(ev.ev[w1], s)) != cudaSuccess) return cuda_err("event record");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_err("sync");
  double round_ms = 0.0;
  if (!elapsed(w0, w1, &round_ms)) return cuda_err("timing");
  const int warm = int(std::min<double>(
      20000.0, std::max<double>(reps, std::ceil(kWarmSeconds * 1e3 / std::max(round_ms, 1e-3)))));
  for (int r = 0; r < warm; ++r)
    if ((st = gpu_op(0)) != HCR_OK || (st = gpu_op(1)) != HCR_OK) return st;
  for (int r = 0; r < reps; ++r) {
    // consecutive events: rep r's restore is [2r, 2r+1), its placement [2r+1, 2r+2)
    if ((e = cudaEventRecord(ev.ev[size_t(2) * r], s)) != cudaSuccess)
      return cuda_err("event record");
    if ((st = gpu_op(0)) != HCR_OK) return st;
    if ((e = cudaEventRecord(ev.ev[size_t(2) * r + 1], s)) != cudaSuccess)
      return cuda_err("event record");
    if ((st = gpu_op(1)) != HCR_OK) return st;
  }
  if ((e = cudaEventRecord(ev.ev[w0], s)) != cudaSuccess) return cuda_err("event record");
  // Copy phase: one untimed round, then `reps` timed rounds.
  for (int op = 0; op < 2; ++op)
    if ((e = copy_op(op)) != cudaSuccess) return cuda_err("copy");
  for (int r = 0; r < reps; ++r)
    for (int op = 0; op < 2; ++op) {
      const size_t i = size_t(2) * reps + size_t(2) * r + op;
      if ((e = cudaEventRecord(ev.ev[i], s)) != cudaSuccess) return cuda_err("event record");
      if ((e = copy_op(op)) != cudaSuccess) return cuda_err("copy");
    }
  if ((e = cudaEventRecord(ev.ev[w1], s)) != cudaSuccess) return cuda_err("event record");
  uint32_t flags = 0;
  st = hcr_check_device_error(h, stream, &flags);   // synchronises the stream
  if (st != HCR_OK) return st;
  double sum[4] = {0, 0, 0, 0};   // restore, place, hidden copy, K/V copy
  for (int r = 0; r < reps; ++r) {
    double ms = 0.0;
    const size_t g = size_t(2) * r;
    // the end of rep r's placement is the start of rep r+1's restore, or the
    // event recorded after the GPU phase
    const size_t g_end = r + 1 < reps ? g + 2 : w0;
    if (!elapsed(g, g + 1, &ms)) return cuda_err("timing");
    sum[0] += ms;
    if (!elapsed(g + 1, g_end, &ms)) return cuda_err("timing");
    sum[1] += ms;
    const size_t c = size_t(2) * reps + g;
    const size_t c_end = r + 1 < reps ? c + 2 : w1;
    if (!elapsed(c, c + 1, &ms)) return cuda_err("timing");
    sum[2] += ms;
    if (!elapsed(c + 1, c_end, &ms)) return cuda_err("timing");
    sum[3] += ms;
  }
  const double per = 1e-3 / (double(reps) * nl);   // ms over reps and layers -> s per layer
  out->restore_s = sum[0] * per;
  out->kv_place_s = sum[1] * per;
  out->hidden_copy_s = sum[2] * per;
  out->kv_copy_s = sum[3] * per;
  return HCR_OK;
}
