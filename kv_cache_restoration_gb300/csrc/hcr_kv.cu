// The KV-offload side of a layer-split restore.
//
// HCache episode ("Fast State Restoration for Evicted LLM KV Caches", cue
// 18): the bubble-free scheduler restores most layers from hidden states and
// hands a smaller group of layers to a complementary method.  The one built
// here is KV offload: those layers' K and V rows are kept as they were
// (position-embedded K, as the cache holds it) and copied back.
//
// kv_rows_kernel moves whole rows between the paged cache and a dense store
//     dense[layer][0 = K, 1 = V][token][n_kv_heads * head_dim]
// in the token order of cu_seqlens, through the slot map the restore's
// prepare kernel computes (slot -1 rows are skipped; prepare has flagged
// them).  One warp per row, 16-byte vectors, four in flight per lane; the
// grid strides over rows.  Either side may be device memory or mapped host
// memory.
#include "hcr_host.h"

namespace hcr {
namespace {

constexpr int kKvThreads = 256;

template <bool TO_CACHE>
__global__ void __launch_bounds__(kKvThreads) kv_rows_kernel(const KvRowsParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t(blockIdx.x) * kKvThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kKvThreads) >> 5;
  const int64_t rows = int64_t(p.n_layers) * 2 * p.n_tokens;
  for (int64_t row = warp0; row < rows; row += nwarps) {
    const int64_t t = row % p.n_tokens;
    const int64_t lk = row / p.n_tokens;   // layer * 2 + (0: K, 1: V)
    const int64_t slot = __ldg(p.slot + t);
    if (slot < 0) continue;
    uint4* cache = static_cast<uint4*>((lk & 1) ? p.v_cache : p.k_cache) +
                   (lk >> 1) * p.layer_stride_vecs + slot * p.row_vecs;
    uint4* dense = p.dense + row * p.row_vecs;
#pragma unroll 4
    for (int v = lane; v < p.row_vecs; v += 32) {
      if constexpr (TO_CACHE)
        cache[v] = __ldg(dense + v);
      else
        dense[v] = cache[v];
    }
  }
}

}  // namespace

cudaError_t launch_kv_rows(const KvRowsParams& p, bool to_cache, int num_sms, cudaStream_t s) {
  const int64_t rows = int64_t(p.n_layers) * 2 * p.n_tokens;
  if (rows <= 0) return cudaSuccess;
  const int64_t want = (rows * 32 + kKvThreads - 1) / kKvThreads;
  const int64_t grid = std::min<int64_t>(want, int64_t(num_sms) * 8);
  if (to_cache)
    kv_rows_kernel<true><<<unsigned(grid), kKvThreads, 0, s>>>(p);
  else
    kv_rows_kernel<false><<<unsigned(grid), kKvThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hcr
