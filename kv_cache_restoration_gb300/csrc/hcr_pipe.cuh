// Device-side pieces shared by the projection kernels (hcr_project.cu: the
// token-row tiles; hcr_project_swap.cu: the weight-row tiles): the pipeline's
// barrier state, bounded waits with their diagnostics record, packing to the
// storage type, and the epilogue arithmetic.  The arithmetic is written with
// explicitly rounded intrinsics so that every kernel variant computes the
// same value for a (token, column) bit for bit, whatever the compiler would
// have contracted.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hcr_internal.h"
#include "ptx.cuh"

namespace hcr {
namespace pipe {

struct __align__(8) PipeState {
  uint64_t full[kStagesMax];    // TMA -> MMA: stage filled
  uint64_t empty[kStagesMax];   // MMA -> TMA: stage consumed
  uint64_t tfull[kAccums];   // MMA -> epilogue: accumulator complete
  uint64_t tempty[kAccums];  // epilogue -> MMA: accumulator drained
  uint64_t drain;            // MMA completion on shutdown
  uint64_t tab_full;         // weight-row tiles: the tile's token table is written
  uint64_t tab_free;         // weight-row tiles: every epilogue warp is done with it
  uint64_t slot_full[kSwapSlotsMax];    // weight-row tiles: MMA -> epilogue, per TMEM slot
  uint64_t slot_empty[kSwapSlotsMax];   // weight-row tiles: epilogue -> MMA, per TMEM slot
  uint32_t tmem_base;
  int32_t abort;
};

// Records where a bounded wait gave up (first one wins): which wait, the CTA
// and thread, and two call-site values (tile index, k-block or accumulator).
__device__ __forceinline__ void record_timeout(const ProjectParams& p, uint32_t code,
                                               uint32_t a, uint32_t b, uint32_t parity) {
  atomicOr(p.err, uint32_t(HCR_DEVERR_TIMEOUT));
  uint32_t* d = p.err + kDiagOffset;
  if (atomicCAS(d, 0u, code) == 0u) {
    d[1] = blockIdx.x;
    d[2] = threadIdx.x;
    d[3] = a;
    d[4] = b;
    d[5] = parity;
    __threadfence();
  }
}

// Waits for the phase of `bar` with the given parity.  Gives up when another
// role raised the abort flag or after kWaitLimitNs, raising it itself.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                           const ProjectParams& p, uint32_t code, uint32_t a,
                                           uint32_t b) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_timeout(p, code, a, b, parity);
      return false;
    }
  }
}

// wait_phase whose probes may sleep up to sleep_ns each until the phase
// completes (same bound, same abort and diagnostics).
__device__ __forceinline__ bool wait_phase_sleep(uint32_t bar, uint32_t parity,
                                                 volatile int32_t* abort, const ProjectParams& p,
                                                 uint32_t code, uint32_t a, uint32_t b,
                                                 uint32_t sleep_ns) {
  if (ptx::mbar_try_wait_sleep(bar, parity, sleep_ns)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, sleep_ns)) return true;
    if (*abort) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_timeout(p, code, a, b, parity);
      return false;
    }
  }
}

// Bounded wait for a flag in global memory that another CTA of the same
// kernel sets (with a release store) to a non-zero value; the acquire load
// that sees it orders this thread's later reads after the writer's earlier
// writes.  Same bound, abort and diagnostics as wait_phase.
__device__ __forceinline__ bool wait_flag(const int32_t* flag, volatile int32_t* abort,
                                          const ProjectParams& p, uint32_t code, uint32_t a,
                                          uint32_t b) {
  if (ptx::ld_acquire_gpu(flag) != 0) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    __nanosleep(256);
    if (ptx::ld_acquire_gpu(flag) != 0) return true;
    if (*abort) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_timeout(p, code, a, b, 0);
      return false;
    }
  }
}

// Bounded wait used only while shutting down after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs / 4) return;
  }
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (DT == HCR_DTYPE_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int DT>
__device__ __forceinline__ void store16(uint16_t* dst, const float (&x)[16]) {
  uint4 lo, hi;
  lo.x = pack2<DT>(x[0], x[1]);
  lo.y = pack2<DT>(x[2], x[3]);
  lo.z = pack2<DT>(x[4], x[5]);
  lo.w = pack2<DT>(x[6], x[7]);
  hi.x = pack2<DT>(x[8], x[9]);
  hi.y = pack2<DT>(x[10], x[11]);
  hi.z = pack2<DT>(x[12], x[13]);
  hi.w = pack2<DT>(x[14], x[15]);
  reinterpret_cast<uint4*>(dst)[0] = lo;
  reinterpret_cast<uint4*>(dst)[1] = hi;
}


// Norm scale of one accumulator element: RMSNorm x = acc * rstd; LayerNorm
// (folded) x = rstd * (acc - mean * colsum_j).
__device__ __forceinline__ float norm_scale(float acc, float rstd, float mean, float col_sum,
                                            bool layer_norm) {
  return layer_norm ? __fmul_rn(rstd, __fmaf_rn(-mean, col_sum, acc)) : __fmul_rn(acc, rstd);
}

// Rotate-half RoPE of one pair (a = dim i, b = dim i + dh/2) by the angle
// whose cosine and sine are c and s: (a c - b s, b c + a s).
__device__ __forceinline__ void rope_pair(float& a, float& b, float c, float s) {
  const float a0 = a, b0 = b;
  a = __fmaf_rn(a0, c, __fmul_rn(-b0, s));
  b = __fmaf_rn(b0, c, __fmul_rn(a0, s));
}

}  // namespace pipe
}  // namespace hcr
