// Device pieces of the decode kernel kept apart from its main loop: the
// balanced split of work over CTAs, the SwiGLU activations, the grid-wide
// counters of the cooperative launch, and the slot-order combine.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "route.cuh"

namespace mxmoe {

// Balanced split of U units over n CTAs (the first U % n CTAs get one more).
__device__ __forceinline__ int range_begin(int v, int U, int n) {
  const int q = U / n, rem = U % n;
  return v * q + (v < rem ? v : rem);
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// SwiGLU-OAI ("MXFP4 MoE decode kernels", Design, Fused epilogues): gate capped
// at 7 (no lower cap), up clamped to [-7, 7], gate * sigmoid(1.702 gate) *
// (up + 1). Comparisons keep a NaN input NaN.
__device__ __forceinline__ float swiglu_oai_f32(float gate, float up) {
  gate = gate > 7.0f ? 7.0f : gate;
  up = up > 7.0f ? 7.0f : (up < -7.0f ? -7.0f : up);
  return gate / (1.0f + expf(-1.702f * gate)) * (up + 1.0f);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const int* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Order this thread's generic global writes before later async-proxy (bulk
// copy) reads of them by any CTA.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until the grid counter reaches target; false when it gave up.
__device__ __forceinline__ bool grid_wait(const int* ctr, uint32_t target) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    __nanosleep(64);
  }
  return false;
}

// y [T, K] = bf16 of the slot-order (j = 0 .. topk-1) fp32 sum of the
// weighted route outputs P [R, K] of each token's valid routes ("MXFP4 MoE
// decode kernels", Design, "Fused epilogues": the weighted top-k sum). This
// CTA writes an equal contiguous share of the 8-column groups; threads
// tid0, tid0 + nthr, ... of the CTA take part.
__device__ __forceinline__ void combine_share(const DecodeArgs& a, int cta, int nCta, int tid0,
                                              int nthr) {
  const int per_row = a.K / 8;
  if (a.per_route) {   // y [R, K]: each computed route's row, zero rows for skipped routes
    const int total = a.T * a.topk * per_row;
    const int c0 = range_begin(cta, total, nCta);
    const int c1 = range_begin(cta + 1, total, nCta);
    for (int i = c0 + tid0; i < c1; i += nthr) {
      const int r = i / per_row, m8 = (i - r * per_row) * 8;
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (local_expert(a.ids[r], a.ebase, a.window, a.E) >= 0) {
        const uint4 lo = ldcg16(a.P + (size_t)r * a.K + m8);
        const uint4 hi = ldcg16(a.P + (size_t)r * a.K + m8 + 4);
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out.x) : "f"(__uint_as_float(lo.y)), "f"(__uint_as_float(lo.x)));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out.y) : "f"(__uint_as_float(lo.w)), "f"(__uint_as_float(lo.z)));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out.z) : "f"(__uint_as_float(hi.y)), "f"(__uint_as_float(hi.x)));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out.w) : "f"(__uint_as_float(hi.w)), "f"(__uint_as_float(hi.z)));
      }
      *reinterpret_cast<uint4*>(a.y + (size_t)r * a.K + m8) = out;
    }
    return;
  }
  const int total = a.T * per_row;
  const int c0 = range_begin(cta, total, nCta);
  const int c1 = range_begin(cta + 1, total, nCta);
  for (int i = c0 + tid0; i < c1; i += nthr) {
    const int tt = i / per_row, m8 = (i - tt * per_row) * 8;
    float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < a.topk; ++j) {
      const int r = tt * a.topk + j;
      if (local_expert(a.ids[r], a.ebase, a.window, a.E) < 0) continue;
      const uint4 lo = ldcg16(a.P + (size_t)r * a.K + m8);
      const uint4 hi = ldcg16(a.P + (size_t)r * a.K + m8 + 4);
      sum[0] += __uint_as_float(lo.x);
      sum[1] += __uint_as_float(lo.y);
      sum[2] += __uint_as_float(lo.z);
      sum[3] += __uint_as_float(lo.w);
      sum[4] += __uint_as_float(hi.x);
      sum[5] += __uint_as_float(hi.y);
      sum[6] += __uint_as_float(hi.z);
      sum[7] += __uint_as_float(hi.w);
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[q]) : "f"(sum[2 * q + 1]), "f"(sum[2 * q]));
    *reinterpret_cast<uint4*>(a.y + (size_t)tt * a.K + m8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace mxmoe
