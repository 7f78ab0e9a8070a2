// Router: the step before routing/permute. Per token, the top-k experts of
// the router logits and their weights (the workload shapes of the "MXFP4 MoE
// decode kernels" page: top-k softmax for the gpt-oss shapes, sigmoid scores
// renormalised over the chosen k for the GLM shapes, an optional per-expert
// bias added to the logits; the "GLM-5.2 and GLM-5.3 (744B) in MXFP4 on
// Gaudi 2" page names grouped top-k).
//
// Selection runs on x = fp32(logit + bias) (one IEEE addition, the same value
// any fp32 implementation gets; NaN ranks as -inf): the k largest x in order,
// ties to the lower expert index; sigmoid is increasing, so this is the top-k
// by score without ties that the rounding of sigmoid near 1 would add.
// Grouped top-k: n_group equal groups of consecutive ids, a group's score its
// largest x; only the topk_group best groups (ties to the lower group) stay
// eligible. Weights in fp32 from v = x of the chosen (or their unbiased
// logits when the bias steers the choice only): softmax over the chosen v, or
// sigmoid(v) of the chosen over their sum.
//
// One warp per token: lane l holds x of experts l, l + 32, ... (E <= 1024);
// with groups, one warp max per group and topk_group rounds of a warp arg-max
// over the group scores mark the experts of the other groups as taken; then
// k rounds of a warp arg-max over the experts not yet taken; lane r keeps the
// r-th choice and computes its weight.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mxmoe {
namespace {

constexpr int kRouterWarps = 8;

struct Cand {
  float x;
  int e;   // INT32_MAX: no candidate
};

// a before b: larger x, then lower index; "no candidate" last
__device__ __forceinline__ bool before(const Cand& a, const Cand& b) {
  if (a.e == INT32_MAX) return false;
  if (b.e == INT32_MAX) return true;
  return a.x > b.x || (a.x == b.x && a.e < b.e);
}

// NPL: experts per lane (a power of two >= ceil(E / 32)), so every scan is
// exactly as long as the lane's share.
template <int NPL>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E,
                  int topk, int scoring, int n_group, int topk_group, int bias_in_weights,
                  int32_t* __restrict__ ids, float* __restrict__ wts) {
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * kRouterWarps + (threadIdx.x >> 5); t < T;
       t += gridDim.x * kRouterWarps) {
    float x[NPL];
    const float* row = logits + (size_t)t * E;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int e = lane + 32 * j;
      x[j] = 0.f;
      if (e < E) {
        const float v = bias != nullptr ? __fadd_rn(row[e], bias[e]) : row[e];
        x[j] = v != v ? -INFINITY : v;   // NaN ranks as -inf
      }
    }
    uint32_t taken = 0;
    if (n_group > 1) {   // warp-uniform
      const int gs = E / n_group;
      float my_g = -INFINITY;   // lane g < n_group: the score of group g
      for (int g = 0; g < n_group; ++g) {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
          const int e = lane + 32 * j;
          if (e < E && e / gs == g) m = fmaxf(m, x[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == g) my_g = m;
      }
      uint32_t kept = 0;
      for (int r = 0; r < topk_group; ++r) {
        Cand c = {0.f, INT32_MAX};
        if (lane < n_group && !((kept >> lane) & 1u)) c = Cand{my_g, lane};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          Cand d;
          d.x = __shfl_xor_sync(0xffffffffu, c.x, o);
          d.e = __shfl_xor_sync(0xffffffffu, c.e, o);
          if (before(d, c)) c = d;
        }
        kept |= 1u << c.e;
      }
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((kept >> (e / gs)) & 1u)) taken |= 1u << j;
      }
    }
    int my_e = 0;
    float my_x = 0.f;
    for (int r = 0; r < topk; ++r) {
      Cand c = {0.f, INT32_MAX};
#pragma unroll
      for (int j = 0; j < NPL; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u)) {
          const Cand d = {x[j], e};
          if (before(d, c)) c = d;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        Cand d;
        d.x = __shfl_xor_sync(0xffffffffu, c.x, o);
        d.e = __shfl_xor_sync(0xffffffffu, c.e, o);
        if (before(d, c)) c = d;
      }
      if ((c.e & 31) == lane) taken |= 1u << (c.e >> 5);
      if (lane == r) {
        my_e = c.e;
        my_x = c.x;
      }
    }
    // weights of the chosen (lanes 0 .. topk-1)
    if (!bias_in_weights && lane < topk) {   // the unbiased logit of the choice
      const float u = row[my_e];
      my_x = u != u ? -INFINITY : u;
    }
    float vmax = lane < topk ? my_x : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    float v = 0.f;
    if (lane < topk) v = scoring == 0 ? expf(my_x - vmax) : 1.0f / (1.0f + expf(-my_x));
    float sum = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < topk) {
      ids[(size_t)t * topk + lane] = my_e;
      wts[(size_t)t * topk + lane] = v / sum;
    }
  }
}

}  // namespace

cudaError_t launch_router(const float* logits, const float* bias, int T, int E, int topk,
                          int scoring, int n_group, int topk_group, int bias_in_weights,
                          int32_t* ids, float* wts, int num_sms, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  int blocks = (T + kRouterWarps - 1) / kRouterWarps;
  if (blocks > num_sms * 8) blocks = num_sms * 8;
  const int npl = (E + 31) / 32;
#define MXMOE_ROUTER(N)                                                                         \
  router_kernel<N><<<blocks, kRouterWarps * 32, 0, stream>>>(                                  \
      logits, bias, T, E, topk, scoring, n_group, topk_group, bias_in_weights, ids, wts)
  if (npl <= 1) MXMOE_ROUTER(1);
  else if (npl <= 2) MXMOE_ROUTER(2);
  else if (npl <= 4) MXMOE_ROUTER(4);
  else if (npl <= 8) MXMOE_ROUTER(8);
  else if (npl <= 16) MXMOE_ROUTER(16);
  else MXMOE_ROUTER(32);
#undef MXMOE_ROUTER
  return cudaGetLastError();
}

}  // namespace mxmoe
