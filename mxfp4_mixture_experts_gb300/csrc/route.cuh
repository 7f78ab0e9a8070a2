// Routing / permute: a stable counting sort of the routes r = t*topk + j by
// expert ("MXFP4 MoE decode kernels", Design, "Routing inside the kernel":
// a prologue counting-sorts the routes by expert and skips the ones that do
// not belong to a present expert).
//
// Two forms:
//  * cta_route_small: one CTA sorts up to kDecodeMaxRoutes routes into shared
//    memory (used as the prologue of each decode CTA, so the decode call needs
//    no separate routing launch);
//  * route_kernel: one 1024-thread CTA sorts any number of routes into global
//    memory (the mxfp4_moe_route entry point and the prefill path).
// Both are warp-synchronous: __match_any_sync groups equal experts inside a
// warp, a popc of the lower-lane mask gives the stable rank, and a ballot
// compacts the touched-expert list.
#pragma once

#include "common.cuh"

namespace mxmoe {

// Shared-memory routing tables of one CTA.
struct RouteTables {
  int* cnt;      // [E]   routes per expert
  int* off;      // [E+1] exclusive prefix sum
  int* run;      // [E]   scratch: routes already placed
  int* lst;      // [R]   route ids grouped by expert, ascending inside a group
  int* touched;  // [E]   experts with cnt > 0, ascending; first nD entries valid
  int* misc;     // [4]   misc[0] = nD, misc[1] = invalid route count
};

// Local expert of a route id: id - ebase when that lies in [0, E); -1 to skip
// the route (a negative id is padding; with window != 0 every id outside the
// window belongs to another expert-parallel rank); -2 for an invalid id
// (>= E, no window), which is counted.
__device__ __forceinline__ int local_expert(int id, int ebase, int window, int E) {
  const int e = id - ebase;
  if (e >= 0 && e < E) return e;
  return (!window && id >= E) ? -2 : -1;
}

// All threads of the CTA must call this. Ends with __syncthreads().
__device__ __forceinline__ void cta_route_small(const int32_t* __restrict__ ids, int R, int E,
                                                int ebase, int window, RouteTables tb) {
  const int tid = threadIdx.x;
  for (int i = tid; i < E; i += blockDim.x) {
    tb.cnt[i] = 0;
    tb.run[i] = 0;
  }
  if (tid < 4) tb.misc[tid] = 0;
  __syncthreads();
  int inv = 0;
  for (int r = tid; r < R; r += blockDim.x) {
    const int e = local_expert(ids[r], ebase, window, E);
    if (e == -2) ++inv;
    else if (e >= 0) atomicAdd(&tb.cnt[e], 1);   // integer counts: order-independent
  }
  if (inv) atomicAdd(&tb.misc[1], inv);
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const uint32_t lt = lanemask_lt();
    // exclusive scan of the counts and compaction of the touched experts
    int carry = 0, dcarry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? tb.cnt[e] : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) tb.off[e] = carry + x - c;
      carry += __shfl_sync(0xffffffffu, x, 31);
      const uint32_t m = __ballot_sync(0xffffffffu, c > 0);
      if (c > 0) tb.touched[dcarry + __popc(m & lt)] = e;
      dcarry += __popc(m);
    }
    if (lane == 0) {
      tb.off[E] = carry;
      tb.misc[0] = dcarry;
    }
    __syncwarp();
    // stable placement, 32 routes at a time in route order
    for (int base = 0; base < R; base += 32) {
      const int r = base + lane;
      const int e = r < R ? local_expert(ids[r], ebase, window, E) : -1;
      const bool ok = e >= 0;
      const int key = ok ? e : (E + lane);          // invalid lanes stay alone
      const uint32_t grp = __match_any_sync(0xffffffffu, key);
      const int rank = __popc(grp & lt);
      const int before = ok ? tb.run[e] : 0;
      __syncwarp();
      if (ok) {
        tb.lst[tb.off[e] + before + rank] = r;
        if (rank == 0) tb.run[e] = before + __popc(grp);
      }
      __syncwarp();
    }
  }
  __syncthreads();
}

}  // namespace mxmoe
