// Standalone routing / permute kernel: stable counting sort of any number of
// routes by expert, one 1024-thread CTA. Each warp owns a contiguous segment
// of the routes; per-segment counts give every (segment, expert) its base, so
// the placement pass runs in all 32 warps at once and stays in route order.
#include "common.cuh"
#include "kernels.h"
#include "route.cuh"

namespace mxmoe {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

__global__ void __launch_bounds__(kRouteThreads, 1)
route_kernel(const int32_t* __restrict__ ids, int R, int E, int ebase, int window,
             int32_t* __restrict__ count, int32_t* __restrict__ offset,
             int32_t* __restrict__ list, int32_t* status) {
  extern __shared__ int sm[];
  int* seg = sm;                        // [32][E] per-segment counts, then bases
  int* off = seg + kRouteWarps * E;     // [E+1]
  __shared__ int s_inv, s_nd;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = lanemask_lt();

  grid_dependency_wait();
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) seg[i] = 0;
  if (tid == 0) s_inv = 0;
  __syncthreads();

  const int rb = (int)((int64_t)R * warp / kRouteWarps);
  const int re = (int)((int64_t)R * (warp + 1) / kRouteWarps);
  int* myseg = seg + warp * E;
  int inv = 0;
  for (int base = rb; base < re; base += 32) {
    const int r = base + lane;
    const int e = r < re ? local_expert(ids[r], ebase, window, E) : -1;
    const bool ok = e >= 0;
    if (e == -2) ++inv;
    const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : E + lane);
    if (ok && (grp & lt) == 0) myseg[e] += __popc(grp);
    __syncwarp();
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) inv += __shfl_xor_sync(0xffffffffu, inv, o);
  if (lane == 0 && inv) atomicAdd(&s_inv, inv);
  __syncthreads();

  // per expert: exclusive prefix over segments, total in off[e] (temporarily)
  for (int e = tid; e < E; e += kRouteThreads) {
    int run = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = seg[w * E + e];
      seg[w * E + e] = run;
      run += c;
    }
    off[e] = run;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0, nd = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? off[e] : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) {
        count[e] = c;
        off[e] = carry + x - c;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
      nd += __popc(__ballot_sync(0xffffffffu, c > 0));
    }
    if (lane == 0) {
      off[E] = carry;
      s_nd = nd;
    }
  }
  __syncthreads();

  for (int base = rb; base < re; base += 32) {
    const int r = base + lane;
    const int e = r < re ? local_expert(ids[r], ebase, window, E) : -1;
    const bool ok = e >= 0;
    const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : E + lane);
    const int rank = __popc(grp & lt);
    const int before = ok ? myseg[e] : 0;
    __syncwarp();
    if (ok) {
      list[off[e] + before + rank] = r;
      if (rank == 0) myseg[e] = before + __popc(grp);
    }
    __syncwarp();
  }
  for (int e = tid; e <= E; e += kRouteThreads) offset[e] = off[e];
  for (int p = off[E] + tid; p < R; p += kRouteThreads) list[p] = -1;
  if (tid == 0 && status != nullptr) {
    status[0] = s_inv;
    status[1] = s_nd;
    status[2] = 0;
    status[3] = 0;
  }
}

// ---------------------------------------------------------------------------
// Many routes (the prefill path): the same stable counting sort over up to
// kRoutePartCtas CTAs. Each CTA owns a contiguous chunk of the routes:
//   route_count_kernel  per chunk and expert, the chunk's route count
//                       (part[e][b]) and its invalid ids (part[E][b]);
//   route_scan_kernel   one CTA: per expert, exclusive prefix over the chunks
//                       (a warp per expert), the expert offsets, status;
//                       part[e][b] becomes the position of chunk b's first
//                       route of expert e;
//   route_place_kernel  per chunk, one warp walks its routes in order and
//                       places them (match_any ranks inside each 32 routes).
// ---------------------------------------------------------------------------
constexpr int kPartThreads = 256;

__global__ void __launch_bounds__(kPartThreads)
route_count_kernel(const int32_t* __restrict__ ids, int R, int E, int ebase, int window,
                   int32_t* __restrict__ part) {
  extern __shared__ int cnt[];   // [E]
  __shared__ int s_inv;
  const int B = gridDim.x, b = blockIdx.x, tid = threadIdx.x;
  grid_dependency_wait();
  for (int e = tid; e < E; e += kPartThreads) cnt[e] = 0;
  if (tid == 0) s_inv = 0;
  __syncthreads();
  const int r0 = (int)((int64_t)R * b / B), r1 = (int)((int64_t)R * (b + 1) / B);
  int inv = 0;
  for (int r = r0 + tid; r < r1; r += kPartThreads) {
    const int e = local_expert(ids[r], ebase, window, E);
    if (e >= 0) atomicAdd(&cnt[e], 1);   // integer counts: order-independent
    else if (e == -2) ++inv;
  }
  if (inv) atomicAdd(&s_inv, inv);
  __syncthreads();
  for (int e = tid; e < E; e += kPartThreads) part[(size_t)e * B + b] = cnt[e];
  if (tid == 0) part[(size_t)E * B + b] = s_inv;
}

__global__ void __launch_bounds__(1024, 1)
route_scan_kernel(int R, int E, int B, int32_t* __restrict__ part, int32_t* __restrict__ count,
                  int32_t* __restrict__ offset, int32_t* __restrict__ list, int32_t* status) {
  extern __shared__ int tot[];   // [E + 1]
  __shared__ int s_inv, s_nd;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = lanemask_lt();
  // per expert (a warp each): exclusive prefix of its chunk counts
  for (int e = warp; e <= E; e += 32) {   // row E: the chunks' invalid ids
    int carry = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      const int c = b < B ? part[(size_t)e * B + b] : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (b < B && e < E) part[(size_t)e * B + b] = carry + x - c;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) tot[e] = carry;
  }
  __syncthreads();
  if (warp == 0) {   // expert offsets
    int carry = 0, nd = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? tot[e] : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) {
        count[e] = c;
        offset[e] = carry + x - c;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
      nd += __popc(__ballot_sync(0xffffffffu, c > 0));
    }
    (void)lt;
    if (lane == 0) {
      offset[E] = carry;
      s_inv = tot[E];
      s_nd = nd;
      tot[E] = carry;   // (now the number of placed routes)
    }
  }
  __syncthreads();
  // chunk bases become absolute positions; routes past the placed ones: -1
  for (int i = tid; i < E * B; i += 1024) {
    const int e = i / B;
    part[i] += offset[e];
  }
  for (int p = tot[E] + tid; p < R; p += 1024) list[p] = -1;
  if (tid == 0 && status != nullptr) {
    status[0] = s_inv;
    status[1] = s_nd;
    status[2] = 0;
    status[3] = 0;
  }
}

__global__ void __launch_bounds__(32)
route_place_kernel(const int32_t* __restrict__ ids, int R, int E, int ebase, int window,
                   const int32_t* __restrict__ part, int32_t* __restrict__ list) {
  extern __shared__ int run[];   // [E] next position of each expert in this chunk
  const int B = gridDim.x, b = blockIdx.x, lane = threadIdx.x;
  const uint32_t lt = lanemask_lt();
  for (int e = lane; e < E; e += 32) run[e] = part[(size_t)e * B + b];
  __syncwarp();
  const int r0 = (int)((int64_t)R * b / B), r1 = (int)((int64_t)R * (b + 1) / B);
  for (int base = r0; base < r1; base += 32) {
    const int r = base + lane;
    const int e = r < r1 ? local_expert(ids[r], ebase, window, E) : -1;
    const bool ok = e >= 0;
    const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : E + lane);
    const int rank = __popc(grp & lt);
    const int before = ok ? run[e] : 0;
    __syncwarp();
    if (ok) {
      list[before + rank] = r;
      if (rank == 0) run[e] = before + __popc(grp);
    }
    __syncwarp();
  }
}

size_t route_part_ints(int E) { return (size_t)kRoutePartCtas * (E + 1); }

cudaError_t launch_route_parts(const int32_t* ids, int R, int E, int ebase, int window,
                               int32_t* count, int32_t* offset, int32_t* list, int32_t* status,
                               int32_t* part, cudaStream_t stream) {
  if (R < kRoutePartMin)
    return launch_route(ids, R, E, ebase, window, count, offset, list, status, stream);
  int B = (R + 511) / 512;
  if (B > kRoutePartCtas) B = kRoutePartCtas;
  route_count_kernel<<<B, kPartThreads, sizeof(int) * E, stream>>>(ids, R, E, ebase, window, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  route_scan_kernel<<<1, 1024, sizeof(int) * (E + 1), stream>>>(R, E, B, part, count, offset, list,
                                                                status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  route_place_kernel<<<B, 32, sizeof(int) * E, stream>>>(ids, R, E, ebase, window, part, list);
  return cudaGetLastError();
}

cudaError_t launch_route(const int32_t* ids, int R, int E, int ebase, int window, int32_t* count,
                         int32_t* offset, int32_t* list, int32_t* status, cudaStream_t stream) {
  static size_t granted = 48 * 1024;
  const size_t smem = sizeof(int) * ((size_t)kRouteWarps * E + E + 1);
  if (smem > granted) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    granted = smem;
  }
  route_kernel<<<1, kRouteThreads, smem, stream>>>(ids, R, E, ebase, window, count, offset, list,
                                                   status);
  return cudaGetLastError();
}

}  // namespace mxmoe
