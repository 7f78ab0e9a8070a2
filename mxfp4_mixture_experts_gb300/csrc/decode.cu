// Decode kernels (1..32 tokens): the routed experts run straight from the
// packed MXFP4 bytes ("MXFP4 MoE decode kernels", Design).
//
// Two launches per layer call:
//   phase 1 (w13): per touched expert, gate and up rows are streamed once,
//                  dequantised in registers, multiplied with the expert's
//                  tokens on the tensor cores (mma.sync m16n8k16, fp32
//                  accumulators) and finished with SwiGLU -> bf16 h [R, I];
//   phase 2 (w2):  per touched expert, the w2 rows are streamed the same way
//                  against h, scaled by the routing weight into fp32 route
//                  outputs P [R, K]; the last contribution to each 16-row
//                  output tile sums the k slots of every token in slot order
//                  and writes bf16 y [T, K].
//
// Work decomposition. A work *item* is (touched expert d, row tile nt, token
// group gr): 16 weight rows against up to 8 of the expert's tokens (phase 1:
// gate rows nt*8..nt*8+7 and the matching up rows, so SwiGLU sees gate and up
// of one output in the same thread; phase 2: w2 rows nt*16..nt*16+15). An item
// has S = ceil(K_red/128) *steps*; in one step a warp consumes 4 scale blocks
// (lane t of each quad owns one 32-value block of one gate/w2 row and of the
// paired up/w2 row). Items are ordered (d, nt, gr) and their steps are dealt to
// warps in equal contiguous ranges ("stream-K"), so every warp streams the same
// number of bytes whatever the routing. An item cut between warps is finished
// by whichever of its warps arrives last (an integer counter per item): it adds
// the fp32 partials in fixed warp order, so the result is deterministic.
//
// Register dequantisation (see e2m1_pair_raw): nibbles p and p+4 of a 32-bit
// word become one bf16x2 A-fragment register, so lane t's physical k indices
// in a step are a fixed permutation of its block; the B fragment (activations)
// is gathered in the same permutation with byte permutes.
#include "common.cuh"
#include "route.cuh"
#include "kernels.h"

namespace mxmoe {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kPrefetch = 4;       // steps of weight bytes in flight per warp
constexpr int kGroup = 8;          // tokens per mma n-tile

struct Cursor {
  int s;    // step inside the item
  int nt;   // row tile
  int gr;   // token group
  int d;    // index into the touched-expert list
  int ng;   // token groups of expert d
  int e;    // expert id
};

struct DecodeCtx {
  const DecodeArgs* a;
  RouteTables tb;
  const int* gbase;   // [nD+1] token-group prefix over touched experts
  int nD, NT, S, nblk, rows_per_e, row_bytes, G;
  // activation rows staged in shared memory: list positions [p_lo, p_lo + nrows)
  const char* stage;
  int p_lo, nrows, stage_stride;
};

__device__ __forceinline__ void cursor_load_expert(Cursor& c, const DecodeCtx& x) {
  if (c.d < x.nD) {
    c.e = x.tb.touched[c.d];
    c.ng = (x.tb.cnt[c.e] + kGroup - 1) / kGroup;
  }
}

// Position of global unit u (item u / S, step u % S).
__device__ __forceinline__ Cursor cursor_at(int64_t u, const DecodeCtx& x) {
  Cursor c;
  const int64_t item = u / x.S;
  c.s = (int)(u - item * x.S);
  // items of expert d start at NT * gbase[d]; find d by binary search
  int lo = 0, hi = x.nD;   // invariant: NT*gbase[lo] <= item < NT*gbase[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)x.NT * x.gbase[mid] <= item) lo = mid; else hi = mid;
  }
  c.d = lo;
  cursor_load_expert(c, x);
  const int local = (int)(item - (int64_t)x.NT * x.gbase[lo]);
  c.nt = local / c.ng;
  c.gr = local - c.nt * c.ng;
  return c;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const DecodeCtx& x) {
  if (++c.s == x.S) {
    c.s = 0;
    if (++c.gr == c.ng) {
      c.gr = 0;
      if (++c.nt == x.NT) {
        c.nt = 0;
        ++c.d;
        cursor_load_expert(c, x);
      }
    }
  }
}

__device__ __forceinline__ int64_t cursor_item(const Cursor& c, const DecodeCtx& x) {
  return (int64_t)x.NT * x.gbase[c.d] + (int64_t)c.nt * c.ng + c.gr;
}

// Weight rows of the item for this lane's quad row g: first row (gate / w2
// row g) and second row (up / w2 row g+8).
template <int PHASE>
__device__ __forceinline__ void item_rows(const Cursor& c, const DecodeCtx& x, int g,
                                          int64_t& r0, int64_t& r1) {
  const DecodeArgs& a = *x.a;
  if (PHASE == 1) {
    r0 = (int64_t)c.e * (2 * a.I) + c.nt * 8 + g;
    r1 = r0 + a.I;
  } else {
    r0 = (int64_t)c.e * a.K + c.nt * 16 + g;
    r1 = r0 + 8;
  }
}

struct Slot {
  uint4 w0, w1;
  uint32_t s0, s1;
};

template <int PHASE>
__device__ __forceinline__ void load_slot(Slot& sl, const Cursor& c, const DecodeCtx& x, int g,
                                          int t) {
  const int b = c.s * 4 + t;
  if (b < x.nblk) {
    int64_t r0, r1;
    item_rows<PHASE>(c, x, g, r0, r1);
    const DecodeArgs& a = *x.a;
    sl.w0 = ldg_stream16(a.wq + r0 * x.row_bytes + b * 16);
    sl.w1 = ldg_stream16(a.wq + r1 * x.row_bytes + b * 16);
    sl.s0 = ldg_u8(a.wsc + r0 * x.nblk + b);
    sl.s1 = ldg_u8(a.wsc + r1 * x.nblk + b);
  } else {
    sl.w0 = make_uint4(0, 0, 0, 0);
    sl.w1 = make_uint4(0, 0, 0, 0);
    sl.s0 = 127;
    sl.s1 = 127;
  }
}

// Pairs of one 16-byte chunk of 8 consecutive activations x[8i..8i+7]:
// (x[8i+p], x[8i+p+4]) for p = 0..3, matching e2m1_pair_raw<p> of word i.
__device__ __forceinline__ uint4 chunk_to_pairs(uint4 v) {
  return make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u),
                    prmt(v.y, v.w, 0x5410u), prmt(v.y, v.w, 0x7632u));
}

// Global source row of list position p (a token row of hidden, or a route row of h).
template <int PHASE>
__device__ __forceinline__ const uint16_t* src_row(const DecodeCtx& x, int p) {
  const DecodeArgs& a = *x.a;
  const int r = x.tb.lst[p];
  if (PHASE == 1) return a.x + (int64_t)(r / a.topk) * a.K;
  return a.x + (int64_t)r * a.I;
}

// Shared-memory layout of a staged row: block b (32 values) takes 64 bytes,
// its 16-byte chunk i (pairs of x[32b+8i .. 32b+8i+7]) sits at position
// i ^ (b & 3), so the four lanes of a quad (consecutive blocks) and two quads
// (row stride = 64 mod 128 bytes) hit distinct banks.
__device__ __forceinline__ int stage_offset(int b, int i) { return b * 64 + ((i ^ (b & 3)) << 4); }

// B fragment pairs of token column g for block b, in [word i][pair p] order.
template <int PHASE>
__device__ __forceinline__ void load_b(uint32_t (&bp)[16], const Cursor& c, const DecodeCtx& x,
                                       int g, int b) {
  const int j = c.gr * kGroup + g;
  if (b < x.nblk && j < x.tb.cnt[c.e]) {
    const int p = x.tb.off[c.e] + j;
    const int idx = p - x.p_lo;
    if (idx >= 0 && idx < x.nrows) {
      const char* row = x.stage + (size_t)idx * x.stage_stride;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + stage_offset(b, i));
        bp[4 * i + 0] = v.x;
        bp[4 * i + 1] = v.y;
        bp[4 * i + 2] = v.z;
        bp[4 * i + 3] = v.w;
      }
    } else {
      // row not staged (shared memory full): read it from L2 and permute here
      const uint4* src = reinterpret_cast<const uint4*>(src_row<PHASE>(x, p) + b * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = chunk_to_pairs(ldcg16(src + i));
        bp[4 * i + 0] = v.x;
        bp[4 * i + 1] = v.y;
        bp[4 * i + 2] = v.z;
        bp[4 * i + 3] = v.w;
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) bp[q] = 0;
  }
}

template <int WI>
__device__ __forceinline__ void mma_word(float (&acc)[4], uint32_t wa, uint32_t wb,
                                         const ScaleMul& ma, const ScaleMul& mb,
                                         const uint32_t (&bp)[16]) {
  const uint32_t a0 = apply_scale(e2m1_pair_raw<0>(wa), ma);
  const uint32_t a1 = apply_scale(e2m1_pair_raw<1>(wa), ma);
  const uint32_t a2 = apply_scale(e2m1_pair_raw<2>(wa), ma);
  const uint32_t a3 = apply_scale(e2m1_pair_raw<3>(wa), ma);
  const uint32_t c0 = apply_scale(e2m1_pair_raw<0>(wb), mb);
  const uint32_t c1 = apply_scale(e2m1_pair_raw<1>(wb), mb);
  const uint32_t c2 = apply_scale(e2m1_pair_raw<2>(wb), mb);
  const uint32_t c3 = apply_scale(e2m1_pair_raw<3>(wb), mb);
  // A rows: g -> word wa, g+8 -> word wb; logical k (2t,2t+1) then (2t+8,2t+9)
  mma_bf16_16816(acc, a0, c0, a1, c1, bp[4 * WI + 0], bp[4 * WI + 1]);
  mma_bf16_16816(acc, a2, c2, a3, c3, bp[4 * WI + 2], bp[4 * WI + 3]);
}

template <int PHASE>
__device__ __forceinline__ void compute_step(float (&acc)[4], const Slot& sl, const Cursor& c,
                                             const DecodeCtx& x, int g, int t) {
  uint32_t bp[16];
  load_b<PHASE>(bp, c, x, g, c.s * 4 + t);
  const ScaleMul ma = scale_mul(sl.s0), mb = scale_mul(sl.s1);
  mma_word<0>(acc, sl.w0.x, sl.w1.x, ma, mb, bp);
  mma_word<1>(acc, sl.w0.y, sl.w1.y, ma, mb, bp);
  mma_word<2>(acc, sl.w0.z, sl.w1.z, ma, mb, bp);
  mma_word<3>(acc, sl.w0.w, sl.w1.w, ma, mb, bp);
}

// Balanced split of U units over NW warps: warp v gets q = U / NW units plus
// one more if v < U % NW, in order. Warps left empty (U < NW) are all at the
// end, so the warps covering one item are always consecutive and non-empty.
__device__ __forceinline__ int64_t range_begin(int v, int64_t U, int NW) {
  const int64_t q = U / NW, rem = U % NW;
  return (int64_t)v * q + (v < rem ? v : rem);
}
__device__ __forceinline__ int warp_of_unit(int64_t u, int64_t U, int NW) {
  const int64_t q = U / NW, rem = U % NW;
  if (u < rem * (q + 1)) return (int)(u / (q + 1));
  return (int)(rem + (u - rem * (q + 1)) / q);
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// Item epilogue, phase 1: SwiGLU of (gate, up) and bf16 store into h.
__device__ __forceinline__ void finish_w13(const float (&acc)[4], const Cursor& c,
                                           const DecodeCtx& x, int g, int t) {
  const DecodeArgs& a = *x.a;
  const int n = c.nt * 8 + g;
  const int ntok = min(kGroup, x.tb.cnt[c.e] - c.gr * kGroup);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int col = 2 * t + q;
    if (col < ntok) {
      const int r = x.tb.lst[x.tb.off[c.e] + c.gr * kGroup + col];
      const float hv = silu_f32(acc[q]) * acc[2 + q];
      reinterpret_cast<uint16_t*>(a.h)[(int64_t)r * a.I + n] = f32_to_bf16_rne(hv);
    }
  }
}

// Item epilogue, phase 2: weighted route outputs, then (last contribution to
// the row tile) the slot-order combine into y.
__device__ __forceinline__ void finish_w2(const float (&acc)[4], const Cursor& c,
                                          const DecodeCtx& x, int g, int t, int lane) {
  const DecodeArgs& a = *x.a;
  const int m0 = c.nt * 16;
  const int ntok = min(kGroup, x.tb.cnt[c.e] - c.gr * kGroup);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int col = 2 * t + q;
    if (col < ntok) {
      const int r = x.tb.lst[x.tb.off[c.e] + c.gr * kGroup + col];
      const float w = a.wts[r];
      a.P[(int64_t)r * a.K + m0 + g] = w * acc[q];
      a.P[(int64_t)r * a.K + m0 + g + 8] = w * acc[2 + q];
    }
  }
  __syncwarp();
  __threadfence();
  int old = 0;
  if (lane == 0) old = atomicAdd(&a.tile_ctr[c.nt], 1);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != x.G - 1) return;
  __threadfence();
  const int k = a.topk;
  for (int idx = lane; idx < a.T * 16; idx += 32) {
    const int tok = idx >> 4;
    const int m = m0 + (idx & 15);
    float s = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int r = tok * k + j;
      const int e = a.ids[r];
      if (e >= 0 && e < a.E) s += ldcg_f32(a.P + (int64_t)r * a.K + m);
    }
    a.y[(int64_t)tok * a.K + m] = f32_to_bf16_rne(s);
  }
  __syncwarp();
  if (lane == 0) a.tile_ctr[c.nt] = 0;
}

template <int PHASE>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs args) {
  extern __shared__ int smem[];
  const DecodeArgs& a = args;
  const int E = a.E;
  const int R = a.T * a.topk;
  RouteTables tb;
  tb.cnt = smem;
  tb.off = tb.cnt + E;
  tb.run = tb.off + E + 1;
  tb.touched = tb.run + E;
  tb.lst = tb.touched + E;
  tb.misc = tb.lst + R;
  int* gbase = tb.misc + 4;   // [E+1]

  // Phase 1 reads inputs that the previous kernel in the stream may produce;
  // phase 2 only needs h after the wait (its routing and weight prefetch use
  // inputs that were complete before phase 1 started).
  if (PHASE == 1) grid_dependency_wait();
  cta_route_small(a.ids, R, E, tb);
  const int nD = tb.misc[0];
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < nD; base += 32) {
      const int d = base + lane;
      const int ng = d < nD ? (tb.cnt[tb.touched[d]] + kGroup - 1) / kGroup : 0;
      int xs = ng;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) xs += y;
      }
      if (d < nD) gbase[d] = carry + xs - ng;
      carry += __shfl_sync(0xffffffffu, xs, 31);
    }
    if (lane == 0) gbase[nD] = carry;
  }
  __syncthreads();
  launch_dependents();

  DecodeCtx x;
  x.a = &a;
  x.tb = tb;
  x.gbase = gbase;
  x.nD = nD;
  x.G = gbase[nD];
  x.NT = PHASE == 1 ? a.I / 8 : a.K / 16;
  const int kred = PHASE == 1 ? a.K : a.I;
  x.nblk = kred / kScaleBlock;
  x.S = (x.nblk + 3) / 4;
  x.rows_per_e = PHASE == 1 ? 2 * a.I : a.K;
  x.row_bytes = kred / 2;

  if (PHASE == 1 && blockIdx.x == 0 && threadIdx.x == 0 && a.status != nullptr) {
    a.status[0] = tb.misc[1];
    a.status[1] = nD;
    a.status[2] = 0;
    a.status[3] = 0;
  }

  const int64_t U = (int64_t)x.NT * x.G * x.S;
  if (U == 0) {
    // no valid route at all: y is zero
    if (PHASE == 2) {
      grid_dependency_wait();
      const int64_t n = (int64_t)a.T * a.K;
      for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
           i += (int64_t)gridDim.x * blockDim.x)
        a.y[i] = 0;
    }
    return;
  }

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int NW = gridDim.x * kDecWarps;
  const int v = blockIdx.x * kDecWarps + warp;
  const int64_t cta_ub = range_begin(blockIdx.x * kDecWarps, U, NW);
  const int64_t cta_ue = range_begin((blockIdx.x + 1) * kDecWarps, U, NW);
  if (cta_ub >= cta_ue) return;     // the whole CTA has no work (U < number of warps)
  const int64_t ub = range_begin(v, U, NW);
  const int64_t ue = range_begin(v + 1, U, NW);

  // Activation rows this CTA can need: every route of the touched experts its
  // unit range covers (a contiguous stretch of the route list).
  {
    const Cursor c0 = cursor_at(cta_ub, x);
    const Cursor c1 = cursor_at(cta_ue - 1, x);
    const int e0 = tb.touched[c0.d], e1 = tb.touched[c1.d];
    x.p_lo = tb.off[e0];
    const int need = tb.off[e1] + tb.cnt[e1] - x.p_lo;
    x.stage_stride = ((kred * 2 + 127) / 128) * 128 + 64;
    const size_t tables = decode_smem_bytes(a.T, a.topk, E);
    const size_t stage_at = (tables + 127) / 128 * 128;
    x.stage = reinterpret_cast<const char*>(smem) + stage_at;
    const int fit = (int)((a.smem_bytes - stage_at) / x.stage_stride);
    x.nrows = need < fit ? need : fit;
  }

  Cursor lc = ub < ue ? cursor_at(ub, x) : cursor_at(cta_ub, x);    // loader
  Cursor cc = lc;                                                    // consumer
  Slot ring[kPrefetch];
#pragma unroll
  for (int q = 0; q < kPrefetch; ++q) {
    if (ub + q < ue) {
      load_slot<PHASE>(ring[q], lc, x, g, t);
      cursor_next(lc, x);
    }
  }
  if (PHASE == 2) grid_dependency_wait();   // h is ready from here on

  // stage: 16-byte chunks, permuted into MMA pair order
  {
    char* st = const_cast<char*>(x.stage);
    const int chunks = kred / 8;
    const int total = x.nrows * chunks;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
      const int row = i / chunks, c16 = i - row * chunks;
      const uint4 v4 = ldcg16(src_row<PHASE>(x, x.p_lo + row) + c16 * 8);
      *reinterpret_cast<uint4*>(st + (size_t)row * x.stage_stride + stage_offset(c16 >> 2, c16 & 3)) =
          chunk_to_pairs(v4);
    }
  }
  __syncthreads();
  if (ub >= ue) return;

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool seg_from_start = (cc.s == 0);   // current segment began at step 0 of its item
  bool first_seg = true;               // current segment is this warp's first
  for (int64_t u = ub; u < ue; u += kPrefetch) {
#pragma unroll
    for (int q = 0; q < kPrefetch; ++q) {
      if (u + q < ue) {
        compute_step<PHASE>(acc, ring[q], cc, x, g, t);
        if (u + q + kPrefetch < ue) {
          load_slot<PHASE>(ring[q], lc, x, g, t);
          cursor_next(lc, x);
        }
        const bool item_end = (cc.s == x.S - 1);
        const bool range_end = (u + q + 1 == ue);
        if (item_end || range_end) {
          const bool whole = seg_from_start && item_end;
          if (whole) {
            if (PHASE == 1) finish_w13(acc, cc, x, g, t);
            else finish_w2(acc, cc, x, g, t, lane);
          } else {
            // partial item: publish, count, and let the last arrival finish
            const int64_t item = cursor_item(cc, x);
            const int va = warp_of_unit(item * x.S, U, NW);
            const int vb = warp_of_unit(item * x.S + x.S - 1, U, NW);
            const int slot = first_seg ? 0 : 1;
            float4* mine = reinterpret_cast<float4*>(a.parts + ((int64_t)v * 2 + slot) * 128);
            mine[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            __syncwarp();
            __threadfence();
            int old = 0;
            if (lane == 0) old = atomicAdd(&a.item_ctr[va], 1);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == vb - va) {
              __threadfence();
              float tot[4] = {0.f, 0.f, 0.f, 0.f};
              const bool va_first = range_begin(va, U, NW) == item * x.S;
              for (int w = va; w <= vb; ++w) {
                const int sl = (w == va && !va_first) ? 1 : 0;
                const uint4 pv = ldcg16(a.parts + ((int64_t)w * 2 + sl) * 128 + lane * 4);
                tot[0] += __uint_as_float(pv.x);
                tot[1] += __uint_as_float(pv.y);
                tot[2] += __uint_as_float(pv.z);
                tot[3] += __uint_as_float(pv.w);
              }
              if (PHASE == 1) finish_w13(tot, cc, x, g, t);
              else finish_w2(tot, cc, x, g, t, lane);
              if (lane == 0) a.item_ctr[va] = 0;
            }
          }
          acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
          seg_from_start = true;
          first_seg = false;
        }
        cursor_next(cc, x);
      }
    }
  }
}


// Raises a kernel's dynamic shared-memory limit only when a launch needs more
// than was granted before (per process; one device per process is assumed for
// the cache, a second device simply repeats the call).
template <typename K>
static cudaError_t ensure_smem(K kernel, size_t bytes, size_t& granted) {
  if (bytes <= 48 * 1024 || bytes <= granted) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) granted = bytes;
  return e;
}

cudaError_t launch_decode(const DecodeArgs& a, int phase, int num_sms, cudaStream_t stream,
                          bool pdl) {
  static size_t granted1 = 0, granted2 = 0;
  const size_t smem = a.smem_bytes;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (phase == 1) {
    cudaError_t e = ensure_smem(decode_kernel<1>, smem, granted1);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, decode_kernel<1>, a);
  }
  cudaError_t e = ensure_smem(decode_kernel<2>, smem, granted2);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_kernel<2>, a);
}

}  // namespace mxmoe
