// Decode kernels (1..32 tokens): the routed experts run straight from the
// packed MXFP4 bytes ("MXFP4 MoE decode kernels", Design).
//
// Three launches per layer call (each may start while the previous one
// drains: programmatic dependent launch):
//   phase 1 (w13): per touched expert, gate and up rows are streamed once,
//                  decoded in registers, multiplied with the expert's tokens
//                  on the tensor cores and finished with SwiGLU -> bf16 h [R, I];
//   phase 2 (w2):  per touched expert, the w2 rows are streamed the same way
//                  against h and scaled by the routing weight into fp32 route
//                  outputs P [R, K];
//   combine:       y [T, K] = bf16 of the sum of each token's k route outputs,
//                  in slot order.
//
// CTA = 1 producer warp + 12 consumer warps, one CTA per SM.
//  * The producer streams weight tiles with 2-D TMA (cp.async.bulk.tensor,
//    128-byte swizzle) into a ring of shared-memory stages, and each item's
//    E8M0 scale rows with 1-D bulk copies; mbarriers track both.
//  * Consumers decode E2M1 with the hardware e2m1x2 -> f16x2 conversion
//    (exact), run one m16n8k16 f16 MMA pair per 32-value scale block into a
//    fresh fp32 fragment and fold it into the accumulator with one FFMA by
//    2^(s-127) (exact for every scale byte, 0 and 255 included).
//  * Activations (hidden rows for phase 1, h rows for phase 2) are staged once
//    per CTA in shared memory as f16 after an exact power-of-two prescale per
//    row (max |x| lands in [2^14, 2^15)); the epilogue multiplies it back.
//
// Work decomposition. An *item* is (touched expert d, row tile nt, token
// group gr): 32 weight rows against up to 8 of the expert's tokens (phase 1:
// gate rows 16nt..16nt+15 and the matching up rows; phase 2: w2 rows
// 32nt..32nt+31). Its K range is cut into *chunks* of 48 scale blocks (one
// pipeline stage each). The (item, chunk) units are dealt to CTAs in equal
// contiguous ranges, so every SM streams the same number of bytes whatever
// the routing; an item cut between CTAs is finished by whichever CTA arrives
// last (an integer counter per item), adding the fp32 partials in fixed CTA
// order, so the result is deterministic.
#include <cuda.h>

#include "common.cuh"
#include "route.cuh"
#include "kernels.h"

namespace mxmoe {

constexpr int kConsumerWarps = 12;   // 13 warps: at most 4 per SM sub-partition, 128 registers each
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kGroup = 8;            // tokens per mma n-tile
constexpr int kItemRows = 32;        // weight rows per item (two m16 tiles)
constexpr int kChunkBlocks = 48;     // scale blocks per stage (6 TMA columns of 128 B)
constexpr int kWarpBlocks = kChunkBlocks / kConsumerWarps;   // blocks per consumer warp per stage
constexpr int kStageBytes = kItemRows * kChunkBlocks * 16;   // 24 KB
constexpr int kBoxBytes = 16 * 128;  // one TMA box: 16 rows x 128 bytes
constexpr int kScaleSlots = 3;
constexpr int kBarConsumers = 1;     // named barrier id of the consumer warps
constexpr int kRowBars = 16;         // barriers of the staged activation rows
constexpr uint32_t kRowBarBytes = 32768;   // bytes tracked by one of them (at most)

__host__ __device__ inline size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

// Shared-memory plan (byte offsets from a 1024-byte aligned base).
struct DecodeSmem {
  size_t stage, scale, scale_slot, bars, red, fin, flags, ints, row_sh, xs, total;
};

__host__ __device__ inline DecodeSmem decode_smem_plan(int phase, int T, int K, int I, int E,
                                                       int topk, int stages, int rows_cap,
                                                       int xs_rows, int xs_stride) {
  DecodeSmem m;
  const int kred = phase == 1 ? K : I;
  const int nblk = kred / kScaleBlock;
  const int R = T * topk;
  size_t o = 0;
  m.stage = o;
  o += (size_t)stages * kStageBytes;
  m.scale_slot = round_up((size_t)kItemRows * nblk, 128);
  m.scale = o;
  o += kScaleSlots * m.scale_slot;
  m.bars = o;
  o += round_up((size_t)(2 * stages + 2 * kScaleSlots + kRowBars) * 8, 16);
  m.red = o;
  o += (size_t)kConsumerWarps * 2 * 32 * 4 * sizeof(float);
  m.fin = o;
  o += 256 * sizeof(float);
  m.flags = o;
  o += 32;   // int flags[4] + a 16-byte zero chunk
  m.ints = o;
  o += (size_t)(5 * E + R + 6) * sizeof(int);
  m.row_sh = o;
  o += (size_t)rows_cap * sizeof(int);
  o = round_up(o, 128);
  m.xs = o;
  o += (size_t)xs_rows * xs_stride;
  m.total = o;
  return m;
}

struct Cursor {
  int nt, gr, d, ng, e;
};

struct Ctx {
  RouteTables tb;
  const int* gbase;
  int nD, NT, G;
};

__device__ __forceinline__ void cursor_expert(Cursor& c, const Ctx& x) {
  if (c.d < x.nD) {
    c.e = x.tb.touched[c.d];
    c.ng = (x.tb.cnt[c.e] + kGroup - 1) / kGroup;
  }
}

// Item index -> (d, nt, gr); items of expert d start at NT * gbase[d].
__device__ __forceinline__ Cursor cursor_of_item(int64_t item, const Ctx& x) {
  Cursor c;
  int lo = 0, hi = x.nD;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)x.NT * x.gbase[mid] <= item) lo = mid; else hi = mid;
  }
  c.d = lo;
  cursor_expert(c, x);
  const int local = (int)(item - (int64_t)x.NT * x.gbase[lo]);
  c.nt = local / c.ng;
  c.gr = local - c.nt * c.ng;
  return c;
}

__device__ __forceinline__ void cursor_next_item(Cursor& c, const Ctx& x) {
  if (++c.gr == c.ng) {
    c.gr = 0;
    if (++c.nt == x.NT) {
      c.nt = 0;
      ++c.d;
      cursor_expert(c, x);
    }
  }
}

// Balanced split of U units over n CTAs (first U % n CTAs get one more).
__device__ __forceinline__ int64_t range_begin(int v, int64_t U, int n) {
  const int64_t q = U / n, rem = U % n;
  return (int64_t)v * q + (v < rem ? v : rem);
}
__device__ __forceinline__ int owner_of_unit(int64_t u, int64_t U, int n) {
  const int64_t q = U / n, rem = U % n;
  if (u < rem * (q + 1)) return (int)(u / (q + 1));
  return (int)(rem + (u - rem * (q + 1)) / q);
}

// First weight row of TMA box h (0, 1) of an item.
template <int PHASE>
__device__ __forceinline__ int box_row(const Cursor& c, const DecodeArgs& a, int h) {
  if (PHASE == 1) return c.e * (2 * a.I) + h * a.I + c.nt * 16;
  return c.e * a.K + c.nt * kItemRows + h * 16;
}

// Scale rows of an item into [32][nblk]: phase 1 two runs of 16 rows (gate,
// up), phase 2 one run of 32 rows.
template <int PHASE>
__device__ __forceinline__ void issue_scales(const Cursor& c, const DecodeArgs& a, int nblk,
                                             uint8_t* dst, uint64_t* bar) {
  const uint32_t run = 16u * nblk;
  mbar_arrive_expect_tx(bar, 2 * run);
  if (PHASE == 1) {
    bulk_load_split(dst, a.wsc + (size_t)box_row<1>(c, a, 0) * nblk, run, bar);
    bulk_load_split(dst + run, a.wsc + (size_t)box_row<1>(c, a, 1) * nblk, run, bar);
  } else {
    bulk_load_split(dst, a.wsc + (size_t)box_row<2>(c, a, 0) * nblk, 2 * run, bar);
  }
}

// Activation row (bf16) of route-list position q.
template <int PHASE>
__device__ __forceinline__ const uint16_t* act_row(const DecodeArgs& a, const RouteTables& tb,
                                                   int q) {
  const int r = tb.lst[q];
  if (PHASE == 1) return a.x + (size_t)(r / a.topk) * a.K;
  return a.x + (size_t)r * a.I;
}

__device__ __forceinline__ float pow2f(int e) {   // 2^e, -126 <= e <= 127
  return __uint_as_float((uint32_t)(e + 127) << 23);
}

// 8 bf16 (one uint4) times a power of two -> 8 f16, round to nearest even.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float mul) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16) * mul;
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * mul;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(hi), "f"(lo));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// Epilogue of one item from the 256 reduced values (thread o = consumer
// thread ctid holds output (tile tt, lane l, element q): MMA row
// tt*16 + l/4 + 8*(q/2), token column 2*(l%4) + q%2). All 256 consumer
// threads call it.
template <int PHASE>
__device__ void finish_item(float v, const Cursor& c, const Ctx& x, const DecodeArgs& a,
                            float* fin, int ctid, int p_lo, int n_sh, const int* row_sh,
                            int* flags) {
  const bool own = ctid < 256;     // threads 256.. only join the barriers
  const int tt = (ctid >> 7) & 1, l = (ctid >> 2) & 31, q = ctid & 3;
  const int g = l >> 2, t = l & 3;
  const int col = 2 * t + (q & 1);
  const int ntok = own ? min(kGroup, x.tb.cnt[c.e] - c.gr * kGroup) : 0;
  const int qpos = x.tb.off[c.e] + c.gr * kGroup + col;   // route-list position of the column
  float colmul = 1.0f;
  int r = -1;
  if (col < ntok) {
    r = x.tb.lst[qpos];
    const int idx = qpos - p_lo;
    colmul = pow2f(idx >= 0 && idx < n_sh ? row_sh[idx] : 0);
  }
  if (PHASE == 1) {
    if (own) fin[ctid] = v;
    named_barrier(kBarConsumers, kConsumerThreads);
    if (q < 2 && col < ntok) {
      const float gate = fin[ctid] * colmul, up = fin[ctid + 2] * colmul;
      const int n = c.nt * 16 + tt * 8 + g;
      a.h[(size_t)r * a.I + n] = f32_to_bf16_rne(silu_f32(gate) * up);
    }
  } else {
    // weighted route output; the slot-order sum over each token's routes is
    // done by combine_kernel once every route is complete
    const int m = c.nt * kItemRows + tt * 16 + g + 8 * (q >> 1);
    if (col < ntok) a.P[(size_t)r * a.K + m] = a.wts[r] * (v * colmul);
  }
}

// y[t][m] = bf16( sum over slots j = 0..k-1 with a valid expert of
// P[t*k + j][m] ), in slot order (deterministic). 8 outputs per thread.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ P,
                                                      const int32_t* __restrict__ ids, int T,
                                                      int K, int E, int topk,
                                                      uint16_t* __restrict__ y) {
  grid_dependency_wait();   // P comes from the w2 phase
  const int per_row = K / 8;
  const int64_t n = (int64_t)T * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / per_row), m8 = (int)(i - (int64_t)t * per_row) * 8;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < topk; ++j) {
      const int r = t * topk + j;
      const int e = ids[r];
      if (e < 0 || e >= E) continue;
      const uint4 lo = ldcg16(P + (size_t)r * K + m8);
      const uint4 hi = ldcg16(P + (size_t)r * K + m8 + 4);
      s[0] += __uint_as_float(lo.x);
      s[1] += __uint_as_float(lo.y);
      s[2] += __uint_as_float(lo.z);
      s[3] += __uint_as_float(lo.w);
      s[4] += __uint_as_float(hi.x);
      s[5] += __uint_as_float(hi.y);
      s[6] += __uint_as_float(hi.z);
      s[7] += __uint_as_float(hi.w);
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[q]) : "f"(s[2 * q + 1]), "f"(s[2 * q]));
    *reinterpret_cast<uint4*>(y + (size_t)t * K + m8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Lane-constant shared-memory offsets of the consumer warp's kWarpBlocks
// blocks (bi = cw * kWarpBlocks + j) inside a stage / an item.
struct LaneOffsets {
  int a[kWarpBlocks][2][2];   // A word: [j][tile][row g | row g + 8], from the stage base
  int s[kWarpBlocks][2][2];   // scale byte: [j][tile][row], from the item's scale rows + b_lo
  int b[kWarpBlocks];         // B chunk: from the token row + 64 * b_lo
};

// One stage (chunk) of the current item for one consumer warp, both m16 tiles.
// FAST: the item has no E8M0 byte 0 or 255, so 2^(s-127) is a single shift.
// GLOB: some lane's token row is read (and converted) from global memory.
template <bool FAST, bool GLOB>
__device__ __forceinline__ void consume_stage(float (&acc)[2][4], const uint8_t* stg,
                                              const uint8_t* sc, int b_lo, int nb, int cw,
                                              int t, const LaneOffsets& lo, const uint8_t* brow,
                                              const uint8_t* zero16, const uint16_t* bglob,
                                              float bmul) {
#pragma unroll
  for (int j = 0; j < kWarpBlocks; ++j) {
    if (nb < kChunkBlocks && cw * kWarpBlocks + j >= nb) break;
    // B: token column g, physical k = 32b + 8t .. 32b + 8t + 7 (f16); padding
    // columns read a zero chunk
    uint4 bv;
    if (GLOB && bglob != nullptr) {
      const int b = b_lo + cw * kWarpBlocks + j;
      bv = bf16x8_to_f16x8(ldcg16(bglob + b * 32 + t * 8), bmul);
    } else {
      const uint8_t* bp = brow != nullptr ? brow + b_lo * 64 + lo.b[j] : zero16;
      bv = *reinterpret_cast<const uint4*>(bp);
    }
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(stg + lo.a[j][tt][0]);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(stg + lo.a[j][tt][1]);
      const uint32_t sb0 = sc[b_lo + lo.s[j][tt][0]], sb1 = sc[b_lo + lo.s[j][tt][1]];
      uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
      e2m1x8_to_f16x2(w0, a0, a1, a2, a3);
      e2m1x8_to_f16x2(w1, c0, c1, c2, c3);
      float d[4];
      // k16 slot 0 <- physical (8t, 8t+1), (8t+2, 8t+3); slot 1 <- (8t+4 .. 8t+7)
      mma_f16_16816_z(d, a0, c0, a1, c1, bv.x, bv.y);
      mma_f16_16816(d, a2, c2, a3, c3, bv.z, bv.w);
      const float f0 = FAST ? e8m0_to_f32_normal(sb0) : e8m0_to_f32(sb0);
      const float f1 = FAST ? e8m0_to_f32_normal(sb1) : e8m0_to_f32(sb1);
      acc[tt][0] = fmaf(d[0], f0, acc[tt][0]);
      acc[tt][1] = fmaf(d[1], f0, acc[tt][1]);
      acc[tt][2] = fmaf(d[2], f1, acc[tt][2]);
      acc[tt][3] = fmaf(d[3], f1, acc[tt][3]);
    }
  }
}

// All chunks [ch, ch_end) of one item: wait for each stage, consume, release.
template <bool FAST, bool GLOB>
__device__ __forceinline__ void consume_item(float (&acc)[2][4], uint8_t* stage_base,
                                             uint64_t* full, uint64_t* empty, int S, int& st,
                                             uint32_t& phase, bool& ok, const uint8_t* sc,
                                             int ch, int ch_end, int nblk, int cw, int t,
                                             int lane, const LaneOffsets& lo,
                                             const uint8_t* brow, const uint8_t* zero16,
                                             const uint16_t* bglob, float bmul) {
  for (; ch < ch_end; ++ch) {
    if (ok) ok = mbar_wait(&full[st], phase);
    const int b_lo = ch * kChunkBlocks;
    consume_stage<FAST, GLOB>(acc, stage_base + st * kStageBytes, sc, b_lo,
                              min(kChunkBlocks, nblk - b_lo), cw, t, lo, brow, zero16, bglob,
                              bmul);
    // the stage is refilled by tensor copies (async proxy): order the generic
    // reads of it before that write
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (++st == S) {
      st = 0;
      phase ^= 1u;
    }
  }
}

template <int PHASE>
__global__ void __launch_bounds__(kThreads, 1)
decode_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128-byte swizzled TMA tiles); offsetting the array
  // keeps the compiler's knowledge that these are shared-memory addresses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const DecodeArgs& a = P.a;
  const int E = a.E, R = a.T * a.topk;
  const int kred = PHASE == 1 ? a.K : a.I;
  const int nblk = kred / kScaleBlock;
  const int NC = (nblk + kChunkBlocks - 1) / kChunkBlocks;
  const int S = P.stages;
  const DecodeSmem M = decode_smem_plan(PHASE, a.T, a.K, a.I, E, a.topk, S, P.rows_cap,
                                        P.xs_rows_cap, P.xs_stride);
  uint8_t* stage_base = smem + M.stage;
  uint8_t* scale_base = smem + M.scale;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + M.bars);   // [S]
  uint64_t* empty = full + S;                                     // [S]
  uint64_t* sfull = empty + S;                                    // [kScaleSlots]
  uint64_t* sempty = sfull + kScaleSlots;                         // [kScaleSlots]
  uint64_t* xfull = sempty + kScaleSlots;                         // [kRowBars] staged rows
  float* red = reinterpret_cast<float*>(smem + M.red);            // [warps][2][32][4]
  float* fin = reinterpret_cast<float*>(smem + M.fin);            // [256]
  int* flags = reinterpret_cast<int*>(smem + M.flags);
  RouteTables tb;
  tb.cnt = reinterpret_cast<int*>(smem + M.ints);
  tb.off = tb.cnt + E;
  tb.run = tb.off + E + 1;
  tb.touched = tb.run + E;
  tb.lst = tb.touched + E;
  tb.misc = tb.lst + R;
  int* gbase = tb.misc + 4;                                        // [E+1]
  int* row_sh = reinterpret_cast<int*>(smem + M.row_sh);          // [rows_cap]
  uint8_t* xs_base = smem + M.xs;
  const int xs_stride = P.xs_stride;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (PHASE == 1) grid_dependency_wait();   // inputs may come from the previous kernel
  if (tid < 8) flags[tid] = 0;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kScaleSlots; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], kConsumerWarps);
    }
    for (int i = 0; i < kRowBars; ++i) mbar_init(&xfull[i], 1);
    fence_barrier_init();
    prefetch_tensormap(&P.tmap);
  }
  cta_route_small(a.ids, R, E, tb);   // ends with __syncthreads
  const int nD = tb.misc[0];
  if (tid < 32) {
    int carry = 0;
    for (int base = 0; base < nD; base += 32) {
      const int d = base + lane;
      const int ng = d < nD ? (tb.cnt[tb.touched[d]] + kGroup - 1) / kGroup : 0;
      int xsum = ng;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xsum, o);
        if (lane >= o) xsum += y;
      }
      if (d < nD) gbase[d] = carry + xsum - ng;
      carry += __shfl_sync(0xffffffffu, xsum, 31);
    }
    if (lane == 0) gbase[nD] = carry;
  }
  __syncthreads();
  launch_dependents();

  Ctx x;
  x.tb = tb;
  x.gbase = gbase;
  x.nD = nD;
  x.G = gbase[nD];
  x.NT = PHASE == 1 ? a.I / 16 : a.K / kItemRows;

  if (PHASE == 1 && blockIdx.x == 0 && tid == 0 && a.status != nullptr) {
    a.status[0] = tb.misc[1];
    a.status[1] = nD;
    a.status[2] = 0;
    a.status[3] = 0;
  }

  const int64_t U = (int64_t)x.NT * x.G * NC;
  if (U == 0) return;   // no valid route at all (the combine writes y = 0)
  const int nCta = gridDim.x;
  const int64_t cub = range_begin(blockIdx.x, U, nCta);
  const int64_t cue = range_begin(blockIdx.x + 1, U, nCta);
  if (cub >= cue) return;
  const int64_t i_first = cub / NC, i_last = (cue - 1) / NC;

  // activation rows this CTA can need: every route of the touched experts
  // its unit range covers (a contiguous stretch of the route list)
  const Cursor c_first = cursor_of_item(i_first, x);
  const Cursor c_last = cursor_of_item(i_last, x);
  const int p_lo = tb.off[c_first.e];
  const int p_need = tb.off[c_last.e] + tb.cnt[c_last.e] - p_lo;
  const int n_sh = min(p_need, P.rows_cap);
  // staged rows, tracked by kRowBars barriers of at most kRowBarBytes each
  const int rows_per_bar = max(1, (int)(kRowBarBytes / ((uint32_t)kred * 2)));
  const int xs_rows = min(min(n_sh, P.xs_rows_cap), rows_per_bar * kRowBars);

  // ======================= producer warp =======================
  if (warp == 0) {
    if (lane == 0) {
      // raw bf16 activation rows -> shared memory (converted by the consumers)
      auto issue_rows = [&]() {
        for (int r0 = 0; r0 < xs_rows; r0 += rows_per_bar) {
          const int r1 = min(xs_rows, r0 + rows_per_bar);
          uint64_t* bar = &xfull[r0 / rows_per_bar];
          mbar_arrive_expect_tx(bar, (uint32_t)(r1 - r0) * kred * 2);
          for (int r = r0; r < r1; ++r)
            bulk_load_split(xs_base + (size_t)r * xs_stride, act_row<PHASE>(a, tb, p_lo + r),
                            (uint32_t)kred * 2, bar);
        }
      };
      // Phase 2 issues the h rows once phase 1 is complete, and always before
      // its first blocking wait: the consumers need the rows before they can
      // free any stage or scale slot.
      bool rows_issued = false;
      auto ensure_rows = [&]() {
        if (rows_issued) return;
        if (PHASE == 2) grid_dependency_wait();
        issue_rows();
        rows_issued = true;
      };
      int fail_site = 0;
      if (PHASE == 1) ensure_rows();
      Cursor c = cursor_of_item(i_first, x);
      int ch = (int)(cub - i_first * NC);
      int k = 0, seq = 0, st = 0;
      uint32_t phase = 0;      // parity of the current pass over the stages
      bool ok = true;
      for (int64_t u = cub; u < cue && ok; ++u) {
        if (u == cub || ch == 0) {
          const int slot = seq % kScaleSlots;
          if (seq >= kScaleSlots) {
            ensure_rows();
            ok = mbar_wait(&sempty[slot], ((seq / kScaleSlots) - 1) & 1);
          }
          if (!ok) {
            fail_site |= 1;
            break;
          }
          issue_scales<PHASE>(c, a, nblk, scale_base + slot * M.scale_slot, &sfull[slot]);
          ++seq;
        }
        if (k >= S) {
          ensure_rows();
          ok = mbar_wait(&empty[st], phase ^ 1u);
        }
        if (!ok) {
          fail_site |= 2;
          break;
        }
        uint8_t* dst = stage_base + (size_t)st * kStageBytes;
        // columns of 8 blocks that start inside the row (a partial last
        // column reads zeros past the row end)
        const int ncols = min(kChunkBlocks / 8, (nblk - ch * kChunkBlocks + 7) / 8);
        mbar_arrive_expect_tx(&full[st], ncols * 2 * kBoxBytes);
        const int x0 = ch * kChunkBlocks * 16;
        for (int col = 0; col < ncols; ++col) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(dst + (col * 2 + h) * kBoxBytes, &P.tmap, x0 + col * 128,
                        box_row<PHASE>(c, a, h), &full[st]);
        }
        ++k;
        if (++st == S) {
          st = 0;
          phase ^= 1u;
        }
        if (++ch == NC) {
          ch = 0;
          cursor_next_item(c, x);
        }
      }
      ensure_rows();
      if (fail_site != 0 && a.status != nullptr) {
        atomicOr(&a.status[2], fail_site << (PHASE == 1 ? 0 : 8));
        atomicCAS(&a.status[3], 0, blockIdx.x + 1);
      }
    }
    return;
  }

  // ======================= consumer warps =======================
  const int cw = warp - 1;        // consumer warp 0..7
  const int ctid = tid - 32;      // 0..255
  const int g = lane >> 2, t = lane & 3;


  if (PHASE == 2) grid_dependency_wait();   // h is complete from here on
  bool ok = true;
  int fail_site = 0;
  for (int i = 0; i * rows_per_bar < xs_rows; ++i) ok = ok && mbar_wait(&xfull[i], 0);
  if (!ok) fail_site |= 4;
  // One warp per row: the largest exponent of the row, then (staged rows)
  // conversion in place to f16 with max |x| * 2^-sh in [2^14, 2^15) -- exact
  // in f16 down to 2^-31 of the row maximum. Rows past the staged ones are
  // only scanned (read from global memory when used).
  for (int r = cw; r < n_sh; r += kConsumerWarps) {
    const bool staged = r < xs_rows;
    uint4* row = reinterpret_cast<uint4*>(xs_base + (size_t)r * xs_stride);
    const uint4* src = reinterpret_cast<const uint4*>(act_row<PHASE>(a, tb, p_lo + r));
    uint32_t emax = 0;
    for (int c16 = lane; c16 < kred / 8; c16 += 32) {
      const uint4 v = staged ? row[c16] : ldcg16(src + c16);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        emax = max(emax, (w[i] >> 7) & 0xFFu);
        emax = max(emax, (w[i] >> 23) & 0xFFu);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    const int sh = max(-100, min(100, emax == 0 ? 0 : (int)emax - 127 - 14));
    if (lane == 0) row_sh[r] = sh;
    if (staged) {
      const float mul = pow2f(-sh);
      for (int c16 = lane; c16 < kred / 8; c16 += 32) row[c16] = bf16x8_to_f16x8(row[c16], mul);
    }
  }
  named_barrier(kBarConsumers, kConsumerThreads);

  Cursor c = c_first;
  int64_t item = i_first;
  int st = 0, seq = 0;
  uint32_t phase = 0;
  float acc[2][4];
  LaneOffsets lo;
#pragma unroll
  for (int j = 0; j < kWarpBlocks; ++j) {
    const int bi = cw * kWarpBlocks + j;
    const int colsw = (bi >> 3) * (2 * kBoxBytes) + ((((bi & 7) ^ g) << 4) + (t << 2));
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      if (PHASE == 1) {   // box 0 = gate rows, box 1 = up rows; tile tt = rows tt*8 ..
        lo.a[j][tt][0] = colsw + (tt * 8 + g) * 128;
        lo.a[j][tt][1] = colsw + kBoxBytes + (tt * 8 + g) * 128;
        lo.s[j][tt][0] = (tt * 8 + g) * nblk + bi;
        lo.s[j][tt][1] = (16 + tt * 8 + g) * nblk + bi;
      } else {            // box tt = rows 16tt .. 16tt+15
        lo.a[j][tt][0] = colsw + tt * kBoxBytes + g * 128;
        lo.a[j][tt][1] = colsw + tt * kBoxBytes + (g + 8) * 128;
        lo.s[j][tt][0] = (tt * 16 + g) * nblk + bi;
        lo.s[j][tt][1] = (tt * 16 + g + 8) * nblk + bi;
      }
    }
    lo.b[j] = bi * 64 + t * 16;
  }
  const uint8_t* zero16 = reinterpret_cast<const uint8_t*>(flags + 4);   // B chunk of padding columns

  int ch = (int)(cub - i_first * NC);
  int64_t u = cub;
  while (u < cue) {
    // ---- item start: its scales, the special-byte flag, this lane's B row
    const int slot = seq % kScaleSlots;
    if (ok) {
      ok = mbar_wait(&sfull[slot], (seq / kScaleSlots) & 1);
      if (!ok) fail_site |= 8;
    }
    const uint8_t* sc = scale_base + slot * M.scale_slot;
    int bad = 0;
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(sc);
    for (int i = ctid; i < (kItemRows * nblk) / 4; i += kConsumerThreads) {
      const uint32_t w = sw[i];
      const uint32_t z = (w - 0x01010101u) & ~w & 0x80808080u;     // some byte == 0
      const uint32_t f = (~w - 0x01010101u) & w & 0x80808080u;     // some byte == 0xFF
      bad |= (z | f) != 0u;
    }
    const bool special = named_barrier_or(kBarConsumers, kConsumerThreads, bad != 0);
    const int ntok = min(kGroup, tb.cnt[c.e] - c.gr * kGroup);
    const uint8_t* brow = nullptr;
    const uint16_t* bglob = nullptr;
    float bmul = 1.0f;
    if (g < ntok) {
      const int qpos = tb.off[c.e] + c.gr * kGroup + g;
      const int r = qpos - p_lo;
      if (r >= 0 && r < xs_rows) {
        brow = xs_base + (size_t)r * xs_stride;
      } else {
        bglob = act_row<PHASE>(a, tb, qpos);
        bmul = pow2f(-(r >= 0 && r < n_sh ? row_sh[r] : 0));
      }
    }
    const bool glob = __any_sync(0xffffffffu, bglob != nullptr);
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[tt][q] = 0.f;
    const int ch_end = (int)min((int64_t)NC, ch + (cue - u));
    const int ch_start = ch;
    if (!special && !glob)
      consume_item<true, false>(acc, stage_base, full, empty, S, st, phase, ok, sc, ch, ch_end,
                                nblk, cw, t, lane, lo, brow, zero16, bglob, bmul);
    else if (!special)
      consume_item<true, true>(acc, stage_base, full, empty, S, st, phase, ok, sc, ch, ch_end,
                               nblk, cw, t, lane, lo, brow, zero16, bglob, bmul);
    else
      consume_item<false, true>(acc, stage_base, full, empty, S, st, phase, ok, sc, ch, ch_end,
                                nblk, cw, t, lane, lo, brow, zero16, bglob, bmul);
    u += ch_end - ch_start;

    // ---- item end: reduce the warps' fragments, then finish or publish
    float* my = red + ((size_t)cw * 2 * 32 + lane) * 4;
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
      *reinterpret_cast<float4*>(my + tt * 32 * 4) =
          make_float4(acc[tt][0], acc[tt][1], acc[tt][2], acc[tt][3]);
    named_barrier(kBarConsumers, kConsumerThreads);
    float v = 0.f;
    if (ctid < 256) {
      const int tt = ctid >> 7, l = (ctid >> 2) & 31, q = ctid & 3;
      for (int w = 0; w < kConsumerWarps; ++w) v += red[(((size_t)w * 2 + tt) * 32 + l) * 4 + q];
    }
    const bool whole = (ch_end == NC) && (item * NC >= cub);
    if (whole) {
      finish_item<PHASE>(v, c, x, a, fin, ctid, p_lo, n_sh, row_sh, flags);
    } else {
      // partial item: publish, count, and let the last CTA to arrive finish it
      const int va = owner_of_unit(item * NC, U, nCta);
      const int vb = owner_of_unit(item * NC + NC - 1, U, nCta);
      const int pslot = (item == i_first) ? 0 : 1;
      if (ctid < 256) a.parts[((size_t)blockIdx.x * 2 + pslot) * 256 + ctid] = v;
      named_barrier(kBarConsumers, kConsumerThreads);
      if (ctid == 0) {
        __threadfence();
        flags[1] = atomicAdd(&a.item_ctr[va], 1);
        __threadfence();
      }
      named_barrier(kBarConsumers, kConsumerThreads);
      if (flags[1] == vb - va) {
        const bool va_first = range_begin(va, U, nCta) == item * NC;
        float tot = 0.f;
        for (int w = va; w <= vb && ctid < 256; ++w) {
          const int sl = (w == va && !va_first) ? 1 : 0;
          tot += ldcg_f32(a.parts + ((size_t)w * 2 + sl) * 256 + ctid);
        }
        finish_item<PHASE>(tot, c, x, a, fin, ctid, p_lo, n_sh, row_sh, flags);
        if (ctid == 0) a.item_ctr[va] = 0;
      }
    }
    fence_proxy_async_smem();   // scale slot: refilled by a bulk copy (async proxy)
    named_barrier(kBarConsumers, kConsumerThreads);
    if (lane == 0) mbar_arrive(&sempty[seq % kScaleSlots]);
    ++seq;
    ch = 0;
    ++item;
    cursor_next_item(c, x);
  }
  if (!ok && lane == 0 && a.status != nullptr) {
    atomicOr(&a.status[2], (fail_site | 16) << (PHASE == 1 ? 0 : 8));
    atomicCAS(&a.status[3], 0, blockIdx.x + 1);
  }
}

cudaError_t launch_combine(const float* P, const int32_t* ids, int T, int K, int E, int topk,
                           uint16_t* y, int num_sms, cudaStream_t stream, bool pdl) {
  const int64_t n = (int64_t)T * (K / 8);
  int64_t blocks = (n + 255) / 256;
  if (blocks > (int64_t)num_sms * 4) blocks = (int64_t)num_sms * 4;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, P, ids, T, K, E, topk, y);
}

size_t decode_fixed_smem(int phase, int T, int K, int I, int E, int topk, int stages) {
  return decode_smem_plan(phase, T, K, I, E, topk, stages, T * topk, 0, 0).total + 1024;
}

template <typename Kern>
static cudaError_t ensure_smem(Kern kernel, size_t bytes, size_t& granted) {
  if (bytes <= 48 * 1024 || bytes <= granted) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) granted = bytes;
  return e;
}

cudaError_t launch_decode(const DecodeArgs& a, int phase, int num_sms, int max_smem,
                          const CUtensorMap& tmap, cudaStream_t stream, bool pdl) {
  static size_t granted1 = 0, granted2 = 0;
  DecodeParams p;
  p.tmap = tmap;
  p.a = a;
  const int kred = phase == 1 ? a.K : a.I;
  const int R = a.T * a.topk;
  p.rows_cap = R;
  p.xs_stride = (int)round_up((size_t)kred * 2, 128) + 64;
  // deepest pipeline (up to 5 stages) that still leaves room for a few rows
  int stages = 5;
  size_t fixed = decode_fixed_smem(phase, a.T, a.K, a.I, a.E, a.topk, stages);
  const size_t want_rows = (size_t)(R < 8 ? R : 8) * p.xs_stride;
  while (stages > 3 && fixed + want_rows > (size_t)max_smem) {
    --stages;
    fixed = decode_fixed_smem(phase, a.T, a.K, a.I, a.E, a.topk, stages);
  }
  if (fixed > (size_t)max_smem) return cudaErrorInvalidValue;
  p.stages = stages;
  size_t rows = ((size_t)max_smem - fixed) / p.xs_stride;
  if (rows > (size_t)R) rows = R;
  p.xs_rows_cap = (int)rows;
  const size_t smem = fixed + rows * p.xs_stride;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
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
    return cudaLaunchKernelEx(&cfg, decode_kernel<1>, p);
  }
  cudaError_t e = ensure_smem(decode_kernel<2>, smem, granted2);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_kernel<2>, p);
}

}  // namespace mxmoe
