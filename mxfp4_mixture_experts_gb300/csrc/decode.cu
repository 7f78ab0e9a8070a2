// Decode (1..32 tokens): the routed experts run straight from the packed
// MXFP4 bytes ("MXFP4 MoE decode kernels", Design), in ONE cooperative
// launch per layer call:
//
//   phase 1 (w13): per touched expert, every gate/up row is streamed once,
//                  decoded on the fly, multiplied with all of the expert's
//                  tokens on the tensor cores and finished with SwiGLU into
//                  bf16 h [R, I];
//   grid barrier   (h complete; each warp's first w2 stages were issued
//                  before it);
//   phase 2 (w2):  the same over the w2 rows against h, scaled by the routing
//                  weight into fp32 route outputs P [R, K];
//   grid barrier;
//   combine:       y [T, K] = bf16 of the slot-order sum of each token's route
//                  outputs.
//
// One CTA per SM: 10 to 12 consumer warps with 3-deep rings when the
// activation rows a CTA is expected to need fit in shared memory next to the
// rings, else 7 consumer warps and a producer warp, which leave the most room
// for rows (decode_warps). In the 10- to 12-warp forms each consumer warp's
// lane 0 issues its own stages; in the 7 + 1 form the producer's lanes issue
// them for all consumer warps.
//  * Work item = 16 weight rows of one touched expert over the whole
//    reduction (phase 1: gate rows i0..i0+7 and the matching up rows; phase 2:
//    16 w2 rows) times up to 32 of the expert's routes. A phase's items are
//    split into equal contiguous ranges, one per CTA, and a CTA's items are
//    dealt round-robin to its warps: a warp owns whole items, so no partial
//    sums cross warps or CTAs, and the SwiGLU of a gate/up pair happens in the
//    thread that holds both.
//  * Each warp streams its own items: lane 0 keeps the next stages of 16 rows
//    x 256 bytes in flight in the warp's private ring (128-byte swizzle; a
//    whole stage is one 4-D (w13) or 3-D (w2) tensor copy, the last partial
//    stage of a row one copy per 128-byte column), running on into its
//    phase-2 items before h exists, and bulk-copies each item's E8M0 rows
//    into one of the warp's two scale slots. Spreading the issue over all
//    warps keeps enough bytes in flight per SM.
//  * Consumers decode E2M1 with the hardware e2m1x2 -> f16x2 conversion
//    (exact), run one m16n8k16 f16 MMA pair per 32-value block into a fresh
//    fp32 fragment and fold it into the accumulator by 2^(s-127) with two
//    packed fp32 FMAs (exact scales for every byte, 0 and 255 included).
//  * Activations (hidden rows for phase 1, h rows for phase 2) are staged in
//    shared memory by thread 0 (bulk copies) and converted to f16 after an
//    exact power-of-two prescale per row (max |x| lands in [2^14, 2^15)); the
//    epilogue multiplies it back. Rows that do not fit are converted once, with
//    the same prescale, into an f16 scratch in global memory and read from
//    there (generic loads that bypass L1). When a phase needs fewer rows than
//    the CTA has warps, several warps share each row's conversion. Thread 0
//    also waits for the grid between the phases.
#include <cuda.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "route.cuh"
#include "kernels.h"

namespace mxmoe {

// stages in each warp's ring: 3 (a 4-deep ring in the 8-warp form took the
// shared memory that activation rows need: measured slower on every shape)
__host__ __device__ constexpr int ring_depth(int) { return 3; }
constexpr int kRows = 16;                    // weight rows per item (one m16 tile)
constexpr int kChunk = 256;                  // packed bytes per row per stage
constexpr int kChunkBlocks = kChunk / 16;    // 16 scale blocks per stage
constexpr int kStageBytes = kRows * kChunk;  // 4 KB
constexpr int kColBytes = kRows * 128;       // one 128-byte column of a stage

constexpr int kGroup = 8;                    // tokens per mma n-tile
constexpr int kBatch = 32;                   // routes of one expert an item multiplies at most
constexpr int kMaxGroups = kBatch / kGroup;
constexpr int kBarConsumers = 1;             // named barrier of the consumer warps
constexpr int kRowBars = 16;                 // barriers of the staged activation rows
constexpr uint32_t kRowBarBytes = 32768;     // bytes tracked by one of them (at most)
// The form with 7 consumer warps has a producer warp besides them (8 warps in
// all): its lanes issue the consumers' weight stages and scale rows, which the
// consumers hand back through per-slot barriers. Only that form has one.
__host__ __device__ constexpr bool has_producer(int cw) { return cw == 7; }
// polls (32 ns apart) without a copy issued before the producer warp gives up
constexpr uint32_t kProducerIdleLimit = 1u << 24;


__host__ __device__ inline size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

// Shared-memory plan (byte offsets from a 1024-byte aligned base).
struct DecodeSmem {
  size_t ring, scales, bars, flags, ints, eb, row_sh, xs, total;
  int slot_bytes;
};

// cw warps, each with a ring_depth(cw)-stage ring and two scale slots.
__host__ __device__ inline DecodeSmem decode_smem_plan(int cw, int K, int I, int E, int R,
                                                       int xs_rows, int xs_stride) {
  DecodeSmem m;
  const int nblk = (K > I ? K : I) / kScaleBlock;
  size_t o = 0;
  m.ring = o;
  o += (size_t)cw * ring_depth(cw) * kStageBytes;
  m.slot_bytes = (int)round_up((size_t)kRows * nblk, 128);
  m.scales = o;
  o += (size_t)2 * cw * m.slot_bytes;
  m.bars = o;
  o += round_up((size_t)((has_producer(cw) ? 2 : 1) * (cw * ring_depth(cw) + 2 * cw) + kRowBars) * 8,
                16);
  m.flags = o;
  o += 64;   // int flags[16]
  m.ints = o;
  o += (size_t)(5 * E + R + 6) * sizeof(int);
  m.eb = o;
  o += (size_t)(E + kDecodeMaxRoutes / kBatch + 2) * sizeof(int);
  m.row_sh = o;
  o += (size_t)R * sizeof(int);
  o = round_up(o, 128);
  m.xs = o;
  o += (size_t)xs_rows * xs_stride;
  m.total = o;
  return m;
}

// Items a warp owns among n items dealt round-robin to CW warps.
template <int CW>
__device__ __forceinline__ int warp_items(int w, int n) { return n / CW + (w < n % CW ? 1 : 0); }

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

// Largest biased exponent of 8 bf16 values (one uint4).
__device__ __forceinline__ uint32_t bf16x8_max_exponent(uint4 q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t e = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e = max(e, (w[i] >> 7) & 0xFFu);
    e = max(e, (w[i] >> 23) & 0xFFu);
  }
  return e;
}

// An item's routes: expert e, route-list positions q0 .. q0 + cnt - 1 (a batch
// of at most kBatch of the expert's routes; more than one batch per expert
// only when a token names the same expert in several slots).
struct ItemRoutes {
  int e, q0, cnt;
};
__device__ __forceinline__ ItemRoutes item_routes(const RouteTables& tb, const int* eb, int j) {
  ItemRoutes r;
  r.e = eb[j] >> 8;
  const int t0 = (eb[j] & 255) * kBatch;
  r.q0 = tb.off[r.e] + t0;
  r.cnt = min(kBatch, tb.cnt[r.e] - t0);
  return r;
}

// Per-phase view of the CTA's item range.
struct PhaseView {
  int kred, nblk, nc, NB;   // reduction length, scale blocks, stages per item, items per batch
  int ib, n;                // first item and count of this CTA
  int p_lo, n_need;         // route-list positions whose activation rows the items use
  int il;                   // the item's scale rows alternate gate / up (gpt-oss w13)
};

__device__ __forceinline__ PhaseView phase_view(int phase, const DecodeArgs& a,
                                                const RouteTables& tb, const int* eb, int nEB) {
  PhaseView v;
  v.kred = phase == 1 ? a.K : a.I;
  v.nblk = v.kred / kScaleBlock;
  v.nc = (v.kred / 2 + kChunk - 1) / kChunk;
  v.NB = phase == 1 ? a.I / 8 : a.K / kRows;
  v.il = phase == 1 && a.oai != 0;
  const int U = nEB * v.NB;
  v.ib = range_begin(blockIdx.x, U, gridDim.x);
  v.n = range_begin(blockIdx.x + 1, U, gridDim.x) - v.ib;
  v.p_lo = 0;
  v.n_need = 0;
  if (v.n > 0) {
    const ItemRoutes r0 = item_routes(tb, eb, v.ib / v.NB);
    const ItemRoutes r1 = item_routes(tb, eb, (v.ib + v.n - 1) / v.NB);
    v.p_lo = r0.q0;
    v.n_need = r1.q0 + r1.cnt - v.p_lo;
  }
  return v;
}

// Activation row (bf16) of route-list position q.
__device__ __forceinline__ const uint16_t* act_row(int phase, const DecodeArgs& a,
                                                   const RouteTables& tb, int q) {
  const int r = tb.lst[q];
  if (phase == 1) return a.x + (size_t)(r / a.topk) * a.K;
  return a.h + (size_t)r * a.I;
}

// Weight row of item row 0 (half 0) or item row 8 (half 1) of item (e, rb).
// Phase 1: the w13 row group of item row 0 (gate row; its up row is one half
// stride later): row e 2I + i of [gate; up], or pair e I + i of the gpt-oss
// interleaved rows (half ignored). Phase 2: the w2 row of item row 0 / row 8.
__device__ __forceinline__ int item_row(int phase, const DecodeArgs& a, int e, int rb, int half) {
  if (phase == 1) return (a.oai ? e * a.I : e * (2 * a.I)) + rb * 8;
  return e * a.K + rb * kRows + half * 8;
}

// Staged activation rows of a phase and the barriers that track them.
struct RowPlan {
  int xs_rows, rows_per_bar, nbars;
};
__device__ __forceinline__ RowPlan row_plan(const PhaseView& v, int xs_rows_cap) {
  RowPlan r;
  r.rows_per_bar = max(1, (int)(kRowBarBytes / ((uint32_t)v.kred * 2)));
  r.xs_rows = min(min(v.n_need, xs_rows_cap), r.rows_per_bar * kRowBars);
  r.nbars = (r.xs_rows + r.rows_per_bar - 1) / r.rows_per_bar;
  return r;
}

// Converts part of staged activation row r (16-byte chunks c0, c0 + step, ..)
// to f16 after the exact power-of-two prescale that puts the row's largest
// exponent emax at 2^14 (the epilogue multiplies it back): in place when the
// row is staged in shared memory, else into the f16 scratch in global memory.
__device__ __forceinline__ void convert_row_part(const DecodeArgs& a, const PhaseView& v,
                                                 uint8_t* xs, int xs_stride, int* row_sh,
                                                 const RowPlan& rp, const RouteTables& tb,
                                                 int phase, int r, uint32_t emax, int c0, int step,
                                                 bool write_sh) {
  const int sh = max(-100, min(100, emax == 0 ? 0 : (int)emax - 127 - 14));
  if (write_sh) row_sh[r] = sh;
  const float mul = pow2f(-sh);
  if (r < rp.xs_rows) {
    uint4* row = reinterpret_cast<uint4*>(xs + (size_t)r * xs_stride);
    for (int c16 = c0; c16 < v.kred / 8; c16 += step) row[c16] = bf16x8_to_f16x8(row[c16], mul);
  } else {   // rows with no room here: converted once into the f16 scratch
    const size_t xf_stride = (size_t)(a.K > a.I ? a.K : a.I);
    const uint4* src = reinterpret_cast<const uint4*>(act_row(phase, a, tb, v.p_lo + r));
    uint4* dst = reinterpret_cast<uint4*>(a.xf + (size_t)(v.p_lo + r) * xf_stride);
    for (int c16 = c0; c16 < v.kred / 8; c16 += step) dst[c16] = bf16x8_to_f16x8(ldcg16(src + c16), mul);
  }
}

// B operand of one token group for this lane (token column g), at block 0:
// the byte offset of its staged f16 row in the activation area (every row of
// an item staged), or a generic pointer to the row's chunk in shared memory or
// in the f16 scratch in global memory (rows with no room in shared memory,
// converted once with the same prescale). Either advances 64 bytes per block.
// Padding columns (tokens past the item's) read the item's first row; their
// columns are never stored.
struct BRows {
  uint32_t off[kMaxGroups];
  const uint8_t* gp[kMaxGroups];
};

// Token group GR's B row for this lane (token column g of the group, padding
// columns: the item's first row q_first); glob is set when it is not staged.
template <int GR>
__device__ __forceinline__ void set_group(BRows& br, bool& glob, int q_first, int cnt, int g, int t,
                                          int xs_rows, int xs_stride, const uint8_t* xs,
                                          const uint8_t* xf_lo, size_t xf_stride) {
  int q = q_first;
  if (GR * kGroup + g < cnt) q = q_first + GR * kGroup + g;
  const bool staged = q < xs_rows;
  glob |= !staged;
  br.off[GR] = (uint32_t)q * (uint32_t)xs_stride + t * 16;
  br.gp[GR] = staged ? xs + br.off[GR] : xf_lo + (size_t)q * xf_stride * 2;
}

// This lane's activation chunk of token group gr at block b: a shared-memory
// load when every row of the item is staged, else a generic load that stays
// out of L1 (the scratch is rewritten between the phases).
template <bool GLOB>
__device__ __forceinline__ const uint8_t* brow_ptr(const BRows& br, const uint8_t* xs, int gr, int b) {
  return GLOB ? br.gp[gr] + b * 64 : xs + br.off[gr] + b * 64;
}
template <bool GLOB>
__device__ __forceinline__ uint4 load_b16(const uint8_t* p) {
  if constexpr (GLOB) return ld_cg_generic16(p);
  else return *reinterpret_cast<const uint4*>(p);
}

// acc[0..1] += d[0..1] * f0 and acc[2..3] += d[2..3] * f1 as two packed fp32
// FMAs (each lane of a pair rounds like a single FFMA).
__device__ __forceinline__ void fold_block(float (&acc)[4], const float (&d)[4], float f0, float f1) {
  const float2 lo = __ffma2_rn(make_float2(d[0], d[1]), make_float2(f0, f0),
                               make_float2(acc[0], acc[1]));
  const float2 hi = __ffma2_rn(make_float2(d[2], d[3]), make_float2(f1, f1),
                               make_float2(acc[2], acc[3]));
  acc[0] = lo.x;
  acc[1] = lo.y;
  acc[2] = hi.x;
  acc[3] = hi.y;
}

// One 32-value block of one item for one warp: both m16 rows' 4-byte words,
// their scales, and one MMA pair per token group.
template <bool FAST, bool GLOB>
__device__ __forceinline__ void block_mma(float (&acc)[kMaxGroups][4], const uint8_t* stg, int b,
                                          int g, int t, const uint8_t* sc_g, const uint8_t* sc_g8,
                                          int bglob, int ng, const BRows& br, const uint8_t* xs) {
  const int off = (b >> 3) * kColBytes + g * 128 + ((((b & 7) ^ g) << 4) + (t << 2));
  const uint32_t w0 = *reinterpret_cast<const uint32_t*>(stg + off);
  const uint32_t w1 = *reinterpret_cast<const uint32_t*>(stg + off + 8 * 128);
  const uint32_t s0 = sc_g[bglob], s1 = sc_g8[bglob];
  uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
  e2m1x8_to_f16x2(w0, a0, a1, a2, a3);
  e2m1x8_to_f16x2(w1, c0, c1, c2, c3);
  const float f0 = FAST ? e8m0_to_f32_normal(s0) : e8m0_to_f32(s0);
  const float f1 = FAST ? e8m0_to_f32_normal(s1) : e8m0_to_f32(s1);
#pragma unroll
  for (int gr = 0; gr < kMaxGroups; ++gr) {
    if (gr >= ng) break;
    // B: token column g of the group, physical k = 32 bglob + 8t .. +7 (f16)
    const uint4 bv = load_b16<GLOB>(brow_ptr<GLOB>(br, xs, gr, bglob));
    float d[4];
    // k16 slot 0 <- physical (8t, 8t+1), (8t+2, 8t+3); slot 1 <- (8t+4 .. 8t+7)
    mma_f16_16816_z(d, a0, c0, a1, c1, bv.x, bv.y);
    mma_f16_16816(d, a2, c2, a3, c3, bv.z, bv.w);
    fold_block(acc[gr], d, f0, f1);
  }
}

// NBAT consecutive 32-value blocks b0 .. b0+NBAT-1 of a stage (b0 a
// compile-time multiple of 8) for an item with a single token group,
// software-pipelined: every load of the batch is issued before the first
// conversion, and the blocks' MMA chains are independent, so their latencies
// overlap. xo[u] is this lane's byte offset of block (8k + u) inside a
// 128-byte column (row g, 128-byte swizzle); brow / scg / scg8 point at block
// b0's activation chunk (shared memory, or generic when GLOB) and scale bytes.
template <bool FAST, bool GLOB, int NBAT, int B0>
__device__ __forceinline__ void blocks_mma(float (&acc)[4], const uint8_t* stg, const int (&xo)[8],
                                           const uint8_t* scg, const uint8_t* scg8,
                                           const uint8_t* brow) {
  uint32_t w0[NBAT], w1[NBAT], s0[NBAT], s1[NBAT];
  uint4 bv[NBAT];
#pragma unroll
  for (int u = 0; u < NBAT; ++u) {
    const uint8_t* p = stg + ((B0 + u) >> 3) * kColBytes + xo[(B0 + u) & 7];
    w0[u] = *reinterpret_cast<const uint32_t*>(p);
    w1[u] = *reinterpret_cast<const uint32_t*>(p + 8 * 128);
    s0[u] = scg[u];
    s1[u] = scg8[u];
    bv[u] = load_b16<GLOB>(brow + u * 64);
  }
#pragma unroll
  for (int u = 0; u < NBAT; ++u) {
    uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
    e2m1x8_to_f16x2(w0[u], a0, a1, a2, a3);
    e2m1x8_to_f16x2(w1[u], c0, c1, c2, c3);
    const float f0 = FAST ? e8m0_to_f32_normal(s0[u]) : e8m0_to_f32(s0[u]);
    const float f1 = FAST ? e8m0_to_f32_normal(s1[u]) : e8m0_to_f32(s1[u]);
    float d[4];
    mma_f16_16816_z(d, a0, c0, a1, c1, bv[u].x, bv[u].y);
    mma_f16_16816(d, a2, c2, a3, c3, bv[u].z, bv[u].w);
    fold_block(acc, d, f0, f1);
  }
}

// As blocks_mma for an item with NG token groups (batches of NBAT blocks):
// the A words and scales of the batch are loaded once, each group's
// activation chunk per block.
template <bool FAST, bool GLOB, int NG, int NBAT, int B0>
__device__ __forceinline__ void blocks_mma_groups(float (&acc)[kMaxGroups][4], const uint8_t* stg,
                                                  const int (&xo)[8], const uint8_t* scg,
                                                  const uint8_t* scg8, int bg, const BRows& br,
                                                  const uint8_t* xs) {
  uint32_t w0[NBAT], w1[NBAT], s0[NBAT], s1[NBAT];
  uint4 bv[NBAT][NG];
#pragma unroll
  for (int u = 0; u < NBAT; ++u) {
    const uint8_t* p = stg + ((B0 + u) >> 3) * kColBytes + xo[(B0 + u) & 7];
    w0[u] = *reinterpret_cast<const uint32_t*>(p);
    w1[u] = *reinterpret_cast<const uint32_t*>(p + 8 * 128);
    s0[u] = scg[u];
    s1[u] = scg8[u];
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) bv[u][gr] = load_b16<GLOB>(brow_ptr<GLOB>(br, xs, gr, bg + u));
  }
#pragma unroll
  for (int u = 0; u < NBAT; ++u) {
    uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
    e2m1x8_to_f16x2(w0[u], a0, a1, a2, a3);
    e2m1x8_to_f16x2(w1[u], c0, c1, c2, c3);
    const float f0 = FAST ? e8m0_to_f32_normal(s0[u]) : e8m0_to_f32(s0[u]);
    const float f1 = FAST ? e8m0_to_f32_normal(s1[u]) : e8m0_to_f32(s1[u]);
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      float d[4];
      mma_f16_16816_z(d, a0, c0, a1, c1, bv[u][gr].x, bv[u][gr].y);
      mma_f16_16816(d, a2, c2, a3, c3, bv[u][gr].z, bv[u][gr].w);
      fold_block(acc[gr], d, f0, f1);
    }
  }
}

// All 16 blocks of a full stage for NG token groups: batches of 4 blocks for
// two groups, of 2 for three or four (register budget).
template <int CW, bool FAST, bool GLOB, int NG, int B0 = 0>
__device__ __forceinline__ void stage_groups(float (&acc)[kMaxGroups][4], const uint8_t* stg,
                                             const int (&xo)[8], const uint8_t* sc_g,
                                             const uint8_t* sc_g8, int bg, const BRows& br,
                                             const uint8_t* xs) {
  constexpr int NBAT = NG <= 2 ? 4 : 2;
  blocks_mma_groups<FAST, GLOB, NG, NBAT, B0>(acc, stg, xo, sc_g + bg + B0, sc_g8 + bg + B0,
                                              bg + B0, br, xs);
  if constexpr (B0 + NBAT < kChunkBlocks)
    stage_groups<CW, FAST, GLOB, NG, B0 + NBAT>(acc, stg, xo, sc_g, sc_g8, bg, br, xs);
}

// The item sequence of one consumer warp across both phases (items k =
// 0, 1, .. of phase 1, then of phase 2): weight rows of item row 0 / row 8.
struct ItemCursor {
  int phase, k;   // phase 3 = past the last item
  int j, rb;      // expert-batch index and row block of the item (it = j NB + rb)
};
// Positions the cursor on the warp's first item of its phase (one division).
template <int CW>
__device__ __forceinline__ void cursor_locate(ItemCursor& c, const PhaseView& v1,
                                              const PhaseView& v2, int cw) {
  if (c.phase > 2) return;
  const PhaseView& v = c.phase == 1 ? v1 : v2;
  const int it = v.ib + c.k * CW + cw;
  c.j = it / v.NB;
  c.rb = it - c.j * v.NB;
}
template <int CW>
__device__ __forceinline__ void cursor_skip_empty(ItemCursor& c, int n1, int n2,
                                                  const PhaseView& v1, const PhaseView& v2, int cw) {
  bool moved = false;
  while (c.phase <= 2 && c.k >= (c.phase == 1 ? n1 : n2)) {
    ++c.phase;
    c.k = 0;
    moved = true;
  }
  if (moved) cursor_locate<CW>(c, v1, v2, cw);
}
// Next item of the warp: CW items further in the CTA's range.
template <int CW>
__device__ __forceinline__ void cursor_next(ItemCursor& c, int n1, int n2, const PhaseView& v1,
                                            const PhaseView& v2, int cw) {
  const PhaseView& v = c.phase == 1 ? v1 : v2;
  ++c.k;
  c.rb += CW;
  while (c.rb >= v.NB) {
    c.rb -= v.NB;
    ++c.j;
  }
  cursor_skip_empty<CW>(c, n1, n2, v1, v2, cw);
}
__device__ __forceinline__ void cursor_rows(const ItemCursor& c, const DecodeArgs& a,
                                            const int* eb, int& r0, int& r1) {
  const int e = eb[c.j] >> 8;
  r0 = item_row(c.phase, a, e, c.rb, 0);
  r1 = item_row(c.phase, a, e, c.rb, 1);
}

// Position in a warp's KD-stage ring: stage n sits in slot n % KD and is the
// (n / KD)-th use of that slot (phase parity), kept incrementally.
struct RingPos {
  int n, slot;
  uint32_t par;
};
template <int KD>
__device__ __forceinline__ void ring_advance(RingPos& r) {
  ++r.n;
  if (++r.slot == KD) {
    r.slot = 0;
    r.par ^= 1u;
  }
}

// Lane 0 of a consumer warp: issues the warp's weight stages in order into
// its KD-stage ring (tracked by full[slot]).
struct StageIssuer {
  ItemCursor cur;
  RingPos q;
  int c, row0, row1;
};
template <int CW>
__device__ __forceinline__ void issue_stage(StageIssuer& is, const DecodeParams& P,
                                            const PhaseView& v1, const PhaseView& v2, int n1,
                                            int n2, const int* eb, int cw, uint8_t* ring_w,
                                            uint64_t* full_w) {
  if (is.cur.phase > 2) return;
  const PhaseView& v = is.cur.phase == 1 ? v1 : v2;
  if (is.c == 0) cursor_rows(is.cur, P.a, eb, is.row0, is.row1);
  constexpr int KD = ring_depth(CW);
  const int slot = is.q.slot;
  uint8_t* dst = ring_w + slot * kStageBytes;
  uint64_t* bar = &full_w[slot];
  const int x0 = is.c * kChunk;
  if (x0 + kChunk <= v.kred / 2) {   // a whole stage: one copy
    mbar_arrive_expect_tx(bar, (uint32_t)kStageBytes);
    if (is.cur.phase == 1)   // [chunk][gate, up][8 rows][128 bytes]
      tma_load_4d(dst, &P.tmap1q, 0, is.row0, 0, 2 * is.c, bar);
    else                     // [chunk][16 rows][128 bytes]
      tma_load_3d(dst, &P.tmap2q, 0, is.row0, 2 * is.c, bar);
  } else {                           // the last, partial stage: 2-D copies
    const int ncols = min(2, (v.kred / 2 - x0 + 127) / 128);
    mbar_arrive_expect_tx(bar, (uint32_t)ncols * kColBytes);
    for (int col = 0; col < ncols; ++col) {
      if (is.cur.phase == 1) {   // 8 gate rows, then the 8 matching up rows
        tma_load_3d(dst + col * kColBytes, &P.tmap1, x0 + col * 128, is.row0, 0, bar);
      } else {                   // 16 consecutive rows
        tma_load_2d(dst + col * kColBytes, &P.tmap2, x0 + col * 128, is.row0, bar);
      }
    }
  }
  ring_advance<KD>(is.q);
  if (++is.c == v.nc) {
    is.c = 0;
    cursor_next<CW>(is.cur, n1, n2, v1, v2, cw);
  }
}

// Lane 0 of a consumer warp: the scale rows of the item at the cursor into
// the warp's scale slot x (tracked by sfull_w[x]).
__device__ __forceinline__ void issue_scales(const ItemCursor& cur, const DecodeArgs& a,
                                             const PhaseView& v1, const PhaseView& v2,
                                             const int* eb, int cw, uint8_t* dst, uint64_t* bar) {
  const PhaseView& v = cur.phase == 1 ? v1 : v2;
  const uint8_t* wsc = cur.phase == 1 ? a.s13 : a.s2;
  int r0, r1;
  cursor_rows(cur, a, eb, r0, r1);
  const uint32_t run = 8u * v.nblk;   // scale bytes of 8 rows
  mbar_arrive_expect_tx(bar, 2 * run);
  if (cur.phase == 1 && !a.oai) {     // 8 gate rows, then the 8 matching up rows
    bulk_load_split(dst, wsc + (size_t)r0 * v.nblk, run, bar);
    bulk_load_split(dst + run, wsc + ((size_t)r0 + a.I) * v.nblk, run, bar);
  } else {                            // 16 consecutive rows (w2, or gate/up pairs)
    const size_t row = cur.phase == 1 ? 2 * (size_t)r0 : (size_t)r0;
    bulk_load_split(dst, wsc + row * v.nblk, 2 * run, bar);
  }
}

// All stages of one item for one warp; false when a wait gave up. s is the
// warp's running stage number (both phases).
template <int CW, bool FAST, bool GLOB>
__device__ __forceinline__ bool item_stages(float (&acc)[kMaxGroups][4], const int (&xo)[8],
                                            const uint8_t* ring_w,
                                            uint64_t* full_w, RingPos& s, const PhaseView& v,
                                            int lane, const uint8_t* sc, int ng, const BRows& br,
                                            const uint8_t* xs, StageIssuer& is, const DecodeParams& P,
                                            const PhaseView& v1, const PhaseView& v2, int n1,
                                            int n2, const int* eb, int cw, uint64_t* empty_w) {
  constexpr int KD = ring_depth(CW);
  const int g = lane >> 2, t = lane & 3;
  // scale rows of MMA rows g (gate / w2 row g) and g + 8 (up / w2 row g + 8)
  const uint8_t* sc_g = sc + (v.il ? 2 * g : g) * v.nblk;
  const uint8_t* sc_g8 = sc + (v.il ? 2 * g + 1 : g + 8) * v.nblk;
  for (int c = 0; c < v.nc; ++c, ring_advance<KD>(s)) {
    // keep KD - 1 stages ahead: the slot refilled now held stage s - 1, which
    // every lane has finished reading (fenced below)
    if constexpr (!has_producer(CW))
      if (lane == 0) issue_stage<CW>(is, P, v1, v2, n1, n2, eb, cw, const_cast<uint8_t*>(ring_w), full_w);
    const int slot = s.slot;
    if (!__all_sync(0xffffffffu, mbar_wait(&full_w[slot], s.par))) return false;
    const uint8_t* stg = ring_w + slot * kStageBytes;
    const int nb = min(kChunkBlocks, v.nblk - c * kChunkBlocks);
    const int bg = c * kChunkBlocks;   // first block of the stage in the row
    // this lane's activation chunk of block bg (token group 0)
    const uint8_t* brow0 = brow_ptr<GLOB>(br, xs, 0, bg);
    if (ng == 1 && nb == kChunkBlocks && GLOB && CW >= 10) {   // (registers: batches of 4)
#pragma unroll 1
      for (int col = 0; col < 2; ++col) {
        const int b8 = bg + 8 * col;
        blocks_mma<FAST, GLOB, 4, 0>(acc[0], stg + col * kColBytes, xo, sc_g + b8, sc_g8 + b8,
                                     brow0 + col * 8 * 64);
        blocks_mma<FAST, GLOB, 4, 4>(acc[0], stg + col * kColBytes, xo, sc_g + b8 + 4, sc_g8 + b8 + 4,
                                     brow0 + col * 8 * 64 + 4 * 64);
      }
    } else if (ng == 1 && nb == kChunkBlocks) {
      blocks_mma<FAST, GLOB, 8, 0>(acc[0], stg, xo, sc_g + bg, sc_g8 + bg, brow0);
      blocks_mma<FAST, GLOB, 8, 8>(acc[0], stg, xo, sc_g + bg + 8, sc_g8 + bg + 8, brow0 + 8 * 64);
    } else if (ng == 1) {   // partial last stage: a batch of 8 (2 x 4), then single blocks
      int b = 0;
      if (nb >= 8) {
        if (GLOB && CW >= 10) {
          blocks_mma<FAST, GLOB, 4, 0>(acc[0], stg, xo, sc_g + bg, sc_g8 + bg, brow0);
          blocks_mma<FAST, GLOB, 4, 4>(acc[0], stg, xo, sc_g + bg + 4, sc_g8 + bg + 4, brow0 + 4 * 64);
        } else {
          blocks_mma<FAST, GLOB, 8, 0>(acc[0], stg, xo, sc_g + bg, sc_g8 + bg, brow0);
        }
        b = 8;
      }
      for (; b < nb; ++b)
        block_mma<FAST, GLOB>(acc, stg, b, g, t, sc_g, sc_g8, bg + b, ng, br, xs);
    } else if (nb == kChunkBlocks && CW < 10) {   // (the 10- to 12-warp forms have no registers to spare)
      if (ng == 2)
        stage_groups<CW, FAST, GLOB, 2>(acc, stg, xo, sc_g, sc_g8, bg, br, xs);
      else if (ng == 3)
        stage_groups<CW, FAST, GLOB, 3>(acc, stg, xo, sc_g, sc_g8, bg, br, xs);
      else
        stage_groups<CW, FAST, GLOB, 4>(acc, stg, xo, sc_g, sc_g8, bg, br, xs);
    } else if (nb == kChunkBlocks) {
#pragma unroll 4
      for (int b = 0; b < kChunkBlocks; ++b)
        block_mma<FAST, GLOB>(acc, stg, b, g, t, sc_g, sc_g8, bg + b, ng, br, xs);
    } else {
      for (int b = 0; b < nb; ++b)
        block_mma<FAST, GLOB>(acc, stg, b, g, t, sc_g, sc_g8, bg + b, ng, br, xs);
    }
    // the slot is refilled by tensor copies (async proxy): order the generic
    // reads of it before that write (and hand it back to a producer warp)
    fence_proxy_async_smem();
    __syncwarp();
    if constexpr (has_producer(CW))
      if (lane == 0) mbar_arrive(&empty_w[slot]);
  }
  return true;
}

// Stages the activation rows of a phase into shared memory (one thread).
__device__ __forceinline__ void issue_rows(int phase, const PhaseView& v, const RowPlan& rp,
                                           const DecodeArgs& a, const RouteTables& tb, uint8_t* xs,
                                           int xs_stride, uint64_t* xfull) {
  for (int r0 = 0; r0 < rp.xs_rows; r0 += rp.rows_per_bar) {
    const int r1 = min(rp.xs_rows, r0 + rp.rows_per_bar);
    uint64_t* bar = &xfull[r0 / rp.rows_per_bar];
    mbar_arrive_expect_tx(bar, (uint32_t)(r1 - r0) * v.kred * 2);
    for (int r = r0; r < r1; ++r)
      bulk_load_split(xs + (size_t)r * xs_stride, act_row(phase, a, tb, v.p_lo + r),
                      (uint32_t)v.kred * 2, bar);
  }
}

// CW warps, all of them consumers; warp 0's lane 0 also stages the activation
// rows and waits for the grid between the phases.
template <int CW>
__global__ void __launch_bounds__((CW + (has_producer(CW) ? 1 : 0)) * 32, 1)
    decode_kernel(const __grid_constant__ DecodeParams P) {
  constexpr int kThreadsCW = CW * 32;
  constexpr int KD = ring_depth(CW);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128-byte swizzled TMA tiles); offsetting the array
  // keeps the compiler's knowledge that these are shared-memory addresses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const DecodeArgs& a = P.a;
  const int E = a.E, R = a.T * a.topk;
  const DecodeSmem M = decode_smem_plan(CW, a.K, a.I, E, R, P.xs_rows_cap, P.xs_stride);
  uint8_t* ring = smem + M.ring;
  uint8_t* scales = smem + M.scales;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + M.bars);  // [CW][KD] stage landed
  uint64_t* sfull = wfull + CW * KD;                              // [CW][2] scale rows landed
  uint64_t* xfull = sfull + 2 * CW;                               // [kRowBars]
  uint64_t* wempty = xfull + kRowBars;                            // producer form: [CW][KD] consumed
  uint64_t* sempty = wempty + CW * KD;                            // producer form: [CW][2] consumed
  int* flags = reinterpret_cast<int*>(smem + M.flags);
  RouteTables tb;
  tb.cnt = reinterpret_cast<int*>(smem + M.ints);
  tb.off = tb.cnt + E;
  tb.run = tb.off + E + 1;
  tb.touched = tb.run + E;
  tb.lst = tb.touched + E;
  tb.misc = tb.lst + R;
  // flags[0..2]: grid waits passed, expert-batch count; flags[4..15]: the
  // exponent maxima of rows whose conversion several warps share (fewer rows
  // than warps, at most 11)
  int* rmax = flags + 4;
  int* row_sh = reinterpret_cast<int*>(smem + M.row_sh);          // [R]
  int* eb = reinterpret_cast<int*>(smem + M.eb);                  // [nEB] (expert << 8) | batch
  uint8_t* xs = smem + M.xs;
  const int xs_stride = P.xs_stride;
  const size_t xf_stride = (size_t)(a.K > a.I ? a.K : a.I);   // f16 scratch row, elements

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int nCta = gridDim.x;

  if (tid < 16) flags[tid] = 0;
  if (tid == 0) {
    for (int i = 0; i < CW * KD; ++i) mbar_init(&wfull[i], 1);
    for (int i = 0; i < 2 * CW; ++i) mbar_init(&sfull[i], 1);
    if constexpr (has_producer(CW)) {
      for (int i = 0; i < CW * KD; ++i) mbar_init(&wempty[i], 1);
      for (int i = 0; i < 2 * CW; ++i) mbar_init(&sempty[i], 1);
    }
    for (int i = 0; i < kRowBars; ++i) mbar_init(&xfull[i], 1);
    fence_barrier_init();
    prefetch_tensormap(&P.tmap1q);
    prefetch_tensormap(&P.tmap2q);
    prefetch_tensormap(&P.tmap1);
    prefetch_tensormap(&P.tmap2);
  }
  cta_route_small(a.ids, R, E, a.ebase, a.window, tb);   // ends with __syncthreads
  const int nD = tb.misc[0];
  if (warp == 0) {   // expert-batch table: each touched expert's routes in batches of kBatch
    int carry = 0;
    for (int base = 0; base < nD; base += 32) {
      const int d = base + lane;
      const int e = d < nD ? tb.touched[d] : 0;
      const int nb = d < nD ? (tb.cnt[e] + kBatch - 1) / kBatch : 0;
      int x = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      for (int b = 0; b < nb; ++b) eb[carry + x - nb + b] = (e << 8) | b;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) flags[2] = carry;
  }
  __syncthreads();
  const int nEB = flags[2];
  if (blockIdx.x == 0 && tid == 0 && a.status != nullptr) {
    a.status[0] = tb.misc[1];
    a.status[1] = nD;
    a.status[2] = 0;
    a.status[3] = 0;
  }
  const PhaseView v1 = phase_view(1, a, tb, eb, nEB);
  const PhaseView v2 = phase_view(2, a, tb, eb, nEB);
  const RowPlan rp1 = row_plan(v1, P.xs_rows_cap);
  const RowPlan rp2 = row_plan(v2, P.xs_rows_cap);
  int* gbar = a.gbar;   // [0] phase arrivals (two per CTA and call), [1] CTAs done

  if constexpr (has_producer(CW)) {
    if (warp == CW) {
      // ===================== producer warp =====================
      // Lane w issues consumer warp w's weight stages into its KD-stage ring
      // and its items' scale rows into its two scale slots, in the order the
      // warp consumes them, refilling a slot as soon as the warp hands it back
      // (one warp instruction issues for all consumer warps). Phase-2 stages
      // go out before h exists.
      const bool live = lane < CW;
      const int w = live ? lane : 0;
      const int pn1 = warp_items<CW>(w, v1.n), pn2 = warp_items<CW>(w, v2.n);
      uint8_t* ring_p = ring + (size_t)w * KD * kStageBytes;
      uint64_t* full_p = wfull + w * KD;
      uint64_t* empty_p = wempty + w * KD;
      uint8_t* scale_p = scales + (size_t)w * 2 * M.slot_bytes;
      uint64_t* sfull_p = sfull + w * 2;
      uint64_t* sempty_p = sempty + w * 2;
      StageIssuer is;
      is.cur.phase = live ? 1 : 3;
      is.cur.k = 0;
      is.c = 0;
      is.q = {0, 0, 0u};
      is.row0 = is.row1 = 0;
      is.cur.j = is.cur.rb = 0;
      cursor_locate<CW>(is.cur, v1, v2, w);
      cursor_skip_empty<CW>(is.cur, pn1, pn2, v1, v2, w);
      ItemCursor scc = is.cur;   // next item whose scale rows are to be issued
      int nsc = 0;               // scale copies issued
      bool pfail = false;
      uint32_t idle = 0;
      for (;;) {
        bool progress = false;
        if (is.cur.phase <= 2) {   // stage n into slot n % KD once stage n - KD was consumed
          const int n = is.q.n;
          if (n < KD || mbar_test(&empty_p[is.q.slot], (uint32_t)(n / KD - 1) & 1u)) {
            issue_stage<CW>(is, P, v1, v2, pn1, pn2, eb, w, ring_p, full_p);
            progress = true;
          }
        }
        if (scc.phase <= 2) {      // scale copy n into slot n & 1 once item n - 2 is done
          const int x = nsc & 1;
          if (nsc < 2 || mbar_test(&sempty_p[x], (uint32_t)((nsc >> 1) - 1) & 1u)) {
            issue_scales(scc, a, v1, v2, eb, w, scale_p + x * M.slot_bytes, &sfull_p[x]);
            ++nsc;
            cursor_next<CW>(scc, pn1, pn2, v1, v2, w);
            progress = true;
          }
        }
        if (__all_sync(0xffffffffu, is.cur.phase > 2 && scc.phase > 2)) break;
        if (__any_sync(0xffffffffu, progress)) {
          idle = 0;
        } else {
          __nanosleep(32);
          if (++idle > kProducerIdleLimit) {   // the consumers stopped taking stages
            pfail = true;
            break;
          }
        }
      }
      // every copy issued lands before the CTA can exit
      if (live) {
        for (int n = max(0, is.q.n - KD); n < is.q.n; ++n)
          mbar_wait(&full_p[n % KD], (uint32_t)(n / KD) & 1u);
        for (int n = max(0, nsc - 2); n < nsc; ++n)
          mbar_wait(&sfull_p[n & 1], (uint32_t)(n >> 1) & 1u);
      }
      if (pfail && lane == 0 && a.status != nullptr) {
        atomicOr(&a.status[2], 1);
        atomicCAS(&a.status[3], 0, blockIdx.x + 1);
      }
      return;
    }
  }

  // ======================= consumer warps =======================
  const int cw = warp;
  const int ctid = tid;
  if (ctid == 0) issue_rows(1, v1, rp1, a, tb, xs, xs_stride, xfull);
  const int g = lane >> 2, t = lane & 3;
  int xo[8];   // byte offset of this lane's word of block u (0..7) in a 128-byte column
#pragma unroll
  for (int u = 0; u < 8; ++u) xo[u] = g * 128 + (((u ^ g) << 4) + (t << 2));
  uint8_t* ring_w = ring + (size_t)cw * KD * kStageBytes;
  uint64_t* full_w = wfull + cw * KD;
  uint64_t* empty_w = wempty + cw * KD;   // (producer form)
  uint64_t* sfull_w = sfull + cw * 2;
  uint64_t* sempty_w = sempty + cw * 2;   // (producer form)
  uint8_t* scale_w = scales + (size_t)cw * 2 * M.slot_bytes;
  const int n1 = warp_items<CW>(cw, v1.n), n2 = warp_items<CW>(cw, v2.n);
  bool ok = true;
  int fail = 0;
  RingPos s = {0, 0, 0u};    // running stage of this warp
  int kitems = 0;            // items this warp has started
  uint32_t rows_used = 0;    // staged-row barriers used in phase 1
  // stage and scale pipelines: the first KD - 1 stages and the first item's scales
  StageIssuer is;
  is.cur.phase = 1;
  is.cur.k = 0;
  is.c = 0;
  is.q = {0, 0, 0u};
  is.row0 = is.row1 = 0;
  is.cur.j = is.cur.rb = 0;
  cursor_locate<CW>(is.cur, v1, v2, cw);
  cursor_skip_empty<CW>(is.cur, n1, n2, v1, v2, cw);
  ItemCursor sc_next = is.cur;   // next item whose scale rows are to be issued
  int sc_count = 0;              // scale copies issued (lane 0)
  if (!has_producer(CW) && lane == 0) {
    for (int i = 0; i < KD - 1; ++i) issue_stage<CW>(is, P, v1, v2, n1, n2, eb, cw, ring_w, full_w);
    if (sc_next.phase <= 2) {
      issue_scales(sc_next, a, v1, v2, eb, cw, scale_w, &sfull_w[0]);
      ++sc_count;
    }
  }
  cursor_next<CW>(sc_next, n1, n2, v1, v2, cw);

  for (int phase = 1; phase <= 2; ++phase) {
    const PhaseView& v = phase == 1 ? v1 : v2;
    const RowPlan& rp = phase == 1 ? rp1 : rp2;
    if (phase == 2) {   // h of every CTA is complete (also for rows read from global)
      if constexpr (CW >= 10)
        if (ctid >= 32 && ctid < 44) rmax[ctid - 32] = 0;
      if (ctid == 0) {
        flags[1] = grid_wait(gbar, (uint32_t)nCta) ? 1 : 0;
        if (flags[1] != 0) {
          fence_proxy_async_global();
          issue_rows(2, v2, rp2, a, tb, xs, xs_stride, xfull);
        }
      }
      named_barrier(kBarConsumers, kThreadsCW);
      if (flags[1] == 0 && ok) {
        ok = false;
        fail |= 2;
      }
    }
    // -- activation rows: wait, prescale (one warp per row), convert to f16
    for (int i = 0; i < rp.nbars && ok; ++i) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&xfull[i], phase == 2 ? (rows_used >> i & 1u) : 0u));
      if (!ok) fail |= 4;
    }
    if (phase == 1) rows_used = (1u << rp.nbars) - 1u;
    bool shared_rows = false;   // fewer rows than warps: G warps share each row
    if constexpr (CW >= 10) shared_rows = v.n_need > 0 && v.n_need < CW;
    if (!shared_rows) {   // one warp per row
      for (int r = cw; r < v.n_need && ok; r += CW) {
        const bool staged = r < rp.xs_rows;
        uint4* row = reinterpret_cast<uint4*>(xs + (size_t)r * xs_stride);
        const uint4* src = reinterpret_cast<const uint4*>(act_row(phase, a, tb, v.p_lo + r));
        uint32_t emax = 0;
        for (int c16 = lane; c16 < v.kred / 8; c16 += 32) {
          const uint4 q = staged ? row[c16] : ldcg16(src + c16);
          const uint32_t wq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            emax = max(emax, (wq[i] >> 7) & 0xFFu);
            emax = max(emax, (wq[i] >> 23) & 0xFFu);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
        const int sh = max(-100, min(100, emax == 0 ? 0 : (int)emax - 127 - 14));
        if (lane == 0) row_sh[r] = sh;
        const float mul = pow2f(-sh);
        if (staged) {
          for (int c16 = lane; c16 < v.kred / 8; c16 += 32) row[c16] = bf16x8_to_f16x8(row[c16], mul);
        } else {   // rows with no room here: converted once into the f16 scratch
          uint4* dst = reinterpret_cast<uint4*>(a.xf + (size_t)(v.p_lo + r) * xf_stride);
          for (int c16 = lane; c16 < v.kred / 8; c16 += 32) dst[c16] = bf16x8_to_f16x8(ldcg16(src + c16), mul);
        }
      }
    } else {
      const int G = CW / v.n_need;
      const int r = cw / G, part = cw - r * G;
      const bool mine = r < v.n_need && ok;
      if (mine) {
        const bool staged = r < rp.xs_rows;
        const uint4* row = reinterpret_cast<const uint4*>(xs + (size_t)r * xs_stride);
        const uint4* src = reinterpret_cast<const uint4*>(act_row(phase, a, tb, v.p_lo + r));
        uint32_t emax = 0;
        for (int c16 = part * 32 + lane; c16 < v.kred / 8; c16 += G * 32)
          emax = max(emax, bf16x8_max_exponent(staged ? row[c16] : ldcg16(src + c16)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
        if (lane == 0) atomicMax(&rmax[r], (int)emax);
      }
      named_barrier(kBarConsumers, kThreadsCW);
      if (mine)
        convert_row_part(a, v, xs, xs_stride, row_sh, rp, tb, phase, r, (uint32_t)rmax[r],
                         part * 32 + lane, G * 32, part == 0 && lane == 0);
    }
    named_barrier(kBarConsumers, kThreadsCW);

    // -- this warp's items of the phase: item k of the warp is CTA item ib + k CW + cw
    const int my_n = phase == 1 ? n1 : n2;
    int cj = 0, crb = 0;   // expert batch and row block of the warp's next item
    if (my_n > 0) {
      const int it0 = v.ib + cw;
      cj = it0 / v.NB;
      crb = it0 - cj * v.NB;
    }
    for (int k = 0; k < my_n && ok; ++k) {
      const ItemRoutes ir = item_routes(tb, eb, cj);
      const int rb = crb;
      crb += CW;
      while (crb >= v.NB) {
        crb -= v.NB;
        ++cj;
      }
      const int sx = kitems & 1;
      // the next item's scale rows go to the other slot, which the previous
      // item (finished and fenced) no longer reads
      if (!has_producer(CW) && lane == 0 && sc_next.phase <= 2) {
        issue_scales(sc_next, a, v1, v2, eb, cw, scale_w + (sx ^ 1) * M.slot_bytes, &sfull_w[sx ^ 1]);
        ++sc_count;
      }
      cursor_next<CW>(sc_next, n1, n2, v1, v2, cw);
      ok = __all_sync(0xffffffffu, mbar_wait(&sfull_w[sx], (uint32_t)(kitems >> 1) & 1u));
      if (!ok) {
        fail |= 8;
        break;
      }
      const uint8_t* sc = scale_w + sx * M.slot_bytes;
      // E8M0 bytes 0 / 255 in this item: take the exact general conversion.
      // A byte is 0x00 or 0xFF exactly when its bits are all equal, i.e. when
      // b ^ (b >> 1) is 0 in bits 0..6; subtracting 1 from each such 7-bit
      // value sets bit 7 of some byte exactly when one of them is 0.
      uint32_t hit = 0;
      const uint4* sw = reinterpret_cast<const uint4*>(sc);
      for (int i = lane; i < v.nblk; i += 32) {   // 16 rows x nblk bytes = nblk 16-byte words
        const uint4 x = sw[i];
        hit |= ((x.x ^ (x.x >> 1)) & 0x7F7F7F7Fu) - 0x01010101u;
        hit |= ((x.y ^ (x.y >> 1)) & 0x7F7F7F7Fu) - 0x01010101u;
        hit |= ((x.z ^ (x.z >> 1)) & 0x7F7F7F7Fu) - 0x01010101u;
        hit |= ((x.w ^ (x.w >> 1)) & 0x7F7F7F7Fu) - 0x01010101u;
      }
      const bool special = __any_sync(0xffffffffu, (hit & 0x80808080u) != 0u);
      // B rows of the item's token groups for this lane's token column g
      const int cnt = ir.cnt;
      const int ng = (cnt + kGroup - 1) / kGroup;
      // (groups past ng are never read)
      BRows br;
      bool glob = false;
      const int q_first = ir.q0 - v.p_lo;
      const uint8_t* xf_lo = reinterpret_cast<const uint8_t*>(a.xf + (size_t)v.p_lo * xf_stride) + t * 16;
      set_group<0>(br, glob, q_first, cnt, g, t, rp.xs_rows, xs_stride, xs, xf_lo, xf_stride);
      if (ng > 1) {
        set_group<1>(br, glob, q_first, cnt, g, t, rp.xs_rows, xs_stride, xs, xf_lo, xf_stride);
        if (ng > 2) {
          set_group<2>(br, glob, q_first, cnt, g, t, rp.xs_rows, xs_stride, xs, xf_lo, xf_stride);
          if (ng > 3) set_group<3>(br, glob, q_first, cnt, g, t, rp.xs_rows, xs_stride, xs, xf_lo, xf_stride);
        }
      }
      glob = __any_sync(0xffffffffu, glob);
      float acc[kMaxGroups][4];
#pragma unroll
      for (int gr = 0; gr < kMaxGroups; ++gr)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[gr][q] = 0.f;
      if (!special && !glob)
        ok = item_stages<CW, true, false>(acc, xo, ring_w, full_w, s, v, lane, sc, ng, br, xs, is, P,
                                          v1, v2, n1, n2, eb, cw, empty_w);
      else if (special && !glob)
        ok = item_stages<CW, false, false>(acc, xo, ring_w, full_w, s, v, lane, sc, ng, br, xs, is, P,
                                           v1, v2, n1, n2, eb, cw, empty_w);
      else if (!special)
        ok = item_stages<CW, true, true>(acc, xo, ring_w, full_w, s, v, lane, sc, ng, br, xs, is,
                                              P, v1, v2, n1, n2, eb, cw, empty_w);
      else
        ok = item_stages<CW, false, true>(acc, xo, ring_w, full_w, s, v, lane, sc, ng, br, xs, is,
                                               P, v1, v2, n1, n2, eb, cw, empty_w);
      if (!ok) {
        fail |= 16;
        break;
      }
      // -- epilogue: rows g, g+8 and token columns 2t, 2t+1 of each group
#pragma unroll
      for (int gr = 0; gr < kMaxGroups; ++gr) {
        if (gr >= ng) break;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int n = gr * kGroup + 2 * t + j;
          if (n >= cnt) continue;
          const int qpos = ir.q0 + n;
          const int r = tb.lst[qpos];
          const float colmul = pow2f(row_sh[qpos - v.p_lo]);
          if (phase == 1) {
            const int i = rb * 8 + g;
            float gate = acc[gr][j] * colmul, up = acc[gr][2 + j] * colmul;
            float hv;
            if (a.oai) {
              gate += a.b13[((size_t)ir.e * a.I + i) * 2];
              up += a.b13[((size_t)ir.e * a.I + i) * 2 + 1];
              hv = swiglu_oai_f32(gate, up);
            } else {
              hv = silu_f32(gate) * up;
            }
            a.h[(size_t)r * a.I + i] = f32_to_bf16_rne(hv);
          } else {
            const int m = rb * kRows + g;
            const float wr = a.per_route ? 1.0f : a.wts[r];   // per-route rows: unweighted
            float o0 = acc[gr][j] * colmul, o1 = acc[gr][2 + j] * colmul;
            if (a.oai) {
              o0 += a.b2[(size_t)ir.e * a.K + m];
              o1 += a.b2[(size_t)ir.e * a.K + m + 8];
            }
            a.P[(size_t)r * a.K + m] = wr * o0;
            a.P[(size_t)r * a.K + m + 8] = wr * o1;
          }
        }
      }
      // the scale slot is refilled by a bulk copy (async proxy)
      fence_proxy_async_smem();
      __syncwarp();
      if constexpr (has_producer(CW))
        if (lane == 0) mbar_arrive(&sempty_w[sx]);
      ++kitems;
    }
    // -- grid arrival: this CTA's outputs of the phase are written
    if (phase == 1) fence_proxy_async_global();   // h is read next by bulk copies
    __threadfence();
    named_barrier(kBarConsumers, kThreadsCW);
    if (ctid == 0 && !(phase == 1 && (int)blockIdx.x == a.skip_arrival_cta)) atomicAdd(gbar, 1);
  }

  // -- combine: y [T, K] (this CTA's slice), once every route output exists
  if (ctid == 0) flags[0] = grid_wait(gbar, 2u * nCta) ? 1 : 0;
  named_barrier(kBarConsumers, kThreadsCW);
  if (flags[0] == 0) {
    ok = false;
    fail |= 32;
  } else {
    combine_share(a, blockIdx.x, nCta, ctid, kThreadsCW);
  }
  // the last CTA out leaves the grid counters at zero for the next call
  named_barrier(kBarConsumers, kThreadsCW);
  if (ctid == 0) {
    __threadfence();
    if (atomicAdd(&gbar[1], 1) == nCta - 1) {
      atomicExch(&gbar[0], 0);
      atomicExch(&gbar[1], 0);
    }
  }
  // stages issued ahead but never consumed (only after a failed wait) must
  // land before the CTA exits
  if (!has_producer(CW) && lane == 0) {
    for (int n = s.n; n < is.q.n; ++n) mbar_wait(&full_w[n % KD], (uint32_t)(n / KD) & 1u);
    for (int n = kitems; n < sc_count; ++n) mbar_wait(&sfull_w[n & 1], (uint32_t)(n >> 1) & 1u);
  }
  if (!ok && lane == 0 && a.status != nullptr) {
    atomicOr(&a.status[2], (fail | 128) << 8);
    atomicCAS(&a.status[3], 0, blockIdx.x + 1);
  }
}

size_t decode_smem_bytes(int cw, int K, int I, int E, int R, int xs_rows, int xs_stride) {
  return decode_smem_plan(cw, K, I, E, R, xs_rows, xs_stride).total + 1024;
}

int decode_row_stride(int K, int I) { return (int)round_up((size_t)(K > I ? K : I) * 2, 128) + 64; }

// The smallest m with P(max over E experts of routes per expert <= m) >= 0.99
// when each of T tokens names an expert with probability topk / E
// (binomial counts, independent across experts).
static int routes_per_expert_p99(int T, int topk, int E) {
  const double p = (double)topk / E;
  double cdf = 0.0, pmf = pow(1.0 - p, (double)T);   // P(X = 0)
  for (int m = 0; m <= T; ++m) {
    cdf += pmf;
    if (pow(cdf > 1.0 ? 1.0 : cdf, (double)E) >= 0.99) return m;
    pmf *= (double)(T - m) / (m + 1) * p / (1.0 - p);
  }
  return T;
}

// Warps per CTA: the most of 12, 11 or 10 (more warps hide more of the
// latency of the conversion and MMA chain) whose rings, scale slots and the
// activation rows a CTA is expected to need all fit. A CTA's items span one
// or two expert batches, so it needs the rows of those experts' routes: at
// most 2 m99 (m99 from routes_per_expert_p99), and 3 rho + 3 covered the
// largest need of every CTA on the workload shapes (rho = R / (E (1 - (1 -
// 1/E)^R)), the expected routes per touched expert). When those rows do not
// fit next to any of them: 7 consumer warps and a producer, the form with the
// most room for rows
// (and batched paths for rows read from the f16 scratch and for items with
// several token groups) -- an item whose rows are not all staged reads them
// through L2 on every block and runs about 1.5x longer, which decides the
// call's time through the slowest CTA. 0 when even that form does not fit. Rows
// beyond the staged ones are read from the f16 scratch in global memory
// (correct for any routing, only slower).
static int decode_warps_at(int K, int I, int E, int T, int topk, int max_smem) {
  const int R = T * topk;
  const int stride = decode_row_stride(K, I);
  const double rho = (double)R / ((double)E * (1.0 - pow(1.0 - 1.0 / E, (double)R)));
  const int m99 = routes_per_expert_p99(T, topk, E);
  int want = (int)ceil(3.0 * rho + 3.0);
  if (want > 2 * m99) want = 2 * m99;
  if (want > R) want = R;
  for (int cw = 12; cw >= 10; --cw)
    if (decode_smem_bytes(cw, K, I, E, R, want, stride) <= (size_t)max_smem) return cw;
  if (decode_smem_bytes(7, K, I, E, R, 1, stride) <= (size_t)max_smem) return 7;
  return 0;
}

// The form of a call: the one its own T needs, except that when the largest
// decode T of the layer shape runs one of the 10- to 12-warp forms, every T of
// the shape runs that form. Serving interleaves calls of different T, and on
// gptoss128 a sequence of T = 1, 4, 16, 32 whose calls moved between the 12-
// and 11-warp forms took about 8 us more per change than the same calls on
// one form; the 11-warp form costs the small calls a little on their own
// (T = 4 / 16 ran 1.5 / 4.5 us slower than on 12 warps). (All T on the 12-warp
// form, with one staged row fewer at T = 32, was slower: T = 32 routings whose
// CTAs need more rows than 12 warps leave room for read them through L2.)
int decode_warps(int K, int I, int E, int T, int topk, int max_smem) {
  const int cw = decode_warps_at(K, I, E, T, topk, max_smem);
  int t_max = kDecodeMaxTokens;
  if (t_max * topk > kDecodeMaxRoutes) t_max = kDecodeMaxRoutes / topk;
  if (cw == 0 || t_max <= T) return cw;
  const int cw_max = decode_warps_at(K, I, E, t_max, topk, max_smem);
  return cw_max >= 10 && cw_max < cw ? cw_max : cw;
}

bool decode_fits(int K, int I, int E, int T, int topk, int max_smem) {
  return decode_warps(K, I, E, T, topk, max_smem) != 0;
}

template <int CW>
static cudaError_t launch_cw(const DecodeParams& p, size_t smem, int num_sms, cudaStream_t stream) {
  // the shared-memory grant is a per-device attribute of the kernel
  static size_t granted[kGrantDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kGrantDevices) return cudaErrorInvalidDevice;
  if (smem > granted[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<CW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    granted[dev] = smem;
  }
  // every CTA must be resident at once (grid barriers): one per SM, cooperative launch
  int per_sm = 0;
  constexpr int kThreads = (CW + (has_producer(CW) ? 1 : 0)) * 32;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<CW>, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<CW>, p);
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmap1, const CUtensorMap& tmap2,
                          const CUtensorMap& tmap1q, const CUtensorMap& tmap2q, int num_sms,
                          int max_smem, cudaStream_t stream) {
  DecodeParams p;
  p.tmap1 = tmap1;
  p.tmap2 = tmap2;
  p.tmap1q = tmap1q;
  p.tmap2q = tmap2q;
  p.a = a;
  const int R = a.T * a.topk;
  const int cw = decode_warps(a.K, a.I, a.E, a.T, a.topk, max_smem);
  if (cw == 0) return cudaErrorInvalidValue;
  p.xs_stride = decode_row_stride(a.K, a.I);
  const size_t fixed = decode_smem_bytes(cw, a.K, a.I, a.E, R, 0, p.xs_stride);
  size_t rows = ((size_t)max_smem - fixed) / p.xs_stride;
  if (rows > (size_t)R) rows = R;
  p.xs_rows_cap = (int)rows;
  p.stages = ring_depth(cw);
  const size_t smem = decode_smem_bytes(cw, a.K, a.I, a.E, R, (int)rows, p.xs_stride);
  if (cw == 12) return launch_cw<12>(p, smem, num_sms, stream);
  if (cw == 11) return launch_cw<11>(p, smem, num_sms, stream);
  if (cw == 10) return launch_cw<10>(p, smem, num_sms, stream);
  return launch_cw<7>(p, smem, num_sms, stream);
}

}  // namespace mxmoe
