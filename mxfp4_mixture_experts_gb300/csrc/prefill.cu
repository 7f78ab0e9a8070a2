// Prefill path (many tokens): the routed experts as grouped GEMMs on the
// 5th-generation tensor cores ("MXFP4 MoE decode kernels", Prefill: on large
// MoE models the routed experts are most of the prefill; the pages unpack the
// weights to bf16 and run a stock bf16 MoE op -- here the unpack is fused
// into the GEMM's shared-memory tiles instead).
//
//   route   stable counting sort of the routes by expert (route.cu)
//   gather  xp[pos] = hidden[token of route list[pos]]: rows in expert order,
//           each group of 8 values in pair order (0 4 1 5 2 6 3 7)
//   GEMM1   per expert: [M_e x K] x [K x 2I]^T -> SwiGLU -> hp [M_e x I] bf16
//           (pair order inside each group of 8 intermediate values)
//   GEMM2   per expert: [M_e x I] x [I x K]^T -> P[pos] fp32 (expert order)
//   combine y[t] = bf16(sum over the token's slots of w * P[pos of the route]),
//           slot order
//
// GEMM kernel: weight-stationary, one persistent CTA per SM. A tile is
// (expert, 128 weight rows, a chunk of up to 384 of the expert's tokens); the
// MMA computes D[weight row][token] with the bf16 weights as operand A in
// tensor memory and the tokens as operand B in shared memory (N = tokens
// rounded up to 16, so an expert's tokens cost no padding beyond that).
// Warp roles:
// The token tile and the dequantised weights of a k-stage share one ring
// slot and one pair of barriers (full: the token bytes and the 8 dequant
// warps; empty: the MMAs that read the slot), so the MMA issuer waits and
// commits once per stage.
//   warp 0      TMA producer of token tiles (128 rows x 64 bf16, 128-byte swizzle)
//   warp 1      MMA issuer: tcgen05.mma M128 N<=256 K16, A from tensor memory
//   warp 2      TMA producer of packed weight bytes (2 x 64 rows x 32 bytes a stage)
//   warps 4..7  epilogue: tcgen05.ld of D -> SwiGLU / routing weight -> global
// Both GEMMs take the reduction dimension in pair order inside each group of
// 8 values, on the weights (as dequant32_bf16_pairs makes them) and on the
// token rows alike, so the dot products are those of row order.
//   warps 8..15 dequant: packed E2M1 + E8M0 -> exact bf16, tcgen05.st into the
//               tensor-memory ring of operand A (two warps per lane quarter,
//               32 of the stage's 64 K values each)
// GEMM1 puts gate row i at lane 16g + r and up row i at lane 16g + 8 + r
// (i = i0 + 8g + r), so one 16x256b tensor-memory load hands a thread both
// factors of its SwiGLU products.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "prefill.h"
#include "route.cuh"

namespace mxmoe {

constexpr int kPfWarps = 20;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kBM = 128;                  // weight rows per tile (MMA M)
constexpr int kBK = 64;                   // K values per stage (128 bytes of bf16)
constexpr int kMaxTok = 320;              // tokens per tile (accumulator columns)
constexpr int kXBox = 64;                 // token rows per TMA copy (<= 5 a stage)
constexpr int kS = 4, kSP = 12;          // rings: operand stages (tokens in smem + bf16 weights in TMEM), packed bytes (smem)
constexpr int kXStage = kMaxTok * kBK * 2;   // 40 KB
constexpr int kXBoxBytes = kXBox * kBK * 2;  // 8 KB
constexpr int kPStage = kBM * kBK / 2;       // 4 KB of packed bytes
constexpr int kPBoxRows = 64;
constexpr int kTmemCols = 512;
constexpr int kWCol0 = kMaxTok;           // operand-A ring: columns 320..511
constexpr int kWCols = kBK / 2;           // 32 columns (bf16 pairs) a stage
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpTmaW = 2, kWarpEpi = 4, kWarpDeq = 8;
constexpr int kWarpEpi2 = 16;            // second epilogue group: the upper half of the tokens
constexpr int kEpiWarps = 8;
constexpr int kDeqWarps = 8;
constexpr int kScaleAhead = 8;            // k-stages of scale bytes held in registers
static_assert(kWCol0 + kS * kWCols <= kTmemCols, "tensor memory budget");
static_assert(kMaxTok % kXBox == 0 && kMaxTok % 16 == 0, "token boxes fill a stage exactly");

struct GemmParams {
  CUtensorMap tmapX;   // tokens bf16 [R][kred], box {64, 128}, 128-byte swizzle
  // packed weights: GEMM1 u8 {K/2 bytes, row groups, 2 halves (gate, up)}, box
  // {32, 64, 2} (64 gate rows, then the 64 matching up rows); GEMM2 u8
  // [rows][I/2], box {32, 64}
  CUtensorMap tmapW;
  const uint8_t* wsc;  // scales u8 [rows][kred/32]
  const int32_t* count;
  const int32_t* offset;
  const int32_t* list;
  const float* wts;
  uint16_t* hp;        // GEMM1 output bf16 [R][I]
  float* P;            // GEMM2 output fp32 [R][K] (expert order, unweighted)
  int E, K, I, kred, NT;
  int32_t* status;
  const float* bias;   // gpt-oss form: GEMM1 b13 [E][2I] (interleaved), GEMM2 b2 [E][K]
  int oai;             // gpt-oss form: interleaved w13 rows, biases, SwiGLU-OAI
};

// Token chunks of one expert: nch chunks of cs tokens (cs a multiple of 16,
// at most kMaxTok), the last one possibly shorter, none empty.
__host__ __device__ __forceinline__ void chunk_plan(int c, int& nch, int& cs) {
  if (c <= 0) { nch = 0; cs = 0; return; }
  const int n0 = (c + kMaxTok - 1) / kMaxTok;
  cs = (((c + n0 - 1) / n0) + 15) & ~15;
  nch = (c + cs - 1) / cs;
}

struct TileId {
  int e, nt, t0, n;   // expert, weight-row block, first token (within the expert), tokens
};

__device__ __forceinline__ TileId decode_tile(int t, const int* tile_base, const int32_t* count,
                                              int E) {
  int lo = 0, hi = E;   // tile_base[lo] <= t < tile_base[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_base[mid] <= t) lo = mid; else hi = mid;
  }
  TileId id;
  id.e = lo;
  const int c = count[lo];
  int nch, cs;
  chunk_plan(c, nch, cs);
  const int local = t - tile_base[lo];
  id.nt = local / nch;
  const int ch = local - id.nt * nch;
  id.t0 = ch * cs;
  id.n = min(cs, c - id.t0);
  return id;
}

// Lane m of operand A <-> weight row. GEMM1: gate/up of i = 64 nt + 8g + r at
// lanes 16g + r / 16g + 8 + r; its packed bytes sit at shared row up*64 + 8g + r.
// GEMM2: output column k = 128 nt + m, packed row m.
template <int PHASE>
__device__ __forceinline__ int packed_row(int m) {
  return PHASE == 1 ? ((m >> 3) & 1) * 64 + (m >> 4) * 8 + (m & 7) : m;
}
template <int PHASE>
__device__ __forceinline__ int weight_row(int e, int nt, const GemmParams& p, int m) {
  if (PHASE == 1) {
    const int pr = packed_row<1>(m);
    if (p.oai) return e * (2 * p.I) + 2 * (nt * 64 + (pr & 63)) + (pr >= 64 ? 1 : 0);
    return e * (2 * p.I) + (pr >= 64 ? p.I : 0) + nt * 64 + (pr & 63);
  }
  const int k = nt * kBM + m;
  return e * p.K + (k < p.K ? k : nt * kBM);   // rows past K (a partial last tile): never stored
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

template <int PHASE, bool OAI>
__global__ void __launch_bounds__(kPfThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sX = smem;
  uint8_t* sP = sX + kS * kXStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(sP + kSP * kPStage);   // [kS]
  uint64_t* empty = full + kS;                                        // [kS]
  uint64_t* p_full = empty + kS;
  uint64_t* p_empty = p_full + kSP;
  uint64_t* d_full = p_empty + kSP;
  uint64_t* d_empty = d_full + 1;
  uint64_t* drain = d_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* tile_base = reinterpret_cast<int*>(tmem_slot + 4);   // [E+1]
  // the experts' route counts and list offsets, read at every tile change by
  // every role: shared copies keep global round trips out of the tile switch
  int* s_cnt = tile_base + p.E + 1;                          // [E]
  int* s_off = s_cnt + p.E;                                  // [E]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  for (int i = threadIdx.x; i < E; i += kPfThreads) {
    s_cnt[i] = p.count[i];
    s_off[i] = p.offset[i];
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kS; ++i) { mbar_init(&full[i], 1 + kDeqWarps); mbar_init(&empty[i], 1); }
    for (int i = 0; i < kSP; ++i) { mbar_init(&p_full[i], 1); mbar_init(&p_empty[i], kDeqWarps); }
    mbar_init(d_full, 1);
    mbar_init(d_empty, kEpiWarps);
    mbar_init(drain, 1);
    fence_barrier_init();
    prefetch_tensormap(&p.tmapX);
    prefetch_tensormap(&p.tmapW);
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  if (warp == 3) {   // tile table: experts in order, (weight block, token chunk) inside
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int nch = 0, cs;
      if (e < E) chunk_plan(p.count[e], nch, cs);
      const int tiles = nch * p.NT;
      int x = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) tile_base[e] = carry + x - tiles;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) tile_base[E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = tile_base[E];
  const int nK = p.kred / kBK;
  int fail = 0;

  if (warp == kWarpTma && lane == 0) {
    // ------------------------------------------------------------ token producer
    int sx = 0, kx = 0;
    uint32_t px = 0, xpar = 0;   // parity of each stage's last fill
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const TileId id = decode_tile(t, tile_base, s_cnt, E);
      const int row0 = s_off[id.e] + id.t0;
      const int nbox = (id.n + kXBox - 1) / kXBox;
      for (int kc = 0; kc < nK; ++kc) {
        if (kx >= kS && !mbar_wait(&empty[sx], px ^ 1u)) { fail = 1; break; }
        xpar = (xpar & ~(1u << sx)) | (px << sx);
        mbar_arrive_expect_tx(&full[sx], nbox * kXBoxBytes);
        for (int b = 0; b < nbox; ++b)
          tma_load_2d(sX + sx * kXStage + b * kXBoxBytes, &p.tmapX, kc * kBK, row0 + b * kXBox,
                      &full[sx]);
        if (++sx == kS) { sx = 0; px ^= 1u; }
        ++kx;
      }
    }
    // no copy may still be landing in shared memory when the CTA exits
    for (int i = 0; i < kS && i < kx; ++i) mbar_wait(&full[i], (xpar >> i) & 1u);
  } else if (warp == kWarpTmaW && lane == 0) {
    // ------------------------------------------------------------ packed-weight producer
    int sp = 0, kp = 0;
    uint32_t pp = 0, ppar = 0;
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const TileId id = decode_tile(t, tile_base, s_cnt, E);
      // GEMM1: 64 gate rows then the 64 matching up rows (one copy: row group
      // e 2I + i of [gate; up], or pair e I + i of the interleaved rows);
      // GEMM2: 128 rows (past the matrix: other experts' rows or zeros, never
      // stored)
      const int r0 = PHASE == 1 ? (OAI ? id.e * p.I : id.e * 2 * p.I) + id.nt * 64
                                : id.e * p.K + id.nt * kBM;
      for (int kc = 0; kc < nK; ++kc) {
        if (kp >= kSP && !mbar_wait(&p_empty[sp], pp ^ 1u)) { fail = 2; break; }
        ppar = (ppar & ~(1u << sp)) | (pp << sp);
        mbar_arrive_expect_tx(&p_full[sp], kPStage);
        if (PHASE == 1) {
          tma_load_3d(sP + sp * kPStage, &p.tmapW, kc * (kBK / 2), r0, 0, &p_full[sp]);
        } else {
          tma_load_2d(sP + sp * kPStage, &p.tmapW, kc * (kBK / 2), r0, &p_full[sp]);
          tma_load_2d(sP + sp * kPStage + kPBoxRows * (kBK / 2), &p.tmapW, kc * (kBK / 2),
                      r0 + 64, &p_full[sp]);
        }
        if (++sp == kSP) { sp = 0; pp ^= 1u; }
        ++kp;
      }
    }
    for (int i = 0; i < kSP && i < kp; ++i) mbar_wait(&p_full[i], (ppar >> i) & 1u);
  } else if (warp == kWarpMma && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // The issuing thread is the pipe's bottleneck (each tcgen05 instruction,
    // barrier test and commit costs it tens of cycles), so a stage is one
    // barrier test, four MMAs on precomputed descriptors and one commit; the
    // next stage's barrier is tested while the current stage's last MMA is
    // queued, and a blocking wait is only taken when that test failed.
    const uint64_t desc0 = umma_desc_sw128(smem_u32(sX));
    int s = 0, tiles = 0;
    uint32_t ph = 0;
    bool ready = false;   // operands of stage s known to have landed
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x, ++tiles) {
      const TileId id = decode_tile(t, tile_base, s_cnt, E);
      const int n16 = (id.n + 15) & ~15;
      const int n_a = min(n16, 256), n_b = n16 - n_a;   // MMA N of the two column groups
      const uint32_t idesc_a = umma_idesc_bf16(kBM, n_a);
      const uint32_t idesc_b = umma_idesc_bf16(kBM, n_b > 0 ? n_b : 16);
      if (tiles > 0) {   // the epilogue must have read the previous tile's accumulators
        if (!mbar_wait(d_empty, (tiles - 1) & 1)) { fail = 4; break; }
        tc_fence_after();
      }
      for (int kc = 0; kc < nK; ++kc) {
        if (!ready && !mbar_wait(&full[s], ph)) { fail = 8; break; }
        tc_fence_after();
        const uint32_t a_col = tmem + kWCol0 + s * kWCols;
        // start-address field (bytes / 16): stage s, k16 step 32 bytes, token 256 at 32 KB
        const uint64_t dsc = desc0 + (uint64_t)(s * (kXStage >> 4));
        const int s1 = s + 1 == kS ? 0 : s + 1;
        const uint32_t ph1 = s + 1 == kS ? ph ^ 1u : ph;
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16) {
          if (k16 == kBK / 16 - 1) ready = mbar_test(&full[s1], ph1);
          const bool acc = kc > 0 || k16 > 0;
          umma_bf16_ts(tmem, a_col + k16 * 8, dsc + 2 * k16, idesc_a, acc);
          if (n_b > 0)
            umma_bf16_ts(tmem + 256, a_col + k16 * 8, dsc + ((256 * 128) >> 4) + 2 * k16, idesc_b,
                         acc);
        }
        umma_commit(&empty[s]);
        s = s1;
        ph = ph1;
      }
      if (fail) break;
      umma_commit(d_full);
    }
    // every issued MMA has finished before tensor memory is released
    umma_commit(drain);
    mbar_wait(drain, 0);
  } else if (warp >= kWarpDeq && warp < kWarpDeq + kDeqWarps) {
    // ------------------------------------------------------------ dequant
    const int q = warp & 3;                    // lane quarter
    const int h = (warp - kWarpDeq) >> 2;      // which 32 of the stage's 64 K values
    const int m = q * 32 + lane;               // operand-A row (TMEM lane)
    const int prow = packed_row<PHASE>(m);
    const uint32_t wlane = tmem + ((uint32_t)(q * 32) << 16) + kWCol0 + h * 16;
    int sp = 0, sw = 0, kw = 0;   // packed-ring slot, operand-ring slot, stages done
    uint32_t pp = 0, pw = 0;
    // scale row of this thread's weight row in tile t (its half's bytes)
    auto scale_row = [&](int t) {
      const TileId id = decode_tile(t, tile_base, s_cnt, E);
      return p.wsc + (size_t)weight_row<PHASE>(id.e, id.nt, p, m) * (p.kred / kScaleBlock) + h;
    };
    // the scale byte of each of the next kScaleAhead stages, loaded one window
    // early (the next tile's first window during the current tile's last one)
    uint32_t sc[kScaleAhead];
    const uint8_t* srow = blockIdx.x < ntiles ? scale_row(blockIdx.x) : nullptr;
#pragma unroll
    for (int i = 0; i < kScaleAhead; ++i) sc[i] = (srow != nullptr && i < nK) ? ldg_u8(srow + 2 * i) : 0u;
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const int tn = t + gridDim.x;
      const uint8_t* srow_n = tn < ntiles ? scale_row(tn) : nullptr;
      for (int k0 = 0; k0 < nK && !fail; k0 += kScaleAhead) {
        uint32_t nx[kScaleAhead];
        if (k0 + kScaleAhead < nK) {
#pragma unroll
          for (int i = 0; i < kScaleAhead; ++i)
            nx[i] = k0 + kScaleAhead + i < nK ? ldg_u8(srow + 2 * (k0 + kScaleAhead + i)) : 0u;
        } else {
#pragma unroll
          for (int i = 0; i < kScaleAhead; ++i)
            nx[i] = (srow_n != nullptr && i < nK) ? ldg_u8(srow_n + 2 * i) : 0u;
        }
#pragma unroll
        for (int i = 0; i < kScaleAhead; ++i) {
          if (k0 + i >= nK || fail) break;
          if (!warp_wait(&p_full[sp], pp)) { fail = 16; break; }
          const uint4 qv = *reinterpret_cast<const uint4*>(sP + sp * kPStage + prow * (kBK / 2) + h * 16);
          // the stage is refilled by the tensor-copy engine (async proxy): the
          // generic read above must be ordered before that write
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_empty[sp]);
          if (++sp == kSP) { sp = 0; pp ^= 1u; }
          const uint32_t wd[4] = {qv.x, qv.y, qv.z, qv.w};
          uint32_t o[16];   // this thread's 32 values, in row order (bf16 pairs)
          dequant32_bf16_pairs(wd, scale_mul(sc[i]), o);
          if (kw >= kS) {   // the MMAs that read this ring slot have completed
            if (!warp_wait(&empty[sw], pw ^ 1u)) { fail = 32; break; }
            tc_fence_after();
          }
          tmem_st16(wlane + sw * kWCols, o);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[sw]);
          if (++sw == kS) { sw = 0; pw ^= 1u; }
          ++kw;
        }
#pragma unroll
        for (int i = 0; i < kScaleAhead; ++i) sc[i] = nx[i];
      }
      srow = srow_n;
    }
  } else if ((warp >= kWarpEpi && warp < kWarpEpi + 4) || warp >= kWarpEpi2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const int half = warp >= kWarpEpi2;   // which half of the tile's tokens (32-column blocks)
    int tiles = 0;
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x, ++tiles) {
      const TileId id = decode_tile(t, tile_base, s_cnt, E);
      if (!warp_wait(d_full, tiles & 1)) { fail = 64; break; }
      tc_fence_after();
      const int pos0 = s_off[id.e] + id.t0;
      if (PHASE == 1) {
        // lane groups g = 2q, 2q + 1: this thread's SwiGLU pairs are
        // i = 64 nt + 8g + lane/4, tokens 8b + 2(lane%4) + {0, 1}
#pragma unroll 1
        for (int s = 0; s < 2; ++s) {
          const int g = 2 * q + s;
          const int i = id.nt * 64 + 8 * g + (lane >> 2);
          const int ip = (i & ~7) | pair_order_pos(i & 7);   // its column of hp
          const uint32_t taddr = tmem + ((uint32_t)(16 * g) << 16);
          float bg = 0.f, bu = 0.f;   // gpt-oss biases of pair i (interleaved order)
          if (OAI) {
            bg = p.bias[((size_t)id.e * p.I + i) * 2];
            bu = p.bias[((size_t)id.e * p.I + i) * 2 + 1];
          }
          const int n32 = (id.n + 31) >> 5, lo32 = (n32 + 1) >> 1;
#pragma unroll 1
          for (int b = (half ? lo32 : 0) * 4; b < (half ? n32 : lo32) * 4; b += 4) {
            uint32_t v[4][4];
            tmem_ld_16x256b_x4(taddr + b * 8, v);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
#pragma unroll
              for (int x = 0; x < 2; ++x) {
                const int n = (b + u) * 8 + 2 * (lane & 3) + x;
                float gt = __uint_as_float(v[u][x]), up = __uint_as_float(v[u][2 + x]);
                float hv;
                if (OAI) {
                  gt += bg;
                  up += bu;
                  hv = swiglu_oai_fast(gt, up);
                } else {
                  hv = silu_fast(gt) * up;
                }
                if (n < id.n) p.hp[(size_t)(pos0 + n) * p.I + ip] = f32_to_bf16_rne(hv);
              }
            }
          }
        }
      } else {
        const int k = id.nt * kBM + q * 32 + lane;
        const bool kvalid = k < p.K;
        // gpt-oss: the expert's w2 bias, weighted with the route in the combine
        const float bk = (OAI && kvalid) ? p.bias[(size_t)id.e * p.K + k] : 0.f;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        const int n32 = (id.n + 31) >> 5, lo32 = (n32 + 1) >> 1;
#pragma unroll 1
        for (int c0 = (half ? lo32 : 0) * 32; c0 < (half ? n32 : lo32) * 32; c0 += 32) {
          float v[32];
          tmem_ld32(taddr + c0, v);
          // one 128-byte row segment per token: 32 consecutive output columns
          float* dst = p.P + (size_t)(pos0 + c0) * p.K + k;
          const int nv = min(32, id.n - c0);
          if (kvalid) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nv) dst[(size_t)j * p.K] = v[j] + bk;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(d_empty);
    }
  }
  __syncwarp();
  if (fail && p.status != nullptr) {
    atomicOr(&p.status[2], fail << (PHASE == 1 ? 16 : 24));
    atomicCAS(&p.status[3], 0, blockIdx.x + 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// xp[pos] = hidden[list[pos] / topk] for the valid (expert-sorted) routes,
// each group of 8 values in pair order (0 4 1 5 2 6 3 7); one warp per row,
// 16-byte chunks (one group each) in batches of 8 per lane (all loads of a
// batch in flight before its stores); the rows of xp are written with an
// evict-first hint, so the hidden rows (each read topk times) stay in L2.
// Also inv[route] = pos, the row of the route's output in P.
__device__ __forceinline__ void st_cs16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ hidden,
                                                     const int32_t* __restrict__ list,
                                                     const int32_t* __restrict__ n_valid, int K,
                                                     int topk, uint16_t* __restrict__ xp,
                                                     int32_t* __restrict__ inv) {
  constexpr int kB = 8;
  const int n = *n_valid;
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int per_row = K / 8;   // 16-byte chunks
  for (int pos = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < n; pos += warps) {
    const int r = list[pos];
    if (lane == 0) inv[r] = pos;
    const uint4* src = reinterpret_cast<const uint4*>(hidden + (size_t)(r / topk) * K);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)pos * K);
    for (int c0 = lane; c0 < per_row; c0 += 32 * kB) {
      uint4 v[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j)
        if (c0 + 32 * j < per_row) v[j] = src[c0 + 32 * j];
#pragma unroll
      for (int j = 0; j < kB; ++j)
        if (c0 + 32 * j < per_row) {
          const uint4 u = v[j];   // words (0 1) (2 3) (4 5) (6 7) -> (0 4) (1 5) (2 6) (3 7)
          st_cs16(dst + c0 + 32 * j, make_uint4(prmt(u.x, u.z, 0x5410u), prmt(u.x, u.z, 0x7632u),
                                                prmt(u.y, u.w, 0x5410u), prmt(u.y, u.w, 0x7632u)));
        }
    }
  }
}

// y[t][m] = bf16( sum over slots j = 0..k-1 with a valid expert of
// w[t][j] * P[inv[t*k + j]][m] ), in slot order (deterministic). 8 outputs a thread.
__global__ void __launch_bounds__(256) combine_pos_kernel(const float* __restrict__ P,
                                                          const int32_t* __restrict__ ids,
                                                          const float* __restrict__ wts,
                                                          const int32_t* __restrict__ inv, int T,
                                                          int K, int E, int topk, int ebase,
                                                          int window, uint16_t* __restrict__ y) {
  const int per_row = K / 8;
  const int64_t n = (int64_t)T * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / per_row), m8 = (int)(i - (int64_t)t * per_row) * 8;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < topk; ++j) {
      const int r = t * topk + j;
      if (local_expert(ids[r], ebase, window, E) < 0) continue;
      const float w = wts[r];
      const float* row = P + (size_t)inv[r] * K + m8;
      const uint4 lo = ldcg16(row);
      const uint4 hi = ldcg16(row + 4);
      s[0] += w * __uint_as_float(lo.x);
      s[1] += w * __uint_as_float(lo.y);
      s[2] += w * __uint_as_float(lo.z);
      s[3] += w * __uint_as_float(lo.w);
      s[4] += w * __uint_as_float(hi.x);
      s[5] += w * __uint_as_float(hi.y);
      s[6] += w * __uint_as_float(hi.z);
      s[7] += w * __uint_as_float(hi.w);
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[q]) : "f"(s[2 * q + 1]), "f"(s[2 * q]));
    *reinterpret_cast<uint4*>(y + (size_t)t * K + m8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Per-route output: y[r][m] = bf16(P[inv[r]][m]) for the computed routes, zero
// rows for skipped ones (8 outputs a thread).
__global__ void __launch_bounds__(256) route_rows_kernel(const float* __restrict__ P,
                                                         const int32_t* __restrict__ ids,
                                                         const int32_t* __restrict__ inv, int R,
                                                         int K, int E, int ebase, int window,
                                                         uint16_t* __restrict__ y) {
  const int per_row = K / 8;
  const int64_t n = (int64_t)R * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_row), m8 = (int)(i - (int64_t)r * per_row) * 8;
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (local_expert(ids[r], ebase, window, E) >= 0) {
      const float* row = P + (size_t)inv[r] * K + m8;
      const uint4 lo = ldcg16(row);
      const uint4 hi = ldcg16(row + 4);
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.x) : "f"(__uint_as_float(lo.y)), "f"(__uint_as_float(lo.x)));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.y) : "f"(__uint_as_float(lo.w)), "f"(__uint_as_float(lo.z)));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.z) : "f"(__uint_as_float(hi.y)), "f"(__uint_as_float(hi.x)));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.w) : "f"(__uint_as_float(hi.w)), "f"(__uint_as_float(hi.z)));
    }
    *reinterpret_cast<uint4*>(y + (size_t)r * K + m8) = o;
  }
}

static size_t gemm_smem_bytes(int E) {
  return 1024 + (size_t)kS * kXStage + (size_t)kSP * kPStage +
         (size_t)(2 * kS + 2 * kSP + 3) * 8 + 16 + (size_t)(3 * E + 1) * 4;
}

template <int PHASE, bool OAI>
static cudaError_t launch_gemm_form(const GemmParams& gp, int num_sms, cudaStream_t stream) {
  // the shared-memory grant is a per-device attribute of the kernel
  static size_t granted[kGrantDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kGrantDevices) return cudaErrorInvalidDevice;
  const size_t smem = gemm_smem_bytes(gp.E);
  if (smem > granted[dev]) {
    e = cudaFuncSetAttribute(gemm_kernel<PHASE, OAI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    granted[dev] = smem;
  }
  gemm_kernel<PHASE, OAI><<<num_sms, kPfThreads, smem, stream>>>(gp);
  return cudaGetLastError();
}
template <int PHASE>
static cudaError_t launch_gemm(const GemmParams& gp, int num_sms, cudaStream_t stream) {
  return gp.oai ? launch_gemm_form<PHASE, true>(gp, num_sms, stream)
                : launch_gemm_form<PHASE, false>(gp, num_sms, stream);
}

// GEMM1's packed weights as row groups: {K/2 bytes, groups, 2 halves}, box
// {32, 64, 2}. [gate; up]: group e 2I + i, the up half I rows later;
// interleaved (gpt-oss): group e I + i (pair), the up half the next row.
static bool encode_w13_groups(CUtensorMap* m, const PrefillArgs& a) {
  const uint64_t rb = (uint64_t)a.K / 2;
  const uint64_t dims[3] = {rb, a.oai ? (uint64_t)a.E * a.I : (uint64_t)a.E * 2 * a.I, 2};
  const uint64_t strides[2] = {a.oai ? 2 * rb : rb, a.oai ? rb : (uint64_t)a.I * rb};
  const uint32_t box[3] = {32, kPBoxRows, 2};
  return encode_tiled_u8(m, a.w13, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream, void* const* phase_events,
                           int n_events) {
  auto rec = [&](int i) {
    if (phase_events != nullptr && i < n_events)
      cudaEventRecord(static_cast<cudaEvent_t>(phase_events[i]), stream);
  };
  const int R = a.T * a.topk;
  rec(0);
  cudaError_t e = launch_route_parts(a.ids, R, a.E, a.ebase, a.window, a.count, a.offset, a.list,
                                     a.status, a.rpart, stream);
  if (e != cudaSuccess) return e;
  int gblocks = a.num_sms * 8;
  gather_kernel<<<gblocks, 256, 0, stream>>>(a.hidden, a.list, a.offset + a.E, a.K, a.topk, a.xp,
                                             a.inv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  rec(1);

  GemmParams g1 = {};
  if (!encode_tiled_2d(&g1.tmapX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.xp, (uint64_t)a.K, (uint64_t)R,
                       (uint64_t)a.K * 2, kBK, kXBox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_w13_groups(&g1.tmapW, a))
    return cudaErrorInvalidValue;
  g1.wsc = a.s13;
  g1.count = a.count;
  g1.offset = a.offset;
  g1.list = a.list;
  g1.wts = a.wts;
  g1.hp = a.hp;
  g1.P = a.P;
  g1.E = a.E;
  g1.K = a.K;
  g1.I = a.I;
  g1.kred = a.K;
  g1.NT = a.I / 64;   // 64 gate + 64 up rows a tile
  g1.status = a.status;
  g1.bias = a.b13;
  g1.oai = a.oai;
  if ((e = launch_gemm<1>(g1, a.num_sms, stream)) != cudaSuccess) return e;
  rec(2);

  GemmParams g2 = g1;
  if (!encode_tiled_2d(&g2.tmapX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.hp, (uint64_t)a.I, (uint64_t)R,
                       (uint64_t)a.I * 2, kBK, kXBox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_2d(&g2.tmapW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w2, (uint64_t)a.I / 2,
                       (uint64_t)a.E * a.K, (uint64_t)a.I / 2, 32, kPBoxRows,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  g2.wsc = a.s2;
  g2.bias = a.b2;
  g2.kred = a.I;
  g2.NT = (a.K + kBM - 1) / kBM;   // K % 64 == 0: the last tile may hold 64 rows
  if ((e = launch_gemm<2>(g2, a.num_sms, stream)) != cudaSuccess) return e;
  rec(3);
  {
    const int64_t n = (int64_t)(a.per_route ? R : a.T) * (a.K / 8);
    int64_t blocks = (n + 255) / 256;
    if (blocks > (int64_t)a.num_sms * 8) blocks = (int64_t)a.num_sms * 8;
    if (a.per_route)
      route_rows_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a.P, a.ids, a.inv, R, a.K, a.E,
                                                              a.ebase, a.window, a.y);
    else
      combine_pos_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a.P, a.ids, a.wts, a.inv, a.T, a.K,
                                                               a.E, a.topk, a.ebase, a.window,
                                                               a.y);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  rec(4);
  return cudaSuccess;
}

}  // namespace mxmoe
