// Prefill path (many tokens): the routed experts as grouped GEMMs on the
// 5th-generation tensor cores ("MXFP4 MoE decode kernels", Prefill: on large
// MoE models the routed experts are most of the prefill; the pages unpack the
// weights to bf16 and run a stock bf16 MoE op -- here the unpack is fused
// into the GEMM's shared-memory tiles instead).
//
//   route   stable counting sort of the routes by expert (route.cu)
//   gather  xp[pos] = hidden[token of route list[pos]]: rows in expert order
//   GEMM1   per expert: [M_e x K] x [K x 2I]^T -> SwiGLU -> hp [M_e x I] bf16
//   GEMM2   per expert: [M_e x I] x [I x K]^T -> x routing weight -> P[route] fp32
//   combine y[t] = bf16(sum of the token's route outputs, slot order)
//
// GEMM kernel: one persistent CTA per SM, tiles (expert, 256 weight rows, up to
// 2 x 128 tokens) dealt round-robin. Warp roles:
//   warp 0      TMA producer of activation tiles (128 rows x 64 bf16, 128-byte
//               swizzle)
//   warp 1      MMA issuer: tcgen05.mma M128 N256 K16 (bf16, fp32 accumulators
//               in tensor memory: 2 m-tiles x 256 columns)
//   warp 2      TMA producer of packed weight bytes (256 rows x 32 bytes a stage)
//   warps 4..7  epilogue: tcgen05.ld of the accumulators (one TMEM lane per
//               token row) -> SwiGLU / routing weight -> global
//   warps 8..15 dequant: packed E2M1 + E8M0 -> exact bf16 in the canonical
//               K-major 128-byte-swizzled layout the MMA reads, one row a thread
// The two m-tiles' accumulators are released separately, so the next tile's
// first MMAs start as soon as the epilogue has read the first m-tile.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "prefill.h"

namespace mxmoe {

constexpr int kPfWarps = 16;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kBM = 128;                  // tokens per m-tile
constexpr int kBN = 256;                  // weight rows per tile (MMA N)
constexpr int kHalf = kBN / 2;            // GEMM1: gate rows, then as many up rows
constexpr int kBK = 64;                   // K values per stage (128 bytes of bf16)
constexpr int kMT = 2;                    // m-tiles per tile
constexpr int kSA = 3, kSB = 3, kSP = 3;  // ring depths: activations, bf16 weights, packed
constexpr int kATile = kBM * kBK * 2;     // 16 KB
constexpr int kAStage = kMT * kATile;     // 32 KB
constexpr int kPStage = kBN * kBK / 2;    // 8 KB of packed bytes
constexpr int kBStage = kBN * kBK * 2;    // 32 KB of bf16
constexpr int kPBoxRows = 128;            // packed-weight copies are 128 rows x 32 bytes
constexpr int kTmemCols = kMT * kBN;      // 512: both m-tiles' accumulators
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpTmaW = 2, kWarpEpi = 4, kWarpDeq = 8;
constexpr int kDeqWarps = 8;              // one weight row per thread
constexpr int kScaleAhead = 8;            // k-stages of scale bytes held in registers
constexpr int kTokensPerTile = kMT * kBM;
static_assert(kDeqWarps * 32 == kBN, "one dequant thread per B row");

struct GemmParams {
  CUtensorMap tmapA;   // activations bf16 [R][kred], box {64, 128}, 128-byte swizzle
  CUtensorMap tmapB;   // packed weights u8 [rows][kred/2], box {32, 128}
  const uint8_t* wsc;  // scales u8 [rows][kred/32]
  const int32_t* count;
  const int32_t* offset;
  const int32_t* list;
  const float* wts;
  uint16_t* hp;        // GEMM1 output bf16 [R][I]
  float* P;            // GEMM2 output fp32 [R][K] (route order)
  int E, K, I, kred, NT;
  int32_t* status;
};

struct TileId {
  int e, nt, mp, nm;
};

__device__ __forceinline__ TileId decode_tile(int t, const int* tile_base, const int32_t* count,
                                              int E, int NT) {
  int lo = 0, hi = E;   // tile_base[lo] <= t < tile_base[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_base[mid] <= t) lo = mid; else hi = mid;
  }
  TileId id;
  id.e = lo;
  const int c = count[lo];
  const int mps = (c + kTokensPerTile - 1) / kTokensPerTile;
  const int local = t - tile_base[lo];
  id.nt = local / mps;
  id.mp = local - id.nt * mps;
  const int rem = c - id.mp * kTokensPerTile;
  id.nm = rem > kBM ? 2 : 1;
  return id;
}

// Output index (GEMM1: intermediate index, GEMM2: output column) of B row j,
// and whether it exists (the last tile of a dimension may be partial).
template <int PHASE>
__device__ __forceinline__ int out_index(const TileId& id, int j) {
  return PHASE == 1 ? id.nt * kHalf + (j & (kHalf - 1)) : id.nt * kBN + j;
}
template <int PHASE>
__device__ __forceinline__ bool row_valid(const TileId& id, const GemmParams& p, int j) {
  return out_index<PHASE>(id, j) < (PHASE == 1 ? p.I : p.K);
}
// Weight row of B row j: GEMM1 takes 128 gate rows then the matching 128 up rows.
template <int PHASE>
__device__ __forceinline__ int weight_row(const TileId& id, const GemmParams& p, int j) {
  if (PHASE == 1) return id.e * (2 * p.I) + (j < kHalf ? 0 : p.I) + out_index<1>(id, j);
  return id.e * p.K + out_index<2>(id, j);
}

// Bounded wait taken by a whole warp: every lane gets the same answer, so the
// warp stays converged for the .sync.aligned tensor-memory instructions.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// silu(z) = z * sigmoid(z) with the fast exponential and division (a few ulp
// of fp32; the product is rounded to bf16 afterwards).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

template <int PHASE>
__global__ void __launch_bounds__(kPfThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kSA * kAStage;
  uint8_t* sP = sB + kSB * kBStage;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(sP + kSP * kPStage);
  uint64_t* a_empty = a_full + kSA;
  uint64_t* p_full = a_empty + kSA;
  uint64_t* p_empty = p_full + kSP;
  uint64_t* b_full = p_empty + kSP;
  uint64_t* b_empty = b_full + kSB;
  uint64_t* d_full = b_empty + kSB;    // [kMT]
  uint64_t* d_empty = d_full + kMT;    // [kMT]
  uint64_t* drain = d_empty + kMT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* tile_base = reinterpret_cast<int*>(tmem_slot + 4);   // [E+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSA; ++i) { mbar_init(&a_full[i], 1); mbar_init(&a_empty[i], 1); }
    for (int i = 0; i < kSP; ++i) { mbar_init(&p_full[i], 1); mbar_init(&p_empty[i], kDeqWarps); }
    for (int i = 0; i < kSB; ++i) { mbar_init(&b_full[i], kDeqWarps); mbar_init(&b_empty[i], 1); }
    for (int i = 0; i < kMT; ++i) { mbar_init(&d_full[i], 1); mbar_init(&d_empty[i], 4); }
    mbar_init(drain, 1);
    fence_barrier_init();
    prefetch_tensormap(&p.tmapA);
    prefetch_tensormap(&p.tmapB);
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  if (warp == 3) {   // tile table: experts in order, (nt, mp) inside an expert
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? p.count[e] : 0;
      const int tiles = ((c + kTokensPerTile - 1) / kTokensPerTile) * p.NT;
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
    // ------------------------------------------------------------ activation producer
    int sa = 0, ka = 0;
    uint32_t pa = 0, apar = 0;   // parity of each stage's last fill
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const TileId id = decode_tile(t, tile_base, p.count, E, p.NT);
      const int m0 = p.offset[id.e] + id.mp * kTokensPerTile;
      for (int kc = 0; kc < nK; ++kc) {
        if (ka >= kSA && !mbar_wait(&a_empty[sa], pa ^ 1u)) { fail = 1; break; }
        apar = (apar & ~(1u << sa)) | (pa << sa);
        mbar_arrive_expect_tx(&a_full[sa], id.nm * kATile);
        for (int mt = 0; mt < id.nm; ++mt)
          tma_load_2d(sA + sa * kAStage + mt * kATile, &p.tmapA, kc * kBK, m0 + mt * kBM, &a_full[sa]);
        if (++sa == kSA) { sa = 0; pa ^= 1u; }
        ++ka;
      }
    }
    // no copy may still be landing in shared memory when the CTA exits
    for (int i = 0; i < kSA && i < ka; ++i) mbar_wait(&a_full[i], (apar >> i) & 1u);
  } else if (warp == kWarpTmaW && lane == 0) {
    // ------------------------------------------------------------ packed-weight producer
    // runs ahead of the dequant warps across tile boundaries
    int sp = 0, kp = 0;
    uint32_t pp = 0, ppar = 0;
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const TileId id = decode_tile(t, tile_base, p.count, E, p.NT);
      // rows of a partial last tile past the matrix read other experts' rows
      // (or zeros past the tensor): never stored
      const int r0 = weight_row<PHASE>(id, p, 0);
      const int r1 = PHASE == 1 ? r0 + p.I : r0 + kPBoxRows;
      for (int kc = 0; kc < nK; ++kc) {
        if (kp >= kSP && !mbar_wait(&p_empty[sp], pp ^ 1u)) { fail = 2; break; }
        ppar = (ppar & ~(1u << sp)) | (pp << sp);
        mbar_arrive_expect_tx(&p_full[sp], kPStage);
        tma_load_2d(sP + sp * kPStage, &p.tmapB, kc * (kBK / 2), r0, &p_full[sp]);
        tma_load_2d(sP + sp * kPStage + kPBoxRows * (kBK / 2), &p.tmapB, kc * (kBK / 2), r1,
                    &p_full[sp]);
        if (++sp == kSP) { sp = 0; pp ^= 1u; }
        ++kp;
      }
    }
    for (int i = 0; i < kSP && i < kp; ++i) mbar_wait(&p_full[i], (ppar >> i) & 1u);
  } else if (warp == kWarpMma && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = umma_idesc_bf16(kBM, kBN);
    int sa = 0, sb = 0;
    uint32_t pa = 0, pb = 0;
    int uses[kMT] = {0, 0};   // earlier tiles that accumulated into each m-tile
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const TileId id = decode_tile(t, tile_base, p.count, E, p.NT);
      for (int kc = 0; kc < nK && !fail; ++kc) {
        if (!mbar_wait(&a_full[sa], pa) || !mbar_wait(&b_full[sb], pb)) { fail = 8; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sA + sa * kAStage);
        const uint32_t b_addr = smem_u32(sB + sb * kBStage);
        for (int mt = 0; mt < id.nm; ++mt) {
          if (kc == 0 && uses[mt] > 0) {   // the epilogue must have read the last tile's m-tile
            if (!mbar_wait(&d_empty[mt], (uses[mt] - 1) & 1)) { fail = 4; break; }
            tc_fence_after();
          }
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16)
            umma_bf16(tmem + mt * kBN, umma_desc_sw128(a_addr + mt * kATile + k16 * 32),
                      umma_desc_sw128(b_addr + k16 * 32), idesc, kc > 0 || k16 > 0);
        }
        umma_commit(&a_empty[sa]);
        umma_commit(&b_empty[sb]);
        if (++sa == kSA) { sa = 0; pa ^= 1u; }
        if (++sb == kSB) { sb = 0; pb ^= 1u; }
      }
      if (fail) break;
      for (int mt = 0; mt < id.nm; ++mt) {
        umma_commit(&d_full[mt]);
        ++uses[mt];
      }
    }
    // every issued MMA has finished before tensor memory is released
    umma_commit(drain);
    mbar_wait(drain, 0);
  } else if (warp >= kWarpDeq && warp < kWarpDeq + kDeqWarps) {
    // ------------------------------------------------------------ dequant
    // thread j: B row j, all 64 values of each stage
    const int j = threadIdx.x - kWarpDeq * 32;
    int sp = 0, sb = 0, kb = 0;
    uint32_t pp = 0, pb = 0;
    uint8_t* const drow0 = sB + (j >> 3) * 1024 + (j & 7) * 128;
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const TileId id = decode_tile(t, tile_base, p.count, E, p.NT);
      // rows of a partial last tile are never stored: they take any
      // in-bounds scale row
      const int row = weight_row<PHASE>(id, p, row_valid<PHASE>(id, p, j) ? j : 0);
      const uint8_t* srow = p.wsc + (size_t)row * (p.kred / kScaleBlock);
      // the two scale bytes of each of the next kScaleAhead stages, loaded one window early
      uint32_t sc[kScaleAhead];
#pragma unroll
      for (int i = 0; i < kScaleAhead; ++i) sc[i] = i < nK ? ldg_u16(srow + 2 * i) : 0u;
      for (int k0 = 0; k0 < nK && !fail; k0 += kScaleAhead) {
        uint32_t nx[kScaleAhead];
#pragma unroll
        for (int i = 0; i < kScaleAhead; ++i)
          nx[i] = k0 + kScaleAhead + i < nK ? ldg_u16(srow + 2 * (k0 + kScaleAhead + i)) : 0u;
#pragma unroll
        for (int i = 0; i < kScaleAhead; ++i) {
          if (k0 + i >= nK || fail) break;
          if (!warp_wait(&p_full[sp], pp)) { fail = 16; break; }
          const uint4* src = reinterpret_cast<const uint4*>(sP + sp * kPStage + j * (kBK / 2));
          const uint4 q0 = src[0], q1 = src[1];
          // the stage is refilled by the tensor-copy engine (async proxy): the
          // generic reads above must be ordered before that write
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_empty[sp]);
          if (++sp == kSP) { sp = 0; pp ^= 1u; }
          if (kb >= kSB && !warp_wait(&b_empty[sb], pb ^ 1u)) { fail = 32; break; }
          const ScaleMul s0 = scale_mul(sc[i] & 0xFFu), s1 = scale_mul(sc[i] >> 8);
          const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
          uint8_t* drow = drow0 + sb * kBStage;
#pragma unroll
          for (int c = 0; c < 8; ++c) {   // chunk c = values 8c .. 8c+7 of the stage
            const ScaleMul& sm = c < 4 ? s0 : s1;
            const uint32_t p0 = apply_scale(e2m1_pair_raw<0>(w[c]), sm);   // (n0, n4)
            const uint32_t p1 = apply_scale(e2m1_pair_raw<1>(w[c]), sm);   // (n1, n5)
            const uint32_t p2 = apply_scale(e2m1_pair_raw<2>(w[c]), sm);   // (n2, n6)
            const uint32_t p3 = apply_scale(e2m1_pair_raw<3>(w[c]), sm);   // (n3, n7)
            *reinterpret_cast<uint4*>(drow + ((c ^ (j & 7)) << 4)) =
                make_uint4(prmt(p0, p1, 0x5410u), prmt(p2, p3, 0x5410u), prmt(p0, p1, 0x7632u),
                           prmt(p2, p3, 0x7632u));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&b_full[sb]);
          if (++sb == kSB) { sb = 0; pb ^= 1u; }
          ++kb;
        }
#pragma unroll
        for (int i = 0; i < kScaleAhead; ++i) sc[i] = nx[i];
      }
    }
  } else if (warp >= kWarpEpi && warp < kWarpEpi + 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quarter of this warp
    int uses[kMT] = {0, 0};
    for (int t = blockIdx.x; t < ntiles && !fail; t += gridDim.x) {
      const TileId id = decode_tile(t, tile_base, p.count, E, p.NT);
      const int c = p.count[id.e];
      for (int mt = 0; mt < id.nm; ++mt) {
        if (!warp_wait(&d_full[mt], uses[mt] & 1)) { fail = 64; break; }
        tc_fence_after();
        const int local = id.mp * kTokensPerTile + mt * kBM + q * 32 + lane;
        const bool valid = local < c;
        const int pos = p.offset[id.e] + local;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + mt * kBN;
        if (PHASE == 1) {
          const int n32 = min(kHalf, p.I - id.nt * kHalf) >> 5;
#pragma unroll 1
          for (int c32 = 0; c32 < n32; ++c32) {
            float gv[32], uv[32];
            tmem_ld32(taddr + c32 * 32, gv);
            tmem_ld32(taddr + kHalf + c32 * 32, uv);
            uint32_t hb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = silu_fast(gv[2 * i]) * uv[2 * i];
              const float h1 = silu_fast(gv[2 * i + 1]) * uv[2 * i + 1];
              asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hb[i]) : "f"(h1), "f"(h0));
            }
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(p.hp + (size_t)pos * p.I + id.nt * kHalf + c32 * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
            }
          }
        } else {
          const int r = valid ? p.list[pos] : 0;
          const float wr = valid ? p.wts[r] : 0.f;
          const int n32 = min(kBN, p.K - id.nt * kBN) >> 5;
#pragma unroll 1
          for (int c32 = 0; c32 < n32; ++c32) {
            float v[32];
            tmem_ld32(taddr + c32 * 32, v);
            if (valid) {
              float4* dst = reinterpret_cast<float4*>(p.P + (size_t)r * p.K + id.nt * kBN + c32 * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(wr * v[4 * i], wr * v[4 * i + 1], wr * v[4 * i + 2],
                                     wr * v[4 * i + 3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_empty[mt]);
        ++uses[mt];
      }
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

// xp[pos] = hidden[list[pos] / topk] for the valid (expert-sorted) routes.
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ hidden,
                                                     const int32_t* __restrict__ list,
                                                     const int32_t* __restrict__ n_valid, int K,
                                                     int topk, uint16_t* __restrict__ xp) {
  const int n = *n_valid;
  const int per_row = K / 8;
  const int64_t total = (int64_t)n * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int pos = (int)(i / per_row), c = (int)(i - (int64_t)pos * per_row);
    const int tok = list[pos] / topk;
    reinterpret_cast<uint4*>(xp + (size_t)pos * K)[c] =
        reinterpret_cast<const uint4*>(hidden + (size_t)tok * K)[c];
  }
}

static size_t gemm_smem_bytes(int E) {
  return 1024 + (size_t)kSA * kAStage + (size_t)kSB * kBStage + (size_t)kSP * kPStage +
         (size_t)(2 * kSA + 2 * kSP + 2 * kSB + 2 * kMT + 1) * 8 + 16 + (size_t)(E + 1) * 4;
}

size_t prefill_counter_bytes(int, int, int, int, int) { return 256; }

template <int PHASE>
static cudaError_t launch_gemm(const GemmParams& gp, int num_sms, cudaStream_t stream) {
  static size_t granted = 0;
  const size_t smem = gemm_smem_bytes(gp.E);
  if (smem > granted) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<PHASE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    granted = smem;
  }
  gemm_kernel<PHASE><<<num_sms, kPfThreads, smem, stream>>>(gp);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream, void* const* phase_events,
                           int n_events) {
  auto rec = [&](int i) {
    if (phase_events != nullptr && i < n_events)
      cudaEventRecord(static_cast<cudaEvent_t>(phase_events[i]), stream);
  };
  const int R = a.T * a.topk;
  rec(0);
  cudaError_t e = launch_route(a.ids, R, a.E, a.count, a.offset, a.list, a.status, stream);
  if (e != cudaSuccess) return e;
  int gblocks = a.num_sms * 8;
  gather_kernel<<<gblocks, 256, 0, stream>>>(a.hidden, a.list, a.offset + a.E, a.K, a.topk, a.xp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  rec(1);

  GemmParams g1 = {};
  if (!encode_tiled_2d(&g1.tmapA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.xp, (uint64_t)a.K, (uint64_t)R,
                       (uint64_t)a.K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_2d(&g1.tmapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w13, (uint64_t)a.K / 2,
                       (uint64_t)a.E * 2 * a.I, (uint64_t)a.K / 2, 32, kPBoxRows,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
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
  g1.NT = (a.I + kHalf - 1) / kHalf;   // I % 64 == 0: the last tile may hold 64 rows
  g1.status = a.status;
  if ((e = launch_gemm<1>(g1, a.num_sms, stream)) != cudaSuccess) return e;
  rec(2);

  GemmParams g2 = g1;
  if (!encode_tiled_2d(&g2.tmapA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.hp, (uint64_t)a.I, (uint64_t)R,
                       (uint64_t)a.I * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_2d(&g2.tmapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w2, (uint64_t)a.I / 2,
                       (uint64_t)a.E * a.K, (uint64_t)a.I / 2, 32, kPBoxRows,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  g2.wsc = a.s2;
  g2.kred = a.I;
  g2.NT = (a.K + kBN - 1) / kBN;   // K % 64 == 0: the last tile may be partial
  if ((e = launch_gemm<2>(g2, a.num_sms, stream)) != cudaSuccess) return e;
  rec(3);
  if ((e = launch_combine(a.P, a.ids, a.T, a.K, a.E, a.topk, a.y, a.num_sms, stream, false)) !=
      cudaSuccess)
    return e;
  rec(4);
  return cudaSuccess;
}

}  // namespace mxmoe
