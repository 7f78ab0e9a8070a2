// Device helpers shared by the kernels of the MXFP4 MoE library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mxmoe {

constexpr int kScaleBlock = 32;        // E2M1 values per E8M0 scale
constexpr int kMaxExperts = 1024;
constexpr int kDecodeMaxTokens = 32;
constexpr int kDecodeMaxRoutes = 1024;
constexpr int kGrantDevices = 64;      // devices whose kernel attributes are tracked

// ---------------------------------------------------------------------------
// Small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// 16 bytes through a generic address (shared or global memory), not cached in
// L1 when global.
__device__ __forceinline__ uint4 ld_cg_generic16(const void* p) {
  uint4 v;
  asm volatile("ld.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// 16-byte load that skips L1, for data other SMs wrote during this kernel.
__device__ __forceinline__ uint4 ldcg16(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

// Programmatic dependent launch: wait until the grid this one depends on has
// finished (or triggered) before reading its results.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}



// Exact bf16x2 product (inputs and results may be subnormal).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  // fma with a -0 addend returns the rounded product, sign of zero included
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// ---------------------------------------------------------------------------
// E2M1 -> bf16
//
// An E2M1 code s.e1e0.m (sign bit 3) has magnitude (1 + m/2) * 2^(e-1) for
// e > 0 and m/2 for e = 0. Writing (e1, e0, m) into bits 8..6 of a bf16 gives
// exponent field e and leading mantissa bit m, i.e. exactly magnitude *
// 2^-126 -- including the two e = 0 codes, which land on bf16 subnormals --
// and the sign goes to bit 15. One exact bf16 multiply by 2^126 * 2^(s-127)
// then gives E2M1 * 2^(s-127).
//
// e2m1_word_raw(w, r) places nibbles P and P+4 of the 32-bit word w (bits
// 4P..4P+3 and 4P+16..4P+19, which sit 16 bits apart) into the low and high
// bf16 of r[P]. A code c isolated at bits 0..3 of a half, times 0x1040, is
// c << 6 + c << 12 with no carries (bits 6..9 and 12..15): the magnitude lands
// on bits 6..8 and the sign on bit 15, the mask clears the two copies' other
// bits. Odd nibbles sit 4 bits higher and take 0x104 instead. One integer
// multiply does the work of two shifts and a merge.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t mul_lo(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.lo.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void e2m1_word_raw(uint32_t w, uint32_t (&r)[4]) {
  constexpr uint32_t kKeep = 0x81C081C0u;   // bits 6..8 and 15 of each half
  const uint32_t w8 = w >> 8;
  r[0] = mul_lo(w & 0x000F000Fu, 0x1040u) & kKeep;    // nibbles 0, 4
  r[1] = mul_lo(w & 0x00F000F0u, 0x0104u) & kKeep;    // nibbles 1, 5
  r[2] = mul_lo(w8 & 0x000F000Fu, 0x1040u) & kKeep;   // nibbles 2, 6
  r[3] = mul_lo(w8 & 0x00F000F0u, 0x0104u) & kKeep;   // nibbles 3, 7
}

// Multiplier pair for one E8M0 scale byte s. For s <= 128 a single exact
// multiply by 2^(s-1) turns a raw pair into E2M1 * 2^(s-127). Larger bytes
// need two steps (2^126, then 2^(s-127)); 255 is NaN.
struct ScaleMul {
  uint32_t m1;    // bf16x2
  uint32_t m2;    // bf16x2, only used when two == true
  bool two;
};

__device__ __forceinline__ ScaleMul scale_mul(uint32_t s) {
  ScaleMul r;
  if (s <= 128u) {
    const uint32_t b = (s + 126u) << 7;            // bf16 bits of 2^(s-1)
    r.m1 = b | (b << 16);
    r.m2 = 0;
    r.two = false;
  } else {
    r.m1 = 0x7E807E80u;                            // 2^126
    const uint32_t b = (s == 255u) ? 0x7FC0u : (s << 7);   // 2^(s-127) or NaN
    r.m2 = b | (b << 16);
    r.two = true;
  }
  return r;
}


// One 32-value scale block as exact bf16 by integer bit placement and bf16
// multiplies (the prefill GEMM's operand A): wd holds the 16 packed bytes
// (value 2i in the low nibble of byte i), sm the block's scale multipliers.
// Pair order, the order in which the bit placement produces them:
// o[4c + P] = values (8c + P, 8c + P + 4) as a bf16 pair (low half first), so
// each group of 8 values is held in the order 0 4 1 5 2 6 3 7. The GEMM's
// token rows carry the same order inside each group of 8 (the dot products
// are unchanged), which saves the byte permutes of row order.
__device__ __forceinline__ void dequant32_bf16_pairs(const uint32_t (&wd)[4], const ScaleMul& sm,
                                                     uint32_t (&o)[16]) {
  uint32_t r[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {   // values 8c .. 8c+7: o[4c + P] = (n_P, n_P+4)
    e2m1_word_raw(wd[c], r);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[4 * c + q] = bf16x2_mul(r[q], sm.m1);
  }
  if (__builtin_expect(sm.two, 0)) {   // scale bytes above 128: the second exact step
#pragma unroll
    for (int q = 0; q < 16; ++q) o[q] = bf16x2_mul(o[q], sm.m2);
  }
}
// The same block in row order: o[4c .. 4c+3] = values 8c .. 8c+7 as bf16
// pairs (low half first).
__device__ __forceinline__ void dequant32_bf16(const uint32_t (&wd)[4], const ScaleMul& sm,
                                               uint32_t (&o)[16]) {
  uint32_t q[16];
  dequant32_bf16_pairs(wd, sm, q);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    o[4 * c + 0] = prmt(q[4 * c + 0], q[4 * c + 1], 0x5410u);   // (n0, n1)
    o[4 * c + 1] = prmt(q[4 * c + 2], q[4 * c + 3], 0x5410u);   // (n2, n3)
    o[4 * c + 2] = prmt(q[4 * c + 0], q[4 * c + 1], 0x7632u);   // (n4, n5)
    o[4 * c + 3] = prmt(q[4 * c + 2], q[4 * c + 3], 0x7632u);   // (n6, n7)
  }
}
// Position of value k of a group of 8 in pair order (0 4 1 5 2 6 3 7).
__host__ __device__ __forceinline__ int pair_order_pos(int k) { return 2 * (k & 3) + (k >> 2); }

// silu(z) = z * sigmoid(z) with the fast exponential and division (a few ulp
// of fp32; the product is rounded to bf16 afterwards).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// SwiGLU-OAI ("MXFP4 MoE decode kernels", Design, Fused epilogues) with the
// same fast exponential and division: gate capped at 7 (no lower cap), up
// clamped to [-7, 7], gate * sigmoid(1.702 gate) * (up + 1); comparisons keep
// a NaN input NaN.
__device__ __forceinline__ float swiglu_oai_fast(float gate, float up) {
  gate = gate > 7.0f ? 7.0f : gate;
  up = up > 7.0f ? 7.0f : (up < -7.0f ? -7.0f : up);
  return __fdividef(gate, 1.0f + __expf(-1.702f * gate)) * (up + 1.0f);
}

// fp32 -> bf16 bits, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

}  // namespace mxmoe

// ---------------------------------------------------------------------------
// Shared-memory barriers, bulk / tensor copies (TMA), FP4 conversion, f16 MMA
// ---------------------------------------------------------------------------
namespace mxmoe {

// Upper bound on polls of one mbarrier wait; a wait that runs out reports an
// error through the status word instead of spinning forever.
constexpr uint32_t kWaitLimit = 1u << 20;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity; false when it gave up.
// A phase that has already completed is seen by one non-blocking test, which
// answers sooner than the potentially blocking try_wait.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 2-D tensor copy global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// 3-D and 4-D tensor copies global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
// Contiguous bulk copy global -> shared (16-byte aligned addresses and size).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// A contiguous copy as pieces of at most 4 KB (larger single bulk copies were
// seen never to complete their transaction count on this part).
constexpr uint32_t kBulkPiece = 4096;
__device__ __forceinline__ void bulk_load_split(void* dst, const void* src, uint32_t bytes,
                                                uint64_t* bar) {
  for (uint32_t o = 0; o < bytes; o += kBulkPiece)
    bulk_load(static_cast<uint8_t*>(dst) + o, static_cast<const uint8_t*>(src) + o,
              bytes - o < kBulkPiece ? bytes - o : kBulkPiece, bar);
}
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Named barrier for a subset of the CTA's warps.
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Eight E2M1 codes (one 32-bit word, low nibble first) -> four f16x2, exact:
// result j holds the codes of byte j (low nibble in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& o0, uint32_t& o1,
                                                uint32_t& o2, uint32_t& o3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}

// E8M0 byte -> fp32 2^(s-127), exact for every byte (0 -> 2^-127 subnormal,
// 255 -> NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  uint32_t b = s << 23;
  if (((s + 1u) & 0xFEu) == 0u) b |= 0x00400000u;   // s == 0 or s == 255
  return __uint_as_float(b);
}
// The same for bytes known to be in 1..254: a single shift.
__device__ __forceinline__ float e8m0_to_f32_normal(uint32_t s) { return __uint_as_float(s << 23); }

// D += A * B for one m16n8k16 tile, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A * B (zero accumulator in).
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1,
                                                uint32_t a2, uint32_t a3, uint32_t b0,
                                                uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

}  // namespace mxmoe

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, tensor memory)
// ---------------------------------------------------------------------------
namespace mxmoe {

// Shared-memory matrix descriptor of a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes (64 bf16), 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)1 << 16;                                 // leading offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                      // stride between 8-row atoms
  d |= (uint64_t)1 << 46;                                 // descriptor version
  d |= (uint64_t)2 << 61;                                 // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 x bf16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// D[tmem] (+)= A[tmem] * B[smem]^T: operand A (M rows = lanes, K values as bf16
// pairs along columns) read from tensor memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// Arrive on an mbarrier once all tcgen05.mma issued so far by this thread completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the async proxy (tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Tensor-memory allocation by one whole warp; the base address lands in *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane (warp = lane quarter).
// The wait is in the same asm statement, so no use of the registers can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (warp = lane quarter),
// waiting for the write to complete.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Four 16x256b loads (16 lanes x 8 columns each, columns c0, c0+8, c0+16,
// c0+24) and their wait in one asm statement. For block u, thread t gets lane
// t/4 in v[u][0], v[u][1] (columns 2(t%4), 2(t%4)+1 of the block) and lane
// 8 + t/4 in v[u][2], v[u][3] (same columns).
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&v)[4][4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%16];\n"
      "tcgen05.ld.sync.aligned.16x256b.x1.b32 {%4,%5,%6,%7}, [%17];\n"
      "tcgen05.ld.sync.aligned.16x256b.x1.b32 {%8,%9,%10,%11}, [%18];\n"
      "tcgen05.ld.sync.aligned.16x256b.x1.b32 {%12,%13,%14,%15}, [%19];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0][0]), "=r"(v[0][1]), "=r"(v[0][2]), "=r"(v[0][3]), "=r"(v[1][0]),
        "=r"(v[1][1]), "=r"(v[1][2]), "=r"(v[1][3]), "=r"(v[2][0]), "=r"(v[2][1]),
        "=r"(v[2][2]), "=r"(v[2][3]), "=r"(v[3][0]), "=r"(v[3][1]), "=r"(v[3][2]),
        "=r"(v[3][3])
      : "r"(taddr), "r"(taddr + 8), "r"(taddr + 16), "r"(taddr + 24)
      : "memory");
}

}  // namespace mxmoe
