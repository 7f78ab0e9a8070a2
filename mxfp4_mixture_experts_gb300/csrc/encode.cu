// MXFP4 encoder: bf16 [rows, cols] -> E2M1 codes packed two per byte (value
// 2i in the low nibble of byte i) and one E8M0 scale per 32 values along the
// row ("GLM-5.2 and GLM-5.3 (744B) in MXFP4 on Gaudi 2", What was built,
// "MXFP4 encoder": the OCP shared exponent X = floor(log2(amax)) - 2; the
// Quark rule raises X by one when amax / 2^X >= 7).
//
// X is clamped to [-127, 127] (an all-zero block: byte 0); a block with a
// NaN or infinite value gets byte 255 and codes 0. Each element v / 2^X (an
// exact fp32 product) is rounded to E2M1 by the hardware conversion
// cvt.rn.satfinite.e2m1x2.f32: nearest, ties to the even code, magnitudes
// above 6 saturate to 6, the sign kept (-0 stays -0).
//
// One thread per 8 consecutive values (16 bytes in, 4 bytes of codes out);
// the 4 threads of a 32-value block share the block maximum through two
// shuffles, and the first of them writes the scale byte. HBM-bound: 2 + 17/32
// bytes per value.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mxmoe {
namespace {

constexpr int kEncThreads = 256;

// Eight fp32 values -> four bytes of E2M1 codes, value 2j in the low nibble
// of byte j (each conversion puts its second source in the low nibble).
__device__ __forceinline__ uint32_t e2m1x8_rn_sat(const float (&v)[8]) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

__global__ void __launch_bounds__(kEncThreads)
    encode_kernel(const uint4* __restrict__ in, int64_t n8, int quark,
                  uint32_t* __restrict__ packed, uint8_t* __restrict__ scale) {
  const int64_t stride = (int64_t)gridDim.x * kEncThreads;
  // every iteration covers whole warps, so the shuffles always see all lanes
  for (int64_t i = (int64_t)blockIdx.x * kEncThreads + threadIdx.x; i - (threadIdx.x & 31) < n8;
       i += stride) {
    const bool valid = i < n8;
    const uint4 q = valid ? in[i] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t m = 0;   // largest |v| as bf16 magnitude bits (integer order = magnitude order)
#pragma unroll
    for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const bool nonfinite = m >= 0x7F80u;
    const int E = (int)(m >> 7);   // bf16 exponent field of amax
    // floor(log2(amax)) = E - 127 for a normal amax; zero or subnormal: X = -127
    int X = E >= 1 ? E - 129 : -127;
    if (X < -127) X = -127;
    // Quark: amax / 2^X = 1.m x 4 >= 7  <=>  mantissa >= 0.75 (unclamped X only)
    if (quark && E >= 2 && (m & 0x7Fu) >= 96u) ++X;
    const float inv = __uint_as_float((uint32_t)(127 - X) << 23);   // 2^-X, exact
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16) * inv;
      v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * inv;
    }
    const uint32_t out = nonfinite ? 0u : e2m1x8_rn_sat(v);
    if (valid) {
      packed[i] = out;
      if ((threadIdx.x & 3) == 0) scale[i >> 2] = nonfinite ? 255u : (uint8_t)(X + 127);
    }
  }
}

}  // namespace

cudaError_t launch_encode(const uint16_t* x, int64_t rows, int64_t cols, int quark,
                          uint8_t* packed, uint8_t* scale, int num_sms, cudaStream_t stream) {
  const int64_t n8 = rows * cols / 8;
  if (n8 == 0) return cudaSuccess;
  int64_t blocks = (n8 + kEncThreads - 1) / kEncThreads;
  if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
  encode_kernel<<<(unsigned)blocks, kEncThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(x), n8, quark, reinterpret_cast<uint32_t*>(packed), scale);
  return cudaGetLastError();
}

}  // namespace mxmoe
