// Packed MXFP4 rows -> bf16 ("MXFP4 MoE decode kernels", Prefill: mxk_deq
// unpacks an expert's weights straight to bf16), in either of the two ways
// the layer's kernels decode weights, so that a bit-exact test of this entry
// point pins the decode of each path:
//  form 1  the decode kernels' conversion: hardware e2m1x2 -> f16x2 (exact),
//          then an exact fp32 multiply by 2^(s-127) (e8m0_to_f32). Every
//          product is representable in fp32 (E2M1 has two significant bits),
//          so the only rounding is the final fp32 -> bf16 one.
//  form 2  the prefill GEMM's operand A (dequant32_bf16_pairs, the device
//          function the GEMM's dequant warps call, then put in row order): the
//          E2M1 fields placed in a bf16 bit pattern, then one or two exact
//          bf16 multiplies.
// Both are exact except where the product leaves the bf16 range.
#include "common.cuh"
#include "kernels.h"

namespace mxmoe {

__device__ __forceinline__ uint32_t f16x2_scale_to_bf16x2(uint32_t h2, float s) {
  float lo, hi;
  asm("{\n .reg .f16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  uint32_t o;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(hi * s), "f"(lo * s));
  return o;
}

// One thread per 32-value scale block: 16 packed bytes + 1 scale byte -> 64 B.
template <int FORM>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ packed,
                                                      const uint8_t* __restrict__ scale,
                                                      int rows, int cols,
                                                      uint32_t* __restrict__ out) {
  grid_dependency_wait();
  const int nblk = cols / kScaleBlock;
  const int64_t total = (int64_t)rows * nblk;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = *reinterpret_cast<const uint4*>(packed + i * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t* o = out + i * 16;   // 32 bf16 = 16 words
    if constexpr (FORM == 1) {
      const float s = e8m0_to_f32(scale[i]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t h0, h1, h2, h3;   // byte j of word q -> values 8q+2j, 8q+2j+1
        e2m1x8_to_f16x2(w[q], h0, h1, h2, h3);
        o[4 * q + 0] = f16x2_scale_to_bf16x2(h0, s);
        o[4 * q + 1] = f16x2_scale_to_bf16x2(h1, s);
        o[4 * q + 2] = f16x2_scale_to_bf16x2(h2, s);
        o[4 * q + 3] = f16x2_scale_to_bf16x2(h3, s);
      }
    } else {
      uint32_t r[16];
      dequant32_bf16(w, scale_mul(scale[i]), r);
#pragma unroll
      for (int q = 0; q < 16; ++q) o[q] = r[q];
    }
  }
}

cudaError_t launch_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                           int form, uint16_t* out, int num_sms, cudaStream_t stream) {
  const int64_t total = (int64_t)rows * (cols / kScaleBlock);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  uint32_t* o = reinterpret_cast<uint32_t*>(out);
  if (form == 2)
    dequant_kernel<2><<<(unsigned)blocks, 256, 0, stream>>>(packed, scale, rows, cols, o);
  else
    dequant_kernel<1><<<(unsigned)blocks, 256, 0, stream>>>(packed, scale, rows, cols, o);
  return cudaGetLastError();
}

}  // namespace mxmoe
