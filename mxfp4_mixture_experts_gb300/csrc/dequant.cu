// Packed MXFP4 rows -> bf16 ("MXFP4 MoE decode kernels", Prefill: mxk_deq
// unpacks an expert's weights straight to bf16). It uses the same register
// decode and exact scale multiply as the decode and prefill kernels, so the
// bit-exact test of this entry point also pins their dequantisation.
#include "common.cuh"
#include "kernels.h"

namespace mxmoe {

// One thread per 32-value scale block: 16 packed bytes + 1 scale byte -> 64 B.
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
    const ScaleMul sm = scale_mul(scale[i]);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t* o = out + i * 16;   // 32 bf16 = 16 words
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t p0 = apply_scale(e2m1_pair_raw<0>(w[q]), sm);   // (n0, n4)
      const uint32_t p1 = apply_scale(e2m1_pair_raw<1>(w[q]), sm);   // (n1, n5)
      const uint32_t p2 = apply_scale(e2m1_pair_raw<2>(w[q]), sm);   // (n2, n6)
      const uint32_t p3 = apply_scale(e2m1_pair_raw<3>(w[q]), sm);   // (n3, n7)
      // back to natural order: (n0,n1), (n2,n3), (n4,n5), (n6,n7)
      o[4 * q + 0] = prmt(p0, p1, 0x5410u);
      o[4 * q + 1] = prmt(p2, p3, 0x5410u);
      o[4 * q + 2] = prmt(p0, p1, 0x7632u);
      o[4 * q + 3] = prmt(p2, p3, 0x7632u);
    }
  }
}

cudaError_t launch_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                           uint16_t* out, int num_sms, cudaStream_t stream) {
  const int64_t total = (int64_t)rows * (cols / kScaleBlock);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  dequant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(packed, scale, rows, cols,
                                                       reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

}  // namespace mxmoe
