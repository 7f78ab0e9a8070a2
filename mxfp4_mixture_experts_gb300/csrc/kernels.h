// Host-side declarations shared by the kernel translation units and the C-ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mxmoe {

// One decode phase (1: w13 + SwiGLU, 2: w2 + weighted combine).
struct DecodeArgs {
  const uint16_t* x;      // phase 1: hidden bf16 [T, K]; phase 2: h bf16 [R, I]
  const int32_t* ids;     // [T * topk]
  const float* wts;       // [T * topk]
  const uint8_t* wq;      // packed weights of the phase
  const uint8_t* wsc;     // scales of the phase
  int T, K, I, E, topk;
  uint16_t* h;            // phase 1 output, bf16 [R, I]
  float* P;               // phase 2 weighted route outputs, fp32 [R, K]
  uint16_t* y;            // phase 2 output, bf16 [T, K]
  float* parts;           // stream-K partials [warps][2][128]
  int* item_ctr;          // [warps], zero between calls
  int* tile_ctr;          // [K / 16], zero between calls (phase 2)
  int32_t* status;        // [4] or null (phase 1 writes it)
  size_t smem_bytes;      // dynamic shared memory of the launch (tables + staged rows)
};

constexpr int kDecodeWarpsPerCta = 16;
constexpr int kMaxCtas = 256;            // grid cap; sizes the stream-K bookkeeping

// Shared-memory routing tables of a decode CTA (the staged activation rows
// follow them, 128-byte aligned).
__host__ __device__ inline size_t decode_smem_bytes(int T, int topk, int E) {
  const int R = T * topk;
  return sizeof(int) * (size_t)(E /*cnt*/ + (E + 1) /*off*/ + E /*run*/ + E /*touched*/ +
                                R /*lst*/ + 4 /*misc*/ + (E + 1) /*gbase*/);
}
cudaError_t launch_decode(const DecodeArgs& a, int phase, int num_sms, cudaStream_t stream,
                          bool pdl);

cudaError_t launch_route(const int32_t* ids, int R, int E, int32_t* count, int32_t* offset,
                         int32_t* list, int32_t* status, cudaStream_t stream);

cudaError_t launch_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                           uint16_t* out, int num_sms, cudaStream_t stream);

}  // namespace mxmoe
