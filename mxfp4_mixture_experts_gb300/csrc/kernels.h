// Host-side declarations shared by the kernel translation units and the C-ABI.
#pragma once

#include <cuda.h>
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
  float* parts;           // stream-K partials [CTAs][2][256]
  int* item_ctr;          // [CTAs], zero between calls
  int32_t* status;        // [4] or null (phase 1 writes it)
};

constexpr int kMaxCtas = 256;            // grid cap; sizes the stream-K bookkeeping

// Kernel parameter block of one decode phase: the weight tensor map (TMA
// descriptor, 64-byte aligned) and the launch-time shared-memory plan.
struct DecodeParams {
  CUtensorMap tmap;       // packed weights of the phase as 2-D u8 [rows][row bytes]
  DecodeArgs a;
  int stages;             // weight pipeline depth (24 KB stages)
  int rows_cap;           // activation rows whose prescale is tracked (>= routes)
  int xs_rows_cap;        // activation rows staged in shared memory
  int xs_stride;          // bytes per staged row (f16), = 64 mod 128
};

// Shared-memory plan of a decode phase for a given stage count; returns the
// bytes needed before the staged activation rows (and their offset).
size_t decode_fixed_smem(int phase, int T, int K, int I, int E, int topk, int stages);

cudaError_t launch_decode(const DecodeArgs& a, int phase, int num_sms, int max_smem,
                          const CUtensorMap& tmap, cudaStream_t stream, bool pdl);

cudaError_t launch_combine(const float* P, const int32_t* ids, int T, int K, int E, int topk,
                           uint16_t* y, int num_sms, cudaStream_t stream, bool pdl);

// 2-D tiled tensor map [dim1 rows][dim0 elements] with the given row pitch,
// box {box0, box1}; reads past the tensor return zeros (api.cu).
bool encode_tiled_2d(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t dim0,
                     uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
                     CUtensorMapSwizzle swizzle);

cudaError_t launch_route(const int32_t* ids, int R, int E, int32_t* count, int32_t* offset,
                         int32_t* list, int32_t* status, cudaStream_t stream);

cudaError_t launch_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                           uint16_t* out, int num_sms, cudaStream_t stream);

}  // namespace mxmoe
