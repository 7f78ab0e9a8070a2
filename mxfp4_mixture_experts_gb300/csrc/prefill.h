// Prefill path (many tokens): route -> gather -> grouped GEMM1 (+SwiGLU) ->
// grouped GEMM2 (+routing weight) -> slot-order combine.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mxmoe {

struct PrefillArgs {
  const uint16_t* hidden;   // bf16 [T, K]
  const int32_t* ids;       // [T * topk]
  const float* wts;         // [T * topk]
  const uint8_t *w13, *s13, *w2, *s2;
  int T, K, I, E, topk;
  uint16_t* y;              // bf16 [T, K]
  int32_t* status;
  // workspace regions
  int32_t* count;           // [E]
  int32_t* offset;          // [E+1]
  int32_t* list;            // [R]
  uint16_t* xp;             // bf16 [R, K], rows in expert order
  uint16_t* hp;             // bf16 [R, I], rows in expert order
  float* P;                 // fp32 [R, K], rows in expert order, unweighted
  int32_t* inv;             // [R] route -> row of P
  int32_t* rpart;           // route_part_ints(E): scratch of the many-CTA route sort
  int num_sms;
  // gpt-oss form (oai != 0): w13 rows interleaved (row 2i gate i, row 2i + 1
  // up i), f32 biases b13 [E, 2I] (same row order) and b2 [E, K], SwiGLU-OAI
  const float* b13;
  const float* b2;
  int oai;
  // expert window and per-route output, as in DecodeArgs
  int ebase, window, per_route;
};

cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream, void* const* phase_events,
                           int n_events);

}  // namespace mxmoe
