// Host-side declarations shared by the kernel translation units and the C-ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mxmoe {

// One decode call (1..32 tokens): w13 + SwiGLU, w2 + routing weight, combine.
struct DecodeArgs {
  const uint16_t* x;      // hidden bf16 [T, K]
  const int32_t* ids;     // [T * topk]
  const float* wts;       // [T * topk]
  const uint8_t *w13, *s13, *w2, *s2;
  int T, K, I, E, topk;
  uint16_t* h;            // bf16 [R, I] (SwiGLU output)
  uint16_t* xf;           // f16 [R, max(K, I)]: prescaled activation rows that have no
                          // room in shared memory, by route-list position
  float* P;               // weighted route outputs, fp32 [R, K]
  uint16_t* y;            // bf16 [T, K]
  int* gbar;              // [2] grid-barrier counters, zero between calls
  int32_t* status;        // [4] or null
  // gpt-oss form (oai != 0): w13 rows interleaved (row 2i gate i, row 2i + 1
  // up i), f32 biases b13 [E, 2I] (same row order) and b2 [E, K], SwiGLU-OAI
  const float* b13;
  const float* b2;
  int oai;
  // expert window (window != 0): the weights hold experts ebase .. ebase+E-1,
  // other ids are skipped; per_route != 0: y is [T * topk, K], each route's
  // unweighted w2 output (zero rows for skipped routes)
  int ebase, window, per_route;
  // test only (-1 = off): this CTA does not arrive at the grid barrier after
  // phase 1, so every CTA's bounded waits on it run out and report it
  int skip_arrival_cta;
};

// Kernel parameter block: the two weight tensor maps (TMA descriptors,
// 64-byte aligned) and the launch-time shared-memory plan.
struct DecodeParams {
  // w13 as 3-D u8 {K/2 bytes, row groups, 2 halves}, box {128, 8, 2}: 8 gate
  // rows then the 8 matching up rows of one 128-byte column (row groups: rows
  // with the up half I rows later, or gate/up pairs of the gpt-oss form)
  CUtensorMap tmap1;
  CUtensorMap tmap2;      // w2 packed as 2-D u8 [E*K rows][I/2], box {128, 16}
  // whole 4 KB stages in one copy: w13 as 4-D u8 {128 bytes, row groups, 2
  // halves, whole 128-byte chunks of a row}, box {128, 8, 2, 2}; w2 as 3-D u8
  // {128 bytes, E*K rows, whole chunks}, box {128, 16, 2}
  CUtensorMap tmap1q;
  CUtensorMap tmap2q;
  DecodeArgs a;
  int stages;             // weight ring depth (4 KB stages)
  int xs_rows_cap;        // activation rows staged in shared memory
  int xs_stride;          // bytes per staged row (f16), = 64 mod 128
};

// Bytes at the start of every workspace that must be zero when a call starts
// (api.cu).
size_t workspace_zero_kept_bytes();

// Whether the decode kernel's shared-memory plan fits for these sizes.
bool decode_fits(int K, int I, int E, int T, int topk, int max_smem);
// Warps per CTA of the decode form a call would run (7: 7 consumers + producer).
int decode_warps(int K, int I, int E, int T, int topk, int max_smem);

// One cooperative launch (one CTA per SM, all resident) per decode call.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& tmap1, const CUtensorMap& tmap2,
                          const CUtensorMap& tmap1q, const CUtensorMap& tmap2q, int num_sms,
                          int max_smem, cudaStream_t stream);

// 2-D tiled tensor map [dim1 rows][dim0 elements] with the given row pitch,
// box {box0, box1}; reads past the tensor return zeros (api.cu).
bool encode_tiled_2d(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t dim0,
                     uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
                     CUtensorMapSwizzle swizzle);

// Tiled u8 tensor map of the given rank (2..5): dims and box innermost first,
// strides[i] = bytes between consecutive coordinates of dimension i + 1 (any
// order; the views may overlap); reads past a dimension return zeros (api.cu).
bool encode_tiled_u8(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle);

// ids outside [ebase, ebase + E) are skipped; without a window (window == 0,
// ebase == 0) ids >= E are counted as invalid in status[0].
cudaError_t launch_route(const int32_t* ids, int R, int E, int ebase, int window, int32_t* count,
                         int32_t* offset, int32_t* list, int32_t* status, cudaStream_t stream);

// The same sort over many CTAs for many routes (R >= kRoutePartMin; fewer go
// to launch_route): part is device scratch of route_part_ints(E) ints.
constexpr int kRoutePartCtas = 128;
constexpr int kRoutePartMin = 8192;
size_t route_part_ints(int E);
cudaError_t launch_route_parts(const int32_t* ids, int R, int E, int ebase, int window,
                               int32_t* count, int32_t* offset, int32_t* list, int32_t* status,
                               int32_t* part, cudaStream_t stream);

// MXFP4 encoder: bf16 [rows, cols] (cols % 32 == 0) -> packed [rows, cols/2]
// and E8M0 scales [rows, cols/32]; quark != 0 takes the Quark exponent rule
// (encode.cu).
cudaError_t launch_encode(const uint16_t* x, int64_t rows, int64_t cols, int quark,
                          uint8_t* packed, uint8_t* scale, int num_sms, cudaStream_t stream);

constexpr int kRouterMaxExperts = 1024;   // 32 per lane of one warp

// Router: logits fp32 [T, E] (+ bias [E] or null) -> top-k ids int32 [T, k]
// and weights fp32 [T, k]; scoring 0 = softmax over the chosen k, 1 = sigmoid
// renormalised over the chosen k (router.cu).
cudaError_t launch_router(const float* logits, const float* bias, int T, int E, int topk,
                          int scoring, int n_group, int topk_group, int bias_in_weights,
                          int32_t* ids, float* wts, int num_sms, cudaStream_t stream);

// form 1: the decode kernels' conversion; form 2: the prefill GEMM's (dequant.cu).
cudaError_t launch_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                           int form, uint16_t* out, int num_sms, cudaStream_t stream);

}  // namespace mxmoe
