// Host side of the C ABI declared in include/mxfp4_moe.h: argument checks,
// workspace layout and kernel dispatch. Nothing here allocates, frees or
// synchronises; every call only enqueues work on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "../../include/mxfp4_moe.h"
#include "common.cuh"
#include "kernels.h"
#include "prefill.h"

namespace {

using namespace mxmoe;

constexpr int kDecodeMaxT = 32;
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool ok = false;
  int num_sms = 0;
  int max_smem = 0;   // opt-in dynamic shared memory per block
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

void* const* g_phase_events = nullptr;
int g_phase_n = 0;
int g_test_skip_arrival = -1;   // mxfp4_moe_test_skip_grid_arrival

// cuTensorMapEncodeTiled, fetched from the driver at first use (no link-time
// dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

bool get_encoder() {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_encode_tiled != nullptr) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// Checks the current device once (sm_103) and caches its SM count.
int current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXFP4_MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return MXFP4_MOE_ERR_CUDA;
    d.probed = true;
    d.ok = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.max_smem = smem;
  }
  if (!d.ok) return MXFP4_MOE_ERR_DEVICE;
  *out = &d;
  return MXFP4_MOE_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

// Workspace layout. The bookkeeping that must be zero between calls comes
// first; the scratch regions after it are overwritten by every call.
struct Layout {
  size_t gbar;                                             // zero-kept, fixed size
  size_t h, P, rcount, roffset, rlist, rinv, rpart, xp;    // scratch
  size_t total;
};

bool shape_ok(int T, int K, int I, int E, int topk) {
  if (T < 0 || K < 32 || I < 32 || K > 16384 || I > 16384) return false;
  if (K % 32 || I % 32) return false;
  if (E < 1 || E > kMaxExperts || topk < 1 || topk > 32 || topk > E) return false;
  if ((int64_t)T * topk * (int64_t)K >= ((int64_t)1 << 31)) return false;
  return true;
}

Layout layout(int T, int K, int I, int E, int topk) {
  Layout L;
  const size_t R = (size_t)T * topk;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += up256(bytes); return at; };
  // the zero-kept prefix has the same size for every call, so workspaces
  // sized for one T serve calls of any smaller T
  L.gbar = take(4 * sizeof(int));
  L.h = take(R * I * 2);
  L.P = take(R * K * sizeof(float));
  L.rcount = take((size_t)E * sizeof(int));
  L.roffset = take((size_t)(E + 1) * sizeof(int));
  L.rlist = take(R * sizeof(int));
  L.rinv = take(R * sizeof(int));
  L.rpart = take(route_part_ints(E) * sizeof(int));
  L.xp = take(R * (size_t)(K > I ? K : I) * 2);   // (decode: the f16 row scratch)
  L.total = o;
  return L;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MXFP4_MOE_OK : MXFP4_MOE_ERR_CUDA; }

void record_phase(int i, cudaStream_t s) {
  if (g_phase_events != nullptr && i < g_phase_n)
    cudaEventRecord(static_cast<cudaEvent_t>(g_phase_events[i]), s);
}

}  // namespace

namespace mxmoe {
// Bytes at the start of every workspace that must be zero when a call starts
// (the decode launch's counters; the same for all sizes).
size_t workspace_zero_kept_bytes() { return layout(1, 64, 64, 1, 1).h; }

bool encode_tiled_2d(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t dim0,
                     uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
                     CUtensorMapSwizzle swizzle) {
  if (!get_encoder()) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t es[2] = {1, 1};
  return g_encode_tiled(m, type, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool encode_tiled_u8(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  if (!get_encoder() || rank < 2 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides[i];
  return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d,
                        st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}
// Which routes a forward call computes and what it writes: an expert window
// (ids outside [ebase, ebase + E) skipped, not counted as invalid) and the
// per-route output (y [T * topk, K], unweighted) instead of the token sums.
struct RouteMode {
  int ebase = 0, window = 0, per_route = 0;
};

// The decode path (one cooperative launch) of both forward forms: tensor maps
// over the packed weights, then the kernel.
int run_decode(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
               const uint8_t* w13, const uint8_t* s13, const float* b13, const uint8_t* w2,
               const uint8_t* s2, const float* b2, int T, int K, int I, int E, int topk, void* out,
               int32_t* status, char* ws, const Layout& L, int oai, DeviceInfo* d, cudaStream_t s,
               RouteMode rm = RouteMode()) {
  DecodeArgs a = {};
  a.x = static_cast<const uint16_t*>(hidden);
  a.ids = topk_ids;
  a.wts = topk_weights;
  a.w13 = w13;
  a.s13 = s13;
  a.w2 = w2;
  a.s2 = s2;
  a.T = T;
  a.K = K;
  a.I = I;
  a.E = E;
  a.topk = topk;
  a.h = reinterpret_cast<uint16_t*>(ws + L.h);
  a.xf = reinterpret_cast<uint16_t*>(ws + L.xp);
  a.P = reinterpret_cast<float*>(ws + L.P);
  a.y = static_cast<uint16_t*>(out);
  a.gbar = reinterpret_cast<int*>(ws + L.gbar);
  a.status = status;
  a.b13 = b13;
  a.b2 = b2;
  a.oai = oai;
  a.ebase = rm.ebase;
  a.window = rm.window;
  a.per_route = rm.per_route;
  a.skip_arrival_cta = g_test_skip_arrival;
  // w13 row groups: the gate row of group p and its up row one half-stride
  // later -- [gate; up] per expert: p = e 2I + i, up I rows later; gpt-oss
  // (interleaved): p = e I + i, up the next row
  const uint64_t rb = (uint64_t)K / 2;                       // bytes per packed row
  const uint64_t groups = oai ? (uint64_t)E * I : (uint64_t)E * 2 * I;
  const uint64_t group_stride = oai ? 2 * rb : rb;
  const uint64_t half_stride = oai ? rb : (uint64_t)I * rb;
  // one 128-byte column of 8 gate + 8 up rows per copy, reads past the row
  // return zeros (the last, partial stage)
  CUtensorMap map1, map2;
  const uint64_t d1c[3] = {rb, groups, 2};
  const uint64_t st1c[2] = {group_stride, half_stride};
  const uint32_t b1c[3] = {128, 8, 2};
  if (!encode_tiled_u8(&map1, w13, 3, d1c, st1c, b1c, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_2d(&map2, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2, (uint64_t)I / 2, (uint64_t)E * K,
                       (uint64_t)I / 2, 128, 16, CU_TENSOR_MAP_SWIZZLE_128B))
    return MXFP4_MOE_ERR_CUDA;
  // whole stages (two 128-byte chunks of 8 gate + 8 up rows / 16 w2 rows) in
  // one copy; the chunk extent counts only whole chunks of a row, so a box
  // never reaches past a row (the last, partial stage takes the maps above)
  CUtensorMap map1q, map2q;
  const uint64_t nc1 = (uint64_t)K / 2 / 128, nc2 = (uint64_t)I / 2 / 128;
  // (rows with fewer than two whole chunks never take these maps)
  const uint64_t d1[4] = {128, groups, 2, nc1 > 2 ? nc1 : 2};
  const uint64_t st1[3] = {group_stride, half_stride, 128};
  const uint32_t b1[4] = {128, 8, 2, 2};
  const uint64_t d2[3] = {128, (uint64_t)E * K, nc2 > 2 ? nc2 : 2};
  const uint64_t st2[2] = {(uint64_t)I / 2, 128};
  const uint32_t b2q[3] = {128, 16, 2};
  if (!encode_tiled_u8(&map1q, w13, 4, d1, st1, b1, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_u8(&map2q, w2, 3, d2, st2, b2q, CU_TENSOR_MAP_SWIZZLE_128B))
    return MXFP4_MOE_ERR_CUDA;
  record_phase(0, s);
  const cudaError_t e = launch_decode(a, map1, map2, map1q, map2q, d->num_sms, d->max_smem, s);
  if (e != cudaSuccess) return MXFP4_MOE_ERR_CUDA;
  record_phase(1, s);
  return MXFP4_MOE_OK;
}

// The prefill path (route, gather, two grouped GEMMs, combine) of both
// forward forms.
int run_prefill(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                const uint8_t* w13, const uint8_t* s13, const float* b13, const uint8_t* w2,
                const uint8_t* s2, const float* b2, int T, int K, int I, int E, int topk,
                void* out, int32_t* status, char* ws, const Layout& L, int oai, DeviceInfo* d,
                cudaStream_t s, RouteMode rm = RouteMode()) {
  PrefillArgs p = {};
  p.hidden = static_cast<const uint16_t*>(hidden);
  p.ids = topk_ids;
  p.wts = topk_weights;
  p.w13 = w13;
  p.s13 = s13;
  p.w2 = w2;
  p.s2 = s2;
  p.T = T;
  p.K = K;
  p.I = I;
  p.E = E;
  p.topk = topk;
  p.y = static_cast<uint16_t*>(out);
  p.status = status;
  p.count = reinterpret_cast<int32_t*>(ws + L.rcount);
  p.offset = reinterpret_cast<int32_t*>(ws + L.roffset);
  p.list = reinterpret_cast<int32_t*>(ws + L.rlist);
  p.xp = reinterpret_cast<uint16_t*>(ws + L.xp);
  p.hp = reinterpret_cast<uint16_t*>(ws + L.h);   // SwiGLU output, expert order
  p.P = reinterpret_cast<float*>(ws + L.P);
  p.inv = reinterpret_cast<int32_t*>(ws + L.rinv);
  p.rpart = reinterpret_cast<int32_t*>(ws + L.rpart);
  p.num_sms = d->num_sms;
  p.b13 = b13;
  p.b2 = b2;
  p.oai = oai;
  p.ebase = rm.ebase;
  p.window = rm.window;
  p.per_route = rm.per_route;
  return cuda_status(launch_prefill(p, s, g_phase_events, g_phase_n));
}

}  // namespace mxmoe

extern "C" {

size_t mxfp4_moe_workspace_size(int T, int K, int I, int E, int topk) {
  if (!shape_ok(T, K, I, E, topk)) return 0;
  return layout(T, K, I, E, topk).total;
}

size_t mxfp4_moe_workspace_zero_bytes(void) { return mxmoe::workspace_zero_kept_bytes(); }

int mxfp4_moe_route(const int32_t* topk_ids, int T, int topk, int E, int32_t* expert_count,
                    int32_t* expert_offset, int32_t* route_list, int32_t* status, void* stream) {
  if (T < 0 || topk < 1 || topk > 32 || E < 1 || E > kMaxExperts) return MXFP4_MOE_ERR_SHAPE;
  if (expert_count == nullptr || expert_offset == nullptr) return MXFP4_MOE_ERR_ARG;
  if (T > 0 && (topk_ids == nullptr || route_list == nullptr)) return MXFP4_MOE_ERR_ARG;
  if ((int64_t)T * topk >= ((int64_t)1 << 30)) return MXFP4_MOE_ERR_SHAPE;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  return cuda_status(launch_route(topk_ids, T * topk, E, 0, 0, expert_count, expert_offset, route_list,
                                  status, static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_moe_route_workspace_size(int T, int topk, int E) {
  if (T < 0 || topk < 1 || topk > 32 || E < 1 || E > kMaxExperts) return 0;
  return route_part_ints(E) * sizeof(int);
}

int mxfp4_moe_route_ws(const int32_t* topk_ids, int T, int topk, int E, int32_t* expert_count,
                       int32_t* expert_offset, int32_t* route_list, int32_t* status,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || topk < 1 || topk > 32 || E < 1 || E > kMaxExperts) return MXFP4_MOE_ERR_SHAPE;
  if (expert_count == nullptr || expert_offset == nullptr) return MXFP4_MOE_ERR_ARG;
  if (T > 0 && (topk_ids == nullptr || route_list == nullptr)) return MXFP4_MOE_ERR_ARG;
  if ((int64_t)T * topk >= ((int64_t)1 << 30)) return MXFP4_MOE_ERR_SHAPE;
  if (workspace == nullptr || workspace_bytes < route_part_ints(E) * sizeof(int))
    return MXFP4_MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return MXFP4_MOE_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  return cuda_status(launch_route_parts(topk_ids, T * topk, E, 0, 0, expert_count, expert_offset,
                                        route_list, status, static_cast<int32_t*>(workspace),
                                        static_cast<cudaStream_t>(stream)));
}

int mxfp4_moe_forward(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                      const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                      const uint8_t* s2, int T, int K, int I, int E, int topk, void* out,
                      int32_t* status, void* workspace, size_t workspace_bytes, int path,
                      void* stream) {
  if (!shape_ok(T, K, I, E, topk)) return MXFP4_MOE_ERR_SHAPE;
  if (path < 0 || path > 2) return MXFP4_MOE_ERR_ARG;
  if (T == 0) return MXFP4_MOE_OK;
  if (!hidden || !topk_ids || !topk_weights || !w13 || !s13 || !w2 || !s2 || !out)
    return MXFP4_MOE_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(out, 16) || !aligned(w13, 16) || !aligned(w2, 16) ||
      !aligned(s13, 16) || !aligned(s2, 16))
    return MXFP4_MOE_ERR_ALIGN;
  if (workspace == nullptr) return MXFP4_MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MXFP4_MOE_ERR_ALIGN;
  const Layout L = layout(T, K, I, E, topk);
  if (workspace_bytes < L.total) return MXFP4_MOE_ERR_WORKSPACE;
  const bool decode = path == 1 || (path == 0 && T <= kDecodeMaxT);
  if (decode && (T > kDecodeMaxT || T * topk > kDecodeMaxRoutes || K % 64 || I % 64))
    return MXFP4_MOE_ERR_SHAPE;
  if (!decode && (K % 64 || I % 64)) return MXFP4_MOE_ERR_SHAPE;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  if (decode && !decode_fits(K, I, E, T, topk, d->max_smem)) return MXFP4_MOE_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);

  if (decode)
    return run_decode(hidden, topk_ids, topk_weights, w13, s13, nullptr, w2, s2, nullptr, T, K, I, E,
                      topk, out, status, ws, L, 0, d, s);

  return run_prefill(hidden, topk_ids, topk_weights, w13, s13, nullptr, w2, s2, nullptr, T, K, I, E,
                     topk, out, status, ws, L, 0, d, s);
}

int mxfp4_moe_forward_window(const void* hidden, const int32_t* topk_ids,
                             const float* topk_weights, const uint8_t* w13, const uint8_t* s13,
                             const uint8_t* w2, const uint8_t* s2, int T, int K, int I, int E,
                             int topk, int expert_base, int per_route, void* out, int32_t* status,
                             void* workspace, size_t workspace_bytes, int path, void* stream) {
  if (!shape_ok(T, K, I, E, topk)) return MXFP4_MOE_ERR_SHAPE;
  if (path < 0 || path > 2 || expert_base < 0 || (per_route != 0 && per_route != 1))
    return MXFP4_MOE_ERR_ARG;
  if (T == 0) return MXFP4_MOE_OK;
  if (!hidden || !topk_ids || (!topk_weights && !per_route) || !w13 || !s13 || !w2 || !s2 || !out)
    return MXFP4_MOE_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(out, 16) || !aligned(w13, 16) || !aligned(w2, 16) ||
      !aligned(s13, 16) || !aligned(s2, 16))
    return MXFP4_MOE_ERR_ALIGN;
  if (workspace == nullptr) return MXFP4_MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MXFP4_MOE_ERR_ALIGN;
  const Layout L = layout(T, K, I, E, topk);
  if (workspace_bytes < L.total) return MXFP4_MOE_ERR_WORKSPACE;
  const bool decode = path == 1 || (path == 0 && T <= kDecodeMaxT);
  if (decode && (T > kDecodeMaxT || T * topk > kDecodeMaxRoutes || K % 64 || I % 64))
    return MXFP4_MOE_ERR_SHAPE;
  if (!decode && (K % 64 || I % 64)) return MXFP4_MOE_ERR_SHAPE;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  if (decode && !decode_fits(K, I, E, T, topk, d->max_smem)) return MXFP4_MOE_ERR_SHAPE;
  RouteMode rm;
  rm.ebase = expert_base;
  rm.window = 1;
  rm.per_route = per_route;
  // per-route outputs ignore the routing weights (the caller applies them)
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (decode)
    return run_decode(hidden, topk_ids, topk_weights, w13, s13, nullptr, w2, s2, nullptr, T, K, I, E,
                      topk, out, status, ws, L, 0, d, s, rm);
  return run_prefill(hidden, topk_ids, topk_weights, w13, s13, nullptr, w2, s2, nullptr, T, K, I, E,
                     topk, out, status, ws, L, 0, d, s, rm);
}

int mxfp4_moe_forward_oai(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                          const uint8_t* w13, const uint8_t* s13, const float* b13,
                          const uint8_t* w2, const uint8_t* s2, const float* b2, int T, int K,
                          int I, int E, int topk, void* out, int32_t* status, void* workspace,
                          size_t workspace_bytes, int path, void* stream) {
  if (!shape_ok(T, K, I, E, topk)) return MXFP4_MOE_ERR_SHAPE;
  if (path < 0 || path > 2) return MXFP4_MOE_ERR_ARG;
  if (T == 0) return MXFP4_MOE_OK;
  if (!hidden || !topk_ids || !topk_weights || !w13 || !s13 || !b13 || !w2 || !s2 || !b2 || !out)
    return MXFP4_MOE_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(out, 16) || !aligned(w13, 16) || !aligned(w2, 16) ||
      !aligned(s13, 16) || !aligned(s2, 16) || !aligned(b13, 4) || !aligned(b2, 4))
    return MXFP4_MOE_ERR_ALIGN;
  if (workspace == nullptr) return MXFP4_MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MXFP4_MOE_ERR_ALIGN;
  const Layout L = layout(T, K, I, E, topk);
  if (workspace_bytes < L.total) return MXFP4_MOE_ERR_WORKSPACE;
  const bool decode = path == 1 || (path == 0 && T <= kDecodeMaxT);
  if (decode && (T > kDecodeMaxT || T * topk > kDecodeMaxRoutes || K % 64 || I % 64))
    return MXFP4_MOE_ERR_SHAPE;
  if (!decode && (K % 64 || I % 64)) return MXFP4_MOE_ERR_SHAPE;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  if (decode && !decode_fits(K, I, E, T, topk, d->max_smem)) return MXFP4_MOE_ERR_SHAPE;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (decode)
    return run_decode(hidden, topk_ids, topk_weights, w13, s13, b13, w2, s2, b2, T, K, I, E, topk,
                      out, status, ws, L, 1, d, s);
  return run_prefill(hidden, topk_ids, topk_weights, w13, s13, b13, w2, s2, b2, T, K, I, E, topk,
                     out, status, ws, L, 1, d, s);
}

int mxfp4_moe_router_grouped(const float* logits, const float* bias, int T, int E, int topk,
                             int scoring, int n_group, int topk_group, int bias_in_weights,
                             int32_t* topk_ids, float* topk_weights, void* stream) {
  if (T < 0 || E < 1 || E > kRouterMaxExperts || topk < 1 || topk > 32 || topk > E)
    return MXFP4_MOE_ERR_SHAPE;
  if (n_group < 1 || n_group > 32 || E % n_group || topk_group < 1 || topk_group > n_group ||
      topk > topk_group * (E / n_group))
    return MXFP4_MOE_ERR_SHAPE;
  if (scoring != 0 && scoring != 1) return MXFP4_MOE_ERR_ARG;
  if (bias_in_weights != 0 && bias_in_weights != 1) return MXFP4_MOE_ERR_ARG;
  if (T == 0) return MXFP4_MOE_OK;
  if (!logits || !topk_ids || !topk_weights) return MXFP4_MOE_ERR_ARG;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4) ||
      (bias != nullptr && !aligned(bias, 4)))
    return MXFP4_MOE_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  return cuda_status(launch_router(logits, bias, T, E, topk, scoring, n_group, topk_group,
                                   bias_in_weights, topk_ids, topk_weights, d->num_sms,
                                   static_cast<cudaStream_t>(stream)));
}

int mxfp4_moe_router(const float* logits, const float* bias, int T, int E, int topk, int scoring,
                     int32_t* topk_ids, float* topk_weights, void* stream) {
  return mxfp4_moe_router_grouped(logits, bias, T, E, topk, scoring, 1, 1, 1, topk_ids,
                                  topk_weights, stream);
}

int mxfp4_moe_encode(const void* x, int rows, int cols, int rule, uint8_t* packed,
                     uint8_t* scale, void* stream) {
  if (rows < 0 || cols < 32 || cols % 32) return MXFP4_MOE_ERR_SHAPE;
  if (rule != 0 && rule != 1) return MXFP4_MOE_ERR_ARG;
  if (rows == 0) return MXFP4_MOE_OK;
  if (!x || !packed || !scale) return MXFP4_MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(packed, 4)) return MXFP4_MOE_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  return cuda_status(launch_encode(static_cast<const uint16_t*>(x), rows, cols, rule, packed, scale,
                                   d->num_sms, static_cast<cudaStream_t>(stream)));
}

int mxfp4_moe_dequant_form(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                           int form, void* out, void* stream) {
  if (rows < 0 || cols < 0 || (form != 1 && form != 2)) return MXFP4_MOE_ERR_ARG;
  if (cols % 32) return MXFP4_MOE_ERR_SHAPE;
  if (rows == 0 || cols == 0) return MXFP4_MOE_OK;
  if (!packed || !scale || !out) return MXFP4_MOE_ERR_ARG;
  if (!aligned(packed, 16) || !aligned(out, 4)) return MXFP4_MOE_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  if (int rc = current_device(&d)) return rc;
  return cuda_status(launch_dequant(packed, scale, rows, cols, form, static_cast<uint16_t*>(out),
                                    d->num_sms, static_cast<cudaStream_t>(stream)));
}

int mxfp4_moe_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols, void* out,
                      void* stream) {
  return mxfp4_moe_dequant_form(packed, scale, rows, cols, 1, out, stream);
}

void mxfp4_moe_set_phase_events(void* const* events, int n) {
  if (events == nullptr || n < 3) {
    g_phase_events = nullptr;
    g_phase_n = 0;
  } else {
    g_phase_events = events;
    g_phase_n = n;
  }
}

void mxfp4_moe_test_skip_grid_arrival(int cta) { g_test_skip_arrival = cta < 0 ? -1 : cta; }

int mxfp4_moe_test_decode_form(int T, int K, int I, int E, int topk, int max_smem) {
  if (T < 1 || T > kDecodeMaxT || topk < 1 || topk > 32 || topk > E || E < 1 || E > kMaxExperts ||
      T * topk > kDecodeMaxRoutes || K < 64 || I < 64 || K % 64 || I % 64 || max_smem < 0)
    return -1;
  return mxmoe::decode_warps(K, I, E, T, topk, max_smem);
}

const char* mxfp4_moe_strerror(int code) {
  switch (code) {
    case MXFP4_MOE_OK: return "ok";
    case MXFP4_MOE_ERR_ARG: return "invalid argument (null pointer, negative size or bad path)";
    case MXFP4_MOE_ERR_SHAPE: return "unsupported shape (see the limits in mxfp4_moe.h)";
    case MXFP4_MOE_ERR_ALIGN: return "pointer alignment rule violated";
    case MXFP4_MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MXFP4_MOE_ERR_CUDA: return "CUDA runtime error";
    case MXFP4_MOE_ERR_DEVICE: return "current device is not an sm_103 GPU";
    default: return "unknown error code";
  }
}

int mxfp4_moe_version(void) { return 100; }

}  // extern "C"
