/*
 * mxfp4_moe.h -- C ABI of the routed-expert MXFP4 mixture-of-experts layer
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * The layer reads each expert's weights in the served packed layout
 * ("MXFP4 MoE decode kernels", Design, "Read the served layout"):
 *   w13  uint8 [E, 2I, K/2]   two E2M1 values per byte, low nibble first
 *   s13  uint8 [E, 2I, K/32]  one E8M0 scale per 32 values along K
 *   w2   uint8 [E, K, I/2]
 *   s2   uint8 [E, K, I/32]
 * and computes, for every token t and slot j of its top-k routing,
 *   g, u = split([gate; up] rows of dequant(w13[e])) . x_t     (fp32 accumulate)
 *   h    = bf16( silu(g) * u )                                  (one bf16 rounding)
 *   o    = dequant(w2[e]) . h                                   (fp32 accumulate)
 *   y_t  = bf16( sum_{j=0..k-1} w_tj * o_(t,j) )                (slot order)
 * where dequant(v) = E2M1(nibble) * 2^(E8M0 - 127) ("GLM-5.2 and GLM-5.3 (744B)
 * in MXFP4 on Gaudi 2", What was built, "Byte-exact repack"; "MXFP4 MoE decode
 * kernels", Design, "Unpack in registers" and "Fused epilogues"; Beyond
 * gpt-oss, "mxk_w13x: SiLU without bias for [gate; up] row layouts").
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer owned by the caller (for
 *    example a PyTorch CUDA tensor's data_ptr()), unless it is marked "host".
 *    The library never allocates device memory, never frees, and never
 *    synchronises the device: each call validates its arguments on the host,
 *    enqueues its kernels on `stream` (a cudaStream_t passed as void*, NULL =
 *    the legacy default stream) and returns.
 *  - A non-zero return value is an mxfp4_moe_status code and means nothing
 *    was enqueued (except MXFP4_MOE_ERR_CUDA, which reports a failed launch).
 *  - Conditions only the device can see are written to `status` (device
 *    int32[4]) by the enqueued work:
 *       status[0] = number of routes whose expert id is >= E (skipped)
 *       status[1] = number of distinct experts touched by the call
 *       status[2] = non-zero when a bounded wait inside a kernel gave up (the
 *                   output of that call is then not valid; never expected);
 *                   the bits name the wait: bits 0..7 the decode kernel's
 *                   producer, 8..15 its consumers, 16..23 the prefill path's
 *                   first GEMM, 24..31 its second. The workspace stays
 *                   usable after such a call: the decode kernel's last CTA
 *                   resets its counters on every exit path, and the prefill
 *                   path keeps no state in the workspace between calls
 *       status[3] = 1 + the first CTA that reported such a wait, else 0
 *    Negative expert ids are padding and are skipped silently.
 *  - Every call is deterministic: repeating it on the same inputs gives
 *    bit-identical outputs (no floating-point atomics anywhere).
 */
#ifndef MXFP4_MOE_H_
#define MXFP4_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXFP4_MOE_OK = 0,
  MXFP4_MOE_ERR_ARG = 1,        /* null pointer where one is required, negative size */
  MXFP4_MOE_ERR_SHAPE = 2,      /* shape outside the supported limits listed below */
  MXFP4_MOE_ERR_ALIGN = 3,      /* a pointer breaks its alignment rule */
  MXFP4_MOE_ERR_WORKSPACE = 4,  /* workspace missing or smaller than mxfp4_moe_workspace_size */
  MXFP4_MOE_ERR_CUDA = 5,       /* a CUDA runtime call failed (device query or launch) */
  MXFP4_MOE_ERR_DEVICE = 6      /* current device is not an sm_103 GPU */
} mxfp4_moe_status;

/* Shape limits (checked on the host, MXFP4_MOE_ERR_SHAPE otherwise):
 *   K % 32 == 0, I % 32 == 0, 32 <= K, I <= 16384
 *   1 <= E <= 1024, 1 <= topk <= 32, topk <= E, 0 <= T
 *   decode path: T <= 32, T * topk <= 1024, K % 64 == 0, I % 64 == 0 (scale
 *                rows are copied 8 rows at a time) and the kernel's shared-memory
 *                plan must fit: about 12 * max(K, I) + 20 * E + 2 * max(K, I)
 *                + 66 KB <= 227 KB (K, I <= 8192 always fit for E <= 256)
 *   prefill path: K % 64 == 0, I % 64 == 0 (tensor-core tiles), T * topk < 2^31 / K
 * Alignment (MXFP4_MOE_ERR_ALIGN otherwise): w13, s13, w2, s2, hidden and out
 * 16-byte aligned; workspace 256-byte aligned. */

/* Bytes of device workspace a forward call with these sizes needs (either
 * path). The bookkeeping part (the first mxfp4_moe_workspace_zero_bytes()
 * bytes) must be zero before the first call that uses a workspace; every call
 * leaves it zero again (also one whose bounded wait gave up), so a workspace
 * can be reused without clearing. Returns 0 for invalid sizes. */
size_t mxfp4_moe_workspace_size(int T, int K, int I, int E, int topk);

/* Bytes at the start of every workspace that hold the bookkeeping: they must
 * be zero before the first call (clearing only them is enough) and every call
 * leaves them zero. The same for all sizes (a few KB), so a workspace
 * sized for the largest call serves calls of any smaller size. */
size_t mxfp4_moe_workspace_zero_bytes(void);

/* Routing / permute ("MXFP4 MoE decode kernels", Design, "Routing inside the
 * kernel": a counting sort of the routes by expert; absent experts skipped).
 * Route r = t * topk + j. Outputs:
 *   expert_count  int32 [E]     routes per expert
 *   expert_offset int32 [E+1]   exclusive prefix sum, expert_offset[E] = valid routes
 *   route_list    int32 [T*topk] route ids grouped by expert in ascending
 *                 expert order, ascending r inside a group; entries past
 *                 expert_offset[E] are set to -1
 *   status        int32 [4]     as above (may be NULL)
 * topk_ids int32 [T, topk]. No workspace needed. */
int mxfp4_moe_route(const int32_t* topk_ids, int T, int topk, int E,
                    int32_t* expert_count, int32_t* expert_offset, int32_t* route_list,
                    int32_t* status, void* stream);

/* The same routing with device scratch for many routes: identical outputs
 * (bit for bit) to mxfp4_moe_route. From 8192 routes on it sorts over many
 * CTAs -- per-chunk expert counts, one prefix pass, an in-order placement per
 * chunk -- which is the form the prefill path runs; fewer routes take the
 * one-CTA sort. workspace: device memory of at least
 * mxfp4_moe_route_workspace_size(T, topk, E) bytes, 16-byte aligned
 * (MXFP4_MOE_ERR_WORKSPACE / MXFP4_MOE_ERR_ALIGN), no initial contents
 * required, not shared by calls that may run concurrently. Other arguments,
 * limits and errors as mxfp4_moe_route. */
size_t mxfp4_moe_route_workspace_size(int T, int topk, int E);
int mxfp4_moe_route_ws(const int32_t* topk_ids, int T, int topk, int E,
                       int32_t* expert_count, int32_t* expert_offset, int32_t* route_list,
                       int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/* Router: the step before routing ("MXFP4 MoE decode kernels", Design, "Routing
 * inside the kernel" takes its top-k ids; the workload shapes fix the
 * scoring). Per token t:
 *   x_e = fp32(logits[t][e] + bias[e])   (bias may be NULL: x_e = logits[t][e];
 *                                          a NaN x ranks as -inf)
 *   topk_ids[t][0..k-1]  the k largest x in descending order, ties to the
 *                        lower expert index (sigmoid is increasing, so this is
 *                        also the top-k by sigmoid score)
 *   topk_weights[t][j]   scoring 0 ("softmax_topk"): exp(x_j - x_0) / sum over
 *                        the chosen; scoring 1 ("sigmoid_renorm"): sigmoid(x_j)
 *                        / sum of the chosen sigmoids; fp32
 *   logits fp32 [T, E], bias fp32 [E] or NULL, topk_ids int32 [T, k],
 *   topk_weights fp32 [T, k]: device pointers owned by the caller, 4-byte
 *   aligned (MXFP4_MOE_ERR_ALIGN). Limits: 1 <= E <= 1024, 1 <= k <= min(32, E),
 *   0 <= T (MXFP4_MOE_ERR_SHAPE); scoring 0 or 1 and non-NULL logits/outputs
 *   (MXFP4_MOE_ERR_ARG). T == 0 enqueues nothing. The outputs feed
 *   mxfp4_moe_forward directly. */
int mxfp4_moe_router(const float* logits, const float* bias, int T, int E, int topk, int scoring,
                     int32_t* topk_ids, float* topk_weights, void* stream);

/* Router with grouped top-k and a choice of what the bias moves ("GLM-5.2 and
 * GLM-5.3 (744B) in MXFP4 on Gaudi 2", Why it needed a port, item 4, names
 * grouped top-k without defining it). As mxfp4_moe_router, plus:
 *   n_group       the E experts form n_group equal groups of consecutive ids
 *                 (group of e = e / (E / n_group)); a group's score is its
 *                 largest x; only the topk_group highest-scoring groups (ties
 *                 to the lower group index) stay eligible, and the k largest x
 *                 among their experts are chosen as above. n_group = 1 is the
 *                 plain router.
 *   bias_in_weights  1: the weights use x (the bias moves selection and
 *                 weights, as mxfp4_moe_router); 0: the bias steers the
 *                 choice only, the weights use the chosen experts' unbiased
 *                 logits (a NaN logit as -inf); softmax over the chosen then
 *                 subtracts their largest value.
 * Limits (MXFP4_MOE_ERR_SHAPE): those of mxfp4_moe_router, 1 <= n_group <= 32,
 * E % n_group == 0, 1 <= topk_group <= n_group, k <= topk_group * E / n_group;
 * bias_in_weights 0 or 1 (MXFP4_MOE_ERR_ARG). */
int mxfp4_moe_router_grouped(const float* logits, const float* bias, int T, int E, int topk,
                             int scoring, int n_group, int topk_group, int bias_in_weights,
                             int32_t* topk_ids, float* topk_weights, void* stream);

/* The MoE layer, y = sum_j w_tj * W2[e] silu(W_gate[e] x) * (W_up[e] x).
 *   hidden        bf16  [T, K]
 *   topk_ids      int32 [T, topk]   (negative = padding, >= E = invalid, both skipped)
 *   topk_weights  fp32  [T, topk]
 *   w13/s13/w2/s2 packed weights and scales, layouts in the file header
 *   out           bf16  [T, K]      written completely (zero for tokens with no valid route)
 *   status        int32 [4]         may be NULL
 *   workspace     device scratch of at least mxfp4_moe_workspace_size(T,K,I,E,topk)
 *                 bytes, zero before first use (see above); not shared by
 *                 calls that may run concurrently
 *   path          0 = automatic (decode for T <= 32, else prefill),
 *                 1 = decode kernels, 2 = prefill (tensor-core grouped GEMM)
 * T == 0 returns MXFP4_MOE_OK and enqueues nothing. */
int mxfp4_moe_forward(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                      const uint8_t* w13, const uint8_t* s13,
                      const uint8_t* w2, const uint8_t* s2,
                      int T, int K, int I, int E, int topk,
                      void* out, int32_t* status,
                      void* workspace, size_t workspace_bytes,
                      int path, void* stream);

/* The layer over an expert-parallel window, optionally per route ("MXFP4 MoE
 * decode kernels", Design, "Routing inside the kernel": routes to experts on
 * other expert-parallel ranks are skipped and cost nothing; Beyond gpt-oss:
 * mxk_w2xr, a per-route w2 output for models that apply a per-route operation
 * before the token sum).
 *   w13/s13/w2/s2 hold the E local experts, global ids expert_base ..
 *                 expert_base + E - 1 (expert_base >= 0); a route whose id lies
 *                 outside that window is skipped silently (no status count)
 *   per_route 0   out bf16 [T, K]: y_t = sum over the window's routes of
 *                 w_tj * W2[e] h (this rank's part of the token sums)
 *   per_route 1   out bf16 [T * topk, K]: row t * topk + j = W2[e] h of route
 *                 (t, j), unweighted (topk_weights may be NULL), zero rows for
 *                 skipped routes
 * Everything else (paths, limits, alignment, workspace, errors) as
 * mxfp4_moe_forward; path, per_route or expert_base out of range give
 * MXFP4_MOE_ERR_ARG. */
int mxfp4_moe_forward_window(const void* hidden, const int32_t* topk_ids,
                             const float* topk_weights,
                             const uint8_t* w13, const uint8_t* s13,
                             const uint8_t* w2, const uint8_t* s2,
                             int T, int K, int I, int E, int topk,
                             int expert_base, int per_route,
                             void* out, int32_t* status,
                             void* workspace, size_t workspace_bytes,
                             int path, void* stream);

/* The gpt-oss form of the layer ("MXFP4 MoE decode kernels", Design, "Read
 * the served layout" and "Fused epilogues"):
 *   y_t = sum_j w_tj * (W2[e] h + b2[e]),  h = SwiGLU-OAI(W_gate[e] x + b_gate[e],
 *                                                     W_up[e] x + b_up[e])
 *   SwiGLU-OAI(g, u) = min(g, 7) * sigmoid(1.702 min(g, 7)) * (clamp(u, -7, 7) + 1)
 * with h rounded once to bf16 between the projections and all sums in fp32.
 *   w13 / s13     uint8 [E, 2I, K/2] / [E, 2I, K/32] with the gate and up rows
 *                 INTERLEAVED: row 2i is gate row i, row 2i + 1 is up row i
 *   b13           fp32  [E, 2I] in the same (interleaved) row order
 *   w2 / s2       as for mxfp4_moe_forward
 *   b2            fp32  [E, K]; each route adds its expert's b2 before the
 *                 routing weight, so a token gets sum_j w_tj * b2[e_tj]
 * Other arguments, paths (decode for T <= 32, else the tensor-core prefill),
 * limits and errors as mxfp4_moe_forward. b13 and b2 are device pointers, 4-byte
 * aligned (MXFP4_MOE_ERR_ALIGN), non-NULL (MXFP4_MOE_ERR_ARG); the caller owns
 * every buffer. NaN in a pre-activation stays NaN (the cap and clamp do not
 * replace it). */
int mxfp4_moe_forward_oai(const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                          const uint8_t* w13, const uint8_t* s13, const float* b13,
                          const uint8_t* w2, const uint8_t* s2, const float* b2,
                          int T, int K, int I, int E, int topk,
                          void* out, int32_t* status,
                          void* workspace, size_t workspace_bytes,
                          int path, void* stream);

/* The forward call for callers that cannot allocate device memory. The pages
 * have no counterpart of this entry point: it is a convenience of this
 * library. Some callers may not call cudaMalloc at all -- code that runs under
 * a host framework that owns every device allocation (a plugin interface that
 * hands out no scratch space), latency-critical serving loops that must never
 * synchronise the device (cudaMalloc and cudaFree can), or pipelines that fix
 * their memory footprint before they start. This variant takes the same
 * arguments as mxfp4_moe_forward without the workspace, and uses instead a
 * fixed device array of MXFP4_MOE_NOALLOC_BYTES bytes compiled into the
 * library: every GPU that loads the library holds that array until the
 * process exits. Nothing is allocated by this call (no cudaMalloc, cudaFree or
 * allocating library routine).
 *  - Sizes whose mxfp4_moe_workspace_size(T, K, I, E, topk) exceeds
 *    MXFP4_MOE_NOALLOC_BYTES are rejected with MXFP4_MOE_ERR_WORKSPACE (the
 *    decode path of the four workload shapes fits up to T = 32).
 *  - The first call on a device performs the set-up for that device: it looks
 *    up the array's device address, which makes the CUDA driver load this part
 *    of the library and place the array on that device (a one-time driver
 *    allocation that may synchronise), and clears the array's bookkeeping part
 *    on `stream`. Make that first call in set-up code, before any stream
 *    capture and before any loop that must not synchronise; the promise that
 *    nothing is allocated holds for every later call.
 *  - The library leaves the array's bookkeeping part zero after every call,
 *    also after one whose bounded wait gave up (status[2] != 0), so the array
 *    never needs clearing by the caller (who could not reach it anyway).
 *  - All calls share the one array, and it keeps the last call's contents:
 *    calls whose work may overlap on the GPU (different streams without
 *    ordering) race on it; issue them on one stream or order them. */
#define MXFP4_MOE_NOALLOC_BYTES (16u * 1024u * 1024u)
int mxfp4_moe_forward_noalloc(const void* hidden, const int32_t* topk_ids,
                              const float* topk_weights,
                              const uint8_t* w13, const uint8_t* s13,
                              const uint8_t* w2, const uint8_t* s2,
                              int T, int K, int I, int E, int topk,
                              void* out, int32_t* status, int path, void* stream);

/* MXFP4 encoder ("GLM-5.2 and GLM-5.3 (744B) in MXFP4 on Gaudi 2", What was
 * built, "MXFP4 encoder"): bf16 rows -> the packed form the forward calls read.
 *   x       bf16  [rows, cols], cols % 32 == 0 (MXFP4_MOE_ERR_SHAPE), 16-byte aligned
 *   packed  uint8 [rows, cols/2]  value 2i in the low nibble of byte i, 4-byte aligned
 *   scale   uint8 [rows, cols/32] E8M0
 *   rule    0 = OCP: per 32-value block X = floor(log2(amax)) - 2;
 *           1 = Quark: the same, raised by one when amax / 2^X >= 7
 * X is clamped to [-127, 127] (an all-zero block gets byte 0); a block with a
 * NaN or infinite value gets byte 255 and codes 0. Each element v / 2^X is
 * rounded to the nearest E2M1 value, ties to the even code, saturating at 6,
 * keeping its sign (-0 stays -0). Device pointers owned by the caller;
 * rows == 0 enqueues nothing. */
int mxfp4_moe_encode(const void* x, int rows, int cols, int rule, uint8_t* packed,
                     uint8_t* scale, void* stream);

/* Dequantise packed rows to bf16 ("MXFP4 MoE decode kernels", Prefill:
 * mxk_deq unpacks an expert's MXFP4 weights straight to bf16).
 *   packed uint8 [rows, cols/2], scale uint8 [rows, cols/32] -> out bf16 [rows, cols]
 * Each value is E2M1(nibble) * 2^(s - 127) rounded once to bf16, which is
 * exact except that products beyond the bf16 range become +-inf and the
 * scale byte 255 gives NaN. cols % 32 == 0 (MXFP4_MOE_ERR_SHAPE); packed
 * 16-byte and out 4-byte aligned (MXFP4_MOE_ERR_ALIGN). Uses the decode
 * kernels' conversion (form 1 of mxfp4_moe_dequant_form). */
int mxfp4_moe_dequant(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                      void* out, void* stream);

/* The same dequantisation through the conversion of one path of the layer,
 * so that a bit-exact check pins the weights each path computes with:
 *   form 1  the decode kernels': hardware E2M1 -> f16 (exact), then an exact
 *           fp32 multiply by 2^(s - 127), rounded once to bf16;
 *   form 2  the prefill GEMM's operand A: the E2M1 fields placed in a bf16
 *           bit pattern (magnitude x 2^-126), then exact bf16 multiplies by
 *           2^(s - 1), or by 2^126 and 2^(s - 127) for bytes above 128 --
 *           the same device routine that feeds the GEMM's tensor memory.
 * Both give the value stated for mxfp4_moe_dequant, bit for bit; form
 * outside {1, 2} gives MXFP4_MOE_ERR_ARG; other rules as mxfp4_moe_dequant. */
int mxfp4_moe_dequant_form(const uint8_t* packed, const uint8_t* scale, int rows, int cols,
                           int form, void* out, void* stream);

/* Profiling hook: when events (host array of n cudaEvent_t handles, n >= 2)
 * is non-NULL, each later forward call on this process records events[0]
 * before its first kernel and events[i] after its i-th kernel (while i < n),
 * on its stream; the decode path runs 1 kernel (one cooperative launch), the
 * prefill path 5 (the first two events bracket route + gather). Pass NULL to
 * turn it off.
 * Not thread-safe; meant for benchmarks. */
void mxfp4_moe_set_phase_events(void* const* events, int n);

/* Test only: from the next forward call on, the decode kernel's CTA `cta`
 * does not arrive at the grid barrier between its two phases, so every
 * bounded wait on that barrier (in all CTAs) runs out and the call reports it
 * in status[2] and status[3] instead of computing the output; a negative cta
 * turns this off (the default). It exists so tests can exercise the failure
 * reporting without faulting or hanging a GPU. Not thread-safe. */
void mxfp4_moe_test_skip_grid_arrival(int cta);

/* Test only: the warps per CTA of the decode kernel form that a decode call of
 * this shape and T would run on a device with max_smem bytes of opt-in shared
 * memory per block: 12, 11 or 10 (every warp a consumer), 7 (7 consumer warps
 * and a producer warp), or 0 when no form fits. The form is the one the call's
 * own T needs, except that every T of a layer shape runs the form of its
 * largest decode T when that is a 10- to 12-warp form. Host only; no device
 * is touched. -1 for shapes the decode path does not take (T outside 1..32,
 * T * topk > 1024, K or I not a multiple of 64, E or topk out of range). */
int mxfp4_moe_test_decode_form(int T, int K, int I, int E, int topk, int max_smem);

/* Static description of an error code (never NULL). */
const char* mxfp4_moe_strerror(int code);

/* Library ABI version: 100 * major + minor. */
int mxfp4_moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_MOE_H_ */
