#include "prefill.h"

namespace mxmoe {

size_t prefill_counter_bytes(int, int, int, int, int) { return 256; }

cudaError_t launch_prefill(const PrefillArgs&, cudaStream_t, void* const*, int) {
  return cudaErrorNotSupported;
}

}  // namespace mxmoe
