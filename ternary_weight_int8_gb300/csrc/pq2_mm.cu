// pq2_mm.cu — prefill (M >= 16) ternary x INT8 matmul on tcgen05 tensor
// cores (sm_103a).
#include "pq2_device.cuh"
#include "pq2_internal.h"

namespace pq2 {

int launch_mm(const uint16_t*, const float*, const uint8_t*, const uint16_t*, void*, int,
              int32_t*, int64_t, int64_t, int64_t, int, int32_t*, cudaStream_t) {
  return PQ2_ERR_LAUNCH;
}

}  // namespace pq2
