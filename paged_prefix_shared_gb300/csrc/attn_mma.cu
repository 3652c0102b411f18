// Tensor-core (tcgen05) attention tiles for prefill chunks, verify rows and
// wide shared-prefix groups.  Not built yet: the planner routes every task to
// the bandwidth kernel while this reports the path unavailable.
#include <cuda_runtime.h>

#include "pps_internal.h"

namespace pps {

bool mma_path_available() { return false; }

int launch_mma_attention(const Shape&, const DeviceTables&, int64_t, const void*, const pps_pool&,
                         void*, int32_t*, void*) {
  return (int)cudaErrorNotSupported;
}

}  // namespace pps
