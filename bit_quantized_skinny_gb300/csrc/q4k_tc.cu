// q4k_tc.cu — tensor-core (tcgen05) variant of the skinny Q4K x bf16 product.
// Not built yet: every shape is reported unsupported, so dispatch keeps the CUDA-core kernel.
#include "q4k_internal.h"

namespace q4k {

bool tc_supports(int, int64_t, int64_t) { return false; }

cudaError_t launch_tc(const Job*, int, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace q4k
