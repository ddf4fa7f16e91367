// Placeholder translation unit for the tcgen05 prefill kernel.
#include <cuda_runtime.h>

#include "kernels.h"

namespace pkv {

cudaError_t launch_paged_prefill(const PrefillArgs&, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace pkv
