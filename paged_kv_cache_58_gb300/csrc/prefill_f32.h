// CUDA-core prefill for fp32 pools (paged_prefill_f32.cu).
#pragma once

#include <cuda_runtime.h>

#include "kernels.h"

namespace pkv {

// Same arguments and result as launch_paged_prefill (cascade mode unsupported); K/V
// stay fp32 end to end.
cudaError_t launch_paged_prefill_f32(const PrefillArgs& a, int group, cudaStream_t stream);

}  // namespace pkv
