// prefill.cu — tiled causal prefill (placeholder until the tcgen05 kernels land).
#include <cuda_runtime.h>

#include "internal.h"

namespace kascade {
cudaError_t launch_prefill_dense(const PrefillArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_prefill_lse(const PrefillArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_prefill_anchor_main(const PrefillArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_prefill_reuse(const PrefillArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kascade
