// Sparse MLA on tcgen05 tensor cores (placeholder until the kernel lands).
#include "kernels.h"

namespace dsi {

bool tc_mla_supported(int) { return false; }

cudaError_t launch_sparse_mla_tc(const bf16*, const CacheView&, const int32_t*, int, int, int, int,
                                 int64_t, float, bf16*, float*, void*, size_t, int*,
                                 cudaStream_t) {
  return cudaErrorInvalidValue;
}

}  // namespace dsi
