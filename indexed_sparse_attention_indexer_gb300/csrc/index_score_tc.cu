// Indexer scoring on tcgen05 tensor cores (placeholder until the kernel lands).
#include "kernels.h"

namespace dsi {

bool tc_score_supported(const CacheView&, int) { return false; }

cudaError_t launch_index_score_tc(const bf16*, const float*, const CacheView&, int, int, int64_t,
                                  float*, int64_t, int*, cudaStream_t) {
  return cudaErrorInvalidValue;
}

}  // namespace dsi
