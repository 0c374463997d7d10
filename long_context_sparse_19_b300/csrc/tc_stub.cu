// Placeholder until the tcgen05 kernels land: reports the tensor-core path as unavailable.
#include "tc.h"

namespace csa {
bool tc_enabled() { return false; }
int tc_attn_split_len() { return 128; }
size_t tc_workspace_bytes(int, int, int64_t, int) { return 0; }
cudaError_t tc_index_scores(int, int, const int64_t*, const void*, const float*, const void*, int64_t, int,
                            const RopeTab&, float*, void*, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t tc_sparse_attn(int, const AttnParams&, void*, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace csa
