// The tcgen05 attention kernel is not built yet: report it unavailable.
#include "tc.h"

namespace csa {
bool tc_index_available() { return true; }
bool tc_attn_available() { return false; }
int tc_attn_split_len() { return 128; }
size_t tc_workspace_bytes(int, int, int64_t, int) { return 0; }
cudaError_t tc_sparse_attn(int, const AttnParams&, void*, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace csa
