// Tensor-core paged decode attention (placeholder: not yet selected).
#include "swa_internal.h"

namespace swa {
bool mma_decode_supported(const Ctx &, int) { return false; }
size_t mma_decode_ws_bytes(const Ctx &, int, int64_t, int) { return 0; }
cudaError_t launch_attn_decode_mma(Ctx &, const AttnArgs &, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace swa
