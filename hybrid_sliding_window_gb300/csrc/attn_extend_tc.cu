// tcgen05 chunked-prefill attention (placeholder: not yet selected).
#include "swa_internal.h"

namespace swa {
bool tc_extend_supported(const Ctx &, int) { return false; }
size_t tc_extend_ws_bytes(const Ctx &, int, int64_t, int) { return 0; }
cudaError_t launch_attn_extend_tc(Ctx &, const AttnArgs &, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace swa
