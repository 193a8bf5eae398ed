// Tensor-core chunked prefill (tcgen05 + TMA + TMEM).  Not enabled yet: every call takes the
// token-serial kernel.
#include "gdn_internal.cuh"

namespace gdn {

bool tc_prefill_eligible(int, int, int, int, int, int) { return false; }
size_t tc_prefill_workspace_bytes(int, int, int, int, bool) { return 0; }
cudaError_t launch_tc_prefill(const PrefillArgs&, void**, int) { return cudaErrorNotSupported; }

}  // namespace gdn
