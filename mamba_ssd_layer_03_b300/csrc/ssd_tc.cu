// Tensor-core (tcgen05) path of the SSD forward scan -- not built yet.
#include "ssd_internal.h"

namespace ssd {
size_t tc_workspace_bytes(const Problem &) { return 0; }
int tc_supported(const Problem &) { return SSD_ERR_UNSUPPORTED; }
cudaError_t tc_launch(const Problem &) { return cudaErrorNotSupported; }
}  // namespace ssd
