// kda_prefill.cu -- chunked KDA prefill (filled in below).
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
bool prefill_supported(int, int, int, int) { return false; }
size_t prefill_workspace_bytes(int, int, int, int, int64_t, int) { return 0; }
int launch_prefill(const PrefillArgs &, int, int, cudaStream_t) { return KDA_ERR_UNSUPPORTED_SHAPE; }
}  // namespace kda
