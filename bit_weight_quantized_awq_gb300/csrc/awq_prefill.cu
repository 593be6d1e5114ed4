// awq_prefill.cu -- prefill path (large M). Not built yet: reports unsupported.
#include "awq_internal.h"
namespace awq {
bool prefill_supported(int64_t, int64_t, int64_t, int64_t) { return false; }
cudaError_t launch_prefill(const Problem &, cudaStream_t) { return cudaErrorNotSupported; }
} // namespace awq
