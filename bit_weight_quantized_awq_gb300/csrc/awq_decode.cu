// awq_decode.cu -- decode path (small M). Not built yet: reports unsupported.
#include "awq_internal.h"
namespace awq {
bool decode_supported(int64_t, int64_t, int64_t, int64_t) { return false; }
cudaError_t launch_decode(const Problem &, cudaStream_t) { return cudaErrorNotSupported; }
} // namespace awq
