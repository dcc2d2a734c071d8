// tcgen05 + TMA kernel of the linear / Titans scan (not available yet: every
// shape is reported as unsupported so the dispatcher uses the CUDA-core kernel).
#include "kernels.h"

namespace ttm {
bool linear_tc_supported(const LinearArgs&) { return false; }
cudaError_t linear_tc_launch(const LinearArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace ttm
