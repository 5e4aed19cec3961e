// Entry points of a tensor-core backward for V = 128, not built: they report
// "not supported", so the dispatcher runs the V = 128 backward on the fp32
// SIMT kernel (simt.cu).  The V = 64 and V = 16 backwards are the warp-MMA
// kernels (mma_backward.cu, mv_backward.cu).
#include "internal.h"

namespace m2rnn {
bool tc_backward_supported(int, int) { return false; }
int tc_backward_parts(int, int) { return 1; }
size_t tc_backward_scratch_bytes(int, int, int, int, int) { return 0; }
cudaError_t launch_tc_backward(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace m2rnn
