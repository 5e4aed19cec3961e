// tcgen05 backward scan (placeholder until the tensor-core backward lands).
#include "internal.h"

namespace m2rnn {
bool tc_backward_supported(int, int) { return false; }
int tc_backward_parts(int, int) { return 1; }
size_t tc_backward_scratch_bytes(int, int, int, int, int) { return 0; }
cudaError_t launch_tc_backward(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace m2rnn
