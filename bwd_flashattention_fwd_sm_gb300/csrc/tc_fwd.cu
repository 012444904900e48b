#include "tc_kernels.h"
namespace gbattn {
bool tc_available() { return false; }
cudaError_t launch_tc_fwd(const KParams&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd(const KParams&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gbattn
