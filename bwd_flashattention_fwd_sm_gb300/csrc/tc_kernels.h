// Tensor-core (tcgen05 / TMEM / TMA) attention kernels for sm_103a.
#pragma once

#include "common.cuh"

namespace gbattn {

// True when this build carries the tensor-core forward / backward kernels.
bool tc_fwd_available();
bool tc_bwd_available();

// bf16, head_dim 128.  Persistent kernels: one CTA per SM takes units from
// p.unit_counter over the cost-ordered work list p.units (forward: 256 query
// rows per unit; backward: 128 keys per unit).
cudaError_t launch_tc_fwd(const KParams& p, int sms, cudaStream_t st);
cudaError_t launch_tc_bwd(const KParams& p, int sms, cudaStream_t st);

}  // namespace gbattn
