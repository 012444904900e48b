// Tensor-core (tcgen05 / TMEM / TMA) attention kernels for sm_103a.
#pragma once

#include "common.cuh"

namespace gbattn {

// True when this build carries the tensor-core forward / backward kernels.
bool tc_fwd_available();
bool tc_bwd_available();

// bf16, head_dim 128.  Persistent kernels: one CTA per SM takes units from
// p.unit_counter over the cost-ordered work list p.units (forward and dQ pass:
// 256 query rows per unit; backward: 128 keys per unit).
cudaError_t launch_tc_fwd(const KParams& p, int sms, cudaStream_t st);
// with_dq: also add dQ into p.dq_accum (L2 reductions, order not fixed);
// otherwise dK and dV only.
cudaError_t launch_tc_bwd(const KParams& p, int sms, cudaStream_t st, bool with_dq);
// Head dim 256: each 128-key unit taken twice (tickets 2u and 2u + 1 of
// p.unit_counter), once per half of the head dim; dQ added into p.dq_accum.
cudaError_t launch_tc_bwd256(const KParams& p, int sms, cudaStream_t st);
// Query-stationary dQ (fixed summation order) straight to p.dq as bf16; needs
// p.delta from the preprocess and the forward's work list.
cudaError_t launch_tc_dq(const KParams& p, int sms, cudaStream_t st);

}  // namespace gbattn
