// FP8 (e4m3) forward: quantisation and the tensor-core forward on 8-bit operands.
// Internal to the library (the public interface is include/gbattn.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace gbattn {

// One tensor to quantise: bf16 source [B, heads, S, 128] by element strides,
// codes at dst (row-major, or transposed when `transpose`), one float32 scale per
// (batch, head, 128-row tile) at scale.
struct Fp8QuantJob {
  const __nv_bfloat16* src;
  long long sb, sh, ss;
  uint8_t* dst;
  float* scale;
  int heads;
  int transpose;
};

// Quantises the three jobs (Q, K, V) in one launch; ld_t is the row length in
// bytes of transposed outputs (S rounded up to 16).
cudaError_t launch_quant_fp8(const Fp8QuantJob (&jobs)[3], int batch, int seqlen, int ld_t, cudaStream_t st);

// Inputs of the FP8 forward: codes and per-tile scales as launch_quant_fp8 writes them.
struct Fp8Operands {
  const uint8_t* q8;   // [B, Hq, S, 128]
  const uint8_t* k8;   // [B, Hkv, S, 128]
  const uint8_t* v8t;  // [B, Hkv, 128, ld_t]
  const float* qs;     // [B, Hq, n_tiles]
  const float* ks;     // [B, Hkv, n_tiles]
  const float* vs;     // [B, Hkv, n_tiles]
  int ld_t;
};

// Forward on the tensor cores with e4m3 Q K^T and P V products (head_dim 128,
// fixed length); O and LSE as for launch_tc_fwd.
cudaError_t launch_tc_fwd_fp8(const KParams& p, int sms, cudaStream_t st, const Fp8Operands& f);

}  // namespace gbattn
