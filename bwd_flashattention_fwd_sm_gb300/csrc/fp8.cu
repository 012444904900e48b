// Per-tile e4m3 quantisation of Q, K and V for the FP8 forward.
//
// Newer accelerators multiply 8-bit floats so that every transfer and every
// matrix instruction handles more numbers, while sums stay in a wider format
// (smzdm contest article, closing section on precision).  Each 128-row tile of
// one head gets its own scale: amax = max |x| over the tile, scale = amax / 448,
// code = e4m3(x * (448 / amax)) with the division and the product rounded to
// float32 and the conversion rounding to nearest even, saturating at 448.
//
// Outputs (contiguous):
//   Q codes [B, Hq, S, 128], K codes [B, Hkv, S, 128] (one 128-byte row per position),
//   V codes transposed, [B, Hkv, 128, ld] with ld = S rounded up to 16: the P V
//   product then reads V with the keys along each 128-byte row, the same
//   K-major operand layout as K in Q K^T;
//   scales [B, H, ceil(S / 128)] float32 for each of the three.
// The kernel is bound by device-memory bandwidth: 2 bytes read and 1 written per
// element.  One CTA per (tensor, batch, head, tile).
#include <cuda_bf16.h>

#include "common.cuh"
#include "fp8.h"
#include "ptx.cuh"

namespace gbattn {

namespace {

constexpr int kThreads = 256;

struct QuantArgs {
  Fp8QuantJob job[3];
  int seqlen, n_tiles, ld_t;
  long long first_block[4];  // job j owns blocks [first_block[j], first_block[j + 1])
};

__device__ __forceinline__ float absmax8(const uint4& u, float m) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
  }
  return m;
}

// bf16 element e (0-7) of a 16-byte vector, as float32.
__device__ __forceinline__ float elem(const uint4& u, int e) {
  const uint32_t w = e < 2 ? u.x : e < 4 ? u.y : e < 6 ? u.z : u.w;
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

__global__ void __launch_bounds__(kThreads) k_quant_fp8(const __grid_constant__ QuantArgs a) {
  // transposed codes of one V tile: row d holds 128 keys; its eight 16-byte
  // chunks are permuted by (d / 8) % 8 so that the column writes spread over banks
  __shared__ __align__(16) uint32_t tr[128][32];
  __shared__ float red[kThreads / 32];

  long long blk = blockIdx.x;
  const int j = blk >= a.first_block[2] ? 2 : blk >= a.first_block[1] ? 1 : 0;
  blk -= a.first_block[j];
  const Fp8QuantJob& J = a.job[j];
  const int t = (int)(blk % a.n_tiles);
  const long long bh = blk / a.n_tiles;
  const int h = (int)(bh % J.heads);
  const int b = (int)(bh / J.heads);
  const int r0 = t * 128;
  const int rows = min(128, a.seqlen - r0);
  const __nv_bfloat16* src = J.src + (long long)b * J.sb + (long long)h * J.sh + (long long)r0 * J.ss;
  const int tid = threadIdx.x;

  uint4 x[8];
  float m = 0.f;
  if (!J.transpose) {
    // vector c = tid + 256 i: row c / 16, columns 8 (c % 16) .. + 7
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = tid + i * kThreads, r = c >> 4, col = (c & 15) * 8;
      x[i] = r < rows ? *reinterpret_cast<const uint4*>(src + (long long)r * J.ss + col) : make_uint4(0, 0, 0, 0);
      m = absmax8(x[i], m);
    }
  } else {
    // item c = tid + 256 i (i < 2): keys 4 (c / 16) .. + 3, columns 8 (c % 16) .. + 7
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + i * kThreads, kg = c >> 4, col = (c & 15) * 8;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = kg * 4 + e;
        x[i * 4 + e] =
            r < rows ? *reinterpret_cast<const uint4*>(src + (long long)r * J.ss + col) : make_uint4(0, 0, 0, 0);
        m = absmax8(x[i * 4 + e], m);
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  float amax = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  if (tid == 0) J.scale[bh * a.n_tiles + t] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;

  if (!J.transpose) {
    uint8_t* dst = J.dst + (bh * a.seqlen + r0) * 128;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = tid + i * kThreads, r = c >> 4, col = (c & 15) * 8;
      if (r < rows) {
        uint2 w;
        w.x = ptx::pack_e4m3x4(__fmul_rn(elem(x[i], 0), inv), __fmul_rn(elem(x[i], 1), inv),
                               __fmul_rn(elem(x[i], 2), inv), __fmul_rn(elem(x[i], 3), inv));
        w.y = ptx::pack_e4m3x4(__fmul_rn(elem(x[i], 4), inv), __fmul_rn(elem(x[i], 5), inv),
                               __fmul_rn(elem(x[i], 6), inv), __fmul_rn(elem(x[i], 7), inv));
        *reinterpret_cast<uint2*>(dst + (long long)r * 128 + col) = w;
      }
    }
    return;
  }
  // transposed: word (d, keys 4 kg .. 4 kg + 3) at row d, chunk (kg / 4) ^ ((d / 8) % 8)
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = tid + i * kThreads, kg = c >> 4, col = (c & 15) * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int d = col + e;
      const uint32_t w = ptx::pack_e4m3x4(__fmul_rn(elem(x[i * 4 + 0], e), inv), __fmul_rn(elem(x[i * 4 + 1], e), inv),
                                          __fmul_rn(elem(x[i * 4 + 2], e), inv), __fmul_rn(elem(x[i * 4 + 3], e), inv));
      tr[d][(((kg >> 2) ^ ((d >> 3) & 7)) << 2) | (kg & 3)] = w;
    }
  }
  __syncthreads();
  uint8_t* dst = J.dst + bh * 128 * (long long)a.ld_t + r0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = tid + i * kThreads, d = c >> 3, ch = c & 7;
    if (r0 + ch * 16 < a.seqlen) {
      const uint4 v = *reinterpret_cast<const uint4*>(&tr[d][(ch ^ ((d >> 3) & 7)) << 2]);
      *reinterpret_cast<uint4*>(dst + (long long)d * a.ld_t + ch * 16) = v;
    }
  }
}

}  // namespace

cudaError_t launch_quant_fp8(const Fp8QuantJob (&jobs)[3], int batch, int seqlen, int ld_t, cudaStream_t st) {
  QuantArgs a;
  a.seqlen = seqlen;
  a.n_tiles = (seqlen + 127) / 128;
  a.ld_t = ld_t;
  a.first_block[0] = 0;
  for (int j = 0; j < 3; ++j) {
    a.job[j] = jobs[j];
    a.first_block[j + 1] = a.first_block[j] + (long long)batch * jobs[j].heads * a.n_tiles;
  }
  const long long blocks = a.first_block[3];
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  k_quant_fp8<<<(unsigned)blocks, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbattn
