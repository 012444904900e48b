// Memory-bound pieces of the backward pass.
//
//  * preprocess: D_i = <dO_i, O_i> in float32 for every query row, and a zeroed
//    float32 dQ accumulator.  With P recomputed block by block (smzdm contest
//    article, section 03: the forward drops the attention matrix, so the backward
//    recomputes it per block), sum_j P_ij dP_ij = <dO_i, O_i> gives the softmax
//    Jacobian's row term without a second pass over the keys.
//  * dQ conversion: dQ = scale * accumulator, rounded to the output type.  dQ is
//    the gradient whose accumulation runs against the key-block loop, so every key
//    tile adds into it (same section: "many cores accumulate into the same place").
//
// Both are pure streaming kernels: one warp per row, 128-bit or 64-bit loads per
// lane, a grid sized in multiples of the SM count.
#include "common.cuh"
#include "ptx.cuh"

namespace gbattn {

namespace {

// Loads N contiguous elements of T starting at ptr (N * sizeof(T) in {4, 8, 16} bytes).
template <class T, int N>
__device__ __forceinline__ void load_vec(const T* ptr, float (&out)[N]) {
  constexpr int kBytes = N * (int)sizeof(T);
  static_assert(kBytes == 4 || kBytes == 8 || kBytes == 16, "vector width");
  union {
    uint4 u4;
    uint2 u2[2];
    unsigned u1[4];
    T t[N];
  } buf;
  if constexpr (kBytes == 16) buf.u4 = __ldg(reinterpret_cast<const uint4*>(ptr));
  else if constexpr (kBytes == 8) buf.u2[0] = __ldg(reinterpret_cast<const uint2*>(ptr));
  else buf.u1[0] = __ldg(reinterpret_cast<const unsigned*>(ptr));
#pragma unroll
  for (int i = 0; i < N; ++i) out[i] = to_f32(buf.t[i]);
}

template <class T, int N>
__device__ __forceinline__ void store_vec(T* ptr, const float (&in)[N]) {
  constexpr int kBytes = N * (int)sizeof(T);
  union {
    uint4 u4;
    uint2 u2[2];
    unsigned u1[4];
    T t[N];
  } buf;
#pragma unroll
  for (int i = 0; i < N; ++i) buf.t[i] = from_f32<T>(in[i]);
  if constexpr (kBytes == 16) *reinterpret_cast<uint4*>(ptr) = buf.u4;
  else if constexpr (kBytes == 8) *reinterpret_cast<uint2*>(ptr) = buf.u2[0];
  else *reinterpret_cast<unsigned*>(ptr) = buf.u1[0];
}

struct RowRef {
  long long q;      // element offset in q-like tensors
  long long lse;    // index into lse / delta
  long long acc;    // element offset in the dQ accumulator
};

// Flat row r (over all positions of all sequences and all query heads) to offsets.
__device__ __forceinline__ RowRef row_ref(const KParams& p, long long r) {
  RowRef x;
  const int H = p.heads_q;
  if (p.varlen) {
    const long long tok = r / H;
    const int h = (int)(r - tok * H);
    x.q = tok * p.q_ss + (long long)h * p.q_sh;
    x.lse = (long long)h * p.total_tokens + tok;
    x.acc = (tok * H + h) * (long long)p.head_dim;
  } else {
    const long long S = p.seqlen;
    const long long bh = r / S;
    const long long pos = r - bh * S;
    const int b = (int)(bh / H), h = (int)(bh % H);
    x.q = (long long)b * p.q_sb + (long long)h * p.q_sh + pos * p.q_ss;
    x.lse = r;
    x.acc = r * (long long)p.head_dim;
  }
  return x;
}

template <class T, int D>
__global__ void __launch_bounds__(256) k_bwd_preprocess(KParams p, long long n_rows) {
  constexpr int N = D / 32;
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const T* o = static_cast<const T*>(p.o);
  const T* dO = static_cast<const T*>(p.dout);
  for (long long r = warp0; r < n_rows; r += nwarps) {
    const RowRef x = row_ref(p, r);
    float a[N], b[N];
    load_vec<T, N>(o + x.q + lane * N, a);
    load_vec<T, N>(dO + x.q + lane * N, b);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) s = fmaf(a[i], b[i], s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) p.delta[x.lse] = s;
    if (p.dq_accum) {  // no accumulator in the deterministic (query-stationary dQ) mode
      float z[N];
#pragma unroll
      for (int i = 0; i < N; ++i) z[i] = 0.f;
      store_vec<float, N>(p.dq_accum + x.acc + lane * N, z);
    }
  }
}

template <class T, int D>
__global__ void __launch_bounds__(256) k_dq_convert(KParams p, long long n_rows) {
  constexpr int N = D / 32;
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  T* dq = static_cast<T*>(p.dq);
  for (long long r = warp0; r < n_rows; r += nwarps) {
    const RowRef x = row_ref(p, r);
    float a[N];
    const float4* src = reinterpret_cast<const float4*>(p.dq_accum + x.acc + lane * N);
    if constexpr (N == 4) {
      float4 f = __ldcs(src);
      a[0] = f.x; a[1] = f.y; a[2] = f.z; a[3] = f.w;
    } else {
      float2 f = __ldcs(reinterpret_cast<const float2*>(src));
      a[0] = f.x; a[1] = f.y;
    }
#pragma unroll
    for (int i = 0; i < N; ++i) a[i] *= p.scale;
    store_vec<T, N>(dq + x.q + lane * N, a);
  }
}

long long total_rows(const KParams& p) {
  if (p.varlen) return p.total_tokens * p.heads_q;
  return (long long)p.batch * p.heads_q * p.seqlen;
}

int grid_for(long long rows) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long want = (rows + 7) / 8;  // 8 warps per block
  long long cap = (long long)sms * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const KParams& p, bool bf16, cudaStream_t st) {
  const long long rows = total_rows(p);
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows);
  if (bf16) {
    if (p.head_dim == 128) k_bwd_preprocess<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(p, rows);
    else k_bwd_preprocess<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(p, rows);
  } else {
    if (p.head_dim == 128) k_bwd_preprocess<float, 128><<<grid, 256, 0, st>>>(p, rows);
    else k_bwd_preprocess<float, 64><<<grid, 256, 0, st>>>(p, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const KParams& p, bool bf16, cudaStream_t st) {
  const long long rows = total_rows(p);
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows);
  if (bf16) {
    if (p.head_dim == 128) k_dq_convert<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(p, rows);
    else k_dq_convert<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(p, rows);
  } else {
    if (p.head_dim == 128) k_dq_convert<float, 128><<<grid, 256, 0, st>>>(p, rows);
    else k_dq_convert<float, 64><<<grid, 256, 0, st>>>(p, rows);
  }
  return cudaGetLastError();
}

namespace {

__global__ void k_wait_probe(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ ptx::Abort abort;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);  // one arrival completes it; none comes
    abort.flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::mbar_wait(&bar, 0, &abort, status, limit_ns);
  __syncwarp();
}

}  // namespace

cudaError_t launch_wait_probe(int* status, unsigned long long limit_ns, cudaStream_t st) {
  k_wait_probe<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace gbattn
