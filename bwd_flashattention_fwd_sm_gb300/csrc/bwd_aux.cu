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
// Both are pure streaming kernels: a warp takes a batch of rows at a time
// (16-byte loads and stores per lane, all loads issued before use), a grid
// sized in multiples of the SM count.
#include "common.cuh"
#include "ptx.cuh"

namespace gbattn {

namespace {

// Loads N contiguous elements of T starting at ptr (N * sizeof(T) in {4, 8, 16} bytes) into out[0, N).
template <class T, int N>
__device__ __forceinline__ void load_vec(const T* ptr, float* out) {
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
__device__ __forceinline__ void store_vec(T* ptr, const float* in) {
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
  bool ok;          // checked builds: the row's batch entry, head and position lie in the tensors
};

// Flat row r (over all positions of all sequences and all query heads) to offsets.
// The divisions run in 32 bits (rows, heads and lengths all fit; the host caps
// problems well below 2^31 rows).
__device__ __forceinline__ RowRef row_ref(const KParams& p, long long r) {
  RowRef x;
  const unsigned H = (unsigned)p.heads_q, ur = (unsigned)r;
  if (p.varlen) {
    const unsigned tok = ur / H;
    const int h = (int)(ur - tok * H);
    x.q = (long long)tok * p.q_ss + (long long)h * p.q_sh;
    x.lse = (long long)h * p.total_tokens + tok;
    x.acc = r * (long long)p.head_dim;
    x.ok = bounds_ok(!GBATTN_CHECKED || row_in_range(1, 1, p.seqlen, p.total_tokens, p.heads_q, 0, h, 0, tok),
                     p.status);
  } else {
    const unsigned S = (unsigned)p.seqlen;
    const unsigned bh = ur / S;
    const long long pos = (long long)(ur - bh * S);
    const int b = (int)(bh / H), h = (int)(bh - (bh / H) * H);
    x.q = (long long)b * p.q_sb + (long long)h * p.q_sh + pos * p.q_ss;
    x.lse = r;
    x.acc = r * (long long)p.head_dim;
    x.ok = bounds_ok(!GBATTN_CHECKED || row_in_range(0, p.batch, p.seqlen, 0, p.heads_q, b, h, 0, pos), p.status);
  }
  return x;
}

// Rows a warp is given at least (grid sizing); each kernel takes its own batch
// per iteration, all loads issued before use, so HBM sees tens of KB in flight
// per SM.
constexpr int kRows = 4;

// Preprocess with 16-byte loads: L = min(32, D / E) lanes cover one row, each
// with NV vectors of E elements (16 bytes), so one load instruction covers
// 32 / L rows; a warp takes kPreRows rows per iteration, all loads issued
// before use.
constexpr int kPreRows = 8;

// Dot product of two 16-byte vectors of T, added to s.
template <class T>
__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, float s) {
  constexpr int N = 16 / (int)sizeof(T);
  union U {
    uint4 u;
    T t[N];
  };
  U ua, ub;
  ua.u = a;
  ub.u = b;
#pragma unroll
  for (int i = 0; i < N; ++i) s = fmaf(to_f32(ua.t[i]), to_f32(ub.t[i]), s);
  return s;
}

template <class T, int D>
__global__ void __launch_bounds__(256) k_bwd_preprocess(KParams p, long long n_rows) {
  constexpr int E0 = 16 / (int)sizeof(T);  // elements per 16-byte load
  constexpr int L = D / E0 < 32 ? D / E0 : 32;  // lanes per row
  constexpr int E = D / L;                 // elements per lane (E / E0 loads)
  constexpr int RP = 32 / L;               // rows per load instruction
  constexpr int NL = kPreRows / RP;        // load instructions per tensor per iteration
  static_assert(L <= 32 && 32 % L == 0 && kPreRows % RP == 0 && E % E0 == 0, "row geometry");
  const int lane = threadIdx.x & 31;
  const int sub = lane % L, part = lane / L;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const T* o = static_cast<const T*>(p.o);
  const T* dO = static_cast<const T*>(p.dout);
  for (long long r0 = warp0 * kPreRows; r0 < n_rows; r0 += nwarps * kPreRows) {
    // raw 16-byte vectors, widened only in the dot product: the loads of a whole
    // iteration stay in flight in few registers (widened on load, the bf16
    // head-dim-128 kernel took 86 registers, two blocks per SM, and ran at 62%
    // of the copy bandwidth)
    uint4 a[NL][E / E0], b[NL][E / E0];
    RowRef x[NL];
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const long long r = r0 + j * RP + part;
      x[j].ok = false;
      if (r < n_rows && (x[j] = row_ref(p, r)).ok) {
#pragma unroll
        for (int v = 0; v < E / E0; ++v) {
          a[j][v] = __ldg(reinterpret_cast<const uint4*>(o + x[j].q + (sub + v * L) * E0));
          b[j][v] = __ldg(reinterpret_cast<const uint4*>(dO + x[j].q + (sub + v * L) * E0));
        }
      } else {
#pragma unroll
        for (int v = 0; v < E / E0; ++v) a[j][v] = b[j][v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const long long r = r0 + j * RP + part;
      float s = 0.f;
#pragma unroll
      for (int v = 0; v < E / E0; ++v) s = dot16<T>(a[j][v], b[j][v], s);
#pragma unroll
      for (int off = L / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (sub == 0 && r < n_rows && x[j].ok) p.delta[x[j].lse] = s;
    }
    if (p.dq_accum) {  // no accumulator in the deterministic (query-stationary dQ) mode
      // zero the rows' float32 accumulator: LZ lanes of 16 bytes per row, NZ stores each
      constexpr int LZ = D / 4 < 32 ? D / 4 : 32, NZ = D / 4 / LZ, RZ = 32 / LZ;
      const int subz = lane % LZ, partz = lane / LZ;
#pragma unroll
      for (int j = 0; j < kPreRows / RZ; ++j) {
        const long long r = r0 + j * RZ + partz;
        // the accumulator is contiguous over flat rows: row r starts at r * D
        if (r < n_rows) {
#pragma unroll
          for (int z = 0; z < NZ; ++z)
            *reinterpret_cast<float4*>(p.dq_accum + r * D + (subz + z * LZ) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
}

// dQ conversion with 16-byte stores: a lane converts E = 16 / sizeof(T)
// consecutive elements (E float32 read as E / 4 16-byte loads), L = D / E
// lanes per row; a warp takes kCvtRows rows per iteration.
constexpr int kCvtRows = 8;

template <class T, int D>
__global__ void __launch_bounds__(256) k_dq_convert(KParams p, long long n_rows) {
  constexpr int E0 = 16 / (int)sizeof(T);
  constexpr int L = D / E0 < 32 ? D / E0 : 32, E = D / L, RP = 32 / L, NL = kCvtRows / RP;
  static_assert(L <= 32 && 32 % L == 0 && kCvtRows % RP == 0 && E % E0 == 0 && E0 % 4 == 0, "row geometry");
  const int lane = threadIdx.x & 31;
  const int sub = lane % L, part = lane / L;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  T* dq = static_cast<T*>(p.dq);
  for (long long r0 = warp0 * kCvtRows; r0 < n_rows; r0 += nwarps * kCvtRows) {
    float a[NL][E];
    RowRef x[NL];
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const long long r = r0 + j * RP + part;
      x[j].ok = false;
      if (r < n_rows && (x[j] = row_ref(p, r)).ok) {
#pragma unroll
        for (int w = 0; w < E / E0; ++w) {
          const float4* src = reinterpret_cast<const float4*>(p.dq_accum + x[j].acc + (sub + w * L) * E0);
#pragma unroll
          for (int v = 0; v < E0 / 4; ++v) {
            const float4 f = __ldcs(src + v);
            float* d = a[j] + w * E0 + 4 * v;
            d[0] = f.x; d[1] = f.y; d[2] = f.z; d[3] = f.w;
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const long long r = r0 + j * RP + part;
      if (r >= n_rows || !x[j].ok) continue;
#pragma unroll
      for (int i = 0; i < E; ++i) a[j][i] *= p.scale;
#pragma unroll
      for (int w = 0; w < E / E0; ++w) store_vec<T, E0>(dq + x[j].q + (sub + w * L) * E0, a[j] + w * E0);
    }
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
  long long want = (rows + 8 * kRows - 1) / (8 * kRows);  // 8 warps per block, kRows (or more) rows per warp
  long long cap = (long long)sms * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

// Forward with a split key range: per row, the parts' unnormalised O_s, row
// max m_s and row sum l_s (log2 units) merge as M = max_s m_s,
// L = sum_s 2^(m_s - M) l_s, O = sum_s 2^(m_s - M) O_s / L, LSE = ln 2 (M + log2 L),
// the same correction the online softmax applies between key tiles (zwxr.cn
// CANN article, section 3.3).  One warp per row; a lane holds D / 32
// consecutive columns.  Bound by device memory: reads n_split (4 D + 8) bytes
// per row, writes 2 D + 4.
template <int D>
__global__ void __launch_bounds__(256) k_fwd_combine(KParams p, long long n_rows) {
  constexpr int NC = D / 32;
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int ns = p.n_split;
  __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o);
  for (long long r = warp0; r < n_rows; r += nwarps) {
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, p.part_ml[((long long)s * n_rows + r) * 2]);
    float L = 0.f, acc[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[c] = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + ((long long)s * n_rows + r) * 2);
      if (ml.x == -INFINITY) continue;
      const float w = exp2f(ml.x - M);
      L = fmaf(w, ml.y, L);
      float v[NC];
      load_vec<float, NC>(p.part_o + ((long long)s * n_rows + r) * D + lane * NC, v);
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = fmaf(w, v[c], acc[c]);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[c] *= inv;
    const RowRef x = row_ref(p, r);
    if (!x.ok) continue;
    store_vec<__nv_bfloat16, NC>(O + x.q + lane * NC, acc);
    if (lane == 0) p.lse[x.lse] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_fwd_combine(const KParams& p, cudaStream_t st) {
  const long long rows = total_rows(p);
  if (rows == 0 || p.n_split <= 1) return cudaSuccess;
  const int grid = grid_for(rows);
  if (p.head_dim == 128) k_fwd_combine<128><<<grid, 256, 0, st>>>(p, rows);
  else if (p.head_dim == 64) k_fwd_combine<64><<<grid, 256, 0, st>>>(p, rows);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const KParams& p, bool bf16, cudaStream_t st) {
  const long long rows = total_rows(p);
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows);
  if (bf16) {
    if (p.head_dim == 256) k_bwd_preprocess<__nv_bfloat16, 256><<<grid, 256, 0, st>>>(p, rows);
    else if (p.head_dim == 128) k_bwd_preprocess<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(p, rows);
    else k_bwd_preprocess<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(p, rows);
  } else {
    if (p.head_dim == 256) k_bwd_preprocess<float, 256><<<grid, 256, 0, st>>>(p, rows);
    else if (p.head_dim == 128) k_bwd_preprocess<float, 128><<<grid, 256, 0, st>>>(p, rows);
    else k_bwd_preprocess<float, 64><<<grid, 256, 0, st>>>(p, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const KParams& p, bool bf16, cudaStream_t st) {
  const long long rows = total_rows(p);
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows);
  if (bf16) {
    if (p.head_dim == 256) k_dq_convert<__nv_bfloat16, 256><<<grid, 256, 0, st>>>(p, rows);
    else if (p.head_dim == 128) k_dq_convert<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(p, rows);
    else k_dq_convert<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(p, rows);
  } else {
    if (p.head_dim == 256) k_dq_convert<float, 256><<<grid, 256, 0, st>>>(p, rows);
    else if (p.head_dim == 128) k_dq_convert<float, 128><<<grid, 256, 0, st>>>(p, rows);
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
