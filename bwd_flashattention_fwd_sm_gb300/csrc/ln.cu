// Fused residual add + LayerNorm (lpqz.cn CUDA tutorial, sections 5.1-5.3):
// one pass over HBM per row, statistics merged in registers.
//
// A CTA of 256 threads normalises one row at a time (grid-stride over rows).
// Long rows (more than two 16-byte vectors per thread) that are whole vectors
// at aligned addresses stream through a ring of shared-memory stages filled by
// bulk copies, several rows ahead; other rows are loaded straight into
// registers, every load of the row issued before any is used.  Each thread holds its
// 16-byte vectors of the row in registers (8 bf16 or 4 float32 elements each),
// adds the residual, and summarises every vector
// as (count, mean, M2) computed from its registers.  Summaries are merged with
// the parallel form of Welford's update - n = na + nb, d = mb - ma,
// mean = ma + d nb / n, M2 = M2a + M2b + d^2 na nb / n - first within the
// thread, then across the warp with shuffles, then across the eight warps
// through shared memory (the reduction scheme of the tutorial's section 5.2).
// The row is then normalised from the registers it is already in, so x and
// the residual are read once and y (and h) written once: the bytes moved set
// the time (section 5.1 on arithmetic intensity below 1).  When every thread
// holds the same number of whole vectors, all merges join equal counts and run
// without the division.  rstd uses the IEEE square root and division, once per
// row, not the approximate reciprocal square root the tutorial warns against
// for LayerNorm (section 4).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/gbln.h"
#include "common.cuh"
#include "ptx.cuh"

#include <algorithm>

namespace gbattn {
void set_last_error_text(const char* text);
attn_status_t device_status(int** status, int* sms, unsigned long long* wait_ns);
}

namespace gbattn {

namespace {

constexpr int kThreadsLn = 256;

struct Stats {
  float n, mean, m2;
};

__device__ __forceinline__ Stats merge(Stats a, Stats b) {
  const float n = a.n + b.n;
  if (n == 0.f) return a;
  const float d = b.mean - a.mean;
  const float wb = b.n / n;
  Stats r;
  r.n = n;
  r.mean = a.mean + d * wb;
  r.m2 = a.m2 + b.m2 + d * d * a.n * wb;
  return r;
}

// merge() for two summaries of equal counts, where n_b / n is exactly 1/2: the
// same update without the division.  Rows that every thread covers with the
// same number of whole vectors merge only equal counts (in a tree within the
// thread, then across lanes and warps), and the divisions' latency was a
// fifth of the row's time on [16384, 4096] bf16.
__device__ __forceinline__ Stats merge_eq(Stats a, Stats b) {
  const float d = b.mean - a.mean;
  Stats r;
  r.n = a.n + b.n;
  r.mean = a.mean + d * 0.5f;
  r.m2 = a.m2 + b.m2 + d * d * a.n * 0.5f;
  return r;
}

// The (count, mean, M2) summary of one whole vector of E values.
template <int E>
__device__ __forceinline__ Stats vec_stats(const float (&v)[E]) {
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) sum += v[e];
  const float m = sum * (1.f / E);
  float q = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) q += (v[e] - m) * (v[e] - m);
  return Stats{(float)E, m, q};
}

// Summaries of all threads merged into warp_stats (lane 0 of each warp), then
// by warp 0 into row_stats and the row's rstd; `eq`: every summary has the
// same count.  Leaves row_stats / row_rstd valid after its second barrier.
__device__ __forceinline__ void block_stats(Stats st, bool eq, int lane, int warp, float cols, float eps,
                                            Stats* warp_stats, Stats& row_stats, float& row_rstd, float* mean_out,
                                            float* rstd_out) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Stats o;
    o.n = __shfl_xor_sync(0xffffffffu, st.n, off);
    o.mean = __shfl_xor_sync(0xffffffffu, st.mean, off);
    o.m2 = __shfl_xor_sync(0xffffffffu, st.m2, off);
    st = eq ? merge_eq(st, o) : merge(st, o);
  }
  if (lane == 0) warp_stats[warp] = st;
  __syncthreads();
  if (warp == 0) {
    // lanes 8.. hold empty summaries; the xor offsets below 8 keep them apart
    Stats w = lane < kThreadsLn / 32 ? warp_stats[lane] : Stats{0.f, 0.f, 0.f};
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {
      Stats o;
      o.n = __shfl_xor_sync(0xffffffffu, w.n, off);
      o.mean = __shfl_xor_sync(0xffffffffu, w.mean, off);
      o.m2 = __shfl_xor_sync(0xffffffffu, w.m2, off);
      w = eq ? merge_eq(w, o) : merge(w, o);
    }
    if (lane == 0) {
      row_stats = w;
      row_rstd = 1.f / sqrtf(w.m2 / cols + eps);
      if (mean_out) *mean_out = w.mean;
      if (rstd_out) *rstd_out = row_rstd;
    }
  }
  __syncthreads();
}

template <class T>
struct Vec;  // one 16-byte vector of T
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) { unpack(*reinterpret_cast<const uint4*>(p), v); }
  __device__ static void unpack(const uint4& u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};
template <>
struct Vec<float> {
  static constexpr int E = 4;
  __device__ static void load(const float* p, float (&v)[4]) { unpack(*reinterpret_cast<const uint4*>(p), v); }
  __device__ static void unpack(const uint4& u, float (&v)[4]) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y); v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __device__ static float load1(const float* p) { return *p; }
  __device__ static void store1(float* p, float v) { *p = v; }
};

struct LnArgs {
  ln_params_t p;
  const void* x;
  const void* r;
  const float* gamma;
  const float* beta;
  void* y;
  void* h;
  float* mean;
  float* rstd;
  int vec;  // every pointer (gamma, beta included) 16-byte aligned and every stride a whole number of vectors
};

// gamma and beta of columns c0 .. c0 + E - 1 (1 and 0 when absent), as float4
// loads when the vector is whole and a.vec says gamma and beta are 16-byte
// aligned (c0 is a multiple of E, so gamma + c0 then is too).
template <int E>
__device__ __forceinline__ void affine(const LnArgs& a, int64_t c0, int64_t cols, float (&g)[E], float (&b)[E]) {
  if (a.vec && c0 + E <= cols) {
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 gv = a.gamma ? __ldg(reinterpret_cast<const float4*>(a.gamma + c0 + e)) : make_float4(1.f, 1.f, 1.f, 1.f);
      const float4 bv = a.beta ? __ldg(reinterpret_cast<const float4*>(a.beta + c0 + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
      g[e] = gv.x; g[e + 1] = gv.y; g[e + 2] = gv.z; g[e + 3] = gv.w;
      b[e] = bv.x; b[e + 1] = bv.y; b[e + 2] = bv.z; b[e + 3] = bv.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int64_t c = c0 + e < cols ? c0 + e : cols - 1;
      g[e] = a.gamma ? __ldg(a.gamma + c) : 1.f;
      b[e] = a.beta ? __ldg(a.beta + c) : 0.f;
    }
  }
}

// kVpt: 16-byte vectors per thread (cols <= 256 * kVpt * E).  Short rows leave
// registers to spare: several CTAs per SM then keep more loads in flight.
template <class T, int kVpt>
__global__ void __launch_bounds__(kThreadsLn, kVpt >= 8 ? 1 : (kVpt >= 4 ? 2 : 4)) k_ln_residual(const LnArgs a) {
  constexpr int E = Vec<T>::E;
  __shared__ Stats warp_stats[kThreadsLn / 32];
  __shared__ Stats row_stats;
  __shared__ float row_rstd;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t cols = a.p.cols;
  const int64_t nvec = (cols + E - 1) / E;
  const bool ragged = cols % E != 0 || !a.vec;  // element loads where vectors do not fit
  // every thread holds kVpt whole vectors: summaries of equal counts throughout
  const bool uniform = !ragged && nvec == (int64_t)kThreadsLn * kVpt;
  const T* X = static_cast<const T*>(a.x);
  const T* R = static_cast<const T*>(a.r);
  T* Y = static_cast<T*>(a.y);
  T* H = static_cast<T*>(a.h);
  for (int64_t row = blockIdx.x; row < a.p.rows; row += gridDim.x) {
    const T* xr = X + row * a.p.x_stride;
    const T* rr = R ? R + row * a.p.r_stride : nullptr;
    float v[kVpt][E];
    Stats st{0.f, 0.f, 0.f};
    Stats sv[kVpt];
    // whole vectors: every load of the row issued first, as raw 16-byte words
    // (widened only afterwards, so they are all in flight at once)
    uint4 ux[kVpt], ur[kVpt];
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
      const int64_t vi = tid + (int64_t)j * kThreadsLn;
      const int64_t c0 = vi * E;
      ux[j] = ur[j] = make_uint4(0u, 0u, 0u, 0u);
      if (vi < nvec && (!ragged || (a.vec && c0 + E <= cols))) {
        ux[j] = *reinterpret_cast<const uint4*>(xr + c0);
        if (rr) ur[j] = *reinterpret_cast<const uint4*>(rr + c0);
      }
    }
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
      const int64_t vi = tid + (int64_t)j * kThreadsLn;
      const int64_t c0 = vi * E;
      int cnt = 0;
      sv[j] = Stats{0.f, 0.f, 0.f};
      if (vi < nvec) {
        if (!ragged || (a.vec && c0 + E <= cols)) {
          Vec<T>::unpack(ux[j], v[j]);
          if (rr) {
            float t[E];
            Vec<T>::unpack(ur[j], t);
#pragma unroll
            for (int e = 0; e < E; ++e) v[j][e] += t[e];
          }
          cnt = E;
          if (uniform) {
            sv[j] = vec_stats<E>(v[j]);
            continue;
          }
        } else {  // the row's last, partial vector
#pragma unroll
          for (int e = 0; e < E; ++e) {
            v[j][e] = 0.f;
            if (c0 + e < cols) {
              v[j][e] = Vec<T>::load1(xr + c0 + e) + (rr ? Vec<T>::load1(rr + c0 + e) : 0.f);
              ++cnt;
            }
          }
        }
      }
      if (cnt > 0) {  // this vector's (count, mean, M2) from its registers
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) s += (e < cnt) ? v[j][e] : 0.f;
        const float m = s / (float)cnt;
        float q = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float d = v[j][e] - m;
          q += (e < cnt) ? d * d : 0.f;
        }
        st = merge(st, Stats{(float)cnt, m, q});
      }
    }
    if (uniform) {  // the thread's vectors in a tree of equal counts
#pragma unroll
      for (int w = 1; w < kVpt; w <<= 1)
#pragma unroll
        for (int j = 0; j + w < kVpt; j += 2 * w) sv[j] = merge_eq(sv[j], sv[j + w]);
      st = sv[0];
    }
    // warp, then block
    block_stats(st, uniform, lane, warp, (float)cols, a.p.eps, warp_stats, row_stats, row_rstd,
                a.mean ? a.mean + row : nullptr, a.rstd ? a.rstd + row : nullptr);
    const float mu = row_stats.mean;
    const float rs = row_rstd;
    T* yr = Y + row * a.p.y_stride;
    T* hr = H ? H + row * a.p.h_stride : nullptr;
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
      const int64_t vi = tid + (int64_t)j * kThreadsLn;
      const int64_t c0 = vi * E;
      if (vi >= nvec) continue;
      float o[E], g[E], b[E];
      affine<E>(a, c0, cols, g, b);
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = (v[j][e] - mu) * rs * g[e] + b[e];
      if (!ragged || (a.vec && c0 + E <= cols)) {
        Vec<T>::store(yr + c0, o);
        if (hr) Vec<T>::store(hr + c0, v[j]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (c0 + e < cols) {
            Vec<T>::store1(yr + c0 + e, o[e]);
            if (hr) Vec<T>::store1(hr + c0 + e, v[j][e]);
          }
      }
    }
    __syncthreads();  // row_stats / warp_stats are rewritten for the next row
  }
}

// Persistent grid: as many CTAs as fit on the SMs at once (at most one per row).
template <class T, int kVpt>
cudaError_t launch_ln_v(const LnArgs& a, int sms, cudaStream_t st) {
  int per_sm = 1;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ln_residual<T, kVpt>, kThreadsLn, 0);
  if (e != cudaSuccess) return e;
  const int64_t want = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  const int grid = (int)(a.p.rows < want ? a.p.rows : want);
  k_ln_residual<T, kVpt><<<grid, kThreadsLn, 0, st>>>(a);
  return cudaGetLastError();
}

// Whole rows through a ring of shared-memory stages filled by bulk copies:
// thread 0 keeps `stages` rows of x (and the residual) in flight per CTA while
// the CTA works on the oldest, so HBM always has loads outstanding.  Used when
// rows are whole 16-byte vectors at 16-byte aligned addresses.  The wait on a
// stage is bounded: a CTA that gives up records ATTN_ERR_DEVICE_TIMEOUT, waits
// (bounded) for its own copies and returns.
constexpr int kMaxStages = 8;
// CTAs per SM the ring kernel is built for: several CTAs, each with a short
// ring, beat one CTA with a deep ring (measured on [16384, 4096] bf16: four CTAs
// x 3 stages 4.7 TB/s, three x 4 4.5, two x 6 3.7, one x 12 2.3), because a
// CTA's barriers and stores serialise its rows.
template <int kVpt>
constexpr int ring_ctas() { return kVpt <= 2 ? 4 : (kVpt == 4 ? 2 : 1); }

template <class T, int kVpt>
__global__ void __launch_bounds__(kThreadsLn, ring_ctas<kVpt>()) k_ln_ring(const LnArgs a, int stages, uint32_t row_bytes,
                                                           int* status, unsigned long long wait_ns) {
  constexpr int E = Vec<T>::E;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ Stats warp_stats[kThreadsLn / 32];
  __shared__ Stats row_stats;
  __shared__ float row_rstd;
  __shared__ ptx::Abort abort;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t cols = a.p.cols, nvec = cols / E;
  const bool uniform = nvec == (int64_t)kThreadsLn * kVpt;  // equal summary counts throughout
  const bool has_r = a.r != nullptr;
  const uint32_t stage_bytes = row_bytes * (has_r ? 2 : 1);
  const char* X = static_cast<const char*>(a.x);
  const char* R = static_cast<const char*>(a.r);
  const int64_t xs = a.p.x_stride * (int64_t)sizeof(T), rs_ = a.p.r_stride * (int64_t)sizeof(T);
  auto issue = [&](int s, int64_t row) {  // thread 0 only
    uint8_t* dst = ring + (size_t)s * stage_bytes;
    ptx::mbar_arrive_expect_tx(&full[s], stage_bytes);
    ptx::bulk_load(dst, X + row * xs, row_bytes, &full[s]);
    if (has_r) ptx::bulk_load(dst + row_bytes, R + row * rs_, row_bytes, &full[s]);
  };
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) ptx::mbar_init(&full[s], 1);
    abort.flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < stages; ++s) {
      const int64_t row = blockIdx.x + (int64_t)s * gridDim.x;
      if (row < a.p.rows) issue(s, row);
    }
  T* Y = static_cast<T*>(a.y);
  T* H = static_cast<T*>(a.h);
  int64_t it = 0;
  bool ok = true;
  for (int64_t row = blockIdx.x; row < a.p.rows; row += gridDim.x, ++it) {
    const int s = (int)(it % stages);
    const uint32_t ph = (uint32_t)((it / stages) & 1);
    // a thread whose wait gives up reads whatever the stage holds; the
    // block-wide agreement below stops everyone before anything is stored
    const bool mine = ptx::mbar_wait(&full[s], ph, &abort, status, wait_ns);
    const uint8_t* xsm = ring + (size_t)s * stage_bytes;
    float v[kVpt][E];
    Stats st{0.f, 0.f, 0.f};
    Stats sv[kVpt];
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
      const int64_t vi = tid + (int64_t)j * kThreadsLn;
      sv[j] = Stats{0.f, 0.f, 0.f};
      if (vi < nvec) {
        Vec<T>::load(reinterpret_cast<const T*>(xsm) + vi * E, v[j]);
        if (has_r) {
          float t[E];
          Vec<T>::load(reinterpret_cast<const T*>(xsm + row_bytes) + vi * E, t);
#pragma unroll
          for (int e = 0; e < E; ++e) v[j][e] += t[e];
        }
        sv[j] = vec_stats<E>(v[j]);
        if (!uniform) st = merge(st, sv[j]);
      }
    }
    if (uniform) {  // the thread's vectors in a tree of equal counts
#pragma unroll
      for (int w = 1; w < kVpt; w <<= 1)
#pragma unroll
        for (int j = 0; j + w < kVpt; j += 2 * w) sv[j] = merge_eq(sv[j], sv[j + w]);
      st = sv[0];
    }
    // every thread has read stage s (and agrees on the wait): refill the stage
    // with the row `stages` iterations ahead at once (refilling after the
    // reduction instead measured 30% slower)
    if (__syncthreads_or(!mine)) { ok = false; break; }
    if (tid == 0) {
      const int64_t next = row + (int64_t)stages * gridDim.x;
      if (next < a.p.rows) issue(s, next);
    }
    block_stats(st, uniform, lane, warp, (float)cols, a.p.eps, warp_stats, row_stats, row_rstd,
                a.mean ? a.mean + row : nullptr, a.rstd ? a.rstd + row : nullptr);
    const float mu = row_stats.mean;
    const float r_s = row_rstd;
    T* yr = Y + row * a.p.y_stride;
    T* hr = H ? H + row * a.p.h_stride : nullptr;
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
      const int64_t vi = tid + (int64_t)j * kThreadsLn;
      if (vi >= nvec) continue;
      const int64_t c0 = vi * E;
      float o[E], g[E], b[E];
      affine<E>(a, c0, cols, g, b);
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = (v[j][e] - mu) * r_s * g[e] + b[e];
      Vec<T>::store(yr + c0, o);
      if (hr) Vec<T>::store(hr + c0, v[j]);
    }
    // row_stats / warp_stats are rewritten for the next row only after this
    // barrier (the next iteration's first barrier comes before any rewrite)
  }
  if (!ok && tid == 0) {
    // copies this CTA issued and did not consume: wait (bounded) for them
    ptx::Abort none;
    none.flag = 0;
    for (int64_t j = it; j < it + stages; ++j) {
      const int64_t row = blockIdx.x + j * gridDim.x;
      if (row >= a.p.rows) break;
      ptx::mbar_wait(&full[j % stages], (uint32_t)((j / stages) & 1), &none, status, wait_ns);
    }
  }
}

template <class T>
cudaError_t launch_ln(const LnArgs& a, int sms, int* status, unsigned long long wait_ns, cudaStream_t st) {
  constexpr int E = Vec<T>::E;
  const int64_t per = (a.p.cols + (int64_t)kThreadsLn * E - 1) / ((int64_t)kThreadsLn * E);
  const uint32_t row_bytes = (uint32_t)(a.p.cols * (int64_t)sizeof(T));
  const uint32_t stage_bytes = row_bytes * (a.r ? 2 : 1);
  // ring: whole vectors, aligned rows; 192 KB of stages per SM split over the
  // CTAs the kernel is built for
  const int ctas = per <= 2 ? ring_ctas<2>() : (per <= 4 ? ring_ctas<4>() : ring_ctas<8>());
  const int stages = (int)std::min<int64_t>(kMaxStages, (192 * 1024 / ctas) / stage_bytes);
  // the ring for rows of more than two vectors per thread; shorter rows (4096
  // bf16 or 2048 float32 columns and below) go through registers: on [16384,
  // 4096] bf16 the register path with its loads issued first and division-free
  // statistics measured 5.03-5.08 TB/s against 4.66-4.75 for the ring
  if (a.vec && a.p.cols % E == 0 && stages >= 2 && per > 2 && per <= 8) {
    auto launch = [&](auto kernel) -> cudaError_t {
      const size_t smem = (size_t)stages * stage_bytes;
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      int per_sm = 1;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreadsLn, smem);
      if (e != cudaSuccess) return e;
      const int64_t want = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
      const int grid = (int)(a.p.rows < want ? a.p.rows : want);
      kernel<<<grid, kThreadsLn, smem, st>>>(a, stages, row_bytes, status, wait_ns);
      return cudaGetLastError();
    };
    if (per <= 1) return launch(k_ln_ring<T, 1>);
    if (per <= 2) return launch(k_ln_ring<T, 2>);
    if (per <= 4) return launch(k_ln_ring<T, 4>);
    return launch(k_ln_ring<T, 8>);
  }
  if (per <= 1) return launch_ln_v<T, 1>(a, sms, st);
  if (per <= 2) return launch_ln_v<T, 2>(a, sms, st);
  if (per <= 4) return launch_ln_v<T, 4>(a, sms, st);
  if (per <= 8) return launch_ln_v<T, 8>(a, sms, st);
  if (per <= 16) return launch_ln_v<T, 16>(a, sms, st);
  return cudaErrorInvalidValue;
}

attn_status_t ln_fail(attn_status_t s, const char* msg) {
  set_last_error_text(msg);
  return s;
}

}  // namespace

}  // namespace gbattn

extern "C" attn_status_t ln_residual_fwd(const ln_params_t* p, const void* x, const void* residual,
                                         const float* gamma, const float* beta, void* y, void* h, float* mean,
                                         float* rstd, void* stream) {
  using namespace gbattn;
  if (!p) return ln_fail(ATTN_ERR_INVALID_ARG, "ln_residual_fwd: params is NULL");
  if (p->dtype != ATTN_BF16 && p->dtype != ATTN_F32)
    return ln_fail(ATTN_ERR_INVALID_ARG, "ln_residual_fwd: dtype is not ATTN_F32 or ATTN_BF16");
  if (p->rows < 0 || p->cols < 1) return ln_fail(ATTN_ERR_INVALID_ARG, "ln_residual_fwd: rows < 0 or cols < 1");
  if (p->cols > 16384) return ln_fail(ATTN_ERR_UNSUPPORTED, "ln_residual_fwd: cols above 16384");
  if (!(p->eps >= 0.f)) return ln_fail(ATTN_ERR_INVALID_ARG, "ln_residual_fwd: eps must be >= 0");
  const int64_t esize = p->dtype == ATTN_BF16 ? 2 : 4, per_vec = 16 / esize;
  auto bad_stride = [&](int64_t s, bool used) { return used && s < p->cols; };
  if (bad_stride(p->x_stride, true) || bad_stride(p->y_stride, true) || bad_stride(p->r_stride, residual != nullptr) ||
      bad_stride(p->h_stride, h != nullptr))
    return ln_fail(ATTN_ERR_INVALID_ARG, "ln_residual_fwd: a row stride is below cols");
  if (p->rows == 0) return ATTN_OK;
  if (!x || !y) return ln_fail(ATTN_ERR_INVALID_ARG, "ln_residual_fwd: x or y is NULL");
  auto off = [](const void* q, uintptr_t m) { return (reinterpret_cast<uintptr_t>(q) & m) != 0; };
  const uintptr_t em = (uintptr_t)esize - 1;
  if (off(x, em) || off(y, em) || off(residual, em) || off(h, em) || off(gamma, 3) || off(beta, 3) ||
      off(mean, 3) || off(rstd, 3))
    return ln_fail(ATTN_ERR_INVALID_ARG, "ln_residual_fwd: a pointer is not aligned to its element size");
  auto strided = [&](int64_t s, bool used) { return !used || s % per_vec == 0; };
  const bool vec = !off(x, 15) && !off(y, 15) && !off(residual, 15) && !off(h, 15) && !off(gamma, 15) &&
                   !off(beta, 15) && strided(p->x_stride, true) &&
                   strided(p->y_stride, true) && strided(p->r_stride, residual != nullptr) &&
                   strided(p->h_stride, h != nullptr);
  int* status = nullptr;
  int sms = 0;
  unsigned long long wait_ns = 0;
  attn_status_t ds = device_status(&status, &sms, &wait_ns);
  if (ds != ATTN_OK) return ds;
  LnArgs a{*p, x, residual, gamma, beta, y, h, mean, rstd, vec ? 1 : 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = p->dtype == ATTN_BF16 ? launch_ln<__nv_bfloat16>(a, sms, status, wait_ns, st)
                                        : launch_ln<float>(a, sms, status, wait_ns, st);
  if (e != cudaSuccess) return ln_fail(ATTN_ERR_CUDA, "ln_residual_fwd: launch failed");
  return ATTN_OK;
}
