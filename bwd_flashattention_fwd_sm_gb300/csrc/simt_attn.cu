// Tiled fused attention in float32 arithmetic on the CUDA cores.
//
// This is the path for float32 inputs (true float32 FMA, no TF32), where the
// tensor-core path does not apply.  It follows the same tiling as the tensor-core
// kernels: the forward streams 64-key blocks past a 64-row query tile with the
// running max/sum correction (zwxr.cn CANN ops-nn fused-attention article,
// sections 3.2-3.3), so no score matrix is stored; the backward keeps a 64-key
// block of K and V on chip, gathers dK and dV along the query direction and adds
// each block's share of dQ into a float32 accumulator (smzdm contest article,
// section 03, on recomputation and the direction conflict between the three
// gradients).  Masked tiles are never visited.
#include "common.cuh"

namespace gbattn {

namespace {

constexpr int kRows = 64;     // query rows per forward unit; keys per backward unit
constexpr int kCols = 64;     // keys per forward step; query rows per backward step
constexpr int kThreads = 256;

template <class T>
__device__ __forceinline__ void load_row_f32(float* dst, const T* src, int D, bool valid, int lane,
                                             int nlanes) {
  for (int d = lane; d < D; d += nlanes) dst[d] = valid ? to_f32(src[d]) : 0.f;
}

// Key blocks visited by a forward unit, in order.
struct KeyBlocks {
  int n;        // number of blocks
  int e0;       // block mask: first CSR entry
  int mode;     // mask kind
  __device__ int get(const KParams& p, int i) const {
    if (mode != kMaskBlock) return i;
    const int c = p.col_idx[e0 + i];
    return check_block(p, c, p.n_col_blocks) ? c : INT_MAX / (2 * kCols);  // failed: past every sequence
  }
};

// ---------------------------------------------------------------------------
// Forward: one CTA per (sequence, query head, 64-row query tile).
// Warp w owns query rows 8w..8w+7 of the tile; lane handles keys lane and lane+32
// for the scores and head-dim columns lane + 32c for the output.
// ---------------------------------------------------------------------------
template <class T, int D>
__global__ void __launch_bounds__(kThreads) k_simt_fwd(KParams p) {
  constexpr int NC = D / 32;      // output columns per lane
  constexpr int KS = D + 1;       // padded K row stride (conflict-free column reads)
  extern __shared__ float smem[];
  float* Qs = smem;                       // [64][D]
  float* Ks = Qs + kRows * D;             // [64][D+1]
  float* Vs = Ks + kCols * KS;            // [64][D]
  float* Ps = Vs + kCols * D;             // [8 warps][8 rows][64]

  const Unit u = p.units[blockIdx.x];
  if (!check_unit(p, u, false, kRows)) return;
  const SeqInfo si = seq_info(p, u.seq);
  const int h = u.head, g = h / p.group;
  const int q0 = u.tile * kRows;
  if (q0 >= si.len) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* Q = static_cast<const T*>(p.q);
  const T* K = static_cast<const T*>(p.k);
  const T* V = static_cast<const T*>(p.v);

  for (int r = warp; r < kRows; r += kThreads / 32) {
    const bool ok = q0 + r < si.len && check_q_row(p, si, h, q0 + r);
    load_row_f32(Qs + r * D, Q + (ok ? q_off(p, si, h, q0 + r) : 0), D, ok, lane, 32);
  }

  KeyBlocks kb;
  kb.mode = p.mask;
  kb.e0 = 0;
  const int nkb_seq = (si.len + kCols - 1) / kCols;
  if (p.mask == kMaskNone) kb.n = nkb_seq;
  else if (p.mask == kMaskCausal) kb.n = (min(si.len, q0 + kRows) - 1) / kCols + 1;
  else {
    kb.e0 = p.row_ptr[u.tile];
    kb.n = p.row_ptr[u.tile + 1] - kb.e0;
  }
  const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);

  float m[8], l[8], acc[8][NC];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;
  }
  float* Pw = Ps + warp * 8 * kCols;

  for (int it = 0; it < kb.n; ++it) {
    const int blk = kb.get(p, it);
    const int k0 = blk * kCols;
    if (k0 >= si.len) continue;
    __syncthreads();  // previous block's K/V no longer in use
    for (int r = warp; r < kCols; r += kThreads / 32) {
      const bool ok = k0 + r < si.len && check_kv_row(p, si, g, k0 + r);
      const long long off = ok ? kv_off(p, si, g, k0 + r) : 0;
      for (int d = lane; d < D; d += 32) {
        Ks[r * KS + d] = ok ? to_f32(K[off + d]) : 0.f;
        Vs[r * D + d] = ok ? to_f32(V[off + d]) : 0.f;
      }
    }
    __syncthreads();

    // scores for this warp's 8 rows against keys lane, lane+32
    float s[8][2];
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r][0] = s[r][1] = 0.f;
    const float* q8 = Qs + (warp * 8) * D;
    for (int d = 0; d < D; ++d) {
      const float ka = Ks[lane * KS + d], kb2 = Ks[(lane + 32) * KS + d];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float qv = q8[r * D + d];
        s[r][0] = fmaf(qv, ka, s[r][0]);
        s[r][1] = fmaf(qv, kb2, s[r][1]);
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = q0 + warp * 8 + r;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = k0 + lane + 32 * c;
        bool keep = j < si.len;
        if (elem_causal) keep = keep && j <= i;
        s[r][c] = keep ? s[r][c] * p.scale_log2 : -INFINITY;
      }
      float mb = fmaxf(s[r][0], s[r][1]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float mn = fmaxf(m[r], mb);
      const float mu = mn == -INFINITY ? 0.f : mn;
      const float alpha = exp2f(m[r] - mu);
      const float p0 = exp2f(s[r][0] - mu), p1 = exp2f(s[r][1] - mu);
      float ps = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[r] = l[r] * alpha + ps;
      m[r] = mn;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[r][c] *= alpha;
      Pw[r * kCols + lane] = p0;
      Pw[r * kCols + lane + 32] = p1;
    }
    __syncwarp();
    for (int j = 0; j < kCols; ++j) {
      float vv[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) vv[c] = Vs[j * D + lane + 32 * c];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float pj = Pw[r * kCols + j];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[r][c] = fmaf(pj, vv[c], acc[r][c]);
      }
    }
    __syncwarp();
  }

  T* O = static_cast<T*>(p.o);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = q0 + warp * 8 + r;
    if (i >= si.len || !check_q_row(p, si, h, i)) continue;
    const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
    const long long off = q_off(p, si, h, i);
#pragma unroll
    for (int c = 0; c < NC; ++c) O[off + lane + 32 * c] = from_f32<T>(acc[r][c] * inv);
    if (lane == 0)
      p.lse[row_index(p, si, h, i)] =
          l[r] > 0.f ? (m[r] + log2f(l[r])) * 0.69314718055994530942f : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Backward: one CTA per (sequence, kv head, 64-key tile); loops over the group's
// query heads and the query blocks that see this key block.
// Thread (j = tid/4, part = tid%4) owns key row j and head-dim columns 4t + part.
// ---------------------------------------------------------------------------
template <class T, int D>
__global__ void __launch_bounds__(kThreads) k_simt_bwd(KParams p) {
  constexpr int NT = D / 4;
  constexpr int SS = kCols + 1;  // padded dS row stride
  extern __shared__ float smem[];
  float* Ks = smem;                 // [64][D]
  float* Qs = Ks + kRows * D;       // [64][D]
  float* dOs = Qs + kCols * D;      // [64][D]
  float* dSs = dOs + kCols * D;     // [64 q][65]
  float* lse2 = dSs + kCols * SS;   // [64]  lse * log2(e)
  float* dlt = lse2 + kCols;        // [64]

  const Unit u = p.units[blockIdx.x];
  if (!check_unit(p, u, true, kRows)) return;
  const SeqInfo si = seq_info(p, u.seq);
  const int g = u.head;
  const int k0 = u.tile * kRows;
  if (k0 >= si.len) return;
  const int tid = threadIdx.x, j = tid >> 2, part = tid & 3;
  const int warp = tid >> 5, lane = tid & 31;
  const T* Q = static_cast<const T*>(p.q);
  const T* K = static_cast<const T*>(p.k);
  const T* V = static_cast<const T*>(p.v);
  const T* dO = static_cast<const T*>(p.dout);

  const bool kvalid = k0 + j < si.len && check_kv_row(p, si, g, k0 + j);
  float kr[NT], vr[NT], dk[NT], dv[NT];
  {
    const long long off = kvalid ? kv_off(p, si, g, k0 + j) : 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      kr[t] = kvalid ? to_f32(K[off + 4 * t + part]) : 0.f;
      vr[t] = kvalid ? to_f32(V[off + 4 * t + part]) : 0.f;
      dk[t] = dv[t] = 0.f;
      Ks[j * D + 4 * t + part] = kr[t];
    }
  }

  const int nqb_seq = (si.len + kCols - 1) / kCols;
  const int kblk = u.tile;
  int qb_begin = 0, qb_count = nqb_seq, e0 = 0;
  if (p.mask == kMaskCausal) {
    qb_begin = kblk;
    qb_count = nqb_seq - kblk;
  } else if (p.mask == kMaskBlock) {
    e0 = p.csc_ptr[kblk];
    qb_count = p.csc_ptr[kblk + 1] - e0;
  }
  const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);

  for (int hh = 0; hh < p.group; ++hh) {
    const int h = g * p.group + hh;
    for (int it = 0; it < qb_count; ++it) {
      int qb = p.mask == kMaskBlock ? p.csc_idx[e0 + it] : qb_begin + it;
      if (p.mask == kMaskBlock && !check_block(p, qb, p.n_row_blocks)) qb = INT_MAX / (2 * kCols);
      const int q0 = qb * kCols;
      if (q0 >= si.len) continue;
      __syncthreads();  // previous step done with Qs, dOs, dSs
      for (int r = warp; r < kCols; r += kThreads / 32) {
        const bool ok = q0 + r < si.len && check_q_row(p, si, h, q0 + r);
        const long long off = ok ? q_off(p, si, h, q0 + r) : 0;
        for (int d = lane; d < D; d += 32) {
          Qs[r * D + d] = ok ? to_f32(Q[off + d]) : 0.f;
          dOs[r * D + d] = ok ? to_f32(dO[off + d]) : 0.f;
        }
      }
      if (tid < kCols) {
        const bool ok = q0 + tid < si.len && check_q_row(p, si, h, q0 + tid);
        const long long ri = ok ? row_index(p, si, h, q0 + tid) : 0;
        const float L = ok ? p.lse[ri] : -INFINITY;
        lse2[tid] = L * 1.4426950408889634f;
        dlt[tid] = ok ? p.delta[ri] : 0.f;
      }
      __syncthreads();

      for (int i = 0; i < kCols; ++i) {
        const float* qi = Qs + i * D;
        const float* doi = dOs + i * D;
        float qv[NT], dov[NT];
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          qv[t] = qi[4 * t + part];
          dov[t] = doi[4 * t + part];
          s = fmaf(qv[t], kr[t], s);
          dp = fmaf(dov[t], vr[t], dp);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 2);
        const int ii = q0 + i, jj = k0 + j;
        bool keep = kvalid && ii < si.len && lse2[i] != -INFINITY;
        if (elem_causal) keep = keep && jj <= ii;
        const float pij = keep ? exp2f(s * p.scale_log2 - lse2[i]) : 0.f;
        const float ds = pij * (dp - dlt[i]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          dv[t] = fmaf(pij, dov[t], dv[t]);
          dk[t] = fmaf(ds, qv[t], dk[t]);
        }
        if (part == 0) dSs[i * SS + j] = ds;
      }
      __syncthreads();

      // dQ rows of this block: row i = tid/4, columns 4t + part
      {
        const int i = tid >> 2;
        if (q0 + i < si.len && check_q_row(p, si, h, q0 + i)) {
          float a[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) a[t] = 0.f;
          for (int jj = 0; jj < kRows; ++jj) {
            const float dsv = dSs[i * SS + jj];
#pragma unroll
            for (int t = 0; t < NT; ++t) a[t] = fmaf(dsv, Ks[jj * D + 4 * t + part], a[t]);
          }
          float* dst = p.dq_accum + dqacc_off(p, si, h, q0 + i);
#pragma unroll
          for (int t = 0; t < NT; ++t) atomicAdd(dst + 4 * t + part, a[t]);
        }
      }
    }
  }

  if (kvalid) {
    T* dK = static_cast<T*>(p.dk);
    T* dV = static_cast<T*>(p.dv);
    const long long off = kv_off(p, si, g, k0 + j);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      dK[off + 4 * t + part] = from_f32<T>(dk[t] * p.scale);
      dV[off + 4 * t + part] = from_f32<T>(dv[t]);
    }
  }
}

// ---------------------------------------------------------------------------
// Backward at head dim 256.  The layout above would hold K, V, dK and dV rows in
// registers (4 x 64 per thread), more than a thread has, so here K and V stay
// in shared memory (rows padded to 260 floats so the eight key rows a warp
// reads fall in different banks) and only dK and dV are in registers; query
// rows are staged 32 at a time.  Thread (j = tid/4, part = tid%4) still owns key
// row j and columns 4t + part.
// ---------------------------------------------------------------------------
constexpr int kQStep256 = 32;

template <class T>
__global__ void __launch_bounds__(kThreads) k_simt_bwd256(KParams p) {
  constexpr int D = 256, NT = D / 4, KS = D + 4, SS = kRows + 1;
  extern __shared__ float smem[];
  float* Ks = smem;                    // [64][260]
  float* Vs = Ks + kRows * KS;         // [64][260]
  float* Qs = Vs + kRows * KS;         // [32][256]
  float* dOs = Qs + kQStep256 * D;     // [32][256]
  float* dSs = dOs + kQStep256 * D;    // [32 q][65]
  float* lse2 = dSs + kQStep256 * SS;  // [32]
  float* dlt = lse2 + kQStep256;       // [32]

  const Unit u = p.units[blockIdx.x];
  if (!check_unit(p, u, true, kRows)) return;
  const SeqInfo si = seq_info(p, u.seq);
  const int g = u.head;
  const int k0 = u.tile * kRows;
  if (k0 >= si.len) return;
  const int tid = threadIdx.x, j = tid >> 2, part = tid & 3;
  const int warp = tid >> 5, lane = tid & 31;
  const T* Q = static_cast<const T*>(p.q);
  const T* K = static_cast<const T*>(p.k);
  const T* V = static_cast<const T*>(p.v);
  const T* dO = static_cast<const T*>(p.dout);

  for (int r = warp; r < kRows; r += kThreads / 32) {
    const bool ok = k0 + r < si.len && check_kv_row(p, si, g, k0 + r);
    const long long off = ok ? kv_off(p, si, g, k0 + r) : 0;
    for (int d = lane; d < D; d += 32) {
      Ks[r * KS + d] = ok ? to_f32(K[off + d]) : 0.f;
      Vs[r * KS + d] = ok ? to_f32(V[off + d]) : 0.f;
    }
  }
  const bool kvalid = k0 + j < si.len && check_kv_row(p, si, g, k0 + j);
  float dk[NT], dv[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) dk[t] = dv[t] = 0.f;

  const int nqb_seq = (si.len + kCols - 1) / kCols;
  const int kblk = u.tile;
  int qb_begin = 0, qb_count = nqb_seq, e0 = 0;
  if (p.mask == kMaskCausal) {
    qb_begin = kblk;
    qb_count = nqb_seq - kblk;
  } else if (p.mask == kMaskBlock) {
    e0 = p.csc_ptr[kblk];
    qb_count = p.csc_ptr[kblk + 1] - e0;
  }
  const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);
  const float* krow = Ks + j * KS;
  const float* vrow = Vs + j * KS;

  for (int hh = 0; hh < p.group; ++hh) {
    const int h = g * p.group + hh;
    for (int it = 0; it < qb_count; ++it) {
      int qb = p.mask == kMaskBlock ? p.csc_idx[e0 + it] : qb_begin + it;
      if (p.mask == kMaskBlock && !check_block(p, qb, p.n_row_blocks)) qb = INT_MAX / (2 * kCols);
      for (int half = 0; half < kCols / kQStep256; ++half) {
        const int q0 = qb * kCols + half * kQStep256;
        if (q0 >= si.len) continue;
        __syncthreads();  // previous step done with Qs, dOs, dSs (and K, V written)
        for (int r = warp; r < kQStep256; r += kThreads / 32) {
          const bool ok = q0 + r < si.len && check_q_row(p, si, h, q0 + r);
          const long long off = ok ? q_off(p, si, h, q0 + r) : 0;
          for (int d = lane; d < D; d += 32) {
            Qs[r * D + d] = ok ? to_f32(Q[off + d]) : 0.f;
            dOs[r * D + d] = ok ? to_f32(dO[off + d]) : 0.f;
          }
        }
        if (tid < kQStep256) {
          const bool ok = q0 + tid < si.len && check_q_row(p, si, h, q0 + tid);
          const long long ri = ok ? row_index(p, si, h, q0 + tid) : 0;
          const float L = ok ? p.lse[ri] : -INFINITY;
          lse2[tid] = L * 1.4426950408889634f;
          dlt[tid] = ok ? p.delta[ri] : 0.f;
        }
        __syncthreads();

        for (int i = 0; i < kQStep256; ++i) {
          const float* qi = Qs + i * D;
          const float* doi = dOs + i * D;
          float s = 0.f, dp = 0.f;
#pragma unroll 16
          for (int t = 0; t < NT; ++t) {
            s = fmaf(qi[4 * t + part], krow[4 * t + part], s);
            dp = fmaf(doi[4 * t + part], vrow[4 * t + part], dp);
          }
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          s += __shfl_xor_sync(0xffffffffu, s, 2);
          dp += __shfl_xor_sync(0xffffffffu, dp, 1);
          dp += __shfl_xor_sync(0xffffffffu, dp, 2);
          const int ii = q0 + i, jj = k0 + j;
          bool keep = kvalid && ii < si.len && lse2[i] != -INFINITY;
          if (elem_causal) keep = keep && jj <= ii;
          const float pij = keep ? exp2f(s * p.scale_log2 - lse2[i]) : 0.f;
          const float ds = pij * (dp - dlt[i]);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            dv[t] = fmaf(pij, doi[4 * t + part], dv[t]);
            dk[t] = fmaf(ds, qi[4 * t + part], dk[t]);
          }
          if (part == 0) dSs[i * SS + j] = ds;
        }
        __syncthreads();

        // dQ rows of this step: row i = tid / 8, columns 8t + sub
        {
          const int i = tid >> 3, sub = tid & 7;
          if (q0 + i < si.len && check_q_row(p, si, h, q0 + i)) {
            float a[D / 8];
#pragma unroll
            for (int t = 0; t < D / 8; ++t) a[t] = 0.f;
            for (int jj = 0; jj < kRows; ++jj) {
              const float dsv = dSs[i * SS + jj];
#pragma unroll
              for (int t = 0; t < D / 8; ++t) a[t] = fmaf(dsv, Ks[jj * KS + 8 * t + sub], a[t]);
            }
            float* dst = p.dq_accum + dqacc_off(p, si, h, q0 + i);
#pragma unroll
            for (int t = 0; t < D / 8; ++t) atomicAdd(dst + 8 * t + sub, a[t]);
          }
        }
      }
    }
  }

  if (kvalid) {
    T* dK = static_cast<T*>(p.dk);
    T* dV = static_cast<T*>(p.dv);
    const long long off = kv_off(p, si, g, k0 + j);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      dK[off + 4 * t + part] = from_f32<T>(dk[t] * p.scale);
      dV[off + 4 * t + part] = from_f32<T>(dv[t]);
    }
  }
}

template <class T>
cudaError_t launch_bwd256_t(const KParams& p, cudaStream_t st) {
  constexpr size_t smem =
      sizeof(float) * (2 * kRows * (256 + 4) + 2 * kQStep256 * 256 + kQStep256 * (kRows + 1) + 2 * kQStep256);
  cudaError_t e = cudaFuncSetAttribute(k_simt_bwd256<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_simt_bwd256<T><<<p.n_units, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template <class T, int D>
cudaError_t launch_fwd_t(const KParams& p, cudaStream_t st) {
  constexpr size_t smem = sizeof(float) * (kRows * D + kCols * (D + 1) + kCols * D + 8 * 8 * kCols);
  cudaError_t e = cudaFuncSetAttribute(k_simt_fwd<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  k_simt_fwd<T, D><<<p.n_units, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template <class T, int D>
cudaError_t launch_bwd_t(const KParams& p, cudaStream_t st) {
  constexpr size_t smem = sizeof(float) * (3 * kRows * D + kCols * (kCols + 1) + 2 * kCols);
  cudaError_t e = cudaFuncSetAttribute(k_simt_bwd<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  k_simt_bwd<T, D><<<p.n_units, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_fwd(const KParams& p, bool bf16, cudaStream_t st) {
  if (p.n_units == 0) return cudaSuccess;
  if (bf16) return p.head_dim == 256   ? launch_fwd_t<__nv_bfloat16, 256>(p, st)
                   : p.head_dim == 128 ? launch_fwd_t<__nv_bfloat16, 128>(p, st)
                                       : launch_fwd_t<__nv_bfloat16, 64>(p, st);
  return p.head_dim == 256   ? launch_fwd_t<float, 256>(p, st)
         : p.head_dim == 128 ? launch_fwd_t<float, 128>(p, st)
                             : launch_fwd_t<float, 64>(p, st);
}

cudaError_t launch_simt_bwd(const KParams& p, bool bf16, cudaStream_t st) {
  if (p.n_units == 0) return cudaSuccess;
  if (p.head_dim == 256) return bf16 ? launch_bwd256_t<__nv_bfloat16>(p, st) : launch_bwd256_t<float>(p, st);
  if (bf16) return p.head_dim == 128 ? launch_bwd_t<__nv_bfloat16, 128>(p, st)
                                     : launch_bwd_t<__nv_bfloat16, 64>(p, st);
  return p.head_dim == 128 ? launch_bwd_t<float, 128>(p, st) : launch_bwd_t<float, 64>(p, st);
}

}  // namespace gbattn
