// Backward attention on the fifth-generation tensor cores (sm_103a).
//
// The forward drops the attention matrix, so the backward recomputes it block
// by block and produces three gradients; walking the keys' blocks gathers dK and
// dV, while dQ accumulates in the opposite direction and many blocks add into
// the same rows (smzdm contest article "杀进决赛!这 28 支队伍把算子优化卷疯了!",
// section 03).  This kernel keeps one 128-key tile of K and V on chip, walks the
// query blocks (of every query head of the KV head's group) that see it, and
// accumulates dK and dV in tensor memory; each block's dQ share is added into a
// float32 accumulator with atomic adds.
//
// Per 64-row query block i (all five products on the tensor cores, bf16 operands,
// float32 accumulation in tensor memory):
//   S^T  = K Q_i^T            P^T = exp(S^T * scale - LSE_i)   (masked: 0)
//   dP^T = V dO_i^T           dS^T = P^T o (dP^T - D_i),  D_i = <dO_i, O_i>
//   dV  += P^T dO_i           (P^T read from tensor memory)
//   dK  += dS^T Q_i           (dS^T from shared memory)
//   dQ_i^T = K^T dS^T         -> float32 atomics into the accumulator
//
// Warp roles (320 threads):
//   warps 0-3  thread t owns key row t: P^T, dS^T, then the dK epilogue
//   warps 4-7  thread t owns head-dim column t of dQ_i^T: atomics; dV epilogue
//   warp 8     TMA producer (K, V once; Q_i, dO_i double-buffered) + LSE, D rows
//   warp 9     tensor-core issuer (one thread)
// Every wait is bounded; a CTA that gives up records ATTN_ERR_DEVICE_TIMEOUT,
// drains its copies and tensor-core work, frees tensor memory and returns.
#include <cuda.h>

#include "tc_common.cuh"
#include "tc_kernels.h"
#include "tma_host.h"

namespace gbattn {

namespace {

constexpr int kQB = 64;                          // query rows per step
constexpr uint32_t kQBoxBytes = kQB * 128;       // 64 rows x 64 bf16 columns (128-byte rows)
constexpr uint32_t kQTileBytes = 2 * kQBoxBytes; // 64 x 128 bf16
constexpr uint32_t kDsBytes = kTile * kQB * 2;   // dS^T: 128 key rows x 64 bf16 query columns
constexpr int kBwdThreads = 320;
constexpr uint32_t kTmemCols = 512;
// dV [0,128) dK [128,256) S^T buffers [256,320) [320,384) dP^T [384,448) dQ^T [448,512)
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384, kColDQ = 448;

struct BwdArgs {
  CUtensorMap tq, tk, tv, tdo;
  int q_rows_inner, kv_rows_inner;
  KParams p;
};

struct BwdSmem {
  uint8_t k[kTileBytes];
  uint8_t v[kTileBytes];
  uint8_t q[2][kQTileBytes];   // Q_i stages; dK staging in the epilogue
  uint8_t dO[2][kQTileBytes];  // dO_i stages; dV staging in the epilogue
  uint8_t ds[2][kDsBytes];     // dS^T buffers (128-byte swizzled rows)
  float lse2[2][kQB];          // LSE * log2(e) of the stage's query rows (+inf: no key)
  float dlt[2][kQB];           // D of the stage's query rows
  uint64_t kv_full, qdo_full[2], qdo_empty[2], st_full[2], pt_full[2], dp_full, dp_free;
  uint64_t ds_full[2], ds_free[2], dq_full, dq_free, mma_done, drain;
  uint32_t tmem_base;
  ptx::Abort abort;
};

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, BwdSmem& sm, const KParams& p) {
  bool ok = ptx::mbar_wait(bar, parity, &sm.abort, p.status, p.wait_limit_ns);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool wait_one(uint64_t* bar, uint32_t parity, BwdSmem& sm, const KParams& p) {
  return ptx::mbar_wait(bar, parity, &sm.abort, p.status, p.wait_limit_ns);
}

__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, const KParams& p) {
  ptx::Abort none;
  none.flag = 0;
  ptx::mbar_wait(bar, parity, &none, p.status, p.wait_limit_ns);
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// Writes 32 float32 accumulator columns (x scale) of this thread's row as bf16
// into a 256-byte-row staging tile, 16-byte chunk c of row r at chunk c ^ (r & 15).
__device__ __forceinline__ void stage_row_chunks(uint8_t* stage, int r, int cc, const uint32_t (&v)[32],
                                                 float scale) {
#pragma unroll
  for (int w4 = 0; w4 < 4; ++w4) {
    uint4 o;
    o.x = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 0]) * scale, __uint_as_float(v[w4 * 8 + 1]) * scale);
    o.y = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 2]) * scale, __uint_as_float(v[w4 * 8 + 3]) * scale);
    o.z = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 4]) * scale, __uint_as_float(v[w4 * 8 + 5]) * scale);
    o.w = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 6]) * scale, __uint_as_float(v[w4 * 8 + 7]) * scale);
    const int ch = cc * 4 + w4;
    *reinterpret_cast<uint4*>(stage + r * 256 + ((ch ^ (r & 15)) * 16)) = o;
  }
}

// One warp: reads its 32 rows of a 128-column accumulator from tensor memory
// (or zeros), scales, rounds to bf16 and writes them to global memory rows
// k0 + row (row < len) of head g through a staging tile.
__device__ __forceinline__ void write_kv_rows(uint32_t taddr_row, bool have, float scale, uint8_t* stage,
                                              int wq, int lane, const KParams& p, const SeqInfo& si, int g,
                                              int k0, void* out) {
  const int r = wq * 32 + lane;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t v[32];
    if (have) {
      ptx::tmem_ld32(taddr_row + cc * 32, v);
      ptx::tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
    stage_row_chunks(stage, r, cc, v, scale);
  }
  __syncwarp();
  __nv_bfloat16* O = static_cast<__nv_bfloat16*>(out);
#pragma unroll 4
  for (int it = 0; it < 16; ++it) {
    const int row = wq * 32 + it * 2 + (lane >> 4), ch = lane & 15;
    if (k0 + row < si.len) {
      const uint4 v4 = *reinterpret_cast<const uint4*>(stage + row * 256 + ((ch ^ (row & 15)) * 16));
      *reinterpret_cast<uint4*>(O + kv_off(p, si, g, k0 + row) + ch * 8) = v4;
    }
  }
}

__global__ void __launch_bounds__(kBwdThreads, 1) k_tc_bwd(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KParams& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Unit u = p.units[blockIdx.x];
  const SeqInfo si = seq_info(p, u.seq);
  const int g = u.head;
  const int kt = u.tile, k0 = kt * kTile;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sm.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.qdo_full[s], 2);  // TMA transaction arrival + LSE/D rows written
      ptx::mbar_init(&sm.qdo_empty[s], 1);
      ptx::mbar_init(&sm.st_full[s], 1);
      ptx::mbar_init(&sm.pt_full[s], 4);
      ptx::mbar_init(&sm.ds_full[s], 4);
      ptx::mbar_init(&sm.ds_free[s], 1);
    }
    ptx::mbar_init(&sm.dp_full, 1);
    ptx::mbar_init(&sm.dp_free, 4);
    ptx::mbar_init(&sm.dq_full, 1);
    ptx::mbar_init(&sm.dq_free, 4);
    ptx::mbar_init(&sm.mma_done, 1);
    ptx::mbar_init(&sm.drain, 1);
    sm.abort.flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  BwdSteps steps;
  steps.init(p, si.len, kt);
  int n_steps = 0;
  {
    BwdSteps t = steps;
    int hh, qb, bits;
    while (t.next(hh, qb, bits)) ++n_steps;
  }
  const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    int last_phase[2] = {-1, -1};
    if (n_steps > 0) {
      if (lane == 0) {
        ptx::tma_prefetch_desc(&a.tq);
        ptx::tma_prefetch_desc(&a.tdo);
        ptx::mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
        tma_tile(sm.k, &a.tk, a.kv_rows_inner, &sm.kv_full, map_row(si, k0), g, si.b, kHalfTileBytes);
        tma_tile(sm.v, &a.tv, a.kv_rows_inner, &sm.kv_full, map_row(si, k0), g, si.b, kHalfTileBytes);
      }
      BwdSteps t = steps;
      int hh, qb, bits, i = 0;
      while (t.next(hh, qb, bits)) {
        const int st = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!wait_warp(&sm.qdo_empty[st], ph ^ 1, sm, p)) break;
        const int h = g * p.group + hh, q0 = qb * kQB;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(&sm.qdo_full[st], 2 * kQTileBytes);
          tma_tile(sm.q[st], &a.tq, a.q_rows_inner, &sm.qdo_full[st], map_row(si, q0), h, si.b, kQBoxBytes);
          tma_tile(sm.dO[st], &a.tdo, a.q_rows_inner, &sm.qdo_full[st], map_row(si, q0), h, si.b, kQBoxBytes);
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = lane + 32 * c2, qi = q0 + c;
          float l2 = INFINITY, dl = 0.f;
          if (qi < si.len) {
            const long long ri = row_index(p, si, h, qi);
            const float L = p.lse[ri];
            l2 = L == -INFINITY ? INFINITY : L * 1.4426950408889634f;
            dl = p.delta[ri];
          }
          sm.lse2[st][c] = l2;
          sm.dlt[st][c] = dl;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.qdo_full[st]);
        last_phase[st] = (int)ph;
        ++i;
      }
      if (lane == 0) {
        wait_drain(&sm.kv_full, 0, p);
        for (int s = 0; s < 2; ++s)
          if (last_phase[s] >= 0) wait_drain(&sm.qdo_full[s], (uint32_t)last_phase[s], p);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if (n_steps > 0) {
        constexpr uint32_t id_st = ptx::idesc_bf16(128, 64, false, false);   // S^T, dP^T
        constexpr uint32_t id_acc = ptx::idesc_bf16(128, 128, false, true);  // dV, dK
        constexpr uint32_t id_dq = ptx::idesc_bf16(128, 64, true, true);     // dQ^T
        const uint32_t k_addr = ptx::smem_u32(sm.k), v_addr = ptx::smem_u32(sm.v);
        bool ok = wait_one(&sm.kv_full, 0, sm, p);
        ptx::tc_fence_after();

        // S^T_i = K Q_i^T: A = K (key rows, head dim contiguous), B = Q_i (query rows).
        auto issue_s = [&](int i) -> bool {
          const int st = i & 1;
          if (!wait_one(&sm.qdo_full[st], (i >> 1) & 1, sm, p)) return false;
          ptx::tc_fence_after();
          const uint32_t q_addr = ptx::smem_u32(sm.q[st]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = ptx::sdesc_sw128(k_addr + (kk >> 2) * kHalfTileBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = ptx::sdesc_sw128(q_addr + (kk >> 2) * kQBoxBytes + (kk & 3) * 32, 16, 1024);
            ptx::mma_ss(tmem + kColS + st * 64, ad, bd, id_st, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&sm.st_full[st]);
          return true;
        };
        // dP^T_i = V dO_i^T (the stage is already known to be loaded).
        auto issue_dp = [&](int i) -> bool {
          const int st = i & 1;
          if (i > 0 && !wait_one(&sm.dp_free, (i - 1) & 1, sm, p)) return false;
          ptx::tc_fence_after();
          const uint32_t do_addr = ptx::smem_u32(sm.dO[st]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = ptx::sdesc_sw128(v_addr + (kk >> 2) * kHalfTileBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = ptx::sdesc_sw128(do_addr + (kk >> 2) * kQBoxBytes + (kk & 3) * 32, 16, 1024);
            ptx::mma_ss(tmem + kColDP, ad, bd, id_st, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&sm.dp_full);
          return true;
        };

        ok = ok && issue_s(0) && issue_dp(0);
        for (int i = 0; ok && i < n_steps; ++i) {
          const int st = i & 1;
          if (i + 1 < n_steps && !issue_s(i + 1)) { ok = false; break; }
          // dV += P^T_i dO_i: A = P^T from tensor memory, B = dO_i as (head dim, query) MN-major.
          if (!wait_one(&sm.pt_full[st], (i >> 1) & 1, sm, p)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t q_addr = ptx::smem_u32(sm.q[st]), do_addr = ptx::smem_u32(sm.dO[st]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = ptx::sdesc_sw128(do_addr + kk * 2048, kQBoxBytes, 1024);
            ptx::mma_ts(tmem + kColDV, tmem + kColS + st * 64 + kk * 8, bd, id_acc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          if (i + 1 < n_steps && !issue_dp(i + 1)) { ok = false; break; }
          // dK += dS^T_i Q_i: A = dS^T (key rows, query contiguous), B = Q_i MN-major.
          if (!wait_one(&sm.ds_full[st], (i >> 1) & 1, sm, p)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t ds_addr = ptx::smem_u32(sm.ds[st]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = ptx::sdesc_sw128(ds_addr + kk * 32, 16, 1024);
            const uint64_t bd = ptx::sdesc_sw128(q_addr + kk * 2048, kQBoxBytes, 1024);
            ptx::mma_ss(tmem + kColDK, ad, bd, id_acc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          // dQ_i^T = K^T dS^T_i: A = K^T (head dim contiguous: MN-major), B = dS^T as
          // (query, key) with query contiguous: MN-major.
          if (i > 0 && !wait_one(&sm.dq_free, (i - 1) & 1, sm, p)) { ok = false; break; }
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = ptx::sdesc_sw128(k_addr + kk * 2048, kHalfTileBytes, 1024);
            const uint64_t bd = ptx::sdesc_sw128(ds_addr + kk * 2048, kDsBytes, 1024);
            ptx::mma_ss(tmem + kColDQ, ad, bd, id_dq, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&sm.dq_full);
          ptx::mma_commit(&sm.qdo_empty[st]);
          ptx::mma_commit(&sm.ds_free[st]);
        }
      }
      ptx::mma_commit(&sm.mma_done);
      ptx::mma_commit(&sm.drain);
      wait_drain(&sm.drain, 0, p);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ P^T / dS^T warps
    const int t = threadIdx.x;  // key row in the tile = TMEM lane
    const int kj = k0 + t;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float c = p.scale_log2;
    const int key_half = t >= 64 ? 1 : 0;
    bool ok = true;
    BwdSteps s = steps;
    int hh, qb, bits, i = 0;
    while (s.next(hh, qb, bits)) {
      const int st = i & 1;
      const int q0 = qb * kQB;
      if (!wait_warp(&sm.qdo_full[st], (i >> 1) & 1, sm, p) || !wait_warp(&sm.st_full[st], (i >> 1) & 1, sm, p)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t sr[64];
      ptx::tmem_ld32(tmem + lane_base + kColS + st * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      ptx::tmem_ld32(tmem + lane_base + kColS + st * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      ptx::tmem_ld_wait();
      const bool need_mask = (k0 + kTile > si.len) || (elem_causal && q0 < k0 + kTile - 1) || bits != 3;
      const bool row_listed = (bits >> key_half) & 1;
      float pv[64];
      uint32_t pk[32];
#pragma unroll
      for (int cc = 0; cc < 64; ++cc) {
        bool keep = true;
        if (need_mask) {
          keep = row_listed && kj < si.len;
          if (elem_causal) keep = keep && kj <= q0 + cc;
        }
        pv[cc] = keep ? fast_exp2(__uint_as_float(sr[cc]) * c - sm.lse2[st][cc]) : 0.f;
      }
#pragma unroll
      for (int w = 0; w < 32; ++w) pk[w] = ptx::pack_bf16x2(pv[2 * w], pv[2 * w + 1]);
      ptx::tmem_st32(tmem + lane_base + kColS + st * 64, pk);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.pt_full[st]);

      if (!wait_warp(&sm.dp_full, i & 1, sm, p)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t dr[64];
      ptx::tmem_ld32(tmem + lane_base + kColDP, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      ptx::tmem_ld32(tmem + lane_base + kColDP + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.dp_free);

      if (!wait_warp(&sm.ds_free[st], ((i >> 1) & 1) ^ 1, sm, p)) {
        ok = false;
        break;
      }
      uint8_t* dsrow = sm.ds[st] + t * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint4 o;
        float d[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int cc = ch * 8 + e;
          d[e] = pv[cc] * (__uint_as_float(dr[cc]) - sm.dlt[st][cc]);
        }
        o.x = ptx::pack_bf16x2(d[0], d[1]);
        o.y = ptx::pack_bf16x2(d[2], d[3]);
        o.z = ptx::pack_bf16x2(d[4], d[5]);
        o.w = ptx::pack_bf16x2(d[6], d[7]);
        *reinterpret_cast<uint4*>(dsrow + ((ch ^ (t & 7)) * 16)) = o;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.ds_full[st]);
      ++i;
    }
    // dK epilogue
    if (ok && wait_warp(&sm.mma_done, 0, sm, p) && !sm.abort.flag) {
      ptx::tc_fence_after();
      write_kv_rows(tmem + lane_base + kColDK, n_steps > 0, p.scale, sm.q[0], warp, lane, p, si, g, k0, p.dk);
    }
  } else {
    // ------------------------------------------------------------ dQ warps
    const int wq = warp - 4;
    const int d = wq * 32 + lane;  // head-dim column = TMEM lane
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    bool ok = true;
    BwdSteps s = steps;
    int hh, qb, bits, i = 0;
    while (s.next(hh, qb, bits)) {
      if (!wait_warp(&sm.dq_full, i & 1, sm, p)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t vr[64];
      ptx::tmem_ld32(tmem + lane_base + kColDQ, *reinterpret_cast<uint32_t(*)[32]>(&vr[0]));
      ptx::tmem_ld32(tmem + lane_base + kColDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&vr[32]));
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.dq_free);
      const int h = g * p.group + hh, q0 = qb * kQB;
      const int nrows = min(kQB, si.len - q0);
      float* base = p.dq_accum + dqacc_off(p, si, h, q0) + d;
      const long long rstride = p.varlen ? (long long)p.heads_q * p.head_dim : p.head_dim;
#pragma unroll
      for (int cc = 0; cc < 64; ++cc)
        if (cc < nrows) red_add_f32(base + cc * rstride, __uint_as_float(vr[cc]));
      ++i;
    }
    // dV epilogue
    if (ok && wait_warp(&sm.mma_done, 0, sm, p) && !sm.abort.flag) {
      ptx::tc_fence_after();
      write_kv_rows(tmem + lane_base + kColDV, n_steps > 0, 1.f, sm.dO[0], wq, lane, p, si, g, k0, p.dv);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool tc_bwd_available() { return true; }

cudaError_t launch_tc_bwd(const KParams& p, int sms, cudaStream_t st) {
  (void)sms;
  if (p.n_units == 0) return cudaSuccess;
  BwdArgs a;
  TileMap mq, mk, mv, mdo;
  cudaError_t e;
  if ((e = make_tile_map(&mq, p.q, p, false, kQB)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mdo, p.dout, p, false, kQB)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mk, p.k, p, true)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mv, p.v, p, true)) != cudaSuccess) return e;
  a.tq = mq.map;
  a.tdo = mdo.map;
  a.tk = mk.map;
  a.tv = mv.map;
  a.q_rows_inner = mq.rows_inner;
  a.kv_rows_inner = mk.rows_inner;
  a.p = p;
  const size_t smem = sizeof(BwdSmem) + 1024;
  e = cudaFuncSetAttribute(k_tc_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_tc_bwd<<<p.n_units, kBwdThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbattn
