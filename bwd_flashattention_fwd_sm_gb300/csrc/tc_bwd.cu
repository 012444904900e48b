// Backward attention on the fifth-generation tensor cores (sm_103a): persistent
// CTAs, dQ reduced through TMA.
//
// The forward drops the attention matrix, so the backward recomputes it block
// by block and produces three gradients; walking the key blocks gathers dK and
// dV, while dQ accumulates in the opposite direction and many blocks add into
// the same rows (smzdm contest article "杀进决赛!这 28 支队伍把算子优化卷疯了!",
// section 03).  A unit keeps one 128-key tile of K and V on chip, walks the
// 64-row query blocks (of every query head of the KV head's group) that see it,
// and accumulates dK and dV in tensor memory.
//
// Per query block i (five tcgen05 products, bf16 operands, float32 accumulation):
//   S^T  = K Q_i^T            P^T = exp(S^T * scale - LSE_i)   (masked: 0)
//   dP^T = V dO_i^T           dS^T = P^T o (dP^T - D_i),  D_i = <dO_i, O_i>
//   dV  += P^T dO_i           (P^T read from tensor memory)
//   dK  += dS^T Q_i           (dS^T from shared memory)
//   dQ_i^T = K^T dS^T         -> staged in shared memory, added into the float32
//                                accumulator by one TMA reduce-add (the L2 adds)
//
// CTAs are persistent (one per SM): the TMA warp takes the next unit from an
// atomic counter over the cost-ordered work list (zwxr.cn CANN ops-nn article,
// section 4.2: whoever finishes first takes the next block) and hands it to the
// other roles through a two-slot ring in shared memory.
//
// V is the A operand of dP^T only, so it sits in tensor memory (packed bf16
// pairs, D / 2 columns), written once per unit by the compute warps: dP^T then
// reads only dO_i from shared memory, and its N = 64 products run at the full
// rate instead of being paced by shared-memory reads.  Tensor memory:
//   dV [0,128)  dK [128,256)  S^T / P^T [256,320)  V [320,384)  dP^T [384,448)
//   dQ^T [448,512).
// With one S^T buffer, the next step's S^T is issued after this step's dV
// product, which reads P^T in place.
//
// Warp roles (480 threads):
//   warps 0-7    compute: warp w covers TMEM lane quarter w % 4 (key rows) and
//                query columns 32 (w / 4) .. +31 of the step.  Per step: P^T and
//                dS^T.  Per unit: head-dim half w / 4 of V for their key rows
//                into tensor memory.  Unit epilogue: warps 0-3 dK, warps 4-7 dV.
//   warp 8       TMA producer (K per unit; Q_i, dO_i in a 3-stage ring; LSE, D rows)
//   warp 9       tensor-core issuer for S^T, dP^T and dV (whole warp, one
//                elected lane issues)
//   warp 14      tensor-core issuer for dK and dQ^T.  tcgen05.mma holds its
//                thread until the tensor core takes it, so with one issuer every
//                barrier wait left the tensor core idle; with two, one waits
//                while the other's products run.
//   warps 10-13  dQ writers: warp w reads head-dim rows 32 (w % 4) .. +31 of
//                dQ_i^T from tensor memory, stages them in shared memory as
//                [query][head dim], and one thread adds the tile into the float32
//                accumulator with a TMA reduce; this runs beside the next step's
//                P^T / dS^T work instead of inside it.
// Every mbarrier wait is bounded; a CTA that gives up records
// ATTN_ERR_DEVICE_TIMEOUT, drains its copies and tensor-core work, frees tensor
// memory and returns.
#include <cuda.h>

#include <cstring>

#include "tc_common.cuh"
#include "tc_kernels.h"
#include "tma_host.h"

namespace gbattn {

namespace {

constexpr int kQB = 64;                           // query rows per step
constexpr uint32_t kQBoxBytes = kQB * 128;        // 64 rows x 64 bf16 (128-byte rows)
constexpr uint32_t kQTileBytes = 2 * kQBoxBytes;  // 64 x 128 bf16
constexpr uint32_t kDsBytes = kTile * kQB * 2;    // dS^T: 128 key rows x 64 bf16 query columns
constexpr int kStages = 3;  // Q_i / dO_i ring: loads run two steps ahead of the products
constexpr int kThreads = 480;
constexpr uint32_t kTmemCols = 512;
// dV [0,128) dK [128,256) S^T [256,320) V [320,384) dP^T [384,448) dQ^T [448,512)
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColV = 320, kColDP = 384, kColDQ = 448;

struct BwdArgs {
  CUtensorMap tq, tk, tdo, tacc;
  int q_rows_inner, kv_rows_inner, acc_rows_inner;
  KParams p;
};

struct Smem {
  uint8_t k[kTileBytes];
  uint8_t q[kStages][kQTileBytes];
  uint8_t dO[kStages][kQTileBytes];
  uint8_t ds[2][kDsBytes];   // dS^T (128-byte swizzled rows)
  float dq[kQB * kHeadDim];  // dQ_i staging, row-major [query][head dim]
  float nlse2[kStages][kQB];  // -LSE * log2(e) of the stage's query rows (-inf: no key / past the end)
  float ndlt[kStages][kQB];   // -D of the stage's query rows
  uint64_t unit_full[2], unit_empty[2];
  uint64_t k_full, k_empty, v_full, qdo_full[kStages], qdo_empty[kStages];
  uint64_t st_full[2], pt_full[2], dp_full, dp_free, ds_full[2], ds_free[2], dq_full, dq_free;
  uint64_t acc_done, acc_free, drain[2];
  int unit_slot[2][4];
  uint32_t tmem_base;
  ptx::Abort abort;
};

static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory per CTA is at most 227 KiB");

struct Waiter {
  Smem& sm;
  const KParams& p;
  __device__ bool one(uint64_t* bar, uint32_t parity) {
    return ptx::mbar_wait(bar, parity, &sm.abort, p.status, p.wait_limit_ns);
  }
  __device__ bool warp(uint64_t* bar, uint32_t parity) {
    const bool ok = one(bar, parity);
    return __all_sync(0xffffffffu, ok);
  }
  __device__ void drain(uint64_t* bar, uint32_t parity) {
    ptx::Abort none;
    none.flag = 0;
    ptx::mbar_wait(bar, parity, &none, p.status, p.wait_limit_ns);
  }
};

__device__ __forceinline__ bool read_unit(const Smem& sm, int slot, Unit& un) {
  const volatile int* s = sm.unit_slot[slot];
  un.seq = s[0];
  un.head = s[1];
  un.tile = s[2];
  return s[3] != 0;
}

// AND of `pred` over the 256 compute threads (named barrier 1).  Named barriers
// have no time limit, so every compute thread reaches this exactly once per step
// and per unit whatever its own waits returned, and the group acts on the result.
__device__ __forceinline__ bool group_all(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}
// The same over the 128 dQ-writer threads (named barrier 2).
__device__ __forceinline__ bool dq_all(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void dq_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// One warp writes its 32 key rows of a D-column accumulator (x scale, bf16)
// straight from tensor memory to global memory rows k0 + row < len of head g.
template <int D>
__device__ __forceinline__ void store_kv_rows(uint32_t taddr_row, bool have, float scale, int row,
                                              const KParams& p, const SeqInfo& si, int g, int k0, void* out) {
  const bool ok = k0 + row < si.len && check_kv_row(p, si, g, k0 + row);
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + (ok ? kv_off(p, si, g, k0 + row) : 0);
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t v[32];
    if (have) {
      ptx::tmem_ld32(taddr_row + cc * 32, v);
      ptx::tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
    if (ok) {
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) {
        uint4 o;
        o.x = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 0]) * scale, __uint_as_float(v[w4 * 8 + 1]) * scale);
        o.y = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 2]) * scale, __uint_as_float(v[w4 * 8 + 3]) * scale);
        o.z = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 4]) * scale, __uint_as_float(v[w4 * 8 + 5]) * scale);
        o.w = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 6]) * scale, __uint_as_float(v[w4 * 8 + 7]) * scale);
        *reinterpret_cast<uint4*>(dst + cc * 32 + w4 * 8) = o;
      }
    }
  }
}

// One warp copies head-dim columns c0 .. c0 + D / 2 - 1 of its 32 key rows of
// V (row k0 + row of head g; zeros past the sequence end) into tensor memory at
// taddr_row as packed bf16 pairs, the layout of an A operand read from tensor
// memory (column j holds elements 2j and 2j + 1 of the row).
template <int D>
__device__ __forceinline__ void load_v_rows(uint32_t taddr_row, int row, int c0, const KParams& p,
                                            const SeqInfo& si, int g, int k0) {
  constexpr int kCols = D / 4;  // packed columns per warp: D / 2 elements
  const bool ok = k0 + row < si.len && check_kv_row(p, si, g, k0 + row);
  const uint4* src =
      reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.v) + (ok ? kv_off(p, si, g, k0 + row) : 0) + c0);
  uint32_t r[kCols];
#pragma unroll
  for (int j = 0; j < kCols / 4; ++j) {
    const uint4 x = ok ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
    r[4 * j] = x.x;
    r[4 * j + 1] = x.y;
    r[4 * j + 2] = x.z;
    r[4 * j + 3] = x.w;
  }
  if constexpr (kCols == 32) ptx::tmem_st32(taddr_row, r);
  else ptx::tmem_st16(taddr_row, r);
  ptx::tmem_st_wait();
}

// kDq false: dK and dV only (dQ comes from the query-stationary pass).
// D: head dim, 64 or 128 (shared memory is laid out for 128 either way).  With
// D = 64 the dQ^T product still runs with M = 128: the upper half of the K tile
// buffer holds zeros, so head-dim rows 64-127 of dQ^T are zero and unused.
template <bool kDq, int D>
__global__ void __launch_bounds__(kThreads, 1) k_tc_bwd(const __grid_constant__ BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KParams& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Waiter W{sm, p};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sm.qdo_full[s], 2);  // TMA transaction arrival + LSE/D rows written
      ptx::mbar_init(&sm.qdo_empty[s], 2);  // one commit per MMA warp
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.unit_full[s], 1);
      ptx::mbar_init(&sm.unit_empty[s], 14);  // 2 MMA warps + 8 compute warps + 4 dQ writers
      ptx::mbar_init(&sm.st_full[s], 1);
      ptx::mbar_init(&sm.pt_full[s], 8);
      ptx::mbar_init(&sm.ds_full[s], 8);
      ptx::mbar_init(&sm.ds_free[s], 1);
    }
    ptx::mbar_init(&sm.k_full, 1);
    ptx::mbar_init(&sm.k_empty, 2);  // one commit per MMA warp
    ptx::mbar_init(&sm.v_full, 8);   // compute warps
    ptx::mbar_init(&sm.dp_full, 1);
    ptx::mbar_init(&sm.dp_free, 8);
    ptx::mbar_init(&sm.dq_full, 1);
    ptx::mbar_init(&sm.dq_free, 4);  // dQ writer warps
    ptx::mbar_init(&sm.acc_done, 2);  // dV issuer + dK issuer
    ptx::mbar_init(&sm.acc_free, 8);  // dK writers (warps 0-3) + dV writers (warps 4-7)
    ptx::mbar_init(&sm.drain[0], 1);
    ptx::mbar_init(&sm.drain[1], 1);
    sm.abort.flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if constexpr (D == 64) {  // zero upper half of the K buffer (the A operand of dQ^T reads it)
    for (int i = threadIdx.x; i < (int)(kHalfTileBytes / 16); i += blockDim.x)
      reinterpret_cast<uint4*>(sm.k + kHalfTileBytes)[i] = make_uint4(0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);

  if (warp == 8) {
    // ================================================================ producer
    uint32_t n_units = 0, n_steps = 0;
    int last_qdo_phase[kStages] = {-1, -1, -1};
    bool kv_loaded = false;
    uint32_t last_kv_phase = 0;
    for (;;) {
      const int slot = n_units & 1;
      if (!W.warp(&sm.unit_empty[slot], ((n_units >> 1) & 1) ^ 1)) break;
      int idx = 0;
      if (lane == 0) idx = atomicAdd(p.unit_counter, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      bool valid = idx < p.n_units;
      Unit un{0, 0, 0, 0};
      if (valid) {
        un = p.units[idx];
        valid = check_unit(p, un, true, kTile);
      }
      if (lane == 0) {
        volatile int* s = sm.unit_slot[slot];
        s[0] = un.seq;
        s[1] = un.head;
        s[2] = un.tile;
        s[3] = valid ? 1 : 0;
        ptx::mbar_arrive(&sm.unit_full[slot]);
      }
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      const int g = un.head, k0 = un.tile * kTile;
      // The unit is known a few steps before the previous one ends: start its K
      // on its way into L2, so the load below does not wait on memory.
      if (lane == 0) tma_prefetch_tile(&a.tk, a.kv_rows_inner, map_row(si, k0), g, si.b, D / 64);
      // K of the unit, once the previous unit's products are done with it
      if (!W.warp(&sm.k_empty, (n_units & 1) ^ 1)) break;
      if (lane == 0) {
        check_kv_row(p, si, g, k0);
        ptx::mbar_arrive_expect_tx(&sm.k_full, tile_bytes<D>());
        tma_tile(sm.k, &a.tk, a.kv_rows_inner, &sm.k_full, map_row(si, k0), g, si.b, kHalfTileBytes, D / 64);
      }
      kv_loaded = true;
      last_kv_phase = n_units & 1;
      ++n_units;
      BwdSteps steps;
      steps.init(p, si.len, un.tile);
      int hh, qb, bits;
      bool ok = true;
      while (steps.next(hh, qb, bits)) {
        const int st = n_steps % kStages;
        const uint32_t ph = (n_steps / kStages) & 1;
        if (!W.warp(&sm.qdo_empty[st], ph ^ 1)) { ok = false; break; }
        const int h = g * p.group + hh, q0 = qb * kQB;
        if (lane == 0) {
          check_q_row(p, si, h, q0);
          ptx::mbar_arrive_expect_tx(&sm.qdo_full[st], 2 * kQBoxBytes * (D / 64));
          tma_tile(sm.q[st], &a.tq, a.q_rows_inner, &sm.qdo_full[st], map_row(si, q0), h, si.b, kQBoxBytes, D / 64);
          tma_tile(sm.dO[st], &a.tdo, a.q_rows_inner, &sm.qdo_full[st], map_row(si, q0), h, si.b, kQBoxBytes,
                   D / 64);
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = lane + 32 * c2, qi = q0 + c;
          float nl2 = -INFINITY, ndl = 0.f;
          if (qi < si.len && check_q_row(p, si, h, qi)) {
            const long long ri = row_index(p, si, h, qi);
            const float L = p.lse[ri];
            nl2 = L == -INFINITY ? -INFINITY : -L * 1.4426950408889634f;
            ndl = -p.delta[ri];
          }
          sm.nlse2[st][c] = nl2;
          sm.ndlt[st][c] = ndl;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.qdo_full[st]);
        last_qdo_phase[st] = (int)ph;
        ++n_steps;
      }
      if (!ok) break;
    }
    if (lane == 0) {
      if (kv_loaded) W.drain(&sm.k_full, last_kv_phase);
      for (int s = 0; s < kStages; ++s)
        if (last_qdo_phase[s] >= 0) W.drain(&sm.qdo_full[s], (uint32_t)last_qdo_phase[s]);
    }
  } else if (warp == 9 || warp == 14) {
    // ================================================================ MMA issuers
    // The whole warp runs the control flow in step; one elected lane issues the
    // tensor-core instructions and commits (a lone diverged thread is starved of
    // issue slots by the compute warps on its sub-partition).  elect.sync on the
    // full, converged warp picks the same lane every time, so each commit covers
    // every product that lane issued before it.  Both warps walk the same steps;
    // barriers that free a resource both use (Q_i / dO_i stage, K / V tiles, the
    // unit's accumulators) count one commit from each.
    const int side = warp == 9 ? 0 : 1;  // 0: S^T, dP^T, dV   1: dK, dQ^T
    constexpr uint32_t id_st = ptx::idesc_bf16(128, 64, false, false);   // S^T, dP^T
    constexpr uint32_t id_acc = ptx::idesc_bf16(128, D, false, true);    // dV, dK
    constexpr uint32_t id_dq = ptx::idesc_bf16(128, 64, true, true);     // dQ^T
    const uint32_t k_addr = ptx::smem_u32(sm.k);
    uint32_t n_units = 0, gi = 0;  // gi: global step counter (all units)
    bool ok = true;

    auto issue_s = [&](uint32_t i) -> bool {  // S^T_i = K Q_i^T
      const int st = i & 1, qs = i % kStages;
      if (!W.warp(&sm.qdo_full[qs], (i / kStages) & 1)) return false;
      ptx::tc_fence_after();
      const uint32_t q_addr = ptx::smem_u32(sm.q[qs]);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = ptx::sdesc_sw128(k_addr + (kk >> 2) * kHalfTileBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = ptx::sdesc_sw128(q_addr + (kk >> 2) * kQBoxBytes + (kk & 3) * 32, 16, 1024);
          ptx::mma_ss(tmem + kColS, ad, bd, id_st, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&sm.st_full[st]);
      }
      __syncwarp();
      return true;
    };
    // dP^T_i = V dO_i^T (stage known loaded): A = V from tensor memory (8
    // packed columns per 16 head-dim columns), B = dO_i K-major.  It overwrites
    // dP^T_{i-1}, so the compute warps must have read that.
    auto issue_dp = [&](uint32_t i) -> bool {
      const int qs = i % kStages;
      if (i > 0 && !W.warp(&sm.dp_free, (i - 1) & 1)) return false;
      ptx::tc_fence_after();
      const uint32_t do_addr = ptx::smem_u32(sm.dO[qs]);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t bd = ptx::sdesc_sw128(do_addr + (kk >> 2) * kQBoxBytes + (kk & 3) * 32, 16, 1024);
          ptx::mma_ts(tmem + kColDP, tmem + kColV + 8 * kk, bd, id_st, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&sm.dp_full);
      }
      __syncwarp();
      return true;
    };

    for (;;) {
      const int slot = n_units & 1;
      if (!W.warp(&sm.unit_full[slot], (n_units >> 1) & 1)) { ok = false; break; }
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      int n = 0;
      {
        BwdSteps t;
        t.init(p, si.len, un.tile);
        int hh, qb, bits;
        while (t.next(hh, qb, bits)) ++n;
      }
      if (!W.warp(&sm.k_full, n_units & 1)) { ok = false; break; }
      ptx::tc_fence_after();
      if (side == 0) {
        // the unit's V is in tensor memory before its first dP^T product
        if (n > 0) ok = issue_s(gi) && W.warp(&sm.v_full, n_units & 1) && issue_dp(gi);
        else ok = W.warp(&sm.v_full, n_units & 1);
        for (int s = 0; ok && s < n; ++s) {
          const uint32_t i = gi + s;
          const int st = i & 1, qs = i % kStages;
          // dV += P^T_i dO_i: A = P^T from tensor memory, B = dO_i as (head dim, query) MN-major
          if (!W.warp(&sm.pt_full[st], (i >> 1) & 1)) { ok = false; break; }
          // before the unit's first dV product: the previous unit's epilogue has
          // read the accumulators
          if (s == 0 && !W.warp(&sm.acc_free, (n_units & 1) ^ 1)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t do_addr = ptx::smem_u32(sm.dO[qs]);
          if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // P^T of query columns 16 kk .. +15: the compute warps of column half
              // kk / 2 write their 16 packed columns at 32 (kk / 2) within the S^T buffer
              const uint32_t a_col = kColS + 32 * (kk >> 1) + (kk & 1) * 8;
              const uint64_t bd = ptx::sdesc_sw128(do_addr + kk * 2048, kQBoxBytes, 1024);
              ptx::mma_ts(tmem + kColDV, tmem + a_col, bd, id_acc, (s > 0 || kk > 0) ? 1u : 0u);
            }
            // this side is done with Q_i / dO_i once S^T_i, dP^T_i and dV's product are
            ptx::mma_commit(&sm.qdo_empty[qs]);
          }
          __syncwarp();
          // one S^T buffer: the next S^T overwrites P^T_i after the dV product just
          // issued has read it (products of one thread run in order)
          if (s + 1 < n && !(issue_s(i + 1) && issue_dp(i + 1))) { ok = false; break; }
        }
      } else {
        for (int s = 0; ok && s < n; ++s) {
          const uint32_t i = gi + s;
          const int st = i & 1, qs = i % kStages;
          // dK += dS^T_i Q_i: A = dS^T (key rows, query contiguous), B = Q_i MN-major
          if (!W.warp(&sm.qdo_full[qs], (i / kStages) & 1)) { ok = false; break; }
          if (!W.warp(&sm.ds_full[st], (i >> 1) & 1)) { ok = false; break; }
          if (s == 0 && !W.warp(&sm.acc_free, (n_units & 1) ^ 1)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t q_addr = ptx::smem_u32(sm.q[qs]), ds_addr = ptx::smem_u32(sm.ds[st]);
          if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = ptx::sdesc_sw128(ds_addr + kk * 32, 16, 1024);
              const uint64_t bd = ptx::sdesc_sw128(q_addr + kk * 2048, kQBoxBytes, 1024);
              ptx::mma_ss(tmem + kColDK, ad, bd, id_acc, (s > 0 || kk > 0) ? 1u : 0u);
            }
          }
          __syncwarp();
          // dQ_i^T = K^T dS^T_i: A = K^T (head dim contiguous: MN-major), B = dS^T as
          // (query, key) with query contiguous: MN-major
          if (kDq && i > 0 && !W.warp(&sm.dq_free, (i - 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            if constexpr (kDq) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = ptx::sdesc_sw128(k_addr + kk * 2048, kHalfTileBytes, 1024);
                const uint64_t bd = ptx::sdesc_sw128(ds_addr + kk * 2048, kDsBytes, 1024);
                ptx::mma_ss(tmem + kColDQ, ad, bd, id_dq, kk > 0 ? 1u : 0u);
              }
              ptx::mma_commit(&sm.dq_full);
            }
            ptx::mma_commit(&sm.qdo_empty[qs]);
            ptx::mma_commit(&sm.ds_free[st]);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (n == 0 && !W.warp(&sm.acc_free, (n_units & 1) ^ 1)) { ok = false; break; }
      gi += n;
      if (ptx::elect_one()) {
        ptx::mma_commit(&sm.k_empty);
        ptx::mma_commit(&sm.acc_done);
      }
      __syncwarp();
      ++n_units;
    }
    (void)ok;
    __syncwarp();
    if (ptx::elect_one()) ptx::mma_commit(&sm.drain[side]);
    __syncwarp();
    if (lane == 0) W.drain(&sm.drain[side], 0);
    __syncwarp();
  } else if (warp < 8) {
    // ================================================================ compute warps
    const int qr = warp & 3, ch = warp >> 2;  // TMEM lane quarter, query-column half
    const int t = qr * 32 + lane;              // key row of S^T / dP^T
    const uint32_t lane_base = (uint32_t)(qr * 32) << 16;
    const float c = p.scale_log2;
    const int key_half = t >= 64 ? 1 : 0;
    uint32_t n_units = 0, i = 0;
    for (;;) {
      const int slot = n_units & 1;
      if (!group_all(W.warp(&sm.unit_full[slot], (n_units >> 1) & 1))) break;
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      const int g = un.head, k0 = un.tile * kTile, kj = k0 + t;
      // V of the unit into tensor memory (warp column half ch: head-dim columns
      // D/2 ch ..).  Its previous readers, the dP^T products of the previous
      // unit, completed before that unit's last dp_full, which this warp has seen.
      load_v_rows<D>(tmem + lane_base + kColV + (D / 4) * ch, t, (D / 2) * ch, p, si, g, k0);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.v_full);
      BwdSteps steps;
      steps.init(p, si.len, un.tile);
      int hh, qb, bits, n = 0;
      // A warp whose wait gave up skips the rest of the unit's steps but still
      // reaches the unit's group-wide agreement below, like every other warp.
      bool alive = true;
      while (steps.next(hh, qb, bits)) {
        const int st = i & 1, qs = i % kStages;
        const int q0 = qb * kQB;
        bool mine = alive && W.warp(&sm.qdo_full[qs], (i / kStages) & 1) && W.warp(&sm.st_full[st], (i >> 1) & 1);
        float pv[32];
        if (mine) {
          // P^T = exp2(S^T * scale * log2 e - LSE * log2 e) for 32 query columns
          ptx::tc_fence_after();
          uint32_t sr[32];
          ptx::tmem_ld32(tmem + lane_base + kColS + 32 * ch, sr);
          ptx::tmem_ld_wait();
          const bool need_mask = (k0 + kTile > si.len) || (elem_causal && q0 < k0 + kTile - 1) || bits != 3;
          // visible: key listed for this query block, inside the sequence and
          // (causal) not after the query: q0 + 32 ch + cc >= kj
          const bool row_ok = ((bits >> key_half) & 1) && kj < si.len;
          const int lo = elem_causal ? kj - q0 - 32 * ch : -1;
          uint32_t pk[16];
          const float2 c2 = make_float2(c, c);
          const float2* nl2 = reinterpret_cast<const float2*>(&sm.nlse2[qs][32 * ch]);
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[2 * w]), __uint_as_float(sr[2 * w + 1])), c2, nl2[w]);
            pv[2 * w] = fast_exp2(x.x);
            pv[2 * w + 1] = fast_exp2(x.y);
          }
          if (need_mask) {
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
              if (!(row_ok && cc >= lo)) pv[cc] = 0.f;
          }
#pragma unroll
          for (int w = 0; w < 16; ++w) pk[w] = ptx::pack_bf16x2(pv[2 * w], pv[2 * w + 1]);
          ptx::tmem_st16(tmem + lane_base + kColS + 32 * ch, pk);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.pt_full[st]);
          mine = W.warp(&sm.dp_full, i & 1);
        }
        if (mine) {
          ptx::tc_fence_after();
          uint32_t dr[32];
          ptx::tmem_ld32(tmem + lane_base + kColDP + 32 * ch, dr);
          ptx::tmem_ld_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.dp_free);
          mine = W.warp(&sm.ds_free[st], ((i >> 1) & 1) ^ 1);
          if (mine) {
            // dS^T = P^T o (dP^T - D), bf16, 128-byte swizzled row t of the dS^T tile
            uint8_t* dsrow = sm.ds[st] + t * 128;
            const float2* nd2 = reinterpret_cast<const float2*>(&sm.ndlt[qs][32 * ch]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float d[8];
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const int cc = j * 8 + e;
                const float2 t2 = __fadd2_rn(make_float2(__uint_as_float(dr[cc]), __uint_as_float(dr[cc + 1])), nd2[cc >> 1]);
                const float2 d2 = __fmul2_rn(make_float2(pv[cc], pv[cc + 1]), t2);
                d[e] = d2.x;
                d[e + 1] = d2.y;
              }
              uint4 o;
              o.x = ptx::pack_bf16x2(d[0], d[1]);
              o.y = ptx::pack_bf16x2(d[2], d[3]);
              o.z = ptx::pack_bf16x2(d[4], d[5]);
              o.w = ptx::pack_bf16x2(d[6], d[7]);
              const int chunk = 4 * ch + j;
              *reinterpret_cast<uint4*>(dsrow + ((chunk ^ (t & 7)) * 16)) = o;
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.ds_full[st]);
          }
        }
        alive = mine;
        (void)hh;
        ++i;
        ++n;
      }
      // unit epilogue: warps 0-3 write dK (x scale), warps 4-7 dV
      if (!group_all(alive && W.warp(&sm.acc_done, n_units & 1))) break;
      ptx::tc_fence_after();
      if (ch == 0) store_kv_rows<D>(tmem + lane_base + kColDK, n > 0, p.scale, t, p, si, g, k0, p.dk);
      else store_kv_rows<D>(tmem + lane_base + kColDV, n > 0, 1.f, t, p, si, g, k0, p.dv);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.acc_free);
      ++n_units;
    }
  } else if (warp >= 10 && warp < 14) {
    // ================================================================ dQ writers
    const int qr = warp & 3;
    const int d = qr * 32 + lane;  // head-dim column of dQ = TMEM lane of dQ^T
    const uint32_t lane_base = (uint32_t)(qr * 32) << 16;
    const bool issuer = warp == 10 && lane == 0;  // issues the reduce-adds
    uint32_t n_units = 0, i = 0;
    bool ok = true;
    for (;;) {
      const int slot = n_units & 1;
      if (!dq_all(W.warp(&sm.unit_full[slot], (n_units >> 1) & 1))) { ok = false; break; }
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      BwdSteps steps;
      steps.init(p, si.len, un.tile);
      int hh, qb, bits;
      while (kDq && steps.next(hh, qb, bits)) {
        // named barriers below: the four warps agree on the wait first
        if (!dq_all(W.warp(&sm.dq_full, i & 1))) { ok = false; break; }
        ptx::tc_fence_after();
        uint32_t v0[32], v1[32];
        ptx::tmem_ld32(tmem + lane_base + kColDQ, v0);
        ptx::tmem_ld32(tmem + lane_base + kColDQ + 32, v1);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.dq_free);
        if (issuer) ptx::bulk_wait_group_read<0>();  // the previous tile has left the staging buffer
        dq_sync();
        if (D == 128 || qr * 32 < D) {  // head-dim rows past D hold zeros (see above)
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) sm.dq[cc * D + d] = __uint_as_float(v0[cc]);
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) sm.dq[(32 + cc) * D + d] = __uint_as_float(v1[cc]);
        }
        ptx::fence_proxy_async_smem();
        dq_sync();
        if (issuer) {
          // rows past the sequence end carry exact zeros (their P is 0); the map
          // clips rows past the tensor end
          const int h = un.head * p.group + hh, q0 = qb * kQB;
          check_q_row(p, si, h, q0);
          if (a.acc_rows_inner) ptx::tma_reduce_add_4d(&a.tacc, sm.dq, 0, (int)(si.tok0 + q0), h, si.b);
          else ptx::tma_reduce_add_4d(&a.tacc, sm.dq, 0, h, (int)(si.tok0 + q0), 0);
          ptx::bulk_commit_group();
        }
        (void)bits;
        ++i;
      }
      if (!ok) break;
      ++n_units;
    }
    (void)ok;
    if (issuer) ptx::bulk_wait_group<0>();
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

cudaError_t launch_tc_bwd(const KParams& p, int sms, cudaStream_t st, bool with_dq) {
  if (p.n_units == 0) return cudaSuccess;
  BwdArgs a;
  TileMap mq, mk, mdo, macc;
  cudaError_t e;
  if ((e = make_tile_map(&mq, p.q, p, false, kQB)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mdo, p.dout, p, false, kQB)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mk, p.k, p, true)) != cudaSuccess) return e;
  if (with_dq && (e = make_acc_map(&macc, p.dq_accum, p, kQB)) != cudaSuccess) return e;
  if (!with_dq) std::memset(&macc, 0, sizeof(macc));
  a.tq = mq.map;
  a.tdo = mdo.map;
  a.tk = mk.map;
  a.tacc = macc.map;
  a.q_rows_inner = mq.rows_inner;
  a.kv_rows_inner = mk.rows_inner;
  a.acc_rows_inner = macc.rows_inner;
  a.p = p;
  const size_t smem = sizeof(Smem) + 1024;
  auto kernel = p.head_dim == 64 ? (with_dq ? k_tc_bwd<true, 64> : k_tc_bwd<false, 64>)
                                 : (with_dq ? k_tc_bwd<true, 128> : k_tc_bwd<false, 128>);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = p.n_units < sms ? p.n_units : sms;
  kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbattn
