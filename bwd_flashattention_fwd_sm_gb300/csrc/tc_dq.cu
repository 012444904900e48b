// Deterministic dQ on the fifth-generation tensor cores (sm_103a): a
// query-stationary pass, so every dQ row is one sum taken in a fixed order.
//
// The dK/dV-stationary backward reaches each dQ row from many key tiles, and
// the float32 adds land in whatever order the CTAs reach L2; the result is
// correct but its last bits vary from run to run (zwxr.cn CANN article,
// section 6.1, on accumulation order and precision).  The pages also name the
// way round it: loop over the query blocks on the outside and walk the key
// blocks inside, the other loop order of the two (smzdm contest article,
// section 03, on the backward's two loop directions).  This kernel does that
// for dQ alone; the dK/dV pass then skips its dQ product.
//
// Per 128-row query tile and key tile (three tcgen05 products, bf16 operands,
// float32 accumulation in tensor memory):
//   S  = Q K^T      dP = dO V^T      P = exp(S * scale - LSE)   (masked: 0)
//   dS = P o (dP - D)  (bf16, written to tensor memory)
//   dQ += dS K      (dS from tensor memory, K as an MN-major smem operand)
// and at the tile's end dQ * scale goes straight to global memory as bf16.
// Key tiles are walked in ascending order, so the sum order is fixed.
//
// Work distribution: the forward's work list (256 query rows per unit, longest
// first) and persistent CTAs that take units from an atomic counter; a unit's
// two 128-row tiles are done one after the other.
//
// Warp roles (320 threads):
//   warps 0-7  compute: warps w and w + 4 share TMEM lane quarter w mod 4
//              (query rows 32 (w mod 4) ..), warp w the keys [0, 64) of each
//              tile and warp w + 4 the keys [64, 128): P and dS need no row-wide
//              reduction (the forward's LSE fixes P), so the two halves of a
//              row are independent and a tile's elementwise work is split
//              over eight warps
//   warp 8     TMA producer and unit fetcher
//   warp 9     tensor-core issuer (whole warp; one elected lane issues)
// Every wait is bounded; a CTA that gives up records ATTN_ERR_DEVICE_TIMEOUT,
// drains its copies and tensor-core work, frees tensor memory and returns.
#include <cuda.h>

#include "tc_common.cuh"
#include "tc_kernels.h"
#include "tma_host.h"

namespace gbattn {

namespace {

// K is held until the tile's dQ product has read it, V only until dP has: K's
// ring is one stage deeper, so its next load starts a tile earlier (with two K
// stages the issuer waited about 1250 clocks per tile for K to arrive).
constexpr int kKStages = 3, kVStages = 2;
constexpr int kThreads = 320;
constexpr int kComputeWarps = 8;
constexpr uint32_t kTmemCols = 512;
// S [0,128)  dP [128,256)  dS (bf16 pairs) [256,320)  dQ [384,512)
constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 384;

struct DqArgs {
  CUtensorMap tq, tdo, tk, tv;
  int q_rows_inner, kv_rows_inner;
  KParams p;
};

struct Smem {
  uint8_t q[kTileBytes];
  uint8_t dO[kTileBytes];
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[kVStages][kTileBytes];
  uint64_t unit_full[2], unit_empty[2];
  uint64_t qd_full, qd_empty;
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t sdp_full, sdp_free, ds_full, ds_free, dq_final, dq_free, drain;
  int unit_slot[2][4];  // seq, head, 256-row tile, valid
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

// Key tiles of query tile q (0 or 1) of a 256-row unit that have visible keys.
template <bool kSparse>
__device__ __forceinline__ int count_active(const KParams& p, int len, int q0_unit, int q) {
  KvTileList2<kSparse> t;
  t.init(p, len, q0_unit);
  int kt, bits, n = 0;
  while (t.next(kt, bits)) n += ((bits >> (4 * q)) & 0xF) != 0;
  return n;
}

// D: head dim, 64 or 128 (shared memory is laid out for 128 either way).
template <bool kSparse, int D>
__global__ void __launch_bounds__(kThreads, 1) k_tc_dq(const __grid_constant__ DqArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KParams& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Waiter W{sm, p};

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sm.unit_full[i], 1);
      ptx::mbar_init(&sm.unit_empty[i], 1 + kComputeWarps);  // MMA warp + compute warps
    }
    ptx::mbar_init(&sm.qd_full, 1);
    ptx::mbar_init(&sm.qd_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      ptx::mbar_init(&sm.k_full[s], 1);
      ptx::mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      ptx::mbar_init(&sm.v_full[s], 1);
      ptx::mbar_init(&sm.v_empty[s], 1);
    }
    ptx::mbar_init(&sm.sdp_full, 1);
    ptx::mbar_init(&sm.sdp_free, kComputeWarps);
    ptx::mbar_init(&sm.ds_full, kComputeWarps);
    ptx::mbar_init(&sm.ds_free, 1);
    ptx::mbar_init(&sm.dq_final, 1);
    ptx::mbar_init(&sm.dq_free, kComputeWarps);
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

  if (warp == 8) {
    // ================================================================ producer
    uint32_t n_units = 0, n_qd = 0, n_kv = 0;
    int last_qd_phase = -1, last_k_phase[kKStages], last_v_phase[kVStages];
    for (int s = 0; s < kKStages; ++s) last_k_phase[s] = -1;
    for (int s = 0; s < kVStages; ++s) last_v_phase[s] = -1;
    bool ok = true;
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
        valid = check_unit(p, un, false, 2 * kTile);
      }
      if (lane == 0) {
        volatile int* s = sm.unit_slot[slot];
        s[0] = un.seq;
        s[1] = un.head;
        s[2] = un.tile;
        s[3] = valid ? 1 : 0;
        ptx::mbar_arrive(&sm.unit_full[slot]);
      }
      ++n_units;
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      const int h = un.head, g = h / p.group, q0u = un.tile * 2 * kTile;
      for (int q = 0; q < 2 && ok; ++q) {
        const int q0 = q0u + q * kTile;
        if (q0 >= si.len || count_active<kSparse>(p, si.len, q0u, q) == 0) continue;
        if (!W.warp(&sm.qd_empty, (n_qd & 1) ^ 1)) { ok = false; break; }
        if (lane == 0) {
          check_q_row(p, si, h, q0);
          ptx::mbar_arrive_expect_tx(&sm.qd_full, 2 * tile_bytes<D>());
          tma_tile(sm.q, &a.tq, a.q_rows_inner, &sm.qd_full, map_row(si, q0), h, si.b, kHalfTileBytes, D / 64);
          tma_tile(sm.dO, &a.tdo, a.q_rows_inner, &sm.qd_full, map_row(si, q0), h, si.b, kHalfTileBytes, D / 64);
        }
        last_qd_phase = (int)(n_qd & 1);
        ++n_qd;
        KvTileList2<kSparse> t;
        t.init(p, si.len, q0u);
        int kt, bits;
        while (t.next(kt, bits)) {
          if (!((bits >> (4 * q)) & 0xF)) continue;
          const int kst = n_kv % kKStages, vst = n_kv % kVStages;
          const uint32_t kph = (n_kv / kKStages) & 1, vph = (n_kv / kVStages) & 1;
          if (!W.warp(&sm.k_empty[kst], kph ^ 1) || !W.warp(&sm.v_empty[vst], vph ^ 1)) { ok = false; break; }
          if (lane == 0) {
            check_kv_row(p, si, g, kt * kTile);
            ptx::mbar_arrive_expect_tx(&sm.k_full[kst], tile_bytes<D>());
            tma_tile(sm.k[kst], &a.tk, a.kv_rows_inner, &sm.k_full[kst], map_row(si, kt * kTile), g, si.b,
                     kHalfTileBytes, D / 64);
            ptx::mbar_arrive_expect_tx(&sm.v_full[vst], tile_bytes<D>());
            tma_tile(sm.v[vst], &a.tv, a.kv_rows_inner, &sm.v_full[vst], map_row(si, kt * kTile), g, si.b,
                     kHalfTileBytes, D / 64);
          }
          last_k_phase[kst] = (int)kph;
          last_v_phase[vst] = (int)vph;
          ++n_kv;
        }
      }
      if (!ok) break;
    }
    // wait for this warp's own copies before the CTA may exit
    if (lane == 0) {
      if (last_qd_phase >= 0) W.drain(&sm.qd_full, (uint32_t)last_qd_phase);
      for (int s = 0; s < kKStages; ++s)
        if (last_k_phase[s] >= 0) W.drain(&sm.k_full[s], (uint32_t)last_k_phase[s]);
      for (int s = 0; s < kVStages; ++s)
        if (last_v_phase[s] >= 0) W.drain(&sm.v_full[s], (uint32_t)last_v_phase[s]);
    }
  } else if (warp == 9) {
    // ================================================================ MMA issuer
    // The whole warp runs the control flow; elect.sync on the full, converged
    // warp picks the same lane every time, so each commit covers every product
    // that lane issued before it.
    constexpr uint32_t idesc_ss = ptx::idesc_bf16(128, 128, false, false);  // S, dP
    constexpr uint32_t idesc_dq = ptx::idesc_bf16(128, D, false, true);     // dQ: B = K MN-major
    const uint32_t q_addr = ptx::smem_u32(sm.q), do_addr = ptx::smem_u32(sm.dO);
    uint32_t n_units = 0, n_qd = 0, n_kv = 0, n_sdp = 0, n_ds = 0, n_tiles = 0;
    bool ok = true;

    // dQ (+)= dS K of the key tile in stage st; first: the query tile's first product
    auto issue_dq = [&](int st, bool first) -> bool {
      if (!W.warp(&sm.ds_full, n_ds & 1)) return false;
      ++n_ds;
      // before the tile's first product, the previous tile's epilogue has read dQ
      if (first && !W.warp(&sm.dq_free, (n_tiles & 1) ^ 1)) return false;
      ptx::tc_fence_after();
      const uint32_t k_addr = ptx::smem_u32(sm.k[st]);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // B = K as (N = head dim, K = keys), head dim contiguous: MN-major
          const uint64_t bdesc = ptx::sdesc_sw128(k_addr + kk * 2048, kHalfTileBytes, 1024);
          ptx::mma_ts(tmem + kColDQ, tmem + kColDS + kk * 8, bdesc, idesc_dq, (first && kk == 0) ? 0u : 1u);
        }
        ptx::mma_commit(&sm.ds_free);
        ptx::mma_commit(&sm.k_empty[st]);
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
      ++n_units;
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      const int q0u = un.tile * 2 * kTile;
      for (int q = 0; q < 2 && ok; ++q) {
        const int q0 = q0u + q * kTile;
        if (q0 >= si.len) continue;
        const int n_act = count_active<kSparse>(p, si.len, q0u, q);
        if (n_act == 0) continue;
        KvTileList2<kSparse> t;
        t.init(p, si.len, q0u);
        int kt, bits, act = 0, prev_st = 0;
        while (t.next(kt, bits)) {
          if (!((bits >> (4 * q)) & 0xF)) continue;
          const int st = n_kv % kKStages, vst = n_kv % kVStages;
          if (!W.warp(&sm.k_full[st], (n_kv / kKStages) & 1) || !W.warp(&sm.v_full[vst], (n_kv / kVStages) & 1)) {
            ok = false;
            break;
          }
          ++n_kv;
          if (act == 0) {  // Q and dO of this query tile
            if (!W.warp(&sm.qd_full, n_qd & 1)) { ok = false; break; }
            ++n_qd;
          }
          // S and dP of the previous tile have been read by the compute warps
          if (n_sdp > 0 && !W.warp(&sm.sdp_free, (n_sdp - 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t k_addr = ptx::smem_u32(sm.k[st]), v_addr = ptx::smem_u32(sm.v[vst]);
          if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
              ptx::mma_ss(tmem + kColS, ptx::sdesc_sw128(q_addr + off, 16, 1024),
                          ptx::sdesc_sw128(k_addr + off, 16, 1024), idesc_ss, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
              ptx::mma_ss(tmem + kColDP, ptx::sdesc_sw128(do_addr + off, 16, 1024),
                          ptx::sdesc_sw128(v_addr + off, 16, 1024), idesc_ss, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(&sm.sdp_full);
            ptx::mma_commit(&sm.v_empty[vst]);
            if (act == n_act - 1) ptx::mma_commit(&sm.qd_empty);
          }
          __syncwarp();
          ++n_sdp;
          // the previous key tile's dQ product, now that this tile's S and dP are queued
          if (act > 0 && !issue_dq(prev_st, act == 1)) { ok = false; break; }
          prev_st = st;
          ++act;
        }
        if (!ok) break;
        if (!issue_dq(prev_st, act == 1)) { ok = false; break; }
        if (ptx::elect_one()) ptx::mma_commit(&sm.dq_final);
        __syncwarp();
        ++n_tiles;
      }
      if (!ok) break;
    }
    (void)ok;
    __syncwarp();
    if (ptx::elect_one()) ptx::mma_commit(&sm.drain);
    __syncwarp();
    if (lane == 0) W.drain(&sm.drain, 0);
    __syncwarp();
  } else if (warp < kComputeWarps) {
    // ================================================================ compute
    const int wq = warp & 3, hf = warp >> 2;  // TMEM lane quarter; key half of each tile
    const int r = wq * 32 + lane;             // query row in the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);
    const float c = p.scale_log2;
    const int row_half = r >= 64 ? 2 : 0;
    uint32_t n_units = 0, n_sdp = 0, n_ds = 0, n_tiles = 0;
    bool ok = true;
    for (;;) {
      const int slot = n_units & 1;
      if (!W.warp(&sm.unit_full[slot], (n_units >> 1) & 1)) { ok = false; break; }
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      ++n_units;
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      const int h = un.head, q0u = un.tile * 2 * kTile;
      for (int q = 0; q < 2 && ok; ++q) {
        const int q0 = q0u + q * kTile;
        if (q0 >= si.len) continue;
        const int qi = q0 + r;
        const bool row_ok = qi < si.len && check_q_row(p, si, h, qi);
        const int n_act = count_active<kSparse>(p, si.len, q0u, q);
        __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.dq) + (row_ok ? q_off(p, si, h, qi) : 0);
        if (n_act == 0) {  // no visible key: dQ rows are zero (each warp its half of the columns)
          if (row_ok) {
#pragma unroll
            for (int w = 0; w < D / 16; ++w)
              *reinterpret_cast<uint4*>(drow + hf * (D / 2) + w * 8) = make_uint4(0u, 0u, 0u, 0u);
          }
          continue;
        }
        // this row's -LSE log2(e) (-inf: no visible key or past the end) and -D
        float nl2 = -INFINITY, ndl = 0.f;
        if (row_ok) {
          const long long ri = row_index(p, si, h, qi);
          const float L = p.lse[ri];
          nl2 = L == -INFINITY ? -INFINITY : -L * 1.4426950408889634f;
          ndl = -p.delta[ri];
        }
        const float2 c2 = make_float2(c, c), nl22 = make_float2(nl2, nl2), nd2 = make_float2(ndl, ndl);
        KvTileList2<kSparse> t;
        t.init(p, si.len, q0u);
        int kt, bits8;
        while (t.next(kt, bits8)) {
          const int bits = (bits8 >> (4 * q)) & 0xF;
          if (!bits) continue;
          if (!W.warp(&sm.sdp_full, n_sdp & 1)) { ok = false; break; }
          ++n_sdp;
          ptx::tc_fence_after();
          const int k0 = kt * kTile;
          const bool need_mask = (k0 + kTile > si.len) || (elem_causal && k0 + kTile - 1 > q0) || bits != 0xF;
          int thr = si.len - k0;
          if (elem_causal) thr = min(thr, qi - k0 + 1);
          const bool lo_ok = (bits >> row_half) & 1, hi_ok = (bits >> (row_half + 1)) & 1;
          // dS = P o (dP - D) as bf16 pairs over this warp's 64 keys of the row
          const bool half_ok = hf == 0 ? lo_ok : hi_ok;
          uint32_t pk[32];
          {
            uint32_t sr[64], dr[64];
            ptx::tmem_ld32(tmem + lane_base + kColS + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            ptx::tmem_ld32(tmem + lane_base + kColS + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            ptx::tmem_ld32(tmem + lane_base + kColDP + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
            ptx::tmem_ld32(tmem + lane_base + kColDP + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
              const int k = hf * 64 + i;
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), c2, nl22);
              float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
              if (need_mask) {
                if (!(k < thr && half_ok)) pp.x = 0.f;
                if (!(k + 1 < thr && half_ok)) pp.y = 0.f;
              }
              const float2 t2 = __fadd2_rn(make_float2(__uint_as_float(dr[i]), __uint_as_float(dr[i + 1])), nd2);
              const float2 d2 = __fmul2_rn(pp, t2);
              pk[i / 2] = ptx::pack_bf16x2(d2.x, d2.y);
            }
          }
          // S and dP of this tile are in registers: the next tile's may overwrite them
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.sdp_free);
          // the previous tile's dQ product has read the dS buffer
          if (!W.warp(&sm.ds_free, (n_ds & 1) ^ 1)) { ok = false; break; }
          ++n_ds;
          ptx::tc_fence_after();
          ptx::tmem_st32(tmem + lane_base + kColDS + hf * 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.ds_full);
        }
        if (!ok) break;
        // epilogue: dQ * scale straight from tensor memory to global memory,
        // each of the row's two warps half of its columns
        if (!W.warp(&sm.dq_final, n_tiles & 1)) { ok = false; break; }
        ++n_tiles;
        ptx::tc_fence_after();
#pragma unroll
        for (int cc = hf * (D / 64); cc < (hf + 1) * (D / 64); ++cc) {
          uint32_t v[32];
          ptx::tmem_ld32(tmem + lane_base + kColDQ + cc * 32, v);
          ptx::tmem_ld_wait();
          if (row_ok) {
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              uint4 o;
              o.x = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 0]) * p.scale, __uint_as_float(v[w4 * 8 + 1]) * p.scale);
              o.y = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 2]) * p.scale, __uint_as_float(v[w4 * 8 + 3]) * p.scale);
              o.z = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 4]) * p.scale, __uint_as_float(v[w4 * 8 + 5]) * p.scale);
              o.w = ptx::pack_bf16x2(__uint_as_float(v[w4 * 8 + 6]) * p.scale, __uint_as_float(v[w4 * 8 + 7]) * p.scale);
              *reinterpret_cast<uint4*>(drow + cc * 32 + w4 * 8) = o;
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.dq_free);
      }
      if (!ok) break;
    }
    (void)ok;
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_tc_dq(const KParams& p, int sms, cudaStream_t st) {
  if (p.n_units == 0) return cudaSuccess;
  DqArgs a;
  TileMap mq, mdo, mk, mv;
  cudaError_t e;
  if ((e = make_tile_map(&mq, p.q, p, false)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mdo, p.dout, p, false)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mk, p.k, p, true)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mv, p.v, p, true)) != cudaSuccess) return e;
  a.tq = mq.map;
  a.tdo = mdo.map;
  a.tk = mk.map;
  a.tv = mv.map;
  a.q_rows_inner = mq.rows_inner;
  a.kv_rows_inner = mk.rows_inner;
  a.p = p;
  const size_t smem = sizeof(Smem) + 1024;
  const int grid = p.n_units < sms ? p.n_units : sms;
  auto kernel = p.head_dim == 64 ? (p.mask == kMaskBlock ? k_tc_dq<true, 64> : k_tc_dq<false, 64>)
                                 : (p.mask == kMaskBlock ? k_tc_dq<true, 128> : k_tc_dq<false, 128>);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbattn
