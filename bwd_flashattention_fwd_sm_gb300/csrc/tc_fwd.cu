// Forward attention on the fifth-generation tensor cores (sm_103a):
// persistent CTAs, two query tiles per CTA sharing every K/V tile.
//
// The method is the block-by-block attention of the zwxr.cn CANN ops-nn
// fused-attention article (sections 3.2-3.3): query blocks outside, key/value
// blocks streamed inside, a running max and sum correcting the softmax, the
// score matrix never leaving the chip (smzdm contest article, section 03).
//
// GB300 mapping.  A unit is 256 query rows of one head: two 128-row tiles Q0,
// Q1 whose S = Q K^T products share each K/V tile fetched by TMA.  Each query
// tile has its own softmax warpgroup, S buffer and O accumulator in tensor
// memory (S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512) columns; P_q is
// written back as bf16 over S_q and read by the P V product from tensor
// memory, so P never leaves the SM: zwxr.cn article, section 5.4).  The
// tensor core alternates between the two tiles: while warpgroup 0 turns S0
// into P0, the tensor core runs P1 V and the next Q1 K^T, and the other way
// round, so matrix work overlaps the exponentials.  At head dim 64 the O
// accumulators take half the columns and P_q gets its own (O0 [256,320) O1
// [320,384) P0 [384,448) P1 [448,512)): the next S_q is then issued as soon as
// the softmax has read S_q, and each softmax warpgroup runs tile after tile.
//
// Few units (fewer than the SMs): units of one 128-row query tile (kPair).
// Both slots then hold that tile; the key tiles it sees go to the two slots in
// turn, so each warpgroup keeps a partial (row max, row sum, O) over half of
// them, and at the end the second hands its max and sum to the first through
// shared memory, which merges the two halves and writes the rows.
//
// Work distribution.  CTAs are persistent (one per SM); the TMA warp takes the
// next unit from an atomic counter over the cost-ordered work list and hands
// it to the other roles through a two-slot ring in shared memory, so long
// units start first and no SM idles while work remains (zwxr.cn article,
// section 4.2: whoever finishes first takes the next block; smzdm article,
// section 02, on uneven work).
//
// Warp roles (384 threads):
//   warps 0-3 / 4-7  softmax for query tile 0 / 1: thread r owns row r (the
//                    whole 128-column S row in registers; max and sum in 8
//                    independent partials to keep dependency chains short)
//   warp 8           TMA producer and unit fetcher
//   warps 9 / 10     tensor-core issuers for query tile 0 / 1 (each waits on
//                    its own tile's barriers while the other's products run)
//   warp 11          idle (it completes the third warpgroup, whose registers
//                    the softmax warpgroups borrow)
// Every wait is bounded; a CTA that gives up records ATTN_ERR_DEVICE_TIMEOUT,
// drains its copies and tensor-core work, frees tensor memory and returns.
#include <cuda.h>

#include "fp8.h"
#include "tc_common.cuh"
#include "tc_kernels.h"
#include "tma_host.h"

namespace gbattn {

namespace {

constexpr int kThreads = 384;  // three full warpgroups
// Register split: launched at 168 per thread (384 x 168 = 64512 registers); the
// two softmax warpgroups raise theirs, the producer/issuer warpgroup lowers its:
// 256 x 192 + 128 x 112 = 256 x 200 + 128 x 96 = 63488 <= 64512.  Dense and
// causal units take 192 / 112 (at 96 the issuers' loop spills); block-sparse
// units, whose tile lists hold more state in the softmax, 200 / 96.
template <bool kSparse>
struct RegSplit {
  static constexpr uint32_t kSoftmax = 192, kControl = 112;
};
template <>
struct RegSplit<true> {
  static constexpr uint32_t kSoftmax = 200, kControl = 96;
};

// Shared-memory tile size and ring depths: bf16 tiles are 32 KiB (two Q tiles,
// K and V rings), e4m3 tiles 16 KiB, so the FP8 rings are twice as deep in less
// space.
template <bool kFp8>
struct FwdCfg {
  static constexpr uint32_t kTileB = kTileBytes;
  static constexpr int kKStages = 2, kVStages = 2;
};
template <>
struct FwdCfg<true> {
  static constexpr uint32_t kTileB = (uint32_t)kTile * 128;
  static constexpr int kKStages = 4, kVStages = 4;
};
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the row max grows by more than 2^8
constexpr uint32_t kTmemCols = 512;

struct FwdArgs {
  CUtensorMap tq, tk, tv;
  int q_rows_inner, kv_rows_inner;
  KParams p;
  // FP8 operands: per-tile scales [batch, heads, n_tiles] of Q, K, V
  const float* qs;
  const float* ks;
  const float* vs;
  int n_tiles;
};

template <class C>
struct Smem {
  static constexpr int kKStages = C::kKStages, kVStages = C::kVStages;
  uint8_t q[2][C::kTileB];
  uint8_t k[kKStages][C::kTileB];
  uint8_t v[kVStages][C::kTileB];
  uint64_t unit_full[2], unit_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kKStages], v_full[kVStages], k_empty[kKStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2], o_final[2], o_free[2];
  uint64_t turn[2];  // turn[q]: issuer q has issued its products for a key tile
  uint64_t drain[2];
  int unit_slot[2][4];  // seq, head, 256-row tile, valid
  uint32_t tmem_base;
  ptx::Abort abort;
  // 128-row units: the second softmax warpgroup's row max and sum for the
  // first, which merges the two halves of the key range
  uint64_t pair_full, pair_free;
  float pair_m[kTile], pair_l[kTile];
  int pair_have;
  // head dim 64 (P in its own columns): s_free[q], the softmax has read S_q;
  // pv_done[q], the P_q V product has finished
  uint64_t s_free[2], pv_done[2];
};

static_assert(sizeof(Smem<FwdCfg<false>>) + 1024 <= 232448, "shared memory per CTA is at most 227 KiB");
static_assert(sizeof(Smem<FwdCfg<true>>) + 1024 <= 232448, "shared memory per CTA is at most 227 KiB");

template <class SM>
struct Waiter {
  SM& sm;
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

// Reads unit slot `u` (after its full barrier); false for the end sentinel.
// Slot word 3 is 0 for the sentinel, else 1 + the unit's part of a split key
// range (returned in un.cost; 0 when the range is not split).
template <class SM>
__device__ __forceinline__ bool read_unit(const SM& sm, int slot, Unit& un) {
  const volatile int* s = sm.unit_slot[slot];
  un.seq = s[0];
  un.head = s[1];
  un.tile = s[2];
  un.cost = s[3] > 0 ? s[3] - 1 : 0;
  return s[3] != 0;
}

// The key tiles of a unit that one part of a split forward takes: entries
// [lo, hi) of the unit's tile list, cut into p.n_split near-equal runs (dense
// and causal lists, of n_dense entries; no split: the whole list).  Every role
// walks the same entries, so the pipeline's rings stay in step.
//
// kPair (128-row units): the unit owns one of the two query tiles (keep: its
// bits, 0x0F for tile 0 or 0xF0 for tile 1).  Key tiles without its bits are
// skipped, and the kept ones alternate between the two slots (bits 0-3, then
// 4-7, ...), so that the CTA's two halves split the tile's key range.
template <bool kSparse, bool kPair = false>
struct PartList {
  KvTileList2<kSparse> t;
  int e, lo, hi;
  __device__ void init(const KParams& p, int len, int q0, int part, int = 0xFF) {
    t.init(p, len, q0);
    e = 0;
    lo = 0;
    hi = INT_MAX;
    if constexpr (!kSparse) {
      if (p.n_split > 1) {
        lo = part * t.n_dense / p.n_split;
        hi = (part + 1) * t.n_dense / p.n_split;
      }
    }
  }
  __device__ bool next(int& kt, int& bits) {
    while (e < hi && t.next(kt, bits))
      if (e++ >= lo) return true;
    return false;
  }
};
template <bool kSparse>
struct PartList<kSparse, true> {
  KvTileList2<kSparse> t;
  int keep, kept;
  __device__ void init(const KParams& p, int len, int q0, int, int keep_) {
    t.init(p, len, q0);
    keep = keep_;
    kept = 0;
  }
  __device__ bool next(int& kt, int& bits) {
    while (t.next(kt, bits)) {
      const int nib = (bits & keep) >> (keep == 0xF0 ? 4 : 0);
      if (nib == 0) continue;
      bits = nib << (4 * (kept++ & 1));
      return true;
    }
    return false;
  }
};

// The rows of a forward unit: the first row of its 256-row pair of query tiles
// and the bits of the tiles it owns (both; with 128-row units one, whose key
// tiles the two halves of the CTA then share, see PartList).
struct UnitRows {
  int q0, keep;
};
template <bool kPair>
__device__ __forceinline__ UnitRows unit_rows(const Unit& un) {
  if constexpr (kPair) return UnitRows{(un.tile >> 1) * 2 * kTile, (un.tile & 1) ? 0xF0 : 0x0F};
  return UnitRows{un.tile * 2 * kTile, 0xFF};
}
// First row of the query rows of slot q (with 128-row units both slots hold
// the unit's one tile).
template <bool kPair>
__device__ __forceinline__ int slot_row(const Unit& un, int q) {
  return kPair ? un.tile * kTile : un.tile * 2 * kTile + q * kTile;
}

// Stores P = 0 over eight tensor-memory columns (a 64-key half that no row of
// the warp sees: nothing of it is read or exponentiated).
__device__ __forceinline__ void zero_p8(uint32_t taddr) {
  uint32_t z[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) z[i] = 0u;
  ptx::tmem_st8(taddr, z);
}

// P = exp2(s * c - mu) for one 128-key row (two elements per packed FFMA2 /
// FADD2), rounded to bf16 pairs and stored to tensor memory at `taddr` 8
// columns at a time; keys at or past the visibility threshold get P = 0 when
// kMask.  kHalf (block-sparse): the 64-key halves the row's block does not list
// (lo_ok / hi_ok false, the same for the whole warp) are written as zeros
// without reading S.  Returns the row sum of the float32 P values.
template <bool kMask, bool kHalf>
__device__ __forceinline__ float write_p(const uint32_t (&sr)[128], float c, float mu, int thr, bool lo_ok,
                                         bool hi_ok, uint32_t taddr);

// The P of keys [K0, K0 + 64) of one row (see write_p), accumulated into rs2.
template <bool kMask, int K0>
__device__ __forceinline__ void write_p_half(const uint32_t (&sr)[128], float2 c2, float2 nmu2, int thr,
                                             uint32_t taddr, float2 (&rs2)[2]) {
#pragma unroll
  for (int cc = K0 / 16; cc < K0 / 16 + 4; ++cc) {
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = cc * 16 + 2 * i;
      const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nmu2);
      float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
      if constexpr (kMask) {
        if (!(k < thr)) pp.x = 0.f;
        if (!(k + 1 < thr)) pp.y = 0.f;
      }
      rs2[i & 1] = __fadd2_rn(rs2[i & 1], pp);
      pk[i] = ptx::pack_bf16x2(pp.x, pp.y);
    }
    ptx::tmem_st8(taddr + cc * 8, pk);
  }
}

template <bool kMask, bool kHalf>
__device__ __forceinline__ float write_p(const uint32_t (&sr)[128], float c, float mu, int thr, bool lo_ok,
                                         bool hi_ok, uint32_t taddr) {
  const float2 c2 = make_float2(c, c), nmu2 = make_float2(-mu, -mu);
  float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  if constexpr (kHalf) {
    // Block-sparse: lo_ok and hi_ok are the same for the whole warp, so each
    // half is one straight run of exponentials (or of zeros), decided once.
    if (lo_ok) {
      write_p_half<kMask, 0>(sr, c2, nmu2, thr, taddr, rs2);
    } else {
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) zero_p8(taddr + cc * 8);
    }
    if (hi_ok) {
      write_p_half<kMask, 64>(sr, c2, nmu2, thr, taddr, rs2);
    } else {
#pragma unroll
      for (int cc = 4; cc < 8; ++cc) zero_p8(taddr + cc * 8);
    }
    return (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
  } else {
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = cc * 16 + 2 * i;
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nmu2);
        float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        if constexpr (kMask) {
          if (!(k < thr)) pp.x = 0.f;
          if (!(k + 1 < thr)) pp.y = 0.f;
        }
        rs2[i & 1] = __fadd2_rn(rs2[i & 1], pp);
        pk[i] = ptx::pack_bf16x2(pp.x, pp.y);
      }
      ptx::tmem_st8(taddr + cc * 8, pk);
    }
    return (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
  }
}

// The FP8 form of write_p: P-hat = exp2(s * c - mu) rounded to e4m3 (mu also
// carries the V tile's scale ratio, so P-hat stays below 2^8 < 448), four keys
// per 32-bit column (key 4i + b in byte b), stored 8 columns = 32 keys at a time.
// Masks as write_p.  Returns the row sum of the float32 P-hat values.
template <bool kMask, bool kHalf>
__device__ __forceinline__ float write_p8(const uint32_t (&sr)[128], float c, float mu, int thr, bool lo_ok,
                                          bool hi_ok, uint32_t taddr) {
  const float2 c2 = make_float2(c, c), nmu2 = make_float2(-mu, -mu);
  float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    if constexpr (kHalf) {
      if (!(cc < 2 ? lo_ok : hi_ok)) {
        zero_p8(taddr + cc * 8);
        continue;
      }
    }
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = cc * 32 + 4 * i;
      const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nmu2);
      const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3])), c2, nmu2);
      float2 p0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
      float2 p1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
      if constexpr (kMask) {
        if (!(k < thr)) p0.x = 0.f;
        if (!(k + 1 < thr)) p0.y = 0.f;
        if (!(k + 2 < thr)) p1.x = 0.f;
        if (!(k + 3 < thr)) p1.y = 0.f;
      }
      rs2[0] = __fadd2_rn(rs2[0], p0);
      rs2[1] = __fadd2_rn(rs2[1], p1);
      pk[i] = ptx::pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
    }
    ptx::tmem_st8(taddr + cc * 8, pk);
  }
  return (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
}

// D: head dim, 64 or 128 (shared memory is laid out for 128 either way).
// kFp8: e4m3 operands (D = 128): Q and K tiles of 128 rows x 128 bytes, V
// transposed (128 head-dim rows x 128 keys), both products kind::f8f6f4 with
// K = 32 per instruction; P rounded to e4m3 into tensor memory; per-tile scales
// folded into the softmax constant (Q and K) and into P (V, relative to the
// head's largest V scale, which multiplies O in the epilogue).
template <bool kSparse, int D, bool kFp8, bool kPair = false>
__global__ void __launch_bounds__(kThreads, 1) k_tc_fwd(const __grid_constant__ FwdArgs a) {
  using SM = Smem<FwdCfg<kFp8>>;
  constexpr int kKStages = SM::kKStages, kVStages = SM::kVStages;
  extern __shared__ uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KParams& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Waiter<SM> W{sm, p};
  static_assert(!kFp8 || D == 128, "the FP8 forward has head dim 128");
  static_assert(!kPair || (!kSparse && !kFp8), "128-row units: dense and causal bf16 only");
  // At head dim 64 the O accumulators take 128 columns, so P_q gets columns of
  // its own ([384, 448) and [448, 512)) instead of S_q's: the next S_q can then
  // be issued as soon as the softmax holds this S_q in registers, and each
  // softmax warpgroup runs tile after tile without waiting for its own P V and
  // S products.
  constexpr bool kSepP = D == 64 && !kFp8;
  constexpr uint32_t kLoadBytes = kFp8 ? (uint32_t)kTile * 128 : tile_bytes<D>();

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sm.unit_full[i], 1);
      ptx::mbar_init(&sm.unit_empty[i], 10);  // 2 MMA warps + 8 softmax warps
      ptx::mbar_init(&sm.q_full[i], 1);
      ptx::mbar_init(&sm.q_empty[i], 1);
      ptx::mbar_init(&sm.s_full[i], 1);
      ptx::mbar_init(&sm.p_full[i], 4);
      ptx::mbar_init(&sm.o_final[i], 1);
      ptx::mbar_init(&sm.o_free[i], 4);
    }
    for (int s = 0; s < kKStages; ++s) {
      ptx::mbar_init(&sm.k_full[s], 1);
      ptx::mbar_init(&sm.k_empty[s], 2);  // one commit per MMA warp
    }
    for (int s = 0; s < kVStages; ++s) {
      ptx::mbar_init(&sm.v_full[s], 1);
      ptx::mbar_init(&sm.v_empty[s], 2);
    }
    ptx::mbar_init(&sm.turn[0], 1);
    ptx::mbar_init(&sm.turn[1], 1);
    ptx::mbar_init(&sm.drain[0], 1);
    ptx::mbar_init(&sm.drain[1], 1);
    if constexpr (kPair) {
      ptx::mbar_init(&sm.pair_full, 4);  // the second warpgroup's warps
      ptx::mbar_init(&sm.pair_free, 4);  // the first warpgroup's warps
    }
    if constexpr (kSepP) {
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(&sm.s_free[i], 4);  // the softmax warpgroup's warps
        ptx::mbar_init(&sm.pv_done[i], 1);
      }
    }
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
  if (warp >= 8) ptx::regs_decrease<RegSplit<kSparse>::kControl>();
  if (warp == 8) {
    // ================================================================ producer
    uint32_t n_units_seen = 0, n_q_loads[2] = {0, 0}, n_k = 0, n_v = 0;
    int last_q_phase[2] = {-1, -1}, last_k_phase[kKStages], last_v_phase[kVStages];
    for (int s = 0; s < kKStages; ++s) last_k_phase[s] = -1;
    for (int s = 0; s < kVStages; ++s) last_v_phase[s] = -1;
    bool ok = true;
    for (;;) {
      const int slot = n_units_seen & 1;
      // claim the slot (its previous unit has been read by every role)
      if (!W.warp(&sm.unit_empty[slot], ((n_units_seen >> 1) & 1) ^ 1)) { ok = false; break; }
      int idx = 0;
      if (lane == 0) idx = atomicAdd(p.unit_counter, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      bool valid = idx < p.n_units;
      Unit un{0, 0, 0, 0};
      if (valid) {
        un = p.units[idx];
        valid = check_unit(p, un, false, kPair ? kTile : 2 * kTile);
      }
      if (lane == 0) {
        volatile int* s = sm.unit_slot[slot];
        s[0] = un.seq;
        s[1] = un.head;
        s[2] = un.tile;
        s[3] = valid ? 1 + (p.n_split > 1 ? un.cost : 0) : 0;
        ptx::mbar_arrive(&sm.unit_full[slot]);
      }
      ++n_units_seen;
      if (!valid) break;

      const SeqInfo si = seq_info(p, un.seq);
      const UnitRows ur = unit_rows<kPair>(un);
      const int h = un.head, g = h / p.group, q0 = ur.q0;
      // which query tiles have work, for the Q loads
      bool act[2] = {false, false};
      const int part = p.n_split > 1 ? un.cost : 0;
      {
        PartList<kSparse, kPair> t;
        t.init(p, si.len, q0, part, ur.keep);
        int kt, bits;
        while (t.next(kt, bits)) {
          act[0] |= (bits & 0xF) != 0;
          act[1] |= (bits & 0xF0) != 0;
        }
      }
      for (int q = 0; q < 2 && ok; ++q) {
        if (!act[q]) continue;
        const uint32_t c = n_q_loads[q];
        if (!W.warp(&sm.q_empty[q], ((c & 1) ^ 1))) { ok = false; break; }
        if (lane == 0) {
          const int qr0 = slot_row<kPair>(un, q);
          check_q_row(p, si, h, qr0);
          ptx::mbar_arrive_expect_tx(&sm.q_full[q], kLoadBytes);
          if constexpr (kFp8)
            ptx::tma_load_4d(sm.q[q], &a.tq, &sm.q_full[q], 0, qr0, h, si.b);
          else
            tma_tile(sm.q[q], &a.tq, a.q_rows_inner, &sm.q_full[q], map_row(si, qr0), h, si.b, kHalfTileBytes,
                     D / 64);
        }
        last_q_phase[q] = c & 1;
        ++n_q_loads[q];
      }
      if (!ok) break;
      // K runs one tile ahead of V: K is released as soon as the S products of
      // its tile are done, V only after the P V products, so loading K(j+1)
      // before V(j) gives it the longest lead.
      auto load_k = [&](int kt_) -> bool {
        const int st = n_k % kKStages;
        const uint32_t ph = (n_k / kKStages) & 1;
        if (!W.warp(&sm.k_empty[st], ph ^ 1)) return false;
        if (lane == 0) {
          check_kv_row(p, si, g, kt_ * kTile);
          ptx::mbar_arrive_expect_tx(&sm.k_full[st], kLoadBytes);
          if constexpr (kFp8)
            ptx::tma_load_4d(sm.k[st], &a.tk, &sm.k_full[st], 0, kt_ * kTile, g, si.b);
          else
            tma_tile(sm.k[st], &a.tk, a.kv_rows_inner, &sm.k_full[st], map_row(si, kt_ * kTile), g, si.b,
                     kHalfTileBytes, D / 64);
        }
        last_k_phase[st] = (int)ph;
        ++n_k;
        return true;
      };
      auto load_v = [&](int kt_) -> bool {
        const int st = n_v % kVStages;
        const uint32_t ph = (n_v / kVStages) & 1;
        if (!W.warp(&sm.v_empty[st], ph ^ 1)) return false;
        if (lane == 0) {
          check_kv_row(p, si, g, kt_ * kTile);
          ptx::mbar_arrive_expect_tx(&sm.v_full[st], kLoadBytes);
          if constexpr (kFp8)  // V transposed: keys along x, head dim along y
            ptx::tma_load_4d(sm.v[st], &a.tv, &sm.v_full[st], kt_ * kTile, 0, g, si.b);
          else
            tma_tile(sm.v[st], &a.tv, a.kv_rows_inner, &sm.v_full[st], map_row(si, kt_ * kTile), g, si.b,
                     kHalfTileBytes, D / 64);
        }
        last_v_phase[st] = (int)ph;
        ++n_v;
        return true;
      };
      // K(j) then V(j): the first P V product, which the next tile's S waits
      // behind, needs V(0) before K(1)
      PartList<kSparse, kPair> t;
      t.init(p, si.len, q0, part, ur.keep);
      int kt, bits;
      while (t.next(kt, bits)) {
        if (!load_k(kt) || !load_v(kt)) { ok = false; break; }
      }
      if (!ok) break;
    }
    (void)ok;
    if (lane == 0) {
      for (int q = 0; q < 2; ++q)
        if (last_q_phase[q] >= 0) W.drain(&sm.q_full[q], (uint32_t)last_q_phase[q]);
      for (int s = 0; s < kKStages; ++s)
        if (last_k_phase[s] >= 0) W.drain(&sm.k_full[s], (uint32_t)last_k_phase[s]);
      for (int s = 0; s < kVStages; ++s)
        if (last_v_phase[s] >= 0) W.drain(&sm.v_full[s], (uint32_t)last_v_phase[s]);
    }
  } else if (warp == 9 || warp == 10) {
    // ================================================================ MMA issuers
    // Warp 9 + q issues the products of query tile q: S_q = Q_q K^T and
    // O_q += P_q V.  Each tcgen05.mma holds its issuing thread until the tensor
    // core takes it, so a single issuer's barrier waits left the tensor core
    // idle; with one issuer per tile, one waits while the other's products run.
    // Both issuers walk every key tile of the unit and commit once per K / V
    // stage (the empty barriers count two), so the ring stays in step even for
    // tiles where one query tile has no visible keys.
    // Per key tile the two issuers take turns (tile 0's products, then tile
    // 1's, ...): left free-running, both warpgroups drift into the same phase,
    // their products interleave and each waits for both; taking turns keeps one
    // warpgroup's exponentials under the other's products.
    // The whole warp runs the control flow; elect.sync on the full, converged
    // warp picks the same lane every time, so each commit covers every product
    // that lane issued before it.
    const int q = warp - 9;
    constexpr uint32_t idesc_s = kFp8 ? ptx::idesc_e4m3(128, 128) : ptx::idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_pv = kFp8 ? ptx::idesc_e4m3(128, D) : ptx::idesc_bf16(128, D, false, true);
    const uint32_t q_addr = ptx::smem_u32(sm.q[q]);
    const uint32_t t_s = tmem + q * 128, t_o = tmem + 256 + q * D;
    const uint32_t t_p = kSepP ? tmem + 384 + q * 64 : t_s;  // P_q, the A operand of P_q V
    uint32_t n_units_seen = 0, n_q = 0, n_p = 0, n_o = 0, n_k = 0, n_v = 0;
    uint32_t n_si = 0;  // S_q products issued (all units)
    uint32_t n_turn = 0;  // key tiles walked so far (all units)
    bool ok = true;
    for (;;) {
      const int slot = n_units_seen & 1;
      if (!W.warp(&sm.unit_full[slot], (n_units_seen >> 1) & 1)) { ok = false; break; }
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      ++n_units_seen;
      if (!valid) break;

      const SeqInfo si = seq_info(p, un.seq);
      const UnitRows ur = unit_rows<kPair>(un);
      PartList<kSparse, kPair> tl;
      tl.init(p, si.len, ur.q0, un.cost, ur.keep);
      int n_act = 0;
      {
        PartList<kSparse, kPair> t = tl;
        int kt, bits;
        while (t.next(kt, bits)) n_act += ((bits >> (4 * q)) & 0xF) != 0;
      }
      int s_issued = 0, pv_issued = 0;
      // S_q = Q_q K^T into S_q; after the unit's last one, Q_q may be refilled.
      auto issue_s = [&](uint32_t k_addr) -> bool {
        if constexpr (kSepP) {  // the softmax has read the previous S_q
          if (n_si > 0 && !W.warp(&sm.s_free[q], (n_si - 1) & 1)) return false;
          ++n_si;
        }
        if (s_issued == 0) {
          if (!W.warp(&sm.q_full[q], n_q & 1)) return false;
          ++n_q;
          ptx::tc_fence_after();
        }
        const bool last = ++s_issued == n_act;
        if (ptx::elect_one()) {
          if constexpr (kFp8) {
            // one 128-byte row per position: four K-steps of 32 bytes
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_ss_f8(t_s, ptx::sdesc_sw128(q_addr + kk * 32, 16, 1024),
                             ptx::sdesc_sw128(k_addr + kk * 32, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
              ptx::mma_ss(t_s, ptx::sdesc_sw128(q_addr + off, 16, 1024), ptx::sdesc_sw128(k_addr + off, 16, 1024),
                          idesc_s, kk > 0 ? 1u : 0u);
            }
          }
          ptx::mma_commit(&sm.s_full[q]);
          if (last) ptx::mma_commit(&sm.q_empty[q]);
        }
        __syncwarp();
        return true;
      };

      // O_q += P_q V (V from stage vst_); the unit's last one frees O_q for the epilogue.
      auto issue_pv = [&](uint32_t vst_) {
        ptx::tc_fence_after();
        const uint32_t v_addr = ptx::smem_u32(sm.v[vst_]);
        const uint32_t acc0 = pv_issued > 0 ? 1u : 0u;
        const bool last = ++pv_issued == n_act;
        if (ptx::elect_one()) {
          if constexpr (kFp8) {
            // B = V^T as (N = head dim, K = keys), keys contiguous: K-major;
            // A = P, 32 keys per 8 tensor-memory columns
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_ts_f8(t_o, t_p + kk * 8, ptx::sdesc_sw128(v_addr + kk * 32, 16, 1024), idesc_pv,
                             kk > 0 ? 1u : acc0);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // B = V as (N = head dim, K = keys), head dim contiguous: MN-major.
              const uint64_t bdesc = ptx::sdesc_sw128(v_addr + kk * 2048, kHalfTileBytes, 1024);
              ptx::mma_ts(t_o, t_p + kk * 8, bdesc, idesc_pv, kk > 0 ? 1u : acc0);
            }
          }
          if constexpr (kSepP) ptx::mma_commit(&sm.pv_done[q]);
          if (last) ptx::mma_commit(&sm.o_final[q]);
        }
        __syncwarp();
        if (last) ++n_o;
      };

      PartList<kSparse, kPair> t = tl;
      int kt, bits;
      bool have = t.next(kt, bits);
      uint32_t cur_stage = 0;
      int cur_bits = bits;
      if (have) {  // prologue: S of the first tile
        cur_stage = n_k % kKStages;
        if (!W.warp(&sm.k_full[cur_stage], (n_k / kKStages) & 1)) { ok = false; break; }
        ++n_k;
        ptx::tc_fence_after();
        if ((bits >> (4 * q)) & 0xF) ok = issue_s(ptx::smem_u32(sm.k[cur_stage]));
        if (!ok) break;
        // K of tile 0 is free once its S products are done
        if (ptx::elect_one()) ptx::mma_commit(&sm.k_empty[cur_stage]);
        __syncwarp();
      }
      while (have) {
        int nkt, nbits = 0;
        const bool nhave = t.next(nkt, nbits);
        const uint32_t nst = n_k % kKStages, vst = n_v % kVStages;
        if constexpr (kSepP) {
          // S_q of the next tile first: issue_s waits only until the softmax has
          // read this tile's S_q; then this tile's P_q V once P_q is written.
          // The issuers do not take turns: each softmax warpgroup runs on as
          // soon as its next S_q is there.
          if (nhave) {
            if (!W.warp(&sm.k_full[nst], (n_k / kKStages) & 1)) { ok = false; break; }
            ++n_k;
            if ((nbits >> (4 * q)) & 0xF) {
              ptx::tc_fence_after();
              if (!issue_s(ptx::smem_u32(sm.k[nst]))) { ok = false; break; }
            }
            if (ptx::elect_one()) ptx::mma_commit(&sm.k_empty[nst]);  // this warp's S product issued
            __syncwarp();
          }
          if (!W.warp(&sm.v_full[vst], (n_v / kVStages) & 1)) { ok = false; break; }
          ++n_v;
          if ((cur_bits >> (4 * q)) & 0xF) {
            if (!W.warp(&sm.p_full[q], n_p & 1)) { ok = false; break; }
            ++n_p;
            if (pv_issued == 0 && !W.warp(&sm.o_free[q], (n_o & 1) ^ 1)) { ok = false; break; }
            issue_pv(vst);
          }
          if (ptx::elect_one()) ptx::mma_commit(&sm.v_empty[vst]);  // this warp's P V product issued
          __syncwarp();
          have = nhave;
          cur_bits = nbits;
          cur_stage = nst;
          continue;
        }
        if (!W.warp(&sm.v_full[vst], (n_v / kVStages) & 1)) { ok = false; break; }
        ++n_v;
        // K of the next tile is waited for before P_q: it is normally there long
        // before P_q, so the wait stays off the softmax -> products -> softmax chain.
        if (nhave) {
          if (!W.warp(&sm.k_full[nst], (n_k / kKStages) & 1)) { ok = false; break; }
          ++n_k;
        }
        if ((cur_bits >> (4 * q)) & 0xF) {
          // O_q += P_q V.  Before the unit's first product, the previous unit's
          // epilogue must have read O_q.
          if (!W.warp(&sm.p_full[q], n_p & 1)) { ok = false; break; }
          ++n_p;
          if (pv_issued == 0 && !W.warp(&sm.o_free[q], (n_o & 1) ^ 1)) { ok = false; break; }
        }
        // this tile's turn: issuer 0 after issuer 1's previous tile, issuer 1
        // after issuer 0's same tile
        if (q == 0 ? (n_turn > 0 && !W.warp(&sm.turn[1], (n_turn - 1) & 1)) : !W.warp(&sm.turn[0], n_turn & 1)) {
          ok = false;
          break;
        }
        if ((cur_bits >> (4 * q)) & 0xF) issue_pv(vst);
        // S_q of the next tile: the S_q buffer held P_q, consumed by the product above
        if (nhave && ((nbits >> (4 * q)) & 0xF)) {
          ptx::tc_fence_after();
          if (!issue_s(ptx::smem_u32(sm.k[nst]))) { ok = false; break; }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.turn[q]);  // hand the turn to the other issuer
        ++n_turn;
        if (ptx::elect_one()) {
          ptx::mma_commit(&sm.v_empty[vst]);             // V of this tile: this warp's P V product issued
          if (nhave) ptx::mma_commit(&sm.k_empty[nst]);  // K of the next tile: this warp's S product issued
        }
        __syncwarp();
        have = nhave;
        cur_bits = nbits;
        cur_stage = nst;
      }
      if (!ok) break;
    }
    (void)ok;
    __syncwarp();
    if (ptx::elect_one()) ptx::mma_commit(&sm.drain[q]);
    __syncwarp();
    if (lane == 0) W.drain(&sm.drain[q], 0);
    __syncwarp();
  } else if (warp < 8) {
    // ================================================================ softmax
    ptx::regs_increase<RegSplit<kSparse>::kSoftmax>();
    const int q = warp >> 2;          // query tile of this warpgroup
    const int wq = warp & 3;          // warp within the group = TMEM lane quarter
    const int r = wq * 32 + lane;     // row in the query tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t col_s = q * 128, col_o = 256 + q * D;
    const uint32_t col_p = kSepP ? 384 + q * 64 : col_s;  // where P_q is written
    const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);
    const float c = p.scale_log2;
    const int row_half = r >= 64 ? 2 : 0;
    uint32_t n_units_seen = 0, n_s = 0, n_o = 0, n_pair = 0;
    uint32_t n_pw = 0;  // P_q tiles written (all units)
    bool ok = true;
    for (;;) {
      const int slot = n_units_seen & 1;
      if (!W.warp(&sm.unit_full[slot], (n_units_seen >> 1) & 1)) { ok = false; break; }
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      ++n_units_seen;
      if (!valid) break;

      const SeqInfo si = seq_info(p, un.seq);
      const int h = un.head;
      const UnitRows ur = unit_rows<kPair>(un);
      const int q0 = slot_row<kPair>(un, q);  // this tile's first row
      const int qi = q0 + r;
      float m_used = -INFINITY, l = 0.f;
      // FP8: this Q tile's scale and the KV head's largest V tile scale
      float sq = 1.f, sv_ref = 1.f;
      const float *ks_row = nullptr, *vs_row = nullptr;
      if constexpr (kFp8) {
        const long long kv_base = ((long long)si.b * p.heads_kv + h / p.group) * a.n_tiles;
        ks_row = a.ks + kv_base;
        vs_row = a.vs + kv_base;
        sq = q0 < si.len ? a.qs[((long long)si.b * p.heads_q + h) * a.n_tiles + q0 / kTile] : 0.f;
        float mx = 0.f;
        for (int t2 = lane; t2 < a.n_tiles; t2 += 32) mx = fmaxf(mx, vs_row[t2]);
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        sv_ref = mx;
      }
      int n_done = 0;
      PartList<kSparse, kPair> t;
      t.init(p, si.len, ur.q0, un.cost, ur.keep);
      int kt, bits8;
      while (t.next(kt, bits8)) {
        const int bits = (bits8 >> (4 * q)) & 0xF;
        if (!bits) continue;
        float sk = 1.f, sv = 1.f;
        if constexpr (kFp8) {  // read before the wait so that the loads overlap it
          sk = ks_row[kt];
          sv = vs_row[kt];
        }
        if (!W.warp(&sm.s_full[q], n_s & 1)) { ok = false; break; }
        ++n_s;
        ptx::tc_fence_after();
        const int k0 = kt * kTile;
        const bool need_mask = (k0 + kTile > si.len) || (elem_causal && k0 + kTile - 1 > q0);
        // Visibility of key k of this tile from this row: k < thr (sequence end and,
        // for causal rows, the diagonal) and, block-sparse, the row block's listed
        // 64-key halves (lo_ok / hi_ok: one row block per warp, so the same for the
        // whole warp; an unlisted half is neither read nor exponentiated).
        int thr = si.len - k0;
        if (elem_causal) thr = min(thr, qi - k0 + 1);
        const bool lo_ok = !kSparse || ((bits >> row_half) & 1), hi_ok = !kSparse || ((bits >> (row_half + 1)) & 1);
        // The 128-column S row (its listed halves), read from tensor memory at once.
        uint32_t sr[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          ptx::tmem_ld32(tmem + lane_base + col_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
        ptx::tmem_ld_wait();
        if constexpr (kSepP) {  // S_q is in registers: the next S_q may overwrite it
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.s_free[q]);
        }
        // x = s * scale * log2(e) = s' * |c| with s' = s or -s by the sign of the
        // scale, so the row max of x is |c| times the max of s' (8 partials keep the
        // dependency chains short).  Masked keys are left out.
        if (c < 0.f) {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k < 64 ? lo_ok : hi_ok) sr[k] ^= 0x80000000u;
        }
        const float ca = kFp8 ? fabsf(c) * sq * sk : fabsf(c);
        // FP8: P-hat = P r with r = sv / sv_ref in (0, 1], as 2^lr in the exponent
        // (lr >= -64: a tile with r below 2^-64 holds only zero codes or values
        // under 2^-55 of the head's largest); the row sum takes P-hat / r.
        float lr = 0.f, inv_r = 1.f;
        if constexpr (kFp8) {
          const float rr = sv_ref > 0.f ? sv / sv_ref : 1.f;
          lr = rr > 0.f ? fmaxf(fast_log2(rr), -64.f) : -64.f;
          inv_r = fast_exp2(-lr);
        }
        float e8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) e8[u] = -INFINITY;
        if (!need_mask) {
          // two scores per max instruction at head dim 128; at 64 the
          // two-input form measured 3% faster (register allocation)
          if constexpr (D == 128) {
            if (lo_ok) {
#pragma unroll
              for (int k = 0; k < 64; k += 2)
                e8[(k >> 1) & 7] = fmax3f(e8[(k >> 1) & 7], __uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
            }
            if (hi_ok) {
#pragma unroll
              for (int k = 64; k < 128; k += 2)
                e8[(k >> 1) & 7] = fmax3f(e8[(k >> 1) & 7], __uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
            }
          } else {
            if (lo_ok) {
#pragma unroll
              for (int k = 0; k < 64; ++k) e8[k & 7] = fmaxf(e8[k & 7], __uint_as_float(sr[k]));
            }
            if (hi_ok) {
#pragma unroll
              for (int k = 64; k < 128; ++k) e8[k & 7] = fmaxf(e8[k & 7], __uint_as_float(sr[k]));
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k < thr && (k < 64 ? lo_ok : hi_ok)) e8[k & 7] = fmaxf(e8[k & 7], __uint_as_float(sr[k]));
        }
        const float ext = fmaxf(fmaxf(fmaxf(e8[0], e8[1]), fmaxf(e8[2], e8[3])),
                                fmaxf(fmaxf(e8[4], e8[5]), fmaxf(e8[6], e8[7])));
        const float mx = ext == -INFINITY ? -INFINITY : ext * ca;
        const float m_new = fmaxf(m_used, mx);
        const bool resc = m_new > m_used + kRescaleLog2;
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m_used - m_new);
          l *= alpha;
          m_used = m_new;
        }
        const float mu = m_used == -INFINITY ? 0.f : m_used;
        if constexpr (kSepP) {
          // P_q's columns are free, and O_q stable, once the previous P_q V
          // product has finished
          if (n_pw > 0 && !W.warp(&sm.pv_done[q], (n_pw - 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
        }
        // P = exp2(s' |c| - m) as bf16 pairs, written 8 columns at a time over
        // S_q (at head dim 64 into P_q's own columns)
        float rs;
        if constexpr (kFp8)
          rs = (need_mask ? write_p8<true, kSparse>(sr, ca, mu - lr, thr, lo_ok, hi_ok, tmem + lane_base + col_s)
                          : write_p8<false, kSparse>(sr, ca, mu - lr, thr, lo_ok, hi_ok, tmem + lane_base + col_s)) *
               inv_r;
        else
          rs = need_mask ? write_p<true, kSparse>(sr, ca, mu, thr, lo_ok, hi_ok, tmem + lane_base + col_p)
                         : write_p<false, kSparse>(sr, ca, mu, thr, lo_ok, hi_ok, tmem + lane_base + col_p);
        // O_q is stable here: S_q of this tile was issued after the previous P_q V
        // product, whose completion its completion covers (at head dim 64 the
        // wait above covers it); the next product waits for p_full, so rescaling
        // O_q now (after P is written) is in time.
        if (n_done > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            ptx::tmem_ld32(tmem + lane_base + col_o + cc * 32, orr);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            ptx::tmem_st32(tmem + lane_base + col_o + cc * 32, orr);
          }
        }
        l += rs;
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.p_full[q]);
        ++n_done;
        ++n_pw;
      }
      if (!ok) break;
      if (q0 >= si.len) continue;  // this query tile lies past the sequence end
      // epilogue: O_q / l straight from tensor memory to global memory
      if (n_done > 0) {
        if (!W.warp(&sm.o_final[q], n_o & 1)) { ok = false; break; }
        ptx::tc_fence_after();
      }
      if constexpr (kPair) {
        // 128-row unit: both warpgroups hold partial results of the same rows
        // over alternate key tiles.  The second hands its row max and sum to the
        // first, which merges the two halves (each scaled to the larger max)
        // and writes the rows; the first also frees the second's O columns.
        if (q == 1) {
          if (!W.warp(&sm.pair_free, (n_pair & 1) ^ 1)) { ok = false; break; }
          sm.pair_m[r] = m_used;
          sm.pair_l[r] = l;
          if (r == 0) sm.pair_have = n_done > 0 ? 1 : 0;
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.pair_full);
          if (n_done > 0) ++n_o;
          ++n_pair;
          continue;
        }
        if (!W.warp(&sm.pair_full, n_pair & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const float m1 = sm.pair_m[r], l1 = sm.pair_l[r];
        const bool have1 = sm.pair_have != 0;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.pair_free);
        ++n_pair;
        const bool in0 = l > 0.f, in1 = have1 && l1 > 0.f;
        const float mm = in0 ? (in1 ? fmaxf(m_used, m1) : m_used) : (in1 ? m1 : 0.f);
        const float a0 = in0 ? fast_exp2(m_used - mm) : 0.f, a1 = in1 ? fast_exp2(m1 - mm) : 0.f;
        const float lt = l * a0 + (in1 ? l1 * a1 : 0.f);
        const float inv = lt > 0.f ? (kFp8 ? sv_ref / lt : 1.f / lt) : 0.f;
        const float w0 = a0 * inv, w1 = a1 * inv;
        __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o);
        const bool row_ok = qi < si.len && check_q_row(p, si, h, qi);
        __nv_bfloat16* orow = O + (row_ok ? q_off(p, si, h, qi) : 0);
        const float v0 = n_done > 0 ? w0 : 0.f, v1 = have1 ? w1 : 0.f;
#pragma unroll 1
        for (int cc = 0; cc < D / 16; ++cc) {
          uint32_t o0[16], o1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o0[i] = o1[i] = 0u;
          if (n_done > 0) ptx::tmem_ld16(tmem + lane_base + 256 + cc * 16, o0);
          if (have1) ptx::tmem_ld16(tmem + lane_base + 256 + D + cc * 16, o1);
          ptx::tmem_ld_wait();
          if (row_ok) {
#pragma unroll
            for (int w4 = 0; w4 < 2; ++w4) {
              uint32_t pk[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int i = w4 * 8 + 2 * j;
                pk[j] = ptx::pack_bf16x2(__uint_as_float(o0[i]) * v0 + __uint_as_float(o1[i]) * v1,
                                         __uint_as_float(o0[i + 1]) * v0 + __uint_as_float(o1[i + 1]) * v1);
              }
              *reinterpret_cast<uint4*>(orow + cc * 16 + w4 * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (n_done > 0) ptx::mbar_arrive(&sm.o_free[0]);
          if (have1) ptx::mbar_arrive(&sm.o_free[1]);
        }
        if (n_done > 0) ++n_o;
        if (row_ok) p.lse[row_index(p, si, h, qi)] = lt > 0.f ? (mm + fast_log2(lt)) * 0.69314718055994530942f : -INFINITY;
        continue;
      }
      if (p.n_split > 1) {
        // one part of a split key range: the unnormalised O (times the V
        // reference scale of FP8), the row max (log2 units) and the row sum
        const bool row_ok = qi < si.len && check_q_row(p, si, h, qi);
        const long long rows = (long long)p.batch * p.heads_q * p.seqlen;
        const long long ri = (long long)un.cost * rows + row_index(p, si, h, qi);
        const float osc = kFp8 ? sv_ref : 1.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t orr[32];
          if (n_done > 0) {
            ptx::tmem_ld32(tmem + lane_base + col_o + cc * 32, orr);
            ptx::tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = 0u;
          }
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(p.part_o + ri * D + cc * 32);
#pragma unroll
            for (int w4 = 0; w4 < 8; ++w4)
              dst[w4] = make_float4(__uint_as_float(orr[w4 * 4 + 0]) * osc, __uint_as_float(orr[w4 * 4 + 1]) * osc,
                                    __uint_as_float(orr[w4 * 4 + 2]) * osc, __uint_as_float(orr[w4 * 4 + 3]) * osc);
          }
        }
        if (n_done > 0) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.o_free[q]);
          ++n_o;
        }
        if (row_ok) *reinterpret_cast<float2*>(p.part_ml + ri * 2) = make_float2(l > 0.f ? m_used : -INFINITY, l);
        continue;
      }
      const float inv = l > 0.f ? (kFp8 ? sv_ref / l : 1.f / l) : 0.f;
      __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o);
      const bool row_ok = qi < si.len && check_q_row(p, si, h, qi);
      __nv_bfloat16* orow = O + (row_ok ? q_off(p, si, h, qi) : 0);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t orr[32];
        if (n_done > 0) {
          ptx::tmem_ld32(tmem + lane_base + col_o + cc * 32, orr);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            uint4 v4;
            v4.x = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 0]) * inv, __uint_as_float(orr[w4 * 8 + 1]) * inv);
            v4.y = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 2]) * inv, __uint_as_float(orr[w4 * 8 + 3]) * inv);
            v4.z = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 4]) * inv, __uint_as_float(orr[w4 * 8 + 5]) * inv);
            v4.w = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 6]) * inv, __uint_as_float(orr[w4 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + cc * 32 + w4 * 8) = v4;
          }
        }
      }
      if (n_done > 0) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.o_free[q]);
        ++n_o;
      }
      if (row_ok)
        p.lse[row_index(p, si, h, qi)] = l > 0.f ? (m_used + fast_log2(l)) * 0.69314718055994530942f : -INFINITY;
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

// ===========================================================================
// Head dim 256.  Two query tiles' O accumulators (2 x 256 columns) and S
// buffers would need 768 tensor-memory columns, so a unit is one 128-row query
// tile: S0 [0,128) S1 [128,256) O [256,512).  S of the CTA's k-th key tile goes
// to buffer k % 2, so the tensor core computes S(k+1) while the softmax works on
// S(k); P(k) is written over S(k) as bf16 and read by the P V products, and only
// then does S(k+2) overwrite the buffer (the tensor core runs one thread's
// products in issue order).  The products per key tile (2 x 1024 clocks) exceed
// the softmax (about 1150), so the tensor core sets the pace.
//
// Shared memory: Q (128 x 256, four 64-column boxes, 64 KiB) and a ring of
// 32 KiB chunks (128 rows x 128 columns, two boxes), each released by its own
// eight products: per key tile K[:, 0:128), K[:, 128:256), then, one tile
// behind, V[:, 0:128), V[:, 128:256), in the order the issuer uses them.
//
// Warps (256 threads): 0-3 softmax (thread r owns row r), 4 TMA producer and
// unit fetcher, 5 tensor-core issuer, 6-7 idle.  Every wait is bounded.
// ===========================================================================
constexpr int kThreads256 = 256;
constexpr int kRing256 = 5;
constexpr uint32_t kChunk256 = 2 * kHalfTileBytes;  // 128 rows x 128 bf16 columns

struct Smem256 {
  uint8_t q[4][kHalfTileBytes];
  uint8_t ring[kRing256][kChunk256];
  uint64_t unit_full[2], unit_empty[2];
  uint64_t q_full, q_empty;
  uint64_t c_full[kRing256], c_empty[kRing256];
  uint64_t s_full[2], p_full[2], pv_done, o_final, o_free;
  uint64_t drain;
  int unit_slot[2][4];
  uint32_t tmem_base;
  ptx::Abort abort;
};
static_assert(sizeof(Smem256) + 1024 <= 232448, "shared memory per CTA is at most 227 KiB");

template <bool kSparse>
__global__ void __launch_bounds__(kThreads256, 1) k_tc_fwd256(const __grid_constant__ FwdArgs a) {
  using SM = Smem256;
  extern __shared__ uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KParams& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Waiter<SM> W{sm, p};

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sm.unit_full[i], 1);
      ptx::mbar_init(&sm.unit_empty[i], 5);  // 4 softmax warps + the issuer
      ptx::mbar_init(&sm.s_full[i], 1);
      ptx::mbar_init(&sm.p_full[i], 4);
    }
    ptx::mbar_init(&sm.q_full, 1);
    ptx::mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < kRing256; ++s) {
      ptx::mbar_init(&sm.c_full[s], 1);
      ptx::mbar_init(&sm.c_empty[s], 1);
    }
    ptx::mbar_init(&sm.pv_done, 1);
    ptx::mbar_init(&sm.o_final, 1);
    ptx::mbar_init(&sm.o_free, 4);
    ptx::mbar_init(&sm.drain, 1);
    sm.abort.flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 4) {
    // ================================================================ producer
    uint32_t n_units_seen = 0, n_q = 0, n_c = 0;
    int last_q_phase = -1, last_c_phase[kRing256];
    for (int s = 0; s < kRing256; ++s) last_c_phase[s] = -1;
    bool ok = true;
    for (;;) {
      const int slot = n_units_seen & 1;
      if (!W.warp(&sm.unit_empty[slot], ((n_units_seen >> 1) & 1) ^ 1)) { ok = false; break; }
      int idx = 0;
      if (lane == 0) idx = atomicAdd(p.unit_counter, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      bool valid = idx < p.n_units;
      Unit un{0, 0, 0, 0};
      if (valid) {
        un = p.units[idx];
        valid = check_unit(p, un, false, kTile);
      }
      if (lane == 0) {
        volatile int* s = sm.unit_slot[slot];
        s[0] = un.seq;
        s[1] = un.head;
        s[2] = un.tile;
        s[3] = valid ? 1 : 0;
        ptx::mbar_arrive(&sm.unit_full[slot]);
      }
      ++n_units_seen;
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      const int h = un.head, g = h / p.group, q0 = un.tile * kTile;
      bool any = false;
      {
        KvTileList2<kSparse> t;
        t.init(p, si.len, q0);
        int kt, bits;
        while (t.next(kt, bits)) any |= (bits & 0xF) != 0;
      }
      if (!any) continue;
      if (!W.warp(&sm.q_empty, (n_q & 1) ^ 1)) { ok = false; break; }
      if (lane == 0) {
        check_q_row(p, si, h, q0);
        ptx::mbar_arrive_expect_tx(&sm.q_full, 4 * kHalfTileBytes);
        for (int c = 0; c < 4; ++c) {
          if (a.q_rows_inner) ptx::tma_load_4d(sm.q[c], &a.tq, &sm.q_full, c * 64, map_row(si, q0), h, si.b);
          else ptx::tma_load_4d(sm.q[c], &a.tq, &sm.q_full, c * 64, h, map_row(si, q0), si.b);
        }
      }
      last_q_phase = (int)(n_q & 1);
      ++n_q;
      // two chunks (columns 0-127, 128-255) of K or V for key tile kt_
      auto load_pair = [&](const CUtensorMap* map, int kt_) -> bool {
        for (int half = 0; half < 2; ++half) {
          const int st = n_c % kRing256;
          const uint32_t ph = (n_c / kRing256) & 1;
          if (!W.warp(&sm.c_empty[st], ph ^ 1)) return false;
          if (lane == 0) {
            check_kv_row(p, si, g, kt_ * kTile);
            ptx::mbar_arrive_expect_tx(&sm.c_full[st], kChunk256);
            for (int c = 0; c < 2; ++c) {
              const int x = half * 128 + c * 64;
              uint8_t* d = sm.ring[st] + c * kHalfTileBytes;
              if (a.kv_rows_inner) ptx::tma_load_4d(d, map, &sm.c_full[st], x, map_row(si, kt_ * kTile), g, si.b);
              else ptx::tma_load_4d(d, map, &sm.c_full[st], x, g, map_row(si, kt_ * kTile), si.b);
            }
          }
          last_c_phase[st] = (int)ph;
          ++n_c;
        }
        return true;
      };
      // K runs one key tile ahead of V: the issuer's order is S(0), S(1), PV(0), S(2), PV(1), ...
      KvTileList2<kSparse> t;
      t.init(p, si.len, q0);
      int kt = 0, bits = 0;
      bool have = t.next(kt, bits);
      while (have && !(bits & 0xF)) have = t.next(kt, bits);
      if (have && !load_pair(&a.tk, kt)) { ok = false; break; }
      while (have) {
        int nkt = 0, nbits = 0;
        bool nhave = t.next(nkt, nbits);
        while (nhave && !(nbits & 0xF)) nhave = t.next(nkt, nbits);
        if (nhave && !load_pair(&a.tk, nkt)) { ok = false; break; }
        if (!load_pair(&a.tv, kt)) { ok = false; break; }
        have = nhave;
        kt = nkt;
      }
      if (!ok) break;
    }
    (void)ok;
    if (lane == 0) {
      if (last_q_phase >= 0) W.drain(&sm.q_full, (uint32_t)last_q_phase);
      for (int s = 0; s < kRing256; ++s)
        if (last_c_phase[s] >= 0) W.drain(&sm.c_full[s], (uint32_t)last_c_phase[s]);
    }
  } else if (warp == 5) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc_s = ptx::idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_pv = ptx::idesc_bf16(128, 128, false, true);
    const uint32_t q_addr = ptx::smem_u32(sm.q[0]);
    const uint32_t t_o = tmem + 256;
    uint32_t n_units_seen = 0, n_q = 0, n_c = 0, n_s = 0, n_p = 0, n_o = 0;
    bool ok = true;
    // waits for the next ring chunk; returns its shared address (0 on a timeout)
    auto next_chunk = [&](uint32_t& st) -> uint32_t {
      st = n_c % kRing256;
      if (!W.warp(&sm.c_full[st], (n_c / kRing256) & 1)) return 0;
      ++n_c;
      ptx::tc_fence_after();
      return ptx::smem_u32(sm.ring[st]);
    };
    // S of the unit's next key tile into buffer n_s % 2: Q K^T over head-dim
    // columns 0-127 (first chunk) and 128-255 (second chunk)
    auto issue_s = [&](bool last_of_unit) -> bool {
      const uint32_t t_s = tmem + (n_s & 1) * 128;
      for (int half = 0; half < 2; ++half) {
        uint32_t st;
        const uint32_t k_addr = next_chunk(st);
        if (!k_addr) return false;
        if (ptx::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t qo = (uint32_t)(half * 2 + (kk >> 2)) * kHalfTileBytes + (kk & 3) * 32;
            const uint32_t ko = (uint32_t)(kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
            ptx::mma_ss(t_s, ptx::sdesc_sw128(q_addr + qo, 16, 1024), ptx::sdesc_sw128(k_addr + ko, 16, 1024),
                        idesc_s, (half > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&sm.c_empty[st]);
          if (half == 1) {
            ptx::mma_commit(&sm.s_full[n_s & 1]);
            if (last_of_unit) ptx::mma_commit(&sm.q_empty);
          }
        }
        __syncwarp();
      }
      ++n_s;
      return true;
    };
    for (;;) {
      const int slot = n_units_seen & 1;
      if (!W.warp(&sm.unit_full[slot], (n_units_seen >> 1) & 1)) { ok = false; break; }
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      ++n_units_seen;
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      int n_act = 0;
      {
        KvTileList2<kSparse> t;
        t.init(p, si.len, un.tile * kTile);
        int kt, bits;
        while (t.next(kt, bits)) n_act += (bits & 0xF) != 0;
      }
      if (n_act == 0) continue;
      if (!W.warp(&sm.q_full, n_q & 1)) { ok = false; break; }
      ++n_q;
      ptx::tc_fence_after();
      if (!issue_s(n_act == 1)) { ok = false; break; }
      if (n_act > 1 && !issue_s(n_act == 2)) { ok = false; break; }
      for (int i = 0; i < n_act && ok; ++i) {
        // O += P(i) V(i) once the softmax has written P(i); before the unit's
        // first product, the previous unit's epilogue must have read O
        const uint32_t b = n_p & 1;
        if (!W.warp(&sm.p_full[b], (n_p >> 1) & 1)) { ok = false; break; }
        ++n_p;
        if (i == 0 && !W.warp(&sm.o_free, (n_o & 1) ^ 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t t_p = tmem + b * 128;
        for (int half = 0; half < 2; ++half) {
          uint32_t st;
          const uint32_t v_addr = next_chunk(st);
          if (!v_addr) { ok = false; break; }
          if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // B = V as (N = head dim, K = keys), head dim contiguous: MN-major
              const uint64_t bdesc = ptx::sdesc_sw128(v_addr + kk * 2048, kHalfTileBytes, 1024);
              ptx::mma_ts(t_o + half * 128, t_p + kk * 8, bdesc, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::mma_commit(&sm.c_empty[st]);
            if (half == 1) {
              ptx::mma_commit(&sm.pv_done);
              if (i == n_act - 1) ptx::mma_commit(&sm.o_final);
            }
          }
          __syncwarp();
        }
        if (!ok) break;
        if (i + 2 < n_act && !issue_s(i + 3 == n_act)) { ok = false; break; }
      }
      if (!ok) break;
      ++n_o;
    }
    (void)ok;
    __syncwarp();
    if (ptx::elect_one()) ptx::mma_commit(&sm.drain);
    __syncwarp();
    if (lane == 0) W.drain(&sm.drain, 0);
    __syncwarp();
  } else if (warp < 4) {
    // ================================================================ softmax
    const int r = warp * 32 + lane;  // row in the query tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t col_o = 256;
    const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);
    const float c = p.scale_log2;
    const int row_half = r >= 64 ? 2 : 0;
    uint32_t n_units_seen = 0, n_t = 0, n_o = 0;
    bool ok = true;
    for (;;) {
      const int slot = n_units_seen & 1;
      if (!W.warp(&sm.unit_full[slot], (n_units_seen >> 1) & 1)) { ok = false; break; }
      Unit un;
      const bool valid = read_unit(sm, slot, un);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.unit_empty[slot]);
      ++n_units_seen;
      if (!valid) break;
      const SeqInfo si = seq_info(p, un.seq);
      const int h = un.head;
      const int q0 = un.tile * kTile;
      const int qi = q0 + r;
      float m_used = -INFINITY, l = 0.f;
      int n_done = 0;
      KvTileList2<kSparse> t;
      t.init(p, si.len, q0);
      int kt, bits8;
      while (t.next(kt, bits8)) {
        const int bits = bits8 & 0xF;
        if (!bits) continue;
        const uint32_t b = n_t & 1, col_s = b * 128;
        if (!W.warp(&sm.s_full[b], (n_t >> 1) & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const int k0 = kt * kTile;
        const bool need_mask = (k0 + kTile > si.len) || (elem_causal && k0 + kTile - 1 > q0);
        int thr = si.len - k0;
        if (elem_causal) thr = min(thr, qi - k0 + 1);
        const bool lo_ok = !kSparse || ((bits >> row_half) & 1), hi_ok = !kSparse || ((bits >> (row_half + 1)) & 1);
        uint32_t sr[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          ptx::tmem_ld32(tmem + lane_base + col_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
        ptx::tmem_ld_wait();
        if (c < 0.f) {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k < 64 ? lo_ok : hi_ok) sr[k] ^= 0x80000000u;
        }
        const float ca = fabsf(c);
        float e8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) e8[u] = -INFINITY;
        if (!need_mask) {
          if (lo_ok) {
#pragma unroll
            for (int k = 0; k < 64; k += 2)
              e8[(k >> 1) & 7] = fmax3f(e8[(k >> 1) & 7], __uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
          }
          if (hi_ok) {
#pragma unroll
            for (int k = 64; k < 128; k += 2)
              e8[(k >> 1) & 7] = fmax3f(e8[(k >> 1) & 7], __uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
          }
        } else {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k < thr && (k < 64 ? lo_ok : hi_ok)) e8[k & 7] = fmaxf(e8[k & 7], __uint_as_float(sr[k]));
        }
        const float ext = fmaxf(fmaxf(fmaxf(e8[0], e8[1]), fmaxf(e8[2], e8[3])),
                                fmaxf(fmaxf(e8[4], e8[5]), fmaxf(e8[6], e8[7])));
        const float mx = ext == -INFINITY ? -INFINITY : ext * ca;
        const float m_new = fmaxf(m_used, mx);
        const bool resc = m_new > m_used + kRescaleLog2;
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m_used - m_new);
          l *= alpha;
          m_used = m_new;
        }
        const float mu = m_used == -INFINITY ? 0.f : m_used;
        const float rs = need_mask ? write_p<true, kSparse>(sr, ca, mu, thr, lo_ok, hi_ok, tmem + lane_base + col_s)
                                   : write_p<false, kSparse>(sr, ca, mu, thr, lo_ok, hi_ok, tmem + lane_base + col_s);
        // Rescaling O: the previous tile's P V products may still run (S of this
        // tile was issued before them), so wait for them first.  The products
        // of this tile wait for p_full, so rescaling now is in time.
        if (n_done > 0 && __any_sync(0xffffffffu, resc)) {
          if (!W.warp(&sm.pv_done, (n_t - 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t orr[32];
            ptx::tmem_ld32(tmem + lane_base + col_o + cc * 32, orr);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            ptx::tmem_st32(tmem + lane_base + col_o + cc * 32, orr);
          }
        }
        l += rs;
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.p_full[b]);
        ++n_t;
        ++n_done;
      }
      if (!ok) break;
      if (q0 >= si.len) continue;
      if (n_done > 0) {
        if (!W.warp(&sm.o_final, n_o & 1)) { ok = false; break; }
        ptx::tc_fence_after();
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o);
      const bool row_ok = qi < si.len && check_q_row(p, si, h, qi);
      __nv_bfloat16* orow = O + (row_ok ? q_off(p, si, h, qi) : 0);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t orr[32];
        if (n_done > 0) {
          ptx::tmem_ld32(tmem + lane_base + col_o + cc * 32, orr);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            uint4 v4;
            v4.x = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 0]) * inv, __uint_as_float(orr[w4 * 8 + 1]) * inv);
            v4.y = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 2]) * inv, __uint_as_float(orr[w4 * 8 + 3]) * inv);
            v4.z = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 4]) * inv, __uint_as_float(orr[w4 * 8 + 5]) * inv);
            v4.w = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 6]) * inv, __uint_as_float(orr[w4 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + cc * 32 + w4 * 8) = v4;
          }
        }
      }
      if (n_done > 0) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.o_free);
        ++n_o;
      }
      if (row_ok)
        p.lse[row_index(p, si, h, qi)] = l > 0.f ? (m_used + fast_log2(l)) * 0.69314718055994530942f : -INFINITY;
    }
    (void)ok;
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool tc_fwd_available() { return true; }

cudaError_t launch_tc_fwd256(const KParams& p, int sms, cudaStream_t st) {
  FwdArgs a;
  TileMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_tile_map(&mq, p.q, p, false)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mk, p.k, p, true)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mv, p.v, p, true)) != cudaSuccess) return e;
  a.tq = mq.map;
  a.tk = mk.map;
  a.tv = mv.map;
  a.q_rows_inner = mq.rows_inner;
  a.kv_rows_inner = mk.rows_inner;
  a.p = p;
  const size_t smem = sizeof(Smem256) + 1024;
  const int grid = p.n_units < sms ? p.n_units : sms;
  auto kernel = p.mask == kMaskBlock ? k_tc_fwd256<true> : k_tc_fwd256<false>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const KParams& p, int sms, cudaStream_t st) {
  if (p.n_units == 0) return cudaSuccess;
  if (p.head_dim == 256) return launch_tc_fwd256(p, sms, st);
  FwdArgs a;
  TileMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_tile_map(&mq, p.q, p, false)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mk, p.k, p, true)) != cudaSuccess) return e;
  if ((e = make_tile_map(&mv, p.v, p, true)) != cudaSuccess) return e;
  a.tq = mq.map;
  a.tk = mk.map;
  a.tv = mv.map;
  a.q_rows_inner = mq.rows_inner;
  a.kv_rows_inner = mk.rows_inner;
  a.p = p;
  const size_t smem = sizeof(Smem<FwdCfg<false>>) + 1024;
  const int grid = p.n_units < sms ? p.n_units : sms;
  auto kernel = p.fwd_half
                    ? (p.head_dim == 64 ? k_tc_fwd<false, 64, false, true> : k_tc_fwd<false, 128, false, true>)
                : p.head_dim == 64
                    ? (p.mask == kMaskBlock ? k_tc_fwd<true, 64, false> : k_tc_fwd<false, 64, false>)
                    : (p.mask == kMaskBlock ? k_tc_fwd<true, 128, false> : k_tc_fwd<false, 128, false>);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd_fp8(const KParams& p, int sms, cudaStream_t st, const Fp8Operands& f) {
  if (p.n_units == 0) return cudaSuccess;
  FwdArgs a;
  TileMap mq, mk, mv;
  cudaError_t e;
  const long long S = p.seqlen;
  // Q and K codes: 128-byte rows, one per position; V codes: one row per head dim, keys along it
  if ((e = make_byte_map(&mq, f.q8, 128, S, p.heads_q, p.batch, 128)) != cudaSuccess) return e;
  if ((e = make_byte_map(&mk, f.k8, 128, S, p.heads_kv, p.batch, 128)) != cudaSuccess) return e;
  if ((e = make_byte_map(&mv, f.v8t, S, 128, p.heads_kv, p.batch, f.ld_t)) != cudaSuccess) return e;
  a.tq = mq.map;
  a.tk = mk.map;
  a.tv = mv.map;
  a.q_rows_inner = a.kv_rows_inner = 1;
  a.p = p;
  a.qs = f.qs;
  a.ks = f.ks;
  a.vs = f.vs;
  a.n_tiles = (int)((S + kTile - 1) / kTile);
  const size_t smem = sizeof(Smem<FwdCfg<true>>) + 1024;
  const int grid = p.n_units < sms ? p.n_units : sms;
  auto kernel = p.mask == kMaskBlock ? k_tc_fwd<true, 128, true> : k_tc_fwd<false, 128, true>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbattn
