// Forward attention on the fifth-generation tensor cores (sm_103a).
//
// One CTA computes one 128-row query tile of one head (zwxr.cn CANN ops-nn
// fused-attention article, sections 3.2-3.3: the outer loop takes a query block,
// the inner loop streams key/value blocks, and a running max and sum correct
// the softmax across blocks, so the score matrix never leaves the chip; smzdm
// contest article, section 03, on FlashAttention as tiling plus fusion).
//
// Warp roles (192 threads):
//   warp 4     TMA producer: Q once, then K_j and V_j into a two-stage ring
//              (prefetch the next block while the current one is used: zwxr.cn
//              article, section 4.1, double buffering).
//   warp 5     tensor-core issuer: S_j = Q K_j^T into tensor memory (two S
//              buffers), then O += P_j V_j with P read from tensor memory.  The
//              matrix products run on the matrix unit (smzdm article, the team
//              that moved the matmul to the cube unit).
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r).  It reads S_j,
//              masks, updates the running max m and sum l, writes P_j as bf16
//              over S_j in tensor memory (P is never written to shared or global
//              memory: zwxr.cn article, section 5.4), rescales O when m grew by
//              more than 2^8, and finally writes O / l and LSE.
// Every wait is bounded; a CTA that gives up records ATTN_ERR_DEVICE_TIMEOUT,
// drains its copies and tensor-core work, frees tensor memory and returns.
#include <cuda.h>

#include "tc_common.cuh"
#include "tc_kernels.h"
#include "tma_host.h"

namespace gbattn {

namespace {

constexpr int kStages = 2;
constexpr int kFwdThreads = 192;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the row max grows by more than 2^8
constexpr uint32_t kTmemCols = 512;   // S0 [0,128) S1 [128,256) O [256,384)
constexpr uint32_t kColO = 256;

struct FwdArgs {
  CUtensorMap tq, tk, tv;
  int q_rows_inner, kv_rows_inner;
  KParams p;
};

struct FwdSmem {
  uint8_t q[kTileBytes];  // Q tile; O staging in the epilogue
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint64_t q_full, k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2], o_ready, o_final, drain;
  uint32_t tmem_base;
  ptx::Abort abort;
};

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, FwdSmem& sm, const KParams& p) {
  bool ok = ptx::mbar_wait(bar, parity, &sm.abort, p.status, p.wait_limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// Wait that ignores the abort flag (used only to drain in-flight work).
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, FwdSmem& sm, const KParams& p) {
  ptx::Abort none;
  none.flag = 0;
  ptx::mbar_wait(bar, parity, &none, p.status, p.wait_limit_ns);
}

__global__ void __launch_bounds__(kFwdThreads, 1) k_tc_fwd(const __grid_constant__ FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KParams& p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Unit u = p.units[blockIdx.x];
  const SeqInfo si = seq_info(p, u.seq);
  const int h = u.head, g = h / p.group;
  const int q0 = u.tile * kTile;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sm.k_full[s], 1);
      ptx::mbar_init(&sm.v_full[s], 1);
      ptx::mbar_init(&sm.kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sm.s_full[b], 1);
      ptx::mbar_init(&sm.p_full[b], 4);
    }
    ptx::mbar_init(&sm.o_ready, 1);
    ptx::mbar_init(&sm.o_final, 1);
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

  KvTileList tiles;
  tiles.init(p, si.len, q0);
  int n_tiles = 0;
  {
    KvTileList t = tiles;
    int kt, bits;
    while (t.next(kt, bits)) ++n_tiles;
  }

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      ptx::tma_prefetch_desc(&a.tq);
      ptx::tma_prefetch_desc(&a.tk);
      ptx::tma_prefetch_desc(&a.tv);
      ptx::mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
      tma_tile(sm.q, &a.tq, a.q_rows_inner, &sm.q_full, map_row(si, q0), h, si.b, kHalfTileBytes);
      int last_phase[kStages];
      for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
      KvTileList t = tiles;
      int kt, bits, j = 0;
      while (t.next(kt, bits)) {
        const int st = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!ptx::mbar_wait(&sm.kv_empty[st], ph ^ 1, &sm.abort, p.status, p.wait_limit_ns)) break;
        ptx::mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
        tma_tile(sm.k[st], &a.tk, a.kv_rows_inner, &sm.k_full[st], map_row(si, kt * kTile), g, si.b,
                 kHalfTileBytes);
        ptx::mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
        tma_tile(sm.v[st], &a.tv, a.kv_rows_inner, &sm.v_full[st], map_row(si, kt * kTile), g, si.b,
                 kHalfTileBytes);
        last_phase[st] = (int)ph;
        ++j;
      }
      // every copy this thread started has landed before the CTA winds down
      wait_drain(&sm.q_full, 0, sm, p);
      for (int s = 0; s < kStages; ++s)
        if (last_phase[s] >= 0) {
          wait_drain(&sm.k_full[s], (uint32_t)last_phase[s], sm, p);
          wait_drain(&sm.v_full[s], (uint32_t)last_phase[s], sm, p);
        }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16(128, 128, false, true);
      const uint32_t q_addr = ptx::smem_u32(sm.q);
      bool ok = ptx::mbar_wait(&sm.q_full, 0, &sm.abort, p.status, p.wait_limit_ns);
      ptx::tc_fence_after();

      // o_ready completes after every P V product (the softmax waits on it only
      // right after seeing S_j, when it is at most one phase behind); o_final
      // completes once, after the last one.
      auto issue_pv = [&](int i, bool last) -> bool {
        const int b = i & 1, st = i % kStages;
        if (!ptx::mbar_wait(&sm.p_full[b], (i >> 1) & 1, &sm.abort, p.status, p.wait_limit_ns)) return false;
        if (!ptx::mbar_wait(&sm.v_full[st], (i / kStages) & 1, &sm.abort, p.status, p.wait_limit_ns))
          return false;
        ptx::tc_fence_after();
        const uint32_t v_addr = ptx::smem_u32(sm.v[st]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // B = V as (N = head dim, K = keys), head dim contiguous: MN-major.
          const uint64_t bdesc = ptx::sdesc_sw128(v_addr + kk * 2048, kHalfTileBytes, 1024);
          ptx::mma_ts(tmem + kColO, tmem + b * 128 + kk * 8, bdesc, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&sm.kv_empty[st]);
        ptx::mma_commit(&sm.o_ready);
        if (last) ptx::mma_commit(&sm.o_final);
        return true;
      };

      KvTileList t = tiles;
      int kt, bits, j = 0;
      while (ok && t.next(kt, bits)) {
        const int b = j & 1, st = j % kStages;
        if (!ptx::mbar_wait(&sm.k_full[st], (j / kStages) & 1, &sm.abort, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t k_addr = ptx::smem_u32(sm.k[st]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
          ptx::mma_ss(tmem + b * 128, ptx::sdesc_sw128(q_addr + off, 16, 1024),
                      ptx::sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&sm.s_full[b]);
        if (j > 0 && !issue_pv(j - 1, false)) {
          ok = false;
          break;
        }
        ++j;
      }
      if (ok && j > 0) issue_pv(j - 1, true);
      // every tensor-core operation issued so far is finished before tensor memory is freed
      ptx::mma_commit(&sm.drain);
      wait_drain(&sm.drain, 0, sm, p);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int r = threadIdx.x;  // row in the tile = TMEM lane
    const int qi = q0 + r;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const bool elem_causal = p.mask == kMaskCausal || (p.mask == kMaskBlock && p.causal_in_block);
    const float c = p.scale_log2;
    const int row_half = r >= 64 ? 2 : 0;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int j = 0;
    {
      KvTileList t = tiles;
      int kt, bits;
      while (t.next(kt, bits)) {
        const int b = j & 1;
        if (!wait_warp(&sm.s_full[b], (j >> 1) & 1, sm, p)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          ptx::tmem_ld32(tmem + lane_base + b * 128 + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
        ptx::tmem_ld_wait();
        const int k0 = kt * kTile;
        const bool need_mask = (k0 + kTile > si.len) || (elem_causal && k0 + kTile - 1 > q0) || bits != 0xF;
        float x[128];
        float mx = -INFINITY;
        if (need_mask) {
#pragma unroll
          for (int k = 0; k < 128; ++k) {
            const int kj = k0 + k;
            bool keep = kj < si.len && ((bits >> (row_half + (k >= 64 ? 1 : 0))) & 1);
            if (elem_causal) keep = keep && kj <= qi;
            x[k] = keep ? __uint_as_float(sr[k]) * c : -INFINITY;
            mx = fmaxf(mx, x[k]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 128; ++k) {
            x[k] = __uint_as_float(sr[k]) * c;
            mx = fmaxf(mx, x[k]);
          }
        }
        const float m_new = fmaxf(m_used, mx);
        const bool resc = m_new > m_used + kRescaleLog2;
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m_used - m_new);  // 0 when m_used is -inf
          l *= alpha;
          m_used = m_new;
        }
        const float mu = m_used == -INFINITY ? 0.f : m_used;
        uint32_t pk[64];
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float p0 = fast_exp2(x[2 * i] - mu), p1 = fast_exp2(x[2 * i + 1] - mu);
          rs += p0 + p1;
          pk[i] = ptx::pack_bf16x2(p0, p1);
        }
        l += rs;
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O holds sum_{t<j} P_t V_t once the previous product is done; rescale it
          if (!wait_warp(&sm.o_ready, (j - 1) & 1, sm, p)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t orr[32];
            ptx::tmem_ld32(tmem + lane_base + kColO + cc * 32, orr);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            ptx::tmem_st32(tmem + lane_base + kColO + cc * 32, orr);
          }
        }
        ptx::tmem_st32(tmem + lane_base + b * 128, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        ptx::tmem_st32(tmem + lane_base + b * 128 + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.p_full[b]);
        ++j;
      }
    }
    if (ok && j > 0) ok = wait_warp(&sm.o_final, 0, sm, p);
    ok = ok && !sm.abort.flag;
    if (ok) {
      ptx::tc_fence_after();
      // O / l to bf16, staged in shared memory (the Q buffer: every S product is
      // done once the last P V product is), 16-byte chunk c of row r at chunk c ^ (r & 15).
      uint8_t* stage = sm.q;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t orr[32];
        if (j > 0) {
          ptx::tmem_ld32(tmem + lane_base + kColO + cc * 32, orr);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = 0u;
        }
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          uint4 v4;
          v4.x = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 0]) * inv, __uint_as_float(orr[w4 * 8 + 1]) * inv);
          v4.y = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 2]) * inv, __uint_as_float(orr[w4 * 8 + 3]) * inv);
          v4.z = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 4]) * inv, __uint_as_float(orr[w4 * 8 + 5]) * inv);
          v4.w = ptx::pack_bf16x2(__uint_as_float(orr[w4 * 8 + 6]) * inv, __uint_as_float(orr[w4 * 8 + 7]) * inv);
          const int ch = cc * 4 + w4;
          *reinterpret_cast<uint4*>(stage + r * 256 + ((ch ^ (r & 15)) * 16)) = v4;
        }
      }
      if (qi < si.len)
        p.lse[row_index(p, si, h, qi)] = l > 0.f ? (m_used + fast_log2(l)) * 0.69314718055994530942f : -INFINITY;
      __syncwarp();
      // each warp copies its own 32 rows out: two full 256-byte rows per instruction
      __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o);
#pragma unroll 4
      for (int it = 0; it < 16; ++it) {
        const int row = warp * 32 + it * 2 + (lane >> 4), ch = lane & 15;
        if (q0 + row < si.len) {
          const uint4 v4 = *reinterpret_cast<const uint4*>(stage + row * 256 + ((ch ^ (row & 15)) * 16));
          *reinterpret_cast<uint4*>(O + q_off(p, si, h, q0 + row) + ch * 8) = v4;
        }
      }
    }
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

cudaError_t launch_tc_fwd(const KParams& p, int sms, cudaStream_t st) {
  (void)sms;
  if (p.n_units == 0) return cudaSuccess;
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
  const size_t smem = sizeof(FwdSmem) + 1024;
  e = cudaFuncSetAttribute(k_tc_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_tc_fwd<<<p.n_units, kFwdThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gbattn
