// Pieces shared by the tensor-core forward and backward kernels: tile loads
// through TMA and the lists of score tiles a unit visits.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace gbattn {

constexpr int kTile = 128;                       // rows of a Q tile / keys of a K,V tile
constexpr int kHeadDim = 128;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;  // bf16 128 x 128 = 32 KiB
constexpr uint32_t kHalfTileBytes = kTileBytes / 2;    // one 128 x 64 box (128-byte rows)
// bf16 bytes of a 128-row tile of head dim D (64: one box, 128: two boxes)
template <int D>
constexpr uint32_t tile_bytes() { return (uint32_t)kTile * D * 2; }

// Loads rows [row, row + rows) x all nbox * 64 columns of one head as nbox
// 64-column boxes (each rows x 128 bytes, 128-byte swizzled) at dst,
// dst + box_bytes, ...
__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* map, int rows_inner, uint64_t* bar,
                                         int row, int head, int b, uint32_t box_bytes, int nbox = 2) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (c >= nbox) break;
    void* d = static_cast<char*>(dst) + c * box_bytes;
    if (rows_inner) ptx::tma_load_4d(d, map, bar, c * 64, row, head, b);
    else ptx::tma_load_4d(d, map, bar, c * 64, head, row, b);
  }
}

// L2 prefetch of the same tile tma_tile would load.
__device__ __forceinline__ void tma_prefetch_tile(const CUtensorMap* map, int rows_inner, int row, int head, int b,
                                                  int nbox = 2) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (c >= nbox) break;
    if (rows_inner) ptx::tma_prefetch_4d(map, c * 64, row, head, b);
    else ptx::tma_prefetch_4d(map, c * 64, head, row, b);
  }
}

// Row coordinate and batch coordinate of position `pos` of a sequence in a tile map.
__device__ __forceinline__ int map_row(const SeqInfo& s, int pos) { return (int)(s.tok0 + pos); }

}  // namespace gbattn

namespace gbattn {

// The 64-row query blocks a backward unit (one 128-key tile) visits for one
// query head, ascending, with a 2-bit mask of which 64x64 sub-blocks are listed:
//   bit 0 (keys 0-63 of the tile), bit 1 (keys 64-127).
// Dense units visit every query block; causal units start at the block holding
// the tile's first key; block-sparse units take the union of the two key
// blocks' transposed (per key block) lists.
struct QBlockList {
  int mode;
  int first, count, it;      // dense / causal range
  const int* row;            // transposed lists (query blocks per key block)
  int a0, ea, b0, eb, ia, ib;
  int nblk;
  const KParams* kp;         // checked builds: extents and status word

  // Transposed-list entry i in [s, e): a query block below the sequence's block
  // count, else INT_MAX (ascending: every later entry is past the end too).
  __device__ int entry(int i, int e) const {
    if (i >= e) return INT_MAX;
    const int r = row[i];
    if (!check_block(*kp, r, kp->n_row_blocks)) return INT_MAX;
    return r < nblk ? r : INT_MAX;
  }

  __device__ void init(const KParams& p, int len, int kt) {
    kp = &p;
    mode = p.mask;
    nblk = (len + 63) / 64;
    it = 0;
    a0 = ea = b0 = eb = 0;
    row = nullptr;
    if (mode == kMaskNone) {
      first = 0;
      count = nblk;
    } else if (mode == kMaskCausal) {
      first = 2 * kt;
      count = nblk > first ? nblk - first : 0;
    } else {
      row = p.csc_idx;
      const int cb0 = 2 * kt, cb1 = cb0 + 1;
      if (check_block(p, cb0, p.n_col_blocks)) {
        a0 = p.csc_ptr[cb0];
        ea = p.csc_ptr[cb0 + 1];
      }
      if (cb1 < p.n_col_blocks && cb1 * 64 < len) {
        b0 = p.csc_ptr[cb1];
        eb = p.csc_ptr[cb1 + 1];
      } else {
        b0 = eb = 0;
      }
      // each key block's list lies inside the transposed index array
      const int nnz = p.csc_ptr[p.n_col_blocks];
      if (!bounds_ok(!GBATTN_CHECKED || (0 <= a0 && a0 <= ea && ea <= nnz && 0 <= b0 && b0 <= eb && eb <= nnz),
                     p.status))
        a0 = ea = b0 = eb = 0;
    }
    restart();
  }

  __device__ void restart() {
    it = 0;
    ia = a0;
    ib = b0;
  }

  __device__ bool next(int& qb, int& bits) {
    if (mode != kMaskBlock) {
      if (it >= count) return false;
      qb = first + it++;
      bits = 3;
      return true;
    }
    const int a = entry(ia, ea);
    const int b = entry(ib, eb);
    const int m = a < b ? a : b;
    if (m == INT_MAX) return false;
    qb = m;
    bits = (a == m ? 1 : 0) | (b == m ? 2 : 0);
    if (a == m) ++ia;
    if (b == m) ++ib;
    return true;
  }
};

// Steps of a backward unit: every query head of the KV head's group, each with
// its query-block list.
struct BwdSteps {
  QBlockList list;
  int group, hh;

  __device__ void init(const KParams& p, int len, int kt) {
    list.init(p, len, kt);
    group = p.group;
    hh = 0;
  }
  // Next step: query head offset in the group, query block, sub-block bits.
  __device__ bool next(int& head_off, int& qb, int& bits) {
    while (hh < group) {
      if (list.next(qb, bits)) {
        head_off = hh;
        return true;
      }
      ++hh;
      list.restart();
    }
    return false;
  }
};

}  // namespace gbattn

namespace gbattn {

// The score tiles a 256-row forward unit (two 128-row query tiles, four 64-row
// query blocks) visits: the ascending union over its query blocks, each with an
// 8-bit mask of listed 64x64 sub-blocks, bit 2r + c for query block r (0-3) and
// key half c (0-1).  Query tile q uses bits 4q..4q+3 and skips a tile whose
// four bits are all clear.  Dense and causal units list every key tile up to
// the last one any of their rows sees; a query tile past the sequence end, or
// (causal) whose rows all precede a key tile, gets clear bits for it.
template <bool kSparse>
struct KvTileList2 {
  int n_dense, it, len, q0;
  const int* col;
  // Block-sparse: per query block r, the next two listed key blocks below the
  // sequence's block count (w0 < w1; INT_MAX past the list) and the index of the
  // entry after them.  A key tile holds at most two of a block's entries, so the
  // window always covers it; each call refills what it used, and those loads are
  // first read by the next call, so no call waits on its own loads.
  int s[kSparse ? 4 : 1], e[kSparse ? 4 : 1];
  int w0[kSparse ? 4 : 1], w1[kSparse ? 4 : 1];
  int nblk;
  bool causal;

  int* status;
  int n_col_blocks;

  __device__ int entry(int i, int end) const {
    if (i >= end) return INT_MAX;
    const int c = __ldg(col + i);
    if (!bounds_ok(!GBATTN_CHECKED || (c >= 0 && c < n_col_blocks), status)) return INT_MAX;
    return c < nblk ? c : INT_MAX;  // ascending: every later entry is past the end too
  }

  __device__ void init(const KParams& p, int len_, int q0_) {
    status = p.status;
    n_col_blocks = p.n_col_blocks;
    len = len_;
    q0 = q0_;
    it = 0;
    nblk = (len + 63) / 64;
    causal = p.mask == kMaskCausal;
    const int last = min(len, q0 + 2 * kTile) - 1;
    if constexpr (!kSparse) {
      n_dense = causal ? last / kTile + 1 : (len + kTile - 1) / kTile;
    } else {
      n_dense = 0;
      col = p.col_idx;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int rb = q0 / 64 + r;
        if (rb < p.n_row_blocks && rb * 64 < len) {
          s[r] = p.row_ptr[rb];
          e[r] = p.row_ptr[rb + 1];
        } else {
          s[r] = e[r] = 0;
        }
        w0[r] = entry(s[r], e[r]);
        w1[r] = entry(s[r] + 1, e[r]);
        s[r] += 2;
      }
    }
  }

  __device__ bool next(int& kt, int& bits) {
    if constexpr (!kSparse) {
      if (it >= n_dense) return false;
      kt = it++;
      bits = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int r0 = q0 + q * kTile;
        if (r0 >= len) continue;
        const int rl = min(len, r0 + kTile) - 1;
        if (causal && kt * kTile > rl) continue;
        bits |= 0xF << (4 * q);
      }
      return true;
    } else {
      const int m = min(min(w0[0], w0[1]), min(w0[2], w0[3]));
      if (m == INT_MAX) return false;
      kt = m >> 1;
      bits = 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        if ((w0[r] >> 1) != kt) continue;
        bits |= 1 << (2 * r + (w0[r] & 1));
        if ((w1[r] >> 1) == kt) {  // both key halves listed
          bits |= 1 << (2 * r + (w1[r] & 1));
          w0[r] = entry(s[r], e[r]);
          w1[r] = entry(s[r] + 1, e[r]);
          s[r] += 2;
        } else {
          w0[r] = w1[r];
          w1[r] = entry(s[r], e[r]);
          s[r] += 1;
        }
      }
      return true;
    }
  }
};

}  // namespace gbattn
