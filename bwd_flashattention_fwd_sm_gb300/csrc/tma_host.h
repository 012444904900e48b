// Host-side TMA descriptor construction for 128-row x 64-column bf16 tiles
// (128-byte swizzle) of q-like and kv-like tensors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace gbattn {

// Where a tile's rows sit among the tensor map's dimensions.
//   rows_inner = 1: dims (d, position, head, batch)  -- head-major storage
//   rows_inner = 0: dims (d, head, position, batch)  -- position-major storage
//                   (also packed variable-length tensors: position = token, batch = 1)
struct TileMap {
  CUtensorMap map;
  int rows_inner;
};

// Builds the map for the q-like (kv = false) or kv-like (kv = true) tensor at
// `base`, with boxes of `box_rows` positions x 64 columns.
cudaError_t make_tile_map(TileMap* out, const void* base, const KParams& p, bool kv, int box_rows = 128);

// Map of a 4-D byte tensor (x, row, head, batch) with x contiguous, `row_bytes`
// between rows and rows packed per head and heads per batch entry, for TMA loads
// of 128 x 128-byte boxes with the 128-byte swizzle (the FP8 operands: x = head
// dim for Q and K codes, x = key for the transposed V codes).  x and rows past
// the extents read as zero.
cudaError_t make_byte_map(TileMap* out, const void* base, long long x_extent, long long rows, long long heads,
                          long long batch, long long row_bytes);

// Map of the float32 dQ accumulator (rows laid out like a contiguous q) for
// TMA reduce-adds of box_rows x box_cols tiles (no swizzle; box_cols 0: the
// whole head dim).
//   fixed length: dims (d, position, head, batch); variable: (d, head, token, 1).
cudaError_t make_acc_map(TileMap* out, float* base, const KParams& p, int box_rows, int box_cols = 0);

}  // namespace gbattn
