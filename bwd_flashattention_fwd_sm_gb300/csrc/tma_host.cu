#include "tma_host.h"

#include <cstring>
#include <mutex>

namespace gbattn {

namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static std::once_flag once;
  static EncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}

}  // namespace

cudaError_t make_tile_map(TileMap* out, const void* base, const KParams& p, bool kv, int box_rows) {
  EncodeFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const long long sh = kv ? p.kv_sh : p.q_sh;
  const long long ss = kv ? p.kv_ss : p.q_ss;
  const long long sb = kv ? p.kv_sb : p.q_sb;
  const long long H = kv ? p.heads_kv : p.heads_q;
  const long long E = 2;  // bf16
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  if (p.varlen) {
    out->rows_inner = 0;
    dims[0] = p.head_dim; dims[1] = H; dims[2] = p.total_tokens; dims[3] = 1;
    strides[0] = (H > 1 ? sh : p.head_dim) * E;
    strides[1] = ss * E;
    strides[2] = ss * E * (p.total_tokens > 0 ? p.total_tokens : 1);
    box[0] = 64; box[1] = 1; box[2] = box_rows; box[3] = 1;
  } else if (H == 1 || ss <= sh) {
    out->rows_inner = 1;
    dims[0] = p.head_dim; dims[1] = p.seqlen; dims[2] = H; dims[3] = p.batch;
    strides[0] = ss * E;
    strides[1] = (H > 1 ? sh : ss * p.seqlen) * E;
    strides[2] = (p.batch > 1 ? sb : strides[1] / E * H) * E;
    box[0] = 64; box[1] = box_rows; box[2] = 1; box[3] = 1;
  } else {
    out->rows_inner = 0;
    dims[0] = p.head_dim; dims[1] = H; dims[2] = p.seqlen; dims[3] = p.batch;
    strides[0] = sh * E;
    strides[1] = ss * E;
    strides[2] = (p.batch > 1 ? sb : ss * p.seqlen) * E;
    box[0] = 64; box[1] = 1; box[2] = box_rows; box[3] = 1;
  }
  std::memset(&out->map, 0, sizeof(out->map));
  CUresult r = enc(&out->map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_byte_map(TileMap* out, const void* base, long long x_extent, long long rows, long long heads,
                          long long batch, long long row_bytes) {
  EncodeFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (x_extent < 1 || rows < 1 || heads < 1 || batch < 1 || row_bytes % 16) return cudaErrorInvalidValue;
  out->rows_inner = 1;
  cuuint64_t dims[4] = {(cuuint64_t)x_extent, (cuuint64_t)rows, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)row_bytes, (cuuint64_t)(row_bytes * rows),
                           (cuuint64_t)(row_bytes * rows * heads)};
  cuuint32_t box[4] = {128, 128, 1, 1}, estr[4] = {1, 1, 1, 1};
  std::memset(&out->map, 0, sizeof(out->map));
  CUresult r = enc(&out->map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_acc_map(TileMap* out, float* base, const KParams& p, int box_rows, int box_cols) {
  EncodeFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const long long D = p.head_dim, H = p.heads_q, E = 4;
  const cuuint32_t bc = (cuuint32_t)(box_cols > 0 ? box_cols : D);
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  if (p.varlen) {
    out->rows_inner = 0;
    dims[0] = D; dims[1] = H; dims[2] = p.total_tokens; dims[3] = 1;
    strides[0] = D * E;
    strides[1] = H * D * E;
    strides[2] = H * D * E * (p.total_tokens > 0 ? p.total_tokens : 1);
    box[0] = bc; box[1] = 1; box[2] = box_rows; box[3] = 1;
  } else {
    out->rows_inner = 1;
    dims[0] = D; dims[1] = p.seqlen; dims[2] = H; dims[3] = p.batch;
    strides[0] = D * E;
    strides[1] = (long long)p.seqlen * D * E;
    strides[2] = H * p.seqlen * D * E;
    box[0] = bc; box[1] = box_rows; box[2] = 1; box[3] = 1;
  }
  std::memset(&out->map, 0, sizeof(out->map));
  CUresult r = enc(&out->map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gbattn
