// Internal definitions shared by the kernels and the C ABI layer of gbattn.
// Not part of the public interface (that is include/gbattn.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbattn {

// Device status codes (same values as attn_status_t).
enum : int { kStatusOk = 0, kStatusTimeout = 5, kStatusBounds = 6 };

// Mask kinds (same values as attn_mask_t).
enum : int { kMaskNone = 0, kMaskCausal = 1, kMaskBlock = 2 };

constexpr int kMaskBlockSize = 64;  // block-sparse tile edge (query and key)

// A work unit: one output tile of one head of one sequence.
//   forward : (sequence, query head, query tile)
//   backward: (sequence, kv head,   key tile)
// `cost` is the number of 64x64 score tiles the unit computes (for ordering only).
struct Unit {
  int seq, head, tile, cost;
};

// Everything a kernel needs, resolved on the host.  Element strides are in
// elements of the I/O type; the head dimension is contiguous.
struct KParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;

  int batch, heads_q, heads_kv, group, seqlen, head_dim;
  int varlen, n_seqs;           // variable length: sequence starts in cu_seqlens
  const int* cu_seqlens;        // device, [n_seqs + 1] (NULL for fixed length)
  long long total_tokens;       // variable length: T

  long long q_sb, q_sh, q_ss;   // q, o, dout, dq strides
  long long kv_sb, kv_sh, kv_ss;// k, v, dk, dv strides

  float scale;       // score scale
  float scale_log2;  // scale * log2(e): exp(scale * x) = exp2(scale_log2 * x)

  int mask;
  const int* row_ptr;   // block mask CSR (device)
  const int* col_idx;
  int n_row_blocks, n_col_blocks, causal_in_block;
  int nnz;              // block mask: listed tiles (the host copy's count)
  const int* csc_ptr;   // block mask transposed: query blocks per key block (device)
  const int* csc_idx;

  float* dq_accum;      // backward: float32 dQ accumulator, rows like q, contiguous D
  float* delta;         // backward: D_i = <dO_i, O_i>, laid out like lse

  const Unit* units;
  int n_units;
  int* unit_counter;    // persistent kernels: next unit to take (zeroed by the work-list build)

  // Forward with the key range split (few units): each unit's key tiles are cut
  // into n_split parts, one work-list entry each (its part in Unit::cost once the
  // list is ordered); each part writes its unnormalised O (float32
  // [n_split][rows][D]) and its row max and sum (log2 units, [n_split][rows][2])
  // for the combine kernel.  n_split <= 1: no split.
  int n_split;
  float* part_o;
  float* part_ml;
  // Forward on the tensor cores with few units: units of one 128-row query
  // tile instead of two (Unit::tile counts 128-row tiles); the kernel leaves
  // the pair's other tile idle.
  int fwd_half;

  int* status;               // device status word
  unsigned long long wait_limit_ns;  // bounded-wait limit for pipeline barriers
};

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Checked builds
// ---------------------------------------------------------------------------
//
// A library built with GBATTN_CHECKED=1 compares every index it computes on the
// device (work-list entries, block-mask entries, the positions, heads and batch
// entries behind each tile load, reduce-add, row read and row store) with the
// extent of the tensor it addresses before the access.  A failed check records
// kStatusBounds in the status word and the access is skipped (a tile load whose
// start is out of range still runs, since the tensor map clips it; its data are
// not used as a valid result).  The host validates all arguments before any
// launch, so with valid arguments no check fails; the checks catch a device-side
// index bug instead of letting it read or write another tensor's memory.  Other
// builds compile every check to `true`.
#ifndef GBATTN_CHECKED
#define GBATTN_CHECKED 0
#endif

__device__ __forceinline__ bool bounds_ok(bool ok, int* status) {
#if GBATTN_CHECKED
  if (!ok) set_status(status, kStatusBounds);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}

// Extents of the tensors the kernels address, from the launch parameters:
// position `pos` (relative to the sequence start s_tok0) of batch entry b and
// head h lies inside a q-like (heads = heads_q) or kv-like (heads_kv) tensor.
__host__ __device__ inline bool row_in_range(int varlen, int batch, long long seqlen, long long total_tokens,
                                             int heads, int b, int h, long long s_tok0, long long pos) {
  const long long rows = varlen ? total_tokens : seqlen;
  const int nb = varlen ? 1 : batch;
  const long long r = s_tok0 + pos;
  return b >= 0 && b < nb && h >= 0 && h < heads && pos >= 0 && r >= 0 && r < rows;
}

// ---------------------------------------------------------------------------
// Sequence geometry
// ---------------------------------------------------------------------------

struct SeqInfo {
  int len;             // number of positions
  long long tok0;      // variable length: first token; fixed: 0
  int b;               // fixed length: batch index; variable: 0
};

__host__ __device__ inline SeqInfo seq_info(const KParams& p, int n) {
  SeqInfo s;
  if (p.varlen) {
    int a = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
    s.len = e - a;
    s.tok0 = a;
    s.b = 0;
  } else {
    s.len = p.seqlen;
    s.tok0 = 0;
    s.b = n;
  }
  return s;
}

// Element offset of (sequence, head, position) in a q-like tensor.
__device__ __forceinline__ long long q_off(const KParams& p, const SeqInfo& s, int h, int pos) {
  return (long long)s.b * p.q_sb + (long long)h * p.q_sh + (s.tok0 + pos) * p.q_ss;
}
__device__ __forceinline__ long long kv_off(const KParams& p, const SeqInfo& s, int h, int pos) {
  return (long long)s.b * p.kv_sb + (long long)h * p.kv_sh + (s.tok0 + pos) * p.kv_ss;
}
// Index into lse / delta.
__device__ __forceinline__ long long row_index(const KParams& p, const SeqInfo& s, int h, int pos) {
  if (p.varlen) return (long long)h * p.total_tokens + s.tok0 + pos;
  return ((long long)s.b * p.heads_q + h) * p.seqlen + pos;
}
// Checked-build guards for one row of a q-like / kv-like tensor (see above).
__device__ __forceinline__ bool check_q_row(const KParams& p, const SeqInfo& s, int h, long long pos) {
  return bounds_ok(!GBATTN_CHECKED ||
                       row_in_range(p.varlen, p.batch, p.seqlen, p.total_tokens, p.heads_q, s.b, h, s.tok0, pos),
                   p.status);
}
__device__ __forceinline__ bool check_kv_row(const KParams& p, const SeqInfo& s, int h, long long pos) {
  return bounds_ok(!GBATTN_CHECKED ||
                       row_in_range(p.varlen, p.batch, p.seqlen, p.total_tokens, p.heads_kv, s.b, h, s.tok0, pos),
                   p.status);
}
// A work-list unit names an existing sequence and head (q heads for the forward,
// kv heads for the backward) and a tile that starts inside the sequence.
__device__ __forceinline__ bool check_unit(const KParams& p, const Unit& u, bool backward, int tile_rows) {
  if (!GBATTN_CHECKED) return true;
  const int n_seq = p.varlen ? p.n_seqs : p.batch;
  bool ok = u.seq >= 0 && u.seq < n_seq && u.head >= 0 && u.head < (backward ? p.heads_kv : p.heads_q) &&
            u.tile >= 0;
  if (ok) {
    const SeqInfo s = seq_info(p, u.seq);
    ok = (long long)u.tile * tile_rows < s.len;
  }
  return bounds_ok(ok, p.status);
}
// A block-mask entry (a 64-row or 64-column block index) lies inside the mask.
__device__ __forceinline__ bool check_block(const KParams& p, int blk, int n_blocks) {
  return bounds_ok(!GBATTN_CHECKED || (blk >= 0 && blk < n_blocks), p.status);
}

// Element offset of a row of the float32 dQ accumulator (contiguous, like q).
__device__ __forceinline__ long long dqacc_off(const KParams& p, const SeqInfo& s, int h, int pos) {
  if (p.varlen) return ((s.tok0 + pos) * p.heads_q + h) * (long long)p.head_dim;
  return (((long long)s.b * p.heads_q + h) * p.seqlen + pos) * (long long)p.head_dim;
}

// ---------------------------------------------------------------------------
// Element conversion
// ---------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <class T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// max(a, b, c) in one instruction (the three-input max.f32 of sm_100 and later)
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Host-side launchers (one per kernel family)
// ---------------------------------------------------------------------------

// Work list: units for the forward (tile = query rows per unit) or the
// backward (tile = key rows per unit), ordered by decreasing cost.
cudaError_t launch_build_worklist(const KParams& p, bool backward, int tile_rows, Unit* units,
                                  int n_units, int* scratch, cudaStream_t st);
// Block mask: per key block, the ascending list of query blocks that list it.
cudaError_t launch_csr_to_csc(const KParams& p, int* csc_ptr, int* csc_idx, cudaStream_t st);

// Forward with a split key range: O and LSE from the parts' partial results.
cudaError_t launch_fwd_combine(const KParams& p, cudaStream_t st);

// Backward preprocess (D_i and zeroed dQ accumulator) and dQ conversion.
cudaError_t launch_bwd_preprocess(const KParams& p, bool bf16, cudaStream_t st);
cudaError_t launch_dq_convert(const KParams& p, bool bf16, cudaStream_t st);
// One warp waits, through the kernels' bounded mbarrier wait, on a barrier that
// nothing completes: after limit_ns it records kStatusTimeout in *status and
// returns (a check of the device-side timeout path).
cudaError_t launch_wait_probe(int* status, unsigned long long limit_ns, cudaStream_t st);

// float32-arithmetic SIMT kernels (any dtype, D in {64, 128, 256}).
cudaError_t launch_simt_fwd(const KParams& p, bool bf16, cudaStream_t st);
cudaError_t launch_simt_bwd(const KParams& p, bool bf16, cudaStream_t st);

// Units per query tile for a given tile height (host helper).
long long count_units(const KParams& p, const int* cu_host, bool backward, int tile_rows);

}  // namespace gbattn
