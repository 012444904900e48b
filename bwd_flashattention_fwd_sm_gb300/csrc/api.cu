// C ABI of gbattn: argument validation, workspace layout, launch orchestration.
//
// Every check runs on the host before anything is queued, so a bad call never
// reaches the device (zwxr.cn CANN ops-nn article, section 2.3: declare layout,
// dtype and tiling up front, or the mismatch only shows up later; section 6.2:
// boundary indices are checked, never trusted, because an out-of-range index
// shows up as a rare hang).  Device-side failures (a bounded wait that ran out)
// go to a per-device status word, read back by attn_get_status().
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/gbattn.h"
#include "common.cuh"
#include "fp8.h"
#include "tc_kernels.h"

using namespace gbattn;

namespace {

thread_local std::string g_last_error;
// [which][start/stop]: 0 forward main kernel, 1 backward main kernel(s), 2 backward
// preprocess, 3 dQ conversion
thread_local cudaEvent_t g_timing_events[4][2] = {};

__device__ int g_status_word;  // one per device; set by kernels, cleared by attn_get_status

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int* g_status_ptr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};

attn_status_t fail(attn_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
attn_status_t fail(attn_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

// Per-device state (status word address and SM count), looked up once per device.
attn_status_t device_state(int** status, int* sms) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(ATTN_ERR_CUDA, "no usable CUDA device (%s)", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "status word lookup failed: %s", cudaGetErrorString(e));
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "SM count query failed: %s", cudaGetErrorString(e));
    g_sm_count[dev] = n;
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  *status = g_status_ptr[dev];
  *sms = g_sm_count[dev];
  return ATTN_OK;
}

unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* s = std::getenv("GBATTN_WAIT_LIMIT_MS");
    long long ms = s ? std::atoll(s) : 0;
    if (ms <= 0) ms = 4000;
    return (unsigned long long)ms * 1000000ull;
  }();
  return v;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Which kernel family serves these parameters: the tensor-core kernels for bf16
// (head_dim 64, 128 or 256; the backward at 256 takes each key tile once per
// half of the head dim), the float32-arithmetic kernels for float32 I/O.
bool use_tensor_cores(const attn_params_t* p, bool backward) {
  const bool avail = backward ? tc_bwd_available() : tc_fwd_available();
  return avail && p->dtype == ATTN_BF16 && (p->head_dim == 128 || p->head_dim == 64 || p->head_dim == 256);
}

struct Problem {
  bool varlen;
  int n_seqs;
  long long total_tokens;  // rows per head (sum of lengths)
  bool empty;
};

// Validates everything about the parameters that does not involve data pointers.
attn_status_t validate_params(const attn_params_t* p, Problem* pr) {
  g_last_error.clear();
  if (!p) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
  if (p->dtype != ATTN_F32 && p->dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, "dtype %d is not ATTN_F32 or ATTN_BF16", (int)p->dtype);
  if (p->mask != ATTN_MASK_NONE && p->mask != ATTN_MASK_CAUSAL && p->mask != ATTN_MASK_BLOCK)
    return fail(ATTN_ERR_INVALID_ARG, "mask %d is not a known mask kind", (int)p->mask);
  if (p->heads_q <= 0 || p->heads_kv <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "heads_q=%d and heads_kv=%d must be positive", p->heads_q, p->heads_kv);
  if (p->heads_q % p->heads_kv)
    return fail(ATTN_ERR_INVALID_ARG, "heads_q=%d is not a multiple of heads_kv=%d", p->heads_q, p->heads_kv);
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256)
    return fail(ATTN_ERR_UNSUPPORTED, "head_dim=%d: only 64, 128 and 256 are implemented", p->head_dim);
  if (!std::isfinite(p->scale)) return fail(ATTN_ERR_INVALID_ARG, "scale is not finite");
  if (p->seqlen < 0) return fail(ATTN_ERR_INVALID_ARG, "seqlen=%d is negative", p->seqlen);
  if (p->seqlen > (1 << 30)) return fail(ATTN_ERR_UNSUPPORTED, "seqlen=%d exceeds 2^30", p->seqlen);

  pr->varlen = p->cu_seqlens != nullptr;
  if (pr->varlen) {
    if (!p->cu_seqlens_host) return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens_host is required with cu_seqlens");
    if (p->n_seqs < 0) return fail(ATTN_ERR_INVALID_ARG, "n_seqs=%d is negative", p->n_seqs);
    if (p->cu_seqlens_host[0] != 0) return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens[0]=%d must be 0", p->cu_seqlens_host[0]);
    for (int n = 0; n < p->n_seqs; ++n) {
      const int L = p->cu_seqlens_host[n + 1] - p->cu_seqlens_host[n];
      if (L < 0) return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens decreases at %d", n);
      if (L > p->seqlen)
        return fail(ATTN_ERR_INVALID_ARG, "sequence %d has length %d > seqlen %d", n, L, p->seqlen);
    }
    if (p->mask == ATTN_MASK_BLOCK)
      return fail(ATTN_ERR_UNSUPPORTED, "block-sparse masks with variable-length batches are not implemented");
    pr->n_seqs = p->n_seqs;
    pr->total_tokens = p->cu_seqlens_host[p->n_seqs];
  } else {
    if (p->batch < 0) return fail(ATTN_ERR_INVALID_ARG, "batch=%d is negative", p->batch);
    pr->n_seqs = p->batch;
    pr->total_tokens = (long long)p->batch * p->seqlen;
  }
  pr->empty = pr->total_tokens == 0;
  if (pr->empty) return ATTN_OK;  // nothing is read or written
  // query rows over all heads are indexed in 32 bits on the device
  if (pr->total_tokens * (long long)p->heads_q >= (1ll << 31))
    return fail(ATTN_ERR_UNSUPPORTED, "%lld query rows over all heads: at most 2^31 - 1 are supported",
                pr->total_tokens * (long long)p->heads_q);

  const int align = p->dtype == ATTN_BF16 ? 8 : 4;
  const long long strides[6] = {p->q_stride_b, p->q_stride_h, p->q_stride_s,
                                p->kv_stride_b, p->kv_stride_h, p->kv_stride_s};
  const char* names[6] = {"q_stride_b", "q_stride_h", "q_stride_s", "kv_stride_b", "kv_stride_h", "kv_stride_s"};
  for (int i = 0; i < 6; ++i) {
    if (pr->varlen && (i == 0 || i == 3)) continue;
    if (strides[i] < 0 || strides[i] % align)
      return fail(ATTN_ERR_INVALID_ARG, "%s=%lld must be a non-negative multiple of %d elements",
                  names[i], strides[i], align);
  }
  if (p->q_stride_s < p->head_dim || p->kv_stride_s < p->head_dim)
    return fail(ATTN_ERR_INVALID_ARG, "row strides (q %lld, kv %lld) are smaller than head_dim %d",
                (long long)p->q_stride_s, (long long)p->kv_stride_s, p->head_dim);
  if ((p->heads_q > 1 && p->q_stride_h < p->head_dim) || (p->heads_kv > 1 && p->kv_stride_h < p->head_dim))
    return fail(ATTN_ERR_INVALID_ARG, "head strides smaller than head_dim");

  if (p->mask == ATTN_MASK_BLOCK) {
    const attn_block_mask_t* bm = p->block_mask;
    if (!bm) return fail(ATTN_ERR_INVALID_ARG, "mask is ATTN_MASK_BLOCK but block_mask is NULL");
    if (bm->block_q != kMaskBlockSize || bm->block_k != kMaskBlockSize)
      return fail(ATTN_ERR_UNSUPPORTED, "block mask tiles %dx%d: only 64x64 is implemented", bm->block_q, bm->block_k);
    const int nb = (p->seqlen + kMaskBlockSize - 1) / kMaskBlockSize;
    if (bm->n_row_blocks != nb || bm->n_col_blocks != nb)
      return fail(ATTN_ERR_INVALID_ARG, "block mask is %dx%d tiles, seqlen %d needs %dx%d",
                  bm->n_row_blocks, bm->n_col_blocks, p->seqlen, nb, nb);
    if (!bm->row_ptr_host || (bm->nnz > 0 && !bm->col_idx_host))
      return fail(ATTN_ERR_INVALID_ARG, "block mask host copies are required");
    if (!pr->empty && (!bm->row_ptr || (bm->nnz > 0 && !bm->col_idx)))
      return fail(ATTN_ERR_INVALID_ARG, "block mask device arrays are NULL");
    if (bm->row_ptr_host[0] != 0) return fail(ATTN_ERR_INVALID_ARG, "block mask row_ptr[0] must be 0");
    for (int r = 0; r < nb; ++r) {
      const int a = bm->row_ptr_host[r], e = bm->row_ptr_host[r + 1];
      if (e < a) return fail(ATTN_ERR_INVALID_ARG, "block mask row_ptr decreases at row %d", r);
      for (int i = a; i < e; ++i) {
        const int c = bm->col_idx_host[i];
        if (c < 0 || c >= nb)
          return fail(ATTN_ERR_INVALID_ARG, "block mask row %d lists column %d outside [0, %d)", r, c, nb);
        if (i > a && c <= bm->col_idx_host[i - 1])
          return fail(ATTN_ERR_INVALID_ARG, "block mask row %d columns are not strictly ascending", r);
      }
    }
    if (bm->row_ptr_host[nb] != bm->nnz)
      return fail(ATTN_ERR_INVALID_ARG, "block mask nnz=%d but row_ptr ends at %d", bm->nnz, bm->row_ptr_host[nb]);
  }
  return ATTN_OK;
}

struct Layout {
  int tile_rows;       // rows per work unit (query rows fwd, key rows bwd)
  long long n_units;
  size_t counter, units, sched, csc_ptr, csc_idx, dq_acc, delta, total;
  // backward on the tensor cores: the query-stationary dQ pass's work list
  // (forward-style units of 256 query rows), used by the deterministic mode
  long long q_units;
  size_t q_counter, q_list, q_sched;
  // forward with a split key range: parts per unit and the parts' partial results
  int n_split;
  size_t part_o, part_ml;
  // forward on the tensor cores in units of one 128-row query tile
  bool fwd_half;
};

// Parts to cut each forward unit's key range into.  With fewer units than a
// GPU has SMs, a whole unit per CTA leaves SMs idle; parts of at least
// kSplitMinTiles key tiles each (a unit's fixed costs and the combine outweigh
// shorter parts: at 16 key tiles, two parts of 8 were slower than one), up to
// four parts, for a target of kSplitTarget CTAs' worth of units (a fixed
// target, so that the workspace size needs no device query).  Dense and causal
// fixed-length forwards on the tensor cores at head_dim 64 and 128 only.
constexpr long long kSplitTarget = 128, kSplitMinTiles = 16;
int forward_split(const attn_params_t* p, const Problem& pr, long long n_units) {
  if (!use_tensor_cores(p, false) || p->head_dim == 256 || pr.varlen || p->mask == ATTN_MASK_BLOCK || n_units <= 0)
    return 1;
  const long long key_tiles = (p->seqlen + 127) / 128;
  long long ns = kSplitTarget / n_units;
  if (ns > 4) ns = 4;
  if (ns > key_tiles / kSplitMinTiles) ns = key_tiles / kSplitMinTiles;
  return ns > 1 ? (int)ns : 1;
}

// Forward units of one 128-row query tile instead of two when the two-tile
// units would be fewer than a GB300's 152 SMs (a fixed count, so that the
// workspace size needs no device query).  The CTA's two softmax warpgroups then
// split the tile's key range and merge at the end.  Measured on B1 H8 S2048
// (64 two-tile units): forward 399 -> 472 TFLOP/s; on B2 H16 S2048 causal (256
// units, more than one per SM) it lost 25%, hence the threshold.
constexpr long long kHalfUnitsBelow = 152;

KParams base_kparams(const attn_params_t* p, const Problem& pr) {
  KParams k;
  std::memset(&k, 0, sizeof(k));
  k.batch = p->batch;
  k.heads_q = p->heads_q;
  k.heads_kv = p->heads_kv;
  k.group = p->heads_q / p->heads_kv;
  k.seqlen = p->seqlen;
  k.head_dim = p->head_dim;
  k.varlen = pr.varlen ? 1 : 0;
  k.n_seqs = pr.n_seqs;
  k.cu_seqlens = p->cu_seqlens;
  k.total_tokens = pr.total_tokens;
  k.q_sb = p->q_stride_b;
  k.q_sh = p->q_stride_h;
  k.q_ss = p->q_stride_s;
  k.kv_sb = p->kv_stride_b;
  k.kv_sh = p->kv_stride_h;
  k.kv_ss = p->kv_stride_s;
  k.scale = p->scale;
  k.scale_log2 = (float)((double)p->scale * 1.4426950408889634);
  k.mask = (int)p->mask;
  if (p->mask == ATTN_MASK_BLOCK) {
    k.row_ptr = p->block_mask->row_ptr;
    k.col_idx = p->block_mask->col_idx;
    k.n_row_blocks = p->block_mask->n_row_blocks;
    k.n_col_blocks = p->block_mask->n_col_blocks;
    k.nnz = p->block_mask->nnz;
    k.causal_in_block = p->block_mask->causal_in_block ? 1 : 0;
  }
  k.wait_limit_ns = wait_limit_ns();
  return k;
}

// allow_half: the bf16 forward may take 128-row units (kHalfUnitsBelow); the
// FP8 forward and block masks keep 256-row units.
Layout layout_for(const attn_params_t* p, const Problem& pr, bool backward, bool allow_half = false) {
  Layout L;
  std::memset(&L, 0, sizeof(L));
  // tensor cores: forward units are 256 query rows (two 128-row tiles sharing
  // each K/V tile; one 128-row tile at head_dim 256), backward units 128 keys;
  // float32 path: 64 rows
  L.tile_rows = use_tensor_cores(p, backward) ? (backward ? 128 : (p->head_dim == 256 ? 128 : 256)) : 64;
  KParams k = base_kparams(p, pr);
  L.n_units = count_units(k, p->cu_seqlens_host, backward, L.tile_rows);
  L.n_split = backward ? 1 : forward_split(p, pr, L.n_units);
  if (allow_half && !backward && L.n_split == 1 && L.tile_rows == 256 && p->mask != ATTN_MASK_BLOCK &&
      L.n_units < kHalfUnitsBelow) {
    L.fwd_half = true;
    L.tile_rows = 128;
    L.n_units = count_units(k, p->cu_seqlens_host, backward, L.tile_rows);
  }
  L.n_units *= L.n_split;
  size_t off = 0;
  L.counter = off;
  off = align_up(off + sizeof(int), 256);
  L.units = off;
  off = align_up(off + sizeof(Unit) * (size_t)L.n_units, 256);
  L.sched = off;
  // work-list scratch: tile prefix, sequence order and sequence starts, then the units
  off = align_up(off + sizeof(int) * 3 * align_up((size_t)pr.n_seqs + 1, 4) + sizeof(Unit) * (size_t)L.n_units, 256);
  if (L.n_split > 1) {
    const size_t rows = (size_t)pr.total_tokens * (size_t)p->heads_q;
    L.part_o = off;
    off = align_up(off + sizeof(float) * (size_t)L.n_split * rows * (size_t)p->head_dim, 256);
    L.part_ml = off;
    off = align_up(off + sizeof(float) * 2 * (size_t)L.n_split * rows, 256);
  }
  if (backward) {
    if (p->mask == ATTN_MASK_BLOCK) {
      L.csc_ptr = off;
      off = align_up(off + sizeof(int) * ((size_t)p->block_mask->n_col_blocks + 1), 256);
      L.csc_idx = off;
      off = align_up(off + sizeof(int) * ((size_t)p->block_mask->nnz + 1), 256);
    }
    const size_t rows = (size_t)pr.total_tokens * (size_t)p->heads_q;
    L.dq_acc = off;
    off = align_up(off + sizeof(float) * rows * (size_t)p->head_dim, 256);
    L.delta = off;
    off = align_up(off + sizeof(float) * rows, 256);
    if (use_tensor_cores(p, true)) {
      L.q_units = count_units(k, p->cu_seqlens_host, false, 256);
      L.q_counter = off;
      off = align_up(off + sizeof(int), 256);
      L.q_list = off;
      off = align_up(off + sizeof(Unit) * (size_t)L.q_units, 256);
      L.q_sched = off;
      off = align_up(off + sizeof(int) * 3 * align_up((size_t)pr.n_seqs + 1, 4) + sizeof(Unit) * (size_t)L.q_units, 256);
    }
  }
  L.total = off;
  return L;
}

// The forward's split key range (parts and partial buffers) from the layout.
void set_split(KParams& kp, const Layout& L, char* ws) {
  kp.n_split = L.n_split;
  kp.fwd_half = L.fwd_half ? 1 : 0;
  if (L.n_split > 1) {
    kp.part_o = reinterpret_cast<float*>(ws + L.part_o);
    kp.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
  }
}

attn_status_t check_ptr(const void* ptr, const char* name) {
  if (!ptr) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(ptr)) return fail(ATTN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return ATTN_OK;
}

attn_status_t check_workspace(void* ws, size_t bytes, size_t need) {
  if (need == 0) return ATTN_OK;
  if (!ws) return fail(ATTN_ERR_WORKSPACE, "workspace is NULL but %zu bytes are needed", need);
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(ATTN_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (bytes < need) return fail(ATTN_ERR_WORKSPACE, "workspace has %zu bytes, %zu are needed", bytes, need);
  return ATTN_OK;
}

attn_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Row length in bytes of the transposed V codes: S rounded up to 16.
int fp8_vt_ld(int seqlen) { return (seqlen + 15) / 16 * 16; }

attn_status_t check_scale_ptr(const float* ptr, const char* name) {
  if (!ptr) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(ptr) & 3u) return fail(ATTN_ERR_INVALID_ARG, "%s is not 4-byte aligned", name);
  return ATTN_OK;
}

// The FP8 forward's extra constraints on top of validate_params.
attn_status_t validate_fp8_params(const attn_params_t* p, Problem* pr) {
  attn_status_t s = validate_params(p, pr);
  if (s != ATTN_OK) return s;
  if (p->dtype != ATTN_BF16)
    return fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward takes bf16 inputs and writes a bf16 O (dtype must be ATTN_BF16)");
  if (p->head_dim != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "head_dim=%d: the FP8 forward has head_dim 128 only", p->head_dim);
  if (p->cu_seqlens)
    return fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward takes fixed-length batches only (cu_seqlens must be NULL)");
  if (!tc_fwd_available()) return fail(ATTN_ERR_UNSUPPORTED, "this build has no tensor-core forward");
  return ATTN_OK;
}

}  // namespace

namespace gbattn {
// Lets other translation units of the library report an argument error.
void set_last_error_text(const char* text) { g_last_error = text; }
// The device status word, SM count and wait limit, for kernels in other
// translation units of the library.
attn_status_t device_status(int** status, int* sms, unsigned long long* wait_ns) {
  *wait_ns = wait_limit_ns();
  return device_state(status, sms);
}
}  // namespace gbattn

extern "C" {

size_t attn_fwd_workspace_size(const attn_params_t* p) {
  Problem pr;
  if (validate_params(p, &pr) != ATTN_OK) return SIZE_MAX;
  if (pr.empty) return 0;
  // enough for the bf16 forward and for the FP8 forward, which may lay it out differently
  return std::max(layout_for(p, pr, false, true).total, layout_for(p, pr, false, false).total);
}

size_t attn_bwd_workspace_size(const attn_params_t* p) {
  Problem pr;
  if (validate_params(p, &pr) != ATTN_OK) return SIZE_MAX;
  if (pr.empty) return 0;
  return layout_for(p, pr, true).total;
}

attn_status_t attn_fwd(const attn_params_t* p, const void* q, const void* k, const void* v, void* o,
                       float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  Problem pr;
  attn_status_t s = validate_params(p, &pr);
  if (s != ATTN_OK) return s;
  if (pr.empty) return ATTN_OK;
  if ((s = check_ptr(q, "q")) || (s = check_ptr(k, "k")) || (s = check_ptr(v, "v")) ||
      (s = check_ptr(o, "o")) || (s = check_ptr(lse, "lse")))
    return s;
  const Layout L = layout_for(p, pr, false, true);
  if ((s = check_workspace(workspace, workspace_bytes, L.total))) return s;

  int* status = nullptr;
  int sms = 0;
  if ((s = device_state(&status, &sms))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);

  KParams kp = base_kparams(p, pr);
  kp.q = q;
  kp.k = k;
  kp.v = v;
  kp.o = o;
  kp.lse = lse;
  kp.status = status;
  kp.units = reinterpret_cast<const Unit*>(ws + L.units);
  kp.n_units = (int)L.n_units;
  kp.unit_counter = reinterpret_cast<int*>(ws + L.counter);
  set_split(kp, L, ws);

  cudaError_t e = launch_build_worklist(kp, false, L.tile_rows, reinterpret_cast<Unit*>(ws + L.units),
                                        (int)L.n_units, reinterpret_cast<int*>(ws + L.sched), st);
  if (e != cudaSuccess) return cuda_fail(e, "work-list launch");
  if (g_timing_events[0][0] && (e = cudaEventRecord(g_timing_events[0][0], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  if (use_tensor_cores(p, false)) e = launch_tc_fwd(kp, sms, st);
  else e = launch_simt_fwd(kp, p->dtype == ATTN_BF16, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (kp.n_split > 1 && (e = launch_fwd_combine(kp, st)) != cudaSuccess) return cuda_fail(e, "combine launch");
  if (g_timing_events[0][1] && (e = cudaEventRecord(g_timing_events[0][1], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  return ATTN_OK;
}

// ---------------------------------------------------------------------------
// FP8 (e4m3) forward
// ---------------------------------------------------------------------------

attn_status_t attn_quantize_fp8(const attn_params_t* p, const void* q, const void* k, const void* v, void* q8,
                                void* k8, void* v8t, float* q_scale, float* k_scale, float* v_scale, void* stream) {
  Problem pr;
  attn_status_t s = validate_fp8_params(p, &pr);
  if (s != ATTN_OK) return s;
  if (pr.empty) return ATTN_OK;
  if ((s = check_ptr(q, "q")) || (s = check_ptr(k, "k")) || (s = check_ptr(v, "v")) || (s = check_ptr(q8, "q8")) ||
      (s = check_ptr(k8, "k8")) || (s = check_ptr(v8t, "v8t")) || (s = check_scale_ptr(q_scale, "q_scale")) ||
      (s = check_scale_ptr(k_scale, "k_scale")) || (s = check_scale_ptr(v_scale, "v_scale")))
    return s;
  Fp8QuantJob jobs[3];
  jobs[0] = {static_cast<const __nv_bfloat16*>(q), p->q_stride_b, p->q_stride_h, p->q_stride_s,
             static_cast<uint8_t*>(q8), q_scale, p->heads_q, 0};
  jobs[1] = {static_cast<const __nv_bfloat16*>(k), p->kv_stride_b, p->kv_stride_h, p->kv_stride_s,
             static_cast<uint8_t*>(k8), k_scale, p->heads_kv, 0};
  jobs[2] = {static_cast<const __nv_bfloat16*>(v), p->kv_stride_b, p->kv_stride_h, p->kv_stride_s,
             static_cast<uint8_t*>(v8t), v_scale, p->heads_kv, 1};
  cudaError_t e = launch_quant_fp8(jobs, p->batch, p->seqlen, fp8_vt_ld(p->seqlen), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantisation launch");
  return ATTN_OK;
}

attn_status_t attn_fwd_fp8(const attn_params_t* p, const void* q8, const void* k8, const void* v8t,
                           const float* q_scale, const float* k_scale, const float* v_scale, void* o, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream) {
  Problem pr;
  attn_status_t s = validate_fp8_params(p, &pr);
  if (s != ATTN_OK) return s;
  if (pr.empty) return ATTN_OK;
  if ((s = check_ptr(q8, "q8")) || (s = check_ptr(k8, "k8")) || (s = check_ptr(v8t, "v8t")) ||
      (s = check_scale_ptr(q_scale, "q_scale")) || (s = check_scale_ptr(k_scale, "k_scale")) ||
      (s = check_scale_ptr(v_scale, "v_scale")) || (s = check_ptr(o, "o")) || (s = check_ptr(lse, "lse")))
    return s;
  const Layout L = layout_for(p, pr, false);
  if ((s = check_workspace(workspace, workspace_bytes, L.total))) return s;
  int* status = nullptr;
  int sms = 0;
  if ((s = device_state(&status, &sms))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);

  KParams kp = base_kparams(p, pr);
  kp.o = o;
  kp.lse = lse;
  kp.status = status;
  kp.units = reinterpret_cast<const Unit*>(ws + L.units);
  kp.n_units = (int)L.n_units;
  kp.unit_counter = reinterpret_cast<int*>(ws + L.counter);
  set_split(kp, L, ws);
  cudaError_t e = launch_build_worklist(kp, false, L.tile_rows, reinterpret_cast<Unit*>(ws + L.units),
                                        (int)L.n_units, reinterpret_cast<int*>(ws + L.sched), st);
  if (e != cudaSuccess) return cuda_fail(e, "work-list launch");
  Fp8Operands f;
  f.q8 = static_cast<const uint8_t*>(q8);
  f.k8 = static_cast<const uint8_t*>(k8);
  f.v8t = static_cast<const uint8_t*>(v8t);
  f.qs = q_scale;
  f.ks = k_scale;
  f.vs = v_scale;
  f.ld_t = fp8_vt_ld(p->seqlen);
  if (g_timing_events[0][0] && (e = cudaEventRecord(g_timing_events[0][0], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  if ((e = launch_tc_fwd_fp8(kp, sms, st, f)) != cudaSuccess) return cuda_fail(e, "FP8 forward launch");
  if (kp.n_split > 1 && (e = launch_fwd_combine(kp, st)) != cudaSuccess) return cuda_fail(e, "combine launch");
  if (g_timing_events[0][1] && (e = cudaEventRecord(g_timing_events[0][1], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  return ATTN_OK;
}

}  // extern "C"

namespace {

// The backward pass.  deterministic: dK and dV from the dK/dV-stationary pass
// without its dQ product, then dQ from the query-stationary pass (fixed sum
// order, no accumulator); otherwise dQ is added into the float32 accumulator
// by L2 reductions and converted at the end.
attn_status_t bwd_impl(const attn_params_t* p, const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                       size_t workspace_bytes, void* stream, bool deterministic) {
  Problem pr;
  attn_status_t s = validate_params(p, &pr);
  if (s != ATTN_OK) return s;
  if (deterministic && (!use_tensor_cores(p, true) || p->head_dim == 256))
    return fail(ATTN_ERR_UNSUPPORTED,
                "the deterministic backward runs on the tensor-core path only (bf16, head_dim 64 or 128)");
  if (pr.empty) return ATTN_OK;
  if ((s = check_ptr(q, "q")) || (s = check_ptr(k, "k")) || (s = check_ptr(v, "v")) ||
      (s = check_ptr(o, "o")) || (s = check_ptr(dout, "dout")) || (s = check_ptr(lse, "lse")) ||
      (s = check_ptr(dq, "dq")) || (s = check_ptr(dk, "dk")) || (s = check_ptr(dv, "dv")))
    return s;
  const Layout L = layout_for(p, pr, true);
  if ((s = check_workspace(workspace, workspace_bytes, L.total))) return s;

  int* status = nullptr;
  int sms = 0;
  if ((s = device_state(&status, &sms))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const bool bf16 = p->dtype == ATTN_BF16;

  KParams kp = base_kparams(p, pr);
  kp.q = q;
  kp.k = k;
  kp.v = v;
  kp.o = const_cast<void*>(o);
  kp.lse = const_cast<float*>(lse);
  kp.dout = dout;
  kp.dq = dq;
  kp.dk = dk;
  kp.dv = dv;
  kp.status = status;
  kp.dq_accum = deterministic ? nullptr : reinterpret_cast<float*>(ws + L.dq_acc);
  kp.delta = reinterpret_cast<float*>(ws + L.delta);
  kp.units = reinterpret_cast<const Unit*>(ws + L.units);
  kp.n_units = (int)L.n_units;
  kp.unit_counter = reinterpret_cast<int*>(ws + L.counter);

  cudaError_t e = cudaSuccess;
  if (p->mask == ATTN_MASK_BLOCK) {
    kp.csc_ptr = reinterpret_cast<int*>(ws + L.csc_ptr);
    kp.csc_idx = reinterpret_cast<int*>(ws + L.csc_idx);
    e = launch_csr_to_csc(kp, reinterpret_cast<int*>(ws + L.csc_ptr), reinterpret_cast<int*>(ws + L.csc_idx), st);
    if (e != cudaSuccess) return cuda_fail(e, "mask transpose launch");
  }
  e = launch_build_worklist(kp, true, L.tile_rows, reinterpret_cast<Unit*>(ws + L.units), (int)L.n_units,
                            reinterpret_cast<int*>(ws + L.sched), st);
  if (e != cudaSuccess) return cuda_fail(e, "work-list launch");
  KParams kq = kp;  // the dQ pass: forward-style work list
  if (deterministic) {
    kq.units = reinterpret_cast<const Unit*>(ws + L.q_list);
    kq.n_units = (int)L.q_units;
    kq.unit_counter = reinterpret_cast<int*>(ws + L.q_counter);
    e = launch_build_worklist(kq, false, 256, reinterpret_cast<Unit*>(ws + L.q_list), (int)L.q_units,
                              reinterpret_cast<int*>(ws + L.q_sched), st);
    if (e != cudaSuccess) return cuda_fail(e, "work-list launch");
  }
  if (g_timing_events[2][0] && (e = cudaEventRecord(g_timing_events[2][0], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  e = launch_bwd_preprocess(kp, bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "preprocess launch");
  if (g_timing_events[2][1] && (e = cudaEventRecord(g_timing_events[2][1], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  if (g_timing_events[1][0] && (e = cudaEventRecord(g_timing_events[1][0], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  if (use_tensor_cores(p, true))
    e = p->head_dim == 256 ? launch_tc_bwd256(kp, sms, st) : launch_tc_bwd(kp, sms, st, !deterministic);
  else e = launch_simt_bwd(kp, bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  if (deterministic && (e = launch_tc_dq(kq, sms, st)) != cudaSuccess) return cuda_fail(e, "dQ pass launch");
  if (g_timing_events[1][1] && (e = cudaEventRecord(g_timing_events[1][1], st)) != cudaSuccess)
    return cuda_fail(e, "timing event");
  if (!deterministic) {
    if (g_timing_events[3][0] && (e = cudaEventRecord(g_timing_events[3][0], st)) != cudaSuccess)
      return cuda_fail(e, "timing event");
    e = launch_dq_convert(kp, bf16, st);
    if (e != cudaSuccess) return cuda_fail(e, "dQ conversion launch");
    if (g_timing_events[3][1] && (e = cudaEventRecord(g_timing_events[3][1], st)) != cudaSuccess)
      return cuda_fail(e, "timing event");
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_bwd(const attn_params_t* p, const void* q, const void* k, const void* v,
                       const void* o, const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(p, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, stream, false);
}

attn_status_t attn_bwd_deterministic(const attn_params_t* p, const void* q, const void* k, const void* v,
                                     const void* o, const void* dout, const float* lse, void* dq, void* dk,
                                     void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(p, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, stream, true);
}

attn_status_t attn_get_status(void* stream) {
  int* status = nullptr;
  int sms = 0;
  attn_status_t s = device_state(&status, &sms);
  if (s != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int host = 0;
  e = cudaMemcpy(&host, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (host != 0) {
    const int zero = 0;
    e = cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
  }
  return static_cast<attn_status_t>(host);
}

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_DEVICE_BOUNDS: return "ATTN_ERR_DEVICE_BOUNDS";
  }
  return "ATTN_ERR_UNKNOWN";
}

const char* attn_last_error(void) { return g_last_error.c_str(); }

attn_status_t attn_set_timing_events(int which, void* start, void* stop) {
  if (which < 0 || which > 3) return fail(ATTN_ERR_INVALID_ARG, "timing hook %d is not 0, 1, 2 or 3", which);
  g_timing_events[which][0] = static_cast<cudaEvent_t>(start);
  g_timing_events[which][1] = static_cast<cudaEvent_t>(stop);
  return ATTN_OK;
}

const char* attn_version(void) { return GBATTN_CHECKED ? "gbattn 0.1.0 sm_103a checked" : "gbattn 0.1.0 sm_103a"; }

attn_status_t attn_selftest_bounded_wait(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 1000000u)
    return fail(ATTN_ERR_INVALID_ARG, "limit_us=%u: must be in [1, 1000000]", limit_us);
  int* status = nullptr;
  int sms = 0;
  attn_status_t s = device_state(&status, &sms);
  if (s != ATTN_OK) return s;
  cudaError_t e = launch_wait_probe(status, (unsigned long long)limit_us * 1000ull, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
  return ATTN_OK;
}

}  // extern "C"
