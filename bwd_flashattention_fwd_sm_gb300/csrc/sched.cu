// Work lists and block-mask metadata, built on the device.
//
// Uneven work is the rule here: causal masks, skipped tiles and sequences of
// different lengths give query (or key) tiles very different amounts of work,
// and a core that draws only short tiles idles while another finishes a long
// one (smzdm contest article, section 02 on splitting work across cores, and
// section 03 on sparsity).  Handing out work dynamically, longest first, beats
// a static even split (zwxr.cn CANN ops-nn article, section 4.2).  The work
// list below orders units by decreasing cost; the kernels take units in that
// order, so the longest ones start first.  The list is built on the device in
// one small launch, so no slow host-side statistics step precedes the kernels
// (smzdm article, the team that removed an idle 147 us start-up step).
#include "common.cuh"

namespace gbattn {

namespace {

constexpr int kThreads = 1024;
constexpr int kBuckets = 4096;  // costs are clamped into this many buckets
constexpr int kTileGroup = 16;  // fixed-length causal backward: tiles per group, at most (see below)

__device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Number of distinct entries in the union of ascending lists [a0,a1) and [b0,b1)
// of `idx`, counting only values < limit.
__device__ int union_count(const int* idx, int a0, int a1, int b0, int b1, int limit) {
  int n = 0;
  while (a0 < a1 || b0 < b1) {
    int x = a0 < a1 ? idx[a0] : INT_MAX;
    int y = b0 < b1 ? idx[b0] : INT_MAX;
    int m = x < y ? x : y;
    if (m >= limit) break;
    ++n;
    if (x == m) ++a0;
    if (y == m) ++b0;
  }
  return n;
}

// Cost (in 64x64 tiles) of one unit.
__device__ int unit_cost(const KParams& p, bool backward, int tile_rows, int len, int t) {
  const int nb = cdiv(len, kMaskBlockSize);  // 64-blocks in this sequence
  const int r0 = t * tile_rows;
  const int r1 = min(len, r0 + tile_rows);
  const int b0 = r0 / kMaskBlockSize, b1 = cdiv(r1, kMaskBlockSize);  // blocks of this tile
  if (!backward) {
    if (p.mask == kMaskNone) return nb;
    if (p.mask == kMaskCausal) return b1;
    // block mask: union of the listed key blocks of the tile's query blocks
    if (b1 - b0 == 1) return union_count(p.col_idx, p.row_ptr[b0], p.row_ptr[b0 + 1], 0, 0, nb);
    int c = 0;
    // tiles of more than two blocks are not used; fall back to a sum (upper bound)
    if (b1 - b0 == 2)
      return union_count(p.col_idx, p.row_ptr[b0], p.row_ptr[b0 + 1], p.row_ptr[b0 + 1],
                         p.row_ptr[b0 + 2], nb);
    for (int b = b0; b < b1; ++b) c += p.row_ptr[b + 1] - p.row_ptr[b];
    return c;
  }
  int per_head;
  if (p.mask == kMaskNone) per_head = nb;
  else if (p.mask == kMaskCausal) per_head = nb - b0;
  else if (b1 - b0 == 1) per_head = union_count(p.csc_idx, p.csc_ptr[b0], p.csc_ptr[b0 + 1], 0, 0, nb);
  else if (b1 - b0 == 2)
    per_head = union_count(p.csc_idx, p.csc_ptr[b0], p.csc_ptr[b0 + 1], p.csc_ptr[b0 + 1],
                           p.csc_ptr[b0 + 2], nb);
  else {
    per_head = 0;
    for (int b = b0; b < b1; ++b) per_head += p.csc_ptr[b + 1] - p.csc_ptr[b];
  }
  return per_head * p.group;
}

// Block-wide exclusive scan of one int per thread (kThreads threads).
__device__ int block_exclusive_scan(int x, int* smem, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) smem[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (kThreads / 32) ? smem[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    smem[32 + lane] = wi - w;
    if (lane == 31) smem[64] = wi;
  }
  __syncthreads();
  int r = smem[32 + warp] + incl - x;
  *total = smem[64];
  __syncthreads();
  return r;
}

// Turns hist (counts per cost bucket) into the first list position of each
// bucket, highest bucket first.  All threads of the block call it.
__device__ void bucket_starts_desc(int* hist, int* scan_smem) {
  const int tid = threadIdx.x;
  const int per = kBuckets / kThreads;  // buckets per thread, thread 0 owns the highest
  int vals[kBuckets / kThreads];
  int s = 0;
  for (int i = 0; i < per; ++i) {
    vals[i] = hist[kBuckets - 1 - (tid * per + i)];
    s += vals[i];
  }
  int tot;
  int b = block_exclusive_scan(s, scan_smem, &tot);
  for (int i = 0; i < per; ++i) {
    hist[kBuckets - 1 - (tid * per + i)] = b;
    b += vals[i];
  }
  __syncthreads();
}

// Words of int scratch before the unit array: tile prefix, sequence order and
// sequence starts, [n_seqs + 1] each, rounded to 4.
__host__ __device__ inline int sched_ints(int n_seqs) { return 3 * ((n_seqs + 1 + 3) & ~3); }

// One block.  scratch: [n_seqs + 1] tile prefix, [n_seqs + 1] sequence order,
// [n_seqs + 1] sequence starts (each rounded to 4 ints), then [n_units]
// unsorted units (as int4).
__global__ void __launch_bounds__(kThreads) k_build_worklist(KParams p, int backward, int tile_rows,
                                                           Unit* out, int n_units, int* scratch) {
  __shared__ int hist[kBuckets];
  __shared__ int scan_smem[72];
  const int tid = threadIdx.x;
  const int n_seqs = p.varlen ? p.n_seqs : p.batch;
  const int heads = backward ? p.heads_kv : p.heads_q;
  const int seq_words = (n_seqs + 1 + 3) & ~3;
  int* prefix = scratch;                                  // [n_seqs + 1]
  int* seq_order = scratch + seq_words;                   // [n_seqs]
  int* seq_start = scratch + 2 * seq_words;               // [n_seqs]
  Unit* tmp = reinterpret_cast<Unit*>(scratch + sched_ints(n_seqs));

  // 1. prefix of tiles per sequence (chunked block scan)
  const int chunk = cdiv(n_seqs, kThreads);
  int local = 0;
  for (int n = tid * chunk; n < min(n_seqs, (tid + 1) * chunk); ++n)
    local += cdiv(seq_info(p, n).len, tile_rows);
  int total;
  int base = block_exclusive_scan(local, scan_smem, &total);
  // The device's sequence lengths give as many units as the host counted from
  // its copy (a checked build stops here otherwise: the list would not fit).
  if (!bounds_ok(!GBATTN_CHECKED ||
                     (long long)total * heads * (backward ? 1 : max(1, p.n_split)) == (long long)n_units,
                 p.status)) {
    if (tid == 0 && p.unit_counter) *p.unit_counter = n_units;  // the kernels take no unit
    return;
  }
  for (int n = tid * chunk; n < min(n_seqs, (tid + 1) * chunk); ++n) {
    prefix[n] = base;
    base += cdiv(seq_info(p, n).len, tile_rows);
  }
  if (tid == 0) {
    prefix[n_seqs] = total;
    if (p.unit_counter) *p.unit_counter = 0;
  }
  for (int i = tid; i < kBuckets; i += kThreads) hist[i] = 0;
  __syncthreads();

  if (p.varlen) {
    // Packed sequences: sequence by sequence, longest first (a sequence's cost
    // grows with its length, for every mask a packed batch takes), each head by
    // head and each head's tiles longest first (causal: tile 0 first backward,
    // the last tile first forward).  Units of one sequence and head then run at
    // the same time and share its Q and dO (or K and V) in L2; ordered by unit
    // cost alone, the units running at once came from hundreds of different
    // (sequence, head) pairs and shared nothing.
    for (int n = tid; n < n_seqs; n += kThreads)
      atomicAdd(&hist[min(prefix[n + 1] - prefix[n], kBuckets - 1)], 1);
    __syncthreads();
    bucket_starts_desc(hist, scan_smem);
    for (int n = tid; n < n_seqs; n += kThreads)
      seq_order[atomicAdd(&hist[min(prefix[n + 1] - prefix[n], kBuckets - 1)], 1)] = n;
    __syncthreads();
    int local2 = 0;
    for (int i = tid * chunk; i < min(n_seqs, (tid + 1) * chunk); ++i) {
      const int n = seq_order[i];
      local2 += heads * (prefix[n + 1] - prefix[n]);
    }
    int total2;
    int base2 = block_exclusive_scan(local2, scan_smem, &total2);
    for (int i = tid * chunk; i < min(n_seqs, (tid + 1) * chunk); ++i) {
      const int n = seq_order[i];
      seq_start[n] = base2;
      base2 += heads * (prefix[n + 1] - prefix[n]);
    }
    __syncthreads();
    for (int u = tid; u < n_units; u += kThreads) {
      int lo = 0, hi = n_seqs - 1;
      while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((long long)heads * prefix[mid] <= u) lo = mid; else hi = mid - 1;
      }
      const int n = lo, tiles = prefix[n + 1] - prefix[n];
      const int local = u - heads * prefix[n];
      const int h = local / tiles, t = local % tiles;
      const int len = seq_info(p, n).len;
      Unit un;
      un.seq = n;
      un.head = h;
      un.tile = t;
      un.cost = (t * tile_rows < len) ? unit_cost(p, backward, tile_rows, len, t) : 0;
      const int r = (p.mask == kMaskCausal && !backward) ? tiles - 1 - t : t;
      const int at = seq_start[n] + h * tiles + r;
      if (bounds_ok(!GBATTN_CHECKED || (at >= 0 && at < n_units), p.status)) out[at] = un;
    }
    return;
  }

  if (backward && p.mask == kMaskCausal && n_seqs > 0 && prefix[1] - prefix[0] >= 2 * kTileGroup) {
    // Fixed-length causal backward: every (batch, head) pair has the same tiles,
    // tile t costing more the smaller t is.  Ordered by cost alone, the units
    // running at once held about five tiles of each pair, so each pair's Q and
    // dO were fetched about once per five units.  Groups of tg tiles in cost
    // order, and inside a group pair by pair, keep the longest units first
    // while a group's units of one pair share their Q and dO in L2.  Only pairs
    // of at least 2 * kTileGroup tiles are grouped: with fewer (S = 2048 at
    // 128-key tiles) there are only a few units per SM, and balancing them
    // longest first matters more (groups of 8 there: 0.135 against 0.118 ms).
    // Measured at S = 8192 and 4096: groups of 16 beat 8, 32 and 64.  (The
    // forward keeps the plain cost order: grouping slowed it.)
    const int nt = prefix[1] - prefix[0], n_pairs = n_seqs * heads;
    const int tg = kTileGroup;
    for (int u = tid; u < n_units; u += kThreads) {
      const int pair = u / nt, t = u % nt, n = pair / heads, h = pair - n * heads;
      const int len = seq_info(p, n).len;
      Unit un;
      un.seq = n;
      un.head = h;
      un.tile = t;
      un.cost = (t * tile_rows < len) ? unit_cost(p, backward, tile_rows, len, t) : 0;
      const int g = t / tg, sz = min(tg, nt - g * tg);
      const int at = g * tg * n_pairs + pair * sz + (t - g * tg);
      if (bounds_ok(!GBATTN_CHECKED || (at >= 0 && at < n_units), p.status)) out[at] = un;
    }
    return;
  }

  // 2. enumerate units, compute costs, histogram.  Units are numbered sequence
  // by sequence, head by head, tile fastest, so that among equal costs (every
  // unit of a dense mask) the units running at the same time share a few heads'
  // K and V (or Q and dO) in L2 instead of touching every head at once.
  // A forward with a split key range lists each unit once per part (u = base
  // unit * ns + part), at the part's share of the cost.
  const int ns = backward ? 1 : max(1, p.n_split);
  for (int u = tid; u < n_units; u += kThreads) {
    const int ub = u / ns;
    int lo = 0, hi = n_seqs - 1;  // last n with heads * prefix[n] <= ub
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if ((long long)heads * prefix[mid] <= ub) lo = mid; else hi = mid - 1;
    }
    const int n = lo;
    const int tiles = prefix[n + 1] - prefix[n];
    const int local = ub - heads * prefix[n];
    const int h = local / tiles, t = local % tiles;
    const int len = seq_info(p, n).len;
    Unit un;
    un.seq = n;
    un.head = h;
    un.tile = t;
    un.cost = (t * tile_rows < len) ? cdiv(unit_cost(p, backward, tile_rows, len, t), ns) : 0;
    tmp[u] = un;
    atomicAdd(&hist[min(un.cost, kBuckets - 1)], 1);
  }
  __syncthreads();

  // 3. bucket starts, highest cost first
  bucket_starts_desc(hist, scan_smem);

  // 4. scatter (a split forward's entries carry their part in `cost` from here on)
  for (int u = tid; u < n_units; u += kThreads) {
    Unit un = tmp[u];
    int pos = atomicAdd(&hist[min(un.cost, kBuckets - 1)], 1);
    if (ns > 1) un.cost = u % ns;
    if (bounds_ok(!GBATTN_CHECKED || (pos >= 0 && pos < n_units), p.status)) out[pos] = un;
  }
}

// One block.  For each key block c: csc_ptr[c] = start, csc_idx = ascending query blocks.
__global__ void __launch_bounds__(kThreads) k_csr_to_csc(KParams p, int* csc_ptr, int* csc_idx) {
  __shared__ int scan_smem[72];
  const int nrb = p.n_row_blocks, ncb = p.n_col_blocks;
  const int chunk = cdiv(ncb, kThreads);
  const int c0 = threadIdx.x * chunk, c1 = min(ncb, c0 + chunk);
  auto listed = [&](int r, int c) {
    int lo = p.row_ptr[r], hi = p.row_ptr[r + 1] - 1;
    // the device copy of row r lies inside the column array
    if (!bounds_ok(!GBATTN_CHECKED || (0 <= lo && hi < p.nnz), p.status)) return false;
    while (lo <= hi) {
      int mid = (lo + hi) >> 1;
      int v = p.col_idx[mid];
      if (v == c) return true;
      if (v < c) lo = mid + 1; else hi = mid - 1;
    }
    return false;
  };
  int local = 0;
  for (int c = c0; c < c1; ++c)
    for (int r = 0; r < nrb; ++r) local += listed(r, c);
  int total;
  int base = block_exclusive_scan(local, scan_smem, &total);
  for (int c = c0; c < c1; ++c) {
    csc_ptr[c] = base;
    for (int r = 0; r < nrb; ++r)
      if (listed(r, c) && bounds_ok(!GBATTN_CHECKED || base < p.nnz, p.status)) csc_idx[base++] = r;
  }
  if (threadIdx.x == 0) csc_ptr[ncb] = total;
}

}  // namespace

cudaError_t launch_build_worklist(const KParams& p, bool backward, int tile_rows, Unit* units,
                                  int n_units, int* scratch, cudaStream_t st) {
  if (n_units <= 0) return cudaSuccess;
  k_build_worklist<<<1, kThreads, 0, st>>>(p, backward ? 1 : 0, tile_rows, units, n_units, scratch);
  return cudaGetLastError();
}

cudaError_t launch_csr_to_csc(const KParams& p, int* csc_ptr, int* csc_idx, cudaStream_t st) {
  k_csr_to_csc<<<1, kThreads, 0, st>>>(p, csc_ptr, csc_idx);
  return cudaGetLastError();
}

long long count_units(const KParams& p, const int* cu_host, bool backward, int tile_rows) {
  const int heads = backward ? p.heads_kv : p.heads_q;
  long long tiles = 0;
  if (p.varlen) {
    for (int n = 0; n < p.n_seqs; ++n) {
      int L = cu_host[n + 1] - cu_host[n];
      tiles += (L + tile_rows - 1) / tile_rows;
    }
  } else {
    tiles = (long long)p.batch * ((p.seqlen + tile_rows - 1) / tile_rows);
  }
  return tiles * heads;
}

}  // namespace gbattn
