// Oracle: plain, slow, float64 CPU attention (forward and analytic backward).
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
// leg of the benchmark may load this library.  The GPU library never links, loads
// or calls it, and the two share no code, headers or tables.
//
// What it computes (the plain definition, not the tiled algorithm):
//   * "Standard attention": Q.K^T gives a full score matrix, softmax over each
//     row, then a weighted sum of V (smzdm article "杀进决赛!这 28 支队伍把算子优化卷疯了!",
//     section 03, the paragraph describing how standard Attention is computed).
//     FlashAttention reaches the same numbers block by block (same section, next
//     paragraph), so the oracle is the unblocked definition.
//   * Inputs Q, K, V shaped [batch, head, seq_len, head_dim], optional mask, output
//     of the same shape (zwxr.cn CANN ops-nn fused-attention article, section 3.1).
//   * score = dot(q_i, k_j) * scale; masked positions become -inf before the
//     softmax (same article, section 3.3 pseudocode; the comparison operator was
//     lost in extraction and is read as "mask == 0 means masked").
//   * Backward: the three gradients dQ, dK, dV from the recomputed attention
//     matrix (smzdm article, section 03, the paragraph on why the backward is
//     harder).  The pages print no formula; the oracle uses the textbook softmax
//     Jacobian:  dP = dO.V^T, delta_i = sum_j P_ij dP_ij, dS = P * (dP - delta),
//     dQ = scale dS.K, dK = scale dS^T.Q, dV = P^T.dO.
//
// Layouts (all contiguous float64):
//   fixed length : q, o, do, dq  [B][Hq][S][D];  k, v, dk, dv  [B][Hkv][S][D];
//                  lse [B][Hq][S]
//   variable len : q, o, do, dq  [T][Hq][D];     k, v, dk, dv  [T][Hkv][D];
//                  lse [Hq][T];  sequence n covers rows cu_seqlens[n] .. cu_seqlens[n+1]-1
// Query head h reads KV head h / (Hq / Hkv) (contiguous groups).
// LSE is natural-log log-sum-exp of the scaled scores: LSE_i = m_i + ln(l_i).
// A row with no allowed key gets O = 0, LSE = -inf and contributes nothing to any
// gradient.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

extern "C" {

typedef struct {
  int32_t batch, heads_q, heads_kv, seqlen, head_dim;
  const int32_t* cu_seqlens;  // host, [n_seqs + 1], or NULL for fixed length
  int32_t n_seqs;
  double scale;
  int32_t mask;               // 0 none, 1 causal, 2 block-sparse
  const int32_t* row_ptr;     // block-sparse CSR over (block_q x block_k) tiles
  const int32_t* col_idx;
  int32_t n_row_blocks, n_col_blocks, block_q, block_k;
  int32_t causal_in_block;    // 1: inside listed tiles also require j <= i
} oracle_params_t;

}  // extern "C"

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// Position i may attend to position j (both relative to the sequence start).
bool keep(const oracle_params_t* p, int i, int j, int len) {
  if (j < 0 || j >= len) return false;
  if (p->mask == 1) return j <= i;
  if (p->mask == 2) {
    int rb = i / p->block_q, cb = j / p->block_k;
    if (rb >= p->n_row_blocks || cb >= p->n_col_blocks) return false;
    bool listed = false;
    for (int e = p->row_ptr[rb]; e < p->row_ptr[rb + 1]; ++e)
      if (p->col_idx[e] == cb) { listed = true; break; }
    if (!listed) return false;
    if (p->causal_in_block) return j <= i;
    return true;
  }
  return true;
}

int n_sequences(const oracle_params_t* p) { return p->cu_seqlens ? p->n_seqs : p->batch; }

int seq_len(const oracle_params_t* p, int n) {
  return p->cu_seqlens ? p->cu_seqlens[n + 1] - p->cu_seqlens[n] : p->seqlen;
}

// Offset (in doubles) of row `pos` of head `h` of sequence `n` in a tensor with `H` heads.
int64_t row_off(const oracle_params_t* p, int n, int h, int H, int pos) {
  const int64_t D = p->head_dim;
  if (p->cu_seqlens) return ((int64_t)(p->cu_seqlens[n] + pos) * H + h) * D;
  return (((int64_t)n * H + h) * p->seqlen + pos) * D;
}

int64_t lse_off(const oracle_params_t* p, int n, int h, int pos) {
  if (p->cu_seqlens) {
    int64_t T = p->cu_seqlens[p->n_seqs];
    return (int64_t)h * T + p->cu_seqlens[n] + pos;
  }
  return ((int64_t)n * p->heads_q + h) * p->seqlen + pos;
}

double dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int t = 0; t < d; ++t) s += a[t] * b[t];
  return s;
}

// Rows per work item (rows of one head are independent in the forward and in
// the per-row pass of the backward; keys are independent in the per-key pass).
const int kRowChunk = 64;

int row_chunks(const oracle_params_t* p) {
  int maxlen = p->seqlen;
  if (p->cu_seqlens)
    for (int n = 0; n < p->n_seqs; ++n) {
      const int L = p->cu_seqlens[n + 1] - p->cu_seqlens[n];
      if (L > maxlen) maxlen = L;
    }
  return maxlen > 0 ? (maxlen + kRowChunk - 1) / kRowChunk : 1;
}

template <class F>
void parallel_for(int n_items, int nthreads, F&& fn) {
  if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n_items) nthreads = n_items;
  if (nthreads <= 1) {
    for (int i = 0; i < n_items; ++i) fn(i);
    return;
  }
  std::atomic<int> next(0);
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t)
    pool.emplace_back([&]() {
      for (int i = next.fetch_add(1); i < n_items; i = next.fetch_add(1)) fn(i);
    });
  for (auto& th : pool) th.join();
}

// Scores of one query row against every allowed key: fills s[j] (scaled) for j in
// the allowed set, kNegInf elsewhere; returns the row max (kNegInf if none allowed).
double row_scores(const oracle_params_t* p, const double* q, const double* k, int n, int h,
                  int i, std::vector<double>& s) {
  const int L = seq_len(p, n), D = p->head_dim;
  const int G = p->heads_q / p->heads_kv, g = h / G;
  const double* qi = q + row_off(p, n, h, p->heads_q, i);
  double m = kNegInf;
  for (int j = 0; j < L; ++j) {
    if (!keep(p, i, j, L)) { s[j] = kNegInf; continue; }
    s[j] = p->scale * dot(qi, k + row_off(p, n, g, p->heads_kv, j), D);
    if (s[j] > m) m = s[j];
  }
  return m;
}

}  // namespace

extern "C" {

// Forward: O and LSE by the plain definition (full softmax over each row).
// Rows are independent, so work items are (sequence, query head, chunk of rows).
int oracle_attn_fwd(const oracle_params_t* p, const double* q, const double* k, const double* v,
                    double* o, double* lse, int nthreads) {
  const int NS = n_sequences(p), Hq = p->heads_q, D = p->head_dim;
  if (Hq <= 0 || p->heads_kv <= 0 || Hq % p->heads_kv) return 1;
  const int chunks = row_chunks(p);
  parallel_for(NS * Hq * chunks, nthreads, [&](int item) {
    const int n = item / (Hq * chunks), h = (item / chunks) % Hq, c = item % chunks;
    const int L = seq_len(p, n);
    const int G = Hq / p->heads_kv, g = h / G;
    std::vector<double> s(L > 0 ? L : 1);
    for (int i = c * kRowChunk; i < L && i < (c + 1) * kRowChunk; ++i) {
      double* oi = o + row_off(p, n, h, Hq, i);
      for (int t = 0; t < D; ++t) oi[t] = 0.0;
      const double m = row_scores(p, q, k, n, h, i, s);
      if (m == kNegInf) { lse[lse_off(p, n, h, i)] = kNegInf; continue; }
      double l = 0.0;
      for (int j = 0; j < L; ++j)
        if (s[j] != kNegInf) l += std::exp(s[j] - m);
      for (int j = 0; j < L; ++j) {
        if (s[j] == kNegInf) continue;
        const double pij = std::exp(s[j] - m) / l;
        const double* vj = v + row_off(p, n, g, p->heads_kv, j);
        for (int t = 0; t < D; ++t) oi[t] += pij * vj[t];
      }
      lse[lse_off(p, n, h, i)] = m + std::log(l);
    }
  });
  return 0;
}

// Forward by the block-by-block algorithm of the zwxr.cn CANN ops-nn article,
// sections 3.2-3.3: the outer loop takes one query row at a time, the inner loop
// streams key blocks of `block` keys; each block gives a local max, the running
// max and sum are corrected by exp(old_max - new_max), the accumulator is scaled by
// the same factor and gains exp(score - new_max) * v; O = acc / sum at the end.
// It exists so that tests can show the streamed algorithm reaches the plain
// definition; nothing else uses it.
int oracle_attn_fwd_blocked(const oracle_params_t* p, const double* q, const double* k,
                            const double* v, double* o, double* lse, int block, int nthreads) {
  const int NS = n_sequences(p), Hq = p->heads_q, D = p->head_dim;
  if (block <= 0 || Hq <= 0 || p->heads_kv <= 0 || Hq % p->heads_kv) return 1;
  parallel_for(NS * Hq, nthreads, [&](int item) {
    const int n = item / Hq, h = item % Hq;
    const int L = seq_len(p, n);
    const int G = Hq / p->heads_kv, g = h / G;
    std::vector<double> acc(D), sblk(block);
    for (int i = 0; i < L; ++i) {
      const double* qi = q + row_off(p, n, h, Hq, i);
      double gmax = kNegInf, gsum = 0.0;
      for (int t = 0; t < D; ++t) acc[t] = 0.0;
      for (int j0 = 0; j0 < L; j0 += block) {
        const int j1 = j0 + block < L ? j0 + block : L;
        double lmax = kNegInf;
        for (int j = j0; j < j1; ++j) {
          sblk[j - j0] = keep(p, i, j, L)
                             ? p->scale * dot(qi, k + row_off(p, n, g, p->heads_kv, j), D)
                             : kNegInf;
          if (sblk[j - j0] > lmax) lmax = sblk[j - j0];
        }
        if (lmax == kNegInf) continue;  // block fully masked for this row
        const double nmax = gmax > lmax ? gmax : lmax;
        const double corr = gmax == kNegInf ? 0.0 : std::exp(gmax - nmax);
        gsum *= corr;
        for (int t = 0; t < D; ++t) acc[t] *= corr;
        for (int j = j0; j < j1; ++j) {
          if (sblk[j - j0] == kNegInf) continue;
          const double e = std::exp(sblk[j - j0] - nmax);
          gsum += e;
          const double* vj = v + row_off(p, n, g, p->heads_kv, j);
          for (int t = 0; t < D; ++t) acc[t] += e * vj[t];
        }
        gmax = nmax;
      }
      double* oi = o + row_off(p, n, h, Hq, i);
      if (gmax == kNegInf) {
        for (int t = 0; t < D; ++t) oi[t] = 0.0;
        lse[lse_off(p, n, h, i)] = kNegInf;
      } else {
        for (int t = 0; t < D; ++t) oi[t] = acc[t] / gsum;
        lse[lse_off(p, n, h, i)] = gmax + std::log(gsum);
      }
    }
  });
  return 0;
}

// Backward: dQ, dK, dV by the softmax Jacobian, recomputing P from the scores.
//   pass 1, per query row i (items: sequence, query head, chunk of rows):
//     m_i, l_i (max and sum of the row's softmax), dP_ij = <dO_i, v_j>,
//     delta_i = sum_j P_ij dP_ij and dQ_i = scale sum_j dS_ij k_j;
//   pass 2, per key row j (items: sequence, KV head, chunk of keys):
//     dK_j = scale sum_{h in group} sum_i dS_ij q_i,  dV_j = sum_{h in group} sum_i P_ij dO_i,
//     with P_ij = exp(s_ij - m_i) / l_i and dS_ij = P_ij (dP_ij - delta_i) taken from
//     the row quantities of pass 1.
int oracle_attn_bwd(const oracle_params_t* p, const double* q, const double* k, const double* v,
                    const double* dout, double* dq, double* dk, double* dv, int nthreads) {
  const int NS = n_sequences(p), Hq = p->heads_q, Hkv = p->heads_kv, D = p->head_dim;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv) return 1;
  const int G = Hq / Hkv;
  const int chunks = row_chunks(p);
  // Row statistics, laid out like lse.
  int64_t n_rows = 0;
  for (int n = 0; n < NS; ++n) n_rows += (int64_t)seq_len(p, n) * Hq;
  std::vector<double> row_m(n_rows), row_l(n_rows), row_delta(n_rows);

  parallel_for(NS * Hq * chunks, nthreads, [&](int item) {
    const int n = item / (Hq * chunks), h = (item / chunks) % Hq, c = item % chunks;
    const int L = seq_len(p, n), g = h / G;
    std::vector<double> s(L > 0 ? L : 1), dp(L > 0 ? L : 1);
    for (int i = c * kRowChunk; i < L && i < (c + 1) * kRowChunk; ++i) {
      double* dqi = dq + row_off(p, n, h, Hq, i);
      for (int t = 0; t < D; ++t) dqi[t] = 0.0;
      const int64_t r = lse_off(p, n, h, i);
      const double m = row_scores(p, q, k, n, h, i, s);
      row_m[r] = m;
      row_l[r] = 0.0;
      row_delta[r] = 0.0;
      if (m == kNegInf) continue;
      double l = 0.0;
      for (int j = 0; j < L; ++j)
        if (s[j] != kNegInf) l += std::exp(s[j] - m);
      const double* doi = dout + row_off(p, n, h, Hq, i);
      double delta = 0.0;
      for (int j = 0; j < L; ++j) {
        if (s[j] == kNegInf) { s[j] = 0.0; dp[j] = 0.0; continue; }
        s[j] = std::exp(s[j] - m) / l;  // P_ij
        dp[j] = dot(doi, v + row_off(p, n, g, Hkv, j), D);
        delta += s[j] * dp[j];
      }
      for (int j = 0; j < L; ++j) {
        if (s[j] == 0.0) continue;
        const double ds = s[j] * (dp[j] - delta);
        const double* kj = k + row_off(p, n, g, Hkv, j);
        for (int t = 0; t < D; ++t) dqi[t] += p->scale * ds * kj[t];
      }
      row_l[r] = l;
      row_delta[r] = delta;
    }
  });

  parallel_for(NS * Hkv * chunks, nthreads, [&](int item) {
    const int n = item / (Hkv * chunks), g = (item / chunks) % Hkv, c = item % chunks;
    const int L = seq_len(p, n);
    for (int j = c * kRowChunk; j < L && j < (c + 1) * kRowChunk; ++j) {
      double* dkj = dk + row_off(p, n, g, Hkv, j);
      double* dvj = dv + row_off(p, n, g, Hkv, j);
      for (int t = 0; t < D; ++t) dkj[t] = dvj[t] = 0.0;
      const double* kj = k + row_off(p, n, g, Hkv, j);
      const double* vj = v + row_off(p, n, g, Hkv, j);
      for (int h = g * G; h < (g + 1) * G; ++h) {
        for (int i = 0; i < L; ++i) {
          if (!keep(p, i, j, L)) continue;
          const int64_t r = lse_off(p, n, h, i);
          if (row_m[r] == kNegInf) continue;
          const double* qi = q + row_off(p, n, h, Hq, i);
          const double* doi = dout + row_off(p, n, h, Hq, i);
          const double pij = std::exp(p->scale * dot(qi, kj, D) - row_m[r]) / row_l[r];
          const double ds = pij * (dot(doi, vj, D) - row_delta[r]);
          for (int t = 0; t < D; ++t) {
            dkj[t] += p->scale * ds * qi[t];
            dvj[t] += pij * doi[t];
          }
        }
      }
    }
  });
  return 0;
}

}  // extern "C"
