// attn_oracle.cpp -- fp64 CPU oracle for exact softmax attention.
//
// TEST INFRASTRUCTURE ONLY: used by the test suite, the smoke check and the
// benchmark's CPU-baseline leg to check the CUDA library.  It shares no code
// with the CUDA path.  Declarations and the conventions are in attn_oracle.h.
//
// The forward is the definition written out, one query row at a time:
//   S = scale * Q K^T, P = softmax(S), O = P V
// ("LLM 注意力与计算内核精读笔记 · 02 FlashAttention", §2, the three-step
// definition), with the softmax taken as the 3-pass safe softmax of
// "从Online-Softmax到FlashAttention V1/V2/V3", 0x02: pass 1 the row max, pass 2
// the sum of exp(x - max), pass 3 the normalisation.  The score row is
// computed once into a buffer and then read three times.
//
// The backward is the analytic derivative of that forward (the pages' own
// backward formulas did not survive; 0x04 of the same page only says that S
// and P are recomputed).  With dL/dO = dO:
//   D_i    = sum_k dO_ik O_ik           (= sum_j p_ij dP_ij)
//   dP_ij  = <dO_i, v_j>
//   dS_ij  = p_ij (dP_ij - D_i)
//   dQ_i   = scale * sum_j dS_ij k_j
//   dK_j   = scale * sum_{heads in group} sum_i dS_ij q_i
//   dV_j   = sum_{heads in group} sum_i p_ij dO_i
// Masked (i, j) pairs contribute nothing.

#include "attn_oracle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// Run f(idx) for idx in [0, n) on `threads` worker threads.
template <class F>
void parallel_for(int64_t n, int threads, F f) {
  int nt = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  if (nt < 1) nt = 1;
  if (n < nt) nt = (int)std::max<int64_t>(n, 1);
  if (nt == 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next(0);
  const int64_t chunk = std::max<int64_t>(1, n / (nt * 16));
  std::vector<std::thread> pool;
  pool.reserve(nt);
  for (int t = 0; t < nt; ++t) {
    pool.emplace_back([&]() {
      for (;;) {
        int64_t s = next.fetch_add(chunk);
        if (s >= n) break;
        int64_t e = std::min(n, s + chunk);
        for (int64_t i = s; i < e; ++i) f(i);
      }
    });
  }
  for (auto& th : pool) th.join();
}

double dot(const double* a, const double* b, int d) {
  double acc = 0.0;
  for (int k = 0; k < d; ++k) acc += a[k] * b[k];
  return acc;
}

bool bad_shape(int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d) {
  return B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || d < 1 || (Hq % Hkv) != 0;
}

struct Shape {
  int B, Hq, Hkv;
  int64_t Nq, Nk;
  int d;
  double scale;
  int causal;
  // Block-sparse mask (NULL: none): bmask[hm][i / bsize][j / bsize] != 0
  // keeps the block, hm = 0 when one mask serves every head, else the query
  // head ("从Online-Softmax…" 0x04: Block-Sparse FlashAttention skips the
  // masked blocks outright, i.e. their scores take no part in the softmax).
  const uint8_t* bmask = nullptr;
  int bmask_heads = 1;
  int64_t bsize = 128;
  int group() const { return Hq / Hkv; }
};

// Does query i of query head h keep key j?  The causal rule, then the block mask.
bool keep(const Shape& sh, int h, int64_t i, int64_t j) {
  if (sh.causal && !oracle_causal_keep(i, j, sh.Nq, sh.Nk)) return false;
  if (!sh.bmask) return true;
  const int64_t nqb = (sh.Nq + sh.bsize - 1) / sh.bsize, nkb = (sh.Nk + sh.bsize - 1) / sh.bsize;
  const int64_t hm = sh.bmask_heads == 1 ? 0 : h;
  return sh.bmask[(hm * nqb + i / sh.bsize) * nkb + j / sh.bsize] != 0;
}

// One query row of the forward: fills s (scores of kept keys, Nk entries,
// masked ones set to -inf), returns m and l, writes O (d) and LSE.
// Follows the 3-pass safe softmax order.
void fwd_row(const Shape& sh, const double* Q, const double* K, const double* V,
             int64_t row, std::vector<double>& s, double* O, double* LSE) {
  const int64_t i = row % sh.Nq;
  const int64_t bh = row / sh.Nq;
  const int h = (int)(bh % sh.Hq);
  const int b = (int)(bh / sh.Hq);
  const int hk = h / sh.group();  // contiguous query-head groups (0x09 GQA)
  const double* q = Q + row * sh.d;
  const double* Kh = K + ((int64_t)b * sh.Hkv + hk) * sh.Nk * sh.d;
  const double* Vh = V + ((int64_t)b * sh.Hkv + hk) * sh.Nk * sh.d;
  s.assign((size_t)sh.Nk, kNegInf);
  // Pass 1: logits and their max.
  double m = kNegInf;
  for (int64_t j = 0; j < sh.Nk; ++j) {
    if (!keep(sh, h, i, j)) continue;
    s[j] = sh.scale * dot(q, Kh + j * sh.d, sh.d);
    if (s[j] > m) m = s[j];
  }
  for (int k = 0; k < sh.d; ++k) O[k] = 0.0;
  if (m == kNegInf) {  // no kept key: output zero ("从Online-Softmax…", 0x09)
    *LSE = kNegInf;
    return;
  }
  // Pass 2: the denominator.
  double l = 0.0;
  for (int64_t j = 0; j < sh.Nk; ++j)
    if (s[j] != kNegInf) l += std::exp(s[j] - m);
  // Pass 3: normalised probabilities times V.
  for (int64_t j = 0; j < sh.Nk; ++j) {
    if (s[j] == kNegInf) continue;
    const double p = std::exp(s[j] - m) / l;
    const double* v = Vh + j * sh.d;
    for (int k = 0; k < sh.d; ++k) O[k] += p * v[k];
  }
  *LSE = m + std::log(l);
}

// dQ of one query row, recomputing everything of the row in fp64.
void dq_row(const Shape& sh, const double* Q, const double* K, const double* V,
            const double* dO, int64_t row, std::vector<double>& s, std::vector<double>& o,
            double* dQ, double* LSE_out, double* O_out, double* D_out) {
  const int64_t bh = row / sh.Nq;
  const int h = (int)(bh % sh.Hq);
  const int b = (int)(bh / sh.Hq);
  const int hk = h / sh.group();
  const double* Kh = K + ((int64_t)b * sh.Hkv + hk) * sh.Nk * sh.d;
  const double* Vh = V + ((int64_t)b * sh.Hkv + hk) * sh.Nk * sh.d;
  const double* dOi = dO + row * sh.d;
  o.assign((size_t)sh.d, 0.0);
  double lse;
  fwd_row(sh, Q, K, V, row, s, o.data(), &lse);
  double Di = dot(dOi, o.data(), sh.d);
  for (int k = 0; k < sh.d; ++k) dQ[k] = 0.0;
  if (lse != kNegInf) {
    for (int64_t j = 0; j < sh.Nk; ++j) {
      if (s[j] == kNegInf) continue;
      const double p = std::exp(s[j] - lse);
      const double dP = dot(dOi, Vh + j * sh.d, sh.d);
      const double dS = p * (dP - Di);
      const double* kj = Kh + j * sh.d;
      for (int k = 0; k < sh.d; ++k) dQ[k] += sh.scale * dS * kj[k];
    }
  }
  if (LSE_out) *LSE_out = lse;
  if (O_out)
    for (int k = 0; k < sh.d; ++k) O_out[k] = o[k];
  if (D_out) *D_out = Di;
}

// dK and dV of one key row, given LSE and D of every query row.
void dkv_row(const Shape& sh, const double* Q, const double* K, const double* V,
             const double* dO, const double* LSE, const double* Dv, int64_t kvrow,
             double* dK, double* dV) {
  const int64_t j = kvrow % sh.Nk;
  const int64_t bhk = kvrow / sh.Nk;
  const int hk = (int)(bhk % sh.Hkv);
  const int b = (int)(bhk / sh.Hkv);
  const double* kj = K + kvrow * sh.d;
  const double* vj = V + kvrow * sh.d;
  for (int k = 0; k < sh.d; ++k) dK[k] = dV[k] = 0.0;
  const int G = sh.group();
  for (int g = 0; g < G; ++g) {
    const int h = hk * G + g;
    const int64_t base = ((int64_t)b * sh.Hq + h) * sh.Nq;
    for (int64_t i = 0; i < sh.Nq; ++i) {
      if (!keep(sh, h, i, j)) continue;
      const double lse = LSE[base + i];
      if (lse == kNegInf) continue;
      const double* qi = Q + (base + i) * sh.d;
      const double* dOi = dO + (base + i) * sh.d;
      const double sij = sh.scale * dot(qi, kj, sh.d);
      const double p = std::exp(sij - lse);
      const double dP = dot(dOi, vj, sh.d);
      const double dS = p * (dP - Dv[base + i]);
      for (int k = 0; k < sh.d; ++k) {
        dK[k] += sh.scale * dS * qi[k];
        dV[k] += p * dOi[k];
      }
    }
  }
}

}  // namespace

extern "C" {

int oracle_causal_keep(int64_t i, int64_t j, int64_t Nq, int64_t Nk) {
  // Bottom-right alignment ("从Online-Softmax…", 0x09): the last query row sees
  // every key; row i sees keys j <= i + (Nk - Nq).
  return j <= i + (Nk - Nq) ? 1 : 0;
}

int oracle_softmax3(const double* x, int64_t n, double* out) {
  if (!x || !out || n < 1) return -1;
  double m = kNegInf;
  for (int64_t j = 0; j < n; ++j) m = std::max(m, x[j]);  // pass 1
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) l += std::exp(x[j] - m);  // pass 2
  for (int64_t j = 0; j < n; ++j) out[j] = std::exp(x[j] - m) / l;  // pass 3
  return 0;
}

int oracle_softmax3_f32(const float* x, int64_t n, float* out) {
  if (!x || !out || n < 1) return -1;
  float m = -std::numeric_limits<float>::infinity();
  for (int64_t j = 0; j < n; ++j) m = std::max(m, x[j]);
  float l = 0.0f;
  for (int64_t j = 0; j < n; ++j) l += std::exp(x[j] - m);
  for (int64_t j = 0; j < n; ++j) out[j] = std::exp(x[j] - m) / l;
  return 0;
}

int oracle_online_row(const double* s, const double* v, int64_t n, int64_t dv,
                      const int64_t* block_sizes, int64_t nblocks,
                      double* O_out, double* m_trace, double* l_trace, double* O_trace) {
  if (!s || !v || !block_sizes || !O_out || n < 1 || dv < 1 || nblocks < 1) return -1;
  int64_t total = 0;
  for (int64_t t = 0; t < nblocks; ++t) {
    if (block_sizes[t] < 1) return -1;
    total += block_sizes[t];
  }
  if (total != n) return -1;
  // Running state before any block: m = -inf, l = 0, O = 0.
  double m = kNegInf, l = 0.0;
  std::vector<double> O((size_t)dv, 0.0), pv((size_t)dv);
  int64_t start = 0;
  for (int64_t t = 0; t < nblocks; ++t) {
    const int64_t nb = block_sizes[t];
    // In-block statistics: m~ = block max, P~ = exp(s - m~), l~ = sum P~,
    // and the in-block product P~ V.
    double mt = kNegInf;
    for (int64_t j = 0; j < nb; ++j) mt = std::max(mt, s[start + j]);
    double lt = 0.0;
    std::fill(pv.begin(), pv.end(), 0.0);
    for (int64_t j = 0; j < nb; ++j) {
      const double p = std::exp(s[start + j] - mt);
      lt += p;
      for (int64_t k = 0; k < dv; ++k) pv[k] += p * v[(start + j) * dv + k];
    }
    // Merge ("02 FlashAttention", §5): m+ = max(m, m~);
    // l+ = e^{m - m+} l + e^{m~ - m+} l~;
    // O+ = (e^{m - m+} l O + e^{m~ - m+} P~V) / l+.
    const double mn = std::max(m, mt);
    const double a_old = (m == kNegInf) ? 0.0 : std::exp(m - mn);
    const double a_new = std::exp(mt - mn);
    const double ln = a_old * l + a_new * lt;
    for (int64_t k = 0; k < dv; ++k) O[k] = (a_old * l * O[k] + a_new * pv[k]) / ln;
    m = mn;
    l = ln;
    if (m_trace) m_trace[t] = m;
    if (l_trace) l_trace[t] = l;
    if (O_trace)
      for (int64_t k = 0; k < dv; ++k) O_trace[t * dv + k] = O[k];
    start += nb;
  }
  for (int64_t k = 0; k < dv; ++k) O_out[k] = O[k];
  return 0;
}

int oracle_online_softmax_f32(const float* x, int64_t n, int64_t block, float* out) {
  if (!x || !out || n < 1 || block < 1) return -1;
  // Running max m and running denominator d' of "Flash-attention 学习", §0:
  // m_i = max(m_{i-1}, x_i), d'_i = d'_{i-1} e^{m_{i-1} - m_i} + e^{x_i - m_i},
  // taken one block at a time (block max first, then the block's terms).
  float m = -std::numeric_limits<float>::infinity();
  float d = 0.0f;
  for (int64_t s0 = 0; s0 < n; s0 += block) {
    const int64_t e = std::min(n, s0 + block);
    float mb = -std::numeric_limits<float>::infinity();
    for (int64_t j = s0; j < e; ++j) mb = std::max(mb, x[j]);
    const float mn = std::max(m, mb);
    float db = 0.0f;
    for (int64_t j = s0; j < e; ++j) db += std::exp(x[j] - mn);
    d = (d == 0.0f ? 0.0f : d * std::exp(m - mn)) + db;
    m = mn;
  }
  for (int64_t j = 0; j < n; ++j) out[j] = std::exp(x[j] - m) / d;
  return 0;
}

int oracle_fwd(const double* Q, const double* K, const double* V,
               int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
               double scale, int causal, double* O, double* LSE, int threads) {
  if (!Q || !K || !V || !O || !LSE || bad_shape(B, Hq, Hkv, Nq, Nk, d)) return -1;
  const Shape sh{B, Hq, Hkv, Nq, Nk, d, scale, causal};
  const int64_t rows = (int64_t)B * Hq * Nq;
  parallel_for(rows, threads, [&](int64_t r) {
    thread_local std::vector<double> s;
    fwd_row(sh, Q, K, V, r, s, O + r * d, LSE + r);
  });
  return 0;
}

int oracle_fwd_rows(const double* Q, const double* K, const double* V,
                    int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                    double scale, int causal, const int64_t* rows, int64_t nrows,
                    double* O_rows, double* LSE_rows, int threads) {
  if (!Q || !K || !V || !rows || !O_rows || !LSE_rows || nrows < 0 ||
      bad_shape(B, Hq, Hkv, Nq, Nk, d))
    return -1;
  const int64_t total = (int64_t)B * Hq * Nq;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -2;
  const Shape sh{B, Hq, Hkv, Nq, Nk, d, scale, causal};
  parallel_for(nrows, threads, [&](int64_t r) {
    thread_local std::vector<double> s;
    fwd_row(sh, Q, K, V, rows[r], s, O_rows + r * d, LSE_rows + r);
  });
  return 0;
}

int oracle_bwd(const double* Q, const double* K, const double* V, const double* dO,
               int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
               double scale, int causal,
               double* dQ, double* dK, double* dV,
               double* O, double* LSE, double* Dvec, int threads) {
  if (!Q || !K || !V || !dO || !dQ || !dK || !dV || bad_shape(B, Hq, Hkv, Nq, Nk, d))
    return -1;
  const Shape sh{B, Hq, Hkv, Nq, Nk, d, scale, causal};
  const int64_t qrows = (int64_t)B * Hq * Nq;
  const int64_t kvrows = (int64_t)B * Hkv * Nk;
  std::vector<double> lse_buf(LSE ? 0 : (size_t)qrows), d_buf(Dvec ? 0 : (size_t)qrows);
  double* lse = LSE ? LSE : lse_buf.data();
  double* dv = Dvec ? Dvec : d_buf.data();
  // Phase 1, per query row: O, LSE, D and dQ.
  parallel_for(qrows, threads, [&](int64_t r) {
    thread_local std::vector<double> s, o;
    dq_row(sh, Q, K, V, dO, r, s, o, dQ + r * d, lse + r, O ? O + r * d : nullptr, dv + r);
  });
  // Phase 2, per key row: dK and dV from the row statistics of phase 1.
  parallel_for(kvrows, threads, [&](int64_t r) {
    dkv_row(sh, Q, K, V, dO, lse, dv, r, dK + r * d, dV + r * d);
  });
  return 0;
}

int oracle_bwd_dq_rows(const double* Q, const double* K, const double* V, const double* dO,
                       int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                       double scale, int causal, const int64_t* rows, int64_t nrows,
                       double* dQ_rows, int threads) {
  if (!Q || !K || !V || !dO || !rows || !dQ_rows || nrows < 0 ||
      bad_shape(B, Hq, Hkv, Nq, Nk, d))
    return -1;
  const int64_t total = (int64_t)B * Hq * Nq;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -2;
  const Shape sh{B, Hq, Hkv, Nq, Nk, d, scale, causal};
  parallel_for(nrows, threads, [&](int64_t r) {
    thread_local std::vector<double> s, o;
    dq_row(sh, Q, K, V, dO, rows[r], s, o, dQ_rows + r * d, nullptr, nullptr, nullptr);
  });
  return 0;
}

int oracle_bwd_dkv_rows(const double* Q, const double* K, const double* V, const double* dO,
                        const double* LSE, const double* Dvec,
                        int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                        double scale, int causal, const int64_t* kv_rows, int64_t nrows,
                        double* dK_rows, double* dV_rows, int threads) {
  if (!Q || !K || !V || !dO || !LSE || !Dvec || !kv_rows || !dK_rows || !dV_rows ||
      nrows < 0 || bad_shape(B, Hq, Hkv, Nq, Nk, d))
    return -1;
  const int64_t total = (int64_t)B * Hkv * Nk;
  for (int64_t r = 0; r < nrows; ++r)
    if (kv_rows[r] < 0 || kv_rows[r] >= total) return -2;
  const Shape sh{B, Hq, Hkv, Nq, Nk, d, scale, causal};
  parallel_for(nrows, threads, [&](int64_t r) {
    dkv_row(sh, Q, K, V, dO, LSE, Dvec, kv_rows[r], dK_rows + r * d, dV_rows + r * d);
  });
  return 0;
}

int oracle_fwd_masked(const double* Q, const double* K, const double* V,
                      int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                      double scale, int causal, const uint8_t* bmask, int bmask_heads, int64_t bsize,
                      double* O, double* LSE, int threads) {
  if (!Q || !K || !V || !O || !LSE || !bmask || bsize < 1 || bad_shape(B, Hq, Hkv, Nq, Nk, d) ||
      (bmask_heads != 1 && bmask_heads != Hq))
    return -1;
  Shape sh{B, Hq, Hkv, Nq, Nk, d, scale, causal};
  sh.bmask = bmask;
  sh.bmask_heads = bmask_heads;
  sh.bsize = bsize;
  const int64_t rows = (int64_t)B * Hq * Nq;
  parallel_for(rows, threads, [&](int64_t r) {
    thread_local std::vector<double> s;
    fwd_row(sh, Q, K, V, r, s, O + r * d, LSE + r);
  });
  return 0;
}

int oracle_bwd_masked(const double* Q, const double* K, const double* V, const double* dO,
                      int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                      double scale, int causal, const uint8_t* bmask, int bmask_heads, int64_t bsize,
                      double* dQ, double* dK, double* dV, double* O, double* LSE, int threads) {
  if (!Q || !K || !V || !dO || !dQ || !dK || !dV || !bmask || bsize < 1 ||
      bad_shape(B, Hq, Hkv, Nq, Nk, d) || (bmask_heads != 1 && bmask_heads != Hq))
    return -1;
  Shape sh{B, Hq, Hkv, Nq, Nk, d, scale, causal};
  sh.bmask = bmask;
  sh.bmask_heads = bmask_heads;
  sh.bsize = bsize;
  const int64_t qrows = (int64_t)B * Hq * Nq;
  const int64_t kvrows = (int64_t)B * Hkv * Nk;
  std::vector<double> lse_buf(LSE ? 0 : (size_t)qrows), d_buf((size_t)qrows);
  double* lse = LSE ? LSE : lse_buf.data();
  parallel_for(qrows, threads, [&](int64_t r) {
    thread_local std::vector<double> s, o;
    dq_row(sh, Q, K, V, dO, r, s, o, dQ + r * d, lse + r, O ? O + r * d : nullptr, d_buf.data() + r);
  });
  parallel_for(kvrows, threads, [&](int64_t r) {
    dkv_row(sh, Q, K, V, dO, lse, d_buf.data(), r, dK + r * d, dV + r * d);
  });
  return 0;
}

}  // extern "C"
