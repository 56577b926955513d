/*
 * attn_oracle.h -- plain, slow, fp64 CPU oracle for exact softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists to check the CUDA library.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA
 * path, and it never calls into it.
 *
 * Sources it restates (page title, section):
 *  [P1] "[Attention优化][2w字]原理&图解: 从Online-Softmax到FlashAttention V1/V2/V3"
 *       (qinglite.cn): 0x01 standard 3-step attention, 0x02 3-pass safe softmax,
 *       0x09 GQA head indexing and the bottom-right causal alignment example.
 *  [P2] "LLM 注意力与计算内核精读笔记 · 02 FlashAttention：IO 感知的精确注意力"
 *       (zzszmyf.github.io): §2 the three-step S/P/O definition, §5 the online
 *       (m, l, O) block merge and §5.1 its shift invariance, §8 the worked example.
 *  [P3] "Flash-attention 学习" (s1mplewind.github.io): §0 online softmax
 *       recurrence for m_i and d'_i.
 *
 * Conventions (readings where the pages are silent):
 *  - Layout is row-major [B, H, N, d] with d contiguous.  Q, O, dQ use H = Hq;
 *    K, V, dK, dV use H = Hkv.  LSE and D are [B, Hq, Nq].
 *  - Query head h uses key/value head h / (Hq / Hkv) (contiguous groups).
 *  - Logits are s_ij = scale * <q_i, k_j>.  LSE_i = m_i + ln(l_i) in natural-log
 *    units of the scaled logits.
 *  - Causal keeps key j for query i when j <= i + (Nk - Nq) (bottom-right
 *    alignment).  A query row with no kept key gives O = 0 and LSE = -inf.
 *  - The backward is the analytic gradient of O alone (dL/dO = dO given); no
 *    gradient flows through LSE.
 *
 * Every entry point returns 0 on success and a negative number on a bad
 * argument.  `threads` <= 0 means "all hardware threads".
 */
#ifndef ATTN_ORACLE_H
#define ATTN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 1 if query i keeps key j under the causal rule above, else 0. */
int oracle_causal_keep(int64_t i, int64_t j, int64_t Nq, int64_t Nk);

/* 3-pass safe softmax of one row x[0..n): max, sum of exp(x - max), normalise. */
int oracle_softmax3(const double* x, int64_t n, double* out);

/* The online (m, l, O) merge of [P2] §5 applied to one score row s[0..n) with
 * value rows v[n][dv], consuming the row in consecutive blocks of the given
 * sizes.  After block t it records m, l and the normalised O (dv values) in
 * m_trace[t], l_trace[t], O_trace[t*dv ..].  O_out gets the final O.
 * Used only to pin the oracle against the pages' worked example and to check
 * that the online form equals the 3-pass form. */
int oracle_online_row(const double* s, const double* v, int64_t n, int64_t dv,
                      const int64_t* block_sizes, int64_t nblocks,
                      double* O_out, double* m_trace, double* l_trace, double* O_trace);

/* The same online softmax carried out in fp32 arithmetic ([P3] §0 recurrence,
 * block version): returns the probabilities of x (n floats) consumed in blocks
 * of `block` elements.  Used for the blocked-softmax rounding study. */
int oracle_online_softmax_f32(const float* x, int64_t n, int64_t block, float* out);
/* Plain fp32 3-pass softmax, the baseline of that study. */
int oracle_softmax3_f32(const float* x, int64_t n, float* out);

/* Full forward: O [B,Hq,Nq,d], LSE [B,Hq,Nq]. */
int oracle_fwd(const double* Q, const double* K, const double* V,
               int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
               double scale, int causal, double* O, double* LSE, int threads);

/* Forward on selected query rows only.  rows[r] = (b*Hq + h)*Nq + i.
 * O_rows is [nrows, d], LSE_rows is [nrows]. */
int oracle_fwd_rows(const double* Q, const double* K, const double* V,
                    int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                    double scale, int causal, const int64_t* rows, int64_t nrows,
                    double* O_rows, double* LSE_rows, int threads);

/* Full backward.  Outputs dQ [B,Hq,Nq,d], dK and dV [B,Hkv,Nk,d].  O, LSE and
 * D = rowsum(dO * O) [B,Hq,Nq] are also returned (any may be NULL). */
int oracle_bwd(const double* Q, const double* K, const double* V, const double* dO,
               int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
               double scale, int causal,
               double* dQ, double* dK, double* dV,
               double* O, double* LSE, double* Dvec, int threads);

/* dQ on selected query rows (rows as in oracle_fwd_rows).  Fully independent:
 * every quantity of the row is recomputed in fp64.  dQ_rows is [nrows, d]. */
int oracle_bwd_dq_rows(const double* Q, const double* K, const double* V, const double* dO,
                       int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                       double scale, int causal, const int64_t* rows, int64_t nrows,
                       double* dQ_rows, int threads);

/* dK and dV on selected key rows, kv_rows[r] = (b*Hkv + hk)*Nk + j, given the
 * per-query-row LSE and D = rowsum(dO * O) as inputs ([B,Hq,Nq] each).  The
 * probabilities are rebuilt as p_ij = exp(s_ij - LSE_i).  dK_rows, dV_rows are
 * [nrows, d]. */
int oracle_bwd_dkv_rows(const double* Q, const double* K, const double* V, const double* dO,
                        const double* LSE, const double* Dvec,
                        int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                        double scale, int causal, const int64_t* kv_rows, int64_t nrows,
                        double* dK_rows, double* dV_rows, int threads);

/* Block-sparse forward and backward: as oracle_fwd / oracle_bwd with a block
 * mask on top of the causal rule.  bmask is uint8 [bmask_heads][ceil(Nq/bsize)]
 * [ceil(Nk/bsize)] with bmask_heads 1 (one mask for every head) or Hq; a zero
 * entry removes the block's keys from its queries' softmax ("从Online-Softmax…"
 * 0x04, Block-Sparse FlashAttention skips masked blocks).  A row left with no
 * key gives O = 0, LSE = -inf (and zero gradients). */
int oracle_fwd_masked(const double* Q, const double* K, const double* V,
                      int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                      double scale, int causal, const uint8_t* bmask, int bmask_heads, int64_t bsize,
                      double* O, double* LSE, int threads);
int oracle_bwd_masked(const double* Q, const double* K, const double* V, const double* dO,
                      int B, int Hq, int Hkv, int64_t Nq, int64_t Nk, int d,
                      double scale, int causal, const uint8_t* bmask, int bmask_heads, int64_t bsize,
                      double* dQ, double* dK, double* dV, double* O, double* LSE, int threads);

#ifdef __cplusplus
}
#endif

#endif
