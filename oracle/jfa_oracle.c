/*
 * jfa_oracle.c -- plain fp64 CPU oracle for jagged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the libjfa CUDA
 * library and its Python binding) may include, link, load or call this file.
 * It exists so that tests, the smoke check and the CPU baseline leg of the
 * benchmark can compare the GPU kernels with an obviously-correct definition.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (one sequence b and one head h at a time, every value in
 * double precision, no tiling, no blocking, no online rescaling):
 *
 *   Jagged layout.  Sequence b owns rows offs_q[b] .. offs_q[b+1]-1 of Q/O/dO
 *   and rows offs_k[b] .. offs_k[b+1]-1 of K/V.  No padding exists anywhere.
 *   Source: Meta GEM MFU co-design write-up (piletech.kr/articles/112134),
 *   "상세 정리" (details) section, jagged-input bullet and Jagged Flash
 *   Attention bullet: attention works directly on variable-length tensors.
 *
 *   Valid set.  V(i) = { j : j < Lk_b }, and additionally j <= i when causal
 *   (causal is defined only for self-attention, Lq_b == Lk_b).
 *
 *   Softmax attention (the JFA bullet of the same page):
 *     s_ij   = scale * <q_i, k_j>
 *     m_i    = max_{j in V(i)} s_ij
 *     P_ij   = exp(s_ij - m_i) / sum_{j' in V(i)} exp(s_ij' - m_i)
 *     o_i    = sum_j P_ij v_j
 *     lse_i  = m_i + log(sum_{j in V(i)} exp(s_ij - m_i))
 *   A query row with an empty valid set (Lk_b == 0, cross-attention only)
 *   gets o_i = 0 and lse_i = -infinity.
 *
 *   Generalized dot-product attention, non-softmax (the GDPA bullet of the
 *   same page: a pipeline for non-softmax activations).  The activation used
 *   by this library is SiLU of the scaled score divided by the sequence
 *   length Lq_b:
 *     u_ij = scale * <q_i, k_j>
 *     P_ij = u_ij * sigmoid(u_ij) / Lq_b   for j in V(i), 0 otherwise
 *     o_i  = sum_j P_ij v_j                 (no lse is produced)
 *
 *   Backward passes are the analytic gradients of the loss L(o) with
 *   dL/do_i = dO_i, obtained by the chain rule through the formulas above:
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = <dO_i, v_j>
 *     softmax:  D_i = sum_j P_ij dP_ij,  dS_ij = P_ij (dP_ij - D_i)
 *     GDPA:     dS_ij = dP_ij * SiLU'(u_ij) / Lq_b,
 *               SiLU'(u) = sigmoid(u) (1 + u (1 - sigmoid(u)))
 *     dQ_i  = scale * sum_j dS_ij k_j
 *     dK_j  = scale * sum_i dS_ij q_i
 *
 * Layouts: Q is [Tq, H, Dqk], K is [Tk, H, Dqk], V is [Tk, H, Dv], O and dO
 * are [Tq, H, Dv], lse is [Tq, H]; all row-major, all double.  offs_q and
 * offs_k are int64 [B+1].
 *
 * Parallelism: one OpenMP task per (sequence, head); the outputs of different
 * tasks never overlap, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS 1
#define ORACLE_BAD_OFFSETS 2
#define ORACLE_NO_MEMORY 3

#define ACT_SOFTMAX 0
#define ACT_SILU_OVER_LEN 1

static double dot(const double* a, const double* b, int n) {
  double acc = 0.0;
  for (int d = 0; d < n; ++d) acc += a[d] * b[d];
  return acc;
}

static double sigmoid(double u) { return 1.0 / (1.0 + exp(-u)); }

static int check_offsets(int64_t B, const int64_t* offs_q, const int64_t* offs_k,
                         int causal) {
  if (offs_q[0] != 0 || offs_k[0] != 0) return ORACLE_BAD_OFFSETS;
  for (int64_t b = 0; b < B; ++b) {
    if (offs_q[b + 1] < offs_q[b] || offs_k[b + 1] < offs_k[b])
      return ORACLE_BAD_OFFSETS;
    if (causal && offs_q[b + 1] - offs_q[b] != offs_k[b + 1] - offs_k[b])
      return ORACLE_BAD_OFFSETS;
  }
  return ORACLE_OK;
}

/* Number of valid key columns for query row i: V(i) is a prefix of the keys. */
static int64_t valid_count(int64_t i, int64_t Lk, int causal) {
  if (!causal) return Lk;
  return (i + 1 < Lk) ? i + 1 : Lk;
}

/*
 * Fills p[0..n) with the attention weights P_ij of one query row, j < n.
 * s holds the scores u_ij = scale * <q_i, k_j> on entry and is left as is.
 * Returns lse (softmax) or 0 (GDPA).
 */
static double row_weights(const double* s, int64_t n, int64_t Lq, int act,
                          double* p) {
  if (act == ACT_SOFTMAX) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) sum += exp(s[j] - m);
    for (int64_t j = 0; j < n; ++j) p[j] = exp(s[j] - m) / sum;
    return m + log(sum);
  }
  for (int64_t j = 0; j < n; ++j) p[j] = s[j] * sigmoid(s[j]) / (double)Lq;
  return 0.0;
}

int oracle_fwd(int64_t B, int32_t H, int32_t Dqk, int32_t Dv,
               const int64_t* offs_q, const int64_t* offs_k,
               const double* q, const double* k, const double* v,
               double scale, int32_t causal, int32_t act,
               double* o, double* lse) {
  if (B < 0 || H <= 0 || Dqk <= 0 || Dv <= 0) return ORACLE_BAD_ARGS;
  if (act != ACT_SOFTMAX && act != ACT_SILU_OVER_LEN) return ORACLE_BAD_ARGS;
  if (B == 0) return ORACLE_OK;
  int rc = check_offsets(B, offs_q, offs_k, causal);
  if (rc != ORACLE_OK) return rc;
  int64_t ntask = B * (int64_t)H;
  int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t task = 0; task < ntask; ++task) {
    int64_t b = task / H;
    int32_t h = (int32_t)(task % H);
    int64_t q0 = offs_q[b], Lq = offs_q[b + 1] - q0;
    int64_t k0 = offs_k[b], Lk = offs_k[b + 1] - k0;
    if (Lq == 0) continue;
    double* s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
    double* p = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
    if (!s || !p) {
      free(s); free(p);
#pragma omp atomic write
      failed = 1;
      continue;
    }
    for (int64_t i = 0; i < Lq; ++i) {
      const double* qi = q + ((q0 + i) * H + h) * Dqk;
      double* oi = o + ((q0 + i) * H + h) * Dv;
      int64_t n = valid_count(i, Lk, causal);
      for (int d = 0; d < Dv; ++d) oi[d] = 0.0;
      if (n == 0) {
        if (lse) lse[(q0 + i) * H + h] = (act == ACT_SOFTMAX) ? -INFINITY : 0.0;
        continue;
      }
      for (int64_t j = 0; j < n; ++j)
        s[j] = scale * dot(qi, k + ((k0 + j) * H + h) * Dqk, Dqk);
      double l = row_weights(s, n, Lq, act, p);
      for (int64_t j = 0; j < n; ++j) {
        const double* vj = v + ((k0 + j) * H + h) * Dv;
        for (int d = 0; d < Dv; ++d) oi[d] += p[j] * vj[d];
      }
      if (lse) lse[(q0 + i) * H + h] = (act == ACT_SOFTMAX) ? l : 0.0;
    }
    free(s);
    free(p);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

int oracle_bwd(int64_t B, int32_t H, int32_t Dqk, int32_t Dv,
               const int64_t* offs_q, const int64_t* offs_k,
               const double* q, const double* k, const double* v,
               const double* dout, double scale, int32_t causal, int32_t act,
               double* dq, double* dk, double* dv) {
  if (B < 0 || H <= 0 || Dqk <= 0 || Dv <= 0) return ORACLE_BAD_ARGS;
  if (act != ACT_SOFTMAX && act != ACT_SILU_OVER_LEN) return ORACLE_BAD_ARGS;
  if (B == 0) return ORACLE_OK;
  int rc = check_offsets(B, offs_q, offs_k, causal);
  if (rc != ORACLE_OK) return rc;
  int64_t ntask = B * (int64_t)H;
  int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t task = 0; task < ntask; ++task) {
    int64_t b = task / H;
    int32_t h = (int32_t)(task % H);
    int64_t q0 = offs_q[b], Lq = offs_q[b + 1] - q0;
    int64_t k0 = offs_k[b], Lk = offs_k[b + 1] - k0;
    /* dK and dV are sums over the query rows of this sequence: start at 0. */
    for (int64_t j = 0; j < Lk; ++j) {
      double* dkj = dk + ((k0 + j) * H + h) * Dqk;
      double* dvj = dv + ((k0 + j) * H + h) * Dv;
      for (int d = 0; d < Dqk; ++d) dkj[d] = 0.0;
      for (int d = 0; d < Dv; ++d) dvj[d] = 0.0;
    }
    for (int64_t i = 0; i < Lq; ++i) {
      double* dqi = dq + ((q0 + i) * H + h) * Dqk;
      for (int d = 0; d < Dqk; ++d) dqi[d] = 0.0;
    }
    if (Lq == 0 || Lk == 0) continue;
    double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
    double* p = (double*)malloc(sizeof(double) * (size_t)Lk);
    double* dp = (double*)malloc(sizeof(double) * (size_t)Lk);
    if (!s || !p || !dp) {
      free(s); free(p); free(dp);
#pragma omp atomic write
      failed = 1;
      continue;
    }
    for (int64_t i = 0; i < Lq; ++i) {
      const double* qi = q + ((q0 + i) * H + h) * Dqk;
      const double* doi = dout + ((q0 + i) * H + h) * Dv;
      double* dqi = dq + ((q0 + i) * H + h) * Dqk;
      int64_t n = valid_count(i, Lk, causal);
      for (int64_t j = 0; j < n; ++j)
        s[j] = scale * dot(qi, k + ((k0 + j) * H + h) * Dqk, Dqk);
      row_weights(s, n, Lq, act, p);
      for (int64_t j = 0; j < n; ++j)
        dp[j] = dot(doi, v + ((k0 + j) * H + h) * Dv, Dv);
      double Di = 0.0;
      if (act == ACT_SOFTMAX)
        for (int64_t j = 0; j < n; ++j) Di += p[j] * dp[j];
      for (int64_t j = 0; j < n; ++j) {
        double ds;
        if (act == ACT_SOFTMAX) {
          ds = p[j] * (dp[j] - Di);
        } else {
          double sg = sigmoid(s[j]);
          ds = dp[j] * sg * (1.0 + s[j] * (1.0 - sg)) / (double)Lq;
        }
        const double* kj = k + ((k0 + j) * H + h) * Dqk;
        double* dkj = dk + ((k0 + j) * H + h) * Dqk;
        double* dvj = dv + ((k0 + j) * H + h) * Dv;
        for (int d = 0; d < Dqk; ++d) dqi[d] += scale * ds * kj[d];
        for (int d = 0; d < Dqk; ++d) dkj[d] += scale * ds * qi[d];
        for (int d = 0; d < Dv; ++d) dvj[d] += p[j] * doi[d];
      }
    }
    free(s);
    free(p);
    free(dp);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}
