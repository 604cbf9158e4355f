/*
 * fp64 CPU oracle for the exact attention forward pass and its backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference arm may load or run this file.  It shares no code
 * with the CUDA path.
 *
 * What it computes is the plain definition, row by row:
 *
 *   S = scale * Q K^T,  P = softmax(S) row-wise,  O = P V
 *     ("Flash Attention 4 on Blackwell" (GPU-HPC book, ch. 13), section
 *      "Attention's real bottleneck", the formula O = softmax(QK^T/sqrt(d)) V;
 *      "Infra: Flash Attention", opening formula S = QK^T/sqrt(d), P, O = PV)
 *
 *   with the stable (safe) softmax: m = max_j s_j, l = sum_j exp(s_j - m),
 *   p_j = exp(s_j - m) / l
 *     ("Infra: Flash Attention", section "How softmax is computed in pieces")
 *
 *   and the per-row log-sum-exp  L_i = m_i + log l_i = log sum_j exp(S_ij)
 *     ("Infra: Flash Attention", Algorithm 1 (FlashAttention forward) and
 *      section "Why backward recomputes")
 *
 * Masks and head mapping:
 *   - causal is bottom-right aligned: query i sees key j iff
 *     j <= i + Sk - Sq  ("Flash Attention 4 on Blackwell", section
 *     "Causal attention and GQA").
 *   - GQA/MQA: query head h reads key/value head h / (Hq / Hkv) (same
 *     section: q_head = kv_head * ratio + offset).
 *   - A row with no visible key has no defined softmax; the pages leave its
 *     output to the operator ("Infra: Flash Attention", "Notation and boundary
 *     conditions").  Reading taken here: O = 0 and L = -inf.
 *
 * Everything is double precision with libm exp/log.  Inputs are decoded from
 * bf16 bit patterns exactly, or taken as doubles.  Layouts are contiguous
 * BSHD: q [B,Sq,Hq,dqk], k [B,Sk,Hkv,dqk], v [B,Sk,Hkv,dv].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* element i of a tensor stored as doubles (elem == 0) or bf16 bits (elem == 1) */
static inline double elem_at(const void* p, int64_t i, int elem) {
  return elem ? bf16_to_double(((const uint16_t*)p)[i]) : ((const double*)p)[i];
}

/* Number of keys query row i sees (keys 0 .. n-1): j < Sk, and under the
 * causal mask j <= i + Sk - Sq. */
static inline int64_t visible_keys(int64_t i, int64_t Sq, int64_t Sk, int causal) {
  int64_t nvis = Sk;
  if (causal) {
    int64_t last = i + Sk - Sq;
    nvis = last + 1 < Sk ? last + 1 : Sk;
    if (nvis < 0) nvis = 0;
  }
  return nvis;
}

typedef struct {
  const void *q, *k, *v;
  int elem;
  int64_t B, Hq, Hkv, Sq, Sk, dqk, dv;
  int causal;
  double scale;
  const int64_t* rows; /* NULL: rows 0 .. nrows-1 */
  int64_t nrows;
  double *o, *lse;
  int64_t first, step; /* this thread takes requests first, first + step, ... */
  int status;
} job_t;

/* One output row: linear row id r = (b * Sq + i) * Hq + h. */
static int one_row(const job_t* J, int64_t r, double* s, double* o_row, double* lse_out) {
  const int64_t h = r % J->Hq;
  const int64_t i = (r / J->Hq) % J->Sq;
  const int64_t b = r / (J->Hq * J->Sq);
  const int64_t kvh = h / (J->Hq / J->Hkv);

  const int64_t nvis = visible_keys(i, J->Sq, J->Sk, J->causal);
  if (nvis == 0) {
    for (int64_t c = 0; c < J->dv; ++c) o_row[c] = 0.0;
    *lse_out = -INFINITY;
    return 0;
  }

  /* scores s_j = scale * q_i . k_j */
  const int64_t qoff = ((b * J->Sq + i) * J->Hq + h) * J->dqk;
  for (int64_t j = 0; j < nvis; ++j) {
    const int64_t koff = ((b * J->Sk + j) * J->Hkv + kvh) * J->dqk;
    double acc = 0.0;
    for (int64_t c = 0; c < J->dqk; ++c)
      acc += elem_at(J->q, qoff + c, J->elem) * elem_at(J->k, koff + c, J->elem);
    s[j] = J->scale * acc;
  }

  /* stable softmax: m = max s, l = sum exp(s - m) */
  double m = s[0];
  for (int64_t j = 1; j < nvis; ++j)
    if (s[j] > m) m = s[j];
  double l = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    s[j] = exp(s[j] - m); /* s now holds the unnormalised weights */
    l += s[j];
  }

  /* O = (sum_j w_j v_j) / l */
  for (int64_t c = 0; c < J->dv; ++c) o_row[c] = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    const int64_t voff = ((b * J->Sk + j) * J->Hkv + kvh) * J->dv;
    for (int64_t c = 0; c < J->dv; ++c) o_row[c] += s[j] * elem_at(J->v, voff + c, J->elem);
  }
  for (int64_t c = 0; c < J->dv; ++c) o_row[c] /= l;

  /* L = m + log l */
  *lse_out = m + log(l);
  return 0;
}

static void* run_job(void* arg) {
  job_t* J = (job_t*)arg;
  double* s = (double*)malloc(sizeof(double) * (size_t)(J->Sk > 0 ? J->Sk : 1));
  if (!s) {
    J->status = -2;
    return 0;
  }
  const int64_t total = J->B * J->Sq * J->Hq;
  for (int64_t n = J->first; n < J->nrows; n += J->step) {
    int64_t r = J->rows ? J->rows[n] : n;
    if (r < 0 || r >= total) {
      J->status = -3;
      break;
    }
    one_row(J, r, s, J->o + n * J->dv, J->lse + n);
  }
  free(s);
  return 0;
}

/*
 * Compute O (nrows x dv, double) and L (nrows, double) for the requested rows.
 * rows == NULL computes rows 0 .. nrows-1 in linear order (b, i, h), which for
 * nrows = B*Sq*Hq is the whole output in BSHD order.
 * Returns 0, -1 on bad arguments, -2 on allocation failure, -3 on a bad row id.
 */
int oracle_attn_fwd(const void* q, const void* k, const void* v, int elem, int64_t B, int64_t Hq,
                    int64_t Hkv, int64_t Sq, int64_t Sk, int64_t dqk, int64_t dv, int causal,
                    double scale, const int64_t* rows, int64_t nrows, double* o, double* lse,
                    int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || dqk <= 0 || dv <= 0 || nrows < 0)
    return -1;
  if (Hq % Hkv != 0) return -1;
  if (nrows == 0) return 0;
  if (!q || !k || !v || !o || !lse) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if (nthreads > nrows) nthreads = (int)nrows;

  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  int* live = (int*)calloc((size_t)nthreads, sizeof(int));
  if (!jobs || !th || !live) {
    free(jobs);
    free(th);
    free(live);
    return -2;
  }
  /* interleaved requests keep the threads' costs even under the causal mask */
  for (int t = 0; t < nthreads; ++t) {
    job_t* J = &jobs[t];
    J->q = q, J->k = k, J->v = v, J->elem = elem;
    J->B = B, J->Hq = Hq, J->Hkv = Hkv, J->Sq = Sq, J->Sk = Sk, J->dqk = dqk, J->dv = dv;
    J->causal = causal, J->scale = scale, J->rows = rows, J->nrows = nrows, J->o = o, J->lse = lse;
    J->first = t;
    J->step = nthreads;
    if (t > 0 && pthread_create(&th[t], 0, run_job, J) == 0) live[t] = 1;
    else if (t > 0) run_job(J);
  }
  run_job(&jobs[0]);
  int status = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (t > 0 && live[t]) pthread_join(th[t], 0);
    if (jobs[t].status) status = jobs[t].status;
  }
  free(jobs);
  free(th);
  free(live);
  return status;
}

/* ---------------------------------------------------------------------------
 * Backward: the gradients of a scalar loss through O = softmax(S) V, given
 * dO = dLoss/dO.  The chain rule through the three steps gives
 * ("Infra: Flash Attention", section "Why backward recomputes" and its detail
 * on computing the gradients block by block):
 *
 *   dV = P^T dO,        dP = dO V^T,
 *   dS_ij = P_ij (dP_ij - D_i)   with D_i = sum_j P_ij dP_ij
 *     (the softmax Jacobian; the pages rewrite D_i as dO_i . O_i, which is
 *      the same number because O_i = sum_j P_ij V_j),
 *   dQ = scale dS K,    dK = scale dS^T Q    (S = scale Q K^T).
 *
 * Masks and heads as in the forward: a hidden key has P = 0 and receives no
 * gradient; a row with no visible key contributes nothing; a shared key/value
 * head (GQA/MQA) receives the sum over the query heads that read it.
 *
 * P is recomputed from the definition (stable softmax of the visible scores),
 * in double precision, row by row.  One thread owns a (batch, key/value head)
 * unit: all its query heads and rows, so dK and dV of the unit accumulate in
 * place without sharing.
 * ------------------------------------------------------------------------- */
typedef struct {
  const void *q, *k, *v, *dout;
  int elem;
  int64_t B, Hq, Hkv, Sq, Sk, dqk, dv;
  int causal;
  double scale;
  double *dq, *dk, *dvv;
  int64_t first, step;
  int status;
} bjob_t;

static void* run_bwd(void* arg) {
  bjob_t* J = (bjob_t*)arg;
  const size_t n = (size_t)(J->Sk > 0 ? J->Sk : 1);
  double* p = (double*)malloc(sizeof(double) * n);
  double* dp = (double*)malloc(sizeof(double) * n);
  if (!p || !dp) {
    free(p);
    free(dp);
    J->status = -2;
    return 0;
  }
  const int64_t ratio = J->Hq / J->Hkv;
  for (int64_t u = J->first; u < J->B * J->Hkv; u += J->step) {
    const int64_t b = u / J->Hkv, kvh = u % J->Hkv;
    for (int64_t h = kvh * ratio; h < (kvh + 1) * ratio; ++h) {
      for (int64_t i = 0; i < J->Sq; ++i) {
        const int64_t qoff = ((b * J->Sq + i) * J->Hq + h) * J->dqk;
        const int64_t ooff = ((b * J->Sq + i) * J->Hq + h) * J->dv;
        double* dq_row = J->dq + qoff;
        for (int64_t c = 0; c < J->dqk; ++c) dq_row[c] = 0.0;
        const int64_t nvis = visible_keys(i, J->Sq, J->Sk, J->causal);
        if (nvis == 0) continue;

        /* P_i. : stable softmax of the visible scores */
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) {
          const int64_t koff = ((b * J->Sk + j) * J->Hkv + kvh) * J->dqk;
          double acc = 0.0;
          for (int64_t c = 0; c < J->dqk; ++c)
            acc += elem_at(J->q, qoff + c, J->elem) * elem_at(J->k, koff + c, J->elem);
          p[j] = J->scale * acc;
          if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
          p[j] = exp(p[j] - m);
          l += p[j];
        }
        for (int64_t j = 0; j < nvis; ++j) p[j] /= l;

        /* dP_ij = dO_i . V_j and D_i = sum_j P_ij dP_ij */
        double D = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
          const int64_t voff = ((b * J->Sk + j) * J->Hkv + kvh) * J->dv;
          double acc = 0.0;
          for (int64_t c = 0; c < J->dv; ++c)
            acc += elem_at(J->dout, ooff + c, J->elem) * elem_at(J->v, voff + c, J->elem);
          dp[j] = acc;
          D += p[j] * acc;
        }

        /* dS_ij = P_ij (dP_ij - D_i); dQ_i, dK_j, dV_j */
        for (int64_t j = 0; j < nvis; ++j) {
          const double ds = p[j] * (dp[j] - D);
          const int64_t koff = ((b * J->Sk + j) * J->Hkv + kvh) * J->dqk;
          const int64_t voff = ((b * J->Sk + j) * J->Hkv + kvh) * J->dv;
          for (int64_t c = 0; c < J->dqk; ++c) {
            dq_row[c] += J->scale * ds * elem_at(J->k, koff + c, J->elem);
            J->dk[koff + c] += J->scale * ds * elem_at(J->q, qoff + c, J->elem);
          }
          for (int64_t c = 0; c < J->dv; ++c) J->dvv[voff + c] += p[j] * elem_at(J->dout, ooff + c, J->elem);
        }
      }
    }
  }
  free(p);
  free(dp);
  return 0;
}

/*
 * dq [B,Sq,Hq,dqk], dk [B,Sk,Hkv,dqk], dv [B,Sk,Hkv,dv] (doubles, written
 * whole) for q, k, v and dout [B,Sq,Hq,dv] given as doubles (elem 0) or bf16
 * bits (elem 1).  Returns 0, -1 on bad arguments, -2 on allocation failure.
 */
int oracle_attn_bwd(const void* q, const void* k, const void* v, const void* dout, int elem, int64_t B,
                    int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t dqk, int64_t dv, int causal,
                    double scale, double* dq, double* dk, double* dvv, int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || dqk <= 0 || dv <= 0) return -1;
  if (Hq % Hkv != 0) return -1;
  if (B == 0) return 0;
  if (!q || !k || !v || !dout || !dq || !dk || !dvv) return -1;
  memset(dk, 0, sizeof(double) * (size_t)(B * Sk * Hkv * dqk));
  memset(dvv, 0, sizeof(double) * (size_t)(B * Sk * Hkv * dv));
  const int64_t units = B * Hkv;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if (nthreads > units) nthreads = (int)units;
  bjob_t* jobs = (bjob_t*)calloc((size_t)nthreads, sizeof(bjob_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  int* live = (int*)calloc((size_t)nthreads, sizeof(int));
  if (!jobs || !th || !live) {
    free(jobs);
    free(th);
    free(live);
    return -2;
  }
  for (int t = 0; t < nthreads; ++t) {
    bjob_t* J = &jobs[t];
    J->q = q, J->k = k, J->v = v, J->dout = dout, J->elem = elem;
    J->B = B, J->Hq = Hq, J->Hkv = Hkv, J->Sq = Sq, J->Sk = Sk, J->dqk = dqk, J->dv = dv;
    J->causal = causal, J->scale = scale, J->dq = dq, J->dk = dk, J->dvv = dvv;
    J->first = t;
    J->step = nthreads;
    if (t > 0 && pthread_create(&th[t], 0, run_bwd, J) == 0) live[t] = 1;
    else if (t > 0) run_bwd(J);
  }
  run_bwd(&jobs[0]);
  int status = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (t > 0 && live[t]) pthread_join(th[t], 0);
    if (jobs[t].status) status = jobs[t].status;
  }
  free(jobs);
  free(th);
  free(live);
  return status;
}
