/*
 * fp64 CPU oracle of the Kimi Delta Attention (KDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the library's product path links,
 * loads or calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code with the CUDA kernels.
 *
 * What it computes (per sequence and head, token by token, in fp64):
 *   - gate, page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.3
 *     (lower-bounded decay): the per-key-channel log-decay is
 *     g_min * Sigmoid(logit) with g_min = -5, and alpha = exp(log-decay).
 *     The caller's logit already contains the per-head scale e^{A^h}.
 *     Variant map (decay_map = 1): the predecessor model's unbounded map that
 *     page "Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽" contrasts with the bound
 *     (section "最被低估的一个细节：下界衰减"), log-decay = -Softplus(logit)
 *     = -ln(1 + e^logit), which has no lower limit.
 *   - recurrence, same page §3.1 (KDA equation) and page "Kimi K3 架构篇：一文详解
 *     2.8 万亿参数的巨型怪兽", section "KDA 到底在算什么":
 *        S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *        o_t = S_t^T q_t,
 *     with S_t of shape d_k x d_v; Diag(alpha_t) multiplies from the left, so
 *     it scales the ROWS of S (one row per key channel).
 *   - the step order of §3.2 of the first page, which is the same equation
 *     written out: decay the rows, read the old prediction with k, write the
 *     beta-weighted error back along k, then read the output with q from the
 *     UPDATED state (so o_t includes token t).
 *
 * Inputs are read exactly as stored: fp32, bf16 (raw bit patterns, widened
 * exactly) or fp64.  beta is fp32 (already in (0, 1)); no normalisation or
 * scaling of q or k is applied.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

#define ORACLE_DECAY_BOUNDED 0
#define ORACLE_DECAY_SOFTPLUS 1

static double load_elem(const void* p, int dtype, int64_t i) {
  if (dtype == ORACLE_F64) return ((const double*)p)[i];
  if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
  /* bf16: the 16 stored bits are the high half of an fp32 */
  uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* The log-decay of one channel, then alpha = exp of it:
 *   bounded:  g_min * Sigmoid(x), g_min = -5;
 *   softplus: -ln(1 + e^x), written max(x, 0) + ln(1 + e^{-|x|}) so that no
 *             intermediate overflows (x = +inf gives alpha = 0, -inf gives 1). */
static double decay_alpha(double logit, int decay_map) {
  if (decay_map == ORACLE_DECAY_SOFTPLUS) {
    const double softplus = (logit > 0.0 ? logit : 0.0) + log1p(exp(-fabs(logit)));
    return exp(-softplus);
  }
  const double sig = 1.0 / (1.0 + exp(-logit));
  return exp(-5.0 * sig);
}

/*
 * One (sequence, head) chain.
 *   q, k, g: token rows of d_k values, v: token rows of d_v values; the row of
 *   token j (0 <= j < n) of this chain starts at element (row0 + j*row_stride)*d
 *   of its array (d = d_k or d_v).  beta: element row0 + j*row_stride.
 *   s0: d_k x d_v initial state (row major, d_v contiguous) or NULL for zeros.
 *   o:  n x d_v outputs; s_out: d_k x d_v final state (both fp64, may be NULL).
 *   snaps: with snap_every > 0, the state after the first m * snap_every tokens
 *   (the prefix-cache snapshots of the first page's §9) for m = 1 .. n / snap_every,
 *   one d_k x d_v matrix each (may be NULL).
 */
static void run_chain(const void* q, const void* k, const void* v, const void* g, int dtype,
                      const float* beta, int64_t row0, int64_t row_stride, int64_t n,
                      int32_t d_k, int32_t d_v, const double* s0, double* o, double* s_out,
                      int64_t snap_every, double* snaps, int decay_map) {
  double* S = (double*)calloc((size_t)d_k * d_v, sizeof(double));
  double* kk = (double*)malloc(sizeof(double) * d_k);
  double* qq = (double*)malloc(sizeof(double) * d_k);
  double* alpha = (double*)malloc(sizeof(double) * d_k);
  double* err = (double*)malloc(sizeof(double) * d_v);
  if (s0) memcpy(S, s0, sizeof(double) * (size_t)d_k * d_v);

  for (int64_t j = 0; j < n; ++j) {
    const int64_t row = row0 + j * row_stride;
    const double b = (double)beta[row];
    for (int32_t i = 0; i < d_k; ++i) {
      kk[i] = load_elem(k, dtype, row * d_k + i);
      qq[i] = load_elem(q, dtype, row * d_k + i);
      alpha[i] = decay_alpha(load_elem(g, dtype, row * d_k + i), decay_map);
    }
    /* 1. decay: S_bar = Diag(alpha) S  (row i scaled by alpha_i) */
    for (int32_t i = 0; i < d_k; ++i)
      for (int32_t c = 0; c < d_v; ++c) S[(int64_t)i * d_v + c] *= alpha[i];
    /* 2. read the old prediction v_hat = S_bar^T k, and 3. the weighted error */
    for (int32_t c = 0; c < d_v; ++c) {
      double vhat = 0.0;
      for (int32_t i = 0; i < d_k; ++i) vhat += S[(int64_t)i * d_v + c] * kk[i];
      err[c] = b * (load_elem(v, dtype, row * d_v + c) - vhat);
    }
    /* 4. write: S = S_bar + k err^T */
    for (int32_t i = 0; i < d_k; ++i)
      for (int32_t c = 0; c < d_v; ++c) S[(int64_t)i * d_v + c] += kk[i] * err[c];
    /* 5. read out from the updated state: o = S^T q */
    if (o) {
      for (int32_t c = 0; c < d_v; ++c) {
        double acc = 0.0;
        for (int32_t i = 0; i < d_k; ++i) acc += S[(int64_t)i * d_v + c] * qq[i];
        o[j * d_v + c] = acc;
      }
    }
    /* 6. snapshot of the state after j + 1 tokens */
    if (snaps && snap_every > 0 && (j + 1) % snap_every == 0)
      memcpy(snaps + ((j + 1) / snap_every - 1) * (int64_t)d_k * d_v, S, sizeof(double) * (size_t)d_k * d_v);
  }
  if (s_out) memcpy(s_out, S, sizeof(double) * (size_t)d_k * d_v);
  free(S);
  free(kk);
  free(qq);
  free(alpha);
  free(err);
}

/*
 * Many independent chains, OpenMP over chains.  Chain c covers n[c] tokens
 * whose first row is row0[c] (rows advance by row_stride); its initial state is
 * s0 + c*d_k*d_v (s0 may be NULL), its outputs go to o + o_off[c] (n[c] x d_v)
 * and s_out + c*d_k*d_v (either may be NULL).  With snap_every > 0 its
 * n[c] / snap_every snapshots go to snaps + snap_off[c]*d_k*d_v.  decay_map
 * selects the gate (ORACLE_DECAY_BOUNDED or ORACLE_DECAY_SOFTPLUS).
 * Returns the number of threads used, or -1 on bad arguments.
 */
int kda_oracle_chains_map(const void* q, const void* k, const void* v, const void* g, int32_t dtype,
                          const float* beta, int64_t row_stride, int32_t d_k, int32_t d_v, int32_t nchains,
                          const int64_t* row0, const int64_t* n, const double* s0, double* o,
                          const int64_t* o_off, double* s_out, int64_t snap_every, double* snaps,
                          const int64_t* snap_off, int32_t decay_map) {
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return -1;
  if (decay_map != ORACLE_DECAY_BOUNDED && decay_map != ORACLE_DECAY_SOFTPLUS) return -1;
  if (d_k <= 0 || d_v <= 0 || nchains < 0 || row_stride <= 0 || snap_every < 0) return -1;
  if (snap_every > 0 && snaps && !snap_off) return -1;
  int used = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      used = omp_get_num_threads();
#endif
    }
#pragma omp for schedule(dynamic, 1)
    for (int32_t c = 0; c < nchains; ++c) {
      const int64_t dd = (int64_t)d_k * d_v;
      run_chain(q, k, v, g, dtype, beta, row0[c], row_stride, n[c], d_k, d_v, s0 ? s0 + c * dd : NULL,
                o ? o + o_off[c] : NULL, s_out ? s_out + c * dd : NULL, snap_every,
                (snap_every > 0 && snaps) ? snaps + snap_off[c] * dd : NULL, decay_map);
    }
  }
  return used;
}

int kda_oracle_chains_snap(const void* q, const void* k, const void* v, const void* g, int32_t dtype,
                           const float* beta, int64_t row_stride, int32_t d_k, int32_t d_v, int32_t nchains,
                           const int64_t* row0, const int64_t* n, const double* s0, double* o,
                           const int64_t* o_off, double* s_out, int64_t snap_every, double* snaps,
                           const int64_t* snap_off) {
  return kda_oracle_chains_map(q, k, v, g, dtype, beta, row_stride, d_k, d_v, nchains, row0, n, s0, o, o_off,
                               s_out, snap_every, snaps, snap_off, ORACLE_DECAY_BOUNDED);
}

int kda_oracle_chains(const void* q, const void* k, const void* v, const void* g, int32_t dtype,
                      const float* beta, int64_t row_stride, int32_t d_k, int32_t d_v, int32_t nchains,
                      const int64_t* row0, const int64_t* n, const double* s0, double* o,
                      const int64_t* o_off, double* s_out) {
  return kda_oracle_chains_snap(q, k, v, g, dtype, beta, row_stride, d_k, d_v, nchains, row0, n, s0, o, o_off,
                                s_out, 0, NULL, NULL);
}

int kda_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
