/*
 * Gated DeltaNet recurrence, per token, in fp64 -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark load
 * this library.  It shares no code with the CUDA library.
 *
 * Definition (qiita Nyysyyan, "Gated-DeltaNet" section):
 *     S_i = alpha_i S_{i-1} (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,  h_i = S_i q_i
 * computed in the equivalent order gate -> predict -> correct -> write
 * (kkkzoz "linear-attention", "Gated DeltaNet" section):
 *     S <- alpha S;  p = S k;  S <- S + beta (v - p) k^T;  h = S q.
 * Optional separate erase e and write w strengths give
 *     S <- alpha S;  p = S k;  S <- S - e p k^T + w v k^T
 * (e = w = beta is the definition; e = 0, w = 1 is Mamba2).
 *
 * Inputs are fp32 arrays (bf16 values are exact in fp32); all arithmetic is fp64.
 * Token-major layout with heads inner: x[token][head][dim].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * One "unit" is one (sequence, head) recurrence.
 *   unit_start[u]  first token of the sequence (row index into q/k/v)
 *   unit_len[u]    number of tokens
 *   unit_head[u]   head index
 *   unit_out[u]    first row of this unit's outputs in `out` ([rows][dv])
 * S0: [n_units][dv][dk] fp32 or NULL (zeros).  S_final: [n_units][dv][dk] fp64.
 * erase, write: same layout as beta, or NULL (then beta).
 * Returns 0 on success, 1 on allocation failure, 2 on bad sizes.
 */
int oracle_gdn_units(const float* q, const float* k, const float* v,
                     const float* log_alpha, const float* beta,
                     const float* erase, const float* write,
                     const float* S0, int H, int dk, int dv,
                     const int64_t* unit_start, const int64_t* unit_len,
                     const int32_t* unit_head, const int64_t* unit_out, int n_units,
                     double* out, double* S_final, int n_threads) {
  if (H <= 0 || dk <= 0 || dv <= 0 || n_units < 0) return 2;
  int failed = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
  for (int u = 0; u < n_units; ++u) {
    double* S = (double*)malloc(sizeof(double) * (size_t)dv * dk);
    double* kk = (double*)malloc(sizeof(double) * (size_t)dk);
    double* qq = (double*)malloc(sizeof(double) * (size_t)dk);
    double* p = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!S || !kk || !qq || !p) {
      failed |= 1;
      free(S); free(kk); free(qq); free(p);
      continue;
    }
    const int h = unit_head[u];
    if (S0) {
      const float* s0 = S0 + (size_t)u * dv * dk;
      for (size_t i = 0; i < (size_t)dv * dk; ++i) S[i] = (double)s0[i];
    } else {
      memset(S, 0, sizeof(double) * (size_t)dv * dk);
    }
    for (int64_t t = 0; t < unit_len[u]; ++t) {
      const int64_t row = unit_start[u] + t;
      const size_t gi = (size_t)row * H + h;            /* gate / beta index */
      const float* kr = k + gi * dk;
      const float* qr = q + gi * dk;
      const float* vr = v + gi * dv;
      const double a = exp((double)log_alpha[gi]);
      const double b = (double)beta[gi];
      const double e = erase ? (double)erase[gi] : b;
      const double w = write ? (double)write[gi] : b;
      for (int j = 0; j < dk; ++j) { kk[j] = (double)kr[j]; qq[j] = (double)qr[j]; }
      /* gate, then predict with the gated state */
      for (int i = 0; i < dv; ++i) {
        double* Si = S + (size_t)i * dk;
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) { Si[j] *= a; acc += Si[j] * kk[j]; }
        p[i] = acc;
      }
      /* correct and write along k: S += (w v - e p) k^T, then read with q */
      double* o = out + (size_t)(unit_out[u] + t) * dv;
      for (int i = 0; i < dv; ++i) {
        double* Si = S + (size_t)i * dk;
        const double c = w * (double)vr[i] - e * p[i];
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) { Si[j] += c * kk[j]; acc += Si[j] * qq[j]; }
        o[i] = acc;
      }
    }
    memcpy(S_final + (size_t)u * dv * dk, S, sizeof(double) * (size_t)dv * dk);
    free(S); free(kk); free(qq); free(p);
  }
  return failed ? 1 : 0;
}

/* Number of threads OpenMP would use (for reporting the CPU baseline). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
