/*
 * gdn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously-correct fp64 CPU oracle for the Gated DeltaNet
 * (gated delta rule) recurrence.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library; the GPU
 * library shares no code, header, table or helper with it.
 *
 * Source: "Long-Context Aware Upcycling: A New Frontier for Hybrid LLM
 * Scaling", Appendix A.3 "GDN Layer Architecture", Eq. (16)-(19):
 *
 *   Eq. 16   S~_t = e^{g_t} S_{t-1}                 (S in R^{dk x dv})
 *   Eq. 17   v'_t = v_t - S~_t^T k_t
 *   Eq. 18   S_t  = S~_t + k_t (beta_t v'_t)^T
 *   Eq. 19   o_t  = S_t^T q_t / sqrt(dk)             (the UPDATED state)
 *
 * The oracle keeps the state in that paper orientation (dk rows, dv columns)
 * and walks the tokens one at a time in sequence order, exactly in the order of
 * the four equations.  At the library boundary states are exchanged in the
 * transposed layout [dv][dk] (row i of the boundary state is column i of the
 * paper's S), so S0 is transposed on entry and S_final on exit.  alpha_t is
 * the decay e^{g_t} itself (the caller supplies it, not g_t).
 *
 * Every step here is a textbook loop; there is no blocking, chunking, fusion
 * or reordering.  Parity status: pinned (see the tests' closed-form,
 * brute-force rational and invariant checks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* io dtype codes shared only with this file's Python wrapper */
#define ORACLE_F32 0
#define ORACLE_BF16 1

/* exact widening of one input element to fp64 */
static double load_elem(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  /* bfloat16: the top 16 bits of an IEEE-754 binary32 */
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/*
 * One token of the recurrence, Eq. (16)-(19), paper orientation.
 *   Sp     : dk x dv state, row-major (Sp[i*dv + j]), updated in place
 *   q, k   : dk vectors;  v : dv vector;  alpha = e^{g_t};  beta = beta_t
 *   o      : dv output;   vp : dv scratch for v'_t
 */
static void gdn_token(double* Sp, const double* q, const double* k, const double* v,
                      double alpha, double beta, int dk, int dv, double* o, double* vp) {
  /* Eq. 16: S~ = e^{g} S */
  for (int64_t a = 0; a < (int64_t)dk * dv; ++a) Sp[a] *= alpha;
  /* Eq. 17: v' = v - S~^T k */
  for (int j = 0; j < dv; ++j) vp[j] = 0.0;
  for (int i = 0; i < dk; ++i) {
    const double ki = k[i];
    const double* row = Sp + (int64_t)i * dv;
    for (int j = 0; j < dv; ++j) vp[j] += row[j] * ki;
  }
  for (int j = 0; j < dv; ++j) vp[j] = v[j] - vp[j];
  /* Eq. 18: S = S~ + k (beta v')^T */
  for (int i = 0; i < dk; ++i) {
    const double ki = k[i];
    double* row = Sp + (int64_t)i * dv;
    for (int j = 0; j < dv; ++j) row[j] += ki * (beta * vp[j]);
  }
  /* Eq. 19: o = S^T q / sqrt(dk), with the updated S */
  for (int j = 0; j < dv; ++j) o[j] = 0.0;
  for (int i = 0; i < dk; ++i) {
    const double qi = q[i];
    const double* row = Sp + (int64_t)i * dv;
    for (int j = 0; j < dv; ++j) o[j] += row[j] * qi;
  }
  const double inv_sqrt_dk = 1.0 / sqrt((double)dk);
  for (int j = 0; j < dv; ++j) o[j] *= inv_sqrt_dk;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Prefill over N packed sequences.
 *   q, k       : [T_total][H][dk]   (dtype io_dtype)
 *   v          : [T_total][H][dv]   (dtype io_dtype)
 *   alpha,beta : [T_total][H]       fp32
 *   S0         : [N][H][dv][dk] fp64, or NULL for a zero initial state
 *   cu_seqlens : N+1 int64 offsets into the token axis (cu[0] = 0)
 *   out        : [T_total][H][dv] fp64
 *   S_final    : [N][H][dv][dk] fp64, or NULL
 * Independent (sequence, head) units are distributed over nthreads OpenMP
 * threads (nthreads <= 0: the runtime default).  Returns the thread count
 * used, or a negative value on allocation failure.
 */
int oracle_gdn_prefill(const void* q, const void* k, const void* v, int io_dtype,
                       const float* alpha, const float* beta, const double* S0,
                       const int64_t* cu_seqlens, int N, int H, int dk, int dv,
                       double* out, double* S_final, int nthreads) {
  int used = 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
  used = nthreads;
#else
  (void)nthreads;
#endif
  int failed = 0;
  const int64_t units = (int64_t)N * H;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
  {
    double* Sp = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* qd = (double*)malloc(sizeof(double) * (size_t)dk);
    double* kd = (double*)malloc(sizeof(double) * (size_t)dk);
    double* vd = (double*)malloc(sizeof(double) * (size_t)dv);
    double* vp = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!Sp || !qd || !kd || !vd || !vp) {
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t u = 0; u < units; ++u) {
        const int n = (int)(u / H), h = (int)(u % H);
        /* boundary state [dv][dk] -> paper state [dk][dv] */
        for (int i = 0; i < dk; ++i)
          for (int j = 0; j < dv; ++j)
            Sp[(int64_t)i * dv + j] =
                S0 ? S0[(((int64_t)n * H + h) * dv + j) * dk + i] : 0.0;
        for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
          const int64_t qk_base = (t * H + h) * dk, v_base = (t * H + h) * dv;
          for (int i = 0; i < dk; ++i) {
            qd[i] = load_elem(q, io_dtype, qk_base + i);
            kd[i] = load_elem(k, io_dtype, qk_base + i);
          }
          for (int j = 0; j < dv; ++j) vd[j] = load_elem(v, io_dtype, v_base + j);
          gdn_token(Sp, qd, kd, vd, (double)alpha[t * H + h], (double)beta[t * H + h], dk, dv,
                    out + v_base, vp);
        }
        if (S_final)
          for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
              S_final[(((int64_t)n * H + h) * dv + j) * dk + i] = Sp[(int64_t)i * dv + j];
      }
    }
    free(Sp); free(qd); free(kd); free(vd); free(vp);
  }
  return failed ? -1 : used;
}

/*
 * One decode step for N independent sequences (one new token each): the same
 * recurrence at T = 1 against a cached state.
 *   q, k : [N][H][dk];  v : [N][H][dv];  alpha, beta : [N][H] fp32
 *   S    : [N][H][dv][dk] fp64, updated in place
 *   out  : [N][H][dv] fp64
 */
int oracle_gdn_decode_step(const void* q, const void* k, const void* v, int io_dtype,
                           const float* alpha, const float* beta, double* S, int N, int H,
                           int dk, int dv, double* out, int nthreads) {
  int64_t* cu = (int64_t*)malloc(sizeof(int64_t) * ((size_t)N + 1));
  if (!cu) return -1;
  for (int n = 0; n <= N; ++n) cu[n] = n;
  int r = oracle_gdn_prefill(q, k, v, io_dtype, alpha, beta, S, cu, N, H, dk, dv, out, S,
                             nthreads);
  free(cu);
  return r;
}
