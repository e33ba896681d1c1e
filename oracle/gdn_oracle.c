/*
 * Oracle for the forward pass of the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes, token by token, in IEEE double precision, per
 * (sequence, head):
 *
 *     S_t = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t                      alpha_t = exp(g_t)
 *
 * This is the gated delta rule of Yang et al., "Gated Delta Networks"
 * (arXiv 2412.06464), the algorithm that "v1.0 Architecture & Design Spec",
 * section 2.3 (Gated Delta Net block) and section 12a.1 name for the GDN
 * kernel.  The token loop with one state update and one read per step follows
 * the eager recurrence of "Model Architecture Walkthrough", section 5.5
 * (Step 5: Gated Delta Rule Recurrence); the decay alpha = exp(gate) follows
 * the same page, section 5.2.1.  The product S (I - beta k k^T) is expanded
 * as S - beta (S k) k^T, which is the same matrix written without forming
 * the dv x dk identity.
 *
 * A second mode, GDN_ORACLE_GLA, drops beta and the erase term and keeps a
 * scalar decay:  S_t = alpha_t S_{t-1} + v_t k_t^T.  That is the recurrence
 * the HyMo pages print ("Model Architecture Walkthrough", section 5.2.1, and
 * "Optimization Quartet", Triton GDN kernel section 3.2) with the write key
 * b = k, the read key c = q and one decay value shared by all key
 * dimensions.  It exists only to pin the decay and write paths against the
 * closed form of the unrolled decay ("Model Architecture Walkthrough",
 * section 5.3.1).
 *
 * Data layout (all arrays dense, row-major, double):
 *   q, k   [T_total, H, dk]      v, o   [T_total, H, dv]
 *   g, beta [T_total, H]
 *   s0, sN  [num_seqs, H, dk, dv]  -- the state is stored transposed,
 *            element (i, j) = S[j][i], i.e. H = S^T with key index first.
 *   cu      [num_seqs + 1]        sequence n covers rows cu[n] .. cu[n+1]-1.
 * s0 may be NULL (zero initial state); sN may be NULL (not returned).
 *
 * Optional q/k normalisation (qk_l2norm != 0): x / sqrt(sum(x^2) + 1e-6),
 * applied to each q_t and k_t before use.
 *
 * Work is spread over (sequence, head) units with POSIX threads; every unit
 * is computed by exactly one thread with the same operation order, so the
 * result does not depend on the thread count.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no fused
 * multiply-add contraction, so x86 and Arm hosts round identically).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

enum { GDN_ORACLE_DELTA = 0, GDN_ORACLE_GLA = 1 };

typedef struct {
  const double *q, *k, *v, *g, *beta, *s0;
  const long long *cu;
  int num_seqs, H, dk, dv, mode, qk_l2norm;
  double *o, *sN;
  int next_unit;
  pthread_mutex_t lock;
} oracle_job;

static void l2normalise(const double *x, double *y, int n) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + 1e-6);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv;
}

/* One (sequence, head) unit.  S is held as dv rows of dk columns. */
static void run_unit(const oracle_job *J, int n, int h, double *S, double *Sk,
                     double *qn, double *kn) {
  const int H = J->H, dk = J->dk, dv = J->dv;
  const size_t state_off = ((size_t)n * H + h) * (size_t)dk * dv;

  /* S_0: the stored state is H0 = S0^T, element (i, j) at i*dv + j. */
  for (int j = 0; j < dv; ++j)
    for (int i = 0; i < dk; ++i)
      S[(size_t)j * dk + i] = J->s0 ? J->s0[state_off + (size_t)i * dv + j] : 0.0;

  for (long long t = J->cu[n]; t < J->cu[n + 1]; ++t) {
    const size_t row = (size_t)t * H + h;
    const double *q = J->q + row * dk;
    const double *k = J->k + row * dk;
    const double *v = J->v + row * dv;
    if (J->qk_l2norm) {
      l2normalise(q, qn, dk);
      l2normalise(k, kn, dk);
      q = qn;
      k = kn;
    }
    const double alpha = exp(J->g[row]);

    if (J->mode == GDN_ORACLE_DELTA) {
      const double beta = J->beta[row];
      /* Sk = S_{t-1} k_t */
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(size_t)j * dk + i] * k[i];
        Sk[j] = acc;
      }
      /* S_t = alpha (S - beta Sk k^T) + beta v k^T */
      for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i) {
          double *s = &S[(size_t)j * dk + i];
          *s = alpha * (*s - beta * Sk[j] * k[i]) + beta * v[j] * k[i];
        }
    } else {
      /* S_t = alpha S + v k^T */
      for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i) {
          double *s = &S[(size_t)j * dk + i];
          *s = alpha * (*s) + v[j] * k[i];
        }
    }

    /* o_t = S_t q_t (read after the update) */
    double *o = J->o + row * dv;
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)j * dk + i] * q[i];
      o[j] = acc;
    }
  }

  if (J->sN)
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j)
        J->sN[state_off + (size_t)i * dv + j] = S[(size_t)j * dk + i];
}

static void *worker(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  const int units = J->num_seqs * J->H;
  double *S = (double *)malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double *Sk = (double *)malloc(sizeof(double) * (size_t)J->dv);
  double *qn = (double *)malloc(sizeof(double) * (size_t)J->dk);
  double *kn = (double *)malloc(sizeof(double) * (size_t)J->dk);
  if (!S || !Sk || !qn || !kn) {
    free(S); free(Sk); free(qn); free(kn);
    return (void *)1;
  }
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int u = J->next_unit++;
    pthread_mutex_unlock(&J->lock);
    if (u >= units) break;
    run_unit(J, u / J->H, u % J->H, S, Sk, qn, kn);
  }
  free(S); free(Sk); free(qn); free(kn);
  return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 if a thread failed. */
int gdn_oracle_forward(const double *q, const double *k, const double *v,
                       const double *g, const double *beta, const double *s0,
                       const long long *cu, int num_seqs, int H, int dk, int dv,
                       int mode, int qk_l2norm, double *o, double *sN,
                       int nthreads) {
  if (!q || !k || !v || !g || !cu || !o || num_seqs < 0 || H <= 0 || dk <= 0 ||
      dv <= 0 || (mode != GDN_ORACLE_DELTA && mode != GDN_ORACLE_GLA) ||
      (mode == GDN_ORACLE_DELTA && !beta))
    return -1;
  for (int n = 0; n < num_seqs; ++n)
    if (cu[n + 1] < cu[n]) return -1;
  if (nthreads < 1) nthreads = 1;
  const int units = num_seqs * H;
  if (nthreads > units) nthreads = units > 0 ? units : 1;

  oracle_job J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.s0 = s0; J.cu = cu;
  J.num_seqs = num_seqs; J.H = H; J.dk = dk; J.dv = dv; J.mode = mode;
  J.qk_l2norm = qk_l2norm; J.o = o; J.sN = sN; J.next_unit = 0;
  pthread_mutex_init(&J.lock, NULL);

  int rc = 0;
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!tid) { pthread_mutex_destroy(&J.lock); return -2; }
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&tid[i], NULL, worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) {
    if (worker(&J) != NULL) rc = -2;
  }
  for (int i = 0; i < started; ++i) {
    void *ret = NULL;
    pthread_join(tid[i], &ret);
    if (ret != NULL) rc = -2;
  }
  free(tid);
  pthread_mutex_destroy(&J.lock);
  return rc;
}
