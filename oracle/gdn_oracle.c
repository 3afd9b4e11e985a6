/*
 * GDN forward, float64 CPU oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
 * load this file's library.  It shares no code, header, table or helper with
 * the CUDA path, and nothing here is tuned: it is the plain definition,
 * written out token by token.
 *
 * What it computes (the gated delta rule of the GDN layer):
 *   Named by the FlashQLA pages ("FlashQLA: fused linear-attention kernels for
 *   CP/backward (GDN)", section "Optimising GDN chunked prefill"): the layer
 *   whose chunked prefill is being accelerated is the Gated Delta Network.
 *   The recurrence is the published gated delta rule (Yang, Kautz and
 *   Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule",
 *   ICLR 2025, section "Gated delta rule"):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = scale * S_t q_t,            alpha_t = exp(g_t), scale = 1/sqrt(d_k)
 *
 *   with S_t a d_v x d_k matrix per sequence and value head.  Value head j
 *   reads query/key head floor(j * h_qk / h_v) (grouped heads).  Chunked
 *   prefill evaluates this same layer chunk by chunk, so its exact result is
 *   this recurrence's result; the context-parallel split is an exact
 *   re-association of it (pages, section "AutoCP": segment start states are
 *   combined exactly).
 *
 * Layouts (all row-major, float64, token-major and head-interleaved):
 *   q, k   [T_total, h_qk, d_k]     v, o [T_total, h_v, d_v]
 *   g, beta [T_total, h_v]           h0, hT [n_seqs, h_v, d_k, d_v]
 * The stored state is H = S^T (d_k x d_v), the key-by-value orientation.
 * Sequence n covers tokens [cu_seqlens[n], cu_seqlens[n+1]).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int n_seqs, h_qk, h_v, d_k, d_v;
  double scale;
  const int64_t *cu;
  const double *q, *k, *v, *g, *beta, *h0;
  double *o, *hT;
  const int32_t *head_mask; /* optional: only heads with mask[j] != 0 */
  int next_task;            /* guarded by lock */
  pthread_mutex_t lock;
} oracle_job;

/* One (sequence, value head): the recurrence above, literally. */
static void run_one(const oracle_job *J, int n, int j) {
  const int dk = J->d_k, dv = J->d_v, hqk = J->h_qk, hv = J->h_v;
  const int i = (int)(((int64_t)j * hqk) / hv); /* grouped-head mapping */
  double *S = (double *)calloc((size_t)dv * dk, sizeof(double));
  double *Sk = (double *)malloc((size_t)dv * sizeof(double));
  if (!S || !Sk) { free(S); free(Sk); return; }
  if (J->h0) { /* S = H0^T */
    const double *H0 = J->h0 + ((size_t)n * hv + j) * dk * dv;
    for (int a = 0; a < dv; a++)
      for (int c = 0; c < dk; c++) S[(size_t)a * dk + c] = H0[(size_t)c * dv + a];
  }
  for (int64_t t = J->cu[n]; t < J->cu[n + 1]; t++) {
    const double *kt = J->k + ((size_t)t * hqk + i) * dk;
    const double *qt = J->q + ((size_t)t * hqk + i) * dk;
    const double *vt = J->v + ((size_t)t * hv + j) * dv;
    const double alpha = exp(J->g[(size_t)t * hv + j]);
    const double b = J->beta[(size_t)t * hv + j];
    /* Sk = S_{t-1} k_t */
    for (int a = 0; a < dv; a++) {
      double acc = 0.0;
      for (int c = 0; c < dk; c++) acc += S[(size_t)a * dk + c] * kt[c];
      Sk[a] = acc;
    }
    /* S_t = alpha (S_{t-1} - beta (S_{t-1} k) k^T) + beta v k^T */
    for (int a = 0; a < dv; a++)
      for (int c = 0; c < dk; c++) {
        double s = S[(size_t)a * dk + c];
        S[(size_t)a * dk + c] = alpha * (s - b * Sk[a] * kt[c]) + b * vt[a] * kt[c];
      }
    /* o_t = scale * S_t q_t */
    double *ot = J->o + ((size_t)t * hv + j) * dv;
    for (int a = 0; a < dv; a++) {
      double acc = 0.0;
      for (int c = 0; c < dk; c++) acc += S[(size_t)a * dk + c] * qt[c];
      ot[a] = J->scale * acc;
    }
  }
  if (J->hT) { /* H_T = S_T^T */
    double *HT = J->hT + ((size_t)n * hv + j) * dk * dv;
    for (int c = 0; c < dk; c++)
      for (int a = 0; a < dv; a++) HT[(size_t)c * dv + a] = S[(size_t)a * dk + c];
  }
  free(S);
  free(Sk);
}

static void *worker(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  const int n_tasks = J->n_seqs * J->h_v;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int task = J->next_task++;
    pthread_mutex_unlock(&J->lock);
    if (task >= n_tasks) break;
    int n = task / J->h_v, j = task % J->h_v;
    if (J->head_mask && !J->head_mask[j]) continue;
    run_one(J, n, j);
  }
  return NULL;
}

/*
 * Runs the recurrence for every (sequence, value head) whose head_mask entry
 * is nonzero (all heads when head_mask is NULL).  h0 may be NULL (zero initial
 * state); hT may be NULL (final state not written).  Outputs of masked-out
 * heads are left untouched.  Returns 0, or -1 on a bad argument.
 */
int gdn_oracle_recurrence(int n_seqs, const int64_t *cu_seqlens, int h_qk, int h_v, int d_k,
                          int d_v, double scale, const double *q, const double *k,
                          const double *v, const double *g, const double *beta,
                          const double *h0, double *o, double *hT, const int32_t *head_mask,
                          int n_threads) {
  if (n_seqs < 0 || h_qk <= 0 || h_v <= 0 || d_k <= 0 || d_v <= 0 || !cu_seqlens) return -1;
  if (!q || !k || !v || !g || !beta || !o) return -1;
  for (int n = 0; n < n_seqs; n++)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  oracle_job J;
  memset(&J, 0, sizeof(J));
  J.n_seqs = n_seqs; J.h_qk = h_qk; J.h_v = h_v; J.d_k = d_k; J.d_v = d_v;
  J.scale = scale; J.cu = cu_seqlens;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
  J.o = o; J.hT = hT; J.head_mask = head_mask;
  pthread_mutex_init(&J.lock, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  int started = 0;
  for (int w = 1; w < n_threads; w++)
    if (pthread_create(&th[started], NULL, worker, &J) == 0) started++;
  worker(&J);
  for (int w = 0; w < started; w++) pthread_join(th[w], NULL);
  pthread_mutex_destroy(&J.lock);
  return 0;
}
