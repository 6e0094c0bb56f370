/*
 * gdr_oracle.c -- the CPU oracle for the gated delta rule.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load this code.  The
 * GPU library shares nothing with it: no header, no helper, no constant.
 *
 * What it computes: the plain token-by-token recurrence in fp64, for every (sequence, head)
 * pair independently (pairs are spread over POSIX threads; each pair is one sequential loop).
 *
 * Sources (web pages; sections as numbered on each page):
 *   [HH] heqinghuang.com "gpt2-to-kimi" (22,580 GPT-2s fit inside one Kimi K3)
 *   [DT] dev.to "From GPT-2 to Kimi K3: How Language Models Learned to Manage Memory"
 *   [EM] engineermaxxing.com "From GPT-2 to Kimi K3: one memory, seven eviction policies"
 *   [KH] kylehh.github.io "Kimi K3: From KV Cache to Selective Memory"
 *
 * State convention ([EM] §03b "convention flag"; [DT] §4): S is d_k x d_v, row i is key
 * channel i; the read of a key is v_hat = S^T k and the read-out is o = S^T q ([KH] §5).
 *
 * Gated delta rule, one token t (per-channel gate = Kimi Delta Attention, [DT] §5, [EM] §06b;
 * scalar gate = Gated DeltaNet, [DT] §4, [EM] §05c; alpha = 1 gives DeltaNet, [HH] §09):
 *   1. fade:    S <- Diag(a_t) S           (a_t the d_k-vector gate, or the scalar broadcast)
 *   2. read:    v_hat = S^T k_t            (the read is of the already-faded state, [DT] §4)
 *   3. correct: S <- S + beta_t k_t (v_t - v_hat)^T
 *   4. output:  o_t = S^T q_t              (read after the write, [HH] §09 and §10)
 * Plain (unnormalised) linear attention ([EM] §03b: the identity transition): S <- S + k_t v_t^T,
 * o_t = S^T q_t.  No feature map, no normaliser, no 1/sqrt(d) on q.
 * Gated linear attention (the decayed additive update without the erase term, [EM] §05b and
 * [HH] §11 for a scalar gate; one gate per key channel = row of S as in [DT] §5):
 * S <- Diag(a_t) S + k_t v_t^T, o_t = S^T q_t.  No beta.
 * A decode step is this loop run for one token from a given state.
 *
 * Layouts (all row-major, fp64):
 *   q, k  [T_total, H, d_k]   v, out [T_total, H, d_v]
 *   alpha [T_total, H, d_k] (per channel) or [T_total, H] (scalar)    beta [T_total, H]
 *   S0, S_final [n_seqs, H, d_k, d_v]       cu_seqlens [n_seqs + 1] (int64 offsets)
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_GATED_DELTA = 0, ORACLE_LINEAR = 1, ORACLE_GATED_LINEAR = 2 };

typedef struct {
  int mode;
  int n_seqs, H, dk, dv;
  const int64_t* cu;
  const double *q, *k, *v, *alpha, *beta, *S0;
  int alpha_per_channel;
  double *out, *S_final;
  const int32_t* pairs; /* optional list of (seq, head) pairs, flattened; NULL = all */
  int n_pairs;
  int n_threads;
} oracle_job;

typedef struct {
  const oracle_job* job;
  int tid;
} oracle_worker;

/* One (sequence, head) pair, token by token. */
static void run_pair(const oracle_job* J, int n, int h, double* S, double* vhat) {
  const int H = J->H, dk = J->dk, dv = J->dv;
  const size_t sidx = ((size_t)n * H + h) * (size_t)dk * dv;
  if (J->S0)
    memcpy(S, J->S0 + sidx, sizeof(double) * (size_t)dk * dv);
  else
    memset(S, 0, sizeof(double) * (size_t)dk * dv);

  for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
    const double* qt = J->q + ((size_t)t * H + h) * dk;
    const double* kt = J->k + ((size_t)t * H + h) * dk;
    const double* vt = J->v + ((size_t)t * H + h) * dv;
    double* ot = J->out + ((size_t)t * H + h) * dv;

    if (J->mode == ORACLE_LINEAR) {
      /* S <- S + k v^T */
      for (int i = 0; i < dk; ++i) {
        double* Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) Si[j] += kt[i] * vt[j];
      }
    } else if (J->mode == ORACLE_GATED_LINEAR) {
      /* S <- Diag(a) S + k v^T: each row i faded by its channel's gate, then the outer product */
      for (int i = 0; i < dk; ++i) {
        const double ai = J->alpha_per_channel ? J->alpha[((size_t)t * H + h) * dk + i]
                                               : J->alpha[(size_t)t * H + h];
        double* Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) Si[j] = ai * Si[j] + kt[i] * vt[j];
      }
    } else {
      const double bt = J->beta[(size_t)t * H + h];
      /* 1. fade every row i of S by its channel's gate */
      if (J->alpha_per_channel) {
        const double* at = J->alpha + ((size_t)t * H + h) * dk;
        for (int i = 0; i < dk; ++i) {
          double* Si = S + (size_t)i * dv;
          for (int j = 0; j < dv; ++j) Si[j] *= at[i];
        }
      } else {
        const double at = J->alpha[(size_t)t * H + h];
        for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] *= at;
      }
      /* 2. read the faded state at the key: v_hat = S^T k */
      for (int j = 0; j < dv; ++j) vhat[j] = 0.0;
      for (int i = 0; i < dk; ++i) {
        const double* Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) vhat[j] += Si[j] * kt[i];
      }
      /* 3. write the correction: S <- S + beta k (v - v_hat)^T */
      for (int j = 0; j < dv; ++j) vhat[j] = bt * (vt[j] - vhat[j]);
      for (int i = 0; i < dk; ++i) {
        double* Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) Si[j] += kt[i] * vhat[j];
      }
    }
    /* 4. read-out of the updated state: o = S^T q */
    for (int j = 0; j < dv; ++j) ot[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
      const double* Si = S + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) ot[j] += Si[j] * qt[i];
    }
  }
  if (J->S_final) memcpy(J->S_final + sidx, S, sizeof(double) * (size_t)dk * dv);
}

static void* worker_main(void* arg) {
  const oracle_worker* w = (const oracle_worker*)arg;
  const oracle_job* J = w->job;
  double* S = (double*)malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double* vhat = (double*)malloc(sizeof(double) * (size_t)J->dv);
  if (!S || !vhat) {
    free(S);
    free(vhat);
    return (void*)1;
  }
  const int total = J->pairs ? J->n_pairs : J->n_seqs * J->H;
  for (int p = w->tid; p < total; p += J->n_threads) {
    int n, h;
    if (J->pairs) {
      n = J->pairs[2 * p];
      h = J->pairs[2 * p + 1];
    } else {
      n = p / J->H;
      h = p % J->H;
    }
    run_pair(J, n, h, S, vhat);
  }
  free(S);
  free(vhat);
  return NULL;
}

/*
 * Run the recurrence.  mode 0: gated delta rule (alpha and beta required); mode 1: plain linear
 * attention (alpha and beta ignored); mode 2: gated linear attention (alpha required, beta
 * ignored).  S0 may be NULL (zeros), S_final may be NULL.  pairs (if
 * not NULL) restricts the work to n_pairs (seq, head) pairs; outputs of other pairs are left
 * untouched.  Returns 0 on success, -1 on a bad argument, -2 if a thread could not be run.
 */
int gdr_oracle_run(int mode, int n_seqs, int H, int dk, int dv, const int64_t* cu_seqlens,
                   const double* q, const double* k, const double* v, const double* alpha,
                   int alpha_per_channel, const double* beta, const double* S0, double* out,
                   double* S_final, const int32_t* pairs, int n_pairs, int n_threads) {
  if (n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens || !out) return -1;
  if (mode != ORACLE_GATED_DELTA && mode != ORACLE_LINEAR && mode != ORACLE_GATED_LINEAR) return -1;
  if (mode == ORACLE_GATED_DELTA && (!alpha || !beta)) return -1;
  if (mode == ORACLE_GATED_LINEAR && !alpha) return -1;
  for (int n = 0; n < n_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  if (n_threads < 1) n_threads = 1;
  const int total = pairs ? n_pairs : n_seqs * H;
  if (n_threads > total) n_threads = total > 0 ? total : 1;

  oracle_job J = {mode, n_seqs, H, dk, dv, cu_seqlens, q, k, v, alpha, beta, S0,
                  alpha_per_channel, out, S_final, pairs, n_pairs, n_threads};
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  oracle_worker* ws = (oracle_worker*)malloc(sizeof(oracle_worker) * (size_t)n_threads);
  if (!th || !ws) {
    free(th);
    free(ws);
    return -2;
  }
  int rc = 0, started = 0;
  for (int i = 0; i < n_threads; ++i) {
    ws[i].job = &J;
    ws[i].tid = i;
    if (pthread_create(&th[i], NULL, worker_main, &ws[i]) != 0) {
      rc = -2;
      break;
    }
    ++started;
  }
  for (int i = 0; i < started; ++i) {
    void* r = NULL;
    pthread_join(th[i], &r);
    if (r) rc = -2;
  }
  free(th);
  free(ws);
  return rc;
}
