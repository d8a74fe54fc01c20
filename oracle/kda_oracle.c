/*
 * kda_oracle.c -- fp64 CPU oracle for KDA (Kimi Delta Attention).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path and the CUDA path never calls it.
 *
 * What it computes (plain definition, token by token, in fp64):
 *   For each logical sequence n (packed tokens cu[n] .. cu[n+1]-1) and value
 *   head j, with query/key head h = j / (HV/H) (contiguous groups of value heads
 *   share one q/k head):
 *     S = h0[n,j]            (K x V; zero when no initial state is given)
 *     for each token t:
 *       a     = 2^g[t,j,:]                      per-channel decay (log2 gate)
 *       P     = diag(a) S                        decay first
 *       e     = P^T k[t,h]                       prediction from the decayed state
 *       delta = beta[t,j] (v[t,j] - e)           delta-rule correction
 *       S     = P + k[t,h] delta^T               rank-1 write
 *       o[t,j]= S^T (q[t,h] / sqrt(K))           read-out from the updated state
 *     hT[n,j] = S
 * The per-token log2 gate, the fixed 1/sqrt(K) query scale, the fp32 state
 * with one entry per logical sequence and the packed offsets with repeated
 * offsets as empty slots are the contract of the ``recurrent_kda`` entry
 * point ("kda in torchtitan (training)", pytorch/torchtitan PR #4164, agent
 * note).  An empty slot runs zero tokens, so hT = h0 and dh0 = dhT.
 *
 * Backward (derived by hand from the step above, walked in reverse):
 *   dS += q~ dO^T ;  dq~ = S_t dO                       (o = S_t^T q~)
 *   dk += dS delta ; ddelta = dS^T k ; dP = dS          (S_t = P + k delta^T)
 *   dbeta = ddelta . (v - e) ; dv = beta ddelta ; de = -beta ddelta
 *   dP += k de^T ; dk += P de                           (e = P^T k)
 *   dg = ln2 * a * rowsum(dP .* S_{t-1}) ; dS = diag(a) dP
 *   dh0 = dS after the first token.  dq, dk are summed over the value heads
 *   of a group; dq carries the 1/sqrt(K) factor.
 * States are checkpointed every SEG tokens and recomputed inside a segment.
 *
 * Layout (row-major, packed token axis of T rows):
 *   q,k,dq,dk [T][H][K]   v,o,dO,dv [T][HV][V]   g,dg [T][HV][K]
 *   beta,dbeta [T][HV]    h0,hT,dhT,dh0 [N][HV][K][V]
 * Tokens outside every sequence are neither read nor written.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define SEG 64

typedef struct {
  int64_t T;
  int N, H, HV, K, V;
  const int32_t *cu;
  const double *q, *k, *v, *g, *beta, *h0;
  double *o, *hT;
  const double *dout, *dhT;
  double *dq_part, *dk_part; /* [T][HV][K] per-value-head partials */
  double *dv, *dg, *dbeta, *dh0;
  int backward;
  int next_unit; /* work counter, atomically incremented */
  int status;
} job_t;

static inline const double *row_qk(const job_t *J, const double *base, int64_t t, int h) {
  return base + ((size_t)t * J->H + h) * J->K;
}

/* One token of the recurrence.  S (K x V) is updated in place.  Writes the
 * prediction e[V] and the correction delta[V]. */
static void token_step(int K, int V, double *S, const double *kt, const double *gt, double bt,
                       const double *vt, double *e, double *delta) {
  for (int c = 0; c < K; ++c) {
    double a = exp2(gt[c]);
    double *row = S + (size_t)c * V;
    for (int x = 0; x < V; ++x) row[x] *= a;
  }
  for (int x = 0; x < V; ++x) e[x] = 0.0;
  for (int c = 0; c < K; ++c) {
    const double *row = S + (size_t)c * V;
    for (int x = 0; x < V; ++x) e[x] += row[x] * kt[c];
  }
  for (int x = 0; x < V; ++x) delta[x] = bt * (vt[x] - e[x]);
  for (int c = 0; c < K; ++c) {
    double *row = S + (size_t)c * V;
    for (int x = 0; x < V; ++x) row[x] += kt[c] * delta[x];
  }
}

static void fwd_unit(job_t *J, int n, int j) {
  const int K = J->K, V = J->V, HV = J->HV, r = J->HV / J->H, h = j / r;
  const double scale = 1.0 / sqrt((double)K);
  double *S = calloc((size_t)K * V, sizeof(double));
  double *e = malloc(sizeof(double) * V), *delta = malloc(sizeof(double) * V);
  if (!S || !e || !delta) { J->status = -1; free(S); free(e); free(delta); return; }
  if (J->h0) memcpy(S, J->h0 + ((size_t)n * HV + j) * K * V, sizeof(double) * K * V);
  for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
    const double *kt = row_qk(J, J->k, t, h), *qt = row_qk(J, J->q, t, h);
    const double *gt = J->g + ((size_t)t * HV + j) * K;
    const double *vt = J->v + ((size_t)t * HV + j) * V;
    token_step(K, V, S, kt, gt, J->beta[(size_t)t * HV + j], vt, e, delta);
    double *ot = J->o + ((size_t)t * HV + j) * V;
    for (int x = 0; x < V; ++x) ot[x] = 0.0;
    for (int c = 0; c < K; ++c) {
      const double *row = S + (size_t)c * V;
      const double qc = qt[c] * scale;
      for (int x = 0; x < V; ++x) ot[x] += row[x] * qc;
    }
  }
  if (J->hT) memcpy(J->hT + ((size_t)n * HV + j) * K * V, S, sizeof(double) * K * V);
  free(S); free(e); free(delta);
}

static void bwd_unit(job_t *J, int n, int j) {
  const int K = J->K, V = J->V, HV = J->HV, r = J->HV / J->H, h = j / r;
  const double scale = 1.0 / sqrt((double)K), ln2 = log(2.0);
  const int64_t t0 = J->cu[n], len = J->cu[n + 1] - J->cu[n];
  const size_t KV = (size_t)K * V;
  const int64_t nseg = (len + SEG - 1) / SEG;
  double *ck = malloc(sizeof(double) * KV * (nseg > 0 ? nseg : 1));
  double *St = malloc(sizeof(double) * KV * (SEG + 1));
  double *E = malloc(sizeof(double) * V * SEG), *D = malloc(sizeof(double) * V * SEG);
  double *dS = calloc(KV, sizeof(double)), *dP = malloc(sizeof(double) * KV);
  double *P = malloc(sizeof(double) * KV);
  double *ddel = malloc(sizeof(double) * V), *de = malloc(sizeof(double) * V);
  if (!ck || !St || !E || !D || !dS || !dP || !P || !ddel || !de) {
    J->status = -1;
    goto done;
  }
  /* forward pass, keeping the state at every segment start */
  {
    double *S = St; /* reuse slot 0 as the running state */
    if (J->h0) memcpy(S, J->h0 + ((size_t)n * HV + j) * KV, sizeof(double) * KV);
    else memset(S, 0, sizeof(double) * KV);
    for (int64_t s = 0; s < nseg; ++s) {
      memcpy(ck + (size_t)s * KV, S, sizeof(double) * KV);
      for (int64_t i = 0; i < SEG && s * SEG + i < len; ++i) {
        int64_t t = t0 + s * SEG + i;
        token_step(K, V, S, row_qk(J, J->k, t, h), J->g + ((size_t)t * HV + j) * K,
                   J->beta[(size_t)t * HV + j], J->v + ((size_t)t * HV + j) * V, E, D);
      }
    }
  }
  if (J->dhT) memcpy(dS, J->dhT + ((size_t)n * HV + j) * KV, sizeof(double) * KV);
  for (int64_t s = nseg - 1; s >= 0; --s) {
    const int64_t L = (len - s * SEG) < SEG ? (len - s * SEG) : SEG;
    /* recompute the states of this segment: St[i] = state before token i */
    memcpy(St, ck + (size_t)s * KV, sizeof(double) * KV);
    for (int64_t i = 0; i < L; ++i) {
      int64_t t = t0 + s * SEG + i;
      memcpy(St + (size_t)(i + 1) * KV, St + (size_t)i * KV, sizeof(double) * KV);
      token_step(K, V, St + (size_t)(i + 1) * KV, row_qk(J, J->k, t, h),
                 J->g + ((size_t)t * HV + j) * K, J->beta[(size_t)t * HV + j],
                 J->v + ((size_t)t * HV + j) * V, E + (size_t)i * V, D + (size_t)i * V);
    }
    for (int64_t i = L - 1; i >= 0; --i) {
      const int64_t t = t0 + s * SEG + i;
      const double *Sprev = St + (size_t)i * KV, *Scur = St + (size_t)(i + 1) * KV;
      const double *qt = row_qk(J, J->q, t, h), *kt = row_qk(J, J->k, t, h);
      const double *gt = J->g + ((size_t)t * HV + j) * K;
      const double *vt = J->v + ((size_t)t * HV + j) * V;
      const double *dot = J->dout + ((size_t)t * HV + j) * V;
      const double bt = J->beta[(size_t)t * HV + j];
      const double *e = E + (size_t)i * V, *delta = D + (size_t)i * V;
      double *dqp = J->dq_part + ((size_t)t * HV + j) * K;
      double *dkp = J->dk_part + ((size_t)t * HV + j) * K;
      double *dvt = J->dv + ((size_t)t * HV + j) * V;
      double *dgt = J->dg + ((size_t)t * HV + j) * K;
      /* o_t = S_t^T (q scale) */
      for (int c = 0; c < K; ++c) {
        double acc = 0.0;
        const double *row = Scur + (size_t)c * V;
        double *drow = dS + (size_t)c * V;
        for (int x = 0; x < V; ++x) {
          acc += row[x] * dot[x];
          drow[x] += qt[c] * scale * dot[x];
        }
        dqp[c] = acc * scale;
      }
      /* S_t = P + k delta^T */
      for (int x = 0; x < V; ++x) ddel[x] = 0.0;
      for (int c = 0; c < K; ++c) {
        double acc = 0.0;
        const double *drow = dS + (size_t)c * V;
        for (int x = 0; x < V; ++x) {
          acc += drow[x] * delta[x];
          ddel[x] += drow[x] * kt[c];
        }
        dkp[c] = acc;
      }
      /* delta = beta (v - e) */
      double db = 0.0;
      for (int x = 0; x < V; ++x) {
        db += ddel[x] * (vt[x] - e[x]);
        dvt[x] = bt * ddel[x];
        de[x] = -bt * ddel[x];
      }
      J->dbeta[(size_t)t * HV + j] = db;
      /* P = diag(a) Sprev ;  e = P^T k */
      for (int c = 0; c < K; ++c) {
        const double a = exp2(gt[c]);
        const double *srow = Sprev + (size_t)c * V, *dsrow = dS + (size_t)c * V;
        double *prow = P + (size_t)c * V, *dprow = dP + (size_t)c * V;
        double acc = 0.0;
        for (int x = 0; x < V; ++x) {
          prow[x] = a * srow[x];
          dprow[x] = dsrow[x] + kt[c] * de[x];
          acc += prow[x] * de[x];
        }
        dkp[c] += acc;
      }
      /* dg and the gradient into S_{t-1} */
      for (int c = 0; c < K; ++c) {
        const double a = exp2(gt[c]);
        const double *srow = Sprev + (size_t)c * V, *dprow = dP + (size_t)c * V;
        double *dsrow = dS + (size_t)c * V;
        double acc = 0.0;
        for (int x = 0; x < V; ++x) {
          acc += dprow[x] * srow[x];
          dsrow[x] = a * dprow[x];
        }
        dgt[c] = ln2 * a * acc;
      }
    }
  }
  if (J->dh0) memcpy(J->dh0 + ((size_t)n * HV + j) * KV, dS, sizeof(double) * KV);
done:
  free(ck); free(St); free(E); free(D); free(dS); free(dP); free(P); free(ddel); free(de);
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int units = J->N * J->HV;
  for (;;) {
    int u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
    if (u >= units) break;
    /* longest-first would balance better; plain order keeps it obvious */
    int n = u / J->HV, j = u % J->HV;
    if (J->backward) bwd_unit(J, n, j);
    else fwd_unit(J, n, j);
  }
  return NULL;
}

static int run(job_t *J, int nthreads) {
  if (J->H <= 0 || J->HV % J->H != 0 || J->K <= 0 || J->V <= 0 || J->N < 0) return -2;
  for (int n = 0; n < J->N; ++n)
    if (J->cu[n + 1] < J->cu[n] || J->cu[n] < 0 || J->cu[n + 1] > J->T) return -3;
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  const int units = J->N * J->HV;
  if (nthreads > units) nthreads = units > 0 ? units : 1;
  J->next_unit = 0;
  J->status = 0;
  pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
  if (!th) return -1;
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, J) == 0) ++started;
  }
  if (started == 0) worker(J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  return J->status;
}

/* Forward.  hT and h0 may be NULL.  Returns 0 on success. */
int kda_oracle_fwd(int64_t T, int N, int H, int HV, int K, int V, const int32_t *cu,
                   const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const double *h0, double *o, double *hT, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof(J));
  J.T = T; J.N = N; J.H = H; J.HV = HV; J.K = K; J.V = V; J.cu = cu;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0; J.o = o; J.hT = hT;
  return run(&J, nthreads);
}

/* Backward.  h0, dhT, dh0 may be NULL.  dq_part/dk_part are caller scratch of
 * T*HV*K doubles each; dq, dk receive the group sums. */
int kda_oracle_bwd(int64_t T, int N, int H, int HV, int K, int V, const int32_t *cu,
                   const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const double *h0, const double *dout, const double *dhT,
                   double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dh0,
                   double *dq_part, double *dk_part, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof(J));
  J.T = T; J.N = N; J.H = H; J.HV = HV; J.K = K; J.V = V; J.cu = cu;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
  J.dout = dout; J.dhT = dhT; J.dv = dv; J.dg = dg; J.dbeta = dbeta; J.dh0 = dh0;
  J.dq_part = dq_part; J.dk_part = dk_part;
  J.backward = 1;
  int st = run(&J, nthreads);
  if (st != 0) return st;
  /* group sums of the per-value-head query/key gradients */
  const int r = HV / H;
  for (int n = 0; n < N; ++n) {
    for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
      for (int h = 0; h < H; ++h) {
        double *dqt = dq + ((size_t)t * H + h) * K, *dkt = dk + ((size_t)t * H + h) * K;
        for (int c = 0; c < K; ++c) { dqt[c] = 0.0; dkt[c] = 0.0; }
        for (int jj = 0; jj < r; ++jj) {
          const int j = h * r + jj;
          const double *a = dq_part + ((size_t)t * HV + j) * K;
          const double *b = dk_part + ((size_t)t * HV + j) * K;
          for (int c = 0; c < K; ++c) { dqt[c] += a[c]; dkt[c] += b[c]; }
        }
      }
    }
  }
  return 0;
}
