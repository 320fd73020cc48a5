/*
 * ssd_oracle.c -- plain, sequential fp64 CPU oracle of the Mamba2 SSD scan
 * and of its reverse-mode gradient.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark load this file. The CUDA library shares no
 * code, header, table or helper with it, and it includes nothing from there.
 *
 * What it computes ("Deterministic bwd kernel for mamba2", Mamba PR #827: the
 * page names the forward/backward pair of the mamba2 SSD; the recurrence
 * itself is the one the library is specified by):
 *
 *   for every batch row b and head h (group g = h / (H/G)), token by token:
 *     state_{t-1} := init[seq(t)] (or 0) when t starts a sequence
 *     state_t     = exp(dt_t * A_h) * state_{t-1} + dt_t * x_t (outer) B_t
 *     y_t         = state_t . C_t + D_h * x_t
 *
 * with state_t a (P x N) matrix stored p-major ([p][n]), x_t a P-vector and
 * B_t, C_t the N-vectors of the head's group.  A token t starts a sequence
 * when t == 0 or seq_idx[b][t] != seq_idx[b][t-1].
 *
 * The backward is the reverse sweep of that recurrence (one adjoint matrix
 * dState per task, walked from the last token to the first), written out by
 * hand from the chain rule:
 *   dC_t    += state_t^T g_t                   dState += g_t (outer) C_t
 *   dD      += g_t . x_t                        dx_t    = D g_t + dt_t dState B_t
 *   dB_t    += dt_t dState^T x_t                dalpha  = <state_{t-1}, dState>
 *   ddt_t    = A alpha_t dalpha + x_t^T dState B_t
 *   dA      += dt_t alpha_t dalpha              dState  = alpha_t dState
 *   at a sequence start: dinit[seq] += dState; dState = 0
 * The states state_{t-1} are recomputed from checkpoints taken every
 * ORACLE_CKPT tokens (a spacing unrelated to any chunk size).
 *
 * Work is split over (b, h) tasks on nthreads POSIX threads.  The per-head
 * dB/dC contributions are summed into the group arrays in ascending task
 * order after each wave, so the oracle's own result does not depend on the
 * thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_CKPT 256

typedef struct {
  int64_t b, T, H, P, G, N;
  int64_t nseq;
  const double *x, *dt, *A, *B, *C, *D, *init, *dout;
  const int32_t *seq_idx;
  int64_t chunk;        /* > 0: also record the state entering each chunk */
  double *y, *chunk_states;
  /* backward outputs */
  double *dx, *ddt, *dA, *dD, *dinit;
} problem;

typedef struct {
  const problem *pr;
  int64_t task;        /* b * H + h */
  double *dBh, *dCh;   /* (T, N) per-head contributions (backward only) */
  double *scratch;     /* checkpoints + segment states */
  int is_bwd;
  int status;
} job;

static int starts_seq(const problem *pr, int64_t bi, int64_t t) {
  if (t == 0) return 1;
  if (!pr->seq_idx) return 0;
  return pr->seq_idx[bi * pr->T + t] != pr->seq_idx[bi * pr->T + t - 1];
}

static int64_t seq_of(const problem *pr, int64_t bi, int64_t t) {
  return pr->seq_idx ? (int64_t)pr->seq_idx[bi * pr->T + t] : bi;
}

/* Reset the running state at a sequence start: initial state or zero. */
static void reset_state(const problem *pr, int64_t bi, int64_t h, int64_t t,
                        double *st) {
  const int64_t PN = pr->P * pr->N;
  if (pr->init) {
    const double *src = pr->init + (seq_of(pr, bi, t) * pr->H + h) * PN;
    memcpy(st, src, (size_t)PN * sizeof(double));
  } else {
    memset(st, 0, (size_t)PN * sizeof(double));
  }
}

/* One step of the recurrence: st <- alpha * st + dt * x (outer) B. */
static void step_state(const problem *pr, int64_t bi, int64_t h, int64_t t,
                       double *st) {
  const int64_t H = pr->H, P = pr->P, N = pr->N, G = pr->G;
  const int64_t g = h / (H / G);
  const double dt = pr->dt[(bi * pr->T + t) * H + h];
  const double alpha = exp(dt * pr->A[h]);
  const double *x = pr->x + ((bi * pr->T + t) * H + h) * P;
  const double *Bv = pr->B + ((bi * pr->T + t) * G + g) * N;
  for (int64_t p = 0; p < P; ++p)
    for (int64_t n = 0; n < N; ++n)
      st[p * N + n] = alpha * st[p * N + n] + dt * x[p] * Bv[n];
}

static void fwd_task(job *jb) {
  const problem *pr = jb->pr;
  const int64_t H = pr->H, P = pr->P, N = pr->N, G = pr->G, T = pr->T;
  const int64_t bi = jb->task / H, h = jb->task % H, g = h / (H / G);
  double *st = jb->scratch;
  for (int64_t t = 0; t < T; ++t) {
    if (starts_seq(pr, bi, t)) reset_state(pr, bi, h, t, st);
    if (pr->chunk > 0 && pr->chunk_states && t % pr->chunk == 0) {
      const int64_t nc = (T + pr->chunk - 1) / pr->chunk;
      double *dst = pr->chunk_states + ((bi * nc + t / pr->chunk) * H + h) * P * N;
      memcpy(dst, st, (size_t)(P * N) * sizeof(double));
    }
    step_state(pr, bi, h, t, st);
    const double *Cv = pr->C + ((bi * T + t) * G + g) * N;
    const double *x = pr->x + ((bi * T + t) * H + h) * P;
    double *y = pr->y + ((bi * T + t) * H + h) * P;
    for (int64_t p = 0; p < P; ++p) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += st[p * N + n] * Cv[n];
      y[p] = acc + pr->D[h] * x[p];
    }
  }
}

static void bwd_task(job *jb) {
  const problem *pr = jb->pr;
  const int64_t H = pr->H, P = pr->P, N = pr->N, G = pr->G, T = pr->T;
  const int64_t PN = P * N;
  const int64_t bi = jb->task / H, h = jb->task % H, g = h / (H / G);
  const int64_t nseg = (T + ORACLE_CKPT - 1) / ORACLE_CKPT;
  double *ckpt = jb->scratch;                 /* nseg * PN: state before token k*CKPT (after reset) */
  double *prev = ckpt + nseg * PN;            /* CKPT * PN: state_{t-1} of each token of a segment */
  double *dS = prev + ORACLE_CKPT * PN;       /* PN adjoint */
  double *cur = dS + PN;                      /* PN: state_t */
  const double Ah = pr->A[h], Dh = pr->D[h];

  /* forward sweep, keeping checkpoints */
  memset(cur, 0, (size_t)PN * sizeof(double));
  for (int64_t t = 0; t < T; ++t) {
    if (starts_seq(pr, bi, t)) reset_state(pr, bi, h, t, cur);
    if (t % ORACLE_CKPT == 0) memcpy(ckpt + (t / ORACLE_CKPT) * PN, cur, (size_t)PN * sizeof(double));
    step_state(pr, bi, h, t, cur);
  }

  memset(dS, 0, (size_t)PN * sizeof(double));
  double dA_acc = 0.0, dD_acc = 0.0;
  for (int64_t k = nseg - 1; k >= 0; --k) {
    const int64_t t0 = k * ORACLE_CKPT;
    const int64_t t1 = (t0 + ORACLE_CKPT < T) ? t0 + ORACLE_CKPT : T;
    /* recompute state_{t-1} (as seen by token t, i.e. after any reset) */
    memcpy(cur, ckpt + k * PN, (size_t)PN * sizeof(double));
    for (int64_t t = t0; t < t1; ++t) {
      if (t > t0 && starts_seq(pr, bi, t)) reset_state(pr, bi, h, t, cur);
      memcpy(prev + (t - t0) * PN, cur, (size_t)PN * sizeof(double));
      step_state(pr, bi, h, t, cur);
    }
    for (int64_t t = t1 - 1; t >= t0; --t) {
      const double *sp = prev + (t - t0) * PN;     /* state_{t-1} */
      const double dt = pr->dt[(bi * T + t) * H + h];
      const double alpha = exp(dt * Ah);
      const double *x = pr->x + ((bi * T + t) * H + h) * P;
      const double *gv = pr->dout + ((bi * T + t) * H + h) * P;
      const double *Bv = pr->B + ((bi * T + t) * G + g) * N;
      const double *Cv = pr->C + ((bi * T + t) * G + g) * N;
      double *dCt = jb->dCh + t * N;
      double *dBt = jb->dBh + t * N;
      double *dxt = pr->dx + ((bi * T + t) * H + h) * P;

      /* y_t = state_t . C_t + D x_t ; state_t = alpha state_{t-1} + dt x B^T */
      for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t p = 0; p < P; ++p) {
          const double st_pn = alpha * sp[p * N + n] + dt * x[p] * Bv[n];
          acc += st_pn * gv[p];
        }
        dCt[n] = acc;
      }
      for (int64_t p = 0; p < P; ++p) {
        dD_acc += gv[p] * x[p];
        for (int64_t n = 0; n < N; ++n) dS[p * N + n] += gv[p] * Cv[n];
      }
      double dalpha = 0.0, xdSB = 0.0;
      for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          acc += dS[p * N + n] * Bv[n];
          dalpha += sp[p * N + n] * dS[p * N + n];
        }
        dxt[p] = Dh * gv[p] + dt * acc;
        xdSB += x[p] * acc;
      }
      for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t p = 0; p < P; ++p) acc += dS[p * N + n] * x[p];
        dBt[n] = dt * acc;
      }
      pr->ddt[(bi * T + t) * H + h] = Ah * alpha * dalpha + xdSB;
      dA_acc += dt * alpha * dalpha;
      for (int64_t e = 0; e < PN; ++e) dS[e] *= alpha;
      if (starts_seq(pr, bi, t)) {
        if (pr->init && pr->dinit) {
          double *di = pr->dinit + (seq_of(pr, bi, t) * H + h) * PN;
          for (int64_t e = 0; e < PN; ++e) di[e] += dS[e];
        }
        memset(dS, 0, (size_t)PN * sizeof(double));
      }
    }
  }
  jb->dBh[T * N] = dA_acc;   /* two trailing slots carry the per-task scalars */
  jb->dBh[T * N + 1] = dD_acc;
}

static void *run_job(void *arg) {
  job *jb = (job *)arg;
  if (jb->is_bwd) bwd_task(jb);
  else fwd_task(jb);
  return NULL;
}

static int check_dims(const problem *pr) {
  if (pr->b <= 0 || pr->T <= 0 || pr->H <= 0 || pr->P <= 0 || pr->G <= 0 || pr->N <= 0) return 1;
  if (pr->H % pr->G != 0) return 2;
  if (pr->seq_idx) {
    for (int64_t bi = 0; bi < pr->b; ++bi)
      for (int64_t t = 0; t < pr->T; ++t) {
        int32_t s = pr->seq_idx[bi * pr->T + t];
        if (s < 0 || s >= pr->nseq) return 3;
      }
  } else if (pr->init && pr->nseq != pr->b) {
    return 4;
  }
  return 0;
}

/* Runs all (b, h) tasks in waves of nthreads; for the backward, folds the
   per-head dB/dC/dA/dD of each wave into the outputs in task order. */
static int run_all(problem *pr, int is_bwd, int nthreads, double *dB, double *dC) {
  const int64_t ntask = pr->b * pr->H;
  const int64_t PN = pr->P * pr->N;
  const int64_t nseg = (pr->T + ORACLE_CKPT - 1) / ORACLE_CKPT;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > ntask) nthreads = (int)ntask;
  const int64_t scratch_len = is_bwd ? (nseg + ORACLE_CKPT + 2) * PN : PN;
  const int64_t dbc_len = is_bwd ? pr->T * pr->N + 2 : 0;
  job *jobs = (job *)calloc((size_t)nthreads, sizeof(job));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  double *mem = (double *)malloc((size_t)nthreads * (size_t)(scratch_len + 2 * dbc_len) * sizeof(double));
  if (!jobs || !th || !mem) { free(jobs); free(th); free(mem); return 10; }
  for (int i = 0; i < nthreads; ++i) {
    double *base = mem + (size_t)i * (size_t)(scratch_len + 2 * dbc_len);
    jobs[i].pr = pr;
    jobs[i].scratch = base;
    jobs[i].dBh = base + scratch_len;
    jobs[i].dCh = base + scratch_len + dbc_len;
    jobs[i].is_bwd = is_bwd;
  }
  for (int64_t first = 0; first < ntask; first += nthreads) {
    int nw = (int)((ntask - first < nthreads) ? ntask - first : nthreads);
    for (int i = 0; i < nw; ++i) {
      jobs[i].task = first + i;
      if (nw == 1) run_job(&jobs[i]);
      else pthread_create(&th[i], NULL, run_job, &jobs[i]);
    }
    if (nw > 1)
      for (int i = 0; i < nw; ++i) pthread_join(th[i], NULL);
    if (is_bwd) {
      for (int i = 0; i < nw; ++i) {   /* ascending task order */
        const int64_t task = first + i, bi = task / pr->H, h = task % pr->H;
        const int64_t g = h / (pr->H / pr->G);
        for (int64_t t = 0; t < pr->T; ++t)
          for (int64_t n = 0; n < pr->N; ++n) {
            const int64_t o = ((bi * pr->T + t) * pr->G + g) * pr->N + n;
            dB[o] += jobs[i].dBh[t * pr->N + n];
            dC[o] += jobs[i].dCh[t * pr->N + n];
          }
        pr->dA[h] += jobs[i].dBh[pr->T * pr->N];
        pr->dD[h] += jobs[i].dBh[pr->T * pr->N + 1];
      }
    }
  }
  free(jobs); free(th); free(mem);
  return 0;
}

/* Forward.  y: (b,T,H,P).  chunk_states (nullable, needs chunk > 0):
   (b, ceil(T/chunk), H, P, N), the state entering each chunk, i.e. the
   running state after token c*chunk-1, or init/zero when token c*chunk starts
   a sequence.  Returns 0 on success. */
int ssd_oracle_fwd(int64_t b, int64_t T, int64_t H, int64_t P, int64_t G, int64_t N,
                   int64_t nseq, const double *x, const double *dt, const double *A,
                   const double *B, const double *C, const double *D,
                   const int32_t *seq_idx, const double *init, int64_t chunk,
                   double *y, double *chunk_states, int nthreads) {
  problem pr;
  memset(&pr, 0, sizeof(pr));
  pr.b = b; pr.T = T; pr.H = H; pr.P = P; pr.G = G; pr.N = N; pr.nseq = nseq;
  pr.x = x; pr.dt = dt; pr.A = A; pr.B = B; pr.C = C; pr.D = D;
  pr.seq_idx = seq_idx; pr.init = init; pr.chunk = chunk;
  pr.y = y; pr.chunk_states = chunk_states;
  int rc = check_dims(&pr);
  if (rc) return rc;
  return run_all(&pr, 0, nthreads, NULL, NULL);
}

/* Backward of L = sum(y * dout).  Outputs are overwritten:
   dx (b,T,H,P), ddt (b,T,H), dA (H), dB, dC (b,T,G,N), dD (H),
   dinit (nseq,H,P,N; nullable, only with init).  Returns 0 on success. */
int ssd_oracle_bwd(int64_t b, int64_t T, int64_t H, int64_t P, int64_t G, int64_t N,
                   int64_t nseq, const double *x, const double *dt, const double *A,
                   const double *B, const double *C, const double *D,
                   const int32_t *seq_idx, const double *init, const double *dout,
                   double *dx, double *ddt, double *dA, double *dB, double *dC,
                   double *dD, double *dinit, int nthreads) {
  problem pr;
  memset(&pr, 0, sizeof(pr));
  pr.b = b; pr.T = T; pr.H = H; pr.P = P; pr.G = G; pr.N = N; pr.nseq = nseq;
  pr.x = x; pr.dt = dt; pr.A = A; pr.B = B; pr.C = C; pr.D = D;
  pr.seq_idx = seq_idx; pr.init = init; pr.dout = dout;
  pr.dx = dx; pr.ddt = ddt; pr.dA = dA; pr.dD = dD; pr.dinit = dinit;
  int rc = check_dims(&pr);
  if (rc) return rc;
  memset(dA, 0, (size_t)H * sizeof(double));
  memset(dD, 0, (size_t)H * sizeof(double));
  memset(dB, 0, (size_t)(b * T * G * N) * sizeof(double));
  memset(dC, 0, (size_t)(b * T * G * N) * sizeof(double));
  if (init && dinit) memset(dinit, 0, (size_t)(nseq * H * P * N) * sizeof(double));
  return run_all(&pr, 1, nthreads, dB, dC);
}
