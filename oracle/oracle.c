/*
 * ORACLE -- test infrastructure, not part of the product.
 *
 * A plain, slow, float64 CPU implementation of one data-parallel training
 * step, written from its definition.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it; the product library
 * never calls it and shares no code with it.
 *
 * What it computes (one step over a flat parameter space of psi elements,
 * n data-parallel replicas, a accumulation micro-steps):
 *
 *   G[i]   = sum over ranks r and micro-steps k of g_{r,k}[i]
 *            -- each rank sums its a micro-step gradients, an all-reduce
 *               sums the ranks ("Distributed Training: Split along the Four
 *               Axes", data-parallelism paragraphs on averaging and
 *               accumulation, B_global = b x n x a);
 *   gbar   = G / (n * S)
 *            -- the average over the n replicas, unscaled by the loss
 *               scale S (same page: gbar = (sum_r g_r) / n);
 *   found  = some input is inf/NaN, or fl32(G) or fl32(gbar) is not finite;
 *            when found, nothing is updated and the step count stays;
 *   Adam   -- standard Adam with bias correction, epsilon added to the
 *             square root, no weight decay (Kingma & Ba 2015; the page only
 *             names Adam's first and second moments, memory-budget
 *             paragraph), t counted from 1 on the first applied step:
 *               m'  = b1 m + (1-b1) gbar ;  v' = b2 v + (1-b2) gbar^2
 *               mh  = m' / (1 - b1^t)    ;  vh = v' / (1 - b2^t)
 *               th' = th - lr mh / (sqrt(vh) + eps)
 *   stores -- fp32 (round to nearest even) for master / m / v, and the bf16
 *             image (round to nearest even) of the fp32 master in every
 *             one of the n replicas (the all-gather of the ZeRO pages:
 *             "ZeRO-1 shards optimizer state ... parameters are aggregated
 *             on demand").
 *
 * Sharding changes only where state lives, not what is computed ("sharding
 * changes the storage layout and communication pattern, not the update
 * semantics", ZeRO/FSDP paragraph).  Stage 1-3: element i of segment
 * (global_off, len, owner, local_off) keeps its master/m/v in owner's shard
 * arrays at local_off + (i - global_off).  Stage 0 (plain data parallelism):
 * every rank keeps full-length master/m/v arrays and updates all of them.
 *
 * All arithmetic is float64 with the user's fp32 constants widened exactly;
 * the sum of at most 64 bf16 values is exact in float64 unless their
 * exponents span more than ~45 binades.  Compiled with -ffp-contract=off so
 * every operation is rounded on its own, on every host.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int64_t psi;
  int32_t n, a, stage, nseg;
  const int64_t* seg;              /* nseg rows of {global_off, len, owner, local_off} */
  const uint16_t* const* grads;    /* n*a arrays of psi bf16 bit patterns, index r*a + k */
  float* const* master;            /* n arrays (shards, or full length for stage 0) */
  float* const* m;
  float* const* v;
  uint16_t* const* replicas;       /* n arrays of psi bf16, or NULL */
  double* gbar;                    /* optional psi doubles: the exact averaged gradient */
  float lr, beta1, beta2, eps, loss_scale;
  int32_t t;                       /* in: applied steps so far; out: after this step */
  int32_t found;                   /* out: 1 if the step was skipped */
  int64_t nonfinite;               /* out: elements whose reduced gradient is not finite */
  int32_t nthreads;
  int32_t pad;
} oracle_problem_t;

/* ---- value conversions -------------------------------------------------- */

double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Nearest bf16 value to an fp32 value, ties to even: keep 8 significant
 * bits inside binary32's exponent range. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return (uint16_t)0x7FC0u;
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  double x = fabs((double)f);
  if (x == 0.0) return sign;
  if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
  int e;
  (void)frexp(x, &e);                 /* x = fr * 2^e, fr in [0.5, 1) */
  int q = e - 8;                      /* weight of the 8th significant bit */
  if (q < -133) q = -133;             /* bf16 subnormal spacing */
  double y = ldexp(nearbyint(ldexp(x, -q)), q);
  if (y > 0x1.FEp127) return (uint16_t)(sign | 0x7F80u);
  float g = (float)y;
  uint32_t w;
  memcpy(&w, &g, 4);
  return (uint16_t)(sign | (uint16_t)((w >> 16) & 0x7FFFu));
}

/* ---- work split ----------------------------------------------------------- */

typedef struct {
  oracle_problem_t* p;
  int64_t lo, hi;          /* global index range of this worker */
  int pass;                /* 1 = reduce, 2 = update */
  double* gbar;
  int32_t t_new;
  int found;
  int64_t count;
} work_t;

static void reduce_range(work_t* w) {
  oracle_problem_t* p = w->p;
  const int na = p->n * p->a;
  const double nS = (double)p->n * (double)p->loss_scale;
  for (int64_t i = w->lo; i < w->hi; ++i) {
    double G = 0.0;
    int bad = 0;
    for (int q = 0; q < na; ++q) {
      double x = oracle_bf16_to_double(p->grads[q][i]);
      if (!isfinite(x)) bad = 1;
      G += x;
    }
    double gb = G / nS;
    if (!bad) {
      float G32 = (float)G, gb32 = (float)gb;
      if (!isfinite(G32) || !isfinite(gb32)) bad = 1;
    }
    if (bad) {
      w->found = 1;
      w->count += 1;
    }
    w->gbar[i] = gb;
  }
}

static void adam_one(double g, float* th, float* mm, float* vv, double lr, double b1, double b2, double eps,
                     double bc1, double bc2) {
  double m1 = b1 * (double)*mm + (1.0 - b1) * g;
  double v1 = b2 * (double)*vv + (1.0 - b2) * g * g;
  double mh = m1 / bc1;
  double vh = v1 / bc2;
  double t1 = (double)*th - lr * mh / (sqrt(vh) + eps);
  *mm = (float)m1;
  *vv = (float)v1;
  *th = (float)t1;
}

static void update_range(work_t* w) {
  oracle_problem_t* p = w->p;
  const double lr = p->lr, b1 = p->beta1, b2 = p->beta2, eps = p->eps;
  const double bc1 = 1.0 - pow(b1, (double)w->t_new);
  const double bc2 = 1.0 - pow(b2, (double)w->t_new);
  for (int s = 0; s < p->nseg; ++s) {
    const int64_t* row = p->seg + 4 * s;
    int64_t g0 = row[0], len = row[1], owner = row[2], l0 = row[3];
    int64_t lo = g0 > w->lo ? g0 : w->lo;
    int64_t hi = (g0 + len) < w->hi ? (g0 + len) : w->hi;
    for (int64_t i = lo; i < hi; ++i) {
      double g = w->gbar[i];
      if (p->stage == 0) {
        for (int r = 0; r < p->n; ++r) {
          adam_one(g, &p->master[r][i], &p->m[r][i], &p->v[r][i], lr, b1, b2, eps, bc1, bc2);
          if (p->replicas) p->replicas[r][i] = oracle_f32_to_bf16(p->master[r][i]);
        }
      } else {
        int64_t j = l0 + (i - g0);
        adam_one(g, &p->master[owner][j], &p->m[owner][j], &p->v[owner][j], lr, b1, b2, eps, bc1, bc2);
        if (p->replicas) {
          uint16_t b = oracle_f32_to_bf16(p->master[owner][j]);
          for (int r = 0; r < p->n; ++r) p->replicas[r][i] = b;
        }
      }
    }
  }
}

static void* worker(void* arg) {
  work_t* w = (work_t*)arg;
  if (w->pass == 1)
    reduce_range(w);
  else
    update_range(w);
  return 0;
}

static void run_pass(oracle_problem_t* p, int pass, double* gbar, int32_t t_new, int* found, int64_t* count) {
  int nt = p->nthreads < 1 ? 1 : (p->nthreads > 256 ? 256 : p->nthreads);
  if (p->psi < 4096) nt = 1;
  work_t ws[256];
  pthread_t th[256];
  int64_t chunk = (p->psi + nt - 1) / nt;
  if (chunk < 1) chunk = 1;
  int used = 0;
  for (int t = 0; t < nt; ++t) {
    int64_t lo = (int64_t)t * chunk, hi = lo + chunk;
    if (hi > p->psi) hi = p->psi;
    if (lo >= hi && t > 0) break;
    ws[t].p = p;
    ws[t].lo = lo;
    ws[t].hi = hi > lo ? hi : lo;
    ws[t].pass = pass;
    ws[t].gbar = gbar;
    ws[t].t_new = t_new;
    ws[t].found = 0;
    ws[t].count = 0;
    used = t + 1;
  }
  int spawned[256] = {0};
  for (int t = 1; t < used; ++t) spawned[t] = pthread_create(&th[t], 0, worker, &ws[t]) == 0;
  worker(&ws[0]);
  for (int t = 1; t < used; ++t) {
    if (spawned[t])
      pthread_join(th[t], 0);
    else
      worker(&ws[t]);
  }
  for (int t = 0; t < used; ++t) {
    *found |= ws[t].found;
    *count += ws[t].count;
  }
}

/* Reduce only: fills p->gbar (required), p->found and p->nonfinite. */
int oracle_reduce(oracle_problem_t* p) {
  if (!p || p->n < 1 || p->a < 1 || p->psi < 0 || (p->psi > 0 && !p->gbar)) return 1;
  int found = 0;
  int64_t count = 0;
  run_pass(p, 1, p->gbar, 0, &found, &count);
  p->found = found;
  p->nonfinite = count;
  return 0;
}

/* One full step, in place on master/m/v/replicas and t. */
int oracle_step(oracle_problem_t* p) {
  if (!p || p->n < 1 || p->a < 1 || p->psi < 0 || p->stage < 0 || p->stage > 3) return 1;
  double* gb = p->gbar;
  int owned = 0;
  if (!gb && p->psi > 0) {
    gb = (double*)malloc(sizeof(double) * (size_t)p->psi);
    if (!gb) return 2;
    owned = 1;
  }
  int found = 0;
  int64_t count = 0;
  run_pass(p, 1, gb, 0, &found, &count);
  p->found = found;
  p->nonfinite = count;
  if (!found) {
    int32_t t_new = p->t + 1;
    int f2 = 0;
    int64_t c2 = 0;
    run_pass(p, 2, gb, t_new, &f2, &c2);
    p->t = t_new;
  }
  if (owned) free(gb);
  return 0;
}
