/*
 * Seeded synthetic inputs for the data-parallel step: counter-based random
 * streams and the value distributions of the workloads.
 *
 * This file holds no arithmetic of the step itself (no reduction, no
 * optimizer, no rounding of results).  It turns (seed, role, rank,
 * micro-step, element index) into a value, so that any element of any
 * buffer can be regenerated on its own, in any order, on any thread.
 *
 * Generator: Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11), the 4-word / 64-bit / 10-round
 * member of the family, with the published multipliers and Weyl key
 * increments.  Normals: the Box-Muller transform in double precision
 * (Box & Muller 1958).  bf16 inputs are the round-to-nearest-even image of
 * the double sample (8 significant bits, binary32 exponent range).
 *
 * Stream layout for one buffer (key = {seed, role<<48 | rank<<24 | micro}):
 *   block b = element / 2 uses counter {b, 0, 0, 0};
 *   words 0,1 -> one Box-Muller pair (cos -> even element, sin -> odd);
 *   words 2,3 -> the heavy-tail draw of the even / odd element.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2E7470EE14C6C93ULL
#define PHILOX_M1 0xCA5A826395121157ULL
#define PHILOX_W0 0x9E3779B97F4A7C15ULL
#define PHILOX_W1 0xBB67AE8584CAA73BULL

static inline void mulhilo64(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
  unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
  *hi = (uint64_t)(p >> 64);
  *lo = (uint64_t)p;
}

void synth_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2], uint64_t out[4]) {
  uint64_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint64_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t hi0, lo0, hi1, lo1;
    mulhilo64(PHILOX_M0, c0, &hi0, &lo0);
    mulhilo64(PHILOX_M1, c2, &hi1, &lo1);
    uint64_t n0 = hi1 ^ c1 ^ k0;
    uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

static inline void stream_key(uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, uint64_t key[2]) {
  key[0] = seed;
  key[1] = ((uint64_t)(role & 0xFFFFu) << 48) | ((uint64_t)(rank & 0xFFFFFFu) << 24) | (uint64_t)(micro & 0xFFFFFFu);
}

/* Uniform in the open interval (0, 1) from the top 53 bits of a word. */
static inline double u01_open(uint64_t w) { return ((double)(w >> 11) + 0.5) * 0x1p-53; }

/* Standard normal sample of element i of the stream, plus its heavy-tail
 * uniform in *tail_u. */
static inline double normal_at(const uint64_t key[2], int64_t i, double* tail_u) {
  uint64_t ctr[4] = {(uint64_t)i >> 1, 0, 0, 0};
  uint64_t w[4];
  synth_philox4x64_10(ctr, key, w);
  double u1 = u01_open(w[0]);
  double u2 = u01_open(w[1]);
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  double sn, cs;
  sincos(th, &sn, &cs);
  int odd = (int)(i & 1);
  if (tail_u) *tail_u = u01_open(w[2 + odd]);
  return odd ? r * sn : r * cs;
}

/* Round a double to the nearest bf16 value, ties to even.  bf16 keeps 8
 * significant bits and binary32's exponent range (subnormal spacing 2^-133). */
uint16_t synth_f64_to_bf16(double x) {
  /* Fast path for the normal bf16 range: round the 52-bit fraction to 7 bits
   * by adding half a unit (minus one, plus the kept LSB for ties-to-even) and
   * truncating; a carry ripples into the exponent as it should. */
  uint64_t b;
  memcpy(&b, &x, 8);
  uint64_t ex = (b >> 52) & 0x7FFu;
  if (ex >= 1023u - 126u && ex <= 1023u + 127u) {
    uint64_t r = b + 0x00000FFFFFFFFFFFull + ((b >> 45) & 1u);
    r &= ~0x00001FFFFFFFFFFFull;
    uint64_t rex = (r >> 52) & 0x7FFu;
    if (rex <= 1023u + 127u) {
      uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
      uint16_t e8 = (uint16_t)(rex - 1023u + 127u);
      uint16_t frac = (uint16_t)((r >> 45) & 0x7Fu);
      return (uint16_t)(sign | (uint16_t)(e8 << 7) | frac);
    }
  }
  if (isnan(x)) return (uint16_t)0x7FC0u;
  uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0;
  double ax = fabs(x);
  if (ax == 0.0) return sign;
  if (isinf(ax)) return (uint16_t)(sign | 0x7F80u);
  int e;
  (void)frexp(ax, &e);          /* ax = f * 2^e, f in [0.5, 1) */
  int q = e - 8;                /* weight of the last kept bit */
  if (q < -133) q = -133;
  double r = nearbyint(ldexp(ax, -q));  /* default rounding mode: nearest-even */
  double y = ldexp(r, q);
  if (y > 0x1.FEp127) return (uint16_t)(sign | 0x7F80u);  /* beyond bf16 max -> inf */
  float f = (float)y;           /* exact: y has <= 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFFu));
}

typedef struct {
  uint64_t key[2];
  int64_t start, count;
  const int64_t* idx; /* gather variant when non-null */
  double sigma, tail_p, tail_mult;
  int kind;           /* 0 = bf16, 1 = f32, 2 = f64 */
  void* out;
} job_t;

static inline void store_one(const job_t* j, int64_t t, double z, double tu) {
  double x = j->sigma * z;
  if (j->tail_p > 0.0 && tu < j->tail_p) x *= j->tail_mult;
  if (j->kind == 0) {
    ((uint16_t*)j->out)[t] = synth_f64_to_bf16(x);
  } else if (j->kind == 1) {
    ((float*)j->out)[t] = (float)x;
  } else {
    ((double*)j->out)[t] = x;
  }
}

static void run_range(const job_t* j, int64_t lo, int64_t hi) {
  if (j->idx) {
    for (int64_t t = lo; t < hi; ++t) {
      double tu = 1.0;
      double z = normal_at(j->key, j->idx[t], &tu);
      store_one(j, t, z, tu);
    }
    return;
  }
  /* Contiguous range: one Philox block and one Box-Muller pair per two elements. */
  int64_t t = lo;
  while (t < hi) {
    int64_t i = j->start + t;
    uint64_t ctr[4] = {(uint64_t)i >> 1, 0, 0, 0};
    uint64_t w[4];
    synth_philox4x64_10(ctr, j->key, w);
    double r = sqrt(-2.0 * log(u01_open(w[0])));
    double th = 6.283185307179586476925286766559 * u01_open(w[1]);
    double sn, cs;
    sincos(th, &sn, &cs);
    if ((i & 1) == 0) {
      store_one(j, t, r * cs, u01_open(w[2]));
      ++t;
      if (t >= hi) break;
    }
    store_one(j, t, r * sn, u01_open(w[3]));
    ++t;
  }
}

typedef struct {
  const job_t* job;
  int64_t lo, hi;
} part_t;

static void* run_part(void* p) {
  const part_t* q = (const part_t*)p;
  run_range(q->job, q->lo, q->hi);
  return 0;
}

static void run_job(const job_t* j, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (j->count < 65536 || nthreads == 1) {
    run_range(j, 0, j->count);
    return;
  }
  pthread_t th[256];
  part_t parts[256];
  int64_t chunk = (j->count + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t lo = (int64_t)t * chunk, hi = lo + chunk;
    if (hi > j->count) hi = j->count;
    if (lo >= hi) break;
    parts[t].job = j;
    parts[t].lo = lo;
    parts[t].hi = hi;
    if (pthread_create(&th[t], 0, run_part, &parts[t]) != 0) {
      run_range(j, lo, hi);
      parts[t].job = 0;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (parts[t].job) pthread_join(th[t], 0);
}

static void fill(int kind, uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, int64_t start,
                 int64_t count, const int64_t* idx, double sigma, double tail_p, double tail_mult, void* out,
                 int nthreads) {
  job_t j;
  stream_key(seed, role, rank, micro, j.key);
  j.start = start;
  j.count = count;
  j.idx = idx;
  j.sigma = sigma;
  j.tail_p = tail_p;
  j.tail_mult = tail_mult;
  j.kind = kind;
  j.out = out;
  run_job(&j, nthreads);
}

void synth_bf16_normal(uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, int64_t start, int64_t count,
                       double sigma, double tail_p, double tail_mult, uint16_t* out, int nthreads) {
  fill(0, seed, role, rank, micro, start, count, 0, sigma, tail_p, tail_mult, out, nthreads);
}

void synth_bf16_normal_at(uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, const int64_t* idx,
                          int64_t count, double sigma, double tail_p, double tail_mult, uint16_t* out, int nthreads) {
  fill(0, seed, role, rank, micro, 0, count, idx, sigma, tail_p, tail_mult, out, nthreads);
}

void synth_f32_normal(uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, int64_t start, int64_t count,
                      double sigma, float* out, int nthreads) {
  fill(1, seed, role, rank, micro, start, count, 0, sigma, 0.0, 1.0, out, nthreads);
}

void synth_f32_normal_at(uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, const int64_t* idx,
                         int64_t count, double sigma, float* out, int nthreads) {
  fill(1, seed, role, rank, micro, 0, count, idx, sigma, 0.0, 1.0, out, nthreads);
}

void synth_f64_normal(uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, int64_t start, int64_t count,
                      double* out, int nthreads) {
  fill(2, seed, role, rank, micro, start, count, 0, 1.0, 0.0, 1.0, out, nthreads);
}

/* Raw 64-bit words of a stream: word w of block b is element 4b + w. */
void synth_u64(uint64_t seed, uint32_t role, uint32_t rank, uint32_t micro, int64_t start, int64_t count,
               uint64_t* out) {
  uint64_t key[2];
  stream_key(seed, role, rank, micro, key);
  for (int64_t t = 0; t < count; ++t) {
    int64_t i = start + t;
    uint64_t ctr[4] = {(uint64_t)i >> 2, 0, 0, 0};
    uint64_t w[4];
    synth_philox4x64_10(ctr, key, w);
    out[t] = w[i & 3];
  }
}
