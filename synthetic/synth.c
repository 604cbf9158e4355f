/*
 * Seeded synthetic inputs shared by the fp64 oracle and the CUDA path.
 *
 * This file holds no attention arithmetic: it only draws numbers.  Both
 * sides consume the same host-generated bf16 bit patterns.
 *
 * Generator: a counter-based splitmix64 stream (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014; the
 * finaliser constants are the published ones).  Draw i of stream (seed, id)
 * is mix64(base + (i + 1) * GAMMA) with base = mix64(seed * GAMMA ^ id).
 * Two draws give two uniforms in (0, 1); the Box-Muller transform (Box &
 * Muller 1958) turns them into two standard normals, computed in double.
 * A value is multiplied by `mul`, optionally offset, rounded to float32
 * (round to nearest even) and then to bfloat16 (round to nearest even).
 *
 * Work is split over POSIX threads by index range; the result does not
 * depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t id) {
  return mix64(seed * GAMMA ^ (id + 0x632BE59BD9B4E019ULL));
}

/* uniform in the open interval (0, 1): 53 random bits, centred in the cell */
static inline double to_unit(uint64_t r) {
  return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) { /* inf / nan: keep, quiet nan */
    return (uint16_t)((u >> 16) | ((u & 0x007FFFFFu) ? 0x40u : 0u));
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* standard normal number n of stream (base): pair k = n / 2, cos or sin leg */
static inline double normal_at(uint64_t base, int64_t n) {
  int64_t k = n >> 1;
  uint64_t r1 = mix64(base + (uint64_t)(2 * k + 1) * GAMMA);
  uint64_t r2 = mix64(base + (uint64_t)(2 * k + 2) * GAMMA);
  double u1 = to_unit(r1), u2 = to_unit(r2);
  double rad = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586476925286766559 * u2;
  return (n & 1) ? rad * sin(ang) : rad * cos(ang);
}

typedef struct {
  uint16_t* out;
  int64_t lo, hi;
  uint64_t base;
  double mul;
  /* optional per-row offset: value += off_max * (row / (rows - 1)), where
   * row = (n / row_inner) % rows.  rows <= 1 disables it. */
  double off_max;
  int64_t row_inner, rows;
} job_t;

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  for (int64_t n = j->lo; n < j->hi; ++n) {
    double x = j->mul * normal_at(j->base, n);
    if (j->rows > 1) {
      int64_t row = (n / j->row_inner) % j->rows;
      x += j->off_max * ((double)row / (double)(j->rows - 1));
    }
    j->out[n] = f32_to_bf16_rne((float)x);
  }
  return 0;
}

static int run_parallel(uint16_t* out, int64_t count, uint64_t seed, uint64_t id, double mul,
                        double off_max, int64_t row_inner, int64_t rows, int nthreads) {
  if (count <= 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (count < 65536) nthreads = 1;
  pthread_t th[256];
  int live[256];
  job_t jobs[256];
  uint64_t base = stream_base(seed, id);
  int64_t per = (count + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    int64_t lo = (int64_t)t * per, hi = lo + per;
    live[t] = 0;
    if (lo >= count) continue;
    if (hi > count) hi = count;
    jobs[t] = (job_t){out, lo, hi, base, mul, off_max, row_inner, rows};
    if (t > 0 && pthread_create(&th[t], 0, run_job, &jobs[t]) == 0) {
      live[t] = 1;
    } else if (t > 0) {
      run_job(&jobs[t]); /* thread creation failed: do the slice here */
    }
  }
  run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (live[t]) pthread_join(th[t], 0);
  return 0;
}

/* out[n] = bf16(mul * N(0,1)_n) for n < count */
int synth_normal_bf16(uint16_t* out, int64_t count, uint64_t seed, uint64_t id, double mul,
                      int nthreads) {
  return run_parallel(out, count, seed, id, mul, 0.0, 1, 0, nthreads);
}

/* out[n] = bf16(mul * N(0,1)_n + off_max * row / (rows - 1)) with
 * row = (n / row_inner) % rows: for a [B, S, H, D] tensor, row_inner = H * D
 * and rows = S gives an offset that rises linearly along the sequence. */
int synth_normal_offset_bf16(uint16_t* out, int64_t count, uint64_t seed, uint64_t id, double mul,
                             double off_max, int64_t row_inner, int64_t rows, int nthreads) {
  if (row_inner < 1) return -1;
  return run_parallel(out, count, seed, id, mul, off_max, row_inner, rows, nthreads);
}
