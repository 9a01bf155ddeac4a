/*
 * Seeded synthetic input generator, shared by the tests, the oracle-side
 * checks and the bench.  It draws random tensors and nothing else: it holds
 * none of the normalisation arithmetic, and neither the oracle nor the CUDA
 * library links against it.
 *
 * Stream definition (counter based, so any element can be drawn alone and the
 * fill is trivially parallel):
 *   sub-seed  s_t = mix64(seed ^ (tensor_id * 0x9E3779B97F4A7C15))
 *   word      w(i) = mix64(s_t + (i + 1) * 0x9E3779B97F4A7C15)        (SplitMix64)
 *   uniform   u(i) = (w(i) >> 11) * 2^-53                            in [0, 1)
 *   normal    for the pair p: a = sqrt(-2 ln(1 - u(2p))), b = 2 pi u(2p+1);
 *             element 2p = a cos b, element 2p+1 = a sin b          (Box-Muller)
 * Values are drawn in double precision and rounded once to the storage type:
 * fp32 by the C conversion (round to nearest even), bf16 by the rounding
 * written below (round to nearest even, straight from double).
 *
 * Outliers: exactly K distinct positions of the tensor are chosen uniformly
 * (Floyd's sampling over a bitmap, driven by the sub-stream of tensor_id +
 * 0x1000); at each one the stored value becomes round(scale * z), z being that
 * element's own normal draw.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL
#define GEN_F32 0
#define GEN_BF16 1
#define DIST_NORMAL 0
#define DIST_UNIFORM 1

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t sub_seed(uint64_t seed, uint64_t tensor_id) {
  return mix64(seed ^ (tensor_id * GOLDEN));
}

static double uniform_at(uint64_t s, uint64_t i) {
  uint64_t w = mix64(s + (i + 1) * GOLDEN);
  return (double)(w >> 11) * (1.0 / 9007199254740992.0);
}

static double normal_at(uint64_t s, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t p = i >> 1;
  double u1 = uniform_at(s, 2 * p);
  double u2 = uniform_at(s, 2 * p + 1);
  double a = sqrt(-2.0 * log(1.0 - u1));
  return (i & 1) ? a * sin(two_pi * u2) : a * cos(two_pi * u2);
}

/* Round a double to the nearest bf16 bit pattern, ties to even.  Written from
 * the format: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static uint16_t to_bf16_bits(double v) {
  if (isnan(v)) return (uint16_t)(signbit(v) ? 0xFFC0 : 0x7FC0);
  uint16_t sign = (uint16_t)(signbit(v) ? 0x8000 : 0);
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1) */
  int exp_unb = e - 1;          /* a = 1.f * 2^exp_unb */
  if (exp_unb < -126) exp_unb = -126; /* subnormal range shares the step 2^-133 */
  double step = ldexp(1.0, exp_unb - 7);
  double q = a / step;          /* exact: power-of-two scaling */
  double fl = floor(q);
  double rem = q - fl;
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  double r = fl * step;
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  /* re-encode r exactly */
  if (r < ldexp(1.0, -126)) {
    uint16_t frac = (uint16_t)(r / ldexp(1.0, -133));
    return (uint16_t)(sign | frac);
  }
  int e2;
  double f2 = frexp(r, &e2);    /* r = f2 * 2^e2 */
  uint16_t biased = (uint16_t)(e2 - 1 + 127);
  uint16_t frac = (uint16_t)((f2 * 2.0 - 1.0) * 128.0);
  return (uint16_t)(sign | (uint16_t)(biased << 7) | frac);
}

typedef struct {
  uint64_t s;
  int dist;
  double p0, p1;
  int dtype;
  void* out;
  int64_t begin, end;
} fill_job;

static void store_value(void* out, int dtype, int64_t i, double v) {
  if (dtype == GEN_F32)
    ((float*)out)[i] = (float)v;
  else
    ((uint16_t*)out)[i] = to_bf16_bits(v);
}

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  for (int64_t i = j->begin; i < j->end; ++i) {
    double v;
    if (j->dist == DIST_NORMAL)
      v = j->p0 + j->p1 * normal_at(j->s, (uint64_t)i);
    else
      v = j->p0 + (j->p1 - j->p0) * uniform_at(j->s, (uint64_t)i);
    store_value(j->out, j->dtype, i, v);
  }
  return NULL;
}

/* Fill out[0..n) with the tensor (seed, tensor_id).  dist: 0 normal(p0 = mean,
 * p1 = std), 1 uniform[p0, p1).  dtype: 0 fp32, 1 bf16 bits.  threads <= 0
 * picks one thread per 4M elements, at most 64.  Returns 0, or -1 on bad
 * arguments. */
int gen_fill(uint64_t seed, uint64_t tensor_id, int dist, double p0, double p1,
             int64_t n, int dtype, void* out, int threads) {
  if (n < 0 || (n > 0 && out == NULL)) return -1;
  if (dtype != GEN_F32 && dtype != GEN_BF16) return -1;
  if (dist != DIST_NORMAL && dist != DIST_UNIFORM) return -1;
  uint64_t s = sub_seed(seed, tensor_id);
  if (threads <= 0) {
    int64_t t = n / (4 << 20) + 1;
    threads = (int)(t > 64 ? 64 : t);
  }
  if (threads > 256) threads = 256;
  fill_job jobs[256];
  pthread_t tids[256];
  int joined[256];
  int64_t chunk = (n + threads - 1) / threads;
  chunk = (chunk + 1) & ~(int64_t)1; /* keep Box-Muller pairs in one job */
  int njobs = 0;
  for (int t = 0; t < threads; ++t) {
    int64_t b = (int64_t)t * chunk, e = b + chunk;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[njobs] = (fill_job){s, dist, p0, p1, dtype, out, b, e};
    joined[njobs] = 0;
    ++njobs;
  }
  for (int t = 1; t < njobs; ++t)
    joined[t] = pthread_create(&tids[t], NULL, fill_worker, &jobs[t]) == 0;
  for (int t = 0; t < njobs; ++t)
    if (!joined[t]) fill_worker(&jobs[t]);
  for (int t = 1; t < njobs; ++t)
    if (joined[t]) pthread_join(tids[t], NULL);
  return 0;
}

/* Choose k distinct positions of [0, n) uniformly (Floyd) from the
 * sub-stream (seed, tensor_id + 0x1000); writes them, ascending, to pos[0..k).
 * Returns 0, or -1 on bad arguments / allocation failure. */
int gen_outlier_positions(uint64_t seed, uint64_t tensor_id, int64_t n, int64_t k,
                          int64_t* pos) {
  if (n < 0 || k < 0 || k > n || (k > 0 && pos == NULL)) return -1;
  if (k == 0) return 0;
  uint64_t s = sub_seed(seed, tensor_id + 0x1000);
  size_t words = (size_t)((n + 63) / 64);
  uint64_t* bits = (uint64_t*)calloc(words, sizeof(uint64_t));
  if (!bits) return -1;
  uint64_t draw = 0;
  for (int64_t j = n - k; j < n; ++j) {
    int64_t t = (int64_t)(uniform_at(s, draw++) * (double)(j + 1));
    if (t > j) t = j;
    int64_t pick = (bits[t >> 6] >> (t & 63)) & 1 ? j : t;
    bits[pick >> 6] |= 1ULL << (pick & 63);
  }
  int64_t c = 0;
  for (size_t w = 0; w < words; ++w) {
    uint64_t b = bits[w];
    while (b) {
      int bit = __builtin_ctzll(b);
      pos[c++] = (int64_t)(w * 64 + (size_t)bit);
      b &= b - 1;
    }
  }
  free(bits);
  return c == k ? 0 : -1;
}

/* Overwrite out[pos[q]] with round(p0 + p1 * scale * z), z being the normal
 * draw of that element in the stream (seed, tensor_id): the element's own
 * value, scaled.  p0/p1 are the tensor's mean/std as passed to gen_fill. */
int gen_apply_outliers(uint64_t seed, uint64_t tensor_id, double p0, double p1,
                       double scale, const int64_t* pos, int64_t k, int dtype,
                       void* out) {
  if (k < 0 || (k > 0 && (pos == NULL || out == NULL))) return -1;
  if (dtype != GEN_F32 && dtype != GEN_BF16) return -1;
  uint64_t s = sub_seed(seed, tensor_id);
  for (int64_t q = 0; q < k; ++q) {
    double z = normal_at(s, (uint64_t)pos[q]);
    store_value(out, dtype, pos[q], p0 + p1 * scale * z);
  }
  return 0;
}

/* The raw streams, for tests of the generator itself. */
double gen_uniform_at(uint64_t seed, uint64_t tensor_id, uint64_t i) {
  return uniform_at(sub_seed(seed, tensor_id), i);
}
double gen_normal_at(uint64_t seed, uint64_t tensor_id, uint64_t i) {
  return normal_at(sub_seed(seed, tensor_id), i);
}
uint64_t gen_splitmix64_next(uint64_t state) { return mix64(state + GOLDEN); }
