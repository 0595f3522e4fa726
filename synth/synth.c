/*
 * synth.c -- seeded, counter-based normal generator shared by the tests, the
 * benchmark and (through them) both the CUDA path and the oracle.
 *
 * It holds none of the convolution's arithmetic: it only turns (stream, index)
 * into an N(0, std^2) sample rounded to float32.
 *
 *   word j of a stream:  splitmix64 output for state  base + (j+1) * 0x9E3779B97F4A7C15,
 *                        base = splitmix64 finaliser of (stream id)        [Steele, Lea &
 *                        Flood, "Fast splittable pseudorandom number generators", 2014]
 *   uniform:             u = (word >> 11) * 2^-53  in [0, 1)
 *   normal pair i:       Box-Muller on (1 - u_{2i}, u_{2i+1}):
 *                        r = sqrt(-2 ln(1 - u_{2i})), t = 2 pi u_{2i+1},
 *                        element 2i = r cos t, element 2i+1 = r sin t   [Box & Muller 1958]
 *
 * Element i depends only on (stream, i), so slices are generated in parallel.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <unistd.h>

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static const uint64_t kGolden = 0x9E3779B97F4A7C15ULL;

static double word_uniform(uint64_t base, uint64_t j) {
  return (double)(mix64(base + (j + 1) * kGolden) >> 11) * (1.0 / 9007199254740992.0);
}

typedef struct { uint64_t base; int64_t lo, hi, n; double std; float* out; } part_t;

static void* fill(void* p) {
  part_t* t = (part_t*)p;
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t i = t->lo; i < t->hi; ++i) {
    int64_t pair = i >> 1;
    double u1 = 1.0 - word_uniform(t->base, (uint64_t)(2 * pair));
    double u2 = word_uniform(t->base, (uint64_t)(2 * pair + 1));
    double r = sqrt(-2.0 * log(u1));
    double z = (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
    t->out[i] = (float)(z * t->std);
  }
  return NULL;
}

/* out[0..n) = std * N(0,1) samples of stream `stream`. */
void synth_normal_f32(uint64_t stream, int64_t n, double std, float* out) {
  uint64_t base = mix64(stream ^ 0x5851F42D4C957F2DULL);
  long nt = sysconf(_SC_NPROCESSORS_ONLN);
  if (nt < 1) nt = 1;
  if (nt > 64) nt = 64;
  if (n < (int64_t)1 << 16) nt = 1;
  pthread_t th[64];
  part_t parts[64];
  int ok[64];
  for (long t = 0; t < nt; ++t) {
    parts[t].base = base;
    parts[t].lo = n * t / nt;
    parts[t].hi = n * (t + 1) / nt;
    parts[t].n = n;
    parts[t].std = std;
    parts[t].out = out;
    ok[t] = nt > 1 && pthread_create(&th[t], NULL, fill, &parts[t]) == 0;
    if (!ok[t]) fill(&parts[t]);
  }
  for (long t = 0; t < nt; ++t)
    if (ok[t]) pthread_join(th[t], NULL);
}
