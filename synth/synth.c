/*
 * Seeded synthetic input generator shared by the tests, the bench and the
 * oracle's test drivers.
 *
 * It holds none of the decode step's arithmetic: it only turns (seed, tag,
 * index) into reproducible random numbers and writes them in a storage type.
 *
 *   key(seed, tag) = splitmix64_mix(seed) ^ fnv1a64(tag)
 *   draw(key, i)   = splitmix64_mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 *
 * splitmix64 is the generator of Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators" (OOPSLA 2014); FNV-1a is the Fowler-Noll-Vo
 * string hash (64-bit offset basis and prime). Both are written here from
 * their published definitions. Being counter based, element i of a stream
 * never depends on how many threads produced the stream.
 *
 * Normals use the Box-Muller transform (Box and Muller, 1958) in double:
 * pair j takes draws 2j and 2j+1, u = ((x >> 11) + 0.5) * 2^-53, and gives
 * r*cos(2*pi*u2) to element 2j and r*sin(2*pi*u2) to element 2j+1, where
 * r = sqrt(-2 ln u1). The value mean + std*n is rounded once, in the
 * default round-to-nearest-even mode, to the target storage type.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t fnv1a64(const char* s) {
  uint64_t h = 0xcbf29ce484222325ULL;
  for (; *s; ++s) {
    h ^= (uint8_t)*s;
    h *= 0x100000001b3ULL;
  }
  return h;
}

uint64_t synth_key(uint64_t seed, const char* tag) { return mix64(seed) ^ fnv1a64(tag); }

uint64_t synth_draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * SYNTH_GOLDEN); }

static double to_unit(uint64_t x) { return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

void synth_uniform_f64(uint64_t seed, const char* tag, int64_t n, double* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = to_unit(synth_draw(key, (uint64_t)i));
}

void synth_u64(uint64_t seed, const char* tag, int64_t n, uint64_t* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = synth_draw(key, (uint64_t)i);
}

/* Normals for stream elements [offset, offset + n), so that a large tensor can
 * be produced in slices that concatenate to the same values; each Box-Muller
 * pair is computed once and both of its values are used. */
#define SYNTH_NORMAL_LOOP(STORE)                                                   \
  uint64_t key = synth_key(seed, tag);                                             \
  int64_t j0 = offset >> 1, j1 = (offset + n + 1) >> 1;                            \
  _Pragma("omp parallel for schedule(static)")                                     \
  for (int64_t j = j0; j < j1; ++j) {                                              \
    double u1 = to_unit(synth_draw(key, 2 * (uint64_t)j));                         \
    double u2 = to_unit(synth_draw(key, 2 * (uint64_t)j + 1));                     \
    double r = sqrt(-2.0 * log(u1));                                               \
    double a = 6.283185307179586476925286766559 * u2;                              \
    double v0 = mean + std * (r * cos(a)), v1 = mean + std * (r * sin(a));         \
    int64_t i0 = 2 * j - offset, i1 = i0 + 1;                                       \
    if (i0 >= 0 && i0 < n) STORE(i0, v0);                                          \
    if (i1 >= 0 && i1 < n) STORE(i1, v1);                                          \
  }

void synth_normal_f64(uint64_t seed, const char* tag, int64_t offset, int64_t n, double mean, double std,
                      double* out) {
#define ST64(i, v) out[i] = (v)
  SYNTH_NORMAL_LOOP(ST64)
#undef ST64
}

void synth_normal_f32(uint64_t seed, const char* tag, int64_t offset, int64_t n, double mean, double std,
                      float* out) {
#define ST32(i, v) out[i] = (float)(v)
  SYNTH_NORMAL_LOOP(ST32)
#undef ST32
}

/* Storage as IEEE binary16 bits; the compiler's _Float16 conversion rounds
 * to nearest even from double in one step. */
static void store_f16(uint16_t* out, int64_t i, double v) {
  _Float16 h = (_Float16)v;
  memcpy(out + i, &h, 2);
}

void synth_normal_f16(uint64_t seed, const char* tag, int64_t offset, int64_t n, double mean, double std,
                      uint16_t* out) {
#define ST16(i, v) store_f16(out, i, v)
  SYNTH_NORMAL_LOOP(ST16)
#undef ST16
}

/* Uniform on [lo, hi) rounded to fp32. */
void synth_uniform_f32(uint64_t seed, const char* tag, int64_t n, double lo, double hi, float* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * to_unit(synth_draw(key, (uint64_t)i)));
}
