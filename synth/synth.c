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

/* One standard normal: element i of the stream keyed by `key`. */
static double normal_at(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  double u1 = to_unit(synth_draw(key, 2 * j));
  double u2 = to_unit(synth_draw(key, 2 * j + 1));
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(a) : r * cos(a);
}

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

/* Normals starting at stream element `offset`, so that a large tensor can be
 * produced in slices that concatenate to the same values. */
void synth_normal_f64(uint64_t seed, const char* tag, int64_t offset, int64_t n, double mean, double std,
                      double* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = mean + std * normal_at(key, (uint64_t)(offset + i));
}

void synth_normal_f32(uint64_t seed, const char* tag, int64_t offset, int64_t n, double mean, double std,
                      float* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + std * normal_at(key, (uint64_t)(offset + i)));
}

/* Storage as IEEE binary16 bits; the compiler's _Float16 conversion rounds
 * to nearest even from double in one step. */
void synth_normal_f16(uint64_t seed, const char* tag, int64_t offset, int64_t n, double mean, double std,
                      uint16_t* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    _Float16 h = (_Float16)(mean + std * normal_at(key, (uint64_t)(offset + i)));
    uint16_t bits;
    memcpy(&bits, &h, 2);
    out[i] = bits;
  }
}

/* Uniform on [lo, hi) rounded to fp32. */
void synth_uniform_f32(uint64_t seed, const char* tag, int64_t n, double lo, double hi, float* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * to_unit(synth_draw(key, (uint64_t)i)));
}
