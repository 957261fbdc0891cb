/* Host implementation of the seeded input generator defined in synth.py.
 *
 * Same definition, element by element: two SplitMix64 words per element from a
 * Weyl counter, the sum of their eight 16-bit lanes (Irwin-Hall, n = 8), centred,
 * times one fp32 scale.  Only integer operations and one IEEE single-precision multiply are involved, so the bits
 * equal those of the torch implementation on any device.  Output is fp32; the
 * caller rounds to bf16 with torch, as the torch path does.  Build with
 * -ffp-contract=off (there is nothing to contract, but keep it explicit).
 */
#include <stdint.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline int64_t lanes(uint64_t w) {
  return (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) +
         (int64_t)((w >> 32) & 0xFFFF) + (int64_t)(w >> 48);
}

static inline float value(uint64_t key, int64_t i, float scale) {
  uint64_t c = 2ULL * (uint64_t)i;
  uint64_t w0 = mix64(key + (c + 1ULL) * GOLDEN);
  uint64_t w1 = mix64(key + (c + 2ULL) * GOLDEN);
  int64_t s2 = 2 * (lanes(w0) + lanes(w1)) - 8 * 65535;
  return (float)s2 * scale; /* (float)s2 is exact: |s2| < 2^21 */
}

void synth_fill_f32(uint64_t key, int64_t offset, int64_t n, float scale, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = value(key, offset + i, scale);
}

void synth_gather_f32(uint64_t key, const int64_t* idx, int64_t n, float scale, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = value(key, idx[i], scale);
}
