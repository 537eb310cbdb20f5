/* Seeded synthetic-input generator (host C, OpenMP).
 *
 * Counter-based: element i of a stream with keys (k1, k2) is a function of
 * (k1, k2, i) alone, so any slice of any tensor can be regenerated on its
 * own and the result does not depend on the thread count.  The mixing
 * function is the 32-bit MurmurHash3 finaliser (Appleby, public domain),
 * applied twice.
 *
 * This file produces inputs only (weights, prompts, uniforms, codes); it
 * contains none of the Dual-AR arithmetic.
 */
#include <stdint.h>

static inline uint32_t fmix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x85EBCA6Bu;
  x ^= x >> 13;
  x *= 0xC2B2AE35u;
  x ^= x >> 16;
  return x;
}

static inline uint32_t counter_hash(int64_t i, uint32_t k1, uint32_t k2) {
  uint32_t lo = (uint32_t)((uint64_t)i & 0xFFFFFFFFu);
  uint32_t hi = (uint32_t)((uint64_t)i >> 32);
  return fmix32(fmix32(lo + k1) ^ (k2 + hi * 0x9E3779B9u));
}

/* out[i] = table[hash(i) >> 16]: a 65,536-entry quantile table turns the
 * 16-bit hash into a (discretised) draw from the table's distribution. */
void dualar_gen_table16(uint16_t* out, int64_t n, const uint16_t* table,
                        uint32_t k1, uint32_t k2) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = table[counter_hash(i, k1, k2) >> 16];
}

/* Uniform floats on [0, 1) with 24 random bits (exact in fp32). */
void dualar_gen_uniform(float* out, int64_t n, uint32_t k1, uint32_t k2) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = (float)(counter_hash(i, k1, k2) >> 8) * (1.0f / 16777216.0f);
}

/* Integers uniform on [lo, hi): lo + floor(hash * (hi - lo) / 2^32). */
void dualar_gen_randint(int64_t* out, int64_t n, uint32_t k1, uint32_t k2,
                        int64_t lo, int64_t hi) {
  uint64_t span = (uint64_t)(hi - lo);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = lo + (int64_t)(((uint64_t)counter_hash(i, k1, k2) * span) >> 32);
}
