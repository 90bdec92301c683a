/* Host (C) copy of the seeded synthetic-input generator defined in synth/gen.py.
 * It holds none of the decode step's arithmetic; it only fills buffers fast
 * enough for multi-GB weight tensors.  Bit-identical to the numpy definition
 * (checked by the tests) and to the CUDA copy in synth_gen.cu. */
#include <stdint.h>
#include <string.h>

#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t syn_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t syn_key(uint64_t seed, uint64_t tid) { return syn_mix64(seed * SYN_GOLDEN + tid); }

static inline uint16_t syn_f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

/* IEEE float32 -> binary16, round to nearest even, for finite positive normal
 * inputs in the fp16 normal range (the scales generated here). */
static inline uint16_t syn_f32_to_f16_pos(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  int32_t e = (int32_t)((b >> 23) & 0xFF) - 127 + 15;
  uint32_t m = b & 0x7FFFFFu;
  uint32_t h = ((uint32_t)e << 10) | (m >> 13);
  uint32_t rem = m & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
  return (uint16_t)h;
}

void synh_fill_normal_bf16(uint16_t* dst, uint64_t n, uint64_t seed, uint64_t tid, float scale, uint64_t start) {
  const uint64_t key = syn_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) {
    uint64_t w = syn_mix64(key + ((uint64_t)i + start + 1ULL) * SYN_GOLDEN);
    int64_t s = (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) + (int64_t)((w >> 32) & 0xFFFF) + (int64_t)(w >> 48);
    float c = (float)(s - 131070);
    dst[i] = syn_f32_to_bf16(c * scale);
  }
}

void synh_fill_q4_packed(uint8_t* dst, uint64_t nbytes, uint64_t seed, uint64_t tid) {
  const uint64_t key = syn_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)nbytes; ++i) {
    uint64_t w = syn_mix64(key + ((uint64_t)i / 8ULL + 1ULL) * SYN_GOLDEN);
    dst[i] = (uint8_t)((w >> (8 * ((uint64_t)i % 8ULL))) & 0xFF);
  }
}

void synh_fill_q4_scales(uint16_t* dst, uint64_t nblocks, uint64_t seed, uint64_t tid, float mult) {
  const uint64_t key = syn_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)nblocks; ++i) {
    uint64_t w = syn_mix64(key + ((uint64_t)i + 1ULL) * SYN_GOLDEN);
    float u = (float)((int64_t)(w & 0xFFFF) + 49152);
    dst[i] = syn_f32_to_f16_pos(u * mult);
  }
}

void synh_fill_uniform_ids(int32_t* dst, uint64_t n, uint64_t seed, uint64_t tid, uint32_t upper, uint64_t start) {
  const uint64_t key = syn_key(seed, tid);
  for (uint64_t i = 0; i < n; ++i) {
    uint64_t w = syn_mix64(key + (i + start + 1ULL) * SYN_GOLDEN);
    dst[i] = (int32_t)(((w >> 32) * (uint64_t)upper) >> 32);
  }
}
