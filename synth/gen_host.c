/*
 * Seeded synthetic input generator, host side (plain C, OpenMP).
 *
 * This file is test and benchmark infrastructure: it produces the inputs that
 * both the CUDA path and the CPU oracle consume. It holds none of the MoE
 * layer's arithmetic.
 *
 * Definition (shared word for word with synth/gen_device.cu, which must stay
 * bit-identical to this file):
 *
 *   mix64(z)     : SplitMix64 output finaliser (Steele, Lea & Flood, "Fast
 *                  splittable pseudorandom number generators", OOPSLA 2014,
 *                  with Stafford's "Mix13" constants as used by Vigna's
 *                  splitmix64.c):
 *                    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                    z =  z ^ (z >> 31)
 *   key(seed, id): mix64(seed * 0x9E3779B97F4A7C15 + id * 0xD1B54A32D192ED03)
 *   bits(i)      : mix64(key + (i + 1) * 0x9E3779B97F4A7C15)   (the (i+1)-th
 *                  SplitMix64 output of a generator whose state is key)
 *   S(i)         : sum of the four 16-bit fields of bits(i), in [0, 262140]
 *   c(i)         : 2 * S(i) - 262140 (an even integer, |c| <= 262140 < 2^24)
 *   value(i)     : (float)c(i) * scale, one IEEE binary32 multiply (RNE),
 *                  where scale = sigma / (2 * sqrt((65536^2 - 1) / 3)) rounded
 *                  once to binary32 by the caller
 *   bf16(i)      : value(i) rounded to bfloat16, round-to-nearest-even
 *
 * c is an Irwin-Hall(4) sum of discrete uniforms, centred and scaled to unit
 * variance, so value(i) approximates N(0, sigma^2) with tails cut at about
 * +-3.46 sigma.
 */
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_stream_key(uint64_t seed, uint64_t tensor_id) {
  return mix64(seed * 0x9E3779B97F4A7C15ULL + tensor_id * 0xD1B54A32D192ED03ULL);
}

static inline int32_t centred_sum(uint64_t key, uint64_t i) {
  uint64_t b = mix64(key + (i + 1ULL) * 0x9E3779B97F4A7C15ULL);
  uint32_t s = (uint32_t)(b & 0xFFFFu) + (uint32_t)((b >> 16) & 0xFFFFu) +
               (uint32_t)((b >> 32) & 0xFFFFu) + (uint32_t)((b >> 48) & 0xFFFFu);
  return 2 * (int32_t)s - 262140;
}

static inline uint16_t f32_to_bf16_rne(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* out[j] = value(start + j) for j < n. */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t n,
                      float scale, float* out) {
  const uint64_t key = synth_stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)n; ++j) {
    float c = (float)centred_sum(key, start + (uint64_t)j);
    out[j] = c * scale;
  }
}

/* out[j] = bf16(start + j) as raw bit patterns. */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t n,
                       float scale, uint16_t* out) {
  const uint64_t key = synth_stream_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)n; ++j) {
    float c = (float)centred_sum(key, start + (uint64_t)j);
    float v = c * scale;
    out[j] = f32_to_bf16_rne(v);
  }
}
