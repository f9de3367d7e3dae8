/*
 * Seeded synthetic inputs for the SCAPE optimizer step: per-worker bf16
 * gradients and the fp32 initial parameters.
 *
 * This header is the single definition of the generator.  It is compiled by
 * gcc for the CPU side (synth_cpu.c, which feeds the oracle) and by nvcc for
 * the GPU side (synth_gpu.cu, which feeds the CUDA path), so both sides draw
 * the same bytes.  It holds none of the optimizer's arithmetic.
 *
 * Every value is a pure function of (seed, stream, worker, step, index):
 *   - counter hash: the SplitMix64 output function (Steele, Lea and Flood,
 *     "Fast splittable pseudorandom number generators", OOPSLA 2014) applied
 *     in a chain over the five counters;
 *   - normal deviates: Marsaglia's polar method (Marsaglia and Bray, 1964),
 *     with candidate pairs drawn from successive hashes of the key;
 *   - the natural log the polar method needs is evaluated here from the
 *     series ln m = 2 atanh((m-1)/(m+1)) after a frexp range reduction, so no
 *     platform math library is involved.
 * Only IEEE-754 single-precision +, -, *, / and sqrt (all correctly rounded
 * on both sides), frexpf, rintf and integer operations are used; both
 * compilers must be told not to contract a*b+c into an FMA (gcc:
 * -ffp-contract=off, nvcc: -fmad=false).  With that the CPU and GPU outputs
 * are bit-identical, which a GPU test checks.
 *
 * Workloads (the parameter-layout shapes of the models the SCAPE pages train):
 *   SYN_GAUSS:     mu_i = sigma_i * Z_i (fixed per coordinate),
 *                  g_{w,t,i} = mu_i + (0.5 sigma_i) * xi_{w,t,i},  xi ~ N(0,1)
 *   SYN_STUDENT_Q: mu_i = sigma * T3_i with T3 = Z0 / sqrt((Z1^2+Z2^2+Z3^2)/3)
 *                  (Student-t, nu = 3); g as above, then rounded half-even to a
 *                  multiple of 2^-14 (many exact ties in |a|).
 *   theta_0,i = 0.02 * Z_i.
 * Gradients are rounded to bf16 with round-to-nearest-even.
 */
#ifndef SCAPE_SYNTH_CORE_H
#define SCAPE_SYNTH_CORE_H

#include <stdint.h>
#include <math.h>
#include <string.h>

#ifdef __CUDACC__
#define SYN_HD __host__ __device__ __forceinline__
#else
#define SYN_HD static inline
#endif

enum { SYN_GAUSS = 0, SYN_STUDENT_Q = 1 };
enum { SYN_STREAM_MU = 1, SYN_STREAM_XI = 2, SYN_STREAM_THETA = 3 };

/* SplitMix64 output function. */
SYN_HD uint64_t syn_mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Key of one draw: a chain of SplitMix64 over the five counters. */
SYN_HD uint64_t syn_key(uint64_t seed, uint64_t stream, uint64_t worker,
                        uint64_t step, uint64_t index) {
  uint64_t h = syn_mix64(seed);
  h = syn_mix64(h ^ stream);
  h = syn_mix64(h ^ worker);
  h = syn_mix64(h ^ step);
  h = syn_mix64(h ^ index);
  return h;
}

/* 24 random bits -> uniform on [-1, 1), exact in fp32. */
SYN_HD float syn_unit2(uint64_t bits24) {
  return ((float)(bits24 & 0xFFFFFFull) * (1.0f / 16777216.0f)) * 2.0f - 1.0f;
}

/* Natural log for 0 < x < 1 (normal range): frexp reduction to
 * m in [1/sqrt2, sqrt2), then 2*atanh(s) = 2(s + s^3/3 + ... + s^13/13),
 * |s| < 0.172 so the dropped tail is below 1e-12 relative. */
SYN_HD float syn_logf(float x) {
  int ex = 0;
  float m = frexpf(x, &ex);
  if (m < 0.70710678f) {
    m = m * 2.0f;
    ex = ex - 1;
  }
  float s = (m - 1.0f) / (m + 1.0f);
  float s2 = s * s;
  float term = s;
  float sum = s;
  term = term * s2; sum = sum + term / 3.0f;
  term = term * s2; sum = sum + term / 5.0f;
  term = term * s2; sum = sum + term / 7.0f;
  term = term * s2; sum = sum + term / 9.0f;
  term = term * s2; sum = sum + term / 11.0f;
  term = term * s2; sum = sum + term / 13.0f;
  return (float)ex * 0.693147182f + 2.0f * sum;
}

/* One N(0,1) deviate by the polar method; attempt j uses hash(key + j).
 * Gives up (returns 0) after 64 rejected pairs, probability ~ 0.2146^64. */
SYN_HD float syn_normal(uint64_t key) {
  for (uint64_t j = 0; j < 64; j++) {
    uint64_t h = syn_mix64(key + j);
    float v1 = syn_unit2(h >> 40);
    float v2 = syn_unit2(h >> 16);
    float s = v1 * v1 + v2 * v2;
    if (s > 0.0f && s < 1.0f) {
      return v1 * sqrtf((-2.0f * syn_logf(s)) / s);
    }
  }
  return 0.0f;
}

SYN_HD uint32_t syn_f32_bits(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  uint32_t b;
  memcpy(&b, &f, 4);
  return b;
#endif
}

/* fp32 -> bf16 with round-to-nearest-even (inputs are finite). */
SYN_HD uint16_t syn_f32_to_bf16(float f) {
  uint32_t b = syn_f32_bits(f);
  b = b + 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

/* Index of the tensor holding flat coordinate i: starts[] has n+1 ascending
 * entries, starts[0] = 0, starts[n] = N. */
SYN_HD uint32_t syn_tensor_of(const uint64_t* starts, uint32_t n, uint64_t i) {
  uint32_t lo = 0, hi = n;
  while (hi - lo > 1) {
    uint32_t mid = (lo + hi) >> 1;
    if (starts[mid] <= i) lo = mid; else hi = mid;
  }
  return lo;
}

/* Per-coordinate mean mu_i. */
SYN_HD float syn_mu(int kind, uint64_t seed, uint64_t i, float sigma) {
  if (kind == SYN_STUDENT_Q) {
    float z0 = syn_normal(syn_key(seed, SYN_STREAM_MU, 0, 0, i));
    float z1 = syn_normal(syn_key(seed, SYN_STREAM_MU, 1, 0, i));
    float z2 = syn_normal(syn_key(seed, SYN_STREAM_MU, 2, 0, i));
    float z3 = syn_normal(syn_key(seed, SYN_STREAM_MU, 3, 0, i));
    float den = sqrtf((z1 * z1 + z2 * z2 + z3 * z3) / 3.0f);
    if (!(den > 0.0f)) return 0.0f;
    return sigma * (z0 / den);
  }
  return sigma * syn_normal(syn_key(seed, SYN_STREAM_MU, 0, 0, i));
}

/* Gradient of worker w at step t, coordinate i, as bf16 bits. */
SYN_HD uint16_t syn_grad_bf16(int kind, uint64_t seed, uint64_t w, uint64_t t,
                              uint64_t i, float sigma) {
  float mu = syn_mu(kind, seed, i, sigma);
  float xi = syn_normal(syn_key(seed, SYN_STREAM_XI, w, t, i));
  float g = mu + (0.5f * sigma) * xi;
  if (kind == SYN_STUDENT_Q) g = rintf(g * 16384.0f) / 16384.0f;
  return syn_f32_to_bf16(g);
}

/* Initial parameter theta_0 at coordinate i. */
SYN_HD float syn_theta0(uint64_t seed, uint64_t i) {
  return 0.02f * syn_normal(syn_key(seed, SYN_STREAM_THETA, 0, 0, i));
}

#endif
