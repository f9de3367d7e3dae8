/*
 * CPU side of the seeded input generator (definitions in synth_core.h).
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (see synth/build.py).
 */
#include "synth_core.h"

#define SYN_API __attribute__((visibility("default")))

/* Gradients of worker w at step t for coordinates [i0, i0+n). */
SYN_API int syn_cpu_grads_range(int kind, uint64_t seed, const uint64_t* starts,
                                const float* sigmas, uint32_t n_tensors, uint32_t w,
                                uint32_t t, uint64_t i0, uint64_t n, uint16_t* out) {
  if (!starts || !sigmas || !out || n_tensors == 0) return -1;
  for (uint64_t j = 0; j < n; j++) {
    uint64_t i = i0 + j;
    float sig = sigmas[syn_tensor_of(starts, n_tensors, i)];
    out[j] = syn_grad_bf16(kind, seed, w, t, i, sig);
  }
  return 0;
}

/* Gradients of worker w at step t for an explicit list of coordinates. */
SYN_API int syn_cpu_grads_list(int kind, uint64_t seed, const uint64_t* starts,
                               const float* sigmas, uint32_t n_tensors, uint32_t w,
                               uint32_t t, const uint64_t* idx, uint64_t n, uint16_t* out) {
  if (!starts || !sigmas || !out || !idx || n_tensors == 0) return -1;
  for (uint64_t j = 0; j < n; j++) {
    float sig = sigmas[syn_tensor_of(starts, n_tensors, idx[j])];
    out[j] = syn_grad_bf16(kind, seed, w, t, idx[j], sig);
  }
  return 0;
}

/* theta_0 for an explicit list of coordinates. */
SYN_API int syn_cpu_theta_list(uint64_t seed, const uint64_t* idx, uint64_t n, float* out) {
  if (!idx || !out) return -1;
  for (uint64_t j = 0; j < n; j++) out[j] = syn_theta0(seed, idx[j]);
  return 0;
}

/* Standard normals Z(seed, stream, w, t, i) for i in [i0, i0+n) (test hook
 * for the distribution checks). */
SYN_API int syn_cpu_normals(uint64_t seed, uint64_t stream, uint32_t w, uint32_t t,
                            uint64_t i0, uint64_t n, float* out) {
  if (!out) return -1;
  for (uint64_t j = 0; j < n; j++) out[j] = syn_normal(syn_key(seed, stream, w, t, i0 + j));
  return 0;
}

/* The series log, exposed so a test can hold it against libm. */
SYN_API float syn_cpu_logf(float x) { return syn_logf(x); }
