/*
 * GPU side of the seeded input generator (definitions in synth_core.h):
 * fills device buffers with the same bytes synth_cpu.c produces.
 * Build: nvcc -gencode arch=compute_103a,code=sm_103a -fmad=false -shared.
 */
#include <cuda_runtime.h>
#include "synth_core.h"

#define SYN_API extern "C" __attribute__((visibility("default")))

namespace {

__global__ void grads_kernel(int kind, uint64_t seed, const uint64_t* __restrict__ starts,
                             const float* __restrict__ sigmas, uint32_t n_tensors, uint32_t w,
                             uint32_t t, uint64_t i0, uint64_t n, uint16_t* __restrict__ out) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    uint64_t i = i0 + j;
    float sig = sigmas[syn_tensor_of(starts, n_tensors, i)];
    out[j] = syn_grad_bf16(kind, seed, w, t, i, sig);
  }
}

__global__ void theta_kernel(uint64_t seed, uint64_t i0, uint64_t n, float* __restrict__ out) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    out[j] = syn_theta0(seed, i0 + j);
}

unsigned grid_for(uint64_t n) {
  uint64_t b = (n + 255) / 256;
  if (b > 152ull * 64) b = 152ull * 64;
  if (b == 0) b = 1;
  return (unsigned)b;
}

}  // namespace

/* Gradients of worker w at step t for [i0, i0+n) into device d_out.
 * starts/sigmas are DEVICE arrays (n_tensors+1 and n_tensors entries). */
SYN_API int syn_gpu_grads_range(int kind, uint64_t seed, const uint64_t* d_starts,
                                const float* d_sigmas, uint32_t n_tensors, uint32_t w,
                                uint32_t t, uint64_t i0, uint64_t n, uint16_t* d_out,
                                cudaStream_t stream) {
  if (!d_starts || !d_sigmas || !d_out || n_tensors == 0) return -1;
  if (n == 0) return 0;
  grads_kernel<<<grid_for(n), 256, 0, stream>>>(kind, seed, d_starts, d_sigmas, n_tensors, w, t,
                                                i0, n, d_out);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

SYN_API int syn_gpu_theta_range(uint64_t seed, uint64_t i0, uint64_t n, float* d_out,
                                cudaStream_t stream) {
  if (!d_out) return -1;
  if (n == 0) return 0;
  theta_kernel<<<grid_for(n), 256, 0, stream>>>(seed, i0, n, d_out);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
