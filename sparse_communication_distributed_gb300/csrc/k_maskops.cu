// Word-wise operations on packed masks, used by the mask diagnostics:
// OR-accumulation of per-worker masks and popcounts of (a & b).
#include "scape_device.cuh"
#include "scape_kernels.cuh"

namespace scape {
namespace {

__global__ __launch_bounds__(256) void mask_or(uint32_t* __restrict__ acc,
                                               const uint32_t* __restrict__ m, uint64_t n,
                                               int first) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    acc[i] = first ? m[i] : (acc[i] | m[i]);
}

// The union variant's compact layout: set bits of every chunk of a mask, one
// warp per chunk (bits past the chunk's end in its last word are ignored).
__global__ __launch_bounds__(256) void chunk_counts(const uint32_t* __restrict__ mask,
                                                    const ChunkDesc* __restrict__ chunks,
                                                    uint64_t n_ch, uint32_t C, uint64_t N,
                                                    uint32_t* __restrict__ counts) {
  const int lane = threadIdx.x & 31;
  const uint64_t nwarps = (uint64_t)gridDim.x * (blockDim.x / 32);
  for (uint64_t c = (uint64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); c < n_ch;
       c += nwarps) {  // warp-uniform
    uint64_t c0;
    uint32_t L;
    if (chunks) {
      c0 = chunks[c].start;
      L = chunks[c].len;
    } else {
      c0 = c * C;
      L = (uint32_t)((N - c0) < C ? (N - c0) : C);
    }
    const uint32_t nw = (L + 31) / 32;
    const uint32_t* m = mask + c0 / 32;
    uint32_t cnt = 0;
    for (uint32_t j = lane; j < nw; j += 32) {
      uint32_t word = m[j];
      if (j == nw - 1 && (L & 31)) word &= (1u << (L & 31)) - 1u;
      cnt += __popc(word);
    }
    cnt = __reduce_add_sync(kFull, cnt);
    if (lane == 0) counts[c] = cnt;
  }
}

// Exclusive prefix of the chunk counts (one CTA, tiles of 1024 with a running
// carry): cbase[c] = packed position of chunk c's first kept value,
// cbase[n_ch] = the total.
__global__ __launch_bounds__(1024) void chunk_scan(const uint32_t* __restrict__ counts,
                                                   uint64_t n_ch, uint64_t* __restrict__ cbase) {
  __shared__ uint32_t part[33];
  __shared__ unsigned long long carry;
  if (threadIdx.x == 0) carry = 0ull;
  __syncthreads();
  for (uint64_t b0 = 0; b0 < n_ch; b0 += 1024) {
    const uint64_t c = b0 + threadIdx.x;
    const uint32_t x = c < n_ch ? counts[c] : 0u;
    uint32_t total;  // at most 1024 * 65536: fits
    const uint32_t inc = block_incl_scan<1024>(x, part, &total);
    const unsigned long long cb = carry;
    if (c < n_ch) cbase[c] = cb + (inc - x);
    __syncthreads();
    if (threadIdx.x == 0) carry = cb + total;
    __syncthreads();
  }
  if (threadIdx.x == 0) cbase[n_ch] = carry;
}

__global__ __launch_bounds__(256) void mask_popcount(const uint32_t* __restrict__ a,
                                                     const uint32_t* __restrict__ b, uint64_t n,
                                                     unsigned long long* __restrict__ out) {
  __shared__ uint32_t part[9];
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint32_t cnt = 0;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    cnt += __popc(b ? (a[i] & b[i]) : a[i]);
  uint32_t total;
  block_incl_scan<256>(cnt, part, &total);
  if (threadIdx.x == 0 && total) atomicAdd(out, (unsigned long long)total);
}

unsigned grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  const uint64_t cap = (uint64_t)num_sms() * 8;
  if (g > cap) g = cap;
  return (unsigned)(g ? g : 1);
}

}  // namespace

cudaError_t launch_mask_or(uint32_t* acc, const uint32_t* m, uint64_t nwords, bool first,
                           cudaStream_t s) {
  mask_or<<<grid_for(nwords), 256, 0, s>>>(acc, m, nwords, first ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_mask_popcount(const uint32_t* a, const uint32_t* b, uint64_t nwords,
                                 unsigned long long* out, cudaStream_t s) {
  mask_popcount<<<grid_for(nwords), 256, 0, s>>>(a, b, nwords, out);
  return cudaGetLastError();
}

cudaError_t launch_chunk_bases(const uint32_t* mask, const ChunkDesc* chunks, uint64_t n_ch,
                               uint32_t C, uint64_t N, uint32_t* counts, uint64_t* cbase,
                               cudaStream_t s) {
  uint64_t grid = (n_ch + 7) / 8;
  const uint64_t cap = (uint64_t)num_sms() * 8;
  if (grid > cap) grid = cap;
  chunk_counts<<<(unsigned)(grid ? grid : 1), 256, 0, s>>>(mask, chunks, n_ch, C, N, counts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  chunk_scan<<<1, 1024, 0, s>>>(counts, n_ch, cbase);
  return cudaGetLastError();
}

}  // namespace scape

// ---- unpack: dense[idx[r]] = vals[r] ----------------------------------------

#include <cstdarg>
#include <cstdio>

#include "../../include/scape.h"

namespace scape {
namespace {

__global__ __launch_bounds__(256) void unpack_kernel(const uint32_t* __restrict__ idx,
                                                     const float* __restrict__ vals, uint64_t K,
                                                     float* __restrict__ dense, uint64_t N,
                                                     uint32_t* __restrict__ bad) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t r = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; r < K; r += stride) {
    const uint32_t i = idx[r];
    if (i < N) dense[i] = vals[r];
    else if (bad) atomicAdd(bad, 1u);  // out-of-range coordinate: skipped and counted
  }
}

int unpack_fail(int code, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  set_thread_error(buf);
  return code;
}

}  // namespace
}  // namespace scape

extern "C" __attribute__((visibility("default"))) int scape_unpack(
    const uint32_t* idx, const float* vals, uint64_t K, float* dense, uint64_t N,
    uint32_t* bad_count, void* stream) {
  using namespace scape;
  if (K == 0) return SCAPE_OK;
  if (!idx || !vals || !dense || N == 0)
    return unpack_fail(SCAPE_EINVAL, "idx, vals and dense must be device pointers, N > 0");
  uint64_t grid = (K + 255) / 256;
  const uint64_t cap = (uint64_t)num_sms() * 8;
  if (grid > cap) grid = cap;
  unpack_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(idx, vals, K, dense,
                                                                               N, bad_count);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SCAPE_OK
                          : unpack_fail(SCAPE_ECUDA, "unpack: %s", cudaGetErrorString(e));
}
