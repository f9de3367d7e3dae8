// scape_step_noalloc: the fused SCAPE step on caller-owned buffers, with no
// device allocation at all.
//
// The fused step kernel needs a little global scratch beyond its inputs and
// outputs: one flag per chunk (chunks whose top-k must be redone by the
// standalone select) and a counter.  A handle gets that scratch from
// cudaMalloc at scape_create.  This entry point instead takes it from the
// file-scope array below, sized for kMaxChunks chunks, which every GPU that
// loads the library holds until the process exits.  Host code cannot use
// the array's name as a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress (with that device current),
// clears the array once and keeps the address.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/scape.h"
#include "scape_kernels.cuh"

#define SCAPE_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr uint64_t kMaxChunks = 65536;  // 256 KiB of flags
constexpr int kMaxDevices = 64;

// [0, kMaxChunks): per-chunk fallback flags; [kMaxChunks]: fallback counter.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kMaxChunks + 64];

std::mutex g_mu;
uint32_t* g_scratch_ptr[kMaxDevices] = {};

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  scape::set_thread_error(buf);
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device (or managed) memory of the current device "dev".  A host pointer, a
// freed pointer or another device's memory would fault the kernels, so it is
// rejected here; the query allocates nothing.  Without a usable CUDA device
// the query itself fails, which is reported the same way.
int check_device_ptr(const void* p, int dev, const char* what) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // the query's error is not sticky; do not leave it behind
    return fail(SCAPE_EINVAL, "%s is not a device pointer (%s)", what, cudaGetErrorString(e));
  }
  const bool ok = at.type == cudaMemoryTypeManaged ||
                  (at.type == cudaMemoryTypeDevice && at.device == dev);
  if (!ok)
    return fail(SCAPE_EINVAL, "%s must be device memory of the current device %d "
                "(memory type %d, device %d)", what, dev, (int)at.type, at.device);
  return SCAPE_OK;
}

}  // namespace

SCAPE_API int scape_step_noalloc(const scape_step_buffers* b, const void* const* grad_ptrs,
                                 void* stream) {
  using namespace scape;
  if (!b || !b->layout || !b->layout->numel || b->layout->n_tensors == 0)
    return fail(SCAPE_EINVAL, "buffers and layout are required");
  const int W = b->W;
  if (W < 1 || W > kMaxW) return fail(SCAPE_EINVAL, "W=%d outside [1, %d]", W, kMaxW);
  if (!(b->density > 0.0 && b->density <= 1.0))
    return fail(SCAPE_EINVAL, "density %g outside (0, 1]", b->density);
  const uint32_t C = b->layout->chunk;
  if (C < 32 || C > kMaxChunk || C % 32)
    return fail(SCAPE_EINVAL, "chunk %u must be a multiple of 32 in [32, %u]", C, kMaxChunk);
  uint64_t N = 0;
  for (uint32_t i = 0; i < b->layout->n_tensors; i++) {
    if (b->layout->numel[i] > (1ull << 32)) return fail(SCAPE_EINVAL, "tensor too large");
    N += b->layout->numel[i];
    if (N >= (1ull << 32)) break;  // rejected below; stops the sum before it can wrap
  }
  if (N == 0 || N >= (1ull << 32)) return fail(SCAPE_EINVAL, "N must be in [1, 2^32)");
  const uint64_t n_ch = (N + C - 1) / C;
  if (n_ch > kMaxChunks)
    return fail(SCAPE_EINVAL, "%llu chunks exceed the %llu this entry point supports",
                (unsigned long long)n_ch, (unsigned long long)kMaxChunks);
  if (!std::isfinite(b->beta1) || !std::isfinite(b->beta2) || !std::isfinite(b->lr) ||
      !std::isfinite(b->wd) || !(b->eps > 0.0f) || !std::isfinite(b->eps))
    return fail(SCAPE_EINVAL, "hyper-parameters must be finite and eps > 0");
  const uint32_t k_full = (uint32_t)std::floor(b->density * (double)C);
  const uint32_t k_last = (uint32_t)std::floor(b->density * (double)(N - (n_ch - 1) * C));
  const uint64_t K = (n_ch - 1) * (uint64_t)k_full + k_last;
  if (b->row_stride < (N + 3) / 4 * 4 || b->row_stride % 4)
    return fail(SCAPE_EINVAL, "row_stride must be a multiple of 4 and >= N rounded up to 4");
  if (b->vals_stride < K) return fail(SCAPE_EINVAL, "vals_stride must be >= K = %llu",
                                      (unsigned long long)K);
  const void* ptrs[] = {b->theta, b->v, b->u, b->e, b->mask_prev, b->mask_next, b->vals,
                        b->bbar, b->idx};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(SCAPE_EINVAL, "every buffer must be a 16-byte aligned device pointer");
  if (b->mask_prev == b->mask_next) return fail(SCAPE_EINVAL, "mask_prev and mask_next must differ");
  if (!grad_ptrs) return fail(SCAPE_EINVAL, "grad_ptrs is NULL");
  for (int w = 0; w < W; w++)
    if (!grad_ptrs[w] || !aligned16(grad_ptrs[w]))
      return fail(SCAPE_EINVAL, "grad_ptrs[%d] must be a 16-byte aligned device pointer", w);

  // every buffer must be memory of the current device (checked before any launch)
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  static const char* const names[] = {"theta", "v", "u", "e", "mask_prev", "mask_next", "vals",
                                      "bbar", "idx"};
  for (int j = 0; j < 9; j++)
    if (int rc = check_device_ptr(ptrs[j], dev, names[j])) return rc;
  for (int w = 0; w < W; w++) {
    char what[32];
    snprintf(what, sizeof what, "grad_ptrs[%d]", w);
    if (int rc = check_device_ptr(grad_ptrs[w], dev, what)) return rc;
  }

  // first call on this device: the device address of the scratch array, and
  // one clear of the whole array (it stays clear: see below)
  if (dev < 0 || dev >= kMaxDevices) return fail(SCAPE_EINVAL, "device %d not supported", dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  uint32_t* scratch;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return fail(SCAPE_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      if ((e = cudaMemsetAsync(p, 0, sizeof(g_noalloc_scratch), s)) != cudaSuccess ||
          (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return fail(SCAPE_ECUDA, "clearing the scratch: %s", cudaGetErrorString(e));
      g_scratch_ptr[dev] = static_cast<uint32_t*>(p);
    }
    scratch = g_scratch_ptr[dev];
  }
  // scratch layout within the array: flags at [0, n_ch), counter at [kMaxChunks].
  // The step kernel sets the flag of a chunk it leaves to the standalone
  // select, and the select clears every flag it handles, so a call that
  // completes leaves the flags clear for the next.  (A call that failed
  // between its launches may leave flags set; the next call then redoes
  // those chunks' selection from the same state, which gives the same mask.)
  // The counter only counts flagged chunks and is never read here.
  uint32_t* flags = scratch;
  uint32_t* counter = scratch + kMaxChunks;

  SelectArgs sa{};
  for (int w = 0; w < W; w++) sa.grads[w] = static_cast<const uint16_t*>(grad_ptrs[w]);
  sa.e = b->e;
  sa.u = b->u;
  sa.vals = b->vals;
  sa.b1 = b->beta1;
  sa.c1 = 1.0f - b->beta1;
  sa.N = N;
  sa.Np = b->row_stride;
  sa.Kp = b->vals_stride;
  sa.n_ch = n_ch;
  sa.q = (n_ch + W - 1) / W;
  sa.C = C;
  sa.k_full = k_full;
  sa.k_last = k_last;
  if (b->first_step) {
    sa.mprev = nullptr;
    sa.mout = b->mask_prev;
    sa.flags = nullptr;
    if ((e = launch_select(sa, true, s)) != cudaSuccess)
      return fail(SCAPE_ECUDA, "select (step 0): %s", cudaGetErrorString(e));
  }
  FusedArgs a{};
  for (int w = 0; w < W; w++) a.grads[w] = sa.grads[w];
  a.u = b->u;
  a.e = b->e;
  a.vals = b->vals;
  a.theta = b->theta;
  a.v = b->v;
  a.bbar = b->bbar;
  a.idx = b->idx;
  a.mprev = b->mask_prev;
  a.mout = b->mask_next;
  a.fallback = flags;
  a.n_fallback = counter;
  a.N = N;
  a.Np = b->row_stride;
  a.Kp = b->vals_stride;
  a.n_ch = n_ch;
  a.q = sa.q;
  a.C = C;
  a.k_full = k_full;
  a.k_last = k_last;
  a.W = W;
  a.b1 = b->beta1;
  a.c1 = 1.0f - b->beta1;
  a.b2 = b->beta2;
  a.c2 = 1.0f - b->beta2;
  a.lr = b->lr;
  a.wd = b->wd;
  a.eps = b->eps;
  a.invW = 1.0f / (float)W;
  if ((e = launch_step_chunks(a, s)) != cudaSuccess)
    return fail(SCAPE_ECUDA, "step kernel: %s", cudaGetErrorString(e));
  sa.mprev = b->mask_prev;
  sa.mout = b->mask_next;
  sa.flags = flags;
  if ((e = launch_select(sa, false, s)) != cudaSuccess)
    return fail(SCAPE_ECUDA, "select (fallback): %s", cudaGetErrorString(e));
  return SCAPE_OK;
}
