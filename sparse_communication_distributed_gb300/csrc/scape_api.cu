// Host side of libscape: argument checks, the chunk/shard table, device
// allocation, the launch sequence of one step and state read-back.  The
// operations are documented in include/scape.h.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/scape.h"
#include "scape_kernels.cuh"

#define SCAPE_API extern "C" __attribute__((visibility("default")))

namespace scape {
// SM count of the current device (cached per device).
int num_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 152;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace scape

using namespace scape;

struct scape_handle {
  // geometry
  uint64_t N = 0, Np = 0, mask_words = 0, mask_alloc = 0;
  uint32_t C = 0;
  int W = 0;
  double density = 0;
  uint64_t n_ch = 0, q = 0, K = 0, Kp = 0;
  uint32_t k_full = 0, k_last = 0;
  // hyper-parameters (fp32, as used)
  float b1 = 0, b2 = 0, lr = 0, wd = 0, eps = 0, c1 = 0, c2 = 0, invW = 0;
  // device state
  float *theta = nullptr, *v = nullptr, *u = nullptr, *e = nullptr;
  float *vals = nullptr, *bbar = nullptr;
  uint32_t* idx = nullptr;
  uint32_t* mask[2] = {nullptr, nullptr};
  uint32_t* fallback = nullptr;    // per chunk, see k_fused.cu
  uint32_t* n_fallback = nullptr;  // chunks redone by the standalone select (running total)
  uint32_t* dbg = nullptr;         // check-failure record of debug builds (4 words)
  uint32_t* pending = nullptr;     // two counters of flagged chunks, used in turn by the
  uint32_t launches = 0;           // step-kernel launches (launch i counts into slot i % 2)
  uint16_t* stage = nullptr;  // scape_step_host staging, W x N bf16
  uint32_t* diag = nullptr;   // scape_mask_stats: two masks + 3 counters (first use)
  uint32_t flags = 0;         // SCAPE_CHUNK_PER_TENSOR | SCAPE_RESIDUAL_HOST | SCAPE_UNION_MASK
  // union variant: packed base of every chunk of mask[b] (n_ch + 1 entries;
  // the last is the mask's total) and the per-chunk counts behind it
  uint64_t* cbase[2] = {nullptr, nullptr};
  uint32_t* ccount = nullptr;
  std::vector<ChunkDesc> chunks;     // chunk table (host copy, every mode)
  ChunkDesc* chunks_dev = nullptr;   // device copy, per-tensor mode only
  uint64_t host_bytes = 0;           // page-locked host memory held (residuals)
  int n_allocs = 0, fail_alloc = -1;  // allocation count, injected failure (tests)
  int prev = 0;               // mask[prev] = M_{t-1} for the next step
  bool has_mask = false;      // a mask exists (built by a step or loaded)
  bool stepped = false;       // compact buffers hold a step's output
  int64_t t = 0;
  cudaStream_t last_stream = nullptr;
  uint64_t device_bytes = 0;
  // profiling
  bool profiling = false;
  // scape_mask_async: per mask buffer, the event after its last enqueued read
  // and whether a step must still wait for it before overwriting the buffer
  cudaEvent_t ev_written = nullptr, ev_read[2] = {nullptr, nullptr};
  bool read_pending[2] = {false, false};
  std::vector<cudaEvent_t> ev_pool;
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> ev_rec;
  std::string err;
};

namespace {

thread_local std::string g_create_err;

int fail(scape_handle* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->err = buf; else g_create_err = buf;
  return code;
}

int cuda_fail(scape_handle* h, cudaError_t e, const char* what) {
  return fail(h, SCAPE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Fault injection for tests: with SCAPE_TEST_FAIL_ALLOC=n in the environment,
// the n-th device allocation (0-based) of each scape_create reports
// cudaErrorMemoryAllocation without calling cudaMalloc.
int fail_alloc_at() {
  const char* v = std::getenv("SCAPE_TEST_FAIL_ALLOC");
  return v ? std::atoi(v) : -1;
}

template <class T>
cudaError_t dalloc(scape_handle* h, T** p, uint64_t count) {
  const uint64_t bytes = (count ? count : 1) * sizeof(T);
  if (h->n_allocs++ == h->fail_alloc) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), bytes);
  if (e == cudaSuccess) {
    h->device_bytes += bytes;
    e = cudaMemset(*p, 0, bytes);
  }
  return e;
}

void release(scape_handle* h) {
  void* ps[] = {h->theta, h->v, h->u, h->vals, h->bbar, h->idx, h->mask[0], h->mask[1],
                h->fallback, h->n_fallback, h->stage, h->diag, h->chunks_dev, h->dbg,
                h->pending, h->cbase[0], h->cbase[1], h->ccount};
  for (void* p : ps)
    if (p) cudaFree(p);
  if (h->e) {
    if (h->flags & SCAPE_RESIDUAL_HOST) cudaFreeHost(h->e);
    else cudaFree(h->e);
  }
  for (cudaEvent_t ev : {h->ev_written, h->ev_read[0], h->ev_read[1]})
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : h->ev_pool) cudaEventDestroy(ev);
  for (auto& r : h->ev_rec) {
    cudaEventDestroy(r.second.first);
    cudaEventDestroy(r.second.second);
  }
}

cudaEvent_t get_event(scape_handle* h) {
  if (!h->ev_pool.empty()) {
    cudaEvent_t ev = h->ev_pool.back();
    h->ev_pool.pop_back();
    return ev;
  }
  cudaEvent_t ev = nullptr;
  cudaEventCreate(&ev);
  return ev;
}

// Records an event pair around one phase when profiling.
struct PhaseTimer {
  scape_handle* h;
  int ph;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  PhaseTimer(scape_handle* h_, int ph_, cudaStream_t s_) : h(h_), ph(ph_), s(s_) {
    if (h->profiling) {
      a = get_event(h);
      cudaEventRecord(a, s);
    }
  }
  void done() {
    if (a) {
      cudaEvent_t b = get_event(h);
      cudaEventRecord(b, s);
      h->ev_rec.push_back({ph, {a, b}});
      a = nullptr;
    }
  }
};

bool is_field(int which) { return which >= SCAPE_THETA && which <= SCAPE_STEP; }

// Waits for the last step and for every mask read still in flight.
cudaError_t wait_last(scape_handle* h) {
  cudaError_t e = h->last_stream ? cudaStreamSynchronize(h->last_stream) : cudaDeviceSynchronize();
  for (int b = 0; b < 2 && e == cudaSuccess; b++)
    if (h->read_pending[b]) {
      e = cudaEventSynchronize(h->ev_read[b]);
      if (e == cudaSuccess) h->read_pending[b] = false;
    }
  return e;
}

// Checks that a 0/1 bitmap (host copy) carries exactly k_c bits in every chunk
// (in the union variant between k_c and min(len, W * k_c)) and none past N.
bool mask_valid(const scape_handle* h, const std::vector<uint32_t>& m, std::string& why) {
  const bool uni = (h->flags & SCAPE_UNION_MASK) != 0;
  for (uint64_t c = 0; c < h->n_ch; c++) {
    const ChunkDesc& d = h->chunks[c];
    const uint64_t w0 = d.start / 32;
    const uint64_t nw = (d.len + 31) / 32;
    uint64_t cnt = 0;
    for (uint64_t j = 0; j < nw; j++) {
      uint32_t word = m[w0 + j];
      if (j == nw - 1 && (d.len & 31)) word &= (1u << (d.len & 31)) - 1u;
      cnt += __builtin_popcount(word);
    }
    const uint64_t hi = uni ? std::min<uint64_t>(d.len, (uint64_t)h->W * d.k) : d.k;
    if (cnt < d.k || cnt > hi) {
      why = "chunk " + std::to_string(c) + " has " + std::to_string(cnt) + " bits, needs " +
            (uni ? "between " + std::to_string(d.k) + " and " + std::to_string(hi)
                 : std::to_string(d.k));
      return false;
    }
  }
  if (h->N % 32) {
    const uint32_t tail = m[h->mask_words - 1] >> (h->N % 32);
    if (tail) {
      why = "bits set past the last coordinate";
      return false;
    }
  }
  return true;
}

}  // namespace

namespace scape {
// Sets the message scape_last_error(NULL) returns on this thread.
void set_thread_error(const char* msg) { g_create_err = msg; }
}  // namespace scape

SCAPE_API int scape_create_ex(const scape_layout* layout, int W, double density, float beta1,
                              float beta2, float lr, float wd, float eps, uint32_t flags,
                              scape_handle** out) {
  if (!out) return fail(nullptr, SCAPE_EINVAL, "out is NULL");
  *out = nullptr;
  if (!layout || !layout->numel || layout->n_tensors == 0)
    return fail(nullptr, SCAPE_EINVAL, "layout must list at least one tensor");
  if (W < 1 || W > kMaxW) return fail(nullptr, SCAPE_EINVAL, "W=%d outside [1, %d]", W, kMaxW);
  if (!(density > 0.0 && density <= 1.0))
    return fail(nullptr, SCAPE_EINVAL, "density %g outside (0, 1]", density);
  const uint32_t C = layout->chunk;
  if (C < 32 || C > kMaxChunk || C % 32)
    return fail(nullptr, SCAPE_EINVAL, "chunk %u must be a multiple of 32 in [32, %u]", C,
                kMaxChunk);
  uint64_t N = 0;
  for (uint32_t i = 0; i < layout->n_tensors; i++) {
    if (layout->numel[i] > (1ull << 32)) return fail(nullptr, SCAPE_EINVAL, "tensor too large");
    N += layout->numel[i];
    if (N >= (1ull << 32)) break;  // rejected below; stops the sum before it can wrap
  }
  if (N == 0 || N >= (1ull << 32))
    return fail(nullptr, SCAPE_EINVAL, "N=%llu must be in [1, 2^32)", (unsigned long long)N);
  if (!std::isfinite(beta1) || !std::isfinite(beta2) || !std::isfinite(lr) ||
      !std::isfinite(wd) || !(eps > 0.0f) || !std::isfinite(eps))
    return fail(nullptr, SCAPE_EINVAL, "hyper-parameters must be finite and eps > 0");
  if (flags & ~(uint32_t)(SCAPE_CHUNK_PER_TENSOR | SCAPE_RESIDUAL_HOST | SCAPE_UNION_MASK))
    return fail(nullptr, SCAPE_EINVAL, "unknown flags 0x%x", flags);
  if (flags & SCAPE_CHUNK_PER_TENSOR)
    for (uint32_t i = 0; i + 1 < layout->n_tensors; i++)
      if (layout->numel[i] % 32)
        return fail(nullptr, SCAPE_EINVAL,
                    "per-tensor chunks need every tensor but the last to hold a multiple of 32 "
                    "coordinates (tensor %u has %llu)", i, (unsigned long long)layout->numel[i]);

  scape_handle* h = new (std::nothrow) scape_handle();
  if (!h) return fail(nullptr, SCAPE_ENOMEM, "host allocation failed");
  h->fail_alloc = fail_alloc_at();
  h->N = N;
  h->C = C;
  h->W = W;
  h->density = density;
  h->b1 = beta1; h->b2 = beta2; h->lr = lr; h->wd = wd; h->eps = eps;
  h->c1 = 1.0f - beta1;
  h->c2 = 1.0f - beta2;
  h->invW = 1.0f / (float)W;
  h->Np = (N + kTile - 1) / kTile * kTile;
  h->mask_words = (N + 31) / 32;
  h->mask_alloc = h->Np / 32;
  h->flags = flags;
  // chunk table: every C coordinates of the flat vector, or of each tensor
  {
    uint64_t off = 0, base = 0;
    auto add = [&](uint64_t start, uint64_t len) {
      ChunkDesc d;
      d.start = start;
      d.len = (uint32_t)len;
      d.k = (uint32_t)std::floor(density * (double)len);
      d.base = base;
      base += d.k;
      h->chunks.push_back(d);
    };
    if (flags & SCAPE_CHUNK_PER_TENSOR) {
      for (uint32_t t = 0; t < layout->n_tensors; t++) {
        for (uint64_t x = 0; x < layout->numel[t]; x += C)
          add(off + x, std::min<uint64_t>(C, layout->numel[t] - x));
        off += layout->numel[t];
      }
    } else {
      for (uint64_t x = 0; x < N; x += C) add(x, std::min<uint64_t>(C, N - x));
    }
    h->K = base;
  }
  h->n_ch = h->chunks.size();
  h->q = (h->n_ch + W - 1) / W;
  h->k_full = (uint32_t)std::floor(density * (double)C);
  h->k_last = h->chunks.back().k;
  uint64_t kmax = h->K;  // compact values per worker at most
  if (flags & SCAPE_UNION_MASK) {
    kmax = 0;
    for (const ChunkDesc& d : h->chunks) kmax += std::min<uint64_t>(d.len, (uint64_t)W * d.k);
  }
  h->Kp = (kmax + 3) / 4 * 4;

  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = dalloc(h, &h->theta, h->Np);
  if (e == cudaSuccess) e = dalloc(h, &h->v, h->Np);
  if (e == cudaSuccess) e = dalloc(h, &h->u, (uint64_t)W * h->Np);
  if (flags & SCAPE_RESIDUAL_HOST) {
    // residuals in page-locked host memory, read and written by the step
    // kernel in place over the CPU-GPU link
    const uint64_t bytes = (uint64_t)W * h->Np * sizeof(float);
    void* hp = nullptr;
    if (e == cudaSuccess) e = cudaHostAlloc(&hp, bytes, cudaHostAllocMapped);
    if (e == cudaSuccess) {
      void* dp = nullptr;
      std::memset(hp, 0, bytes);
      e = cudaHostGetDevicePointer(&dp, hp, 0);
      if (e == cudaSuccess) {
        h->e = static_cast<float*>(dp);
        h->host_bytes += bytes;
      } else {
        cudaFreeHost(hp);
      }
    }
  } else if (e == cudaSuccess) {
    e = dalloc(h, &h->e, (uint64_t)W * h->Np);
  }
  if (e == cudaSuccess) e = dalloc(h, &h->vals, (uint64_t)W * h->Kp);
  if (e == cudaSuccess) e = dalloc(h, &h->bbar, h->Kp);
  if (e == cudaSuccess) e = dalloc(h, &h->idx, h->Kp);
  if (e == cudaSuccess) e = dalloc(h, &h->mask[0], h->mask_alloc);
  if (e == cudaSuccess) e = dalloc(h, &h->mask[1], h->mask_alloc);
  if (e == cudaSuccess) e = dalloc(h, &h->fallback, h->n_ch);
  if (e == cudaSuccess) e = dalloc(h, &h->n_fallback, 1);
  if (e == cudaSuccess) e = dalloc(h, &h->dbg, 4);
  if (e == cudaSuccess) e = dalloc(h, &h->pending, 2);
  if (flags & SCAPE_UNION_MASK) {
    if (e == cudaSuccess) e = dalloc(h, &h->cbase[0], h->n_ch + 1);
    if (e == cudaSuccess) e = dalloc(h, &h->cbase[1], h->n_ch + 1);
    if (e == cudaSuccess) e = dalloc(h, &h->ccount, h->n_ch);
  }
  if (e == cudaSuccess && (flags & SCAPE_CHUNK_PER_TENSOR)) {
    e = dalloc(h, &h->chunks_dev, h->n_ch);
    if (e == cudaSuccess)
      e = cudaMemcpy(h->chunks_dev, h->chunks.data(), h->n_ch * sizeof(ChunkDesc),
                     cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    const int code = (e == cudaErrorMemoryAllocation) ? SCAPE_ENOMEM : SCAPE_ECUDA;
    fail(nullptr, code, "device allocation of %.3f GB failed: %s",
         (double)h->device_bytes / 1e9, cudaGetErrorString(e));
    cudaGetLastError();
    release(h);
    delete h;
    return code;
  }
  *out = h;
  return SCAPE_OK;
}

SCAPE_API int scape_create(const scape_layout* layout, int W, double density, float beta1,
                           float beta2, float lr, float wd, float eps, scape_handle** out) {
  return scape_create_ex(layout, W, density, beta1, beta2, lr, wd, eps, 0u, out);
}

SCAPE_API void scape_destroy(scape_handle* h) {
  if (!h) return;
  wait_last(h);
  release(h);
  delete h;
}

SCAPE_API const char* scape_last_error(const scape_handle* h) {
  return h ? h->err.c_str() : g_create_err.c_str();
}

// Compact values per worker of the last step: sum_c k_c, or in the union
// variant the count of the mask that step applied (read from the device; the
// caller has waited for the step).
static cudaError_t last_K(const scape_handle* h, uint64_t* K) {
  *K = h->K;
  if (!(h->flags & SCAPE_UNION_MASK)) return cudaSuccess;
  if (!h->stepped) {
    *K = 0;
    return cudaSuccess;
  }
  return cudaMemcpy(K, h->cbase[1 - h->prev] + h->n_ch, sizeof(uint64_t), cudaMemcpyDeviceToHost);
}

SCAPE_API int scape_info(const scape_handle* h, scape_info_t* out) {
  if (!h || !out) return SCAPE_EINVAL;
  out->N = h->N;
  out->W = (uint32_t)h->W;
  out->chunk = h->C;
  out->n_chunks = h->n_ch;
  out->chunks_per_worker = h->q;
  out->k_full = h->k_full;
  out->k_last = h->k_last;
  out->K = h->K;
  out->mask_words = h->mask_words;
  out->step = h->t;
  out->device_bytes = h->device_bytes;
  uint32_t nf = 0;
  scape_handle* hm = const_cast<scape_handle*>(h);
  if (wait_last(hm) != cudaSuccess ||
      cudaMemcpy(&nf, h->n_fallback, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_fail(hm, cudaGetLastError(), "scape_info");
  out->select_fallbacks = nf;
  if (last_K(h, &out->K) != cudaSuccess) return cuda_fail(hm, cudaGetLastError(), "scape_info");
  out->flags = h->flags;
  out->host_bytes = h->host_bytes;
  uint32_t dbg[4] = {0, 0, 0, 0};
  if (cudaMemcpy(dbg, h->dbg, sizeof dbg, cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_fail(hm, cudaGetLastError(), "scape_info");
  out->check_code = dbg[0];
  out->check_count = dbg[1];
  out->check_where = (uint64_t)dbg[2] | ((uint64_t)dbg[3] << 32);
#ifdef SCAPE_DEBUG_CHECKS
  out->checks_compiled = 1;
#else
  out->checks_compiled = 0;
#endif
  return SCAPE_OK;
}

// Arguments of the fused step kernel (normal mode).
static void fill_fused(const scape_handle* h, const uint16_t* const* g, const uint32_t* mprev,
                       uint32_t* mout, FusedArgs& a) {
  a = FusedArgs{};
  for (int w = 0; w < h->W; w++) a.grads[w] = g[w];
  a.u = h->u;
  a.e = h->e;
  a.vals = h->vals;
  a.theta = h->theta;
  a.v = h->v;
  a.bbar = h->bbar;
  a.idx = h->idx;
  a.mprev = mprev;
  a.mout = mout;
  a.fallback = h->fallback;
  a.n_fallback = h->n_fallback;
  a.chunks = h->chunks_dev;
  a.dbg = h->dbg;
  a.N = h->N;
  a.Np = h->Np;
  a.Kp = h->Kp;
  a.n_ch = h->n_ch;
  a.q = h->q;
  a.C = h->C;
  a.k_full = h->k_full;
  a.k_last = h->k_last;
  a.W = h->W;
  a.boot = 0;
  a.e_host = (h->flags & SCAPE_RESIDUAL_HOST) ? 1 : 0;
  a.b1 = h->b1;
  a.c1 = h->c1;
  a.b2 = h->b2;
  a.c2 = h->c2;
  a.lr = h->lr;
  a.wd = h->wd;
  a.eps = h->eps;
  a.invW = h->invW;
  if (h->flags & SCAPE_UNION_MASK) {
    a.union_mask = 1;
    a.cbase = h->cbase[h->prev];  // bases of M_{t-1}
  }
}

// Launch i of the step kernel counts the chunks it flags into pending[i % 2]
// and zeroes the other slot for launch i + 1; the select after launch i-1,
// the only reader of that slot, has finished by then (same stream).  No
// per-step memset is needed.
static void take_pending_slot(scape_handle* h, FusedArgs& a, SelectArgs& sa) {
  const uint32_t i = h->launches++ & 1u;
  a.pending = h->pending + i;
  a.pending_clear = h->pending + (1u - i);
  sa.pending = h->pending + i;
}

static int step_device(scape_handle* h, const uint16_t* const* g, cudaStream_t s) {
  cudaError_t e;
  uint32_t* mprev = h->mask[h->prev];
  uint32_t* mcur = h->mask[1 - h->prev];

  SelectArgs sa{};
  for (int w = 0; w < h->W; w++) sa.grads[w] = g[w];
  sa.e = h->e;
  sa.u = h->u;
  sa.vals = h->vals;
  sa.b1 = h->b1;
  sa.c1 = h->c1;
  sa.N = h->N;
  sa.Np = h->Np;
  sa.Kp = h->Kp;
  sa.n_ch = h->n_ch;
  sa.q = h->q;
  sa.C = h->C;
  sa.k_full = h->k_full;
  sa.k_last = h->k_last;
  sa.chunks = h->chunks_dev;
  sa.dbg = h->dbg;
  const bool uni = (h->flags & SCAPE_UNION_MASK) != 0;
  if (uni) {
    sa.union_mask = 1;
    sa.W = h->W;
    sa.cbase = h->cbase[h->prev];  // keys rebuilt from the compact values on M_{t-1}
  }

  // a mask read enqueued by scape_mask_async on another stream must finish
  // before this step overwrites its buffer (M_t here; M_{-1} too at step 0)
  for (int b = 0; b < 2; b++) {
    const bool written = b == 1 - h->prev || !h->has_mask;
    if (written && h->read_pending[b]) {
      if ((e = cudaStreamWaitEvent(s, h->ev_read[b], 0)) != cudaSuccess)
        return cuda_fail(h, e, "wait for a mask read");
      h->read_pending[b] = false;
    }
  }

  FusedArgs a{};
  if (!h->has_mask) {  // step 0: M_{-1} from the step-0 accumulators
    PhaseTimer pt(h, SCAPE_PH_SELECT_BOOT, s);
    fill_fused(h, g, mprev, mprev, a);
    a.mprev = nullptr;
    a.boot = 1;
    take_pending_slot(h, a, sa);
    if ((e = launch_step_chunks(a, s)) != cudaSuccess) return cuda_fail(h, e, "step-0 mask");
    sa.mprev = nullptr;  // chunks with too many tied keys: the standalone select
    sa.mout = mprev;
    sa.flags = h->fallback;
    if ((e = launch_select(sa, true, s)) != cudaSuccess) return cuda_fail(h, e, "select (step 0)");
    if (uni && (e = launch_chunk_bases(mprev, h->chunks_dev, h->n_ch, h->C, h->N, h->ccount,
                                       h->cbase[h->prev], s)) != cudaSuccess)
      return cuda_fail(h, e, "chunk bases (step 0)");
    pt.done();
  }
  {
    fill_fused(h, g, mprev, mcur, a);
    take_pending_slot(h, a, sa);
    PhaseTimer pt(h, SCAPE_PH_STEP, s);
    if ((e = launch_step_chunks(a, s)) != cudaSuccess) return cuda_fail(h, e, "step kernel");
    pt.done();
  }
  {  // chunks whose threshold bucket overflowed the on-chip candidate list
    sa.mprev = mprev;
    sa.mout = mcur;
    sa.flags = h->fallback;
    PhaseTimer pt(h, SCAPE_PH_SELECT_FALLBACK, s);
    if ((e = launch_select(sa, false, s)) != cudaSuccess) return cuda_fail(h, e, "select (fallback)");
    // union variant: the compact layout of M_t, for the next step
    if (uni && (e = launch_chunk_bases(mcur, h->chunks_dev, h->n_ch, h->C, h->N, h->ccount,
                                       h->cbase[1 - h->prev], s)) != cudaSuccess)
      return cuda_fail(h, e, "chunk bases");
    pt.done();
  }
  h->prev = 1 - h->prev;
  h->has_mask = true;
  h->stepped = true;
  h->t += 1;
  h->last_stream = s;
  return SCAPE_OK;
}

static int check_grad_ptrs(scape_handle* h, const void* const* gp, bool device) {
  if (!gp) return fail(h, SCAPE_EINVAL, "grad_ptrs is NULL");
  for (int w = 0; w < h->W; w++) {
    if (!gp[w]) return fail(h, SCAPE_EINVAL, "grad_ptrs[%d] is NULL", w);
    if (device && (reinterpret_cast<uintptr_t>(gp[w]) & 15))
      return fail(h, SCAPE_EINVAL, "grad_ptrs[%d] is not 16-byte aligned", w);
  }
  return SCAPE_OK;
}

SCAPE_API int scape_step(scape_handle* h, const void* const* grad_ptrs, void* stream) {
  if (!h) return SCAPE_EINVAL;
  int rc = check_grad_ptrs(h, grad_ptrs, true);
  if (rc) return rc;
  std::vector<const uint16_t*> g(h->W);
  for (int w = 0; w < h->W; w++) g[w] = static_cast<const uint16_t*>(grad_ptrs[w]);
  return step_device(h, g.data(), static_cast<cudaStream_t>(stream));
}

// Device-visible address of a page-locked host buffer, or nullptr when the
// buffer is ordinary (pageable) host memory.
static const void* pinned_device_ptr(const void* host) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  return at.devicePointer;
}

SCAPE_API int scape_step_host(scape_handle* h, const void* const* host_grad_ptrs, void* stream) {
  if (!h) return SCAPE_EINVAL;
  int rc = check_grad_ptrs(h, host_grad_ptrs, false);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  std::vector<const uint16_t*> g(h->W);
  // Page-locked buffers: the step kernel reads them in place over the
  // CPU-GPU link (each gradient is read once), no copy and no staging.
  bool direct = true;
  for (int w = 0; w < h->W && direct; w++) {
    const void* d = pinned_device_ptr(host_grad_ptrs[w]);
    if (!d || (reinterpret_cast<uintptr_t>(d) & 15)) direct = false;
    else g[w] = static_cast<const uint16_t*>(d);
  }
  if (direct) return step_device(h, g.data(), s);

  const uint64_t per = (h->N + 7) / 8 * 8;  // keep every worker's slice 16-byte aligned
  if (!h->stage) {
    if ((e = cudaMalloc(&h->stage, (uint64_t)h->W * per * sizeof(uint16_t))) != cudaSuccess) {
      h->stage = nullptr;
      cudaGetLastError();
      return fail(h, e == cudaErrorMemoryAllocation ? SCAPE_ENOMEM : SCAPE_ECUDA,
                  "staging allocation failed: %s", cudaGetErrorString(e));
    }
    h->device_bytes += (uint64_t)h->W * per * sizeof(uint16_t);
  }
  {
    PhaseTimer pt(h, SCAPE_PH_H2D, s);
    for (int w = 0; w < h->W; w++) {
      uint16_t* dst = h->stage + (uint64_t)w * per;
      if ((e = cudaMemcpyAsync(dst, host_grad_ptrs[w], h->N * sizeof(uint16_t),
                               cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(h, e, "gradient copy");
      g[w] = dst;
    }
    pt.done();
  }
  return step_device(h, g.data(), s);
}

SCAPE_API int scape_mask(scape_handle* h, uint32_t* out_bits) {
  if (!h) return SCAPE_EINVAL;
  if (!out_bits) return fail(h, SCAPE_EINVAL, "out_bits is NULL");
  if (!h->has_mask) return fail(h, SCAPE_ESTATE, "no mask before the first step");
  cudaError_t e = wait_last(h);
  if (e == cudaSuccess)
    e = cudaMemcpy(out_bits, h->mask[h->prev], h->mask_words * 4, cudaMemcpyDefault);
  return e == cudaSuccess ? SCAPE_OK : cuda_fail(h, e, "scape_mask");
}

SCAPE_API int scape_mask_async(scape_handle* h, uint32_t* out_bits, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!out_bits) return fail(h, SCAPE_EINVAL, "out_bits is NULL");
  if (!h->has_mask) return fail(h, SCAPE_ESTATE, "no mask before the first step");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (!h->ev_written) e = cudaEventCreateWithFlags(&h->ev_written, cudaEventDisableTiming);
  for (int b = 0; b < 2 && e == cudaSuccess; b++)
    if (!h->ev_read[b]) e = cudaEventCreateWithFlags(&h->ev_read[b], cudaEventDisableTiming);
  const int b = h->prev;  // M_t
  // the copy starts after everything enqueued so far on the last step's stream
  if (e == cudaSuccess && s != h->last_stream) {
    e = cudaEventRecord(h->ev_written, h->last_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_written, 0);
  }
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(out_bits, h->mask[b], h->mask_words * 4, cudaMemcpyDefault, s);
  if (e == cudaSuccess) e = cudaEventRecord(h->ev_read[b], s);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_mask_async");
  h->read_pending[b] = true;
  return SCAPE_OK;
}

static int field_ptr(scape_handle* h, int which, int w, char** base, uint64_t* count,
                     uint64_t* esize) {
  if (!is_field(which)) return fail(h, SCAPE_EINVAL, "unknown state field %d", which);
  if ((which == SCAPE_U || which == SCAPE_E) && (w < 0 || w >= h->W))
    return fail(h, SCAPE_EINVAL, "worker %d outside [0, %d)", w, h->W);
  switch (which) {
    case SCAPE_THETA: *base = (char*)h->theta; *count = h->N; *esize = 4; break;
    case SCAPE_V: *base = (char*)h->v; *count = h->N; *esize = 4; break;
    case SCAPE_U: *base = (char*)(h->u + (uint64_t)w * h->Np); *count = h->N; *esize = 4; break;
    case SCAPE_E: *base = (char*)(h->e + (uint64_t)w * h->Np); *count = h->N; *esize = 4; break;
    case SCAPE_MASK: *base = (char*)h->mask[h->prev]; *count = h->mask_words; *esize = 4; break;
    default: *base = nullptr; *count = 1; *esize = 8; break;
  }
  return SCAPE_OK;
}

SCAPE_API int scape_read_state(scape_handle* h, int which, int w, void* dst, uint64_t offset,
                               uint64_t count) {
  if (!h) return SCAPE_EINVAL;
  if (!dst) return fail(h, SCAPE_EINVAL, "dst is NULL");
  char* base;
  uint64_t n, es;
  int rc = field_ptr(h, which, w, &base, &n, &es);
  if (rc) return rc;
  if (offset > n || count > n - offset) return fail(h, SCAPE_EINVAL, "range outside the field");
  cudaError_t e = wait_last(h);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_read_state");
  if (which == SCAPE_STEP) {
    int64_t t = h->t;
    e = cudaMemcpy(dst, &t, 8, cudaMemcpyDefault);
  } else {
    e = cudaMemcpy(dst, base + offset * es, count * es, cudaMemcpyDefault);
  }
  return e == cudaSuccess ? SCAPE_OK : cuda_fail(h, e, "scape_read_state");
}

SCAPE_API int scape_load_state(scape_handle* h, int which, int w, const void* src, uint64_t offset,
                               uint64_t count) {
  if (!h) return SCAPE_EINVAL;
  if (!src) return fail(h, SCAPE_EINVAL, "src is NULL");
  char* base;
  uint64_t n, es;
  int rc = field_ptr(h, which, w, &base, &n, &es);
  if (rc) return rc;
  if (offset > n || count > n - offset) return fail(h, SCAPE_EINVAL, "range outside the field");
  cudaError_t e = wait_last(h);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_load_state");
  if (which == SCAPE_STEP) {
    int64_t t;
    if ((e = cudaMemcpy(&t, src, 8, cudaMemcpyDefault)) != cudaSuccess)
      return cuda_fail(h, e, "scape_load_state");
    if (t < 0) return fail(h, SCAPE_EINVAL, "step must be >= 0");
    h->t = t;
    return SCAPE_OK;
  }
  if (which == SCAPE_MASK) {
    if (offset != 0 || count != h->mask_words)
      return fail(h, SCAPE_EINVAL, "a mask load must cover all %llu words",
                  (unsigned long long)h->mask_words);
    std::vector<uint32_t> m(count);
    if ((e = cudaMemcpy(m.data(), src, count * 4, cudaMemcpyDefault)) != cudaSuccess)
      return cuda_fail(h, e, "scape_load_state");
    std::string why;
    const char* skip = std::getenv("SCAPE_TEST_SKIP_MASK_CHECK");  // tests of debug checks
    if (!(skip && skip[0] == '1') && !mask_valid(h, m, why))
      return fail(h, SCAPE_EINVAL, "invalid mask: %s", why.c_str());
    if ((e = cudaMemcpy(base, m.data(), count * 4, cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(h, e, "scape_load_state");
    if ((h->flags & SCAPE_UNION_MASK) &&  // the next step's compact layout
        ((e = launch_chunk_bases(h->mask[h->prev], h->chunks_dev, h->n_ch, h->C, h->N, h->ccount,
                                 h->cbase[h->prev], nullptr)) != cudaSuccess ||
         (e = cudaDeviceSynchronize()) != cudaSuccess))
      return cuda_fail(h, e, "scape_load_state");
    h->has_mask = true;
    return SCAPE_OK;
  }
  e = cudaMemcpy(base + offset * es, src, count * es, cudaMemcpyDefault);
  return e == cudaSuccess ? SCAPE_OK : cuda_fail(h, e, "scape_load_state");
}

SCAPE_API int scape_read_sparse(scape_handle* h, int w, uint32_t* idx, float* vals,
                                uint64_t offset, uint64_t count, uint64_t* total) {
  if (!h) return SCAPE_EINVAL;
  if (w < -1 || w >= h->W) return fail(h, SCAPE_EINVAL, "worker %d outside [-1, %d)", w, h->W);
  if (!h->stepped) {
    if (total) *total = (h->flags & SCAPE_UNION_MASK) ? 0 : h->K;
    return fail(h, SCAPE_ESTATE, "no step has run");
  }
  cudaError_t e = wait_last(h);
  uint64_t K = h->K;
  if (e == cudaSuccess) e = last_K(h, &K);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_read_sparse");
  if (total) *total = K;
  if (offset > K || count > K - offset) return fail(h, SCAPE_EINVAL, "range outside [0, K)");
  if (e == cudaSuccess && idx && count)
    e = cudaMemcpy(idx, h->idx + offset, count * 4, cudaMemcpyDefault);
  if (e == cudaSuccess && vals && count) {
    const float* src = w < 0 ? h->bbar : h->vals + (uint64_t)w * h->Kp;
    e = cudaMemcpy(vals, src + offset, count * 4, cudaMemcpyDefault);
  }
  return e == cudaSuccess ? SCAPE_OK : cuda_fail(h, e, "scape_read_sparse");
}

SCAPE_API int scape_profile(scape_handle* h, int enable) {
  if (!h) return SCAPE_EINVAL;
  h->profiling = enable != 0;
  return SCAPE_OK;
}

SCAPE_API int scape_profile_read(scape_handle* h, double* ms, uint32_t* launches) {
  if (!h) return SCAPE_EINVAL;
  if (ms)
    for (int i = 0; i < SCAPE_N_PHASES; i++) ms[i] = 0;
  if (launches)
    for (int i = 0; i < SCAPE_N_PHASES; i++) launches[i] = 0;
  for (auto& r : h->ev_rec) {
    cudaError_t e = cudaEventSynchronize(r.second.second);
    float t = 0;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.second.first, r.second.second);
    if (e != cudaSuccess) return cuda_fail(h, e, "scape_profile_read");
    if (ms) ms[r.first] += t;
    if (launches) launches[r.first] += 1;
    h->ev_pool.push_back(r.second.first);
    h->ev_pool.push_back(r.second.second);
  }
  h->ev_rec.clear();
  return SCAPE_OK;
}

SCAPE_API int scape_mask_stats(scape_handle* h, scape_mask_stats_t* out) {
  if (!h) return SCAPE_EINVAL;
  if (!out) return fail(h, SCAPE_EINVAL, "out is NULL");
  if (!h->stepped) return fail(h, SCAPE_ESTATE, "no step has run");
  cudaError_t e = wait_last(h);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_mask_stats");
  const uint64_t nw = h->mask_alloc;
  if (!h->diag) {
    const uint64_t bytes = (2 * nw + 8) * sizeof(uint32_t);
    if ((e = cudaMalloc(&h->diag, bytes)) != cudaSuccess) {
      h->diag = nullptr;
      cudaGetLastError();
      return fail(h, e == cudaErrorMemoryAllocation ? SCAPE_ENOMEM : SCAPE_ECUDA,
                  "diagnostics allocation failed: %s", cudaGetErrorString(e));
    }
    h->device_bytes += bytes;
    if ((e = cudaMemset(h->diag, 0, bytes)) != cudaSuccess) return cuda_fail(h, e, "memset");
  }
  uint32_t* tmp = h->diag;
  uint32_t* uni = h->diag + nw;
  unsigned long long* cnt = reinterpret_cast<unsigned long long*>(h->diag + 2 * nw);
  cudaStream_t s = h->last_stream;
  const uint32_t* m_new = h->mask[h->prev];       // M_t, built by the last step
  const uint32_t* m_used = h->mask[1 - h->prev];  // M_{t-1}, applied in the last step
  if ((e = cudaMemsetAsync(cnt, 0, 3 * sizeof(unsigned long long), s)) != cudaSuccess)
    return cuda_fail(h, e, "memset");
  SelectArgs sa{};
  sa.e = h->e;
  sa.u = h->u;
  sa.vals = h->vals;
  sa.mprev = m_used;
  sa.b1 = h->b1;
  sa.c1 = h->c1;
  sa.N = h->N;
  sa.Np = h->Np;
  sa.Kp = h->Kp;
  sa.n_ch = h->n_ch;
  sa.q = h->q;
  sa.C = h->C;
  sa.k_full = h->k_full;
  sa.k_last = h->k_last;
  sa.flags = nullptr;
  sa.chunks = h->chunks_dev;
  sa.dbg = h->dbg;
  sa.mout = tmp;
  if (h->flags & SCAPE_UNION_MASK) sa.cbase = h->cbase[1 - h->prev];  // layout of M_{t-1}
  for (int w = 0; w < h->W; w++) {
    sa.rank_worker = w + 1;
    if ((e = launch_select(sa, false, s)) != cudaSuccess) return cuda_fail(h, e, "select");
    if ((e = launch_mask_or(uni, tmp, nw, w == 0, s)) != cudaSuccess)
      return cuda_fail(h, e, "mask_or");
  }
  if ((e = launch_mask_popcount(m_new, nullptr, nw, cnt, s)) != cudaSuccess ||
      (e = launch_mask_popcount(m_new, m_used, nw, cnt + 1, s)) != cudaSuccess ||
      (e = launch_mask_popcount(uni, nullptr, nw, cnt + 2, s)) != cudaSuccess)
    return cuda_fail(h, e, "popcount");
  unsigned long long host[3];
  if ((e = cudaMemcpyAsync(host, cnt, sizeof host, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess)
    return cuda_fail(h, e, "scape_mask_stats");
  out->kept = host[0];
  out->overlap_prev = host[1];
  out->union_global_topk = host[2];
  return SCAPE_OK;
}
