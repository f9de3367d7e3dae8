/*
 * libscape — the SCAPE sparse-communication optimizer step on one GPU
 * (sm_103a), as a C ABI.
 *
 * Method: "SCAPE: Accurate and Efficient LLM Training with Extreme Sparse
 * Communication" (arXiv 2607.01678) — abstract; gist.science technical
 * summary §2 "Methodology" (AdamS base optimizer; partitioned mask
 * synchronization; delayed mask usage; single-buffer second-moment
 * reconstruction; packed single-bit masks).  W data-parallel workers are
 * emulated as W gradient replicas in one GPU's memory; the all-reduce of the
 * sparse buffer becomes a fixed-order sum and the all-gather of the shard
 * masks becomes their concatenation in one bitmap.
 *
 * One step t, per coordinate i and worker w (fp32, no fused multiply-add):
 *   u_w   = b1*u_w + (1-b1)*g_w
 *   a_w   = e_w + u_w
 *   b_w   = M_{t-1}[i] ? a_w : +0          (mask built at step t-1)
 *   e_w   = a_w - b_w
 *   bbar  = (b_0 + b_1 + ... + b_{W-1}) * (1/W)   (left to right)
 *   v     = b2*v + (1-b2)*(bbar*bbar)
 *   theta = theta - lr*(bbar/(sqrt(v)+eps) + wd*theta)
 * then M_t: the flat vector is cut into chunks of C coordinates; worker w owns
 * chunks [w*q, (w+1)*q), q = ceil(n_chunks/W), and in each of them keeps the
 * k_c = floor(density*len_c) coordinates of largest |a_w| (as fp32 bits with
 * the sign cleared), equal keys going to the lower index.  Every chunk thus
 * carries exactly k_c coordinates and K = sum_c k_c values are exchanged per
 * worker per step.  At step 0, M_{-1} is this selection applied to the step-0
 * accumulators (before anything is written).
 *
 * Conventions for every entry point:
 *   - Return value: SCAPE_OK (0) or a negative SCAPE_E* code; the handle's
 *     message (scape_last_error) says what failed.  Argument errors are found
 *     before anything is enqueued; SCAPE_ECUDA reports a CUDA runtime error.
 *   - "stream" is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  scape_step* only enqueue work on it and return; readers
 *     (scape_mask, scape_read_*) first wait for the last step's stream.
 *     Consecutive steps of one handle must run in order: on one stream, or
 *     on streams the caller orders (each step reads what the previous one
 *     wrote; the library adds no wait between them).  A step is not meant to
 *     be captured into a CUDA graph and replayed: the handle's host-side
 *     state (which mask buffer is M_{t-1}, the step count) advances once per
 *     call, not per replay.
 *   - Pointers documented as "host or device" may be either (copies use
 *     cudaMemcpyDefault under unified addressing).
 *   - A handle is not thread-safe; separate handles are independent.
 *   - Limits: 1 <= W <= 64; 0 < density <= 1; chunk a multiple of 32 in
 *     [32, 65536]; 0 < N < 2^32.
 */
#ifndef SCAPE_H
#define SCAPE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct scape_handle scape_handle; /* opaque, owned by the library */

/* Flat parameter layout: the concatenation of n_tensors tensors of numel[]
 * coordinates (N = sum numel).  Chunks tile the flat vector and ignore tensor
 * boundaries, unless scape_create_ex is given SCAPE_CHUNK_PER_TENSOR.  numel
 * is read during scape_create only. */
typedef struct {
  uint32_t n_tensors;
  const uint64_t* numel;
  uint32_t chunk;
} scape_layout;

enum {
  SCAPE_OK = 0,
  SCAPE_EINVAL = -1, /* bad argument */
  SCAPE_ENOMEM = -2, /* device or host allocation failed */
  SCAPE_ECUDA = -3,  /* CUDA runtime error (message has the CUDA error string) */
  SCAPE_ESTATE = -4  /* call not valid in the handle's state (e.g. no mask yet) */
};

/* State fields for scape_read_state / scape_load_state. Element types:
 * THETA, V, U, E: fp32; MASK: uint32 words (bit j of word i = coordinate
 * 32i+j); STEP: one int64 (the step counter t). */
enum { SCAPE_THETA = 0, SCAPE_V = 1, SCAPE_U = 2, SCAPE_E = 3, SCAPE_MASK = 4, SCAPE_STEP = 5 };

/* Kernel phases reported by scape_profile_read. */
enum {
  SCAPE_PH_SELECT_BOOT = 0,     /* step 0 only: M_{-1} from the step-0 accumulators */
  SCAPE_PH_STEP = 1,            /* the fused step: every rule line, chunk by chunk, incl. M_t */
  SCAPE_PH_SELECT_FALLBACK = 2, /* standalone top-k of chunks with too many tied keys */
  SCAPE_PH_H2D = 3,             /* scape_step_host: host -> device gradient copies */
  SCAPE_N_PHASES = 4
};

/* Options of scape_create_ex (bitwise OR). */
enum {
  /* Chunks tile every tensor separately ("partitioned layers", gist.science
   * technical summary §2): tensor t is cut into ceil(numel_t / C) chunks, its
   * last one shorter, k_c = floor(density * len_c) each.  Every tensor but the
   * last must hold a multiple of 32 coordinates (chunks own whole mask words). */
  SCAPE_CHUNK_PER_TENSOR = 1u,
  /* The residuals e_w live in page-locked host memory (cudaHostAlloc, mapped)
   * instead of HBM, read and written by the step kernel in place over the
   * CPU-GPU link: W*N*4 bytes less device memory, at the link's bandwidth.
   * The SCAPE pages offload residual buffers to CPU memory (technical summary
   * §2 "Memory Optimization", §4). */
  SCAPE_RESIDUAL_HOST = 2u,
  /* The non-partitioned alternative that SCAPE replaces (technical summary
   * §2 "Partitioned Mask Synchronization"): in every chunk each worker keeps
   * the top-k_c of its own |a_w| (same key and tie rule) and M_t is the union
   * of the W selections, so a chunk keeps between k_c and min(len, W * k_c)
   * coordinates ("fill-in").  The compact buffers then hold as many values
   * per worker as the applied mask has bits: K of scape_info and the total
   * of scape_read_sparse change from step to step (at most
   * sum_c min(len_c, W * k_c), which the buffers are sized for).  A loaded
   * mask must keep between k_c and min(len, W * k_c) bits per chunk. */
  SCAPE_UNION_MASK = 4u
};

typedef struct {
  uint64_t N;          /* coordinates */
  uint32_t W;          /* emulated workers */
  uint32_t chunk;      /* C */
  uint64_t n_chunks;   /* ceil(N / C); with SCAPE_CHUNK_PER_TENSOR the sum over tensors */
  uint64_t chunks_per_worker; /* q */
  uint32_t k_full;     /* k of a full chunk */
  uint32_t k_last;     /* k of the last chunk */
  uint64_t K;          /* values per worker per step (SCAPE_UNION_MASK: in the last step) */
  uint64_t mask_words; /* ceil(N / 32) */
  int64_t step;        /* steps taken (t) */
  uint64_t device_bytes; /* device memory held by the handle */
  uint64_t select_fallbacks; /* chunks (over all steps) whose top-k the standalone select
                                redid because their threshold bucket held too many ties */
  uint32_t flags;      /* scape_create_ex options */
  uint64_t host_bytes; /* page-locked host memory held (SCAPE_RESIDUAL_HOST) */
  /* Debug builds (libscape_debug.so, compiled with SCAPE_DEBUG_CHECKS) check in
   * the kernels every index that depends on the applied mask carrying exactly
   * k_c bits per chunk; a failed check skips the access and is recorded here.
   * Release builds report checks_compiled = 0 and zeros. */
  uint32_t checks_compiled;
  uint32_t check_code;  /* first failed check (0 = none) */
  uint32_t check_count; /* failed checks so far */
  uint64_t check_where; /* coordinate of the first failure */
} scape_info_t;

/* Create a handle: computes the chunk/shard table, allocates all state on the
 * current CUDA device (theta, v: N fp32; u, e: W x N fp32; two N-bit masks;
 * K-entry compact buffers) and zeroes it.  Set theta with scape_load_state.
 * On failure *out is NULL and nothing is leaked.  For tests of that path,
 * SCAPE_TEST_FAIL_ALLOC=n in the environment makes the n-th (0-based) device
 * allocation of each create fail with SCAPE_ENOMEM. */
int scape_create(const scape_layout* layout, int W, double density, float beta1, float beta2,
                 float lr, float wd, float eps, scape_handle** out);

/* scape_create with options (SCAPE_CHUNK_PER_TENSOR, SCAPE_RESIDUAL_HOST,
 * SCAPE_UNION_MASK, combinable);
 * flags = 0 is scape_create.  k_full and k_last of scape_info are then
 * floor(density * C) and the last chunk's k. */
int scape_create_ex(const scape_layout* layout, int W, double density, float beta1, float beta2,
                    float lr, float wd, float eps, uint32_t flags, scape_handle** out);

/* One optimizer step.  grad_ptrs: HOST array of W DEVICE pointers, each to N
 * bf16 gradients (16-byte aligned), borrowed read-only until the step has
 * completed on "stream".  Enqueues the step's kernels and returns. */
int scape_step(scape_handle* h, const void* const* grad_ptrs, void* stream);

/* The same step from HOST gradients: W host pointers to N bf16 each,
 * borrowed until the step has completed on "stream".  Page-locked buffers
 * (cudaHostAlloc / cudaHostRegister, 16-byte aligned) are read by the step
 * kernel in place over the CPU-GPU link: no copy, no staging buffer.  Other
 * host memory is first copied (cudaMemcpyAsync per worker) into a W x N bf16
 * device staging buffer that the first such call allocates and the handle
 * owns.  Enqueues the work on "stream" and returns. */
int scape_step_host(scape_handle* h, const void* const* host_grad_ptrs, void* stream);

/* Copy M_t, the mask built by the last step (applied at the next one), into
 * out_bits (mask_words uint32, host or device).  Waits for the last step.
 * SCAPE_ESTATE before the first step (unless a mask was loaded). */
int scape_mask(scape_handle* h, uint32_t* out_bits);

/* Stream-ordered copy of M_t into out_bits (mask_words uint32, host or
 * device; page-locked host memory lets the copy overlap other work).  The
 * copy is enqueued on "stream" after everything already enqueued on the last
 * step's stream, and the call returns at once.  out_bits is written when
 * "stream" reaches the copy and must stay valid until then.  Later steps may
 * be enqueued at once: a step that would overwrite the buffer being read
 * (every second step reuses it) first waits, on the GPU, for the copy; the
 * synchronous readers, scape_load_state and scape_destroy wait for it on the
 * host.  So the read-back of step t's mask runs while step t+1 runs.
 * SCAPE_ESTATE before the first step (unless a mask was loaded); CUDA
 * failures give SCAPE_ECUDA. */
int scape_mask_async(scape_handle* h, uint32_t* out_bits, void* stream);

/* Free everything the handle owns (waits for its last step). NULL is a no-op. */
void scape_destroy(scape_handle* h);

/* Sizes and counters of the handle (waits for the last step). */
int scape_info(const scape_handle* h, scape_info_t* out);

/* Copy elements [offset, offset+count) of a state field (worker w for U and
 * E; ignored otherwise) to dst (host or device).  MASK counts words and gives
 * M_t; STEP copies one int64 (offset 0, count 1).  Waits for the last step. */
int scape_read_state(scape_handle* h, int which, int w, void* dst, uint64_t offset,
                     uint64_t count);

/* Overwrite elements [offset, offset+count) of a state field from src (host
 * or device).  A MASK load must cover all words and carry exactly k_c bits in
 * every chunk (checked; SCAPE_EINVAL otherwise); it becomes the mask the next
 * step applies, so that step does no step-0 selection.  STEP sets t.
 * (SCAPE_TEST_SKIP_MASK_CHECK=1 in the environment skips the mask check; it
 * exists for tests of the debug build's kernel checks.) */
int scape_load_state(scape_handle* h, int which, int w, const void* src, uint64_t offset,
                     uint64_t count);

/* The last step's compact buffers, in ascending coordinate order: w in [0,W)
 * gives worker w's kept values b_w, w = -1 the synchronized buffer bbar.
 * Copies entries [offset, offset+count) to idx (uint32 coordinates, may be
 * NULL) and vals (fp32, may be NULL), host or device; *total (may be NULL)
 * receives K.  SCAPE_ESTATE before the first step. */
int scape_read_sparse(scape_handle* h, int w, uint32_t* idx, float* vals, uint64_t offset,
                      uint64_t count, uint64_t* total);

/* Message of the handle's last error ("" if none).  Valid until the next call
 * on the handle.  h == NULL gives the message of the last failure, on this
 * thread, of a call that has no handle: scape_create, scape_create_ex,
 * scape_unpack, scape_dense_adams_step, scape_step_noalloc. */
const char* scape_last_error(const scape_handle* h);

/* enable != 0: every later step records CUDA events around each kernel phase
 * on its stream (no extra synchronisation). enable == 0 stops recording. */
int scape_profile(scape_handle* h, int enable);

/* Sum of the recorded phase durations in ms (ms[SCAPE_N_PHASES]) and the
 * number of recorded launches of each (launches[SCAPE_N_PHASES]); waits for
 * the recorded events, then clears the record. */
int scape_profile_read(scape_handle* h, double* ms, uint32_t* launches);

/* ---- Mask diagnostics -------------------------------------------------------
 * Two properties the SCAPE pages build on (gist.science technical summary
 * §2): the top-k structure of the first moment is stable from one step to the
 * next (which is what lets the mask be used one step late), and letting every
 * worker select over the whole vector instead of its own shard "fills in" the
 * global mask as W grows.  After a step:
 *   kept              = |M_t| (= K)
 *   overlap_prev      = |M_t AND M_{t-1}|: coordinates kept two steps running
 *   union_global_topk = | OR_w S_w |, S_w = worker w's own top-k_c of |a_w| in
 *                       EVERY chunk (not only its shard), from the same
 *                       accumulators; the partitioned rule keeps K of them.
 * Waits for the last step; the first call allocates 2 masks of diagnostics
 * buffers on the device (freed with the handle).  SCAPE_ESTATE before the
 * first step. */
typedef struct {
  uint64_t kept;
  uint64_t overlap_prev;
  uint64_t union_global_topk;
} scape_mask_stats_t;

int scape_mask_stats(scape_handle* h, scape_mask_stats_t* out);

/* ---- Unpack ------------------------------------------------------------------
 * The receiving side of a compact buffer (the single synchronized sparse
 * buffer of SCAPE, gist.science technical summary §2; the pages pack masks and
 * values with dedicated kernels, §2 "Memory Optimization"): scatter
 *   dense[idx[r]] = vals[r]   for r in [0, K)
 * into a dense fp32 vector of N coordinates; coordinates not listed are left
 * as they are (clear dense first for a dense copy of b_w or bbar).  idx, vals
 * (K entries, e.g. from scape_read_sparse) and dense are DEVICE pointers owned
 * by the caller; idx entries >= N are skipped and counted into *bad_count (a
 * DEVICE uint32, may be NULL).  Allocates nothing; enqueues one kernel on
 * "stream" and returns.  K = 0 is a no-op. */
int scape_unpack(const uint32_t* idx, const float* vals, uint64_t K, float* dense, uint64_t N,
                 uint32_t* bad_count, void* stream);

/* ---- Dense AdamS baseline --------------------------------------------------
 * The comparator of the SCAPE pages ("3.26x speedup per step compared to
 * dense AdamS": abstract; gist.science technical summary §4): dense data
 * parallelism, where every worker's full gradient is averaged (the dense
 * all-reduce, here a fixed-order sum over the W replicas) and one AdamS update
 * follows on every coordinate:
 *   gbar = (g_0 + ... + g_{W-1}) * (1/W);  m = b1*m + (1-b1)*gbar;
 *   v = b2*v + (1-b2)*(m*m);  theta = theta - lr*(m/(sqrt(v)+eps) + wd*theta)
 * (fp32, no fused multiply-add, correctly rounded sqrt and /).
 * theta, m, v: N fp32 each, DEVICE, 16-byte aligned, caller-owned and updated
 * in place.  grad_ptrs: HOST array of W DEVICE pointers to N bf16 each
 * (16-byte aligned), read-only.  Allocates nothing; enqueues one kernel on
 * "stream" and returns.  SCAPE_EINVAL on bad arguments (message from
 * scape_last_error(NULL)), SCAPE_ECUDA on a launch error. */
int scape_dense_adams_step(float* theta, float* m, float* v, const void* const* grad_ptrs, int W,
                           uint64_t N, float beta1, float beta2, float lr, float wd, float eps,
                           void* stream);

/* ---- Allocation-free step ------------------------------------------------
 * The SCAPE pages have no counterpart to this entry point; it exists for
 * callers that may not call cudaMalloc: programs whose device memory is all
 * owned by another allocator (a framework's caching pool, a fixed arena
 * handed out at start-up) and programs that must not allocate inside their
 * step loop because cudaMalloc can synchronise the device and changes the
 * memory footprint they budgeted for.  Such a caller owns every buffer of
 * the optimizer state and passes them in; the library allocates nothing.
 *
 * Buffers (all DEVICE pointers, 16-byte aligned, owned by the caller):
 *   theta, v        N fp32 each
 *   u, e            W rows of N fp32, row w starting at w * row_stride
 *                   (row_stride a multiple of 4, >= N rounded up to 4)
 *   mask_prev       M_{t-1}: ceil(N/32) words, bit j of word i = coordinate 32i+j
 *   mask_next       M_t is written here (ceil(N/32) words; must differ from mask_prev)
 *   vals            W rows of K fp32 (row stride vals_stride >= K): kept values
 *   bbar, idx       K fp32 / K uint32: synchronized buffer and its coordinates
 * K = sum over chunks of floor(density * chunk length), as scape_info gives.
 * The step is the partitioned rule on flat chunks (scape_create with no
 * options): no per-tensor chunks, host-resident residuals or union variant.
 * first_step != 0 means there is no M_{t-1} yet: the call first writes the
 * step-0 mask into mask_prev, as scape_step does on a new handle.  Between
 * calls the caller swaps mask_prev and mask_next.
 *
 * Every buffer and gradient pointer must be device (or managed) memory of
 * the current device; a host, freed or foreign pointer -> SCAPE_EINVAL
 * (checked with cudaPointerGetAttributes before anything is enqueued).
 *
 * Scratch: the step needs one flag per chunk and a counter.  They live in a
 * static device array inside the library, sized for at most 65536 chunks
 * (256 KiB), which every GPU that loads the library holds until the process
 * exits.  More chunks -> SCAPE_EINVAL.  The array keeps the last call's
 * contents: a call that completes leaves every flag clear again (the
 * standalone select clears each flag it handles).  All calls share the one
 * array, so calls whose work overlaps on the GPU (different streams without
 * ordering, or several threads) race on it: order them on one stream.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress), clears the whole array (cudaMemsetAsync on
 * "stream", then cudaStreamSynchronize) and sets the kernel's shared-memory
 * limit; make that first call before any stream capture.  No call allocates
 * device or pinned memory, and nothing calls cudaMalloc, cudaFree or an
 * allocating library routine.
 *
 * Returns SCAPE_OK or SCAPE_EINVAL / SCAPE_ECUDA; the message is available
 * from scape_last_error(NULL) on the calling thread.  The work is enqueued on
 * "stream" and the call returns. */
typedef struct {
  const scape_layout* layout;
  int W;
  double density;
  float beta1, beta2, lr, wd, eps;
  float* theta;
  float* v;
  float* u;
  float* e;
  uint64_t row_stride;
  uint32_t* mask_prev;
  uint32_t* mask_next;
  float* vals;
  uint64_t vals_stride;
  float* bbar;
  uint32_t* idx;
  int first_step;
} scape_step_buffers;

int scape_step_noalloc(const scape_step_buffers* buffers, const void* const* grad_ptrs,
                       void* stream);

#ifdef __cplusplus
}
#endif

#endif
