// Kernel interfaces of libscape (internal).
//
// Data layout in HBM (all allocations by the library):
//   theta, v      fp32[Np]            Np = N rounded up to 256
//   u, e          fp32[W][Np]
//   mask[2]       uint32[Np/32]       M_{t-1} / M_t, bit j of word i = coord 32i+j
//   vals          fp32[W][Kp]         compact b_w, ascending coordinate
//   bbar          fp32[Kp]            compact synchronized buffer
//   idx           uint32[Kp]          coordinates of the compact entries
//   fallback      uint32[n_ch]        chunks whose selection the standalone select redoes
//   cbase[2]      uint64[n_ch+1]      union variant: packed base of every chunk of mask[b]
// Chunk c (C coordinates, the last one ragged) keeps exactly k_c coordinates,
// so its kept values start at packed position c * k_full.  In the union
// variant (every worker's own top-k, OR-ed) a chunk keeps between k_c and
// W * k_c, and its base comes from the scan of the mask's per-chunk counts.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace scape {

constexpr int kMaxW = 64;
constexpr int kTile = 256;             // coordinates per warp tile (8 per thread)
constexpr uint32_t kMaxChunk = 65536;  // largest chunk (16-bit in-chunk index)

// One chunk of the per-tensor variant (chunks restart at every tensor).
struct ChunkDesc {
  uint64_t start;  // first coordinate (a multiple of 32)
  uint64_t base;   // packed position of its first kept value
  uint32_t len;    // coordinates
  uint32_t k;      // kept coordinates
};

struct FusedArgs {
  const uint16_t* grads[kMaxW];
  float* u;
  float* e;
  float* vals;
  float* theta;
  float* v;
  float* bbar;
  uint32_t* idx;
  const uint32_t* mprev;
  uint32_t* mout;
  uint32_t* fallback;    // per chunk: 1 = selection left to the standalone select
  uint32_t* n_fallback;  // count of such chunks (diagnostic)
  uint32_t* pending;     // chunks flagged by this launch (zero at its start; may be NULL)
  uint32_t* pending_clear;  // zeroed by the launch (the next launch's counter); may be NULL
  const ChunkDesc* chunks;  // NULL: chunk c = [c*C, c*C + C) of the flat vector
  uint64_t N, Np, Kp, n_ch, q;
  uint32_t C, k_full, k_last;
  int W;
  int boot;  // 1: only build M_{-1} into mout from the step-0 accumulators (no writes)
  int e_host;  // 1: e lives in mapped host memory (whole-sector access mapping)
  int union_mask;  // 1: the non-partitioned variant (mout = union of every worker's top-k)
  const uint64_t* cbase;  // union variant: packed base of each chunk of mprev (n_ch + 1)
  uint32_t* dbg;  // debug builds: check-failure record (4 words), may be NULL
  float b1, c1, b2, c2, lr, wd, eps, invW;
};

struct SelectArgs {
  // key source after the step: e (new residual) and vals of the owner, M_{t-1}
  const float* e;
  const float* vals;
  const uint32_t* mprev;
  // key source at step 0: the accumulator b1*u + c1*g + e, nothing written
  const uint16_t* grads[kMaxW];
  const float* u;
  float b1, c1;
  uint32_t* mout;
  uint32_t* flags;  // NULL: every chunk; else only chunks with flags[c] != 0 (cleared)
  const uint32_t* pending;  // if set and zero, no chunk is flagged: the launch returns at once
  int rank_worker;  // 0: each chunk ranks its owner's accumulator (the SCAPE rule);
                    // w + 1: every chunk ranks worker w's (mask diagnostics)
  int union_mask;   // 1: a chunk's words are the union of every worker's selection
  int W;            // workers (union variant)
  const uint64_t* cbase;  // set: packed base of each chunk of mprev (n_ch + 1; union
                          // variant), else chunk c's values start at c * k_full
  const ChunkDesc* chunks;  // NULL: chunk c = [c*C, c*C + C) of the flat vector
  uint32_t* dbg;            // debug builds: check-failure record (4 words), may be NULL
  uint64_t N, Np, Kp, n_ch, q;
  uint32_t C, k_full, k_last;
};

// Launchers; all enqueue on "s" and return cudaGetLastError().
cudaError_t launch_step_chunks(const FusedArgs& a, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, bool boot, cudaStream_t s);
// acc = first ? m : (acc | m), over nwords words.
cudaError_t launch_mask_or(uint32_t* acc, const uint32_t* m, uint64_t nwords, bool first,
                           cudaStream_t s);
// Union variant: counts[c] = set bits of chunk c of mask, cbase[c] = their
// exclusive prefix over the chunks, cbase[n_ch] = the total.
cudaError_t launch_chunk_bases(const uint32_t* mask, const ChunkDesc* chunks, uint64_t n_ch,
                               uint32_t C, uint64_t N, uint32_t* counts, uint64_t* cbase,
                               cudaStream_t s);
// *out += popcount(a & b) (b may be NULL: popcount(a)), over nwords words.
cudaError_t launch_mask_popcount(const uint32_t* a, const uint32_t* b, uint64_t nwords,
                                 unsigned long long* out, cudaStream_t s);

int num_sms();
void set_thread_error(const char* msg);

}  // namespace scape
