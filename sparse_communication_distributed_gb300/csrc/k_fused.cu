// The SCAPE step, one chunk at a time, in one persistent kernel.
//
// SCAPE (arXiv 2607.01678; gist.science technical summary §2) aligns mask
// generation with optimizer sharding: worker w builds the top-k mask only for
// the chunks of its own shard, from its first-moment accumulator, and the mask
// is applied one step later.  Here the chunk is the unit of work: a CTA takes
// chunk c (C coordinates, owner w_c = c / q) and runs every step of the rule on
// it before moving to the next chunk, so each state array is streamed through
// HBM exactly once per step and the selection runs on-chip.
//
// Phases per chunk (one 1024-thread CTA per SM with 188.8 KB of shared memory;
// chunks of at most 16384 coordinates: two 512-thread CTAs per SM):
//  0. load the chunk's words of M_{t-1} and their exclusive popcount prefix:
//     the packed position of a kept coordinate i is
//       base_c + popcount(M_{t-1} bits of the chunk before i),
//     base_c = c * k_full (every earlier chunk keeps exactly k coordinates),
//     or the chunk table's base in the per-tensor variant, where chunks
//     restart at every tensor (each tensor starts on a mask word);
//  1. the owner's streaming pass (momentum, accumulate, mask select, residual,
//     compaction into vals_owner), which also keeps every |a| as a 16-bit
//     truncated key (fp32 bits 30..15) in shared memory and counts its top 12
//     bits in a 4096-bin histogram;
//  2. exact top-k_c of the owner's |a| with ties to the lower index: the
//     histogram gives the 12-bit bin of the k-th largest, a 16-bin pass over
//     the stored keys its 16-bit bucket; every key above that bucket is kept,
//     every key below dropped, and the coordinates inside it (usually a few
//     hundred) get their full 31-bit keys back from what phase 1 wrote (vals
//     on the applied mask, else the new residual) and are ranked on the
//     unique composite (key << 16 | 0xFFFF - index); one pass over the stored
//     keys both assembles the chunk's mask words in shared memory and lists
//     the bucket's coordinates.  A bucket with more than
//     kCap coordinates (massive ties) flags the chunk; the standalone radix
//     select redoes such chunks after this kernel;
//  3. the streaming pass of every other worker;
//  4. the "all-reduce": bbar = (vals_0 + ... + vals_{W-1}) * (1/W) for the
//     chunk's kept coordinates, read back from the compact buffers the
//     workers wrote (the only place worker data meets), then v and theta for
//     every coordinate of the chunk.
// At step 0 a first launch in boot mode builds M_{-1} the same way: phases 1
// and 2 on the owner's step-0 accumulator a = e + (b1*u + c1*g), computed
// read-only, with nothing else written.
// The union variant (the non-partitioned alternative) runs phases 1 and 2 for
// every worker of the chunk in turn, OR-ing the W selections into M_t, and
// takes base_c from the prefix of M_{t-1}'s per-chunk counts.
// The grid is persistent and balanced (the fewest rounds, the last one as
// full as possible); launches use programmatic dependent launch, and the
// count of chunks left to the standalone select lives in a two-slot ring.
// Arithmetic is the fp32 rule of the library header, with the same
// parenthesisation and no FMA contraction (built with -fmad=false).
//
// Per coordinate the HBM traffic is W*(2 g + 8 u + 8 e + 1/8 mask) + 8 theta +
// 8 v + 1/8 new mask bytes, plus 4 B per kept value per worker written and
// read back and 8 B per kept coordinate (bbar, idx) -- the compulsory bytes.
#include <atomic>
#include "scape_device.cuh"
#include "scape_kernels.cuh"

namespace scape {
namespace {

constexpr uint32_t kCap = 2048;          // candidates ranked in shared memory
constexpr uint32_t kRankCountMax = 1024; // up to this many: direct rank count
constexpr int kTB = 47;                  // composite key bits

// The CTA shape: NT threads, chunks of up to MAXC coordinates, MINB CTAs per
// SM.  Dynamic shared memory layout (bytes) at the end.  L1 and shared memory
// share one 256 KB array per SM and loads in flight are staged in L1: the
// shapes below stay inside the 196 KB carve-out (about 60 KB of L1 left).
// Anything past 196 KB moves the kernel to the 228 KB carve-out, where 28 KB
// of L1 cannot hold enough loads in flight (measured: 24 KB more made the step
// 16% slower; 24 KB less made no difference).
template <int NT_, uint32_t MAXC_, int MINB_>
struct Shape {
  static constexpr int NT = NT_;
  static constexpr int NW = NT / 32;
  static constexpr uint32_t MAXC = MAXC_;
  static constexpr uint32_t NWORDS = MAXC / 32;
  static constexpr int MINB = MINB_;
  static constexpr uint32_t OffKey16 = 0;                      // uint16[MAXC]
  static constexpr uint32_t OffHist = OffKey16 + MAXC * 2;     // uint32[4096]
  static constexpr uint32_t OffWprev = OffHist + 4096 * 4;     // uint32[NWORDS]
  static constexpr uint32_t OffMword = OffWprev + NWORDS * 4;  // uint32[NWORDS]
  static constexpr uint32_t OffWpre = OffMword + NWORDS * 4;   // uint16[NWORDS]
  static constexpr uint32_t OffCand = OffWpre + NWORDS * 2;    // uint64[kCap]
  static constexpr uint32_t OffScan = OffCand + kCap * 8;      // uint32[64]
  static constexpr uint32_t OffCtl = OffScan + 64 * 4;         // uint32[32]
  static constexpr uint32_t OffStage = OffCtl + 32 * 4;        // float[NW][32]
  static constexpr uint32_t SmemBytes = OffStage + NW * 32 * 4;
  static_assert(NWORDS <= 2 * NT, "phase 0 takes two mask words per thread");
  static_assert(OffCand % 8 == 0, "candidate keys are 8-byte aligned");
  static_assert(NW <= 32, "block scans keep one total per warp");
  static_assert(MINB * (SmemBytes + 1024) <= 196 * 1024, "inside the 196 KB carve-out");
};
// Big: one 1024-thread CTA per SM, chunks up to 65536 (188.8 KB).  Small:
// chunks up to 16384 leave most of a 1024-thread CTA idle and too few chunks
// in flight, so two 512-thread CTAs share an SM (71.4 KB each).
using Big = Shape<1024, kMaxChunk, 1>;
using Small = Shape<512, 16384, 2>;

// ctl[] slots
enum { C_BIN = 0, C_ABOVE = 1, C_CNT = 2, C_NCAND = 3, C_SUB = 8 /* 16 entries */ };

struct Shared {
  uint16_t* key16;
  uint32_t* hist;
  uint32_t* wprev;
  uint32_t* mword;
  uint16_t* wpre;
  unsigned long long* cand;
  uint32_t* scan;
  uint32_t* ctl;
  float* stage;  // per warp: the tile's first 32 kept values, for one coalesced store
};

template <class K>
__device__ __forceinline__ Shared carve(unsigned char* s) {
  Shared sh;
  sh.key16 = reinterpret_cast<uint16_t*>(s + K::OffKey16);
  sh.hist = reinterpret_cast<uint32_t*>(s + K::OffHist);
  sh.wprev = reinterpret_cast<uint32_t*>(s + K::OffWprev);
  sh.mword = reinterpret_cast<uint32_t*>(s + K::OffMword);
  sh.wpre = reinterpret_cast<uint16_t*>(s + K::OffWpre);
  sh.cand = reinterpret_cast<unsigned long long*>(s + K::OffCand);
  sh.scan = reinterpret_cast<uint32_t*>(s + K::OffScan);
  sh.ctl = reinterpret_cast<uint32_t*>(s + K::OffCtl);
  sh.stage = reinterpret_cast<float*>(s + K::OffStage);
  return sh;
}

struct Chunk {
  uint64_t c, c0, base;  // index, first coordinate, first packed position
  uint32_t L, k, nw;     // length, coordinates to select, mask words
  uint32_t cap;          // compact slots of the chunk: k, or M_{t-1}'s count (union variant)
  int owner;             // the worker whose accumulator is ranked
};

enum { PASS_OTHER = 0, PASS_OWNER = 1, PASS_BOOT = 2 };

// Phases 1 and 3: worker w's streaming pass over the chunk.  One warp per
// 256-coordinate tile, 8 consecutive coordinates per thread (16-byte loads).
// PASS_OWNER also keeps the keys of |a| and their histogram; PASS_BOOT only
// computes the step-0 accumulator a = e + (b1*u + c1*g) for its keys and
// writes nothing to memory.
template <class K, int PASS>
__device__ __forceinline__ void stream_worker(const FusedArgs& p, const Shared& sh,
                                              const Chunk& ch, int w) {
  constexpr bool KEYS = PASS != PASS_OTHER;
  constexpr bool WRITE = PASS != PASS_BOOT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint16_t* __restrict__ g = p.grads[w] + ch.c0;
  float* __restrict__ u = p.u + (uint64_t)w * p.Np + ch.c0;
  float* __restrict__ e = p.e + (uint64_t)w * p.Np + ch.c0;
  float* __restrict__ vals = p.vals + (uint64_t)w * p.Kp + ch.base;
  const float b1 = p.b1, c1 = p.c1;
  float* stage = sh.stage + warp * 32;
  const uint32_t ntile = (ch.L + 255) / 256;
  for (uint32_t t = warp; t < ntile; t += K::NW) {  // warp-uniform: every lane takes part
    const uint32_t i0 = t * 256 + lane * 8;
    const bool active = i0 < ch.L;
    uint32_t byte = 0, rank0 = 0, tile0 = 0;
    if (WRITE) {
      if (active) {
        const uint32_t j = i0 >> 5;
        const uint32_t word = sh.wprev[j];
        const uint32_t sft = (lane & 3) * 8;
        byte = (word >> sft) & 0xFFu;
        rank0 = sh.wpre[j] + __popc(word & ((1u << sft) - 1u));
      }
      tile0 = sh.wpre[t * 8];  // the tile's kept values occupy [tile0, tile0 + cnt)
    }
    // kept value of element jj: tile rank < 32 -> staged, else stored directly
#define SCAPE_KEEP(jj, bval)                                              \
    do {                                                                  \
      const uint32_t r_ = rank0 + __popc(byte & ((1u << (jj)) - 1u));     \
      if (r_ - tile0 < 32u) stage[r_ - tile0] = (bval);                   \
      else if (SCAPE_CHECK(p.dbg, r_ < ch.cap, CHK_VALS_WRITE,              \
                           ch.c0 + i0 + (jj))) vals[r_] = (bval);         \
    } while (0)
    if (!active) {
      // nothing to stream; the lane still joins the warp's coalesced store
    } else if (i0 + 8 <= ch.L) {
      const uint4 gr = ld_stream_u4(g + i0);
      float4* up = reinterpret_cast<float4*>(u + i0);
      float4* ep = reinterpret_cast<float4*>(e + i0);
      const float4 u0 = up[0], u1 = up[1], e0 = ep[0], e1 = ep[1];
      float gf[8] = {bf16lo(gr.x), bf16hi(gr.x), bf16lo(gr.y), bf16hi(gr.y),
                     bf16lo(gr.z), bf16hi(gr.z), bf16lo(gr.w), bf16hi(gr.w)};
      float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      float ee[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
      uint32_t k16[8];
#pragma unroll
      for (int jj = 0; jj < 8; jj++) {
        const float un = (b1 * uu[jj]) + (c1 * gf[jj]);
        const float a = ee[jj] + un;
        if (WRITE) {
          const bool m = (byte >> jj) & 1u;
          const float b = m ? a : 0.0f;
          uu[jj] = un;
          ee[jj] = a - b;
          if (m) SCAPE_KEEP(jj, b);
        }
        if (KEYS) {
          const uint32_t key = __float_as_uint(a) & 0x7FFFFFFFu;
          k16[jj] = key >> 15;
          atomicAdd(&sh.hist[key >> 19], 1u);
        }
      }
      if (WRITE) {
        up[0] = make_float4(uu[0], uu[1], uu[2], uu[3]);
        up[1] = make_float4(uu[4], uu[5], uu[6], uu[7]);
        ep[0] = make_float4(ee[0], ee[1], ee[2], ee[3]);
        ep[1] = make_float4(ee[4], ee[5], ee[6], ee[7]);
      }
      if (KEYS) {
        uint4 kv;
        kv.x = k16[0] | (k16[1] << 16);
        kv.y = k16[2] | (k16[3] << 16);
        kv.z = k16[4] | (k16[5] << 16);
        kv.w = k16[6] | (k16[7] << 16);
        *reinterpret_cast<uint4*>(sh.key16 + i0) = kv;
      }
    } else {
      const uint32_t nv = ch.L - i0;
      for (uint32_t jj = 0; jj < nv; jj++) {
        const float un = (b1 * u[i0 + jj]) + (c1 * bf16f(g[i0 + jj]));
        const float a = e[i0 + jj] + un;
        if (WRITE) {
          const bool m = (byte >> jj) & 1u;
          const float b = m ? a : 0.0f;
          u[i0 + jj] = un;
          e[i0 + jj] = a - b;
          if (m) SCAPE_KEEP(jj, b);
        }
        if (KEYS) {
          const uint32_t key = __float_as_uint(a) & 0x7FFFFFFFu;
          sh.key16[i0 + jj] = (uint16_t)(key >> 15);
          atomicAdd(&sh.hist[key >> 19], 1u);
        }
      }
    }
#undef SCAPE_KEEP
    if (WRITE) {
      const uint32_t cnt = __reduce_add_sync(kFull, (uint32_t)__popc(byte));
      __syncwarp();
      if (lane < cnt && SCAPE_CHECK(p.dbg, tile0 + lane < ch.cap, CHK_VALS_STAGE, ch.c0 + t * 256))
        vals[tile0 + lane] = stage[lane];
      __syncwarp();
    }
  }
}

// The same pass for residuals held in mapped host memory.  Each lane takes two
// groups of 4 consecutive coordinates, 128 apart, one group after the other,
// so that every warp access of u and e covers 512 contiguous bytes.  Over the
// CPU-GPU link an access that covers half of each 32-byte sector (the layout
// above) moves half the useful bytes per transfer; in HBM, L2 merges the
// halves and the layout above, with twice the bytes in flight per thread, is
// faster.
template <class K, int PASS>
__device__ __forceinline__ void stream_worker_contig(const FusedArgs& p, const Shared& sh,
                                              const Chunk& ch, int w) {
  constexpr bool KEYS = PASS != PASS_OTHER;
  constexpr bool WRITE = PASS != PASS_BOOT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint16_t* __restrict__ g = p.grads[w] + ch.c0;
  float* __restrict__ u = p.u + (uint64_t)w * p.Np + ch.c0;
  float* __restrict__ e = p.e + (uint64_t)w * p.Np + ch.c0;
  float* __restrict__ vals = p.vals + (uint64_t)w * p.Kp + ch.base;
  const float b1 = p.b1, c1 = p.c1;
  float* stage = sh.stage + warp * 32;
  const uint32_t ntile = (ch.L + 255) / 256;
  const uint32_t sft = (lane & 7) * 4;  // the group's nibble in its mask word
  for (uint32_t t = warp; t < ntile; t += K::NW) {  // warp-uniform: every lane takes part
    const uint32_t tile0 = WRITE ? (uint32_t)sh.wpre[t * 8] : 0u;  // first kept value's rank
    const uint32_t ia = t * 256 + lane * 4;  // group h starts at ia + 128 h
    uint32_t nr[2] = {0u, 0u};  // group h: mask nibble << 28 | rank of its first coordinate
    uint2 gr[2];
    float4 uv[2], ev[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const uint32_t i0 = ia + h * 128;
      if (WRITE && i0 < ch.L) {
        const uint32_t j = i0 >> 5;
        const uint32_t word = sh.wprev[j];
        nr[h] = (((word >> sft) & 0xFu) << 28) | (sh.wpre[j] + __popc(word & ((1u << sft) - 1u)));
      }
    }
    // kept value of element jj of group h: tile rank < 32 -> staged, else stored directly
#define SCAPE_KEEP(h, jj, bval)                                                     \
    do {                                                                            \
      const uint32_t r_ = (nr[h] & 0x0FFFFFFFu) + __popc((nr[h] >> 28) & ((1u << (jj)) - 1u)); \
      if (r_ - tile0 < 32u) stage[r_ - tile0] = (bval);                             \
      else if (SCAPE_CHECK(p.dbg, r_ < ch.cap, CHK_VALS_WRITE,                        \
                           ch.c0 + ia + (h) * 128 + (jj))) vals[r_] = (bval);       \
    } while (0)
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const uint32_t i0 = ia + h * 128;
      if (i0 + 4 <= ch.L) {
        gr[h] = ld_stream_u2(g + i0);
        uv[h] = *reinterpret_cast<const float4*>(u + i0);
        ev[h] = *reinterpret_cast<const float4*>(e + i0);
        float gf[4] = {bf16lo(gr[h].x), bf16hi(gr[h].x), bf16lo(gr[h].y), bf16hi(gr[h].y)};
        float uu[4] = {uv[h].x, uv[h].y, uv[h].z, uv[h].w};
        float ee[4] = {ev[h].x, ev[h].y, ev[h].z, ev[h].w};
        uint32_t k16[4];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          const float un = (b1 * uu[jj]) + (c1 * gf[jj]);
          const float a = ee[jj] + un;
          if (WRITE) {
            const bool m = (nr[h] >> (28 + jj)) & 1u;
            const float b = m ? a : 0.0f;
            uu[jj] = un;
            ee[jj] = a - b;
            if (m) SCAPE_KEEP(h, jj, b);
          }
          if (KEYS) {
            const uint32_t key = __float_as_uint(a) & 0x7FFFFFFFu;
            k16[jj] = key >> 15;
            atomicAdd(&sh.hist[key >> 19], 1u);
          }
        }
        if (WRITE) {
          *reinterpret_cast<float4*>(u + i0) = make_float4(uu[0], uu[1], uu[2], uu[3]);
          *reinterpret_cast<float4*>(e + i0) = make_float4(ee[0], ee[1], ee[2], ee[3]);
        }
        if (KEYS)
          *reinterpret_cast<uint2*>(sh.key16 + i0) =
              make_uint2(k16[0] | (k16[1] << 16), k16[2] | (k16[3] << 16));
      } else if (i0 < ch.L) {  // the chunk's ragged end
        const uint32_t nv = ch.L - i0;
        for (uint32_t jj = 0; jj < nv; jj++) {
          const uint32_t i = i0 + jj;
          const float un = (b1 * u[i]) + (c1 * bf16f(g[i]));
          const float a = e[i] + un;
          if (WRITE) {
            const bool m = (nr[h] >> (28 + jj)) & 1u;
            const float b = m ? a : 0.0f;
            u[i] = un;
            e[i] = a - b;
            if (m) SCAPE_KEEP(h, jj, b);
          }
          if (KEYS) {
            const uint32_t key = __float_as_uint(a) & 0x7FFFFFFFu;
            sh.key16[i] = (uint16_t)(key >> 15);
            atomicAdd(&sh.hist[key >> 19], 1u);
          }
        }
      }
    }
#undef SCAPE_KEEP
    if (WRITE) {
      const uint32_t cnt = __reduce_add_sync(kFull, (uint32_t)(__popc(nr[0] >> 28) + __popc(nr[1] >> 28)));
      __syncwarp();
      if (lane < cnt && SCAPE_CHECK(p.dbg, tile0 + lane < ch.cap, CHK_VALS_STAGE, ch.c0 + t * 256))
        vals[tile0 + lane] = stage[lane];
      __syncwarp();
    }
  }
}

// Full 31-bit key of the owner's accumulator at chunk coordinate i, rebuilt
// from what phase 1 wrote: the kept value on M_{t-1}, else the residual (or,
// in the step-0 pass, recomputed from the untouched state and gradient).
__device__ __forceinline__ uint32_t owner_key(const FusedArgs& p, const Shared& sh,
                                              const Chunk& ch, uint32_t i) {
  if (p.boot) {  // step 0: nothing written yet, a = e + (b1*u + c1*g)
    const uint64_t x = (uint64_t)ch.owner * p.Np + ch.c0 + i;
    const float un = (p.b1 * p.u[x]) + (p.c1 * bf16f(p.grads[ch.owner][ch.c0 + i]));
    return __float_as_uint(p.e[x] + un) & 0x7FFFFFFFu;
  }
  const uint32_t j = i >> 5, bit = i & 31;
  const uint32_t word = sh.wprev[j];
  float a;
  if ((word >> bit) & 1u) {
    const uint32_t r = sh.wpre[j] + __popc(word & ((1u << bit) - 1u));
    a = SCAPE_CHECK(p.dbg, r < ch.cap, CHK_OWNER_KEY, ch.c0 + i)
            ? p.vals[(uint64_t)ch.owner * p.Kp + ch.base + r]
            : 0.0f;
  } else {
    a = p.e[(uint64_t)ch.owner * p.Np + ch.c0 + i];
  }
  return __float_as_uint(a) & 0x7FFFFFFFu;
}

// Phase 2.  Leaves the chunk's mask words in sh.mword; returns false when the
// chunk must be redone by the standalone select (too many tied candidates).
template <class K>
__device__ bool select_chunk(const FusedArgs& p, const Shared& sh, const Chunk& ch) {
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t L = ch.L, k = ch.k;
  uint32_t T16 = 0;     // keys above this 16-bit bucket are kept
  bool take_bucket;     // keep the whole bucket T16 too
  bool ranked = false;  // bucket T16 resolved through candidates
  uint32_t r2 = 0, ncand = 0;

  if (k == 0 || k == L) {
    for (uint32_t j = tid; j < ch.nw; j += K::NT) {
      uint32_t word = 0u;
      if (k != 0) word = (j == ch.nw - 1 && (L & 31)) ? ((1u << (L & 31)) - 1u) : 0xFFFFFFFFu;
      sh.mword[j] = word;
    }
    __syncthreads();
    return true;
  }
  find_bin<K::NT>(sh.hist, 4096, k, sh.scan, sh.ctl);
  const uint32_t b12 = sh.ctl[C_BIN], cnt12 = sh.ctl[C_CNT];
  const uint32_t r1 = k - sh.ctl[C_ABOVE];
  if (r1 == cnt12) {
    T16 = b12 << 4;
    take_bucket = true;
  } else {
    // 16 sub-buckets of the threshold bin
    if (tid < 16) sh.ctl[C_SUB + tid] = 0;
    __syncthreads();
    const uint32_t L8 = L & ~7u;  // 8 keys per 16-byte load, then the ragged end
    for (uint32_t i = tid * 8; i < L8; i += K::NT * 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(sh.key16 + i);
      const uint32_t kw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 8; q++) {
        const uint32_t k16 = (kw[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
        if ((k16 >> 4) == b12) atomicAdd(&sh.ctl[C_SUB + (k16 & 15u)], 1u);
      }
    }
    for (uint32_t i = L8 + tid; i < L; i += K::NT) {
      const uint32_t k16 = sh.key16[i];
      if ((k16 >> 4) == b12) atomicAdd(&sh.ctl[C_SUB + (k16 & 15u)], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t acc = 0;
      for (int b = 15; b >= 0; b--) {
        const uint32_t h = sh.ctl[C_SUB + b];
        if (acc + h >= r1) {
          sh.ctl[C_BIN] = (b12 << 4) | (uint32_t)b;
          sh.ctl[C_ABOVE] = r1 - acc;
          sh.ctl[C_CNT] = h;
          break;
        }
        acc += h;
      }
      sh.ctl[C_NCAND] = 0;
    }
    __syncthreads();
    T16 = sh.ctl[C_BIN];
    r2 = sh.ctl[C_ABOVE];
    const uint32_t cnt16 = sh.ctl[C_CNT];
    take_bucket = (r2 == cnt16);
    if (!take_bucket) {
      if (cnt16 > kCap) return false;  // uniform: every thread read the same cnt16
      ranked = true;
    }
  }

  // One pass over the stored keys builds the chunk's mask words (kept iff
  // key16 >= tb) and, when the threshold bucket must be ranked, lists its
  // coordinates with their full composite keys.  Lane l of a warp tests keys
  // [b0 + 8 l, b0 + 8 l + 8) (one 16-byte load; a warp covers 8 words) into a
  // byte, and the 4 lanes of a word merge their bytes by two xor-shuffles;
  // the rare rounds where some lane holds a bucket key allocate list slots by
  // a warp scan.
  const int warp = tid >> 5;
  const uint32_t tb = take_bucket ? T16 : T16 + 1;  // kept iff key16 >= tb
  for (uint32_t b0 = (uint32_t)warp * 256; b0 < ch.nw * 32; b0 += K::NT * 8) {
    const uint32_t i0 = b0 + lane * 8;
    uint32_t byte = 0u, m8 = 0u;  // m8 bit j: coordinate i0 + j is in the bucket
    if (i0 + 8 <= L) {
      const uint4 v = *reinterpret_cast<const uint4*>(sh.key16 + i0);
      const uint32_t kw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 8; q++) {
        const uint32_t k16 = (kw[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
        byte |= (uint32_t)(k16 >= tb) << q;
        m8 |= (uint32_t)(k16 == T16) << q;
      }
    } else {
      for (uint32_t q = 0; i0 + q < L; q++) {
        const uint32_t k16 = sh.key16[i0 + q];
        byte |= (uint32_t)(k16 >= tb) << q;
        m8 |= (uint32_t)(k16 == T16) << q;
      }
    }
    uint32_t word = byte << (8 * (lane & 3));
    word |= __shfl_xor_sync(kFull, word, 1);
    word |= __shfl_xor_sync(kFull, word, 2);
    if ((lane & 3) == 0 && (i0 >> 5) < ch.nw) sh.mword[i0 >> 5] = word;
    if (!ranked) continue;
    if (!__any_sync(kFull, m8 != 0u)) continue;  // warp-uniform
    const uint32_t n = __popc(m8);
    const uint32_t incl = warp_incl_scan(n, lane);
    uint32_t pos = 0;
    if (lane == 31) pos = atomicAdd(&sh.ctl[C_NCAND], incl);
    pos = __shfl_sync(kFull, pos, 31) + incl - n;
    for (uint32_t mm = m8; mm; mm &= mm - 1u) {
      const uint32_t i = i0 + (uint32_t)(__ffs(mm) - 1);
      const uint32_t slot = pos++;
      if (SCAPE_CHECK(p.dbg, slot < kCap, CHK_CAND, ch.c0 + i)) {
        const uint32_t key = owner_key(p, sh, ch, i);
        sh.cand[slot] = ((unsigned long long)key << 16) | (unsigned long long)(0xFFFFu - i);
      }
    }
  }
  __syncthreads();
  if (ranked) ncand = sh.ctl[C_NCAND];

  if (ranked) {
    if (ncand <= kRankCountMax) {
      // direct rank: keep candidate m iff fewer than r2 candidates are larger
      for (uint32_t m = tid; m < ncand; m += K::NT) {
        const unsigned long long X = sh.cand[m];
        uint32_t above = 0;
        for (uint32_t o = 0; o < ncand; o++) above += sh.cand[o] > X;
        if (above < r2) {
          const uint32_t i = 0xFFFFu - (uint32_t)(X & 0xFFFFu);
          atomicOr(&sh.mword[i >> 5], 1u << (i & 31));
        }
      }
    } else {
      // radix over the low 31 bits (all candidates share the top 16 = T16)
      unsigned long long pf = T16;
      int pb = 16;
      uint32_t rr = r2;
      while (true) {
        const int d = (kTB - pb) < 12 ? (kTB - pb) : 12;
        const int nb = 1 << d;
        const int shift = kTB - pb - d;
        for (int i = tid; i < nb; i += K::NT) sh.hist[i] = 0;
        __syncthreads();
        for (uint32_t m = tid; m < ncand; m += K::NT) {
          const unsigned long long X = sh.cand[m];
          if ((X >> (kTB - pb)) == pf)
            atomicAdd(&sh.hist[(uint32_t)(X >> shift) & (uint32_t)(nb - 1)], 1u);
        }
        __syncthreads();
        find_bin<K::NT>(sh.hist, nb, rr, sh.scan, sh.ctl);
        const uint32_t b = sh.ctl[C_BIN], above = sh.ctl[C_ABOVE], cnt = sh.ctl[C_CNT];
        __syncthreads();
        rr -= above;
        pf = (pf << d) | b;
        pb += d;
        if (rr == cnt) break;
      }
      const unsigned long long T = pf << (kTB - pb);
      for (uint32_t m = tid; m < ncand; m += K::NT) {
        const unsigned long long X = sh.cand[m];
        if (X >= T) {
          const uint32_t i = 0xFFFFu - (uint32_t)(X & 0xFFFFu);
          atomicOr(&sh.mword[i >> 5], 1u << (i & 31));
        }
      }
    }
    __syncthreads();
  }
  return true;
}

// vals_0[r] + vals_1[r] + ... + vals_{W-1}[r], added left to right.  The loads
// of each group of 8 workers are issued before any of them is added, so their
// memory latencies overlap instead of queueing one after another.
__device__ __forceinline__ float ordered_sum(const FusedArgs& p, uint32_t r) {
  const float* v = p.vals + r;
  float s = 0.0f;
  for (int w0 = 0; w0 < p.W; w0 += 8) {
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; j++) x[j] = (w0 + j < p.W) ? v[(uint64_t)(w0 + j) * p.Kp] : 0.0f;
#pragma unroll
    for (int j = 0; j < 8; j++)
      if (w0 + j < p.W) s = (w0 + j == 0) ? x[j] : s + x[j];
  }
  return s;
}

__device__ __forceinline__ void prefetch_l2(const void* q) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
}

// Before a barrier: ask L2 for this thread's first tile of the next phase, so
// the memory pipe does not run dry while the CTA waits and restarts.
__device__ __forceinline__ void prefetch_worker_tile(const FusedArgs& p, uint64_t c0, uint32_t L,
                                                     int w) {
  const uint32_t i0 = (threadIdx.x >> 5) * 256 + (threadIdx.x & 31) * 8;
  if (i0 + 8 > L) return;
  prefetch_l2(p.grads[w] + c0 + i0);
  prefetch_l2(p.u + (uint64_t)w * p.Np + c0 + i0);
  prefetch_l2(p.e + (uint64_t)w * p.Np + c0 + i0);
}

// Phase 4: fixed-order W-way sum of the compact buffers and the AdamS update.
// The kept coordinates of a 256-coordinate tile have consecutive packed
// positions [R0, R0 + cnt), so the warp computes their bbar together: lane l
// takes positions R0 + l, R0 + l + 32, ... (coalesced reads of the W rows, one
// memory round trip per 32 kept coordinates) and hands each value to the lane
// that holds the coordinate with a shuffle.
template <class K>
__device__ __forceinline__ void update_chunk(const FusedArgs& p, const Shared& sh,
                                             const Chunk& ch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* __restrict__ th = p.theta + ch.c0;
  float* __restrict__ vv = p.v + ch.c0;
  const float b2 = p.b2, c2 = p.c2, lr = p.lr, wd = p.wd, eps = p.eps, invW = p.invW;
  const uint32_t ntile = (ch.L + 255) / 256;
  for (uint32_t t = warp; t < ntile; t += K::NW) {  // warp-uniform: every lane takes part
    const uint32_t i0 = t * 256 + lane * 8;
    const bool active = i0 < ch.L;
    uint32_t byte = 0, local0 = 0;
    if (active) {
      const uint32_t j = i0 >> 5;
      const uint32_t word = sh.wprev[j];
      const uint32_t sft = (lane & 3) * 8;
      byte = (word >> sft) & 0xFFu;
      local0 = sh.wpre[j] + __popc(word & ((1u << sft) - 1u));
    }
    const uint32_t tile0 = sh.wpre[t * 8];  // in-chunk position of the tile's first kept value
    const uint32_t cnt = __reduce_add_sync(kFull, (uint32_t)__popc(byte));
    const uint32_t nv = active ? ((ch.L - i0) < 8 ? (ch.L - i0) : 8) : 0;
    if (nv == 8) {  // theta and v travel to L2 while bbar is being summed
      prefetch_l2(th + i0);
      prefetch_l2(vv + i0);
    }
    // bbar of the tile's kept coordinates, computed cooperatively
    float bb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const uint32_t R0 = (uint32_t)ch.base + tile0;
    for (uint32_t r0 = 0; r0 < cnt; r0 += 32) {
      float mine = 0.0f;
      if (r0 + lane < cnt &&
          SCAPE_CHECK(p.dbg, tile0 + r0 + lane < ch.cap, CHK_BBAR, ch.c0 + t * 256)) {
        mine = ordered_sum(p, R0 + r0 + lane) * invW;
        p.bbar[R0 + r0 + lane] = mine;
      }
#pragma unroll
      for (int jj = 0; jj < 8; jj++) {
        const uint32_t need = local0 - tile0 + __popc(byte & ((1u << jj) - 1u));
        const float got = __shfl_sync(kFull, mine, need & 31);
        if (((byte >> jj) & 1u) && need >= r0 && need < r0 + 32) bb[jj] = got;
      }
    }
    float tt[8], vo[8];
    if (nv == 8) {
      const float4 t0 = reinterpret_cast<const float4*>(th + i0)[0];
      const float4 t1 = reinterpret_cast<const float4*>(th + i0)[1];
      const float4 v0 = reinterpret_cast<const float4*>(vv + i0)[0];
      const float4 v1 = reinterpret_cast<const float4*>(vv + i0)[1];
      tt[0] = t0.x; tt[1] = t0.y; tt[2] = t0.z; tt[3] = t0.w;
      tt[4] = t1.x; tt[5] = t1.y; tt[6] = t1.z; tt[7] = t1.w;
      vo[0] = v0.x; vo[1] = v0.y; vo[2] = v0.z; vo[3] = v0.w;
      vo[4] = v1.x; vo[5] = v1.y; vo[6] = v1.z; vo[7] = v1.w;
    } else {
#pragma unroll
      for (uint32_t jj = 0; jj < 8; jj++) {
        tt[jj] = jj < nv ? th[i0 + jj] : 0.0f;
        vo[jj] = jj < nv ? vv[i0 + jj] : 0.0f;
      }
    }
#pragma unroll
    for (int jj = 0; jj < 8; jj++) {
      const bool m = (byte >> jj) & 1u;
      if (m) {
        const uint32_t r = local0 + __popc(byte & ((1u << jj) - 1u));
        if (SCAPE_CHECK(p.dbg, r < ch.cap, CHK_IDX, ch.c0 + i0 + jj))
          p.idx[ch.base + r] = (uint32_t)(ch.c0 + i0 + jj);
      }
      const float vn = (b2 * vo[jj]) + (c2 * (bb[jj] * bb[jj]));
      const float q = m ? bb[jj] / (sqrtf(vn) + eps) : 0.0f;
      vo[jj] = vn;
      tt[jj] = tt[jj] - (lr * (q + (wd * tt[jj])));
    }
    if (nv == 8) {
      reinterpret_cast<float4*>(th + i0)[0] = make_float4(tt[0], tt[1], tt[2], tt[3]);
      reinterpret_cast<float4*>(th + i0)[1] = make_float4(tt[4], tt[5], tt[6], tt[7]);
      reinterpret_cast<float4*>(vv + i0)[0] = make_float4(vo[0], vo[1], vo[2], vo[3]);
      reinterpret_cast<float4*>(vv + i0)[1] = make_float4(vo[4], vo[5], vo[6], vo[7]);
    } else {
#pragma unroll
      for (uint32_t jj = 0; jj < 8; jj++)
        if (jj < nv) {
          th[i0 + jj] = tt[jj];
          vv[i0 + jj] = vo[jj];
        }
    }
  }
}

template <class K, int PASS, bool CONTIG>
__device__ __forceinline__ void stream_pass(const FusedArgs& p, const Shared& sh, const Chunk& ch,
                                            int w) {
  if (CONTIG) stream_worker_contig<K, PASS>(p, sh, ch, w);
  else stream_worker<K, PASS>(p, sh, ch, w);
}

// The selection's outcome for the chunk: its mask words into M_t (OR-ed into
// what the earlier workers selected when "merge"), or a flag for the
// standalone select, which then redoes the whole chunk.
template <int NT>
__device__ __forceinline__ void publish_mask(const FusedArgs& p, const Shared& sh,
                                             const Chunk& ch, bool ok, bool merge) {
  const int tid = threadIdx.x;
  if (ok) {
    uint32_t* mo = p.mout + ch.c0 / 32;
    for (uint32_t j = tid; j < ch.nw; j += NT) mo[j] = merge ? (mo[j] | sh.mword[j]) : sh.mword[j];
  } else if (tid == 0) {
    p.fallback[ch.c] = 1u;
    atomicAdd(p.n_fallback, 1u);
    if (p.pending) atomicAdd(p.pending, 1u);
  }
}

// CONTIG: residual rows in mapped host memory (whole-sector access mapping).
// UNION: the non-partitioned variant: in every chunk each worker's own
// accumulator is ranked in turn (its pass keeps its keys) and M_t is the
// union of the W selections; the compact buffers follow M_{t-1}'s per-chunk
// counts (cbase) instead of k_c.
template <class K, bool CONTIG, bool UNION>
__global__ __launch_bounds__(K::NT, K::MINB) void step_chunks(const FusedArgs p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const Shared sh = carve<K>(smem_raw);
  const int tid = threadIdx.x;
  grid_dependency_wait();    // the previous step's select has finished
  grid_launch_dependents();  // every CTA is resident: the select may launch
  if (p.pending_clear && blockIdx.x == 0 && tid == 0) *p.pending_clear = 0u;

  for (uint64_t c = blockIdx.x; c < p.n_ch; c += gridDim.x) {
    Chunk ch;
    ch.c = c;
    if (p.chunks) {
      const ChunkDesc d = p.chunks[c];
      ch.c0 = d.start;
      ch.L = d.len;
      ch.k = d.k;
      ch.base = d.base;
    } else {
      ch.c0 = c * p.C;
      ch.L = (uint32_t)((p.N - ch.c0) < p.C ? (p.N - ch.c0) : p.C);
      ch.k = (c == p.n_ch - 1) ? p.k_last : p.k_full;
      ch.base = c * (uint64_t)p.k_full;
    }
    ch.cap = ch.k;
    if (UNION) {
      ch.base = p.cbase ? p.cbase[c] : 0;
      ch.cap = p.cbase ? (uint32_t)(p.cbase[c + 1] - p.cbase[c]) : 0u;
    }
    ch.nw = (ch.L + 31) / 32;
    ch.owner = (int)(c / p.q);
    if (!SCAPE_CHECK(p.dbg, ch.c0 + ch.L <= p.N && ch.L <= K::MAXC, CHK_CHUNK, ch.c0)) continue;

    // phase 0: M_{t-1} words of the chunk, their popcount prefix; clear the histogram
    {
      const uint32_t j0 = tid * 2;
      uint32_t w0 = 0u, w1 = 0u;
      if (!p.boot) {  // no M_{t-1} at step 0
        const uint32_t* mp = p.mprev + ch.c0 / 32;
        if (j0 < ch.nw) w0 = mp[j0];
        if (j0 + 1 < ch.nw) w1 = mp[j0 + 1];
      }
      const uint32_t cnt = __popc(w0) + __popc(w1);
      uint32_t total;
      const uint32_t inc = block_incl_scan<K::NT>(cnt, sh.scan, &total);
      if (j0 < K::NWORDS) {
        sh.wprev[j0] = w0;
        sh.wprev[j0 + 1] = w1;
        sh.wpre[j0] = (uint16_t)(inc - cnt);
        sh.wpre[j0 + 1] = (uint16_t)(inc - cnt + __popc(w0));
      }
      for (int i = tid; i < 4096; i += K::NT) sh.hist[i] = 0;
      __syncthreads();
    }

    if (p.boot) {
      // step 0, first launch: M_{-1} of this chunk from the step-0
      // accumulators (read only), ranked on chip like M_t below: the
      // owner's, or every worker's in turn in the union variant
      const int wa = UNION ? 0 : ch.owner, wb = UNION ? p.W : ch.owner + 1;
      for (int w = wa; w < wb; w++) {
        Chunk cw = ch;
        cw.owner = w;
        stream_pass<K, PASS_BOOT, CONTIG>(p, sh, cw, w);
        __syncthreads();
        publish_mask<K::NT>(p, sh, cw, select_chunk<K>(p, sh, cw), w > wa);
        for (int i = tid; i < 4096; i += K::NT) sh.hist[i] = 0;  // the next worker's
        __syncthreads();
      }
      continue;
    }

    if (UNION) {
      for (int w = 0; w < p.W; w++) {
        Chunk cw = ch;
        cw.owner = w;
        // phase 1 for worker w: its pass, keeping its keys
        stream_pass<K, PASS_OWNER, CONTIG>(p, sh, cw, w);
        if (w + 1 < p.W) {
          prefetch_worker_tile(p, ch.c0, ch.L, w + 1);
        } else {
          const uint32_t i0 = (tid >> 5) * 256 + (tid & 31) * 8;
          if (i0 + 8 <= ch.L) {
            prefetch_l2(p.theta + ch.c0 + i0);
            prefetch_l2(p.v + ch.c0 + i0);
          }
        }
        __syncthreads();
        // phase 2 for worker w: its top-k, OR-ed into M_t
        publish_mask<K::NT>(p, sh, cw, select_chunk<K>(p, sh, cw), w > 0);
        for (int i = tid; i < 4096; i += K::NT) sh.hist[i] = 0;  // the next worker's
        __syncthreads();
      }
      // phase 4: synchronized buffer, second moment, parameters
      update_chunk<K>(p, sh, ch);
    } else {
      // phase 1: the owner's pass, keeping its keys
      stream_pass<K, PASS_OWNER, CONTIG>(p, sh, ch, ch.owner);
      if (p.W > 1) prefetch_worker_tile(p, ch.c0, ch.L, ch.owner == 0 ? 1 : 0);
      __syncthreads();

      // phase 2: top-k of the owner's |a| -> mask words of M_t
      publish_mask<K::NT>(p, sh, ch, select_chunk<K>(p, sh, ch), false);

      // phase 3: every other worker
      for (int w = 0; w < p.W; w++)
        if (w != ch.owner) stream_pass<K, PASS_OTHER, CONTIG>(p, sh, ch, w);
      {
        const uint32_t i0 = (tid >> 5) * 256 + (tid & 31) * 8;
        if (i0 + 8 <= ch.L) {
          prefetch_l2(p.theta + ch.c0 + i0);
          prefetch_l2(p.v + ch.c0 + i0);
        }
      }
      // A warp's tiles are the same in every pass, so the compact values its
      // update reads were all written by the warp itself: the two-CTA shape
      // goes on without waiting for the other warps (2% faster on 4096-long
      // chunks); on the 1024-thread shape the barrier measured 0.3% faster.
      if (K::MINB > 1) __syncwarp();
      else __syncthreads();

      // phase 4: synchronized buffer, second moment, parameters
      update_chunk<K>(p, sh, ch);
    }
    {
      const uint64_t cn = c + gridDim.x;
      if (cn < p.n_ch && !p.chunks && !p.boot) {
        const uint64_t c0n = cn * p.C;
        const uint32_t Ln = (uint32_t)((p.N - c0n) < p.C ? (p.N - c0n) : p.C);
        if ((uint32_t)tid * 2 < (Ln + 31) / 32) prefetch_l2(p.mprev + c0n / 32 + tid * 2);
        prefetch_worker_tile(p, c0n, Ln, UNION ? 0 : (int)(cn / p.q));
      }
    }
    __syncthreads();
  }
}

}  // namespace

namespace {

// The shared-memory opt-in is per device and per instantiation.
template <class K, bool CONTIG, bool UNION>
cudaError_t launch_shape(const FusedArgs& a, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;  // devices past 64: set every launch
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(step_chunks<K, CONTIG, UNION>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)K::SmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  uint64_t grid = (uint64_t)num_sms() * K::MINB;
  if (grid > a.n_ch) grid = a.n_ch;
  {  // the same number of rounds with the last one as full as it gets
    const uint64_t rounds = (a.n_ch + grid - 1) / grid;
    grid = (a.n_ch + rounds - 1) / rounds;
  }
  // launched while the grid ahead of it drains (it waits for it on the GPU)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(K::NT);
  cfg.dynamicSmemBytes = K::SmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_chunks<K, CONTIG, UNION>, a);
}

template <class K>
cudaError_t launch_variant(const FusedArgs& a, cudaStream_t s) {
  if (a.union_mask)
    return a.e_host ? launch_shape<K, true, true>(a, s) : launch_shape<K, false, true>(a, s);
  return a.e_host ? launch_shape<K, true, false>(a, s) : launch_shape<K, false, false>(a, s);
}

}  // namespace

// Chunks of up to 16384 coordinates take the two-CTAs-per-SM shape; every
// chunk of the handle is at most C long (per-tensor chunks too).
cudaError_t launch_step_chunks(const FusedArgs& a, cudaStream_t s) {
  return a.C <= Small::MAXC ? launch_variant<Small>(a, s) : launch_variant<Big>(a, s);
}

}  // namespace scape
