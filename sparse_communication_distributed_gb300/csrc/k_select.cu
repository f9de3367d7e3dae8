// Standalone partitioned mask generation of SCAPE (radix select).
//
// Used for the step-0 mask M_{-1} (every chunk, from the step-0 accumulators)
// and, after the fused step kernel, for the few chunks whose 16-bit threshold
// bucket held more tied coordinates than its shared-memory candidate list
// (those chunks are flagged; this kernel redoes exactly them and clears the
// flags).  One CTA per chunk at a time, grid-strided over the chunks.
//
// SCAPE builds the mask from first-moment statistics, each worker only over
// its own optimizer shard, and the shard masks together form the global mask
// used one step later (gist.science technical summary §2 "Partitioned Mask
// Synchronization", "Delayed Mask Usage"; abstract).  Here: chunk c of C
// coordinates is owned by worker w = c / q; it keeps the k_c coordinates of
// largest |a_w|, the key being the fp32 bit pattern of a_w with the sign
// cleared (an unsigned integer order on |a|), equal keys going to the lower
// coordinate.  Appending the coordinate's complement below the key,
//   X = (key << 16) | (0xFFFF - i_local)      (47 bits, unique in the chunk)
// turns this into "keep the k_c largest X", and the kept set is exactly
// { X >= T } for the k_c-th largest X = T.
//
// T is found by radix selection, one CTA (512 threads) per chunk:
//   1. histogram of the next 12-bit digit of X (shared-memory counters) over
//      the coordinates that match the digits fixed so far; a block scan from
//      the top bin finds the bin holding the r-th largest; repeat while that
//      bin holds more than kCap coordinates (heavy ties) and is not taken
//      whole;
//   2. one more pass writes the chunk's mask words for every coordinate
//      above the fixed prefix (warp-ballot style nibble merge, coalesced
//      32-bit stores) and copies the coordinates equal to the prefix (at
//      most kCap) into shared memory;
//   3. the remaining digits are resolved among those candidates in shared
//      memory, and the kept candidates are OR-ed into the mask words.
// Keys are read with 16-byte loads.  After a step the owner's accumulator is
// rebuilt from what the step wrote: a = vals_w[position] on M_{t-1}, else the
// new residual e_w (which equals a there).  At step 0 it is computed from the
// old state and the gradient, b1*u + c1*g + e, without writing anything.
#include "scape_device.cuh"
#include "scape_kernels.cuh"

namespace scape {
namespace {

constexpr int kNT = 512;
constexpr int kCap = 2048;
constexpr int kTB = 47;
constexpr int kDigit = 12;
constexpr int kMaxWords = kMaxChunk / 32;

struct SelectSmem {
  uint32_t hist[1 << kDigit];
  uint32_t wprev[kMaxWords];
  uint16_t wpre[kMaxWords];
  unsigned long long cand[kCap];
  uint32_t scan[kNT / 32 + 1];
  uint32_t bin, above, cnt;  // written together by find_bin (3 consecutive words)
  uint32_t ncand;
};

enum { SRC_STATE = 0, SRC_BOOT = 1 };

// sm.bin / sm.above / sm.cnt: the bin holding the r-th largest element of
// the histogram, the count in the bins above it, and its count.
__device__ __forceinline__ void find_bin(SelectSmem& sm, int nb, uint32_t r) {
  scape::find_bin<kNT>(sm.hist, nb, r, sm.scan, &sm.bin);
}

// The four composite keys of quad qd (coordinates 4qd..4qd+3 of the chunk);
// returns how many of them lie inside the chunk.
template <int SRC>
__device__ __forceinline__ int quad_keys(const SelectArgs& p, const SelectSmem& sm, int w,
                                         uint64_t c0, uint32_t L, uint32_t kc, uint64_t base_c,
                                         uint32_t qd, unsigned long long X[4]) {
  const uint32_t i4 = qd * 4;
  const int nv = (L - i4) >= 4 ? 4 : (int)(L - i4);
  float a[4];
  const float4 ev = *reinterpret_cast<const float4*>(p.e + (uint64_t)w * p.Np + c0 + i4);
  a[0] = ev.x; a[1] = ev.y; a[2] = ev.z; a[3] = ev.w;
  if (SRC == SRC_STATE) {
    const uint32_t j = qd >> 3, bit0 = (qd & 7) * 4;
    const uint32_t wb = sm.wprev[j];
    const uint32_t nib = (wb >> bit0) & 0xFu;
    if (nib) {
      const float* vw = p.vals + (uint64_t)w * p.Kp + base_c;
      const uint32_t r0 = sm.wpre[j] + __popc(wb & ((1u << bit0) - 1u));
#pragma unroll
      for (int s = 0; s < 4; s++)
        if ((nib >> s) & 1u) {
          const uint32_t r = r0 + __popc(nib & ((1u << s) - 1u));
          if (SCAPE_CHECK(p.dbg, r < kc, CHK_SELECT_VALS, c0 + i4 + s)) a[s] = vw[r];
        }
    }
  } else {
    const float4 uv = *reinterpret_cast<const float4*>(p.u + (uint64_t)w * p.Np + c0 + i4);
    const float uu[4] = {uv.x, uv.y, uv.z, uv.w};
    const uint16_t* gw = p.grads[w] + c0 + i4;
    float gf[4] = {0.f, 0.f, 0.f, 0.f};
    if (nv == 4) {
      const uint2 gr = *reinterpret_cast<const uint2*>(gw);
      gf[0] = bf16lo(gr.x); gf[1] = bf16hi(gr.x); gf[2] = bf16lo(gr.y); gf[3] = bf16hi(gr.y);
    } else {
      for (int s = 0; s < nv; s++) gf[s] = bf16f(gw[s]);
    }
#pragma unroll
    for (int s = 0; s < 4; s++) a[s] = a[s] + ((p.b1 * uu[s]) + (p.c1 * gf[s]));
  }
#pragma unroll
  for (int s = 0; s < 4; s++) {
    const uint32_t key = __float_as_uint(a[s]) & 0x7FFFFFFFu;
    X[s] = ((unsigned long long)key << 16) | (unsigned long long)(0xFFFFu - (i4 + s));
  }
  return nv;
}

// Ranks worker w's accumulator in chunk c and writes the chunk's mask words
// (OR-ed into the words already there when "merge": the union variant).
template <int SRC>
__device__ void select_one(const SelectArgs& p, SelectSmem& sm, const uint64_t c, const int w,
                           const bool merge) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t c0, base_c;
  uint32_t L, k;
  if (p.chunks) {
    const ChunkDesc d = p.chunks[c];
    c0 = d.start;
    L = d.len;
    k = d.k;
    base_c = d.base;
  } else {
    c0 = c * p.C;
    L = (uint32_t)((p.N - c0) < p.C ? (p.N - c0) : p.C);
    k = (c == p.n_ch - 1) ? p.k_last : p.k_full;
    base_c = c * (uint64_t)p.k_full;
  }
  uint32_t kcap = k;  // compact slots of the chunk (M_{t-1}'s count in the union variant)
  if (p.cbase) {  // the union variant's compact layout
    base_c = p.cbase[c];
    kcap = (uint32_t)(p.cbase[c + 1] - p.cbase[c]);
  }
  const uint32_t nwc = (L + 31) / 32;
  uint32_t* mout = p.mout + c0 / 32;

  if (k == 0 || k == L) {
    for (uint32_t j = tid; j < nwc; j += kNT) {
      uint32_t word = 0u;
      if (k != 0) word = (j == nwc - 1 && (L & 31)) ? ((1u << (L & 31)) - 1u) : 0xFFFFFFFFu;
      mout[j] = merge ? (mout[j] | word) : word;
    }
    return;
  }

  if (SRC == SRC_STATE) {
    // M_{t-1} words of the chunk and their exclusive popcount prefix.
    const uint32_t* mp = p.mprev + c0 / 32;
    uint32_t wv[4], cnt = 0;
#pragma unroll
    for (int s = 0; s < 4; s++) {
      const uint32_t j = tid * 4 + s;
      wv[s] = j < nwc ? mp[j] : 0u;
      cnt += __popc(wv[s]);
    }
    uint32_t total;
    uint32_t run = block_incl_scan<kNT>(cnt, sm.scan, &total) - cnt;
#pragma unroll
    for (int s = 0; s < 4; s++) {
      const uint32_t j = tid * 4 + s;
      if (j < nwc) {
        sm.wprev[j] = wv[s];
        sm.wpre[j] = (uint16_t)run;
      }
      run += __popc(wv[s]);
    }
    __syncthreads();
  }

  const uint32_t nq = (L + 3) / 4;

  // 1. digit passes over the chunk
  unsigned long long prefix = 0;
  int pbits = 0;
  uint32_t r = k;
  bool resolved = false;
  while (true) {
    const int d = (kTB - pbits) < kDigit ? (kTB - pbits) : kDigit;
    const int nb = 1 << d;
    const int shift = kTB - pbits - d;
    for (int i = tid; i < nb; i += kNT) sm.hist[i] = 0;
    __syncthreads();
    for (uint32_t base = warp * 32; base < nq; base += kNT) {
      const uint32_t qd = base + lane;
      if (qd < nq) {
        unsigned long long X[4];
        const int nv = quad_keys<SRC>(p, sm, w, c0, L, kcap, base_c, qd, X);
        for (int s = 0; s < nv; s++)
          if ((X[s] >> (kTB - pbits)) == prefix)
            atomicAdd(&sm.hist[(uint32_t)(X[s] >> shift) & (uint32_t)(nb - 1)], 1u);
      }
    }
    __syncthreads();
    find_bin(sm, nb, r);
    const uint32_t b = sm.bin, above = sm.above, cnt = sm.cnt;
    __syncthreads();
    r -= above;
    prefix = (prefix << d) | b;
    pbits += d;
    if (r == cnt) {
      resolved = true;
      break;
    }
    if (cnt <= (uint32_t)kCap) break;
  }

  // 2. mask words for everything above the prefix; candidates to shared memory
  if (tid == 0) sm.ncand = 0;
  __syncthreads();
  const int rem = kTB - pbits;
  for (uint32_t base = warp * 32; base < nq; base += kNT) {
    const uint32_t qd = base + lane;
    uint32_t nib = 0, cc = 0;
    unsigned long long Xc[4];
    if (qd < nq) {
      unsigned long long X[4];
      const int nv = quad_keys<SRC>(p, sm, w, c0, L, kcap, base_c, qd, X);
      for (int s = 0; s < nv; s++) {
        const unsigned long long hi = X[s] >> rem;
        if (resolved ? (hi >= prefix) : (hi > prefix)) nib |= 1u << s;
        else if (!resolved && hi == prefix) Xc[cc++] = X[s];
      }
    }
    if (!resolved) {
      const uint32_t inc = warp_incl_scan(cc, lane);
      uint32_t pos = 0;
      if (lane == 31 && inc) pos = atomicAdd(&sm.ncand, inc);
      pos = __shfl_sync(kFull, pos, 31) + inc - cc;
      for (uint32_t m = 0; m < cc; m++)
        if (pos + m < (uint32_t)kCap) sm.cand[pos + m] = Xc[m];
    }
    uint32_t part = nib << ((lane & 7) * 4);
    part |= __shfl_xor_sync(kFull, part, 1);
    part |= __shfl_xor_sync(kFull, part, 2);
    part |= __shfl_xor_sync(kFull, part, 4);
    const uint32_t j = (base >> 3) + (lane >> 3);
    if ((lane & 7) == 0 && j < nwc) mout[j] = merge ? (mout[j] | part) : part;
  }
  __syncthreads();

  // 3. resolve the remaining digits among the candidates
  if (!resolved) {
    const uint32_t nc = sm.ncand < (uint32_t)kCap ? sm.ncand : (uint32_t)kCap;
    unsigned long long pf = prefix;
    int pb = pbits;
    uint32_t rr = r;
    while (true) {
      const int d = (kTB - pb) < kDigit ? (kTB - pb) : kDigit;
      const int nb = 1 << d;
      const int shift = kTB - pb - d;
      for (int i = tid; i < nb; i += kNT) sm.hist[i] = 0;
      __syncthreads();
      for (uint32_t i = tid; i < nc; i += kNT) {
        const unsigned long long X = sm.cand[i];
        if ((X >> (kTB - pb)) == pf)
          atomicAdd(&sm.hist[(uint32_t)(X >> shift) & (uint32_t)(nb - 1)], 1u);
      }
      __syncthreads();
      find_bin(sm, nb, rr);
      const uint32_t b = sm.bin, above = sm.above, cnt = sm.cnt;
      __syncthreads();
      rr -= above;
      pf = (pf << d) | b;
      pb += d;
      if (rr == cnt) break;
    }
    const unsigned long long T = pf << (kTB - pb);
    for (uint32_t i = tid; i < nc; i += kNT) {
      const unsigned long long X = sm.cand[i];
      if (X >= T) {
        const uint32_t il = 0xFFFFu - (uint32_t)(X & 0xFFFFu);
        atomicOr(&mout[il >> 5], 1u << (il & 31));
      }
    }
  }
}

template <int SRC>
__global__ __launch_bounds__(kNT, 2) void select_topk(const SelectArgs p) {
  __shared__ SelectSmem sm;
  grid_dependency_wait();    // the step kernel has finished
  grid_launch_dependents();  // every CTA is resident: the next step may launch
  if (p.pending && *p.pending == 0u) return;  // the step kernel flagged no chunk
  for (uint64_t c = blockIdx.x; c < p.n_ch; c += gridDim.x) {
    if (p.flags && p.flags[c] == 0u) continue;
    if (p.union_mask) {  // the chunk's words: the union of every worker's selection
      for (int w = 0; w < p.W; w++) {
        select_one<SRC>(p, sm, c, w, w > 0);
        __syncthreads();
      }
    } else {
      select_one<SRC>(p, sm, c, p.rank_worker > 0 ? p.rank_worker - 1 : (int)(c / p.q), false);
      __syncthreads();
    }
    if (p.flags && threadIdx.x == 0) p.flags[c] = 0u;
  }
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, bool boot, cudaStream_t s) {
  uint64_t grid = (uint64_t)num_sms() * 2;
  if (grid > a.n_ch) grid = a.n_ch;
  // launched while the step kernel drains (it waits for it on the GPU)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kNT);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return boot ? cudaLaunchKernelEx(&cfg, select_topk<SRC_BOOT>, a)
              : cudaLaunchKernelEx(&cfg, select_topk<SRC_STATE>, a);
}

}  // namespace scape
