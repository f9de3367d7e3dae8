// Compaction offsets of the applied mask M_{t-1}.
//
// The kept values of a step are packed in ascending coordinate order (the
// packed single-bit masks of the SCAPE pages, gist.science technical summary
// §2 "Memory Optimization", and the one sparse buffer b that is reduced,
// §2 "Single-Buffer Second-Moment Reconstruction").  The position of a kept
// coordinate is the number of set mask bits before it.  These two kernels
// give that count at the start of every 256-coordinate tile:
//   offsets_local: per 65536-coordinate block, one thread per tile, popcount
//                  of the tile's 8 words and a block scan -> toff_local, and
//                  the block's total -> bsum;
//   scan_bsum:     one CTA turns bsum into exclusive prefix sums in place.
// A tile's offset is then toff_local[tile] + bsum[tile / 256].
#include "scape_device.cuh"
#include "scape_kernels.cuh"

namespace scape {
namespace {

__global__ __launch_bounds__(256) void offsets_local(const uint32_t* __restrict__ mask,
                                                     uint32_t* __restrict__ toff_local,
                                                     uint32_t* __restrict__ bsum, uint64_t n_wt) {
  __shared__ uint32_t wt_tot[9];
  const uint64_t wt = (uint64_t)blockIdx.x * kTilesPerBlk + threadIdx.x;
  uint32_t cnt = 0;
  if (wt < n_wt) {
    const uint4* p = reinterpret_cast<const uint4*>(mask + wt * 8);
    uint4 a = __ldg(p), b = __ldg(p + 1);
    cnt = __popc(a.x) + __popc(a.y) + __popc(a.z) + __popc(a.w) + __popc(b.x) + __popc(b.y) +
          __popc(b.z) + __popc(b.w);
  }
  uint32_t total;
  uint32_t inc = block_incl_scan<256>(cnt, wt_tot, &total);
  if (wt < n_wt) toff_local[wt] = inc - cnt;
  if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

__global__ __launch_bounds__(1024) void scan_bsum(uint32_t* __restrict__ bsum, uint64_t n) {
  __shared__ uint32_t wt_tot[33];
  uint32_t carry = 0;
  for (uint64_t base = 0; base < n; base += 1024) {
    uint64_t i = base + threadIdx.x;
    uint32_t x = i < n ? bsum[i] : 0u;
    uint32_t total;
    uint32_t inc = block_incl_scan<1024>(x, wt_tot, &total);
    if (i < n) bsum[i] = carry + inc - x;
    carry += total;
  }
}

}  // namespace

cudaError_t launch_offsets(const uint32_t* mask, uint32_t* toff_local, uint32_t* bsum,
                           uint64_t n_wt, cudaStream_t s) {
  const uint64_t n_blk = (n_wt + kTilesPerBlk - 1) / kTilesPerBlk;
  offsets_local<<<(unsigned)n_blk, 256, 0, s>>>(mask, toff_local, bsum, n_wt);
  scan_bsum<<<1, 1024, 0, s>>>(bsum, n_blk);
  return cudaGetLastError();
}

}  // namespace scape
