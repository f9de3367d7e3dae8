// Kernel interfaces of libscape (internal).
//
// Data layout in HBM (all allocations by the library):
//   theta, v      fp32[Np]            Np = N rounded up to 256
//   u, e          fp32[W][Np]
//   mask[2]       uint32[n_wt*8]      M_{t-1} / M_t, bit j of word i = coord 32i+j
//   vals          fp32[W][Kp]         compact b_w, ascending coordinate
//   bbar          fp32[Kp]            compact synchronized buffer
//   idx           uint32[Kp]          coordinates of the compact entries
//   toff_local    uint32[n_wt]        kept-count before each 256-coordinate tile,
//                                     counted from its 65536-coordinate block
//   bsum          uint32[n_blk]       kept-count before each block (after the scan)
// A "tile" is 256 consecutive coordinates = 8 mask words = one warp of 32
// threads x 8 coordinates; blocks are 256 tiles.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace scape {

constexpr int kMaxW = 64;
constexpr int kTile = 256;             // coordinates per warp tile
constexpr int kTilesPerBlk = 256;      // warp tiles per offsets block
constexpr uint32_t kMaxChunk = 65536;  // largest chunk (16-bit in-chunk index)

struct StreamArgs {
  const uint16_t* grads[kMaxW];
  float* u;
  float* e;
  float* vals;
  const uint32_t* mprev;
  const uint32_t* toff_local;
  const uint32_t* bsum;
  uint64_t N, Np, Kp, n_wt;
  float b1, c1;
};

struct UpdateArgs {
  float* theta;
  float* v;
  const float* vals;
  float* bbar;
  uint32_t* idx;
  const uint32_t* mprev;
  const uint32_t* toff_local;
  const uint32_t* bsum;
  uint64_t N, Kp, n_wt;
  int W;
  float b2, c2, lr, wd, eps, invW;
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
  uint64_t N, Np, Kp, n_ch, q;
  uint32_t C, k_full, k_last;
};

// Launchers; all enqueue on "s" and return cudaGetLastError().
cudaError_t launch_offsets(const uint32_t* mask, uint32_t* toff_local, uint32_t* bsum,
                           uint64_t n_wt, cudaStream_t s);
cudaError_t launch_stream_compact(const StreamArgs& a, int W, cudaStream_t s);
cudaError_t launch_reduce_update(const UpdateArgs& a, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, bool boot, cudaStream_t s);

int num_sms();

}  // namespace scape
