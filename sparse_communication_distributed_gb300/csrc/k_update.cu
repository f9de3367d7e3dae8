// Kernel (b): the synchronized buffer and the AdamS update of a SCAPE step.
//
// SCAPE reduces one sparse buffer per step and rebuilds the second-moment
// input from it (gist.science technical summary §2 "Single-Buffer
// Second-Moment Reconstruction"; abstract).  With W workers emulated in one
// memory the all-reduce is the fixed-order sum of the W compact buffers:
//   bbar = (vals_0 + vals_1 + ... + vals_{W-1}) * (1/W)   (left to right)
// and for every coordinate (bbar = +0 where M_{t-1} is clear):
//   v     = b2*v + c2*(bbar*bbar)                 (c2 = 1 - b2 in fp32)
//   theta = theta - lr*(bbar/(sqrt(v)+eps) + wd*theta)
// sqrt and / are the IEEE correctly rounded operations (no fast-math).  Off
// the mask bbar/(sqrt(v)+eps) is exactly +0, so the division is skipped there
// and +0 used in its place.  The kernel also writes bbar and the coordinate
// list idx of the compact entries (what a real run's collective returns).
//
// Mapping as in kernel (a): one warp per 256-coordinate tile, 8 coordinates
// per thread, two 16-byte loads and stores each of theta and v.  HBM traffic
// per coordinate: 8 (theta) + 8 (v) + 1/8 (mask) bytes, plus per kept entry
// 4W bytes of vals read and 8 bytes of bbar and idx written.
#include "scape_device.cuh"
#include "scape_kernels.cuh"

namespace scape {
namespace {

__device__ __forceinline__ float sync_value(const UpdateArgs& p, uint32_t r) {
  float s = p.vals[r];
  for (int w = 1; w < p.W; w++) s = s + p.vals[(uint64_t)w * p.Kp + r];
  return s * p.invW;
}

__global__ __launch_bounds__(256) void reduce_update(const UpdateArgs p) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const float b2 = p.b2, c2 = p.c2, lr = p.lr, wd = p.wd, eps = p.eps;

  for (uint64_t wt = (uint64_t)blockIdx.x * 8 + warp; wt < p.n_wt; wt += (uint64_t)gridDim.x * 8) {
    const uint64_t i0 = wt * kTile + (uint64_t)lane * 8;
    const uint32_t word = __ldg(p.mprev + wt * 8 + (lane >> 2));
    const uint32_t byte = (word >> ((lane & 3) * 8)) & 0xFFu;
    const uint32_t cnt = __popc(byte);
    const uint32_t inc = warp_incl_scan(cnt, lane);
    const uint32_t rank0 = __ldg(p.toff_local + wt) + __ldg(p.bsum + (wt >> 8)) + inc - cnt;

    if (i0 + 8 <= p.N) {
      float4* tp = reinterpret_cast<float4*>(p.theta + i0);
      float4* vp = reinterpret_cast<float4*>(p.v + i0);
      const float4 t0 = tp[0], t1 = tp[1], v0 = vp[0], v1 = vp[1];
      float th[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const bool m = (byte >> j) & 1u;
        float bb = 0.0f;
        if (m) {
          const uint32_t r = rank0 + __popc(byte & ((1u << j) - 1u));
          bb = sync_value(p, r);
          p.bbar[r] = bb;
          p.idx[r] = (uint32_t)(i0 + j);
        }
        const float vn = (b2 * vv[j]) + (c2 * (bb * bb));
        const float q = m ? bb / (sqrtf(vn) + eps) : 0.0f;
        vv[j] = vn;
        th[j] = th[j] - (lr * (q + (wd * th[j])));
      }
      tp[0] = make_float4(th[0], th[1], th[2], th[3]);
      tp[1] = make_float4(th[4], th[5], th[6], th[7]);
      vp[0] = make_float4(vv[0], vv[1], vv[2], vv[3]);
      vp[1] = make_float4(vv[4], vv[5], vv[6], vv[7]);
    } else if (i0 < p.N) {
      const int nv = (int)(p.N - i0);
      for (int j = 0; j < nv; j++) {
        const bool m = (byte >> j) & 1u;
        float bb = 0.0f;
        if (m) {
          const uint32_t r = rank0 + __popc(byte & ((1u << j) - 1u));
          bb = sync_value(p, r);
          p.bbar[r] = bb;
          p.idx[r] = (uint32_t)(i0 + j);
        }
        const float vn = (b2 * p.v[i0 + j]) + (c2 * (bb * bb));
        const float q = m ? bb / (sqrtf(vn) + eps) : 0.0f;
        p.v[i0 + j] = vn;
        p.theta[i0 + j] = p.theta[i0 + j] - (lr * (q + (wd * p.theta[i0 + j])));
      }
    }
  }
}

}  // namespace

cudaError_t launch_reduce_update(const UpdateArgs& a, cudaStream_t s) {
  uint64_t want = (a.n_wt + 7) / 8;
  uint64_t cap = (uint64_t)num_sms() * 8 * 4;
  if (want > cap) want = cap;
  reduce_update<<<(unsigned)want, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace scape
