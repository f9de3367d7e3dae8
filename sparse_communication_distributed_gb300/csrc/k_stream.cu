// Kernel (a): the per-worker streaming pass of a SCAPE step.
//
// For every worker w and coordinate i (SCAPE, gist.science technical summary
// §2: first moment of AdamS, error feedback with residual buffers, the mask
// built one step earlier applied now):
//   u = b1*u + c1*g          (c1 = 1 - b1 in fp32)
//   a = e + u
//   b = M_{t-1}[i] ? a : +0
//   e = a - b
// and the kept b are packed, in ascending coordinate order, into worker w's
// compact buffer vals_w (the buffer a real data-parallel run would reduce).
//
// Mapping: one warp per 256-coordinate tile and worker, 8 consecutive
// coordinates per thread, so every thread issues one 16-byte load of bf16
// gradients and two 16-byte loads each of u and e (128-bit, coalesced), and
// reads one byte of the mask word its 4-lane group shares.  The packed
// position of a kept coordinate is the tile offset (from the offsets kernels)
// plus a warp scan of the per-thread mask-byte popcounts plus a popcount
// inside the byte.  HBM traffic per coordinate and worker: 2 (g) + 8 (u) +
// 8 (e) + 1/8 (mask) bytes, plus 4 bytes per kept value.
#include "scape_device.cuh"
#include "scape_kernels.cuh"

namespace scape {
namespace {

__global__ __launch_bounds__(256) void stream_compact(const StreamArgs p) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int w = blockIdx.y;
  const uint16_t* __restrict__ g = p.grads[w];
  float* __restrict__ u = p.u + (uint64_t)w * p.Np;
  float* __restrict__ e = p.e + (uint64_t)w * p.Np;
  float* __restrict__ vals = p.vals + (uint64_t)w * p.Kp;
  const float b1 = p.b1, c1 = p.c1;

  for (uint64_t wt = (uint64_t)blockIdx.x * 8 + warp; wt < p.n_wt; wt += (uint64_t)gridDim.x * 8) {
    const uint64_t i0 = wt * kTile + (uint64_t)lane * 8;
    const uint32_t word = __ldg(p.mprev + wt * 8 + (lane >> 2));
    const uint32_t byte = (word >> ((lane & 3) * 8)) & 0xFFu;
    const uint32_t cnt = __popc(byte);
    const uint32_t inc = warp_incl_scan(cnt, lane);
    const uint32_t rank0 = __ldg(p.toff_local + wt) + __ldg(p.bsum + (wt >> 8)) + inc - cnt;

    if (i0 + 8 <= p.N) {
      const uint4 gr = ld_stream_u4(g + i0);
      float4* up = reinterpret_cast<float4*>(u + i0);
      float4* ep = reinterpret_cast<float4*>(e + i0);
      const float4 u0 = up[0], u1 = up[1], e0 = ep[0], e1 = ep[1];
      float gf[8] = {bf16lo(gr.x), bf16hi(gr.x), bf16lo(gr.y), bf16hi(gr.y),
                     bf16lo(gr.z), bf16hi(gr.z), bf16lo(gr.w), bf16hi(gr.w)};
      float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      float ee[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const float un = (b1 * uu[j]) + (c1 * gf[j]);
        const float a = ee[j] + un;
        const bool m = (byte >> j) & 1u;
        const float b = m ? a : 0.0f;
        uu[j] = un;
        ee[j] = a - b;
        if (m) vals[rank0 + __popc(byte & ((1u << j) - 1u))] = b;
      }
      up[0] = make_float4(uu[0], uu[1], uu[2], uu[3]);
      up[1] = make_float4(uu[4], uu[5], uu[6], uu[7]);
      ep[0] = make_float4(ee[0], ee[1], ee[2], ee[3]);
      ep[1] = make_float4(ee[4], ee[5], ee[6], ee[7]);
    } else if (i0 < p.N) {
      const int nv = (int)(p.N - i0);
      for (int j = 0; j < nv; j++) {
        const float gj = bf16f(g[i0 + j]);
        const float un = (b1 * u[i0 + j]) + (c1 * gj);
        const float a = e[i0 + j] + un;
        const bool m = (byte >> j) & 1u;
        const float b = m ? a : 0.0f;
        u[i0 + j] = un;
        e[i0 + j] = a - b;
        if (m) vals[rank0 + __popc(byte & ((1u << j) - 1u))] = b;
      }
    }
  }
}

}  // namespace

cudaError_t launch_stream_compact(const StreamArgs& a, int W, cudaStream_t s) {
  const uint64_t tiles_per_cta = 8;
  uint64_t want = (a.n_wt + tiles_per_cta - 1) / tiles_per_cta;
  uint64_t cap = (uint64_t)num_sms() * 8 * 4 / (uint64_t)W + 1;  // a few waves of resident CTAs
  if (want > cap) want = cap;
  dim3 grid((unsigned)want, (unsigned)W);
  stream_compact<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace scape
