// Device helpers shared by the libscape kernels (internal).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace scape {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Debug builds (-DSCAPE_DEBUG_CHECKS) check every index that depends on the
// applied mask carrying exactly k_c bits per chunk.  A failed check records
// the first failure's code and coordinate in dbg[0..3] (code, count, where
// low, where high) and skips the access; nothing traps.  Release builds
// compile the checks away.
#ifdef SCAPE_DEBUG_CHECKS
__device__ __forceinline__ bool dbg_ok(uint32_t* dbg, bool ok, uint32_t code, uint64_t where) {
  if (!ok && dbg) {
    if (atomicCAS(dbg, 0u, code) == 0u) {
      dbg[2] = (uint32_t)where;
      dbg[3] = (uint32_t)(where >> 32);
    }
    atomicAdd(dbg + 1, 1u);
  }
  return ok;
}
#define SCAPE_CHECK(dbg, cond, code, where) (::scape::dbg_ok((dbg), (cond), (code), (where)))
#else
#define SCAPE_CHECK(dbg, cond, code, where) (true)
#endif

// check codes
enum : uint32_t {
  CHK_VALS_WRITE = 1,   // kept value past the chunk's k
  CHK_VALS_STAGE = 2,   // staged kept values past the chunk's k
  CHK_BBAR = 3,         // synchronized-sum position past the chunk's k
  CHK_IDX = 4,          // coordinate-list position past the chunk's k
  CHK_OWNER_KEY = 5,    // kept value read past the chunk's k (selection)
  CHK_CAND = 6,         // candidate list overflow
  CHK_SELECT_VALS = 7,  // standalone select: kept value read past k
  CHK_CHUNK = 8         // chunk extends past N
};

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint32_t y = __shfl_up_sync(kFull, x, d);
    if (lane >= d) x += y;
  }
  return x;
}

// Block-wide inclusive scan of one value per thread; "warp_tot" is shared
// scratch of at least blockDim.x/32 + 1 entries.  Returns the inclusive
// prefix; *total receives the block total.  Contains __syncthreads().
template <int NT>
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t x, uint32_t* warp_tot,
                                                    uint32_t* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t inc = warp_incl_scan(x, lane);
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    uint32_t t = lane < NW ? warp_tot[lane] : 0u;
    uint32_t ti = warp_incl_scan(t, lane);
    if (lane < NW) warp_tot[lane] = ti - t;  // exclusive warp offsets
    if (lane == NW - 1) warp_tot[NW] = ti;
  }
  __syncthreads();
  uint32_t r = inc + warp_tot[wid];
  *total = warp_tot[NW];
  __syncthreads();
  return r;
}

// Finds, in hist[0..nb) (nb a power of two), the bin holding the r-th largest
// element (1-based, r <= total): out[0] = bin, out[1] = count in the bins above
// it, out[2] = its count.  Block-wide (NT threads); ends with __syncthreads().
template <int NT>
__device__ void find_bin(const uint32_t* hist, int nb, uint32_t r, uint32_t* scan,
                         uint32_t* out) {
  const int t = threadIdx.x;
  const int bpt = nb >= NT ? nb / NT : 1;
  const int b0 = t * bpt;
  uint32_t s = 0;
  if (b0 < nb)
    for (int j = 0; j < bpt; j++) s += hist[b0 + j];
  uint32_t total;
  const uint32_t inc = block_incl_scan<NT>(s, scan, &total);
  const uint32_t above = total - inc;
  if (b0 < nb && above < r && r <= above + s) {
    uint32_t acc = above;
    for (int j = bpt - 1; j >= 0; j--) {
      const uint32_t h = hist[b0 + j];
      if (acc + h >= r) {
        out[0] = (uint32_t)(b0 + j);
        out[1] = acc;
        out[2] = h;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Programmatic dependent launch.  A grid launched with the programmatic
// stream serialization attribute may start before the grid ahead of it on the
// stream has finished; grid_dependency_wait() returns once that grid has
// completed and its memory is visible (at once for a plain launch), and no
// thread touches global memory before it.  grid_launch_dependents() lets the
// next such grid launch; it then waits in its own grid_dependency_wait().
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Streaming 8- and 16-byte loads that are not kept in L1 (read-once data).
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace scape
