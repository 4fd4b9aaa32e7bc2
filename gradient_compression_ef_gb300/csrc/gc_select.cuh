// gc_select.cuh -- block- and warp-level building blocks of the radix
// select shared by the per-call and the bucketed Top-K kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gc {

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Block-wide exclusive scan of one 32-bit value per thread (NT threads);
// returns the exclusive prefix and writes the block total.  warp_sums holds
// NT / 32 + 1 words.  Contains barriers: every thread must call it.
template <int NT>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* warp_sums,
                                               uint32_t* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = lane < NW ? warp_sums[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NW) warp_sums[lane] = wi - w;  // exclusive warp offsets
    if (lane == NW - 1) warp_sums[NW] = wi;
  }
  __syncthreads();
  const uint32_t res = warp_sums[warp] + incl - v;
  *total = warp_sums[NW];
  __syncthreads();
  return res;
}

// Over `bins` counts in shared memory (bin index = digit value), finds the
// digit D whose cumulative count from the top crosses `need`:
// above(D) < need <= above(D) + hist[D].  Writes D and above(D) (left
// untouched when need is 0 or exceeds the total) and returns the total of
// all bins.  Called by all NT threads; ends with a barrier.
template <int NT>
__device__ uint32_t find_digit(const uint32_t* hist, int bins, uint32_t need,
                               uint32_t* warp_sums, uint32_t* out_digit, uint32_t* out_above) {
  const int per = bins >= NT ? bins / NT : 1;
  const bool owner = (int)threadIdx.x * per < bins;
  // thread t owns bins [bins - per*(t+1), bins - per*t): thread 0 the top
  const int hi = bins - per * (int)threadIdx.x;
  uint32_t s = 0;
  if (owner)
    for (int b = hi - 1; b >= hi - per; --b) s += hist[b];
  uint32_t total;
  const uint32_t before = block_scan<NT>(s, warp_sums, &total);
  if (owner && before < need && need <= before + s) {
    uint32_t acc = before;
    for (int b = hi - 1; b >= hi - per; --b) {
      if (acc + hist[b] >= need) {
        *out_digit = (uint32_t)b;
        *out_above = acc;
        break;
      }
      acc += hist[b];
    }
  }
  __syncthreads();
  return total;
}

}  // namespace gc
