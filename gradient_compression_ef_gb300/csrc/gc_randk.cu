// gc_randk.cu -- random sparsification with error feedback.
//
// "分布式训练中的梯度压缩算法" 二.2 随机稀疏化 (keep each element with
// probability p, mask = rand(n) < p) with the unsent entries left in the
// residual (error feedback, "梯度聚合通信优化实战方案" 梯度压缩原理):
//   c = g + e;  keep i when u_i < p, u_i the Philox-4x32-10 draw of element i
//   (the draw stochastic rounding uses);  emit the kept (i, c_i) in ascending
//   index order;  e'_i = +0 when kept, c_i otherwise.
//
// Two launches over the same partition (block i owns a contiguous range of
// 2048-element segments, a warp per segment):
//   mark  : c = g + e, the draws, e' written directly (so the kept entries
//           need no second, scattered write), and per segment the ordered
//           list of the kept (index, c) pairs; per block its total.
//   write : each block adds up the totals of the blocks before it, scans its
//           segments' list lengths and copies the lists to the output; the
//           last block writes the count.
#include <algorithm>

#include "gc_internal.cuh"
#include "gc_select.cuh"

namespace gc {
namespace {

constexpr int kRkThreads = 256;
constexpr int kRkWarps = kRkThreads / 32;

template <bool EF>
__global__ void __launch_bounds__(kRkThreads, 3) randk_mark_kernel(
    const float* __restrict__ grad, float* __restrict__ err, int64_t n, int64_t nseg, float p,
    uint64_t seed, uint64_t step, uint2* __restrict__ list, uint32_t* __restrict__ seg_cnt,
    uint32_t* __restrict__ block_tot) {
  __shared__ uint32_t tot;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = lanemask_lt();
  if (threadIdx.x == 0) tot = 0u;
  __syncthreads();
  int64_t s, s_hi;
  seg_range(nseg, gridDim.x, blockIdx.x, &s, &s_hi);
  for (int64_t seg = s + warp; seg < s_hi; seg += kRkWarps) {
    const int64_t l0 = seg << kSegShift;
    const int64_t l1 = std::min<int64_t>(l0 + kSegElems, n);
    uint2* out = list + l0;
    uint32_t cnt = 0u;
    for (int64_t p0 = l0; p0 < l1; p0 += 512) {
      float4 gv[4], ev[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = p0 + 128 * u + 4 * lane;
        if (i + 3 < l1) {
          gv[u] = __ldcs(reinterpret_cast<const float4*>(grad + i));
          if (EF) ev[u] = *reinterpret_cast<const float4*>(err + i);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = p0 + 128 * u + 4 * lane;
        float c[4];
        bool valid[4];
        if (i + 3 < l1) {
          c[0] = gv[u].x; c[1] = gv[u].y; c[2] = gv[u].z; c[3] = gv[u].w;
          if (EF) {
            c[0] = __fadd_rn(c[0], ev[u].x);
            c[1] = __fadd_rn(c[1], ev[u].y);
            c[2] = __fadd_rn(c[2], ev[u].z);
            c[3] = __fadd_rn(c[3], ev[u].w);
          }
          valid[0] = valid[1] = valid[2] = valid[3] = true;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            valid[j] = i + j < l1;
            c[j] = valid[j] ? grad[i + j] : 0.0f;
            if (EF && valid[j]) c[j] = __fadd_rn(c[j], err[i + j]);
          }
        }
        float ud[4];
        uniform4((uint64_t)i >> 2, seed, step, ud);  // lanes past n draw and discard
        bool keep[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) keep[j] = valid[j] && ud[j] < p;
        if (EF) {
          if (i + 3 < l1) {
            *reinterpret_cast<float4*>(err + i) =
                make_float4(keep[0] ? 0.0f : c[0], keep[1] ? 0.0f : c[1], keep[2] ? 0.0f : c[2],
                            keep[3] ? 0.0f : c[3]);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (valid[j]) err[i + j] = keep[j] ? 0.0f : c[j];
          }
        }
        // ordered append: index order is (lane, j) within the row
        const uint32_t b0 = __ballot_sync(0xffffffffu, keep[0]);
        const uint32_t b1 = __ballot_sync(0xffffffffu, keep[1]);
        const uint32_t b2 = __ballot_sync(0xffffffffu, keep[2]);
        const uint32_t b3 = __ballot_sync(0xffffffffu, keep[3]);
        uint32_t pos = cnt + __popc(b0 & lt) + __popc(b1 & lt) + __popc(b2 & lt) +
                       __popc(b3 & lt);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (keep[j]) out[pos++] = make_uint2(__float_as_uint(c[j]), (uint32_t)(i + j));
        cnt += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
      }
    }
    if (lane == 0) {
      seg_cnt[seg] = cnt;
      atomicAdd(&tot, cnt);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) block_tot[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kRkThreads) randk_write_kernel(
    int64_t nseg, const uint2* __restrict__ list, const uint32_t* __restrict__ seg_cnt,
    const uint32_t* __restrict__ block_tot, int32_t* __restrict__ idx_out,
    float* __restrict__ val_out, int64_t capacity, int64_t* __restrict__ count_out,
    uint32_t* __restrict__ status) {
  __shared__ uint32_t warp_sums[kRkThreads / 32 + 1];
  __shared__ uint64_t base_s;
  __shared__ uint32_t offs[kRkThreads], cnts[kRkThreads];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // entries kept by the blocks before this one (64-bit: n may be near 2^31)
  uint64_t before = 0;
  for (int b = threadIdx.x; b < (int)blockIdx.x; b += kRkThreads) before += block_tot[b];
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (threadIdx.x == 0) base_s = 0;
  __syncthreads();
  if (lane == 0 && before) atomicAdd(reinterpret_cast<unsigned long long*>(&base_s), before);
  __syncthreads();
  uint64_t base = base_s;
  int64_t s, s_hi;
  seg_range(nseg, gridDim.x, blockIdx.x, &s, &s_hi);
  // segments in rounds of kRkThreads: scan their lengths, then a warp per
  // segment copies its list
  for (int64_t r0 = s; r0 < s_hi; r0 += kRkThreads) {
    const int64_t sg = r0 + threadIdx.x;
    const uint32_t c = sg < s_hi ? seg_cnt[sg] : 0u;
    uint32_t total;
    offs[threadIdx.x] = block_scan<kRkThreads>(c, warp_sums, &total);
    cnts[threadIdx.x] = c;
    __syncthreads();
    const int nr = (int)std::min<int64_t>(kRkThreads, s_hi - r0);
    for (int q = warp; q < nr; q += kRkWarps) {
      const uint32_t cnt = cnts[q];
      const uint64_t o = base + offs[q];
      const uint2* in = list + ((r0 + q) << kSegShift);
      for (uint32_t j = lane; j < cnt; j += 32) {
        const uint64_t pos = o + j;
        const uint2 e = in[j];
        if (pos < (uint64_t)capacity) {
          idx_out[pos] = (int32_t)e.y;
          val_out[pos] = __uint_as_float(e.x);
        }
      }
    }
    base += total;
    __syncthreads();
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    *count_out = (int64_t)base;
    if (base > (uint64_t)capacity) atomicOr(status, kStatusTopkOverflow);
  }
}

}  // namespace

gc_status launch_ef_randk(gc_ctx* ctx, const float* grad, float* err, int64_t n, float p,
                          uint64_t seed, uint64_t step, int32_t* idx_out, float* val_out,
                          int64_t capacity, int64_t* count_out) {
  const int64_t nseg = ceil_div(n, kSegElems);
  uint2* list = ctx->ws.cand;
  uint32_t* seg_cnt = reinterpret_cast<uint32_t*>(ctx->ws.vals);
  // per-block totals: a scratch array that every Top-K call writes before
  // it reads it (unlike the histograms and tile_kept, which must stay zero)
  uint32_t* block_tot = ctx->ws.tile_above;
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>({(int64_t)ctx->num_sms * 8, nseg, (int64_t)kMaxTiles}));
  cudaStream_t s = ctx->stream;
  {
    LaunchScope L(ctx, GC_PHASE_RANDK_MARK);
    if (err)
      randk_mark_kernel<true><<<grid, kRkThreads, 0, s>>>(grad, err, n, nseg, p, seed, step,
                                                          list, seg_cnt, block_tot);
    else
      randk_mark_kernel<false><<<grid, kRkThreads, 0, s>>>(grad, err, n, nseg, p, seed, step,
                                                           list, seg_cnt, block_tot);
  }
  {
    LaunchScope L(ctx, GC_PHASE_RANDK_WRITE);
    randk_write_kernel<<<grid, kRkThreads, 0, s>>>(nseg, list, seg_cnt, block_tot, idx_out,
                                                   val_out, capacity, count_out,
                                                   ctx->ws.status);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace gc
