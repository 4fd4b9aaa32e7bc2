// gc_aggregate.cu -- sum of several ranks' compressed gradients into one
// dense fp32 buffer.
//
// "分布式训练中的梯度压缩算法" 四 (gradient compression with All-Reduce):
// every worker compresses its local gradient, the compressed gradients are
// aggregated and decompressed.  With Top-K each rank has its own positions
// and, quantised, its own scales, so the aggregate is the sum of the ranks'
// decompressed sparse vectors, added in rank order:
//   out[i] = 0;  for w = 0 .. W-1: out[idx_w[j]] += v_w[j]   (binary32 adds)
//
// Rank w's indices are strictly increasing, so no two of its entries touch
// the same element and the rank order is the only order that matters.  The
// output is cut into ranges of kAggRange elements, one block each:
//   bounds     : for every rank, the first entry of each range (one thread
//                per entry boundary; each range is written exactly once).
//   accumulate : a block gathers the entries of its range, rank by rank, in
//                chunks into shared memory (all loads of a chunk in flight at
//                once), adds them to its shared accumulator in rank order
//                (a barrier between ranks) and writes its range once.
#include <algorithm>

#include "gc_internal.cuh"

namespace gc {
namespace {

constexpr int kAggShift = 13;
constexpr int kAggRange = 1 << kAggShift;   // output elements per block
constexpr int kAggThreads = 512;
constexpr int kAggSlots = 4096;             // gathered entries per chunk
constexpr int kAggMaxRanks = 1024;

// Per-rank stride of the index and value arrays: k rounded up to 4 entries,
// so every rank's entries start on a 16-byte boundary.
__host__ __device__ __forceinline__ int64_t round_up4(int64_t k) { return (k + 3) / 4 * 4; }

// start[w * (nblk + 1) + b] = first entry of rank w whose index is in range
// b or later (k when none).
__global__ void agg_bounds_kernel(const int32_t* __restrict__ idx, int W, int64_t k, int64_t n,
                                  int64_t nblk, int32_t* __restrict__ start,
                                  uint32_t* __restrict__ status) {
  const int64_t per = k + 1;  // boundary positions j = 0 .. k of one rank
  const int64_t total = (int64_t)W * per;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t w = t / per, j = t - w * per;
    const int32_t* iw = idx + w * round_up4(k);
    auto blk = [&](int64_t jj) -> int64_t {
      const int64_t v = iw[jj];
      if (v < 0 || v >= n) {
        atomicOr(status, kStatusScatterIndex);
        return v < 0 ? 0 : nblk - 1;
      }
      return v >> kAggShift;
    };
    int64_t lo = j == 0 ? 0 : blk(j - 1) + 1;
    int64_t hi = j == k ? nblk : blk(j);
    if (j > 0 && j < k && iw[j] <= iw[j - 1]) atomicOr(status, kStatusScatterIndex);
    lo = std::min<int64_t>(std::max<int64_t>(lo, 0), nblk);
    hi = std::min<int64_t>(hi, nblk);
    int32_t* sw = start + w * (nblk + 1);
    for (int64_t b = lo; b <= hi; ++b) sw[b] = (int32_t)j;
  }
}

struct AggSmem {
  float acc[kAggRange];
  float val[kAggSlots];
  uint16_t loc[kAggSlots];
  int32_t first[kAggMaxRanks + 1];  // rank w's entries of this range: [first, first + cnt)
  int32_t pre[kAggMaxRanks + 1];    // exclusive prefix of the counts
};

// Value of entry j of rank w: val[w*K + j] (K = k rounded up to 4), or for QSGD codes
// +-fl(q * scale) with rank w's codes at w * cb and scales at w * sf (sf a
// multiple of 4).
template <int BITS>
__device__ __forceinline__ float agg_value(const float* __restrict__ val,
                                           const uint8_t* __restrict__ codes,
                                           const float* __restrict__ scales, int64_t k,
                                           int64_t cb, int64_t mag, int64_t sf, int64_t G,
                                           int w, int64_t j) {
  if (BITS == 0) return val[(int64_t)w * round_up4(k) + j];
  const uint8_t* cw = codes + (int64_t)w * cb;
  const int64_t bit = j * BITS;
  const uint32_t q = (uint32_t)(cw[bit >> 3] >> (bit & 7)) & ((1u << BITS) - 1u);
  const bool neg = (cw[mag + (j >> 3)] >> (j & 7)) & 1u;
  const float m = __fmul_rn((float)q, scales[(int64_t)w * sf + j / G]);
  return neg ? -m : m;
}

template <int BITS>
__global__ void __launch_bounds__(kAggThreads) agg_accumulate_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ val,
    const uint8_t* __restrict__ codes, const float* __restrict__ scales, int W, int64_t k,
    int64_t cb, int64_t mag, int64_t sf, int64_t G, int64_t n, int64_t nblk,
    const int32_t* __restrict__ start, float* __restrict__ out, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char agg_smem_raw[];
  AggSmem& sm = *reinterpret_cast<AggSmem*>(agg_smem_raw);
  const int64_t b = blockIdx.x;
  const int64_t a = b << kAggShift;
  const int len = (int)std::min<int64_t>(kAggRange, n - a);
  for (int i = threadIdx.x; i < kAggRange; i += kAggThreads) sm.acc[i] = 0.0f;
  for (int w = threadIdx.x; w < W; w += kAggThreads) {
    // clamped to [0, k): bounds from invalid (flagged) indices stay in range
    const int32_t* sw = start + (int64_t)w * (nblk + 1);
    const int64_t f = std::min<int64_t>(std::max<int32_t>(sw[b], 0), k);
    const int64_t l = std::min<int64_t>(std::max<int32_t>(sw[b + 1], 0), k);
    sm.first[w] = (int32_t)f;
    // a range holds at most kAggRange entries of one rank (distinct indices)
    sm.pre[w] = (int32_t)std::min<int64_t>(l > f ? l - f : 0, kAggRange);  // scanned below
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t run = 0;
    for (int w = 0; w < W; ++w) {
      const int32_t c = sm.pre[w];
      sm.pre[w] = run;
      run += c;
    }
    sm.pre[W] = run;
  }
  __syncthreads();
  const int32_t total = sm.pre[W];
  // chunks of the block's entries in rank-major order
  for (int32_t c0 = 0; c0 < total; c0 += kAggSlots) {
    const int32_t c1 = min(c0 + kAggSlots, total);
    for (int32_t e = c0 + threadIdx.x; e < c1; e += kAggThreads) {
      int w = 0;  // rank of flat entry e: the last w with pre[w] <= e
      int lo = 0, hi = W - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.pre[mid] <= e) lo = mid;
        else hi = mid - 1;
      }
      w = lo;
      const int64_t j = (int64_t)sm.first[w] + (e - sm.pre[w]);
      const int64_t i = (int64_t)idx[(int64_t)w * round_up4(k) + j] - a;
      const bool ok = i >= 0 && i < len;
      if (!ok) atomicOr(status, kStatusScatterIndex);
      sm.loc[e - c0] = ok ? (uint16_t)i : (uint16_t)0xffffu;
      sm.val[e - c0] = agg_value<BITS>(val, codes, scales, k, cb, mag, sf, G, w, j);
    }
    __syncthreads();
    // rank by rank: within a rank the locations are distinct
    int w0 = 0;
    while (w0 < W && sm.pre[w0 + 1] <= c0) ++w0;
    for (int w = w0; w < W && sm.pre[w] < c1; ++w) {
      const int32_t e0 = max(sm.pre[w], c0), e1 = min(sm.pre[w + 1], c1);
      for (int32_t e = e0 + threadIdx.x; e < e1; e += kAggThreads) {
        const uint16_t l = sm.loc[e - c0];
        if (l != 0xffffu) sm.acc[l] = __fadd_rn(sm.acc[l], sm.val[e - c0]);
      }
      __syncthreads();
    }
  }
  __syncthreads();
  float* o = out + a;
  if (len == kAggRange) {
    for (int i = threadIdx.x; i < kAggRange / 4; i += kAggThreads)
      reinterpret_cast<float4*>(o)[i] = reinterpret_cast<const float4*>(sm.acc)[i];
  } else {
    for (int i = threadIdx.x; i < len; i += kAggThreads) o[i] = sm.acc[i];
  }
}

template <int BITS>
gc_status run_accumulate(gc_ctx* ctx, const int32_t* idx, const float* val, const uint8_t* codes,
                         const float* scales, int W, int64_t k, int64_t cb, int64_t mag,
                         int64_t sf, int64_t G, int64_t n, int64_t nblk, const int32_t* start,
                         float* out) {
  LaunchScope L(ctx, GC_PHASE_AGG_ACCUMULATE);
  agg_accumulate_kernel<BITS><<<(unsigned)nblk, kAggThreads, sizeof(AggSmem), ctx->stream>>>(
      idx, val, codes, scales, W, k, cb, mag, sf, G, n, nblk, start, out, ctx->ws.status);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace

gc_status prepare_aggregate_kernels() {
  const int bytes = (int)sizeof(AggSmem);
  const bool ok =
      cudaFuncSetAttribute(agg_accumulate_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
      cudaFuncSetAttribute(agg_accumulate_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
      cudaFuncSetAttribute(agg_accumulate_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
      cudaFuncSetAttribute(agg_accumulate_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
      cudaFuncSetAttribute(agg_accumulate_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
  return ok ? GC_OK : GC_ERR_CUDA;
}

int64_t aggregate_scratch_ints(int W, int64_t n) {
  return (int64_t)W * (ceil_div(n, kAggRange) + 1);
}

int aggregate_max_ranks() { return kAggMaxRanks; }

gc_status launch_aggregate(gc_ctx* ctx, int W, int64_t k, const int32_t* idx, const float* val,
                           const uint8_t* codes, const float* scales, int bits, int64_t group,
                           int64_t n, float* out) {
  if (n == 0) return GC_OK;
  const int64_t nblk = ceil_div(n, kAggRange);
  int32_t* start = reinterpret_cast<int32_t*>(ctx->ws.cand);
  {
    LaunchScope L(ctx, GC_PHASE_AGG_BOUNDS);
    const int64_t total = (int64_t)W * (k + 1);
    const int grid = (int)std::max<int64_t>(
        1, std::min<int64_t>(ceil_div(total, 256), (int64_t)ctx->num_sms * 8));
    agg_bounds_kernel<<<grid, 256, 0, ctx->stream>>>(idx, W, k, n, nblk, start, ctx->ws.status);
  }
  if (cudaGetLastError() != cudaSuccess) return GC_ERR_CUDA;
  if (bits == 0)
    return run_accumulate<0>(ctx, idx, val, nullptr, nullptr, W, k, 0, 0, 0, 1, n, nblk, start,
                             out);
  const int64_t mag = round_up((k * bits + 7) / 8, 16);
  const int64_t cb = mag + round_up((k + 7) / 8, 16);
  const int64_t G = group == 0 ? std::max<int64_t>(k, 1) : group;  // 0: one group of all k
  const int64_t sf = round_up(ceil_div(k, G), 4);  // rank stride: 16-byte aligned
  switch (bits) {
    case 1: return run_accumulate<1>(ctx, idx, nullptr, codes, scales, W, k, cb, mag, sf, G, n, nblk, start, out);
    case 2: return run_accumulate<2>(ctx, idx, nullptr, codes, scales, W, k, cb, mag, sf, G, n, nblk, start, out);
    case 4: return run_accumulate<4>(ctx, idx, nullptr, codes, scales, W, k, cb, mag, sf, G, n, nblk, start, out);
    default: return run_accumulate<8>(ctx, idx, nullptr, codes, scales, W, k, cb, mag, sf, G, n, nblk, start, out);
  }
}

}  // namespace gc
