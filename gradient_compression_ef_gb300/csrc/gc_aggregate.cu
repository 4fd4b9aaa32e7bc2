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
// output is cut into ranges of kAggRange elements, one warp each:
//   bounds     : for every rank, the first entry of each range (threads
//                stride over the rank's entry boundaries eight at a time,
//                loading the next eight while they write; each range is
//                written exactly once).
//   accumulate : a warp takes the ranks 32 at a time and packs their
//                entries of its range into one flat list, rank after rank,
//                read in rows of 32 (lane e of a row finds its rank from a
//                ballot of the ranks that start before the row and a
//                redux of those that start in it; three rows of loads in
//                flight at once).  It adds each row to its own accumulator
//                one rank at a time (__syncwarp between ranks) and writes
//                its range once.  Warps share nothing, so no block barrier
//                holds a range back; each SM keeps forty-eight warps, each
//                loading its next range's bounds while it works on one.
#include <algorithm>

#include "gc_internal.cuh"

namespace gc {
namespace {

constexpr int kAggShift = 10;
constexpr int kAggRange = 1 << kAggShift;   // output elements per warp
constexpr int kAggWarps = 8;                // warps (ranges) per block
constexpr int kAggThreads = 32 * kAggWarps;
constexpr int kAggMaxRanks = 1024;

// Per-rank stride of the index and value arrays: k rounded up to 4 entries,
// so every rank's entries start on a 16-byte boundary.
__host__ __device__ __forceinline__ int64_t round_up4(int64_t k) { return (k + 3) / 4 * 4; }

// start[w * (nblk + 1) + b] = first entry of rank w whose index is in range
// b or later (k when none).  Boundary position j (0 .. k) of rank w owns the
// ranges (range(idx[j-1]), range(idx[j])], so every range is written by
// exactly one position.
constexpr int kBoundsPer = 8;   // boundary positions per thread and step (two 16-byte loads)
constexpr int kBoundsThreads = 256;
constexpr int kBoundsBlocksPerSm = 6;

__global__ void __launch_bounds__(kBoundsThreads, kBoundsBlocksPerSm) agg_bounds_kernel(
    const int32_t* __restrict__ idx, int W, int64_t k, int64_t n, int64_t nblk,
    int32_t* __restrict__ start, uint32_t* __restrict__ status) {
  // rank w = blockIdx.y; the blocks of a rank stride over its positions
  // 0 .. k, kBoundsPer at a time, loading the next step's indices while
  // they write this step's boundaries
  const int64_t w = blockIdx.y;
  const int32_t* iw = idx + w * round_up4(k);
  int32_t* sw = start + w * (nblk + 1);
  // positions and strides in 32 bits: k < 2^31 and a stride < 2^31, so
  // j0 + stride < 2^32
  const uint32_t kk = (uint32_t)k, nb = (uint32_t)nblk, n32 = (uint32_t)n;
  const uint32_t stride = gridDim.x * kBoundsThreads * kBoundsPer;
  // indices of positions j0 - 1 .. j0 + kBoundsPer - 1 (0 where absent)
  auto load = [&](uint32_t j0, int32_t (&v)[kBoundsPer + 1]) {
#pragma unroll
    for (int u = 0; u <= kBoundsPer; ++u) v[u] = 0;
    if (j0 > kk) return;
    if (j0 > 0) v[0] = iw[j0 - 1];
    if (j0 + kBoundsPer <= kk) {
#pragma unroll
      for (int q = 0; q < kBoundsPer / 4; ++q) {
        const int4 x = *reinterpret_cast<const int4*>(iw + j0 + 4 * q);
        v[4 * q + 1] = x.x; v[4 * q + 2] = x.y; v[4 * q + 3] = x.z; v[4 * q + 4] = x.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kBoundsPer; ++u)
        if (j0 + u < kk) v[1 + u] = iw[j0 + u];
    }
  };
  // the range of an index; one outside [0, n) (negative ones are large as
  // unsigned) is flagged and taken as the last range
  bool bad = false;
  auto range_of = [&](int32_t x) -> uint32_t {
    bad |= (uint32_t)x >= n32;
    return min((uint32_t)x >> kAggShift, nb - 1);
  };
  uint32_t j0 = (blockIdx.x * kBoundsThreads + threadIdx.x) * kBoundsPer;
  int32_t v[kBoundsPer + 1], nv[kBoundsPer + 1];
  load(j0, v);
  for (; j0 <= kk; j0 += stride) {
    load(j0 + stride, nv);
    // c[u] = the range of position j0 + u - 1 (nb for position k, and the
    // one before it past k), c[0] that of position j0 - 1 (-1 before 0)
    int32_t c[kBoundsPer + 1];
    if (j0 > 0 && j0 + kBoundsPer <= kk) {
      // a quad inside the rank's entries: no position is 0 or k
#pragma unroll
      for (int u = 0; u <= kBoundsPer; ++u) c[u] = (int32_t)range_of(v[u]);
#pragma unroll
      for (int u = 1; u <= kBoundsPer; ++u) bad |= v[u] <= v[u - 1];
    } else {
      c[0] = j0 > 0 ? (int32_t)range_of(v[0]) : -1;
#pragma unroll
      for (int u = 1; u <= kBoundsPer; ++u) {
        const uint32_t j = j0 + u - 1;
        c[u] = j < kk ? (int32_t)range_of(v[u]) : j == kk ? (int32_t)nb : c[u - 1];
        bad |= j > 0 && j < kk && v[u] <= v[u - 1];
      }
    }
    int32_t hi = c[0];
#pragma unroll
    for (int u = 1; u <= kBoundsPer; ++u) hi = max(hi, c[u]);
    // ranges c[0] + 1 .. max c (at most nb): each starts at the first
    // position whose range reaches it
    for (int32_t b = c[0] + 1; b <= hi; ++b) {
      uint32_t j = j0 + kBoundsPer - 1;
#pragma unroll
      for (int u = kBoundsPer - 1; u >= 1; --u) j = c[u] >= b ? j0 + u - 1 : j;
      sw[b] = (int32_t)j;
    }
#pragma unroll
    for (int u = 0; u <= kBoundsPer; ++u) v[u] = nv[u];
  }
  if (bad) atomicOr(status, kStatusScatterIndex);
}

// Shared memory of one warp: the accumulator of its range, and for the
// current group of 32 ranks the non-empty ones in rank order (their lane in
// the group and the offset from a flat-list position to the rank's entry).
// Aligned to 16 bytes: the accumulator is cleared and written as float4.
struct __align__(16) AggWarpSmem {
  float acc[kAggRange];
  int2 nz[32];
};
static_assert(sizeof(AggWarpSmem) % 16 == 0, "float4 access to each warp's accumulator");

// Value of entry j of rank w: val[w*K + j] (K = k rounded up to 4), or for QSGD codes
// +-fl(q * scale) with rank w's codes at w * cb and scales at w * sf (sf a
// multiple of 4).  Entries and groups fit 32 bits (indices are int32, so
// k < 2^31); the group of entry j is j >> gshift for a power-of-two group
// (POW2), else j / G.
template <int BITS, bool POW2>
__device__ __forceinline__ float agg_value(const float* __restrict__ val,
                                           const uint8_t* __restrict__ codes,
                                           const float* __restrict__ scales, int64_t K,
                                           int64_t cb, int64_t mag, int64_t sf, uint32_t G,
                                           int gshift, int64_t w, uint32_t j) {
  if (BITS == 0) return val[w * K + j];
  const uint8_t* cw = codes + w * cb;
  constexpr int kPerByte = (BITS >= 8 || BITS == 0) ? 1 : 8 / BITS;  // codes per byte
  constexpr int kByteShift = BITS == 8 ? 0 : BITS == 4 ? 1 : BITS == 2 ? 2 : 3;
  const uint32_t q = (uint32_t)(cw[j >> kByteShift] >> ((j & (kPerByte - 1)) * BITS)) &
                     ((1u << BITS) - 1u);
  const bool neg = (cw[mag + (j >> 3)] >> (j & 7)) & 1u;
  const uint32_t g = POW2 ? j >> gshift : j / G;
  const float m = __fmul_rn((float)q, scales[w * sf + g]);
  return neg ? -m : m;
}

constexpr int kAggRows = 3;  // rows of 32 flat entries whose loads are in flight together
template <int BITS>
constexpr int agg_blocks_per_sm() { return BITS == 0 ? 5 : 6; }

template <int BITS, bool POW2>
__global__ void __launch_bounds__(kAggThreads, agg_blocks_per_sm<BITS>()) agg_accumulate_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ val,
    const uint8_t* __restrict__ codes, const float* __restrict__ scales, int W, int64_t k,
    int64_t cb, int64_t mag, int64_t sf, uint32_t G, int gshift, int64_t n, int64_t nblk,
    const int32_t* __restrict__ start, float* __restrict__ out, uint32_t* __restrict__ status) {
  __shared__ AggWarpSmem warps[kAggWarps];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  AggWarpSmem& sm = warps[wi];
  const int64_t K = round_up4(k);
  const int64_t stride = (int64_t)gridDim.x * kAggWarps;
  const uint32_t lanes_le = 0xffffffffu >> (31 - lane);
  bool bad = false;
  // lane r: the first entries of rank r0 + r in ranges bb and bb + 1
  // (0, 0 past the last rank or range)
  auto load_bounds = [&](int r0, int64_t bb, int32_t& lo, int32_t& hi) {
    lo = 0;
    hi = 0;
    if (bb < nblk && lane < min(32, W - r0)) {
      const int32_t* sw = start + (int64_t)(r0 + lane) * (nblk + 1);
      lo = sw[bb];
      hi = sw[bb + 1];
    }
  };
  // persistent warps: the first group's bounds of the next range load while
  // the warp works on this one
  int64_t b = (int64_t)blockIdx.x * kAggWarps + wi;
  int32_t next_lo, next_hi;
  load_bounds(0, b, next_lo, next_hi);
  for (; b < nblk; b += stride) {
    int32_t blo = next_lo, bhi = next_hi;
    load_bounds(0, b + stride, next_lo, next_hi);
    const int64_t a = b << kAggShift;
    const int32_t a32 = (int32_t)a;  // n <= 2^31 - 1
    const uint32_t len = (uint32_t)std::min<int64_t>(kAggRange, n - a);
    __syncwarp();  // the previous range's output reads are done
#pragma unroll
    for (int q = 0; q < kAggRange / 128; ++q)
      reinterpret_cast<float4*>(sm.acc)[q * 32 + lane] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int r0 = 0; r0 < W; r0 += 32) {
      if (r0 > 0) load_bounds(r0, b, blo, bhi);
      // lane r: rank r0 + r's first entry and count in the range (clamped to
      // [0, k): bounds from invalid, flagged indices stay in range; a range
      // holds at most kAggRange entries of one rank), and the position of
      // its entries in the warp's flat list (a scan)
      const int64_t f64 = std::min<int64_t>(std::max<int32_t>(blo, 0), k);
      const int64_t l64 = std::min<int64_t>(std::max<int32_t>(bhi, 0), k);
      const int32_t f = (int32_t)f64;
      const int32_t cnt = (int32_t)std::min<int64_t>(l64 > f64 ? l64 - f64 : 0, kAggRange);
      int32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
      const int32_t pre = incl - cnt;
      const bool nonempty = cnt > 0;
      // the non-empty ranks in order: the i-th one covers flat positions
      // [pre, pre + cnt) and its entry j = position + (f - pre)
      const uint32_t ne = __ballot_sync(0xffffffffu, nonempty);
      __syncwarp();  // the previous group's reads of nz (and the clearing) are done
      if (nonempty) sm.nz[__popc(ne & (lanes_le >> 1))] = make_int2(lane, f - pre);
      __syncwarp();
      for (int32_t c0 = 0; c0 < total; c0 += 32 * kAggRows) {
        // each lane's flat entries of this chunk: their rank (the non-empty
        // ranks that start before a row, plus those that start in it at or
        // before the lane), then all loads in flight
        int32_t iq[kAggRows], rq[kAggRows];
        float vq[kAggRows];
#pragma unroll
        for (int t = 0; t < kAggRows; ++t) {
          const int32_t row = c0 + 32 * t;
          iq[t] = 0;
          vq[t] = 0.0f;
          rq[t] = -1;
          if (row >= total) continue;  // warp-uniform
          const bool in_row = nonempty && pre >= row && pre < row + 32;
          const uint32_t starts = __reduce_or_sync(0xffffffffu, in_row ? 1u << (pre - row) : 0u);
          const int before = __popc(__ballot_sync(0xffffffffu, nonempty && pre < row));
          const int e = row + lane;
          if (e < total) {
            const int ri = before + __popc(starts & lanes_le) - 1;
            const int2 z = sm.nz[ri];
            const int64_t w = r0 + z.x;
            const uint32_t j = (uint32_t)(e + z.y);
            iq[t] = idx[w * K + j];
            vq[t] = agg_value<BITS, POW2>(val, codes, scales, K, cb, mag, sf, G, gshift, w, j);
            rq[t] = ri;
          }
        }
        // adds in rank order: one round per rank present in the row (within
        // a rank the locations are distinct; the warp meets between ranks)
#pragma unroll
        for (int t = 0; t < kAggRows; ++t) {
          const int32_t row = c0 + 32 * t;
          if (row >= total) break;  // warp-uniform
          const int lo = __shfl_sync(0xffffffffu, rq[t], 0);
          const int hi = __shfl_sync(0xffffffffu, rq[t], min(31, total - 1 - row));
          for (int r = lo; r <= hi; ++r) {
            if (rq[t] == r) {
              const uint32_t i = (uint32_t)iq[t] - (uint32_t)a32;
              if (iq[t] >= 0 && i < len) sm.acc[i] = __fadd_rn(sm.acc[i], vq[t]);
              else bad = true;
            }
            __syncwarp();
          }
        }
      }
    }
    float* o = out + a;
    if (len == kAggRange) {
#pragma unroll
      for (int q = 0; q < kAggRange / 128; ++q)
        reinterpret_cast<float4*>(o)[q * 32 + lane] =
            reinterpret_cast<const float4*>(sm.acc)[q * 32 + lane];
    } else {
      for (int i = lane; i < (int)len; i += 32) o[i] = sm.acc[i];
    }
  }
  if (bad) atomicOr(status, kStatusScatterIndex);
}

template <int BITS>
gc_status run_accumulate(gc_ctx* ctx, const int32_t* idx, const float* val, const uint8_t* codes,
                         const float* scales, int W, int64_t k, int64_t cb, int64_t mag,
                         int64_t sf, int64_t G, int64_t n, int64_t nblk, const int32_t* start,
                         float* out) {
  LaunchScope L(ctx, GC_PHASE_AGG_ACCUMULATE);
  // k < 2^31 (int32 indices): G fits 32 bits once clamped to k
  const uint32_t G32 = (uint32_t)std::min<int64_t>(std::max<int64_t>(G, 1), INT32_MAX);
  int gshift = -1;
  if ((G32 & (G32 - 1)) == 0)
    for (gshift = 0; (1u << gshift) != G32; ++gshift) {}
  // persistent: as many blocks as fit on the GPU at once, at most one range a warp
  const unsigned grid = (unsigned)std::min<int64_t>(
      ceil_div(nblk, kAggWarps), (int64_t)std::max(ctx->num_sms, 1) * agg_blocks_per_sm<BITS>());
  if constexpr (BITS != 0) {
    if (gshift < 0) {
      agg_accumulate_kernel<BITS, false><<<grid, kAggThreads, 0, ctx->stream>>>(
          idx, val, codes, scales, W, k, cb, mag, sf, G32, gshift, n, nblk, start, out,
          ctx->ws.status);
      return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
    }
  }
  agg_accumulate_kernel<BITS, true><<<grid, kAggThreads, 0, ctx->stream>>>(
      idx, val, codes, scales, W, k, cb, mag, sf, G32, std::max(gshift, 0), n, nblk, start, out,
      ctx->ws.status);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace

gc_status prepare_aggregate_kernels() {
  // static shared memory only (34 KB a block); prefer the largest carve-out
  // so that six blocks (forty-eight ranges) fit on an SM
  auto carve = [](auto kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) ==
           cudaSuccess;
  };
  const bool ok = carve(agg_accumulate_kernel<0, true>) && carve(agg_accumulate_kernel<1, true>) &&
                  carve(agg_accumulate_kernel<2, true>) && carve(agg_accumulate_kernel<4, true>) &&
                  carve(agg_accumulate_kernel<8, true>) && carve(agg_accumulate_kernel<1, false>) &&
                  carve(agg_accumulate_kernel<2, false>) && carve(agg_accumulate_kernel<4, false>) &&
                  carve(agg_accumulate_kernel<8, false>);
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
    // enough blocks over all ranks to fill the GPU once, at most one step a thread
    const int64_t per_rank = std::max<int64_t>(
        1, (int64_t)std::max(ctx->num_sms, 1) * kBoundsBlocksPerSm / W);
    const dim3 grid((unsigned)std::min<int64_t>(
                        ceil_div(ceil_div(k + 1, kBoundsPer), kBoundsThreads), per_rank),
                    (unsigned)W);
    agg_bounds_kernel<<<grid, kBoundsThreads, 0, ctx->stream>>>(idx, W, k, n, nblk, start,
                                                                 ctx->ws.status);
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
