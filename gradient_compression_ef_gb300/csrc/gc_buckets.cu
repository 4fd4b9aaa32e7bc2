// gc_buckets.cu -- error feedback + exact Top-K over every bucket of a flat
// gradient, one kernel launch per pass for all buckets.
//
// Per bucket the result is that of gc_ef_topk on the bucket's slice
// ("分布式训练中的梯度压缩算法" 二.2 Top-K; "4、梯度累积与梯度压缩" 4.2.1 and
// 4.3, which compresses bucket by bucket; "梯度聚合通信优化实战方案" Python
// 演示 error_feedback_compress): c = g + e, keep the k_b entries of largest
// |c| (ties: smaller index), emit them in ascending index order, e' = c with
// the kept entries cleared.
//
// Work unit: a segment of 2048 consecutive elements of one bucket, owned by
// one warp.  Each pass gives every block a contiguous range of segments; a
// block that reaches the end of a bucket's part of its range flushes its
// shared-memory histogram and takes a ticket, and the last block of the
// bucket (the number of blocks per bucket is fixed by the plan) finishes
// that bucket's selection step -- no block ever waits for another.
//   hist    : c = g + e written over e; 12-bit histogram of the key bits(|c|)
//             per bucket; last block: first-level bin B.
//   collect : per segment, the entries with bin >= B in index order (the
//             kept set is among them) with their count and the count above
//             B; histogram of bits 18..8 of the bin-B entries; last block:
//             second digit B2.
//   refine  : per segment, entries above (B, B2); the (B, B2) entries are
//             set aside with a histogram of bits 7..0; last block: exact
//             threshold key T, kept ties per segment, and the per-segment
//             output offsets of the bucket (one block scan).
//   write   : per segment, the ordered (index, value) writes (warp ballots)
//             and, without quantisation, e' = +0 at the kept positions.
#include <algorithm>
#include <vector>

#include "gc_internal.cuh"
#include "gc_select.cuh"

namespace gc {
namespace {

constexpr int kBkHistThreads = 1024;
constexpr int kBkThreads = 256;
constexpr int kPass = 512;            // elements a warp loads at once (4 x float4 per lane)
constexpr uint32_t kNone = 0xffffffffu;

__device__ __forceinline__ int64_t dev_round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// Warp 0 of block 0: byte / float offsets of every bucket's QSGD codes and
// scales for (bits, group), the running sums of gc_codes_bytes(k_b) and of
// gc_scales_floats(k_b) rounded up to 4 floats.
__device__ void layout_quant_outputs(const BucketWs& w, int bits, int64_t group, int lane) {
  int64_t carry_c = 0, carry_s = 0;
  for (int b0 = 0; b0 < w.nb; b0 += 32) {
    const int b = b0 + lane;
    int64_t cb = 0, sf = 0;
    if (b < w.nb) {
      const int64_t k = w.desc[b].k;
      cb = dev_round_up((k * bits + 7) / 8, 16) + dev_round_up((k + 7) / 8, 16);
      sf = dev_round_up((k + group - 1) / group, 4);
    }
    int64_t ic = cb, is = sf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t tc = __shfl_up_sync(0xffffffffu, ic, o);
      const int64_t ts = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) {
        ic += tc;
        is += ts;
      }
    }
    if (b < w.nb) {
      w.qoff[2 * b] = carry_c + ic - cb;
      w.qoff[2 * b + 1] = carry_s + is - sf;
    }
    carry_c += __shfl_sync(0xffffffffu, ic, 31);
    carry_s += __shfl_sync(0xffffffffu, is, 31);
  }
}

// ---------------------------------------------------------------------------
// hist: c = g + e and the first-level histogram.
// ---------------------------------------------------------------------------
template <bool EF>
__global__ void __launch_bounds__(kBkHistThreads, 1) bk_hist_kernel(
    const float* __restrict__ grad, float* __restrict__ err, BucketWs w, int qbits,
    int64_t qgroup) {
  constexpr int NW = kBkHistThreads / 32;
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t warp_sums[NW + 1];
  __shared__ uint32_t digit, above;
  __shared__ int last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (blockIdx.x == 0 && warp == 0 && qbits > 0) layout_quant_outputs(w, qbits, qgroup, lane);
  for (int i = threadIdx.x; i < kHistBins; i += kBkHistThreads) h[i] = 0u;
  __syncthreads();
  int64_t s, s_hi;
  seg_range(w.nseg, gridDim.x, blockIdx.x, &s, &s_hi);
  while (s < s_hi) {
    const int b = w.seg_bucket[s];
    const BucketDesc* dp = w.desc + b;
    const int32_t seg_first = dp->seg_first, bn = dp->n, bk = dp->k;
    const int64_t sub_hi = std::min<int64_t>(s_hi, (int64_t)seg_first + dp->nseg);
    const bool select = bk > 0;
    const float* g = grad + dp->start;
    float* e = EF ? err + dp->start : nullptr;
    for (int64_t seg = s + warp; seg < sub_hi; seg += NW) {
      // bucket-local offsets fit 32 bits (n <= 2^31 - 1)
      const int32_t l0 = (int32_t)(seg - seg_first) << kSegShift;
      const int32_t l1 = min(l0 + kSegElems, bn);
      for (int32_t p = l0; p < l1; p += kPass) {
        const float4* gp = reinterpret_cast<const float4*>(g + p) + lane;
        float4* ep = reinterpret_cast<float4*>(e + p) + lane;
        const int32_t rem = l1 - p - 4 * lane;  // elements from this lane's first one on
        float4 gv[4], ev[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (128 * u + 3 < rem) {
            gv[u] = __ldcs(gp + 32 * u);
            if (EF) ev[u] = ep[32 * u];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (128 * u + 3 < rem) {
            float4 c = gv[u];
            if (EF) {
              c.x = __fadd_rn(c.x, ev[u].x);
              c.y = __fadd_rn(c.y, ev[u].y);
              c.z = __fadd_rn(c.z, ev[u].z);
              c.w = __fadd_rn(c.w, ev[u].w);
              ep[32 * u] = c;
            }
            if (select) {
              atomicAdd(&h[mag_key(c.x) >> kHistShift], 1u);
              atomicAdd(&h[mag_key(c.y) >> kHistShift], 1u);
              atomicAdd(&h[mag_key(c.z) >> kHistShift], 1u);
              atomicAdd(&h[mag_key(c.w) >> kHistShift], 1u);
            }
          } else {
            const int32_t i = p + 128 * u + 4 * lane;
            for (int j = 0; j < 4; ++j) {
              if (i + j < l1) {
                float c = g[i + j];
                if (EF) {
                  c = __fadd_rn(c, e[i + j]);
                  e[i + j] = c;
                }
                if (select) atomicAdd(&h[mag_key(c) >> kHistShift], 1u);
              }
            }
          }
        }
      }
    }
    __syncthreads();
    if (select) {
      uint32_t* hb = w.hist + (int64_t)b * kHistBins;
      for (int i = threadIdx.x; i < kHistBins; i += kBkHistThreads) {
        if (h[i]) atomicAdd(&hb[i], h[i]);
        h[i] = 0u;
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0)
        last = atomicAdd(&w.sel[b].ticket_hist, 1u) == (uint32_t)dp->blk_hist - 1u;
      __syncthreads();
      if (last) {
        // every block of the bucket has added its counts: first-level bin
        __threadfence();
        for (int i = threadIdx.x; i < kHistBins; i += kBkHistThreads) {
          h[i] = __ldcg(&hb[i]);
          hb[i] = 0u;
        }
        if (threadIdx.x == 0) {
          digit = kNone;
          above = 0u;
        }
        __syncthreads();
        find_digit<kBkHistThreads>(h, kHistBins, (uint32_t)bk, warp_sums, &digit, &above);
        if (threadIdx.x == 0) {
          BucketSel* q = &w.sel[b];
          q->B = digit;
          q->above1 = above;
          q->need1 = (uint32_t)bk - above;
          q->cntB = digit != kNone ? h[digit] : 0u;
          q->ticket_hist = 0u;
          if (digit == kNone) atomicOr(w.status, kStatusTopkSelect);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kHistBins; i += kBkHistThreads) h[i] = 0u;
        __syncthreads();
      }
    }
    s = sub_hi;
  }
}

// ---------------------------------------------------------------------------
// collect: per-segment ordered lists of the entries with bin >= B.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBkThreads) bk_collect_kernel(const float* __restrict__ csrc,
                                                                BucketWs w) {
  constexpr int NW = kBkThreads / 32;
  __shared__ uint32_t mid[kMidBins];
  __shared__ uint32_t warp_sums[NW + 1];
  __shared__ uint32_t digit, above;
  __shared__ int last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = lanemask_lt();
  for (int i = threadIdx.x; i < kMidBins; i += kBkThreads) mid[i] = 0u;
  __syncthreads();
  int64_t s, s_hi;
  seg_range(w.nseg, gridDim.x, blockIdx.x, &s, &s_hi);
  while (s < s_hi) {
    const int b = w.seg_bucket[s];
    const BucketDesc d = w.desc[b];
    const int64_t sub_hi = std::min<int64_t>(s_hi, (int64_t)d.seg_first + d.nseg);
    if (d.k == 0) {
      s = sub_hi;
      continue;
    }
    const uint32_t B = __ldcg(&w.sel[b].B);
    const float* c = csrc + d.start;
    for (int64_t seg = s + warp; seg < sub_hi; seg += NW) {
      const int64_t l0 = (seg - d.seg_first) << kSegShift;
      const int64_t l1 = std::min<int64_t>(l0 + kSegElems, d.n);
      uint2* out = w.list + (seg << kSegShift);
      uint32_t cnt = 0u, above_l = 0u;
      for (int64_t p = l0; p < l1; p += kPass) {
        float v[16];
        bool valid[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = p + 128 * u + 4 * lane;
          if (i + 3 < l1) {
            const float4 x = *reinterpret_cast<const float4*>(c + i);
            v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
            valid[4 * u] = valid[4 * u + 1] = valid[4 * u + 2] = valid[4 * u + 3] = true;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              valid[4 * u + j] = i + j < l1;
              v[4 * u + j] = valid[4 * u + j] ? c[i + j] : 0.0f;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          bool ge[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t key = mag_key(v[4 * u + j]);
            const uint32_t bin = key >> kHistShift;
            ge[j] = valid[4 * u + j] && bin >= B;
            above_l += (valid[4 * u + j] && bin > B) ? 1u : 0u;
            if (valid[4 * u + j] && bin == B)
              atomicAdd(&mid[(key >> kLowBits) & (kMidBins - 1)], 1u);
          }
          // index order is (u, lane, j): lanes below come first
          const uint32_t b0 = __ballot_sync(0xffffffffu, ge[0]);
          const uint32_t b1 = __ballot_sync(0xffffffffu, ge[1]);
          const uint32_t b2 = __ballot_sync(0xffffffffu, ge[2]);
          const uint32_t b3 = __ballot_sync(0xffffffffu, ge[3]);
          uint32_t pos = cnt + __popc(b0 & lt) + __popc(b1 & lt) + __popc(b2 & lt) +
                         __popc(b3 & lt);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (ge[j]) {
              out[pos++] = make_uint2(__float_as_uint(v[4 * u + j]),
                                      (uint32_t)(p + 128 * u + 4 * lane + j));
            }
          }
          cnt += __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
        }
      }
      above_l = __reduce_add_sync(0xffffffffu, above_l);
      if (lane == 0) {
        w.seg_cnt[seg] = cnt;
        w.seg_above[seg] = above_l;
      }
    }
    __syncthreads();
    uint32_t* mb = w.mid + (int64_t)b * kMidBins;
    for (int i = threadIdx.x; i < kMidBins; i += kBkThreads) {
      if (mid[i]) atomicAdd(&mb[i], mid[i]);
      mid[i] = 0u;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      last = atomicAdd(&w.sel[b].ticket_coll, 1u) == (uint32_t)d.blk_coll - 1u;
    __syncthreads();
    if (last) {
      // second digit over the bin-B entries of the whole bucket
      __threadfence();
      for (int i = threadIdx.x; i < kMidBins; i += kBkThreads) {
        mid[i] = __ldcg(&mb[i]);
        mb[i] = 0u;
      }
      if (threadIdx.x == 0) {
        digit = kNone;
        above = 0u;
      }
      __syncthreads();
      BucketSel* q = &w.sel[b];
      const uint32_t need1 = __ldcg(&q->need1);
      const uint32_t total = find_digit<kBkThreads>(mid, kMidBins, need1, warp_sums, &digit, &above);
      if (threadIdx.x == 0) {
        q->B2 = digit;
        q->need2 = need1 - above;
        q->ticket_coll = 0u;
        if (digit == kNone) atomicOr(w.status, kStatusTopkSelect);
        if (total != __ldcg(&q->cntB)) atomicOr(w.status, kStatusTopkCount);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < kMidBins; i += kBkThreads) mid[i] = 0u;
      __syncthreads();
    }
    s = sub_hi;
  }
}

// ---------------------------------------------------------------------------
// refine: counts above (B, B2); the last block of a bucket finds T and the
// segments' output offsets.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void classify_at_T(const BucketWs& w, uint32_t key, uint32_t seg,
                                              uint32_t T) {
  if (key > T) atomicAdd(&w.seg_kept[seg], 1u);
  else if (key == T) atomicAdd(&w.seg_tie[seg], 1u);
}

__global__ void __launch_bounds__(kBkThreads) bk_refine_kernel(BucketWs w) {
  constexpr int NW = kBkThreads / 32;
  __shared__ uint32_t low[kLowBins];
  __shared__ uint32_t warp_sums[NW + 1];
  __shared__ uint32_t digit, above;
  __shared__ int last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kLowBins; i += kBkThreads) low[i] = 0u;
  __syncthreads();
  int64_t s, s_hi;
  seg_range(w.nseg, gridDim.x, blockIdx.x, &s, &s_hi);
  while (s < s_hi) {
    const int b = w.seg_bucket[s];
    const BucketDesc d = w.desc[b];
    const int64_t sub_hi = std::min<int64_t>(s_hi, (int64_t)d.seg_first + d.nseg);
    if (d.k == 0) {
      s = sub_hi;
      continue;
    }
    BucketSel* q = &w.sel[b];
    const uint32_t B = __ldcg(&q->B), B2 = __ldcg(&q->B2);
    uint2* stash = w.stash + (int64_t)b * kBkStash;
    for (int64_t seg = s + warp; seg < sub_hi; seg += NW) {
      const uint32_t cnt = w.seg_cnt[seg];
      const uint2* in = w.list + (seg << kSegShift);
      uint32_t strict = 0u;
      for (uint32_t j = lane; j < cnt; j += 32) {
        const uint32_t key = in[j].x & 0x7fffffffu;
        if ((key >> kHistShift) != B) continue;
        const uint32_t m = (key >> kLowBits) & (kMidBins - 1);
        if (m > B2) {
          ++strict;
        } else if (m == B2) {
          atomicAdd(&low[key & (kLowBins - 1)], 1u);
          const uint32_t slot = atomicAdd(&q->stash_count, 1u);
          if (slot < (uint32_t)kBkStash) stash[slot] = make_uint2(key, (uint32_t)seg);
        }
      }
      strict = __reduce_add_sync(0xffffffffu, strict);
      if (lane == 0) {
        w.seg_kept[seg] = w.seg_above[seg] + strict;
        w.seg_tie[seg] = 0u;
      }
    }
    __syncthreads();
    uint32_t* lb = w.low + (int64_t)b * kLowBins;
    for (int i = threadIdx.x; i < kLowBins; i += kBkThreads) {
      if (low[i]) atomicAdd(&lb[i], low[i]);
      low[i] = 0u;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      last = atomicAdd(&q->ticket_ref, 1u) == (uint32_t)d.blk_ref - 1u;
    __syncthreads();
    if (last) {
      __threadfence();
      for (int i = threadIdx.x; i < kLowBins; i += kBkThreads) {
        low[i] = __ldcg(&lb[i]);
        lb[i] = 0u;
      }
      if (threadIdx.x == 0) {
        digit = kNone;
        above = 0u;
      }
      __syncthreads();
      const uint32_t need2 = __ldcg(&q->need2);
      find_digit<kBkThreads>(low, kLowBins, need2, warp_sums, &digit, &above);
      const uint32_t B3 = digit;
      const uint32_t T = (B << kHistShift) | (B2 << kLowBits) | (B3 & (kLowBins - 1));
      const uint32_t needT = need2 - above;
      // the set-aside entries above T and at T, per segment
      const uint32_t nst = __ldcg(&q->stash_count);
      if (nst <= (uint32_t)kBkStash) {
        for (uint32_t j = threadIdx.x; j < nst; j += kBkThreads) {
          const uint2 e = __ldcg(&stash[j]);
          classify_at_T(w, e.x, e.y, T);
        }
      } else {  // more (B, B2) entries than the stash holds: rescan the lists
        for (int64_t seg = d.seg_first + warp; seg < (int64_t)d.seg_first + d.nseg; seg += NW) {
          const uint32_t cnt = w.seg_cnt[seg];
          const uint2* in = w.list + (seg << kSegShift);
          for (uint32_t j = lane; j < cnt; j += 32) {
            const uint32_t key = in[j].x & 0x7fffffffu;
            if ((key >> kLowBits) == ((B << (kHistShift - kLowBits)) | B2))
              classify_at_T(w, key, (uint32_t)seg, T);
          }
        }
      }
      __syncthreads();
      // output offsets: the ties at T go to the segments in index order
      uint32_t tie_carry = 0u, out_carry = 0u;
      for (int64_t base = 0; base < d.nseg; base += kBkThreads) {
        const int64_t sg = d.seg_first + base + threadIdx.x;
        const bool valid = base + threadIdx.x < d.nseg;
        const uint32_t tie = valid ? __ldcg(&w.seg_tie[sg]) : 0u;
        const uint32_t kept = valid ? __ldcg(&w.seg_kept[sg]) : 0u;
        uint32_t tt, ot;
        const uint32_t tie_ex = tie_carry + block_scan<kBkThreads>(tie, warp_sums, &tt);
        const uint32_t rem = needT > tie_ex ? needT - tie_ex : 0u;
        const uint32_t kk = kept + (tie < rem ? tie : rem);
        const uint32_t out_ex = out_carry + block_scan<kBkThreads>(kk, warp_sums, &ot);
        if (valid) {
          w.seg_out[sg] = out_ex;
          w.seg_tieb[sg] = tie_ex;
        }
        tie_carry += tt;
        out_carry += ot;
      }
      if (threadIdx.x == 0) {
        q->T = T;
        q->needT = needT;
        q->stash_count = 0u;
        q->ticket_ref = 0u;
        if (B == kNone || B2 == kNone || B3 == kNone) atomicOr(w.status, kStatusTopkSelect);
        if (out_carry != (uint32_t)d.k) atomicOr(w.status, kStatusTopkOverflow);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < kLowBins; i += kBkThreads) low[i] = 0u;
      __syncthreads();
    }
    s = sub_hi;
  }
}

// ---------------------------------------------------------------------------
// write: ordered (index, value) of the kept entries.
// ---------------------------------------------------------------------------
template <bool ZERO>
__global__ void __launch_bounds__(kBkThreads) bk_write_kernel(float* __restrict__ err,
                                                              BucketWs w,
                                                              int32_t* __restrict__ idx_out,
                                                              float* __restrict__ val_out) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = lanemask_lt();
  const int64_t gwarp = ((int64_t)blockIdx.x * kBkThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kBkThreads) >> 5;
  for (int64_t seg = gwarp; seg < w.nseg; seg += nwarps) {
    const int b = w.seg_bucket[seg];
    const BucketDesc* dp = w.desc + b;
    const uint32_t bk = (uint32_t)dp->k, bn = (uint32_t)dp->n;
    if (bk == 0u) continue;
    const int64_t idx_off = dp->idx_off;
    float* eb = err + dp->start;
    const uint32_t T = w.sel[b].T, needT = w.sel[b].needT;
    const uint32_t out = w.seg_out[seg], tieb = w.seg_tieb[seg], cnt = w.seg_cnt[seg];
    const uint32_t rem = needT > tieb ? needT - tieb : 0u;
    const uint2* in = w.list + (seg << kSegShift);
    int32_t* io = idx_out + idx_off;
    float* vo = val_out + idx_off;
    uint32_t run = 0u, tie_run = 0u;
    for (uint32_t j0 = 0; j0 < cnt; j0 += 32) {
      const bool valid = j0 + lane < cnt;
      const uint2 e = valid ? in[j0 + lane] : make_uint2(0u, 0u);
      const uint32_t key = e.x & 0x7fffffffu;
      const bool gt = valid && key > T, eq = valid && key == T;
      const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
      const bool keep = gt || (eq && tie_run + __popc(eqb & lt) < rem);
      const uint32_t kb = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const uint32_t pos = out + run + __popc(kb & lt);
        if (pos < bk && e.y < bn) {
          io[pos] = (int32_t)e.y;
          vo[pos] = __uint_as_float(e.x);
          if (ZERO) eb[e.y] = 0.0f;
        } else {
          atomicOr(w.status, kStatusTopkOverflow);
        }
      }
      run += __popc(kb);
      tie_run += __popc(eqb);
    }
  }
}

template <class K>
int blocks_per_sm(K kernel, int threads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return std::max(n, 1);
}

}  // namespace

gc_status launch_ef_topk_buckets(gc_ctx* ctx, const float* grad, float* err, int32_t* idx_out,
                                 float* val_out, bool zero_err, int qbits, int64_t qgroup) {
  const BucketWs& w = ctx->bk;
  cudaStream_t s = ctx->stream;
  {
    LaunchScope L(ctx, GC_PHASE_BK_HIST);
    if (err)
      bk_hist_kernel<true><<<w.g_hist, kBkHistThreads, 0, s>>>(grad, err, w, qbits, qgroup);
    else
      bk_hist_kernel<false><<<w.g_hist, kBkHistThreads, 0, s>>>(grad, err, w, qbits, qgroup);
  }
  {
    LaunchScope L(ctx, GC_PHASE_BK_COLLECT);
    bk_collect_kernel<<<w.g_coll, kBkThreads, 0, s>>>(err ? err : grad, w);
  }
  {
    LaunchScope L(ctx, GC_PHASE_BK_REFINE);
    bk_refine_kernel<<<w.g_ref, kBkThreads, 0, s>>>(w);
  }
  {
    LaunchScope L(ctx, GC_PHASE_BK_WRITE);
    if (zero_err && err)
      bk_write_kernel<true><<<w.g_write, kBkThreads, 0, s>>>(err, w, idx_out, val_out);
    else
      bk_write_kernel<false><<<w.g_write, kBkThreads, 0, s>>>(err, w, idx_out, val_out);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

void free_buckets(gc_ctx* ctx) {
  if (ctx->bk_base) cudaFree(ctx->bk_base);
  ctx->bk_base = nullptr;
  ctx->bk = BucketWs{};
}

gc_status plan_buckets(gc_ctx* ctx, int nb, const int64_t* bucket_n, const int64_t* bucket_k) {
  std::vector<BucketDesc> desc(nb);
  int64_t start = 0, nseg = 0, nchunk = 0, voff = 0;
  for (int b = 0; b < nb; ++b) {
    BucketDesc& d = desc[b];
    d = BucketDesc{};
    d.start = start;
    d.idx_off = voff;
    d.n = (int32_t)bucket_n[b];
    d.k = (int32_t)bucket_k[b];
    d.seg_first = (int32_t)nseg;
    d.nseg = (int32_t)ceil_div(bucket_n[b], kSegElems);
    d.chunk_first = (int32_t)nchunk;
    d.nchunk = (int32_t)ceil_div(bucket_k[b], kChunkVals);
    start += bucket_n[b];
    nseg += d.nseg;
    nchunk += d.nchunk;
    voff += round_up(bucket_k[b], 4);
    if (nseg > INT32_MAX || nchunk > INT32_MAX) return GC_ERR_INVALID_ARG;
  }
  std::vector<int32_t> seg_bucket(nseg), chunk_bucket(std::max<int64_t>(nchunk, 1));
  for (int b = 0; b < nb; ++b) {
    for (int32_t i = 0; i < desc[b].nseg; ++i) seg_bucket[desc[b].seg_first + i] = b;
    for (int32_t i = 0; i < desc[b].nchunk; ++i) chunk_bucket[desc[b].chunk_first + i] = b;
  }
  const int sms = ctx->num_sms;
  BucketWs w{};
  w.nb = nb;
  w.total_n = start;
  w.nseg = nseg;
  w.nchunk = nchunk;
  w.vals_total = voff;
  auto grid = [&](int per_sm) { return (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)sms * per_sm, nseg)); };
  w.g_hist = grid(blocks_per_sm(bk_hist_kernel<true>, kBkHistThreads));
  w.g_coll = grid(blocks_per_sm(bk_collect_kernel, kBkThreads));
  w.g_ref = grid(blocks_per_sm(bk_refine_kernel, kBkThreads));
  w.g_write = grid(blocks_per_sm(bk_write_kernel<true>, kBkThreads));
  // blocks of each ticketed pass that touch each bucket
  auto count_blocks = [&](int G, int32_t BucketDesc::*field) {
    for (int i = 0; i < G; ++i) {
      int64_t lo, hi;
      seg_range(nseg, G, i, &lo, &hi);
      if (lo >= hi) continue;
      for (int b = seg_bucket[lo]; b <= seg_bucket[hi - 1]; ++b) ++(desc[b].*field);
    }
  };
  count_blocks(w.g_hist, &BucketDesc::blk_hist);
  count_blocks(w.g_coll, &BucketDesc::blk_coll);
  count_blocks(w.g_ref, &BucketDesc::blk_ref);

  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) / 256 * 256; return o; };
  const size_t o_desc = take(sizeof(BucketDesc) * nb);
  const size_t o_sel = take(sizeof(BucketSel) * nb);
  const size_t o_segb = take(sizeof(int32_t) * nseg);
  const size_t o_chb = take(sizeof(int32_t) * chunk_bucket.size());
  const size_t o_hist = take(sizeof(uint32_t) * kHistBins * (size_t)nb);
  const size_t o_mid = take(sizeof(uint32_t) * kMidBins * (size_t)nb);
  const size_t o_low = take(sizeof(uint32_t) * kLowBins * (size_t)nb);
  size_t o_seg[6];
  for (int i = 0; i < 6; ++i) o_seg[i] = take(sizeof(uint32_t) * nseg);
  const size_t o_list = take(sizeof(uint2) * (size_t)nseg * kSegElems);
  const size_t o_stash = take(sizeof(uint2) * kBkStash * (size_t)nb);
  const size_t o_qoff = take(sizeof(int64_t) * 2 * (size_t)nb);
  const size_t o_vals = take(sizeof(float) * (size_t)std::max<int64_t>(voff, 1));

  free_buckets(ctx);
  void* base = nullptr;
  const cudaError_t e = cudaMalloc(&base, off);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? GC_ERR_NO_MEMORY : GC_ERR_CUDA;
  }
  char* p = static_cast<char*>(base);
  w.desc = reinterpret_cast<BucketDesc*>(p + o_desc);
  w.sel = reinterpret_cast<BucketSel*>(p + o_sel);
  w.seg_bucket = reinterpret_cast<int32_t*>(p + o_segb);
  w.chunk_bucket = reinterpret_cast<int32_t*>(p + o_chb);
  w.hist = reinterpret_cast<uint32_t*>(p + o_hist);
  w.mid = reinterpret_cast<uint32_t*>(p + o_mid);
  w.low = reinterpret_cast<uint32_t*>(p + o_low);
  w.seg_cnt = reinterpret_cast<uint32_t*>(p + o_seg[0]);
  w.seg_above = reinterpret_cast<uint32_t*>(p + o_seg[1]);
  w.seg_kept = reinterpret_cast<uint32_t*>(p + o_seg[2]);
  w.seg_tie = reinterpret_cast<uint32_t*>(p + o_seg[3]);
  w.seg_out = reinterpret_cast<uint32_t*>(p + o_seg[4]);
  w.seg_tieb = reinterpret_cast<uint32_t*>(p + o_seg[5]);
  w.list = reinterpret_cast<uint2*>(p + o_list);
  w.stash = reinterpret_cast<uint2*>(p + o_stash);
  w.qoff = reinterpret_cast<int64_t*>(p + o_qoff);
  w.vals = reinterpret_cast<float*>(p + o_vals);
  w.status = ctx->ws.status;
  // zero the state that must start at zero; the list, segment arrays and
  // outputs are written before they are read
  bool ok = cudaMemset(p + o_sel, 0, o_segb - o_sel) == cudaSuccess &&
            cudaMemset(p + o_hist, 0, o_seg[0] - o_hist) == cudaSuccess &&
            cudaMemcpy(w.desc, desc.data(), sizeof(BucketDesc) * nb, cudaMemcpyHostToDevice) ==
                cudaSuccess &&
            cudaMemcpy(w.seg_bucket, seg_bucket.data(), sizeof(int32_t) * nseg,
                       cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(w.chunk_bucket, chunk_bucket.data(),
                       sizeof(int32_t) * chunk_bucket.size(), cudaMemcpyHostToDevice) ==
                cudaSuccess;
  // the memsets run on the legacy stream: finish them before any launch
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaFree(base);
    return GC_ERR_CUDA;
  }
  ctx->bk_base = base;
  ctx->bk = w;
  return GC_OK;
}

}  // namespace gc
