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

// Appends the entries flagged in ge[0..3] of this lane (elements base + 4 *
// lane + j of one 128-element row, j = 0..3) to a segment list in index
// order; every lane of the warp calls it.  Returns the new list length.
__device__ __forceinline__ uint32_t append4(uint2* out, uint32_t cnt, const bool ge[4],
                                            const float c[4], uint32_t base, int lane,
                                            uint32_t lt) {
  const uint32_t b0 = __ballot_sync(0xffffffffu, ge[0]);
  const uint32_t b1 = __ballot_sync(0xffffffffu, ge[1]);
  const uint32_t b2 = __ballot_sync(0xffffffffu, ge[2]);
  const uint32_t b3 = __ballot_sync(0xffffffffu, ge[3]);
  // index order is (lane, j): the lanes below come first
  uint32_t pos = cnt + __popc(b0 & lt) + __popc(b1 & lt) + __popc(b2 & lt) + __popc(b3 & lt);
  // the lists are read again by the next passes: ask L2 to keep them while
  // the hist pass streams the gradient past
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (ge[j]) {
      uint2* a = out + pos++;
      asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(a),
                   "r"(__float_as_uint(c[j])), "r"(base + 4 * lane + j), "l"(pol)
                   : "memory");
    }
  }
  return cnt + __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
}

// ---------------------------------------------------------------------------
// hist: c = g + e, the first-level histogram and, when the bucket has a
// threshold guess, the per-segment lists of the entries whose key is at or
// above the guess.
//
// Each warp streams its segments in passes of 256 elements.  g and e of
// the next kStages - 1 passes are in flight as asynchronous copies into the
// warp's shared-memory stages (cp.async, completed with cp.async.wait_group)
// while the current pass is processed, so the memory system always has
// about 10 KB per warp outstanding without holding registers for it.  Each
// lane copies and later reads back the same 16-byte chunks of a pass.
// ---------------------------------------------------------------------------
constexpr int kH1Threads = 512;
constexpr int kH1Warps = kH1Threads / 32;
constexpr int kH1Rows = 2;                 // rows of 128 elements per pass
constexpr int kH1Pass = 128 * kH1Rows;     // elements per pass
constexpr int kStages = 6;

struct HistSmem {
  float4 sg[kH1Warps][kStages][32 * kH1Rows];  // g of a pass
  float4 se[kH1Warps][kStages][32 * kH1Rows];  // e of a pass
  uint32_t h[kHistBins];
  uint32_t warp_sums[kH1Warps + 1];
  uint32_t digit, above, listed;
  int last;
};

// Position of a warp in its work: segment seg (bucket-local element offset
// l0 .. l1) and pass p.
struct PassCursor {
  int32_t seg, l1, p;
  __device__ __forceinline__ bool valid(int32_t sub_hi) const { return seg < sub_hi; }
};

// With PATCH, e is first brought up to date with the residuals of the kept
// entries of the previous (deferred) hybrid call, when the plan's ready flag
// says the patch list holds any (the collect pass clears the flag, the
// deferred QSGD pass sets it, a flush clears it): segment s's entries are
// patch[seg_out[s] .. seg_out[s + 1]) (the last segment of a bucket ends at
// k), sorted by position.  A warp holds a window of 64 of them in registers
// (two per lane), fetched for its next segment while it works on the
// current one, and writes each into the shared-memory stage of e of the
// pass that holds its position, before c is formed.  The ragged end of a
// bucket is read from err directly; its residuals were written there.
template <bool EF, bool DIAG, bool PATCH = false>
__global__ void __launch_bounds__(kH1Threads, 1) bk_hist_kernel(
    const float* __restrict__ grad, float* __restrict__ err, BucketWs w, int qbits,
    int64_t qgroup) {
  extern __shared__ __align__(16) unsigned char hist_smem_raw[];
  HistSmem& sm = *reinterpret_cast<HistSmem*>(hist_smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = lanemask_lt();
  if (blockIdx.x == 0 && warp == 0 && qbits > 0) layout_quant_outputs(w, qbits, qgroup, lane);
  const bool patch_ready = PATCH && __ldcg(w.patch_ready) != 0u;
  for (int i = threadIdx.x; i < kHistBins; i += kH1Threads) sm.h[i] = 0u;
  if (threadIdx.x == 0) sm.listed = 0u;
  __syncthreads();
  int64_t s64, s_hi64;
  seg_range(w.nseg, gridDim.x, blockIdx.x, &s64, &s_hi64);
  // segment numbers fit 32 bits (the plan checks it)
  int32_t s = (int32_t)s64;
  const int32_t s_hi = (int32_t)s_hi64;
  while (s < s_hi) {
    const int b = w.seg_bucket[s];
    const BucketDesc* dp = w.desc + b;
    const int32_t seg_first = dp->seg_first, bn = dp->n, bk = dp->k;
    const int32_t sub_hi = min(s_hi, seg_first + dp->nseg);
    const bool select = bk > 0;
    const uint32_t g1 = select ? __ldcg(&w.sel[b].guess1) : 0u;
    const bool emit = g1 != 0u;
    const uint32_t kg = g1 - 1u;
    const float* g = grad + dp->start;
    float* e = EF ? err + dp->start : nullptr;

    // this warp's passes: segments s + warp, s + warp + NW, ...; 4 passes each
    auto first = [&](int32_t seg) {
      PassCursor c;
      c.seg = seg;
      const int32_t l0 = (seg - seg_first) << kSegShift;  // bucket-local (n <= 2^31 - 2^16)
      c.p = l0;
      c.l1 = min(l0 + kSegElems, bn);
      return c;
    };
    auto advance = [&](PassCursor& c) {
      c.p += kH1Pass;
      if (c.p >= c.l1) c = first(c.seg + kH1Warps);
    };
    // copies of the whole 16-byte chunks of a pass; the ragged end of the
    // last bucket is read directly when the pass is processed
    auto issue = [&](const PassCursor& c, int st) {
      if (c.valid(sub_hi)) {
#pragma unroll
        for (int u = 0; u < kH1Rows; ++u) {
          const int32_t i = c.p + 128 * u + 4 * lane;
          if (i + 3 < c.l1) {
            cp_async16(&sm.sg[warp][st][32 * u + lane], g + i);
            if (EF) cp_async16(&sm.se[warp][st][32 * u + lane], e + i);
          }
        }
      }
      cp_async_commit();  // one group per pass (possibly empty)
    };

    PassCursor ic = first(s + warp), uc = ic;
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
      issue(ic, k);
      if (ic.valid(sub_hi)) advance(ic);
    }

    // pending residuals: entries [pu, pz) of the current segment are still
    // to be applied, lane l holds entries pw + l and pw + 32 + l
    const uint2* plist = PATCH ? w.patch + dp->idx_off : nullptr;
    const int32_t seg_end = seg_first + dp->nseg;
    auto seg_entries = [&](int32_t seg, uint32_t* a, uint32_t* z) {
      const uint32_t z0 = seg + 1 < seg_end ? __ldcg(&w.seg_out[seg + 1]) : (uint32_t)bk;
      *z = min(z0, (uint32_t)bk);  // never past the bucket's entries
      *a = min(__ldcg(&w.seg_out[seg]), *z);
    };
    auto window = [&](uint32_t base, uint32_t z, uint2* e0, uint2* e1) {
      const uint32_t j0 = base + lane, j1 = j0 + 32u;
      *e0 = j0 < z ? __ldcg(&plist[j0]) : make_uint2(0xffffffffu, 0u);
      *e1 = j1 < z ? __ldcg(&plist[j1]) : make_uint2(0xffffffffu, 0u);
    };
    int32_t p_seg = -1, n_seg = -1;
    int n_stage = 0;  // next segment: 1 = range requested, 2 = window requested
    uint32_t pu = 0u, pz = 0u, pw = 0u, na = 0u, nz = 0u;
    uint2 pe0 = make_uint2(0xffffffffu, 0u), pe1 = pe0, ne0 = pe0, ne1 = pe0;
    const bool patching = PATCH && EF && select && patch_ready;
    int st_use = 0, st_issue = kStages - 1;
    uint32_t cnt = 0u;
    float d_all = 0.0f, d_unl = 0.0f;  // sums of c^2: all, key below the guess
    while (uc.valid(sub_hi)) {
      if (patching) {
        if (uc.seg != p_seg) {
          // a new segment: take the prefetched window, or fetch it now
          p_seg = uc.seg;
          if (n_seg == p_seg && n_stage == 2) {
            pu = na; pz = nz; pe0 = ne0; pe1 = ne1;
          } else {
            seg_entries(p_seg, &pu, &pz);
            window(pu, pz, &pe0, &pe1);
          }
          pw = pu;
          n_seg = p_seg + kH1Warps;
          n_stage = 0;
          if (n_seg < sub_hi) {
            seg_entries(n_seg, &na, &nz);
            n_stage = 1;
          }
        } else if (n_stage == 1) {
          window(na, nz, &ne0, &ne1);
          n_stage = 2;
        }
      }
      cp_async_wait<kStages - 2>();  // the oldest pass has landed
      const int32_t p = uc.p, l1 = uc.l1;
      if (patching && pu < pz) {
        const uint32_t pend = (uint32_t)(p + kH1Pass), fend = (uint32_t)(l1 & ~3);
        float* stg = reinterpret_cast<float*>(sm.se[warp][st_use]);
        bool synced = false;
        for (;;) {
          // the entries of this pass are a run from pu (sorted positions)
          const bool in0 = pw + lane >= pu && pw + lane < pz && pe0.x < pend;
          const bool in1 = pw + 32u + lane >= pu && pw + 32u + lane < pz && pe1.x < pend;
          const uint32_t b0 = __ballot_sync(0xffffffffu, in0);
          const uint32_t b1 = __ballot_sync(0xffffffffu, in1);
          if ((b0 | b1) == 0u) break;
          if (!synced) {
            __syncwarp();  // every lane's copies of this pass have landed
            synced = true;
          }
          if (in0 && pe0.x >= (uint32_t)p && pe0.x < fend) stg[pe0.x - p] = __uint_as_float(pe0.y);
          if (in1 && pe1.x >= (uint32_t)p && pe1.x < fend) stg[pe1.x - p] = __uint_as_float(pe1.y);
          pu += __popc(b0) + __popc(b1);
          if (pu < pw + 64u || pu >= pz) break;
          pw += 64u;  // the window is used up inside this pass: the next 64
          window(pw, pz, &pe0, &pe1);
        }
        if (synced) __syncwarp();
      }
      float4 cv[kH1Rows];
#pragma unroll
      for (int u = 0; u < kH1Rows; ++u) {
        const int32_t i = p + 128 * u + 4 * lane;
        if (i + 3 < l1) {
          cv[u] = sm.sg[warp][st_use][32 * u + lane];
          if (EF) {
            const float4 ev = sm.se[warp][st_use][32 * u + lane];
            cv[u].x = __fadd_rn(cv[u].x, ev.x);
            cv[u].y = __fadd_rn(cv[u].y, ev.y);
            cv[u].z = __fadd_rn(cv[u].z, ev.z);
            cv[u].w = __fadd_rn(cv[u].w, ev.w);
            *reinterpret_cast<float4*>(e + i) = cv[u];
          }
          if (select) {
            atomicAdd(&sm.h[mag_key(cv[u].x) >> kHistShift], 1u);
            atomicAdd(&sm.h[mag_key(cv[u].y) >> kHistShift], 1u);
            atomicAdd(&sm.h[mag_key(cv[u].z) >> kHistShift], 1u);
            atomicAdd(&sm.h[mag_key(cv[u].w) >> kHistShift], 1u);
          }
        } else {
          float c[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            c[j] = 0.0f;
            if (i + j < l1) {
              c[j] = g[i + j];
              if (EF) {
                c[j] = __fadd_rn(c[j], e[i + j]);
                e[i + j] = c[j];
              }
              if (select) atomicAdd(&sm.h[mag_key(c[j]) >> kHistShift], 1u);
            }
          }
          cv[u] = make_float4(c[0], c[1], c[2], c[3]);
        }
      }
      if (DIAG) {
        // entries past the end hold 0 and add nothing
#pragma unroll
        for (int u = 0; u < kH1Rows; ++u) {
          const float c[4] = {cv[u].x, cv[u].y, cv[u].z, cv[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            d_all = __fmaf_rn(c[j], c[j], d_all);
            if (mag_key(c[j]) < kg) d_unl = __fmaf_rn(c[j], c[j], d_unl);
          }
        }
      }
      // this stage is free again: start the pass kStages - 1 ahead
      issue(ic, st_issue);
      if (ic.valid(sub_hi)) advance(ic);
      st_issue = st_issue + 1 == kStages ? 0 : st_issue + 1;
      st_use = st_use + 1 == kStages ? 0 : st_use + 1;
      if (emit) {
        uint2* out = w.list + ((int64_t)uc.seg << kSegShift);
#pragma unroll
        for (int u = 0; u < kH1Rows; ++u) {
          const int32_t i = p + 128 * u + 4 * lane;
          const float c[4] = {cv[u].x, cv[u].y, cv[u].z, cv[u].w};
          bool ge[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) ge[j] = i + j < l1 && mag_key(c[j]) >= kg;
          cnt = append4(out, cnt, ge, c, (uint32_t)(p + 128 * u), lane, lt);
        }
      }
      const int32_t seg_done = uc.seg;
      advance(uc);
      if (uc.seg != seg_done) {  // last pass of the segment
        if (emit && lane == 0) {
          w.seg_cnt[seg_done] = cnt;
          atomicAdd(&sm.listed, cnt);
        }
        cnt = 0u;
        if (DIAG) {
          float v2[2] = {d_all, d_unl};
          const float t = warp_sum_many<2>(v2, lane);  // lane 0: all, lane 16: unlisted
          if (lane == 0) w.seg_c2[seg_done] = t;
          if (lane == 16 && emit) w.seg_drop[seg_done] = t;
          d_all = d_unl = 0.0f;
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();
    if (select) {
      uint32_t* hb = w.hist + (int64_t)b * kHistBins;
      for (int i = threadIdx.x; i < kHistBins; i += kH1Threads) {
        if (sm.h[i]) atomicAdd(&hb[i], sm.h[i]);
        sm.h[i] = 0u;
      }
      if (threadIdx.x == 0 && emit) {
        atomicAdd(&w.sel[b].list_total, sm.listed);
        sm.listed = 0u;
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0)
        sm.last = atomicAdd(&w.sel[b].ticket_hist, 1u) == (uint32_t)dp->blk_hist - 1u;
      __syncthreads();
      if (sm.last) {
        // every block of the bucket has added its counts: first-level bin
        __threadfence();
        for (int i = threadIdx.x; i < kHistBins; i += kH1Threads) {
          sm.h[i] = __ldcg(&hb[i]);
          hb[i] = 0u;
        }
        if (threadIdx.x == 0) {
          sm.digit = kNone;
          sm.above = 0u;
        }
        __syncthreads();
        find_digit<kH1Threads>(sm.h, kHistBins, (uint32_t)bk, sm.warp_sums, &sm.digit, &sm.above);
        if (threadIdx.x == 0) {
          BucketSel* q = &w.sel[b];
          const uint32_t B = sm.digit;
          q->B = B;
          q->above1 = sm.above;
          q->need1 = (uint32_t)bk - sm.above;
          q->cntB = B != kNone ? sm.h[B] : 0u;
          q->ticket_hist = 0u;
          // at least k entries with key >= guess: the threshold T is not
          // below the guess, so the lists hold every entry with key >= T
          const uint32_t L = emit ? __ldcg(&q->list_total) : 0u;
          q->list_len = L;
          q->list_total = 0u;
          q->list_ok = (emit && L >= (uint32_t)bk) ? 1u : 0u;
          if (B == kNone) atomicOr(w.status, kStatusTopkSelect);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kHistBins; i += kH1Threads) sm.h[i] = 0u;
        __syncthreads();
      }
    }
    s = sub_hi;
  }
}

// List walkers take eight consecutive segments per warp and load up to 64
// entries of each per round (16 loads per lane in flight).  Lane r < 8
// keeps segment r's counters; every lane gets the list lengths.
constexpr int kWalkSegs = 8;
constexpr int kWalkRows = 2;

// The list lengths of a warp's group of segments s0 .. s0 + 7 (lane r < the
// group's size loads segment s0 + r; 0 past hi), loaded one group ahead of
// the walk: the walk then waits for the entries only, not for their counts
// first.  A warp's groups belong to it alone, so the counts it reads ahead
// are final.
__device__ __forceinline__ uint32_t group_counts(const BucketWs& w, int64_t s0, int64_t hi,
                                                 int lane) {
  return (s0 < hi && s0 + lane < hi && lane < kWalkSegs) ? __ldcg(&w.seg_cnt[s0 + lane]) : 0u;
}
__device__ __forceinline__ uint32_t spread_counts(uint32_t c_l, uint32_t cnt[kWalkSegs]) {
#pragma unroll
  for (int r = 0; r < kWalkSegs; ++r) cnt[r] = __shfl_sync(0xffffffffu, c_l, r);
  return __reduce_max_sync(0xffffffffu, c_l);
}

// Entries j0 + 32 u + lane (u < kWalkRows) of the lists of segments s0 ..
// s0 + 7; (0, 0) past each list's end.
__device__ __forceinline__ void walk_load(const BucketWs& w, int64_t s0, uint32_t j0,
                                          const uint32_t cnt[kWalkSegs], int lane,
                                          uint2 e[kWalkSegs][kWalkRows]) {
#pragma unroll
  for (int r = 0; r < kWalkSegs; ++r) {
#pragma unroll
    for (int u = 0; u < kWalkRows; ++u) {
      const uint32_t j = j0 + 32 * u + lane;
      e[r][u] = j < cnt[r] ? __ldcg(&w.list[((s0 + r) << kSegShift) + j]) : make_uint2(0u, 0u);
    }
  }
}

// ---------------------------------------------------------------------------
// collect: with usable lists, per segment the count above B, the histogram
// of bits 18..8 of the bin-B entries, and the lists compacted in place to
// the entries of bin >= B; otherwise c is read again and the lists of
// bin >= B are built.
// ---------------------------------------------------------------------------
template <bool DIAG>
__global__ void __launch_bounds__(kBkThreads, 4) bk_collect_kernel(const float* __restrict__ csrc,
                                                                   BucketWs w) {
  constexpr bool diag = DIAG;
  constexpr int NW = kBkThreads / 32;
  __shared__ uint32_t mid[kMidBins];
  __shared__ uint32_t warp_sums[NW + 1];
  __shared__ uint32_t digit, above;
  __shared__ int last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = lanemask_lt();
  // the hist pass before this one has applied any pending residuals
  if (blockIdx.x == 0 && threadIdx.x == 0) *w.patch_ready = 0u;
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
    if (__ldcg(&w.sel[b].list_ok)) {
      uint32_t c_next = group_counts(w, s + kWalkSegs * warp, sub_hi, lane);
      for (int64_t s0 = s + kWalkSegs * warp; s0 < sub_hi; s0 += kWalkSegs * NW) {
        const int nq = (int)std::min<int64_t>(kWalkSegs, sub_hi - s0);
        uint32_t cnt[kWalkSegs];
        const uint32_t c_l = c_next;
        c_next = group_counts(w, s0 + kWalkSegs * NW, sub_hi, lane);
        const uint32_t mx = spread_counts(c_l, cnt);
        uint32_t abv_l = 0u, wpos_l = 0u;
        float drop[kWalkSegs];  // this lane's sums of c^2 of the dropped entries
#pragma unroll
        for (int r = 0; r < kWalkSegs; ++r) drop[r] = 0.0f;
        // lane r < nq: segment s0 + r's sum of the entries the hist pass left out
        const float drop0 = (diag && lane < nq) ? w.seg_drop[s0 + lane] : 0.0f;
        for (uint32_t j0 = 0; j0 < mx; j0 += 32 * kWalkRows) {
          uint2 e[kWalkSegs][kWalkRows];
          walk_load(w, s0, j0, cnt, lane, e);
#pragma unroll
          for (int r = 0; r < kWalkSegs; ++r) {
            if (j0 >= cnt[r]) continue;  // warp-uniform
            uint2* list = w.list + ((s0 + r) << kSegShift);
            uint32_t wpos = __shfl_sync(0xffffffffu, wpos_l, r), abv = 0u;
#pragma unroll
            for (int u = 0; u < kWalkRows; ++u) {
              if (j0 + 32 * u >= cnt[r]) break;  // warp-uniform
              const bool valid = j0 + 32 * u + lane < cnt[r];
              const uint32_t key = e[r][u].x & 0x7fffffffu;
              const uint32_t bin = key >> kHistShift;
              const bool keep = valid && bin >= B;
              if (diag && valid && bin < B) {
                const float v = __uint_as_float(e[r][u].x);
                drop[r] = __fmaf_rn(v, v, drop[r]);
              }
              abv += (valid && bin > B) ? 1u : 0u;
              if (valid && bin == B) atomicAdd(&mid[(key >> kLowBits) & (kMidBins - 1)], 1u);
              // in place: every position written was read by an earlier ballot
              const uint32_t kb = __ballot_sync(0xffffffffu, keep);
              if (keep) list[wpos + __popc(kb & lt)] = e[r][u];
              wpos += __popc(kb);
            }
            abv = __reduce_add_sync(0xffffffffu, abv);
            if (lane == r) {
              wpos_l = wpos;
              abv_l += abv;
            }
          }
        }
        if (lane < nq) {
          w.seg_above[s0 + lane] = abv_l;
          w.seg_cnt[s0 + lane] = wpos_l;
        }
        if (diag) {
          // segment r's total lands on lanes 4r .. 4r + 3
          const float t = warp_sum_many<kWalkSegs>(drop, lane);
          const float mine = __shfl_sync(0xffffffffu, t, (4 * lane) & 31);
          if (lane < nq) w.seg_drop[s0 + lane] = __fadd_rn(drop0, mine);
        }
      }
    } else {
      const float* c = csrc + d.start;
      for (int64_t seg = s + warp; seg < sub_hi; seg += NW) {
        const int64_t l0 = (seg - d.seg_first) << kSegShift;
        const int64_t l1 = std::min<int64_t>(l0 + kSegElems, d.n);
        uint2* out = w.list + (seg << kSegShift);
        uint32_t cnt = 0u, above_l = 0u;
        float drop = 0.0f;  // this lane's sum of c^2 below bin B
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
              if (diag && valid[4 * u + j] && bin < B)
                drop = __fmaf_rn(v[4 * u + j], v[4 * u + j], drop);
              above_l += (valid[4 * u + j] && bin > B) ? 1u : 0u;
              if (valid[4 * u + j] && bin == B)
                atomicAdd(&mid[(key >> kLowBits) & (kMidBins - 1)], 1u);
            }
            cnt = append4(out, cnt, ge, &v[4 * u], (uint32_t)(p + 128 * u), lane, lt);
          }
        }
        above_l = __reduce_add_sync(0xffffffffu, above_l);
        if (diag) drop = warp_allsum(drop);
        if (lane == 0) {
          w.seg_cnt[seg] = cnt;
          w.seg_above[seg] = above_l;
          if (diag) w.seg_drop[seg] = drop;
        }
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
        // with lists that start inside bin B only part of the bin is seen
        const uint32_t cntB = __ldcg(&q->cntB);
        if (__ldcg(&q->list_ok) ? total > cntB : total != cntB)
          atomicOr(w.status, kStatusTopkCount);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < kMidBins; i += kBkThreads) mid[i] = 0u;
      __syncthreads();
    }
    s = sub_hi;
  }
}

// ---------------------------------------------------------------------------
// refine: counts above (B, B2); the last block of a bucket finds T, the
// segments' output offsets and the next call's threshold guess.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void classify_at_T(const BucketWs& w, uint32_t key, uint32_t seg,
                                              uint32_t T) {
  if (key > T) atomicAdd(&w.seg_kept[seg], 1u);
  else if (key == T) atomicAdd(&w.seg_tie[seg], 1u);
}

constexpr int kScanPer = 16;                          // segments per thread in the offset scan
constexpr int kScanRound = kBkThreads * kScanPer;     // segments per round of the scan
constexpr int kStashPer = kBkStash / kBkThreads;      // stash entries per thread
constexpr uint32_t kNoSeg = 0xffffffffu;              // an empty stash slot
// Shared-memory slot of scan entry i: one word of padding per 32 entries,
// so that threads reading kScanPer consecutive entries hit distinct banks.
__device__ __forceinline__ int scan_pad(int i) { return i + (i >> 5); }
constexpr int kScanPadded = kScanRound + kScanRound / 32;

__global__ void __launch_bounds__(kBkThreads, 4) bk_refine_kernel(BucketWs w) {
  constexpr int NW = kBkThreads / 32;
  __shared__ uint32_t low[kLowBins];
  __shared__ uint32_t adj_kept[kScanPadded], adj_tie[kScanPadded];
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
    uint32_t c_next = group_counts(w, s + kWalkSegs * warp, sub_hi, lane);
    for (int64_t s0 = s + kWalkSegs * warp; s0 < sub_hi; s0 += kWalkSegs * NW) {
      const int nq = (int)std::min<int64_t>(kWalkSegs, sub_hi - s0);
      uint32_t cnt[kWalkSegs];
      const uint32_t c_l = c_next;
      c_next = group_counts(w, s0 + kWalkSegs * NW, sub_hi, lane);
      const uint32_t mx = spread_counts(c_l, cnt);
      uint32_t strict_l = 0u;
      for (uint32_t j0 = 0; j0 < mx; j0 += 32 * kWalkRows) {
        uint2 e[kWalkSegs][kWalkRows];
        walk_load(w, s0, j0, cnt, lane, e);
#pragma unroll
        for (int r = 0; r < kWalkSegs; ++r) {
          if (j0 >= cnt[r]) continue;  // warp-uniform
          uint32_t strict = 0u;
#pragma unroll
          for (int u = 0; u < kWalkRows; ++u) {
            const uint32_t key = e[r][u].x & 0x7fffffffu;
            if (j0 + 32 * u + lane < cnt[r] && (key >> kHistShift) == B) {
              const uint32_t m = (key >> kLowBits) & (kMidBins - 1);
              if (m > B2) {
                ++strict;
              } else if (m == B2) {
                atomicAdd(&low[key & (kLowBins - 1)], 1u);
                const uint32_t slot = atomicAdd(&q->stash_count, 1u);
                if (slot < (uint32_t)kBkStash) stash[slot] = make_uint2(key, (uint32_t)(s0 + r));
              }
            }
          }
          strict = __reduce_add_sync(0xffffffffu, strict);
          if (lane == r) strict_l += strict;
        }
      }
      // lane r < nq writes segment r (entries above B come from collect)
      if (lane < nq) {
        w.seg_kept[s0 + lane] = __ldcg(&w.seg_above[s0 + lane]) + strict_l;
        w.seg_tie[s0 + lane] = 0u;
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
      // one round of independent loads: the low bins, the bucket's scalars,
      // the stash and the first round of per-segment counts (staged in shared
      // memory with coalesced loads)
      for (int i = threadIdx.x; i < kLowBins; i += kBkThreads) {
        low[i] = __ldcg(&lb[i]);
        lb[i] = 0u;
      }
      const uint32_t need2 = __ldcg(&q->need2);
      const uint32_t nst = __ldcg(&q->stash_count);
      const bool in_stash = nst <= (uint32_t)kBkStash;
      uint2 se[kStashPer];  // this thread's stash entries (key, segment)
#pragma unroll
      for (int r = 0; r < kStashPer; ++r) {
        const uint32_t j = threadIdx.x + (uint32_t)r * kBkThreads;
        se[r] = (in_stash && j < nst) ? __ldcg(&stash[j]) : make_uint2(0u, kNoSeg);
      }
      // kept counts of segments base .. base + kScanRound - 1 into adj_kept
      // (and, after a rescan, the tie counts into adj_tie)
      auto stage = [&](int64_t base) {
        const int64_t nr = std::min<int64_t>(kScanRound, d.nseg - base);
        for (int i = threadIdx.x; i < kScanRound; i += kBkThreads) {
          const int64_t sg = d.seg_first + base + i;
          adj_kept[scan_pad(i)] = i < nr ? __ldcg(&w.seg_kept[sg]) : 0u;
          adj_tie[scan_pad(i)] = (i < nr && !in_stash) ? __ldcg(&w.seg_tie[sg]) : 0u;
        }
      };
      if (in_stash) stage(0);
      if (threadIdx.x == 0) {
        digit = kNone;
        above = 0u;
      }
      __syncthreads();
      find_digit<kBkThreads>(low, kLowBins, need2, warp_sums, &digit, &above);
      const uint32_t B3 = digit;
      const uint32_t T = (B << kHistShift) | (B2 << kLowBits) | (B3 & (kLowBins - 1));
      const uint32_t needT = need2 - above;
      if (!in_stash) {  // more (B, B2) entries than the stash holds: rescan the lists
        const uint32_t prefix = (B << (kHistShift - kLowBits)) | B2;
        for (int64_t seg = d.seg_first + warp; seg < (int64_t)d.seg_first + d.nseg; seg += NW) {
          const uint32_t cnt = w.seg_cnt[seg];
          const uint2* in = w.list + (seg << kSegShift);
          for (uint32_t j = lane; j < cnt; j += 32) {
            const uint32_t key = in[j].x & 0x7fffffffu;
            if ((key >> kLowBits) == prefix) classify_at_T(w, key, (uint32_t)seg, T);
          }
        }
        __syncthreads();
      }
      // output offsets: the ties at T go to the segments in index order;
      // each thread takes kScanPer consecutive segments of a round from
      // shared memory, the stash entries of the round classified at T there
      uint32_t tie_carry = 0u, out_carry = 0u;
      for (int64_t base = 0; base < d.nseg; base += kScanRound) {
        const int64_t nr = std::min<int64_t>(kScanRound, d.nseg - base);
        if (base > 0 || !in_stash) {
          __syncthreads();
          stage(base);
        }
        __syncthreads();
        if (in_stash) {
#pragma unroll
          for (int r = 0; r < kStashPer; ++r) {
            if (se[r].y == kNoSeg) continue;
            const int64_t rel = (int64_t)se[r].y - d.seg_first - base;
            if (rel < 0 || rel >= nr) continue;
            if (se[r].x > T) atomicAdd(&adj_kept[scan_pad((int)rel)], 1u);
            else if (se[r].x == T) atomicAdd(&adj_tie[scan_pad((int)rel)], 1u);
          }
          __syncthreads();
        }
        uint32_t kept[kScanPer], tie[kScanPer];
#pragma unroll
        for (int r = 0; r < kScanPer; ++r) {
          kept[r] = adj_kept[scan_pad((int)threadIdx.x * kScanPer + r)];
          tie[r] = adj_tie[scan_pad((int)threadIdx.x * kScanPer + r)];
        }
        uint32_t tsum = 0u;
#pragma unroll
        for (int r = 0; r < kScanPer; ++r) tsum += tie[r];
        uint32_t tt, ot;
        const uint32_t tie0 = tie_carry + block_scan<kBkThreads>(tsum, warp_sums, &tt);
        uint32_t run = tie0, ksum = 0u;
#pragma unroll
        for (int r = 0; r < kScanPer; ++r) {
          const uint32_t rem = needT > run ? needT - run : 0u;
          kept[r] += tie[r] < rem ? tie[r] : rem;  // kept + ties kept here
          run += tie[r];
          ksum += kept[r];
        }
        const uint32_t out0 = out_carry + block_scan<kBkThreads>(ksum, warp_sums, &ot);
        // offsets back through shared memory, then coalesced stores
        uint32_t ro = out0, rt = tie0;
#pragma unroll
        for (int r = 0; r < kScanPer; ++r) {
          adj_kept[scan_pad((int)threadIdx.x * kScanPer + r)] = ro;
          adj_tie[scan_pad((int)threadIdx.x * kScanPer + r)] = rt;
          ro += kept[r];
          rt += tie[r];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nr; i += kBkThreads) {
          w.seg_out[d.seg_first + base + i] = adj_kept[scan_pad(i)];
          w.seg_tieb[d.seg_first + base + i] = adj_tie[scan_pad(i)];
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
        // next call's guess: a margin below T, widened after a miss and
        // tuned so that the lists hold about 1.5 to 3 times k entries
        uint32_t m = __ldcg(&q->margin);
        const uint32_t L = __ldcg(&q->list_len), k = (uint32_t)d.k;
        if (m == 0u) m = kMarginInit;
        else if (!__ldcg(&q->list_ok)) m = m <= kMarginMax / 2 ? 2u * m : kMarginMax;
        else if (L > 3u * k) m -= m / 4u;
        else if (L < k + k / 2u) m += m / 4u + 1u;
        m = min(max(m, kMarginMin), kMarginMax);
        q->margin = m;
        q->guess1 = (T > m ? T - m : 0u) + 1u;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < kLowBins; i += kBkThreads) low[i] = 0u;
      __syncthreads();
    }
    s = sub_hi;
  }
}

// ---------------------------------------------------------------------------
// write: ordered (index, value) of the kept entries, four segments per warp
// (lane r < 4 holds segment r's bookkeeping).
// ---------------------------------------------------------------------------
// With ZERO and defer, the kept entries' e' = +0 goes to the plan's patch
// list as (position, 0) pairs in output order, for the next call's hist
// pass, instead of a store at each random position of e (the ragged end of
// a bucket, which the hist pass reads from e directly, is stored at once).
template <bool ZERO, bool DIAG>
__global__ void __launch_bounds__(kBkThreads) bk_write_kernel(float* __restrict__ err,
                                                              BucketWs w,
                                                              int32_t* __restrict__ idx_out,
                                                              float* __restrict__ val_out,
                                                              int defer) {
  const int lane = threadIdx.x & 31;
  if (ZERO && defer && blockIdx.x == 0 && threadIdx.x == 0) *w.patch_ready = 1u;
  const uint32_t lt = lanemask_lt();
  const int64_t gwarp = ((int64_t)blockIdx.x * kBkThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kBkThreads) >> 5;
  // the per-segment words of a group (bucket, count, output offset, ties
  // before) are loaded one group ahead, so that a group waits for its list
  // entries only; the bucket's words that depend on them stay in L1
  auto seg_words = [&](int64_t s0, int& b, uint32_t& c, uint32_t& o, uint32_t& t) {
    b = -1;
    c = o = t = 0u;
    if (s0 < w.nseg && s0 + lane < w.nseg && lane < kWalkSegs) {
      const int64_t sg = s0 + lane;
      b = w.seg_bucket[sg];
      c = w.seg_cnt[sg];
      o = w.seg_out[sg];
      t = w.seg_tieb[sg];
    }
  };
  int b_nx;
  uint32_t c_nx, o_nx, t_nx;
  seg_words(kWalkSegs * gwarp, b_nx, c_nx, o_nx, t_nx);
  for (int64_t s0 = kWalkSegs * gwarp; s0 < w.nseg; s0 += kWalkSegs * nwarps) {
    const int nq = (int)std::min<int64_t>(kWalkSegs, w.nseg - s0);
    const int b_cur = b_nx;
    const uint32_t c_cur = c_nx, o_cur = o_nx, t_cur = t_nx;
    seg_words(s0 + kWalkSegs * nwarps, b_nx, c_nx, o_nx, t_nx);
    // lane r < nq: segment s0 + r
    uint32_t cnt_l = 0u, out_l = 0u, rem_l = 0u, T_l = 0u, k_l = 0u, n_l = 0u;
    int64_t off_l = 0, start_l = 0;
    if (lane < nq) {
      const int b = b_cur;
      const BucketDesc* dp = w.desc + b;
      k_l = (uint32_t)dp->k;
      n_l = (uint32_t)dp->n;
      off_l = dp->idx_off;
      start_l = dp->start;
      if (k_l != 0u) {
        cnt_l = c_cur;
        out_l = o_cur;
        const uint32_t tieb = t_cur;
        const uint32_t needT = w.sel[b].needT;
        T_l = w.sel[b].T;
        rem_l = needT > tieb ? needT - tieb : 0u;
      }
    }
    uint32_t cnt[kWalkSegs];
#pragma unroll
    for (int r = 0; r < kWalkSegs; ++r) cnt[r] = __shfl_sync(0xffffffffu, cnt_l, r);
    const uint32_t mx = __reduce_max_sync(0xffffffffu, cnt_l);
    uint32_t run_l = 0u, tr_l = 0u;
    // this lane's sums of c^2: [r] dropped, [kWalkSegs + r] kept, of segment r
    float dk[2 * kWalkSegs];
#pragma unroll
    for (int r = 0; r < 2 * kWalkSegs; ++r) dk[r] = 0.0f;
    // lane r < nq: segment s0 + r's sum of the entries dropped before
    const float drop0 = (DIAG && k_l != 0u) ? w.seg_drop[s0 + lane] : 0.0f;
    for (uint32_t j0 = 0; j0 < mx; j0 += 32 * kWalkRows) {
      uint2 e[kWalkSegs][kWalkRows];
      walk_load(w, s0, j0, cnt, lane, e);
#pragma unroll
      for (int r = 0; r < kWalkSegs; ++r) {
        if (j0 >= cnt[r]) continue;  // warp-uniform
        const uint32_t T = __shfl_sync(0xffffffffu, T_l, r);
        const uint32_t rem = __shfl_sync(0xffffffffu, rem_l, r);
        const uint32_t out = __shfl_sync(0xffffffffu, out_l, r);
        const uint32_t bk = __shfl_sync(0xffffffffu, k_l, r);
        const uint32_t bn = __shfl_sync(0xffffffffu, n_l, r);
        const int64_t off = __shfl_sync(0xffffffffu, off_l, r);
        const int64_t start = __shfl_sync(0xffffffffu, start_l, r);
        uint32_t run = __shfl_sync(0xffffffffu, run_l, r);
        uint32_t tr = __shfl_sync(0xffffffffu, tr_l, r);
#pragma unroll
        for (int u = 0; u < kWalkRows; ++u) {
          if (j0 + 32 * u >= cnt[r]) break;  // warp-uniform
          const bool valid = j0 + 32 * u + lane < cnt[r];
          const uint32_t key = e[r][u].x & 0x7fffffffu;
          const bool gt = valid && key > T, eq = valid && key == T;
          const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
          const bool keep = gt || (eq && tr + __popc(eqb & lt) < rem);
          const uint32_t kb = __ballot_sync(0xffffffffu, keep);
          if (DIAG && valid) {
            const float v = __uint_as_float(e[r][u].x);
            if (keep) dk[kWalkSegs + r] = __fmaf_rn(v, v, dk[kWalkSegs + r]);
            else dk[r] = __fmaf_rn(v, v, dk[r]);
          }
          if (keep) {
            const uint32_t pos = out + run + __popc(kb & lt);
            if (pos < bk && e[r][u].y < bn) {
              idx_out[off + pos] = (int32_t)e[r][u].y;
              val_out[off + pos] = __uint_as_float(e[r][u].x);
              if (ZERO) {
                if (!defer) {
                  err[start + e[r][u].y] = 0.0f;
                } else {
                  w.patch[off + pos] = make_uint2(e[r][u].y, 0u);
                  if (e[r][u].y >= (bn & ~3u)) err[start + e[r][u].y] = 0.0f;
                }
              }
            } else {
              atomicOr(w.status, kStatusTopkOverflow);
            }
          }
          run += __popc(kb);
          tr += __popc(eqb);
        }
        if (lane == r) {
          run_l = run;
          tr_l = tr;
        }
      }
    }
    if (DIAG) {
      // value j's total lands on lanes 2j, 2j + 1
      const float t = warp_sum_many<2 * kWalkSegs>(dk, lane);
      const float dt = __shfl_sync(0xffffffffu, t, (2 * lane) & 31);
      const float kt = __shfl_sync(0xffffffffu, t, (2 * lane + 2 * kWalkSegs) & 31);
      if (k_l != 0u) {  // lanes < nq only
        w.seg_drop[s0 + lane] = __fadd_rn(drop0, dt);
        w.seg_keep[s0 + lane] = kt;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// diag: per bucket, the sums of the per-segment (and, for the hybrid,
// per-chunk) partials in a fixed order: each thread adds a strided run in
// index order, then a fixed tree over the threads.
// ---------------------------------------------------------------------------
constexpr int kDiagThreads = 512;

// Compensated binary32 accumulation (Neumaier's variant of Kahan summation,
// with Knuth's TwoSum for the rounding error of each addition): hi + lo
// carries the sum with a relative error of about 2u + n u^2 (u = 2^-24) for
// non-negative terms, without binary64 arithmetic.
struct Acc {
  float hi, lo;
};

__device__ __forceinline__ void acc_add(Acc& a, float x) {
  const float s = __fadd_rn(a.hi, x);
  const float bb = __fsub_rn(s, a.hi);
  const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
  a.hi = s;
  a.lo = __fadd_rn(a.lo, err);
}

__device__ __forceinline__ void acc_merge(Acc& a, const Acc& b) {
  acc_add(a, b.hi);
  a.lo = __fadd_rn(a.lo, b.lo);
}

__global__ void __launch_bounds__(kDiagThreads) bk_diag_kernel(BucketWs w, int quant,
                                                               double* __restrict__ out) {
  __shared__ Acc red[3][kDiagThreads];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const BucketDesc d = w.desc[b];
  const bool kept = d.k != 0;
  // a[0] sum c^2, a[1] sum g_hat^2, a[2] sum e'^2: each thread adds a
  // strided run of the partials in index order
  Acc a[3] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
  for (int i = threadIdx.x; i < d.nseg; i += kDiagThreads) {
    const int64_t sg = (int64_t)d.seg_first + i;
    acc_add(a[0], w.seg_c2[sg]);
    if (kept) {
      acc_add(a[2], w.seg_drop[sg]);
      if (!quant) acc_add(a[1], w.seg_keep[sg]);
    }
  }
  if (quant && kept) {
    for (int i = threadIdx.x; i < d.nchunk; i += kDiagThreads) {
      const int64_t ch = (int64_t)d.chunk_first + i;
      acc_add(a[1], w.chunk_g2[ch]);
      acc_add(a[2], w.chunk_r2[ch]);
    }
  }
  // fixed order: warp 0 merges the threads' sums in thread order (16 per
  // lane), then a butterfly
#pragma unroll
  for (int q = 0; q < 3; ++q) red[q][threadIdx.x] = a[q];
  __syncthreads();
  if (warp == 0) {
    constexpr int per = kDiagThreads / 32;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      Acc t = red[q][lane * per];
      for (int i = 1; i < per; ++i) acc_merge(t, red[q][lane * per + i]);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        Acc u;
        u.hi = __shfl_xor_sync(0xffffffffu, t.hi, o);
        u.lo = __shfl_xor_sync(0xffffffffu, t.lo, o);
        // the lower lane's sum first, so both lanes get the same result
        if (lane & o) {
          acc_merge(u, t);
          t = u;
        } else {
          acc_merge(t, u);
        }
      }
      a[q] = t;
    }
    if (lane == 0) {
      const double s0 = (double)a[0].hi + (double)a[0].lo;
      out[3 * (int64_t)b] = s0;
      out[3 * (int64_t)b + 1] = kept ? (double)a[1].hi + (double)a[1].lo : 0.0;
      out[3 * (int64_t)b + 2] = kept ? (double)a[2].hi + (double)a[2].lo : s0;  // e' = c
    }
  }
}

}  // namespace

gc_status launch_ef_topk_buckets(gc_ctx* ctx, const float* grad, float* err, int32_t* idx_out,
                                 float* val_out, bool zero_err, int qbits, int64_t qgroup,
                                 bool diag, bool patch, bool defer_zero) {
  const BucketWs& w = ctx->bk;
  cudaStream_t s = ctx->stream;
  {
    LaunchScope L(ctx, GC_PHASE_BK_HIST);
    const size_t sm = sizeof(HistSmem);
    if (err && patch && diag)
      bk_hist_kernel<true, true, true><<<w.g_hist, kH1Threads, sm, s>>>(grad, err, w, qbits,
                                                                        qgroup);
    else if (err && patch)
      bk_hist_kernel<true, false, true><<<w.g_hist, kH1Threads, sm, s>>>(grad, err, w, qbits,
                                                                         qgroup);
    else if (err && diag)
      bk_hist_kernel<true, true><<<w.g_hist, kH1Threads, sm, s>>>(grad, err, w, qbits, qgroup);
    else if (err)
      bk_hist_kernel<true, false><<<w.g_hist, kH1Threads, sm, s>>>(grad, err, w, qbits, qgroup);
    else if (diag)
      bk_hist_kernel<false, true><<<w.g_hist, kH1Threads, sm, s>>>(grad, err, w, qbits, qgroup);
    else
      bk_hist_kernel<false, false><<<w.g_hist, kH1Threads, sm, s>>>(grad, err, w, qbits, qgroup);
  }
  {
    LaunchScope L(ctx, GC_PHASE_BK_COLLECT);
    const float* csrc = err ? err : grad;
    if (diag)
      bk_collect_kernel<true><<<w.g_coll, kBkThreads, 0, s>>>(csrc, w);
    else
      bk_collect_kernel<false><<<w.g_coll, kBkThreads, 0, s>>>(csrc, w);
  }
  {
    LaunchScope L(ctx, GC_PHASE_BK_REFINE);
    bk_refine_kernel<<<w.g_ref, kBkThreads, 0, s>>>(w);
  }
  {
    LaunchScope L(ctx, GC_PHASE_BK_WRITE);
    const bool z = zero_err && err;
    const int gd = w.g_write_diag, df = (z && defer_zero) ? 1 : 0;
    if (z && diag)
      bk_write_kernel<true, true><<<gd, kBkThreads, 0, s>>>(err, w, idx_out, val_out, df);
    else if (z)
      bk_write_kernel<true, false><<<w.g_write, kBkThreads, 0, s>>>(err, w, idx_out, val_out, df);
    else if (diag)
      bk_write_kernel<false, true><<<gd, kBkThreads, 0, s>>>(err, w, idx_out, val_out, 0);
    else
      bk_write_kernel<false, false><<<w.g_write, kBkThreads, 0, s>>>(err, w, idx_out, val_out, 0);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

// The pending residuals of the patch list into err: one warp per chunk of
// 128 entries of one bucket.  Nothing is written unless the ready flag is
// set; the last block to finish (every block has read the flag by then)
// clears it.
__global__ void __launch_bounds__(kBkThreads) bk_flush_kernel(float* __restrict__ err,
                                                              BucketWs w) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * kBkThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kBkThreads) >> 5;
  const bool ready = __ldcg(w.patch_ready) != 0u;
  for (int64_t ch = gwarp; ready && ch < w.nchunk; ch += nwarps) {
    const BucketDesc d = w.desc[w.chunk_bucket[ch]];
    const int64_t m0 = (ch - d.chunk_first) * kChunkVals;
#pragma unroll
    for (int j = 0; j < kChunkVals / 32; ++j) {
      const int64_t m = m0 + 32 * j + lane;
      if (m >= d.k) continue;
      const uint2 pr = w.patch[d.idx_off + m];
      if (pr.x < (uint32_t)d.n) err[d.start + pr.x] = __uint_as_float(pr.y);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(w.flush_ticket, 1u) == gridDim.x - 1u) {
      *w.patch_ready = 0u;
      *w.flush_ticket = 0u;
    }
  }
}

gc_status launch_bucket_flush(gc_ctx* ctx, float* err) {
  const BucketWs& w = ctx->bk;
  if (w.nchunk == 0) return GC_OK;
  LaunchScope L(ctx, GC_PHASE_BK_FLUSH);
  const int grid =
      (int)std::min<int64_t>(ceil_div(w.nchunk, kBkThreads / 32), (int64_t)ctx->num_sms * 8);
  bk_flush_kernel<<<grid, kBkThreads, 0, ctx->stream>>>(err, w);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

gc_status launch_bucket_diag(gc_ctx* ctx, bool quant, double* out) {
  const BucketWs& w = ctx->bk;
  LaunchScope L(ctx, GC_PHASE_BK_DIAG);
  bk_diag_kernel<<<w.nb, kDiagThreads, 0, ctx->stream>>>(w, quant ? 1 : 0, out);
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
  const int hsm = (int)sizeof(HistSmem);
  if (cudaFuncSetAttribute(bk_hist_kernel<true, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, hsm) != cudaSuccess ||
      cudaFuncSetAttribute(bk_hist_kernel<false, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, hsm) != cudaSuccess ||
      cudaFuncSetAttribute(bk_hist_kernel<true, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, hsm) != cudaSuccess ||
      cudaFuncSetAttribute(bk_hist_kernel<false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, hsm) != cudaSuccess ||
      cudaFuncSetAttribute(bk_hist_kernel<true, false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, hsm) != cudaSuccess ||
      cudaFuncSetAttribute(bk_hist_kernel<true, true, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, hsm) != cudaSuccess)
    return GC_ERR_CUDA;
  // every instantiation of a pass runs on the same grid (the tickets count
  // its blocks): the smallest resident count of them
  w.g_hist = grid(std::min(
      std::min(blocks_per_sm(bk_hist_kernel<true, false>, kH1Threads, hsm),
               blocks_per_sm(bk_hist_kernel<true, true>, kH1Threads, hsm)),
      std::min(blocks_per_sm(bk_hist_kernel<true, false, true>, kH1Threads, hsm),
               blocks_per_sm(bk_hist_kernel<true, true, true>, kH1Threads, hsm))));
  w.g_coll = grid(std::min(blocks_per_sm(bk_collect_kernel<false>, kBkThreads),
                           blocks_per_sm(bk_collect_kernel<true>, kBkThreads)));
  w.g_ref = grid(blocks_per_sm(bk_refine_kernel, kBkThreads));
  // the write pass takes no tickets: each variant gets its own grid
  w.g_write = grid(blocks_per_sm(bk_write_kernel<true, false>, kBkThreads));
  w.g_write_diag = grid(blocks_per_sm(bk_write_kernel<true, true>, kBkThreads));
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
  const size_t o_flag = take(2 * sizeof(uint32_t));  // zeroed with the selection records
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
  const size_t o_patch = take(sizeof(uint2) * (size_t)std::max<int64_t>(voff, 1));
  size_t o_dseg[3];
  for (int i = 0; i < 3; ++i) o_dseg[i] = take(sizeof(float) * nseg);
  const size_t o_dch = take(sizeof(float) * 2 * chunk_bucket.size());

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
  w.patch_ready = reinterpret_cast<uint32_t*>(p + o_flag);
  w.flush_ticket = w.patch_ready + 1;
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
  w.patch = reinterpret_cast<uint2*>(p + o_patch);
  w.seg_c2 = reinterpret_cast<float*>(p + o_dseg[0]);
  w.seg_drop = reinterpret_cast<float*>(p + o_dseg[1]);
  w.seg_keep = reinterpret_cast<float*>(p + o_dseg[2]);
  w.chunk_g2 = reinterpret_cast<float*>(p + o_dch);
  w.chunk_r2 = w.chunk_g2 + chunk_bucket.size();
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
