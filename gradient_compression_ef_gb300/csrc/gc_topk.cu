// gc_topk.cu -- error feedback + exact Top-K selection and compaction.
//
// Semantics ("分布式训练中的梯度压缩算法" 二.2 Top-K 稀疏化; "4、梯度累积与梯度
// 压缩" 4.2.1; "梯度聚合通信优化实战方案" Python 演示 error_feedback_compress):
//   c = g + e; keep the k entries of largest |c| (ties: smaller index);
//   emit (index, c) in ascending index order; e' = c with kept entries = +0.
//
// The k-th largest key = bits(|c|) (31 bits) is found by a three-level radix
// select (12 + 11 + 8 bits); nothing is sorted and no block waits for
// another (last-block tickets only):
//   pass 1  ef_hist : c = g + e written over e (the HBM pass), and a
//                     4096-bin histogram of bits 30..19 of the key.
//   pass 2  collect : every block derives the threshold bin B from that
//                     histogram; per tile it counts the entries above B and
//                     appends the entries of bin B ("candidates") to a list,
//                     with a histogram of their bits 18..8.  The last block
//                     finds the second digit B2.
//   pass 3  refine  : one grid-wide pass over the candidates: per tile the
//                     count of those above (B, B2), and the (B, B2) ones set
//                     aside with a histogram of bits 7..0.  The last block
//                     finds the exact threshold key T, counts the set-aside
//                     entries above T and at T (ties) per tile, and scans the
//                     tiles into output offsets.
//   pass 4  write   : per tile, a block scan orders the kept entries; writes
//                     (index, value) and e' = +0 at the kept positions.
// Error feedback makes the residuals of unsent entries pile up below the
// threshold, so the threshold bin can hold 1-2 % of a bucket; hence the
// grid-wide refinement rather than a single block.
#include <algorithm>

#include "gc_internal.cuh"
#include "gc_select.cuh"

namespace gc {
namespace {

// ---------------------------------------------------------------------------
// pass 1: c = g + e (written over e) and the 12-bit histogram of |c|.
// ---------------------------------------------------------------------------
constexpr int kHistThreads = 1024;
constexpr int kHistUnroll = 4;  // 16-byte loads of g (and e) in flight per thread

template <bool EF>
__global__ void __launch_bounds__(kHistThreads, 1) ef_hist_kernel(
    const float* __restrict__ grad, float* __restrict__ err, int64_t n, Workspace ws) {
  __shared__ uint32_t h[kHistBins];
  for (int i = threadIdx.x; i < kHistBins; i += kHistThreads) h[i] = 0u;
  __syncthreads();
  const int64_t nvec = n >> 2;
  const int64_t chunk = (int64_t)kHistThreads * kHistUnroll;
  const float4* g4 = reinterpret_cast<const float4*>(grad);
  float4* e4 = reinterpret_cast<float4*>(err);
  for (int64_t base = (int64_t)blockIdx.x * chunk; base < nvec; base += (int64_t)gridDim.x * chunk) {
    float4 gv[kHistUnroll], ev[kHistUnroll];
#pragma unroll
    for (int u = 0; u < kHistUnroll; ++u) {
      const int64_t v = base + u * kHistThreads + threadIdx.x;
      if (v < nvec) {
        gv[u] = __ldcs(g4 + v);
        if (EF) ev[u] = e4[v];
      }
    }
#pragma unroll
    for (int u = 0; u < kHistUnroll; ++u) {
      const int64_t v = base + u * kHistThreads + threadIdx.x;
      if (v < nvec) {
        float4 c = gv[u];
        if (EF) {
          c.x = __fadd_rn(c.x, ev[u].x);
          c.y = __fadd_rn(c.y, ev[u].y);
          c.z = __fadd_rn(c.z, ev[u].z);
          c.w = __fadd_rn(c.w, ev[u].w);
          e4[v] = c;
        }
        atomicAdd(&h[mag_key(c.x) >> kHistShift], 1u);
        atomicAdd(&h[mag_key(c.y) >> kHistShift], 1u);
        atomicAdd(&h[mag_key(c.z) >> kHistShift], 1u);
        atomicAdd(&h[mag_key(c.w) >> kHistShift], 1u);
      }
    }
  }
  const int64_t stride = (int64_t)gridDim.x * kHistThreads;
  for (int64_t i = (nvec << 2) + (int64_t)blockIdx.x * kHistThreads + threadIdx.x; i < n; i += stride) {
    float c = grad[i];
    if (EF) {
      c = __fadd_rn(c, err[i]);
      err[i] = c;
    }
    atomicAdd(&h[mag_key(c) >> kHistShift], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += kHistThreads)
    if (h[i]) atomicAdd(&ws.hist[i], h[i]);
}

// ---------------------------------------------------------------------------
// pass 2: threshold bin, per-tile counts above it, candidates of the bin
// and the histogram of their bits 18..8; the last block finds B2.
// ---------------------------------------------------------------------------
constexpr int kCollThreads = 256;
constexpr int kCollPer = 16;                          // elements per thread per step
constexpr int kCollStep = kCollThreads * kCollPer;    // 4096

struct CollectSmem {
  uint32_t h[kHistBins];
  uint32_t mid[kMidBins];
  uint32_t warp_sums[kCollThreads / 32 + 1];
  uint32_t digit, above, base;
  bool last;
};

__global__ void __launch_bounds__(kCollThreads) collect_kernel(
    const float* __restrict__ c_src, int64_t n, uint32_t k, int ntiles, int tile_shift,
    Workspace ws) {
  __shared__ CollectSmem sm;
  for (int i = threadIdx.x; i < kHistBins; i += kCollThreads) sm.h[i] = __ldcg(&ws.hist[i]);
  for (int i = threadIdx.x; i < kMidBins; i += kCollThreads) sm.mid[i] = 0u;
  if (threadIdx.x == 0) {
    sm.digit = 0xffffffffu;
    sm.above = 0u;
  }
  __syncthreads();
  find_digit<kCollThreads>(sm.h, kHistBins, k, sm.warp_sums, &sm.digit, &sm.above);
  const uint32_t B = sm.digit;
  const int64_t tile_elems = (int64_t)1 << tile_shift;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t_begin = (int64_t)tile * tile_elems;
    const int64_t t_end = t_begin + tile_elems < n ? t_begin + tile_elems : n;
    uint32_t above = 0u;
    for (int64_t base = t_begin; base < t_end; base += kCollStep) {
      // element (u, j) of thread t: base + u * 1024 + 4t + j (coalesced)
      float c[kCollPer];
      bool valid[kCollPer];
#pragma unroll
      for (int u = 0; u < kCollPer / 4; ++u) {
        const int64_t i0 = base + (int64_t)u * (kCollThreads * 4) + 4 * (int64_t)threadIdx.x;
        if (i0 + 3 < t_end) {
          const float4 v = *reinterpret_cast<const float4*>(c_src + i0);
          c[4 * u] = v.x; c[4 * u + 1] = v.y; c[4 * u + 2] = v.z; c[4 * u + 3] = v.w;
          valid[4 * u] = valid[4 * u + 1] = valid[4 * u + 2] = valid[4 * u + 3] = true;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            valid[4 * u + j] = i0 + j < t_end;
            c[4 * u + j] = valid[4 * u + j] ? c_src[i0 + j] : 0.0f;
          }
        }
      }
      uint32_t ncand = 0u;
#pragma unroll
      for (int e = 0; e < kCollPer; ++e) {
        const uint32_t bin = mag_key(c[e]) >> kHistShift;
        above += (valid[e] && bin > B) ? 1u : 0u;
        ncand += (valid[e] && bin == B) ? 1u : 0u;
      }
      uint32_t total;
      const uint32_t off = block_scan<kCollThreads>(ncand, sm.warp_sums, &total);
      if (total == 0u) continue;
      if (threadIdx.x == 0) sm.base = atomicAdd(&ws.sel->cand_count, total);
      __syncthreads();
      if (ncand) {
        uint32_t pos = sm.base + off;
#pragma unroll
        for (int e = 0; e < kCollPer; ++e) {
          const uint32_t key = mag_key(c[e]);
          if (valid[e] && (key >> kHistShift) == B) {
            const int64_t i =
                base + (int64_t)(e >> 2) * (kCollThreads * 4) + 4 * (int64_t)threadIdx.x + (e & 3);
            ws.cand[pos++] = make_uint2(key, (uint32_t)i);
            atomicAdd(&sm.mid[(key >> kLowBits) & (kMidBins - 1)], 1u);
          }
        }
      }
      __syncthreads();
    }
    uint32_t tot;
    block_scan<kCollThreads>(above, sm.warp_sums, &tot);
    if (threadIdx.x == 0) ws.tile_above[tile] = tot;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kMidBins; i += kCollThreads)
    if (sm.mid[i]) atomicAdd(&ws.mid[i], sm.mid[i]);

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sm.last = atomicAdd(&ws.sel->ticket_coll, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  // last block: every other block has read the first-level histogram and
  // added its candidates; find the second digit and reset what it used
  const uint32_t above1 = sm.above, need1 = k - above1;
  for (int i = threadIdx.x; i < kMidBins; i += kCollThreads) {
    sm.mid[i] = __ldcg(&ws.mid[i]);
    ws.mid[i] = 0u;
  }
  for (int i = threadIdx.x; i < kHistBins; i += kCollThreads) ws.hist[i] = 0u;
  __syncthreads();
  if (threadIdx.x == 0) {
    sm.digit = 0xffffffffu;
    sm.above = 0u;
  }
  __syncthreads();
  find_digit<kCollThreads>(sm.mid, kMidBins, need1, sm.warp_sums, &sm.digit, &sm.above);
  if (threadIdx.x == 0) {
    TopkSel* sel = ws.sel;
    const uint32_t cand = __ldcg(&sel->cand_count);
    if (B == 0xffffffffu || sm.digit == 0xffffffffu) atomicOr(ws.status, kStatusTopkSelect);
    if (B != 0xffffffffu && cand != sm.h[B]) atomicOr(ws.status, kStatusTopkCount);
    sel->bin = B;
    sel->above = above1;
    sel->need1 = need1;
    sel->cand_total = B != 0xffffffffu ? sm.h[B] : 0u;
    sel->B2 = sm.digit;
    sel->need2 = need1 - sm.above;
    sel->ticket_coll = 0u;
  }
}

// ---------------------------------------------------------------------------
// pass 3: grid-wide pass over the candidates; the last block finds T and
// the per-tile output offsets.
// ---------------------------------------------------------------------------
constexpr int kRefThreads = 256;
constexpr int kRefUnroll = 4;

struct RefineSmem {
  uint32_t tk[kMaxTiles];
  uint32_t tt[kMaxTiles];
  uint32_t low[kLowBins];
  uint32_t warp_sums[kRefThreads / 32 + 1];
  uint32_t digit, above;
  bool last;
};

__device__ __forceinline__ void count_third_level(RefineSmem& sm, uint2 c, uint32_t T,
                                                  int tile_shift) {
  if (c.x > T) atomicAdd(&sm.tk[c.y >> tile_shift], 1u);
  else if (c.x == T) atomicAdd(&sm.tt[c.y >> tile_shift], 1u);
}

__global__ void __launch_bounds__(kRefThreads) refine_kernel(int ntiles, int tile_shift,
                                                             Workspace ws) {
  __shared__ RefineSmem sm;
  TopkSel* sel = ws.sel;
  for (int i = threadIdx.x; i < ntiles; i += kRefThreads) sm.tk[i] = 0u;
  for (int i = threadIdx.x; i < kLowBins; i += kRefThreads) sm.low[i] = 0u;
  __syncthreads();
  const uint32_t total = __ldcg(&sel->cand_count);
  const uint32_t B2 = __ldcg(&sel->B2);
  const uint32_t step = gridDim.x * kRefThreads * kRefUnroll;
  for (uint32_t j0 = blockIdx.x * kRefThreads * kRefUnroll + threadIdx.x; j0 < total; j0 += step) {
    uint2 c[kRefUnroll];
#pragma unroll
    for (int q = 0; q < kRefUnroll; ++q) {
      const uint32_t j = j0 + q * kRefThreads;
      c[q] = j < total ? __ldcg(&ws.cand[j]) : make_uint2(0u, 0xffffffffu);
    }
#pragma unroll
    for (int q = 0; q < kRefUnroll; ++q) {
      if (c[q].y == 0xffffffffu) continue;
      const uint32_t mid = (c[q].x >> kLowBits) & (kMidBins - 1);
      if (mid > B2) {
        atomicAdd(&sm.tk[c[q].y >> tile_shift], 1u);
      } else if (mid == B2) {
        atomicAdd(&sm.low[c[q].x & (kLowBins - 1)], 1u);
        const uint32_t p = atomicAdd(&sel->stash_count, 1u);
        if (p < kStashMax) ws.stash[p] = c[q];
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ntiles; i += kRefThreads)
    if (sm.tk[i]) atomicAdd(&ws.tile_kept[i], sm.tk[i]);
  for (int i = threadIdx.x; i < kLowBins; i += kRefThreads)
    if (sm.low[i]) atomicAdd(&ws.low[i], sm.low[i]);

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sm.last = atomicAdd(&sel->ticket_refine, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  // last block: third digit, then the per-tile counts of the entries at
  // the threshold's (B, B2) prefix, then the tile offsets
  for (int i = threadIdx.x; i < kLowBins; i += kRefThreads) {
    sm.low[i] = __ldcg(&ws.low[i]);
    ws.low[i] = 0u;
  }
  for (int i = threadIdx.x; i < ntiles; i += kRefThreads) {
    sm.tk[i] = __ldcg(&ws.tile_kept[i]);
    ws.tile_kept[i] = 0u;
    sm.tt[i] = 0u;
  }
  if (threadIdx.x == 0) {
    sm.digit = 0xffffffffu;
    sm.above = 0u;
  }
  __syncthreads();
  const uint32_t need2 = __ldcg(&sel->need2);
  find_digit<kRefThreads>(sm.low, kLowBins, need2, sm.warp_sums, &sm.digit, &sm.above);
  const uint32_t B = __ldcg(&sel->bin), B3 = sm.digit;
  if (B2 == 0xffffffffu || B3 == 0xffffffffu) {
    if (threadIdx.x == 0) atomicOr(ws.status, kStatusTopkSelect);
  }
  const uint32_t T = (B << kHistShift) | (B2 << kLowBits) | (B3 & (kLowBins - 1));
  const uint32_t need_T = need2 - sm.above;
  const uint32_t nstash = __ldcg(&sel->stash_count);
  if (nstash <= kStashMax) {
    for (uint32_t j = threadIdx.x; j < nstash; j += kRefThreads)
      count_third_level(sm, __ldcg(&ws.stash[j]), T, tile_shift);
  } else {  // more than the stash holds (heavy ties): scan the candidates again
    for (uint32_t j = threadIdx.x; j < total; j += kRefThreads) {
      const uint2 c = __ldcg(&ws.cand[j]);
      if (((c.x >> kLowBits) & (kMidBins - 1)) == B2) count_third_level(sm, c, T, tile_shift);
    }
  }
  __syncthreads();
  // tie offsets first, then output offsets including the kept ties
  constexpr int kPerT = kMaxTiles / kRefThreads;  // 8 tiles per thread
  const int t0 = threadIdx.x * kPerT;
  uint32_t ties = 0u;
  for (int t = t0; t < t0 + kPerT && t < ntiles; ++t) ties += sm.tt[t];
  uint32_t tot;
  uint32_t tie_base = block_scan<kRefThreads>(ties, sm.warp_sums, &tot);
  uint32_t kept = 0u;
  {
    uint32_t tb = tie_base;
    for (int t = t0; t < t0 + kPerT && t < ntiles; ++t) {
      const uint32_t rem = need_T > tb ? need_T - tb : 0u;
      kept += __ldcg(&ws.tile_above[t]) + sm.tk[t] + (sm.tt[t] < rem ? sm.tt[t] : rem);
      tb += sm.tt[t];
    }
  }
  uint32_t out_base = block_scan<kRefThreads>(kept, sm.warp_sums, &tot);
  for (int t = t0; t < t0 + kPerT && t < ntiles; ++t) {
    const uint32_t rem = need_T > tie_base ? need_T - tie_base : 0u;
    ws.tile_out[t] = out_base;
    ws.tile_tie[t] = tie_base;
    out_base += __ldcg(&ws.tile_above[t]) + sm.tk[t] + (sm.tt[t] < rem ? sm.tt[t] : rem);
    tie_base += sm.tt[t];
  }
  if (threadIdx.x == 0) {
    sel->T = T;
    sel->need_T = need_T;
    sel->ticket_refine = 0u;
    sel->cand_count = 0u;
    sel->stash_count = 0u;
  }
}

// ---------------------------------------------------------------------------
// pass 4: ordered compaction of the kept entries and e' = 0 at them.
// ---------------------------------------------------------------------------
constexpr int kWrThreads = 256;
constexpr int kWrPer = 16;                      // consecutive elements per thread
constexpr int kWrStep = kWrThreads * kWrPer;    // 4096

template <bool EF>
__global__ void __launch_bounds__(kWrThreads) write_kernel(
    const float* __restrict__ c_src, float* __restrict__ err, int64_t n, uint32_t k,
    int ntiles, int tile_shift, Workspace ws, int32_t* __restrict__ idx_out,
    float* __restrict__ val_out) {
  __shared__ uint32_t warp_sums[kWrThreads / 32 + 1];
  const uint32_t T = ws.sel->T, need_T = ws.sel->need_T;
  const int64_t tile_elems = (int64_t)1 << tile_shift;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t_begin = (int64_t)tile * tile_elems;
    const int64_t t_end = t_begin + tile_elems < n ? t_begin + tile_elems : n;
    uint32_t out = ws.tile_out[tile];
    uint32_t tie_seen = ws.tile_tie[tile];
    for (int64_t base = t_begin; base < t_end; base += kWrStep) {
      // each thread owns 16 consecutive elements, so one block scan per
      // step orders the kept entries by index
      const int64_t i0 = base + (int64_t)kWrPer * threadIdx.x;
      float c[kWrPer];
      bool valid[kWrPer];
#pragma unroll
      for (int u = 0; u < kWrPer / 4; ++u) {
        const int64_t iv = i0 + 4 * u;
        if (iv + 3 < t_end) {
          const float4 v = *reinterpret_cast<const float4*>(c_src + iv);
          c[4 * u] = v.x; c[4 * u + 1] = v.y; c[4 * u + 2] = v.z; c[4 * u + 3] = v.w;
          valid[4 * u] = valid[4 * u + 1] = valid[4 * u + 2] = valid[4 * u + 3] = true;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            valid[4 * u + j] = iv + j < t_end;
            c[4 * u + j] = valid[4 * u + j] ? c_src[iv + j] : 0.0f;
          }
        }
      }
      uint32_t strict = 0u, ties = 0u;
#pragma unroll
      for (int e = 0; e < kWrPer; ++e) {
        const uint32_t key = mag_key(c[e]);
        strict += (valid[e] && key > T) ? 1u : 0u;
        ties += (valid[e] && key == T) ? 1u : 0u;
      }
      uint32_t tot;
      const uint32_t pre = block_scan<kWrThreads>((strict << 16) | ties, warp_sums, &tot);
      const uint32_t strict_pre = pre >> 16, tie_pre = pre & 0xffffu;
      const uint32_t strict_tot = tot >> 16, tie_tot = tot & 0xffffu;
      const uint32_t rem = need_T > tie_seen ? need_T - tie_seen : 0u;
      if (strict + ties != 0u) {
        uint32_t pos = out + strict_pre + (tie_pre < rem ? tie_pre : rem);
        uint32_t tie_rank = tie_pre;
#pragma unroll
        for (int e = 0; e < kWrPer; ++e) {
          const uint32_t key = mag_key(c[e]);
          bool keep = valid[e] && key > T;
          if (valid[e] && key == T) {
            keep = tie_rank < rem;
            ++tie_rank;
          }
          if (keep) {
            if (pos < k) {
              idx_out[pos] = (int32_t)(i0 + e);
              val_out[pos] = c[e];
              if (EF) err[i0 + e] = 0.0f;
            } else {
              atomicOr(ws.status, kStatusTopkOverflow);
            }
            ++pos;
          }
        }
      }
      out += strict_tot + (tie_tot < rem ? tie_tot : rem);
      tie_seen += tie_tot;
    }
  }
}

__global__ void ef_add_kernel(const float* __restrict__ grad, float* __restrict__ err,
                              int64_t n) {
  const int64_t nvec = n >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const float4* g4 = reinterpret_cast<const float4*>(grad);
  float4* e4 = reinterpret_cast<float4*>(err);
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const float4 g = __ldcs(g4 + v);
    float4 e = e4[v];
    e.x = __fadd_rn(g.x, e.x);
    e.y = __fadd_rn(g.y, e.y);
    e.z = __fadd_rn(g.z, e.z);
    e.w = __fadd_rn(g.w, e.w);
    e4[v] = e;
  }
  for (int64_t i = (nvec << 2) + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    err[i] = __fadd_rn(grad[i], err[i]);
}

// Launch geometry of one Top-K call.
struct TopkPlan {
  int tile_shift, ntiles, hist_blocks, coll_blocks, ref_blocks, wr_blocks;
};

TopkPlan topk_plan(int64_t n, int sms) {
  TopkPlan p;
  p.tile_shift = kMinTileShift;
  while (ceil_div(n, (int64_t)1 << p.tile_shift) > kMaxTiles) ++p.tile_shift;
  p.ntiles = (int)ceil_div(n, (int64_t)1 << p.tile_shift);
  p.hist_blocks = (int)std::max<int64_t>(
      1, std::min<int64_t>(ceil_div(ceil_div(n, 4), (int64_t)kHistThreads * kHistUnroll), sms));
  p.coll_blocks = (int)std::min<int64_t>(p.ntiles, (int64_t)sms * 4);
  p.ref_blocks = (int)std::max<int64_t>(
      1, std::min<int64_t>(ceil_div(n, (int64_t)kRefThreads * kRefUnroll * 8), sms));
  p.wr_blocks = (int)std::min<int64_t>(p.ntiles, (int64_t)sms * 6);
  return p;
}

template <class Scope>
gc_status run_topk(const Workspace& ws, cudaStream_t s, int sms, const float* grad,
                   float* err, int64_t n, int64_t k, int32_t* idx_out, float* val_out,
                   Scope&& scope) {
  if (n == 0) return GC_OK;
  if (k == 0) {
    if (err) {
      const int64_t blocks = std::min<int64_t>(ceil_div(ceil_div(n, 4), 256), (int64_t)sms * 8);
      auto L = scope(GC_PHASE_EF_ADD);
      ef_add_kernel<<<(int)blocks, 256, 0, s>>>(grad, err, n);
    }
    return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
  }
  const TopkPlan p = topk_plan(n, sms);
  const float* c_src = err ? err : grad;
  {
    auto L = scope(GC_PHASE_EF_HIST);
    if (err)
      ef_hist_kernel<true><<<p.hist_blocks, kHistThreads, 0, s>>>(grad, err, n, ws);
    else
      ef_hist_kernel<false><<<p.hist_blocks, kHistThreads, 0, s>>>(grad, err, n, ws);
  }
  {
    auto L = scope(GC_PHASE_COLLECT);
    collect_kernel<<<p.coll_blocks, kCollThreads, 0, s>>>(c_src, n, (uint32_t)k, p.ntiles,
                                                          p.tile_shift, ws);
  }
  {
    auto L = scope(GC_PHASE_REFINE);
    refine_kernel<<<p.ref_blocks, kRefThreads, 0, s>>>(p.ntiles, p.tile_shift, ws);
  }
  {
    auto L = scope(GC_PHASE_WRITE);
    if (err)
      write_kernel<true><<<p.wr_blocks, kWrThreads, 0, s>>>(c_src, err, n, (uint32_t)k, p.ntiles,
                                                            p.tile_shift, ws, idx_out, val_out);
    else
      write_kernel<false><<<p.wr_blocks, kWrThreads, 0, s>>>(c_src, err, n, (uint32_t)k,
                                                             p.ntiles, p.tile_shift, ws, idx_out,
                                                             val_out);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

struct NoScope {
  int operator()(int) const { return 0; }
};

}  // namespace

gc_status launch_ef_topk(gc_ctx* ctx, const float* grad, float* err, int64_t n,
                         int64_t k, int32_t* idx_out, float* val_out) {
  return run_topk(ctx->ws, ctx->stream, ctx->num_sms, grad, err, n, k, idx_out, val_out,
                  [ctx](int phase) { return LaunchScope(ctx, phase); });
}

gc_status launch_ef_topk_on(const Workspace& ws, cudaStream_t s, int sms, const float* grad,
                            float* err, int64_t n, int64_t k, int32_t* idx_out,
                            float* val_out) {
  return run_topk(ws, s, sms, grad, err, n, k, idx_out, val_out, NoScope());
}

}  // namespace gc
