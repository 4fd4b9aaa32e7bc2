// gc_topk.cu -- error feedback + exact Top-K selection and compaction.
//
// Semantics ("分布式训练中的梯度压缩算法" 二.2 Top-K 稀疏化; "4、梯度累积与梯度
// 压缩" 4.2.1; "梯度聚合通信优化实战方案" Python 演示 error_feedback_compress):
//   c = g + e; keep the k entries of largest |c| (ties: smaller index);
//   emit (index, c) in ascending index order; e' = c with kept entries = +0.
//
// Design (no sort, no device-wide waits):
//   pass 1  ef_hist   : c = g + e, c written over e, and a 4096-bin histogram
//                       of the top 12 bits of key = bits(|c|).  The last
//                       block to finish (ticket counter) finds the bin B
//                       that holds the k-th largest key.
//   pass 2  collect   : per tile of the array, counts entries above B and
//                       appends the entries of bin B to a candidate list.
//                       The last block refines B to the exact threshold key
//                       T with two more histogram levels over the
//                       candidates (11 + 8 bits), counts per tile the kept
//                       candidates and the ties at T, and scans the tiles
//                       into output offsets.
//   pass 3  write     : per tile, a block scan orders the kept entries and
//                       writes (index, value) and e' = 0 at kept entries.
// Every pass streams 16-byte vectors; pass 1 reads g, e from HBM and the
// re-reads of c in passes 2 and 3 hit L2 when a bucket fits in it.
#include <algorithm>

#include "gc_internal.cuh"

namespace gc {
namespace {

constexpr int kThreads = kTopkThreads;
constexpr int kWarps = kThreads / 32;

// Block-wide exclusive scan of one 32-bit value per thread (kThreads
// threads); returns the exclusive prefix and writes the block total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v,
                                                         uint32_t* warp_sums,
                                                         uint32_t* total) {
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
    uint32_t w = lane < kWarps ? warp_sums[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kWarps) warp_sums[lane] = wi - w;  // exclusive warp offsets
    if (lane == kWarps - 1) warp_sums[kWarps] = wi;
  }
  __syncthreads();
  const uint32_t res = warp_sums[warp] + incl - v;
  *total = warp_sums[kWarps];
  __syncthreads();
  return res;
}

// Finds, over `bins` counts held in shared memory (bin index = value of the
// key digit), the digit D whose cumulative count from the top crosses
// `need`: above(D) < need <= above(D) + hist[D].  Writes D and above(D).
// All threads of the block call it; need >= 1 and the total >= need.
__device__ void find_digit(const uint32_t* hist, int bins, uint32_t need,
                           uint32_t* scratch, uint32_t* out_digit,
                           uint32_t* out_above) {
  const int per = bins / kThreads;  // bins per thread (>= 1 when bins >= kThreads)
  const int nthreads_used = per > 0 ? kThreads : bins;
  const int per_t = per > 0 ? per : 1;
  // thread t owns bins [bins - per_t*(t+1), bins - per_t*t) -- thread 0 the top
  uint32_t s = 0;
  const int hi = bins - per_t * (int)threadIdx.x;
  if ((int)threadIdx.x < nthreads_used)
    for (int b = hi - 1; b >= hi - per_t; --b) s += hist[b];
  uint32_t total;
  const uint32_t before = block_exclusive_scan(s, scratch, &total);
  if ((int)threadIdx.x < nthreads_used && before < need && need <= before + s) {
    uint32_t acc = before;
    for (int b = hi - 1; b >= hi - per_t; --b) {
      if (acc + hist[b] >= need) {
        *out_digit = (uint32_t)b;
        *out_above = acc;
        break;
      }
      acc += hist[b];
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// pass 1: c = g + e (written over e) and the 12-bit histogram of |c|.
// ---------------------------------------------------------------------------
template <bool EF>
__global__ void __launch_bounds__(kThreads) ef_hist_kernel(
    const float* __restrict__ grad, float* __restrict__ err, int64_t n,
    uint32_t k, Workspace ws) {
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t scratch[kWarps + 1];
  __shared__ uint32_t sh_digit, sh_above;
  __shared__ bool last;
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) h[i] = 0u;
  __syncthreads();

  const int64_t nvec = n >> 2;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const float4* g4 = reinterpret_cast<const float4*>(grad);
  float4* e4 = reinterpret_cast<float4*>(err);
  for (int64_t v = (int64_t)blockIdx.x * kThreads + threadIdx.x; v < nvec; v += stride) {
    float4 c = __ldcs(g4 + v);
    if (EF) {
      const float4 e = e4[v];
      c.x = __fadd_rn(c.x, e.x);
      c.y = __fadd_rn(c.y, e.y);
      c.z = __fadd_rn(c.z, e.z);
      c.w = __fadd_rn(c.w, e.w);
      e4[v] = c;
    }
    atomicAdd(&h[mag_key(c.x) >> kHistShift], 1u);
    atomicAdd(&h[mag_key(c.y) >> kHistShift], 1u);
    atomicAdd(&h[mag_key(c.z) >> kHistShift], 1u);
    atomicAdd(&h[mag_key(c.w) >> kHistShift], 1u);
  }
  for (int64_t i = (nvec << 2) + (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride) {
    float c = grad[i];
    if (EF) {
      c = __fadd_rn(c, err[i]);
      err[i] = c;
    }
    atomicAdd(&h[mag_key(c) >> kHistShift], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += kThreads)
    if (h[i]) atomicAdd(&ws.hist[i], h[i]);

  // The last block to arrive owns the complete histogram.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&ws.sel->ticket_hist, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) {
    h[i] = __ldcg(&ws.hist[i]);
    ws.hist[i] = 0u;  // ready for the next call
  }
  if (threadIdx.x == 0) {
    sh_digit = 0xffffffffu;
    sh_above = 0u;
  }
  __syncthreads();
  find_digit(h, kHistBins, k, scratch, &sh_digit, &sh_above);
  if (threadIdx.x == 0) {
    TopkSel* s = ws.sel;
    if (sh_digit == 0xffffffffu) {
      atomicOr(ws.status, kStatusTopkSelect);
      sh_digit = 0u;
    }
    s->bin = sh_digit;
    s->above = sh_above;
    s->need1 = k - sh_above;
    s->cand_total = h[sh_digit];
    s->cand_count = 0u;
    s->ticket_hist = 0u;
  }
}

// Loads the 4 elements of a block step starting at i0 (i0 % 4 == 0).
__device__ __forceinline__ void load4(const float* src, int64_t i0, int64_t end,
                                      float c[4], bool valid[4]) {
  if (i0 + 3 < end) {
    const float4 v = *reinterpret_cast<const float4*>(src + i0);
    c[0] = v.x; c[1] = v.y; c[2] = v.z; c[3] = v.w;
    valid[0] = valid[1] = valid[2] = valid[3] = true;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      valid[j] = i0 + j < end;
      c[j] = valid[j] ? src[i0 + j] : 0.0f;
    }
  }
}

// Refinement inside the last block of pass 2 (kThreads threads).
struct RefineSmem {
  uint32_t mid[kMidBins];
  uint32_t low[kLowBins];
  uint32_t tile_kept[kMaxTiles];
  uint32_t tile_ties[kMaxTiles];
};

__device__ void refine_threshold(Workspace ws, int ntiles, int64_t tile_elems,
                                 RefineSmem& sm, uint32_t* scratch) {
  __shared__ uint32_t sh_digit, sh_above;
  TopkSel* sel = ws.sel;
  const uint32_t total = __ldcg(&sel->cand_count);
  const uint32_t need1 = __ldcg(&sel->need1);
  const uint32_t B = __ldcg(&sel->bin);
  if (threadIdx.x == 0 && total != __ldcg(&sel->cand_total))
    atomicOr(ws.status, kStatusTopkCount);

  // level 2: bits 18..8 of the candidates' keys
  for (int i = threadIdx.x; i < kMidBins; i += kThreads) sm.mid[i] = 0u;
  for (int i = threadIdx.x; i < kLowBins; i += kThreads) sm.low[i] = 0u;
  for (int i = threadIdx.x; i < ntiles; i += kThreads) {
    sm.tile_kept[i] = 0u;
    sm.tile_ties[i] = 0u;
  }
  if (threadIdx.x == 0) { sh_digit = 0xffffffffu; sh_above = 0u; }
  __syncthreads();
  for (uint32_t j = threadIdx.x; j < total; j += kThreads)
    atomicAdd(&sm.mid[(__ldcg(&ws.cand[j].x) >> kLowBits) & (kMidBins - 1)], 1u);
  __syncthreads();
  find_digit(sm.mid, kMidBins, need1, scratch, &sh_digit, &sh_above);
  const uint32_t B2 = sh_digit, above2 = sh_above;
  const uint32_t need2 = need1 - above2;
  __syncthreads();
  if (threadIdx.x == 0) { sh_digit = 0xffffffffu; sh_above = 0u; }
  // level 3: bits 7..0 of the candidates whose bits 18..8 equal B2
  for (uint32_t j = threadIdx.x; j < total; j += kThreads) {
    const uint32_t key = __ldcg(&ws.cand[j].x);
    if (((key >> kLowBits) & (kMidBins - 1)) == B2)
      atomicAdd(&sm.low[key & (kLowBins - 1)], 1u);
  }
  __syncthreads();
  find_digit(sm.low, kLowBins, need2, scratch, &sh_digit, &sh_above);
  const uint32_t B3 = sh_digit, above3 = sh_above;
  if (B2 == 0xffffffffu || B3 == 0xffffffffu) {
    if (threadIdx.x == 0) atomicOr(ws.status, kStatusTopkSelect);
  }
  const uint32_t T = (B << kHistShift) | (B2 << kLowBits) | B3;
  const uint32_t need_T = need2 - above3;
  // per-tile counts of kept candidates (key > T) and ties (key == T)
  for (uint32_t j = threadIdx.x; j < total; j += kThreads) {
    const uint2 c = __ldcg(&ws.cand[j]);
    const int tile = (int)((int64_t)c.y / tile_elems);
    if (c.x > T) atomicAdd(&sm.tile_kept[tile], 1u);
    else if (c.x == T) atomicAdd(&sm.tile_ties[tile], 1u);
  }
  __syncthreads();
  // scan tiles: tie offsets first, then output offsets including kept ties
  const int per = (ntiles + kThreads - 1) / kThreads;
  const int t0 = threadIdx.x * per;
  uint32_t ties = 0u;
  for (int t = t0; t < t0 + per && t < ntiles; ++t) ties += sm.tile_ties[t];
  uint32_t tot;
  uint32_t tie_base = block_exclusive_scan(ties, scratch, &tot);
  uint32_t kept = 0u;
  {
    uint32_t tb = tie_base;
    for (int t = t0; t < t0 + per && t < ntiles; ++t) {
      const uint32_t tt = sm.tile_ties[t];
      const uint32_t rem = need_T > tb ? need_T - tb : 0u;
      kept += __ldcg(&ws.tile_above[t]) + sm.tile_kept[t] + (tt < rem ? tt : rem);
      tb += tt;
    }
  }
  uint32_t out_base = block_exclusive_scan(kept, scratch, &tot);
  for (int t = t0; t < t0 + per && t < ntiles; ++t) {
    const uint32_t tt = sm.tile_ties[t];
    const uint32_t rem = need_T > tie_base ? need_T - tie_base : 0u;
    ws.tile_out[t] = out_base;
    ws.tile_tie[t] = tie_base;
    out_base += __ldcg(&ws.tile_above[t]) + sm.tile_kept[t] + (tt < rem ? tt : rem);
    tie_base += tt;
  }
  if (threadIdx.x == 0) {
    sel->T = T;
    sel->need_T = need_T;
    sel->ticket_coll = 0u;
    sel->cand_count = 0u;
  }
}

// ---------------------------------------------------------------------------
// pass 2: per-tile counts above B and the candidate list of bin B.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) collect_kernel(
    const float* __restrict__ c_src, int64_t n, int ntiles, int64_t tile_elems,
    Workspace ws) {
  __shared__ RefineSmem sm;
  __shared__ uint32_t scratch[kWarps + 1];
  __shared__ uint32_t sh_base;
  __shared__ bool last;
  const uint32_t B = ws.sel->bin;

  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t_begin = (int64_t)tile * tile_elems;
    const int64_t t_end = t_begin + tile_elems < n ? t_begin + tile_elems : n;
    uint32_t above = 0u;
    for (int64_t base = t_begin; base < t_end; base += kTopkSub) {
      const int64_t i0 = base + 4 * (int64_t)threadIdx.x;
      float c[4];
      bool valid[4];
      load4(c_src, i0, t_end, c, valid);
      uint32_t keys[4], ncand = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        keys[j] = mag_key(c[j]);
        const uint32_t bin = keys[j] >> kHistShift;
        above += (valid[j] && bin > B) ? 1u : 0u;
        ncand += (valid[j] && bin == B) ? 1u : 0u;
      }
      uint32_t total;
      const uint32_t off = block_exclusive_scan(ncand, scratch, &total);
      if (total == 0u) continue;
      if (threadIdx.x == 0) sh_base = atomicAdd(&ws.sel->cand_count, total);
      __syncthreads();
      uint32_t pos = sh_base + off;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (valid[j] && (keys[j] >> kHistShift) == B)
          ws.cand[pos++] = make_uint2(keys[j], (uint32_t)(i0 + j));
      __syncthreads();
    }
    uint32_t tot;
    block_exclusive_scan(above, scratch, &tot);
    if (threadIdx.x == 0) ws.tile_above[tile] = tot;
  }

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&ws.sel->ticket_coll, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  refine_threshold(ws, ntiles, tile_elems, sm, scratch);
}

// ---------------------------------------------------------------------------
// pass 3: ordered compaction of the kept entries and e' = 0 at them.
// ---------------------------------------------------------------------------
template <bool EF>
__global__ void __launch_bounds__(kThreads) write_kernel(
    const float* __restrict__ c_src, float* __restrict__ err, int64_t n,
    uint32_t k, int ntiles, int64_t tile_elems, Workspace ws,
    int32_t* __restrict__ idx_out, float* __restrict__ val_out) {
  __shared__ uint32_t scratch[kWarps + 1];
  const uint32_t T = ws.sel->T, need_T = ws.sel->need_T;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t_begin = (int64_t)tile * tile_elems;
    const int64_t t_end = t_begin + tile_elems < n ? t_begin + tile_elems : n;
    uint32_t out = ws.tile_out[tile];
    uint32_t tie_seen = ws.tile_tie[tile];
    for (int64_t base = t_begin; base < t_end; base += kTopkSub) {
      const int64_t i0 = base + 4 * (int64_t)threadIdx.x;
      float c[4];
      bool valid[4];
      load4(c_src, i0, t_end, c, valid);
      uint32_t strict = 0u, ties = 0u;
      bool is_strict[4], is_tie[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t key = mag_key(c[j]);
        is_strict[j] = valid[j] && key > T;
        is_tie[j] = valid[j] && key == T;
        strict += is_strict[j];
        ties += is_tie[j];
      }
      uint32_t tot;
      const uint32_t pre = block_exclusive_scan((strict << 16) | ties, scratch, &tot);
      const uint32_t strict_pre = pre >> 16, tie_pre = pre & 0xffffu;
      const uint32_t strict_tot = tot >> 16, tie_tot = tot & 0xffffu;
      const uint32_t rem = need_T > tie_seen ? need_T - tie_seen : 0u;
      uint32_t pos = out + strict_pre + (tie_pre < rem ? tie_pre : rem);
      uint32_t tie_rank = tie_pre;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bool keep = is_strict[j];
        if (is_tie[j]) {
          keep = tie_rank < rem;
          ++tie_rank;
        }
        if (keep) {
          if (pos < k) {
            idx_out[pos] = (int32_t)(i0 + j);
            val_out[pos] = c[j];
            if (EF) err[i0 + j] = 0.0f;
          } else {
            atomicOr(ws.status, kStatusTopkOverflow);
          }
          ++pos;
        }
      }
      out += strict_tot + (tie_tot < rem ? tie_tot : rem);
      tie_seen += tie_tot;
    }
  }
}

__global__ void ef_add_kernel(const float* __restrict__ grad,
                              float* __restrict__ err, int64_t n) {
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

}  // namespace

gc_status launch_ef_topk(gc_ctx* ctx, const float* grad, float* err, int64_t n,
                         int64_t k, int32_t* idx_out, float* val_out) {
  cudaStream_t s = ctx->stream;
  const int sms = ctx->num_sms;
  if (n == 0) return GC_OK;
  if (k == 0) {
    if (err) {
      const int64_t blocks = std::min<int64_t>(ceil_div(ceil_div(n, 4), 256), (int64_t)sms * 8);
      LaunchScope L(ctx, GC_PHASE_EF_ADD);
      ef_add_kernel<<<(int)blocks, 256, 0, s>>>(grad, err, n);
    }
    return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
  }
  const int64_t tile_elems =
      std::max<int64_t>(kTopkSub, round_up(ceil_div(n, kMaxTiles), kTopkSub));
  const int ntiles = (int)ceil_div(n, tile_elems);
  const int64_t hist_blocks =
      std::max<int64_t>(1, std::min<int64_t>(ceil_div(ceil_div(n, 4), kThreads), (int64_t)sms * 4));
  const int pass_blocks = (int)std::min<int64_t>(ntiles, (int64_t)sms * 4);
  const float* c_src = err ? err : grad;
  {
    LaunchScope L(ctx, GC_PHASE_EF_HIST);
    if (err)
      ef_hist_kernel<true><<<(int)hist_blocks, kThreads, 0, s>>>(grad, err, n, (uint32_t)k, ctx->ws);
    else
      ef_hist_kernel<false><<<(int)hist_blocks, kThreads, 0, s>>>(grad, err, n, (uint32_t)k, ctx->ws);
  }
  {
    LaunchScope L(ctx, GC_PHASE_COLLECT);
    collect_kernel<<<pass_blocks, kThreads, 0, s>>>(c_src, n, ntiles, tile_elems, ctx->ws);
  }
  LaunchScope L(ctx, GC_PHASE_WRITE);
  if (err)
    write_kernel<true><<<pass_blocks, kThreads, 0, s>>>(c_src, err, n, (uint32_t)k, ntiles,
                                                        tile_elems, ctx->ws, idx_out, val_out);
  else
    write_kernel<false><<<pass_blocks, kThreads, 0, s>>>(c_src, err, n, (uint32_t)k, ntiles,
                                                         tile_elems, ctx->ws, idx_out, val_out);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

gc_status launch_ef_topk_on(const Workspace& ws, cudaStream_t s, int sms, const float* grad,
                            float* err, int64_t n, int64_t k, int32_t* idx_out,
                            float* val_out) {
  if (n == 0) return GC_OK;
  if (k == 0) {
    if (err) {
      const int64_t blocks = std::min<int64_t>(ceil_div(ceil_div(n, 4), 256), (int64_t)sms * 8);
      ef_add_kernel<<<(int)blocks, 256, 0, s>>>(grad, err, n);
    }
    return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
  }
  const int64_t tile_elems =
      std::max<int64_t>(kTopkSub, round_up(ceil_div(n, kMaxTiles), kTopkSub));
  const int ntiles = (int)ceil_div(n, tile_elems);
  const int64_t hist_blocks =
      std::max<int64_t>(1, std::min<int64_t>(ceil_div(ceil_div(n, 4), kThreads), (int64_t)sms * 4));
  const int pass_blocks = (int)std::min<int64_t>(ntiles, (int64_t)sms * 4);
  const float* c_src = err ? err : grad;
  if (err)
    ef_hist_kernel<true><<<(int)hist_blocks, kThreads, 0, s>>>(grad, err, n, (uint32_t)k, ws);
  else
    ef_hist_kernel<false><<<(int)hist_blocks, kThreads, 0, s>>>(grad, err, n, (uint32_t)k, ws);
  collect_kernel<<<pass_blocks, kThreads, 0, s>>>(c_src, n, ntiles, tile_elems, ws);
  if (err)
    write_kernel<true><<<pass_blocks, kThreads, 0, s>>>(c_src, err, n, (uint32_t)k, ntiles,
                                                        tile_elems, ws, idx_out, val_out);
  else
    write_kernel<false><<<pass_blocks, kThreads, 0, s>>>(c_src, err, n, (uint32_t)k, ntiles,
                                                         tile_elems, ws, idx_out, val_out);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace gc
