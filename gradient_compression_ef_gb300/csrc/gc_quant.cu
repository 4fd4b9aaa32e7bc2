// gc_quant.cu -- group-wise quantisation, bit packing, dequantisation and
// the error-feedback residual.
//
// Formulas ("分布式训练中的梯度压缩算法" 二.1 线性量化 and 三 误差补偿;
// "gradient-compression-quantization-sparsification" 1.1 QSGD / TernGrad,
// 1.2 groups and rounding):
//   min-max : scale = (max - min) / (2^b - 1), t = (c - min) / scale,
//             g_hat = q * scale + min
//   QSGD    : scale = ||c_group||_2 / (2^b - 1), t = |c| / scale,
//             g_hat = sign * q * scale  (sum of squares as the adjacent-pair
//             binary tree over the group)
//   TernGrad: scale = max |c_group|, t = |c| / scale, q in {0, 1}
//   q = rint(t) or floor(t) + [u < frac(t)], clamped; e' = c - g_hat.
//
// Kernels:
//   quant_fused  : groups of 4..128 elements (a power of two).  One pass:
//                  each lane holds 4 consecutive elements, a group is G/4
//                  lanes and its statistics are warp butterflies.  Reads g
//                  and e (or x), writes codes, scales and e'.  The hybrid
//                  call runs it over the kept values and scatters e'.
//   quant_stats  : other group sizes.  One warp per chunk of a group (the
//                  whole group, or power-of-two chunks of a large group);
//                  with error feedback it also writes c over e.
//   quant_combine: combines the chunk statistics of large groups in the same
//                  tree order.
//   quant_apply  : elementwise quantise + pack (+ e' = c - g_hat).
//   dequant      : elementwise g_hat from codes and scales.
#include <algorithm>

#include "gc_internal.cuh"

namespace gc {

QuantPlan quant_plan(int64_t n, int64_t group) {
  QuantPlan p;
  p.G = group == 0 ? n : group;
  if (p.G < 1) p.G = 1;
  p.ngroups = n == 0 ? 0 : ceil_div(n, p.G);
  if (p.G <= 1024) {
    p.chunk = p.G;
    p.chunks_per_group = 1;
  } else {
    // at most about 4096 chunks per group: enough warps for the statistics
    // pass, few partials for the combine (chunk sizes stay powers of two,
    // so the QSGD summation tree is the same for any of them)
    int64_t target = ceil_div(p.G, 4096);
    int64_t c = 1024;
    while (c < target) c <<= 1;
    p.chunk = c;
    p.chunks_per_group = ceil_div(p.G, c);
  }
  p.nchunks = p.ngroups == 0 ? 0
                             : (p.ngroups - 1) * p.chunks_per_group +
                                   ceil_div(n - (p.ngroups - 1) * p.G, p.chunk);
  return p;
}

namespace {

constexpr int kQThreads = 256;

enum IoKind { IO_PLAIN = 0, IO_EF = 1, IO_SCATTER = 2, IO_DIFF = 3 };

struct QuantOut {
  uint8_t* codes;
  uint8_t* signs;        // QSGD sign plane (NULL otherwise)
  float* scales;
  int64_t zero_begin, zero_end;    // padding bytes of the code section
  int64_t szero_begin, szero_end;  // padding bytes of the sign plane
  int64_t scatter_n;               // length of err for the scattered residual
  uint32_t* status;                // device status word
  float* ref;                      // differential quantisation: the history
  int refresh;                     // differential quantisation: ref taken as 0
  uint2* patch;                    // deferred residuals: (position, bits of e') per entry
  int64_t patch_tail;              // positions from here on are also written to err
};

__device__ __forceinline__ void zero_padding_bytes(const QuantOut& o) {
  for (int64_t b = o.zero_begin; b < o.zero_end; ++b) o.codes[b] = 0;
  if (o.signs)
    for (int64_t b = o.szero_begin; b < o.szero_end; ++b) o.signs[b] = 0;
}

__device__ __forceinline__ void zero_padding(const QuantOut& o) {
  if (blockIdx.x == 0 && threadIdx.x == 0) zero_padding_bytes(o);
}

template <int MODE, int BITS>
__device__ __forceinline__ uint32_t code_bits4(const uint32_t q[4], const bool neg[4]) {
  if (MODE == GC_TERN || MODE == GC_LOG) {  // sign-magnitude
    constexpr int SB = MODE == GC_TERN ? 1 : BITS - 1;
    uint32_t t[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) t[j] = q[j] | ((uint32_t)neg[j] << SB);
    return pack4<(MODE == GC_TERN) ? 2 : BITS>(t);
  }
  return pack4<BITS>(q);
}

// ---------------------------------------------------------------------------
// Fused single-pass kernel for groups of G = 4 * LPG elements.
// ---------------------------------------------------------------------------
// Values of elements i0 .. i0+3 of a chunk: c = x (+ e with error
// feedback); lanes past n get zeros and valid = false.
template <int IO>
__device__ __forceinline__ void quant_load4(const float* __restrict__ x,
                                            const float* __restrict__ err, int64_t n,
                                            int64_t i0, float c[4], bool valid[4]) {
  if (i0 + 3 < n) {
    const float4 v = IO == IO_EF ? __ldcs(reinterpret_cast<const float4*>(x + i0))
                                 : *reinterpret_cast<const float4*>(x + i0);
    c[0] = v.x; c[1] = v.y; c[2] = v.z; c[3] = v.w;
    valid[0] = valid[1] = valid[2] = valid[3] = true;
    if (IO == IO_EF) {
      const float4 e = *reinterpret_cast<const float4*>(err + i0);
      c[0] = __fadd_rn(c[0], e.x);
      c[1] = __fadd_rn(c[1], e.y);
      c[2] = __fadd_rn(c[2], e.z);
      c[3] = __fadd_rn(c[3], e.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      valid[j] = i0 + j < n;
      c[j] = valid[j] ? x[i0 + j] : 0.0f;
      if (IO == IO_EF && valid[j]) c[j] = __fadd_rn(c[j], err[i0 + j]);
    }
  }
}

// One warp quantises elements base .. base+127 of x (groups of G = 4 * LPG
// consecutive lanes, G dividing 128), lane l holding elements base + 4l ..
// base + 4l + 3 with values c[] (from quant_load4).  Every lane of the warp
// must call it.
// With DIAG, dsum[0] and dsum[1] accumulate this lane's g_hat^2 and e'^2.
// IO_DIFF writes no residual: the dequantised values go to ghat_out[4].
template <int MODE, int BITS, int LPG, int IO, bool DIAG = false>
__device__ __forceinline__ void quant_fused_apply(
    float c[4], const bool valid[4], float* __restrict__ err,
    const int32_t* __restrict__ scatter_idx, int64_t n, const QuantOut& o,
    int stochastic, uint64_t seed, uint64_t step, int64_t base, int lane,
    float* dsum = nullptr, float* ghat_out = nullptr) {
  constexpr int G = 4 * LPG;
  constexpr uint32_t top = mode_top<MODE, BITS>();
  const float levels = (float)top;
  const int64_t i0 = base + 4 * lane;
  const bool active = i0 < n;

  // group statistics (lanes of a group are LPG consecutive lanes)
  float scale, offset = 0.0f;
  if (MODE == GC_MINMAX) {
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (valid[j]) { mn = fminf(mn, c[j]); mx = fmaxf(mx, c[j]); }
#pragma unroll
    for (int o2 = 1; o2 < LPG; o2 <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
    }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    scale = __fdiv_rn(__fsub_rn(mx, mn), levels);
    offset = mn;
  } else if (MODE == GC_QSGD) {
    float s = __fadd_rn(__fadd_rn(__fmul_rn(c[0], c[0]), __fmul_rn(c[1], c[1])),
                        __fadd_rn(__fmul_rn(c[2], c[2]), __fmul_rn(c[3], c[3])));
    s = warp_sum_tree(s, LPG);
    scale = __fdiv_rn(__fsqrt_rn(s), levels);
  } else {  // TernGrad, logarithmic: max |c|
    float m = fmaxf(fmaxf(fabsf(c[0]), fabsf(c[1])), fmaxf(fabsf(c[2]), fabsf(c[3])));
#pragma unroll
    for (int o2 = 1; o2 < LPG; o2 <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o2));
    scale = MODE == GC_LOG ? __fdiv_rn(cw_logf(__fadd_rn(m, 1.0f)), levels) : m;
  }
  if (active && (lane % LPG) == 0) {
    const int64_t g = i0 / G;
    if (MODE == GC_MINMAX)
      reinterpret_cast<float2*>(o.scales)[g] = make_float2(scale, offset);
    else
      o.scales[g] = scale;
  }

  float u[4] = {0.f, 0.f, 0.f, 0.f};
  if (stochastic) uniform4((uint64_t)i0 >> 2, seed, step, u);
  uint32_t q[4];
  bool neg[4];
  float r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float gh;
    q[j] = quantize_one<MODE>(c[j], scale, offset, stochastic != 0, u[j], top, &neg[j], &gh);
    if (!valid[j]) { q[j] = 0u; neg[j] = false; }
    if (IO == IO_DIFF) ghat_out[j] = gh;
    r[j] = __fsub_rn(c[j], gh);
    if (DIAG && valid[j]) {
      dsum[0] = __fmaf_rn(gh, gh, dsum[0]);
      dsum[1] = __fmaf_rn(r[j], r[j], dsum[1]);
    }
  }
  store_codes4<(MODE == GC_TERN) ? 2 : BITS>(o.codes, i0, active, code_bits4<MODE, BITS>(q, neg));
  if (MODE == GC_QSGD) {
    const bool s4[4] = {neg[0], neg[1], neg[2], neg[3]};
    uint32_t sb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) sb[j] = s4[j] ? 1u : 0u;
    store_codes4<1>(o.signs, i0, active, pack4<1>(sb));
  }
  if (IO == IO_EF) {
    if (i0 + 3 < n) {
      __stcs(reinterpret_cast<float4*>(err + i0), make_float4(r[0], r[1], r[2], r[3]));
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (valid[j]) err[i0 + j] = r[j];
    }
  } else if (IO == IO_SCATTER) {
    if (o.patch) {
      // deferred: (position, e') pairs in entry order, coalesced; the next
      // read of e applies them.  An entry with a bad position gets one that
      // matches no element.
      uint2 pr[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pr[j] = make_uint2(0xffffffffu, 0u);
        if (!valid[j]) continue;
        const int32_t t = scatter_idx[i0 + j];
        if (t >= 0 && (int64_t)t < o.scatter_n) {
          pr[j] = make_uint2((uint32_t)t, __float_as_uint(r[j]));
          if ((int64_t)t >= o.patch_tail) err[t] = r[j];
        } else {
          atomicOr(o.status, kStatusScatterIndex);
        }
      }
      if (i0 + 3 < n) {
        uint4* dst = reinterpret_cast<uint4*>(o.patch + i0);
        dst[0] = make_uint4(pr[0].x, pr[0].y, pr[1].x, pr[1].y);
        dst[1] = make_uint4(pr[2].x, pr[2].y, pr[3].x, pr[3].y);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (valid[j]) o.patch[i0 + j] = pr[j];
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!valid[j]) continue;
        const int32_t t = scatter_idx[i0 + j];
        if (t >= 0 && (int64_t)t < o.scatter_n) err[t] = r[j];
        else atomicOr(o.status, kStatusScatterIndex);
      }
    }
  }
}

// Load + quantise of one 128-element chunk (the bucketed kernel's unit).
template <int MODE, int BITS, int LPG, int IO, bool DIAG = false>
__device__ __forceinline__ void quant_fused_chunk(
    const float* __restrict__ x, float* __restrict__ err,
    const int32_t* __restrict__ scatter_idx, int64_t n, const QuantOut& o,
    int stochastic, uint64_t seed, uint64_t step, int64_t base, int lane,
    float* dsum = nullptr) {
  float c[4];
  bool valid[4];
  quant_load4<IO>(x, err, n, base + 4 * lane, c, valid);
  quant_fused_apply<MODE, BITS, LPG, IO, DIAG>(c, valid, err, scatter_idx, n, o, stochastic,
                                               seed, step, base, lane, dsum);
}

// The fused kernel gives every warp a contiguous run of 128-element chunks
// and keeps the next kQStages - 1 chunks of x (and e) in flight as
// asynchronous copies into the warp's shared-memory stages while it
// quantises the current one; each lane copies and later reads back its own
// 16-byte pieces, so no barrier is involved.  The grid is one wave of
// resident blocks.
constexpr int kQStages = 4;

template <int MODE, int BITS, int LPG, int IO>
__global__ void __launch_bounds__(kQThreads, 5) quant_fused_kernel(
    const float* __restrict__ x, float* __restrict__ err,
    const int32_t* __restrict__ scatter_idx, int64_t n, QuantOut o,
    int stochastic, uint64_t seed, uint64_t step) {
  constexpr int NW = kQThreads / 32;
  constexpr int S = IO == IO_DIFF ? kQStages - 1 : kQStages;  // 36 KB at most
  // staged arrays: x (and e; and the history for differential quantisation)
  constexpr int NA = IO == IO_DIFF ? 3 : IO == IO_EF ? 2 : 1;
  __shared__ float4 stage[NW][S][NA][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  zero_padding(o);
  const int64_t nch = (n + 127) >> 7;
  const int64_t gw = (int64_t)blockIdx.x * NW + warp, nw = (int64_t)gridDim.x * NW;
  const int64_t c_lo = nch * gw / nw;
  const int cnt = (int)(nch * (gw + 1) / nw - c_lo);  // chunks of this warp
  // lane's piece of the warp's first chunk; whole pieces are copied, the
  // ragged end of x is read directly when its chunk is processed
  const int64_t i_first = (c_lo << 7) + 4 * lane;
  const bool has_err = IO == IO_EF || (IO == IO_DIFF && err != nullptr);
  const bool use_ref = IO == IO_DIFF && !o.refresh;
  auto issue = [&](int j, int st) {
    const int64_t i0 = i_first + ((int64_t)j << 7);
    if (j < cnt && i0 + 3 < n) {
      cp_async16(&stage[warp][st][0][lane], x + i0);
      if (has_err) cp_async16(&stage[warp][st][1][lane], err + i0);
      if (use_ref) cp_async16(&stage[warp][st][NA - 1][lane], o.ref + i0);
    }
    cp_async_commit();  // one group per chunk (possibly empty)
  };
#pragma unroll
  for (int k = 0; k < S - 1; ++k) issue(k, k);
  int st = 0;
  for (int j = 0; j < cnt; ++j) {
    cp_async_wait<S - 2>();  // chunk j has landed
    const int64_t i0 = i_first + ((int64_t)j << 7);
    float c[4], rf[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    bool valid[4];
    if (i0 + 3 < n) {
      const float4 v = stage[warp][st][0][lane];
      c[0] = v.x; c[1] = v.y; c[2] = v.z; c[3] = v.w;
      valid[0] = valid[1] = valid[2] = valid[3] = true;
      if (has_err) {
        const float4 e = stage[warp][st][1][lane];
        c[0] = __fadd_rn(c[0], e.x);
        c[1] = __fadd_rn(c[1], e.y);
        c[2] = __fadd_rn(c[2], e.z);
        c[3] = __fadd_rn(c[3], e.w);
      }
      if (use_ref) {
        const float4 h = stage[warp][st][NA - 1][lane];
        rf[0] = h.x; rf[1] = h.y; rf[2] = h.z; rf[3] = h.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        valid[q] = i0 + q < n;
        c[q] = valid[q] ? x[i0 + q] : 0.0f;
        if (has_err && valid[q]) c[q] = __fadd_rn(c[q], err[i0 + q]);
        if (use_ref && valid[q]) rf[q] = o.ref[i0 + q];
      }
    }
    // the stage read one chunk ago is free: refill it S - 1 ahead
    issue(j + S - 1, st == 0 ? S - 1 : st - 1);
    if (IO == IO_DIFF) {
      // quantise d = c - r; g_hat = r + d_hat; e' = c - g_hat; ref' = g_hat
      float d[4], dh[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) d[q] = valid[q] ? __fsub_rn(c[q], rf[q]) : 0.0f;
      quant_fused_apply<MODE, BITS, LPG, IO>(d, valid, err, scatter_idx, n, o, stochastic,
                                             seed, step, i0 - 4 * lane, lane, nullptr, dh);
      float gh[4], e2[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        gh[q] = __fadd_rn(rf[q], dh[q]);
        e2[q] = __fsub_rn(c[q], gh[q]);
      }
      if (i0 + 3 < n) {
        __stcs(reinterpret_cast<float4*>(o.ref + i0), make_float4(gh[0], gh[1], gh[2], gh[3]));
        if (has_err)
          __stcs(reinterpret_cast<float4*>(err + i0), make_float4(e2[0], e2[1], e2[2], e2[3]));
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (!valid[q]) continue;
          o.ref[i0 + q] = gh[q];
          if (has_err) err[i0 + q] = e2[q];
        }
      }
    } else {
      quant_fused_apply<MODE, BITS, LPG, IO>(c, valid, err, scatter_idx, n, o, stochastic,
                                             seed, step, i0 - 4 * lane, lane);
    }
    st = st + 1 == S ? 0 : st + 1;
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Multi-pass path: statistics per chunk (one warp per chunk).
// ---------------------------------------------------------------------------

// Running adjacent-pair tree over equal-sized consecutive nodes: node j of
// the stream enters as a leaf of the tree of nodes; carry[l] holds a pending
// complete subtree of 2^l nodes (bit l of count).  Identical in all lanes.
struct TreeAcc {
  float carry[32];
  uint32_t count;
  __device__ __forceinline__ void init() { count = 0u; }
  __device__ __forceinline__ void push(float v) {
    int l = 0;
    while (count & (1u << l)) {
      v = __fadd_rn(carry[l], v);
      ++l;
    }
    carry[l] = v;
    count += 1u;
  }
  // Sum of the zero-padded tree: fold pending subtrees right to left.
  __device__ __forceinline__ float finish() const {
    float acc = 0.0f;
    bool any = false;
    for (int l = 0; l < 32; ++l) {
      if (count & (1u << l)) {
        acc = any ? __fadd_rn(carry[l], acc) : carry[l];
        any = true;
      }
    }
    return acc;
  }
};

template <int MODE>
__device__ __forceinline__ void finalize_group(float mn, float mx, float amax, float ss,
                                               uint32_t top, float* scales, int64_t g) {
  const float levels = (float)top;
  if (MODE == GC_MINMAX) {
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    reinterpret_cast<float2*>(scales)[g] =
        make_float2(__fdiv_rn(__fsub_rn(mx, mn), levels), mn);
  } else if (MODE == GC_QSGD) {
    scales[g] = __fdiv_rn(__fsqrt_rn(ss), levels);
  } else if (MODE == GC_LOG) {
    scales[g] = __fdiv_rn(cw_logf(__fadd_rn(amax, 1.0f)), levels);
  } else {
    scales[g] = amax;
  }
}

template <int MODE, int IO>
__global__ void __launch_bounds__(kQThreads) quant_stats_kernel(
    const float* __restrict__ x, float* __restrict__ err, int64_t n, int64_t G,
    int64_t chunk, int64_t cpg, int64_t nchunks, uint32_t top,
    float4* __restrict__ partials, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = ((int64_t)blockIdx.x * kQThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kQThreads) >> 5;
  // 16-byte loads need every group to start on a 4-element boundary (or a
  // single group starting at element 0)
  const bool vec_ok = (G % 4) == 0 || G >= n;
  constexpr int NA = IO == IO_EF ? 2 : 1;
  __shared__ float4 stage[kQThreads / 32][kQStages][NA][32];
  const int warp = threadIdx.x >> 5;
  for (int64_t ch = warp_id; ch < nchunks; ch += nwarps) {
    const int64_t g = ch / cpg, cc = ch % cpg;
    const int64_t g_begin = g * G;
    const int64_t g_end = std::min<int64_t>(g_begin + G, n);
    const int64_t begin = g_begin + cc * chunk;
    const int64_t end = std::min<int64_t>(begin + chunk, g_end);
    float mn = INFINITY, mx = -INFINITY, amax = 0.0f;
    TreeAcc tree;
    tree.init();
    // the chunk's 128-element rows with kQStages - 1 of them in flight as
    // asynchronous copies
    const int niter = (int)((end - begin + 127) >> 7);
    auto issue = [&](int it, int st) {
      const int64_t i0 = begin + ((int64_t)it << 7) + 4 * lane;
      if (it < niter && vec_ok && i0 + 3 < end) {
        cp_async16(&stage[warp][st][0][lane], x + i0);
        if (IO == IO_EF) cp_async16(&stage[warp][st][NA - 1][lane], err + i0);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < kQStages - 1; ++k) issue(k, k);
    int st = 0;
    for (int it = 0; it < niter; ++it) {
      cp_async_wait<kQStages - 2>();
      const int64_t i0 = begin + ((int64_t)it << 7) + 4 * lane;
      float c[4];
      const bool vec = vec_ok && i0 + 3 < end;
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f), ev = v;
      if (vec) {
        v = stage[warp][st][0][lane];
        if (IO == IO_EF) ev = stage[warp][st][NA - 1][lane];
      }
      issue(it + kQStages - 1, st == 0 ? kQStages - 1 : st - 1);
      st = st + 1 == kQStages ? 0 : st + 1;
      if (vec) {
        if (IO == IO_EF) {
          const float4 e = ev;
          v.x = __fadd_rn(v.x, e.x);
          v.y = __fadd_rn(v.y, e.y);
          v.z = __fadd_rn(v.z, e.z);
          v.w = __fadd_rn(v.w, e.w);
          *reinterpret_cast<float4*>(err + i0) = v;
        }
        c[0] = v.x; c[1] = v.y; c[2] = v.z; c[3] = v.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          c[j] = 0.0f;
          if (i0 + j < end) {
            c[j] = x[i0 + j];
            if (IO == IO_EF) {
              c[j] = __fadd_rn(c[j], err[i0 + j]);
              err[i0 + j] = c[j];
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (i0 + j < end) {
          mn = fminf(mn, c[j]);
          mx = fmaxf(mx, c[j]);
          amax = fmaxf(amax, fabsf(c[j]));
        }
      }
      if (MODE == GC_QSGD) {
        float s = __fadd_rn(__fadd_rn(__fmul_rn(c[0], c[0]), __fmul_rn(c[1], c[1])),
                            __fadd_rn(__fmul_rn(c[2], c[2]), __fmul_rn(c[3], c[3])));
        tree.push(warp_sum_tree(s, 32));
      }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
    }
    const float ss = MODE == GC_QSGD ? tree.finish() : 0.0f;
    if (lane == 0) {
      if (cpg == 1)
        finalize_group<MODE>(mn, mx, amax, ss, top, scales, g);
      else
        partials[ch] = make_float4(mn, mx, amax, ss);
    }
  }
}

// One block per group.  min / max / max|c| do not depend on the order, so
// every warp takes a share of the group's chunks; the QSGD sum of squares
// keeps its tree order and runs in warp 0.
template <int MODE>
__global__ void __launch_bounds__(kQThreads) quant_combine_kernel(
    const float4* __restrict__ partials, int64_t cpg, int64_t nchunks,
    int64_t ngroups, uint32_t top, float* __restrict__ scales) {
  constexpr int NW = kQThreads / 32;
  __shared__ float red[3][NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
    const int64_t first = g * cpg;
    const int64_t last = std::min<int64_t>(first + cpg, nchunks);
    float mn = INFINITY, mx = -INFINITY, amax = 0.0f, ss = 0.0f;
    if (MODE == GC_QSGD) {
      if (warp == 0) {
        // eight rows of 32 partials loaded at a time, pushed in order
        TreeAcc tree;
        tree.init();
        for (int64_t b = first; b < last; b += 8 * 32) {
          float sv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int64_t i = b + u * 32 + lane;
            sv[u] = i < last ? partials[i].w : 0.0f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (b + u * 32 < last) tree.push(warp_sum_tree(sv[u], 32));
        }
        ss = tree.finish();
      }
    } else {
      int64_t b = first + threadIdx.x;
      for (; b + 7 * kQThreads < last; b += 8 * kQThreads) {
        float4 p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) p[u] = partials[b + u * kQThreads];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          mn = fminf(mn, p[u].x);
          mx = fmaxf(mx, p[u].y);
          amax = fmaxf(amax, p[u].z);
        }
      }
      for (; b < last; b += kQThreads) {
        const float4 p = partials[b];
        mn = fminf(mn, p.x);
        mx = fmaxf(mx, p.y);
        amax = fmaxf(amax, p.z);
      }
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
      }
      if (lane == 0) {
        red[0][warp] = mn;
        red[1][warp] = mx;
        red[2][warp] = amax;
      }
      __syncthreads();
      if (warp == 0) {
        mn = lane < NW ? red[0][lane] : INFINITY;
        mx = lane < NW ? red[1][lane] : -INFINITY;
        amax = lane < NW ? red[2][lane] : 0.0f;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o2));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) finalize_group<MODE>(mn, mx, amax, ss, top, scales, g);
  }
}

// Group of element i0 + j (0 <= j < 4) from one division per lane: with
// G >= 4 at most one group boundary falls inside the 4 elements.
struct GroupOf4 {
  int64_t g0, r0, G;
  // one group of all n (G >= n) needs no division
  __device__ __forceinline__ GroupOf4(int64_t i0, int64_t G_, int64_t n) : G(G_) {
    g0 = G_ >= n ? 0 : i0 / G_;
    r0 = i0 - g0 * G_;
  }
  __device__ __forceinline__ int64_t operator()(int j) const {
    if (G >= 4) return g0 + ((r0 + j >= G) ? 1 : 0);
    return (g0 * G + r0 + j) / G;
  }
};

// Elementwise quantise + pack (+ residual), group parameters from scales.
template <int MODE, int BITS, int IO>
__global__ void __launch_bounds__(kQThreads) quant_apply_kernel(
    const float* __restrict__ c_src, float* __restrict__ err, int64_t n, int64_t G,
    QuantOut o, int stochastic, uint64_t seed, uint64_t step) {
  constexpr uint32_t top = mode_top<MODE, BITS>();
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = ((int64_t)blockIdx.x * kQThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kQThreads) >> 5;
  zero_padding(o);
  // one group of all n: its parameters once, not per element
  const bool one_group = G >= n;
  float scale1 = 0.0f, offset1 = 0.0f;
  if (one_group) {
    if (MODE == GC_MINMAX) {
      const float2 p = reinterpret_cast<const float2*>(o.scales)[0];
      scale1 = p.x;
      offset1 = p.y;
    } else {
      scale1 = o.scales[0];
    }
  }
  // two chunks per round: their Philox chains interleave
#pragma unroll 2
  for (int64_t base = warp_id * 128; base < n; base += nwarps * 128) {
    const int64_t i0 = base + 4 * lane;
    const bool active = i0 < n;
    float c[4];
    bool valid[4];
    if (i0 + 3 < n) {
      const float4 v = IO == IO_EF ? *reinterpret_cast<const float4*>(c_src + i0)
                                   : __ldcs(reinterpret_cast<const float4*>(c_src + i0));
      c[0] = v.x; c[1] = v.y; c[2] = v.z; c[3] = v.w;
      valid[0] = valid[1] = valid[2] = valid[3] = true;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        valid[j] = i0 + j < n;
        c[j] = valid[j] ? c_src[i0 + j] : 0.0f;
      }
    }
    float u[4] = {0.f, 0.f, 0.f, 0.f};
    if (stochastic) uniform4((uint64_t)i0 >> 2, seed, step, u);
    uint32_t q[4];
    bool neg[4];
    float r[4];
    const GroupOf4 group_of(i0, G, n);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      q[j] = 0u;
      neg[j] = false;
      r[j] = 0.0f;
      if (valid[j]) {
        float scale = scale1, offset = offset1;
        if (!one_group) {
          const int64_t g = group_of(j);
          if (MODE == GC_MINMAX) {
            const float2 p = reinterpret_cast<const float2*>(o.scales)[g];
            scale = p.x;
            offset = p.y;
          } else {
            scale = o.scales[g];
          }
        }
        float gh;
        q[j] = quantize_one<MODE>(c[j], scale, offset, stochastic != 0, u[j], top, &neg[j], &gh);
        r[j] = __fsub_rn(c[j], gh);
      }
    }
    store_codes4<(MODE == GC_TERN) ? 2 : BITS>(o.codes, i0, active, code_bits4<MODE, BITS>(q, neg));
    if (MODE == GC_QSGD) {
      uint32_t sb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) sb[j] = neg[j] ? 1u : 0u;
      store_codes4<1>(o.signs, i0, active, pack4<1>(sb));
    }
    if (IO == IO_EF) {
      if (i0 + 3 < n) {
        *reinterpret_cast<float4*>(err + i0) = make_float4(r[0], r[1], r[2], r[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (valid[j]) err[i0 + j] = r[j];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Dequantisation.
// ---------------------------------------------------------------------------
// acc: 0 writes g_hat; 1 adds it to out (out + g_hat); 2 writes 0 + g_hat
// (the receiving side of differential quantisation, without / with refresh).
template <int MODE, int BITS>
__global__ void __launch_bounds__(kQThreads) dequant_kernel(
    const uint8_t* __restrict__ codes, const uint8_t* __restrict__ signs,
    const float* __restrict__ scales, int64_t n, int64_t G, float* __restrict__ out, int acc) {
  constexpr int CB = (MODE == GC_TERN) ? 2 : BITS;
  const int64_t nvec = (n + 3) >> 2;
  const int64_t stride = (int64_t)gridDim.x * kQThreads;
  for (int64_t v = (int64_t)blockIdx.x * kQThreads + threadIdx.x; v < nvec; v += stride) {
    const int64_t i0 = v << 2;
    uint32_t bits4;
    if (CB == 8) bits4 = *reinterpret_cast<const uint32_t*>(codes + i0);
    else if (CB == 4) bits4 = *reinterpret_cast<const uint16_t*>(codes + (i0 >> 1));
    else if (CB == 2) bits4 = codes[i0 >> 2];
    else bits4 = (uint32_t)(codes[i0 >> 3] >> ((v & 1) * 4)) & 0xfu;
    uint32_t sbits = 0u;
    if (MODE == GC_QSGD) sbits = (uint32_t)(signs[i0 >> 3] >> ((v & 1) * 4)) & 0xfu;
    float r[4];
    const GroupOf4 group_of(i0, G, n);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      r[j] = 0.0f;
      if (i0 + j < n) {
        const uint32_t code = (bits4 >> (j * CB)) & ((1u << CB) - 1u);
        const int64_t g = group_of(j);
        if (MODE == GC_MINMAX) {
          const float2 p = reinterpret_cast<const float2*>(scales)[g];
          r[j] = __fadd_rn(__fmul_rn((float)code, p.x), p.y);
        } else if (MODE == GC_QSGD) {
          const float m = __fmul_rn((float)code, scales[g]);
          r[j] = ((sbits >> j) & 1u) ? -m : m;
        } else if (MODE == GC_LOG) {
          constexpr uint32_t mask = (1u << (BITS - 1)) - 1u;
          const float m =
              __fsub_rn(cw_expf(__fmul_rn((float)(code & mask), scales[g])), 1.0f);
          r[j] = (code >> (BITS - 1)) ? -m : m;
        } else {
          const float m = __fmul_rn((float)(code & 1u), scales[g]);
          r[j] = (code >> 1) ? -m : m;
        }
      }
    }
    if (acc != 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i0 + j < n) r[j] = __fadd_rn(acc == 1 ? out[i0 + j] : 0.0f, r[j]);
    }
    if (i0 + 3 < n) {
      *reinterpret_cast<float4*>(out + i0) = make_float4(r[0], r[1], r[2], r[3]);
    } else {
      for (int j = 0; j < 4; ++j)
        if (i0 + j < n) out[i0 + j] = r[j];
    }
  }
}

// ---------------------------------------------------------------------------
// Host dispatch.
// ---------------------------------------------------------------------------
__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t up64(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// Output pointers and padding ranges of n quantised elements.
__host__ __device__ inline QuantOut make_out(uint8_t* codes, float* scales, int64_t n, int bits,
                                             int mode) {
  QuantOut o;
  const int cb = mode == GC_TERN ? 2 : bits;
  const int64_t mag = up64((n * cb + 7) / 8, 16);
  o.codes = codes;
  o.scales = scales;
  o.signs = mode == GC_QSGD ? codes + mag : nullptr;
  // bytes written by the lanes cover ceil(n/4)*4 elements
  const int64_t n4 = up64(n, 4);
  o.zero_begin = min64((n4 * cb + 7) / 8, mag);
  if (cb == 1) o.zero_begin = min64((n4 + 7) / 8, mag);
  o.zero_end = mag;
  const int64_t smag = up64((n + 7) / 8, 16);
  o.szero_begin = min64((n4 + 7) / 8, smag);
  o.szero_end = smag;
  o.scatter_n = 0;
  o.status = nullptr;
  o.ref = nullptr;
  o.refresh = 0;
  o.patch = nullptr;
  o.patch_tail = 0;
  return o;
}

// QSGD of the kept values of every bucket of a plan: one warp per chunk of
// 128 values of one bucket; bucket b's codes and scales start at the offsets
// the hist pass laid out, its residuals go to err[start_b + idx] or, with
// defer, to the plan's patch list.
template <int BITS, int LPG, bool DIAG>
__global__ void __launch_bounds__(kQThreads) quant_buckets_kernel(
    float* __restrict__ err, const int32_t* __restrict__ idx, BucketWs w,
    uint8_t* __restrict__ codes_out, float* __restrict__ scales_out, int stochastic,
    uint64_t seed, uint64_t step, int defer) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = ((int64_t)blockIdx.x * kQThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kQThreads) >> 5;
  for (int64_t ch = warp_id; ch < w.nchunk; ch += nwarps) {
    const int b = w.chunk_bucket[ch];
    const BucketDesc d = w.desc[b];
    const int64_t lc = ch - d.chunk_first;
    QuantOut o = make_out(codes_out + w.qoff[2 * b], scales_out + w.qoff[2 * b + 1], d.k, BITS,
                          GC_QSGD);
    o.scatter_n = d.n;
    o.status = w.status;
    if (defer) {
      o.patch = w.patch + d.idx_off;
      o.patch_tail = d.n & ~3;  // the ragged end of a bucket is read from err directly
      if (ch == 0 && lane == 0) *w.patch_ready = 1u;  // read by the next call's hist pass
    }
    if (lc == 0 && lane == 0) zero_padding_bytes(o);
    float dsum[2] = {0.0f, 0.0f};
    quant_fused_chunk<GC_QSGD, BITS, LPG, IO_SCATTER, DIAG>(
        w.vals + d.idx_off, err + d.start, idx + d.idx_off, d.k, o, stochastic,
        bucket_seed(seed, b), step, lc * kChunkVals, lane, dsum);
    if (DIAG) {
      const float g2 = warp_allsum(dsum[0]), r2 = warp_allsum(dsum[1]);
      if (lane == 0) {
        w.chunk_g2[ch] = g2;
        w.chunk_r2[ch] = r2;
      }
    }
  }
}

int grid_for(gc_ctx* ctx, int64_t work_items, int per_block, int per_sm) {
  const int64_t want = std::max<int64_t>(1, ceil_div(work_items, per_block));
  return (int)std::min<int64_t>(want, (int64_t)ctx->num_sms * per_sm);
}

template <int MODE, int BITS, int LPG, int IO>
void launch_fused(gc_ctx* ctx, const float* x, float* err, const int32_t* idx, int64_t n,
                  const QuantOut& o, int stoch, uint64_t seed, uint64_t step) {
  auto kernel = quant_fused_kernel<MODE, BITS, LPG, IO>;
  // resident blocks per SM of this instantiation, with shared memory
  // preferred over L1 (the stages bypass L1)
  static const int per_sm = [&] {
    cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaGetLastError();
    return blocks_per_sm(kernel, kQThreads);
  }();
  const int grid = grid_for(ctx, ceil_div(n, 128), kQThreads / 32, per_sm);
  kernel<<<grid, kQThreads, 0, ctx->stream>>>(x, err, idx, n, o, stoch, seed, step);
}

template <int MODE, int BITS, int IO>
gc_status run_fused(gc_ctx* ctx, const float* x, float* err, const int32_t* idx,
                    int64_t n, int64_t G, const QuantOut& o, int stoch, uint64_t seed,
                    uint64_t step) {
  LaunchScope L(ctx, GC_PHASE_QUANT_FUSED);
  switch (G) {
    case 4: launch_fused<MODE, BITS, 1, IO>(ctx, x, err, idx, n, o, stoch, seed, step); break;
    case 8: launch_fused<MODE, BITS, 2, IO>(ctx, x, err, idx, n, o, stoch, seed, step); break;
    case 16: launch_fused<MODE, BITS, 4, IO>(ctx, x, err, idx, n, o, stoch, seed, step); break;
    case 32: launch_fused<MODE, BITS, 8, IO>(ctx, x, err, idx, n, o, stoch, seed, step); break;
    case 64: launch_fused<MODE, BITS, 16, IO>(ctx, x, err, idx, n, o, stoch, seed, step); break;
    default: launch_fused<MODE, BITS, 32, IO>(ctx, x, err, idx, n, o, stoch, seed, step); break;
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

template <int MODE, int BITS, int IO>
gc_status run_multipass(gc_ctx* ctx, const float* x, float* err, int64_t n,
                        int64_t group, const QuantOut& o, int stoch, uint64_t seed,
                        uint64_t step) {
  const QuantPlan p = quant_plan(n, group);
  if (p.chunks_per_group > 1 && p.nchunks > ctx->ws.max_partials) return GC_ERR_WORKSPACE;
  constexpr uint32_t top = mode_top<MODE, BITS>();
  cudaStream_t s = ctx->stream;
  const int warps_per_block = kQThreads / 32;
  {
    LaunchScope L(ctx, GC_PHASE_QUANT_STATS);
    auto kernel = quant_stats_kernel<MODE, IO>;
    static const int per_sm = [&] {
      cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      cudaGetLastError();
      return blocks_per_sm(kernel, kQThreads);
    }();
    kernel<<<grid_for(ctx, p.nchunks, warps_per_block, per_sm), kQThreads, 0, s>>>(
        x, err, n, p.G, p.chunk, p.chunks_per_group, p.nchunks, top, ctx->ws.partials, o.scales);
  }
  if (p.chunks_per_group > 1) {
    LaunchScope L(ctx, GC_PHASE_QUANT_COMBINE);
    quant_combine_kernel<MODE><<<grid_for(ctx, p.ngroups, 1, 8), kQThreads, 0, s>>>(
        ctx->ws.partials, p.chunks_per_group, p.nchunks, p.ngroups, top, o.scales);
  }
  const float* c_src = IO == IO_EF ? err : x;
  {
    LaunchScope L(ctx, GC_PHASE_QUANT_APPLY);
    quant_apply_kernel<MODE, BITS, IO><<<grid_for(ctx, ceil_div(n, 128), warps_per_block, 8), kQThreads, 0, s>>>(
        c_src, err, n, p.G, o, stoch, seed, step);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

template <int MODE, int BITS>
gc_status dispatch_io(gc_ctx* ctx, const float* x, float* err, const int32_t* idx,
                      int64_t n, int64_t group, const QuantOut& o, int stoch,
                      uint64_t seed, uint64_t step) {
  const int64_t G = group == 0 ? n : group;
  if (quant_is_fused(n, group)) {
    if (idx) return run_fused<MODE, BITS, IO_SCATTER>(ctx, x, err, idx, n, G, o, stoch, seed, step);
    if (err) return run_fused<MODE, BITS, IO_EF>(ctx, x, err, idx, n, G, o, stoch, seed, step);
    return run_fused<MODE, BITS, IO_PLAIN>(ctx, x, err, idx, n, G, o, stoch, seed, step);
  }
  if (idx) return GC_ERR_UNSUPPORTED;
  if (n > ctx->ws.max_n) return GC_ERR_WORKSPACE;
  if (err) return run_multipass<MODE, BITS, IO_EF>(ctx, x, err, n, group, o, stoch, seed, step);
  return run_multipass<MODE, BITS, IO_PLAIN>(ctx, x, err, n, group, o, stoch, seed, step);
}

template <int MODE>
gc_status dispatch_bits(gc_ctx* ctx, const float* x, float* err, const int32_t* idx,
                        int64_t n, int bits, int64_t group, const QuantOut& o, int stoch,
                        uint64_t seed, uint64_t step) {
  // bits as validated by the API: TernGrad 2; logarithmic 2, 4, 8
  if constexpr (MODE == GC_TERN) {
    return dispatch_io<GC_TERN, 2>(ctx, x, err, idx, n, group, o, stoch, seed, step);
  } else {
  switch (bits) {
    case 1:
      if (MODE == GC_LOG) return GC_ERR_UNSUPPORTED;
      return dispatch_io<MODE, (MODE == GC_LOG ? 2 : 1)>(ctx, x, err, idx, n, group, o, stoch,
                                                         seed, step);
    case 2: return dispatch_io<MODE, 2>(ctx, x, err, idx, n, group, o, stoch, seed, step);
    case 4: return dispatch_io<MODE, 4>(ctx, x, err, idx, n, group, o, stoch, seed, step);
    default: return dispatch_io<MODE, 8>(ctx, x, err, idx, n, group, o, stoch, seed, step);
  }
  }
}

// Differential quantisation: the fused pass only.
template <int MODE>
gc_status diff_bits(gc_ctx* ctx, const float* grad, float* err, int64_t n, int bits, int64_t G,
                    const QuantOut& o, int stoch, uint64_t seed, uint64_t step) {
  if constexpr (MODE == GC_TERN) {
    return run_fused<GC_TERN, 2, IO_DIFF>(ctx, grad, err, nullptr, n, G, o, stoch, seed, step);
  } else {
  switch (bits) {
    case 1:
      if (MODE == GC_LOG) return GC_ERR_UNSUPPORTED;
      return run_fused<MODE, (MODE == GC_LOG ? 2 : 1), IO_DIFF>(ctx, grad, err, nullptr, n, G,
                                                                o, stoch, seed, step);
    case 2: return run_fused<MODE, 2, IO_DIFF>(ctx, grad, err, nullptr, n, G, o, stoch, seed, step);
    case 4: return run_fused<MODE, 4, IO_DIFF>(ctx, grad, err, nullptr, n, G, o, stoch, seed, step);
    default: return run_fused<MODE, 8, IO_DIFF>(ctx, grad, err, nullptr, n, G, o, stoch, seed, step);
  }
  }
}

// Dequantisation into out (acc 0), added to out (1) or to 0 (2).
gc_status dequant_into(gc_ctx* ctx, const uint8_t* codes, const float* scales, int64_t n,
                       int bits, int64_t group, int mode, float* out, int acc) {
  if (n == 0) return GC_OK;
  const int64_t G = group == 0 ? n : group;
  const int cb = mode == GC_TERN ? 2 : bits;
  const uint8_t* signs = mode == GC_QSGD ? codes + round_up((n * cb + 7) / 8, 16) : nullptr;
  const int grid = grid_for(ctx, ceil_div(n, 4), kQThreads, 8);
  cudaStream_t s = ctx->stream;
  LaunchScope L(ctx, GC_PHASE_DEQUANT);
#define GC_DQ(M, B) \
  dequant_kernel<M, B><<<grid, kQThreads, 0, s>>>(codes, signs, scales, n, G, out, acc)
#define GC_DQ_BITS(M)               \
  switch (bits) {                   \
    case 1: GC_DQ(M, 1); break;     \
    case 2: GC_DQ(M, 2); break;     \
    case 4: GC_DQ(M, 4); break;     \
    default: GC_DQ(M, 8); break;    \
  }
  if (mode == GC_TERN) {
    GC_DQ(GC_TERN, 2);
  } else if (mode == GC_LOG) {
    switch (bits) {
      case 2: GC_DQ(GC_LOG, 2); break;
      case 4: GC_DQ(GC_LOG, 4); break;
      default: GC_DQ(GC_LOG, 8); break;
    }
  } else if (mode == GC_MINMAX) {
    GC_DQ_BITS(GC_MINMAX)
  } else {
    GC_DQ_BITS(GC_QSGD)
  }
#undef GC_DQ_BITS
#undef GC_DQ
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace

gc_status launch_quant(gc_ctx* ctx, const float* x, float* err,
                       const int32_t* scatter_idx, int64_t scatter_n, int64_t n,
                       int bits, int64_t group, int mode, int rounding, uint64_t seed,
                       uint64_t step, uint8_t* codes_out, float* scales_out) {
  QuantOut o = make_out(codes_out, scales_out, n, bits, mode);
  o.scatter_n = scatter_n;
  o.status = ctx->ws.status;
  if (n == 0) return GC_OK;
  const int stoch = rounding == GC_STOCHASTIC;
  if (mode == GC_MINMAX)
    return dispatch_bits<GC_MINMAX>(ctx, x, err, scatter_idx, n, bits, group, o, stoch, seed, step);
  if (mode == GC_QSGD)
    return dispatch_bits<GC_QSGD>(ctx, x, err, scatter_idx, n, bits, group, o, stoch, seed, step);
  if (mode == GC_LOG)
    return dispatch_bits<GC_LOG>(ctx, x, err, scatter_idx, n, bits, group, o, stoch, seed, step);
  return dispatch_bits<GC_TERN>(ctx, x, err, scatter_idx, n, bits, group, o, stoch, seed, step);
}

gc_status launch_dequant(gc_ctx* ctx, const uint8_t* codes, const float* scales,
                         int64_t n, int bits, int64_t group, int mode, float* x_out) {
  return dequant_into(ctx, codes, scales, n, bits, group, mode, x_out, 0);
}

gc_status launch_diff_quant(gc_ctx* ctx, const float* grad, float* err, float* ref, int64_t n,
                            int bits, int64_t group, int mode, int rounding, uint64_t seed,
                            uint64_t step, int refresh, uint8_t* codes_out, float* scales_out) {
  QuantOut o = make_out(codes_out, scales_out, n, bits, mode);
  o.status = ctx->ws.status;
  o.ref = ref;
  o.refresh = refresh ? 1 : 0;
  if (n == 0) return GC_OK;
  const int stoch = rounding == GC_STOCHASTIC;
  const int64_t G = group == 0 ? n : group;
  if (mode == GC_MINMAX) return diff_bits<GC_MINMAX>(ctx, grad, err, n, bits, G, o, stoch, seed, step);
  if (mode == GC_QSGD) return diff_bits<GC_QSGD>(ctx, grad, err, n, bits, G, o, stoch, seed, step);
  if (mode == GC_LOG) return diff_bits<GC_LOG>(ctx, grad, err, n, bits, G, o, stoch, seed, step);
  return diff_bits<GC_TERN>(ctx, grad, err, n, bits, G, o, stoch, seed, step);
}

gc_status launch_diff_dequant(gc_ctx* ctx, const uint8_t* codes, const float* scales,
                              int64_t n, int bits, int64_t group, int mode, int refresh,
                              float* ref) {
  return dequant_into(ctx, codes, scales, n, bits, group, mode, ref, refresh ? 2 : 1);
}

gc_status launch_quant_buckets(gc_ctx* ctx, float* err, const int32_t* idx_out, int bits,
                               int64_t group, int rounding, uint64_t seed, uint64_t step,
                               uint8_t* codes_out, float* scales_out, bool diag,
                               bool defer) {
  const BucketWs& w = ctx->bk;
  if (w.nchunk == 0) return GC_OK;
  const int grid = grid_for(ctx, w.nchunk, kQThreads / 32, 8);
  const int st = rounding == GC_STOCHASTIC;
  const int df = defer ? 1 : 0;
  cudaStream_t s = ctx->stream;
  LaunchScope L(ctx, GC_PHASE_BK_QUANT);
#define GC_BQ(B, LPG)                                                                    \
  do {                                                                                   \
    if (diag)                                                                            \
      quant_buckets_kernel<B, LPG, true><<<grid, kQThreads, 0, s>>>(                     \
          err, idx_out, w, codes_out, scales_out, st, seed, step, df);                   \
    else                                                                                 \
      quant_buckets_kernel<B, LPG, false><<<grid, kQThreads, 0, s>>>(                    \
          err, idx_out, w, codes_out, scales_out, st, seed, step, df);                   \
  } while (0)
#define GC_BQ_G(B)                 \
  switch (group) {                 \
    case 4: GC_BQ(B, 1); break;    \
    case 8: GC_BQ(B, 2); break;    \
    case 16: GC_BQ(B, 4); break;   \
    case 32: GC_BQ(B, 8); break;   \
    case 64: GC_BQ(B, 16); break;  \
    default: GC_BQ(B, 32); break;  \
  }
  switch (bits) {
    case 1: GC_BQ_G(1); break;
    case 2: GC_BQ_G(2); break;
    case 4: GC_BQ_G(4); break;
    default: GC_BQ_G(8); break;
  }
#undef GC_BQ_G
#undef GC_BQ
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace gc
