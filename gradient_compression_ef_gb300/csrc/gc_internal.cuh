// gc_internal.cuh -- shared definitions of the CUDA compressor (sm_103a).
//
// Everything here is internal to libgc.so; the public surface is the C ABI
// in include/gc.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gc.h"

namespace gc {

// ---------------------------------------------------------------------------
// Tunables shared by host and device code.
// ---------------------------------------------------------------------------

// Top-K radix select over the 31-bit magnitude key (IEEE bits of |c|).
constexpr int kHistBits = 12;                    // bits 30..19: 8 exponent + 4 mantissa
constexpr int kHistBins = 1 << kHistBits;
constexpr int kHistShift = 31 - kHistBits;       // 19
constexpr int kMidBits = 11;                     // bits 18..8
constexpr int kMidBins = 1 << kMidBits;
constexpr int kLowBits = 8;                      // bits 7..0
constexpr int kLowBins = 1 << kLowBits;
constexpr int kMaxTiles = 2048;                  // tiles of the ordered compaction
constexpr int kMinTileShift = 12;                // tiles of at least 4096 elements
constexpr int kStashMax = 8192;                  // third-level candidates kept aside

// Device status bits (OR-ed into the context's status word).
constexpr uint32_t kStatusTopkCount = 1u << 0;   // candidate count mismatch
constexpr uint32_t kStatusTopkSelect = 1u << 1;  // threshold search failed
constexpr uint32_t kStatusTopkOverflow = 1u << 2;  // more than k entries kept
constexpr uint32_t kStatusScatterIndex = 1u << 3;  // residual index out of range
constexpr uint32_t kStatusWaitTimeout = 1u << 4;   // a bounded wait on an mbarrier ran out

// Per-context Top-K selection state in device memory.
struct TopkSel {
  uint32_t bin;           // first-level threshold bin B
  uint32_t above;         // elements whose bin is above B
  uint32_t need1;         // k - above: how many of bin B are kept
  uint32_t cand_total;    // elements in bin B
  uint32_t B2;            // second-level digit (bits 18..8)
  uint32_t need2;         // how many of the (B, B2) entries are kept
  uint32_t T;             // exact threshold key
  uint32_t need_T;        // entries with key == T to keep (smallest indices)
  uint32_t ticket_coll;   // last-block ticket of the collection pass
  uint32_t ticket_refine; // last-block ticket of the refinement pass
  uint32_t cand_count;    // fill counter of the candidate buffer
  uint32_t stash_count;   // fill counter of the third-level stash
  uint32_t pad[4];
};

// Device scratch of one context (all pointers into one allocation).  The
// histograms, tile_kept, sel and status must be zero when a call starts;
// every call leaves them zero again.
struct Workspace {
  uint32_t* hist;        // [kHistBins] first level
  uint32_t* mid;         // [kMidBins] candidates' bits 18..8
  uint32_t* low;         // [kLowBins] (B, B2) candidates' bits 7..0
  uint32_t* tile_kept;   // [kMaxTiles] kept candidates per tile
  TopkSel* sel;          // one record
  uint32_t* status;      // device status word
  uint32_t* tile_above;  // [kMaxTiles]
  uint32_t* tile_out;    // [kMaxTiles] exclusive output offsets
  uint32_t* tile_tie;    // [kMaxTiles] exclusive tie offsets
  uint2* cand;           // [max_n] (key, index) candidates
  uint2* stash;          // [kStashMax] third-level candidates
  float* vals;           // [max_n] kept values of the hybrid call
  float4* partials;      // [max_partials] chunk statistics of quantisation
  int64_t max_n;
  int64_t max_partials;
};

// ---------------------------------------------------------------------------
// Bucketed calls: one launch per pass for every bucket of a flat gradient.
// ---------------------------------------------------------------------------
constexpr int kSegShift = 11;                    // segments of 2048 elements, one warp each
constexpr int kSegElems = 1 << kSegShift;
constexpr int kChunkVals = 128;                  // kept values per quantisation warp
constexpr int kBkStash = 2048;                   // third-level entries set aside per bucket
constexpr uint32_t kMarginInit = 1u << 19;       // first guess: one first-level bin below T
constexpr uint32_t kMarginMin = 1u << 12;
constexpr uint32_t kMarginMax = 1u << 23;        // one octave
constexpr int kMaxBuckets = 65536;
constexpr int64_t kMaxBucketElems = INT32_MAX - 65535;  // 32-bit offsets inside a bucket

// One bucket of the plan (device copy written once by gc_ctx_set_buckets).
struct BucketDesc {
  int64_t start;        // first element in the flat gradient
  int64_t idx_off;      // first slot of the bucket's idx / value outputs
  int32_t n, k;
  int32_t seg_first;    // first global segment
  int32_t nseg;
  int32_t chunk_first;  // first 128-value quantisation chunk
  int32_t nchunk;
  int32_t blk_hist;     // blocks of each pass that touch the bucket (last-block tickets)
  int32_t blk_coll;
  int32_t blk_ref;
  int32_t pad;
};

// Per-bucket selection state.  Tickets and the stash counter are zero
// between calls (each pass's last block resets its own).
struct BucketSel {
  uint32_t B, above1, need1, cntB;   // first level
  uint32_t B2, need2;                // second level
  uint32_t T, needT;                 // exact threshold key, ties kept at T
  uint32_t ticket_hist, ticket_coll, ticket_ref;
  uint32_t stash_count;
  // threshold reuse across calls: the hist pass lists the entries with
  // key >= guess1 - 1 (guess1 == 0: no guess); when at least k are listed
  // the lists hold every entry the selection needs
  uint32_t guess1;
  uint32_t list_ok;     // this call's lists are usable
  uint32_t list_total;  // entries listed so far by the hist pass (reset by its last block)
  uint32_t list_len;    // entries listed by this call's hist pass
  uint32_t margin;      // key distance of the next guess below T
  uint32_t pad[3];
};

// Device scratch of a bucket plan (pointers into one allocation).  hist,
// mid, low, sel are zero between calls.
struct BucketWs {
  int nb;
  int64_t total_n;      // elements of the flat gradient
  int64_t nseg;         // segments over all buckets
  int64_t nchunk;       // quantisation chunks over all buckets
  int64_t vals_total;   // slots of the idx / value outputs (sum of k rounded up to 4)
  int g_hist, g_coll, g_ref, g_write;  // grid sizes the tickets were counted for
  int g_write_diag;     // grid of the write pass with diagnostics
  BucketDesc* desc;     // [nb]
  BucketSel* sel;       // [nb]
  int32_t* seg_bucket;  // [nseg]
  int32_t* chunk_bucket;  // [nchunk]
  uint32_t* hist;       // [nb][kHistBins]
  uint32_t* mid;        // [nb][kMidBins]
  uint32_t* low;        // [nb][kLowBins]
  uint32_t* seg_cnt;    // [nseg] list entries of the segment
  uint32_t* seg_above;  // [nseg] entries above the first-level bin
  uint32_t* seg_kept;   // [nseg] entries above the threshold key T
  uint32_t* seg_tie;    // [nseg] entries equal to T
  uint32_t* seg_out;    // [nseg] first output slot (bucket-relative)
  uint32_t* seg_tieb;   // [nseg] ties at T in earlier segments of the bucket
  uint2* list;          // [nseg * kSegElems] (bits of c, bucket index), per segment
  uint2* stash;         // [nb][kBkStash] (key, segment)
  int64_t* qoff;        // [nb][2] codes byte / scales float offset of each bucket
  float* vals;          // [vals_total] kept values of the hybrid call
  uint2* patch;         // [vals_total] (position, bits of e') of the kept entries whose
                        // residual write-back is deferred to the next call
  uint32_t* patch_ready;   // 1 while the patch list holds residuals not yet in e
  uint32_t* flush_ticket;  // last-block ticket of the flush pass
  // per-segment / per-chunk partial sums of the diagnostics
  float* seg_c2;        // [nseg] sum of c^2
  float* seg_drop;      // [nseg] sum of c^2 over the entries not kept
  float* seg_keep;      // [nseg] sum of c^2 over the kept entries
  float* chunk_g2;      // [nchunk] sum of g_hat^2 of a chunk of kept values
  float* chunk_r2;      // [nchunk] sum of e'^2 of a chunk of kept values
  uint32_t* status;     // the context's device status word
};

// Segment range [lo, hi) of block i out of G over S segments.
__host__ __device__ __forceinline__ void seg_range(int64_t S, int G, int i, int64_t* lo,
                                                   int64_t* hi) {
  *lo = S * i / G;
  *hi = S * (i + 1) / G;
}

struct PsgdWorkspace {
  float* q_part;         // [splits][max_n][max_r] partial sums of M^T P
  uint32_t* tickets;     // [strips] last-block tickets
  int64_t max_m, max_n;
  int max_r;
  int64_t bytes;
};

}  // namespace gc

struct gc_ctx {
  int device;
  int num_sms;
  cudaStream_t stream;
  void* ws_base;
  gc::Workspace ws;
  void* psgd_base;
  gc::PsgdWorkspace psgd;
  // per-kernel timing (gc_ctx_enable_timing)
  int timing_cap;           // event pairs available, 0 = off
  int timing_used;          // pairs recorded in the current window
  cudaEvent_t* ev_start;
  cudaEvent_t* ev_stop;
  int* ev_phase;
  int64_t launches;         // kernels launched by this context
  // bucket plan (gc_ctx_set_buckets)
  void* bk_base;
  gc::BucketWs bk;
  int bk_defer;             // deferred residual write-back of the bucketed hybrid
  float* bk_pending;        // error buffer whose kept-entry residuals are pending
};

namespace gc {

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t mag_key(float x) {
  return __float_as_uint(x) & 0x7fffffffu;
}

// Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies whose
// halves are mixed with the other two words and the round key; the key is
// advanced by the golden-ratio and sqrt(3)-1 Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint2 key) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * x.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, x.x);
    const uint32_t lo1 = 0xCD9E8D57u * x.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, x.z);
    x = make_uint4(hi1 ^ x.y ^ key.x, lo1, hi0 ^ x.w ^ key.y, lo0);
    key.x += 0x9E3779B9u;
    key.y += 0xBB67AE85u;
  }
  return x;
}

// The four draws of elements 4b .. 4b+3 of a call: word j of Philox at
// counter (b, step) and key seed, top 24 bits scaled by 2^-24.
__device__ __forceinline__ void uniform4(uint64_t block, uint64_t seed,
                                         uint64_t step, float u[4]) {
  const uint4 r = philox4x32_10(
      make_uint4((uint32_t)block, (uint32_t)(block >> 32), (uint32_t)step,
                 (uint32_t)(step >> 32)),
      make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  u[0] = __fmul_rn(__uint2float_rn(r.x >> 8), 0x1p-24f);
  u[1] = __fmul_rn(__uint2float_rn(r.y >> 8), 0x1p-24f);
  u[2] = __fmul_rn(__uint2float_rn(r.z >> 8), 0x1p-24f);
  u[3] = __fmul_rn(__uint2float_rn(r.w >> 8), 0x1p-24f);
}

// Philox key of bucket b of a bucketed call: the call's seed with b times
// the 64-bit golden-ratio constant xor-ed in.  Bucket 0 keeps the seed, and a
// caller that changes the seed by small steps between calls never makes one
// bucket reuse another bucket's draws (seed + b would: bucket b + 1 under
// seed s would draw what bucket b draws under seed s + 1).
__host__ __device__ __forceinline__ uint64_t bucket_seed(uint64_t seed, int b) {
  return seed ^ ((uint64_t)b * 0x9E3779B97F4A7C15ull);
}

// Natural logarithm and exponential of the logarithmic quantiser, by the
// Cody-Waite method (W. J. Cody, W. Waite, "Software Manual for the
// Elementary Functions", 1980, ALOG and EXP), every step one rounded
// binary32 operation so that any IEEE-754 evaluation of the same steps gives
// the same bits.  ln 2 = kLn2Hi + kLn2Lo with kLn2Hi = 45426 * 2^-16 (16
// significant bits: k * kLn2Hi is exact for |k| < 256) and kLn2Lo the rest
// rounded to binary32; the series coefficients are 1/(2j+1) and 1/j!
// rounded to binary32.
constexpr float kLn2Hi = 0x1.62e4p-1f;
constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
constexpr float kInvLn2 = 0x1.715476p+0f;
constexpr float kSqrt2 = 0x1.6a09e6p+0f;

// log x for finite x >= 1: x = 2^k m with m in [sqrt(2)/2, sqrt(2)],
// s = (m - 1) / (m + 1), log m = 2 atanh s = 2s (1 + z/3 + ... + z^5/11),
// z = s^2; log x = k kLn2Hi + (k kLn2Lo + log m).
__device__ __forceinline__ float cw_logf(float x) {
  uint32_t u = __float_as_uint(x);
  int k = (int)(u >> 23) - 127;
  float m = __uint_as_float((u & 0x007fffffu) | 0x3f800000u);
  if (m > kSqrt2) {
    m = __fmul_rn(m, 0.5f);
    k += 1;
  }
  const float f = __fsub_rn(m, 1.0f);
  const float s = __fdiv_rn(f, __fadd_rn(f, 2.0f));
  const float z = __fmul_rn(s, s);
  float r = 0x1.745d18p-4f;                    // 1/11
  r = __fadd_rn(0x1.c71c72p-4f, __fmul_rn(z, r));  // 1/9
  r = __fadd_rn(0x1.24924ap-3f, __fmul_rn(z, r));  // 1/7
  r = __fadd_rn(0x1.99999ap-3f, __fmul_rn(z, r));  // 1/5
  r = __fadd_rn(0x1.555556p-2f, __fmul_rn(z, r));  // 1/3
  r = __fmul_rn(z, r);
  const float w = __fadd_rn(s, s);
  const float logm = __fadd_rn(w, __fmul_rn(w, r));
  const float kf = (float)k;
  return __fadd_rn(__fmul_rn(kf, kLn2Hi), __fadd_rn(__fmul_rn(kf, kLn2Lo), logm));
}

// exp y for 0 <= y < 89: k = rint(y / ln 2), r = (y - k kLn2Hi) - k kLn2Lo,
// exp r by the Taylor polynomial to r^8/8! (Horner), times 2^k exactly;
// k >= 128 overflows to +inf.
__device__ __forceinline__ float cw_expf(float y) {
  const float kf = rintf(__fmul_rn(y, kInvLn2));
  const float r = __fsub_rn(__fsub_rn(y, __fmul_rn(kf, kLn2Hi)), __fmul_rn(kf, kLn2Lo));
  float p = 0x1.a01a02p-16f;                       // 1/8!
  p = __fadd_rn(0x1.a01a02p-13f, __fmul_rn(r, p));  // 1/7!
  p = __fadd_rn(0x1.6c16c2p-10f, __fmul_rn(r, p));  // 1/6!
  p = __fadd_rn(0x1.111112p-7f, __fmul_rn(r, p));   // 1/5!
  p = __fadd_rn(0x1.555556p-5f, __fmul_rn(r, p));   // 1/4!
  p = __fadd_rn(0x1.555556p-3f, __fmul_rn(r, p));   // 1/3!
  p = __fadd_rn(0.5f, __fmul_rn(r, p));             // 1/2!
  p = __fadd_rn(1.0f, __fmul_rn(r, p));
  p = __fadd_rn(1.0f, __fmul_rn(r, p));
  const int k = (int)kf;
  if (k >= 128) return __int_as_float(0x7f800000);
  return __fmul_rn(p, __uint_as_float((uint32_t)(k + 127) << 23));
}

// Top level of a mode's code: TernGrad 1, logarithmic 2^(b-1) - 1 (one bit
// is the sign), otherwise 2^b - 1.
template <int MODE, int BITS>
__host__ __device__ constexpr uint32_t mode_top() {
  return MODE == GC_TERN ? 1u : MODE == GC_LOG ? ((1u << (BITS - 1)) - 1u) : ((1u << BITS) - 1u);
}

// Level of one element: t >= 0 is its position on the level grid.
// Nearest-even: rint(t).  Stochastic: floor(t) + [u < t - floor(t)].
// Clamped to [0, top].
// The conversions saturate and take NaN to 0, so a NaN t gives level 0 and
// a t beyond the grid gives top.
__device__ __forceinline__ uint32_t round_level(float t, bool stochastic,
                                                float u, uint32_t top) {
  int q;
  if (stochastic) {
    const float fl = floorf(t);
    q = __float2int_rz(fl) + ((u < __fsub_rn(t, fl)) ? 1 : 0);
  } else {
    q = __float2int_rn(t);  // half to even
  }
  return (uint32_t)min(max(q, 0), (int)top);
}


// Quantise one value c against its group parameters; returns the code
// level, the sign flag (QSGD/TernGrad, only when q != 0) and g_hat.
template <int MODE>
__device__ __forceinline__ uint32_t quantize_one(float c, float scale,
                                                 float offset, bool stochastic,
                                                 float u, uint32_t top,
                                                 bool* negative, float* ghat) {
  uint32_t q = 0u;
  if (scale != 0.0f) {
    const float t = (MODE == GC_MINMAX) ? __fdiv_rn(__fsub_rn(c, offset), scale)
                    : (MODE == GC_LOG)  ? __fdiv_rn(cw_logf(__fadd_rn(fabsf(c), 1.0f)), scale)
                                        : __fdiv_rn(fabsf(c), scale);
    if (MODE == GC_TERN) {
      // scale = max |c| of the group, so t is in [0, 1] (or NaN): the level
      // round_level gives is [u < t] stochastically (floor(t) is 0, and
      // u < 1 for t = 1) and [t > 1/2] to nearest (rint(1/2) = 0); NaN
      // compares false, level 0, as there
      q = stochastic ? (u < t ? 1u : 0u) : (t > 0.5f ? 1u : 0u);
    } else {
      q = round_level(t, stochastic, u, top);
    }
  }
  float mag = __fmul_rn((float)q, scale);
  if (MODE == GC_LOG) mag = __fsub_rn(cw_expf(mag), 1.0f);
  if (MODE == GC_MINMAX) {
    *negative = false;
    *ghat = __fadd_rn(mag, offset);
  } else {
    *negative = (q != 0u) && (c < 0.0f);
    *ghat = *negative ? -mag : mag;
  }
  return q;
}

// Pack four b-bit codes of consecutive elements into the low 4b bits.
template <int BITS>
__device__ __forceinline__ uint32_t pack4(const uint32_t q[4]) {
  return q[0] | (q[1] << BITS) | (q[2] << (2 * BITS)) | (q[3] << (3 * BITS));
}

// Stores the packed codes of elements i0..i0+3 (i0 % 4 == 0).  Every lane of
// the warp must call it (1-bit codes pair neighbouring lanes).
template <int BITS>
__device__ __forceinline__ void store_codes4(uint8_t* codes, int64_t i0,
                                             bool lane_active, uint32_t bits4) {
  if (BITS == 8) {
    if (lane_active) *reinterpret_cast<uint32_t*>(codes + i0) = bits4;
  } else if (BITS == 4) {
    if (lane_active) *reinterpret_cast<uint16_t*>(codes + (i0 >> 1)) = (uint16_t)bits4;
  } else if (BITS == 2) {
    if (lane_active) codes[i0 >> 2] = (uint8_t)bits4;
  } else {  // BITS == 1: two lanes form one byte
    const uint32_t hi = __shfl_down_sync(0xffffffffu, bits4, 1);
    if (lane_active && ((i0 >> 2) & 1) == 0)
      codes[i0 >> 3] = (uint8_t)(bits4 | (hi << 4));
  }
}

// Asynchronous 16-byte global -> shared copies (cp.async.cg: cached in L2
// only), grouped per commit and completed with cp.async.wait_group, which
// makes a thread's own copies visible to that thread.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Sums each of v[0 .. N-1] (N a power of two <= 32) over the 32 lanes by a
// transposed butterfly: at the exchange across lane bit 4, 3, ... a lane
// keeps the half of its values picked by that bit and receives the
// partner's copy of the same half, so N values take N + 5 - log2(N)
// shuffles instead of 5 N.  Value j ends on the lanes l with
// l >> (5 - log2 N) == j and is returned there.  Fixed order of additions.
template <int N>
__device__ __forceinline__ float warp_sum_many(float (&v)[N], int lane) {
  int off = 16;
#pragma unroll
  for (int half = N / 2; half >= 1; half >>= 1, off >>= 1) {
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = hi ? v[i + half] : v[i];
      const float send = hi ? v[i] : v[i + half];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  float t = v[0];
#pragma unroll
  for (; off >= 1; off >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, off));
  return t;
}

// Sum over the 32 lanes by the butterfly (the same value on every lane, the
// same order of additions on every call).
__device__ __forceinline__ float warp_allsum(float s) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  return s;
}

__device__ __forceinline__ float warp_sum_tree(float s, int lanes) {
  // Butterfly over `lanes` consecutive lanes: with offsets 1, 2, 4 ... the
  // value after offset o is the sum of an aligned block of 2o lanes, formed
  // from its two aligned halves -- the adjacent-pair binary tree.
  for (int o = 1; o < lanes; o <<= 1)
    s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  return s;
}

// Brackets one kernel launch: counts it and, when timing is on, records a
// start / stop event pair on the context's stream around it.
struct LaunchScope {
  gc_ctx* ctx;
  int slot;
  LaunchScope(gc_ctx* c, int phase) : ctx(c), slot(-1) {
    ++ctx->launches;
    if (ctx->timing_cap > 0 && ctx->timing_used < ctx->timing_cap) {
      slot = ctx->timing_used++;
      ctx->ev_phase[slot] = phase;
      cudaEventRecord(ctx->ev_start[slot], ctx->stream);
    }
  }
  ~LaunchScope() {
    if (slot >= 0) cudaEventRecord(ctx->ev_stop[slot], ctx->stream);
  }
};

// Host helpers.
inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Resident blocks per SM of a kernel at `threads` threads (at least 1).
template <class K>
int blocks_per_sm(K kernel, int threads, size_t smem = 0) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n > 1 ? n : 1;
}

// Launchers implemented in the .cu files (return GC_OK or GC_ERR_CUDA).
gc_status launch_ef_topk(gc_ctx* ctx, const float* grad, float* err, int64_t n,
                         int64_t k, int32_t* idx_out, float* val_out);
// The same Top-K passes on an explicit workspace and stream (no context);
// the workspace's hist, sel and status must be zero on entry.
gc_status launch_ef_topk_on(const Workspace& ws, cudaStream_t s, int sms, const float* grad,
                            float* err, int64_t n, int64_t k, int32_t* idx_out,
                            float* val_out);
// scatter_idx != NULL: x holds kept values and the residual of element j
// goes to err[scatter_idx[j]] (err has scatter_n elements).
gc_status launch_quant(gc_ctx* ctx, const float* x, float* err,
                       const int32_t* scatter_idx, int64_t scatter_n, int64_t n,
                       int bits, int64_t group, int mode, int rounding, uint64_t seed,
                       uint64_t step, uint8_t* codes_out, float* scales_out);
gc_status launch_dequant(gc_ctx* ctx, const uint8_t* codes,
                         const float* scales, int64_t n, int bits,
                         int64_t group, int mode, float* x_out);
gc_status launch_powersgd(gc_ctx* ctx, const float* grad, float* err,
                          int64_t m, int64_t n, int r, float* P_out,
                          float* Q_inout);

// Bucketed Top-K over every bucket of the context's plan; vals != NULL
// receives the kept values at the bucket's idx_off (val_out otherwise);
// zero_err writes e' = +0 at the kept positions.  qbits > 0 also lays out
// the QSGD outputs of (qbits, qgroup) for launch_quant_buckets.
// diag also leaves the per-segment diagnostic partial sums.
// patch applies the residuals a previous deferred call left in the plan's
// patch list to e as it is read (when the plan's ready flag says there are
// any); defer_zero (with zero_err) puts the kept entries' e' = +0 into the
// patch list instead of storing it.
gc_status launch_ef_topk_buckets(gc_ctx* ctx, const float* grad, float* err, int32_t* idx_out,
                                 float* val_out, bool zero_err, int qbits, int64_t qgroup,
                                 bool diag, bool patch = false, bool defer_zero = false);
// Writes the pending residuals of the patch list into err (the kept
// positions of the last deferred bucketed call).
gc_status launch_bucket_flush(gc_ctx* ctx, float* err);
// QSGD of every bucket's kept values (from launch_ef_topk_buckets) with the
// residual scattered to err; bucket b uses bucket_seed(seed, b).  diag also leaves the
// per-chunk diagnostic partial sums.  defer keeps the residuals in the
// plan's patch list instead (only the ragged tail of a bucket, which the
// next read takes directly from err, is also written to err).
gc_status launch_quant_buckets(gc_ctx* ctx, float* err, const int32_t* idx_out, int bits,
                               int64_t group, int rounding, uint64_t seed, uint64_t step,
                               uint8_t* codes_out, float* scales_out, bool diag,
                               bool defer = false);
// Per-bucket diagnostics {sum c^2, sum g_hat^2, sum e'^2} into out[nb][3]
// from the partial sums of the last bucketed call (quant: the hybrid's).
gc_status launch_bucket_diag(gc_ctx* ctx, bool quant, double* out);
// EF + differential quantisation (group 4..128, a power of two) against the
// history ref; refresh treats ref as 0.
gc_status launch_diff_quant(gc_ctx* ctx, const float* grad, float* err, float* ref, int64_t n,
                            int bits, int64_t group, int mode, int rounding, uint64_t seed,
                            uint64_t step, int refresh, uint8_t* codes_out, float* scales_out);
// ref = (refresh ? 0 : ref) + dequant(codes, scales).
gc_status launch_diff_dequant(gc_ctx* ctx, const uint8_t* codes, const float* scales,
                              int64_t n, int bits, int64_t group, int mode, int refresh,
                              float* ref);
// EF + random sparsification over n <= max_n elements (list scratch in the
// context); writes at most `capacity` entries and the kept count.
gc_status launch_ef_randk(gc_ctx* ctx, const float* grad, float* err, int64_t n, float p,
                          uint64_t seed, uint64_t step, int32_t* idx_out, float* val_out,
                          int64_t capacity, int64_t* count_out);

// Sum of W ranks' sparse vectors into out[n] in rank order; bits == 0: fp32
// values val[W*k], else QSGD codes / scales laid out per rank (see gc.h).
gc_status launch_aggregate(gc_ctx* ctx, int W, int64_t k, const int32_t* idx, const float* val,
                           const uint8_t* codes, const float* scales, int bits, int64_t group,
                           int64_t n, float* out);
// int32 scratch the aggregation needs for W ranks over n elements, and the
// largest W.
int64_t aggregate_scratch_ints(int W, int64_t n);
int aggregate_max_ranks();
// Opts the aggregation kernels into their shared memory (once per device).
gc_status prepare_aggregate_kernels();

// Builds the device plan of nb buckets (synchronous; frees the previous).
gc_status plan_buckets(gc_ctx* ctx, int nb, const int64_t* bucket_n, const int64_t* bucket_k);
void free_buckets(gc_ctx* ctx);

// Bytes of PowerSGD scratch for matrices up to max_m x max_n, rank max_r.
int64_t psgd_workspace_bytes(int64_t max_m, int64_t max_n, int max_r, int num_sms);

// Whether (group, n) runs in the fused single-pass quantisation kernel.
inline bool quant_is_fused(int64_t n, int64_t group) {
  const int64_t G = group == 0 ? n : group;
  return G >= 4 && G <= 128 && (G & (G - 1)) == 0;
}

// Chunking of the multi-pass quantisation (groups the fused kernel does
// not take): a group is cut into chunks of `chunk` elements (a power of two
// >= 1024 when the group is larger than that, else the whole group).
struct QuantPlan {
  int64_t G, ngroups, chunk, chunks_per_group, nchunks;
};
QuantPlan quant_plan(int64_t n, int64_t group);

}  // namespace gc
