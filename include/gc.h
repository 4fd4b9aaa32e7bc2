/*
 * gc.h -- C ABI of the GB300 gradient compressor with error feedback.
 *
 * The compressor runs on a flat fp32 gradient before the gradient leaves GPU
 * memory ("gradient-compression-quantization-sparsification" (hotdry blog),
 * 3.2: compression finishes before the data leaves GPU memory and needs
 * custom CUDA kernels).  It adds the error-feedback residual, selects the
 * Top-K entries, quantises with per-group scales, packs the codes,
 * dequantises and writes the new residual; PowerSGD is the low-rank variant.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Buffers are DEVICE pointers owned by the caller (plain C types, no
 *    framework types).  Every buffer must start on a 16-byte boundary
 *    (GC_ERR_ALIGNMENT otherwise); a pointer may be NULL only when the call
 *    touches no element of it (n == 0, k == 0).
 *  - Calls are asynchronous: they validate arguments on the host, enqueue
 *    kernels on the context's CUDA stream and return.  The return value
 *    reports host-side validation and launch errors only (a launch error is
 *    GC_ERR_CUDA).  Device-side self checks set a status word in the
 *    context; gc_ctx_check() synchronises the stream and reports it.
 *  - No call allocates memory.  Scratch space lives in the context and is
 *    reserved by gc_ctx_create / gc_ctx_reserve_powersgd.  Consecutive calls
 *    on one context are ordered by its stream; calls that overlap in time
 *    need one context each.
 *  - n <= 2^31 - 1 (indices are int32) and, for calls that use the context's
 *    scratch (Top-K, hybrid, quantisation with groups that do not fit the
 *    single-pass kernel), n <= the context's max_n (GC_ERR_WORKSPACE).
 *  - Finite inputs are a precondition.  Squares and ranges must not
 *    overflow binary32 (|x| < 1.8e19 for QSGD).
 *  - Arithmetic is IEEE-754 binary32 with one round-to-nearest-even per
 *    operation and no fused multiply-add, so results are bit-identical to a
 *    plain sequential evaluation of the same formulas; PowerSGD is the
 *    exception (fp32 accumulation in an unspecified order).
 *  - err is read and written in place; no other output may alias an input.
 *
 * Compressed formats
 * ------------------
 *  codes: the b-bit codes of elements 0..n-1 as one little-endian bit stream
 *         (element i occupies bits i*b .. i*b+b-1, bit 0 being the least
 *         significant bit of byte 0), zero-padded to a multiple of 16 bytes;
 *         for GC_QSGD a sign plane (1 bit per element, set when the element
 *         is negative and its code is not 0) follows, laid out the same way.
 *         GC_TERN codes are 2 bits, (sign << 1) | q with q in {0, 1};
 *         GC_LOG codes are b-bit sign-magnitude, (sign << (b-1)) | q.
 *         gc_codes_bytes() gives the size.
 *  scales: per group of `group` consecutive elements (group == 0: one group
 *         of all n; the last group may be partial): GC_MINMAX stores
 *         {scale, min} (two floats), GC_QSGD, GC_TERN and GC_LOG store
 *         {scale}.
 *         gc_scales_floats() gives the size in floats.
 */
#ifndef GC_H_
#define GC_H_

#include <stdint.h>

#if defined(__GNUC__)
#define GC_API __attribute__((visibility("default")))
#else
#define GC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gc_status {
  GC_OK = 0,
  GC_ERR_INVALID_ARG = -1,  /* NULL, negative size, k > n, group < 0 ... */
  GC_ERR_UNSUPPORTED = -2,  /* bits not in {1,2,4,8}; TERN with bits != 2;
                               LOG with bits == 1 */
  GC_ERR_ALIGNMENT = -3,    /* a buffer is not 16-byte aligned */
  GC_ERR_WORKSPACE = -4,    /* n above the reserved scratch: the context's
                               capacity, or GC_NOALLOC_MAX_N for
                               gc_ef_topk_noalloc */
  GC_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
  GC_ERR_DEVICE_CHECK = -6, /* a device-side self check failed */
  GC_ERR_NO_MEMORY = -7     /* gc_ctx_create could not reserve scratch */
} gc_status;

typedef enum gc_mode {
  GC_MINMAX = 0, /* linear min-max quantisation */
  GC_QSGD = 1,   /* s = 2^b - 1 levels of the group L2 norm, sign plane */
  GC_TERN = 2,   /* TernGrad: levels {-max|c|, 0, +max|c|} */
  GC_LOG = 3     /* logarithmic: levels exp(q * scale) - 1, sign bit */
} gc_mode;

typedef enum gc_rounding {
  GC_NEAREST_EVEN = 0, /* round half to even */
  GC_STOCHASTIC = 1    /* unbiased, Philox-4x32-10 keyed by (seed, step, i) */
} gc_rounding;

typedef struct gc_ctx gc_ctx;

/* Library version (major * 10000 + minor * 100 + patch). */
GC_API int gc_version(void);

/* Human-readable text for a gc_status value; never NULL. */
GC_API const char* gc_status_string(int status);

/*
 * Creates a context bound to `cuda_stream` (a cudaStream_t; NULL selects the
 * legacy default stream) on the current CUDA device and reserves its scratch
 * for calls of up to `max_n` elements (about 12 bytes per element plus a
 * few tens of KB).  The context owns the scratch; the caller owns every
 * buffer passed to the compute calls.  Returns GC_ERR_NO_MEMORY when the
 * device allocation fails, GC_ERR_CUDA on other CUDA errors.
 */
GC_API gc_status gc_ctx_create(gc_ctx** ctx, void* cuda_stream, int64_t max_n);

/* Waits for the context's stream, then frees its scratch.  NULL is a no-op. */
GC_API gc_status gc_ctx_destroy(gc_ctx* ctx);

/* Rebinds the context to another stream of the same device. */
GC_API gc_status gc_ctx_set_stream(gc_ctx* ctx, void* cuda_stream);

/*
 * Reserves the PowerSGD scratch for matrices up to max_m x max_n and rank
 * up to max_r (1..16); a later call with larger limits grows it.  Must not
 * be called while work is in flight on the context.
 */
GC_API gc_status gc_ctx_reserve_powersgd(gc_ctx* ctx, int64_t max_m, int64_t max_n,
                                  int max_r);

/*
 * Synchronises the context's stream and reports the device status word:
 * GC_OK, or GC_ERR_DEVICE_CHECK when a kernel's self check failed (the word
 * is then cleared), or GC_ERR_CUDA for an asynchronous CUDA error.
 */
GC_API gc_status gc_ctx_check(gc_ctx* ctx);

/*
 * Kernel phases, for per-kernel timing.  Every kernel the library launches
 * belongs to one phase.
 */
typedef enum gc_phase {
  GC_PHASE_EF_HIST = 0,      /* Top-K pass 1: c = g + e, 12-bit histogram */
  GC_PHASE_COLLECT = 1,      /* Top-K pass 2: threshold bin, candidates */
  GC_PHASE_WRITE = 2,        /* Top-K pass 4: ordered compaction, e' = 0 */
  GC_PHASE_EF_ADD = 3,       /* e = g + e (k == 0) */
  GC_PHASE_QUANT_FUSED = 4,  /* single-pass group quantisation */
  GC_PHASE_QUANT_STATS = 5,  /* multi-pass: chunk statistics */
  GC_PHASE_QUANT_COMBINE = 6,/* multi-pass: group statistics */
  GC_PHASE_QUANT_APPLY = 7,  /* multi-pass: quantise + pack + residual */
  GC_PHASE_DEQUANT = 8,
  GC_PHASE_PSGD_MQ = 9,      /* PowerSGD pass 1: M = G + E, P = M Q */
  GC_PHASE_PSGD_MTP = 10,    /* PowerSGD pass 2: Q' = M^T P_hat */
  GC_PHASE_PSGD_RESID = 11,  /* PowerSGD pass 3: E' = M - P_hat Q'^T */
  GC_PHASE_REFINE = 12,      /* Top-K pass 3: exact threshold, tile offsets */
  GC_PHASE_BK_HIST = 13,     /* bucketed: c = g + e, first-level histograms */
  GC_PHASE_BK_COLLECT = 14,  /* bucketed: per-segment lists of entries >= B */
  GC_PHASE_BK_REFINE = 15,   /* bucketed: exact thresholds, segment offsets */
  GC_PHASE_BK_WRITE = 16,    /* bucketed: ordered compaction */
  GC_PHASE_BK_QUANT = 17,    /* bucketed: QSGD of the kept values */
  GC_PHASE_AGG_BOUNDS = 18,  /* aggregation: each rank's entries per output range */
  GC_PHASE_AGG_ACCUMULATE = 19, /* aggregation: rank-ordered sum into the dense output */
  GC_PHASE_RANDK_MARK = 20,  /* random sparsification: draws, residual, kept lists */
  GC_PHASE_RANDK_WRITE = 21, /* random sparsification: ordered output */
  GC_PHASE_BK_DIAG = 22,     /* bucketed: per-bucket diagnostics */
  GC_PHASE_BK_FLUSH = 23,    /* bucketed: pending kept-entry residuals into e */
  GC_PHASE_PSGD_THIN = 24,   /* PowerSGD: Q images, the final reduction of Q' */
  GC_PHASE_COUNT = 25
} gc_phase;

/* Name of a phase ("ef_hist", ...); "?" when out of range. */
GC_API const char* gc_phase_name(int phase);

/*
 * Per-kernel timing.  With max_launches > 0 every later kernel launch on the
 * context is bracketed by two CUDA events recorded on the context's stream
 * (up to max_launches launches between reads; further launches are not
 * timed).  max_launches == 0 turns timing off.  The events are created here
 * (not per call).
 */
GC_API gc_status gc_ctx_enable_timing(gc_ctx* ctx, int max_launches);

/*
 * Synchronises the stream, adds each timed launch's duration (ms) and count
 * to ms_out[phase] and count_out[phase] (arrays of GC_PHASE_COUNT entries,
 * caller-initialised), and starts a new timing window.
 */
GC_API gc_status gc_ctx_read_timing(gc_ctx* ctx, double* ms_out, int64_t* count_out);

/* Number of kernels this context has launched since it was created. */
GC_API int64_t gc_ctx_launch_count(gc_ctx* ctx);

/* Bytes of the packed code buffer for n elements (see "Compressed
 * formats"); -1 for invalid arguments. */
GC_API int64_t gc_codes_bytes(int64_t n, int bits, int mode);

/* Floats of the scale buffer for n elements; -1 for invalid arguments. */
GC_API int64_t gc_scales_floats(int64_t n, int64_t group, int mode);

/*
 * Error feedback + Top-K sparsification.
 * Pages: "分布式训练中的梯度压缩算法" 二.2 (Top-K keeps the K entries of
 * largest |g|); "4、梯度累积与梯度压缩" 4.2.1 (exactly k entries, returned as
 * (indices, values)); "梯度聚合通信优化实战方案" Python 演示
 * error_feedback_compress (c = g + e; the entries not sent stay in the
 * residual).
 *   c = grad + err;  keep the k entries of largest |c|, ties broken by the
 *   smaller index;  idx_out[0..k) = kept positions in ascending order;
 *   val_out[j] = c[idx_out[j]];  err[i] = +0 at kept positions, c[i]
 *   elsewhere.
 * err == NULL selects from grad alone and writes no residual.
 * grad: fp32[n] (read);  err: fp32[n] (read, then overwritten);
 * idx_out: int32[k];  val_out: fp32[k].  0 <= k <= n <= max_n.
 */
GC_API gc_status gc_ef_topk(gc_ctx* ctx, const float* grad, float* err, int64_t n,
                     int64_t k, int32_t* idx_out, float* val_out);

/*
 * Group-wise quantisation of x (no error feedback).
 * Pages: "分布式训练中的梯度压缩算法" 二.1 线性量化 (q = round((g - min) /
 * scale), scale = (max - min) / (2^b - 1)); "gradient-compression-
 * quantization-sparsification" 1.1 (QSGD stochastic rounding, TernGrad
 * {-1, 0, +1} with layer-wise scaling) and 1.2 (groups of e.g. 64;
 * deterministic vs stochastic rounding).
 *   GC_MINMAX: scale = (max - min) / (2^b - 1); t = (x - min) / scale.
 *   GC_QSGD:   scale = ||x_group||_2 / (2^b - 1); t = |x| / scale; the sum of
 *              squares is added as the perfect binary tree over the group
 *              (zero-padded to a power of two, adjacent pairs first).
 *   GC_TERN:   scale = max |x_group|; t = |x| / scale; bits must be 2.
 *   GC_LOG:    ("分布式训练中的梯度压缩算法" 二.1 对数量化)
 *              scale = log(max |x_group| + 1) / (2^(b-1) - 1);
 *              t = log(|x| + 1) / scale; levels 0 .. 2^(b-1) - 1 plus a sign
 *              bit, so bits must be 2, 4 or 8.  log and exp are the
 *              Cody-Waite binary32 functions (W. J. Cody, W. Waite,
 *              "Software Manual for the Elementary Functions", 1980: ln 2
 *              split as 45426 * 2^-16 + rest, the atanh series in
 *              s = (m-1)/(m+1) up to s^11/11 for log, the Taylor polynomial
 *              to r^8/8! on [-ln2/2, ln2/2] for exp), every step one
 *              rounded binary32 operation: within 2 ulp (log) and 1.5 ulp
 *              (exp) of the true functions, and reproducible bit for bit.
 *   q = round(t) (nearest-even) or floor(t) + [u < t - floor(t)]
 *   (stochastic), clamped to [0, top]; scale == 0 gives q = 0.
 *   The draw u of element i is word (i mod 4) of Philox-4x32-10 (Salmon et
 *   al., SC'11) at counter {lo32(i/4), hi32(i/4), lo32(step), hi32(step)}
 *   and key {lo32(seed), hi32(seed)}, taking its top 24 bits times 2^-24.
 * x: fp32[n];  codes_out: gc_codes_bytes(n, bits, mode) bytes;
 * scales_out: gc_scales_floats(n, group, mode) floats.  bits in {1,2,4,8}.
 * Groups of 4..128 elements (a power of two) run in one fused pass and need
 * no scratch; other group sizes need n <= max_n.
 */
GC_API gc_status gc_quant(gc_ctx* ctx, const float* x, int64_t n, int bits,
                   int64_t group, int mode, int rounding, uint64_t seed,
                   uint64_t step, uint8_t* codes_out, float* scales_out);

/*
 * Dequantisation: x_out[i] = q * scale + min (GC_MINMAX, two roundings),
 * +-(q * scale) (GC_QSGD / GC_TERN) or +-(exp(q * scale) - 1) (GC_LOG) --
 * "分布式训练中的梯度压缩算法" 二.1 (g_hat = q * scale + min; g_hat =
 * sign(q) (exp(|q| scale) - 1)).  Arguments as written by gc_quant.
 */
GC_API gc_status gc_dequant(gc_ctx* ctx, const uint8_t* codes, const float* scales,
                     int64_t n, int bits, int64_t group, int mode,
                     float* x_out);

/*
 * Error feedback + quantisation.
 * Pages: "分布式训练中的梯度压缩算法" 三 误差补偿代码示例 (compensate,
 * quantise, keep the quantisation error for the next step).
 *   c = grad + err;  (codes, scales) = gc_quant(c, ...);
 *   err = c - dequant(codes, scales)   (one rounding).
 * grad: fp32[n] (read);  err: fp32[n] (read, then overwritten).
 */
GC_API gc_status gc_ef_quant(gc_ctx* ctx, const float* grad, float* err, int64_t n,
                      int bits, int64_t group, int mode, int rounding,
                      uint64_t seed, uint64_t step, uint8_t* codes_out,
                      float* scales_out);

/*
 * Differential quantisation with error feedback.
 * Page: "分布式训练中的梯度压缩算法" 二.4 差分量化 (send only the change
 * from the previous gradient, at low precision; both sides keep a history;
 * errors pile up unless corrected from time to time).  The history ref is
 * the gradient the receiver reconstructed last (the same on both sides, so
 * quantisation errors do not pile up in it); refresh != 0 is the periodic
 * correction and treats ref as 0 (the full gradient is sent):
 *   c = grad + err (err may be NULL: c = grad);  r = refresh ? 0 : ref;
 *   d = c - r;  (codes, scales) = gc_quant(d, bits, group, mode, ...);
 *   g_hat = r + dequant(codes, scales);  err = c - g_hat (if err);
 *   ref = g_hat.
 * grad: fp32[n] (read); err, ref: fp32[n] (read, then overwritten).
 * group must be a power of two in 4 .. 128 (one fused pass; else
 * GC_ERR_UNSUPPORTED); any mode.
 */
GC_API gc_status gc_ef_diff_quant(gc_ctx* ctx, const float* grad, float* err, float* ref,
                                  int64_t n, int bits, int64_t group, int mode, int rounding,
                                  uint64_t seed, uint64_t step, int refresh,
                                  uint8_t* codes_out, float* scales_out);

/*
 * The receiving side of gc_ef_diff_quant: ref = (refresh ? 0 : ref) +
 * dequant(codes, scales), elementwise in binary32 -- after the same call
 * sequence it holds exactly the sender's ref.  ref: fp32[n] (read, then
 * overwritten).
 */
GC_API gc_status gc_diff_dequant(gc_ctx* ctx, const uint8_t* codes, const float* scales,
                                 int64_t n, int bits, int64_t group, int mode, int refresh,
                                 float* ref);

/*
 * Hybrid: error feedback + Top-K, then QSGD on the kept values.
 * Pages: "4、梯度累积与梯度压缩" 4.3 (TopK 1% + 8-bit QSGD);
 * "gradient-compression-quantization-sparsification" 三 (hybrid
 * compression).
 *   c = grad + err;  (idx_out, val) = Top-K(c) as in gc_ef_topk;
 *   (codes, scales) = QSGD(val[0..k), bits, group, rounding, seed, step),
 *   element j of the quantised array being val[j];
 *   err[idx_out[j]] = val[j] - g_hat[j];  err[i] = c[i] at every other i.
 * idx_out: int32[k];  codes_out: gc_codes_bytes(k, bits, GC_QSGD) bytes;
 * scales_out: gc_scales_floats(k, group, GC_QSGD) floats.  err must not be
 * NULL.  The kept values live in the context's scratch (n <= max_n).
 */
GC_API gc_status gc_ef_topk_quant(gc_ctx* ctx, const float* grad, float* err,
                           int64_t n, int64_t k, int bits, int64_t group,
                           int rounding, uint64_t seed, uint64_t step,
                           int32_t* idx_out, uint8_t* codes_out,
                           float* scales_out);

/*
 * One rank-r PowerSGD step with error feedback.
 * Pages: "gradient-compression-quantization-sparsification" 3.1 (low-rank
 * approximation, send the two thin matrices, rebuild on the receiver);
 * "梯度聚合通信优化实战方案" 梯度压缩原理 (error compensation is what makes
 * PowerSGD work).  Steps (Vogels et al., NeurIPS 2019, Algorithm 1):
 *   M = grad + err  (stored into err);  P = M Q;
 *   P_hat = the orthonormal factor of P (the page's Gram-Schmidt step):
 *     computed as a Cholesky QR, G = P^T P in binary64, G = U^T U with U
 *     upper triangular and positive diagonal, P_hat = P U^-1 -- the same
 *     factor Gram-Schmidt gives, up to rounding; a zero column stays zero;
 *   Q' = M^T P_hat;  err = M - P_hat Q'^T.
 * grad, err: fp32 m x n row-major;  P_out: fp32 m x r (receives P_hat);
 * Q_inout: fp32 n x r (read as Q, overwritten with Q').  1 <= r <= 16;
 * requires gc_ctx_reserve_powersgd with limits covering (m, n, r).
 * Tolerance-based, deterministic: when n is a multiple of 4 (rows of a
 * 16-byte multiple) P = M Q runs on the tensor cores with TF32 operands
 * split in three products (near-fp32 products, fp32 accumulation) and the
 * other products as fp32 FMAs; otherwise every product is an fp32 FMA.
 * Every sum is added in a fixed order, so equal inputs give equal bits.
 */
GC_API gc_status gc_powersgd_step(gc_ctx* ctx, const float* grad, float* err,
                           int64_t m, int64_t n, int r, float* P_out,
                           float* Q_inout);

/*
 * Error feedback + random sparsification.
 * Pages: "分布式训练中的梯度压缩算法" 二.2 随机稀疏化 (keep each element with
 * probability p: mask = rand(n) < p); "gradient-compression-quantization-
 * sparsification" 2.2 (random sparsification keeps the traffic steady);
 * "梯度聚合通信优化实战方案" 梯度压缩原理 (unsent entries stay in the residual).
 *   c = grad + err;  element i is kept when u_i < p, u_i being the draw of
 *   stochastic rounding (word i mod 4 of Philox-4x32-10 at counter {i/4,
 *   step}, key seed, top 24 bits * 2^-24);  the kept (i, c_i) are written in
 *   ascending index order;  err[i] = +0 when kept, c_i otherwise.
 * The number kept is random: *count_out (a DEVICE int64) receives it.  At
 * most `capacity` entries are written to idx_out / val_out; a larger count
 * sets the device status (GC_ERR_DEVICE_CHECK from gc_ctx_check).
 * err == NULL selects from grad alone and writes no residual.  0 <= n <=
 * max_n (the context's scratch holds the candidate lists).
 */
GC_API gc_status gc_ef_randk(gc_ctx* ctx, const float* grad, float* err, int64_t n, float p,
                             uint64_t seed, uint64_t step, int32_t* idx_out, float* val_out,
                             int64_t capacity, int64_t* count_out);

/*
 * Aggregation of several ranks' compressed gradients.
 * Page: "分布式训练中的梯度压缩算法" 四 (gradient compression with All-Reduce:
 * every worker compresses its local gradient, the compressed gradients are
 * aggregated and decompressed, every worker applies the result).  With
 * Top-K each rank keeps its own positions (and, quantised, its own scales),
 * so the aggregate is the sum of the ranks' decompressed sparse vectors:
 *   out[i] = 0;  for w = 0 .. W-1 in order:  out[idx_w[j]] += v_w[j]
 * one binary32 addition per present entry (deterministic).
 * idx: int32[W*K] with K = k rounded up to a multiple of 4: rank w's k
 * indices at idx + w*K (16-byte aligned, as gc_ef_topk writes them),
 * strictly increasing in [0, n) (a violation sets the device status:
 * GC_ERR_DEVICE_CHECK from gc_ctx_check, with the offending entries left
 * out).  val: fp32[W*K], laid out the same way.  out: fp32[n], fully
 * written.  1 <= W <= 1024;
 * 0 <= k <= n <= 2^31 - 1.  Scratch: W * (ceil(n / 1024) + 1) int32 (the
 * first entry of every rank in every 1024-element range of the output) of
 * the context's Top-K scratch, which holds 2 * max_n of them; a larger call
 * returns GC_ERR_WORKSPACE.
 */
GC_API gc_status gc_topk_aggregate(gc_ctx* ctx, int W, int64_t k, const int32_t* idx,
                                   const float* val, int64_t n, float* out);

/*
 * The same for the hybrid's output: rank w's values are its QSGD codes
 * decompressed, v_w[j] = +-fl(q * scale) (gc_dequant), with rank w's codes
 * at codes + w * gc_codes_bytes(k, bits, GC_QSGD) and its scales at
 * scales + w * S, S = gc_scales_floats(k, group, GC_QSGD) rounded up to a
 * multiple of 4 (so every rank's scales start on a 16-byte boundary and
 * gc_ef_topk_quant can write them in place).
 */
GC_API gc_status gc_topk_quant_aggregate(gc_ctx* ctx, int W, int64_t k, const int32_t* idx,
                                         const uint8_t* codes, const float* scales, int bits,
                                         int64_t group, int64_t n, float* out);

/*
 * Bucketed calls.
 * A data-parallel step compresses a flat gradient bucket by bucket ("4、梯度
 * 累积与梯度压缩" 4.3: a compression hook on the gradient buckets;
 * "gradient-compression-quantization-sparsification" 3.2: compression
 * happens before the data leaves GPU memory).  A bucket plan fixes the
 * buckets once; each step then runs every bucket in one launch per pass
 * (a few launches per step, whatever the number of buckets), so the
 * passes stream the whole gradient at full memory bandwidth instead of
 * one bucket at a time.
 *
 * Buckets are consecutive slices of one flat fp32 array: bucket b holds
 * elements [start_b, start_b + bucket_n[b]) with start_b = sum of the
 * earlier sizes, and keeps bucket_k[b] entries.  Per bucket the result is
 * bit-identical to the single-bucket call on the slice (gc_ef_topk, or
 * gc_ef_topk_quant with the key gc_bucket_seed(seed, b)); indices are
 * bucket-local.  The flat array may hold more than 2^31 elements (up to
 * 65536 buckets of up to 2^31 - 2^16 elements each).
 */

/*
 * Philox key of bucket b in a bucketed call with `seed`: seed XOR (b *
 * 0x9E3779B97F4A7C15), the 64-bit golden-ratio constant floor(2^64 / phi).
 * Bucket 0 keeps the seed; calls whose seeds differ by small amounts never
 * give two buckets the same key (seed + b would: bucket b + 1 under seed s
 * would repeat bucket b under seed s + 1).  The pages compress bucket by
 * bucket and fix no random stream per bucket ("4、梯度累积与梯度压缩" 4.3).
 */
GC_API uint64_t gc_bucket_seed(uint64_t seed, int b);

/*
 * Sets the context's bucket plan: nb (1 .. 65536) buckets of bucket_n[b]
 * elements (1 .. 2^31 - 2^16; a multiple of 4 for every bucket but the last,
 * so that every bucket starts on a 16-byte boundary, else
 * GC_ERR_ALIGNMENT) keeping bucket_k[b] (0 .. bucket_n[b]) entries each.
 * bucket_n and bucket_k are HOST arrays, read during the call.  Reserves
 * device scratch of about 8.1 bytes per element plus 40 KB per bucket
 * (replacing any earlier plan) and uploads the plan; synchronises the
 * context's stream first, so it must not be called while work is in flight
 * or during stream capture.  GC_ERR_NO_MEMORY when the reservation fails.
 * Residuals still pending from a deferred bucketed call (below) are written
 * to their error buffer first.
 */
GC_API gc_status gc_ctx_set_buckets(gc_ctx* ctx, int nb, const int64_t* bucket_n,
                                    const int64_t* bucket_k);

/*
 * Host-only layout of the bucketed outputs (no device work, no context).
 * For b = 0 .. nb, writes the start of bucket b's outputs (entry nb = the
 * total size):
 *   idx_off[b]:    int32 / fp32 slots, sum of bucket_k rounded up to 4;
 *   codes_off[b]:  bytes, sum of gc_codes_bytes(bucket_k, bits, GC_QSGD);
 *   scales_off[b]: floats, sum of gc_scales_floats(bucket_k, group, GC_QSGD)
 *                  rounded up to 4.
 * Each output array may be NULL (not written); codes_off / scales_off need
 * valid bits / group.  Every offset is a multiple of 16 bytes.
 */
GC_API gc_status gc_bucket_offsets(int nb, const int64_t* bucket_k, int bits, int64_t group,
                                   int64_t* idx_off, int64_t* codes_off, int64_t* scales_off);

/*
 * Diagnostics of the bucketed calls ("gradient-compression-quantization-
 * sparsification" 3.2: watch the ratio of the gradient norm after and before
 * compression; "梯度聚合通信优化实战方案" Python 演示: the error energy, the
 * sum of the squared residual).  When diag_out is not NULL the call also
 * writes, for every bucket b, three fp64 values at diag_out[3b ..]:
 *   [0] sum over the bucket of c_i^2             (c = g + e, or g)
 *   [1] sum over the kept entries of g_hat_j^2   (what the receiver
 *       reconstructs: the kept c for Top-K, the dequantised value for the
 *       hybrid), so the norm ratio is sqrt([1] / [0]);
 *   [2] sum over the bucket of e'_i^2            (the new residual; kept
 *       Top-K entries contribute 0; with err == NULL the residual the call
 *       would have stored)
 * diag_out is a DEVICE fp64[3 * nb], 16-byte aligned.  The sums are
 * computed inside the passes that already touch each value: fp32 squares
 * accumulated by fused multiply-add in runs of at most 64 per lane, added
 * over the warp into one fp32 partial per 2048-element segment (or 128 kept
 * values), then per bucket by compensated (TwoSum) fp32 summation, all in a
 * fixed order (deterministic); the relative error of each value is below
 * 5e-6 (73 roundings of 2^-24 at most).  One more small launch per call.
 * Requires finite c with |c| < 2^63 (no overflow of c^2 in fp32).
 */

/*
 * gc_ef_topk on every bucket of the plan.
 * grad, err: fp32[total] (err may be NULL: select from grad, no residual);
 * idx_out: int32[idx_off[nb]], val_out: fp32[idx_off[nb]]; bucket b's
 * entries start at idx_off[b] (slots between buckets are not written);
 * diag_out: NULL, or the diagnostics above.
 * GC_ERR_WORKSPACE when the context has no plan.
 */
GC_API gc_status gc_ef_topk_buckets(gc_ctx* ctx, const float* grad, float* err,
                                    int32_t* idx_out, float* val_out, double* diag_out);

/*
 * gc_ef_topk_quant on every bucket of the plan: bucket b is compressed as
 * gc_ef_topk_quant(slice_b, bucket_k[b], bits, group, rounding,
 * gc_bucket_seed(seed, b), step) with its indices at idx_out + idx_off[b], its codes at codes_out +
 * codes_off[b] and its scales at scales_out + scales_off[b]
 * (gc_bucket_offsets).  group must be a power of two in 4 .. 128
 * (GC_ERR_UNSUPPORTED otherwise); err must not be NULL.  diag_out: NULL, or
 * the diagnostics above (g_hat = the dequantised kept values).
 */
GC_API gc_status gc_ef_topk_quant_buckets(gc_ctx* ctx, const float* grad, float* err,
                                          int bits, int64_t group, int rounding,
                                          uint64_t seed, uint64_t step, int32_t* idx_out,
                                          uint8_t* codes_out, float* scales_out,
                                          double* diag_out);

/*
 * Deferred residual write-back of the bucketed calls with error feedback.
 * The pages store the new error e' after every step and add it back at the
 * next ("gradient-compression-quantization-sparsification" 2.1, Top-K with
 * error feedback; "4、梯度累积与梯度压缩" 4.3); they do not say when the
 * kept entries' part has to reach memory.  Written at once it is one 4-byte
 * store per kept entry at a random position of e, and each costs a DRAM
 * sector read and write-back (about 40 us for 1.3 million kept entries, a
 * tenth of the hybrid's step).
 *
 * on = 1: gc_ef_topk_quant_buckets (e' = c - g_hat) and gc_ef_topk_buckets
 * with err (e' = +0) leave e'_i = c_i at the kept positions and keep the
 * kept entries' e' in the plan's scratch; the next bucketed call on the
 * same err applies them as it reads e (no extra pass, no scattered stores).
 * Indices, values, codes, scales and diagnostics of every call are
 * bit-identical to the immediate write-back, and so is err once the
 * residuals are flushed.  Until then err differs from e' at the last
 * call's kept positions: call gc_bucket_flush before reading, changing or
 * freeing err, or before handing it to any other call.
 * on = 0 (the default): flushes pending residuals, then every call writes
 * e' in full again.
 * While residuals are pending, a bucketed call with another err (or none)
 * returns GC_ERR_INVALID_ARG (nothing launched); gc_ctx_set_buckets
 * flushes first; gc_ctx_destroy drops them.
 * The plan also records on the device whether residuals are pending, so a
 * call captured into a CUDA graph applies, at every replay, those the call
 * or replay before it left (none on the first call of a plan or after a
 * flush); gc_bucket_flush after replays writes those of the last one.
 */
GC_API gc_status gc_ctx_set_deferred_residual(gc_ctx* ctx, int on);

/*
 * Writes the pending residuals of the last deferred bucketed call into its
 * err (asynchronous on the context's stream: one small launch); a no-op when
 * none are pending.
 */
GC_API gc_status gc_bucket_flush(gc_ctx* ctx);

/*
 * Largest n accepted by gc_ef_topk_noalloc: its scratch is a fixed device
 * array of about 8 bytes per element up to this size (8.2 MiB in all).
 */
#define GC_NOALLOC_MAX_N 1048576

/*
 * gc_ef_topk without any allocation.  The pages have no counterpart: this
 * entry exists for callers that must not allocate device memory -- code
 * whose device memory all belongs to another allocator (a framework's
 * caching pool, a fixed arena), code with a hard memory budget, or code on
 * a latency-critical path where cudaMalloc's implicit device-wide
 * synchronisation is unacceptable.  gc_ctx_create allocates; this call
 * does not, and takes no context.
 *
 * Same arguments, results and error rules as gc_ef_topk (grad, err,
 * idx_out and val_out are caller-owned device buffers; err may be NULL),
 * plus the CUDA stream to run on, which must belong to the current device.
 * n must be <= GC_NOALLOC_MAX_N, else GC_ERR_WORKSPACE before any device
 * work.
 *
 * Scratch: one library-owned static device array per GPU, reserved when
 * the library's module is loaded on that GPU and held until the process
 * exits.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The address is kept for the life of the
 * process: after cudaDeviceReset (or any reset of the device's primary
 * context) the module is loaded again elsewhere, so do not call this entry
 * point on that device after such a reset.  Every call on a device shares the one
 * array, and each call first clears the part that must start at zero;
 * calls that overlap on the GPU (other streams, other host threads) race on
 * it and give wrong results, so serialise them.  Device self-check status
 * is not reported (there is no context to hold it).  Calls no cudaMalloc,
 * cudaFree or other allocating routine.
 */
GC_API gc_status gc_ef_topk_noalloc(const float* grad, float* err, int64_t n, int64_t k,
                                    int32_t* idx_out, float* val_out, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* GC_H_ */
