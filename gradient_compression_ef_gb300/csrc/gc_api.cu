// gc_api.cu -- the C ABI of include/gc.h: argument validation, context and
// scratch management, and dispatch to the kernel launchers.
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "gc_internal.cuh"

using gc::ceil_div;
using gc::round_up;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_bits(int bits) { return bits == 1 || bits == 2 || bits == 4 || bits == 8; }

gc_status check_quant(int64_t n, int bits, int64_t group, int mode, int rounding) {
  if (n < 0 || n > INT32_MAX || group < 0) return GC_ERR_INVALID_ARG;
  if (mode != GC_MINMAX && mode != GC_QSGD && mode != GC_TERN && mode != GC_LOG)
    return GC_ERR_INVALID_ARG;
  if (rounding != GC_NEAREST_EVEN && rounding != GC_STOCHASTIC) return GC_ERR_INVALID_ARG;
  if (!valid_bits(bits)) return GC_ERR_UNSUPPORTED;
  if (mode == GC_TERN && bits != 2) return GC_ERR_UNSUPPORTED;
  if (mode == GC_LOG && bits == 1) return GC_ERR_UNSUPPORTED;  // no magnitude bit
  return GC_OK;
}

// A buffer that the call touches must be non-NULL and 16-byte aligned.
gc_status check_buf(const void* p, bool used) {
  if (!used) return GC_OK;
  if (!p) return GC_ERR_INVALID_ARG;
  if (!aligned16(p)) return GC_ERR_ALIGNMENT;
  return GC_OK;
}

#define GC_TRY(expr)                    \
  do {                                  \
    const gc_status _st = (expr);       \
    if (_st != GC_OK) return _st;       \
  } while (0)

// Makes the context's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    if (ok && prev >= 0) cudaSetDevice(prev);
  }
};

// Layout of the per-context scratch (one allocation).
struct WsLayout {
  size_t hist, mid, low, tile_kept, sel, status, tile_above, tile_out, tile_tie, cand, stash, vals,
      partials, total;
};

WsLayout ws_layout(int64_t max_n, int64_t max_partials) {
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) / 256 * 256; return o; };
  L.hist = take(sizeof(uint32_t) * gc::kHistBins);
  L.mid = take(sizeof(uint32_t) * gc::kMidBins);
  L.low = take(sizeof(uint32_t) * gc::kLowBins);
  L.tile_kept = take(sizeof(uint32_t) * gc::kMaxTiles);
  L.sel = take(sizeof(gc::TopkSel));
  L.status = take(sizeof(uint32_t) * 4);
  L.tile_above = take(sizeof(uint32_t) * gc::kMaxTiles);
  L.tile_out = take(sizeof(uint32_t) * gc::kMaxTiles);
  L.tile_tie = take(sizeof(uint32_t) * gc::kMaxTiles);
  L.cand = take(sizeof(uint2) * std::max<int64_t>(max_n, 1));
  L.stash = take(sizeof(uint2) * gc::kStashMax);
  L.vals = take(sizeof(float) * std::max<int64_t>(max_n, 1));
  L.partials = take(sizeof(float4) * std::max<int64_t>(max_partials, 1));
  L.total = off;
  return L;
}

}  // namespace

extern "C" {

int gc_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* gc_status_string(int status) {
  switch (status) {
    case GC_OK: return "ok";
    case GC_ERR_INVALID_ARG: return "invalid argument";
    case GC_ERR_UNSUPPORTED: return "unsupported bit width or mode";
    case GC_ERR_ALIGNMENT: return "buffer not 16-byte aligned";
    case GC_ERR_WORKSPACE:
      return "size exceeds the reserved scratch (the context's, or the fixed array of "
             "the allocation-free call)";
    case GC_ERR_CUDA: return "CUDA runtime error";
    case GC_ERR_DEVICE_CHECK: return "device-side self check failed";
    case GC_ERR_NO_MEMORY: return "device allocation failed";
    default: return "unknown status";
  }
}

int64_t gc_codes_bytes(int64_t n, int bits, int mode) {
  if (n < 0 || !valid_bits(bits)) return -1;
  if (mode != GC_MINMAX && mode != GC_QSGD && mode != GC_TERN && mode != GC_LOG) return -1;
  const int cb = mode == GC_TERN ? 2 : bits;
  int64_t bytes = round_up((n * cb + 7) / 8, 16);
  if (mode == GC_QSGD) bytes += round_up((n + 7) / 8, 16);
  return bytes;
}

int64_t gc_scales_floats(int64_t n, int64_t group, int mode) {
  if (n < 0 || group < 0) return -1;
  if (mode != GC_MINMAX && mode != GC_QSGD && mode != GC_TERN && mode != GC_LOG) return -1;
  if (n == 0) return 0;
  const int64_t G = group == 0 ? n : group;
  return ceil_div(n, G) * (mode == GC_MINMAX ? 2 : 1);
}

gc_status gc_ctx_create(gc_ctx** out, void* cuda_stream, int64_t max_n) {
  if (!out || max_n < 0 || max_n > INT32_MAX) return GC_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GC_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GC_ERR_CUDA;
  gc_ctx* ctx = static_cast<gc_ctx*>(calloc(1, sizeof(gc_ctx)));
  if (!ctx) return GC_ERR_NO_MEMORY;
  ctx->device = dev;
  ctx->num_sms = sms;
  ctx->stream = static_cast<cudaStream_t>(cuda_stream);
  // partial statistics of the multi-pass quantisation: at most
  // 2 * ceil(max_n / 1024) chunks of groups larger than 1024 elements
  const int64_t max_partials = 2 * ceil_div(std::max<int64_t>(max_n, 1), 1024) + 2;
  const WsLayout L = ws_layout(max_n, max_partials);
  void* base = nullptr;
  const cudaError_t e = cudaMalloc(&base, L.total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    free(ctx);
    return e == cudaErrorMemoryAllocation ? GC_ERR_NO_MEMORY : GC_ERR_CUDA;
  }
  if (cudaMemset(base, 0, L.total) != cudaSuccess) {
    cudaFree(base);
    free(ctx);
    return GC_ERR_CUDA;
  }
  char* b = static_cast<char*>(base);
  ctx->ws_base = base;
  ctx->ws.hist = reinterpret_cast<uint32_t*>(b + L.hist);
  ctx->ws.mid = reinterpret_cast<uint32_t*>(b + L.mid);
  ctx->ws.low = reinterpret_cast<uint32_t*>(b + L.low);
  ctx->ws.tile_kept = reinterpret_cast<uint32_t*>(b + L.tile_kept);
  ctx->ws.sel = reinterpret_cast<gc::TopkSel*>(b + L.sel);
  ctx->ws.status = reinterpret_cast<uint32_t*>(b + L.status);
  ctx->ws.tile_above = reinterpret_cast<uint32_t*>(b + L.tile_above);
  ctx->ws.tile_out = reinterpret_cast<uint32_t*>(b + L.tile_out);
  ctx->ws.tile_tie = reinterpret_cast<uint32_t*>(b + L.tile_tie);
  ctx->ws.cand = reinterpret_cast<uint2*>(b + L.cand);
  ctx->ws.stash = reinterpret_cast<uint2*>(b + L.stash);
  ctx->ws.vals = reinterpret_cast<float*>(b + L.vals);
  ctx->ws.partials = reinterpret_cast<float4*>(b + L.partials);
  ctx->ws.max_n = max_n;
  ctx->ws.max_partials = max_partials;
  if (gc::prepare_aggregate_kernels() != GC_OK) {
    cudaFree(base);
    free(ctx);
    return GC_ERR_CUDA;
  }
  *out = ctx;
  return GC_OK;
}

namespace {
void free_timing(gc_ctx* ctx) {
  for (int i = 0; i < ctx->timing_cap; ++i) {
    cudaEventDestroy(ctx->ev_start[i]);
    cudaEventDestroy(ctx->ev_stop[i]);
  }
  free(ctx->ev_start);
  free(ctx->ev_stop);
  free(ctx->ev_phase);
  ctx->ev_start = ctx->ev_stop = nullptr;
  ctx->ev_phase = nullptr;
  ctx->timing_cap = ctx->timing_used = 0;
}
}  // namespace

const char* gc_phase_name(int phase) {
  static const char* names[GC_PHASE_COUNT] = {
      "ef_hist", "collect", "write", "ef_add", "quant_fused", "quant_stats",
      "quant_combine", "quant_apply", "dequant", "psgd_mq", "psgd_mtp", "psgd_resid",
      "refine", "bk_hist", "bk_collect", "bk_refine", "bk_write", "bk_quant", "agg_bounds",
      "agg_accumulate", "randk_mark", "randk_write", "bk_diag", "bk_flush", "psgd_thin"};
  return (phase >= 0 && phase < GC_PHASE_COUNT) ? names[phase] : "?";
}

gc_status gc_ctx_enable_timing(gc_ctx* ctx, int max_launches) {
  if (!ctx || max_launches < 0) return GC_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return GC_ERR_CUDA;
  free_timing(ctx);
  if (max_launches == 0) return GC_OK;
  ctx->ev_start = static_cast<cudaEvent_t*>(calloc(max_launches, sizeof(cudaEvent_t)));
  ctx->ev_stop = static_cast<cudaEvent_t*>(calloc(max_launches, sizeof(cudaEvent_t)));
  ctx->ev_phase = static_cast<int*>(calloc(max_launches, sizeof(int)));
  if (!ctx->ev_start || !ctx->ev_stop || !ctx->ev_phase) {
    free_timing(ctx);
    return GC_ERR_NO_MEMORY;
  }
  for (int i = 0; i < max_launches; ++i) {
    if (cudaEventCreate(&ctx->ev_start[i]) != cudaSuccess ||
        cudaEventCreate(&ctx->ev_stop[i]) != cudaSuccess) {
      ctx->timing_cap = i;  // destroy what was made (a failed create leaves garbage)
      free_timing(ctx);
      return GC_ERR_CUDA;
    }
    ctx->timing_cap = i + 1;
  }
  ctx->timing_used = 0;
  return GC_OK;
}

gc_status gc_ctx_read_timing(gc_ctx* ctx, double* ms_out, int64_t* count_out) {
  if (!ctx || !ms_out || !count_out) return GC_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return GC_ERR_CUDA;
  for (int i = 0; i < ctx->timing_used; ++i) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, ctx->ev_start[i], ctx->ev_stop[i]) != cudaSuccess)
      return GC_ERR_CUDA;
    ms_out[ctx->ev_phase[i]] += ms;
    count_out[ctx->ev_phase[i]] += 1;
  }
  ctx->timing_used = 0;
  return GC_OK;
}

int64_t gc_ctx_launch_count(gc_ctx* ctx) { return ctx ? ctx->launches : -1; }

gc_status gc_ctx_destroy(gc_ctx* ctx) {
  if (!ctx) return GC_OK;
  DeviceGuard guard(ctx->device);
  gc_status st = GC_OK;
  if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) st = GC_ERR_CUDA;
  free_timing(ctx);
  if (ctx->ws_base) cudaFree(ctx->ws_base);
  if (ctx->psgd_base) cudaFree(ctx->psgd_base);
  gc::free_buckets(ctx);
  free(ctx);
  return st;
}

gc_status gc_ctx_set_stream(gc_ctx* ctx, void* cuda_stream) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  ctx->stream = static_cast<cudaStream_t>(cuda_stream);
  return GC_OK;
}

gc_status gc_ctx_reserve_powersgd(gc_ctx* ctx, int64_t max_m, int64_t max_n, int max_r) {
  if (!ctx || max_m < 1 || max_n < 1 || max_r < 1 || max_r > 16) return GC_ERR_INVALID_ARG;
  if (ctx->psgd_base && max_m <= ctx->psgd.max_m && max_n <= ctx->psgd.max_n &&
      max_r <= ctx->psgd.max_r)
    return GC_OK;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  max_m = std::max<int64_t>(max_m, ctx->psgd.max_m);
  max_n = std::max<int64_t>(max_n, ctx->psgd.max_n);
  max_r = std::max(max_r, ctx->psgd.max_r);
  const int64_t bytes = gc::psgd_workspace_bytes(max_m, max_n, max_r, ctx->num_sms);
  if (ctx->psgd_base) {
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return GC_ERR_CUDA;
    cudaFree(ctx->psgd_base);
    ctx->psgd_base = nullptr;
  }
  void* base = nullptr;
  const cudaError_t e = cudaMalloc(&base, (size_t)bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    ctx->psgd = gc::PsgdWorkspace{};
    return e == cudaErrorMemoryAllocation ? GC_ERR_NO_MEMORY : GC_ERR_CUDA;
  }
  // the memset runs on the legacy stream: finish it before any launch
  if (cudaMemset(base, 0, (size_t)bytes) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(base);
    return GC_ERR_CUDA;
  }
  ctx->psgd_base = base;
  ctx->psgd.max_m = max_m;
  ctx->psgd.max_n = max_n;
  ctx->psgd.max_r = max_r;
  ctx->psgd.bytes = bytes;
  return GC_OK;
}

gc_status gc_ctx_check(gc_ctx* ctx) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return GC_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ctx->ws.status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GC_ERR_CUDA;
  if (word == 0) return GC_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(ctx->ws.status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return GC_ERR_CUDA;
  return GC_ERR_DEVICE_CHECK;
}

gc_status gc_ef_topk(gc_ctx* ctx, const float* grad, float* err, int64_t n, int64_t k,
                     int32_t* idx_out, float* val_out) {
  if (!ctx || n < 0 || n > INT32_MAX || k < 0 || k > n) return GC_ERR_INVALID_ARG;
  GC_TRY(check_buf(grad, n > 0));
  if (err) GC_TRY(check_buf(err, n > 0));
  GC_TRY(check_buf(idx_out, k > 0));
  GC_TRY(check_buf(val_out, k > 0));
  if (k > 0 && n > ctx->ws.max_n) return GC_ERR_WORKSPACE;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_ef_topk(ctx, grad, err, n, k, idx_out, val_out);
}

gc_status gc_quant(gc_ctx* ctx, const float* x, int64_t n, int bits, int64_t group,
                   int mode, int rounding, uint64_t seed, uint64_t step, uint8_t* codes_out,
                   float* scales_out) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  GC_TRY(check_quant(n, bits, group, mode, rounding));
  GC_TRY(check_buf(x, n > 0));
  GC_TRY(check_buf(codes_out, n > 0));
  GC_TRY(check_buf(scales_out, n > 0));
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_quant(ctx, x, nullptr, nullptr, 0, n, bits, group, mode, rounding, seed,
                          step, codes_out, scales_out);
}

gc_status gc_dequant(gc_ctx* ctx, const uint8_t* codes, const float* scales, int64_t n,
                     int bits, int64_t group, int mode, float* x_out) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  GC_TRY(check_quant(n, bits, group, mode, GC_NEAREST_EVEN));
  GC_TRY(check_buf(codes, n > 0));
  GC_TRY(check_buf(scales, n > 0));
  GC_TRY(check_buf(x_out, n > 0));
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_dequant(ctx, codes, scales, n, bits, group, mode, x_out);
}

gc_status gc_ef_quant(gc_ctx* ctx, const float* grad, float* err, int64_t n, int bits,
                      int64_t group, int mode, int rounding, uint64_t seed, uint64_t step,
                      uint8_t* codes_out, float* scales_out) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  GC_TRY(check_quant(n, bits, group, mode, rounding));
  GC_TRY(check_buf(grad, n > 0));
  GC_TRY(check_buf(err, n > 0));
  GC_TRY(check_buf(codes_out, n > 0));
  GC_TRY(check_buf(scales_out, n > 0));
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_quant(ctx, grad, err, nullptr, 0, n, bits, group, mode, rounding, seed,
                          step, codes_out, scales_out);
}

gc_status gc_ef_diff_quant(gc_ctx* ctx, const float* grad, float* err, float* ref, int64_t n,
                           int bits, int64_t group, int mode, int rounding, uint64_t seed,
                           uint64_t step, int refresh, uint8_t* codes_out, float* scales_out) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  GC_TRY(check_quant(n, bits, group, mode, rounding));
  GC_TRY(check_buf(grad, n > 0));
  if (err) GC_TRY(check_buf(err, n > 0));
  GC_TRY(check_buf(ref, n > 0));
  GC_TRY(check_buf(codes_out, n > 0));
  GC_TRY(check_buf(scales_out, n > 0));
  if (n > 0 && !gc::quant_is_fused(n, group)) return GC_ERR_UNSUPPORTED;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_diff_quant(ctx, grad, err, ref, n, bits, group, mode, rounding, seed, step,
                               refresh, codes_out, scales_out);
}

gc_status gc_diff_dequant(gc_ctx* ctx, const uint8_t* codes, const float* scales, int64_t n,
                          int bits, int64_t group, int mode, int refresh, float* ref) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  GC_TRY(check_quant(n, bits, group, mode, GC_NEAREST_EVEN));
  GC_TRY(check_buf(codes, n > 0));
  GC_TRY(check_buf(scales, n > 0));
  GC_TRY(check_buf(ref, n > 0));
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_diff_dequant(ctx, codes, scales, n, bits, group, mode, refresh, ref);
}

gc_status gc_ef_topk_quant(gc_ctx* ctx, const float* grad, float* err, int64_t n, int64_t k,
                           int bits, int64_t group, int rounding, uint64_t seed,
                           uint64_t step, int32_t* idx_out, uint8_t* codes_out,
                           float* scales_out) {
  if (!ctx || n < 0 || n > INT32_MAX || k < 0 || k > n) return GC_ERR_INVALID_ARG;
  GC_TRY(check_quant(k, bits, group, GC_QSGD, rounding));
  GC_TRY(check_buf(grad, n > 0));
  if (!err && n > 0) return GC_ERR_INVALID_ARG;
  GC_TRY(check_buf(err, n > 0));
  GC_TRY(check_buf(idx_out, k > 0));
  GC_TRY(check_buf(codes_out, k > 0));
  GC_TRY(check_buf(scales_out, k > 0));
  if (k > 0 && n > ctx->ws.max_n) return GC_ERR_WORKSPACE;
  // the kept values are quantised by the single-pass kernel, which takes
  // groups of 4..128 elements (a power of two)
  if (k > 0 && !gc::quant_is_fused(k, group)) return GC_ERR_UNSUPPORTED;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  GC_TRY(gc::launch_ef_topk(ctx, grad, err, n, k, idx_out, ctx->ws.vals));
  if (k == 0) return GC_OK;
  return gc::launch_quant(ctx, ctx->ws.vals, err, idx_out, n, k, bits, group, GC_QSGD,
                          rounding, seed, step, codes_out, scales_out);
}

gc_status gc_powersgd_step(gc_ctx* ctx, const float* grad, float* err, int64_t m, int64_t n,
                           int r, float* P_out, float* Q_inout) {
  if (!ctx || m < 0 || n < 0 || r < 1 || r > 16) return GC_ERR_INVALID_ARG;
  const bool used = m > 0 && n > 0;
  GC_TRY(check_buf(grad, used));
  GC_TRY(check_buf(err, used));
  GC_TRY(check_buf(P_out, used));
  GC_TRY(check_buf(Q_inout, used));
  if (!used) return GC_OK;
  if (!ctx->psgd_base || m > ctx->psgd.max_m || n > ctx->psgd.max_n || r > ctx->psgd.max_r)
    return GC_ERR_WORKSPACE;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_powersgd(ctx, grad, err, m, n, r, P_out, Q_inout);
}

namespace {
// Writes the residuals a deferred bucketed call left pending into its err.
gc_status flush_pending(gc_ctx* ctx) {
  if (!ctx->bk_pending) return GC_OK;
  float* err = ctx->bk_pending;
  ctx->bk_pending = nullptr;
  if (!ctx->bk_base) return GC_OK;
  return gc::launch_bucket_flush(ctx, err);
}
}  // namespace

gc_status gc_ctx_set_buckets(gc_ctx* ctx, int nb, const int64_t* bucket_n,
                             const int64_t* bucket_k) {
  if (!ctx || nb < 1 || nb > gc::kMaxBuckets || !bucket_n || !bucket_k) return GC_ERR_INVALID_ARG;
  for (int b = 0; b < nb; ++b) {
    if (bucket_n[b] < 1 || bucket_n[b] > gc::kMaxBucketElems) return GC_ERR_INVALID_ARG;
    if (bucket_k[b] < 0 || bucket_k[b] > bucket_n[b]) return GC_ERR_INVALID_ARG;
  }
  for (int b = 0; b + 1 < nb; ++b)
    if (bucket_n[b] % 4 != 0) return GC_ERR_ALIGNMENT;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  GC_TRY(flush_pending(ctx));
  if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return GC_ERR_CUDA;
  return gc::plan_buckets(ctx, nb, bucket_n, bucket_k);
}

gc_status gc_ctx_set_deferred_residual(gc_ctx* ctx, int on) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  if (!on) GC_TRY(flush_pending(ctx));
  ctx->bk_defer = on ? 1 : 0;
  return GC_OK;
}

gc_status gc_bucket_flush(gc_ctx* ctx) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return flush_pending(ctx);
}

uint64_t gc_bucket_seed(uint64_t seed, int b) { return gc::bucket_seed(seed, b); }

gc_status gc_bucket_offsets(int nb, const int64_t* bucket_k, int bits, int64_t group,
                            int64_t* idx_off, int64_t* codes_off, int64_t* scales_off) {
  if (nb < 1 || nb > gc::kMaxBuckets || !bucket_k) return GC_ERR_INVALID_ARG;
  for (int b = 0; b < nb; ++b)
    if (bucket_k[b] < 0 || bucket_k[b] > INT32_MAX) return GC_ERR_INVALID_ARG;
  if (codes_off && !valid_bits(bits)) return GC_ERR_UNSUPPORTED;
  if (scales_off && group < 1) return GC_ERR_INVALID_ARG;
  int64_t oi = 0, oc = 0, os = 0;
  for (int b = 0; b <= nb; ++b) {
    if (idx_off) idx_off[b] = oi;
    if (codes_off) codes_off[b] = oc;
    if (scales_off) scales_off[b] = os;
    if (b == nb) break;
    oi += round_up(bucket_k[b], 4);
    if (codes_off) oc += gc_codes_bytes(bucket_k[b], bits, GC_QSGD);
    if (scales_off) os += round_up(gc_scales_floats(bucket_k[b], group, GC_QSGD), 4);
  }
  return GC_OK;
}

gc_status gc_ef_topk_buckets(gc_ctx* ctx, const float* grad, float* err, int32_t* idx_out,
                             float* val_out, double* diag_out) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  if (!ctx->bk_base) return GC_ERR_WORKSPACE;
  const gc::BucketWs& w = ctx->bk;
  GC_TRY(check_buf(grad, true));
  if (err) GC_TRY(check_buf(err, true));
  GC_TRY(check_buf(idx_out, w.vals_total > 0));
  GC_TRY(check_buf(val_out, w.vals_total > 0));
  if (diag_out) GC_TRY(check_buf(diag_out, true));
  // pending residuals belong to one error buffer
  if (ctx->bk_pending && ctx->bk_pending != err) return GC_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  const bool defer = ctx->bk_defer != 0 && err != nullptr;
  ctx->bk_pending = nullptr;
  GC_TRY(gc::launch_ef_topk_buckets(ctx, grad, err, idx_out, val_out, true, 0, 0,
                                    diag_out != nullptr, defer, defer));
  if (defer) ctx->bk_pending = err;
  return diag_out ? gc::launch_bucket_diag(ctx, false, diag_out) : GC_OK;
}

gc_status gc_ef_topk_quant_buckets(gc_ctx* ctx, const float* grad, float* err, int bits,
                                   int64_t group, int rounding, uint64_t seed, uint64_t step,
                                   int32_t* idx_out, uint8_t* codes_out, float* scales_out,
                                   double* diag_out) {
  if (!ctx) return GC_ERR_INVALID_ARG;
  if (!ctx->bk_base) return GC_ERR_WORKSPACE;
  const gc::BucketWs& w = ctx->bk;
  GC_TRY(check_quant(1, bits, group, GC_QSGD, rounding));
  if (group < 4 || group > 128 || (group & (group - 1)) != 0) return GC_ERR_UNSUPPORTED;
  GC_TRY(check_buf(grad, true));
  if (!err) return GC_ERR_INVALID_ARG;
  GC_TRY(check_buf(err, true));
  GC_TRY(check_buf(idx_out, w.vals_total > 0));
  GC_TRY(check_buf(codes_out, w.vals_total > 0));
  GC_TRY(check_buf(scales_out, w.vals_total > 0));
  if (diag_out) GC_TRY(check_buf(diag_out, true));
  // pending residuals belong to one error buffer
  if (ctx->bk_pending && ctx->bk_pending != err) return GC_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  const bool diag = diag_out != nullptr;
  // in deferred mode the hist pass checks the plan's ready flag itself, so a
  // call captured into a graph applies whatever the call before it left
  const bool defer = ctx->bk_defer != 0, patch = defer;
  ctx->bk_pending = nullptr;
  GC_TRY(gc::launch_ef_topk_buckets(ctx, grad, err, idx_out, w.vals, false, bits, group, diag,
                                    patch));
  GC_TRY(gc::launch_quant_buckets(ctx, err, idx_out, bits, group, rounding, seed, step,
                                  codes_out, scales_out, diag, defer));
  if (defer) ctx->bk_pending = err;
  return diag ? gc::launch_bucket_diag(ctx, true, diag_out) : GC_OK;
}

namespace {
gc_status check_aggregate(gc_ctx* ctx, int W, int64_t k, int64_t n, const void* idx,
                          const void* out) {
  if (!ctx || W < 1 || W > gc::aggregate_max_ranks() || k < 0 || n < 0 || k > n ||
      n > INT32_MAX)
    return GC_ERR_INVALID_ARG;
  GC_TRY(check_buf(idx, k > 0));
  GC_TRY(check_buf(out, n > 0));
  if (n > 0 && gc::aggregate_scratch_ints(W, n) > 2 * std::max<int64_t>(ctx->ws.max_n, 1))
    return GC_ERR_WORKSPACE;
  return GC_OK;
}
}  // namespace

gc_status gc_topk_aggregate(gc_ctx* ctx, int W, int64_t k, const int32_t* idx,
                            const float* val, int64_t n, float* out) {
  GC_TRY(check_aggregate(ctx, W, k, n, idx, out));
  GC_TRY(check_buf(val, k > 0));
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_aggregate(ctx, W, k, idx, val, nullptr, nullptr, 0, 0, n, out);
}

gc_status gc_topk_quant_aggregate(gc_ctx* ctx, int W, int64_t k, const int32_t* idx,
                                  const uint8_t* codes, const float* scales, int bits,
                                  int64_t group, int64_t n, float* out) {
  GC_TRY(check_aggregate(ctx, W, k, n, idx, out));
  GC_TRY(check_quant(k, bits, group, GC_QSGD, GC_NEAREST_EVEN));
  GC_TRY(check_buf(codes, k > 0));
  GC_TRY(check_buf(scales, k > 0));
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_aggregate(ctx, W, k, idx, nullptr, codes, scales, bits, group, n, out);
}

gc_status gc_ef_randk(gc_ctx* ctx, const float* grad, float* err, int64_t n, float p,
                      uint64_t seed, uint64_t step, int32_t* idx_out, float* val_out,
                      int64_t capacity, int64_t* count_out) {
  if (!ctx || n < 0 || n > INT32_MAX || capacity < 0 || !count_out || !(p >= 0.0f) ||
      !(p <= 1.0f))
    return GC_ERR_INVALID_ARG;
  GC_TRY(check_buf(grad, n > 0));
  if (err) GC_TRY(check_buf(err, n > 0));
  GC_TRY(check_buf(idx_out, capacity > 0));
  GC_TRY(check_buf(val_out, capacity > 0));
  if (n > ctx->ws.max_n) return GC_ERR_WORKSPACE;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return GC_ERR_CUDA;
  return gc::launch_ef_randk(ctx, grad, err, n, p, seed, step, idx_out, val_out, capacity,
                             count_out);
}

}  // extern "C"
