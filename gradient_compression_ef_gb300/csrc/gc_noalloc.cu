// gc_noalloc.cu -- EF + Top-K whose scratch is a static device array, for
// callers that cannot allocate device memory (see gc_ef_topk_noalloc in
// include/gc.h).  The kernels are the ones gc_ef_topk runs; only where the
// scratch comes from differs.
#include <stddef.h>

#include <mutex>

#include "gc_internal.cuh"

namespace gc {
namespace {

constexpr int64_t kNoAllocMaxN = GC_NOALLOC_MAX_N;
constexpr int kMaxDevices = 128;

// Layout of the static scratch: the leading part (up to tile_above) must
// be zero when a call starts; the rest is fully written by every call.
struct StaticScratch {
  uint32_t hist[kHistBins];
  uint32_t mid[kMidBins];
  uint32_t low[kLowBins];
  uint32_t tile_kept[kMaxTiles];
  TopkSel sel;
  uint32_t status[4];
  uint32_t tile_above[kMaxTiles];
  uint32_t tile_out[kMaxTiles];
  uint32_t tile_tie[kMaxTiles];
  uint2 stash[kStashMax];
  uint2 cand[kNoAllocMaxN];
};

// One copy per GPU that loads the library; lives until the process exits.
static __device__ __align__(256) unsigned char g_topk_scratch[sizeof(StaticScratch)];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];
int g_num_sms[kMaxDevices];

// Once per device, with that device current: the device address of the
// scratch array (the host-side symbol is only a stand-in for it).
gc_status device_scratch(int dev, void** addr, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return GC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GC_ERR_CUDA;
    }
    int n_sms = 0;
    if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GC_ERR_CUDA;
    }
    g_num_sms[dev] = n_sms;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  *sms = g_num_sms[dev];
  return GC_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gc

extern "C" gc_status gc_ef_topk_noalloc(const float* grad, float* err, int64_t n, int64_t k,
                                        int32_t* idx_out, float* val_out, void* cuda_stream) {
  using gc::aligned16;
  if (n < 0 || n > INT32_MAX || k < 0 || k > n) return GC_ERR_INVALID_ARG;
  if (n > 0 && !grad) return GC_ERR_INVALID_ARG;
  if (k > 0 && (!idx_out || !val_out)) return GC_ERR_INVALID_ARG;
  if ((n > 0 && (!aligned16(grad) || (err && !aligned16(err)))) ||
      (k > 0 && (!aligned16(idx_out) || !aligned16(val_out))))
    return GC_ERR_ALIGNMENT;
  if (n > gc::kNoAllocMaxN) return GC_ERR_WORKSPACE;
  if (n == 0) return GC_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GC_ERR_CUDA;
  void* base = nullptr;
  int sms = 0;
  const gc_status st = gc::device_scratch(dev, &base, &sms);
  if (st != GC_OK) return st;
  char* b = static_cast<char*>(base);
  gc::Workspace ws{};
  ws.hist = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, hist));
  ws.mid = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, mid));
  ws.low = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, low));
  ws.tile_kept = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, tile_kept));
  ws.sel = reinterpret_cast<gc::TopkSel*>(b + offsetof(gc::StaticScratch, sel));
  ws.status = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, status));
  ws.tile_above = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, tile_above));
  ws.tile_out = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, tile_out));
  ws.tile_tie = reinterpret_cast<uint32_t*>(b + offsetof(gc::StaticScratch, tile_tie));
  ws.cand = reinterpret_cast<uint2*>(b + offsetof(gc::StaticScratch, cand));
  ws.stash = reinterpret_cast<uint2*>(b + offsetof(gc::StaticScratch, stash));
  ws.vals = nullptr;
  ws.partials = nullptr;
  ws.max_n = gc::kNoAllocMaxN;
  ws.max_partials = 0;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // the array keeps the previous call's contents: clear the counters and
  // the histogram that the passes expect to start at zero
  if (cudaMemsetAsync(base, 0, offsetof(gc::StaticScratch, tile_above), s) != cudaSuccess)
    return GC_ERR_CUDA;
  return gc::launch_ef_topk_on(ws, s, sms, grad, err, n, k, idx_out, val_out);
}
