// Head classification for callers that cannot allocate device memory.
//
// hc_classify needs a workspace (the four fp32 attention-output planes and
// the per-token cosines) that the caller normally allocates.  Some callers
// cannot: a plugin whose host framework owns all device memory and offers no
// allocator at that point, or a real-time loop whose policy forbids any
// allocation after start-up.  hc_classify_static_scratch gives them the same
// classification with its workspace in a fixed array that lives in the
// library's own device image.  The paper has no counterpart to this; it is a
// deployment convenience.
//
// Costs and limits:
//  - every GPU that loads this library holds HC_STATIC_SCRATCH_BYTES of
//    device memory for the array until the process exits;
//  - layers whose workspace exceeds that size are rejected with
//    HC_ERR_SIZE (hc_classify_scratch_bytes gives the size a layer needs);
//  - all calls share the one array, so calls whose kernels overlap on the GPU
//    (two streams, or two host threads) race on it: serialise them.
// The array keeps whatever the previous call left in it.  Nothing needs
// clearing: every byte of the workspace that a call reads it has written
// first (each output plane row and each per-token statistic is stored once
// before it is read).
#include <mutex>

#include "hc_internal.h"

// The fixed workspace.  In host code this name is only a host-side stand-in:
// its device address must come from cudaGetSymbolAddress on the device that
// runs the kernels.
static __device__ __align__(256) unsigned char g_hc_static_scratch[HC_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;

// Device address of the array on the current device, looked up once per
// device (the first call on each device does the lookup).
hc_status static_scratch_address(void** out) {
  static std::mutex mu;
  static void* cached[kMaxDevices] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return hc::record_error(HC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return hc::record_error(HC_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_hc_static_scratch);
    if (e != cudaSuccess || !p)
      return hc::record_error(HC_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    cached[dev] = p;
  }
  *out = cached[dev];
  return HC_OK;
}

}  // namespace

extern "C" hc_status hc_classify_static_scratch(const hc_config* cfg, const void* q, const void* k,
                                                const void* v, int32_t n_key_frames, int8_t* labels_dev,
                                                int8_t* labels_host, float* stats_dev, void* o_full,
                                                void* stream) {
  size_t need = 0;
  hc_status s = hc_classify_scratch_bytes(cfg, n_key_frames, &need);
  if (s != HC_OK) return s;
  if (need > (size_t)HC_STATIC_SCRATCH_BYTES)
    return hc::record_error(HC_ERR_SIZE,
                            "layer needs %zu bytes of classification workspace; the static workspace holds %zu "
                            "(use hc_classify with a caller-allocated workspace)",
                            need, (size_t)HC_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if ((s = static_scratch_address(&scratch)) != HC_OK) return s;
  return hc_classify(cfg, q, k, v, n_key_frames, labels_dev, labels_host, stats_dev, o_full, scratch,
                     (size_t)HC_STATIC_SCRATCH_BYTES, stream);
}
