// moe_expert_ffn_grouped_noalloc: the grouped expert FFN for callers that
// cannot allocate device memory themselves.
//
// The ordinary entry point takes its scratch (the bf16 SwiGLU activations h,
// T*k rows of I values) from a caller-provided workspace.  Some callers have
// no way to provide one: code running inside a host framework that owns every
// byte of device memory and exposes no allocator, firmware-like services with
// a fixed memory budget decided at load time, and serving loops that must
// never call cudaMalloc/cudaFree because those calls can synchronise the whole
// device and stall every other stream.  This variant uses a scratch array
// that is part of the library image instead: it exists once per device that
// loads the library and stays allocated until the process exits.
//
// The first call on each device looks up the array's device address with
// cudaGetSymbolAddress while that device is current (host code cannot use the
// array's name as a device pointer: in host code it names a host-side
// stand-in).  Make that first call before any stream capture begins.
// Every call on a device uses the same array; calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on it.  Nothing
// in the array has to start at zero: every h row is written before it is read.
#include <mutex>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_ffn_scratch[MOE_NOALLOC_FFN_SCRATCH_BYTES];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_ffn_scratch on the current device (looked up once).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_ffn_scratch);
    if (err != cudaSuccess) return err;
    if (ptr == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" int moe_expert_ffn_grouped_noalloc(const moe_cache* cache, int layer, const int32_t* counts,
                                              const int32_t* offsets, const int32_t* perm, const void* x,
                                              const void* x_perm_opt, int T, int k,
                                              const uint8_t* expert_mask_opt, int ffn_mode, float* y_rows,
                                              uint32_t* dev_status, moe_stream_t stream) {
  if (!cache || T < 0 || k < 1) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const size_t need = moe_expert_ffn_workspace_size(T, k, cache->E, cache->H, cache->I, ffn_mode);
  if (need > (size_t)MOE_NOALLOC_FFN_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (moe::scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_expert_ffn_grouped(cache, layer, counts, offsets, perm, x, x_perm_opt, T, k, expert_mask_opt, ffn_mode,
                                y_rows, scratch, (size_t)MOE_NOALLOC_FFN_SCRATCH_BYTES, dev_status, stream);
}
