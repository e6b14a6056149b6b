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
// The first call in each CUDA context (in practice: on each device, and again
// after that device was reset) looks up the array's device address with
// cudaGetSymbolAddress while that device is current; host code cannot use the
// array's name as a device pointer, since in host code it names a host-side
// stand-in.  Make that first call before any stream capture begins.  Every
// call on a device uses the same array; calls whose kernels overlap on the
// GPU (different streams, no ordering between them) race on it.  Nothing in
// the array has to start at zero: every h row is written before it is read.
#include <cuda.h>

#include <mutex>

#include "moe_common.cuh"

namespace moe {
namespace {

static __device__ __align__(256) unsigned char g_ffn_scratch[MOE_NOALLOC_FFN_SCRATCH_BYTES];

// The driver calls that name the current context, fetched through the
// runtime (no link-time dependency on the driver library).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn current = nullptr;
  CtxGetIdFn id = nullptr;
};

const CtxFns& ctx_fns() {
  static const CtxFns fns = [] {
    CtxFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.id = reinterpret_cast<CtxGetIdFn>(p);
    return f;
  }();
  return fns;
}

// Unique id of the calling thread's current context, 0 if there is none or
// it cannot be read.  A device reset destroys the context; the next one
// gets a new id.
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!f.current || !f.id || f.current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  return f.id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

struct ScratchEntry {
  void* ptr = nullptr;
  unsigned long long ctx = 0;   // context the address belongs to
};

std::mutex g_setup_mutex;
ScratchEntry g_scratch[kMaxDevices];

// Device address of g_ffn_scratch in the current device's context: looked
// up once per context, so that an address cached before a device reset is
// never handed to a kernel of the next context.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchEntry& s = g_scratch[dev];
  const unsigned long long ctx = current_ctx_id();
  if (s.ptr == nullptr || ctx == 0 || s.ctx != ctx) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_ffn_scratch);   // makes the device's context current if needed
    if (err != cudaSuccess) return err;
    if (ptr == nullptr) return cudaErrorInvalidSymbol;
    s.ptr = ptr;
    s.ctx = current_ctx_id();
  }
  *out = s.ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" int moe_expert_ffn_grouped_noalloc(const moe_cache* cache, int layer, const int32_t* counts,
                                              const int32_t* offsets, const int32_t* perm, const void* x,
                                              const void* x_perm_opt, int T, int k,
                                              const uint8_t* expert_mask_opt, int ffn_mode, float* y_rows,
                                              uint32_t* dev_status, moe_stream_t stream) {
  // the ordinary call's argument checks first, so an invalid call reports what is invalid
  const int st = moe::ffn_check_args(cache, layer, counts, offsets, perm, x, x_perm_opt, T, k, ffn_mode, y_rows);
  if (st != MOE_OK || T == 0) return st;
  const size_t need = moe_expert_ffn_workspace_size(T, k, cache->E, cache->H, cache->I, ffn_mode);
  if (need > (size_t)MOE_NOALLOC_FFN_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (moe::scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_expert_ffn_grouped(cache, layer, counts, offsets, perm, x, x_perm_opt, T, k, expert_mask_opt, ffn_mode,
                                y_rows, scratch, (size_t)MOE_NOALLOC_FFN_SCRATCH_BYTES, dev_status, stream);
}
