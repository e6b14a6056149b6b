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
  // h, then the grid-barrier words and the per-instance counters of the fused GEMV
  return align_up(R * I * sizeof(__nv_bfloat16), 256) + align_up((4 + R) * sizeof(unsigned int), 256);
}

cudaError_t launch_ffn(const moe_cache& c, int layer, const int32_t* counts, const int32_t* offsets,
                       const int32_t* perm, const __nv_bfloat16* x, const __nv_bfloat16* x_perm,
                       int T, int k, const uint8_t* mask, int mode, float* y_rows, void* ws,
                       uint32_t* status, cudaStream_t s, const int32_t* fused_fills,
                       const int32_t* fused_n_fill, const float* combine_w, __nv_bfloat16* combine_out,
                       __nv_bfloat16* y_rows_bf16) {
  if (T == 0) return cudaSuccess;
  const int R = T * k;
  __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(ws);
  // groups above gemv_max run on the tensor-core GEMM; the rest on the GEMV
  int gemv_max = INT_MAX;
  if (mode == MOE_FFN_GEMM) {
    if (!gemm_shape_ok(c.H, c.I) || !x_perm) return cudaErrorNotSupported;
    gemv_max = 0;
  } else if (mode == MOE_FFN_AUTO && x_perm && gemm_shape_ok(c.H, c.I) && T > kGemvMaxRows) {
    // the GEMM pads a group only to 16 token rows, so it takes small groups too
    gemv_max = 0;
  }
  // A host-resident staging pool is read with plain loads only: the kernels
  // below take the cache pool's experts, and a plain GEMV pass the staged ones.
  const bool host_stage = c.staging.w_gate != nullptr && c.staging.host != 0;
  // bf16 expert rows are written by the GEMM only
  if (y_rows_bf16 != nullptr && (gemv_max != 0 || host_stage)) return cudaErrorNotSupported;
  // a fused fill or combine is only done by the fused GEMV kernel, over every expert
  if ((fused_fills != nullptr || combine_out != nullptr) && (gemv_max != INT_MAX || host_stage))
    return cudaErrorNotSupported;
  if (combine_out != nullptr && !gemv_fused_ok(c.H, c.I)) return cudaErrorNotSupported;
  if (gemv_max > 0) {
    GemvParams p = {};
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
    p.max_rows = gemv_max;
    p.h = h;
    p.y = y_rows;
    p.status = status;
    p.fills = fused_fills;
    p.n_fill = fused_n_fill;
    p.combine_w = combine_w;
    p.combine_out = combine_out;
    p.grid_count = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(ws) +
                                                   align_up((size_t)R * c.I * sizeof(__nv_bfloat16), 256));
    p.inst_done = R <= kMaxFusedInst ? p.grid_count + 4 : nullptr;
    p.pool_filter = host_stage ? kPoolDeviceOnly : kPoolAll;
    cudaError_t err = launch_gemv(p, s);
    if (err != cudaSuccess) return err;
  }
  if (gemv_max != INT_MAX) {
    cudaError_t err = launch_gemm(c, layer, counts, offsets, perm, mask, gemv_max, x_perm, T, R, h, y_rows,
                                  y_rows_bf16, status, s);
    if (err != cudaSuccess) return err;
  }
  if (host_stage) {
    // the staged experts, every group size, on the plain-load GEMV (h and y rows disjoint from the pass above)
    GemvParams q = {};
    q.c = c;
    q.layer = layer;
    q.E = c.E;
    q.H = c.H;
    q.I = c.I;
    q.k = k;
    q.T = T;
    q.counts = counts;
    q.offsets = offsets;
    q.perm = perm;
    q.x = x;
    q.x_perm = x_perm;
    q.mask = mask;
    q.max_rows = INT_MAX;
    q.h = h;
    q.y = y_rows;
    q.status = status;
    q.pool_filter = kPoolStagingOnly;
    return launch_gemv_plain(q, s);
  }
  return cudaSuccess;
}

}  // namespace moe
