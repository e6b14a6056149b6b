// Parameters of the weight-streaming expert GEMV kernels.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kMaxFusedInst = 1024;   // fused launches with at most this many routed rows track instances

struct GemvParams {
  moe_cache c;
  int layer, E, H, I, k, T;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const __nv_bfloat16* x;
  const __nv_bfloat16* x_perm;
  const uint8_t* mask;
  int max_rows;       // experts with more rows are left to the GEMM kernel
  __nv_bfloat16* h;   // [R, I]
  float* y;           // [R, H]
  uint32_t* status;
  // Fused fill (optional): experts admitted to the cache by this call's bind
  // are read from the staging pool and written to their cache slot on the fly.
  const int32_t* fills;     // [n][2]: (staging slot l*E+e, cache slot)
  const int32_t* n_fill;    // device count of valid rows of `fills`
  unsigned int* grid_count; // workspace words for the fused kernel's grid barriers
  // Per-instance phase-A completion counters (zero at launch, one word per
  // instance), or null: the fused kernel then separates its phases with a
  // grid barrier.
  unsigned int* inst_done;
  // Fused combine (optional): out[t] = sum_j combine_w[t*k+j] * y[t*k+j] after the FFN.
  const float* combine_w;
  __nv_bfloat16* combine_out;
  int pool_filter;    // kPoolAll, or the pool whose experts this launch takes (host-resident staging pools)
};

// The plain-load GEMV (no bulk copies): the kernel that may read host memory.
cudaError_t launch_gemv_plain(const GemvParams& p, cudaStream_t s);


cudaError_t launch_gemv(const GemvParams& p, cudaStream_t s);

bool gemm_shape_ok(int H, int I);
cudaError_t launch_gemm(const moe_cache& c, int layer, const int32_t* counts, const int32_t* offsets,
                        const int32_t* perm, const uint8_t* mask, int min_rows, const __nv_bfloat16* x_perm,
                        int T, int R, __nv_bfloat16* h, float* y, __nv_bfloat16* y16, uint32_t* status,
                        cudaStream_t s);

}  // namespace moe
