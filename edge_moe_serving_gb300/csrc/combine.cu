// Gate-weighted combine (FreeToken paper, section 3.2: the partial sums of
// the GPU execution set and of the in-place set merge into the exact layer
// output; Figure 2).  Every routed row's expert output sits in one y_rows
// buffer at its dispatch position, whichever pool served the expert, so the
// merge is one fixed-order sum per token:
//   out[t, :] = sum_{j = 0..k-1} w[t, j] * y_rows[inv_perm[t*k + j], :]
// in ascending expert order, sequential fp32 FMAs, no atomics.  HBM-bound:
// each thread owns 4 consecutive columns (16-byte loads of y).
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
combine_kernel(const float* __restrict__ y_rows, const int32_t* __restrict__ inv_perm,
               const float* __restrict__ topk_w, int T, int k, int H, __nv_bfloat16* __restrict__ out,
               float* __restrict__ out_f32) {
  const int H4 = H >> 2;
  const long long total = (long long)T * H4;
  for (long long idx = (long long)blockIdx.x * kThreads + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * kThreads) {
    const int t = (int)(idx / H4);
    const int c4 = (int)(idx % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float w = __ldg(topk_w + (size_t)t * k + j);
      const int pos = __ldg(inv_perm + (size_t)t * k + j);
      const float4 y = __ldcs(reinterpret_cast<const float4*>(y_rows + (size_t)pos * H) + c4);
      acc.x = fmaf(w, y.x, acc.x);
      acc.y = fmaf(w, y.y, acc.y);
      acc.z = fmaf(w, y.z, acc.z);
      acc.w = fmaf(w, y.w, acc.w);
    }
    if (out) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(out + (size_t)t * H)[c4] = packed;
    }
    if (out_f32) reinterpret_cast<float4*>(out_f32 + (size_t)t * H)[c4] = acc;
  }
}

}  // namespace

cudaError_t launch_combine(const float* y_rows, const int32_t* inv_perm, const float* topk_w, int T,
                           int k, int H, __nv_bfloat16* out, float* out_f32, uint32_t* status,
                           cudaStream_t s) {
  (void)status;
  if (T == 0) return cudaSuccess;
  const long long total = (long long)T * (H / 4);
  long long blocks = (total + kThreads - 1) / kThreads;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  combine_kernel<<<(int)blocks, kThreads, 0, s>>>(y_rows, inv_perm, topk_w, T, k, H, out, out_f32);
  return cudaGetLastError();
}

}  // namespace moe
