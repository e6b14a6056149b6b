// Gate-weighted combine (FreeToken paper, section 3.2: the partial sums of
// the GPU execution set and of the in-place set merge into the exact layer
// output; Figure 2).  Every routed row's expert output sits in one
// token-major y_rows buffer (row t*k + j), whichever pool served the expert,
// so the merge is one fixed-order sum per token over k contiguous rows:
//   out[t, :] = sum_{j = 0..k-1} w[t, j] * y_rows[t*k + j, :]
// in ascending expert order, sequential fp32 FMAs, no atomics.  HBM-bound:
// a work item is (token, 1024 columns); each thread owns 4 consecutive
// columns and has the k row loads (16 bytes each) in flight together.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk4 = kThreads;   // float4 columns per work item

template <int KM>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const float* __restrict__ y_rows, const float* __restrict__ topk_w, int T, int k, int H,
               __nv_bfloat16* __restrict__ out, float* __restrict__ out_f32) {
  pdl_wait();
  pdl_trigger();
  const int H4 = H >> 2;
  const int chunks = (H4 + kChunk4 - 1) / kChunk4;
  const long long items = (long long)T * chunks;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int t = (int)(it / chunks);
    const int c4 = (int)(it % chunks) * kChunk4 + threadIdx.x;
    if (c4 >= H4) continue;
    const float4* rows = reinterpret_cast<const float4*>(y_rows + (size_t)t * k * H) + c4;
    float wv[KM];
    float4 yv[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        wv[j] = __ldg(topk_w + (size_t)t * k + j);
        yv[j] = __ldcs(rows + (size_t)j * H4);
      }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        acc.x = fmaf(wv[j], yv[j].x, acc.x);
        acc.y = fmaf(wv[j], yv[j].y, acc.y);
        acc.z = fmaf(wv[j], yv[j].z, acc.z);
        acc.w = fmaf(wv[j], yv[j].w, acc.w);
      }
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

cudaError_t launch_combine(const float* y_rows, const float* topk_w, int T, int k, int H, __nv_bfloat16* out,
                           float* out_f32, uint32_t* status, cudaStream_t s) {
  (void)status;
  if (T == 0) return cudaSuccess;
  const long long items = (long long)T * ((H / 4 + kChunk4 - 1) / kChunk4);
  long long blocks = items;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (k <= 8) return launch_k(combine_kernel<8>, (int)blocks, kThreads, 0, s, y_rows, topk_w, T, k, H, out, out_f32);
  return launch_k(combine_kernel<kMaxK>, (int)blocks, kThreads, 0, s, y_rows, topk_w, T, k, H, out, out_f32);
}

}  // namespace moe
