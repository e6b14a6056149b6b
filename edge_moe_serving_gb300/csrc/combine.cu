// Gate-weighted combine (FreeToken paper, section 3.2: the partial sums of
// the GPU execution set and of the in-place set merge into the exact layer
// output; Figure 2).  Every routed row's expert output sits in one
// token-major y_rows buffer (row t*k + j), whichever pool served the expert,
// so the merge is one fixed-order sum per token over k contiguous rows:
//   out[t, :] = sum_{j = 0..k-1} w[t, j] * y_rows[t*k + j, :]
// in ascending expert order, sequential fp32 FMAs, no atomics.  HBM-bound:
// a work item is (token, 1024 columns); each thread owns 4 consecutive
// columns and has the k row loads in flight together.  The rows are fp32, or
// bf16 when the layer keeps them internally (half the bytes written and read).
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk4 = kThreads;   // float4 columns per work item

__device__ inline float4 load_row4(const float* rows, size_t i) {
  return __ldcs(reinterpret_cast<const float4*>(rows) + i);
}
__device__ inline float4 load_row4(const __nv_bfloat16* rows, size_t i) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(rows) + i);
  return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

template <int KM, typename YT>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const YT* __restrict__ y_rows, const float* __restrict__ topk_w, int T, int k, int H,
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
    const YT* rows = y_rows + (size_t)t * k * H;
    float wv[KM];
    float4 yv[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        wv[j] = __ldg(topk_w + (size_t)t * k + j);
        yv[j] = load_row4(rows, (size_t)j * H4 + c4);
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

template <typename YT>
cudaError_t launch_combine_t(const YT* y_rows, const float* topk_w, int T, int k, int H, __nv_bfloat16* out,
                             float* out_f32, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const long long items = (long long)T * ((H / 4 + kChunk4 - 1) / kChunk4);
  long long blocks = items;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (k <= 8)
    return launch_k(combine_kernel<8, YT>, (int)blocks, kThreads, 0, s, y_rows, topk_w, T, k, H, out, out_f32);
  return launch_k(combine_kernel<kMaxK, YT>, (int)blocks, kThreads, 0, s, y_rows, topk_w, T, k, H, out, out_f32);
}

}  // namespace

cudaError_t launch_combine(const float* y_rows, const float* topk_w, int T, int k, int H, __nv_bfloat16* out,
                           float* out_f32, uint32_t* status, cudaStream_t s) {
  (void)status;
  return launch_combine_t(y_rows, topk_w, T, k, H, out, out_f32, s);
}

cudaError_t launch_combine(const __nv_bfloat16* y_rows, const float* topk_w, int T, int k, int H,
                           __nv_bfloat16* out, float* out_f32, uint32_t* status, cudaStream_t s) {
  (void)status;
  return launch_combine_t(y_rows, topk_w, T, k, H, out, out_f32, s);
}

}  // namespace moe
