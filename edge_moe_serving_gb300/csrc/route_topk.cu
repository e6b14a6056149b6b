// Router scoring + warp top-k + renormalisation (FreeToken paper, section 3.2:
// the router runs per MoE layer on the GPU and selects the active experts).
//
// Two kernels, chosen by T:
//  * T <= 32 (decode): one CTA per expert streams that expert's fp32 router
//    row once and dots it with every token (the router weights are the only
//    bytes of the step besides the experts).  Up to 4 tokens the last CTA to
//    finish (ticket counter) runs the top-k for all tokens; 5..32 tokens take
//    one pass with a per-token partial sum in every thread, then one warp per
//    token selects.
//  * T > 32 (prefill): the tensor-core router of route_tc.cu when H is a
//    multiple of 64; otherwise a register-blocked fp32 SIMT GEMM where a CTA
//    owns 32 tokens x all E experts, so the top-k runs in its epilogue from
//    shared memory.
// Accumulation is fp32 (bf16 x is exact in fp32).  Top-k order is (logit
// descending, id ascending); ids are written ascending.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kSmallT = 32;
constexpr int kSmallThreads = 256;

// ---------------------------------------------------------------- decode path
// TOPK = false: only the logits are written (the decode front end selects).
template <int NT, bool TOPK>
__global__ void __launch_bounds__(kSmallThreads)
route_small_kernel(const __nv_bfloat16* __restrict__ x, int T, int H,
                   const float* __restrict__ w_router, const float* __restrict__ bias, int E,
                   int k, float* __restrict__ logits, unsigned int* __restrict__ ticket,
                   int32_t* __restrict__ topk_ids, float* __restrict__ topk_w) {
  __shared__ float red[kSmallThreads / 32][NT];
  __shared__ bool is_last;
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float4* wrow = reinterpret_cast<const float4*>(w_router + (size_t)e * H);
  const int H4 = H >> 2;
  for (int t0 = 0; t0 < T; t0 += NT) {
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    for (int h4 = tid; h4 < H4; h4 += kSmallThreads) {
      const float4 w = __ldg(wrow + h4);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t0 + t < T) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + t) * H) + h4);
          float a = acc[t];
          a = fmaf(w.x, bf16_lo(xv.x), a);
          a = fmaf(w.y, bf16_hi(xv.x), a);
          a = fmaf(w.z, bf16_lo(xv.y), a);
          a = fmaf(w.w, bf16_hi(xv.y), a);
          acc[t] = a;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float s = warp_sum(acc[t]);
      if (lane == 0) red[warp][t] = s;
    }
    __syncthreads();
    if (tid < NT && t0 + tid < T) {
      float s = 0.0f;
#pragma unroll
      for (int w = 0; w < kSmallThreads / 32; ++w) s += red[w][tid];
      if (bias) s += bias[e];
      logits[(size_t)(t0 + tid) * E + e] = s;
    }
    __syncthreads();
  }
  if (!TOPK) return;
  // last CTA to finish runs the top-k for every token
  __threadfence();
  if (tid == 0) {
    const unsigned int n = atomicAdd(ticket, 1u);
    is_last = (n == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int t = warp; t < T; t += kSmallThreads / 32) {
    // logits written by other CTAs: read them through L2
    float* row = logits + (size_t)t * E;
    __shared__ float srow[kSmallThreads / 32][kMaxRouteE];
    for (int j = lane; j < E; j += 32) srow[warp][j] = __ldcg(row + j);
    __syncwarp();
    warp_topk(srow[warp], E, k, topk_ids + (size_t)t * k, topk_w + (size_t)t * k);
    __syncwarp();
  }
  if (tid == 0) *ticket = 0u;  // ready for the next call
}

// 4 < T <= 32 tokens, logits only: one CTA per expert streams its fp32 router
// row once, and every thread keeps one partial sum per token.  A butterfly
// across the warp transposes and reduces the 32 partial sums in 31 shuffles
// (lane t ends with token t's warp sum); the warps' sums add up in shared
// memory.  One pass over the row for all tokens.
__global__ void __launch_bounds__(kSmallThreads)
route_wide_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, const float* __restrict__ w_router,
                  const float* __restrict__ bias, int E, float* __restrict__ logits) {
  __shared__ float red[kSmallThreads / 32][32];
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float4* wrow = reinterpret_cast<const float4*>(w_router + (size_t)e * H);
  const int H4 = H >> 2;
  float acc[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) acc[t] = 0.0f;
  for (int h4 = tid; h4 < H4; h4 += kSmallThreads) {
    const float4 w = __ldg(wrow + h4);
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      if (t < T) {
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)t * H) + h4);
        float a = acc[t];
        a = fmaf(w.x, bf16_lo(xv.x), a);
        a = fmaf(w.y, bf16_hi(xv.x), a);
        a = fmaf(w.z, bf16_lo(xv.y), a);
        a = fmaf(w.w, bf16_hi(xv.y), a);
        acc[t] = a;
      }
    }
  }
  // at offset o the lanes whose bit o is set keep the upper half of the 2o live sums
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? acc[i] : acc[i + o];
      const float keep = upper ? acc[i + o] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  red[warp][lane] = acc[0];
  __syncthreads();
  if (tid < T) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kSmallThreads / 32; ++w) s += red[w][tid];
    if (bias) s += bias[e];
    logits[(size_t)tid * E + e] = s;
  }
}

// ---------------------------------------------------------------- prefill path
constexpr int kLT = 32;     // tokens per CTA
constexpr int kLE = 256;    // experts per pass
constexpr int kLK = 32;     // H per k-step
constexpr int kLThreads = 128;

__global__ void __launch_bounds__(kLThreads)
route_large_kernel(const __nv_bfloat16* __restrict__ x, int T, int H,
                   const float* __restrict__ w_router, const float* __restrict__ bias, int E,
                   int k, float* __restrict__ logits_opt, int32_t* __restrict__ topk_ids,
                   float* __restrict__ topk_w) {
  extern __shared__ float smem[];
  pdl_wait();
  pdl_trigger();
  float* xs = smem;                          // [kLK][kLT]
  float* wsm = xs + kLK * kLT;               // [kLK][kLE + 4]
  float* lg = wsm + kLK * (kLE + 4);         // [kLT][E + 1]
  const int tid = threadIdx.x;
  const int ty = tid >> 5, tx = tid & 31;
  const int t_base = blockIdx.x * kLT;
  const int ldl = E + 1;

  for (int eb = 0; eb < E; eb += kLE) {
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    for (int h0 = 0; h0 < H; h0 += kLK) {
      // x tile: 32 tokens x 32 h, bf16 -> fp32, stored [h][token]
      {
        const int tok = tid >> 2, hc = (tid & 3) * 8;
        const int t = t_base + tok;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < T && h0 + hc < H) v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + h0 + hc));
        xs[(hc + 0) * kLT + tok] = bf16_lo(v.x);
        xs[(hc + 1) * kLT + tok] = bf16_hi(v.x);
        xs[(hc + 2) * kLT + tok] = bf16_lo(v.y);
        xs[(hc + 3) * kLT + tok] = bf16_hi(v.y);
        xs[(hc + 4) * kLT + tok] = bf16_lo(v.z);
        xs[(hc + 5) * kLT + tok] = bf16_hi(v.z);
        xs[(hc + 6) * kLT + tok] = bf16_lo(v.w);
        xs[(hc + 7) * kLT + tok] = bf16_hi(v.w);
      }
      // W tile: 256 experts x 32 h fp32, stored [h][expert]
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int el = (tid >> 3) + 16 * i;
        const int hc = (tid & 7) * 4;
        const int e = eb + el;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < E && h0 + hc < H) v = __ldg(reinterpret_cast<const float4*>(w_router + (size_t)e * H + h0 + hc));
        wsm[(hc + 0) * (kLE + 4) + el] = v.x;
        wsm[(hc + 1) * (kLE + 4) + el] = v.y;
        wsm[(hc + 2) * (kLE + 4) + el] = v.z;
        wsm[(hc + 3) * (kLE + 4) + el] = v.w;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kLK; ++kk) {
        const float4 xa = *reinterpret_cast<const float4*>(xs + kk * kLT + ty * 8);
        const float4 xb = *reinterpret_cast<const float4*>(xs + kk * kLT + ty * 8 + 4);
        const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        float wv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) wv[j] = wsm[kk * (kLE + 4) + tx + 32 * j];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = eb + tx + 32 * j;
        if (e < E) lg[(ty * 8 + i) * ldl + e] = acc[i][j] + (bias ? bias[e] : 0.0f);
      }
  }
  __syncthreads();
  const int warp = tid >> 5;
  for (int tl = warp; tl < kLT; tl += kLThreads / 32) {
    const int t = t_base + tl;
    if (t >= T) break;
    if (logits_opt)
      for (int e = tid & 31; e < E; e += 32) logits_opt[(size_t)t * E + e] = lg[tl * ldl + e];
    warp_topk(lg + tl * ldl, E, k, topk_ids + (size_t)t * k, topk_w + (size_t)t * k);
  }
}

size_t large_smem(int E) {
  return sizeof(float) * ((size_t)kLK * kLT + (size_t)kLK * (kLE + 4) + (size_t)kLT * (E + 1));
}

}  // namespace

size_t route_ws_bytes(int T, int H, int E) {
  if (T <= kSmallT) return align_up((size_t)T * E * sizeof(float), 256) + 256;
  if (route_tc_ok(T, H, E)) return route_tc_ws_bytes(T, H, E);
  return 0;
}

cudaError_t launch_route_topk(const __nv_bfloat16* x, int T, int H, const float* w_router,
                              const float* bias, int E, int k, int32_t* topk_ids, float* topk_w,
                              float* logits_opt, void* ws, uint32_t* status, cudaStream_t s) {
  (void)status;
  if (T == 0) return cudaSuccess;
  if (T <= kSmallT) {
    float* logits = logits_opt ? logits_opt : reinterpret_cast<float*>(ws);
    unsigned int* ticket = reinterpret_cast<unsigned int*>(
        reinterpret_cast<char*>(ws) + align_up((size_t)T * E * sizeof(float), 256));
    cudaError_t err = cudaSuccess;
    if (T <= 4) {
      err = cudaMemsetAsync(ticket, 0, sizeof(unsigned int), s);
      if (err != cudaSuccess) return err;
    }
    if (T <= 1)
      return launch_k(route_small_kernel<1, true>, E, kSmallThreads, 0, s, x, T, H, w_router, bias, E, k, logits,
                      ticket, topk_ids, topk_w);
    if (T <= 4)
      return launch_k(route_small_kernel<4, true>, E, kSmallThreads, 0, s, x, T, H, w_router, bias, E, k, logits,
                      ticket, topk_ids, topk_w);
    // more tokens: logits only, then one warp per token selects
    err = launch_k(route_wide_kernel, E, kSmallThreads, 0, s, x, T, H, w_router, bias, E, logits);
    if (err != cudaSuccess) return err;
    return launch_topk(logits, nullptr, T, E, k, false, topk_ids, topk_w, s);
  }
  if (route_tc_ok(T, H, E))
    return launch_route_tc(x, T, H, w_router, bias, E, k, topk_ids, topk_w, logits_opt, ws, status, s);
  const size_t smem = large_smem(E);
  static std::atomic<unsigned char> attr[kMaxDevices];
  {
    cudaError_t err = once_per_device(attr, [] {
      return cudaFuncSetAttribute(route_large_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)large_smem(kMaxRouteE));
    });
    if (err != cudaSuccess) return err;
  }
  const int grid = (T + kLT - 1) / kLT;
  return launch_k(route_large_kernel, grid, kLThreads, smem, s, x, T, H, w_router, bias, E, k, logits_opt, topk_ids,
                  topk_w);
}

// Logits only, T <= 32 (the decode front end does the selection).
cudaError_t launch_route_logits(const __nv_bfloat16* x, int T, int H, const float* w_router, const float* bias,
                                int E, float* logits, cudaStream_t s) {
  if (T <= 1)
    return launch_k(route_small_kernel<1, false>, E, kSmallThreads, 0, s, x, T, H, w_router, bias, E, 1, logits,
                    (unsigned int*)nullptr, (int32_t*)nullptr, (float*)nullptr);
  if (T <= 4)
    return launch_k(route_small_kernel<4, false>, E, kSmallThreads, 0, s, x, T, H, w_router, bias, E, 1, logits,
                    (unsigned int*)nullptr, (int32_t*)nullptr, (float*)nullptr);
  return launch_k(route_wide_kernel, E, kSmallThreads, 0, s, x, T, H, w_router, bias, E, logits);
}

}  // namespace moe
