// Pieces shared by the one-launch decode kernels (bf16 experts in
// decode_layer.cu, FP4 experts in ffn_mxfp4_ring.cu): the router rows every
// CTA scores, and the bounded grid-wide barrier that publishes the logits
// (FreeToken paper, section 3.2: the router runs on the GPU per MoE layer).
#pragma once

#include "ring_gemv.cuh"

namespace moe {
namespace {

constexpr int kDecMaxT = 8;        // token rows a decode CTA scores
constexpr int kDecMaxRows = 4;     // router rows per CTA
constexpr int kDecMaxSlots = 1024; // cache-pool slots whose state the decision copies

// Bounded grid-wide barrier: the CTA barrier orders every thread's stores
// before thread 0's release arrival (release is cumulative), and thread 0's
// acquire poll orders the other CTAs' stores before the closing CTA barrier.
__device__ inline bool grid_barrier(unsigned int* count, volatile int* abort_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
    unsigned long long t0 = 0;
    for (uint32_t it = 0; ld_acquire_u32(count) < gridDim.x; ++it) {
      if ((it & 15) == 15) {
        if (*abort_flag) break;
        const unsigned long long now = gtimer();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > kGridWaitNs) {
          *abort_flag = 1;
          break;
        }
      }
    }
  }
  __syncthreads();
  return !*abort_flag;
}

// Logits of this CTA's R router rows (rows b, b + G, ..., fp32, in wrow) for
// the T <= TT token rows (bf16, in xs): every thread takes the float4 columns
// tid, tid + blockDim, ... of all R x T dot products, then warp sums and a
// sum over the NW warps (red: [NW][kDecMaxRows][kDecMaxT] of shared memory).
// R and TT are compile-time so the loop body carries no per-row or per-token
// branch.  logits[t * E + b + i * G] = sum + bias_sh[i].
template <int R, int TT, int NW>
__device__ inline void router_rows_block(const float* wrow, const __nv_bfloat16* xs, int H, int T, int E,
                                         float (*red)[kDecMaxRows][kDecMaxT], const float* bias_sh, float* logits,
                                         int b, int G) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float acc[R][TT];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[i][t] = 0.0f;
  const int H4 = H >> 2;
  for (int q = tid; q < H4; q += blockDim.x) {
    float4 xv[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const uint2 u = (TT == 1 || t < T) ? reinterpret_cast<const uint2*>(xs + (size_t)t * H)[q] : make_uint2(0u, 0u);
      xv[t] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const float4 w = reinterpret_cast<const float4*>(wrow + (size_t)i * H)[q];
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        float a = acc[i][t];
        a = fmaf(w.x, xv[t].x, a);
        a = fmaf(w.y, xv[t].y, a);
        a = fmaf(w.z, xv[t].z, a);
        a = fmaf(w.w, xv[t].w, a);
        acc[i][t] = a;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const float s = warp_sum(acc[i][t]);
      if (lane == 0) red[warp][i][t] = s;
    }
  __syncthreads();
  if (tid < R * T) {
    const int i = tid / T, t = tid - (tid / T) * T;
    float s = 0.0f;
    for (int w = 0; w < NW; ++w) s += red[w][i][t];
    logits[(size_t)t * E + b + i * G] = s + bias_sh[i];
  }
}

}  // namespace
}  // namespace moe
