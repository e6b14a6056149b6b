// Router scoring on the tensor cores for prefill-sized T (FreeToken paper,
// section 3.2: the router scores every expert for every token of the layer).
//
// The router weights are fp32 and the tokens bf16.  Every fp32 weight w is
// the exact sum of three bf16 numbers (hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid): 8 + 8 + 8 significand bits cover fp32's 24), and a
// bf16 x bf16 product is exact in fp32, so
//     logit[t, e] = sum_h x[t,h] (hi[e,h] + mid[e,h] + lo[e,h])
// is one bf16 GEMM with fp32 accumulation over K = 3H, where the token
// operand is the same x row read three times (TMA coordinate k mod H).
//
//   split_kernel   W3[e, :] = [hi(W_r[e,:]) | mid(...) | lo(...)]   bf16 [E, 3H]
//   logits_kernel  logits^T tile (128 experts x 128 tokens) = W3 x^T on tcgen05
//                  (persistent, one CTA per SM, 6-stage TMA ring, fp32 logits
//                  to [T, E])
//   topk_kernel    one warp per token: + bias, top-k (logit desc, id asc),
//                  softmax renormalised over the selection, ids ascending
//
// The tensor core adds into its fp32 accumulator without rounding to
// nearest, which over K = 3H = 12288 biases a logit towards zero by about
// 2e-5 relative.  The K range is therefore cut into kParts contiguous parts,
// each accumulated in its own TMEM columns, and the epilogue adds the parts
// in fp32 with round-to-nearest: fewer steps per accumulator, each of smaller
// magnitude.
//
// Every mbarrier wait is bounded; on expiry the CTA sets MOE_DEV_ERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and returns.
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kRM = 128;                      // experts per tile (MMA M)
constexpr int kRN = 128;                      // tokens per tile (MMA N)
constexpr int kRStages = 6;
constexpr int kRATile = kRM * kBK * 2;        // 16 KB
constexpr int kRBTile = kRN * kBK * 2;        // 16 KB
constexpr int kRStage = kRATile + kRBTile;
constexpr int kRSmem = kRStages * kRStage + 1024;
constexpr int kRThreads = 192;
constexpr int kParts = 4;                     // K parts, one TMEM accumulator each
constexpr int kRTmemCols = kParts * kRN;

__global__ void __launch_bounds__(256)
split_kernel(const float* __restrict__ w, int E, int H, __nv_bfloat16* __restrict__ w3) {
  pdl_wait();
  pdl_trigger();
  const size_t n4 = (size_t)E * H / 4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(w) + i);
    const size_t e = (i * 4) / H, h = (i * 4) % H;
    const float a[4] = {v.x, v.y, v.z, v.w};
    unsigned short hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 b0 = __float2bfloat16_rn(a[j]);
      const float r1 = a[j] - __bfloat162float(b0);
      const __nv_bfloat16 b1 = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(b1);
      hi[j] = __bfloat16_as_ushort(b0);
      mid[j] = __bfloat16_as_ushort(b1);
      lo[j] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
    }
    unsigned short* row = reinterpret_cast<unsigned short*>(w3) + e * 3 * H + h;
    *reinterpret_cast<uint2*>(row) = make_uint2(hi[0] | (uint32_t)hi[1] << 16, hi[2] | (uint32_t)hi[3] << 16);
    *reinterpret_cast<uint2*>(row + H) = make_uint2(mid[0] | (uint32_t)mid[1] << 16, mid[2] | (uint32_t)mid[3] << 16);
    *reinterpret_cast<uint2*>(row + 2 * H) = make_uint2(lo[0] | (uint32_t)lo[1] << 16, lo[2] | (uint32_t)lo[3] << 16);
  }
}

struct LogitParams {
  int T, E, H;
  int n_mt, n_tiles;
  float* logits;     // [T, E]
  uint32_t* status;
};

__global__ void __launch_bounds__(kRThreads, 1)
logits_kernel(const __grid_constant__ CUtensorMap map_w3, const __grid_constant__ CUtensorMap map_x,
              const LogitParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kRStages], empty_bar[kRStages], tmem_full, tmem_empty, drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kIdesc = make_idesc(kRM, kRN);

  if (tid == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tmem_full, 1);
    mbar_init(&tmem_empty, 128);
    mbar_init(&drain_bar, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                 "r"(kRTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort_flag = &s_abort;
  const int kb_count = 3 * p.H / kBK;
  const int kb_h = p.H / kBK;
  const int nparts = min(kParts, kb_count);   // every part gets at least one k-block

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool armed[kRStages] = {};
      uint32_t armed_parity[kRStages] = {};
      for (int t = blockIdx.x; t < p.n_tiles && !*abort_flag; t += gridDim.x) {
        const int mt = t % p.n_mt, tc_ = t / p.n_mt;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) break;
          uint8_t* sA = smem + stage * kRStage;
          mbar_expect_tx(&full_bar[stage], kRStage);
          armed[stage] = true;
          armed_parity[stage] = phase;
          tma_load_2d(sA, &map_w3, &full_bar[stage], kb * kBK, mt * kRM);
          tma_load_2d(sA + kRATile, &map_x, &full_bar[stage], (kb % kb_h) * kBK, tc_ * kRN);
          if (++stage == kRStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      volatile int no_abort = 0;
      for (int s = 0; s < kRStages; ++s)
        if (armed[s]) mbar_wait(&full_bar[s], armed_parity[s], &no_abort);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, tphase = 0;
      bool issued = false;
      for (int t = blockIdx.x; t < p.n_tiles && !*abort_flag; t += gridDim.x) {
        if (!mbar_wait(&tmem_empty, tphase ^ 1u, abort_flag)) break;
        tc_fence_after();
        bool good = true;
        int prev_part = -1;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
            good = false;
            break;
          }
          tc_fence_after();
          const int part = kb * nparts / kb_count;
          const uint32_t d = tmem_base + part * kRN;
          const bool first = part != prev_part;
          prev_part = part;
          const uint32_t a0 = smem_u32(smem + stage * kRStage);
#pragma unroll
          for (int ks = 0; ks < kBK / kUK; ++ks)
            tc_mma(d, smem_desc(a0 + ks * kUK * 2), smem_desc(a0 + kRATile + ks * kUK * 2), kIdesc,
                   (!first || ks > 0) ? 1u : 0u);
          issued = true;
          tc_commit(&empty_bar[stage]);
          if (++stage == kRStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!good) break;
        tc_commit(&tmem_full);
        tphase ^= 1u;
      }
      if (issued) {
        volatile int no_abort = 0;
        tc_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, &no_abort);
      }
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    uint32_t tphase = 0;
    for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
      const int mt = t % p.n_mt, tc_ = t / p.n_mt;
      if (!mbar_wait(&tmem_full, tphase, abort_flag)) break;
      tphase ^= 1u;
      tc_fence_after();
      const int e = mt * kRM + quarter * 32 + lane;
      const uint32_t addr = tmem_base + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < kRN; c += 32) {
        uint32_t v[32];
        float acc[32];
        tmem_ld32(addr + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(v[j]);
#pragma unroll 1
        for (int q = 1; q < nparts; ++q) {
          tmem_ld32(addr + q * kRN + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] = __fadd_rn(acc[j], __uint_as_float(v[j]));
        }
        const int t0 = tc_ * kRN + c;
        if (e < p.E) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (t0 + j < p.T) p.logits[(size_t)(t0 + j) * p.E + e] = acc[j];
        }
      }
      tc_fence_before();
      mbar_arrive(&tmem_empty);
    }
  }
  pdl_trigger();
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kRTmemCols));
}

// One warp per token.  logits holds the raw products; bias is added here and
// the biased logits are written back when write_back is set.
constexpr int kTopkWarps = 8;

__global__ void __launch_bounds__(32 * kTopkWarps)
topk_kernel(float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k, int write_back,
            int32_t* __restrict__ topk_ids, float* __restrict__ topk_w) {
  __shared__ float srow[kTopkWarps][kMaxRouteE];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = blockIdx.x * kTopkWarps + warp; t < T; t += gridDim.x * kTopkWarps) {
    float* row = logits + (size_t)t * E;
    for (int e = lane; e < E; e += 32) {
      const float v = row[e] + (bias ? bias[e] : 0.0f);
      srow[warp][e] = v;
      if (write_back) row[e] = v;
    }
    __syncwarp();
    warp_topk(srow[warp], E, k, topk_ids + (size_t)t * k, topk_w + (size_t)t * k);
    __syncwarp();
  }
}

}  // namespace

bool route_tc_ok(int T, int H, int E) { return T > 32 && H % kBK == 0 && H >= kBK && E <= kMaxRouteE; }

size_t route_tc_ws_bytes(int T, int H, int E) {
  return align_up((size_t)E * 3 * H * sizeof(__nv_bfloat16), 256) + align_up((size_t)T * E * sizeof(float), 256);
}

cudaError_t launch_route_tc(const __nv_bfloat16* x, int T, int H, const float* w_router, const float* bias, int E,
                            int k, int32_t* topk_ids, float* topk_w, float* logits_opt, void* ws, uint32_t* status,
                            cudaStream_t s) {
  static std::atomic<unsigned char> attr[kMaxDevices];
  {
    cudaError_t e = once_per_device(
        attr, [] { return cudaFuncSetAttribute(logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem); });
    if (e != cudaSuccess) return e;
  }
  __nv_bfloat16* w3 = reinterpret_cast<__nv_bfloat16*>(ws);
  float* logits = logits_opt ? logits_opt
                             : reinterpret_cast<float*>(reinterpret_cast<char*>(ws) +
                                                        align_up((size_t)E * 3 * H * sizeof(__nv_bfloat16), 256));
  const int sms = num_sms();
  const size_t n4 = (size_t)E * H / 4;
  const int sgrid = (int)std::min<size_t>((n4 + 255) / 256, (size_t)sms * 8);
  cudaError_t err = launch_k(split_kernel, sgrid, 256, 0, s, w_router, E, H, w3);
  if (err != cudaSuccess) return err;

  CUtensorMap mw, mx;
  if (!make_map(&mw, w3, 3 * (uint64_t)H, (uint64_t)E, kRM) || !make_map(&mx, x, (uint64_t)H, (uint64_t)T, kRN))
    return cudaErrorInvalidValue;
  LogitParams p;
  p.T = T;
  p.E = E;
  p.H = H;
  p.n_mt = (E + kRM - 1) / kRM;
  p.n_tiles = p.n_mt * ((T + kRN - 1) / kRN);
  p.logits = logits;
  p.status = status;
  err = launch_k(logits_kernel, std::min(p.n_tiles, sms), kRThreads, kRSmem, s, mw, mx, p);
  if (err != cudaSuccess) return err;
  return launch_topk(logits, bias, T, E, k, logits_opt != nullptr, topk_ids, topk_w, s);
}

cudaError_t launch_topk(float* logits, const float* bias, int T, int E, int k, bool write_back, int32_t* topk_ids,
                        float* topk_w, cudaStream_t s) {
  const int tgrid = std::min((T + kTopkWarps - 1) / kTopkWarps, num_sms() * 8);
  return launch_k(topk_kernel, tgrid, 32 * kTopkWarps, 0, s, logits, bias, T, E, k, write_back ? 1 : 0, topk_ids,
                  topk_w);
}

}  // namespace moe
