// Grouped expert FFN over block-scaled FP4 (MXFP4) expert banks: the entry
// point, and the table-decode kernel for calls of more than one token (one-
// token calls of qualifying shapes run on the ring kernel, ffn_mxfp4_ring.cu),
// for decode-sized groups (FreeToken paper, section 5.1 "Models": the routed
// experts of DeepSeek-V4-Flash are natively MXFP4; section 4.1: the expert
// kernels dequantise in-kernel; section 3.2: grouped evaluation through the
// (layer, expert) slot).  Encoding (OCP Microscaling Formats v1.0): FP4 E2M1
// elements, one E8M0 scale per 32 consecutive inputs of a weight row, input
// 2c in the low nibble of code byte c.
//
//  gate/up  h[pos, i] = bf16( silu(Wg[i,:] . x_t) * (Wu[i,:] . x_t) )
//  down     y[perm[pos], o] = Wd[o,:] . h[pos,:]                  (fp32)
//
// Work split as in the bf16 weight-streaming GEMV: an instance is (expert e,
// chunk of up to NT of its rows) with one task per output neuron; CTA b owns
// a contiguous range of the flattened tasks, NG neurons at a time.  A thread
// owns whole 32-input blocks: one 16-byte code vector and its scale byte per
// row.  Codes decode through a byte -> bf16x2 table in shared memory,
// replicated once per lane so that every lane reads its own bank.  A block's
// 32 products are summed in fp32 and then scaled by the block's power of two
// (exact), so the result is the dot product with the dequantised row up to
// fp32 summation order.
#include <climits>

#include "mxfp4.cuh"
#include "ring_gemv.cuh"

namespace moe {
namespace {

constexpr int kMxThreadsMax = 256;

// FP4 E2M1 magnitudes by the low three code bits (the element table of the
// OCP MX specification); bit 3 is the sign.
__device__ inline float e2m1(uint32_t c) {
  const uint32_t m = c & 7u;
  float v = (m < 2u) ? 0.5f * (float)m : 0.0f;
  if (m == 2u) v = 1.0f;
  if (m == 3u) v = 1.5f;
  if (m == 4u) v = 2.0f;
  if (m == 5u) v = 3.0f;
  if (m == 6u) v = 4.0f;
  if (m == 7u) v = 6.0f;
  return (c & 8u) ? -v : v;
}

// Four code bytes (one 32-bit word: 8 inputs) -> 8 bf16 weights through the
// per-lane table.
__device__ inline uint4 mx_decode_word(const uint32_t* lut, uint32_t w, int lane) {
  uint4 r;
  r.x = lut[((w >> 0) & 0xFFu) * 32 + lane];
  r.y = lut[((w >> 8) & 0xFFu) * 32 + lane];
  r.z = lut[((w >> 16) & 0xFFu) * 32 + lane];
  r.w = lut[((w >> 24) & 0xFFu) * 32 + lane];
  return r;
}

// Dot product of one 32-input block (16 code bytes) with 32 bf16 activations.
__device__ inline float mx_block_dot(const uint32_t* lut, const uint4& q, const uint4 (&a)[4], int lane) {
  float part = 0.0f;
  part = dot8(mx_decode_word(lut, q.x, lane), a[0], part);
  part = dot8(mx_decode_word(lut, q.y, lane), a[1], part);
  part = dot8(mx_decode_word(lut, q.z, lane), a[2], part);
  part = dot8(mx_decode_word(lut, q.w, lane), a[3], part);
  return part;
}

template <int NT, int NG, bool GATEUP>
__global__ void __launch_bounds__(kMxThreadsMax)
mx_gemv_kernel(MxParams p) {
  constexpr int NR = GATEUP ? 2 : 1;
  constexpr int NV = NG * NR * NT;
  constexpr int NVP = NV < 32 ? 32 : NV;
  constexpr int PER_LANE = NVP / 32;
  __shared__ uint32_t lut[256 * 32];   // [code byte][lane]: two bf16 weights, low nibble in the low half
  __shared__ int s_pref[kMaxE + 1];
  __shared__ int s_warp[kMxThreadsMax / 32];
  __shared__ float red[2][kMxThreadsMax / 32][NVP];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int K = GATEUP ? p.H : p.I;        // inputs per weight row
  const int NTASK = GATEUP ? p.I : p.H;    // output neurons per instance
  const int KB = K / kMxBlock;             // blocks per row
  const size_t qrow = (size_t)K / 2, srow = (size_t)KB;
  const int sweeps = (KB + nthreads - 1) / nthreads;

  // table: warp w fills entries w, w + nwarps, ...; lane = copy (one bank each)
  for (int b = warp; b < 256; b += nwarps) {
    const uint32_t lo = __float_as_uint(e2m1((uint32_t)b & 15u)) >> 16;
    const uint32_t hi = __float_as_uint(e2m1((uint32_t)b >> 4)) >> 16;
    lut[b * 32 + lane] = lo | (hi << 16);
  }
  pdl_wait();
  pdl_trigger();
  build_group_prefix<NT, kMaxE / 32>(p.counts, p.E, 0, INT_MAX, nullptr, s_pref, s_warp);   // ends with __syncthreads
  const long long total = (long long)s_pref[p.E] * NTASK;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long begin = (long long)blockIdx.x * per;
  const long long end = begin + per < total ? begin + per : total;

  int buf = 0;
  for (long long tau = begin; tau < end;) {
    const int j = (int)(tau / NTASK);
    const int n0 = (int)(tau % NTASK);
    int gsize = NTASK - n0;
    if (gsize > NG) gsize = NG;
    if (end - tau < gsize) gsize = (int)(end - tau);
    const int e = find_group(s_pref, p.E, j);
    const int c = j - s_pref[e];
    const int cnt = p.counts[e];
    const int pos0 = p.offsets[e] + c * NT;
    const int ntok = min(NT, cnt - c * NT);
    MxRows rw;
    if (!mx_resolve<GATEUP>(p, p.slot_table[p.layer * p.E + e], &rw, tid == 0 ? p.status : nullptr)) {
      tau += gsize;   // uniform across the CTA: every thread skips
      continue;
    }
    const uint8_t* q0 = rw.q0 + (size_t)n0 * qrow;
    const uint8_t* s0 = rw.s0 + (size_t)n0 * srow;
    const uint8_t* q1 = rw.q1 + (size_t)n0 * qrow;
    const uint8_t* s1 = rw.s1 + (size_t)n0 * srow;
    const __nv_bfloat16* act[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int pos = pos0 + (t < ntok ? t : 0);
      act[t] = GATEUP ? p.x + (size_t)(p.perm[pos] / p.k) * p.H : p.h + (size_t)pos * p.I;
    }

    float acc[NVP];
#pragma unroll
    for (int q = 0; q < NVP; ++q) acc[q] = 0.0f;
    for (int sw = 0; sw < sweeps; ++sw) {
      const int v = sw * nthreads + tid;
      if (v < KB) {
        uint4 wq[NG][NR];
        float sc[NG][NR];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          if (g < gsize) {
            wq[g][0] = ldg_stream(q0 + (size_t)g * qrow + (size_t)v * 16);
            sc[g][0] = e8m0(__ldg(s0 + (size_t)g * srow + v));
            if (NR == 2) {
              wq[g][NR - 1] = ldg_stream(q1 + (size_t)g * qrow + (size_t)v * 16);
              sc[g][NR - 1] = e8m0(__ldg(s1 + (size_t)g * srow + v));
            }
          } else {
            wq[g][0] = make_uint4(0, 0, 0, 0);
            wq[g][NR - 1] = make_uint4(0, 0, 0, 0);
            sc[g][0] = 0.0f;
            sc[g][NR - 1] = 0.0f;
          }
        }
        uint4 a[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            a[t][i] = (t < ntok) ? ldg_cached(act[t] + (size_t)v * kMxBlock + i * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
          for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const float part = mx_block_dot(lut, wq[g][r], a[t], lane);
              acc[(g * NR + r) * NT + t] = fmaf(part, sc[g][r], acc[(g * NR + r) * NT + t]);
            }
      }
    }
    warp_reduce_scatter<NVP>(acc);
#pragma unroll
    for (int u = 0; u < PER_LANE; ++u) red[buf][warp][lane * PER_LANE + u] = acc[u];
    __syncthreads();
    for (int qi = tid; qi < NG * NT; qi += nthreads) {
      const int g = qi / NT, t = qi % NT;
      if (g < gsize && t < ntok) {
        if (GATEUP) {
          float gs = 0.0f, us = 0.0f;
          for (int w = 0; w < nwarps; ++w) {
            gs += red[buf][w][(g * 2 + 0) * NT + t];
            us += red[buf][w][(g * 2 + 1) * NT + t];
          }
          p.h[(size_t)(pos0 + t) * p.I + n0 + g] = __float2bfloat16_rn(silu(gs) * us);
        } else {
          float ys = 0.0f;
          for (int w = 0; w < nwarps; ++w) ys += red[buf][w][g * NT + t];
          p.y[(size_t)p.perm[pos0 + t] * p.H + n0 + g] = ys;
        }
      }
    }
    buf ^= 1;
    tau += gsize;
  }
}

template <typename Kern>
int mx_grid(Kern kern, int threads, std::atomic<int> (&cache)[kMaxDevices][kMxThreadsMax / 32 + 1]) {
  const int dev = device_index();
  int g = dev >= 0 ? cache[dev][threads / 32].load(std::memory_order_relaxed) : 0;
  if (g) return g;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  g = per_sm * num_sms();
  if (dev >= 0) cache[dev][threads / 32].store(g, std::memory_order_relaxed);
  return g;
}

template <int NT>
cudaError_t launch_mx_nt(const MxParams& p, cudaStream_t s) {
  constexpr int NG_UP = 2, NG_DN = 4;
  const int thr_up = std::min(kMxThreadsMax, (int)align_up((size_t)(p.H / kMxBlock), 32));
  const int thr_dn = std::min(kMxThreadsMax, (int)align_up((size_t)(p.I / kMxBlock), 32));
  static std::atomic<int> grid_up[kMaxDevices][kMxThreadsMax / 32 + 1], grid_dn[kMaxDevices][kMxThreadsMax / 32 + 1];
  const int gu = mx_grid(mx_gemv_kernel<NT, NG_UP, true>, thr_up, grid_up);
  const int gd = mx_grid(mx_gemv_kernel<NT, NG_DN, false>, thr_dn, grid_dn);
  cudaError_t err = launch_k(mx_gemv_kernel<NT, NG_UP, true>, gu, thr_up, 0, s, p);
  if (err != cudaSuccess) return err;
  return launch_k(mx_gemv_kernel<NT, NG_DN, false>, gd, thr_dn, 0, s, p);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_mx_pool(const moe_pool_mxfp4* pool) {
  if (!pool->gate_q || !pool->gate_s || !pool->up_q || !pool->up_s || !pool->down_q || !pool->down_s ||
      pool->n_slots < 1)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(pool->gate_q) || !aligned16(pool->up_q) || !aligned16(pool->down_q)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// An NVFP4 pool in the MXFP4 pool's layout (the same six banks; only the
// scale rows are twice as long) plus its tensor scales.
moe_pool_mxfp4 as_mx_pool(const moe_pool_nvfp4& n) {
  moe_pool_mxfp4 m = {};
  m.gate_q = n.gate_q;
  m.gate_s = n.gate_s;
  m.up_q = n.up_q;
  m.up_s = n.up_s;
  m.down_q = n.down_q;
  m.down_s = n.down_s;
  m.n_slots = n.n_slots;
  return m;
}

int check_nv_pool(const moe_pool_nvfp4* pool) {
  const moe_pool_mxfp4 m = as_mx_pool(*pool);
  const int st = check_mx_pool(&m);
  if (st != MOE_OK) return st;
  if (!pool->tensor_scale) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(pool->tensor_scale) & 3u) != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// h rows (bf16 [T*k, I]), the ring kernel's per-instance counters, then the
// token rows in dispatch order (bf16 [T*k, H], the tensor-core GEMM's operand)
size_t mx_ws_bytes(int T, int k, int H, int I) {
  const size_t R = (size_t)T * k;
  return align_up(R * I * sizeof(__nv_bfloat16), 256) + align_up(R * sizeof(unsigned int), 256) +
         align_up(R * H * sizeof(__nv_bfloat16), 256);
}

// Checks shared by the two FP4 entry points (the pools are checked by the
// caller), then the parameter block.
int fp4_common(const int32_t* slot_table, int n_layers, int layer, int E, int H, int I, const int32_t* counts,
               const int32_t* offsets, const int32_t* perm, const void* x, int T, int k, float* y_rows, void* ws,
               size_t ws_bytes, uint32_t* dev_status, MxParams* p) {
  if (T == 0) return MOE_OK;
  if (!counts || !offsets || !perm || !x || !y_rows) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y_rows)) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < mx_ws_bytes(T, k, H, I)) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_UNSUPPORTED;   // h rows are read as 16-byte vectors
  p->slot_table = slot_table;
  p->layer = layer;
  p->E = E;
  p->H = H;
  p->I = I;
  p->k = k;
  p->counts = counts;
  p->offsets = offsets;
  p->perm = perm;
  p->x = reinterpret_cast<const __nv_bfloat16*>(x);
  p->h = reinterpret_cast<__nv_bfloat16*>(ws);
  const size_t h_bytes = align_up((size_t)T * k * I * sizeof(__nv_bfloat16), 256);
  p->inst_done = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(ws) + h_bytes);
  p->x_perm = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<char*>(ws) + h_bytes +
                                               align_up((size_t)T * k * sizeof(unsigned int), 256));
  p->y = y_rows;
  p->status = dev_status;
  return MOE_OK;
}

int shape_check(const void* cache_pool, const int32_t* slot_table, int n_layers, int layer, int E, int H, int I, int T,
                int k, int block) {
  if (!cache_pool || !slot_table || n_layers < 1 || layer < 0 || layer >= n_layers || E < 1 || T < 0 || k < 1 ||
      k > E || k > kMaxK || H < block || I < block)
    return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || (H % block) || (I % block) || (long long)n_layers * E > MOE_SLOT_MASK ||
      (long long)T * k > INT_MAX / 2)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The tensor-core GEMM: the token rows gathered in dispatch order, then the
// gate/up and down launches.
cudaError_t run_fp4_gemm(const MxParams& p, bool nv, int T, cudaStream_t s) {
  const cudaError_t err = launch_gather(p.x, p.H, p.k, p.perm, p.offsets, p.E, T * p.k, p.x_perm, s);
  if (err != cudaSuccess) return err;
  return launch_fp4_gemm(p, nv, p.x_perm, T, s);
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_expert_ffn_mxfp4_workspace_size(int T, int k, int H, int I) {
  if (T < 0 || k < 1 || H < moe::kMxBlock || I < moe::kMxBlock || (long long)T * k > INT_MAX / 2) return 0;
  return moe::mx_ws_bytes(T, k, H, I);
}

extern "C" int moe_expert_ffn_mxfp4(const moe_pool_mxfp4* cache_pool, const moe_pool_mxfp4* staging_opt,
                                    const int32_t* slot_table, int n_layers, int layer, int E, int H, int I,
                                    const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                                    const void* x, int T, int k, float* y_rows, void* ws, size_t ws_bytes,
                                    uint32_t* dev_status, moe_stream_t stream) {
  using namespace moe;
  int st = shape_check(cache_pool, slot_table, n_layers, layer, E, H, I, T, k, kMxBlock);
  if (st != MOE_OK) return st;
  st = check_mx_pool(cache_pool);
  if (st != MOE_OK) return st;
  if (staging_opt) {
    st = check_mx_pool(staging_opt);
    if (st != MOE_OK) return st;
  }
  MxParams p = {};
  p.a = *cache_pool;
  if (staging_opt) p.b = *staging_opt;   // else n_slots 0: staging entries read as out of range
  st = fp4_common(slot_table, n_layers, layer, E, H, I, counts, offsets, perm, x, T, k, y_rows, ws, ws_bytes,
                  dev_status, &p);
  if (st != MOE_OK || T == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (fp4_ring_ok(p, T, false)) err = launch_fp4_ring(p, T, false, s);
  else if (fp4_gemm_ok(p, false)) err = run_fp4_gemm(p, false, T, s);
  else if (T <= 1) err = launch_mx_nt<1>(p, s);
  else if (T <= 2) err = launch_mx_nt<2>(p, s);
  else err = launch_mx_nt<4>(p, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" size_t moe_expert_ffn_nvfp4_workspace_size(int T, int k, int H, int I) {
  if (T < 0 || k < 1 || H < 16 || I < 16 || (long long)T * k > INT_MAX / 2) return 0;
  return moe::mx_ws_bytes(T, k, H, I);
}

extern "C" int moe_expert_ffn_nvfp4(const moe_pool_nvfp4* cache_pool, const moe_pool_nvfp4* staging_opt,
                                    const int32_t* slot_table, int n_layers, int layer, int E, int H, int I,
                                    const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                                    const void* x, int T, int k, float* y_rows, void* ws, size_t ws_bytes,
                                    uint32_t* dev_status, moe_stream_t stream) {
  using namespace moe;
  int st = shape_check(cache_pool, slot_table, n_layers, layer, E, H, I, T, k, 16);
  if (st != MOE_OK) return st;
  st = check_nv_pool(cache_pool);
  if (st != MOE_OK) return st;
  if (staging_opt) {
    st = check_nv_pool(staging_opt);
    if (st != MOE_OK) return st;
  }
  MxParams p = {};
  p.a = as_mx_pool(*cache_pool);
  p.ts_a = cache_pool->tensor_scale;
  if (staging_opt) {
    p.b = as_mx_pool(*staging_opt);
    p.ts_b = staging_opt->tensor_scale;
  }
  st = fp4_common(slot_table, n_layers, layer, E, H, I, counts, offsets, perm, x, T, k, y_rows, ws, ws_bytes,
                  dev_status, &p);
  if (st != MOE_OK || T == 0) return st;
  // the ring kernel for decode-sized calls, the tensor-core GEMM for the rest
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (fp4_ring_ok(p, T, true)) err = launch_fp4_ring(p, T, true, s);
  else if (fp4_gemm_ok(p, true)) err = run_fp4_gemm(p, true, T, s);
  else return MOE_ERR_UNSUPPORTED;
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
