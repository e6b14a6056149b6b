// Weight-streaming grouped GEMV for decode-sized expert groups (FreeToken
// paper, section 3.2: grouped evaluation of the GPU execution set; section 3:
// experts are reached through their (layer, expert) slot).
//
// Decode reads every routed expert's weights once per step, so these kernels
// are HBM-bound: each CTA streams a contiguous range of weight rows with
// 16-byte non-allocating loads, and every thread of the CTA works on every
// row (a row is split across the CTA, not across warps), so all SMs keep the
// same number of bytes in flight until the end and the grid is balanced to
// within one row group.
//
//  gateup_kernel  h[pos, i]  = bf16( silu(W_gate[i,:] . x_t) * (W_up[i,:] . x_t) )
//  down_kernel    y[pos, o]  = W_down[o,:] . h[pos,:]            (fp32)
//
// Work list: an "instance" is (expert e, chunk c of up to NT of its rows); an
// instance has I (gate/up) or H (down) tasks, one per output neuron, and
// consecutive tasks read consecutive weight rows.  CTA b owns tasks
// [b*per, (b+1)*per) of the flattened list and processes them NG at a time.
// Partial dot products are reduced with a warp reduce-scatter plus a fixed
// order sum over warps, so results do not depend on the grid.
#include "ffn_params.cuh"

namespace moe {
namespace {

constexpr int kMaxThreads = 256;

// Warp reduce-scatter of N (power of two >= 32) values: afterwards lane l
// holds the warp totals of values [l*N/32, (l+1)*N/32) in v[0 .. N/32).
template <int N>
__device__ inline void warp_reduce_scatter(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16, n = N; o > 0; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float keep = upper ? v[j + n / 2] : v[j];
      const float send = upper ? v[j] : v[j + n / 2];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

// Instances per expert (prefix over experts of ceil(rows / NT), eligible only).
template <int NT>
__device__ void build_prefix(const GemvParams& p, int* s_pref, int* s_warp) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int per_thread = (p.E + nthreads - 1) / nthreads;
  const int e0 = tid * per_thread;
  int local[kMaxE / 32];
  int sum = 0;
  for (int u = 0; u < per_thread; ++u) {
    const int e = e0 + u;
    int n = 0;
    if (e < p.E) {
      const int cnt = p.counts[e];
      const bool ok = cnt > 0 && cnt <= p.max_rows && (p.mask == nullptr || p.mask[e] != 0);
      n = ok ? (cnt + NT - 1) / NT : 0;
    }
    local[u] = n;
    sum += n;
  }
  // exclusive scan of per-thread sums
  const int lane = tid & 31, warp = tid >> 5;
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < nthreads / 32; ++w) {
      const int t = s_warp[w];
      s_warp[w] = run;
      run += t;
    }
    s_pref[p.E] = run;
  }
  __syncthreads();
  int run = s_warp[warp] + inc - sum;
  for (int u = 0; u < per_thread; ++u) {
    const int e = e0 + u;
    if (e < p.E) s_pref[e] = run;
    run += local[u];
  }
  __syncthreads();
}

// largest e with s_pref[e] <= j < s_pref[e + 1]
__device__ inline int find_expert(const int* s_pref, int E, int j) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= j) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int NT, int NG, bool GATEUP>
__global__ void __launch_bounds__(kMaxThreads)
gemv_kernel(GemvParams p) {
  constexpr int NR = GATEUP ? 2 : 1;
  constexpr int NV = NG * NR * NT;
  constexpr int NVP = NV < 32 ? 32 : NV;
  constexpr int PER_LANE = NVP / 32;
  __shared__ int s_pref[kMaxE + 1];
  __shared__ int s_warp[kMaxThreads / 32];
  __shared__ float red[2][kMaxThreads / 32][NVP];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int K = GATEUP ? p.H : p.I;        // weight row length
  const int NTASK = GATEUP ? p.I : p.H;    // output neurons per instance
  const int KV = K >> 3;                   // 16-byte vectors per row
  const int sweeps = (KV + nthreads - 1) / nthreads;

  build_prefix<NT>(p, s_pref, s_warp);
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
    const int e = find_expert(s_pref, p.E, j);
    const int c = j - s_pref[e];
    const int cnt = p.counts[e];
    const int pos0 = p.offsets[e] + c * NT;
    const int ntok = min(NT, cnt - c * NT);
    BankSet bs;
    const int32_t entry = p.c.slot_table[p.layer * p.E + e];
    if (!resolve_slot(p.c, entry, p.H, p.I, &bs, tid == 0 ? p.status : nullptr)) {
      tau += gsize;
      continue;
    }
    const __nv_bfloat16* wrow0;
    const __nv_bfloat16* wrow1;
    if (GATEUP) {
      wrow0 = bs.gate + (size_t)n0 * K;
      wrow1 = bs.up + (size_t)n0 * K;
    } else {
      wrow0 = bs.down + (size_t)n0 * K;
      wrow1 = wrow0;
    }
    const __nv_bfloat16* act[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int pos = pos0 + (t < ntok ? t : 0);
      if (GATEUP) {
        act[t] = p.x_perm ? p.x_perm + (size_t)pos * p.H : p.x + (size_t)(p.perm[pos] / p.k) * p.H;
      } else {
        act[t] = p.h + (size_t)pos * p.I;
      }
    }

    float acc[NVP];
#pragma unroll
    for (int q = 0; q < NVP; ++q) acc[q] = 0.0f;
    for (int s = 0; s < sweeps; ++s) {
      const int v = s * nthreads + tid;
      if (v < KV) {
        uint4 w[NG][NR];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          if (g < gsize) {
            w[g][0] = ldg_stream(wrow0 + (size_t)g * K + (size_t)v * 8);
            if (NR == 2) w[g][NR - 1] = ldg_stream(wrow1 + (size_t)g * K + (size_t)v * 8);
          } else {
            w[g][0] = make_uint4(0, 0, 0, 0);
            w[g][NR - 1] = make_uint4(0, 0, 0, 0);
          }
        }
        uint4 a[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t)
          a[t] = (t < ntok) ? ldg_cached(act[t] + (size_t)v * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
          for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t)
              acc[(g * NR + r) * NT + t] = dot8(w[g][r], a[t], acc[(g * NR + r) * NT + t]);
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
          p.y[(size_t)(pos0 + t) * p.H + n0 + g] = ys;
        }
      }
    }
    buf ^= 1;
    tau += gsize;
  }
}


// ---------------------------------------------------------------- TMA-ring variant
// Used when the weight row length K is a multiple of 256 (every lane then owns
// K/256 16-byte vectors of each row).  One producer thread streams "units" of
// consecutive weight rows (about 16 KB: U gate rows + U up rows, or U down rows)
// into a ring of shared-memory stages with cp.async.bulk, so each SM keeps
// ~160 KB of weight reads in flight regardless of how long the reductions
// take; four consumer warps each take every fourth unit, reduce each row with
// warp shuffles and write the outputs.  One CTA per SM; a CTA owns a
// contiguous range of units, so the grid is balanced to within one unit.
constexpr int kRingStages = 12;
constexpr int kUnitBytes = 16384;
constexpr int kConsumerWarps = 4;
constexpr int kRingThreads = (kConsumerWarps + 1) * 32;
constexpr unsigned long long kRingWaitNs = 1000000000ull;

__device__ inline uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ inline unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ inline bool ring_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ inline bool ring_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  unsigned long long start = 0;
  for (uint32_t it = 0;; ++it) {
    if (ring_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (*abort_flag) return false;
      const unsigned long long now = gtimer();
      if (start == 0) start = now;
      else if (now - start > kRingWaitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ inline void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Walks the units of [begin, end) in order: unit u = (instance j, rows n0..n0+rows).
struct UnitCursor {
  int j, n0;
};

template <int NT, bool GATEUP>
__global__ void __launch_bounds__(kRingThreads, 1)
gemv_ring_kernel(GemvParams p) {
  constexpr int NB = GATEUP ? 2 : 1;
  constexpr int kMaxVPL = 16;   // registers hold the single decode row for K <= 4096
  extern __shared__ uint8_t ring_raw[];
  __shared__ int s_pref[kMaxE + 1];
  __shared__ int s_warp[kRingThreads / 32];
  __shared__ int s_off[kMaxE];
  __shared__ int s_ent[kMaxE];
  __shared__ __align__(8) uint64_t full_bar[kRingStages], empty_bar[kRingStages];
  __shared__ int s_abort;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ring_raw) + 127) & ~uintptr_t(127));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = GATEUP ? p.H : p.I;
  const int NTASK = GATEUP ? p.I : p.H;
  const int row_bytes = K * 2;
  const int U = max(1, kUnitBytes / (NB * row_bytes));
  const int upi = (NTASK + U - 1) / U;
  const int bank_stride = kUnitBytes / NB;     // byte offset of the up rows in a stage
  const int VPL = K / 256;                     // 16-byte vectors per lane per row

  if (tid == 0) {
    for (int s = 0; s < kRingStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full_bar[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&empty_bar[s])));
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int e = tid; e < p.E; e += blockDim.x) {
    s_off[e] = p.offsets[e];
    s_ent[e] = p.c.slot_table[p.layer * p.E + e];
  }
  build_prefix<NT>(p, s_pref, s_warp);   // ends with __syncthreads
  volatile int* abort_flag = &s_abort;
  const long long total = (long long)s_pref[p.E] * upi;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long begin = (long long)blockIdx.x * per;
  const long long end = begin + per < total ? begin + per : total;
  const int first_j = (int)(begin / upi);
  const int first_n0 = (int)(begin % upi) * U;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      long long ri = 0, armed_last = -1;
      int j = first_j, n0 = first_n0, cur_j = -1;
      bool ok = false;
      BankSet bs;
      for (long long u = begin; u < end && !*abort_flag; ++u) {
        if (j != cur_j) {
          cur_j = j;
          const int e = find_expert(s_pref, p.E, j);
          ok = resolve_slot(p.c, s_ent[e], p.H, p.I, &bs, nullptr);
        }
        const int rows = min(U, NTASK - n0);
        if (ok) {
          const int stage = (int)(ri % kRingStages);
          const uint32_t use = (uint32_t)(ri / kRingStages);
          if (!ring_wait(&empty_bar[stage], (use & 1u) ^ 1u, abort_flag)) break;
          uint8_t* dst = ring + stage * kUnitBytes;
          const uint32_t bytes = (uint32_t)(rows * row_bytes);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&full_bar[stage])),
                       "r"(bytes * NB)
                       : "memory");
          if (GATEUP) {
            bulk_g2s(dst, bs.gate + (size_t)n0 * K, bytes, &full_bar[stage]);
            bulk_g2s(dst + bank_stride, bs.up + (size_t)n0 * K, bytes, &full_bar[stage]);
          } else {
            bulk_g2s(dst, bs.down + (size_t)n0 * K, bytes, &full_bar[stage]);
          }
          armed_last = ri;
          ++ri;
        }
        n0 += U;
        if (n0 >= NTASK) {
          n0 = 0;
          ++j;
        }
      }
      // drain: the copies of the last ring round land before the CTA exits
      volatile int no_abort = 0;
      for (long long q = armed_last; q >= 0 && q > armed_last - kRingStages; --q)
        ring_wait(&full_bar[q % kRingStages], (uint32_t)(q / kRingStages) & 1u, &no_abort);
    }
  } else {
    // ------------------------------------------------ consumers
    long long ri = 0;
    int j = first_j, n0 = first_n0, cur_j = -1;
    bool ok = false;
    int pos0 = 0, ntok = 0;
    const __nv_bfloat16* act[NT];
    uint4 xr[NT == 1 ? kMaxVPL : 1];
    const bool x_in_regs = (NT == 1) && VPL <= kMaxVPL;
    for (long long u = begin; u < end; ++u) {
      if (j != cur_j) {
        cur_j = j;
        const int e = find_expert(s_pref, p.E, j);
        BankSet bs;
        ok = resolve_slot(p.c, s_ent[e], p.H, p.I, &bs, (tid == 0) ? p.status : nullptr);
        const int c = j - s_pref[e];
        pos0 = s_off[e] + c * NT;
        ntok = min(NT, p.counts[e] - c * NT);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int pos = pos0 + (t < ntok ? t : 0);
          if (GATEUP)
            act[t] = p.x_perm ? p.x_perm + (size_t)pos * p.H : p.x + (size_t)(p.perm[pos] / p.k) * p.H;
          else
            act[t] = p.h + (size_t)pos * p.I;
        }
        if (NT == 1 && x_in_regs) {
#pragma unroll
          for (int c2 = 0; c2 < kMaxVPL; ++c2)
            if (c2 < VPL) xr[c2] = ldg_cached(act[0] + (size_t)(lane + 32 * c2) * 8);
        }
      }
      const int rows = min(U, NTASK - n0);
      const int my_n0 = n0;
      n0 += U;
      if (n0 >= NTASK) {
        n0 = 0;
        ++j;
      }
      if (!ok) continue;
      const long long mine = ri++;
      if ((int)(mine % kConsumerWarps) != warp) continue;
      const int stage = (int)(mine % kRingStages);
      const uint32_t use = (uint32_t)(mine / kRingStages);
      if (!ring_wait(&full_bar[stage], use & 1u, abort_flag)) break;
      const uint8_t* sw = ring + stage * kUnitBytes;
      for (int row = 0; row < rows; ++row) {
        float acc[NB][NT];
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[b][t] = 0.0f;
        const uint8_t* wrow = sw + (size_t)row * row_bytes + (size_t)lane * 16;
        if (NT == 1 && x_in_regs) {
#pragma unroll
          for (int c = 0; c < kMaxVPL; ++c) {
            if (c < VPL) {
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                const uint4 w = *reinterpret_cast<const uint4*>(wrow + b * bank_stride + c * 512);
                acc[b][0] = dot8(w, xr[NT == 1 ? c : 0], acc[b][0]);
              }
            }
          }
        } else {
#pragma unroll 4
          for (int c = 0; c < VPL; ++c) {
            const int v = lane + 32 * c;
            uint4 w[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) w[b] = *reinterpret_cast<const uint4*>(wrow + b * bank_stride + c * 512);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (t < ntok) {
                const uint4 a = ldg_cached(act[t] + (size_t)v * 8);
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[b][t] = dot8(w[b], a, acc[b][t]);
              }
            }
          }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[b][t] = warp_sum(acc[b][t]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (lane == t && t < ntok) {
            if (GATEUP)
              p.h[(size_t)(pos0 + t) * p.I + my_n0 + row] = __float2bfloat16_rn(silu(acc[0][t]) * acc[NB - 1][t]);
            else
              p.y[(size_t)(pos0 + t) * p.H + my_n0 + row] = acc[0][t];
          }
        }
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[stage])) : "memory");
    }
  }
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
}

constexpr int kRingSmem = kRingStages * kUnitBytes + 128;

template <int NT>
cudaError_t launch_ring_nt(const GemvParams& p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e1 = cudaFuncSetAttribute(gemv_ring_kernel<NT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmem);
    cudaError_t e2 = cudaFuncSetAttribute(gemv_ring_kernel<NT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmem);
    if (e1 != cudaSuccess) return e1;
    if (e2 != cudaSuccess) return e2;
    attr = true;
  }
  gemv_ring_kernel<NT, true><<<num_sms(), kRingThreads, kRingSmem, s>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  gemv_ring_kernel<NT, false><<<num_sms(), kRingThreads, kRingSmem, s>>>(p);
  return cudaGetLastError();
}

template <typename Kern>
int grid_for(Kern kern, int threads) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return per_sm * num_sms();
}

template <int NT>
cudaError_t launch_gemv_nt(const GemvParams& p, cudaStream_t s) {
  constexpr int NG_UP = 4, NG_DOWN = 8;
  const int thr_up = std::min(kMaxThreads, (int)align_up((size_t)(p.H / 8), 32));
  const int thr_dn = std::min(kMaxThreads, (int)align_up((size_t)(p.I / 8), 32));
  static int grid_up[kMaxThreads / 32 + 1] = {0};
  static int grid_dn[kMaxThreads / 32 + 1] = {0};
  if (!grid_up[thr_up / 32]) grid_up[thr_up / 32] = grid_for(gemv_kernel<NT, NG_UP, true>, thr_up);
  if (!grid_dn[thr_dn / 32]) grid_dn[thr_dn / 32] = grid_for(gemv_kernel<NT, NG_DOWN, false>, thr_dn);
  gemv_kernel<NT, NG_UP, true><<<grid_up[thr_up / 32], thr_up, 0, s>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  gemv_kernel<NT, NG_DOWN, false><<<grid_dn[thr_dn / 32], thr_dn, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Rows per pass: bounded by the tokens of the call (a group never exceeds T).
// Row lengths that are multiples of 256 take the TMA-ring kernels.
cudaError_t launch_gemv(const GemvParams& p, cudaStream_t s) {
  const int bound = std::min(p.T, p.max_rows);
  // a unit (one gate row + one up row, or one down row) must fit one 16 KB stage
  if (p.H % 256 == 0 && p.I % 256 == 0 && 2 * p.H * 2 <= kUnitBytes && p.I * 2 <= kUnitBytes) {
    if (bound <= 1) return launch_ring_nt<1>(p, s);
    if (bound <= 2) return launch_ring_nt<2>(p, s);
    if (bound <= 4) return launch_ring_nt<4>(p, s);
    return launch_ring_nt<8>(p, s);
  }
  if (bound <= 1) return launch_gemv_nt<1>(p, s);
  if (bound <= 2) return launch_gemv_nt<2>(p, s);
  if (bound <= 4) return launch_gemv_nt<4>(p, s);
  return launch_gemv_nt<8>(p, s);
}

}  // namespace moe
