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
#include "ring_gemv.cuh"

namespace moe {
namespace {

constexpr int kMaxThreads = 256;

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

  pdl_wait();
  pdl_trigger();
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
    const int e = find_group(s_pref, p.E, j);
    const int c = j - s_pref[e];
    const int cnt = p.counts[e];
    const int pos0 = p.offsets[e] + c * NT;
    const int ntok = min(NT, cnt - c * NT);
    BankSet bs;
    const int32_t entry = p.c.slot_table[p.layer * p.E + e];
    if (!resolve_filtered(p.c, entry, p.pool_filter, p.H, p.I, &bs, tid == 0 ? p.status : nullptr)) {
      tau += gsize;
      continue;
    }
    const bool host_src = p.c.staging.host != 0 && (entry & MOE_STAGING_TAG) != 0;
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
          if (g < gsize && host_src) {
            // the host-resident staging pool: plain streaming loads over the CPU-GPU link
            w[g][0] = __ldcs(reinterpret_cast<const uint4*>(wrow0 + (size_t)g * K + (size_t)v * 8));
            if (NR == 2) w[g][NR - 1] = __ldcs(reinterpret_cast<const uint4*>(wrow1 + (size_t)g * K + (size_t)v * 8));
          } else if (g < gsize) {
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
          p.y[(size_t)p.perm[pos0 + t] * p.H + n0 + g] = ys;
        }
      }
    }
    buf ^= 1;
    tau += gsize;
  }
}


// One persistent cooperative launch (one CTA per SM) does both projections;
// see fused_ffn_body.
template <int NT, int VA, int VB>
__global__ void __launch_bounds__(kRingThreads, 1)
gemv_fused_kernel(GemvParams p, unsigned int* grid_count) {
  extern __shared__ __align__(128) uint8_t ring_raw[];
  __shared__ __align__(16) FusedShared fs;
  // the ring is the dynamic shared array itself: pointers derived from it keep the shared
  // address space, so stage reads compile to shared-memory loads
  uint8_t* ring = ring_raw;
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) ring_init(fs.r);
  pdl_wait();
  for (int e = tid; e < p.E; e += blockDim.x) {
    fs.off[e] = p.offsets[e];
    fs.ent[e] = p.c.slot_table[p.layer * p.E + e];
    fs.fill[e] = -1;
  }
  __syncthreads();
  if (p.fills != nullptr && tid < 32) {
    const int nf = *p.n_fill;
    for (int f = lane; f < nf; f += 32) {
      const int e = p.fills[2 * f] - p.layer * p.E;
      if (e >= 0 && e < p.E) fs.fill[e] = p.fills[2 * f + 1];
    }
  }
  fused_ffn_body<NT, VA, VB>(p, grid_count, fs, ring);
  pdl_trigger();
  __syncthreads();
  if (fs.r.abort && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
}


template <int NT, int VA, int VB>
cudaError_t launch_fused_one(const GemvParams& p, unsigned int* grid_count, cudaStream_t s) {
  static std::atomic<unsigned char> attr[kMaxDevices];
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(gemv_fused_kernel<NT, VA, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kRingSmem);
  });
  if (e != cudaSuccess) return e;
  const size_t words = p.inst_done != nullptr ? 4 + (size_t)p.T * p.k : 2;
  cudaError_t err = cudaMemsetAsync(grid_count, 0, words * sizeof(unsigned int), s);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = kRingSmem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: the grid barrier can complete
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, gemv_fused_kernel<NT, VA, VB>, p, grid_count));
}

// Single-token calls with rows of 4096 (gate/up) and 2048 (down) elements,
// the decode shapes, keep the token's row in registers.
template <int NT>
cudaError_t launch_ring_nt(const GemvParams& p, unsigned int* grid_count, cudaStream_t s) {
  if (NT == 1) {
    const bool va = p.H == 4096 && ring_rows(p.H, true) == 1;
    const bool vb = p.I == 2048;
    if (va && vb) return launch_fused_one<NT, 16, 8>(p, grid_count, s);
    if (va) return launch_fused_one<NT, 16, 0>(p, grid_count, s);
    if (vb) return launch_fused_one<NT, 0, 8>(p, grid_count, s);
  }
  return launch_fused_one<NT, 0, 0>(p, grid_count, s);
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
  // grid per (device, block size); 0 = not computed yet
  static std::atomic<int> grid_up[kMaxDevices][kMaxThreads / 32 + 1], grid_dn[kMaxDevices][kMaxThreads / 32 + 1];
  const int dev = device_index();
  int gu = dev >= 0 ? grid_up[dev][thr_up / 32].load(std::memory_order_relaxed) : 0;
  int gd = dev >= 0 ? grid_dn[dev][thr_dn / 32].load(std::memory_order_relaxed) : 0;
  if (!gu) {
    gu = grid_for(gemv_kernel<NT, NG_UP, true>, thr_up);
    if (dev >= 0) grid_up[dev][thr_up / 32].store(gu, std::memory_order_relaxed);
  }
  if (!gd) {
    gd = grid_for(gemv_kernel<NT, NG_DOWN, false>, thr_dn);
    if (dev >= 0) grid_dn[dev][thr_dn / 32].store(gd, std::memory_order_relaxed);
  }
  cudaError_t err = launch_k(gemv_kernel<NT, NG_UP, true>, gu, thr_up, 0, s, p);
  if (err != cudaSuccess) return err;
  return launch_k(gemv_kernel<NT, NG_DOWN, false>, gd, thr_dn, 0, s, p);
}

}  // namespace

// The plain-load kernel for any row length, rows per pass bounded by the
// tokens of the call.
cudaError_t launch_gemv_plain(const GemvParams& p, cudaStream_t s) {
  const int bound = std::min(p.T, p.max_rows);
  if (bound <= 1) return launch_gemv_nt<1>(p, s);
  if (bound <= 2) return launch_gemv_nt<2>(p, s);
  if (bound <= 4) return launch_gemv_nt<4>(p, s);
  return launch_gemv_nt<8>(p, s);
}

// Rows per pass: bounded by the tokens of the call (a group never exceeds T).
// Row lengths that are multiples of 256 take the fused TMA-ring kernel.
cudaError_t launch_gemv(const GemvParams& p, cudaStream_t s) {
  const int bound = std::min(p.T, p.max_rows);
  if (gemv_fused_ok(p.H, p.I)) {
    unsigned int* grid_count = p.grid_count;
    if (bound <= 1) return launch_ring_nt<1>(p, grid_count, s);
    if (bound <= 2) return launch_ring_nt<2>(p, grid_count, s);
    if (bound <= 4) return launch_ring_nt<4>(p, grid_count, s);
    return launch_ring_nt<8>(p, grid_count, s);
  }
  return launch_gemv_plain(p, s);
}

}  // namespace moe
