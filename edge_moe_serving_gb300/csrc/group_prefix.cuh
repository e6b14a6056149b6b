// Per-expert work lists shared by the grouped expert kernels: how many work
// items (row chunks, instances) each expert contributes, their exclusive
// prefix, and the search from an item back to its expert.
#pragma once

#include "moe_common.cuh"

namespace moe {
namespace {

// s_pref[e] = index of expert e's first item, s_pref[E] = number of items,
// where expert e contributes ceil(counts[e] / CHUNK) items when
// lo < counts[e] <= hi and (mask == null or mask[e] != 0), none otherwise.
// Run by a whole CTA (blockDim.x a multiple of 32, E <= blockDim.x * MAXPER);
// s_warp holds one int per warp.  Ends with __syncthreads.
template <int CHUNK, int MAXPER>
__device__ void build_group_prefix(const int32_t* counts, int E, int lo, int hi, const uint8_t* mask, int* s_pref,
                                   int* s_warp) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int per_thread = (E + nthreads - 1) / nthreads;
  const int e0 = tid * per_thread;
  int local[MAXPER];
  int sum = 0;
#pragma unroll
  for (int u = 0; u < MAXPER; ++u) {
    const int e = e0 + u;
    int n = 0;
    if (u < per_thread && e < E) {
      const int cnt = counts[e];
      const bool ok = cnt > lo && cnt <= hi && (mask == nullptr || mask[e] != 0);
      n = ok ? (cnt + CHUNK - 1) / CHUNK : 0;
    }
    local[u] = n;
    sum += n;
  }
  // exclusive scan of the per-thread sums: within the warp, then over the warps
  const int lane = tid & 31, warp = tid >> 5;
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
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
    s_pref[E] = run;
  }
  __syncthreads();
  int run = s_warp[warp] + inc - sum;
#pragma unroll
  for (int u = 0; u < MAXPER; ++u) {
    const int e = e0 + u;
    if (u < per_thread && e < E) s_pref[e] = run;
    run += local[u];
  }
  __syncthreads();
}

// The expert that owns item j: the largest e with s_pref[e] <= j (experts
// without items share their prefix value with the next one, so the largest
// such e is the one whose items start there).
__device__ inline int find_group(const int* s_pref, int E, int j) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= j) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace
}  // namespace moe
