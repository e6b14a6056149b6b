// Single-CTA stable counting sort of routed rows by expert id (1024 threads),
// shared by the dispatch kernels and the fused residency + dispatch kernel.
#pragma once

#include "moe_common.cuh"

namespace moe {
namespace blk {

constexpr int kTile = 1024;

__device__ inline unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan over a 1024-thread block; returns this thread's prefix and
// writes the block total to *total.
__device__ inline int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += n;
    }
    warp_tot[lane] = winc - w;
    if (lane == 31) *total = winc;
  }
  __syncthreads();
  const int res = warp_tot[warp] + inc - v;
  __syncthreads();
  return res;
}

// Scatter one tile of rows [base, base + 1024).  cursor[e] holds the next free
// position of expert e; wcnt is a zeroed [32][E] table (left zeroed on exit).
__device__ inline void scatter_tile(const int32_t* __restrict__ ids, int R, int E, int base, int* cursor,
                             int* wcnt, int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int i = base + tid;
  const int e = (i < R) ? ids[i] : -1;
  const bool valid = (e >= 0 && e < E);
  const int key = valid ? e : -1;
  const unsigned mask = __match_any_sync(0xffffffffu, key);
  const unsigned lt = lanemask_lt();
  const int rank = __popc(mask & lt);
  const bool leader = (mask & lt) == 0;
  const int nwarps = blockDim.x >> 5;
  if (valid && leader) wcnt[warp * E + e] = __popc(mask);
  __syncthreads();
  int pos = 0;
  bool last = false;
  if (valid) {
    int pre = 0, later = 0;
    for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
    for (int w = warp + 1; w < nwarps; ++w) later += wcnt[w * E + e];
    pos = cursor[e] + pre + rank;
    last = (later == 0) && (rank == __popc(mask) - 1);
    perm[pos] = i;
    inv_perm[i] = pos;
  }
  __syncthreads();
  if (valid && last) cursor[e] = pos + 1;
  if (valid && leader) wcnt[warp * E + e] = 0;
  __syncthreads();
}

// Whole dispatch of R <= a few thousand rows by one 1024-thread CTA.
// sm: E * 33 ints of shared memory (cursor [E], per-warp counts [32][E]).
__device__ inline void dispatch_block(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ counts,
                                      int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                      int32_t* __restrict__ inv_perm, uint32_t* status, int* sm) {
  int* cursor = sm;              // [E]
  int* wcnt = cursor + E;        // [32][E]
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int tid = threadIdx.x;
  for (int j = tid; j < E * 33; j += kTile) sm[j] = 0;
  __syncthreads();
  bool bad = false;
  for (int i = tid; i < R; i += kTile) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&cursor[e], 1);
    else bad = true;
  }
  if (bad) set_status(status, MOE_DEV_ERR_BAD_ID);
  __syncthreads();
  for (int e0 = 0; e0 < E; e0 += kTile) {
    // E <= 1024 = kTile: one pass
    const int e = e0 + tid;
    const int c = (e < E) ? cursor[e] : 0;
    const int off = block_exclusive_scan(c, warp_tot, &total);
    if (e < E) {
      counts[e] = c;
      offsets[e] = off;
      cursor[e] = off;
    }
    if (tid == 0) offsets[E] = total;
  }
  __syncthreads();
  for (int base = 0; base < R; base += kTile) scatter_tile(ids, R, E, base, cursor, wcnt, perm, inv_perm);
}

}  // namespace blk
}  // namespace moe
