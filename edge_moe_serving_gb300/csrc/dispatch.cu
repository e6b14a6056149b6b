// Token -> expert dispatch (FreeToken paper, section 3.2: routed rows are
// grouped per expert for a grouped evaluation).  A stable counting sort of the
// flat rows i = t*k + j by expert id, bit-exact and deterministic: no atomic
// decides a position.
//
// Tile = 1024 consecutive rows, one per thread.  Within a warp, rows with the
// same expert are ranked by __match_any_sync; across the 32 warps of a tile,
// a [32][E] shared table of per-warp counts gives each row the number of
// same-expert rows in earlier warps.  Tiles are processed in row order, so
// rows of one expert land in increasing i.
//  * R <= kSingleMaxR: one CTA does histogram, scan and every tile.
//  * larger R: (A) per-tile histograms, (B) one CTA turns them into per-tile
//    bases and the offsets, (C) one CTA per tile scatters.
// The optional gather x_perm[pos] = x[perm[pos] / k] is a separate
// bandwidth-bound kernel (one warp per row).
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kTile = 1024;
constexpr int kSingleMaxR = 4096;

__device__ inline unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan over a 1024-thread block; returns this thread's prefix and
// writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
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
__device__ void scatter_tile(const int32_t* __restrict__ ids, int R, int E, int base, int* cursor,
                             int* wcnt, int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

__global__ void __launch_bounds__(kTile)
dispatch_single_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ counts,
                       int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                       int32_t* __restrict__ inv_perm, uint32_t* status) {
  extern __shared__ int sm[];
  int* cursor = sm;              // [E]
  int* wcnt = cursor + E;        // [32][E]
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
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

__global__ void __launch_bounds__(kTile)
tile_hist_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ tile_counts,
                 uint32_t* status) {
  extern __shared__ int hist[];
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  for (int j = tid; j < E; j += kTile) hist[j] = 0;
  __syncthreads();
  const int i = blockIdx.x * kTile + tid;
  if (i < R) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else set_status(status, MOE_DEV_ERR_BAD_ID);
  }
  __syncthreads();
  for (int j = tid; j < E; j += kTile) tile_counts[(size_t)blockIdx.x * E + j] = hist[j];
}

__global__ void __launch_bounds__(kTile)
tile_scan_kernel(int32_t* __restrict__ tile_counts, int ntiles, int E, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets) {
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int e = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  int run = 0;
  if (e < E) {
    // tile counts -> exclusive prefix over tiles (the tile's base before offsets are added);
    // loads are batched so that they are in flight together
    for (int t0 = 0; t0 < ntiles; t0 += 16) {
      int c[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) c[u] = (t0 + u < ntiles) ? tile_counts[(size_t)(t0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        if (t0 + u < ntiles) tile_counts[(size_t)(t0 + u) * E + e] = run;
        run += c[u];
      }
    }
  }
  const int off = block_exclusive_scan(e < E ? run : 0, warp_tot, &total);
  if (e < E) {
    counts[e] = run;
    offsets[e] = off;
    for (int t = 0; t < ntiles; ++t) tile_counts[(size_t)t * E + e] += off;
  }
  if (e == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(kTile)
tile_scatter_kernel(const int32_t* __restrict__ ids, int R, int E,
                    const int32_t* __restrict__ tile_base, int32_t* __restrict__ perm,
                    int32_t* __restrict__ inv_perm) {
  extern __shared__ int sm[];
  int* cursor = sm;
  int* wcnt = cursor + E;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  for (int j = tid; j < E * 32; j += kTile) wcnt[j] = 0;
  for (int j = tid; j < E; j += kTile) cursor[j] = tile_base[(size_t)blockIdx.x * E + j];
  __syncthreads();
  scatter_tile(ids, R, E, blockIdx.x * kTile, cursor, wcnt, perm, inv_perm);
}

// x_perm[pos, :] = x[perm[pos] / k, :]; one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int k,
                   const int32_t* __restrict__ perm, const int32_t* __restrict__ offsets, int E,
                   int R, __nv_bfloat16* __restrict__ x_perm) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  // rows past offsets[E] exist only when some ids were invalid: nothing to gather
  if (warp >= R || warp >= offsets[E]) return;
  const int t = perm[warp] / k;
  if (t < 0 || t >= T) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)warp * H);
  const int nv = H >> 3;
  for (int v = lane; v < nv; v += 32) dst[v] = __ldg(src + v);
}

}  // namespace

size_t dispatch_ws_bytes(int T, int k, int E) {
  const size_t R = (size_t)T * k;
  if (R <= (size_t)kSingleMaxR) return 0;
  const size_t ntiles = (R + kTile - 1) / kTile;
  return align_up(ntiles * E * sizeof(int32_t), 256);
}

cudaError_t launch_dispatch(const int32_t* ids, int R, int k, int E, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                            const __nv_bfloat16* x, int H, __nv_bfloat16* x_perm, void* ws,
                            uint32_t* status, cudaStream_t s) {
  static int attr_bytes = 0;
  const int need = (int)(sizeof(int) * 33 * (size_t)E);
  if (need > attr_bytes) {
    cudaError_t err = cudaFuncSetAttribute(dispatch_single_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(sizeof(int) * 33 * kMaxE));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(tile_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(sizeof(int) * 33 * kMaxE));
    if (err != cudaSuccess) return err;
    attr_bytes = (int)(sizeof(int) * 33 * kMaxE);
  }
  cudaError_t err;
  if (R <= kSingleMaxR) {
    err = launch_k(dispatch_single_kernel, 1, kTile, need, s, ids, R, E, counts, offsets, perm, inv_perm, status);
  } else {
    const int ntiles = (R + kTile - 1) / kTile;
    int32_t* tile_counts = reinterpret_cast<int32_t*>(ws);
    err = launch_k(tile_hist_kernel, ntiles, kTile, sizeof(int) * E, s, ids, R, E, tile_counts, status);
    if (err == cudaSuccess) err = launch_k(tile_scan_kernel, 1, kTile, 0, s, tile_counts, ntiles, E, counts, offsets);
    if (err == cudaSuccess)
      err = launch_k(tile_scatter_kernel, ntiles, kTile, need, s, ids, R, E, (const int32_t*)tile_counts, perm, inv_perm);
  }
  if (err != cudaSuccess) return err;
  if (x && x_perm && R > 0) {
    const int blocks = (R + 7) / 8;
    err = launch_k(gather_rows_kernel, blocks, 256, 0, s, x, R / k, H, k, (const int32_t*)perm,
                   (const int32_t*)offsets, E, R, x_perm);
  }
  return err;
}

}  // namespace moe
