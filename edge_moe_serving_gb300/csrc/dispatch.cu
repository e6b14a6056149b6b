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
#include "dispatch_block.cuh"

namespace moe {
namespace {

using blk::kTile;
using blk::block_exclusive_scan;
using blk::scatter_tile;
constexpr int kSingleMaxR = 4096;

__global__ void __launch_bounds__(kTile)
dispatch_single_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ counts,
                       int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                       int32_t* __restrict__ inv_perm, uint32_t* status) {
  extern __shared__ int sm[];
  pdl_wait();
  pdl_trigger();
  blk::dispatch_block(ids, R, E, counts, offsets, perm, inv_perm, status, sm);
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
  const int need = (int)(sizeof(int) * 33 * (size_t)E);
  static std::atomic<unsigned char> attr[kMaxDevices];
  cudaError_t err = once_per_device(attr, [] {
    const int max_bytes = (int)(sizeof(int) * 33 * kMaxE);
    cudaError_t e = cudaFuncSetAttribute(dispatch_single_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tile_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_bytes);
  });
  if (err != cudaSuccess) return err;
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
  if (x && x_perm && R > 0) err = launch_gather(x, H, k, perm, offsets, E, R, x_perm, s);
  return err;
}

cudaError_t launch_gather(const __nv_bfloat16* x, int H, int k, const int32_t* perm, const int32_t* offsets, int E,
                          int R, __nv_bfloat16* x_perm, cudaStream_t s) {
  const int blocks = (R + 7) / 8;
  return launch_k(gather_rows_kernel, blocks, 256, 0, s, x, R / k, H, k, perm, offsets, E, R, x_perm);
}

}  // namespace moe
