// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA) for prefill-sized expert groups (FreeToken paper,
// section 3.2: grouped evaluation of the GPU execution set; section 3: every
// expert is reached through its (layer, expert) slot).
//
// The products are computed transposed: the expert's weight rows are the
// MMA's M operand (128 rows a step) and the expert's token rows are its N
// operand, so a group of any size is padded only to a multiple of 16 rows
// (tcgen05 takes N = 16..256 in steps of 16 at M = 128).
//
// Work tile = (expert e, chunk of up to 256 of its rows, feature block).  The
// tile list is built on the device from the dispatch counts, so no host sync
// is needed; a persistent grid of one CTA per SM walks it round-robin.  Tiles
// of one chunk are adjacent, so the chunk's activation rows are read from L2
// by the CTAs working on its feature blocks while every weight tile is
// streamed from HBM once per chunk.
//
//   gate/up kernel  D_g = W_gate[f0:f0+128] X_c^T, D_u = W_up[f0:f0+128] X_c^T
//                   epilogue h[c, f] = bf16(silu(D_g) * D_u)  (one thread per f)
//   down kernel     D_m = W_down[f0+128m : +128] H_c^T (m = 0, 1)
//                   epilogue y[perm[c], f] = D  (token-major rows, fp32 or bf16)
//
// Roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM
// owner), warps 2..9 = epilogue (TMEM lanes 32*(warp%4) .. +31; the two warps
// on one lane quarter take alternate 32-column chunks).  Shared memory holds
// 3 stages of {2 weight tiles 128x64, token tile <=256x64} bf16 in the
// 128-byte swizzled K-major layout TMA writes (calls of at most 32 tokens:
// 6 stages with a token tile of <= 32 rows).  The two accumulators use TMEM
// columns [0, N) and [256, 256 + N).  Every mbarrier wait is bounded (about
// one second of %globaltimer); on expiry the CTA sets MOE_DEV_ERR_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <climits>

#include "ffn_params.cuh"
#include "group_prefix.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;                            // weight rows of one MMA
constexpr int kATile = kBM * kBK * 2;               // 16 KB

// Pipeline shape by the largest token chunk of a tile: 256-row chunks with
// three 64 KB stages, or (calls of at most 32 tokens, where the tiles are
// weight streams with a thin token operand) 32-row chunks with six 36 KB
// stages, twice the bytes in flight.
template <int CHUNK>
struct Shape {
  static constexpr int kStages = CHUNK <= 32 ? 6 : 3;
  static constexpr int kBTileMax = CHUNK * kBK * 2;
  static constexpr int kStageBytes = 2 * kATile + kBTileMax;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
};
static_assert(Shape<256>::kSmemBytes <= 227 * 1024 && Shape<32>::kSmemBytes <= 227 * 1024, "shared memory");
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 512;

struct GemmParams {
  const int32_t* counts;
  const int32_t* offsets;
  const uint8_t* mask;
  const int32_t* slot_table;
  int layer, E, H, I;
  int min_rows;            // groups with more rows than this run here
  int n_fb;                // feature blocks per chunk
  int K;                   // reduction length (H for gate/up, I for down)
  int has_staging;
  int skip_staging;        // the staging pool is host-resident: its experts are left to the plain GEMV
  int32_t cache_slots, staging_slots;
  const int32_t* perm;     // dispatch position -> token-major row
  __nv_bfloat16* h;        // gate/up output [R, I] (dispatch order)
  float* y;                // down output [R, H] (token-major), fp32
  __nv_bfloat16* y16;      // or bf16 when non-null
  uint32_t* status;
};

// ---------------------------------------------------------------- tile list
struct Tile {
  int e, r0, rows, N, fb, pool, slot;
  int32_t entry;
  bool ok, skip;   // skip: a staged expert left to another launch (not an error)
};

template <int kChunk>
__device__ inline Tile decode_tile(const GemmParams& p, const int* s_pref, int t) {
  Tile tl;
  const int ci = t / p.n_fb;
  tl.fb = t - ci * p.n_fb;
  tl.e = find_group(s_pref, p.E, ci);
  const int j = ci - s_pref[tl.e];
  const int cnt = p.counts[tl.e];
  tl.r0 = p.offsets[tl.e] + j * kChunk;
  tl.rows = min(kChunk, cnt - j * kChunk);
  tl.N = (tl.rows + 15) & ~15;
  const int32_t entry = p.slot_table[p.layer * p.E + tl.e];
  tl.entry = entry;
  tl.pool = (entry >= 0 && (entry & MOE_STAGING_TAG)) ? 1 : 0;
  tl.slot = entry & MOE_SLOT_MASK;
  tl.skip = p.skip_staging && entry >= 0 && tl.pool == 1;
  tl.ok = !tl.skip && entry >= 0 && (entry & ~(MOE_STAGING_TAG | MOE_SLOT_MASK)) == 0 &&
          tl.slot < (tl.pool ? p.staging_slots : p.cache_slots) && (tl.pool == 0 || p.has_staging);
  return tl;
}

// ---------------------------------------------------------------- kernel
// map_w{0,1}_{cache,stage}: weight banks [n_slots * rows_per_slot, K] with a
// 128-row box (gate/up: w0 = gate, w1 = up; down: w0 = w1 = down).
// map_b64 / map_b16: the token operand [R, K] with 64- and 16-row boxes.
template <bool GATEUP, int CHUNK>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap map_b64, const __grid_constant__ CUtensorMap map_b16,
            const __grid_constant__ CUtensorMap map_w0_cache, const __grid_constant__ CUtensorMap map_w1_cache,
            const __grid_constant__ CUtensorMap map_w0_stage, const __grid_constant__ CUtensorMap map_w1_stage,
            const GemmParams p) {
  using S = Shape<CHUNK>;
  constexpr int kStages = S::kStages, kStageBytes = S::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_pref[kMaxE + 1];
  __shared__ int s_warp[kThreads / 32];
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], tmem_full, tmem_empty, drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tmem_full, 1);
    mbar_init(&tmem_empty, 32 * kEpiWarps);
    mbar_init(&drain_bar, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  pdl_wait();
  // chunks of CHUNK rows per expert with more than min_rows rows (contains __syncthreads)
  build_group_prefix<CHUNK, (kMaxE + kThreads - 1) / kThreads>(p.counts, p.E, p.min_rows, INT_MAX, p.mask, s_pref,
                                                               s_warp);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort_flag = &s_abort;

  const int total = s_pref[p.E] * p.n_fb;
  const int kb_count = p.K / kBK;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      // Thin calls (every group in one chunk of <= 32 rows) read each weight tile
      // once: load it evict-first so it does not push out the reused token
      // tiles or force write-backs of other lines.  Larger groups span several
      // chunks whose CTAs share the weight tiles through L2 (measured: the
      // hint slows prefill down), so they load with the default policy.
      const uint64_t wpol = l2_evict_first();
      bool armed[kStages] = {};
      uint32_t armed_parity[kStages] = {};
      for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode_tile<CHUNK>(p, s_pref, t);
        if (!tl.ok) continue;
        const CUtensorMap* mw0 = tl.pool ? &map_w0_stage : &map_w0_cache;
        const CUtensorMap* mw1 = tl.pool ? &map_w1_stage : &map_w1_cache;
        // weight rows of this feature block inside the slot's bank
        const int wrow0 = GATEUP ? tl.slot * p.I + tl.fb * kBM : tl.slot * p.H + tl.fb * 2 * kBM;
        const int wrow1 = GATEUP ? wrow0 : wrow0 + kBM;
        const int n64 = tl.N >> 6, n16 = (tl.N & 63) >> 4;
        const uint32_t bytes = 2 * kATile + (uint32_t)tl.N * (kBK * 2);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) break;
          uint8_t* sA = smem + stage * kStageBytes;
          uint8_t* sB = sA + 2 * kATile;
          const int k0 = kb * kBK;
          mbar_expect_tx(&full_bar[stage], bytes);
          armed[stage] = true;
          armed_parity[stage] = phase;
          if (CHUNK <= 32) {
            tma_load_2d_hint(sA, mw0, &full_bar[stage], k0, wrow0, wpol);
            tma_load_2d_hint(sA + kATile, mw1, &full_bar[stage], k0, wrow1, wpol);
          } else {
            tma_load_2d(sA, mw0, &full_bar[stage], k0, wrow0);
            tma_load_2d(sA + kATile, mw1, &full_bar[stage], k0, wrow1);
          }
          for (int i = 0; i < n64; ++i) tma_load_2d(sB + i * 64 * (kBK * 2), &map_b64, &full_bar[stage], k0, tl.r0 + 64 * i);
          for (int i = 0; i < n16; ++i) {
            const int r = 64 * n64 + 16 * i;
            tma_load_2d(sB + r * (kBK * 2), &map_b16, &full_bar[stage], k0, tl.r0 + r);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every armed stage's copies land before the CTA can exit
      volatile int no_abort = 0;
      for (int s = 0; s < kStages; ++s)
        if (armed[s]) mbar_wait(&full_bar[s], armed_parity[s], &no_abort);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, tphase = 0;
      bool issued = false;
      for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode_tile<CHUNK>(p, s_pref, t);
        if (!tl.ok) continue;
        const uint32_t idesc = make_idesc(kBM, tl.N);
        if (!mbar_wait(&tmem_empty, tphase ^ 1u, abort_flag)) break;
        tc_fence_after();
        bool good = true;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
            good = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * kStageBytes);
          const uint32_t b0 = a0 + 2 * kATile;
#pragma unroll
          for (int ks = 0; ks < kBK / kUK; ++ks) {
            const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
            const uint64_t bd = smem_desc(b0 + ks * kUK * 2);
            tc_mma(tmem_base, smem_desc(a0 + ks * kUK * 2), bd, idesc, acc);
            tc_mma(tmem_base + 256, smem_desc(a0 + kATile + ks * kUK * 2), bd, idesc, acc);
          }
          issued = true;
          tc_commit(&empty_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!good) break;
        tc_commit(&tmem_full);
        tphase ^= 1u;
      }
      // drain: all issued MMAs complete before TMEM is released
      if (issued) {
        volatile int no_abort = 0;
        tc_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, &no_abort);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (warps 2..9)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t tphase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode_tile<CHUNK>(p, s_pref, t);
      if (!tl.ok) {
        if (tid == 64 && !tl.skip) set_status(p.status, tl.entry < 0 ? MOE_DEV_ERR_UNBOUND : MOE_DEV_ERR_BAD_SLOT);
        continue;
      }
      if (!mbar_wait(&tmem_full, tphase, abort_flag)) break;
      tc_fence_after();
      if (GATEUP) {
        // this thread's h column: feature f of the block
        const int f = tl.fb * kBM + quarter * 32 + lane;
        unsigned short* hcol = reinterpret_cast<unsigned short*>(p.h) + (size_t)tl.r0 * p.I + f;
#pragma unroll 1
        for (int c = half * 32; c < tl.N; c += 64) {
          uint32_t g[32], u[32];
          tmem_ld32(lane_addr + c, g);
          tmem_ld32(lane_addr + 256 + c, u);
          tmem_ld_wait();
          const int nv = min(32, tl.rows - c);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < nv) {
              const float hv = silu_fast(__uint_as_float(g[j])) * __uint_as_float(u[j]);
              hcol[(size_t)(c + j) * p.I] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
        }
      } else {
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
          const int f = tl.fb * 2 * kBM + m * kBM + quarter * 32 + lane;
#pragma unroll 1
          for (int c = half * 32; c < tl.N; c += 64) {
            uint32_t v[32];
            tmem_ld32(lane_addr + m * 256 + c, v);
            // token-major output rows of these 32 dispatch rows
            const int nv = min(32, tl.rows - c);
            const int prow = lane < nv ? p.perm[tl.r0 + c + lane] : 0;
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int yrow = __shfl_sync(0xffffffffu, prow, j);
              if (j < nv) {
                if (p.y16 != nullptr)
                  p.y16[(size_t)yrow * p.H + f] = __float2bfloat16_rn(__uint_as_float(v[j]));
                else
                  p.y[(size_t)yrow * p.H + f] = __uint_as_float(v[j]);
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tmem_empty);
      tphase ^= 1u;
    }
  }
  pdl_trigger();
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols));
}

template <bool GATEUP, int CHUNK>
cudaError_t launch_one(int grid, cudaStream_t s, const CUtensorMap& b64, const CUtensorMap& b16, const CUtensorMap& w0c,
                       const CUtensorMap& w1c, const CUtensorMap& w0s, const CUtensorMap& w1s, const GemmParams& p) {
  static std::atomic<unsigned char> attr[kMaxDevices];
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(gemm_kernel<GATEUP, CHUNK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Shape<CHUNK>::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  return launch_k(gemm_kernel<GATEUP, CHUNK>, grid, kThreads, Shape<CHUNK>::kSmemBytes, s, b64, b16, w0c, w1c, w0s,
                  w1s, p);
}

}  // namespace

bool gemm_shape_ok(int H, int I) { return H % 256 == 0 && I % 128 == 0 && H >= 256 && I >= 128; }

// Grouped GEMM over the experts with more than min_rows rows (gate/up, then down).
cudaError_t launch_gemm(const moe_cache& c, int layer, const int32_t* counts, const int32_t* offsets,
                        const int32_t* perm, const uint8_t* mask, int min_rows, const __nv_bfloat16* x_perm,
                        int T, int R, __nv_bfloat16* h, float* y, __nv_bfloat16* y16, uint32_t* status,
                        cudaStream_t s) {
  if (!gemm_shape_ok(c.H, c.I)) return cudaErrorNotSupported;
  // a host-resident staging pool gets no tensor map: its experts run on the plain GEMV
  const bool host_stage = c.staging.w_gate != nullptr && c.staging.host != 0;
  const bool has_stage = c.staging.w_gate != nullptr && !host_stage;
  const uint64_t H = (uint64_t)c.H, I = (uint64_t)c.I;
  GemmParams p;
  p.counts = counts;
  p.offsets = offsets;
  p.mask = mask;
  p.perm = perm;
  p.slot_table = c.slot_table;
  p.layer = layer;
  p.E = c.E;
  p.H = c.H;
  p.I = c.I;
  p.min_rows = min_rows;
  p.has_staging = has_stage ? 1 : 0;
  p.skip_staging = host_stage ? 1 : 0;
  p.cache_slots = c.cache.n_slots;
  p.staging_slots = has_stage ? c.staging.n_slots : 0;
  p.h = h;
  p.y = y;
  p.y16 = y16;
  p.status = status;

  CUtensorMap x64, x16, g0, u0, g1, u1;
  if (!make_map(&x64, x_perm, H, (uint64_t)R, 64) || !make_map(&x16, x_perm, H, (uint64_t)R, 16) ||
      !make_map(&g0, c.cache.w_gate, H, (uint64_t)c.cache.n_slots * I, kBM) ||
      !make_map(&u0, c.cache.w_up, H, (uint64_t)c.cache.n_slots * I, kBM))
    return cudaErrorInvalidValue;
  if (has_stage) {
    if (!make_map(&g1, c.staging.w_gate, H, (uint64_t)c.staging.n_slots * I, kBM) ||
        !make_map(&u1, c.staging.w_up, H, (uint64_t)c.staging.n_slots * I, kBM))
      return cudaErrorInvalidValue;
  } else {
    g1 = g0;
    u1 = u0;
  }
  p.K = c.H;
  p.n_fb = c.I / kBM;
  const int grid = num_sms();
  const bool thin = T <= 32;   // a group has at most T rows (one per token)
  cudaError_t err = thin ? launch_one<true, 32>(grid, s, x64, x16, g0, u0, g1, u1, p)
                         : launch_one<true, 256>(grid, s, x64, x16, g0, u0, g1, u1, p);
  if (err != cudaSuccess) return err;

  CUtensorMap h64, h16, d0, d1;
  if (!make_map(&h64, h, I, (uint64_t)R, 64) || !make_map(&h16, h, I, (uint64_t)R, 16) ||
      !make_map(&d0, c.cache.w_down, I, (uint64_t)c.cache.n_slots * H, kBM))
    return cudaErrorInvalidValue;
  if (has_stage) {
    if (!make_map(&d1, c.staging.w_down, I, (uint64_t)c.staging.n_slots * H, kBM)) return cudaErrorInvalidValue;
  } else {
    d1 = d0;
  }
  p.K = c.I;
  p.n_fb = c.H / (2 * kBM);
  return thin ? launch_one<false, 32>(grid, s, h64, h16, d0, d0, d1, d1, p)
              : launch_one<false, 256>(grid, s, h64, h16, d0, d0, d1, d1, p);
}

}  // namespace moe
