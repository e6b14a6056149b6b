// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA) for prefill-sized expert groups (FreeToken paper,
// section 3.2: grouped evaluation of the GPU execution set; section 3: every
// expert is reached through its (layer, expert) slot).
//
// Work tile = (expert e, m-pair of up to 256 of its rows, n-tile).  The tile
// list is built on the device from the dispatch counts, so no host sync is
// needed; a persistent grid of one CTA per SM walks it round-robin.  Tiles
// of one expert are adjacent, so the 256 activation rows of an expert are
// read from L2 by the CTAs working on its n-tiles while each weight tile is
// streamed from HBM once for both 128-row m-tiles.
//
//   gate/up kernel  D_g = X_e W_gate^T, D_u = X_e W_up^T  (N = 128 + 128),
//                   epilogue h = bf16(silu(D_g) * D_u) -> h[pos, :]
//   down kernel     D = H_e W_down^T  (N = 256), epilogue fp32 -> y_rows[pos, :]
//
// Roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM
// owner), warps 2..5 = epilogue (TMEM lanes 32*(warp%4) .. +31).  Shared
// memory holds 3 stages of {2 A tiles 128x64, B tile 256x64} bf16 in the
// 128-byte swizzled K-major layout TMA writes.  The accumulator uses all 512
// TMEM columns (2 m-tiles x 256 fp32 columns).  Every mbarrier wait is
// bounded (about one second of %globaltimer); on expiry the CTA sets
// MOE_DEV_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ffn_params.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;       // rows of one MMA
constexpr int kBK = 64;        // K per stage: one 128-byte swizzle row of bf16
constexpr int kUK = 16;        // K of one tcgen05.mma kind::f16
constexpr int kStages = 3;
constexpr int kATile = kBM * kBK * 2;               // 16 KB
constexpr int kBBytes = 256 * kBK * 2;              // 32 KB
constexpr int kStageBytes = 2 * kATile + kBBytes;   // 64 KB
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;

struct GemmParams {
  const int32_t* counts;
  const int32_t* offsets;
  const uint8_t* mask;
  const int32_t* slot_table;
  int layer, E, H, I;
  int min_rows;            // groups with more rows than this run here
  int n_tiles;             // n-tiles per m-pair
  int K;                   // reduction length (H for gate/up, I for down)
  int has_staging;
  int32_t cache_slots, staging_slots;
  const int32_t* perm;     // dispatch position -> token-major row
  __nv_bfloat16* h;        // gate/up output [R, I] (dispatch order)
  float* y;                // down output [R, H] (token-major)
  uint32_t* status;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ inline uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ inline void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ inline void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ inline void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ inline bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return bounded_wait(bar, parity, abort_flag);
}

__device__ inline void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ inline void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ inline void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ inline void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: this thread's row, columns col..col+31.
__device__ inline void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ inline void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (the layout TMA's 128B swizzle writes).
__device__ inline uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);       // start address
  d |= (uint64_t)(16 >> 4) << 16;                  // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- tile list
__device__ void build_mpair_prefix(const GemmParams& p, int* s_pref, int* s_warp) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int per_thread = (p.E + nthreads - 1) / nthreads;
  const int e0 = tid * per_thread;
  int local[(kMaxE + kThreads - 1) / kThreads];
  int sum = 0;
  for (int u = 0; u < per_thread; ++u) {
    const int e = e0 + u;
    int n = 0;
    if (e < p.E) {
      const int cnt = p.counts[e];
      const bool ok = cnt > p.min_rows && (p.mask == nullptr || p.mask[e] != 0);
      n = ok ? (cnt + 2 * kBM - 1) / (2 * kBM) : 0;
    }
    local[u] = n;
    sum += n;
  }
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

__device__ inline int find_owner(const int* s_pref, int E, int j) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= j) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct Tile {
  int e, r0, m_valid, n_m, n0, pool, slot;
  int32_t entry;
  bool ok;
};

__device__ inline Tile decode_tile(const GemmParams& p, const int* s_pref, int t, int n_width) {
  Tile tl;
  const int mpi = t / p.n_tiles;
  const int nt = t % p.n_tiles;
  tl.e = find_owner(s_pref, p.E, mpi);
  const int mp = mpi - s_pref[tl.e];
  const int cnt = p.counts[tl.e];
  tl.r0 = p.offsets[tl.e] + mp * 2 * kBM;
  tl.m_valid = min(2 * kBM, cnt - mp * 2 * kBM);
  tl.n_m = tl.m_valid > kBM ? 2 : 1;
  tl.n0 = nt * n_width;
  const int32_t entry = p.slot_table[p.layer * p.E + tl.e];
  tl.entry = entry;
  tl.pool = (entry >= 0 && (entry & MOE_STAGING_TAG)) ? 1 : 0;
  tl.slot = entry & MOE_SLOT_MASK;
  tl.ok = entry >= 0 && (entry & ~(MOE_STAGING_TAG | MOE_SLOT_MASK)) == 0 &&
          tl.slot < (tl.pool ? p.staging_slots : p.cache_slots) && (tl.pool == 0 || p.has_staging);
  return tl;
}

// ---------------------------------------------------------------- kernel
template <bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0_cache,
            const __grid_constant__ CUtensorMap map_b1_cache, const __grid_constant__ CUtensorMap map_b0_stage,
            const __grid_constant__ CUtensorMap map_b1_stage, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_pref[kMaxE + 1];
  __shared__ int s_warp[kThreads / 32];
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], tmem_full, tmem_empty, drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kNW = GATEUP ? 128 : 256;                      // output columns per tile
  constexpr uint32_t kIdesc = make_idesc(kBM, GATEUP ? 128 : 256);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
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
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  pdl_wait();
  build_mpair_prefix(p, s_pref, s_warp);   // contains __syncthreads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort_flag = &s_abort;

  const int total = s_pref[p.E] * p.n_tiles;
  const int kb_count = p.K / kBK;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool armed[kStages] = {false, false, false};
      uint32_t armed_parity[kStages] = {0, 0, 0};
      for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode_tile(p, s_pref, t, kNW);
        if (!tl.ok) continue;
        const CUtensorMap* mb0 = tl.pool ? &map_b0_stage : &map_b0_cache;
        const CUtensorMap* mb1 = tl.pool ? &map_b1_stage : &map_b1_cache;
        const int brow = tl.slot * (GATEUP ? p.I : p.H) + tl.n0;
        const uint32_t bytes = tl.n_m * kATile + kBBytes;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) break;
          uint8_t* sA = smem + stage * kStageBytes;
          uint8_t* sB = sA + 2 * kATile;
          mbar_expect_tx(&full_bar[stage], bytes);
          armed[stage] = true;
          armed_parity[stage] = phase;
          for (int mt = 0; mt < tl.n_m; ++mt) tma_load_2d(sA + mt * kATile, &map_a, &full_bar[stage], kb * kBK, tl.r0 + mt * kBM);
          if (GATEUP) {
            tma_load_2d(sB, mb0, &full_bar[stage], kb * kBK, brow);
            tma_load_2d(sB + kBBytes / 2, mb1, &full_bar[stage], kb * kBK, brow);
          } else {
            tma_load_2d(sB, mb0, &full_bar[stage], kb * kBK, brow);
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
        const Tile tl = decode_tile(p, s_pref, t, kNW);
        if (!tl.ok) continue;
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
            for (int mt = 0; mt < tl.n_m; ++mt) {
              const uint64_t ad = smem_desc(a0 + mt * kATile + ks * kUK * 2);
              if (GATEUP) {
                tc_mma(tmem_base + mt * 256, ad, smem_desc(b0 + ks * kUK * 2), kIdesc, acc);
                tc_mma(tmem_base + mt * 256 + 128, ad, smem_desc(b0 + kBBytes / 2 + ks * kUK * 2), kIdesc, acc);
              } else {
                tc_mma(tmem_base + mt * 256, ad, smem_desc(b0 + ks * kUK * 2), kIdesc, acc);
              }
            }
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
    // ------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint32_t tphase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode_tile(p, s_pref, t, kNW);
      if (!tl.ok) {
        if (tid == 64) set_status(p.status, tl.entry < 0 ? MOE_DEV_ERR_UNBOUND : MOE_DEV_ERR_BAD_SLOT);
        continue;
      }
      if (!mbar_wait(&tmem_full, tphase, abort_flag)) break;
      tc_fence_after();
      for (int mt = 0; mt < tl.n_m; ++mt) {
        const int row = mt * kBM + row_in_tile;
        const bool valid = row < tl.m_valid;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quarter * 32) << 16) + mt * 256;
        if (GATEUP) {
          __nv_bfloat16* dst = p.h + (size_t)(tl.r0 + row) * p.I + tl.n0;
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(lane_addr + c, g);
            tmem_ld32(lane_addr + 128 + c, u);
            tmem_ld_wait();
            if (valid) {
              uint32_t packed[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float h0 = silu(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
                const float h1 = silu(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
                __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
                packed[j] = *reinterpret_cast<uint32_t*>(&b2);
              }
              uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                d4[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
            }
          }
        } else {
          // token-major output row of this dispatch row
          const int yrow = valid ? p.perm[tl.r0 + row] : 0;
          float* dst = p.y + (size_t)yrow * p.H + tl.n0;
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            uint32_t v[32];
            tmem_ld32(lane_addr + c, v);
            tmem_ld_wait();
            if (valid) {
              float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                d4[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                    __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
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


// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor [rows, inner] (inner contiguous), box = box_rows x 64, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || base == nullptr || rows == 0) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * sizeof(__nv_bfloat16)};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gemm_shape_ok(int H, int I) { return H % 256 == 0 && I % 128 == 0 && H >= 256 && I >= 128; }

// Grouped GEMM over the experts with more than min_rows rows (gate/up, then down).
cudaError_t launch_gemm(const moe_cache& c, int layer, const int32_t* counts, const int32_t* offsets,
                        const int32_t* perm, const uint8_t* mask, int min_rows, const __nv_bfloat16* x_perm,
                        int R, __nv_bfloat16* h, float* y, uint32_t* status, cudaStream_t s) {
  if (!gemm_shape_ok(c.H, c.I)) return cudaErrorNotSupported;
  static bool attr = false;
  if (!attr) {
    cudaError_t e1 = cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    cudaError_t e2 = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e1 != cudaSuccess) return e1;
    if (e2 != cudaSuccess) return e2;
    attr = true;
  }
  const bool has_stage = c.staging.w_gate != nullptr;
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
  p.cache_slots = c.cache.n_slots;
  p.staging_slots = has_stage ? c.staging.n_slots : 0;
  p.h = h;
  p.y = y;
  p.status = status;

  CUtensorMap a, g0, u0, g1, u1;
  if (!make_map(&a, x_perm, H, (uint64_t)R, kBM) ||
      !make_map(&g0, c.cache.w_gate, H, (uint64_t)c.cache.n_slots * I, 128) ||
      !make_map(&u0, c.cache.w_up, H, (uint64_t)c.cache.n_slots * I, 128))
    return cudaErrorInvalidValue;
  if (has_stage) {
    if (!make_map(&g1, c.staging.w_gate, H, (uint64_t)c.staging.n_slots * I, 128) ||
        !make_map(&u1, c.staging.w_up, H, (uint64_t)c.staging.n_slots * I, 128))
      return cudaErrorInvalidValue;
  } else {
    g1 = g0;
    u1 = u0;
  }
  p.K = c.H;
  p.n_tiles = c.I / 128;
  const int grid = num_sms();
  cudaError_t err = launch_k(gemm_kernel<true>, grid, kThreads, kSmemBytes, s, a, g0, u0, g1, u1, p);
  if (err != cudaSuccess) return err;

  CUtensorMap ha, d0, d1;
  if (!make_map(&ha, h, I, (uint64_t)R, kBM) ||
      !make_map(&d0, c.cache.w_down, I, (uint64_t)c.cache.n_slots * H, 256))
    return cudaErrorInvalidValue;
  if (has_stage) {
    if (!make_map(&d1, c.staging.w_down, I, (uint64_t)c.staging.n_slots * H, 256)) return cudaErrorInvalidValue;
  } else {
    d1 = d0;
  }
  p.K = c.I;
  p.n_tiles = c.H / 256;
  return launch_k(gemm_kernel<false>, grid, kThreads, kSmemBytes, s, ha, d0, d0, d1, d1, p);
}

}  // namespace moe
