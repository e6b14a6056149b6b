// Grouped FP4 expert GEMM on the 5th-generation tensor cores (FreeToken
// paper, section 5.1 "Models": MXFP4 and NVFP4 expert banks; section 4.1: the
// expert kernels dequantise in-kernel; section 3.2: grouped evaluation).
//
// The bf16 grouped GEMM's tiling: the expert's weight rows are the MMA's M
// operand (128 rows a step), a chunk of up to CHUNK of its token rows the N
// operand; work tile = (expert, chunk, feature block), the list built on the
// device from the dispatch counts; one persistent CTA per SM.  The weight
// operand arrives as FP4: TMA brings each stage's E2M1 codes (128 rows x 64
// inputs, 4 KB per operand tile); eight dequantising warps read their rows'
// block scales from global memory (8 bytes at a time, one group ahead) and
// expand the codes into the bf16 K-major 128-byte-swizzled tile that
// tcgen05.mma kind::f16 reads.
//
// Exactness: an E2M1 value times its E8M0 power of two (MXFP4) or its E4M3
// value (NVFP4) has at most 6 significant bits, so the expansion (bf16
// products of exact bf16 factors) is exact while it stays inside bf16's range
// (every MXFP4 code up to the scale 2^125, byte 252; all NVFP4 values); the MMA
// multiplies bf16 by bf16 exactly and accumulates in fp32.  NVFP4's fp32
// tensor scale of each bank multiplies the accumulator in the epilogue.
//
//   gate/up kernel  D_g = Wg[f0:+128] X_c^T, D_u = Wu[f0:+128] X_c^T,
//                   h[c, f] = bf16(silu(D_g * ts_g) * (D_u * ts_u))
//   down kernel     D_m = Wd[f0+128m:+128] H_c^T (m = 0, 1), y[perm[c], f] = D_m * ts_d
//
// Roles (576 threads): warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM
// owner), warps 2..9 = epilogue, warps 10..17 = dequantisers (thread = one
// row of one of the two 128-row operand tiles).  Rings: the load ring (codes
// of both operand tiles + the token tile), released by the dequantisers and
// the MMA; the operand ring (two bf16 tiles), filled by the dequantisers and
// released by the MMA.  Every mbarrier wait is bounded (about a second of %globaltimer);
// on expiry the CTA sets MOE_DEV_ERR_TIMEOUT, drains its in-flight copies and
// MMAs, frees TMEM and returns.
#include <algorithm>
#include <climits>

#include "group_prefix.cuh"
#include "mxfp4.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;                    // weight rows of one MMA
constexpr int kCodeTile = kBM * kBK / 2;    // 4 KB of E2M1 codes: 128 rows x 64 inputs
constexpr int kATile = kBM * kBK * 2;       // 16 KB of bf16: the expanded operand tile
constexpr int kScaleGroup = 8;              // scale bytes a dequantiser loads at a time
constexpr int kEpiWarps = 8;
constexpr int kDeqWarps = 8;
constexpr int kThreads = 64 + 32 * (kEpiWarps + kDeqWarps);
constexpr int kTmemCols = 512;

constexpr int kF4MaxE = 256;   // experts per layer the GEMM takes (its group prefix sits in static shared memory)

template <int CHUNK>
struct F4Shape {
  static constexpr int kLoadStages = CHUNK <= 32 ? 8 : 4;
  static constexpr int kAStages = CHUNK <= 32 ? 3 : 2;
  static constexpr int kBTile = CHUNK * kBK * 2;           // token tile (128-byte rows)
  static constexpr int kLoadBytes = kBTile + 2 * kCodeTile;
  static constexpr int kSmemBytes = kAStages * 2 * kATile + kLoadStages * kLoadBytes + 1024;
};
static_assert(F4Shape<256>::kSmemBytes <= 227 * 1024 && F4Shape<32>::kSmemBytes <= 227 * 1024, "shared memory");
static_assert(F4Shape<256>::kLoadBytes % 1024 == 0 && F4Shape<32>::kLoadBytes % 1024 == 0, "token tiles stay aligned");

struct F4Params {
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* slot_table;
  int layer, E, H, I;
  int n_fb;              // feature blocks per chunk
  int K;                 // reduction length (H for gate/up, I for down)
  int32_t cache_slots, staging_slots;
  const float* ts[2];    // NVFP4 tensor scales [n_slots][3] of each pool (null: MXFP4)
  const uint8_t* sc[2][2];   // scale banks [pool][operand tile] (gate/up: gate, up; down: down twice)
  const int32_t* perm;   // dispatch position -> token-major row
  __nv_bfloat16* h;      // gate/up output [R, I] (dispatch order)
  float* y;              // down output [R, H] (token-major)
  uint32_t* status;
};

struct F4Tile {
  int e, r0, rows, N, fb, pool, slot;
  int32_t entry;
  bool ok;
};

template <int CHUNK>
__device__ inline F4Tile f4_tile(const F4Params& p, const int* s_pref, int t) {
  F4Tile tl;
  const int ci = t / p.n_fb;
  tl.fb = t - ci * p.n_fb;
  tl.e = find_group(s_pref, p.E, ci);
  const int j = ci - s_pref[tl.e];
  tl.r0 = p.offsets[tl.e] + j * CHUNK;
  tl.rows = min(CHUNK, p.counts[tl.e] - j * CHUNK);
  tl.N = (tl.rows + 15) & ~15;
  const int32_t entry = p.slot_table[p.layer * p.E + tl.e];
  tl.entry = entry;
  tl.pool = (entry >= 0 && (entry & MOE_STAGING_TAG)) ? 1 : 0;
  tl.slot = entry & MOE_SLOT_MASK;
  tl.ok = entry >= 0 && (entry & ~(MOE_STAGING_TAG | MOE_SLOT_MASK)) == 0 &&
          tl.slot < (tl.pool ? p.staging_slots : p.cache_slots);
  return tl;
}

// Operand tile rows of a work tile inside its slot's bank: tile 0 and tile 1
// (gate/up: the same rows of the gate and the up bank; down: two consecutive
// 128-row blocks of the down bank).
template <bool GATEUP>
__device__ inline int f4_row(const F4Params& p, const F4Tile& tl, int which) {
  return GATEUP ? tl.slot * p.I + tl.fb * kBM : tl.slot * p.H + tl.fb * 2 * kBM + which * kBM;
}

// Eight E2M1 codes (one 32-bit word, element 2c in the low nibble of byte c)
// -> eight bf16 values (16 bytes) equal to the codes' values times the
// block scale, exactly.  A bf16 whose two low exponent bits and top mantissa
// bit are a code's three magnitude bits is that code's value times 2^-126
// (zero and the subnormal code 0.5 included: exponent field 0 is bf16's
// subnormal range), so each pair is placed by bit operations and scaled by
// exact multiplications: by c1, then by c2 when `two` (c1 = 2^126 times the
// block scale where that is a bf16, else c1 = 2^126 and c2 = the scale).
__device__ inline uint4 expand8(uint32_t w, uint32_t c1, uint32_t c2, bool two) {
  const uint32_t a = w & 0x0F0F0F0Fu;          // byte j: element 2j
  const uint32_t b = (w >> 4) & 0x0F0F0F0Fu;   // byte j: element 2j + 1
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // byte 0 <- a.byte j, byte 2 <- b.byte j; bytes 1 and 3 <- 0 (selector 8 replicates the sign bit of
    // a.byte 0, which is clear)
    uint32_t t;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(a), "r"(b), "r"(0x8080u | (uint32_t)j | ((4u + j) << 8)));
    // magnitude bits 0..2 of each half to bits 6..8, the sign (bit 3) to bit 15: t * (2^6 + 2^12) moves
    // both copies without overlap, the mask keeps one of each
    const uint32_t raw = (t * 0x1040u) & 0x81C081C0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[j]) : "r"(raw), "r"(c1));
    if (two) asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(o[j]) : "r"(c2));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Block scale factors as bf16 pairs (exact).  MXFP4, E8M0 s: 2^(s-127) (s = 0
// is 2^-127, a bf16 subnormal; s = 255 NaN); for s <= 128 and for NaN,
// 2^126 * 2^(s-127) = 2^(s-1) is itself a bf16, so one multiplication does.
// NVFP4, E4M3 b (through its f16 value): 2^126 times it below 4 in magnitude
// and for NaN, else 2^126 then the value.
struct F4Scale {
  uint32_t c1, c2;
  bool two;
};

__device__ inline uint32_t bf16_pair(uint32_t h) { return h | (h << 16); }

__device__ inline F4Scale e8m0_scale(uint32_t s) {
  F4Scale f;
  f.c2 = bf16_pair(s == 0u ? 0x0040u : (s == 255u ? 0x7FC0u : s << 7));
  f.two = s > 128u && s != 255u;
  f.c1 = f.two ? 0x7E807E80u : bf16_pair(s == 255u ? 0x7FC0u : (s + 126u) << 7);
  return f;
}

__device__ inline F4Scale e4m3_scale(uint32_t b) {
  uint32_t h, r, r1;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)(b & 0xFFu)));
  const float f = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(f));
  // below 4 in magnitude (or NaN) 2^126 times the E4M3 value is a bf16: one multiplication
  const bool one = !(fabsf(f) >= 4.0f);
  const float g = f * 0x1p126f;   // exact: a power of two times a value with 4 significant bits
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(r1) : "f"(g));
  return F4Scale{one ? r1 : 0x7E807E80u, r, !one};
}

// 32 lanes x 16 consecutive fp32 columns: this thread's row, columns col..col+15.
__device__ inline void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ inline void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// map_w{0,1}_{cache,stage}: code banks [n_slots * rows, K/2] bytes, box 32 x 128;
// map_b64 / map_b16: the token operand [R, K] bf16 with 64- and 16-row boxes.
template <bool GATEUP, int CHUNK, bool NV>
__global__ void __launch_bounds__(kThreads, 1)
fp4_gemm_kernel(const __grid_constant__ CUtensorMap map_b64, const __grid_constant__ CUtensorMap map_b16,
                const __grid_constant__ CUtensorMap map_w0_cache, const __grid_constant__ CUtensorMap map_w1_cache,
                const __grid_constant__ CUtensorMap map_w0_stage, const __grid_constant__ CUtensorMap map_w1_stage,
                const F4Params p) {
  using S = F4Shape<CHUNK>;
  constexpr int kLS = S::kLoadStages, kAS = S::kAStages;
  constexpr int SB = NV ? 16 : kMxBlock;              // inputs per scale byte
  constexpr int kGroupKb = kScaleGroup * SB / kBK;    // k-blocks per 8 scale bytes (4 MXFP4, 2 NVFP4)
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_pref[kF4MaxE + 1];
  __shared__ int s_warp[kThreads / 32];
  __shared__ __align__(8) uint64_t load_full[kLS], load_empty[kLS], a_full[kAS], a_empty[kAS];
  __shared__ __align__(8) uint64_t tmem_full, tmem_empty, drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_ring = smem;                                   // kAS x {tile 0, tile 1}, 16 KB each
  uint8_t* load_ring = a_ring + kAS * 2 * kATile;           // kLS x {token tile, codes 0, codes 1}

  if (tid == 0) {
    for (int s = 0; s < kLS; ++s) {
      mbar_init(&load_full[s], 1);
      mbar_init(&load_empty[s], kDeqWarps + 1);   // the dequantisers read the codes, the MMA the token tile
    }
    for (int s = 0; s < kAS; ++s) {
      mbar_init(&a_full[s], kDeqWarps);
      mbar_init(&a_empty[s], 1);
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
  // chunks of CHUNK rows of every expert with rows (contains __syncthreads)
  build_group_prefix<CHUNK, (kF4MaxE + kThreads - 1) / kThreads>(p.counts, p.E, 0, INT_MAX, nullptr, s_pref, s_warp);
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
      int ls = 0;
      uint32_t lph = 0;
      bool l_armed[kLS] = {};
      uint32_t l_par[kLS] = {};
      const uint64_t wpol = l2_evict_first();   // codes are read once per chunk
      bool stop = false;
      for (int t = blockIdx.x; t < total && !stop && !*abort_flag; t += gridDim.x) {
        const F4Tile tl = f4_tile<CHUNK>(p, s_pref, t);
        if (!tl.ok) continue;
        const CUtensorMap* mw0 = tl.pool ? &map_w0_stage : &map_w0_cache;
        const CUtensorMap* mw1 = tl.pool ? &map_w1_stage : &map_w1_cache;
        const int row0 = f4_row<GATEUP>(p, tl, 0), row1 = f4_row<GATEUP>(p, tl, 1);
        const int n64 = tl.N >> 6, n16 = (tl.N & 63) >> 4;
        const uint32_t bytes = 2 * kCodeTile + (uint32_t)tl.N * (kBK * 2);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&load_empty[ls], lph ^ 1u, abort_flag)) {
            stop = true;
            break;
          }
          uint8_t* sB = load_ring + ls * S::kLoadBytes;
          uint8_t* sC = sB + S::kBTile;
          const int k0 = kb * kBK;
          mbar_expect_tx(&load_full[ls], bytes);
          l_armed[ls] = true;
          l_par[ls] = lph;
          tma_load_2d_hint(sC, mw0, &load_full[ls], kb * (kBK / 2), row0, wpol);
          tma_load_2d_hint(sC + kCodeTile, mw1, &load_full[ls], kb * (kBK / 2), row1, wpol);
          for (int i = 0; i < n64; ++i) tma_load_2d(sB + i * 64 * (kBK * 2), &map_b64, &load_full[ls], k0, tl.r0 + 64 * i);
          for (int i = 0; i < n16; ++i) {
            const int r = 64 * n64 + 16 * i;
            tma_load_2d(sB + r * (kBK * 2), &map_b16, &load_full[ls], k0, tl.r0 + r);
          }
          if (++ls == kLS) {
            ls = 0;
            lph ^= 1u;
          }
        }
      }
      // drain: every armed stage's copies land before the CTA can exit
      volatile int no_abort = 0;
      for (int s = 0; s < kLS; ++s)
        if (l_armed[s]) mbar_wait(&load_full[s], l_par[s], &no_abort);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int ls = 0, as = 0;
      uint32_t lph = 0, aph = 0, tphase = 0;
      bool issued = false, good = true;
      for (int t = blockIdx.x; t < total && good && !*abort_flag; t += gridDim.x) {
        const F4Tile tl = f4_tile<CHUNK>(p, s_pref, t);
        if (!tl.ok) continue;
        const uint32_t idesc = make_idesc(kBM, tl.N);
        if (!mbar_wait(&tmem_empty, tphase ^ 1u, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&load_full[ls], lph, abort_flag) || !mbar_wait(&a_full[as], aph, abort_flag)) {
            good = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(a_ring + as * 2 * kATile);
          const uint32_t b0 = smem_u32(load_ring + ls * S::kLoadBytes);
#pragma unroll
          for (int ks = 0; ks < kBK / kUK; ++ks) {
            const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
            const uint64_t bd = smem_desc(b0 + ks * kUK * 2);
            tc_mma(tmem_base, smem_desc(a0 + ks * kUK * 2), bd, idesc, acc);
            tc_mma(tmem_base + 256, smem_desc(a0 + kATile + ks * kUK * 2), bd, idesc, acc);
          }
          issued = true;
          tc_commit(&load_empty[ls]);
          tc_commit(&a_empty[as]);
          if (++ls == kLS) {
            ls = 0;
            lph ^= 1u;
          }
          if (++as == kAS) {
            as = 0;
            aph ^= 1u;
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
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------ epilogue (warps 2..9)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t tphase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const F4Tile tl = f4_tile<CHUNK>(p, s_pref, t);
      if (!tl.ok) {
        if (tid == 64) set_status(p.status, tl.entry < 0 ? MOE_DEV_ERR_UNBOUND : MOE_DEV_ERR_BAD_SLOT);
        continue;
      }
      if (!mbar_wait(&tmem_full, tphase, abort_flag)) break;
      tc_fence_after();
      const float* ts = p.ts[tl.pool];
      if (GATEUP) {
        const float tg = ts ? ts[(size_t)tl.slot * 3 + 0] : 1.0f, tu = ts ? ts[(size_t)tl.slot * 3 + 1] : 1.0f;
        const int f = tl.fb * kBM + quarter * 32 + lane;
        unsigned short* hcol = reinterpret_cast<unsigned short*>(p.h) + (size_t)tl.r0 * p.I + f;
        // 16-column chunks, alternating between the two warps of a lane quarter
#pragma unroll 1
        for (int c = half * 16; c < tl.N; c += 32) {
          uint32_t g[16], u[16];
          tmem_ld16(lane_addr + c, g);
          tmem_ld16(lane_addr + 256 + c, u);
          tmem_ld_wait();
          const int nv = min(16, tl.rows - c);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j < nv) {
              const float hv = silu_fast(__uint_as_float(g[j]) * tg) * (__uint_as_float(u[j]) * tu);
              hcol[(size_t)(c + j) * p.I] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
        }
      } else {
        const float td = ts ? ts[(size_t)tl.slot * 3 + 2] : 1.0f;
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
          const int f = tl.fb * 2 * kBM + m * kBM + quarter * 32 + lane;
#pragma unroll 1
          for (int c = half * 32; c < tl.N; c += 64) {
            uint32_t v[32];
            tmem_ld32(lane_addr + m * 256 + c, v);
            const int nv = min(32, tl.rows - c);
            const int prow = lane < nv ? p.perm[tl.r0 + c + lane] : 0;
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int yrow = __shfl_sync(0xffffffffu, prow, j);
              if (j < nv) p.y[(size_t)yrow * p.H + f] = __uint_as_float(v[j]) * td;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tmem_empty);
      tphase ^= 1u;
    }
  } else {
    // ------------------------------------------------ dequantisers (warps 10..17)
    const int dt = tid - 32 * (2 + kEpiWarps);
    const int row = dt & (kBM - 1), which = dt >> 7;   // operand tile 0 or 1
    int ls = 0, as = 0;
    uint32_t lph = 0, aph = 0;
    bool good = true;
    const int srow_bytes = p.K / SB;
    for (int t = blockIdx.x; t < total && good && !*abort_flag; t += gridDim.x) {
      const F4Tile tl = f4_tile<CHUNK>(p, s_pref, t);
      if (!tl.ok) continue;
      // this row's block scales: 8 bytes a group, the next group loaded one group ahead
      const uint8_t* srow = p.sc[tl.pool][which] + (size_t)(f4_row<GATEUP>(p, tl, which) + row) * srow_bytes;
      uint2 cur = __ldg(reinterpret_cast<const uint2*>(srow));
      uint2 nxt = kb_count > kGroupKb ? __ldg(reinterpret_cast<const uint2*>(srow + kScaleGroup)) : cur;
      for (int kb = 0; kb < kb_count; ++kb) {
        if (kb > 0 && kb % kGroupKb == 0) {
          cur = nxt;
          const int g = kb / kGroupKb + 1;
          if (g * kGroupKb < kb_count) nxt = __ldg(reinterpret_cast<const uint2*>(srow + g * kScaleGroup));
        }
        if (!mbar_wait(&load_full[ls], lph, abort_flag)) {
          good = false;
          break;
        }
        // the row's 32 code bytes; rows 4..7 of every 8 read their second half first, so that the eight
        // rows of a 16-byte load phase cover all 32 banks
        const uint8_t* codes = load_ring + ls * S::kLoadBytes + S::kBTile + which * kCodeTile + row * (kBK / 2);
        const int first = (row >> 2) & 1;
        const uint4 q0 = *reinterpret_cast<const uint4*>(codes + 16 * first);
        const uint4 q1 = *reinterpret_cast<const uint4*>(codes + 16 * (first ^ 1));
        const uint4 c0 = first ? q1 : q0;
        const uint4 c1 = first ? q0 : q1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&load_empty[ls]);
        if (++ls == kLS) {
          ls = 0;
          lph ^= 1u;
        }
        // this k-block's scale bytes within the group: 2 (MXFP4, one per 32 inputs) or 4 (NVFP4, per 16)
        const int sbyte = (kb % kGroupKb) * (kBK / SB);
        const uint32_t sw = (sbyte < 4 ? cur.x : cur.y) >> ((sbyte & 3) * 8);
        F4Scale sv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          // scale of inputs 16i .. 16i+15 of the k-block
          const uint32_t b = NV ? (sw >> (8 * i)) & 0xFFu : (sw >> (8 * (i >> 1))) & 0xFFu;
          sv[i] = NV ? e4m3_scale(b) : e8m0_scale(b);
        }
        if (!mbar_wait(&a_empty[as], aph ^ 1u, abort_flag)) {
          good = false;
          break;
        }
        uint8_t* arow = a_ring + as * 2 * kATile + which * kATile + row * 128;
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // chunk j = inputs 8j .. 8j+7; 16-byte chunks of a 128-byte row sit at j ^ (row % 8)
          const F4Scale& f = sv[j >> 1];
          *reinterpret_cast<uint4*>(arow + ((j ^ (row & 7)) << 4)) = expand8(cw[j], f.c1, f.c2, f.two);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
        if (++as == kAS) {
          as = 0;
          aph ^= 1u;
        }
      }
    }
    if (!good) *abort_flag = 1;
  }
  pdl_trigger();
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols));
}

// 2-D uint8 tensor [rows, inner] (inner contiguous), box = box_inner x 128 rows, no swizzle.
bool make_byte_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || base == nullptr || rows == 0) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, (cuuint32_t)kBM};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool GATEUP, int CHUNK, bool NV>
cudaError_t launch_one(int grid, cudaStream_t s, const CUtensorMap (&m)[6], const F4Params& p) {
  static std::atomic<unsigned char> attr[kMaxDevices];
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(fp4_gemm_kernel<GATEUP, CHUNK, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                F4Shape<CHUNK>::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  return launch_k(fp4_gemm_kernel<GATEUP, CHUNK, NV>, grid, kThreads, F4Shape<CHUNK>::kSmemBytes, s, m[0], m[1], m[2],
                  m[3], m[4], m[5], p);
}

template <bool GATEUP, bool NV>
cudaError_t launch_pass(bool thin, int grid, cudaStream_t s, const CUtensorMap (&m)[6], const F4Params& p) {
  return thin ? launch_one<GATEUP, 32, NV>(grid, s, m, p) : launch_one<GATEUP, 256, NV>(grid, s, m, p);
}

}  // namespace

bool fp4_gemm_ok(const MxParams& p, bool nv) {
  const int sb = nv ? 16 : kMxBlock;
  const bool b = p.b.n_slots > 0;
  const auto a8 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 7u) == 0; };
  // gate/up feature blocks of 128 rows, down blocks of 256; every row's scales in whole 8-byte groups
  return p.I % kBM == 0 && p.H % (2 * kBM) == 0 && (p.H / sb) % kScaleGroup == 0 && (p.I / sb) % kScaleGroup == 0 &&
         p.E <= kF4MaxE && a8(p.a.gate_s) && a8(p.a.up_s) && a8(p.a.down_s) &&
         (!b || (a8(p.b.gate_s) && a8(p.b.up_s) && a8(p.b.down_s)));
}

cudaError_t launch_fp4_gemm(const MxParams& p, bool nv, const __nv_bfloat16* x_perm, int T, cudaStream_t s) {
  const int R = T * p.k;
  const bool has_stage = p.b.n_slots > 0;
  const uint64_t H = (uint64_t)p.H, I = (uint64_t)p.I;
  const uint64_t na = (uint64_t)p.a.n_slots;
  const moe_pool_mxfp4& A = p.a;
  const moe_pool_mxfp4& B = has_stage ? p.b : p.a;   // no staging pool: its maps alias the cache pool's (never used)
  const uint64_t nbs = has_stage ? (uint64_t)p.b.n_slots : na;
  F4Params f = {};
  f.counts = p.counts;
  f.offsets = p.offsets;
  f.slot_table = p.slot_table;
  f.layer = p.layer;
  f.E = p.E;
  f.H = p.H;
  f.I = p.I;
  f.cache_slots = p.a.n_slots;
  f.staging_slots = has_stage ? p.b.n_slots : 0;
  f.ts[0] = p.ts_a;
  f.ts[1] = p.ts_b;
  f.perm = p.perm;
  f.h = p.h;
  f.y = p.y;
  f.status = p.status;
  const int grid = num_sms();
  const bool thin = T <= 32;   // a group has at most T rows (one per token)
  auto u8 = [](const void* q) { return static_cast<const uint8_t*>(q); };

  // gate/up: codes [slots * I, H/2]; scales [slots * I, H/sb]
  CUtensorMap m[6];
  if (!make_map(&m[0], x_perm, H, (uint64_t)R, 64) || !make_map(&m[1], x_perm, H, (uint64_t)R, 16) ||
      !make_byte_map(&m[2], A.gate_q, H / 2, na * I, 32) || !make_byte_map(&m[3], A.up_q, H / 2, na * I, 32) ||
      !make_byte_map(&m[4], B.gate_q, H / 2, nbs * I, 32) || !make_byte_map(&m[5], B.up_q, H / 2, nbs * I, 32))
    return cudaErrorInvalidValue;
  f.sc[0][0] = u8(A.gate_s);
  f.sc[0][1] = u8(A.up_s);
  f.sc[1][0] = u8(B.gate_s);
  f.sc[1][1] = u8(B.up_s);
  f.K = p.H;
  f.n_fb = p.I / kBM;
  cudaError_t err = nv ? launch_pass<true, true>(thin, grid, s, m, f) : launch_pass<true, false>(thin, grid, s, m, f);
  if (err != cudaSuccess) return err;

  // down: codes [slots * H, I/2], scales [slots * H, I/sb]; token operand = h
  if (!make_map(&m[0], p.h, I, (uint64_t)R, 64) || !make_map(&m[1], p.h, I, (uint64_t)R, 16) ||
      !make_byte_map(&m[2], A.down_q, I / 2, na * H, 32) || !make_byte_map(&m[4], B.down_q, I / 2, nbs * H, 32))
    return cudaErrorInvalidValue;
  m[3] = m[2];
  m[5] = m[4];
  f.sc[0][0] = f.sc[0][1] = u8(A.down_s);
  f.sc[1][0] = f.sc[1][1] = u8(B.down_s);
  f.K = p.I;
  f.n_fb = p.H / (2 * kBM);
  return nv ? launch_pass<false, true>(thin, grid, s, m, f) : launch_pass<false, false>(thin, grid, s, m, f);
}

}  // namespace moe
