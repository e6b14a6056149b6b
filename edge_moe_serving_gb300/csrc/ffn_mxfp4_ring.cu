// Block-scaled FP4 expert FFN for decode-sized calls: a weight-streaming ring
// kernel over MXFP4 or NVFP4 banks (FreeToken paper, section 3.2: grouped
// evaluation of the GPU execution set through the (layer, expert) slot;
// section 4.1: expert kernels dequantise in-kernel; section 5.1: the routed
// experts of DeepSeek-V4-Flash are MXFP4, those of GLM-5.2 and of the laptop
// Qwen3.6 build NVFP4).  Every routed row is its own instance.
//
// One launch, one CTA per SM.  A producer thread streams "units" (a few
// consecutive weight rows: their FP4 code bytes and E8M0 scale bytes) into a
// ring of shared-memory stages with cp.async.bulk (L2 evict-first: weights
// are read once per call); eight consumer warps each reduce every eighth
// unit (the consumers' dependent convert-and-multiply chains bound the
// stream, so more warps help; eight is the measured best within the
// register file).  Phase A streams gate and up rows and writes
// h = bf16(silu(g) * u);
// phase B streams down rows and writes y.  Per-instance counters let a
// consumer start the down rows of an expert as soon as every CTA finished its
// gate/up rows of that expert, while the producer keeps streaming.
//
// Arithmetic of one 32-input code vector (16 code bytes):
//   * the token's activations of the block are rescaled once per call by a
//     power of two g (largest magnitude into [2^7, 2^8)) and rounded to f16,
//     exact for every element within 2^22 of the block's largest;
//   * the hardware converts each code byte to two f16 E2M1 values (exact);
//   * f16 x f16 products are exact in fp32 and are accumulated in fp32;
//   * MXFP4 (one E8M0 scale s per 32 inputs): the vector's sum is multiplied
//     by 2^(s - 127) / g (exact: a power of two) and added to the row's fp32
//     accumulator, so the result is the dot product with the dequantised row
//     up to fp32 summation order, for any E8M0 scale including 2^-127, 2^127
//     and NaN;
//   * NVFP4 (one E4M3 scale per 16 inputs, one fp32 scale per bank): each
//     half's sum is multiplied by its E4M3 value (converted exactly by the
//     hardware) times 1/g, and the row's sum by the bank's tensor scale.
#include <climits>

#include "decode_front.cuh"
#include "front_warp.cuh"
#include "mxfp4.cuh"
#include "ring_gemv.cuh"

namespace moe {
namespace {

constexpr int kMxStages = 8;   // 8 x 18 KB per SM, one stage per consumer warp: measured best of 6, 8, 11 and 12
constexpr int kMxCodeBytes = 16384;     // code bytes per stage (both banks of a gate/up unit)
constexpr int kMxScaleOff = 16384;      // scale bytes follow the codes
constexpr int kMxStageBytes = 18432;    // 16 KB of codes + up to 2 KB of scales (NVFP4)
constexpr int kMxCW = 8;                // consumer warps (one stage each)
constexpr int kMxThreads = (kMxCW + 1) * 32;
constexpr int kMxSmem = kMxStages * kMxStageBytes + 128;
static_assert(kMxStages % kMxCW == 0, "each ring stage must have one consumer warp");
static_assert(kMxStageBytes % 128 == 0, "stages stay 128-byte aligned");

// Rows per unit: gate/up units hold U rows of each bank (U * K/2 code bytes
// per bank), down units U rows; at most 16.
__host__ __device__ inline int mx_rows_gateup(int H) { return min(16, kMxCodeBytes / H); }
__host__ __device__ inline int mx_rows_down(int I) { return min(16, 2 * kMxCodeBytes / I); }

// The token's activations of the V blocks a lane owns (blocks lane + 32c,
// inputs 32v .. 32v+31), rescaled by a power of two per block and rounded to
// f16: a[c][i] holds inputs 32v + 2i (low half) and 32v + 2i + 1 (high
// half); inv[c] is the block's back-scale 1/g.
template <int V>
struct ActRegs {
  uint32_t a[V][16];
  float inv[V];
};

__device__ inline uint32_t bf16_exp(uint32_t packed_half) { return (packed_half >> 7) & 0xFFu; }

// Loads and rescales one block of 32 bf16 activations (64 bytes at `src`,
// read through L2: h was written by other CTAs of this launch).
__device__ inline void stage_block(const __nv_bfloat16* src, uint32_t (&a)[16], float& inv) {
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) raw[i] = __ldcg(reinterpret_cast<const uint4*>(src) + i);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[4 * i + 0] = raw[i].x;
    w[4 * i + 1] = raw[i].y;
    w[4 * i + 2] = raw[i].z;
    w[4 * i + 3] = raw[i].w;
  }
  uint32_t emax = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) emax = max(emax, max(bf16_exp(w[i] & 0xFFFFu), bf16_exp(w[i] >> 16)));
  // g = 2^n with n = 134 - emax, so the largest magnitude lands in [2^7, 2^8);
  // n is kept within the normal exponents (blocks of zeros or subnormals get
  // 2^127, a block holding an inf or NaN 2^-121: its sum is inf or NaN anyway)
  const int n = min(127, max(-126, 134 - (int)emax));
  const float g = __uint_as_float((uint32_t)(n + 127) << 23);
  inv = (n == 127) ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - n) << 23);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __half lo = __float2half_rn(bf16_lo(w[i]) * g);
    const __half hi = __float2half_rn(bf16_hi(w[i]) * g);
    a[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
}

template <int V>
__device__ inline void stage_row(const __nv_bfloat16* row, ActRegs<V>& r) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < V; ++c) stage_block(row + (size_t)(lane + 32 * c) * kMxBlock, r.a[c], r.inv[c]);
}

// Four code bytes -> four f16 pairs (E2M1 values, exact): pair b holds the
// elements of byte b, low nibble in the low half.
__device__ inline void e2m1x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// s0 += w.lo * a.lo, s1 += w.hi * a.hi: f16 products (exact in fp32) added in fp32.
__device__ inline void fma_f16_pair(uint32_t w, uint32_t a, float& s0, float& s1) {
  asm("{\n .reg .b16 wl, wh, al, ah;\n mov.b32 {wl, wh}, %2;\n mov.b32 {al, ah}, %3;\n"
      " fma.rn.f32.f16 %0, wl, al, %0;\n fma.rn.f32.f16 %1, wh, ah, %1;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "r"(w), "r"(a));
}

// Sums of the products of one code vector with its staged activations: lo
// over inputs 0..15 (words x, y), hi over inputs 16..31 (words z, w).
__device__ inline void block_dot(const uint4& q, const uint32_t (&a)[16], float& lo, float& hi) {
  float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
  uint32_t h[4];
  e2m1x8(q.x, h);
  fma_f16_pair(h[0], a[0], s0, s1);
  fma_f16_pair(h[1], a[1], s0, s1);
  fma_f16_pair(h[2], a[2], s0, s1);
  fma_f16_pair(h[3], a[3], s0, s1);
  e2m1x8(q.z, h);
  fma_f16_pair(h[0], a[8], s2, s3);
  fma_f16_pair(h[1], a[9], s2, s3);
  fma_f16_pair(h[2], a[10], s2, s3);
  fma_f16_pair(h[3], a[11], s2, s3);
  e2m1x8(q.y, h);
  fma_f16_pair(h[0], a[4], s0, s1);
  fma_f16_pair(h[1], a[5], s0, s1);
  fma_f16_pair(h[2], a[6], s0, s1);
  fma_f16_pair(h[3], a[7], s0, s1);
  e2m1x8(q.w, h);
  fma_f16_pair(h[0], a[12], s2, s3);
  fma_f16_pair(h[1], a[13], s2, s3);
  fma_f16_pair(h[2], a[14], s2, s3);
  fma_f16_pair(h[3], a[15], s2, s3);
  lo = s0 + s1;
  hi = s2 + s3;
}

// Two E4M3 scale bytes (the low byte scales inputs 0..15 of the vector) ->
// their values, exactly (every E4M3 value is an f16 value; NaN stays NaN).
__device__ inline float2 e4m3x2(uint16_t b) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
  return make_float2(__half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu))),
                     __half2float(__ushort_as_half((unsigned short)(h >> 16))));
}

// The vector's contribution to a row: MXFP4 scales the whole vector by its
// E8M0 power of two, NVFP4 each half by its E4M3 value; inv undoes the
// activations' power-of-two rescaling.
template <bool NV>
__device__ inline float vector_term(const uint4& q, const uint32_t (&a)[16], const uint8_t* srow, int v, float inv) {
  float lo, hi;
  block_dot(q, a, lo, hi);
  if (NV) {
    const float2 sc = e4m3x2(*reinterpret_cast<const uint16_t*>(srow + 2 * v));
    return fmaf(lo, sc.x * inv, hi * (sc.y * inv));
  }
  return (lo + hi) * (e8m0(srow[v]) * inv);
}


// The ring's barriers, the CTA's abort flag and its bookkeeping.
struct MxRing {
  uint64_t full_bar[kMxStages];
  uint64_t empty_bar[kMxStages];
  int abort;
};

struct MxRingState {
  int base;          // ring index of the current phase's first unit
  int armed_last;    // producer: last ring index with copies in flight
  int last_issued;   // producer: last ring index it completed or armed
  bool stored;       // consumer: issued fused-fill stores (waited for before exit)
};

// The call's instances (one per routed row, at most kFp4RingMaxRows),
// looked up once by the whole CTA so that the producer and the consumers read
// their sources from shared memory: expert, dispatch position, token-major
// expert row and slot-table entry.
struct MxInsts {
  int e[kFp4RingMaxRows], pos[kFp4RingMaxRows], yrow[kFp4RingMaxRows], entry[kFp4RingMaxRows];
  int fill[kFp4RingMaxRows];   // cache slot the instance's expert is admitted to while it streams, or -1
  int n;
};

// One phase over the call's instances: units of U consecutive rows,
// grid-strided over the CTAs (CTA b takes units b, b + G, ...).
template <bool GATEUP, int V, bool NV>
__device__ void mx_phase(const MxParams& p, const MxInsts& in, int* s_cnt, uint8_t* ring, MxRing& rg,
                         MxRingState& st, bool producer) {
  constexpr int NB = GATEUP ? 2 : 1;
  constexpr int KC = 1024 * V;                                   // inputs per weight row
  constexpr int SB = NV ? 16 : kMxBlock;                        // inputs per scale byte
  constexpr int KBC = KC / SB;                                   // scale bytes per row
  constexpr int UC = GATEUP ? 16 / V : (32 / V < 16 ? 32 / V : 16);   // rows per unit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = GATEUP ? p.H : p.I;          // inputs per weight row
  const int NTASK = GATEUP ? p.I : p.H;      // rows per expert
  const int KB = K / SB;                     // scale bytes per row
  const int U = GATEUP ? mx_rows_gateup(p.H) : mx_rows_down(p.I);
  const int upi = (NTASK + U - 1) / U;
  const int G = gridDim.x;
  const int n_local = local_units(in.n * upi);
  const int base = st.base;
  volatile int* abort_flag = &rg.abort;
  st.base += n_local;
  const int bank_codes = kMxCodeBytes / NB;  // offset of the second bank's codes in a stage
  const int bank_scales = bank_codes * 2 / SB;                    // offset of the second bank's scales

  if (producer) {
    int cur_j = -1;
    bool ok = false;
    MxRows rw;
    const uint64_t pol = l2_evict_first();
    for (int i = 0; i < n_local && !*abort_flag; ++i) {
      const int u = (int)blockIdx.x + i * G;
      const int j = u / upi, n0 = (u - j * upi) * U;
      if (j != cur_j) {
        cur_j = j;
        ok = mx_resolve<GATEUP, SB>(p, in.entry[j], &rw, nullptr);
      }
      const int ri = base + i;
      const int stage = ri % kMxStages;
      const uint32_t use = (uint32_t)(ri / kMxStages);
      if (!ring_wait(&rg.empty_bar[stage], (use & 1u) ^ 1u, abort_flag)) break;
      st.last_issued = ri;
      if (!ok) {
        // unbound or bad slot: complete the stage's phase without data
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&rg.full_bar[stage])) : "memory");
        continue;
      }
      const int rows = min(U, NTASK - n0);
      const uint32_t cb = (uint32_t)rows * (uint32_t)(K / 2), sb = (uint32_t)rows * (uint32_t)KB;
      uint8_t* dst = ring + (size_t)stage * kMxStageBytes;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&rg.full_bar[stage])),
                   "r"(NB * (cb + sb))
                   : "memory");
      bulk_g2s_hint(dst, rw.q0 + (size_t)n0 * (K / 2), cb, &rg.full_bar[stage], pol);
      bulk_g2s_hint(dst + kMxScaleOff, rw.s0 + (size_t)n0 * KB, sb, &rg.full_bar[stage], pol);
      if (GATEUP) {
        bulk_g2s_hint(dst + bank_codes, rw.q1 + (size_t)n0 * (K / 2), cb, &rg.full_bar[stage], pol);
        bulk_g2s_hint(dst + kMxScaleOff + bank_scales, rw.s1 + (size_t)n0 * KB, sb, &rg.full_bar[stage], pol);
      }
      st.armed_last = ri;
    }
    return;
  }

  // consumers: this warp's units are the ring indices ri = base + i with ri % kMxCW == warp
  const int ua = mx_rows_gateup(p.H);
  const unsigned need = (unsigned)min(G, (p.I + ua - 1) / ua);   // CTAs holding gate/up units of an instance
  ActRegs<V> act;
  int cur_j = -1, pos = 0, yrow = 0, staged_tok = -1, fill_v = -1;
  bool ok = false;
  MxRows rw;   // the rows sit in the stage; the tensor scales are read from here
  const size_t rows_per_slot = GATEUP ? (size_t)p.I : (size_t)p.H;
  const int i0 = ((warp - base) % kMxCW + kMxCW) % kMxCW;
  for (int i = i0; i < n_local; i += kMxCW) {
    const int u = (int)blockIdx.x + i * G;
    const int j = u / upi, n0 = (u - j * upi) * U;
    if (j != cur_j) {
      cur_j = j;
      pos = in.pos[j];
      yrow = in.yrow[j];
      fill_v = in.fill[j];
      if (!GATEUP) {
        // h of instance j is complete once every CTA holding its gate/up units has published them
        if (lane == 0) {
          unsigned long long t0 = 0;
          for (uint32_t it = 0; ld_acquire_u32(p.inst_done + j) < need; ++it) {
            if ((it & 15) == 15) {
              if (*abort_flag) break;
              const unsigned long long now = gtimer();
              if (t0 == 0) {
                t0 = now;
              } else if (now - t0 > kGridWaitNs) {
                *abort_flag = 1;
                break;
              }
            }
          }
        }
        __syncwarp();
        if (*abort_flag) break;
      }
      // any warp meeting an unbound expert reports it (its units are spread over warps)
      ok = mx_resolve<GATEUP, SB>(p, in.entry[j], &rw, lane == 0 ? p.status : nullptr);
      if (ok) {
        if (!GATEUP) {
          stage_row<V>(p.h + (size_t)pos * p.I, act);
        } else if (yrow / p.k != staged_tok) {
          // every gate/up instance of the token reads the same activations: staged once
          staged_tok = yrow / p.k;
          stage_row<V>(p.x + (size_t)staged_tok * p.H, act);
        }
      }
    }
    const int ri = base + i;
    const int stage = ri % kMxStages;
    const uint32_t use = (uint32_t)(ri / kMxStages);
    if (!ring_wait(&rg.full_bar[stage], use & 1u, abort_flag)) break;
    const bool store = ok && fill_v >= 0;
    if (store && lane == 0) {
      // this expert is being admitted to the cache: write the unit's code and scale rows to its slot
      const uint8_t* sw = ring + (size_t)stage * kMxStageBytes;
      const int rows = min(UC, NTASK - n0);
      const size_t row0 = (size_t)fill_v * rows_per_slot + n0;
      const uint32_t cb = (uint32_t)rows * (uint32_t)(K / 2), sb = (uint32_t)rows * (uint32_t)KB;
      uint8_t* q0 = static_cast<uint8_t*>(const_cast<void*>(GATEUP ? p.a.gate_q : p.a.down_q));
      uint8_t* s0 = static_cast<uint8_t*>(const_cast<void*>(GATEUP ? p.a.gate_s : p.a.down_s));
      bulk_s2g(q0 + row0 * (K / 2), sw, cb);
      bulk_s2g(s0 + row0 * KB, sw + kMxScaleOff, sb);
      if (GATEUP) {
        uint8_t* q1 = static_cast<uint8_t*>(const_cast<void*>(p.a.up_q));
        uint8_t* s1 = static_cast<uint8_t*>(const_cast<void*>(p.a.up_s));
        bulk_s2g(q1 + row0 * (K / 2), sw + bank_codes, cb);
        bulk_s2g(s1 + row0 * KB, sw + kMxScaleOff + bank_scales, sb);
      }
      bulk_commit();
      st.stored = true;
    }
    if (ok) {
      const uint8_t* sw = ring + (size_t)stage * kMxStageBytes;
      const int rows = min(UC, NTASK - n0);
      for (int r = 0; r < rows; ++r) {
        const uint8_t* qrow = sw + (size_t)r * (KC / 2);
        const uint8_t* srow = sw + kMxScaleOff + r * KBC;
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const int v = lane + 32 * c;
          acc0 += vector_term<NV>(*reinterpret_cast<const uint4*>(qrow + v * 16), act.a[c], srow, v, act.inv[c]);
          if (GATEUP)
            acc1 += vector_term<NV>(*reinterpret_cast<const uint4*>(qrow + bank_codes + v * 16), act.a[c],
                                    srow + bank_scales, v, act.inv[c]);
        }
        acc0 = warp_sum(acc0) * rw.t0;
        if (GATEUP) {
          acc1 = warp_sum(acc1) * rw.t1;
          if (lane == 0) p.h[(size_t)pos * p.I + n0 + r] = __float2bfloat16_rn(silu(acc0) * acc1);
        } else if (lane == 0) {
          p.y[(size_t)yrow * p.H + n0 + r] = acc0;
        }
      }
    }
    if (GATEUP) {
      // publish instance j once this CTA's gate/up units of it are all done (as in the bf16 ring kernel:
      // a CTA-scope acquire-release count, then one GPU-scope release add by the completing warp)
      __syncwarp();
      if (lane == 0) {
        const int lo = j * upi, hi = lo + upi;
        const int first = lo + (((int)blockIdx.x - lo) % G + G) % G;
        const int mine = first < hi ? (hi - 1 - first) / G + 1 : 0;
        if (atom_add_acq_rel_cta(&s_cnt[j], 1) + 1 == mine)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.inst_done + j) : "memory");
      }
    }
    if (store && lane == 0) bulk_wait_read_all();   // the stores have read the stage
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&rg.empty_bar[stage])) : "memory");
  }
}

template <int VA, int VB, bool NV>
__global__ void __launch_bounds__(kMxThreads, 1) mx_ring_kernel(MxParams p) {
  extern __shared__ __align__(128) uint8_t ring_raw[];
  __shared__ MxRing rg;
  __shared__ int s_pref[kMaxE + 1];
  __shared__ int s_warp[kMxThreads / 32];
  __shared__ int s_cnt[kFp4RingMaxRows];
  __shared__ MxInsts in;
  // the ring is the dynamic shared array itself: pointers derived from it keep the shared
  // address space, so stage reads compile to shared-memory loads
  uint8_t* ring = ring_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rg.full_bar[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rg.empty_bar[s])));
    }
    rg.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kFp4RingMaxRows) s_cnt[tid] = 0;
  pdl_wait();
  build_group_prefix<1, kMaxE / 32>(p.counts, p.E, 0, INT_MAX, nullptr, s_pref, s_warp);   // ends with __syncthreads
  if (tid < kFp4RingMaxRows) {
    // instance tid: the tid-th routed row in dispatch order (expert ids ascending)
    const int n = min(s_pref[p.E], kFp4RingMaxRows);
    if (tid == 0) in.n = n;
    if (tid < n) {
      const int e = find_group(s_pref, p.E, tid);
      const int pos = p.offsets[e] + (tid - s_pref[e]);
      in.e[tid] = e;
      in.pos[tid] = pos;
      in.yrow[tid] = p.perm[pos];   // token-major expert row: token yrow / k, its (yrow % k)-th expert
      in.entry[tid] = p.slot_table[p.layer * p.E + e];
      in.fill[tid] = -1;
    }
  }
  __syncthreads();
  const bool producer = warp == kMxCW;
  MxRingState st = {0, -1, -1, false};
  if (!producer || lane == 0) {
    mx_phase<true, VA, NV>(p, in, s_cnt, ring, rg, st, producer);
    if (!rg.abort) mx_phase<false, VB, NV>(p, in, s_cnt, ring, rg, st, producer);
    if (producer && st.armed_last >= 0) {
      // drain: the copies of the last ring round land before the CTA exits
      volatile int no_abort = 0;
      for (int q = st.last_issued; q >= 0 && q > st.last_issued - kMxStages; --q)
        ring_wait(&rg.full_bar[q % kMxStages], (uint32_t)(q / kMxStages) & 1u, &no_abort);
    }
  }
  pdl_trigger();
  __syncthreads();
  if (rg.abort && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
}

template <int VA, int VB, bool NV>
cudaError_t launch_vv(const MxParams& p, cudaStream_t s) {
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = ensure_smem(mx_ring_kernel<VA, VB, NV>, kMxSmem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_k(mx_ring_kernel<VA, VB, NV>, num_sms(), kMxThreads, kMxSmem, s, p);
}

template <int VA, bool NV>
cudaError_t launch_va(const MxParams& p, cudaStream_t s) {
  switch (p.I / 1024) {
    case 1: return launch_vv<VA, 1, NV>(p, s);
    case 2: return launch_vv<VA, 2, NV>(p, s);
    default: return launch_vv<VA, 4, NV>(p, s);
  }
}

template <bool NV>
cudaError_t launch_fmt(const MxParams& p, cudaStream_t s) {
  switch (p.H / 1024) {
    case 1: return launch_va<1, NV>(p, s);
    case 2: return launch_va<2, NV>(p, s);
    default: return launch_va<4, NV>(p, s);
  }
}

// ---------------------------------------------------------------- one-launch decode over FP4 banks
// The layer for one token in one cooperative launch, the FP4 counterpart of
// the bf16 decode kernel (FreeToken paper, section 3.2: router, cache lookup
// and q* split, grouped evaluation, combine; section 4.1: device-side cache
// control; section 5.1: FP4 expert banks):
//
//   phase R   every CTA scores its router rows (bulk-copied into the ring's
//             shared memory with the token row and the cache state the
//             decision reads) and writes the logits
//   barrier   bounded grid-wide barrier
//   route     warp 0 of every CTA runs the same top-k and looks up which
//             routed experts the cache pool holds: that fixes every
//             instance's source (a hit its cache slot, a miss its staging
//             slot), so the producer starts streaming; warp 0 then decides
//             the fills and their victims, and CTA 0 commits the decision
//   FFN       the ring kernel's gate/up and down phases over the instances;
//             an admitted expert is written to its victim slot from the
//             ring as it streams (bulk shared -> global stores of each unit)
//   barrier   bounded grid-wide barrier: every expert row is written
//   combine   out = bf16(sum over j of w_j * y_j), fp32 FMAs in j order,
//             each CTA a slice of the columns
//
// It computes exactly what the router, bind, fill copy, dispatch, FFN and
// combine launches compute for such a call.

constexpr int kF4DecMaxSlots = 512;   // cache-pool slots whose state the decision copies (the ring takes the rest)

struct __align__(16) F4DecShared {
  int32_t table[kMaxRouteE];       // this layer's slot-table row
  uint32_t stamp[kF4DecMaxSlots];  // the cache pool's stamps
  int32_t owner[kF4DecMaxSlots];   // and owners
  uint32_t hitmap[kF4DecMaxSlots / 32];
  FrontDecision fr;
  float red[kMxThreads / 32][kDecMaxRows][kDecMaxT];
  float bias[kDecMaxRows];
  uint64_t rbar;
  uint32_t clock;
};

constexpr int kBarF4Consumers = 1;   // the consumer warps, once the decision is complete
constexpr int kBarF4Stream = 2;      // warp 0 -> producer warp: the instances' sources are known

template <int VA, int VB, bool NV>
__global__ void __launch_bounds__(kMxThreads, 1) decode_fp4_kernel(MxParams p, Fp4DecodeArgs d) {
  extern __shared__ __align__(128) uint8_t ring_raw[];
  __shared__ MxRing rg;
  __shared__ int s_cnt[kFp4RingMaxRows];
  __shared__ MxInsts in;
  __shared__ F4DecShared sh;
  uint8_t* ring = ring_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E, H = p.H, G = gridDim.x, b = blockIdx.x;
  const int n_my = b < E ? (E - 1 - b) / G + 1 : 0;
  const int n_slots = d.c.cache.n_slots, base = p.layer * E;
  const int rows_per_cta = (E + G - 1) / G;
  // ring bytes during the prologue: router rows (fp32) | token row (bf16)
  float* wrow = reinterpret_cast<float*>(ring);
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(wrow + (size_t)rows_per_cta * H);
  p.inst_done = d.grid_count + 4;

  if (tid == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rg.full_bar[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rg.empty_bar[s])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.rbar)));
    rg.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kFp4RingMaxRows) s_cnt[tid] = 0;
  __syncthreads();
  pdl_wait();
  // ---------------------------------------------------------------- phase R
  const bool table_bulk = (reinterpret_cast<uintptr_t>(d.c.slot_table + base) & 15) == 0;
  const bool slot_bulk = ((reinterpret_cast<uintptr_t>(d.c.stamp) | reinterpret_cast<uintptr_t>(d.c.owner)) & 15) == 0;
  const int table_bulk_n = table_bulk ? (E & ~3) : 0;
  const int slot_bulk_n = slot_bulk ? (n_slots & ~3) : 0;
  if (tid == 0) {
    const uint32_t row_bytes = (uint32_t)H * 4u, x_bytes = (uint32_t)H * 2u;
    const uint32_t bytes = row_bytes * (uint32_t)n_my + x_bytes + 4u * (uint32_t)table_bulk_n + 8u * (uint32_t)slot_bulk_n;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&sh.rbar)), "r"(bytes)
                 : "memory");
    for (int i = 0; i < n_my; ++i)
      bulk_g2s(wrow + (size_t)i * H, d.w_router + (size_t)(b + i * G) * H, row_bytes, &sh.rbar);
    bulk_g2s(xs, p.x, x_bytes, &sh.rbar);
    if (table_bulk_n > 0) bulk_g2s(sh.table, d.c.slot_table + base, 4u * table_bulk_n, &sh.rbar);
    if (slot_bulk_n > 0) {
      bulk_g2s(sh.stamp, d.c.stamp, 4u * slot_bulk_n, &sh.rbar);
      bulk_g2s(sh.owner, d.c.owner, 4u * slot_bulk_n, &sh.rbar);
    }
  } else if (warp == kMxCW) {
    for (int e = table_bulk_n + lane; e < E; e += 32) sh.table[e] = __ldcg(d.c.slot_table + base + e);
    for (int v = slot_bulk_n + lane; v < n_slots; v += 32) {
      sh.stamp[v] = __ldcg(d.c.stamp + v);
      sh.owner[v] = __ldcg(d.c.owner + v);
    }
    if (lane == 0) sh.clock = __ldcg(d.c.clock);
  } else if (warp == 1 && lane < n_my) {
    sh.bias[lane] = d.bias ? __ldg(d.bias + b + lane * G) : 0.0f;
  }
  if (!bounded_wait(&sh.rbar, 0u, &rg.abort)) rg.abort = 1;
  __syncthreads();
  if (n_my > 0 && !rg.abort) {
    constexpr int NW = kMxThreads / 32;
    switch (n_my) {
      case 1: router_rows_block<1, 1, NW>(wrow, xs, H, 1, E, sh.red, sh.bias, d.logits, b, G); break;
      case 2: router_rows_block<2, 1, NW>(wrow, xs, H, 1, E, sh.red, sh.bias, d.logits, b, G); break;
      case 3: router_rows_block<3, 1, NW>(wrow, xs, H, 1, E, sh.red, sh.bias, d.logits, b, G); break;
      default: router_rows_block<4, 1, NW>(wrow, xs, H, 1, E, sh.red, sh.bias, d.logits, b, G); break;
    }
  }
  // ---------------------------------------------------------------- route, residency
  if (grid_barrier(d.grid_count + 0, &rg.abort)) {
    const int R = p.k;
    if (warp == 0) {
      const FrontLane fl = front_route(d.logits, 1, R, E, n_slots, sh.table, sh.fr);
      // one token: its R distinct experts in ascending order, instance j = routed row j
      if (lane < R) {
        in.e[lane] = fl.e;
        in.pos[lane] = lane;
        in.yrow[lane] = sh.fr.perm[lane];
        in.entry[lane] = fl.hit ? fl.entry : (int)(MOE_STAGING_TAG | (base + fl.e));
      }
      if (lane == 0) in.n = R;
      __syncwarp();
      asm volatile("bar.arrive %0, %1;" ::"n"(kBarF4Stream), "n"(64) : "memory");   // the producer may stream
      front_residency(fl, n_slots, p.layer, sh.stamp, sh.owner, sh.clock, d.phi_q16, d.min_fill, d.policy, d.seed,
                      sh.fr, sh.hitmap);
      // admitted experts are written to their victim slots as they stream (instance j = position j)
      const bool fills = d.fill.n > 0 && lane < R && sh.fr.u_kind[lane] == kFrontFill;
      if (lane < R) in.fill[lane] = fills ? sh.fr.u_slot[lane] : -1;
      if (fills && b == 0 && d.fill.n == 7) {
        // NVFP4: the slot's three tensor scales
        const float* ts_src = reinterpret_cast<const float*>(d.fill.src[6]) + (size_t)(base + fl.e) * 3;
        float* ts_dst = reinterpret_cast<float*>(d.fill.dst[6]) + (size_t)sh.fr.u_slot[lane] * 3;
        for (int q = 0; q < 3; ++q) ts_dst[q] = ts_src[q];
      }
      __syncwarp();
    }
    if (warp == kMxCW) {
      asm volatile("bar.sync %0, %1;" ::"n"(kBarF4Stream), "n"(64) : "memory");
    } else {
      asm volatile("bar.sync %0, %1;" ::"n"(kBarF4Consumers), "n"(kMxCW * 32) : "memory");
      // routing outputs, spread over the CTAs; CTA 0 commits the decision (every CTA read the
      // pre-call state before the barrier)
      for (int e = b + tid * G; e <= E; e += G * kMxCW * 32) {
        int lo, hi;
        dispatch_range(sh.fr.sorted, R, e, lo, hi);
        d.offsets[e] = lo;
        if (e < E) d.counts[e] = hi - lo;
      }
      if (b == (G > 1 ? 1 : 0) && tid < R) {
        d.topk_ids[tid] = sh.fr.ids[tid];
        d.topk_w[tid] = sh.fr.w[tid];
        d.perm[tid] = sh.fr.perm[tid];
        d.inv_perm[tid] = sh.fr.inv_perm[tid];
      }
      if (b == 0 && warp == 0) front_commit(sh.fr, d.c, p.layer, d.stats, p.status);
    }
    // ---------------------------------------------------------------- FFN
    const bool producer = warp == kMxCW;
    MxRingState st = {0, -1, -1, false};
    if (!producer || lane == 0) {
      mx_phase<true, VA, NV>(p, in, s_cnt, ring, rg, st, producer);
      if (!rg.abort) mx_phase<false, VB, NV>(p, in, s_cnt, ring, rg, st, producer);
      if (producer && st.armed_last >= 0) {
        volatile int no_abort = 0;
        for (int q = st.last_issued; q >= 0 && q > st.last_issued - kMxStages; --q)
          ring_wait(&rg.full_bar[q % kMxStages], (uint32_t)(q / kMxStages) & 1u, &no_abort);
      }
    }
    if (st.stored && lane == 0) bulk_wait_all();   // the fused fills' writes complete before the barrier
    // ---------------------------------------------------------------- combine
    if (grid_barrier(d.grid_count + 1, &rg.abort)) {
      const int H4 = H >> 2;
      for (int c4 = b * kMxThreads + tid; c4 < H4; c4 += G * kMxThreads) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < R; ++j) {
          const float w = sh.fr.w[j];
          const float4 y = __ldcg(reinterpret_cast<const float4*>(p.y + (size_t)j * H) + c4);
          acc.x = fmaf(w, y.x, acc.x);
          acc.y = fmaf(w, y.y, acc.y);
          acc.z = fmaf(w, y.z, acc.z);
          acc.w = fmaf(w, y.w, acc.w);
        }
        uint2 o;
        o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.x)) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.y)) << 16);
        o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.z)) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.w)) << 16);
        reinterpret_cast<uint2*>(d.out)[c4] = o;
      }
    }
  }
  pdl_trigger();
  __syncthreads();
  if (rg.abort && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
}

// rows of 1024, 2048 or 4096 inputs: 1, 2 or 4 blocks per lane, whose staged activations stay in registers
inline bool v_ok(int K) { return K == 1024 || K == 2048 || K == 4096; }
inline bool al16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }
inline bool pool_ok(const moe_pool_mxfp4& b) {
  return b.n_slots == 0 || (al16(b.gate_q) && al16(b.up_q) && al16(b.down_q) && al16(b.gate_s) && al16(b.up_s) &&
                            al16(b.down_s));
}

}  // namespace

// At most kFp4RingMaxRows routed rows (each its own instance; its token's
// activations stay in registers), rows of 1024, 2048 or 4096 inputs (each
// lane owns whole 32-input code vectors), 16-byte aligned banks (bulk copies
// of code and scale rows).
bool fp4_ring_ok(const MxParams& p, int T, bool nv) {
  (void)nv;
  return T >= 1 && (long long)T * p.k <= kFp4RingMaxRows && v_ok(p.H) && v_ok(p.I) && pool_ok(p.a) &&
         pool_ok(p.b) && p.inst_done != nullptr;
}

bool fp4_decode_ok(const MxParams& p, int T, int n_slots) {
  const int G = num_sms();
  const int rows = (p.E + G - 1) / G;
  return T == 1 && p.k <= 32 && p.E <= kMaxRouteE && rows <= kDecMaxRows && n_slots >= 1 &&
         n_slots <= kF4DecMaxSlots && v_ok(p.H) && v_ok(p.I) && pool_ok(p.a) && pool_ok(p.b) &&
         (size_t)rows * p.H * 4 + (size_t)p.H * 2 <= (size_t)kMxStages * kMxStageBytes;
}

template <int VA, int VB, bool NV>
cudaError_t launch_decode_vv(const MxParams& p, const Fp4DecodeArgs& a, cudaStream_t s) {
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = ensure_smem(decode_fp4_kernel<VA, VB, NV>, kMxSmem, smem_set);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(a.grid_count, 0, (4 + (size_t)p.k) * sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kMxThreads);
  cfg.dynamicSmemBytes = kMxSmem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: the grid barriers and the cross-CTA waits complete
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, decode_fp4_kernel<VA, VB, NV>, p, a));
}

template <int VA, bool NV>
cudaError_t launch_decode_va(const MxParams& p, const Fp4DecodeArgs& a, cudaStream_t s) {
  switch (p.I / 1024) {
    case 1: return launch_decode_vv<VA, 1, NV>(p, a, s);
    case 2: return launch_decode_vv<VA, 2, NV>(p, a, s);
    default: return launch_decode_vv<VA, 4, NV>(p, a, s);
  }
}

template <bool NV>
cudaError_t launch_decode_fmt(const MxParams& p, const Fp4DecodeArgs& a, cudaStream_t s) {
  switch (p.H / 1024) {
    case 1: return launch_decode_va<1, NV>(p, a, s);
    case 2: return launch_decode_va<2, NV>(p, a, s);
    default: return launch_decode_va<4, NV>(p, a, s);
  }
}

cudaError_t launch_fp4_decode(const MxParams& p, bool nv, const Fp4DecodeArgs& a, cudaStream_t s) {
  return nv ? launch_decode_fmt<true>(p, a, s) : launch_decode_fmt<false>(p, a, s);
}

cudaError_t launch_fp4_ring(const MxParams& p, int T, bool nv, cudaStream_t s) {
  const size_t R = (size_t)T * p.k;
  cudaError_t err = cudaMemsetAsync(p.inst_done, 0, R * sizeof(unsigned int), s);
  if (err != cudaSuccess) return err;
  return nv ? launch_fmt<true>(p, s) : launch_fmt<false>(p, s);
}

}  // namespace moe
