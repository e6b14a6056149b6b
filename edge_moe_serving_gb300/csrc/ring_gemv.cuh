// TMA-ring weight-streaming GEMV machinery shared by the fused expert-FFN
// launch (ffn_gemv.cu) and the one-launch decode layer (decode_layer.cu).
// FreeToken paper, section 3.2: grouped evaluation of the GPU execution set;
// section 3: experts are reached through their (layer, expert) slot.
#pragma once

#include "ffn_params.cuh"
#include "group_prefix.cuh"

namespace moe {
namespace {

// Instances per expert (prefix over experts of ceil(rows / NT), eligible
// only: 0 < counts[e] <= max_rows and mask[e] != 0 when a mask is given).
// Needs blockDim.x >= 32 and E <= kMaxE.
template <int NT>
__device__ void build_prefix(const GemvParams& p, int* s_pref, int* s_warp) {
  build_group_prefix<NT, kMaxE / 32>(p.counts, p.E, 0, p.max_rows, p.mask, s_pref, s_warp);
}

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

// Where instance j of a fused launch reads and writes: its expert, the
// slot-table entry its weights stream from, its fill destination (a cache
// slot, or -1), its first dispatch position and its number of token rows.
struct InstInfo {
  int e, entry, fill, pos0, ntok;
};

// Instances from the per-expert prefix: expert e with c rows has ceil(c / NT)
// instances of up to NT rows each (the general fused expert-FFN launch).
template <int NT>
struct PrefixInsts {
  const int* pref;
  const int* off;
  const int* ent;
  const int* fill;
  const int32_t* counts;
  int E;
  __device__ int count() const { return pref[E]; }
  __device__ InstInfo get(int j) const {
    const int e = find_group(pref, E, j);
    const int c = j - pref[e];
    return {e, ent[e], fill[e], off[e] + c * NT, min(NT, counts[e] - c * NT)};
  }
  // what the weight stream needs: the expert, its entry and fill destination
  __device__ void source(int j, int& e, int& entry, int& fill_dst) const {
    e = find_group(pref, E, j);
    entry = ent[e];
    fill_dst = fill[e];
  }
};

// Instances listed one per entry (the one-launch decode layer: one instance per
// routed expert, every expert's rows fit one instance).  `src` already names
// the pool the weights stream from (a hit's cache slot, else the staging
// slot), so the stream can start before `fill` is decided.
struct DecInst {
  int e, src, fill, pos0, ntok;
};
struct TableInsts {
  const DecInst* t;
  int n;
  __device__ int count() const { return n; }
  __device__ InstInfo get(int j) const { return {t[j].e, t[j].src, t[j].fill, t[j].pos0, t[j].ntok}; }
  __device__ void source(int j, int& e, int& entry, int& fill_dst) const {
    e = t[j].e;
    entry = t[j].src;
    fill_dst = -1;
  }
};

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
constexpr int kConsumerWarps = 6;
// Unit i lives in stage i % kRingStages and is consumed by warp i % kConsumerWarps.
// A parity wait tells only two phases of a stage apart, so a consumer may wait
// for use n+1 of a stage only after use n has completed; that holds when every
// stage is always consumed by the same warp, i.e. when the consumer count
// divides the stage count.
static_assert(kRingStages % kConsumerWarps == 0, "each ring stage must have one consumer warp");
constexpr int kRingThreads = (kConsumerWarps + 1) * 32;
static_assert(kMaxFusedInst <= 1024, "per-instance counters live in shared memory");

__device__ inline uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ inline unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ inline bool ring_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return bounded_wait(bar, parity, abort_flag);
}

__device__ inline void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// bulk_g2s with an L2 cache policy (weights: evict first).
__device__ inline void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
               : "memory");
}

// Shared -> global bulk store, evict-first in L2: a fused cache fill is not
// read again in this call, so its lines are the first to go back to DRAM
// (during the call) rather than lingering dirty behind the weight stream.
__device__ inline void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  const uint64_t pol = l2_evict_first();
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
               ::"l"(dst), "r"(smem_addr(src)), "r"(bytes), "l"(pol)
               : "memory");
}
__device__ inline unsigned ld_acquire_u32(const unsigned* ptr) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ inline int atom_add_acq_rel_cta(int* smem_ptr, int v) {
  int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(smem_ptr)), "r"(v)
               : "memory");
  return old;
}

__device__ inline void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ inline void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ inline void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 8 bf16 products into two partial sums (shorter dependency chains).
__device__ inline void dot8x2(const uint4& w, const uint4& a, float& s0, float& s1) {
  s0 = fmaf(bf16_lo(w.x), bf16_lo(a.x), s0);
  s1 = fmaf(bf16_hi(w.x), bf16_hi(a.x), s1);
  s0 = fmaf(bf16_lo(w.y), bf16_lo(a.y), s0);
  s1 = fmaf(bf16_hi(w.y), bf16_hi(a.y), s1);
  s0 = fmaf(bf16_lo(w.z), bf16_lo(a.z), s0);
  s1 = fmaf(bf16_hi(w.z), bf16_hi(a.z), s1);
  s0 = fmaf(bf16_lo(w.w), bf16_lo(a.w), s0);
  s1 = fmaf(bf16_hi(w.w), bf16_hi(a.w), s1);
}

// Source and (for a fused fill) destination banks of the instance's expert.
struct RingSrc {
  BankSet src;
  __nv_bfloat16* dst_gate;
  __nv_bfloat16* dst_up;
  __nv_bfloat16* dst_down;
  bool ok, fill;
};

__device__ inline RingSrc ring_source(const GemvParams& p, int e, int entry, int fill_dst, uint32_t* status) {
  RingSrc r;
  r.fill = false;
  r.dst_gate = r.dst_up = r.dst_down = nullptr;
  if (fill_dst >= 0) {
    // admitted by this call: read the staging copy, write the cache slot
    r.ok = resolve_slot(p.c, MOE_STAGING_TAG | (p.layer * p.E + e), p.H, p.I, &r.src, status);
    const size_t per = (size_t)p.H * p.I;
    r.dst_gate = reinterpret_cast<__nv_bfloat16*>(p.c.cache.w_gate) + (size_t)fill_dst * per;
    r.dst_up = reinterpret_cast<__nv_bfloat16*>(p.c.cache.w_up) + (size_t)fill_dst * per;
    r.dst_down = reinterpret_cast<__nv_bfloat16*>(p.c.cache.w_down) + (size_t)fill_dst * per;
    r.fill = r.ok;
  } else {
    r.ok = resolve_filtered(p.c, entry, p.pool_filter, p.H, p.I, &r.src, status);
  }
  return r;
}

// Rows per unit (per bank) for a weight row length K: units of ~16 KB, at most 4 rows.
__host__ __device__ inline int ring_rows(int K, bool gateup) {
  const int nb = gateup ? 2 : 1;
  const int u = kUnitBytes / (nb * K * 2);
  return u >= 4 ? 4 : (u >= 2 ? 2 : 1);
}

constexpr unsigned long long kGridWaitNs = 1000000000ull;

// Ring bookkeeping shared by the two phases of one CTA.  Ring index = the
// CTA's running unit count over both phases; unit i sits in stage i % S and
// belongs to consumer warp i % C.  Units of an unbound expert still take a
// ring slot (the producer completes it without data), so every role can
// compute ring indices without seeing the other roles' decisions.
struct RingState {
  int base;               // ring index of the current phase's first unit
  int armed_last;         // producer: last ring index with copies in flight
  int last_issued;        // producer: last ring index it completed or armed (data or not)
  bool stored;            // a consumer issued fused-fill stores
};

// Number of this CTA's units among `total` grid-strided units.
__device__ inline int local_units(int total) {
  const int b = blockIdx.x, G = gridDim.x;
  return b < total ? (total - 1 - b) / G + 1 : 0;
}

// Per-warp consumer of ring units: the state of the current instance and the
// reduction of one unit in shared memory (gate/up: h rows; down: y rows).  An
// admitted expert's unit is also written to its cache slot from the stage.
template <int NT, bool GATEUP, int VC>
struct UnitWorker {
  static constexpr int NB = GATEUP ? 2 : 1;
  static constexpr int PS = (NT == 1) ? 2 : 1;
  static constexpr int XR = (NT == 1 && VC > 0) ? VC : 1;
  static constexpr bool x_in_regs = (NT == 1) && VC > 0;
  int cur_j = -1, pos0 = 0, ntok = 0;
  RingSrc rs;
  const __nv_bfloat16* act[NT];
  int yrow[NT];
  uint4 xr[XR];

  // New instance j.  Down rows wait (bounded) until p.inst_done[j] >= need:
  // h of the instance is then complete.  Returns false on abort.
  template <class Insts>
  __device__ inline bool begin(const GemvParams& p, const Insts& v, int j, unsigned need, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    cur_j = j;
    if (!GATEUP && p.inst_done != nullptr) {
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
      if (*abort_flag) return false;
    }
    const InstInfo in = v.get(j);
    // any warp that meets an unbound expert reports it (units are spread over warps)
    rs = ring_source(p, in.e, in.entry, in.fill, (lane == 0) ? p.status : nullptr);
    pos0 = in.pos0;
    ntok = in.ntok;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int pos = pos0 + (t < ntok ? t : 0);
      if (GATEUP)
        act[t] = p.x_perm ? p.x_perm + (size_t)pos * p.H : p.x + (size_t)(p.perm[pos] / p.k) * p.H;
      else
        act[t] = p.h + (size_t)pos * p.I;
      yrow[t] = GATEUP ? 0 : p.perm[pos];
    }
    if (x_in_regs && rs.ok) {
      // phase B reads h written by other CTAs of this launch: through L2, not the read-only path
#pragma unroll
      for (int c2 = 0; c2 < XR; ++c2)
        xr[c2] = GATEUP ? ldg_cached(act[0] + (size_t)(lane + 32 * c2) * 8)
                        : __ldcg(reinterpret_cast<const uint4*>(act[0] + (size_t)(lane + 32 * c2) * 8));
    }
    return true;
  }

  // Reduce the unit in stage sw: rows n0 .. n0 + U - 1 of the instance's expert.
  __device__ inline void run(const GemvParams& p, const uint8_t* sw, int n0, RingState& st) {
    const int lane = threadIdx.x & 31;
    const int K = GATEUP ? p.H : p.I;
    const int NTASK = GATEUP ? p.I : p.H;
    const int row_bytes = K * 2;
    const int U = ring_rows(K, GATEUP);
    const int bank_stride = kUnitBytes / NB;
    const int VPL = K / 256;
    const int rows = min(U, NTASK - n0);
    if (!rs.ok) return;
    if (rs.fill && lane == 0) {
      // this expert is being admitted to the cache: write the unit to its slot
      const uint32_t bytes = (uint32_t)(rows * row_bytes);
      if (GATEUP) {
        bulk_s2g(rs.dst_gate + (size_t)n0 * K, sw, bytes);
        bulk_s2g(rs.dst_up + (size_t)n0 * K, sw + bank_stride, bytes);
      } else {
        bulk_s2g(rs.dst_down + (size_t)n0 * K, sw, bytes);
      }
      bulk_commit();
      st.stored = true;
    }
    const uint8_t* wbase = sw + (size_t)lane * 16;
    for (int r = 0; r < rows; ++r) {
      float acc[NB][NT][PS];
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int q = 0; q < PS; ++q) acc[b][t][q] = 0.0f;
      const uint8_t* wr = wbase + (size_t)r * row_bytes;
      if (x_in_regs) {
#pragma unroll
        for (int c = 0; c < XR; ++c)
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4 w = *reinterpret_cast<const uint4*>(wr + b * bank_stride + c * 512);
            dot8x2(w, xr[c], acc[b][0][0], acc[b][0][PS - 1]);
          }
      } else {
#pragma unroll 4
        for (int c = 0; c < VPL; ++c) {
          const int v = lane + 32 * c;
          uint4 a[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t)
            a[t] = (t < ntok) ? (GATEUP ? ldg_cached(act[t] + (size_t)v * 8)
                                        : __ldcg(reinterpret_cast<const uint4*>(act[t] + (size_t)v * 8)))
                              : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4 w = *reinterpret_cast<const uint4*>(wr + b * bank_stride + c * 512);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[b][t][0] = dot8(w, a[t], acc[b][t][0]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          float v = acc[b][t][0];
          if (PS == 2) v += acc[b][t][PS - 1];
          acc[b][t][0] = warp_sum(v);
        }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (lane == t && t < ntok) {
          if (GATEUP)
            p.h[(size_t)(pos0 + t) * p.I + n0 + r] = __float2bfloat16_rn(silu(acc[0][t][0]) * acc[NB - 1][t][0]);
          else
            p.y[(size_t)yrow[t] * p.H + n0 + r] = acc[0][t][0];
        }
      }
    }
    if (rs.fill && lane == 0) bulk_wait_read_all();   // the store has read the stage
  }
};

// One phase of the fused GEMV: phase A (GATEUP) streams gate and up rows and
// writes h; phase B streams down rows and writes y.  Units are grid-strided:
// CTA b takes units b, b + G, b + 2G, ...  VC > 0: the single token's
// activation row (K = 256*VC) is held in registers.
// owned (phase B only): instead of the stride, CTA b takes the row blocks
// rb = b, b + G, b + 2G, ... of every instance, instance by instance, so that
// it holds every expert output of those rows and can combine them itself.
template <int NT, bool GATEUP, int VC, class Insts>
__device__ inline void ring_phase(const GemvParams& p, const Insts& v, int* s_cnt, uint8_t* ring, uint64_t* full_bar,
                                  uint64_t* empty_bar, volatile int* abort_flag, RingState& st, bool producer,
                                  bool owned = false) {
  constexpr int NB = GATEUP ? 2 : 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = GATEUP ? p.H : p.I;
  const int NTASK = GATEUP ? p.I : p.H;
  const int row_bytes = K * 2;
  const int U = ring_rows(K, GATEUP);
  const int upi = (NTASK + U - 1) / U;
  const int bank_stride = kUnitBytes / NB;
  const int total = v.count() * upi;
  const int G = gridDim.x;
  owned = owned && !GATEUP;
  const int M = local_units(upi);   // row blocks this CTA owns
  const int n_local = owned ? v.count() * M : local_units(total);
  const int base = st.base;
  st.base += n_local;
  // this CTA's i-th unit: instance j, first row n0
  auto unit_of = [&](int i, int& j, int& n0) {
    if (owned) {
      j = i / M;
      n0 = ((int)blockIdx.x + (i - j * M) * G) * U;
    } else {
      const int u = (int)blockIdx.x + i * G;
      j = u / upi;
      n0 = (u - j * upi) * U;
    }
  };

  if (producer) {
    int cur_j = -1;
    RingSrc rs;
    rs.ok = false;
    const uint64_t wpol = l2_evict_first();   // weights are read once per call
    for (int i = 0; i < n_local && !*abort_flag; ++i) {
      int j, n0;
      unit_of(i, j, n0);
      if (j != cur_j) {
        cur_j = j;
        int e, entry, fill_dst;
        v.source(j, e, entry, fill_dst);
        rs = ring_source(p, e, entry, fill_dst, nullptr);
      }
      const int ri = base + i;
      const int stage = ri % kRingStages;
      const uint32_t use = (uint32_t)(ri / kRingStages);
      if (!ring_wait(&empty_bar[stage], (use & 1u) ^ 1u, abort_flag)) break;
      st.last_issued = ri;
      if (!rs.ok) {
        // nothing to stream: complete the slot's phase without data
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&full_bar[stage])) : "memory");
        continue;
      }
      uint8_t* dst = ring + stage * kUnitBytes;
      const int rows = min(U, NTASK - n0);
      const uint32_t bytes = (uint32_t)(rows * row_bytes);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&full_bar[stage])),
                   "r"(bytes * NB)
                   : "memory");
      if (GATEUP) {
        bulk_g2s_hint(dst, rs.src.gate + (size_t)n0 * K, bytes, &full_bar[stage], wpol);
        bulk_g2s_hint(dst + bank_stride, rs.src.up + (size_t)n0 * K, bytes, &full_bar[stage], wpol);
      } else {
        bulk_g2s_hint(dst, rs.src.down + (size_t)n0 * K, bytes, &full_bar[stage], wpol);
      }
      st.armed_last = ri;
    }
    return;
  }

  UnitWorker<NT, GATEUP, VC> wk;
  const int ua = ring_rows(p.H, true);
  const unsigned need = (unsigned)min(G, (p.I + ua - 1) / ua);   // CTAs holding gate/up units of an instance
  // this warp's units: ring index ri = base + i with ri % C == warp
  const int i0 = ((warp - base) % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
  for (int i = i0; i < n_local; i += kConsumerWarps) {
    int j, n0;
    unit_of(i, j, n0);
    if (j != wk.cur_j && !wk.begin(p, v, j, need, abort_flag)) break;
    const int ri = base + i;
    const int stage = ri % kRingStages;
    const uint32_t use = (uint32_t)(ri / kRingStages);
    if (!ring_wait(&full_bar[stage], use & 1u, abort_flag)) break;
    wk.run(p, ring + stage * kUnitBytes, n0, st);
    if (GATEUP && p.inst_done != nullptr) {
      // Publish the instance once this CTA's units of it are all done: each
      // warp counts its unit with a CTA-scope acquire-release add (ordering
      // its lanes' h stores, which __syncwarp made visible to lane 0); the
      // warp that completes the count raises the instance's counter with a
      // GPU-scope release add, which (release being cumulative) carries every
      // counted warp's stores.
      __syncwarp();
      if (lane == 0) {
        const int lo = j * upi, hi = lo + upi;
        const int first = lo + (((int)blockIdx.x - lo) % G + G) % G;   // first u >= lo with u % G == block
        const int mine = first < hi ? (hi - 1 - first) / G + 1 : 0;
        if (atom_add_acq_rel_cta(&s_cnt[j], 1) + 1 == mine)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.inst_done + j) : "memory");
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[stage])) : "memory");
  }
}

// The ring's barriers and the CTA's abort flag.
struct RingShared {
  uint64_t full_bar[kRingStages];
  uint64_t empty_bar[kRingStages];
  int abort;
};

// Shared memory of a general fused-GEMV CTA besides the ring itself.
struct FusedShared {
  int pref[kMaxE + 1];
  int warp[32];               // per-warp scan partials of build_prefix: any block of up to 1024 threads
  int off[kMaxE];
  int ent[kMaxE];
  int fill[kMaxE];
  int cnt[kMaxFusedInst];     // per-instance count of this CTA's finished gate/up units
  RingShared r;
};

constexpr int kRingSmem = kRingStages * kUnitBytes + 128;

__device__ inline void ring_init(RingShared& rs) {
  for (int s = 0; s < kRingStages; ++s) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rs.full_bar[s])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rs.empty_bar[s])));
  }
  rs.abort = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// The two streaming phases of a fused launch and what follows them, for
// instances described by `v`, run by every thread of the CTA: warp
// kConsumerWarps is the producer (its lane 0 streams; the other lanes return at
// once), the others consume.  Phase A (gate/up -> h) and phase B (down -> y)
// share one weight ring, so the producer keeps streaming down rows while the
// consumers wait for h: per instance (p.inst_done, a bounded wait on the
// counter of the instance about to be read; cnt[j] counts this CTA's finished
// gate/up units of instance j and must be zero) or at a bounded grid-wide
// barrier.  With p.combine_out set, phase B gives each CTA whole output row
// blocks (every instance's rows rb = b, b + G, ...) and the CTA applies the
// gate-weighted combine to its own rows when its units are done.
// grid_count[0] and the p.inst_done words must be zero at launch.
template <int NT, int VA, int VB, class Insts>
__device__ void fused_phases(const GemvParams& p, const Insts& v, unsigned int* grid_count, RingShared& rsh, int* cnt,
                             uint8_t* ring) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &rsh.abort;
  const bool producer = warp == kConsumerWarps;
  RingState st = {0, -1, -1, false};

  if (!producer || lane == 0) {
    ring_phase<NT, true, VA>(p, v, cnt, ring, rsh.full_bar, rsh.empty_bar, abort_flag, st, producer);
    if (!producer && p.inst_done == nullptr) {
      // grid-wide barrier: every h row of phase A is written before any is read
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
      if (tid == 0) {
        __threadfence();
        atomicAdd(grid_count, 1u);
        const unsigned long long t0 = gtimer();
        while (*reinterpret_cast<volatile unsigned int*>(grid_count) < gridDim.x) {
          if (*abort_flag) break;
          if (gtimer() - t0 > kGridWaitNs) {
            *abort_flag = 1;
            break;
          }
        }
        __threadfence();
      }
      asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    }
    if (!*abort_flag)
      ring_phase<NT, false, VB>(p, v, cnt, ring, rsh.full_bar, rsh.empty_bar, abort_flag, st, producer,
                                p.combine_out != nullptr);
    if (producer) {
      // drain: the copies of the last ring round land before the CTA exits (the last
      // kRingStages slots issued: each stage's latest use, whatever it carried)
      volatile int no_abort = 0;
      if (st.armed_last >= 0)
        for (int q = st.last_issued; q >= 0 && q > st.last_issued - kRingStages; --q)
          ring_wait(&rsh.full_bar[q % kRingStages], (uint32_t)(q / kRingStages) & 1u, &no_abort);
    } else {
      if (st.stored && lane == 0) bulk_wait_all();   // fused-fill writes complete before exit
      if (p.combine_out != nullptr) {
        // Phase B ran with owned row blocks: every expert row of this CTA's
        // output rows was written by its own warps, so once they are all done
        // (a CTA barrier) it combines those rows itself, in fixed expert order,
        // with no grid-wide barrier.
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
        if (!*abort_flag) {
          const int U = ring_rows(p.I, false);
          const int M = local_units((p.H + U - 1) / U);
          const int per_t = M * U;
          const int items = p.T * per_t;
          for (int it = tid; it < items; it += kConsumerWarps * 32) {
            const int t = it / per_t, rest = it - t * per_t;
            const int m = rest / U;
            const int row = ((int)blockIdx.x + m * (int)gridDim.x) * U + (rest - m * U);
            if (row < p.H) {
              float acc = 0.0f;
              for (int jj = 0; jj < p.k; ++jj)
                acc = fmaf(p.combine_w[t * p.k + jj], __ldcg(p.y + (size_t)(t * p.k + jj) * p.H + row), acc);
              p.combine_out[(size_t)t * p.H + row] = __float2bfloat16_rn(acc);
            }
          }
        }
      }
    }
  }
}

// The general fused launch after its prologue: fs.off / fs.ent / fs.fill hold
// each expert's first dispatch position, slot-table entry and fill
// destination (-1: none); p.counts / p.perm / p.combine_w may point to shared
// memory.  Builds the per-expert instance prefix, then fused_phases.
template <int NT, int VA, int VB>
__device__ void fused_ffn_body(const GemvParams& p, unsigned int* grid_count, FusedShared& fs, uint8_t* ring) {
  const int tid = threadIdx.x;
  build_prefix<NT>(p, fs.pref, fs.warp);   // ends with __syncthreads
  if (p.inst_done != nullptr) {
    for (int i = tid; i < fs.pref[p.E] && i < kMaxFusedInst; i += blockDim.x) fs.cnt[i] = 0;
    __syncthreads();
  }
  const PrefixInsts<NT> v = {fs.pref, fs.off, fs.ent, fs.fill, p.counts, p.E};
  fused_phases<NT, VA, VB>(p, v, grid_count, fs.r, fs.cnt, ring);
}

}  // namespace
}  // namespace moe
