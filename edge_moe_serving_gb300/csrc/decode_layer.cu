// The whole routed MoE layer for a decode-sized call in one cooperative
// launch (FreeToken paper, section 3.2: router, cache lookup and q* split,
// grouped expert evaluation, combine; section 4.1: device-side cache
// control).  One CTA per SM:
//
//   phase R   every CTA scores its router rows (fp32 rows fetched with
//             cp.async.bulk into the weight ring's shared memory, the token
//             rows converted to fp32 next to them) and writes the logits; the
//             cache state the decision reads (this layer's slot-table row,
//             the pool's stamps, owners and clock) is copied into shared
//             memory in the same round of copies
//   barrier   bounded grid-wide barrier: every logit is written
//   route     warp 0 of every CTA runs the same top-k and dispatch on the
//             logits and looks up which routed experts the cache pool holds;
//             that fixes every expert's weight source, so the producer warp
//             starts streaming here
//   residency warp 0 then decides q, the fill set and the victim slots
//             (front_residency) while the first weights are in flight; the
//             consumer warps start once it is done.  CTA 0 commits the
//             decision to the cache state at once: every CTA read the
//             pre-call state before the barrier
//   FFN       the fused weight-streaming gate/up + down phases, admitted
//             experts copied into their cache slots while they stream; each
//             CTA computes whole output row blocks in the down phase and
//             applies the gate-weighted combine to them (fused_phases)
//
// It computes exactly what the router, bind, dispatch, FFN and combine
// launches compute for such calls; it replaces their four kernel boundaries
// by one grid barrier (after the router) and per-instance completion counters
// (gate/up -> down).
#include <algorithm>

#include "decode_front.cuh"
#include "front_warp.cuh"
#include "ring_gemv.cuh"

namespace moe {
namespace {

struct DecodeParams {
  GemvParams g;                    // perm / combine_w are pointed at shared memory in the kernel
  const float* w_router;           // [E, H] fp32
  const float* bias;               // [E] or null
  uint32_t phi_q16;
  int min_fill, policy;
  unsigned long long seed;
  moe_bind_stats* stats;
  float* logits;                   // [T, E] workspace
  int32_t* topk_ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int rows_per_cta;                // ceil(E / grid)
};

// Shared memory of a decode CTA besides the ring.  The state copies are
// targets of bulk copies: 16-byte aligned, first.
struct __align__(16) DecodeShared {
  int32_t table[kMaxRouteE];       // this layer's slot-table row
  uint32_t stamp[kDecMaxSlots];    // the cache pool's stamps
  int32_t owner[kDecMaxSlots];     // and owners
  uint32_t hitmap[kDecMaxSlots / 32];
  FrontDecision fr;
  DecInst inst[32];                // one instance per distinct routed expert, in dispatch order
  int cnt[32];                     // per instance: this CTA's finished gate/up units
  float red[kRingThreads / 32][kDecMaxRows][kDecMaxT];
  float bias[kDecMaxRows];
  uint64_t rbar;
  RingShared r;
  uint32_t clock;
  int n_inst;
};

// Named barriers besides __syncthreads (0) and the consumers' barrier inside
// fused_phases (1, also used here once the decision is complete).
constexpr int kBarConsumers = 1;
constexpr int kBarStream = 2;      // warp 0 -> producer warp: the weight sources are known

template <int NT, int VA, int VB>
__global__ void __launch_bounds__(kRingThreads, 1)
decode_layer_kernel(DecodeParams d, unsigned int* grid_count) {
  extern __shared__ __align__(128) uint8_t ring_raw[];
  __shared__ DecodeShared sh;
  // the ring is the dynamic shared array itself: pointers derived from it keep the shared
  // address space, so stage reads compile to shared-memory loads
  uint8_t* ring = ring_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  GemvParams p = d.g;
  const int E = p.E, H = p.H, T = p.T, G = gridDim.x, b = blockIdx.x;
  const int n_my = b < E ? (E - 1 - b) / G + 1 : 0;
  // ring bytes during the prologue: router rows (fp32) | token rows (bf16)
  const int n_slots = p.c.cache.n_slots, base = p.layer * E;
  float* wrow = reinterpret_cast<float*>(ring);                                    // [n_my][H]
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(wrow + (size_t)d.rows_per_cta * H);   // [T][H]

  if (tid == 0) {
    ring_init(sh.r);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sh.rbar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < 32) sh.cnt[tid] = 0;
  __syncthreads();
  pdl_wait();
  // ---------------------------------------------------------------- phase R
  // One round of bulk copies brings everything the prologue reads: this CTA's
  // router rows, the token rows, and the cache state the decision reads (this
  // layer's slot-table row, the pool's stamps and owners); 16-byte tails and
  // misaligned rows take plain loads.
  const bool table_bulk = (reinterpret_cast<uintptr_t>(p.c.slot_table + base) & 15) == 0;
  const bool slot_bulk = ((reinterpret_cast<uintptr_t>(p.c.stamp) | reinterpret_cast<uintptr_t>(p.c.owner)) & 15) == 0;
  const int table_bulk_n = table_bulk ? (E & ~3) : 0;
  const int slot_bulk_n = slot_bulk ? (n_slots & ~3) : 0;
  if (tid == 0) {
    const uint32_t row_bytes = (uint32_t)H * 4u;
    const uint32_t x_bytes = (uint32_t)T * H * 2u;
    const uint32_t bytes = row_bytes * (uint32_t)n_my + x_bytes + 4u * (uint32_t)table_bulk_n + 8u * (uint32_t)slot_bulk_n;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&sh.rbar)), "r"(bytes)
                 : "memory");
    for (int i = 0; i < n_my; ++i)
      bulk_g2s(wrow + (size_t)i * H, d.w_router + (size_t)(b + i * G) * H, row_bytes, &sh.rbar);
    bulk_g2s(xs, p.x, x_bytes, &sh.rbar);
    if (table_bulk_n > 0) bulk_g2s(sh.table, p.c.slot_table + base, 4u * table_bulk_n, &sh.rbar);
    if (slot_bulk_n > 0) {
      bulk_g2s(sh.stamp, p.c.stamp, 4u * slot_bulk_n, &sh.rbar);
      bulk_g2s(sh.owner, p.c.owner, 4u * slot_bulk_n, &sh.rbar);
    }
  } else if (warp == kConsumerWarps) {
    for (int e = table_bulk_n + lane; e < E; e += 32) sh.table[e] = __ldcg(p.c.slot_table + base + e);
    for (int v = slot_bulk_n + lane; v < n_slots; v += 32) {
      sh.stamp[v] = __ldcg(p.c.stamp + v);
      sh.owner[v] = __ldcg(p.c.owner + v);
    }
    if (lane == 0) sh.clock = __ldcg(p.c.clock);
  } else if (warp == 1 && lane < n_my) {
    sh.bias[lane] = d.bias ? __ldg(d.bias + b + lane * G) : 0.0f;
  }
  if (!bounded_wait(&sh.rbar, 0u, &sh.r.abort)) sh.r.abort = 1;
  __syncthreads();
  if (n_my > 0 && !sh.r.abort) {
    constexpr int NW = kRingThreads / 32;
    switch (n_my) {
      case 1: router_rows_block<1, NT, NW>(wrow, xs, H, T, E, sh.red, sh.bias, d.logits, b, G); break;
      case 2: router_rows_block<2, NT, NW>(wrow, xs, H, T, E, sh.red, sh.bias, d.logits, b, G); break;
      case 3: router_rows_block<3, NT, NW>(wrow, xs, H, T, E, sh.red, sh.bias, d.logits, b, G); break;
      default: router_rows_block<4, NT, NW>(wrow, xs, H, T, E, sh.red, sh.bias, d.logits, b, G); break;
    }
  }
  // ---------------------------------------------------------------- route, residency
  if (grid_barrier(grid_count + 2, &sh.r.abort)) {
    const int R = T * p.k;
    if (warp == 0) {
      const FrontLane fl = front_route(d.logits, T, p.k, E, n_slots, sh.table, sh.fr);
      // one instance per distinct expert, in dispatch order; a hit streams
      // from its cache slot, a miss (filled or not) from its staging slot
      const unsigned um = __ballot_sync(0xffffffffu, fl.uniq);
      const int j = __popc(um & lane_lt());
      if (fl.uniq) {
        const unsigned later = lane == 31 ? 0u : (um & (0xffffffffu << (lane + 1)));
        sh.inst[j].e = fl.e;
        sh.inst[j].src = fl.hit ? fl.entry : (int)(MOE_STAGING_TAG | (base + fl.e));
        sh.inst[j].pos0 = lane;
        sh.inst[j].ntok = (later ? __ffs(later) - 1 : R) - lane;
      }
      if (lane == 0) sh.n_inst = __popc(um);
      __syncwarp();
      asm volatile("bar.arrive %0, %1;" ::"n"(kBarStream), "n"(64) : "memory");   // the producer may stream
      front_residency(fl, n_slots, p.layer, sh.stamp, sh.owner, sh.clock, d.phi_q16, d.min_fill, d.policy, d.seed,
                      sh.fr, sh.hitmap);
      if (fl.uniq) sh.inst[j].fill = sh.fr.u_kind[lane] == kFrontFill ? sh.fr.u_slot[lane] : -1;
      __syncwarp();
    }
    if (warp == kConsumerWarps) {
      asm volatile("bar.sync %0, %1;" ::"n"(kBarStream), "n"(64) : "memory");
    } else {
      asm volatile("bar.sync %0, %1;" ::"n"(kBarConsumers), "n"(kConsumerWarps * 32) : "memory");
      // routing outputs, spread over the CTAs; CTA 0 commits the decision
      for (int e = b + tid * G; e <= E; e += G * kConsumerWarps * 32) {
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
      if (b == 0 && warp == 0) front_commit(sh.fr, p.c, p.layer, d.stats, p.status);
    }
    // ---------------------------------------------------------------- FFN
    p.counts = nullptr;
    p.offsets = nullptr;
    p.perm = sh.fr.perm;
    p.combine_w = sh.fr.w;
    p.fills = nullptr;
    const TableInsts v = {sh.inst, sh.n_inst};
    fused_phases<NT, VA, VB>(p, v, grid_count, sh.r, sh.cnt, ring);
  }
  pdl_trigger();
  __syncthreads();
  if (sh.r.abort && tid == 0) set_status(p.status, MOE_DEV_ERR_TIMEOUT);
}

template <int NT, int VA, int VB>
cudaError_t launch_one(const DecodeParams& d, unsigned int* grid_count, int grid, cudaStream_t s) {
  static std::atomic<unsigned char> attr[kMaxDevices];
  cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(decode_layer_kernel<NT, VA, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kRingSmem);
  });
  if (e != cudaSuccess) return e;
  const size_t words = 4 + (size_t)d.g.T * d.g.k;   // barrier words, then one counter per instance
  cudaError_t err = cudaMemsetAsync(grid_count, 0, words * sizeof(unsigned int), s);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = kRingSmem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: the grid barrier and the cross-CTA waits can complete
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, decode_layer_kernel<NT, VA, VB>, d, grid_count));
}

}  // namespace

bool decode_layer_ok(int T, int k, int E, int H, int I, int n_slots) {
  const int G = num_sms();
  const int rows = (E + G - 1) / G;
  return T >= 1 && T <= kDecMaxT && T * k <= 32 && E <= kMaxRouteE && rows <= kDecMaxRows && gemv_fused_ok(H, I) &&
         n_slots >= 1 && n_slots <= kDecMaxSlots &&
         (size_t)rows * H * 4 + (size_t)T * H * 2 <= (size_t)kRingStages * kUnitBytes;
}

cudaError_t launch_decode_layer(const moe_cache& c, int layer, const __nv_bfloat16* x, int T, int k,
                                const float* w_router, const float* bias, uint32_t phi_q16, int min_fill, int policy,
                                uint64_t seed, moe_bind_stats* stats, float* logits, int32_t* topk_ids, float* topk_w,
                                int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm, float* y_rows,
                                __nv_bfloat16* h, unsigned int* grid_count, __nv_bfloat16* out, uint32_t* status,
                                cudaStream_t s) {
  DecodeParams d = {};
  GemvParams& p = d.g;
  p.c = c;
  p.layer = layer;
  p.E = c.E;
  p.H = c.H;
  p.I = c.I;
  p.k = k;
  p.T = T;
  p.x = x;
  p.x_perm = nullptr;
  p.mask = nullptr;
  p.max_rows = T;
  p.h = h;
  p.y = y_rows;
  p.status = status;
  p.combine_out = out;
  p.grid_count = grid_count;
  p.inst_done = grid_count + 4;
  d.w_router = w_router;
  d.bias = bias;
  d.phi_q16 = phi_q16;
  d.min_fill = min_fill;
  d.policy = policy;
  d.seed = seed;
  d.stats = stats;
  d.logits = logits;
  d.topk_ids = topk_ids;
  d.topk_w = topk_w;
  d.counts = counts;
  d.offsets = offsets;
  d.perm = perm;
  d.inv_perm = inv_perm;
  const int G = num_sms();
  d.rows_per_cta = (c.E + G - 1) / G;
  if (T <= 1) {
    const bool va = c.H == 4096 && ring_rows(c.H, true) == 1;
    const bool vb = c.I == 2048;
    if (va && vb) return launch_one<1, 16, 8>(d, grid_count, G, s);
    return launch_one<1, 0, 0>(d, grid_count, G, s);
  }
  if (T <= 2) return launch_one<2, 0, 0>(d, grid_count, G, s);
  if (T <= 4) return launch_one<4, 0, 0>(d, grid_count, G, s);
  return launch_one<8, 0, 0>(d, grid_count, G, s);
}

}  // namespace moe
