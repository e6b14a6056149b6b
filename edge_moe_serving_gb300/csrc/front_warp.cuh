// Warp-level decode front end pieces (FreeToken paper, section 3.2: router
// top-k, cache lookup and the q* split; section 4.1: device-side cache
// control; the Q16 rounding of the write-up "FreeToken: bandwidth-adaptive
// edge MoE serving", section "The split, and what it is actually
// optimising"), shared by the one-warp front end (front_small.cu) and the
// one-launch decode layer (decode_layer.cu).
#pragma once

#include "moe_common.cuh"

namespace moe {
namespace {

__device__ inline unsigned long long mix64(unsigned long long z) {
  // SplitMix64 output function (Steele, Lea & Flood 2014)
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ inline int fill_rule(int m, uint32_t phi, int min_fill) {
  const long long mm = m, p = phi;
  const long long lo = (mm * p) >> 16;
  const long long c_lo = max(lo * (65536 - p), (mm - lo) * p);
  const long long c_hi = max((lo + 1) * (65536 - p), (mm - lo - 1) * p);
  long long q = (c_hi < c_lo) ? lo + 1 : lo;
  if (q > mm) q = mm;
  if (min_fill && p > 0 && mm > 0 && q < 1) q = 1;
  return (int)q;
}

__device__ inline unsigned lane_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// One token's top-k through L2 (the logits come from other CTAs of the launch).
__device__ inline void topk_lanes(const float* row, int E, int k, int& id_out, float& w_out) {
  topk_core<true>(row, E, k, id_out, w_out);
}

// The decision of one decode-sized call (at most 32 routed rows), computed by
// one warp from the logits and the cache state as they were before the call,
// without writing either: every CTA that computes it gets the same result,
// and front_commit applies it once.  Same rules as the one-warp front end:
// top-k, stable dispatch by (expert, row), hits / misses, q from the Q16 rule,
// the fill set F (lowest ids or seeded SplitMix64 ranks), victims = the q
// least (stamp, slot) cache slots not used by a hit of this call.  It comes in
// two parts: front_route (routing, dispatch, which experts hit) and
// front_residency (F and the victims), so that a caller can start streaming
// the routed experts' weights, whose pools the first part already fixes,
// while the second part runs.
enum { kFrontNone = 0, kFrontHit = 1, kFrontFill = 2, kFrontStage = 3 };

struct FrontDecision {
  int ids[32];                  // routed row r = t*k + j
  float w[32];
  int perm[32];
  int inv_perm[32];
  int sorted[32];               // routed rows' expert ids in dispatch order (0x7fffffff past R)
  int u_e[32];                  // per sorted position: the expert, where u_kind != kFrontNone
  int u_kind[32];
  int u_slot[32];               // hit: its cache slot; fill: the victim slot
  int u_old[32];                // fill: the victim's previous owner (layer*E + e) or -1
  int n_unique, m, q, n_fill, bad_slot;
  uint32_t now;
};

// What lane r (sorted dispatch position r) hands from front_route to front_residency.
struct FrontLane {
  int e;          // expert at this position (0x7fffffff past R)
  int entry;      // its slot-table entry, where uniq
  bool uniq;      // first position of its expert
  bool hit, miss;
};

// Part 1: top-k of each token, the dispatch permutation, and which distinct
// experts the cache pool holds.  table = this layer's slot-table row (E entries).
__device__ inline FrontLane front_route(const float* logits, int T, int k, int E, int n_slots,
                                        const int32_t* table, FrontDecision& d) {
  const int lane = threadIdx.x & 31;
  const int R = T * k;
  // 1. top-k per token: lane r ends up with routed row r = t*k + j
  int my_id = 0x7fffffff;
  float my_w = 0.0f;
  for (int t = 0; t < T; ++t) {
    int id;
    float w;
    topk_lanes(logits + (size_t)t * E, E, k, id, w);
    const int src = lane - t * k;
    const int sid = __shfl_sync(0xffffffffu, id, src & 31);
    const float sw = __shfl_sync(0xffffffffu, w, src & 31);
    if (src >= 0 && src < k) {
      my_id = sid;
      my_w = sw;
    }
  }
  const bool row = lane < R;
  d.ids[lane] = row ? my_id : -1;
  d.w[lane] = row ? my_w : 0.0f;
  // 2. dispatch: bitonic sort of (expert, row) keys across the warp (one
  // token's ids already come in ascending order, distinct: nothing to sort)
  int key = row ? (my_id << 5) | lane : 0x7fffffff;
  for (int size = 2; T > 1 && size <= 32; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int other = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool up = (lane & size) == 0;
      const bool lower = (lane & stride) == 0;
      const int mn = min(key, other), mx = max(key, other);
      key = (lower == up) ? mn : mx;
    }
  }
  if (lane < R) {
    const int r = key & 31;
    d.perm[lane] = r;
    d.inv_perm[r] = lane;
  }
  const int sorted_id = (lane < R) ? (key >> 5) : 0x7fffffff;
  d.sorted[lane] = sorted_id;
  // 3. residency of the distinct experts (first occurrence in sorted order)
  const int prev_id = __shfl_up_sync(0xffffffffu, sorted_id, 1);
  FrontLane fl;
  fl.e = sorted_id;
  fl.uniq = lane < R && (lane == 0 || prev_id != sorted_id);
  fl.entry = fl.uniq ? table[sorted_id] : -1;
  fl.hit = fl.uniq && fl.entry >= 0 && fl.entry < n_slots;
  fl.miss = fl.uniq && !fl.hit;
  return fl;
}

// Part 2: q, the fill set F and its victims.  stamp / owner = the cache pool's
// (n_slots entries), clock = the pool's clock.  hitmap: ceil(n_slots / 32)
// words of scratch (word l, bit b: slot 32 l + b is used by a hit of this call
// or already taken as a victim).
__device__ inline void front_residency(const FrontLane& fl, int n_slots, int layer, const uint32_t* stamp,
                                       const int32_t* owner, uint32_t clock, uint32_t phi_q16, int min_fill,
                                       int policy, unsigned long long seed, FrontDecision& d, uint32_t* hitmap) {
  const int lane = threadIdx.x & 31;
  const int e = fl.e;
  const bool uniq = fl.uniq, hit = fl.hit, miss = fl.miss;
  const int entry = fl.entry;
  const uint32_t now = clock + 1u;
  const int bad = __any_sync(0xffffffffu, miss && entry >= 0 && entry < MOE_STAGING_TAG) ? 1 : 0;
  const int map_words = (n_slots + 31) / 32;
  for (int w = lane; w < map_words; w += 32) hitmap[w] = 0u;
  __syncwarp();
  if (hit) atomicOr(&hitmap[entry >> 5], 1u << (entry & 31));
  __syncwarp();
  const unsigned miss_mask = __ballot_sync(0xffffffffu, miss);
  const int m = __popc(miss_mask);
  const int n_unique = __popc(__ballot_sync(0xffffffffu, uniq));
  const int q = fill_rule(m, phi_q16, min_fill);
  bool inF = false;
  if (policy == MOE_FILL_RANDOM) {
    const unsigned long long counter = ((unsigned long long)now << 32) |
                                       ((unsigned long long)(layer & 0xFFFF) << 16) |
                                       (unsigned long long)(e & 0xFFFF);
    const unsigned long long mk = miss ? mix64(seed ^ counter) : ~0ull;
    int rank = 0;
    for (int j = 0; j < 32; ++j) {
      const unsigned long long kj = __shfl_sync(0xffffffffu, mk, j);
      const bool mj = (miss_mask >> j) & 1u;
      rank += (mj && (kj < mk || (kj == mk && j < lane))) ? 1 : 0;   // lanes ascend with the id
    }
    inF = miss && rank < q;
  } else {
    inF = miss && __popc(miss_mask & lane_lt()) < q;
  }
  const unsigned f_mask = __ballot_sync(0xffffffffu, inF);
  const int f_idx = __popc(f_mask & lane_lt());
  // victims: the q least (stamp, slot) cache slots not used by a hit of this
  // call; lane b scans slots b, b + 32, ... each round, and the round's victim
  // is marked in the hitmap so that the next round skips it
  int n_fill = 0;
  int my_victim = -1;
  const int per_lane = map_words;
  for (int i = 0; i < q; ++i) {
    unsigned long long best = ~0ull;
    for (int l = 0; l < per_lane; ++l) {
      const int v = lane + 32 * l;
      if (v < n_slots) {
        const uint32_t sv = stamp[v];
        const bool used = ((hitmap[l] >> lane) & 1u) != 0 || sv == now;
        const unsigned long long kk = used ? ~0ull : (((unsigned long long)sv << 32) | (unsigned long long)v);
        best = kk < best ? kk : best;
      }
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      const unsigned long long ov = __shfl_xor_sync(0xffffffffu, best, o2);
      best = ov < best ? ov : best;
    }
    if (best == ~0ull) break;   // no candidate left: the rest of F overflows to C
    const int vv = (int)(best & 0xFFFFFFFFull);
    if (lane == (vv & 31)) hitmap[vv >> 5] |= 1u << (vv & 31);
    if (inF && f_idx == i) my_victim = vv;
    ++n_fill;
    __syncwarp();
  }
  const bool filled = inF && f_idx < n_fill;
  d.u_e[lane] = e;
  d.u_kind[lane] = !uniq ? kFrontNone : (hit ? kFrontHit : (filled ? kFrontFill : kFrontStage));
  d.u_slot[lane] = hit ? entry : (filled ? my_victim : -1);
  d.u_old[lane] = filled ? owner[my_victim] : -1;
  if (lane == 0) {
    d.n_unique = n_unique;
    d.m = m;
    d.q = q;
    d.n_fill = n_fill;
    d.bad_slot = bad;
    d.now = now;
  }
  __syncwarp();
}

// First dispatch position of expert e (and one past its last) in the sorted ids.
__device__ inline void dispatch_range(const int* sorted, int R, int e, int& lo_out, int& hi_out) {
  int lo = 0, hi = R;                    // first position with sorted id >= e
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sorted[mid] < e) lo = mid + 1;
    else hi = mid;
  }
  int lo2 = lo, hi2 = R;                 // first position with sorted id > e
  while (lo2 < hi2) {
    const int mid = (lo2 + hi2) >> 1;
    if (sorted[mid] <= e) lo2 = mid + 1;
    else hi2 = mid;
  }
  lo_out = lo;
  hi_out = lo2;
}

// Applies a decision to the cache state (one warp, once per call, after every
// reader of the pre-call state is done with it).
__device__ inline void front_commit(const FrontDecision& d, const moe_cache& c, int layer, moe_bind_stats* stats,
                                    uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int base = layer * c.E;
  const int kind = d.u_kind[lane], e = d.u_e[lane];
  const uint32_t now = d.now;
  if (kind == kFrontHit) c.stamp[d.u_slot[lane]] = now;
  if (kind == kFrontFill) {
    const int v = d.u_slot[lane], old = d.u_old[lane];
    if (old >= 0) c.slot_table[old] = MOE_STAGING_TAG | old;
    c.slot_table[base + e] = v;
    c.owner[v] = base + e;
    c.stamp[v] = now;
  }
  if (kind == kFrontStage) c.slot_table[base + e] = MOE_STAGING_TAG | (base + e);
  if (lane == 0) {
    *c.clock = now;
    if (d.bad_slot) set_status(status, MOE_DEV_ERR_BAD_SLOT);
    if (stats) {
      stats->n_unique = d.n_unique;
      stats->n_hit = d.n_unique - d.m;
      stats->n_miss = d.m;
      stats->q = d.q;
      stats->n_fill = d.n_fill;
      stats->n_overflow = d.q - d.n_fill;
      stats->n_staged = d.m - d.n_fill;
      stats->clock = now;
    }
  }
}

}  // namespace
}  // namespace moe
