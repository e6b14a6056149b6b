// Decode front end in one warp: top-k of the router logits, residency bind
// and dispatch for calls with at most 32 routed rows (FreeToken paper,
// section 3.2: router, cache lookup, q* split; section 4.1: device-side
// cache control; the Q16 rounding of the write-up "FreeToken: bandwidth-
// adaptive edge MoE serving", section "The split, and what it is actually
// optimising").
//
// It computes exactly what route top-k + bind + dispatch compute for such
// calls, with warp shuffles instead of block barriers: lane r holds routed
// row r (r = t*k + j).  Used by moe_layer_forward on decode-sized calls,
// after a router launch that only writes the logits.
#include "front_warp.cuh"

namespace moe {
namespace {

constexpr int kMaxSlotsPerLane = 128;   // cache pools up to 4096 slots

struct FrontOut {
  int32_t* topk_ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* fills;     // [n][2]
  int32_t* n_fill;
};

__global__ void __launch_bounds__(32)
front_small_kernel(const float* __restrict__ logits, int T, int k, moe_cache c, int layer, uint32_t phi_q16,
                   int min_fill, int policy, unsigned long long seed, moe_bind_stats* stats, FrontOut o,
                   uint32_t* status) {
  __shared__ unsigned long long keys[kMaxSlotsPerLane * 32];
  const int lane = threadIdx.x;
  const int E = c.E, R = T * k, base = layer * E;
  const int n_slots = c.cache.n_slots;
  pdl_wait();
  pdl_trigger();

  // 1. top-k per token: lane r ends up with routed row r = t*k + j
  int my_id = 0x7fffffff;
  float my_w = 0.0f;
  for (int t = 0; t < T; ++t) {
    int id;
    float w;
    topk_lanes(logits + (size_t)t * E, E, k, id, w);
    const int src = lane - t * k;   // lane t*k + j takes rank j
    const int sid = __shfl_sync(0xffffffffu, id, src & 31);
    const float sw = __shfl_sync(0xffffffffu, w, src & 31);
    if (src >= 0 && src < k) {
      my_id = sid;
      my_w = sw;
    }
  }
  const bool row = lane < R;
  if (row) {
    o.topk_ids[lane] = my_id;
    o.topk_w[lane] = my_w;
  }
  // 2. dispatch: sort (expert, row) keys across the warp
  int key = row ? (my_id << 5) | lane : 0x7fffffff;
  for (int size = 2; size <= 32; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int other = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool up = (lane & size) == 0;
      const bool lower = (lane & stride) == 0;
      const int mn = min(key, other), mx = max(key, other);
      key = (lower == up) ? mn : mx;
    }
  }
  // lane p now holds the p-th smallest key: position p of row (key & 31)
  if (lane < R) {
    const int r = key & 31;
    o.perm[lane] = r;
    o.inv_perm[r] = lane;
  }
  const int sorted_id = (lane < R) ? (key >> 5) : 0x7fffffff;
  for (int e0 = 0; e0 < E + 1; e0 += 32) {
    const int e = e0 + lane;
    int below = 0, cnt = 0;
    for (int j = 0; j < R; ++j) {
      const int sj = __shfl_sync(0xffffffffu, sorted_id, j);
      below += (sj < e) ? 1 : 0;
      cnt += (sj == e) ? 1 : 0;
    }
    if (e <= E) o.offsets[e] = below;
    if (e < E) o.counts[e] = cnt;
  }

  // 3. residency: distinct experts in ascending order (first occurrence in sorted order)
  const int prev_id = __shfl_up_sync(0xffffffffu, sorted_id, 1);
  const bool uniq = lane < R && (lane == 0 || prev_id != sorted_id);
  const int e = sorted_id;
  int entry = -1;
  if (uniq) entry = c.slot_table[base + e];
  uint32_t now = 0;
  if (lane == 0) now = *c.clock + 1u;
  now = __shfl_sync(0xffffffffu, now, 0);
  const bool hit = uniq && entry >= 0 && entry < n_slots;
  const bool miss = uniq && !hit;
  if (miss && entry >= 0 && entry < MOE_STAGING_TAG) set_status(status, MOE_DEV_ERR_BAD_SLOT);
  if (hit) c.stamp[entry] = now;
  const unsigned miss_mask = __ballot_sync(0xffffffffu, miss);
  const int m = __popc(miss_mask);
  const int n_unique = __popc(__ballot_sync(0xffffffffu, uniq));
  const int q = fill_rule(m, phi_q16, min_fill);
  // fill set F: the q lowest-id misses, or the q smallest seeded keys
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
  __syncwarp();
  // victims: the q least (stamp, slot) slots not stamped by this call (hit stamps above are
  // visible to the warp after __syncwarp)
  int n_fill = 0;
  int my_victim = -1;
  if (q > 0) {
    int local = 0;
    for (int v = lane; v < n_slots; v += 32, ++local) {
      const uint32_t sv = c.stamp[v];
      keys[local * 32 + lane] = (sv == now) ? ~0ull : (((unsigned long long)sv << 32) | (unsigned long long)v);
    }
    __syncwarp();
    const int per_lane = (n_slots + 31) / 32;
    for (int i = 0; i < q; ++i) {
      unsigned long long best = ~0ull;
      int best_at = -1;
      for (int l = 0; l < per_lane; ++l) {
        const unsigned long long kk = keys[l * 32 + lane];
        if (lane + 32 * l < n_slots && kk < best) {
          best = kk;
          best_at = l;
        }
      }
      unsigned long long wmin = best;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) {
        const unsigned long long ov = __shfl_xor_sync(0xffffffffu, wmin, o2);
        wmin = ov < wmin ? ov : wmin;
      }
      if (wmin == ~0ull) break;   // no candidate left: the rest of F overflows to C
      if (best == wmin && best_at >= 0) keys[best_at * 32 + lane] = ~0ull;
      if (inF && f_idx == i) my_victim = (int)(wmin & 0xFFFFFFFFull);
      ++n_fill;
      __syncwarp();
    }
  }
  // admissions and staging bindings
  const bool filled = inF && f_idx < n_fill;
  if (filled) {
    const int v = my_victim;
    const int32_t old = c.owner[v];
    if (old >= 0) c.slot_table[old] = MOE_STAGING_TAG | old;
    c.slot_table[base + e] = v;
    c.owner[v] = base + e;
    c.stamp[v] = now;
    o.fills[2 * f_idx] = base + e;
    o.fills[2 * f_idx + 1] = v;
  }
  if (miss && !filled) c.slot_table[base + e] = MOE_STAGING_TAG | (base + e);
  if (lane == 0) {
    *c.clock = now;
    *o.n_fill = n_fill;
    if (stats) {
      stats->n_unique = n_unique;
      stats->n_hit = n_unique - m;
      stats->n_miss = m;
      stats->q = q;
      stats->n_fill = n_fill;
      stats->n_overflow = q - n_fill;
      stats->n_staged = m - n_fill;
      stats->clock = now;
    }
  }
}

}  // namespace

bool front_small_ok(int T, int k, int E, int n_slots) {
  return T >= 1 && T * k <= 32 && E <= kMaxRouteE && n_slots <= kMaxSlotsPerLane * 32;
}

cudaError_t launch_front_small(const float* logits, int T, int k, const moe_cache& c, int layer, uint32_t phi_q16,
                               int min_fill, int policy, uint64_t seed, moe_bind_stats* stats, int32_t* topk_ids,
                               float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                               void* bind_ws, uint32_t* status, cudaStream_t s) {
  FrontOut o;
  o.topk_ids = topk_ids;
  o.topk_w = topk_w;
  o.counts = counts;
  o.offsets = offsets;
  o.perm = perm;
  o.inv_perm = inv_perm;
  o.n_fill = reinterpret_cast<int32_t*>(bind_ws);
  o.fills = o.n_fill + 4;
  return launch_k(front_small_kernel, 1, 32, 0, s, logits, T, k, c, layer, phi_q16, min_fill, policy,
                  (unsigned long long)seed, stats, o, status);
}

}  // namespace moe
