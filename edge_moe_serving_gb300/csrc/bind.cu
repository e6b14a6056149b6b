// Device-side expert-cache control and the fused batched fill copy
// (FreeToken paper, section 4.1 "Device-side cache control"; the q* split of
// section 3.2, Eq. 1-4, with the Q16 integer rounding given by the write-up
// "FreeToken: bandwidth-adaptive edge MoE serving", section "The split, and
// what it is actually optimising").
//
// bind_kernel: ONE CTA per MoE layer call.
//   1. now = ++clock (one LRU clock shared by all layers).
//   2. Deduplicate the routed ids (flag per expert) -> U ascending.
//   3. Classify against the slot table: cache-pool entries are hits (stamp
//      refreshed to now), everything else is a miss; M ascending, m = |M|.
//   4. q = fill count of m at phi (Q16 makespan rule, optional floor of 1).
//   5. F = q misses: lowest ids, or the q smallest SplitMix64 keys (seeded).
//   6. Victims in ONE pass over the recency state: every slot not stamped now
//      contributes the key (stamp << 32 | slot); a shared-memory bitonic sort
//      orders them and the miss path consumes the first q (the paper's
//      single-pass K-LRU: the cost does not depend on how many misses occur).
//   7. F[i] takes victim i: the victim's previous pair is rebound to the
//      staging pool, the table/owner/stamp are updated, (src, dst) is appended
//      to the fixed-shape fill list; the other misses (C, including overflow
//      when fewer than q victims exist) are bound to the staging pool.
// fill_copy_kernel: one fixed-shape persistent launch applies the device fill
// list to all three banks, masked by the device fill count.
#include <algorithm>

#include "dispatch_block.cuh"

namespace moe {
namespace {

constexpr int kBindThreads = 1024;
constexpr int kCopyThreads = 256;
constexpr size_t kCopyChunk = 16 * 1024;  // bytes per work item of the fill copy (one load round per CTA)

__device__ inline unsigned long long splitmix64(unsigned long long z) {
  // SplitMix64 output function (Steele, Lea & Flood 2014)
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ inline int q_rule(int m, uint32_t phi, int min_fill) {
  const long long mm = m, p = phi;
  const long long lo = (mm * p) >> 16;
  const long long c_lo = max(lo * (65536 - p), (mm - lo) * p);
  const long long c_hi = max((lo + 1) * (65536 - p), (mm - lo - 1) * p);
  long long q = (c_hi < c_lo) ? lo + 1 : lo;
  if (q > mm) q = mm;
  if (min_fill && p > 0 && mm > 0 && q < 1) q = 1;
  return (int)q;
}

__device__ int scan1024(int v, int* warp_tot, int* total) {
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
    const int w = warp_tot[lane];
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

enum : int { kNotRouted = 0, kHit = 1, kMiss = 2, kFilled = 3 };

// Outputs of the optional fused dispatch (see dispatch_block.cuh).
struct DispatchOut {
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
};

// The kernel reads all the state it needs in one batch of independent loads
// (clock, routed ids, this layer's slot-table entries, every slot's stamp),
// decides everything in shared memory, then writes: two dependent round
// trips to memory instead of one per step of the algorithm.
template <bool DISPATCH>
__global__ void __launch_bounds__(kBindThreads)
bind_kernel(moe_cache c, int layer, const int32_t* __restrict__ ids, int R, uint32_t phi_q16,
            int min_fill, int policy, unsigned long long seed, int np2, moe_bind_stats* stats,
            int32_t* __restrict__ fills, int32_t* __restrict__ n_fill_out,
            int32_t* __restrict__ fills_opt, uint32_t* status, DispatchOut dout) {
  extern __shared__ unsigned long long sm64[];
  const int E = c.E;
  unsigned long long* vkeys = sm64;                       // [np2] (stamp << 32 | slot) of candidate victims
  unsigned long long* mkeys = vkeys + np2;                // [E] random-policy keys of M
  int* st = reinterpret_cast<int*>(mkeys + E);            // [E] per-expert state
  int* ent = st + E;                                      // [E] this layer's slot-table entries
  int* Mlist = ent + E;                                   // [E] misses ascending
  int* Flist = Mlist + E;                                 // [E] fill set ascending
  __shared__ int warp_tot[32];
  __shared__ int s_total, s_m, s_q, s_nU, s_ncand;
  __shared__ uint32_t s_now;
  const int tid = threadIdx.x;
  const int base = layer * E;
  const int n_slots = c.cache.n_slots;
  pdl_wait();
  pdl_trigger();

  // 1. independent loads
  if (tid == 0) {
    s_now = *c.clock + 1u;
    s_ncand = 0;
  }
  for (int e = tid; e < E; e += kBindThreads) {
    st[e] = kNotRouted;
    ent[e] = c.slot_table[base + e];
  }
  int local_cand = 0;
  for (int v = tid; v < np2; v += kBindThreads) {
    unsigned long long key = ~0ull;
    if (v < n_slots) {
      key = ((unsigned long long)c.stamp[v] << 32) | (unsigned long long)v;
      ++local_cand;
    }
    vkeys[v] = key;
  }
  __syncthreads();
  const uint32_t now = s_now;
  bool bad = false;
  for (int i = tid; i < R; i += kBindThreads) {
    const int e = ids[i];
    if (e >= 0 && e < E) st[e] = kMiss;   // provisional: routed
    else bad = true;
  }
  if (bad) set_status(status, MOE_DEV_ERR_BAD_ID);
  __syncthreads();
  // 2. classify (thread e owns expert e; E <= 1024); a hit's slot leaves the victim candidates
  const int e = tid;
  const bool routed = (e < E) && st[e] != kNotRouted;
  bool miss = false;
  int my_slot = -1;
  if (routed) {
    const int32_t en = ent[e];
    if (en >= 0 && en < n_slots) {
      my_slot = en;
      vkeys[en] = ~0ull;
      --local_cand;   // the thread that loaded the slot's key may differ: fixed below by the count
      st[e] = kHit;
    } else {
      if (en >= 0 && en < MOE_STAGING_TAG) set_status(status, MOE_DEV_ERR_BAD_SLOT);
      miss = true;
    }
  }
  atomicAdd(&s_ncand, local_cand);
  scan1024(routed ? 1 : 0, warp_tot, &s_total);
  if (tid == 0) s_nU = s_total;
  __syncthreads();
  const int mpos = scan1024(miss ? 1 : 0, warp_tot, &s_total);
  if (miss) Mlist[mpos] = e;
  if (tid == 0) {
    s_m = s_total;
    s_q = q_rule(s_total, phi_q16, min_fill);
  }
  __syncthreads();
  const int m = s_m, q = s_q;
  // 3. fill set F (ascending ids)
  if (policy == MOE_FILL_RANDOM) {
    if (tid < m) {
      const int me = Mlist[tid];
      const unsigned long long counter = ((unsigned long long)now << 32) |
                                         ((unsigned long long)(layer & 0xFFFF) << 16) |
                                         (unsigned long long)(me & 0xFFFF);
      mkeys[tid] = splitmix64(seed ^ counter);
    }
    __syncthreads();
    bool inF = false;
    if (tid < m) {
      const unsigned long long mk = mkeys[tid];
      int rank = 0;
      for (int j = 0; j < m; ++j) {
        const unsigned long long ok = mkeys[j];
        rank += (ok < mk || (ok == mk && j < tid)) ? 1 : 0;   // Mlist ascending: j < tid <=> lower id
      }
      inF = rank < q;
    }
    const int fpos = scan1024(inF ? 1 : 0, warp_tot, &s_total);
    if (inF) Flist[fpos] = Mlist[tid];
  } else {
    if (tid < q) Flist[tid] = Mlist[tid];
  }
  __syncthreads();
  // 4. victims: the q least (stamp, slot) candidates (one pass over the state, then a
  //    shared-memory bitonic sort; skipped when nothing is filled)
  if (q > 0) {
    for (int kk = 2; kk <= np2; kk <<= 1) {
      for (int j = kk >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < np2; i += kBindThreads) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const unsigned long long a = vkeys[i], b = vkeys[ixj];
            const bool up = (i & kk) == 0;
            if ((a > b) == up) {
              vkeys[i] = b;
              vkeys[ixj] = a;
            }
          }
        }
        __syncthreads();
      }
    }
  }
  const int n_fill = min(q, s_ncand);
  // 5. writes: admit F[i] into victim i, refresh hits, bind C to the staging pool
  if (tid < n_fill) {
    const int fe = Flist[tid];
    const int v = (int)(vkeys[tid] & 0xFFFFFFFFull);
    const int32_t old = c.owner[v];
    if (old >= 0) c.slot_table[old] = MOE_STAGING_TAG | old;
    c.slot_table[base + fe] = v;
    c.owner[v] = base + fe;
    c.stamp[v] = now;
    st[fe] = kFilled;
    fills[2 * tid] = base + fe;
    fills[2 * tid + 1] = v;
    if (fills_opt) {
      fills_opt[2 * tid] = base + fe;
      fills_opt[2 * tid + 1] = v;
    }
  }
  if (my_slot >= 0) c.stamp[my_slot] = now;
  __syncthreads();
  if (tid < m) {
    const int me = Mlist[tid];
    if (st[me] != kFilled) c.slot_table[base + me] = MOE_STAGING_TAG | (base + me);
  }
  if (tid == 0) {
    *c.clock = now;
    *n_fill_out = n_fill;
    if (stats) {
      stats->n_unique = s_nU;
      stats->n_hit = s_nU - m;
      stats->n_miss = m;
      stats->q = q;
      stats->n_fill = n_fill;
      stats->n_overflow = q - n_fill;
      stats->n_staged = m - n_fill;
      stats->clock = now;
    }
  }
  if (DISPATCH) {
    // the routed rows' grouping for the expert FFN, in the same launch
    __syncthreads();
    blk::dispatch_block(ids, R, E, dout.counts, dout.offsets, dout.perm, dout.inv_perm, nullptr,
                        reinterpret_cast<int*>(sm64));
  }
}

// Copies every filled expert's rows of the three banks, staging -> cache.
__global__ void __launch_bounds__(kCopyThreads)
fill_copy_kernel(moe_pool src, moe_pool dst, size_t bank_bytes, const int32_t* __restrict__ fills,
                 const int32_t* __restrict__ n_fill_p, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int n_fill = *n_fill_p;
  // the staging copy is read once (evict first); the cache slot keeps the
  // default policy, since the expert FFN reads it right after this launch
  const uint64_t pol = l2_evict_first();
  const size_t chunks = (bank_bytes + kCopyChunk - 1) / kCopyChunk;
  const size_t items = (size_t)n_fill * 3 * chunks;
  for (size_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int f = (int)(item / (3 * chunks));
    const size_t rem = item % (3 * chunks);
    const int bank = (int)(rem / chunks);
    const size_t chunk = rem % chunks;
    const int s_slot = fills[2 * f] , d_slot = fills[2 * f + 1];
    if (s_slot < 0 || s_slot >= src.n_slots || d_slot < 0 || d_slot >= dst.n_slots) {
      if (threadIdx.x == 0) set_status(status, MOE_DEV_ERR_BAD_SLOT);
      continue;
    }
    const char* sb = reinterpret_cast<const char*>(bank == 0 ? src.w_gate : bank == 1 ? src.w_up : src.w_down);
    char* db = reinterpret_cast<char*>(bank == 0 ? dst.w_gate : bank == 1 ? dst.w_up : dst.w_down);
    const size_t lo = chunk * kCopyChunk;
    const size_t len = min(kCopyChunk, bank_bytes - lo);
    const uint4* s4 = reinterpret_cast<const uint4*>(sb + (size_t)s_slot * bank_bytes + lo);
    uint4* d4 = reinterpret_cast<uint4*>(db + (size_t)d_slot * bank_bytes + lo);
    const size_t nv = len / 16;
    size_t v = threadIdx.x;
    if (src.host) {
      // a host-resident staging pool: plain streaming loads over the CPU-GPU link
      for (; v + 3 * kCopyThreads < nv; v += 4 * kCopyThreads) {
        const uint4 a = __ldcs(s4 + v);
        const uint4 b = __ldcs(s4 + v + kCopyThreads);
        const uint4 cc = __ldcs(s4 + v + 2 * kCopyThreads);
        const uint4 d = __ldcs(s4 + v + 3 * kCopyThreads);
        d4[v] = a;
        d4[v + kCopyThreads] = b;
        d4[v + 2 * kCopyThreads] = cc;
        d4[v + 3 * kCopyThreads] = d;
      }
      for (; v < nv; v += kCopyThreads) d4[v] = __ldcs(s4 + v);
      continue;
    }
    for (; v + 3 * kCopyThreads < nv; v += 4 * kCopyThreads) {
      const uint4 a = ldg_stream_hint(s4 + v, pol);
      const uint4 b = ldg_stream_hint(s4 + v + kCopyThreads, pol);
      const uint4 cc = ldg_stream_hint(s4 + v + 2 * kCopyThreads, pol);
      const uint4 d = ldg_stream_hint(s4 + v + 3 * kCopyThreads, pol);
      d4[v] = a;
      d4[v + kCopyThreads] = b;
      d4[v + 2 * kCopyThreads] = cc;
      d4[v + 3 * kCopyThreads] = d;
    }
    for (; v < nv; v += kCopyThreads) d4[v] = ldg_stream_hint(s4 + v, pol);
  }
}

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace

size_t bind_smem_bytes(int n_slots, int E) {
  const size_t np2 = (size_t)next_pow2(n_slots < 1 ? 1 : n_slots);
  return np2 * 8 + (size_t)E * 8 + (size_t)E * 4 * 4;
}

size_t bind_ws_bytes(int T, int k, int E) {
  const size_t kmax = (size_t)std::min((long long)T * k, (long long)E);
  return align_up(kmax * 2 * sizeof(int32_t) + 16, 256);
}

// Fused residency + dispatch is used when one CTA can sort the routed rows.
bool bind_dispatch_fusable(int R, int E) { return R <= 4096 && E <= kMaxE; }

cudaError_t launch_bind(const moe_cache& c, int layer, const int32_t* ids, int R,
                        uint32_t phi_q16, int min_fill, int policy, uint64_t seed,
                        moe_bind_stats* stats, int32_t* fills_opt, void* ws, uint32_t* status,
                        cudaStream_t s, bool do_copy, int32_t* counts, int32_t* offsets, int32_t* perm,
                        int32_t* inv_perm) {
  const bool fused = counts != nullptr;
  size_t smem = bind_smem_bytes(c.cache.n_slots, c.E);
  if (fused) smem = std::max(smem, (size_t)c.E * 33 * sizeof(int));
  static std::atomic<int> attr_fused[kMaxDevices], attr_plain[kMaxDevices];
  {
    cudaError_t err = fused ? ensure_smem(bind_kernel<true>, (int)smem, attr_fused)
                            : ensure_smem(bind_kernel<false>, (int)smem, attr_plain);
    if (err != cudaSuccess) return err;
  }
  int32_t* n_fill = reinterpret_cast<int32_t*>(ws);
  int32_t* fills = n_fill + 4;
  const int np2 = next_pow2(c.cache.n_slots < 1 ? 1 : c.cache.n_slots);
  DispatchOut d = {counts, offsets, perm, inv_perm};
  cudaError_t err = fused ? launch_k(bind_kernel<true>, 1, kBindThreads, smem, s, c, layer, ids, R, phi_q16, min_fill,
                                     policy, (unsigned long long)seed, np2, stats, fills, n_fill, fills_opt, status, d)
                          : launch_k(bind_kernel<false>, 1, kBindThreads, smem, s, c, layer, ids, R, phi_q16, min_fill,
                                     policy, (unsigned long long)seed, np2, stats, fills, n_fill, fills_opt, status, d);
  if (err != cudaSuccess) return err;
  if (!do_copy || c.staging.w_gate == nullptr) return cudaSuccess;   // copy fused elsewhere / no staging pool
  const size_t bank_bytes = (size_t)c.H * c.I * sizeof(__nv_bfloat16);
  return launch_k(fill_copy_kernel, num_sms() * 4, kCopyThreads, 0, s, c.staging, c.cache, bank_bytes,
                  (const int32_t*)fills, (const int32_t*)n_fill, status);
}

}  // namespace moe
