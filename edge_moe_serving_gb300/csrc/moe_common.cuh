// Shared device helpers and internal launch declarations of libmoe.
#pragma once

#include <atomic>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kNumSMs = 152;          // GB300: 2 dies x 76 SMs (queried at run time too)
constexpr int kMaxE = 1024;           // bind / dispatch limit
constexpr int kMaxRouteE = 512;       // router top-k limit (16 logits per lane)
constexpr int kMaxK = 16;
constexpr int kMaxCacheSlots = 16384; // bind kernel keeps all (stamp, slot) keys in shared memory
constexpr int kGemvMaxRows = 2;       // AUTO mode: calls of up to this many tokens use the GEMV path

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// The fused TMA-ring GEMV handles row lengths that are multiples of 256 whose
// units (one gate row + one up row, or one down row) fit a 16 KB stage.
inline bool gemv_fused_ok(int H, int I) {
  return H % 256 == 0 && I % 256 == 0 && 2 * H * 2 <= 16384 && I * 2 <= 16384;
}

// ---------------------------------------------------------------- launch chaining
// Every kernel of the library is launched with programmatic stream
// serialization: the next kernel on the stream may start its prologue while
// this one drains.  Each kernel calls pdl_wait() before it reads anything a
// previous kernel wrote (on every path, so completion stays transitive), and
// pdl_trigger() once its dependents may be scheduled.  Without the launch
// attribute both are no-ops.
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Kernels this library has launched or captured into a graph in this process
// (host-side count, one per launch call that the runtime accepted).
inline std::atomic<unsigned long long>& launch_counter() {
  static std::atomic<unsigned long long> n{0};
  return n;
}

inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) launch_counter().fetch_add(1, std::memory_order_relaxed);
  return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...));
}

// ---------------------------------------------------------------- bounded waits
// Every wait of a pipelined kernel on an mbarrier goes through bounded_wait:
// it gives up after about one second of %globaltimer, raises the CTA's abort
// flag and returns false; the caller then winds down (drains its copies,
// frees TMEM) and the kernel reports MOE_DEV_ERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ inline unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// L2 policy for bytes read once per call (expert weights): evict first, so
// that a weight stream replaces its own lines rather than reusable ones
// (token rows, h, expert rows) or lines that would need a write-back.
__device__ inline uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ inline bool mbar_try_wait_parity(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ inline bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  unsigned long long start = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_parity(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (*abort_flag) return false;
      const unsigned long long now = globaltimer_ns();
      if (start == 0) start = now;
      else if (now - start > kWaitLimitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- device status
__device__ inline void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------- bf16 helpers
// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits.
__device__ inline float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ inline float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

__device__ inline uint4 ldg_stream(const void* p) {
  // 16-byte load that does not allocate in L1: weights are read once.
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ldg_stream with an L2 cache policy (bytes read once: evict first).
__device__ inline uint4 ldg_stream_hint(const void* p, uint64_t policy) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(policy));
  return r;
}

__device__ inline uint4 ldg_cached(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Dot product of 8 bf16 weights with 8 bf16 activations, accumulated in fp32.
__device__ inline float dot8(const uint4& w, const uint4& a, float acc) {
  acc = fmaf(bf16_lo(w.x), bf16_lo(a.x), acc);
  acc = fmaf(bf16_hi(w.x), bf16_hi(a.x), acc);
  acc = fmaf(bf16_lo(w.y), bf16_lo(a.y), acc);
  acc = fmaf(bf16_hi(w.y), bf16_hi(a.y), acc);
  acc = fmaf(bf16_lo(w.z), bf16_lo(a.z), acc);
  acc = fmaf(bf16_hi(w.z), bf16_hi(a.z), acc);
  acc = fmaf(bf16_lo(w.w), bf16_lo(a.w), acc);
  acc = fmaf(bf16_hi(w.w), bf16_hi(a.w), acc);
  return acc;
}

__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ inline float silu(float g) { return g / (1.0f + expf(-g)); }

// silu with CUDA's fast exponential and division intrinsics, for epilogues
// whose result is rounded to bf16.  As g -> -inf the divisor overflows and the
// intrinsic division returns 0, the limit of silu.
__device__ inline float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Order-preserving map of a float to 32 unsigned bits (larger float, larger
// key; equal floats, equal keys); its inverse.
__device__ inline uint32_t ord_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);   // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ inline float ord_val(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k); }

// One warp selects the top-k of one token's logits (E <= 512; order: logit
// descending, id ascending) and renormalises the softmax over the selection.
// On return lane r < k holds the r-th selected id in ascending order and its
// weight.  Lane l holds experts l + 32 j (j < PER) as 64-bit words
// (key << 32 | ~id), sorted in registers in descending order by a bitonic
// network, so its head is its best candidate (largest logit, then lowest id).
// A round is two warp reductions (largest head key, then the lowest id among
// the lanes whose head holds it), and the lane that owned the winner pops its
// head with a branch-free shift.  L2_ONLY: read the row through L2 (rows
// written by other CTAs of the launch).
template <bool L2_ONLY, int PER>
__device__ inline void topk_sorted(const float* row, int E, int k, int& id_out, float& w_out) {
  const int lane = threadIdx.x & 31;
  unsigned long long c[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    float v = 0.0f;
    if (e < E) v = L2_ONLY ? __ldcg(row + e) : row[e];
    // no expert: 0 (key 0, id field ~0xffffffff = 0) sorts below every expert
    c[j] = (e < E) ? (((unsigned long long)ord_key(v) << 32) | (unsigned long long)(~(uint32_t)e)) : 0ull;
  }
#pragma unroll
  for (int size = 2; size <= PER; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;   // the last merge (size == PER) is descending throughout
          const unsigned long long a = c[i], b = c[j];
          const bool sw = desc ? (a < b) : (a > b);
          c[i] = sw ? b : a;
          c[j] = sw ? a : b;
        }
      }
  float sel_v = -INFINITY;
  int sel_id = 0x7fffffff;
  for (int r = 0; r < k; ++r) {
    const uint32_t hk = (uint32_t)(c[0] >> 32);
    const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t id = __reduce_min_sync(0xffffffffu, hk == m ? ~(uint32_t)c[0] : 0xffffffffu);
    if (lane == r) {
      sel_v = ord_val(m);
      sel_id = (int)id;
    }
    const bool pop = (int)(id & 31u) == lane;
#pragma unroll
    for (int j = 0; j + 1 < PER; ++j) c[j] = pop ? c[j + 1] : c[j];
    c[PER - 1] = pop ? 0ull : c[PER - 1];
  }
  const float vmax = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = (lane < k) ? expf(sel_v - vmax) : 0.0f;
  const float denom = warp_sum(ex);
  int rank = 0;
  for (int j = 0; j < k; ++j) rank += (__shfl_sync(0xffffffffu, sel_id, j) < sel_id) ? 1 : 0;
  // lane `rank` receives the id of rank `rank`
  int out_id = 0x7fffffff;
  float out_w = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int rj = __shfl_sync(0xffffffffu, rank, j);
    const int ij = __shfl_sync(0xffffffffu, sel_id, j);
    const float wj = __shfl_sync(0xffffffffu, ex, j);
    if (lane == rj) {
      out_id = ij;
      out_w = wj / denom;
    }
  }
  id_out = out_id;
  w_out = out_w;
}

// topk_sorted with as few candidates per lane as E allows.
template <bool L2_ONLY>
__device__ inline void topk_core(const float* row, int E, int k, int& id_out, float& w_out) {
  if (E <= 128) topk_sorted<L2_ONLY, 4>(row, E, k, id_out, w_out);
  else if (E <= 256) topk_sorted<L2_ONLY, 8>(row, E, k, id_out, w_out);
  else topk_sorted<L2_ONLY, kMaxRouteE / 32>(row, E, k, id_out, w_out);
}

// topk_core writing the selection: ids_out[0..k) ascending, w_out[0..k).
__device__ inline void warp_topk(const float* row, int E, int k, int32_t* ids_out, float* w_out) {
  int id;
  float w;
  topk_core<false>(row, E, k, id, w);
  const int lane = threadIdx.x & 31;
  if (lane < k) {
    ids_out[lane] = id;
    w_out[lane] = w;
  }
}

// Slot-table decoding: returns the bank base row pointer set for (pool, slot),
// or false when the entry is unbound or out of range.
struct BankSet {
  const __nv_bfloat16* gate;
  const __nv_bfloat16* up;
  const __nv_bfloat16* down;
};

__device__ inline bool resolve_slot(const moe_cache& c, int32_t entry, int H, int I, BankSet* out,
                                    uint32_t* status) {
  if (entry < 0) {
    set_status(status, MOE_DEV_ERR_UNBOUND);
    return false;
  }
  const moe_pool* pool = (entry & MOE_STAGING_TAG) ? &c.staging : &c.cache;
  const int32_t slot = entry & MOE_SLOT_MASK;
  if ((entry & ~(MOE_STAGING_TAG | MOE_SLOT_MASK)) != 0 || slot >= pool->n_slots) {
    set_status(status, MOE_DEV_ERR_BAD_SLOT);
    return false;
  }
  const size_t per = (size_t)H * (size_t)I;
  out->gate = reinterpret_cast<const __nv_bfloat16*>(pool->w_gate) + (size_t)slot * per;
  out->up = reinterpret_cast<const __nv_bfloat16*>(pool->w_up) + (size_t)slot * per;
  out->down = reinterpret_cast<const __nv_bfloat16*>(pool->w_down) + (size_t)slot * per;
  return true;
}

// resolve_slot for kernels that take part of the experts only: filter 1
// skips (silently) experts bound to the staging pool, filter 2 those bound
// to the cache pool; unbound and malformed entries are reported either way.
constexpr int kPoolAll = 0, kPoolDeviceOnly = 1, kPoolStagingOnly = 2;
__device__ inline bool resolve_filtered(const moe_cache& c, int32_t entry, int filter, int H, int I, BankSet* out,
                                        uint32_t* status) {
  if (entry >= 0) {
    const bool staged = (entry & MOE_STAGING_TAG) != 0;
    if ((filter == kPoolDeviceOnly && staged) || (filter == kPoolStagingOnly && !staged)) return false;
  }
  return resolve_slot(c, entry, H, I, out, status);
}

// ---------------------------------------------------------------- internal launchers
int num_sms();   // SMs of the current device

// Host-side setup that must be done once per device (kernel attributes are
// per device): `done` is a zero-initialised static table, one flag per
// device.  fn() runs until it succeeds on the current device; concurrent
// first calls may both run it, so it must be idempotent (setting an
// attribute to the same value is).
constexpr int kMaxDevices = 64;

// Current device, or -1 when it cannot be read or is beyond kMaxDevices.
inline int device_index() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev >= 0 && dev < kMaxDevices ? dev : -1;
}

// Raises `kern`'s dynamic shared memory limit on the current device to at
// least `bytes`.  `cur` holds the limit set so far per device; the attribute
// is only ever raised, under one lock, so a launch that saw cur >= its size
// never meets a lower limit set by another thread.
std::mutex& smem_attr_mutex();
template <class K>
inline cudaError_t ensure_smem(K* kern, int bytes, std::atomic<int> (&cur)[kMaxDevices]) {
  const int dev = device_index();
  if (dev >= 0 && cur[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  std::lock_guard<std::mutex> lock(smem_attr_mutex());
  if (dev >= 0 && cur[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0) cur[dev].store(bytes, std::memory_order_release);
  return e;
}

template <class Fn>
inline cudaError_t once_per_device(std::atomic<unsigned char> (&done)[kMaxDevices], Fn&& fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev].store(1, std::memory_order_release);
  return e;
}

cudaError_t launch_route_topk(const __nv_bfloat16* x, int T, int H, const float* w_router,
                              const float* bias, int E, int k, int32_t* topk_ids, float* topk_w,
                              float* logits_opt, void* ws, uint32_t* status, cudaStream_t s);
size_t route_ws_bytes(int T, int H, int E);
bool route_tc_ok(int T, int H, int E);
// One warp per token: logits (+ bias, written back when asked) -> top-k ids and weights.
cudaError_t launch_topk(float* logits, const float* bias, int T, int E, int k, bool write_back, int32_t* topk_ids,
                        float* topk_w, cudaStream_t s);
size_t route_tc_ws_bytes(int T, int H, int E);
cudaError_t launch_route_tc(const __nv_bfloat16* x, int T, int H, const float* w_router, const float* bias, int E,
                            int k, int32_t* topk_ids, float* topk_w, float* logits_opt, void* ws, uint32_t* status,
                            cudaStream_t s);
cudaError_t launch_route_logits(const __nv_bfloat16* x, int T, int H, const float* w_router, const float* bias,
                                int E, float* logits, cudaStream_t s);
bool decode_layer_ok(int T, int k, int E, int H, int I, int n_slots);
cudaError_t launch_decode_layer(const moe_cache& c, int layer, const __nv_bfloat16* x, int T, int k,
                                const float* w_router, const float* bias, uint32_t phi_q16, int min_fill, int policy,
                                uint64_t seed, moe_bind_stats* stats, float* logits, int32_t* topk_ids, float* topk_w,
                                int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm, float* y_rows,
                                __nv_bfloat16* h, unsigned int* grid_count, __nv_bfloat16* out, uint32_t* status,
                                cudaStream_t s);
bool front_small_ok(int T, int k, int E, int n_slots);
cudaError_t launch_front_small(const float* logits, int T, int k, const moe_cache& c, int layer, uint32_t phi_q16,
                               int min_fill, int policy, uint64_t seed, moe_bind_stats* stats, int32_t* topk_ids,
                               float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                               void* bind_ws, uint32_t* status, cudaStream_t s);

size_t dispatch_ws_bytes(int T, int k, int E);
cudaError_t launch_dispatch(const int32_t* ids, int R, int k, int E, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                            const __nv_bfloat16* x, int H, __nv_bfloat16* x_perm, void* ws,
                            uint32_t* status, cudaStream_t s);

cudaError_t launch_gather(const __nv_bfloat16* x, int H, int k, const int32_t* perm, const int32_t* offsets, int E,
                          int R, __nv_bfloat16* x_perm, cudaStream_t s);

size_t bind_ws_bytes(int T, int k, int E);
size_t bind_smem_bytes(int n_slots, int E);
// ws holds the fill count (int32 at offset 0) and the fill list (from int32 offset 4).
// do_copy = false leaves the copy to a fused-fill FFN launch.
// counts != nullptr: the same single-CTA launch also does the dispatch (R <= 4096).
bool bind_dispatch_fusable(int R, int E);
cudaError_t launch_bind(const moe_cache& c, int layer, const int32_t* ids, int R,
                        uint32_t phi_q16, int min_fill, int policy, uint64_t seed,
                        moe_bind_stats* stats, int32_t* fills_opt, void* ws, uint32_t* status,
                        cudaStream_t s, bool do_copy = true, int32_t* counts = nullptr,
                        int32_t* offsets = nullptr, int32_t* perm = nullptr, int32_t* inv_perm = nullptr);

size_t ffn_ws_bytes(int T, int k, int E, int H, int I, int mode);
int ffn_check_args(const moe_cache* cache, int layer, const int32_t* counts, const int32_t* offsets,
                   const int32_t* perm, const void* x, const void* x_perm_opt, int T, int k, int ffn_mode,
                   const float* y_rows);
bool gemm_shape_ok(int H, int I);
cudaError_t launch_ffn(const moe_cache& c, int layer, const int32_t* counts, const int32_t* offsets,
                       const int32_t* perm, const __nv_bfloat16* x, const __nv_bfloat16* x_perm,
                       int T, int k, const uint8_t* mask, int mode, float* y_rows, void* ws,
                       uint32_t* status, cudaStream_t s, const int32_t* fused_fills = nullptr,
                       const int32_t* fused_n_fill = nullptr, const float* combine_w = nullptr,
                       __nv_bfloat16* combine_out = nullptr, __nv_bfloat16* y_rows_bf16 = nullptr);

cudaError_t launch_combine(const float* y_rows, const float* topk_w, int T, int k, int H,
                           __nv_bfloat16* out, float* out_f32, uint32_t* status, cudaStream_t s);
cudaError_t launch_combine(const __nv_bfloat16* y_rows, const float* topk_w, int T, int k, int H,
                           __nv_bfloat16* out, float* out_f32, uint32_t* status, cudaStream_t s);

}  // namespace moe
