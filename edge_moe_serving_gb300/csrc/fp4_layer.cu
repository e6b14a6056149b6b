// The routed MoE layer over an FP4 expert cache (FreeToken paper, section
// 5.1: DeepSeek-V4-Flash serves MXFP4 experts, GLM-5.2 and the laptop
// Qwen3.6 build NVFP4 ones; section 3.2: router, cache lookup and split,
// grouped evaluation, exact merge; section 4.1: device-side cache control and
// a fill copy that moves every bank of an admitted expert under one list).
//
// Per-step launches: router and top-k, the residency bind (the bf16 layer's
// bind kernel: its decisions only need the residency arrays and the cache
// pool's slot count), the FP4 fill copy below, dispatch (in the bind launch
// when it is small enough), the FP4 expert FFN and the combine.
#include <algorithm>
#include <climits>

#include "mxfp4.cuh"

namespace moe {
namespace {

constexpr int kFillThreads = 256;
constexpr size_t kFillChunk = 64 * 1024;   // bytes of one bank of one fill per work item

// Copies every filled expert's slot of every bank, staging -> cache.  Work
// items are (fill, bank, 64 KB chunk); banks whose slot size is a multiple of
// 16 bytes (every code and scale bank of a supported shape) move 16-byte
// words, the tensor scales (12 bytes per slot) 4-byte words.
__global__ void __launch_bounds__(kFillThreads)
fp4_fill_kernel(Fp4FillBanks fb, const int32_t* __restrict__ fills, const int32_t* __restrict__ n_fill_p,
                uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int n_fill = *n_fill_p;
  size_t max_chunks = 1;
  for (int b = 0; b < fb.n; ++b) max_chunks = max(max_chunks, (fb.slot_bytes[b] + kFillChunk - 1) / kFillChunk);
  const size_t items = (size_t)n_fill * fb.n * max_chunks;
  const uint64_t pol = l2_evict_first();
  for (size_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int f = (int)(item / ((size_t)fb.n * max_chunks));
    const size_t rem = item % ((size_t)fb.n * max_chunks);
    const int b = (int)(rem / max_chunks);
    const size_t chunk = rem % max_chunks;
    const size_t slot_bytes = fb.slot_bytes[b];
    const size_t lo = chunk * kFillChunk;
    if (lo >= slot_bytes) continue;
    const int s_slot = fills[2 * f], d_slot = fills[2 * f + 1];
    if (s_slot < 0 || s_slot >= fb.src_slots || d_slot < 0 || d_slot >= fb.dst_slots) {
      if (threadIdx.x == 0 && chunk == 0 && b == 0) set_status(status, MOE_DEV_ERR_BAD_SLOT);
      continue;
    }
    const size_t len = min(kFillChunk, slot_bytes - lo);
    const uint8_t* src = fb.src[b] + (size_t)s_slot * slot_bytes + lo;
    uint8_t* dst = fb.dst[b] + (size_t)d_slot * slot_bytes + lo;
    if ((slot_bytes & 15) == 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (size_t v = threadIdx.x; v < len / 16; v += kFillThreads) d4[v] = ldg_stream_hint(s4 + v, pol);
    } else {
      const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src);
      uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
      for (size_t v = threadIdx.x; v < len / 4; v += kFillThreads) d1[v] = s1[v];
    }
  }
}

inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ring_dim(int d) { return d == 1024 || d == 2048 || d == 4096; }   // the ring kernel's H and I
// NVFP4 calls run on the ring kernel (at most 64 routed rows, rows of 1024, 2048 or 4096 inputs) or on
// the tensor-core GEMM (I a multiple of 128, H of 256, every row's 16-input scales in 8-byte groups)
inline bool nv_ffn_shape(long long R, int H, int I) {
  return (R <= kFp4RingMaxRows && ring_dim(H) && ring_dim(I)) || (I % 128 == 0 && H % 256 == 0);
}

struct Fp4Ws {
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  float* y_rows;
  void* bind_ws;
  float* dec_logits;
  __nv_bfloat16* dec_h;
  unsigned int* dec_words;
  void* scratch;
  size_t scratch_bytes, bytes;
};

Fp4Ws fp4_ws(void* ws, int T, int k, int E, int H, int I) {
  const size_t R = (size_t)T * k;
  char* base = reinterpret_cast<char*>(ws);
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return p;
  };
  Fp4Ws L;
  L.ids = static_cast<int32_t*>(take(R * 4));
  L.w = static_cast<float*>(take(R * 4));
  L.counts = static_cast<int32_t*>(take((size_t)E * 4));
  L.offsets = static_cast<int32_t*>(take((size_t)(E + 1) * 4));
  L.perm = static_cast<int32_t*>(take(R * 4));
  L.inv_perm = static_cast<int32_t*>(take(R * 4));
  L.y_rows = static_cast<float*>(take(R * H * 4));
  L.bind_ws = take(bind_ws_bytes(T, k, E));
  // one-token calls: the one-launch kernel's logits, h rows and barrier words
  L.dec_logits = static_cast<float*>(T == 1 ? take((size_t)E * 4) : nullptr);
  L.dec_h = static_cast<__nv_bfloat16*>(T == 1 ? take(R * I * 2) : nullptr);
  L.dec_words = static_cast<unsigned int*>(T == 1 ? take((4 + R) * 4) : nullptr);
  L.scratch_bytes = std::max({route_ws_bytes(T, H, E), dispatch_ws_bytes(T, k, E),
                              moe_expert_ffn_mxfp4_workspace_size(T, k, H, I),
                              moe_expert_ffn_nvfp4_workspace_size(T, k, H, I), (size_t)256});
  L.scratch = take(L.scratch_bytes);
  L.bytes = off;
  return L;
}

// The bf16 cache view the bind kernel reads: the residency arrays and the
// pools' slot counts (the bind kernel never reads a bank).
moe_cache bind_view(const moe_cache_fp4& c) {
  moe_cache v = {};
  v.cache.w_gate = const_cast<void*>(c.cache.gate_q);
  v.cache.w_up = const_cast<void*>(c.cache.up_q);
  v.cache.w_down = const_cast<void*>(c.cache.down_q);
  v.cache.n_slots = c.cache.n_slots;
  if (c.staging.gate_q) {
    v.staging.w_gate = const_cast<void*>(c.staging.gate_q);
    v.staging.w_up = const_cast<void*>(c.staging.up_q);
    v.staging.w_down = const_cast<void*>(c.staging.down_q);
    v.staging.n_slots = c.staging.n_slots;
  }
  v.slot_table = c.slot_table;
  v.owner = c.owner;
  v.stamp = c.stamp;
  v.clock = c.clock;
  v.n_layers = c.n_layers;
  v.E = c.E;
  v.H = c.H;
  v.I = c.I;
  return v;
}

// The banks a fill copies, staging slot -> cache slot (only read when there is a staging pool).
Fp4FillBanks fill_banks(const moe_cache_fp4& c, bool nv) {
  Fp4FillBanks fb = {};
  const int SB = nv ? 16 : kMxBlock;
  const size_t H = (size_t)c.H, I = (size_t)c.I;
  const moe_pool_nvfp4& a = c.cache;
  const moe_pool_nvfp4& b = c.staging;
  const size_t gq = I * H / 2, gs = I * H / SB, dq = H * I / 2, ds = H * I / SB;
  const void* srcs[6] = {b.gate_q, b.gate_s, b.up_q, b.up_s, b.down_q, b.down_s};
  const void* dsts[6] = {a.gate_q, a.gate_s, a.up_q, a.up_s, a.down_q, a.down_s};
  const size_t sizes[6] = {gq, gs, gq, gs, dq, ds};
  for (int i = 0; i < 6; ++i) {
    fb.src[i] = static_cast<const uint8_t*>(srcs[i]);
    fb.dst[i] = static_cast<uint8_t*>(const_cast<void*>(dsts[i]));
    fb.slot_bytes[i] = sizes[i];
  }
  fb.n = 6;
  if (nv) {
    fb.src[6] = reinterpret_cast<const uint8_t*>(b.tensor_scale);
    fb.dst[6] = reinterpret_cast<uint8_t*>(const_cast<float*>(a.tensor_scale));
    fb.slot_bytes[6] = 3 * sizeof(float);
    fb.n = 7;
  }
  fb.src_slots = b.gate_q ? b.n_slots : 0;
  fb.dst_slots = a.n_slots;
  return fb;
}

// The ring kernels' parameter block over the FP4 cache's pools.
MxParams mx_params(const moe_cache_fp4& c, bool nv, int layer, int k) {
  MxParams p = {};
  const moe_pool_nvfp4* ps[2] = {&c.cache, &c.staging};
  moe_pool_mxfp4* qs[2] = {&p.a, &p.b};
  for (int i = 0; i < 2; ++i) {
    if (!ps[i]->gate_q) continue;   // no staging pool: n_slots 0, staging entries read as out of range
    qs[i]->gate_q = ps[i]->gate_q;
    qs[i]->gate_s = ps[i]->gate_s;
    qs[i]->up_q = ps[i]->up_q;
    qs[i]->up_s = ps[i]->up_s;
    qs[i]->down_q = ps[i]->down_q;
    qs[i]->down_s = ps[i]->down_s;
    qs[i]->n_slots = ps[i]->n_slots;
  }
  if (nv) {
    p.ts_a = c.cache.tensor_scale;
    p.ts_b = c.staging.gate_q ? c.staging.tensor_scale : nullptr;
  }
  p.slot_table = c.slot_table;
  p.layer = layer;
  p.E = c.E;
  p.H = c.H;
  p.I = c.I;
  p.k = k;
  return p;
}

int pool_check(const moe_pool_nvfp4& p, bool nv, bool required) {
  if (!p.gate_q && !p.up_q && !p.down_q && !required) return MOE_OK;
  if (!p.gate_q || !p.gate_s || !p.up_q || !p.up_s || !p.down_q || !p.down_s || p.n_slots < 1)
    return MOE_ERR_INVALID_ARG;
  if (nv && !p.tensor_scale) return MOE_ERR_INVALID_ARG;
  if (!a16(p.gate_q) || !a16(p.up_q) || !a16(p.down_q) || !a16(p.gate_s) || !a16(p.up_s) || !a16(p.down_s) ||
      (nv && (reinterpret_cast<uintptr_t>(p.tensor_scale) & 3u) != 0))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_layer_fp4_workspace_size(const moe_layer* layer, const moe_cache_fp4* cache, int T) {
  if (!layer || !cache || T < 0 || layer->k < 1 || layer->k > layer->E || layer->k > kMaxK ||
      (long long)T * layer->k > INT_MAX / 2)
    return 0;
  return fp4_ws(nullptr, T, layer->k, layer->E, layer->H, layer->I).bytes;
}

extern "C" int moe_layer_forward_fp4(const moe_layer* layer, const moe_cache_fp4* cache, const void* x, int T,
                                     void* out, uint32_t phi_q16, int min_fill, int fill_policy, uint64_t seed,
                                     void* ws, size_t ws_bytes, uint32_t* dev_status, moe_bind_stats* stats_dev,
                                     moe_stream_t stream) {
  if (!layer || !cache) return MOE_ERR_INVALID_ARG;
  const int E = layer->E, H = layer->H, I = layer->I, k = layer->k;
  if (cache->format != MOE_FP4_MXFP4 && cache->format != MOE_FP4_NVFP4) return MOE_ERR_INVALID_ARG;
  const bool nv = cache->format == MOE_FP4_NVFP4;
  if (cache->E != E || cache->H != H || cache->I != I || layer->layer < 0 || layer->layer >= cache->n_layers)
    return MOE_ERR_INVALID_ARG;
  if (T < 0 || k < 1 || k > E || k > kMaxK || !cache->slot_table || !cache->owner || !cache->stamp || !cache->clock)
    return MOE_ERR_INVALID_ARG;
  // every shape check of the FFN step is made here, before the bind updates the residency state
  const int SB = nv ? 16 : kMxBlock;
  if (H < SB || I < SB) return MOE_ERR_INVALID_ARG;
  if ((long long)T * k > INT_MAX / 2 || E > kMaxE || H % SB || I % SB ||
      (long long)cache->n_layers * E > MOE_SLOT_MASK || cache->cache.n_slots > kMaxCacheSlots)
    return MOE_ERR_UNSUPPORTED;
  if (nv && !nv_ffn_shape((long long)T * k, H, I)) return MOE_ERR_UNSUPPORTED;
  int st = pool_check(cache->cache, nv, true);
  if (st != MOE_OK) return st;
  st = pool_check(cache->staging, nv, false);
  if (st != MOE_OK) return st;
  if (phi_q16 > 65536u || (fill_policy != MOE_FILL_LOWEST_ID && fill_policy != MOE_FILL_RANDOM))
    return MOE_ERR_INVALID_ARG;
  if (phi_q16 > 0 && (!cache->staging.gate_q || (long long)cache->staging.n_slots < (long long)cache->n_layers * E))
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || !layer->w_router) return MOE_ERR_INVALID_ARG;
  if (!a16(x) || !a16(layer->w_router) || E > kMaxRouteE) return MOE_ERR_UNSUPPORTED;   // the router's own limits
  const Fp4Ws need = fp4_ws(nullptr, T, k, E, H, I);
  if (!ws || ws_bytes < need.bytes) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_UNSUPPORTED;
  const Fp4Ws L = fp4_ws(ws, T, k, E, H, I);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int R = T * k;

  MxParams mp = mx_params(*cache, nv, layer->layer, k);
  if (T == 1 && fp4_decode_ok(mp, T, cache->cache.n_slots)) {
    // one token: the whole layer in one cooperative launch
    mp.x = static_cast<const __nv_bfloat16*>(x);
    mp.h = L.dec_h;
    mp.y = L.y_rows;
    mp.status = dev_status;
    Fp4DecodeArgs a = {};
    a.c = bind_view(*cache);
    a.w_router = layer->w_router;
    a.bias = layer->bias;
    a.phi_q16 = phi_q16;
    a.min_fill = min_fill;
    a.policy = fill_policy;
    a.seed = seed;
    a.stats = stats_dev;
    a.logits = L.dec_logits;
    a.topk_ids = L.ids;
    a.topk_w = L.w;
    a.counts = L.counts;
    a.offsets = L.offsets;
    a.perm = L.perm;
    a.inv_perm = L.inv_perm;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.grid_count = L.dec_words;
    a.fill = fill_banks(*cache, nv);
    if (phi_q16 == 0 || !cache->staging.gate_q) a.fill.n = 0;   // no fills are admitted
    return launch_fp4_decode(mp, nv, a, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }

  st = moe_route_topk(x, T, H, layer->w_router, layer->bias, E, k, L.ids, L.w, nullptr, L.scratch, L.scratch_bytes,
                      dev_status, stream);
  if (st != MOE_OK) return st;
  const moe_cache view = bind_view(*cache);
  const bool fuse_dispatch = bind_dispatch_fusable(R, E);
  if (launch_bind(view, layer->layer, L.ids, R, phi_q16, min_fill, fill_policy, seed, stats_dev, nullptr, L.bind_ws,
                  dev_status, s, false, fuse_dispatch ? L.counts : nullptr, L.offsets, L.perm, L.inv_perm) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (cache->staging.gate_q && phi_q16 > 0) {
    // the admitted experts: every bank's slot, staging -> cache
    const Fp4FillBanks fb = fill_banks(*cache, nv);
    const int32_t* n_fill = reinterpret_cast<const int32_t*>(L.bind_ws);
    if (launch_k(fp4_fill_kernel, num_sms() * 4, kFillThreads, 0, s, fb, n_fill + 4, n_fill, dev_status) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (!fuse_dispatch) {
    st = moe_dispatch(L.ids, T, k, E, L.counts, L.offsets, L.perm, L.inv_perm, nullptr, H, nullptr, L.scratch,
                      L.scratch_bytes, dev_status, stream);
    if (st != MOE_OK) return st;
  }
  if (nv) {
    st = moe_expert_ffn_nvfp4(&cache->cache, cache->staging.gate_q ? &cache->staging : nullptr, cache->slot_table,
                              cache->n_layers, layer->layer, E, H, I, L.counts, L.offsets, L.perm, x, T, k, L.y_rows,
                              L.scratch, L.scratch_bytes, dev_status, stream);
  } else {
    st = moe_expert_ffn_mxfp4(&mp.a, cache->staging.gate_q ? &mp.b : nullptr, cache->slot_table, cache->n_layers,
                              layer->layer, E, H, I, L.counts, L.offsets, L.perm, x, T, k, L.y_rows, L.scratch,
                              L.scratch_bytes, dev_status, stream);
  }
  if (st != MOE_OK) return st;
  return moe_combine(L.y_rows, L.w, T, k, H, out, nullptr, dev_status, stream);
}
