// C ABI of libmoe (declared in include/moe.h): argument checks, workspace
// layouts and the layer-level composition.  Every entry point only enqueues
// work on the caller's stream.
#include <algorithm>
#include <climits>
#include <cstdint>

#include "moe_common.cuh"

namespace moe {

std::mutex& smem_attr_mutex() {
  static std::mutex m;
  return m;
}

int num_sms() {
  static std::atomic<int> cached[kMaxDevices];   // per device, 0 = not read yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kNumSMs;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kNumSMs;
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

namespace {

constexpr int kVersion = 100;   // 1.0.0

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// workspaces are carved into 256-byte aligned regions read with vector loads
inline bool ws_aligned(const void* ws) { return (reinterpret_cast<uintptr_t>(ws) & 255u) == 0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int check_pool(const moe_pool& p, bool required) {
  if (p.w_gate == nullptr && p.w_up == nullptr && p.w_down == nullptr && !required) return MOE_OK;
  if (!p.w_gate || !p.w_up || !p.w_down || p.n_slots < 1) return MOE_ERR_INVALID_ARG;
  if (!aligned16(p.w_gate) || !aligned16(p.w_up) || !aligned16(p.w_down)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_cache(const moe_cache* c) {
  if (!c || !c->slot_table || c->n_layers < 1 || c->E < 1 || c->H < 8 || c->I < 8) return MOE_ERR_INVALID_ARG;
  if (c->E > kMaxE || (c->H % 8) || (c->I % 8)) return MOE_ERR_UNSUPPORTED;
  if ((long long)c->n_layers * c->E > MOE_SLOT_MASK) return MOE_ERR_UNSUPPORTED;
  int st = check_pool(c->cache, true);
  if (st != MOE_OK) return st;
  if (c->cache.host != 0) return MOE_ERR_UNSUPPORTED;   // the cache pool is the GPU's own memory
  return check_pool(c->staging, false);
}

int check_bind_args(const moe_cache* cache, int layer, int T, int k, uint32_t phi_q16, int fill_policy) {
  int st = check_cache(cache);
  if (st != MOE_OK) return st;
  if (!cache->owner || !cache->stamp || !cache->clock) return MOE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= cache->n_layers || T < 0 || k < 1 || k > cache->E) return MOE_ERR_INVALID_ARG;
  if (phi_q16 > 65536u) return MOE_ERR_INVALID_ARG;
  if (fill_policy != MOE_FILL_LOWEST_ID && fill_policy != MOE_FILL_RANDOM) return MOE_ERR_INVALID_ARG;
  if (cache->cache.n_slots > kMaxCacheSlots) return MOE_ERR_UNSUPPORTED;
  // any fill copies from the staging pool, which must then hold every (layer, expert) pair
  if (phi_q16 > 0 && (cache->staging.w_gate == nullptr ||
                      (long long)cache->staging.n_slots < (long long)cache->n_layers * cache->E))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

struct Carve {
  char* base;
  size_t off = 0;
  explicit Carve(void* b) : base(reinterpret_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align_up(off + count * sizeof(T), 256);
    return p;
  }
};

// Workspace of moe_layer_forward: intermediates, then one scratch region
// shared by the sequential sub-calls.
struct LayerWs {
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  float* y_rows;
  __nv_bfloat16* x_perm;
  float* logits;     // decode-sized calls: router logits of the one-launch layer
  void* bind_ws;     // fill count + fill list, alive until the FFN has run
  void* scratch;
  size_t bytes;
};

// gathered rows feed the GEMM kernel, which AUTO uses for calls of more than kGemvMaxRows tokens
bool needs_x_perm(int mode, int T) {
  return mode == MOE_FFN_GEMM || (mode == MOE_FFN_AUTO && T > kGemvMaxRows);
}

LayerWs layer_ws(void* ws, const moe_layer_buffers* b, int T, int k, int E, int H, int I, int mode) {
  const size_t R = (size_t)T * k;
  Carve cv(ws);
  LayerWs L;
  // the layout does not depend on bufs_opt: caller buffers only replace pointers
  L.ids = cv.take<int32_t>(R);
  L.w = cv.take<float>(R);
  L.counts = cv.take<int32_t>(E);
  L.offsets = cv.take<int32_t>(E + 1);
  L.perm = cv.take<int32_t>(R);
  L.inv_perm = cv.take<int32_t>(R);
  L.y_rows = cv.take<float>(R * H);
  L.x_perm = needs_x_perm(mode, T) ? cv.take<__nv_bfloat16>(R * H) : nullptr;
  L.logits = R <= 32 ? cv.take<float>((size_t)T * E) : nullptr;
  L.bind_ws = cv.take<char>(bind_ws_bytes(T, k, E));
  if (b) {
    if (b->topk_ids) L.ids = b->topk_ids;
    if (b->topk_w) L.w = b->topk_w;
    if (b->counts) L.counts = b->counts;
    if (b->offsets) L.offsets = b->offsets;
    if (b->perm) L.perm = b->perm;
    if (b->inv_perm) L.inv_perm = b->inv_perm;
    if (b->y_rows) L.y_rows = b->y_rows;
  }
  const size_t scratch = std::max({route_ws_bytes(T, H, E), dispatch_ws_bytes(T, k, E),
                                   ffn_ws_bytes(T, k, E, H, I, mode)});
  L.scratch = cv.take<char>(scratch);
  L.bytes = cv.off;
  return L;
}

// k in [1, min(E, kMaxK)], T * k representable with room for the row offsets
bool layer_shape_ok(const moe_layer* layer, int T) {
  return layer->k >= 1 && layer->k <= layer->E && layer->k <= kMaxK && T >= 0 &&
         (long long)T * layer->k <= INT_MAX / 2;
}

}  // namespace

// Argument checks of moe_expert_ffn_grouped that precede the workspace
// check, in the order the header lists its errors (shared with the
// allocation-free variant, which checks its built-in scratch after them).
int ffn_check_args(const moe_cache* cache, int layer, const int32_t* counts, const int32_t* offsets,
                   const int32_t* perm, const void* x, const void* x_perm_opt, int T, int k, int ffn_mode,
                   const float* y_rows) {
  int st = check_cache(cache);
  if (st != MOE_OK) return st;
  if (layer < 0 || layer >= cache->n_layers || T < 0 || k < 1 || k > cache->E) return MOE_ERR_INVALID_ARG;
  if (ffn_mode != MOE_FFN_AUTO && ffn_mode != MOE_FFN_GEMV && ffn_mode != MOE_FFN_GEMM) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!counts || !offsets || !perm || !x || !y_rows) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y_rows) || (x_perm_opt && !aligned16(x_perm_opt))) return MOE_ERR_UNSUPPORTED;
  if (ffn_mode == MOE_FFN_GEMM && !x_perm_opt) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return kVersion; }

unsigned long long moe_kernel_launch_count(void) { return launch_counter().load(std::memory_order_relaxed); }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or API error";
    default: return "unknown status";
  }
}

size_t moe_route_topk_workspace_size(int T, int H, int E) {
  if (T < 0 || H < 1 || E < 1) return 0;
  return route_ws_bytes(T, H, E);
}

int moe_route_topk(const void* x, int T, int H, const float* w_router, const float* bias, int E, int k,
                   int32_t* topk_ids, float* topk_w, float* logits_opt, void* ws, size_t ws_bytes,
                   uint32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || H < 8 || E < 1 || k < 1 || k > E || k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (E > kMaxRouteE || (H % 8) || !aligned16(x) || !aligned16(w_router)) return MOE_ERR_UNSUPPORTED;
  const size_t need = route_ws_bytes(T, H, E);
  if (need && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  if (need && !ws_aligned(ws)) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_route_topk(reinterpret_cast<const __nv_bfloat16*>(x), T, H, w_router, bias, E, k,
                                       topk_ids, topk_w, logits_opt, ws, dev_status,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_dispatch_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return dispatch_ws_bytes(T, k, E);
}

int moe_dispatch(const int32_t* topk_ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
                 int32_t* perm, int32_t* inv_perm, const void* x_opt, int H, void* x_perm_opt, void* ws,
                 size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || k < 1 || E < 1 || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!topk_ids || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  if (x_opt && x_perm_opt && (H < 8 || (H % 8) || !aligned16(x_opt) || !aligned16(x_perm_opt)))
    return MOE_ERR_UNSUPPORTED;
  const size_t need = dispatch_ws_bytes(T, k, E);
  if (need && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  if (need && !ws_aligned(ws)) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_dispatch(topk_ids, T * k, k, E, counts, offsets, perm, inv_perm,
                                     reinterpret_cast<const __nv_bfloat16*>(x_opt), H,
                                     reinterpret_cast<__nv_bfloat16*>(x_perm_opt), ws, dev_status,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_cache_bind_workspace_size(const moe_cache* cache, int T, int k) {
  if (!cache || T < 0 || k < 1) return 0;
  return bind_ws_bytes(T, k, cache->E);
}

int moe_cache_bind_slots(const moe_cache* cache, int layer, const int32_t* topk_ids, int T, int k,
                         uint32_t phi_q16, int min_fill, int fill_policy, uint64_t seed,
                         moe_bind_stats* stats_dev, int32_t* fills_opt, void* ws, size_t ws_bytes,
                         uint32_t* dev_status, moe_stream_t stream) {
  int st = check_bind_args(cache, layer, T, k, phi_q16, fill_policy);
  if (st != MOE_OK) return st;
  if (T > 0 && !topk_ids) return MOE_ERR_INVALID_ARG;
  const size_t need = bind_ws_bytes(T, k, cache->E);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (!ws_aligned(ws)) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_bind(*cache, layer, topk_ids, T * k, phi_q16, min_fill, fill_policy, seed,
                                 stats_dev, fills_opt, ws, dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_expert_ffn_workspace_size(int T, int k, int E, int H, int I, int ffn_mode) {
  if (T < 0 || k < 1 || E < 1 || H < 8 || I < 8) return 0;
  return ffn_ws_bytes(T, k, E, H, I, ffn_mode);
}

int moe_expert_ffn_grouped(const moe_cache* cache, int layer, const int32_t* counts, const int32_t* offsets,
                           const int32_t* perm, const void* x, const void* x_perm_opt, int T, int k,
                           const uint8_t* expert_mask_opt, int ffn_mode, float* y_rows, void* ws,
                           size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream) {
  const int st = ffn_check_args(cache, layer, counts, offsets, perm, x, x_perm_opt, T, k, ffn_mode, y_rows);
  if (st != MOE_OK || T == 0) return st;
  const size_t need = ffn_ws_bytes(T, k, cache->E, cache->H, cache->I, ffn_mode);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (!ws_aligned(ws)) return MOE_ERR_UNSUPPORTED;
  cudaError_t err = launch_ffn(*cache, layer, counts, offsets, perm, reinterpret_cast<const __nv_bfloat16*>(x),
                               reinterpret_cast<const __nv_bfloat16*>(x_perm_opt), T, k, expert_mask_opt,
                               ffn_mode, y_rows, ws, dev_status, reinterpret_cast<cudaStream_t>(stream));
  if (err == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return cuda_status(err);
}

int moe_combine(const float* y_rows, const float* topk_w, int T, int k, int H, void* out, float* out_f32_opt,
                uint32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > kMaxK || H < 8) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y_rows || !topk_w || (!out && !out_f32_opt)) return MOE_ERR_INVALID_ARG;
  if ((H % 8) || !aligned16(y_rows) || (out && !aligned16(out)) || (out_f32_opt && !aligned16(out_f32_opt)))
    return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_combine(y_rows, topk_w, T, k, H, reinterpret_cast<__nv_bfloat16*>(out), out_f32_opt,
                                    dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_layer_workspace_size(const moe_layer* layer, const moe_cache* cache, int T, int ffn_mode) {
  if (!layer || !cache || !layer_shape_ok(layer, T)) return 0;
  return layer_ws(nullptr, nullptr, T, layer->k, layer->E, layer->H, layer->I, ffn_mode).bytes;
}

int moe_layer_forward(const moe_layer* layer, const moe_cache* cache, const void* x, int T, void* out,
                      uint32_t phi_q16, int min_fill, int fill_policy, uint64_t seed, int ffn_mode,
                      const moe_layer_buffers* bufs_opt, void* ws, size_t ws_bytes, uint32_t* dev_status,
                      moe_bind_stats* stats_dev, moe_stream_t stream) {
  if (!layer || !cache) return MOE_ERR_INVALID_ARG;
  int st = check_cache(cache);
  if (st != MOE_OK) return st;
  if (layer->E != cache->E || layer->H != cache->H || layer->I != cache->I) return MOE_ERR_INVALID_ARG;
  if (T < 0 || layer->k < 1 || layer->k > layer->E || layer->k > kMaxK) return MOE_ERR_INVALID_ARG;
  if ((long long)T * layer->k > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
  const int k = layer->k, E = layer->E, H = layer->H, I = layer->I;
  if (T == 0) return MOE_OK;
  if (!x || !out) return MOE_ERR_INVALID_ARG;
  const LayerWs need = layer_ws(nullptr, nullptr, T, k, E, H, I, ffn_mode);
  if (!ws || ws_bytes < need.bytes) return MOE_ERR_WORKSPACE;
  if (!ws_aligned(ws)) return MOE_ERR_UNSUPPORTED;
  const LayerWs L = layer_ws(ws, bufs_opt, T, k, E, H, I, ffn_mode);
  const size_t scratch_bytes = ws_bytes - (size_t)(reinterpret_cast<char*>(L.scratch) - reinterpret_cast<char*>(ws));
  // A host-resident staging pool is read with plain loads only (the fill copy of the bind step
  // and the plain GEMV pass of the FFN), so its calls take the per-step launches.
  const bool host_stage = cache->staging.w_gate != nullptr && cache->staging.host != 0;
  const bool fuse_fill = ffn_mode != MOE_FFN_GEMM && !L.x_perm && gemv_fused_ok(H, I) && !host_stage;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fuse_fill && L.logits && decode_layer_ok(T, k, E, H, I, cache->cache.n_slots) && layer->w_router &&
      aligned16(x) && aligned16(layer->w_router)) {
    // Decode: the whole layer in one cooperative launch (router, selection,
    // residency decision, fused FFN with fills, combine, state commit).
    st = check_bind_args(cache, layer->layer, T, k, phi_q16, fill_policy);
    if (st != MOE_OK) return st;
    unsigned int* grid_count = reinterpret_cast<unsigned int*>(
        reinterpret_cast<char*>(L.scratch) + align_up((size_t)T * k * I * sizeof(__nv_bfloat16), 256));
    cudaError_t err = launch_decode_layer(*cache, layer->layer, reinterpret_cast<const __nv_bfloat16*>(x), T, k,
                                          layer->w_router, layer->bias, phi_q16, min_fill, fill_policy, seed, stats_dev,
                                          L.logits, L.ids, L.w, L.counts, L.offsets, L.perm, L.inv_perm, L.y_rows,
                                          reinterpret_cast<__nv_bfloat16*>(L.scratch), grid_count,
                                          reinterpret_cast<__nv_bfloat16*>(out), dev_status, s);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (fuse_fill && T <= 32 && E <= kMaxRouteE && front_small_ok(T, k, E, cache->cache.n_slots) &&
      k <= kMaxK && layer->w_router && aligned16(x) && aligned16(layer->w_router)) {
    // Decode: router logits over all SMs, then one warp selects, binds and
    // dispatches, then one fused FFN launch (gate/up, down, fills, combine).
    st = check_bind_args(cache, layer->layer, T, k, phi_q16, fill_policy);
    if (st != MOE_OK) return st;
    float* logits = reinterpret_cast<float*>(L.scratch);
    if (launch_route_logits(reinterpret_cast<const __nv_bfloat16*>(x), T, H, layer->w_router, layer->bias, E, logits,
                            s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (launch_front_small(logits, T, k, *cache, layer->layer, phi_q16, min_fill, fill_policy, seed, stats_dev, L.ids,
                           L.w, L.counts, L.offsets, L.perm, L.inv_perm, L.bind_ws, dev_status, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    const int32_t* n_fill = reinterpret_cast<const int32_t*>(L.bind_ws);
    cudaError_t err = launch_ffn(*cache, layer->layer, L.counts, L.offsets, L.perm,
                                 reinterpret_cast<const __nv_bfloat16*>(x), nullptr, T, k, nullptr, ffn_mode, L.y_rows,
                                 L.scratch, dev_status, s, n_fill + 4, n_fill, L.w,
                                 reinterpret_cast<__nv_bfloat16*>(out));
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  st = moe_route_topk(x, T, H, layer->w_router, layer->bias, E, k, L.ids, L.w, nullptr, L.scratch, scratch_bytes,
                      dev_status, stream);
  if (st != MOE_OK) return st;
  // Decode-sized calls run every group on the fused GEMV kernel, which copies
  // each admitted expert into its cache slot while it streams it (one read of
  // the staging copy instead of two) and ends with the combine; other calls
  // copy in the bind step and combine in their own launch.  Calls with few
  // enough routed rows get the dispatch in the bind launch.
  const int R = T * k;
  const bool fuse_dispatch = bind_dispatch_fusable(R, E);
  st = check_bind_args(cache, layer->layer, T, k, phi_q16, fill_policy);
  if (st != MOE_OK) return st;
  if (launch_bind(*cache, layer->layer, L.ids, R, phi_q16, min_fill, fill_policy, seed, stats_dev, nullptr,
                  L.bind_ws, dev_status, s, !fuse_fill, fuse_dispatch ? L.counts : nullptr, L.offsets, L.perm,
                  L.inv_perm) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!fuse_dispatch) {
    st = moe_dispatch(L.ids, T, k, E, L.counts, L.offsets, L.perm, L.inv_perm, L.x_perm ? x : nullptr, H, L.x_perm,
                      L.scratch, scratch_bytes, dev_status, stream);
    if (st != MOE_OK) return st;
  } else if (L.x_perm) {
    if (launch_gather(reinterpret_cast<const __nv_bfloat16*>(x), H, k, L.perm, L.offsets, E, R, L.x_perm, s) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (fuse_fill) {
    const int32_t* n_fill = reinterpret_cast<const int32_t*>(L.bind_ws);
    cudaError_t err = launch_ffn(*cache, layer->layer, L.counts, L.offsets, L.perm,
                                 reinterpret_cast<const __nv_bfloat16*>(x), nullptr, T, k, nullptr, ffn_mode, L.y_rows,
                                 L.scratch, dev_status, s, n_fill + 4, n_fill, L.w,
                                 reinterpret_cast<__nv_bfloat16*>(out));
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (L.x_perm && gemm_shape_ok(H, I) && !(bufs_opt && bufs_opt->y_rows) && !host_stage) {
    // Every group runs on the GEMM and nobody reads the expert rows but the
    // combine: keep them in bf16 (half the bytes written and read back).
    __nv_bfloat16* y16 = reinterpret_cast<__nv_bfloat16*>(L.y_rows);
    cudaError_t err = launch_ffn(*cache, layer->layer, L.counts, L.offsets, L.perm,
                                 reinterpret_cast<const __nv_bfloat16*>(x), L.x_perm, T, k, nullptr, ffn_mode, nullptr,
                                 L.scratch, dev_status, s, nullptr, nullptr, nullptr, nullptr, y16);
    if (err != cudaSuccess) return err == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : MOE_ERR_CUDA;
    return cuda_status(launch_combine(y16, L.w, T, k, H, reinterpret_cast<__nv_bfloat16*>(out), nullptr, dev_status, s));
  }
  st = moe_expert_ffn_grouped(cache, layer->layer, L.counts, L.offsets, L.perm, x, L.x_perm, T, k, nullptr, ffn_mode,
                              L.y_rows, L.scratch, scratch_bytes, dev_status, stream);
  if (st != MOE_OK) return st;
  return moe_combine(L.y_rows, L.w, T, k, H, out, nullptr, dev_status, stream);
}

}  // extern "C"
