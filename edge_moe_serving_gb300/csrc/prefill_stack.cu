// Full-layer double-buffered prefill (FreeToken paper, section 3.1 and
// Figure 2 (1), prefill codesign: while layer l computes, the experts of
// layer l+1 stream from the host-resident source pool into the GPU; section
// 5.3: it is turned off when the pool cannot spare two layers; the write-up's
// section "Prefill: full-layer double buffering").
//
// Host-side orchestration over two streams, no kernel of its own: the copy
// engine moves a layer's three banks (one cudaMemcpyAsync each: a layer's
// experts are consecutive slots l*E .. l*E+E-1 of the source pool) into one
// of two HBM layer buffers on copy_stream, and moe_layer_forward runs the
// layer on stream from the buffer its copy filled.  Events order the two:
// a layer waits for its copy, and a copy into a buffer waits until the layer
// that last read the buffer has finished.  With one buffer (or overlap off)
// every copy waits for the previous layer: on-demand loading.
#include <vector>

#include "moe_common.cuh"

namespace {

struct EventSet {
  std::vector<cudaEvent_t> ev;
  ~EventSet() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);   // released once the recorded work completes
  }
  cudaError_t make(size_t n) {
    ev.assign(n, nullptr);
    for (size_t i = 0; i < n; ++i) {
      const cudaError_t err = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
      if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
  }
};

bool pool_set(const moe_pool& p) { return p.w_gate && p.w_up && p.w_down; }

// Copies layer l's experts from the source pool into buf (E slots).
cudaError_t copy_layer(const moe_pool& src, const moe_pool& buf, int l, int E, size_t bank_bytes, cudaStream_t s) {
  const size_t off = (size_t)l * E * bank_bytes, len = (size_t)E * bank_bytes;
  const void* from[3] = {src.w_gate, src.w_up, src.w_down};
  void* to[3] = {buf.w_gate, buf.w_up, buf.w_down};
  for (int b = 0; b < 3; ++b) {
    const cudaError_t err = cudaMemcpyAsync(to[b], static_cast<const char*>(from[b]) + off, len,
                                            cudaMemcpyDefault, s);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace

extern "C" int moe_prefill_double_buffered(const moe_layer* layers, int n_layers, const moe_pool* source,
                                           const moe_pool* layer_buf, const moe_cache* state, const void* const* x,
                                           int T, void* const* out, int ffn_mode, int overlap, void* ws,
                                           size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream,
                                           moe_stream_t copy_stream) {
  if (!layers || n_layers < 1 || !source || !layer_buf || !state || T < 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !out)) return MOE_ERR_INVALID_ARG;
  const int E = layers[0].E, H = layers[0].H, I = layers[0].I;
  for (int l = 0; l < n_layers; ++l)
    if (layers[l].E != E || layers[l].H != H || layers[l].I != I || layers[l].layer != l) return MOE_ERR_INVALID_ARG;
  if (E < 1 || H < 8 || I < 8) return MOE_ERR_INVALID_ARG;
  if (!pool_set(*source) || (long long)source->n_slots < (long long)n_layers * E) return MOE_ERR_INVALID_ARG;
  if (!pool_set(layer_buf[0]) || layer_buf[0].n_slots < E) return MOE_ERR_INVALID_ARG;
  // a second buffer of at least E slots allows the overlap; otherwise on-demand loading
  const bool two = overlap != 0 && pool_set(layer_buf[1]) && layer_buf[1].n_slots >= E;
  if (!state->slot_table || !state->owner || !state->stamp || !state->clock || state->n_layers != n_layers ||
      state->E != E || state->H != H || state->I != I)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(copy_stream);
  if (!cs || cs == s) return MOE_ERR_INVALID_ARG;
  const size_t bank_bytes = (size_t)H * I * 2;   // one expert's bank, bf16
  const int nb = two ? 2 : 1;

  // events: copied[l] (layer l is in its buffer), done[l] (layer l has read its buffer), start (fork)
  EventSet evs;
  if (evs.make(2 * (size_t)n_layers + 1) != cudaSuccess) return MOE_ERR_CUDA;
  cudaEvent_t* copied = evs.ev.data();
  cudaEvent_t* done = copied + n_layers;
  cudaEvent_t start = evs.ev[2 * n_layers];
  auto cuda = [](cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; };

  int st = cuda(cudaEventRecord(start, s));   // the copies follow whatever came before the call on `stream`
  if (st != MOE_OK) return st;
  st = cuda(cudaStreamWaitEvent(cs, start, 0));
  if (st != MOE_OK) return st;
  auto issue_copy = [&](int l) -> int {
    // buffer l % nb was last read by layer l - nb
    if (l - nb >= 0) {
      const int r = cuda(cudaStreamWaitEvent(cs, done[l - nb], 0));
      if (r != MOE_OK) return r;
    }
    int r = cuda(copy_layer(*source, layer_buf[l % nb], l, E, bank_bytes, cs));
    if (r != MOE_OK) return r;
    return cuda(cudaEventRecord(copied[l], cs));
  };
  st = issue_copy(0);
  if (st != MOE_OK) return st;
  for (int l = 0; l < n_layers; ++l) {
    // with two buffers the next layer's copy is queued before this layer computes
    if (two && l + 1 < n_layers) {
      st = issue_copy(l + 1);
      if (st != MOE_OK) return st;
    }
    st = cuda(cudaStreamWaitEvent(s, copied[l], 0));
    if (st != MOE_OK) return st;
    moe_cache c = *state;
    c.cache = layer_buf[l % nb];
    c.cache.n_slots = E;
    c.staging = moe_pool{nullptr, nullptr, nullptr, 0};
    st = moe_layer_forward(&layers[l], &c, x[l], T, out[l], 0u, 0, MOE_FILL_LOWEST_ID, 0, ffn_mode, nullptr, ws,
                           ws_bytes, dev_status, nullptr, stream);
    if (st != MOE_OK) return st;
    st = cuda(cudaEventRecord(done[l], s));
    if (st != MOE_OK) return st;
    if (!two && l + 1 < n_layers) {
      st = issue_copy(l + 1);   // on-demand: after this layer has read the only buffer
      if (st != MOE_OK) return st;
    }
  }
  // join: `stream` already waited for every copy before the layer that used it
  return MOE_OK;
}
