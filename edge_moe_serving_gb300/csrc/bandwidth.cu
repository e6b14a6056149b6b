// Bandwidth profile for the q* split (FreeToken paper, section 3.2, Eq. 3-4:
// q* = m * B_P / B_H, and Table 1, which measures B_P and B_H per machine;
// the write-up "FreeToken: bandwidth-adaptive edge MoE serving", sections
// "The split, and what it is actually optimising" (measure both sides while
// they contend) and "When to use it (and when not)" (the hybrid gate
// B_H > 2 B_P)).
//
// On GB300 the source-of-truth expert pool would sit in Grace memory behind
// NVLink-C2C: B_P is the copy engine moving expert bytes from pinned host
// memory into HBM (the fill path), B_H the SMs reading the same host memory
// in place (the in-place path, which runs on the GPU here).
#include <algorithm>
#include <cmath>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kReadThreads = 512;
constexpr int kReadCtasPerSm = 4;
constexpr double kHybridGate = 2.0;   // the split pays only when B_H > 2 B_P

// [0]: XOR checksum of the untimed read pass; [1]: sink of the timed passes.
__device__ uint32_t g_bw_words[2];

__device__ inline uint32_t xor4(const uint4& v) { return v.x ^ v.y ^ v.z ^ v.w; }

// Reads n16 16-byte words in place (grid-stride, four loads in flight per
// thread) and XORs every 32-bit word into *sink, one atomic per warp.  Every
// thread reaches the warp reduction (the loops are per thread).
__global__ void __launch_bounds__(kReadThreads) host_read_kernel(const uint4* __restrict__ src, size_t n16,
                                                                 uint32_t* sink) {
  pdl_wait();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(src + i);
    const uint4 b = __ldcs(src + i + stride);
    const uint4 c = __ldcs(src + i + 2 * stride);
    const uint4 d = __ldcs(src + i + 3 * stride);
    acc ^= xor4(a) ^ xor4(b) ^ xor4(c) ^ xor4(d);
  }
  for (; i < n16; i += stride) acc ^= xor4(__ldcs(src + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

double rate_gbs(size_t bytes, long long reps, float ms) {
  return ms > 0.0f ? (double)bytes * (double)reps / ((double)ms * 1e-3) / 1e9 : 0.0;
}

bool rate_ok(double r) { return std::isfinite(r) && r >= 0.0; }

// Events of one measurement; destroyed with the object.
struct Events {
  cudaEvent_t e[4] = {nullptr, nullptr, nullptr, nullptr};
  bool ok = true;
  Events() {
    for (auto& x : e) ok = ok && cudaEventCreate(&x) == cudaSuccess;
  }
  ~Events() {
    for (auto& x : e)
      if (x) cudaEventDestroy(x);
  }
};

float elapsed_ms(cudaEvent_t a, cudaEvent_t b) {
  float ms = 0.0f;
  if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) return -1.0f;
  return ms;
}

}  // namespace
}  // namespace moe

extern "C" uint32_t moe_phi_to_q16(double phi) {
  if (!(phi > 0.0)) return 0u;   // NaN and phi <= 0
  const double v = phi * 65536.0;
  if (v >= 65536.0) return 65536u;
  return (uint32_t)std::nearbyint(v);   // default rounding mode: to nearest, ties to even
}

extern "C" int moe_bw_derive(moe_bw_profile* prof) {
  if (!prof) return MOE_ERR_INVALID_ARG;
  const double bp = prof->b_p_gbs, bh = prof->b_h_gbs;
  const double bpc = prof->b_p_contended_gbs, bhc = prof->b_h_contended_gbs;
  if (!moe::rate_ok(bp) || !moe::rate_ok(bh) || !moe::rate_ok(bpc) || !moe::rate_ok(bhc)) return MOE_ERR_INVALID_ARG;
  // Eq. 4: phi = B_P / B_H; with no in-place path every miss fills (phi = 1)
  prof->phi = bh > 0.0 ? bp / bh : (bp > 0.0 ? 1.0 : 0.0);
  prof->phi_contended = (bpc + bhc) > 0.0 ? bpc / (bpc + bhc) : 0.0;
  prof->phi_q16 = moe_phi_to_q16(prof->phi);
  prof->phi_contended_q16 = moe_phi_to_q16(prof->phi_contended);
  prof->hybrid_ok = bh > moe::kHybridGate * bp ? 1 : 0;
  return MOE_OK;
}

extern "C" int moe_bench_bandwidth(const void* host_src, void* dev_dst, size_t bytes, int iters, moe_bw_profile* out,
                                   moe_stream_t copy_stream, moe_stream_t read_stream) {
  using namespace moe;
  // two distinct created streams: the legacy default stream (NULL) would serialise the contended pair
  if (!host_src || !dev_dst || !out || iters < 1 || bytes == 0 || (bytes & 15) != 0 || copy_stream == read_stream ||
      !copy_stream || !read_stream)
    return MOE_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(host_src) | reinterpret_cast<uintptr_t>(dev_dst)) & 15) != 0)
    return MOE_ERR_INVALID_ARG;
  void* dsrc = nullptr;
  if (cudaHostGetDevicePointer(&dsrc, const_cast<void*>(host_src), 0) != cudaSuccess || !dsrc ||
      (reinterpret_cast<uintptr_t>(dsrc) & 15) != 0) {
    cudaGetLastError();   // clear the lookup's error: the buffer is not device-addressable pinned memory
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s1 = reinterpret_cast<cudaStream_t>(copy_stream), s2 = reinterpret_cast<cudaStream_t>(read_stream);
  uint32_t* words = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&words), g_bw_words) != cudaSuccess) return MOE_ERR_CUDA;
  Events ev;
  if (!ev.ok) return MOE_ERR_CUDA;
  const uint4* src16 = reinterpret_cast<const uint4*>(dsrc);
  const size_t n16 = bytes / 16;
  const dim3 grid(num_sms() * kReadCtasPerSm);
  auto copy = [&]() { return cudaMemcpyAsync(dev_dst, host_src, bytes, cudaMemcpyHostToDevice, s1); };
  auto read = [&](uint32_t* sink) { return launch_k(host_read_kernel, grid, dim3(kReadThreads), 0, s2, src16, n16, sink); };
  auto fail = [&]() { cudaStreamSynchronize(s1); cudaStreamSynchronize(s2); return MOE_ERR_CUDA; };
  // untimed pass: one copy, one read that leaves the checksum
  if (cudaMemsetAsync(words, 0, 2 * sizeof(uint32_t), s2) != cudaSuccess || copy() != cudaSuccess ||
      read(words) != cudaSuccess)
    return fail();
  if (cudaStreamSynchronize(s1) != cudaSuccess || cudaStreamSynchronize(s2) != cudaSuccess) return MOE_ERR_CUDA;
  moe_bw_profile p = {};
  // B_P alone
  if (cudaEventRecord(ev.e[0], s1) != cudaSuccess) return fail();
  for (int r = 0; r < iters; ++r)
    if (copy() != cudaSuccess) return fail();
  if (cudaEventRecord(ev.e[1], s1) != cudaSuccess || cudaEventSynchronize(ev.e[1]) != cudaSuccess) return fail();
  p.b_p_gbs = rate_gbs(bytes, iters, elapsed_ms(ev.e[0], ev.e[1]));
  // B_H alone
  if (cudaEventRecord(ev.e[0], s2) != cudaSuccess) return fail();
  for (int r = 0; r < iters; ++r)
    if (read(words + 1) != cudaSuccess) return fail();
  if (cudaEventRecord(ev.e[1], s2) != cudaSuccess || cudaEventSynchronize(ev.e[1]) != cudaSuccess) return fail();
  p.b_h_gbs = rate_gbs(bytes, iters, elapsed_ms(ev.e[0], ev.e[1]));
  // contended: both from one start event, the read count scaled so that the
  // two streams run for about the same time
  long long iters_r = iters;
  if (p.b_p_gbs > 0.0) iters_r = std::max(1LL, std::llround((double)iters * p.b_h_gbs / p.b_p_gbs));
  iters_r = std::min(iters_r, 64LL * iters);
  if (cudaEventRecord(ev.e[0], s1) != cudaSuccess || cudaStreamWaitEvent(s2, ev.e[0], 0) != cudaSuccess) return fail();
  for (int r = 0; r < iters; ++r)
    if (copy() != cudaSuccess) return fail();
  if (cudaEventRecord(ev.e[1], s1) != cudaSuccess) return fail();
  for (long long r = 0; r < iters_r; ++r)
    if (read(words + 1) != cudaSuccess) return fail();
  if (cudaEventRecord(ev.e[2], s2) != cudaSuccess) return fail();
  if (cudaEventSynchronize(ev.e[1]) != cudaSuccess || cudaEventSynchronize(ev.e[2]) != cudaSuccess) return fail();
  p.b_p_contended_gbs = rate_gbs(bytes, iters, elapsed_ms(ev.e[0], ev.e[1]));
  p.b_h_contended_gbs = rate_gbs(bytes, iters_r, elapsed_ms(ev.e[0], ev.e[2]));
  if (cudaMemcpy(&p.read_checksum, words, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  const int st = moe_bw_derive(&p);
  if (st != MOE_OK) return st;
  *out = p;
  return MOE_OK;
}
