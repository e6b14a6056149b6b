// Pieces shared by the MXFP4 expert-FFN kernels (FreeToken paper, section 5.1
// "Models": the routed experts of DeepSeek-V4-Flash are natively MXFP4;
// section 4.1: the expert kernels dequantise in-kernel).  Encoding of the OCP
// Microscaling Formats v1.0: FP4 E2M1 elements, one E8M0 scale per 32
// consecutive inputs of a weight row, input 2c in the low nibble of code
// byte c.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kMxBlock = 32;   // inputs per E8M0 scale = one 16-byte code vector

struct MxParams {
  moe_pool_mxfp4 a;   // cache pool
  moe_pool_mxfp4 b;   // staging pool (n_slots 0 when absent)
  const int32_t* slot_table;
  int layer, E, H, I, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const __nv_bfloat16* x;
  __nv_bfloat16* h;   // [R, I] by dispatch position
  float* y;           // [R, H] token-major
  uint32_t* status;
  unsigned int* inst_done;   // ring kernel: per-instance gate/up completion counters (zero at launch)
};

struct MxRows {
  const uint8_t* q0;
  const uint8_t* s0;
  const uint8_t* q1;
  const uint8_t* s1;
};

namespace {

// E8M0 scale 2^(s - 127) as fp32 bits: s = 0 is the subnormal 2^-127, s = 255 NaN.
__device__ inline float e8m0(uint32_t s) {
  return __uint_as_float(s == 0u ? 0x00400000u : (s == 255u ? 0x7FC00000u : s << 23));
}

// Slot-table entry -> the slot's code and scale rows of one projection
// (gate and up, or down twice).
template <bool GATEUP>
__device__ inline bool mx_resolve(const MxParams& p, int32_t entry, MxRows* out, uint32_t* status) {
  if (entry < 0) {
    set_status(status, MOE_DEV_ERR_UNBOUND);
    return false;
  }
  const moe_pool_mxfp4& pool = (entry & MOE_STAGING_TAG) ? p.b : p.a;
  const int32_t slot = entry & MOE_SLOT_MASK;
  if ((entry & ~(MOE_STAGING_TAG | MOE_SLOT_MASK)) != 0 || slot >= pool.n_slots) {
    set_status(status, MOE_DEV_ERR_BAD_SLOT);
    return false;
  }
  const size_t rows = GATEUP ? (size_t)p.I : (size_t)p.H;   // output rows per slot
  const size_t K = GATEUP ? (size_t)p.H : (size_t)p.I;       // inputs per row
  const size_t qper = rows * (K / 2), sper = rows * (K / kMxBlock);
  if (GATEUP) {
    out->q0 = reinterpret_cast<const uint8_t*>(pool.gate_q) + (size_t)slot * qper;
    out->s0 = reinterpret_cast<const uint8_t*>(pool.gate_s) + (size_t)slot * sper;
    out->q1 = reinterpret_cast<const uint8_t*>(pool.up_q) + (size_t)slot * qper;
    out->s1 = reinterpret_cast<const uint8_t*>(pool.up_s) + (size_t)slot * sper;
  } else {
    out->q0 = reinterpret_cast<const uint8_t*>(pool.down_q) + (size_t)slot * qper;
    out->s0 = reinterpret_cast<const uint8_t*>(pool.down_s) + (size_t)slot * sper;
    out->q1 = out->q0;
    out->s1 = out->s0;
  }
  return true;
}

}  // namespace

// One-token calls on the weight-streaming ring kernel (ffn_mxfp4_ring.cu):
// whether the shape and banks qualify, and the launch (counters cleared on
// the stream first).  inst_done: R + 4 words of workspace.
bool mx_ring_ok(const MxParams& p, int T);
cudaError_t launch_mx_ring(const MxParams& p, int T, cudaStream_t s);

}  // namespace moe
