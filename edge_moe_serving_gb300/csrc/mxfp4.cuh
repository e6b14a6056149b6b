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
  __nv_bfloat16* x_perm;   // [R, H] token rows in dispatch order (the tensor-core GEMM's operand)
  float* y;           // [R, H] token-major
  uint32_t* status;
  unsigned int* inst_done;   // ring kernel: per-instance gate/up completion counters (zero at launch)
  // NVFP4 banks only: fp32 tensor scale of every (slot, bank) of each pool, [n_slots][3] (gate, up,
  // down); null for MXFP4
  const float* ts_a;
  const float* ts_b;
};

struct MxRows {
  const uint8_t* q0;
  const uint8_t* s0;
  const uint8_t* q1;
  const uint8_t* s1;
  float t0, t1;       // NVFP4 tensor scales of the two banks (1 for MXFP4)
};

namespace {

// E8M0 scale 2^(s - 127) as fp32 bits: s = 0 is the subnormal 2^-127, s = 255 NaN.
__device__ inline float e8m0(uint32_t s) {
  return __uint_as_float(s == 0u ? 0x00400000u : (s == 255u ? 0x7FC00000u : s << 23));
}

// Slot-table entry -> the slot's code and scale rows of one projection
// (gate and up, or down twice).  SB: inputs per scale byte (32 for MXFP4's
// E8M0 scales, 16 for NVFP4's E4M3 scales).
template <bool GATEUP, int SB = kMxBlock>
__device__ inline bool mx_resolve(const MxParams& p, int32_t entry, MxRows* out, uint32_t* status) {
  if (entry < 0) {
    set_status(status, MOE_DEV_ERR_UNBOUND);
    return false;
  }
  const bool staged = (entry & MOE_STAGING_TAG) != 0;
  const moe_pool_mxfp4& pool = staged ? p.b : p.a;
  const int32_t slot = entry & MOE_SLOT_MASK;
  if ((entry & ~(MOE_STAGING_TAG | MOE_SLOT_MASK)) != 0 || slot >= pool.n_slots) {
    set_status(status, MOE_DEV_ERR_BAD_SLOT);
    return false;
  }
  const size_t rows = GATEUP ? (size_t)p.I : (size_t)p.H;   // output rows per slot
  const size_t K = GATEUP ? (size_t)p.H : (size_t)p.I;       // inputs per row
  const size_t qper = rows * (K / 2), sper = rows * (K / SB);
  const float* ts = staged ? p.ts_b : p.ts_a;
  if (GATEUP) {
    out->q0 = reinterpret_cast<const uint8_t*>(pool.gate_q) + (size_t)slot * qper;
    out->s0 = reinterpret_cast<const uint8_t*>(pool.gate_s) + (size_t)slot * sper;
    out->q1 = reinterpret_cast<const uint8_t*>(pool.up_q) + (size_t)slot * qper;
    out->s1 = reinterpret_cast<const uint8_t*>(pool.up_s) + (size_t)slot * sper;
    out->t0 = ts ? ts[(size_t)slot * 3 + 0] : 1.0f;
    out->t1 = ts ? ts[(size_t)slot * 3 + 1] : 1.0f;
  } else {
    out->q0 = reinterpret_cast<const uint8_t*>(pool.down_q) + (size_t)slot * qper;
    out->s0 = reinterpret_cast<const uint8_t*>(pool.down_s) + (size_t)slot * sper;
    out->q1 = out->q0;
    out->s1 = out->s0;
    out->t0 = out->t1 = ts ? ts[(size_t)slot * 3 + 2] : 1.0f;
  }
  return true;
}

}  // namespace

// The weight-streaming ring kernel (ffn_mxfp4_ring.cu) over MXFP4 or NVFP4
// banks (nv): whether the shape and banks qualify (at most kFp4RingMaxRows
// routed rows, each its own instance), and the launch (the inst_done
// counters, one word per routed row, cleared on the stream first).
constexpr int kFp4RingMaxRows = 64;
bool fp4_ring_ok(const MxParams& p, int T, bool nv);
cudaError_t launch_fp4_ring(const MxParams& p, int T, bool nv, cudaStream_t s);

// The banks a cache fill of an FP4 expert copies, staging slot -> cache slot:
// six code and scale banks, plus the NVFP4 tensor scales (n = 7).
struct Fp4FillBanks {
  const uint8_t* src[7];
  uint8_t* dst[7];
  size_t slot_bytes[7];   // bytes of one slot of the bank
  int n;
  int src_slots, dst_slots;
};

// The whole layer for one token over FP4 banks in one cooperative launch
// (ffn_mxfp4_ring.cu): router rows, a grid barrier, the route and residency
// decision in every CTA (CTA 0 commits it), the ring kernel's gate/up and
// down phases, the cache fills, a grid barrier and the combine.  p: as for
// the ring kernel, with p.h and p.y the call's workspace and p.inst_done
// unused (grid_count + 4 is used instead).  Shapes: see fp4_decode_ok.
struct Fp4DecodeArgs {
  moe_cache c;              // residency arrays and the cache pool's slot count
  const float* w_router;    // [E, H]
  const float* bias;        // [E] or null
  uint32_t phi_q16;
  int min_fill, policy;
  unsigned long long seed;
  moe_bind_stats* stats;    // or null
  float* logits;            // [E]
  int32_t* topk_ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  __nv_bfloat16* out;       // [1, H]
  unsigned int* grid_count; // 4 + k words, cleared on the stream by the launch
  Fp4FillBanks fill;
};
bool fp4_decode_ok(const MxParams& p, int T, int n_slots);
cudaError_t launch_fp4_decode(const MxParams& p, bool nv, const Fp4DecodeArgs& a, cudaStream_t s);

// The tensor-core GEMM over FP4 banks (ffn_fp4_gemm.cu): whether the shape
// qualifies (I a multiple of 128, H of 256, every row's scales a multiple of
// 16 bytes), and the two launches (gate/up into p.h, down into p.y) over the
// token rows gathered in dispatch order (x_perm, bf16 [T*k, H]).
bool fp4_gemm_ok(const MxParams& p, bool nv);
cudaError_t launch_fp4_gemm(const MxParams& p, bool nv, const __nv_bfloat16* x_perm, int T, cudaStream_t s);

}  // namespace moe
