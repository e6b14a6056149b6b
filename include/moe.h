/*
 * moe.h — C ABI of libmoe: one routed Mixture-of-Experts layer's forward pass
 * on an NVIDIA GB300 (sm_103a), with an expert cache addressed through a
 * (layer, expert) -> slot table.
 *
 * Source of the method: "FreeToken: Efficient Edge-Native MoE Serving with
 * Bandwidth-Adaptive Execution" (arXiv 2608.16157), cited below as [P], and
 * the write-up "FreeToken: bandwidth-adaptive edge MoE serving", cited as [W].
 *
 * Conventions shared by every call
 * --------------------------------
 * Pointers.   Every tensor pointer is a DEVICE pointer unless stated, owned by
 *             the caller; the library never allocates, frees or keeps a
 *             pointer after the call returns.  Structs (moe_cache, moe_layer,
 *             moe_layer_buffers) are HOST structs holding device pointers;
 *             they are read during the call only.
 * Layout.     Row-major, densely packed.  x, out: bf16 [T, H].  Expert banks:
 *             W_gate, W_up bf16 [n_slots, I, H]; W_down bf16 [n_slots, H, I]
 *             (nn.Linear out x in); the leading dimension is the slot, as in
 *             [P] section 4.2 (banks share one expert -> slot mapping).  Router
 *             weights fp32 [E, H], bias fp32 [E].  ids / indices int32.
 *             Every device pointer must be 16-byte aligned; H and I must be
 *             multiples of 8.
 * Async.      Every call only enqueues work on `stream` (a cudaStream_t) and
 *             returns; no call synchronises with the host, so a sequence of
 *             calls may be captured into a CUDA graph.  The one exception is
 *             the profiling call moe_bench_bandwidth.
 * Errors.     The return value is a host status (MOE_OK or MOE_ERR_*), from
 *             argument checks before any launch or from the launch itself.
 *             Errors found on the device (bad expert id, unbound slot, a
 *             bounded wait that ran out) are OR-ed into *dev_status (device
 *             uint32, caller-zeroed) as MOE_DEV_ERR_* bits; the kernel skips
 *             the offending work and returns, it never traps.
 * Workspace.  Calls that need scratch take (ws, ws_bytes): a device buffer of
 *             at least the size the matching *_workspace_size() reports,
 *             256-byte aligned, with no content requirement.  A call that
 *             gets a smaller ws returns MOE_ERR_WORKSPACE, and one whose ws
 *             is not 256-byte aligned MOE_ERR_UNSUPPORTED, without launching.
 *             Calls sharing one ws must not overlap on the GPU.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

/* host status codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1  /* null pointer, negative size, k > E, layer out of range ... */
#define MOE_ERR_UNSUPPORTED 2  /* shape or alignment outside what the kernels handle */
#define MOE_ERR_WORKSPACE 3    /* ws_bytes below the reported workspace size */
#define MOE_ERR_CUDA 4         /* a CUDA launch or API call failed */

/* device status bits (OR-ed into *dev_status) */
#define MOE_DEV_ERR_BAD_ID 1u     /* a routed expert id outside [0, E) was skipped */
#define MOE_DEV_ERR_UNBOUND 2u    /* an expert's slot-table entry was -1; its rows were not written */
#define MOE_DEV_ERR_BAD_SLOT 4u   /* a slot-table entry pointed outside its pool; treated as unbound */
#define MOE_DEV_ERR_TIMEOUT 8u    /* a bounded wait in a pipelined kernel ran out; its tile was abandoned */

/* fill policy of moe_cache_bind_slots: which q misses form the fill set F */
#define MOE_FILL_LOWEST_ID 0  /* the q misses with the lowest expert ids */
#define MOE_FILL_RANDOM 1     /* a seeded uniformly random q-subset (SplitMix64 keys) */

/* expert-FFN kernel selection */
#define MOE_FFN_AUTO 0  /* calls of <= 2 tokens (or without gathered rows): the fused weight-streaming
                           GEMV; larger calls: the tensor-core grouped GEMM for every group */
#define MOE_FFN_GEMV 1  /* weight-streaming GEMV for every group */
#define MOE_FFN_GEMM 2  /* tcgen05 grouped GEMM for every non-empty group */

/* slot-table entry encoding: -1 unbound; s (0 <= s < cache.n_slots) = cache pool slot s;
 * MOE_STAGING_TAG | p = staging pool slot p, where p = layer * E + expert. */
#define MOE_STAGING_TAG (1 << 30)
#define MOE_SLOT_MASK ((1 << 30) - 1)

/* One pool of expert banks (bf16, see Layout above).  host = 1: the banks
 * live in host memory that the GPU reads in place (pinned memory of a Grace
 * host over NVLink-C2C: the source-of-truth pool of [P] section 3); the
 * kernels then read it only with plain loads (the fill copy, and a
 * weight-streaming GEMV for the experts computed in place), never with the
 * tensor-memory-accelerator copies of the ring and GEMM kernels.  Only the
 * staging pool may be host-resident. */
typedef struct moe_pool {
  void* w_gate;   /* [n_slots, I, H] */
  void* w_up;     /* [n_slots, I, H] */
  void* w_down;   /* [n_slots, H, I] */
  int32_t n_slots;
  int32_t host;   /* 0: device memory; 1: host memory read in place */
} moe_pool;

/* The expert cache of [P] section 3: one elastic slot pool shared by every
 * MoE layer (pool A, `cache`), plus the staging pool (pool B, `staging`) that
 * holds every (layer, expert) pair at slot layer*E + expert and stands in for
 * the host-resident source-of-truth pool of [P] section 3.  A staging pool with
 * fewer than n_layers*E slots is allowed only if no call ever needs it.
 * Residency state (device arrays, read and written by moe_cache_bind_slots):
 *   slot_table [n_layers*E] int32  entry per (layer, expert), encoding above
 *   owner      [cache.n_slots] int32  layer*E+expert held by a slot, or -1
 *   stamp      [cache.n_slots] uint32 clock value of the slot's last use (0 = never)
 *   clock      [1] uint32           one LRU clock for all layers, +1 per bind call */
typedef struct moe_cache {
  moe_pool cache;
  moe_pool staging;
  int32_t* slot_table;
  int32_t* owner;
  uint32_t* stamp;
  uint32_t* clock;
  int32_t n_layers;
  int32_t E;
  int32_t H;
  int32_t I;
} moe_cache;

/* Per-call counters written by moe_cache_bind_slots (device struct). */
typedef struct moe_bind_stats {
  int32_t n_unique;    /* distinct routed experts of the call */
  int32_t n_hit;       /* |H|: resident in the cache pool */
  int32_t n_miss;      /* m = |M| */
  int32_t q;           /* fetch count from the q* rule */
  int32_t n_fill;      /* fills performed (q minus overflow) */
  int32_t n_overflow;  /* fills that found no victim and stayed in C */
  int32_t n_staged;    /* |C|: misses served from the staging pool */
  uint32_t clock;      /* stamp of this call */
} moe_bind_stats;

/* Router and shape of one MoE layer. */
typedef struct moe_layer {
  const float* w_router;  /* fp32 [E, H] */
  const float* bias;      /* fp32 [E] added to the logits, or NULL */
  int32_t layer;          /* layer index into the slot table */
  int32_t E;
  int32_t k;
  int32_t H;
  int32_t I;
} moe_layer;

/* Optional caller-owned destinations for the intermediates of
 * moe_layer_forward; a NULL field is placed in the workspace instead. */
typedef struct moe_layer_buffers {
  int32_t* topk_ids;  /* [T, k] */
  float* topk_w;      /* [T, k] */
  int32_t* counts;    /* [E] */
  int32_t* offsets;   /* [E + 1] */
  int32_t* perm;      /* [T*k] */
  int32_t* inv_perm;  /* [T*k] */
  float* y_rows;      /* [T*k, H], row t*k+j = output of token t's j-th expert */
} moe_layer_buffers;

int moe_version(void);
const char* moe_status_string(int status);

/* Diagnostic of the failure path of the pipelined kernels (no counterpart in
 * the paper): one launch waits, with the same bounded wait the expert-FFN
 * kernels use, on a barrier that nothing completes; after the wait limit
 * (about one second) it ORs MOE_DEV_ERR_TIMEOUT into *dev_status and returns.
 * The context stays usable. */
int moe_check_bounded_wait(uint32_t* dev_status, moe_stream_t stream);

/* Number of kernels this library has launched, or captured into a CUDA graph,
 * in this process: a host-side counter, incremented once per launch that the
 * CUDA runtime accepted (no counterpart in the paper).  The difference across
 * a graph capture is the number of kernels one replay runs. */
unsigned long long moe_kernel_launch_count(void);

/* ---------------------------------------------------------------- bandwidth profile
 * The two measured bandwidths the q* split is made from ([P] section 3.2,
 * Eq. 3-4: q* = m * B_P / B_H; [P] Table 1 measures them per machine on the
 * deployed tensor shapes, because the ratio cannot be read from
 * specification sheets), the contended pair (the write-up "FreeToken:
 * bandwidth-adaptive edge MoE serving", section "The split, and what it is
 * actually optimising": the preferred fetch fraction comes from measuring
 * both sides while they contend) and the hybrid gate B_H > 2 B_P (same
 * write-up, section "When to use it (and when not)").
 *
 * On GB300 the source-of-truth expert pool would sit in Grace memory behind
 * NVLink-C2C, and the C branch runs on the GPU rather than on host cores:
 * B_P is the copy engine moving expert bytes from pinned host memory into
 * HBM (the fill path F), B_H the SMs reading that host memory in place (the
 * in-place path C).  Rates are in GB/s (1e9 bytes per second). */
typedef struct moe_bw_profile {
  double b_p_gbs;            /* copy engine, pinned host -> device, running alone */
  double b_h_gbs;            /* SMs reading the pinned host buffer in place, running alone */
  double b_p_contended_gbs;  /* the copy while the in-place read runs */
  double b_h_contended_gbs;  /* the in-place read while the copy runs */
  double phi;                /* B_P / B_H (Eq. 4); 1 when B_H is 0 and B_P > 0 (no in-place path: every miss
                                fills), 0 when both are 0 */
  double phi_contended;      /* B_Pc / (B_Pc + B_Hc): the copy's share of the contended total, which is
                                B_P / B_H when the two share the host bandwidth fully (B_Hc = B_H - B_P) */
  uint32_t phi_q16;          /* moe_phi_to_q16(phi): the phi_q16 argument of the bind and layer calls */
  uint32_t phi_contended_q16;
  int32_t hybrid_ok;         /* 1 when B_H > 2 B_P (the split is worth running), else 0 */
  uint32_t read_checksum;    /* moe_bench_bandwidth: XOR of every 32-bit word the in-place read saw */
} moe_bw_profile;

/* phi as the split's Q16 argument: round-half-even(phi * 65536), clamped to
 * [0, 65536]; 0 for NaN or phi <= 0.  Host arithmetic, no GPU needed. */
uint32_t moe_phi_to_q16(double phi);

/* Fills phi, phi_contended, both Q16 forms and hybrid_ok of *prof from its
 * four rates (host arithmetic, no GPU needed).  MOE_ERR_INVALID_ARG when prof
 * is NULL or a rate is negative or not finite. */
int moe_bw_derive(moe_bw_profile* prof);

/* Measures the four rates, then moe_bw_derive.  host_src: `bytes` of pinned
 * (page-locked) host memory that the device can address (cudaHostAlloc or
 * cudaHostRegister; an expert-sized buffer is the deployed shape), owned by
 * the caller; dev_dst: `bytes` of device memory, overwritten.  Each rate
 * moves `iters` x `bytes` after one untimed pass; the contended pair runs the
 * copies on copy_stream and the in-place reads on read_stream at once, with
 * the read count scaled so that both take about as long.  bytes a positive
 * multiple of 16 and both pointers 16-byte aligned, iters >= 1, the two
 * streams distinct and both created streams (not the legacy default stream,
 * which would serialise the contended pair); else MOE_ERR_INVALID_ARG (also
 * when the device cannot address host_src).  A profiling call, not for stream capture: it
 * synchronises both streams and keeps its checksum word in a static device
 * variable, so concurrent calls race.  MOE_ERR_CUDA on a launch or copy
 * error. */
int moe_bench_bandwidth(const void* host_src, void* dev_dst, size_t bytes, int iters, moe_bw_profile* out,
                        moe_stream_t copy_stream, moe_stream_t read_stream);

/* ---------------------------------------------------------------- router
 * Router scoring and top-k with renormalisation ([P] section 3.2: at each
 * MoE layer the router runs on the GPU and selects the active experts).
 *   logits[t, e] = sum_h x[t, h] * w_router[e, h] + bias[e]   (fp32 accumulation)
 *   topk_ids[t, :] = the k largest logits' ids (ties to the lower id), ascending
 *   topk_w[t, j]  = exp(l_j - max_sel) / sum_sel exp(l - max_sel)
 *                   (softmax over all E, renormalised over the k selected)
 * x bf16 [T, H]; logits_opt fp32 [T, E] or NULL.  1 <= k <= 16, k <= E <= 512.
 * T = 0 is a no-op.
 * For T > 32 and H a multiple of 64 the products run on the tensor cores:
 * each fp32 router weight is split exactly into three bf16 parts
 * (hi + mid + lo == w) and the bf16 products are accumulated in fp32 over
 * K = 3H.  The workspace then holds the split weights (E x 3H bf16) and,
 * when logits_opt is NULL, the logits (T x E fp32); its size depends on H. */
size_t moe_route_topk_workspace_size(int T, int H, int E);
int moe_route_topk(const void* x, int T, int H, const float* w_router, const float* bias, int E,
                   int k, int32_t* topk_ids, float* topk_w, float* logits_opt, void* ws,
                   size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- dispatch
 * Token -> expert grouping for the grouped evaluation of [P] section 3.2.
 * Stable counting sort of the flat routed rows i = t*k + j by expert id:
 *   counts[e] = #{i : topk_ids[i] == e};  offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   perm[pos] = i, inv_perm[i] = pos, with rows of one expert in increasing i.
 * x_opt / x_perm_opt: if both non-NULL, x_perm[pos, :] = x[perm[pos] / k, :]
 * (bf16, [T*k, H]).  Ids outside [0, E) set MOE_DEV_ERR_BAD_ID and are
 * counted nowhere; their perm/inv_perm entries are left unwritten. */
size_t moe_dispatch_workspace_size(int T, int k, int E);
int moe_dispatch(const int32_t* topk_ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
                 int32_t* perm, int32_t* inv_perm, const void* x_opt, int H, void* x_perm_opt,
                 void* ws, size_t ws_bytes, uint32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- residency
 * Device-side cache control of [P] section 4.1 for one MoE layer, followed by
 * the fused batched fill copy.  One kernel: deduplicate the routed experts,
 * classify them against the slot table into hits H and misses M (m = |M|),
 * derive q = fill count of m at fetch fraction phi_q16 = B_P/B_H in Q16
 * ([P] section 3.2, Eq. 1-4; integer rule of [W] "The split, and what it is
 * actually optimising"; if min_fill != 0 and phi_q16 > 0 and m > 0 then
 * q >= 1, the "at least one fill" floor of [P] section 3.2), choose F
 * (fill_policy), find the q least-recently-used slots not hit by this call
 * in one pass (victims, ordered by (stamp, slot)), rebind evicted pairs to
 * the staging pool, admit F into the victims (F in ascending id order paired
 * with victims in order), and bind the other misses C to the staging pool.
 * Hits and fills take stamp = ++clock.  Then one fixed-shape copy launch,
 * masked by the device fill count, copies every filled expert's three bank
 * rows from the staging pool to its cache slot.
 * fills_opt: int32 [min(T*k, E), 2] (src staging slot, dst cache slot) rows
 * 0..n_fill-1, or NULL.  stats_dev: moe_bind_stats, or NULL.
 * Limits: E <= 1024, cache.n_slots <= 16384. */
size_t moe_cache_bind_workspace_size(const moe_cache* cache, int T, int k);
int moe_cache_bind_slots(const moe_cache* cache, int layer, const int32_t* topk_ids, int T, int k,
                         uint32_t phi_q16, int min_fill, int fill_policy, uint64_t seed,
                         moe_bind_stats* stats_dev, int32_t* fills_opt, void* ws, size_t ws_bytes,
                         uint32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- expert FFN
 * Grouped SwiGLU expert FFN over the combined execution set of [P] section
 * 3.2, reading every expert's weights through the slot table ([P] section 3:
 * lookup and execution on logical (layer, expert) ids).  For each expert e
 * with counts[e] > 0 (and expert_mask_opt[e] != 0 if a mask is given), with
 * rows pos in [offsets[e], offsets[e+1]) and x row t = perm[pos] / k:
 *   g = x_t W_gate^T, u = x_t W_up^T (fp32 accumulation), h = bf16(silu(g) * u),
 *   y_rows[perm[pos], :] = h W_down^T (fp32 accumulation, stored fp32)
 * i.e. y_rows is token-major: row t*k + j holds the output of token t's j-th
 * routed expert, so the combine reads each token's k rows contiguously.
 * where the banks are those of pool slot_table[layer*E + e].  x bf16 [T, H];
 * x_perm_opt: bf16 [T*k, H] gathered rows (from moe_dispatch), required by
 * the GEMM kernel and used by the GEMV kernel if given.  Rows of experts
 * outside the mask are not written.  An unbound entry sets
 * MOE_DEV_ERR_UNBOUND and leaves that expert's rows unwritten. */
size_t moe_expert_ffn_workspace_size(int T, int k, int E, int H, int I, int ffn_mode);
int moe_expert_ffn_grouped(const moe_cache* cache, int layer, const int32_t* counts,
                           const int32_t* offsets, const int32_t* perm, const void* x,
                           const void* x_perm_opt, int T, int k, const uint8_t* expert_mask_opt,
                           int ffn_mode, float* y_rows, void* ws, size_t ws_bytes,
                           uint32_t* dev_status, moe_stream_t stream);

/* Size of the scratch array built into the library for
 * moe_expert_ffn_grouped_noalloc (4 MiB per device that loads the library). */
#define MOE_NOALLOC_FFN_SCRATCH_BYTES (4u << 20)

/* moe_expert_ffn_grouped without a workspace argument, for callers that cannot
 * allocate device memory: a host framework that owns all device memory and
 * offers no allocator, a service running on a memory budget fixed at load
 * time, or a serving loop that must not call cudaMalloc/cudaFree because they
 * can synchronise the device.  The paper has no counterpart to this call.
 * Same arguments, results and errors as moe_expert_ffn_grouped, checked in
 * the same order; the scratch is a static array of
 * MOE_NOALLOC_FFN_SCRATCH_BYTES inside the library, held by every device that
 * loads it until the process exits.  After the argument checks, returns
 * MOE_ERR_WORKSPACE when the call would need more than that
 * (moe_expert_ffn_workspace_size(T, k, E, H, I, ffn_mode) bytes).  The first
 * call in a CUDA context (on each device, and again after a device reset)
 * looks up the array's device address with that device current; make that
 * first call before any stream capture.  All calls on a device share the
 * array, so calls that overlap on the GPU race; the array needs no clearing
 * between calls.  Allocates nothing. */
int moe_expert_ffn_grouped_noalloc(const moe_cache* cache, int layer, const int32_t* counts,
                                   const int32_t* offsets, const int32_t* perm, const void* x,
                                   const void* x_perm_opt, int T, int k,
                                   const uint8_t* expert_mask_opt, int ffn_mode, float* y_rows,
                                   uint32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- MXFP4 experts
 * Block-scaled FP4 expert banks ([P] section 5.1 "Models": the routed experts
 * of DeepSeek-V4-Flash are natively MXFP4; section 4.1: expert kernels
 * dequantise in-kernel).  Encoding of the OCP Microscaling Formats (MX) v1.0
 * specification: FP4 E2M1 elements (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and
 * their negatives) and one E8M0 scale 2^(s - 127) (s = 255: NaN) per block of
 * 32 consecutive inputs of a weight row.  A row of K inputs is K/2 code bytes,
 * input 2c in the low nibble of byte c and input 2c+1 in the high nibble, and
 * K/32 scale bytes.  Banks are slot-major like the bf16 ones:
 *   gate_q, up_q  [n_slots, I, H/2]   gate_s, up_s  [n_slots, I, H/32]
 *   down_q        [n_slots, H, I/2]   down_s        [n_slots, H, I/32]
 * Code banks 16-byte aligned; scale banks have no alignment requirement. */
typedef struct moe_pool_mxfp4 {
  const void* gate_q;
  const void* gate_s;
  const void* up_q;
  const void* up_s;
  const void* down_q;
  const void* down_s;
  int32_t n_slots;
  int32_t reserved;   /* 0 */
} moe_pool_mxfp4;

/* moe_expert_ffn_grouped (GEMV mode) over MXFP4 banks: for each expert e with
 * counts[e] > 0, rows pos in [offsets[e], offsets[e+1]), x row t = perm[pos]/k,
 *   g = x_t W_gate^T, u = x_t W_up^T, h = bf16(silu(g) * u),
 *   y_rows[perm[pos], :] = h W_down^T
 * with W the dequantised weights of the slot that slot_table[layer*E + e]
 * names (cache_pool, or staging_opt for MOE_STAGING_TAG entries; the same
 * encoding as moe_cache).  Three kernels, by the call's shape:
 * - at most 64 routed rows, H and I in {1024, 2048, 4096}, 16-byte aligned
 *   scale banks: one weight-streaming launch (the token's activations
 *   rescaled per 32-input block by a power of two into f16, exact f16
 *   products of the E2M1 values, each block's sum scaled by its power of two);
 * - otherwise, with I a multiple of 128, H of 256, H/32 and I/32 multiples of
 *   8 and 8-byte aligned scale banks: the tensor-core GEMM (the token rows
 *   gathered in dispatch order; the weights expanded exactly into bf16 in
 *   shared memory, E2M1 value times the block's power of two, then
 *   tcgen05.mma against the bf16 token rows, fp32 accumulation).  The
 *   expansion is exact for weights below 2^128 in magnitude: every code up to
 *   the scale byte 252; larger weights become infinities;
 * - otherwise: a two-launch table-decode kernel.
 * slot_table: [n_layers*E] int32.  x bf16 [T, H]; y_rows fp32 [T*k, H],
 * token-major.  counts / offsets / perm as moe_dispatch writes them.
 * Errors: MOE_ERR_INVALID_ARG for a NULL pool, table or (T > 0) array, a
 * pool missing a bank or with n_slots < 1, layer outside [0, n_layers), k
 * outside [1, min(E, 16)], H or I below 32; MOE_ERR_UNSUPPORTED for H or I
 * not a multiple of 32, E > 1024, T*k > INT_MAX/2, a code bank, x or y_rows
 * not 16-byte aligned; MOE_ERR_WORKSPACE for ws_bytes below
 * moe_expert_ffn_mxfp4_workspace_size(T, k, H, I) (the bf16 h rows, one
 * counter per routed row and the gathered bf16 token rows; 0 for invalid
 * arguments), MOE_ERR_UNSUPPORTED for
 * a ws that is not 256-byte aligned.  T = 0 returns MOE_OK and launches nothing.  On the
 * device, an unbound or out-of-range entry sets MOE_DEV_ERR_UNBOUND /
 * MOE_DEV_ERR_BAD_SLOT and leaves that expert's rows unwritten. */
size_t moe_expert_ffn_mxfp4_workspace_size(int T, int k, int H, int I);
int moe_expert_ffn_mxfp4(const moe_pool_mxfp4* cache_pool, const moe_pool_mxfp4* staging_opt,
                         const int32_t* slot_table, int n_layers, int layer, int E, int H, int I,
                         const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                         const void* x, int T, int k, float* y_rows, void* ws, size_t ws_bytes,
                         uint32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- NVFP4 experts
 * Block-scaled FP4 banks in NVIDIA's NVFP4 format ([P] section 5.1 "Models":
 * the routed experts of GLM-5.2 and of the laptop build of Qwen3.6-35B-A3B
 * are NVFP4; section 4.1: expert kernels dequantise in-kernel): FP4 E2M1
 * elements packed as in MXFP4, one FP8 E4M3 scale byte per block of 16
 * consecutive inputs (the OCP 8-bit E4M3 without infinities: 0x7F and 0xFF
 * are NaN), and one fp32 scale per bank of each expert:
 *   W[r, i] = e2m1(code of i) * e4m3(scale of block i/16) * tensor_scale
 * Banks are slot-major; a row of K inputs is K/2 code bytes and K/16 scale
 * bytes:
 *   gate_q, up_q  [n_slots, I, H/2]   gate_s, up_s  [n_slots, I, H/16]
 *   down_q        [n_slots, H, I/2]   down_s        [n_slots, H, I/16]
 *   tensor_scale  fp32 [n_slots, 3]   (gate, up, down of each slot)
 * Code and scale banks 16-byte aligned, tensor_scale 4-byte aligned. */
typedef struct moe_pool_nvfp4 {
  const void* gate_q;
  const void* gate_s;
  const void* up_q;
  const void* up_s;
  const void* down_q;
  const void* down_s;
  const float* tensor_scale;
  int32_t n_slots;
  int32_t reserved;   /* 0 */
} moe_pool_nvfp4;

/* moe_expert_ffn_mxfp4 over NVFP4 banks, same arguments, layouts, results
 * and device errors.  Two kernels, by the call's shape:
 * - T*k at most 64 routed rows and H, I in {1024, 2048, 4096}: one
 *   weight-streaming launch (every routed row reads its expert's weights
 *   once).  Each 16-input half of a 32-input code vector sums its exact f16
 *   products in fp32 and is scaled by its E4M3 value (exact in fp32) and the
 *   activations' power-of-two back-scale;
 * - otherwise, with I a multiple of 128 and H of 256: the tensor-core GEMM,
 *   the weights expanded exactly into bf16 (E2M1 value times E4M3 value) and
 *   multiplied against the bf16 token rows with fp32 accumulation.
 * Either way the row's fp32 sum is scaled by the bank's tensor scale.
 * Errors: as moe_expert_ffn_mxfp4 with 16 in place of 32 for the H and I
 * checks, plus MOE_ERR_INVALID_ARG for a NULL tensor_scale,
 * MOE_ERR_UNSUPPORTED for a misaligned bank or tensor_scale and for calls
 * that fit neither kernel.  moe_expert_ffn_nvfp4_workspace_size(T, k, H, I)
 * bytes of ws. */
size_t moe_expert_ffn_nvfp4_workspace_size(int T, int k, int H, int I);
int moe_expert_ffn_nvfp4(const moe_pool_nvfp4* cache_pool, const moe_pool_nvfp4* staging_opt,
                         const int32_t* slot_table, int n_layers, int layer, int E, int H, int I,
                         const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                         const void* x, int T, int k, float* y_rows, void* ws, size_t ws_bytes,
                         uint32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- the layer over FP4 experts
 * An expert cache whose pools hold block-scaled FP4 experts ([P] section 5.1:
 * DeepSeek-V4-Flash serves MXFP4 experts, GLM-5.2 and the laptop Qwen3.6
 * NVFP4 ones; [P] section 4.1: the fill copy moves every bank of an admitted
 * expert under one list).  The residency arrays are moe_cache's; both pools
 * have the moe_pool_nvfp4 layout (for MXFP4 the scale banks hold K/32 bytes
 * per row and tensor_scale is NULL). */
#define MOE_FP4_MXFP4 0
#define MOE_FP4_NVFP4 1
typedef struct moe_cache_fp4 {
  moe_pool_nvfp4 cache;     /* pool A: the slots the LRU manages */
  moe_pool_nvfp4 staging;   /* pool B: every (layer, expert) pair at slot layer*E + expert; optional */
  int32_t* slot_table;      /* [n_layers * E], as moe_cache */
  int32_t* owner;           /* [cache.n_slots] */
  uint32_t* stamp;          /* [cache.n_slots] */
  uint32_t* clock;          /* [1] */
  int32_t n_layers, E, H, I;
  int32_t format;           /* MOE_FP4_MXFP4 or MOE_FP4_NVFP4 */
  int32_t reserved;         /* 0 */
} moe_cache_fp4;

/* moe_layer_forward over an FP4 expert cache: router and top-k, the
 * residency bind (the same decisions and state updates as
 * moe_cache_bind_slots) with a fill copy of the admitted experts' six code
 * and scale banks (and tensor scales) from the staging pool into their cache
 * slots, dispatch, the FP4 expert FFN (moe_expert_ffn_mxfp4 /
 * moe_expert_ffn_nvfp4) and the combine.  One-token calls with H and I in
 * {1024, 2048, 4096}, k <= 32, at most 512 cache slots and at most 4 router
 * rows per SM run all of it in one cooperative launch (the FFN on the
 * weight-streaming ring kernel's arithmetic, the fills copied after the
 * expert rows); other calls run per-step launches.  Arguments as
 * moe_layer_forward (layer->E, H, I equal to the cache's); stats_dev
 * optional.  Errors: those of the steps, plus MOE_ERR_INVALID_ARG for an
 * unknown format, a shape mismatch or a NULL router, MOE_ERR_UNSUPPORTED for
 * E > 512 or a router, x or ws not aligned as the router and the FFN need,
 * and MOE_ERR_WORKSPACE below moe_layer_fp4_workspace_size; every check is
 * made before the first launch.  NVFP4 calls that fit neither of
 * moe_expert_ffn_nvfp4's kernels return MOE_ERR_UNSUPPORTED. */
size_t moe_layer_fp4_workspace_size(const moe_layer* layer, const moe_cache_fp4* cache, int T);
int moe_layer_forward_fp4(const moe_layer* layer, const moe_cache_fp4* cache, const void* x, int T, void* out,
                          uint32_t phi_q16, int min_fill, int fill_policy, uint64_t seed, void* ws,
                          size_t ws_bytes, uint32_t* dev_status, moe_bind_stats* stats_dev,
                          moe_stream_t stream);

/* ---------------------------------------------------------------- combine
 * Gate-weighted merge of the expert outputs ([P] section 3.2: the partial
 * sums of the GPU set and the in-place set merge into the exact layer
 * output).  out[t, :] = sum_{j=0}^{k-1} topk_w[t, j] * y_rows[t*k + j, :]
 * summed in j order (ascending expert id) with fp32 FMAs, then rounded to
 * bf16 (out) and/or stored fp32 (out_f32_opt).  The result does not depend
 * on which pool any row's expert was read from.  out or out_f32_opt may be
 * NULL, not both. */
int moe_combine(const float* y_rows, const float* topk_w, int T, int k, int H, void* out,
                float* out_f32_opt, uint32_t* dev_status, moe_stream_t stream);

/* ---------------------------------------------------------------- whole layer
 * moe_route_topk -> moe_cache_bind_slots -> moe_dispatch ->
 * moe_expert_ffn_grouped -> moe_combine on one stream ([P] section 3.2 decode
 * order: cache update, batch copy of F, grouped evaluation, merge).
 * out bf16 [T, H].  bufs_opt may name caller buffers for intermediates.
 * stats_dev: moe_bind_stats or NULL.
 * How it runs (the results are those of the five calls in every case):
 * decode-sized calls (T <= 8, T*k <= 32, E <= 512, at most 1024 cache slots,
 * the fused GEMV's shapes, ffn_mode GEMV or AUTO with T <= 2) run as ONE
 * cooperative launch (router, selection, residency decision and commit,
 * fused FFN with the fills streamed into their slots, combine); other calls
 * of at most 32 routed rows use a one-warp front end and one fused FFN launch;
 * larger calls run the per-step launches, the FFN on the tensor-core GEMM
 * under AUTO when T > 2.  The fused launches are cooperative (one CTA per
 * SM, all resident together), so they start only once every SM can take one
 * of their CTAs.
 * Errors: MOE_ERR_INVALID_ARG when layer->k is outside [1, min(E, 16)], the
 * layer's E, H, I differ from the cache's, or a required pointer is NULL;
 * MOE_ERR_UNSUPPORTED when T * k exceeds INT_MAX / 2; the sub-calls' errors
 * otherwise.  moe_layer_workspace_size returns 0 for such arguments. */
size_t moe_layer_workspace_size(const moe_layer* layer, const moe_cache* cache, int T,
                                int ffn_mode);
int moe_layer_forward(const moe_layer* layer, const moe_cache* cache, const void* x, int T,
                      void* out, uint32_t phi_q16, int min_fill, int fill_policy, uint64_t seed,
                      int ffn_mode, const moe_layer_buffers* bufs_opt, void* ws, size_t ws_bytes,
                      uint32_t* dev_status, moe_bind_stats* stats_dev, moe_stream_t stream);

/* Full-layer double-buffered prefill ([P] section 3.1 and Figure 2 (1),
 * prefill codesign; [W] "Prefill: full-layer double buffering"; [P] section
 * 5.3: disabled when the pool cannot spare two layers).  Runs n_layers
 * stacked layers, each on its own input block x[l] (bf16 [T, H]) into out[l]
 * (bf16 [T, H]), with every expert of every layer in `source`, a pool that
 * may live in host memory (pinned, or any memory the copy engine and the GPU
 * reach): layer l's experts are its slots l*E .. l*E+E-1.  layer_buf[0] and
 * layer_buf[1] are HBM pools of at least E slots.  The copy engine moves
 * layer l's three banks into layer_buf[l % 2] on copy_stream (one
 * cudaMemcpyAsync per bank) while layer l-1 computes from the other buffer
 * on `stream` (moe_layer_forward with phi = 0: every expert is resident in
 * the buffer).  overlap = 0, or a layer_buf[1] with fewer than E slots or a
 * NULL bank, loads on demand into layer_buf[0]: each layer's copy waits for
 * the previous layer.  state: the residency arrays of a cache of n_layers
 * layers and E slots (slot_table [n_layers*E] with entry l*E+e = e; owner,
 * stamp [E]; clock), its pools ignored.  ws: moe_layer_workspace_size(layer,
 * cache, T, ffn_mode) bytes, reused by every layer.  Every launch and copy
 * only enqueues: the copies fork from `stream` at the call and join it
 * before the layer that reads them.  The events the call creates are
 * released once the work completes.  Errors: MOE_ERR_INVALID_ARG for
 * layers whose shapes differ or whose layer index is not their position, a
 * source of fewer than n_layers*E slots, a missing layer_buf[0], state
 * arrays missing or of another shape, copy_stream NULL or equal to stream;
 * any error of moe_layer_forward; MOE_ERR_CUDA for a failed copy or event
 * call.  T = 0 returns MOE_OK and launches nothing. */
int moe_prefill_double_buffered(const moe_layer* layers, int n_layers, const moe_pool* source,
                                const moe_pool* layer_buf, const moe_cache* state, const void* const* x, int T,
                                void* const* out, int ffn_mode, int overlap, void* ws, size_t ws_bytes,
                                uint32_t* dev_status, moe_stream_t stream, moe_stream_t copy_stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
