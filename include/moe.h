/*
 * libmoe -- single-GPU MoE expert layer for GB300 (sm_103a).
 *
 * The layer, as described by three sglang PR reports:
 *   [P1] "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report)
 *   [P2] "Add BF16 support to EP-MoE for DeepGEMM"    (sglang PR #17392 report)
 *   [P3] "[Feature] Support BF16 and batch-invariant inference with DeepEP v2"
 *        (sglang PR #38160 report)
 *
 *   plan_layout      top-k routing -> per-expert row layout      [P1 "实现拆解" 2-3]
 *   quant_scatter    x -> FP8 1x128 / MXFP8 1x32 UE8M0 (or BF16) expert rows
 *                                                                [P1 "实现拆解" 3, "风险与影响" 5; P2 step 3]
 *   grouped_gemm_w13_act   h = silu(a W1^T) * (a W3^T)            [P2 "关键源码片段" deep_gemm.py]
 *   grouped_gemm_w2        y = h W2^T                             [P2 same]
 *   combine          out[t] = sum_j w[t,j] * y[src2dst[t,j]]      [P1 "风险与影响" 2, P3 "实现拆解" 3]
 *   forward          all five, in order, on one stream
 * and, around the layer: load-time weight preparation (UE8M0 requantisation,
 * MXFP8 / MXFP4 scale packing) and the fp32 router that produces the routing
 * input.
 *
 * Conventions for every call below
 * --------------------------------
 * - Pointers named "device" are CUDA device pointers; all of them must be
 *   16-byte aligned.  The caller allocates and owns every buffer (weights,
 *   inputs, outputs, workspace); the library allocates no device memory and
 *   frees nothing of the caller's.
 * - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   The hot calls only enqueue work: no host synchronisation, no allocation,
 *   static shapes, so a sequence of them can be captured in a CUDA graph.
 * - Errors the host can see (bad pointers, sizes, unsupported shapes) are
 *   returned before anything is launched.  Errors in the data (an expert id
 *   outside [-1, E_global), a masked expert with more than max_m rows, a wait
 *   that timed out inside a kernel) set a status word in the workspace; the
 *   offending item is skipped and the call still returns MOE_OK.  The word
 *   holds the first such error since the last moe_plan_layout (which clears
 *   it) and is read with moe_read_device_status().
 * - Sizes are int64; the weights of the large shapes exceed 2^31 elements.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,      /* null / misshaped argument */
  MOE_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. K % 128 != 0) */
  MOE_ERR_BUFFER_TOO_SMALL = 3, /* problem larger than a fixed-size buffer (moe_plan_layout_noalloc) */
  MOE_ERR_MISALIGNED = 4,       /* a pointer is not 16-byte aligned */
  MOE_ERR_CUDA = 5,             /* a CUDA runtime / driver call failed */
  MOE_ERR_EXPERT_ID = 6,        /* device: topk id outside [-1, E_global) */
  MOE_ERR_MASKED_OVERFLOW = 7,  /* device: masked expert got more than max_m rows */
  MOE_ERR_TIMEOUT = 8,          /* device: a bounded wait inside a kernel ran out */
  MOE_ERR_DTYPE_MISMATCH = 9    /* weight arguments contradict the declared dtype */
} moe_status_t;

/* Arithmetic of the expert GEMMs [P1 "实现拆解" 1 and 3; P2 "实现拆解" 2]. */
typedef enum {
  MOE_DTYPE_FP8_E4M3_UE8M0 = 0, /* FP8 e4m3 operands, UE8M0 scales: 1x128 (activations), 128x128 (weights) */
  MOE_DTYPE_BF16 = 1,           /* bf16 operands, no scales */
  MOE_DTYPE_MXFP8 = 2,          /* FP8 e4m3 operands, one UE8M0 scale per 1x32 block for activations, h
                                   and every weight row (the MXFP8 variant [P1 "风险与影响" 5]) */
  MOE_DTYPE_MXFP4 = 3           /* FP4 E2M1 weights with one UE8M0 scale per row and 1x32 block (MXFP4),
                                   activations and h as for MXFP8 (the FP4 variant [P1 "风险与影响" 5]) */
} moe_dtype_t;

/* Row layout of the expert inputs [P1 "实现拆解" 2, "关键源码片段" deep_gemm.py]. */
typedef enum {
  MOE_LAYOUT_AUTO = 0,    /* masked iff E_global > E_local && E_local <= 32, else compact */
  MOE_LAYOUT_COMPACT = 1, /* [all_tokens, K], experts padded to block_e rows, m_indices row->expert */
  MOE_LAYOUT_MASKED = 2   /* [E_local, max_m, K] with masked_m[E_local] valid rows per expert */
} moe_layout_t;

/* Static shape of one layer call (MoeRunnerConfig fields [P1 "关键源码片段"
 * deep_gemm.py; P3 "关键源码片段" layer.py] plus the local expert range of
 * [P3 "实现拆解" 1]). */
typedef struct {
  int64_t T;            /* tokens (>= 0) */
  int64_t K;            /* hidden size, multiple of 128 */
  int64_t I;            /* per-expert intermediate size, multiple of 128 */
  int32_t E_global;     /* experts the router chooses from */
  int32_t E_local;      /* experts held here, 1..1024 */
  int32_t expert_start; /* first local expert; E_local + expert_start <= E_global */
  int32_t topk;         /* experts per token, 1..64 */
  int32_t block_e;      /* compact padding granularity; must be 128 */
  int32_t dtype;        /* moe_dtype_t */
  int32_t layout;       /* moe_layout_t */
  int32_t reserved;
  int64_t max_m;        /* masked layout: rows per expert (>= T); ignored for compact */
} moe_shape_t;

/* Byte offsets of the intermediates inside the caller's workspace (all
 * 1024-byte aligned).  Rows of a/h/y: compact -> all_tokens; masked ->
 * E_local * max_m (expert e's rows start at e * max_m). */
typedef struct {
  uint64_t total_bytes;
  uint64_t status;      /* int32[4]: [0] = first moe_status_t seen on the device */
  uint64_t meta;        /* int32[8]: [0] padded rows, [1] valid 128-row blocks */
  uint64_t counts;      /* int32[E_local] assignments per local expert */
  uint64_t padded;      /* int32[E_local] compact: counts rounded up to 128 */
  uint64_t start;       /* int32[E_local] compact: first row of each expert */
  uint64_t masked_m;    /* int32[E_local] masked: valid rows per expert */
  uint64_t m_indices;   /* int32[all_tokens] compact: local expert per row, -1 = no token */
  uint64_t src2dst;     /* int32[T * topk] destination row per assignment, -1 = dropped */
  uint64_t block_info;  /* int32[4 * blocks]: {expert, first row, tma row, valid rows} */
  uint64_t chunk_hist;  /* int32[E_local * chunks] plan scratch */
  uint64_t chunk_rank;  /* int32[T * topk]         plan scratch */
  uint64_t a;           /* [rows, K]  fp8 bytes or bf16: expert inputs */
  uint64_t a_sf;        /* fp8 / mxfp8: scale chunks of a (see moe_sf_offset); FP8 stores four consecutive
                           128-column groups' scales of a row in one word's four bytes, MXFP8 the four
                           32-column scales of a row and 128-column group */
  uint64_t h;           /* [rows, I]  fp8 bytes or bf16: silu(gate) * up */
  uint64_t h_sf;        /* fp8 / mxfp8: scale chunks of h */
  uint64_t y;           /* [rows, K]  bf16: expert outputs */
  int64_t rows;         /* rows of a / h / y */
  int64_t all_tokens;   /* compact static bound (0 for masked) */
  int64_t blocks;       /* static number of 128-row blocks */
  int32_t layout;       /* resolved moe_layout_t */
  int32_t chunks;       /* plan chunks of 256 assignments */
  /* Masked layout only (0 / empty for compact): each expert GEMM's K loop runs
   * in k_splits fixed segments (from K, I and the dtype alone, never from T or
   * max_m); every segment writes fp32 partial sums of the tile's valid rows,
   * and a second kernel of the same call adds them in segment order. */
  uint64_t block_vrow;  /* int32[blocks]: first valid-row index of each block (rows counted without padding) */
  uint64_t partial;     /* fp32 [k_splits][partial_rows][partial_cols] segment sums */
  int64_t partial_rows; /* min(T * topk, E_local * max_m) */
  int32_t k_splits1;    /* segments of GEMM1 (w13) */
  int32_t k_splits2;    /* segments of GEMM2 (w2) */
} moe_ws_layout_t;

typedef struct moe_ctx moe_ctx;

/* Static compact row bound of [P1 "关键源码片段" deep_gemm.py]:
 * block_e * (min(A, E) + (A - min(A, E)) / block_e).  Returns -1 on negative
 * input or block_e <= 0. */
int64_t moe_compact_all_tokens(int64_t num_assignments, int32_t num_experts, int32_t block_e);

/* Layout choice of [P1 "关键源码片段" deep_gemm.py]: MOE_LAYOUT_MASKED iff
 * E_global > E_local and E_local <= 32, else MOE_LAYOUT_COMPACT. */
int32_t moe_choose_layout(int32_t E_global, int32_t E_local);

/* Create a context for one layer shape and its weights (device pointers):
 *   FP8:  w13 uint8 [E_local, 2I, K] e4m3, w13_sf uint8 [E_local, 2I/128, K/128] UE8M0,
 *         w2  uint8 [E_local, K, I]  e4m3, w2_sf  uint8 [E_local, K/128, I/128]  UE8M0
 *   MXFP8: w13, w2 as for FP8; w13_sf / w2_sf hold one UE8M0 byte per row and
 *         32-column block ([E_local, 2I, K/32] / [E_local, K, I/32]) in the
 *         packed order moe_pack_mx_scales writes (16-byte aligned)
 *   MXFP4: w13 uint8 [E_local, 2I, K/2], w2 uint8 [E_local, K, I/2]: E2M1 codes,
 *         two per byte, element 2j in the low nibble of byte j, 32-byte
 *         aligned (else MOE_ERR_MISALIGNED; the GEMMs multiply the codes as
 *         E2M1 operands without expanding them); scales as for MXFP8
 *   BF16: w13 bf16 [E_local, 2I, K], w2 bf16 [E_local, K, I]; w13_sf = w2_sf = NULL
 * Rows 0..I-1 of w13[e] are the gate projection W1, rows I..2I-1 the up
 * projection W3 [P2 "关键源码片段" deep_gemm.py: the activation splits the
 * GEMM output in halves].  Weights are read, never written, and must stay
 * alive while the context is used.  A scale pointer given for BF16 or missing
 * for FP8 / MXFP8 / MXFP4 is MOE_ERR_DTYPE_MISMATCH.  Host-only: builds the weight TMA
 * descriptors; allocates no device memory. */
moe_status_t moe_ctx_create(const moe_shape_t* shape, const void* w13, const uint8_t* w13_sf,
                            const void* w2, const uint8_t* w2_sf, moe_ctx** out);
void moe_ctx_destroy(moe_ctx* ctx);

/* Workspace the caller must provide to the hot calls (device, 256-byte
 * aligned, at least total_bytes).  No initialisation is needed: every
 * region is written before it is read within one pass of the layer. */
moe_status_t moe_workspace_layout(const moe_ctx* ctx, moe_ws_layout_t* out);
moe_status_t moe_workspace_size(const moe_ctx* ctx, size_t* bytes);

/* Step 1 [P1 "实现拆解" 2-3, "关键源码片段" ep_moe_kernels.py; P3 "实现拆解" 1]:
 * topk_ids int32 [T, topk] (device; -1 = no assignment).  Clears the status
 * word, then writes counts,
 * padded/start/m_indices (compact) or masked_m (masked), src2dst and the
 * 128-row block table into ws.  Inside an expert, assignments keep their
 * flattened t * topk + j order; rows without a token have m_indices -1. */
moe_status_t moe_plan_layout(moe_ctx* ctx, const int32_t* topk_ids, void* ws, void* stream);

/* Caller-owned outputs of moe_plan_layout_noalloc (device pointers, int32,
 * same contents as the workspace regions of the same name).  all_tokens =
 * moe_compact_all_tokens(T * topk, E_local, 128); blocks = all_tokens / 128
 * (compact) or E_local * ceil(max_m / 128) (masked). */
typedef struct {
  int32_t* status;     /* [4]; cleared, then first data error of the call */
  int32_t* meta;       /* [8]; [0] padded rows, [1] valid 128-row blocks */
  int32_t* counts;     /* [E_local] */
  int32_t* padded;     /* [E_local], compact only (NULL allowed for masked) */
  int32_t* start;      /* [E_local], compact only */
  int32_t* masked_m;   /* [E_local], masked only (NULL allowed for compact) */
  int32_t* m_indices;  /* [all_tokens], compact only */
  int32_t* src2dst;    /* [T * topk] */
  int32_t* block_info; /* [4 * blocks], 16-byte aligned */
} moe_plan_outputs_t;

/* No counterpart in the PR reports: a variant of moe_plan_layout for callers
 * that cannot allocate device memory (for example code inside a framework
 * whose memory planner owns the device heap and hands it only the tensors it
 * reads and writes).  It needs no context and no workspace: the caller passes
 * the shape, topk_ids and the output buffers above, and the plan's scratch
 * lives in a 1 MiB array inside the library's device image (held by every
 * GPU that loads the library until the process exits).  Limit:
 * ceil(T * topk / 256) * E_local + T * topk <= 262144 (for example
 * T * topk = 65536 with 256 local experts); larger problems return
 * MOE_ERR_BUFFER_TOO_SMALL.  Allocates nothing (no cudaMalloc/cudaFree or
 * allocating library call).  The first call on a device looks up the
 * array's device address; make it before any stream capture.  The address is
 * cached per device and assumes the primary context is not reset
 * (cudaDeviceReset) while the library is loaded.  Calls share the array:
 * calls that overlap on the GPU race on it.  Masked layouts need
 * E_local * max_m < 2^31 (MOE_ERR_UNSUPPORTED otherwise). */
moe_status_t moe_plan_layout_noalloc(const moe_shape_t* shape, const int32_t* topk_ids,
                                     const moe_plan_outputs_t* out, void* stream);

/* Step 2 [P1 "实现拆解" 3; P2 "实现拆解" 3]: x bf16 [T, K] (device).  FP8:
 * each 128-column group of a token gets the smallest power-of-two scale 2^s
 * with amax <= 448 * 2^s (s clamped to [-127, 127]; byte s + 127) and every
 * element is rounded to e4m3 (nearest-even, saturating) after division by
 * that final scale.  The token row (and its scales) is written to each of its
 * destination rows.  BF16: rows are copied unchanged.  Needs moe_plan_layout
 * earlier on the same stream and workspace. */
moe_status_t moe_quant_scatter(moe_ctx* ctx, const void* x_bf16, void* ws, void* stream);

/* Step 3 [P2 "关键源码片段" deep_gemm.py; P1 "实现拆解" 1]: for every row
 * that carries a token: g = a W1_e^T, u = a W3_e^T (fp32 accumulation over the
 * dequantised operands), h = silu(g) * u in fp32, stored as FP8 with 1x128
 * UE8M0 scales (same rule as step 2) or as bf16.  Rows without a token are
 * skipped (neither read back nor written). */
moe_status_t moe_grouped_gemm_w13_act(moe_ctx* ctx, void* ws, void* stream);

/* Step 4 [P2 "关键源码片段" deep_gemm.py]: y = h W2_e^T, fp32 accumulation,
 * stored bf16, for rows that carry a token. */
moe_status_t moe_grouped_gemm_w2(moe_ctx* ctx, void* ws, void* stream);

/* Step 5 [P1 "风险与影响" 2 (src2dst); P3 "实现拆解" 3 (combine through slot
 * pointers)]: out[t] = bf16(sum over j of topk_weights[t, j] * y[src2dst[t, j]])
 * summed in fp32 in j order; 0 for tokens with no local assignment.
 * topk_weights fp32 [T, topk], out bf16 [T, K] (device). */
moe_status_t moe_combine(moe_ctx* ctx, const float* topk_weights, const void* ws, void* out_bf16,
                         void* stream);

/* Steps 1-5 on one stream, no synchronisation, graph-capturable. */
moe_status_t moe_forward(moe_ctx* ctx, const void* x_bf16, const int32_t* topk_ids,
                         const float* topk_weights, void* ws, void* out_bf16, void* stream);

/* Weight preparation, run once at load time [P1 "实现拆解" 1, "关键源码片段"
 * fp8.py: both expert weight tensors are requantised with UE8M0 block scales
 * through a bfloat16 intermediate].  w_in: e4m3 bytes [E, N, C]; scale_in:
 * fp32 [E, N/128, C/128], the dequantisation multiplier of each 128x128
 * block.  Per block: v = bf16(fp32(q) * s); e = smallest integer with
 * amax|v| <= 448 * 2^e (clamped to [-127, 127]); q' = e4m3(v * 2^-e), round to
 * nearest even, saturating.  Writes w_out [E, N, C] and the UE8M0 bytes e + 127
 * to scale_out [E, N/128, C/128] -- the weight format moe_ctx_create takes.
 * w_out may equal w_in.  N and C must be multiples of 128; inputs must be
 * finite.  Device pointers; enqueued on stream. */
moe_status_t moe_requant_weights_ue8m0(const uint8_t* w_in, const float* scale_in, uint8_t* w_out,
                                       uint8_t* scale_out, int64_t E, int64_t N, int64_t C, void* stream);

/* The router that produces the layer's routing input [P3 "关联脉络": the
 * MoE router GEMM is kept in fp32 so that expert selection does not flip under
 * deterministic inference; P1 "关键源码片段" deep_gemm.py: the layer takes
 * standard top-k ids and weights].
 *
 * moe_router_prepare (load time): splits the fp32 router weights w_router
 * [E_global, K] into three bf16 planes w_planes [3, E_global, K] with
 * plane0 + plane1 + plane2 == w exactly (for |w| >= 2^-110), so that the
 * router's fp32 GEMM runs on the tensor cores with exact products.  K must be
 * a multiple of 128; device pointers, 16-byte aligned; enqueued on stream.
 *
 * moe_route: for x bf16 [T, K] (device),
 *   logits[t, e] = sum_k x[t, k] * w[e, k], products exact, accumulated in
 *     fp32: per 1024-wide K segment on the tensor cores, then the segments
 *     added in order.  The operations for one token do not depend on T, so a
 *     token's results are the same bits at every batch size;
 *   topk_ids[t, :] int32 [T, topk]: the topk largest logits in descending
 *     order, equal logits ordered by the lower expert id;
 *   topk_weights[t, j] fp32 = exp(z_j - z_0) / sum_i exp(z_i - z_0) over the
 *     selected logits, the sum taken in j order.
 * ws: caller-owned device scratch of at least moe_route_workspace_size(T, K,
 * E_global) bytes (MOE_ERR_BUFFER_TOO_SMALL otherwise); its first int32 is the
 * device status word (cleared by each call; MOE_ERR_TIMEOUT if a bounded wait
 * ran out), readable with moe_read_device_status(ws, ...).  K must be a
 * multiple of 128, E_global <= 1024, topk <= min(64, E_global), T <= 2^30
 * (MOE_ERR_UNSUPPORTED otherwise); all pointers device, 16-byte aligned
 * (MOE_ERR_MISALIGNED); enqueued on stream, graph-capturable (the call
 * encodes its TMA descriptors on the host).  Inputs must be finite. */
int64_t moe_route_workspace_size(int64_t T, int64_t K, int32_t E_global);
moe_status_t moe_router_prepare(const float* w_router, void* w_planes, int64_t E_global, int64_t K, void* stream);
moe_status_t moe_route(const void* x_bf16, const void* w_planes, int64_t T, int64_t K, int32_t E_global,
                       int32_t topk, float* logits, int32_t* topk_ids, float* topk_weights, void* ws,
                       int64_t ws_bytes, void* stream);

/* Weight preparation for MOE_DTYPE_MXFP8, run once at load time: reorders
 * the UE8M0 bytes of an MXFP8 weight tensor from the natural row-major
 * layout src [E, N, C/32] (one byte per row and 32-column block, the OCP
 * microscaling layout) into the packed order the grouped GEMMs copy into
 * tensor memory: for every (e, 128-row block, 128-column group) a 512-byte
 * chunk in which row r's four bytes (its four 32-column blocks, in column
 * order) sit at 16 * (r % 32) + 4 * (r / 32).  src_ld is the byte stride
 * between consecutive scale rows of src: C/32, or more when the scale rows
 * are padded (a multiple of 4) [P1 "关联脉络": padded MXFP8 scale row
 * strides].  dst holds E * N * C/32 bytes and must not overlap src.  N and C
 * must be multiples of 128; device pointers, 16-byte aligned; enqueued on
 * stream. */
moe_status_t moe_pack_mx_scales(const uint8_t* src, int64_t src_ld, uint8_t* dst, int64_t E, int64_t N, int64_t C,
                                void* stream);

/* Number of kernel launches one moe_forward enqueues (for launch accounting). */
int32_t moe_forward_launches(const moe_ctx* ctx);

/* Copy the device status word to *out after synchronising stream (test use;
 * not capturable).  moe_clear_device_status zeroes it (enqueued on stream). */
moe_status_t moe_read_device_status(const void* ws, void* stream, int32_t* out);
moe_status_t moe_clear_device_status(void* ws, void* stream);

/* Fault-detection self-test: launches one kernel that waits on an mbarrier
 * nothing will complete, bounded by timeout_ns; the wait gives up, writes
 * MOE_ERR_TIMEOUT to the workspace status word and the kernel returns
 * normally, leaving the context usable.  Enqueued on stream. */
moe_status_t moe_selftest_wait_timeout(void* ws, int64_t timeout_ns, void* stream);

/* Byte offset, inside an FP8 (1x128) scale region (a_sf or h_sf), of the
 * UE8M0 byte for (row block b, 128-column group g, row r in 0..127) when a
 * row block holds n_groups groups.  Each (block, four consecutive groups)
 * chunk is 512 bytes laid out for the tensor-memory scale copy: row r's word
 * at byte 16*(r%32) + 4*(r/32), group g's scale in its byte g % 4, so that
 * one copy serves the MMAs of four K blocks.  (MXFP8: one chunk per group,
 * the word's bytes its four 32-column scales.)  Host helper for tests. */
int64_t moe_sf_offset(int64_t block, int64_t group, int64_t n_groups, int32_t row);

const char* moe_strerror(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
