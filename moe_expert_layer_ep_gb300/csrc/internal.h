// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

// Launch a layer kernel with programmatic dependent launch allowed (it may
// start while the stream's previous kernel runs; see pdl_wait in
// common.cuh).  Inside a stream capture this becomes a programmatic edge of
// the graph.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl for a kernel launched in clusters of cluster_x CTAs.
template <typename... Params, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               int cluster_x, Args&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kPlanChunk = 256;   // assignments per plan CTA (8 warps x 32)
constexpr int kMaxLocalExperts = 1024;
constexpr int kMaxTopk = 64;
constexpr int kBlockM = 128;      // rows per expert block == compact block_e
constexpr int kMaxRouterExperts = 1024;
constexpr int kRouterSegment = 1024;     // K elements per router segment sum (fixed, batch-independent)
constexpr int kMaxKSplits = 8;           // K segments of a masked-layout GEMM tile, at most

struct PlanArgs {
  const int32_t* topk_ids;  // [A]
  int64_t A;                // T * topk
  int32_t E_global, E_local, expert_start;
  int32_t masked;           // 0 compact, 1 masked
  int64_t max_m;            // masked rows per expert
  int64_t all_tokens;       // compact static bound
  int32_t blocks_per_expert;  // masked: ceil(max_m / 128)
  int32_t chunks;
  int32_t* status;
  int32_t* meta;
  int32_t* counts;
  int32_t* padded;
  int32_t* start;
  int32_t* masked_m;
  int32_t* m_indices;
  int32_t* src2dst;
  int32_t* block_info;      // int4 per block
  int32_t* chunk_hist;      // [E_local, chunks]
  int32_t* chunk_rank;      // [A]
  int32_t* block_vrow;      // masked, optional: [blocks] first valid-row index of each block
  int32_t clear_status;     // the one-CTA plan clears the status word itself (no memset launch)
};

struct QuantArgs {
  const void* x;            // bf16 [T, K]
  const int32_t* src2dst;   // [T, topk]
  // small problems (plan_is_small): the kernel forms each token's
  // destinations itself from the routing, by the plan's rule
  const int32_t* topk_ids;  // [T, topk]
  int32_t E_global, E_local, expert_start;
  int64_t T, K;
  int32_t topk;
  int32_t fp8;
  int32_t mx;               // fp8 with 1x32 scales (MXFP8)
  int32_t masked;
  int64_t max_m;
  int32_t blocks_per_expert;
  void* a;                  // fp8 or bf16 [rows, K]
  uint8_t* a_sf;            // scale chunks
};

struct CombineArgs {
  const void* y;            // bf16 [rows, K]
  const int32_t* src2dst;
  const float* topk_weights;
  int64_t T, K;
  int32_t topk;
  void* out;                // bf16 [T, K]
};

// One grouped GEMM launch (either stage).
struct GemmArgs {
  const int32_t* block_info;  // int4 {expert, row0, tma_row0, valid}
  const int32_t* meta;        // meta[1] = valid blocks
  int32_t* status;
  int32_t stage;              // 1: w13 + SiLU*up, 2: w2
  int32_t fp8;
  int32_t mx;                 // fp8 with 1x32 scales; w_sf in the packed chunk order
  int32_t fp4;                // mx with FP4 (E2M1) weights, packed two per byte: an E2M1 MMA operand
  int32_t masked;
  int32_t blocks_per_expert;  // masked
  int32_t n_blocks;           // output column blocks (128 h columns, or 256 y columns)
  int32_t k_blocks;           // 128-byte K blocks of the reduction
  int64_t n_half;             // stage 1: I (row offset of the up projection in w13)
  int64_t n_total;            // output columns (I for stage 1, K for stage 2)
  int32_t w_rows_blocks;      // weight rows / 128 (for the weight-scale table)
  int32_t w_k_groups;         // reduction / 128 (weight-scale table)
  const uint8_t* a_sf;        // fp8: activation scale chunks
  const uint8_t* w_sf;        // fp8: weight scales [E, rows/128, red/128]; mxfp8: packed 512-byte chunks
  void* out;                  // h (stage 1) or y (stage 2)
  int64_t out_ld;             // output row stride in elements
  uint8_t* out_sf;            // stage 1 fp8: h scale chunks
  int32_t out_groups;         // stage 1 fp8: I / 128
  uint64_t timeout_ns;
  // Split K (masked layouts): each tile's K loop runs in k_splits fixed
  // segments; segment s writes the tile's valid rows' fp32 sums to
  // partial[s][row][col] and launch_split_reduce then adds the segments in
  // order and applies the stage's epilogue.
  int32_t k_splits;           // 1: no split
  int32_t max_m;              // masked rows per expert
  const int32_t* block_vrow;  // [blocks] first valid-row index of each block
  float* partial;             // [k_splits][part_rows][part_cols]
  int64_t part_rows;
  int64_t part_cols;          // n_blocks * 256
  // Column-block pairs (compact layout, no split, even n_blocks): launched in
  // clusters of two CTAs that always hold the same row block's column blocks
  // 2m and 2m + 1; each CTA loads one 64-row half of the shared A tile and
  // multicasts it to both.  The A map's box is then 64 rows.
  int32_t pair;
};

// Problems the one-CTA plan handles: at most kPlanSmallMaxA assignments and
// kPlanSmallMaxE local experts.
constexpr int kPlanSmallMaxA = 2048;
constexpr int kPlanSmallMaxE = 256;
inline bool plan_is_small(int64_t A, int32_t E_local) { return A <= kPlanSmallMaxA && E_local <= kPlanSmallMaxE; }
cudaError_t launch_plan(const PlanArgs& p, cudaStream_t s);
int plan_launch_count(int64_t A, int32_t E_local);   // kernels one launch_plan enqueues
cudaError_t launch_quant_scatter(const QuantArgs& q, cudaStream_t s);
// moe_forward's first step for small problems (plan_is_small, with q.topk_ids
// set): the one-CTA plan and the quant-scatter in one launch.
cudaError_t launch_plan_quant_small(const PlanArgs& p, const QuantArgs& q, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs& c, cudaStream_t s);
// Tensor maps of one grouped-GEMM launch.
struct GemmMaps {
  CUtensorMap a;     // A rows (a or h); 64-row boxes when g.pair
  CUtensorMap b;     // weights: w13 as [E][gate, up][I/128][128][K] (one box = a tile's gate and up
                     // rows), w2 as [E][K][I] in 256-row boxes
  CUtensorMap out;   // GEMM2: y, 32-column store boxes
  CUtensorMap wsf;   // MXFP8 / MXFP4: packed weight-scale chunks, a tile's two chunks per box
};
cudaError_t launch_gemm(const GemmArgs& g, const GemmMaps& maps, int grid, cudaStream_t s);
// CTAs of a pair launch (g.pair) that can be resident at once: twice the
// device's co-resident two-CTA clusters of the kernel g selects (0 when the
// query fails).
int gemm_pair_ctas(const GemmArgs& g);
// After a split-K GEMM launch: adds each valid row's segment sums in segment
// order and writes h (stage 1: SiLU*up, then FP8 / MXFP8 / bf16 storage) or y
// (stage 2: bf16).  max_tiles: the static bound on the launch's tiles.
cudaError_t launch_split_reduce(const GemmArgs& g, int64_t max_tiles, cudaStream_t s);
cudaError_t launch_requant(const uint8_t* w_in, const float* s_in, uint8_t* w_out, uint8_t* s_out, int64_t E,
                           int64_t N, int64_t C, cudaStream_t s);
cudaError_t launch_pack_mx_scales(const uint8_t* src, int64_t src_ld, uint8_t* dst, int64_t E, int64_t N, int64_t C,
                                  cudaStream_t s);
struct RouterArgs {
  int64_t T, K;
  int32_t E;
  int32_t segs;             // ceil(K / kRouterSegment)
  int32_t m_tiles, n_tiles; // ceil(T / 128), ceil(E / 128)
  int32_t fold;             // 1: one work item per tile, its segments added in the CTA
  float* partial;           // fold == 0: [segs, T, E] fp32 segment sums
  float* z;                 // fold == 1: the logits [T, E]
  int32_t* status;          // int32[4], cleared by the launch
  uint64_t timeout_ns;
};
// Router work items: when the 128 x 128 tiles fill at least three quarters of
// the SMs, a CTA takes a whole tile and adds its segments itself (the
// partial buffer goes unused); with fewer tiles, every segment of every tile
// is its own item, for parallelism.  Either way the same segment sums are
// added in the same order.
inline bool router_folds(int64_t T, int64_t E, int sms) {
  return ((T + 127) / 128) * ((E + 127) / 128) * 4 >= static_cast<int64_t>(sms) * 3;
}

cudaError_t launch_router_split(const float* w, uint16_t* planes, int64_t E, int64_t K, cudaStream_t s);
cudaError_t launch_route(const CUtensorMap& map_x, const CUtensorMap& map_w, const RouterArgs& r, int grid, int topk,
                         float* logits, int32_t* ids, float* wts, cudaStream_t s);
cudaError_t launch_selftest_wait(int32_t* status, uint64_t timeout_ns, cudaStream_t s);


}  // namespace moe
