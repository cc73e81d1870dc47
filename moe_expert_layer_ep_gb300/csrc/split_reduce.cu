// Second half of a split-K grouped GEMM (masked layouts).
//
// For the masked layout (the expert-parallel decode setting of "Support
// DeepGEMM for standard MoE dispatch" (sglang PR #33128 report), "实现拆解"
// step 2) a few tokens meet many experts, so a tile of 128 rows x 256 columns
// carries few valid rows and the whole K loop of one tile per SM leaves most
// SMs idle.  The grouped GEMM kernel therefore runs each tile's K loop in
// k_splits fixed segments (chosen from K, I and the dtype, never from the
// batch) and writes each segment's fp32 sums of the tile's valid rows to the
// partial buffer.  This kernel adds the segments of every valid row in
// segment order -- ((P0 + P1) + P2) + ... in fp32 -- and applies the stage's
// epilogue with the same arithmetic as the unsplit kernel:
//   stage 1  h = silu(g) * u, stored FP8 with 1x128 UE8M0 scales, MXFP8 with
//            1x32 scales, or bf16 ("Add BF16 support to EP-MoE for DeepGEMM"
//            (sglang PR #17392 report), "关键源码片段" deep_gemm.py)
//   stage 2  y stored bf16
// The sum order of a row depends only on K, I and the dtype, so a token's
// bits are the same at every batch size.
//
// One CTA per (valid 128-row block, column tile) work item, 128 threads:
// stage 1 thread c owns h column c of the tile (gate column c and up column
// 128 + c of the accumulator); stage 2 thread c owns y columns 2c and 2c+1.
// Loads are coalesced across the CTA and all segments of a row are loaded
// before any is added.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRedThreads = 128;

template <bool kFP8, bool kMX>
__global__ void __launch_bounds__(kRedThreads) split_reduce_act_kernel(const GemmArgs g) {
  __shared__ float s_amax[2][4];
  const int c = threadIdx.x, warp = c >> 5, lane = c & 31;
  pdl_wait();
  pdl_trigger();
  const int S = g.k_splits;
  const int64_t plane = g.part_rows * g.part_cols;
  const int64_t n_items = static_cast<int64_t>(g.meta[1]) * g.n_blocks;
  for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int64_t j = it / g.n_blocks;
    const int nb = static_cast<int>(it - j * g.n_blocks);
    const int4 info = reinterpret_cast<const int4*>(g.block_info)[j];
    const int64_t vrow = g.block_vrow[j];
    const int64_t sf_block = static_cast<int64_t>(info.x) * g.blocks_per_expert + (info.z >> 7);
    const int64_t col = static_cast<int64_t>(nb) * 128 + c;
    for (int r = 0; r < info.w; ++r) {
      const float* base = g.partial + (vrow + r) * g.part_cols + static_cast<int64_t>(nb) * 256 + c;
      float gv[kMaxKSplits], uv[kMaxKSplits];
#pragma unroll
      for (int i = 0; i < kMaxKSplits; ++i)
        if (i < S) {
          gv[i] = __ldcg(base + i * plane);
          uv[i] = __ldcg(base + i * plane + 128);
        }
      float gs = gv[0], us = uv[0];
#pragma unroll
      for (int i = 1; i < kMaxKSplits; ++i)
        if (i < S) {
          gs += gv[i];
          us += uv[i];
        }
      const float h = silu_mul(gs, us);
      const int64_t row = static_cast<int64_t>(info.y) + r;
      if (kFP8) {
        // 1x128 group: the whole CTA; MXFP8 1x32 block: one warp
        float amax = fabsf(h);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        if (!kMX) {
          if (lane == 0) s_amax[r & 1][warp] = amax;
          __syncthreads();
          amax = fmaxf(fmaxf(s_amax[r & 1][0], s_amax[r & 1][1]), fmaxf(s_amax[r & 1][2], s_amax[r & 1][3]));
        }
        const int e = ue8m0_exponent(amax);
        static_cast<uint8_t*>(g.out)[row * g.out_ld + col] =
            static_cast<uint8_t>(cvt_e4m3x2(h * exp2_neg(e), 0.0f) & 0xFFu);
        if (kMX) {
          // byte k of the row's scale word: 32-column block k
          uint8_t* sf = g.out_sf + sf_chunk_offset(sf_block, nb, g.out_groups) + sf_row_offset(r);
          if (lane == 0) sf[warp] = static_cast<uint8_t>(e + 127);
        } else if (c == 0) {
          g.out_sf[sf_fp8_offset(sf_block, nb, g.out_groups, r)] = static_cast<uint8_t>(e + 127);
        }
      } else {
        const __nv_bfloat16 v = __float2bfloat16_rn(h);
        static_cast<__nv_bfloat16*>(g.out)[row * g.out_ld + col] = v;
      }
    }
  }
}

__global__ void __launch_bounds__(kRedThreads) split_reduce_y_kernel(const GemmArgs g) {
  const int c = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const int S = g.k_splits;
  const int64_t plane = g.part_rows * g.part_cols;
  const int64_t n_items = static_cast<int64_t>(g.meta[1]) * g.n_blocks;
  for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int64_t j = it / g.n_blocks;
    const int nb = static_cast<int>(it - j * g.n_blocks);
    const int4 info = reinterpret_cast<const int4*>(g.block_info)[j];
    const int64_t vrow = g.block_vrow[j];
    const int64_t col = static_cast<int64_t>(nb) * 256 + 2 * c;
    if (col >= g.n_total) continue;   // (no CTA-wide synchronisation in this kernel)
    for (int r = 0; r < info.w; ++r) {
      const float* base = g.partial + (vrow + r) * g.part_cols + col;
      float2 v[kMaxKSplits];
#pragma unroll
      for (int i = 0; i < kMaxKSplits; ++i)
        if (i < S) v[i] = __ldcg(reinterpret_cast<const float2*>(base + i * plane));
      float2 sum = v[0];
#pragma unroll
      for (int i = 1; i < kMaxKSplits; ++i)
        if (i < S) {
          sum.x += v[i].x;
          sum.y += v[i].y;
        }
      *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(g.out) + (static_cast<int64_t>(info.y) + r) * g.out_ld +
                                   col) = pack_bf16x2(sum.x, sum.y);
    }
  }
}

}  // namespace

cudaError_t launch_split_reduce(const GemmArgs& g, int64_t max_tiles, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  const int grid = static_cast<int>(max_tiles < 1216 ? max_tiles : 1216);
  const dim3 block(kRedThreads);
  if (g.stage == 2) return launch_pdl(split_reduce_y_kernel, dim3(grid), block, 0, s, g);
  if (g.mx) return launch_pdl(split_reduce_act_kernel<true, true>, dim3(grid), block, 0, s, g);
  if (g.fp8) return launch_pdl(split_reduce_act_kernel<true, false>, dim3(grid), block, 0, s, g);
  return launch_pdl(split_reduce_act_kernel<false, false>, dim3(grid), block, 0, s, g);
}

}  // namespace moe
