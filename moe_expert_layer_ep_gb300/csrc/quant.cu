// moe_quant_scatter: token rows -> expert rows, FP8 1x128 UE8M0, MXFP8 1x32
// UE8M0, or BF16.
//
// "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report),
// "实现拆解" step 3: activations are quantised directly with a power-of-two
// (UE8M0) scale rather than quantised with a real scale whose value is
// rounded afterwards.  For each 128-column group the exponent is the smallest
// s with amax <= 448 * 2^s; every element is multiplied by 2^-s (exact) and
// rounded to e4m3 (nearest even, saturating).  MXFP8 applies the same rule
// per 32-column block (the variant listed as uncovered in "风险与影响" item 5).
// "Add BF16 support to EP-MoE for
// DeepGEMM" (sglang PR #17392 report), "实现拆解" step 3: the BF16 path moves
// the rows without scales.
//
// One CTA per token: the row is read once (16-byte loads, 8 columns per
// thread, a 128-column group = 16 consecutive lanes), quantised once, and
// written to each of the token's destination rows (8-byte FP8 / 16-byte BF16
// stores, coalesced per group).
#include "common.cuh"
#include "internal.h"
#include "quant_row.cuh"

namespace moe {

namespace {

template <bool kFP8, bool kMX>
__global__ void __launch_bounds__(kQuantThreads) quant_scatter_kernel(QuantArgs q) {
  __shared__ int64_t s_dst[kMaxTopk];
  __shared__ int64_t s_blk[kMaxTopk];
  __shared__ int s_row[kMaxTopk];
  __shared__ int s_any;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid == 0) s_any = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  if (tid < q.topk) {
    const int64_t d = q.src2dst[t * q.topk + tid];
    s_dst[tid] = d;
    if (d >= 0) {
      s_any = 1;
      dest_block(q, d, &s_blk[tid], &s_row[tid]);
    }
  }
  __syncthreads();
  if (!s_any) return;
  quant_scatter_row<kFP8, kMX>(q, t, s_dst, s_blk, s_row, tid);
}


constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs c) {
  __shared__ int64_t s_dst[kMaxTopk];
  __shared__ float s_w[kMaxTopk];
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (tid < c.topk) {
    s_dst[tid] = c.src2dst[t * c.topk + tid];
    s_w[tid] = c.topk_weights[t * c.topk + tid];
  }
  __syncthreads();
  const uint16_t* y = static_cast<const uint16_t*>(c.y);
  uint16_t* orow = static_cast<uint16_t*>(c.out) + t * c.K;
  for (int64_t col = static_cast<int64_t>(tid) * 8; col < c.K; col += kCombineThreads * 8) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < c.topk; j0 += 8) {
      uint4 v[8];
      // issue all loads of the batch before using them
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        v[jj] = make_uint4(0, 0, 0, 0);
        if (j < c.topk && s_dst[j] >= 0) v[jj] = *reinterpret_cast<const uint4*>(y + s_dst[j] * c.K + col);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        if (j < c.topk && s_dst[j] >= 0) {
          const float w = s_w[j];
          const float2 p0 = unpack_bf16x2(v[jj].x), p1 = unpack_bf16x2(v[jj].y), p2 = unpack_bf16x2(v[jj].z),
                       p3 = unpack_bf16x2(v[jj].w);
          acc[0] = fmaf(w, p0.x, acc[0]);
          acc[1] = fmaf(w, p0.y, acc[1]);
          acc[2] = fmaf(w, p1.x, acc[2]);
          acc[3] = fmaf(w, p1.y, acc[3]);
          acc[4] = fmaf(w, p2.x, acc[4]);
          acc[5] = fmaf(w, p2.y, acc[5]);
          acc[6] = fmaf(w, p3.x, acc[6]);
          acc[7] = fmaf(w, p3.y, acc[7]);
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(orow + col) = o;
  }
}

}  // namespace

cudaError_t launch_quant_scatter(const QuantArgs& q, cudaStream_t s) {
  if (q.T <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(q.T)), block(kQuantThreads);
  if (q.mx) return launch_pdl(quant_scatter_kernel<true, true>, grid, block, 0, s, q);
  if (q.fp8) return launch_pdl(quant_scatter_kernel<true, false>, grid, block, 0, s, q);
  return launch_pdl(quant_scatter_kernel<false, false>, grid, block, 0, s, q);
}

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t s) {
  if (c.T <= 0) return cudaSuccess;
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(c.T)), dim3(kCombineThreads), 0, s, c);
}

}  // namespace moe
