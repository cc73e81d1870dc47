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

namespace moe {

namespace {

constexpr int kQuantThreads = 256;
constexpr int kColsPerIter = kQuantThreads * 8;
constexpr int kLoadBatch = 4;

__device__ __forceinline__ void dest_block(const QuantArgs& q, int64_t d, int64_t* block, int* row) {
  if (!q.masked) {
    *block = d >> 7;
    *row = static_cast<int>(d & 127);
  } else {
    const int64_t e = d / q.max_m;
    const int64_t pos = d - e * q.max_m;
    *block = e * q.blocks_per_expert + (pos >> 7);
    *row = static_cast<int>(pos & 127);
  }
}

// One token row: read once (16-byte loads, 8 columns per thread), quantised
// once, written to each destination row listed in s_dst (-1: none).
// kMX: MXFP8, one exponent per 32 columns (4 lanes); the four exponents of a
// 128-column group fill the four bytes of the row's scale word.
template <bool kFP8, bool kMX>
__device__ __forceinline__ void quant_scatter_row(const QuantArgs& q, int64_t t, const int64_t* s_dst,
                                                  const int64_t* s_blk, const int* s_row) {
  const int tid = threadIdx.x;
  const uint16_t* xrow = static_cast<const uint16_t*>(q.x) + t * q.K;
  const int64_t n_groups = q.K / 128;
  // kLoadBatch row segments per thread are loaded before any is used
  for (int64_t c1 = 0; c1 < q.K; c1 += kLoadBatch * kColsPerIter) {
    uint4 vb[kLoadBatch];
#pragma unroll
    for (int b = 0; b < kLoadBatch; ++b) {
      const int64_t col = c1 + b * kColsPerIter + static_cast<int64_t>(tid) * 8;
      vb[b] = make_uint4(0, 0, 0, 0);
      if (col < q.K) vb[b] = __ldg(reinterpret_cast<const uint4*>(xrow + col));
    }
#pragma unroll
    for (int b = 0; b < kLoadBatch; ++b) {
      const int64_t c0 = c1 + b * kColsPerIter;
      if (c0 >= q.K) break;                 // uniform over the CTA
      const int64_t col = c0 + static_cast<int64_t>(tid) * 8;
      const bool active = col < q.K;
      const uint4 v = vb[b];
      if constexpr (kFP8) {
        float f[8];
        const float2 p0 = unpack_bf16x2(v.x), p1 = unpack_bf16x2(v.y), p2 = unpack_bf16x2(v.z),
                     p3 = unpack_bf16x2(v.w);
        f[0] = p0.x; f[1] = p0.y; f[2] = p1.x; f[3] = p1.y;
        f[4] = p2.x; f[5] = p2.y; f[6] = p3.x; f[7] = p3.y;
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        // 16 lanes = one 128-column group (MXFP8: 4 lanes = one 32-column block)
#pragma unroll
        for (int o = kMX ? 2 : 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const int s = ue8m0_exponent(amax);
        uint32_t sf_word = static_cast<uint32_t>(s + 127);
        if constexpr (kMX) {
          const int lane = tid & 31;
          const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(s + 127), lane + 4);
          const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(s + 127), lane + 8);
          const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(s + 127), lane + 12);
          sf_word = static_cast<uint32_t>(s + 127) | (b1 << 8) | (b2 << 16) | (b3 << 24);   // valid at group leads
        }
        const float mul = exp2_neg(s);
        uint2 packed;
        packed.x = cvt_e4m3x2(f[0] * mul, f[1] * mul) | (cvt_e4m3x2(f[2] * mul, f[3] * mul) << 16);
        packed.y = cvt_e4m3x2(f[4] * mul, f[5] * mul) | (cvt_e4m3x2(f[6] * mul, f[7] * mul) << 16);
        if (active) {
          const int64_t group = col >> 7;
          const bool group_lead = (tid & 15) == 0;
          for (int j = 0; j < q.topk; ++j) {
            const int64_t d = s_dst[j];
            if (d < 0) continue;
            uint8_t* arow = static_cast<uint8_t*>(q.a) + d * q.K;
            *reinterpret_cast<uint2*>(arow + col) = packed;
            if (group_lead) {
              if (kMX)   // the group's four 32-column scales, one word
                *reinterpret_cast<uint32_t*>(q.a_sf + sf_chunk_offset(s_blk[j], group, n_groups) +
                                             sf_row_offset(s_row[j])) = sf_word;
              else       // the group's byte of its four-group word
                q.a_sf[sf_fp8_offset(s_blk[j], group, n_groups, s_row[j])] = static_cast<uint8_t>(sf_word);
            }
          }
        }
      } else {
        if (active) {
          for (int j = 0; j < q.topk; ++j) {
            const int64_t d = s_dst[j];
            if (d < 0) continue;
            uint16_t* arow = static_cast<uint16_t*>(q.a) + d * q.K;
            *reinterpret_cast<uint4*>(arow + col) = v;
          }
        }
      }
    }
  }
}

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
  quant_scatter_row<kFP8, kMX>(q, t, s_dst, s_blk, s_row);
}

// Small problems inside moe_forward (at most kPlanSmallMaxA assignments and
// kPlanSmallMaxE local experts): each CTA forms its token's destination rows
// itself, by the plan's rule (the stable rank of the assignment among its
// expert's assignments in flattened t * topk + j order; compact: after the
// earlier experts' 128-padded segments; masked: e * max_m + rank, dropped
// past max_m), so it runs beside the one-CTA plan instead of after it.  It
// waits for the plan to complete only before it finishes, so the kernels
// after it see the plan's tables complete.
template <bool kFP8, bool kMX>
__global__ void __launch_bounds__(kQuantThreads) quant_scatter_small_kernel(QuantArgs q) {
  __shared__ int16_t s_lid[kPlanSmallMaxA];   // local expert of every assignment, -1: not local
  __shared__ int s_cnt[kPlanSmallMaxE];       // compact: assignments per local expert
  __shared__ int64_t s_dst[kMaxTopk];
  __shared__ int64_t s_blk[kMaxTopk];
  __shared__ int s_row[kMaxTopk];
  __shared__ int s_any;
  const int64_t t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t A = q.T * q.topk;
  for (int x = tid; x < q.E_local; x += kQuantThreads) s_cnt[x] = 0;
  if (tid == 0) s_any = 0;
  __syncthreads();
  for (int64_t i = tid; i < A; i += kQuantThreads) {
    const int32_t gid = q.topk_ids[i];
    const int e = (gid >= 0 && gid < q.E_global) ? gid - q.expert_start : -1;
    const int lid = (e >= 0 && e < q.E_local) ? e : -1;
    s_lid[i] = static_cast<int16_t>(lid);
    if (!q.masked && lid >= 0) atomicAdd(&s_cnt[lid], 1);
  }
  __syncthreads();
  for (int j = warp; j < q.topk; j += kQuantThreads / 32) {
    const int64_t pos = t * q.topk + j;
    const int e = s_lid[pos];
    int rank = 0;
    if (e >= 0)
      for (int64_t i = lane; i < pos; i += 32) rank += s_lid[i] == e;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
    if (lane == 0) {
      int64_t d = -1;
      if (e >= 0) {
        if (q.masked) {
          if (rank < q.max_m) d = static_cast<int64_t>(e) * q.max_m + rank;
        } else {
          int64_t start = 0;
          for (int x = 0; x < e; ++x) start += (s_cnt[x] + kBlockM - 1) / kBlockM * kBlockM;
          d = start + rank;
        }
      }
      s_dst[j] = d;
      if (d >= 0) {
        s_any = 1;
        dest_block(q, d, &s_blk[j], &s_row[j]);
      }
    }
  }
  __syncthreads();
  if (s_any) quant_scatter_row<kFP8, kMX>(q, t, s_dst, s_blk, s_row);
  // finish only after the plan (the previous kernel) has completed
  pdl_wait();
  pdl_trigger();
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
  if (q.topk_ids && plan_is_small(q.T * q.topk, q.E_local)) {
    if (q.mx) return launch_pdl(quant_scatter_small_kernel<true, true>, grid, block, 0, s, q);
    if (q.fp8) return launch_pdl(quant_scatter_small_kernel<true, false>, grid, block, 0, s, q);
    return launch_pdl(quant_scatter_small_kernel<false, false>, grid, block, 0, s, q);
  }
  if (q.mx) return launch_pdl(quant_scatter_kernel<true, true>, grid, block, 0, s, q);
  if (q.fp8) return launch_pdl(quant_scatter_kernel<true, false>, grid, block, 0, s, q);
  return launch_pdl(quant_scatter_kernel<false, false>, grid, block, 0, s, q);
}

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t s) {
  if (c.T <= 0) return cudaSuccess;
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(c.T)), dim3(kCombineThreads), 0, s, c);
}

}  // namespace moe
