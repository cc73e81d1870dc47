// Per-token quantise-and-scatter device code, shared by the quant-scatter
// kernels (quant.cu) and the one-launch plan + quant-scatter of small
// problems (plan.cu).  See quant.cu for the method and its citations.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

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

// One token row, by kQuantThreads threads (tid: the thread's index among
// them): read once (16-byte loads, 8 columns per thread), quantised once,
// written to each destination row listed in s_dst (-1: none).
// kMX: MXFP8, one exponent per 32 columns (4 lanes); the four exponents of a
// 128-column group fill the four bytes of the row's scale word.
template <bool kFP8, bool kMX>
__device__ __forceinline__ void quant_scatter_row(const QuantArgs& q, int64_t t, const int64_t* s_dst,
                                                  const int64_t* s_blk, const int* s_row, int tid) {
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

// Small problems (at most kPlanSmallMaxA assignments and kPlanSmallMaxE local
// experts): a token's destination rows formed from the routing by the plan's
// rule -- the stable rank of the assignment among its expert's assignments in
// flattened t * topk + j order; compact: after the earlier experts'
// 128-padded segments; masked: e * max_m + rank, dropped past max_m -- so the
// quantisation need not wait for the plan.  The caller's threads (nthreads of
// them, tid the thread's index) first fill s_lid (local expert of every
// assignment, -1: not local) and s_cnt (compact: assignments per local
// expert) with fill_routing, synchronise, then give each (token, j) to one
// warp with token_destination.
__device__ __forceinline__ void fill_routing(const QuantArgs& q, int16_t* s_lid, int* s_cnt, int tid, int nthreads) {
  const int64_t A = q.T * q.topk;
  for (int64_t i = tid; i < A; i += nthreads) {
    const int32_t gid = q.topk_ids[i];
    const int e = (gid >= 0 && gid < q.E_global) ? gid - q.expert_start : -1;
    const int lid = (e >= 0 && e < q.E_local) ? e : -1;
    s_lid[i] = static_cast<int16_t>(lid);
    if (!q.masked && lid >= 0) atomicAdd(&s_cnt[lid], 1);
  }
}

// Destination row of assignment (t, j), -1 when none; called by a whole warp.
__device__ __forceinline__ int64_t token_destination(const QuantArgs& q, const int16_t* s_lid, const int* s_cnt,
                                                     int64_t t, int j, int lane) {
  const int64_t pos = t * q.topk + j;
  const int e = s_lid[pos];
  int rank = 0;
  if (e >= 0)
    for (int64_t i = lane; i < pos; i += 32) rank += s_lid[i] == e;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
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
  return d;
}

}  // namespace moe
