// moe_route: the fp32 MoE router that feeds the layer its top-k expert ids
// and weights.
//
// "[Feature] Support BF16 and batch-invariant inference with DeepEP v2"
// (sglang PR #38160 report), section "关联脉络": the router GEMM is kept in
// fp32 so that expert selection does not flip under deterministic inference;
// "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report),
// "关键源码片段" deep_gemm.py: the layer consumes standard top-k ids/weights.
//
// The fp32 GEMM runs on the tensor cores.  At load time every fp32 weight is
// split into three bf16 planes with hi + mid + lo == w exactly
// (router_split_kernel); x is bf16, so each product x * plane is exact in the
// fp32 accumulator and z = x.hi + x.mid + x.lo is the fp32-accumulated fp32
// product.
//   router_logits_tc_kernel  persistent, TMA-fed tcgen05 kernel over 128-token
//                            x 128-expert tiles; each tile's K runs in fixed
//                            1024-wide segments, 12 bf16 MMAs per 64-wide K
//                            block into a TMEM accumulator per segment, and
//                            the logits are the segment sums added in order,
//                            z = ((P0 + P1) + P2) + ... in fp32.  Work items:
//                            fewer tiles than about the SMs (small batches):
//                            one segment of one tile, the segment sums going
//                            to a partial buffer for the top-k kernel to add;
//                            more: a whole tile, its segments added in
//                            registers as they complete and z written
//                            directly.  The same operations in the same order
//                            either way.
//   topk_softmax_kernel      one warp per token: folds the partials in
//                            segment order into the logits (or reads them),
//                            then k rounds of a warp argmax (larger logit
//                            wins, equal logits go to the lower expert id),
//                            then w_j = exp(z_j - z_max) / sum, the sum in j
//                            order.
// Tiles, segments and the fold order do not depend on the batch, so a
// token's logits, ids and weights are the same bits at every batch size.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRtTileM = 128;                   // tokens per tile
constexpr int kRtTileN = 128;                   // experts per tile
constexpr int kRtKBlock = 64;                   // bf16 elements of K per stage (one 128-byte swizzle row)
constexpr int kRtStages = 3;
constexpr int kRtPlanes = 3;
constexpr int kRtABytes = kRtTileM * 128;                  // 16 KB
constexpr int kRtBPlaneBytes = kRtTileN * 128;             // 16 KB per plane
constexpr int kRtBBytes = kRtPlanes * kRtBPlaneBytes;      // 48 KB
constexpr int kRtOffA = 0;
constexpr int kRtOffB = kRtOffA + kRtStages * kRtABytes;
constexpr int kRtOffBar = kRtOffB + kRtStages * kRtBBytes;
constexpr int kRtNumBars = 2 * kRtStages + 2 + 2 + 1;
constexpr int kRtOffHolder = kRtOffBar + kRtNumBars * 8;
constexpr int kRtOffAbort = kRtOffHolder + 8;
constexpr int kRtSmemBytes = kRtOffAbort + 8 + 1024;      // + 1024-byte alignment slack
constexpr uint32_t kRtTmemCols = 2 * kRtTileN;             // two accumulators
constexpr int kRtEpiWarps = 8;                             // two per lane quadrant, 64 columns each
constexpr int kRtThreads = 64 + 32 * kRtEpiWarps;          // producer, MMA, epilogue warps
constexpr uint32_t kRtIdesc = (1u << 4)                    // D f32
                              | (1u << 7) | (1u << 10)     // A, B bf16
                              | (static_cast<uint32_t>(kRtTileN >> 3) << 17) |
                              (static_cast<uint32_t>(kRtTileM >> 4) << 24);
static_assert(kRtSmemBytes <= 227 * 1024, "shared memory");

// A work item: tile (mt, nt) and its segments [seg0, seg1) -- one segment
// when the partials go to memory, all of them when the tile is folded in
// the CTA (r.fold).
struct RtItem {
  int mt, nt, seg0, seg1;
};

__device__ __forceinline__ RtItem rt_item(const RouterArgs& r, int64_t i) {
  RtItem it;
  const int per = r.fold ? 1 : r.segs;   // items per tile
  it.seg0 = r.fold ? 0 : static_cast<int>(i % per);
  it.seg1 = r.fold ? r.segs : it.seg0 + 1;
  const int64_t tile = i / per;
  it.nt = static_cast<int>(tile % r.n_tiles);
  it.mt = static_cast<int>(tile / r.n_tiles);
  return it;
}

// K blocks [kb0, kb0 + nkb) of segment seg.
__device__ __forceinline__ void seg_blocks(const RouterArgs& r, int seg, int* kb0, int* nkb) {
  constexpr int kPerSeg = kRouterSegment / kRtKBlock;
  *kb0 = seg * kPerSeg;
  *nkb = min(kPerSeg, static_cast<int>(r.K / kRtKBlock) - *kb0);
}

// Per segment of a work item: per 64-wide K block, 4 K-steps x 3 weight
// planes = 12 MMAs in the fixed order (step, plane), all into one fp32
// accumulator (two accumulators alternate between consecutive segments).  The
// segment's sums go to partial[seg][t][e], or (r.fold) are added to the
// thread's running row of 128 logits.  A token's partials are the same
// operations whatever the batch (tile rows are independent), and so are the
// folded logits.
__global__ void __launch_bounds__(kRtThreads, 1)
    router_logits_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                            const RouterArgs r) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRtOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kRtStages;
  uint64_t* tfull = bars + 2 * kRtStages;
  uint64_t* tempty = bars + 2 * kRtStages + 2;
  uint64_t* done = bars + 2 * kRtStages + 4;
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + kRtOffHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kRtOffAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 32 * kRtEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_x);
    prefetch_tensormap(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(holder, kRtTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  // x may come from the previous kernel of the stream; the partial buffer
  // may still be read by the previous call's top-k kernel
  pdl_wait();
  pdl_trigger();
  const int64_t n_items = static_cast<int64_t>(r.m_tiles) * r.n_tiles * (r.fold ? 1 : r.segs);

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const RtItem it = rt_item(r, i);
        int kb0, nkb, kb_last, nkb_last;
        seg_blocks(r, it.seg0, &kb0, &nkb);
        seg_blocks(r, it.seg1 - 1, &kb_last, &nkb_last);
        const int kb_end = kb_last + nkb_last;
        for (int kb = kb0; kb < kb_end && ok; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, r.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kRtABytes + kRtBBytes);
          const int kc = kb * kRtKBlock;
          tma_load_3d(smem + kRtOffA + stage * kRtABytes, &map_x, &full[stage], kc, it.mt * kRtTileM, 0);
          for (int p = 0; p < kRtPlanes; ++p)
            tma_load_3d(smem + kRtOffB + stage * kRtBBytes + p * kRtBPlaneBytes, &map_w, &full[stage], kc,
                        it.nt * kRtTileN, p);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kRtStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        set_status(r.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // never leave the CTA with bulk copies still landing in its shared memory
      const int never = 0;
      for (int s = 0; s < kRtStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, &never, r.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0;
      bool ok = true;
      for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const RtItem it = rt_item(r, i);
        for (int seg = it.seg0; seg < it.seg1 && ok; ++seg, ++iter) {
          const int acc = iter & 1;
          if (!mbar_wait_bounded(&tempty[acc], ((iter >> 1) & 1) ^ 1, abort_flag, r.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kRtTileN);
          int kb0, nkb;
          seg_blocks(r, seg, &kb0, &nkb);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait_bounded(&full[stage], phase, abort_flag, r.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a_desc = smem_desc(smem_u32(smem + kRtOffA + stage * kRtABytes), 16, 1024, kSwizzle128B);
            const uint32_t b_addr = smem_u32(smem + kRtOffB + stage * kRtBBytes);
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int p = 0; p < kRtPlanes; ++p)
                mma_bf16(d_tmem, a_desc + 2 * k,
                         smem_desc(b_addr + p * kRtBPlaneBytes, 16, 1024, kSwizzle128B) + 2 * k, kRtIdesc,
                         (kb | k | p) != 0);
            tc_commit(&empty[stage]);
            if (++stage == kRtStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc_commit(&tfull[acc]);
        }
      }
      if (!ok) {
        set_status(r.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      tc_commit(done);
      const int never = 0;
      mbar_wait_bounded(done, 0, &never, r.timeout_ns);
    }
  } else {
    const int quad = warp & 3;            // tensor-memory lane quadrant this warp may read
    const int half = (warp - 2) >> 2;     // columns [64 half, 64 half + 64) of the tile
    constexpr int kCols = kRtTileN / 2;
    int iter = 0;
    bool failed = false;
    for (int64_t i = blockIdx.x; i < n_items && !failed; i += gridDim.x) {
      const RtItem it = rt_item(r, i);
      const int64_t t = static_cast<int64_t>(it.mt) * kRtTileM + quad * 32 + lane;
      float run[kCols];   // r.fold: this row's logits so far in this warp's columns, ((P0 + P1) + ...)
      for (int seg = it.seg0; seg < it.seg1; ++seg, ++iter) {
        const int acc = iter & 1;
        const bool got = mbar_wait_bounded(&tfull[acc], (iter >> 1) & 1, abort_flag, r.timeout_ns);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          set_status(r.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + static_cast<uint32_t>(acc * kRtTileN + half * kCols) +
                               (static_cast<uint32_t>(quad * 32) << 16);
        if (r.fold) {
          const bool first = seg == it.seg0;
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(taddr + c * 32, v);
            tmem_ld_wait();
            if (c == kCols / 32 - 1) {
              tc_fence_before();
              mbar_arrive(&tempty[acc]);
            }
            if (first) {
#pragma unroll
              for (int j = 0; j < 32; ++j) run[c * 32 + j] = __uint_as_float(v[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) run[c * 32 + j] += __uint_as_float(v[j]);
            }
          }
          continue;
        }
        float* dst = r.partial + (static_cast<int64_t>(seg) * r.T + t) * r.E;
#pragma unroll 1
        for (int c = 0; c < kCols / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + c * 32, v);
          tmem_ld_wait();
          if (c == kCols / 32 - 1) {
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
          }
          const int e0 = it.nt * kRtTileN + half * kCols + c * 32;
          if (t < r.T && e0 < r.E) {
            if (e0 + 32 <= r.E && (r.E & 3) == 0) {
              float4* d4 = reinterpret_cast<float4*>(dst + e0);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                d4[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                    __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (e0 + j < r.E) dst[e0 + j] = __uint_as_float(v[j]);
            }
          }
        }
      }
      if (failed || !r.fold || t >= r.T) continue;
      float* zrow = r.z + t * r.E;
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        const int e0 = it.nt * kRtTileN + half * kCols + c * 32;
        if (e0 + 32 <= r.E && (r.E & 3) == 0) {
          float4* d4 = reinterpret_cast<float4*>(zrow + e0);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            d4[j] = make_float4(run[c * 32 + 4 * j], run[c * 32 + 4 * j + 1], run[c * 32 + 4 * j + 2],
                                run[c * 32 + 4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (e0 + j < r.E) zrow[e0 + j] = run[c * 32 + j];
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kRtTmemCols);
  }
}

// Load-time split of fp32 router weights into three bf16 planes with
// hi + mid + lo == w exactly (each residual is exact in fp32 and the last
// one has at most 8 significant bits) for |w| >= 2^-110.
__global__ void __launch_bounds__(256) router_split_kernel(const float4* w, uint2* hi, uint2* mid, uint2* lo,
                                                           int64_t n4) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = w[i];
  const float in[4] = {v.x, v.y, v.z, v.w};
  uint32_t h[4], m[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat16 b1 = __float2bfloat16_rn(in[j]);
    const float r1 = in[j] - __bfloat162float(b1);
    const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(b2);
    const __nv_bfloat16 b3 = __float2bfloat16_rn(r2);
    h[j] = __bfloat16_as_ushort(b1);
    m[j] = __bfloat16_as_ushort(b2);
    l[j] = __bfloat16_as_ushort(b3);
  }
  hi[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  mid[i] = make_uint2(m[0] | (m[1] << 16), m[2] | (m[3] << 16));
  lo[i] = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

// P logits per lane (E <= 32 P).  The j-th selection is kept by lane j % 32
// (slot j / 32), so nothing is indexed dynamically; every lane forms the same
// softmax sum in j order from broadcasts, and lane j writes output j.
template <int P>
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* partial, int segs, int64_t T, int E,
                                                           int topk, float* z, int32_t* ids, float* wts) {
  static_assert(P <= 32, "taken mask is 32 bits");
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_wait();      // the logits kernel's partial sums are complete and visible
  pdl_trigger();
  if (t >= T) return;
  float v[P];
  // logits = the segments' partial sums folded in segment order; the loads
  // of kBatch segments are all issued before any of them is added
  constexpr int kBatch = P >= 32 ? 1 : 32 / P;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? partial[t * E + e] : -INFINITY;
  }
  for (int sg = 1; sg < segs; sg += kBatch) {
    float p[kBatch][P];
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const int e = lane + 32 * i;
        p[q][i] = (sg + q < segs && e < E) ? partial[(static_cast<int64_t>(sg + q) * T + t) * E + e] : 0.0f;
      }
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
#pragma unroll
      for (int i = 0; i < P; ++i)
        if (sg + q < segs && lane + 32 * i < E) v[i] += p[q][i];
  }
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int e = lane + 32 * i;
    if (e < E) z[t * E + e] = v[i];
  }
  uint32_t taken = 0;      // bit i: element lane + 32 i already selected
  float my_v0 = 0.0f, my_v1 = 0.0f;
  int my_e0 = 0, my_e1 = 0;
  for (int j = 0; j < topk; ++j) {
    float bv = -INFINITY;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == (j & 31)) {
      if (j < 32) {
        my_v0 = bv;
        my_e0 = be;
      } else {
        my_v1 = bv;
        my_e1 = be;
      }
    }
  }
  const float zmax = __shfl_sync(0xFFFFFFFFu, my_v0, 0);   // the first selection is the largest
  float sum = 0.0f;
  for (int j = 0; j < topk; ++j) sum += expf(__shfl_sync(0xFFFFFFFFu, j < 32 ? my_v0 : my_v1, j & 31) - zmax);
  if (lane < topk) {
    ids[t * topk + lane] = my_e0;
    wts[t * topk + lane] = expf(my_v0 - zmax) / sum;
  }
  if (lane + 32 < topk) {
    ids[t * topk + lane + 32] = my_e1;
    wts[t * topk + lane + 32] = expf(my_v1 - zmax) / sum;
  }
}

}  // namespace

cudaError_t launch_router_split(const float* w, uint16_t* planes, int64_t E, int64_t K, cudaStream_t s) {
  const int64_t n = E * K;
  if (n <= 0) return cudaSuccess;
  const int64_t n4 = n / 4;   // K is a multiple of 128
  router_split_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const float4*>(w), reinterpret_cast<uint2*>(planes), reinterpret_cast<uint2*>(planes + n),
      reinterpret_cast<uint2*>(planes + 2 * n), n4);
  return cudaGetLastError();
}

cudaError_t launch_route(const CUtensorMap& map_x, const CUtensorMap& map_w, const RouterArgs& r, int grid, int topk,
                         float* logits, int32_t* ids, float* wts, cudaStream_t s) {
  if (r.T <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(router_logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRtSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = cudaMemsetAsync(r.status, 0, 16, s);
  if (e != cudaSuccess) return e;
  e = launch_pdl(router_logits_tc_kernel, dim3(grid), dim3(kRtThreads), kRtSmemBytes, s, map_x, map_w, r);
  if (e != cudaSuccess) return e;
  const int warps = 8;
  const dim3 nb(static_cast<unsigned>((r.T + warps - 1) / warps)), block(warps * 32);
  // folded logits were written by the logits kernel: read back as one segment
  const int segs = r.fold ? 1 : r.segs;
  const int E = r.E;
  const int64_t T = r.T;
  const float* partial = r.fold ? r.z : r.partial;
  if (r.E <= 128) return launch_pdl(topk_softmax_kernel<4>, nb, block, 0, s, partial, segs, T, E, topk, logits, ids, wts);
  if (r.E <= 256) return launch_pdl(topk_softmax_kernel<8>, nb, block, 0, s, partial, segs, T, E, topk, logits, ids, wts);
  if (r.E <= 512)
    return launch_pdl(topk_softmax_kernel<16>, nb, block, 0, s, partial, segs, T, E, topk, logits, ids, wts);
  return launch_pdl(topk_softmax_kernel<32>, nb, block, 0, s, partial, segs, T, E, topk, logits, ids, wts);
}

}  // namespace moe
