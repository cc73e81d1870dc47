// moe_plan_layout: top-k routing -> per-expert row layout.
//
// "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report),
// "实现拆解" steps 2-3 and "关键源码片段" ep_moe_kernels.py: experts are laid
// out one after another, each padded to a multiple of 128 rows; the first
// `valid` rows of an expert's range carry its tokens and the rest are marked
// -1 in m_indices.  "[Feature] Support BF16 and batch-invariant inference
// with DeepEP v2" (sglang PR #38160 report), "实现拆解" step 1: only ids in
// [expert_start, expert_start + E_local) are local.
//
// Destination rows follow the flattened t * topk + j order inside each expert
// (a stable counting sort), which makes the layout deterministic and
// independent of thread scheduling:
//   1. plan_count_rank  one CTA per 256 assignments: per-expert counts of the
//                       chunk and each assignment's rank inside the chunk
//                       (warp match + per-warp counts; integer only).
//   2. plan_scan        one CTA: per-expert exclusive scan over chunks, padded
//                       sizes, expert starts, the 128-row block table.
//   3. plan_finalize    src2dst = start + chunk offset + rank; m_indices.
#include "common.cuh"
#include "internal.h"
#include "quant_row.cuh"

namespace moe {

namespace {

__device__ __forceinline__ int local_expert(int32_t gid, int32_t E_global, int32_t E_local, int32_t expert_start,
                                            bool* bad) {
  *bad = (gid < -1) || (gid >= E_global);
  if (*bad || gid < 0) return -1;
  const int e = gid - expert_start;
  return (e >= 0 && e < E_local) ? e : -1;
}

__global__ void __launch_bounds__(kPlanChunk) plan_count_rank(PlanArgs p) {
  extern __shared__ int32_t s_wcnt[];  // [8 warps][E_local]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E_local;
  for (int i = tid; i < 8 * E; i += kPlanChunk) s_wcnt[i] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  const int64_t i = static_cast<int64_t>(blockIdx.x) * kPlanChunk + tid;
  int e = -1;
  if (i < p.A) {
    bool bad;
    e = local_expert(p.topk_ids[i], p.E_global, p.E_local, p.expert_start, &bad);
    if (bad) set_status(p.status, MOE_ERR_EXPERT_ID);
  }
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
  const unsigned lower = peers & ((1u << lane) - 1u);
  if (e >= 0 && lower == 0) s_wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  if (e >= 0) {
    int prefix = 0;
    for (int w = 0; w < warp; ++w) prefix += s_wcnt[w * E + e];
    p.chunk_rank[i] = prefix + __popc(lower);
  }
  for (int x = tid; x < E; x += kPlanChunk) {
    int total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) total += s_wcnt[w * E + x];
    p.chunk_hist[static_cast<int64_t>(x) * p.chunks + blockIdx.x] = total;  // [E][chunks]
  }
}

// Exclusive scan over a 1024-thread block; returns this thread's prefix and
// writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int warp_base = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[31];
  __syncthreads();
  return warp_base + x - v;
}

// From the per-expert counts (s_count, shared): padded sizes, expert starts,
// masked row counts, the 128-row block table and meta.  Called by all 1024
// threads of the block (thread e handles local expert e).  When s_start is
// given, each expert's first row is also left there.
__device__ void expert_tables(const PlanArgs& p, const int* s_count, int* s_warp, int* s_start) {
  const int e = threadIdx.x;
  const bool act = e < p.E_local;
  const int count = act ? s_count[e] : 0;
  int rows, nblk;
  if (!p.masked) {
    rows = (count + kBlockM - 1) / kBlockM * kBlockM;
    nblk = rows / kBlockM;
  } else {
    if (count > p.max_m) set_status(p.status, MOE_ERR_MASKED_OVERFLOW);
    rows = count < p.max_m ? count : static_cast<int>(p.max_m);
    nblk = (rows + kBlockM - 1) / kBlockM;
  }
  int total_rows, total_blk;
  const int row_start = block_exclusive_scan(act ? rows : 0, s_warp, &total_rows);
  const int blk_start = block_exclusive_scan(act ? nblk : 0, s_warp, &total_blk);
  if (act) {
    if (s_start) s_start[e] = row_start;
    p.counts[e] = count;
    if (!p.masked) {
      p.padded[e] = rows;
      p.start[e] = row_start;
    } else {
      p.masked_m[e] = rows;
    }
    for (int b = 0; b < nblk; ++b) {
      int4 info;
      info.x = e;
      if (!p.masked) {
        info.y = row_start + b * kBlockM;
        info.z = info.y;
        const int left = count - b * kBlockM;
        info.w = left < kBlockM ? left : kBlockM;
      } else {
        info.y = static_cast<int>(static_cast<int64_t>(e) * p.max_m + b * kBlockM);
        info.z = b * kBlockM;
        const int left = rows - b * kBlockM;
        info.w = left < kBlockM ? left : kBlockM;
        // valid rows numbered without padding: expert e's rows start at the
        // sum of the earlier experts' valid rows
        if (p.block_vrow) p.block_vrow[blk_start + b] = row_start + b * kBlockM;
      }
      reinterpret_cast<int4*>(p.block_info)[blk_start + b] = info;
    }
  }
  if (threadIdx.x == 0) {
    p.meta[0] = total_rows;
    p.meta[1] = total_blk;
  }
}

__global__ void __launch_bounds__(1024) plan_scan(PlanArgs p) {
  __shared__ int s_warp[32];
  __shared__ int s_count[kMaxLocalExperts];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();
  pdl_trigger();
  // Warp w scans experts w, w + 32, w + 64, w + 96 (then the next four
  // groups): the exclusive scan of an expert's chunk counts becomes each
  // chunk's offset inside the expert, and its total the expert's count.
  // The counts of all four experts for up to 8 x 32 chunks are loaded
  // together, so the warp waits for memory once per 256 chunks rather than
  // once per expert.
  constexpr int kLoads = 8, kGroup = 4;
  for (int ex0 = warp; ex0 < p.E_local; ex0 += 32 * kGroup) {
    int carry[kGroup] = {0, 0, 0, 0};
    for (int c0 = 0; c0 < p.chunks; c0 += 32 * kLoads) {
      int v[kGroup][kLoads];
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int ex = ex0 + 32 * g;
        const int32_t* row = p.chunk_hist + static_cast<int64_t>(ex) * p.chunks;
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
          const int c = c0 + 32 * j + lane;
          v[g][j] = (ex < p.E_local && c < p.chunks) ? row[c] : 0;
        }
      }
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int ex = ex0 + 32 * g;
        if (ex >= p.E_local) continue;   // warp-uniform
        int32_t* row = p.chunk_hist + static_cast<int64_t>(ex) * p.chunks;
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
          const int c = c0 + 32 * j + lane;
          int x = v[g][j];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
          }
          if (c < p.chunks) row[c] = carry[g] + x - v[g][j];
          carry[g] += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g)
      if (lane == 0 && ex0 + 32 * g < p.E_local) s_count[ex0 + 32 * g] = carry[g];
  }
  __syncthreads();
  expert_tables(p, s_count, s_warp, nullptr);
}

// m_indices[r] for rows r = first, first + stride, ...: the local expert
// whose padded segment holds row r if r is one of its first counts[e] rows,
// else -1.  s_tab: start[E], padded[E], counts[E].
__device__ void fill_m_indices(const PlanArgs& p, const int32_t* s_tab, int64_t first, int64_t stride) {
  const int E = p.E_local;
  for (int64_t r = first; r < p.all_tokens; r += stride) {
    // last expert whose start is <= r (empty experts share starts; the last
    // one with that start owns the rows)
    int lo = 0, hi = E - 1, found = -1;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (s_tab[mid] <= r) {
        found = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    int32_t v = -1;
    if (found >= 0) {
      const int64_t off = r - s_tab[found];
      if (off < s_tab[E + found] && off < s_tab[2 * E + found]) v = found;
    }
    p.m_indices[r] = v;
  }
}

__global__ void __launch_bounds__(256) plan_finalize(PlanArgs p) {
  extern __shared__ int32_t s_tab[];  // start[E], padded[E], counts[E] (compact)
  const int E = p.E_local;
  pdl_wait();
  pdl_trigger();
  if (!p.masked) {
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
      s_tab[x] = p.start[x];
      s_tab[E + x] = p.padded[x];
      s_tab[2 * E + x] = p.counts[x];
    }
    __syncthreads();
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.A; i += stride) {
    bool bad;
    const int e = local_expert(p.topk_ids[i], p.E_global, p.E_local, p.expert_start, &bad);
    int32_t dst = -1;
    if (e >= 0) {
      const int rank = p.chunk_hist[static_cast<int64_t>(e) * p.chunks + i / kPlanChunk] + p.chunk_rank[i];
      if (!p.masked) {
        dst = s_tab[e] + rank;
      } else if (rank < p.max_m) {
        dst = static_cast<int32_t>(static_cast<int64_t>(e) * p.max_m + rank);
      }
    }
    p.src2dst[i] = dst;
  }
  if (!p.masked)
    fill_m_indices(p, s_tab, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x, stride);
}

// Small problems (decode): the whole plan in one CTA.  Assignments are
// taken in 1024-wide chunks in flattened order; an assignment's stable rank
// is the expert's count in earlier chunks + in earlier warps of its chunk +
// in earlier lanes of its warp (warp match), as in the three-kernel path, so
// the outputs are identical to it.

// Called by all 1024 threads of one CTA, after the kernel's wait for its
// predecessor.
__device__ void plan_small_body(const PlanArgs& p) {
  __shared__ int s_wcnt[32 * kPlanSmallMaxE];   // [warp][expert] counts of the current chunk
  __shared__ int s_tab[3 * kPlanSmallMaxE];     // start, padded, counts (the running per-expert counts)
  __shared__ int s_warp[32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E_local;
  // the status word reports the first data error of this pass
  if (p.clear_status && tid < 4) p.status[tid] = 0;
  __syncthreads();
  int* s_count = s_tab + 2 * E;
  for (int x = tid; x < E; x += 1024) s_count[x] = 0;
  int my_e[2] = {-1, -1};
  int rank[2] = {0, 0};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = tid + 1024 * k;
    for (int x = tid; x < 32 * E; x += 1024) s_wcnt[x] = 0;
    int e = -1;
    if (i < p.A) {
      bool bad;
      e = local_expert(p.topk_ids[i], p.E_global, p.E_local, p.expert_start, &bad);
      if (bad) set_status(p.status, MOE_ERR_EXPERT_ID);
    }
    my_e[k] = e;
    __syncthreads();
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    if (e >= 0 && lower == 0) s_wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int prefix = s_count[e];
      for (int w = 0; w < warp; ++w) prefix += s_wcnt[w * E + e];
      rank[k] = prefix + __popc(lower);
    }
    __syncthreads();
    for (int x = tid; x < E; x += 1024) {
      int add = 0;
      for (int w = 0; w < 32; ++w) add += s_wcnt[w * E + x];
      s_count[x] += add;
    }
    __syncthreads();
  }
  expert_tables(p, s_count, s_warp, s_tab);
  if (!p.masked)
    for (int x = tid; x < E; x += 1024) s_tab[E + x] = p.padded[x];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = tid + 1024 * k;
    if (i >= p.A) continue;
    const int e = my_e[k];
    int32_t dst = -1;
    if (e >= 0) {
      if (!p.masked) {
        dst = s_tab[e] + rank[k];
      } else if (rank[k] < p.max_m) {
        dst = static_cast<int32_t>(static_cast<int64_t>(e) * p.max_m + rank[k]);
      }
    }
    p.src2dst[i] = dst;
  }
  if (!p.masked) fill_m_indices(p, s_tab, tid, 1024);
}

__global__ void __launch_bounds__(1024) plan_small(PlanArgs p) {
  pdl_wait();
  pdl_trigger();
  plan_small_body(p);
}

// The first step of moe_forward for small problems, in one launch: CTA 0
// plans the layout (plan_small_body) while every other CTA quantises four
// tokens, one per 256 threads, into destination rows it forms itself from
// the routing by the plan's rule (quant_row.cuh), so neither waits for the
// other.  The kernels after it see both complete.
constexpr int kPqTokens = 1024 / kQuantThreads;   // tokens per quantising CTA

template <bool kFP8, bool kMX>
__global__ void __launch_bounds__(1024) plan_quant_small_kernel(PlanArgs p, QuantArgs q) {
  __shared__ int16_t s_lid[kPlanSmallMaxA];
  __shared__ int s_cnt[kPlanSmallMaxE];
  __shared__ int64_t s_dst[kPqTokens][kMaxTopk];
  __shared__ int64_t s_blk[kPqTokens][kMaxTopk];
  __shared__ int s_row[kPqTokens][kMaxTopk];
  __shared__ int s_any[kPqTokens];
  pdl_wait();     // routing and activations come from earlier kernels
  pdl_trigger();
  if (blockIdx.x == 0) {
    plan_small_body(p);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int x = tid; x < q.E_local; x += 1024) s_cnt[x] = 0;
  if (tid < kPqTokens) s_any[tid] = 0;
  __syncthreads();
  fill_routing(q, s_lid, s_cnt, tid, 1024);
  __syncthreads();
  // warp w: token w / 8 of this CTA, selections j = w % 8, w % 8 + 8, ...
  const int g = warp >> 3;
  const int64_t t = static_cast<int64_t>(blockIdx.x - 1) * kPqTokens + g;
  if (t < q.T) {
    for (int j = warp & 7; j < q.topk; j += 8) {
      const int64_t d = token_destination(q, s_lid, s_cnt, t, j, lane);
      if (lane == 0) {
        s_dst[g][j] = d;
        if (d >= 0) {
          s_any[g] = 1;
          dest_block(q, d, &s_blk[g][j], &s_row[g][j]);
        }
      }
    }
  }
  __syncthreads();
  if (t < q.T && s_any[g]) quant_scatter_row<kFP8, kMX>(q, t, s_dst[g], s_blk[g], s_row[g], tid & (kQuantThreads - 1));
}

}  // namespace


cudaError_t launch_plan_quant_small(const PlanArgs& p, const QuantArgs& q, cudaStream_t s) {
  PlanArgs pc = p;
  pc.clear_status = 1;   // the planning CTA clears the status word; nothing else here sets it
  const dim3 grid(static_cast<unsigned>(1 + (q.T + kPqTokens - 1) / kPqTokens)), block(1024);
  if (q.mx) return launch_pdl(plan_quant_small_kernel<true, true>, grid, block, 0, s, pc, q);
  if (q.fp8) return launch_pdl(plan_quant_small_kernel<true, false>, grid, block, 0, s, pc, q);
  return launch_pdl(plan_quant_small_kernel<false, false>, grid, block, 0, s, pc, q);
}

int plan_launch_count(int64_t A, int32_t E_local) {
  if (plan_is_small(A, E_local)) return 1;
  return (A > 0 ? 1 : 0) + 2;   // count_rank (when there are assignments), scan, finalize
}

cudaError_t launch_plan(const PlanArgs& p, cudaStream_t s) {
  if (plan_is_small(p.A, p.E_local)) {
    PlanArgs q = p;
    q.clear_status = 1;   // the one CTA clears the status word before anything can set it
    return launch_pdl(plan_small, dim3(1), dim3(1024), 0, s, q);
  }
  // the status word reports the first data error of this pass through the layer
  cudaError_t e = cudaMemsetAsync(p.status, 0, 16, s);
  if (e != cudaSuccess) return e;
  if (p.chunks > 0) {
    e = launch_pdl(plan_count_rank, dim3(p.chunks), dim3(kPlanChunk), 8 * p.E_local * sizeof(int32_t), s, p);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(plan_scan, dim3(1), dim3(1024), 0, s, p);
  if (e != cudaSuccess) return e;
  const int64_t work = p.A > p.all_tokens ? p.A : p.all_tokens;
  int grid = static_cast<int>((work + 255) / 256);
  if (grid > 1184) grid = 1184;
  if (grid < 1) grid = 1;
  return launch_pdl(plan_finalize, dim3(grid), dim3(256), 3 * p.E_local * sizeof(int32_t), s, p);
}

}  // namespace moe
