// moe_route: the fp32 MoE router that feeds the layer its top-k expert ids
// and weights.
//
// "[Feature] Support BF16 and batch-invariant inference with DeepEP v2"
// (sglang PR #38160 report), section "关联脉络": the router GEMM is kept in
// fp32 so that expert selection does not flip under deterministic inference;
// "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report),
// "关键源码片段" deep_gemm.py: the layer consumes standard top-k ids/weights.
//
//   router_logits_kernel        z[t, e] = sum_k x[t, k] * W[e, k], bf16 x (exact
//                               in fp32) times fp32 W, fp32 FMA on the CUDA
//                               cores; 64x64 output tiles, K in slabs of 32
//                               through shared memory (large batches).
//   router_logits_small_kernel  8 tokens x 2 experts per CTA with 1024-wide K
//                               slabs, so that many CTAs stream the router
//                               weights (batches of up to 256 tokens).
//   Both sum every output's K terms in four fixed chains (k mod 4, ascending
//   k), combined as (c0 + c1) + (c2 + c3): the same operations for every tile
//   shape and batch size, so a token's logits do not depend on its batch.
//   topk_softmax_kernel         one warp per token: k rounds of a warp argmax
//                               (larger logit wins, equal logits go to the
//                               lower expert id), then w_j = exp(z_j - z_max) /
//                               sum, the sum taken in j order.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRouterThreads = 256;

// One BM x BN output tile per CTA (16 x 16 threads, each TM x TN outputs), K
// in slabs of RK staged through shared memory (k-major) while the next slab
// is already loaded into registers.
template <int BM, int BN, int RK>
__global__ void __launch_bounds__(kRouterThreads, 2) router_logits_kernel(const uint16_t* x, const float* w, float* z,
                                                                       int64_t T, int64_t K, int E) {
  constexpr int TM = BM / 16, TN = BN / 16;
  constexpr int XV = BM * RK / 8 / kRouterThreads;   // 8-element bf16 vectors per thread per slab
  constexpr int WV = BN * RK / 4 / kRouterThreads;   // 4-element fp32 vectors per thread per slab
  static_assert(XV >= 1 && WV >= 1, "tile too small for the thread count");
  __shared__ __align__(16) float xs[RK][BM];
  __shared__ __align__(16) float ws[RK][BN];
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * BM;
  const int e0 = blockIdx.y * BN;
  float acc[4][TM][TN] = {};
  uint4 xr[XV];
  float4 wr[WV];
  auto load = [&](int64_t k0) {
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 8), kk = (i % (RK / 8)) * 8;
      const int64_t t = t0 + r;
      xr[v] = t < T ? __ldg(reinterpret_cast<const uint4*>(x + t * K + k0 + kk)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 4), kk = (i % (RK / 4)) * 4;
      const int e = e0 + r;
      wr[v] = e < E ? __ldg(reinterpret_cast<const float4*>(w + static_cast<int64_t>(e) * K + k0 + kk))
                    : make_float4(0, 0, 0, 0);
    }
  };
  auto stage = [&]() {
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 8), kk = (i % (RK / 8)) * 8;
      const float2 p0 = unpack_bf16x2(xr[v].x), p1 = unpack_bf16x2(xr[v].y), p2 = unpack_bf16x2(xr[v].z),
                   p3 = unpack_bf16x2(xr[v].w);
      xs[kk + 0][r] = p0.x; xs[kk + 1][r] = p0.y; xs[kk + 2][r] = p1.x; xs[kk + 3][r] = p1.y;
      xs[kk + 4][r] = p2.x; xs[kk + 5][r] = p2.y; xs[kk + 6][r] = p3.x; xs[kk + 7][r] = p3.y;
    }
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 4), kk = (i % (RK / 4)) * 4;
      ws[kk + 0][r] = wr[v].x; ws[kk + 1][r] = wr[v].y; ws[kk + 2][r] = wr[v].z; ws[kk + 3][r] = wr[v].w;
    }
  };
  load(0);
  for (int64_t k0 = 0; k0 < K; k0 += RK) {   // K is a multiple of 128, so of RK
    stage();
    __syncthreads();
    if (k0 + RK < K) load(k0 + RK);
#pragma unroll
    for (int k = 0; k < RK; ++k) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = xs[k][ty * TM + i];
#pragma unroll
      for (int j = 0; j < TN; ++j) b[j] = ws[k][tx * TN + j];
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[k & 3][i][j] = fmaf(a[i], b[j], acc[k & 3][i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t t = t0 + ty * TM + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int e = e0 + tx * TN + j;
      if (e < E) z[t * E + e] = (acc[0][i][j] + acc[1][i][j]) + (acc[2][i][j] + acc[3][i][j]);
    }
  }
}

// Small batches: BM tokens x BN experts per CTA, one thread per output, the
// whole CTA loading wide K slabs.  Shared rows are padded by four floats so
// that the rows fall in distinct banks.
template <int BM, int BN, int RK>
__global__ void __launch_bounds__(kRouterThreads) router_logits_small_kernel(const uint16_t* x, const float* w,
                                                                             float* z, int64_t T, int64_t K, int E) {
  constexpr int XV = BM * RK / 8 / kRouterThreads;
  constexpr int WV = BN * RK / 4 / kRouterThreads;
  constexpr int LD = RK + 4;
  static_assert(XV >= 1 && WV >= 1 && BM * BN <= kRouterThreads, "tile");
  __shared__ __align__(16) float xs[BM][LD];
  __shared__ __align__(16) float ws[BN][LD];
  const int tid = threadIdx.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * BM;
  const int e0 = blockIdx.y * BN;
  const int my_r = tid / BN, my_c = tid % BN;
  float c0 = 0.0f, c1 = 0.0f, c2 = 0.0f, c3 = 0.0f;
  uint4 xr[XV];
  float4 wr[WV];
  auto load = [&](int64_t k0) {
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 8), kk = (i % (RK / 8)) * 8;
      const int64_t t = t0 + r;
      xr[v] = (t < T && k0 + kk < K) ? __ldg(reinterpret_cast<const uint4*>(x + t * K + k0 + kk))
                                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 4), kk = (i % (RK / 4)) * 4;
      const int e = e0 + r;
      wr[v] = (e < E && k0 + kk < K)
                  ? __ldg(reinterpret_cast<const float4*>(w + static_cast<int64_t>(e) * K + k0 + kk))
                  : make_float4(0, 0, 0, 0);
    }
  };
  load(0);
  for (int64_t k0 = 0; k0 < K; k0 += RK) {
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 8), kk = (i % (RK / 8)) * 8;
      const float2 p0 = unpack_bf16x2(xr[v].x), p1 = unpack_bf16x2(xr[v].y), p2 = unpack_bf16x2(xr[v].z),
                   p3 = unpack_bf16x2(xr[v].w);
      *reinterpret_cast<float4*>(&xs[r][kk]) = make_float4(p0.x, p0.y, p1.x, p1.y);
      *reinterpret_cast<float4*>(&xs[r][kk + 4]) = make_float4(p2.x, p2.y, p3.x, p3.y);
    }
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + v * kRouterThreads;
      const int r = i / (RK / 4), kk = (i % (RK / 4)) * 4;
      *reinterpret_cast<float4*>(&ws[r][kk]) = wr[v];
    }
    __syncthreads();
    if (k0 + RK < K) load(k0 + RK);
    if (tid < BM * BN) {
      // K is a multiple of 128, so a slab holds whole groups of four; the
      // last slab stops at K (an extra zero product could flip a -0 sum).
      const int kn = static_cast<int>(K - k0 < RK ? K - k0 : RK);
#pragma unroll 4
      for (int k = 0; k < kn; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(&xs[my_r][k]);
        const float4 b = *reinterpret_cast<const float4*>(&ws[my_c][k]);
        c0 = fmaf(a.x, b.x, c0);
        c1 = fmaf(a.y, b.y, c1);
        c2 = fmaf(a.z, b.z, c2);
        c3 = fmaf(a.w, b.w, c3);
      }
    }
    __syncthreads();
  }
  const int64_t t = t0 + my_r;
  const int e = e0 + my_c;
  if (tid < BM * BN && t < T && e < E) z[t * E + e] = (c0 + c1) + (c2 + c3);
}

// P logits per lane (E <= 32 P).  The j-th selection is kept by lane j % 32
// (slot j / 32), so nothing is indexed dynamically; every lane forms the same
// softmax sum in j order from broadcasts, and lane j writes output j.
template <int P>
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* z, int64_t T, int E, int topk, int32_t* ids,
                                                           float* wts) {
  static_assert(P <= 32, "taken mask is 32 bits");
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[P];
  const float* row = z + t * E;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
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

cudaError_t launch_route(const void* x, const float* w, int64_t T, int64_t K, int E, int topk, float* logits,
                         int32_t* ids, float* wts, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  if (T <= kRouterSmallBatch) {
    dim3 grid(static_cast<unsigned>((T + 7) / 8), static_cast<unsigned>((E + 1) / 2));
    router_logits_small_kernel<8, 2, 1024><<<grid, kRouterThreads, 0, s>>>(xb, w, logits, T, K, E);
  } else {
    dim3 grid(static_cast<unsigned>((T + 63) / 64), static_cast<unsigned>((E + 63) / 64));
    router_logits_kernel<64, 64, 32><<<grid, kRouterThreads, 0, s>>>(xb, w, logits, T, K, E);
  }
  const int warps = 8;
  const unsigned nb = static_cast<unsigned>((T + warps - 1) / warps);
  if (E <= 128)
    topk_softmax_kernel<4><<<nb, warps * 32, 0, s>>>(logits, T, E, topk, ids, wts);
  else if (E <= 256)
    topk_softmax_kernel<8><<<nb, warps * 32, 0, s>>>(logits, T, E, topk, ids, wts);
  else if (E <= 512)
    topk_softmax_kernel<16><<<nb, warps * 32, 0, s>>>(logits, T, E, topk, ids, wts);
  else
    topk_softmax_kernel<32><<<nb, warps * 32, 0, s>>>(logits, T, E, topk, ids, wts);
  return cudaGetLastError();
}

}  // namespace moe
