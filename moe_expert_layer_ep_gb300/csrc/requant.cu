// Load-time weight preparation:
//   moe_requant_weights_ue8m0: requantisation of 128x128 block-scaled FP8
//     weights to power-of-two (UE8M0) block scales;
//   moe_pack_mx_scales: MXFP8 weight scales into the chunk order the grouped
//     GEMMs copy into tensor memory.
//
// "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128 report),
// "实现拆解" step 1 and "关键源码片段" fp8.py: both expert weight tensors of
// a standard MoE layer are requantised with UE8M0 block scales for the
// grouped GEMMs, through a bfloat16 intermediate.  Per 128x128 block:
//   v  = bf16(fp32(q) * s)                 (s: the block's fp32 scale)
//   e  = smallest integer with amax|v| <= 448 * 2^e, clamped to [-127, 127]
//   q' = e4m3(v * 2^-e)                    (round to nearest even, saturating)
// One CTA per block: 256 threads, each two quarter rows (rows r and r + 64,
// 32 bytes each), read once, reduced, written once; in-place operation
// (w_out == w_in) is allowed because a CTA reads its whole block before
// writing it.  A thread keeps only its 64 raw e4m3 bytes in registers and
// forms the bf16 intermediate twice (for the block maximum, then for the
// output), the same arithmetic both times: with few registers per thread,
// five blocks are in flight per SM.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRequantThreads = 256;
constexpr int kRequantParts = 2;     // quarter rows per thread

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3);
  return __half2float(__half(hr));
}

__global__ void __launch_bounds__(kRequantThreads, 5) requant_kernel(const uint8_t* w_in, const float* s_in,
                                                                 uint8_t* w_out, uint8_t* s_out, int64_t N,
                                                                 int64_t C) {
  __shared__ float s_red[kRequantThreads / 32];
  const int64_t nbn = N / 128, nbc = C / 128;
  const int64_t blk = blockIdx.x;
  const int64_t e = blk / (nbn * nbc);
  const int64_t rb = (blk / nbc) % nbn;
  const int64_t cb = blk % nbc;
  const float scale = s_in[blk];
  const int tid = threadIdx.x;
  const int64_t row = rb * 128 + (tid >> 2);
  // part p: row + 64 p, 16-byte halves h: raw[2 p + h]
  const int64_t off = (e * N + row) * C + cb * 128 + (tid & 3) * 32;
  const int64_t part_stride = 64 * C;

  uint4 raw[2 * kRequantParts];
#pragma unroll
  for (int i = 0; i < 2 * kRequantParts; ++i)
    raw[i] = *reinterpret_cast<const uint4*>(w_in + off + (i >> 1) * part_stride + 16 * (i & 1));
  // bf16(fp32(q) * scale) of bytes b and b + 1 of a word, packed
  auto bf16_pair = [scale](uint32_t word, int b) {
    const __nv_bfloat162 pr = __floats2bfloat162_rn(e4m3_to_float((word >> (8 * b)) & 0xFFu) * scale,
                                                    e4m3_to_float((word >> (8 * b + 8)) & 0xFFu) * scale);
    return *reinterpret_cast<const uint32_t*>(&pr);
  };
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 2 * kRequantParts; ++i) {
    const uint32_t words[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int b = 0; b < 4; b += 2) {
        const float2 f = unpack_bf16x2(bf16_pair(words[w], b));
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((tid & 31) == 0) s_red[tid >> 5] = amax;
  __syncthreads();
  amax = s_red[0];
#pragma unroll
  for (int i = 1; i < kRequantThreads / 32; ++i) amax = fmaxf(amax, s_red[i]);
  const int s = ue8m0_exponent(amax);
  const float mul = exp2_neg(s);
  // form the intermediate again rather than keep the first pass's values live
  // across the reduction (an empty asm hides that the bytes are unchanged)
#pragma unroll
  for (int i = 0; i < 2 * kRequantParts; ++i)
    asm volatile("" : "+r"(raw[i].x), "+r"(raw[i].y), "+r"(raw[i].z), "+r"(raw[i].w));
#pragma unroll
  for (int i = 0; i < 2 * kRequantParts; ++i) {
    const uint32_t words[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    uint32_t outw[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 lo = unpack_bf16x2(bf16_pair(words[w], 0)), hi = unpack_bf16x2(bf16_pair(words[w], 2));
      outw[w] = cvt_e4m3x2(lo.x * mul, lo.y * mul) | (cvt_e4m3x2(hi.x * mul, hi.y * mul) << 16);
    }
    *reinterpret_cast<uint4*>(w_out + off + (i >> 1) * part_stride + 16 * (i & 1)) =
        make_uint4(outw[0], outw[1], outw[2], outw[3]);
  }
  if (tid == 0) s_out[blk] = static_cast<uint8_t>(s + 127);
}

// MXFP8 weight scales, natural [E, N, C/32] bytes (scale rows ld_words
// 32-bit words apart, padded or not) -> packed 512-byte chunks per (e,
// 128-row block, 128-column group), row r's word at byte 16 * (r % 32) +
// 4 * (r / 32).  A source word (4 consecutive 32-column blocks of one row) is
// a destination word, so one thread moves one word.
__global__ void __launch_bounds__(256) pack_mx_scales_kernel(const uint32_t* src, int64_t ld_words, uint32_t* dst,
                                                             int64_t words, int64_t N, int64_t CG) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= words) return;
  const int64_t kg = i % CG;          // 128-column group
  const int64_t n = (i / CG) % N;     // row
  const int64_t e = i / (CG * N);
  const int r = static_cast<int>(n & 127);
  const int64_t chunk = (e * (N / 128) + (n >> 7)) * CG + kg;
  dst[chunk * 128 + 4 * (r & 31) + (r >> 5)] = src[(e * N + n) * ld_words + kg];
}

}  // namespace

cudaError_t launch_pack_mx_scales(const uint8_t* src, int64_t src_ld, uint8_t* dst, int64_t E, int64_t N, int64_t C,
                                  cudaStream_t st) {
  const int64_t words = E * N * (C / 128);
  if (words <= 0) return cudaSuccess;
  pack_mx_scales_kernel<<<static_cast<unsigned>((words + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const uint32_t*>(src), src_ld / 4, reinterpret_cast<uint32_t*>(dst), words, N, C / 128);
  return cudaGetLastError();
}

cudaError_t launch_requant(const uint8_t* w_in, const float* s_in, uint8_t* w_out, uint8_t* s_out, int64_t E,
                           int64_t N, int64_t C, cudaStream_t st) {
  const int64_t blocks = E * (N / 128) * (C / 128);
  if (blocks <= 0) return cudaSuccess;
  requant_kernel<<<static_cast<unsigned>(blocks), kRequantThreads, 0, st>>>(w_in, s_in, w_out, s_out, N, C);
  return cudaGetLastError();
}

}  // namespace moe
