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
// writing it.
//   amax: |v| = bf16(fp32(|q|) * |s|) (both roundings are odd-symmetric)
//         is non-decreasing in |q|, and the magnitude bits of a finite e4m3
//         code (byte & 0x7f) order like |q|, so amax|v| is that function of
//         the block's largest magnitude byte: four bytes per byte-wise
//         integer max, one conversion per block.
//   q':   two codes per conversion (e4m3x2 -> f16x2 -> two fp32), the two
//         products of each pair in one packed fp32 multiply, both roundings
//         to bf16 in one conversion, the power-of-two rescale again as one
//         packed multiply (exact) and one two-code conversion back.
// About five instructions per byte and 32 registers per thread, so eight
// blocks (128 KB of loads) are in flight per SM and the kernel streams at
// close to HBM speed instead of waiting on its arithmetic.
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

// (a, b) * (m, m) in one packed fp32 multiply, round to nearest even
__device__ __forceinline__ float2 mul_f32x2(float a, float b, float m) {
  float2 r;
  asm("{\n\t.reg .b64 p, q, m2;\n\t"
      "mov.b64 p, {%2, %3};\n\t"
      "mov.b64 m2, {%4, %4};\n\t"
      "mul.rn.f32x2 q, p, m2;\n\t"
      "mov.b64 {%0, %1}, q;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a), "f"(b), "f"(m));
  return r;
}

// two e4m3 codes (low 16 bits of pair) -> e4m3(bf16(fp32(q) * s) * 2^-e), lo first
__device__ __forceinline__ uint32_t requant_pair(uint32_t pair, float s, float mul) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3);
  const float2 q = __half22float2(__half2(h));
  const float2 p = mul_f32x2(q.x, q.y, s);              // fp32 products
  const float2 v = unpack_bf16x2(pack_bf16x2(p.x, p.y));    // the bf16 intermediate
  const float2 r = mul_f32x2(v.x, v.y, mul);            // exact power-of-two rescale
  return cvt_e4m3x2(r.x, r.y);
}

__global__ void __launch_bounds__(kRequantThreads, 8) requant_kernel(const uint8_t* w_in, const float* s_in,
                                                                 uint8_t* w_out, uint8_t* s_out, int64_t N,
                                                                 int64_t C) {
  __shared__ uint32_t s_red[kRequantThreads / 32];
  // blocks in (expert, row block, column block) order: block b starts at row
  // 128 (b / (C / 128)) of the [E * N, C] byte matrix, column 128 (b % (C / 128))
  const int64_t nbc = C / 128;
  const int64_t blk = blockIdx.x;
  const float scale = s_in[blk];
  const int tid = threadIdx.x;
  // part p: row + 64 p, 16-byte halves h: raw[2 p + h]
  const int64_t part_stride = 64 * C;
  const uint8_t* src = w_in + ((blk / nbc) * 128 + (tid >> 2)) * C + (blk % nbc) * 128 + (tid & 3) * 32;

  uint4 raw[2 * kRequantParts];
#pragma unroll
  for (int i = 0; i < 2 * kRequantParts; ++i)
    raw[i] = *reinterpret_cast<const uint4*>(src + (i >> 1) * part_stride + 16 * (i & 1));
  // the block's largest magnitude code
  uint32_t mw = 0;
#pragma unroll
  for (int i = 0; i < 2 * kRequantParts; ++i) {
    const uint32_t a = __vmaxu4(raw[i].x & 0x7F7F7F7Fu, raw[i].y & 0x7F7F7F7Fu);
    const uint32_t b = __vmaxu4(raw[i].z & 0x7F7F7F7Fu, raw[i].w & 0x7F7F7F7Fu);
    mw = __vmaxu4(mw, __vmaxu4(a, b));
  }
  mw = __vmaxu4(mw, mw >> 16);
  mw = __vmaxu4(mw, mw >> 8) & 0xFFu;
  mw = __reduce_max_sync(0xFFFFFFFFu, mw);
  if ((tid & 31) == 0) s_red[tid >> 5] = mw;
  __syncthreads();
  mw = s_red[0];
#pragma unroll
  for (int i = 1; i < kRequantThreads / 32; ++i) mw = max(mw, s_red[i]);
  const float amax = unpack_bf16x2(pack_bf16x2(e4m3_to_float(mw) * fabsf(scale), 0.0f)).x;
  const int s = ue8m0_exponent(amax);
  const float mul = exp2_neg(s);
  // the output address formed again here rather than kept live across the
  // reduction (an empty asm hides that the thread index is unchanged)
  int t2 = tid;
  asm volatile("" : "+r"(t2));
  uint8_t* dst = w_out + ((blk / nbc) * 128 + (t2 >> 2)) * C + (blk % nbc) * 128 + (t2 & 3) * 32;
#pragma unroll
  for (int i = 0; i < 2 * kRequantParts; ++i) {
    const uint32_t words[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    uint32_t outw[4];
#pragma unroll
    for (int w = 0; w < 4; ++w)
      outw[w] = requant_pair(words[w] & 0xFFFFu, scale, mul) | (requant_pair(words[w] >> 16, scale, mul) << 16);
    *reinterpret_cast<uint4*>(dst + (i >> 1) * part_stride + 16 * (i & 1)) =
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
