// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, for sm_103a.
//
//   stage 1 (moe_grouped_gemm_w13_act): h = silu(a W1_e^T) * (a W3_e^T)
//   stage 2 (moe_grouped_gemm_w2):      y = h W2_e^T
//
// The sequence is the one of the BF16 run function in "Add BF16 support to
// EP-MoE for DeepGEMM" (sglang PR #17392 report), "关键源码片段"
// deep_gemm.py -- GEMM (M,K)x(E,N,K) -> (M,N), SiLU*mul -> (M,N/2), GEMM
// (M,N/2)x(E,K,N/2) -> (M,K) -- with the activation fused into the first
// GEMM's epilogue.  FP8 operands carry UE8M0 scales ("Support DeepGEMM for
// standard MoE dispatch" (sglang PR #33128 report), "实现拆解" steps 1 and 3):
// 1x128 per activation row and 128x128 per weight block.  Because the scales
// are powers of two, they are handed to the block-scaled MMA
// (kind::mxf8f6f4, one scale per 32 K-elements) by giving all four 32-element
// sub-blocks of a K block the same scale: the products are the same, exactly.
// A row's scale word holds the scales of four consecutive K blocks, one per
// byte, and the MMAs of K block kb read byte kb % 4 (scale-factor ID), so the
// scale tiles are copied into tensor memory once per four K blocks.
// The MXFP8 variant (1x32 scales everywhere; listed as uncovered in the
// standard-dispatch report's "风险与影响" item 5) hands each 32-element
// sub-block its own scale byte: the k-th MMA of a 128-byte K block reads byte
// k of the scale words (scale-factor ID k), and the weight scales arrive as
// packed chunks (both of a tile's in one TMA box) instead of being expanded
// in shared memory.
//
// Work unit: one 128-row expert block (from the block table written by the
// plan) x one output column block.  Stage 1's B tile is 128 gate rows of w13
// stacked on the matching 128 up rows, so one 128x256 accumulator holds g and
// u for 128 consecutive h columns: the epilogue forms h and, on the FP8 path,
// its 1x128 UE8M0 quantisation without leaving the CTA.  Stage 2's B tile is
// 256 consecutive rows of w2.
//
// The MXFP4 variant (FP4 E2M1 weights with 1x32 scales, the FP4 item of
// the same list) is the MXFP8 kernel with an E2M1 B operand: the block-scaled
// MMA multiplies e4m3 activations by E2M1 weights directly, and TMA unpacks
// each 16 packed codes into the 16-byte shared-memory group that operand
// reads (8 bytes of codes, 8 bytes of gap), so a B tile keeps the FP8 tile's
// geometry while half as many bytes leave L2.
//
// One persistent CTA per SM:
//   warp 0      TMA producer: per K block the A tile, the whole B tile in one
//               box (GEMM1's gate and up rows through a 5-d view of w13) and
//               the activation scale chunk (once per four K blocks for 1x128
//               scales; + both MX weight-scale chunks in one box).  TMA
//               accepts about 130 bytes per cycle per SM, so the producer's
//               loop does nothing else.
//   warp 1      TMEM allocation + single-thread MMA issue (tcgen05.cp of the
//               scale tiles, 4 MMAs of K=32 bytes per 128-byte K block)
//   epilogue    4 or 8 warps (see epi_warps): tcgen05.ld of the accumulator,
//               then activation / quantisation and stores of valid rows
//   scale warp  FP8 with 128x128 weight scales: writes each quad of K
//               blocks' weight-scale tile in shared memory and arrives on
//               every stage beside the producer
// A 4-stage mbarrier ring connects producer and MMA; accumulator barriers
// connect MMA and epilogue (two accumulators on the BF16 path, one on the FP8
// path, whose other tensor-memory columns hold the scale tiles).
//
// Column-block pairs (g.pair: FP8 kinds, compact layout, no split, an even
// number of column blocks): the kernel runs in clusters of two CTAs whose
// work units are always column blocks 2m and 2m + 1 of one row block, so
// they read the same A tile.  Each CTA's producer loads one 64-row half of it
// with TMA multicast into both CTAs' stage (each CTA's barrier counts both
// halves), and each CTA's MMA completion frees the stage in both CTAs, so a
// stage is refilled only once both have read it.  Per CTA, half of the A
// bytes (a sixth of all loaded bytes) leave L2; the MMAs, their operands and
// so the results are those of the unpaired kernel.
//
// Every row is computed by the same instruction sequence with the same K
// order whatever the batch, so results are batch-invariant and reproducible.
// Rows of a block beyond its valid count (padding, -1 in m_indices) are
// computed from whatever the buffer holds and never stored.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// Epilogue warps per (dtype, stage).  The FP8 GEMM1 epilogue (one
// accumulator: its other tensor-memory columns hold the scale tiles) uses 8,
// two per accumulator lane quadrant with half of the columns each, copies the
// accumulator out and releases it before the activation and quantisation.
// The others use 4 warps (measured faster there).
// Split-K kernels (masked layouts) copy the accumulator out to the partial
// buffer in 32-column chunks and use 4 warps.
__host__ __device__ constexpr int epi_warps(bool fp8, int stage, bool split = false) {
  return (fp8 && stage == 1 && !split) ? 8 : 4;
}
// FP8 with 128x128 weight scales: one warp expands each stage's weight-scale
// tile in shared memory, beside the TMA producer (whose loop then only
// issues copies).
__host__ __device__ constexpr int scale_warps(bool fp8, bool mx) { return fp8 && !mx ? 1 : 0; }
__host__ __device__ constexpr int threads_for(bool fp8, bool mx, int stage, bool split) {
  return 64 + 32 * epi_warps(fp8, stage, split) + 32 * scale_warps(fp8, mx);
}
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kKBlockBytes = 128;                  // one 128-byte swizzle atom of K per stage
constexpr int kABytes = kTileM * kKBlockBytes;     // 16 KB
constexpr int kBBytes = kTileN * kKBlockBytes;     // 32 KB
constexpr int kBPBytes = kTileN * kKBlockBytes / 2;   // MXFP4: the codes of a B tile, 16 KB (what its copy counts)
constexpr int kSfaBytes = 512;
constexpr int kSfbBytes = 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemCol = 256;               // FP8: scale tiles live in columns 256..383

// Shared-memory map.
struct Lay {
  static constexpr int kStages = 4;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
  static constexpr int kOffBar = kOffSfb + kStages * kSfbBytes;
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 4 + 1;   // full, empty; acc; done; amax; esync
  static constexpr int kOffHolder = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffHolder + 8;
  static constexpr int kOffAmax = kOffAbort + 8;                 // 2 x 4 x 2 x 32 floats
  // GEMM2 output staging for TMA stores: two 128-row x 32-column bf16 tiles
  static constexpr int kOffStage = (kOffAmax + 2 * 4 * 2 * 32 * 4 + 1023) / 1024 * 1024;
  static constexpr int kStageTileBytes = kTileM * 64;
  static constexpr int kSmemBytes = kOffStage + 2 * kStageTileBytes + 1024;   // + 1024-byte alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// Instruction descriptors (M = 128, N = 256, both operands K-major, fp32 D).
constexpr uint32_t kIdescBF16 = (1u << 4)      // D format f32
                                | (1u << 7)    // A bf16
                                | (1u << 10)   // B bf16
                                | (static_cast<uint32_t>(kTileN >> 3) << 17) |
                                (static_cast<uint32_t>(kTileM >> 4) << 24);
constexpr uint32_t kIdescFP8 = (0u << 7)       // A e4m3
                               | (0u << 10)    // B e4m3
                               | (static_cast<uint32_t>(kTileN >> 3) << 17) |
                               (1u << 23)      // scale factors are UE8M0
                               | (static_cast<uint32_t>(kTileM >> 4) << 24);

struct Tile {
  int expert;
  int64_t row0;    // first row of the block in a / h / y
  int tma_row;     // row coordinate of the block for the A tensor map
  int valid;       // rows of the block that carry a token
  int nb;          // output column block
  int64_t sf_block;
};

__device__ __forceinline__ Tile load_tile(const GemmArgs& g, int64_t t) {
  const int64_t j = t / g.n_blocks;
  const int4 info = reinterpret_cast<const int4*>(g.block_info)[j];
  Tile tl;
  tl.expert = info.x;
  tl.row0 = g.masked ? static_cast<int64_t>(info.y) : static_cast<int64_t>(info.y);
  tl.tma_row = info.z;
  tl.valid = info.w;
  tl.nb = static_cast<int>(t - j * g.n_blocks);
  tl.sf_block = g.masked ? static_cast<int64_t>(info.x) * g.blocks_per_expert + (info.z >> 7) : (info.y >> 7);
  return tl;
}

// Weight rows of the two 128-row B boxes of a tile.
template <int kStage>
__device__ __forceinline__ void tile_b_rows(const GemmArgs& g, const Tile& tl, int* r0, int* r1) {
  if (kStage == 1) {
    *r0 = tl.nb * 128;
    *r1 = static_cast<int>(g.n_half) + tl.nb * 128;
  } else {
    *r0 = tl.nb * kTileN;
    *r1 = *r0 + 128;
  }
}

// First K block of segment seg when the K loop runs in S fixed segments.
__device__ __forceinline__ int seg_begin(int seg, int S, int k_blocks) { return seg * k_blocks / S; }

// Tensor maps: map_a (A rows), map_b (weights; GEMM1 as [E][gate, up][I/128]
// [128 rows][K] so that one box holds a tile's gate and up rows, GEMM2 in
// 256-row boxes), map_out (GEMM2 y stores), map_wsf (MXFP8 weight-scale
// chunks, both of a tile's chunks in one box).
// kFP4: MXFP4 weights, an E2M1 B operand (with kFP8 and kMX).
template <bool kFP8, bool kMX, int kStage, bool kFP4, bool kSplit>
__global__ void __launch_bounds__(threads_for(kFP8, kMX, kStage, kSplit), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_out, const __grid_constant__ CUtensorMap map_wsf,
                        const GemmArgs g) {
  using L = Lay;
  // B operand format: e4m3, or E2M1 (code 5) for FP4 weights
  constexpr uint32_t kIdescB = kIdescFP8 | (kFP4 ? (5u << 10) : 0u);
  constexpr int kStages = L::kStages;
  constexpr int kOffA = L::kOffA, kOffB = L::kOffB, kOffSfa = L::kOffSfa, kOffSfb = L::kOffSfb;
  constexpr int kOffBar = L::kOffBar, kOffHolder = L::kOffHolder, kOffAbort = L::kOffAbort, kOffAmax = L::kOffAmax;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = bars + 2 * kStages + 2;
  uint64_t* done = bars + 2 * kStages + 4;
  uint64_t* xchg = bars + 2 * kStages + 5;  // [4]: the two epilogue warps of a lane quadrant
  uint64_t* esync = bars + 2 * kStages + 9; // GEMM2: the epilogue warps have staged a chunk
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + kOffHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // column-block pair: this CTA loads half `crank` of the shared A tile for
  // both CTAs, and a stage is free only once both CTAs' MMAs have read it
  const bool pair = g.pair != 0;
  const uint32_t crank = pair ? cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1 + scale_warps(kFP8, kMX));   // producer (+ scale warp)
      mbar_init(&empty[s], pair ? 2 : 1);                // this CTA's MMAs (+ the partner's)
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 32 * epi_warps(kFP8, kStage, kSplit));
    }
    mbar_init(done, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&xchg[q], 64);
    mbar_init(esync, 32 * epi_warps(kFP8, kStage, kSplit));
    if (kStage == 2) prefetch_tensormap(&map_out);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
    if (kMX) prefetch_tensormap(&map_wsf);
  }
  if (warp == 1) {
    tmem_alloc(holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  // a pair's barriers are initialised in both CTAs before either CTA's copies
  // or MMA completions can reach them
  if (pair)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  constexpr int kElemsPerKBlock = kFP8 ? 128 : 64;
  const int k_blocks = g.k_blocks;
  // work unit u: tile u / S, K segment u % S (S = 1 unless split)
  const int S = kSplit ? g.k_splits : 1;
  if (warp == 0 && lane == 0) {
    // While the previous kernel finishes, bring the first K blocks of this
    // CTA's first weight tile into L2.  Inside the layer the block table was
    // written two kernels back (by the plan), so it is complete here; were it
    // not, a stale entry would only prefetch other weights (a prefetch reads
    // nothing back and ignores coordinates outside the tensor).
    const int64_t pre_units = static_cast<int64_t>(g.meta[1]) * g.n_blocks * S;
    if (blockIdx.x < pre_units) {
      const int64_t t = blockIdx.x / S;
      const int seg = static_cast<int>(blockIdx.x - t * S);
      const Tile tl = load_tile(g, t);
      int r0, r1;
      tile_b_rows<kStage>(g, tl, &r0, &r1);
      const int kb0 = seg_begin(seg, S, k_blocks);
      const int kb1 = min(seg_begin(seg + 1, S, k_blocks), kb0 + 8);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (kStage == 1)
          tma_prefetch_5d(&map_b, kb * kElemsPerKBlock, 0, tl.nb, 0, tl.expert);
        else
          tma_prefetch_3d(&map_b, kb * kElemsPerKBlock, r0, tl.expert);
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  const int64_t n_tiles = static_cast<int64_t>(g.meta[1]) * g.n_blocks;
  const int64_t n_units = n_tiles * S;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    bool ok = true;

    // the next unit's block-table entry is read while the current unit's
    // copies are issued, so no tile starts with a wait for it
    Tile tl_next;
    if (blockIdx.x < n_units) tl_next = load_tile(g, blockIdx.x / S);
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int64_t t = u / S;
      const int seg = static_cast<int>(u - t * S);
      const Tile tl = tl_next;
      if (u + gridDim.x < n_units) tl_next = load_tile(g, (u + gridDim.x) / S);
      int r0, r1;
      tile_b_rows<kStage>(g, tl, &r0, &r1);
      const int a_e = g.masked ? tl.expert : 0;
      const int kb_end = seg_begin(seg + 1, S, k_blocks);
      const int kb_begin = seg_begin(seg, S, k_blocks);
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        // FP8 1x128: the activation scales of K blocks 4q .. 4q + 3 arrive
        // with the stage of the unit's first K block of quad q
        const bool sfa_new = kFP8 && (kMX || (kb & 3) == 0 || kb == kb_begin);
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, g.timeout_ns);
        w_ok = __shfl_sync(0xFFFFFFFFu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t bytes =
              kABytes + (kFP4 ? kBPBytes : kBBytes) + (sfa_new ? kSfaBytes : 0) + (kMX ? kSfbBytes : 0);
          // (FP4: the unpacking copy leaves the 8-byte gaps of each 16-byte
          // group unwritten and counts only the 16 KB of codes)
          mbar_arrive_expect_tx(&full[stage], bytes);
          const int kc = kb * kElemsPerKBlock;
          if (pair)   // 64 rows of A into both CTAs; the partner brings the other 64
            tma_load_3d_multicast(smem + kOffA + stage * kABytes + crank * (kABytes / 2), &map_a, &full[stage], kc,
                                  tl.tma_row + 64 * static_cast<int>(crank), a_e, 0x3);
          else
            tma_load_3d(smem + kOffA + stage * kABytes, &map_a, &full[stage], kc, tl.tma_row, a_e);
          // the whole B tile in one box: GEMM1 gate rows then up rows, GEMM2
          // 256 consecutive rows (MXFP4: the map counts 4-bit codes)
          uint8_t* bdst = smem + kOffB + stage * kBBytes;
          if (kStage == 1)
            tma_load_5d(bdst, &map_b, &full[stage], kc, 0, tl.nb, 0, tl.expert);
          else
            tma_load_3d(bdst, &map_b, &full[stage], kc, r0, tl.expert);
          if (sfa_new) {
            const int64_t chunk = kMX ? sf_chunk_offset(tl.sf_block, kb, k_blocks)
                                      : sf_chunk_offset(tl.sf_block, kb >> 2, sf_quads(k_blocks));
            bulk_load(smem + kOffSfa + stage * kSfaBytes, g.a_sf + chunk, kSfaBytes, &full[stage]);
          }
          if (kMX) {
            // B scale tile: the packed 512-byte chunks of the tile's two
            // 128-row weight blocks in one box (a block past the end of w2
            // reads as zeros: its weight rows are TMA zeros too)
            uint8_t* sfb = smem + kOffSfb + stage * kSfbBytes;
            if (kStage == 1)
              tma_load_5d(sfb, &map_wsf, &full[stage], 0, kb, tl.nb, 0, tl.expert);
            else
              tma_load_4d(sfb, &map_wsf, &full[stage], 0, kb, 2 * tl.nb, tl.expert);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok) {
      set_status(g.status, MOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    if (lane == 0) {
      // never leave the CTA with bulk copies still landing in its shared memory
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) {
          const int never = 0;
          mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, &never, g.timeout_ns);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0;
      int sf_stage = 0;   // FP8 1x128: the stage whose scale slot holds the current quad's scales
      bool ok = true;
      for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++iter) {
        const int seg = static_cast<int>(u % S);
        const int acc = kFP8 ? 0 : (iter & 1);
        const uint32_t acc_phase = kFP8 ? (iter & 1) : ((iter >> 1) & 1);
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, abort_flag, g.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kTileN);
        const int kb_begin = seg_begin(seg, S, k_blocks), kb_end = seg_begin(seg + 1, S, k_blocks);
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          const uint32_t first = kb == kb_begin;   // the segment's first K block starts the sum
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, g.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + kOffA + stage * kABytes);
          const uint32_t b_addr = smem_u32(smem + kOffB + stage * kBBytes);
          const uint64_t a_desc = smem_desc(a_addr, 16, 1024, kSwizzle128B);
          const uint64_t b_desc = smem_desc(b_addr, 16, 1024, kSwizzle128B);
          if (kFP8) {
            // scale tiles into tensor memory: every K block (MX), or once per
            // quad of K blocks (1x128: byte kb % 4 of each row's word)
            if (kMX || (kb & 3) == 0 || first) {
              const uint32_t sfa_t = tmem + kSfTmemCol + 32u * stage;
              const uint32_t sfb_t = sfa_t + 16u;
              const uint32_t sfa_s = smem_u32(smem + kOffSfa + stage * kSfaBytes);
              const uint32_t sfb_s = smem_u32(smem + kOffSfb + stage * kSfbBytes);
              tmem_cp_32x128b_x4(sfa_t, smem_desc(sfa_s, 16, 128, kSwizzleNone));
              tmem_cp_32x128b_x4(sfb_t, smem_desc(sfb_s, 16, 128, kSwizzleNone));
              tmem_cp_32x128b_x4(sfb_t + 4u, smem_desc(sfb_s + 512u, 16, 128, kSwizzleNone));
              sf_stage = stage;
            }
            const uint32_t sfa_t = tmem + kSfTmemCol + 32u * sf_stage;
            const uint32_t sfb_t = sfa_t + 16u;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t id = kMX ? static_cast<uint32_t>(k) : static_cast<uint32_t>(kb & 3);
              mma_fp8_block_scaled(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdescB | (id << 29) | (id << 4), sfa_t,
                                   sfb_t, !(first && k == 0));
            }
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kIdescBF16, !(first && k == 0));
          }
          if (pair)
            tc_commit_multicast(&empty[stage], 0x3);   // the stage's A halves live in both CTAs
          else
            tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
      }
      if (!ok) {
        set_status(g.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // all issued tensor-core work finished before the TMEM is released
      tc_commit(done);
      const int never = 0;
      mbar_wait_bounded(done, 0, &never, g.timeout_ns);
    }
  } else if (scale_warps(kFP8, kMX) && warp == 2 + epi_warps(kFP8, kStage, kSplit)) {
    // ------------------------------------------------------------------ weight-scale tiles (FP8)
    // B scale tile, written into the stage of a unit's first K block of each
    // quad q of K blocks: 256 rows, rows 0..127 of the first weight row block
    // and 128..255 of the second, each row's word holding the block's scales
    // of K blocks 4q .. 4q + 3 (byte j: K block 4q + j); 1 KB written by the
    // warp.  The warp arrives on every stage's barrier, beside the producer's
    // copies.
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // a weight row block's scales of K blocks 4q .. 4q + 3 as one word
    auto quad_word = [&](int64_t base, int q) {
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (4 * q + j < k_blocks) w |= static_cast<uint32_t>(g.w_sf[base + 4 * q + j]) << (8 * j);
      return w;
    };
    // weight-scale rows of a unit's two weight row blocks, and their words of
    // the 32 quads from the unit's first (one per lane); the next unit's are
    // read while the current unit's tiles are written
    auto unit_scales = [&](int64_t u, int64_t* base_sg, int64_t* base_su, uint32_t* sg, uint32_t* su) {
      const int64_t t = u / S;
      const int seg = static_cast<int>(u - t * S);
      const Tile tl = load_tile(g, t);
      int r0, r1;
      tile_b_rows<kStage>(g, tl, &r0, &r1);
      const int64_t base = static_cast<int64_t>(tl.expert) * g.w_rows_blocks;
      *base_sg = (base + min(r0 >> 7, g.w_rows_blocks - 1)) * g.w_k_groups;
      *base_su = (base + min(r1 >> 7, g.w_rows_blocks - 1)) * g.w_k_groups;
      const int q = (seg_begin(seg, S, k_blocks) >> 2) + lane;
      *sg = quad_word(*base_sg, q);
      *su = quad_word(*base_su, q);
    };
    int64_t nb_sg = 0, nb_su = 0;
    uint32_t n_sg = 0, n_su = 0;
    if (blockIdx.x < n_units) unit_scales(blockIdx.x, &nb_sg, &nb_su, &n_sg, &n_su);
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int64_t t = u / S;
      const int seg = static_cast<int>(u - t * S);
      const int64_t base_sg = nb_sg, base_su = nb_su;
      uint32_t sg_cache = n_sg, su_cache = n_su;
      if (u + gridDim.x < n_units) unit_scales(u + gridDim.x, &nb_sg, &nb_su, &n_sg, &n_su);
      const int kb_begin = seg_begin(seg, S, k_blocks), kb_end = seg_begin(seg + 1, S, k_blocks);
      int q0 = kb_begin >> 2;   // first quad of the lanes' words
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        const int q = kb >> 2;
        if (q - q0 == 32) {
          // the next 32 quads, one per lane
          q0 += 32;
          sg_cache = quad_word(base_sg, q0 + lane);
          su_cache = quad_word(base_su, q0 + lane);
        }
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, g.timeout_ns);
        w_ok = __shfl_sync(0xFFFFFFFFu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        if ((kb & 3) == 0 || kb == kb_begin) {
          const uint32_t sg = __shfl_sync(0xFFFFFFFFu, sg_cache, q - q0);
          const uint32_t su = __shfl_sync(0xFFFFFFFFu, su_cache, q - q0);
          const uint32_t word = lane < 16 ? sg : su;
          uint4* dst = reinterpret_cast<uint4*>(smem + kOffSfb + stage * kSfbBytes) + lane * 2;
          dst[0] = make_uint4(word, word, word, word);
          dst[1] = make_uint4(word, word, word, word);
          fence_proxy_async_smem();   // generic-proxy stores -> visible to the tensor-memory copy
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok) {
      set_status(g.status, MOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    // Eight warps: two per tensor-memory lane quadrant (warp % 4), each
    // owning half of the tile's columns.  A thread copies its accumulator
    // slice to registers and releases the accumulator before any math, so
    // the next tile's MMAs never wait on activation, quantisation or stores.
    constexpr int kEpiWarps = epi_warps(kFP8, kStage, kSplit);
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;  // 0 when there are four epilogue warps
    const int r = quad * 32 + lane;
    float* s_amax = reinterpret_cast<float*>(smem + kOffAmax);  // [2 parities][4 quads][2 halves][32]
    int iter = 0;
    uint32_t chunk_ctr = 0;   // GEMM2: staged chunks so far (staging tile and barrier parity)
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x, ++iter) {
      const int64_t t = u / S;
      const Tile tl = load_tile(g, t);
      const int acc = kFP8 ? 0 : (iter & 1);
      const uint32_t acc_phase = kFP8 ? (iter & 1) : ((iter >> 1) & 1);
      const bool got = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, g.timeout_ns);
      // warp-uniform decision, and the warp converged again before the
      // .sync.aligned tensor-memory loads
      if (!__all_sync(0xFFFFFFFFu, got)) {
        set_status(g.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + static_cast<uint32_t>(acc * kTileN) + (static_cast<uint32_t>(quad * 32) << 16);
      const bool row_ok = r < tl.valid;
      const int64_t row = tl.row0 + r;
      if constexpr (kSplit) {
        // ---- split K: this segment's sums of the valid rows go to the
        // partial buffer; the stage's reduce kernel, launched next, adds the
        // segments in order and applies the epilogue.
        const int seg = static_cast<int>(u - t * S);
        const bool quad_rows = quad * 32 < tl.valid;     // warp-uniform
        const int64_t vrow = g.block_vrow[t / g.n_blocks];
        float* prow = g.partial + (static_cast<int64_t>(seg) * g.part_rows + vrow + r) * g.part_cols +
                      static_cast<int64_t>(tl.nb) * 256;
        if (!quad_rows) {
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          continue;
        }
        {
          // the warp's 32 rows, all 256 accumulator columns, 32 at a time
          constexpr int kChunks = kTileN / 32;
#pragma unroll 1
          for (int c = 0; c < kChunks; ++c) {
            const uint32_t col = static_cast<uint32_t>(32 * c);
            uint32_t v32[32];
            tmem_ld_32x32b_x32(taddr + col, v32);
            tmem_ld_wait();
            if (c == kChunks - 1) {
              tc_fence_before();
              mbar_arrive(&tempty[acc]);
            }
            if (row_ok) {
              float4* d = reinterpret_cast<float4*>(prow + col);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                d[v] = make_float4(__uint_as_float(v32[4 * v]), __uint_as_float(v32[4 * v + 1]),
                                   __uint_as_float(v32[4 * v + 2]), __uint_as_float(v32[4 * v + 3]));
            }
          }
        }
        continue;
      }
      if (kStage == 1 && kEpiWarps == 4) {
        uint16_t* dst = static_cast<uint16_t*>(g.out) + row * g.out_ld + tl.nb * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t gv[32], uv[32];
          tmem_ld_32x32b_x32(taddr + c * 32, gv);
          tmem_ld_32x32b_x32(taddr + 128 + c * 32, uv);
          tmem_ld_wait();
          if (c == 3) {
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
          }
          if (row_ok) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int b = v * 8;
              float hv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) hv[i] = silu_mul(__uint_as_float(gv[b + i]), __uint_as_float(uv[b + i]));
              d4[v] = make_uint4(pack_bf16x2(hv[0], hv[1]), pack_bf16x2(hv[2], hv[3]), pack_bf16x2(hv[4], hv[5]),
                                 pack_bf16x2(hv[6], hv[7]));
            }
          }
        }
      } else if (kStage == 1) {
        // gate columns [64 * half, +64) and the matching up columns 128 later
        uint32_t g0[32], g1[32], u0[32], u1[32];
        const uint32_t c0 = static_cast<uint32_t>(64 * half);
        tmem_ld_32x32b_x32(taddr + c0, g0);
        tmem_ld_32x32b_x32(taddr + c0 + 32, g1);
        tmem_ld_32x32b_x32(taddr + 128 + c0, u0);
        tmem_ld_32x32b_x32(taddr + 128 + c0 + 32, u1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        float h[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          h[i] = silu_mul(__uint_as_float(g0[i]), __uint_as_float(u0[i]));
          h[32 + i] = silu_mul(__uint_as_float(g1[i]), __uint_as_float(u1[i]));
        }
        if (kMX) {
          // MXFP8: this thread's 64 columns are two whole 32-column blocks,
          // each with its own exponent; no exchange with the partner warp
          if (row_ok) {
            uint8_t* dstb = static_cast<uint8_t*>(g.out) + row * g.out_ld + tl.nb * 128 + 64 * half;
            uint32_t sfw = 0;
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
              float amax = 0.0f;
#pragma unroll
              for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[32 * blk + i]));
              const int s = ue8m0_exponent(amax);
              const float mul = exp2_neg(s);
              uint4* dst = reinterpret_cast<uint4*>(dstb + 32 * blk);
#pragma unroll
              for (int v = 0; v < 2; ++v) {
                const int b = 32 * blk + 16 * v;
                uint4 o;
                o.x = cvt_e4m3x2(h[b + 0] * mul, h[b + 1] * mul) | (cvt_e4m3x2(h[b + 2] * mul, h[b + 3] * mul) << 16);
                o.y = cvt_e4m3x2(h[b + 4] * mul, h[b + 5] * mul) | (cvt_e4m3x2(h[b + 6] * mul, h[b + 7] * mul) << 16);
                o.z = cvt_e4m3x2(h[b + 8] * mul, h[b + 9] * mul) |
                      (cvt_e4m3x2(h[b + 10] * mul, h[b + 11] * mul) << 16);
                o.w = cvt_e4m3x2(h[b + 12] * mul, h[b + 13] * mul) |
                      (cvt_e4m3x2(h[b + 14] * mul, h[b + 15] * mul) << 16);
                dst[v] = o;
              }
              sfw |= static_cast<uint32_t>(s + 127) << (8 * blk);
            }
            // bytes 2 * half and 2 * half + 1 of the row's scale word
            *reinterpret_cast<uint16_t*>(g.out_sf + sf_chunk_offset(tl.sf_block, tl.nb, g.out_groups) +
                                         sf_row_offset(r) + 2 * half) = static_cast<uint16_t>(sfw);
          }
        } else if (kFP8) {
          // 1x128 group = this thread's 64 columns + the partner warp's 64
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(h[i]));
          float* slot = s_amax + (((iter & 1) * 4 + quad) * 2) * 32;
          slot[half * 32 + lane] = amax;
          mbar_arrive(&xchg[quad]);
          if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&xchg[quad], iter & 1, abort_flag, g.timeout_ns))) {
            set_status(g.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          amax = fmaxf(amax, slot[(half ^ 1) * 32 + lane]);
          if (row_ok) {
            const int s = ue8m0_exponent(amax);
            const float mul = exp2_neg(s);
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<uint8_t*>(g.out) + row * g.out_ld + tl.nb * 128 + 64 * half);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 o;
              const int b = v * 16;
              o.x = cvt_e4m3x2(h[b + 0] * mul, h[b + 1] * mul) | (cvt_e4m3x2(h[b + 2] * mul, h[b + 3] * mul) << 16);
              o.y = cvt_e4m3x2(h[b + 4] * mul, h[b + 5] * mul) | (cvt_e4m3x2(h[b + 6] * mul, h[b + 7] * mul) << 16);
              o.z = cvt_e4m3x2(h[b + 8] * mul, h[b + 9] * mul) | (cvt_e4m3x2(h[b + 10] * mul, h[b + 11] * mul) << 16);
              o.w = cvt_e4m3x2(h[b + 12] * mul, h[b + 13] * mul) |
                    (cvt_e4m3x2(h[b + 14] * mul, h[b + 15] * mul) << 16);
              dst[v] = o;
            }
            if (half == 0) g.out_sf[sf_fp8_offset(tl.sf_block, tl.nb, g.out_groups, r)] = static_cast<uint8_t>(s + 127);
          }
        } else if (row_ok) {
          uint4* dst =
              reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.out) + row * g.out_ld + tl.nb * 128 + 64 * half);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const int b = v * 8;
            dst[v] = make_uint4(pack_bf16x2(h[b + 0], h[b + 1]), pack_bf16x2(h[b + 2], h[b + 3]),
                                pack_bf16x2(h[b + 4], h[b + 5]), pack_bf16x2(h[b + 6], h[b + 7]));
          }
        }
      } else {
        // y: blocks with at least half of their rows valid go through shared
        // memory and TMA stores (each 32-column chunk packed to bf16 into one
        // of two staging tiles -- 64-byte rows, 64-byte swizzle: 16-byte piece
        // j of row r at r * 64 + ((j ^ ((r >> 1) & 3)) * 16) -- then one
        // thread stores the 128 x 32 tile; rows past the valid count land in
        // the expert's padding (compact) or are clipped at max_m by the map
        // (masked)).  Sparser blocks (decode) store their valid rows directly.
        // FP8 (one accumulator): the thread first packs its whole row to
        // bf16 in registers and frees the accumulator, so the next tile's MMAs
        // do not wait for the stores.  BF16 (two accumulators) interleaves
        // tensor-memory loads and stores chunk by chunk.
        constexpr bool kEarly = kFP8;
        const int64_t col0 = static_cast<int64_t>(tl.nb) * kTileN;
        const bool use_tma = tl.valid >= kTileM / 2;     // uniform over the epilogue warps
        const bool issuer = warp == 2 && lane == 0;
        uint16_t* dst = static_cast<uint16_t*>(g.out) + row * g.out_ld + col0;
        bool ok = true;
        uint32_t pk[kEarly ? kTileN / 2 : 1];
        if constexpr (kEarly) {
#pragma unroll
          for (int c = 0; c < kTileN / 32; c += 2) {
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32(taddr + c * 32, v0);
            tmem_ld_32x32b_x32(taddr + (c + 1) * 32, v1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              pk[c * 16 + i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
              pk[(c + 1) * 16 + i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
        }
#pragma unroll
        for (int c = 0; c < kTileN / 32; ++c) {
          uint4 o[4];
          if constexpr (kEarly) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              o[v] = make_uint4(pk[c * 16 + 4 * v], pk[c * 16 + 4 * v + 1], pk[c * 16 + 4 * v + 2],
                                pk[c * 16 + 4 * v + 3]);
          } else {
            uint32_t v32[32];
            tmem_ld_32x32b_x32(taddr + c * 32, v32);
            tmem_ld_wait();
            if (c == kTileN / 32 - 1) {
              tc_fence_before();
              mbar_arrive(&tempty[acc]);
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int b = v * 8;
              o[v].x = pack_bf16x2(__uint_as_float(v32[b + 0]), __uint_as_float(v32[b + 1]));
              o[v].y = pack_bf16x2(__uint_as_float(v32[b + 2]), __uint_as_float(v32[b + 3]));
              o[v].z = pack_bf16x2(__uint_as_float(v32[b + 4]), __uint_as_float(v32[b + 5]));
              o[v].w = pack_bf16x2(__uint_as_float(v32[b + 6]), __uint_as_float(v32[b + 7]));
            }
          }
          if (!use_tma) {
            if (row_ok && col0 + c * 32 < g.n_total) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) d4[v] = o[v];
            }
            continue;
          }
          uint8_t* stg = smem + L::kOffStage + (chunk_ctr & 1) * L::kStageTileBytes + r * 64;
#pragma unroll
          for (int v = 0; v < 4; ++v) *reinterpret_cast<uint4*>(stg + ((v ^ ((r >> 1) & 3)) << 4)) = o[v];
          fence_proxy_async_smem();
          // the previous chunk's store has read its staging tile, so the next
          // chunk may overwrite it once everyone has passed this point
          if (issuer) bulk_wait_read_all();
          mbar_arrive(esync);
          const bool met = mbar_wait_bounded(esync, chunk_ctr & 1, abort_flag, g.timeout_ns);
          if (!__all_sync(0xFFFFFFFFu, met)) {
            ok = false;
            break;
          }
          if (issuer && col0 + c * 32 < g.n_total) {
            tma_store_3d(&map_out, smem + L::kOffStage + (chunk_ctr & 1) * L::kStageTileBytes,
                         static_cast<int32_t>(col0 + c * 32), tl.tma_row, g.masked ? tl.expert : 0);
            bulk_commit_group();
          }
          ++chunk_ctr;
        }
        if (!ok) {
          set_status(g.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
      }
    }
  }

  if (kStage == 2 && warp == 2 && lane == 0) bulk_wait_all();   // the TMA stores of y have completed
  // a pair leaves together: neither CTA's copies or MMA completions may still
  // be on their way to the other's shared memory
  if (pair)
    cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kFP8, bool kMX, int kStage, bool kFP4, bool kSplit>
cudaError_t launch_one(const GemmArgs& g, const GemmMaps& m, int grid, cudaStream_t s) {
  constexpr int kSmemBytes = Lay::kSmemBytes;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kFP8, kMX, kStage, kFP4, kSplit>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (g.pair)
    return launch_pdl_cluster(grouped_gemm_kernel<kFP8, kMX, kStage, kFP4, kSplit>, dim3(grid),
                              dim3(threads_for(kFP8, kMX, kStage, kSplit)), kSmemBytes, s, 2, m.a, m.b, m.out, m.wsf,
                              g);
  return launch_pdl(grouped_gemm_kernel<kFP8, kMX, kStage, kFP4, kSplit>, dim3(grid),
                    dim3(threads_for(kFP8, kMX, kStage, kSplit)), kSmemBytes, s, m.a, m.b, m.out, m.wsf, g);
}

// Co-resident two-CTA clusters of one (unsplit) kernel variant, x 2.
template <bool kFP8, bool kMX, int kStage, bool kFP4>
int pair_ctas_one() {
  static int cached = -1;
  if (cached >= 0) return cached;
  auto kernel = grouped_gemm_kernel<kFP8, kMX, kStage, kFP4, false>;
  constexpr int kSmemBytes = Lay::kSmemBytes;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess) return 0;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(threads_for(kFP8, kMX, kStage, false));
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    clusters = 0;
  }
  cached = 2 * clusters;
  return cached;
}

template <bool kFP8, bool kMX, bool kFP4>
int pair_ctas_stage(int stage) {
  return stage == 1 ? pair_ctas_one<kFP8, kMX, 1, kFP4>() : pair_ctas_one<kFP8, kMX, 2, kFP4>();
}

template <bool kFP8, bool kMX, bool kFP4, bool kSplit>
cudaError_t launch_stage(const GemmArgs& g, const GemmMaps& m, int grid, cudaStream_t s) {
  return g.stage == 1 ? launch_one<kFP8, kMX, 1, kFP4, kSplit>(g, m, grid, s)
                      : launch_one<kFP8, kMX, 2, kFP4, kSplit>(g, m, grid, s);
}

template <bool kSplit>
cudaError_t launch_dtype(const GemmArgs& g, const GemmMaps& m, int grid, cudaStream_t s) {
  if (g.fp4) return launch_stage<true, true, true, kSplit>(g, m, grid, s);
  if (g.mx) return launch_stage<true, true, false, kSplit>(g, m, grid, s);
  if (g.fp8) return launch_stage<true, false, false, kSplit>(g, m, grid, s);
  return launch_stage<false, false, false, kSplit>(g, m, grid, s);
}

__global__ void selftest_wait_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on this barrier: the wait must give up by itself
    if (!mbar_wait_bounded(&bar, 0, &abort_flag, timeout_ns)) set_status(status, MOE_ERR_TIMEOUT);
  }
}

}  // namespace


cudaError_t launch_gemm(const GemmArgs& g, const GemmMaps& m, int grid, cudaStream_t s) {
  return g.k_splits > 1 ? launch_dtype<true>(g, m, grid, s) : launch_dtype<false>(g, m, grid, s);
}

int gemm_pair_ctas(const GemmArgs& g) {
  if (g.fp4) return pair_ctas_stage<true, true, true>(g.stage);
  if (g.mx) return pair_ctas_stage<true, true, false>(g.stage);
  if (g.fp8) return pair_ctas_stage<true, false, false>(g.stage);
  return pair_ctas_stage<false, false, false>(g.stage);
}

cudaError_t launch_selftest_wait(int32_t* status, uint64_t timeout_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe
