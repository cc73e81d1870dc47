// C-ABI of libmoe: argument checks, workspace layout, TMA descriptors and the
// launch sequence.  Declarations and the contract of every call are in
// include/moe.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

struct moe_ctx {
  moe_shape_t shape;
  int layout;  // resolved: MOE_LAYOUT_COMPACT or MOE_LAYOUT_MASKED
  bool fp8;   // FP8 operands (1x128 / 128x128 or MXFP8 scales)
  bool mx;    // MXFP8 / MXFP4: 1x32 scales
  bool fp4;   // MXFP4: FP4 (E2M1) weights
  const void* w13;
  const uint8_t* w13_sf;
  const void* w2;
  const uint8_t* w2_sf;
  int device;
  int num_sms;
  moe_ws_layout_t ws;
  CUtensorMap map_w13;      // [E][gate, up][I/128][128][K]: one box = a GEMM1 tile's gate and up rows
  CUtensorMap map_w2;       // [E][K][I], 256-row boxes
  CUtensorMap map_w13_sf;   // MX: packed scale chunks as [E][gate, up][I/128][K/128][512 B]
  CUtensorMap map_w2_sf;    // MX: packed scale chunks as [E][K/128][I/128][512 B], two blocks per box
  // descriptors of the workspace activations, rebuilt when ws moves
  const void* ws_for_maps;
  CUtensorMap map_a;
  CUtensorMap map_h;
  CUtensorMap map_y;   // GEMM2 output, 32-column store boxes
  CUtensorMap map_a_half;   // compact: 64-row boxes of a and h (column-block pairs)
  CUtensorMap map_h_half;
  int pair_ctas[2];    // per GEMM stage: CTAs of a pair launch that fit at once (-1: not queried yet)
  uint64_t timeout_ns;
};

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// 3-D K-major tile map over [dim2][dim1][dim0] with a 128-byte inner box and
// box_rows rows, 128-byte swizzle (the layout the MMA descriptors expect).
// store64: a 64-byte inner box with 64-byte swizzle (the GEMM2 output stores).
moe_status_t make_map(CUtensorMap* map, const void* base, bool fp8, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                      bool store64 = false, uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  const uint64_t esize = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {dim0 * esize, dim0 * dim1 * esize};
  cuuint32_t box[3] = {static_cast<cuuint32_t>((store64 ? 64 : 128) / esize), box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  store64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// A tiled map of rank 2..5: dims[0] innermost (elements, contiguous),
// strides[i] the byte stride of dims[i + 1].
moe_status_t make_map_nd(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Weight maps.  GEMM1's B tile (gate rows nb*128.. and up rows I + nb*128..)
// is one box of the 5-d view [E][2][I/128][128][K]; GEMM2's (256 rows) one
// box of [E][K][I].  MXFP4 rows are packed (two codes per byte); the map
// unpacks them into the shared-memory layout of an E2M1 MMA operand.
moe_status_t make_weight_maps(moe_ctx* c, const void* w13, const void* w2) {
  const moe_shape_t& s = c->shape;
  // MXFP4: the map counts 4-bit codes and unpacks each 16 of them into a
  // 16-byte shared-memory group (the layout the MMA's E2M1 operand reads), so
  // a 128-code box fills a 128-byte swizzled row as an FP8 box does.
  const uint64_t es = c->fp8 ? 1 : 2, E = static_cast<uint64_t>(s.E_local);
  const CUtensorMapDataType dt = c->fp4  ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B
                                 : c->fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const uint32_t inner = static_cast<uint32_t>(128 / es);
  const uint64_t K = static_cast<uint64_t>(s.K), I = static_cast<uint64_t>(s.I);
  const uint64_t rb1 = c->fp4 ? K / 2 : K * es;   // w13 row bytes
  const uint64_t d1[5] = {K, 128, I / 128, 2, E};
  const uint64_t s1[4] = {rb1, 128 * rb1, I * rb1, 2 * I * rb1};
  const uint32_t b1[5] = {inner, 128, 1, 2, 1};
  moe_status_t st = make_map_nd(&c->map_w13, w13, dt, 5, d1, s1, b1, sw);
  if (st != MOE_OK) return st;
  const uint64_t rb2 = c->fp4 ? I / 2 : I * es;   // w2 row bytes
  const uint64_t d2[3] = {I, K, E};
  const uint64_t s2[2] = {rb2, K * rb2};
  const uint32_t b2[3] = {inner, 256, 1};
  st = make_map_nd(&c->map_w2, w2, dt, 3, d2, s2, b2, sw);
  if (st != MOE_OK || !c->mx) return st;
  // packed 512-byte scale chunks, chunk (e, row block b, K group k) at
  // ((e * row_blocks + b) * k_groups + k) * 512, read as 128 x u32
  const uint64_t kg1 = K / 128, kg2 = I / 128;
  const uint64_t ds1[5] = {128, kg1, I / 128, 2, E};
  const uint64_t ss1[4] = {512, kg1 * 512, (I / 128) * kg1 * 512, (2 * I / 128) * kg1 * 512};
  const uint32_t bs1[5] = {128, 1, 1, 2, 1};
  st = make_map_nd(&c->map_w13_sf, c->w13_sf, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, ds1, ss1, bs1,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != MOE_OK) return st;
  const uint64_t ds2[4] = {128, kg2, K / 128, E};
  const uint64_t ss2[3] = {512, kg2 * 512, (K / 128) * kg2 * 512};
  const uint32_t bs2[4] = {128, 1, 2, 1};
  return make_map_nd(&c->map_w2_sf, c->w2_sf, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, ds2, ss2, bs2,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

moe_status_t check_shape(const moe_shape_t* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->K <= 0 || s->I <= 0 || s->E_global <= 0 || s->E_local <= 0 || s->expert_start < 0 ||
      s->topk <= 0)
    return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s->E_local) + s->expert_start > s->E_global) return MOE_ERR_INVALID_ARG;
  if (s->dtype != MOE_DTYPE_FP8_E4M3_UE8M0 && s->dtype != MOE_DTYPE_BF16 && s->dtype != MOE_DTYPE_MXFP8 &&
      s->dtype != MOE_DTYPE_MXFP4)
    return MOE_ERR_INVALID_ARG;
  if (s->layout != MOE_LAYOUT_AUTO && s->layout != MOE_LAYOUT_COMPACT && s->layout != MOE_LAYOUT_MASKED)
    return MOE_ERR_INVALID_ARG;
  if (s->K % 128 || s->I % 128 || s->block_e != 128) return MOE_ERR_UNSUPPORTED;
  if (s->E_local > moe::kMaxLocalExperts || s->topk > moe::kMaxTopk) return MOE_ERR_UNSUPPORTED;
  if (s->T * s->topk >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Segments of a masked-layout GEMM's K loop.  Chosen from the tile shape
// alone (column tiles and K blocks, i.e. K, I and the dtype), never from T or
// max_m, so that a token's sums are formed the same way at every batch size:
// about 128 work units per expert (column tiles x segments), at least two K
// blocks per segment and at most kMaxKSplits segments.  A GEMM whose experts
// have 24 or more column tiles is not split: at the decode shapes (the w2
// GEMM, 28 tiles of 256 columns) the split measured slower at every batch
// size, while the w13 GEMM (16 tiles) gained.
int k_splits_for(int64_t n_blocks, int64_t k_blocks) {
  if (n_blocks >= 24) return 1;
  int64_t s = 128 / (n_blocks > 0 ? n_blocks : 1);
  if (s > k_blocks / 2) s = k_blocks / 2;
  if (s > moe::kMaxKSplits) s = moe::kMaxKSplits;
  return s < 1 ? 1 : static_cast<int>(s);
}

int64_t gemm_n_blocks(const moe_shape_t& s, int stage) { return stage == 1 ? s.I / 128 : (s.K + 255) / 256; }
int64_t gemm_k_blocks(const moe_shape_t& s, int stage, bool fp8) { return (stage == 1 ? s.K : s.I) / (fp8 ? 128 : 64); }

void compute_ws_layout(moe_ctx* c) {
  const moe_shape_t& s = c->shape;
  moe_ws_layout_t& w = c->ws;
  memset(&w, 0, sizeof(w));
  const int64_t A = s.T * s.topk;
  const int64_t E = s.E_local;
  w.layout = c->layout;
  if (c->layout == MOE_LAYOUT_COMPACT) {
    w.all_tokens = moe_compact_all_tokens(A, s.E_local, s.block_e);
    w.rows = w.all_tokens;
    w.blocks = w.all_tokens / 128;
  } else {
    const int64_t bpe = (s.max_m + 127) / 128;
    w.all_tokens = 0;
    w.rows = E * s.max_m;
    w.blocks = E * bpe;
  }
  w.chunks = static_cast<int32_t>((A + moe::kPlanChunk - 1) / moe::kPlanChunk);
  const uint64_t esize = c->fp8 ? 1 : 2;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t o = off;
    off = align_up(off + (bytes ? bytes : 1), 1024);
    return o;
  };
  w.status = take(16);
  w.meta = take(32);
  w.counts = take(4 * E);
  w.padded = take(4 * E);
  w.start = take(4 * E);
  w.masked_m = take(4 * E);
  w.m_indices = take(4 * static_cast<uint64_t>(w.all_tokens));
  w.src2dst = take(4 * static_cast<uint64_t>(A));
  w.block_info = take(16 * static_cast<uint64_t>(w.blocks));
  w.chunk_hist = take(4 * static_cast<uint64_t>(w.chunks) * E);
  w.chunk_rank = take(4 * static_cast<uint64_t>(A));
  w.a = take(static_cast<uint64_t>(w.rows) * s.K * esize);
  w.a_sf = take(c->fp8 ? static_cast<uint64_t>(w.blocks) * (s.K / 128) * 512 : 0);
  w.h = take(static_cast<uint64_t>(w.rows) * s.I * esize);
  w.h_sf = take(c->fp8 ? static_cast<uint64_t>(w.blocks) * (s.I / 128) * 512 : 0);
  w.y = take(static_cast<uint64_t>(w.rows) * s.K * 2);
  // masked layout: split-K tables and partial sums (see moe_ws_layout_t)
  const bool masked = c->layout == MOE_LAYOUT_MASKED;
  const int64_t nb1 = gemm_n_blocks(s, 1), nb2 = gemm_n_blocks(s, 2);
  w.k_splits1 = masked ? k_splits_for(nb1, gemm_k_blocks(s, 1, c->fp8)) : 1;
  w.k_splits2 = masked ? k_splits_for(nb2, gemm_k_blocks(s, 2, c->fp8)) : 1;
  const bool split = w.k_splits1 > 1 || w.k_splits2 > 1;
  w.partial_rows = split ? (A < w.rows ? A : w.rows) : 0;
  const uint64_t p1 = static_cast<uint64_t>(w.k_splits1 > 1 ? w.k_splits1 : 0) * nb1 * 256;
  const uint64_t p2 = static_cast<uint64_t>(w.k_splits2 > 1 ? w.k_splits2 : 0) * nb2 * 256;
  w.block_vrow = take(split ? 4 * static_cast<uint64_t>(w.blocks) : 0);
  w.partial = take(4 * static_cast<uint64_t>(w.partial_rows) * (p1 > p2 ? p1 : p2));
  w.total_bytes = off;
}

template <typename T>
T* at(void* ws, uint64_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t check_ws(const moe_ctx* c, const void* ws) {
  if (!c || !ws) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status_t ensure_ws_maps(moe_ctx* c, void* ws) {
  if (c->ws_for_maps == ws) return MOE_OK;
  const moe_shape_t& s = c->shape;
  const bool masked = c->layout == MOE_LAYOUT_MASKED;
  const uint64_t d1 = masked ? static_cast<uint64_t>(s.max_m) : static_cast<uint64_t>(c->ws.rows);
  const uint64_t d2 = masked ? static_cast<uint64_t>(s.E_local) : 1;
  if (c->ws.rows > 0) {
    moe_status_t st = make_map(&c->map_a, at<uint8_t>(ws, c->ws.a), c->fp8, s.K, d1, d2);
    if (st != MOE_OK) return st;
    st = make_map(&c->map_h, at<uint8_t>(ws, c->ws.h), c->fp8, s.I, d1, d2);
    if (st != MOE_OK) return st;
    st = make_map(&c->map_y, at<uint8_t>(ws, c->ws.y), false, s.K, d1, d2, true);
    if (st != MOE_OK) return st;
    if (!masked) {
      st = make_map(&c->map_a_half, at<uint8_t>(ws, c->ws.a), c->fp8, s.K, d1, d2, false, 64);
      if (st != MOE_OK) return st;
      st = make_map(&c->map_h_half, at<uint8_t>(ws, c->ws.h), c->fp8, s.I, d1, d2, false, 64);
      if (st != MOE_OK) return st;
    }
  }
  c->ws_for_maps = ws;
  return MOE_OK;
}

moe::GemmArgs gemm_args(const moe_ctx* c, void* ws, int stage) {
  const moe_shape_t& s = c->shape;
  moe::GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.block_info = at<int32_t>(ws, c->ws.block_info);
  g.meta = at<int32_t>(ws, c->ws.meta);
  g.status = at<int32_t>(ws, c->ws.status);
  g.stage = stage;
  g.fp8 = c->fp8;
  g.mx = c->mx;
  g.fp4 = c->fp4;
  g.masked = c->layout == MOE_LAYOUT_MASKED;
  g.blocks_per_expert = static_cast<int32_t>((s.max_m + 127) / 128);
  g.k_blocks = static_cast<int32_t>(gemm_k_blocks(s, stage, c->fp8));
  g.timeout_ns = c->timeout_ns;
  g.max_m = static_cast<int32_t>(s.max_m);
  g.k_splits = stage == 1 ? c->ws.k_splits1 : c->ws.k_splits2;
  if (g.k_splits > 1) {
    g.block_vrow = at<int32_t>(ws, c->ws.block_vrow);
    g.partial = at<float>(ws, c->ws.partial);
    g.part_rows = c->ws.partial_rows;
    g.part_cols = gemm_n_blocks(s, stage) * 256;
  }
  if (stage == 1) {
    g.n_blocks = static_cast<int32_t>(gemm_n_blocks(s, 1));
    g.n_half = s.I;
    g.n_total = s.I;
    g.w_rows_blocks = static_cast<int32_t>(2 * s.I / 128);
    g.w_k_groups = static_cast<int32_t>(s.K / 128);
    g.a_sf = at<uint8_t>(ws, c->ws.a_sf);
    g.w_sf = c->w13_sf;
    g.out = at<void>(ws, c->ws.h);
    g.out_ld = s.I;
    g.out_sf = at<uint8_t>(ws, c->ws.h_sf);
    g.out_groups = static_cast<int32_t>(s.I / 128);
  } else {
    g.n_blocks = static_cast<int32_t>(gemm_n_blocks(s, 2));
    g.n_half = 0;
    g.n_total = s.K;
    g.w_rows_blocks = static_cast<int32_t>(s.K / 128);
    g.w_k_groups = static_cast<int32_t>(s.I / 128);
    g.a_sf = at<uint8_t>(ws, c->ws.h_sf);
    g.w_sf = c->w2_sf;
    g.out = at<void>(ws, c->ws.y);
    g.out_ld = s.K;
  }
  return g;
}

}  // namespace

extern "C" {

int64_t moe_compact_all_tokens(int64_t num_assignments, int32_t num_experts, int32_t block_e) {
  if (num_assignments < 0 || num_experts < 0 || block_e <= 0) return -1;
  const int64_t nonempty = num_assignments < num_experts ? num_assignments : num_experts;
  return static_cast<int64_t>(block_e) * (nonempty + (num_assignments - nonempty) / block_e);
}

int32_t moe_choose_layout(int32_t E_global, int32_t E_local) {
  return (E_global > E_local && E_local <= 32) ? MOE_LAYOUT_MASKED : MOE_LAYOUT_COMPACT;
}

moe_status_t moe_ctx_create(const moe_shape_t* shape, const void* w13, const uint8_t* w13_sf, const void* w2,
                            const uint8_t* w2_sf, moe_ctx** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status_t st = check_shape(shape);
  if (st != MOE_OK) return st;
  const bool fp4 = shape->dtype == MOE_DTYPE_MXFP4;
  const bool mx = shape->dtype == MOE_DTYPE_MXFP8 || fp4;
  const bool fp8 = shape->dtype == MOE_DTYPE_FP8_E4M3_UE8M0 || mx;
  if (!w13 || !w2) return MOE_ERR_INVALID_ARG;
  if (fp8 != (w13_sf != nullptr) || fp8 != (w2_sf != nullptr)) return MOE_ERR_DTYPE_MISMATCH;
  if (!aligned16(w13) || !aligned16(w2)) return MOE_ERR_MISALIGNED;
  if (mx && (!aligned16(w13_sf) || !aligned16(w2_sf))) return MOE_ERR_MISALIGNED;
  // packed FP4 weights are read by TMA with 32-byte-aligned bases
  if (fp4 && ((reinterpret_cast<uintptr_t>(w13) & 31u) || (reinterpret_cast<uintptr_t>(w2) & 31u)))
    return MOE_ERR_MISALIGNED;
  int layout = shape->layout == MOE_LAYOUT_AUTO ? moe_choose_layout(shape->E_global, shape->E_local) : shape->layout;
  if (layout == MOE_LAYOUT_MASKED && shape->max_m < (shape->T > 0 ? shape->T : 1)) return MOE_ERR_INVALID_ARG;
  if (layout == MOE_LAYOUT_MASKED && static_cast<int64_t>(shape->E_local) * shape->max_m >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;

  moe_ctx* c = new (std::nothrow) moe_ctx;
  if (!c) return MOE_ERR_INVALID_ARG;
  memset(c, 0, sizeof(*c));
  c->shape = *shape;
  c->shape.layout = layout;
  c->layout = layout;
  c->fp8 = fp8;
  c->mx = mx;
  c->fp4 = fp4;
  c->w13 = w13;
  c->w13_sf = w13_sf;
  c->w2 = w2;
  c->w2_sf = w2_sf;
  c->timeout_ns = 2000000000ull;
  c->pair_ctas[0] = c->pair_ctas[1] = -1;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return MOE_ERR_CUDA;
  }
  compute_ws_layout(c);
  st = make_weight_maps(c, w13, w2);
  if (st != MOE_OK) {
    delete c;
    return st;
  }
  *out = c;
  return MOE_OK;
}

void moe_ctx_destroy(moe_ctx* ctx) { delete ctx; }

moe_status_t moe_workspace_layout(const moe_ctx* ctx, moe_ws_layout_t* out) {
  if (!ctx || !out) return MOE_ERR_INVALID_ARG;
  *out = ctx->ws;
  return MOE_OK;
}

moe_status_t moe_workspace_size(const moe_ctx* ctx, size_t* bytes) {
  if (!ctx || !bytes) return MOE_ERR_INVALID_ARG;
  *bytes = static_cast<size_t>(ctx->ws.total_bytes);
  return MOE_OK;
}

// Arguments of the layout step; checks the routing pointer.
static moe_status_t plan_args(moe_ctx* ctx, const int32_t* topk_ids, void* ws, moe::PlanArgs* out) {
  moe_status_t st = check_ws(ctx, ws);
  if (st != MOE_OK) return st;
  const moe_shape_t& s = ctx->shape;
  const int64_t A = s.T * s.topk;
  if (A > 0 && !topk_ids) return MOE_ERR_INVALID_ARG;
  if (topk_ids && !aligned16(topk_ids)) return MOE_ERR_MISALIGNED;
  moe::PlanArgs& p = *out;
  memset(&p, 0, sizeof(p));
  p.topk_ids = topk_ids;
  p.A = A;
  p.E_global = s.E_global;
  p.E_local = s.E_local;
  p.expert_start = s.expert_start;
  p.masked = ctx->layout == MOE_LAYOUT_MASKED;
  p.max_m = s.max_m;
  p.all_tokens = ctx->ws.all_tokens;
  p.blocks_per_expert = static_cast<int32_t>((s.max_m + 127) / 128);
  p.chunks = ctx->ws.chunks;
  p.status = at<int32_t>(ws, ctx->ws.status);
  p.meta = at<int32_t>(ws, ctx->ws.meta);
  p.counts = at<int32_t>(ws, ctx->ws.counts);
  p.padded = at<int32_t>(ws, ctx->ws.padded);
  p.start = at<int32_t>(ws, ctx->ws.start);
  p.masked_m = at<int32_t>(ws, ctx->ws.masked_m);
  p.m_indices = at<int32_t>(ws, ctx->ws.m_indices);
  p.src2dst = at<int32_t>(ws, ctx->ws.src2dst);
  p.block_info = at<int32_t>(ws, ctx->ws.block_info);
  p.chunk_hist = at<int32_t>(ws, ctx->ws.chunk_hist);
  p.chunk_rank = at<int32_t>(ws, ctx->ws.chunk_rank);
  if (ctx->ws.partial_rows > 0) p.block_vrow = at<int32_t>(ws, ctx->ws.block_vrow);
  return MOE_OK;
}

// Arguments of the quant-scatter step; checks the activation pointer.
// topk_ids (moe_forward's small problems): destinations formed from the
// routing instead of read from src2dst.
static moe_status_t quant_args(moe_ctx* ctx, const void* x_bf16, const int32_t* topk_ids, void* ws,
                               moe::QuantArgs* out) {
  moe_status_t st = check_ws(ctx, ws);
  if (st != MOE_OK) return st;
  const moe_shape_t& s = ctx->shape;
  if (s.T > 0 && !x_bf16) return MOE_ERR_INVALID_ARG;
  if (x_bf16 && !aligned16(x_bf16)) return MOE_ERR_MISALIGNED;
  moe::QuantArgs& q = *out;
  memset(&q, 0, sizeof(q));
  q.x = x_bf16;
  q.src2dst = at<int32_t>(ws, ctx->ws.src2dst);
  q.T = s.T;
  q.K = s.K;
  q.topk = s.topk;
  q.fp8 = ctx->fp8;
  q.mx = ctx->mx;
  q.masked = ctx->layout == MOE_LAYOUT_MASKED;
  q.max_m = s.max_m;
  q.blocks_per_expert = static_cast<int32_t>((s.max_m + 127) / 128);
  q.a = at<void>(ws, ctx->ws.a);
  q.a_sf = at<uint8_t>(ws, ctx->ws.a_sf);
  q.topk_ids = topk_ids;
  q.E_global = s.E_global;
  q.E_local = s.E_local;
  q.expert_start = s.expert_start;
  return MOE_OK;
}

moe_status_t moe_plan_layout(moe_ctx* ctx, const int32_t* topk_ids, void* ws, void* stream) {
  moe::PlanArgs p;
  const moe_status_t st = plan_args(ctx, topk_ids, ws, &p);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_plan(p, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quant_scatter(moe_ctx* ctx, const void* x_bf16, void* ws, void* stream) {
  moe::QuantArgs q;
  const moe_status_t st = quant_args(ctx, x_bf16, nullptr, ws, &q);
  if (st != MOE_OK) return st;
  return cuda_status(moe::launch_quant_scatter(q, static_cast<cudaStream_t>(stream)));
}

static moe_status_t run_gemm(moe_ctx* ctx, void* ws, void* stream, int stage) {
  moe_status_t st = check_ws(ctx, ws);
  if (st != MOE_OK) return st;
  if (ctx->ws.blocks == 0) return MOE_OK;
  st = ensure_ws_maps(ctx, ws);
  if (st != MOE_OK) return st;
  moe::GemmArgs g = gemm_args(ctx, ws, stage);
  int64_t max_tiles = ctx->ws.blocks * g.n_blocks * g.k_splits;
  // FP8 kinds, compact, unsplit, an even number of column blocks: column-block
  // pairs share their A tile through cluster multicast (measured 1-2% faster
  // per step on the FP8 prefills; no gain on BF16, which stays unpaired)
  const bool pairable = g.fp8 && !g.masked && g.k_splits == 1 && g.n_blocks % 2 == 0;
  int& pair_ctas = ctx->pair_ctas[stage - 1];
  if (pairable && pair_ctas < 0) pair_ctas = moe::gemm_pair_ctas(g);
  g.pair = pairable && pair_ctas >= 2;
  int grid = g.pair ? (pair_ctas < ctx->num_sms ? pair_ctas : ctx->num_sms) & ~1 : ctx->num_sms;
  if (max_tiles < grid) grid = static_cast<int>(max_tiles);   // (even when paired: n_blocks is)
  moe::GemmMaps m;
  if (g.pair)
    m.a = stage == 1 ? ctx->map_a_half : ctx->map_h_half;
  else
    m.a = stage == 1 ? ctx->map_a : ctx->map_h;
  m.b = stage == 1 ? ctx->map_w13 : ctx->map_w2;
  m.out = stage == 1 ? ctx->map_a : ctx->map_y;   // stage 1 stores through plain writes
  m.wsf = ctx->mx ? (stage == 1 ? ctx->map_w13_sf : ctx->map_w2_sf) : m.b;   // (not read without MX scales)
  cudaError_t e = moe::launch_gemm(g, m, grid, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess && g.k_splits > 1)
    e = moe::launch_split_reduce(g, ctx->ws.blocks * g.n_blocks, static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

moe_status_t moe_grouped_gemm_w13_act(moe_ctx* ctx, void* ws, void* stream) { return run_gemm(ctx, ws, stream, 1); }

moe_status_t moe_grouped_gemm_w2(moe_ctx* ctx, void* ws, void* stream) { return run_gemm(ctx, ws, stream, 2); }

moe_status_t moe_combine(moe_ctx* ctx, const float* topk_weights, const void* ws, void* out_bf16, void* stream) {
  moe_status_t st = check_ws(ctx, ws);
  if (st != MOE_OK) return st;
  const moe_shape_t& s = ctx->shape;
  if (s.T > 0 && (!topk_weights || !out_bf16)) return MOE_ERR_INVALID_ARG;
  if ((topk_weights && !aligned16(topk_weights)) || (out_bf16 && !aligned16(out_bf16))) return MOE_ERR_MISALIGNED;
  moe::CombineArgs c;
  c.y = at<const void>(const_cast<void*>(ws), ctx->ws.y);
  c.src2dst = at<const int32_t>(const_cast<void*>(ws), ctx->ws.src2dst);
  c.topk_weights = topk_weights;
  c.T = s.T;
  c.K = s.K;
  c.topk = s.topk;
  c.out = out_bf16;
  return cuda_status(moe::launch_combine(c, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_forward(moe_ctx* ctx, const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                         void* ws, void* out_bf16, void* stream) {
  moe_status_t st;
  if (ctx && moe::plan_is_small(ctx->shape.T * ctx->shape.topk, ctx->shape.E_local)) {
    // small problems: the plan and the quant-scatter in one launch, the
    // quantising CTAs forming their tokens' destinations from the routing
    moe::PlanArgs p;
    moe::QuantArgs q;
    if ((st = plan_args(ctx, topk_ids, ws, &p)) != MOE_OK) return st;
    if ((st = quant_args(ctx, x_bf16, topk_ids, ws, &q)) != MOE_OK) return st;
    if ((st = cuda_status(moe::launch_plan_quant_small(p, q, static_cast<cudaStream_t>(stream)))) != MOE_OK)
      return st;
  } else {
    if ((st = moe_plan_layout(ctx, topk_ids, ws, stream)) != MOE_OK) return st;
    if ((st = moe_quant_scatter(ctx, x_bf16, ws, stream)) != MOE_OK) return st;
  }
  if ((st = moe_grouped_gemm_w13_act(ctx, ws, stream)) != MOE_OK) return st;
  if ((st = moe_grouped_gemm_w2(ctx, ws, stream)) != MOE_OK) return st;
  return moe_combine(ctx, topk_weights, ws, out_bf16, stream);
}

int32_t moe_forward_launches(const moe_ctx* ctx) {
  if (!ctx) return -1;
  const moe_shape_t& s = ctx->shape;
  int n;
  if (moe::plan_is_small(s.T * s.topk, s.E_local))
    n = 1 + (s.T > 0 ? 1 : 0);                  // plan + quant in one launch, combine
  else
    n = moe::plan_launch_count(s.T * s.topk, s.E_local) + (s.T > 0 ? 2 : 0);   // plan, quant + combine
  if (ctx->ws.blocks > 0) {
    n += 2;                                     // two GEMMs
    n += (ctx->ws.k_splits1 > 1) + (ctx->ws.k_splits2 > 1);   // their split-K reductions
  }
  return n;
}

moe_status_t moe_read_device_status(const void* ws, void* stream, int32_t* out) {
  if (!ws || !out) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(cudaMemcpy(out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost));
}

moe_status_t moe_clear_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, 16, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_selftest_wait_timeout(void* ws, int64_t timeout_ns, void* stream) {
  if (!ws || timeout_ns <= 0) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_selftest_wait(static_cast<int32_t*>(ws), static_cast<uint64_t>(timeout_ns),
                                               static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_requant_weights_ue8m0(const uint8_t* w_in, const float* scale_in, uint8_t* w_out,
                                       uint8_t* scale_out, int64_t E, int64_t N, int64_t C, void* stream) {
  if (E < 0 || N < 0 || C < 0) return MOE_ERR_INVALID_ARG;
  if (N % 128 || C % 128) return MOE_ERR_UNSUPPORTED;
  if (E * N * C == 0) return MOE_OK;
  if (!w_in || !scale_in || !w_out || !scale_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_in) || !aligned16(w_out) || (reinterpret_cast<uintptr_t>(scale_in) & 3u)) return MOE_ERR_MISALIGNED;
  return cuda_status(moe::launch_requant(w_in, scale_in, w_out, scale_out, E, N, C, static_cast<cudaStream_t>(stream)));
}

int64_t moe_route_workspace_size(int64_t T, int64_t K, int32_t E_global) {
  if (T < 0 || K <= 0 || E_global <= 0) return -1;
  const int64_t segs = (K + moe::kRouterSegment - 1) / moe::kRouterSegment;
  return 256 + static_cast<int64_t>(align_up(static_cast<uint64_t>(segs * T * E_global) * 4, 256));
}

moe_status_t moe_router_prepare(const float* w_router, void* w_planes, int64_t E_global, int64_t K, void* stream) {
  if (E_global <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 128) return MOE_ERR_UNSUPPORTED;
  if (!w_router || !w_planes) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_router) || !aligned16(w_planes)) return MOE_ERR_MISALIGNED;
  return cuda_status(moe::launch_router_split(w_router, static_cast<uint16_t*>(w_planes), E_global, K,
                                              static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_route(const void* x_bf16, const void* w_planes, int64_t T, int64_t K, int32_t E_global, int32_t topk,
                       float* logits, int32_t* topk_ids, float* topk_weights, void* ws, int64_t ws_bytes,
                       void* stream) {
  if (T < 0 || K <= 0 || E_global <= 0 || topk <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 128 || E_global > moe::kMaxRouterExperts || topk > moe::kMaxTopk || topk > E_global ||
      T > (int64_t(1) << 30))
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x_bf16 || !w_planes || !logits || !topk_ids || !topk_weights || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(w_planes) || !aligned16(logits) || !aligned16(topk_ids) ||
      !aligned16(topk_weights) || !aligned16(ws))
    return MOE_ERR_MISALIGNED;
  if (ws_bytes < moe_route_workspace_size(T, K, E_global)) return MOE_ERR_BUFFER_TOO_SMALL;
  CUtensorMap map_x, map_w;
  moe_status_t st = make_map(&map_x, x_bf16, false, static_cast<uint64_t>(K), static_cast<uint64_t>(T), 1);
  if (st == MOE_OK)
    st = make_map(&map_w, w_planes, false, static_cast<uint64_t>(K), static_cast<uint64_t>(E_global), 3);
  if (st != MOE_OK) return st;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe::RouterArgs r;
  memset(&r, 0, sizeof(r));
  r.T = T;
  r.K = K;
  r.E = E_global;
  r.segs = static_cast<int32_t>((K + moe::kRouterSegment - 1) / moe::kRouterSegment);
  r.m_tiles = static_cast<int32_t>((T + 127) / 128);
  r.n_tiles = (E_global + 127) / 128;
  r.fold = moe::router_folds(T, E_global, sms) ? 1 : 0;
  r.status = static_cast<int32_t*>(ws);
  r.partial = r.fold ? nullptr : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  r.z = logits;
  r.timeout_ns = 2000000000ull;
  const int64_t items = static_cast<int64_t>(r.m_tiles) * r.n_tiles * (r.fold ? 1 : r.segs);
  const int grid = static_cast<int>(items < sms ? items : sms);
  return cuda_status(moe::launch_route(map_x, map_w, r, grid, topk, logits, topk_ids, topk_weights,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_pack_mx_scales(const uint8_t* src, int64_t src_ld, uint8_t* dst, int64_t E, int64_t N, int64_t C,
                                void* stream) {
  if (E < 0 || N < 0 || C < 0 || src_ld < C / 32 || src_ld % 4) return MOE_ERR_INVALID_ARG;
  if (N % 128 || C % 128) return MOE_ERR_UNSUPPORTED;
  if (E * N * C == 0) return MOE_OK;
  if (!src || !dst) return MOE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_MISALIGNED;
  const int64_t src_bytes = E * N * src_ld, dst_bytes = E * N * (C / 32);
  if (src < dst + dst_bytes && dst < src + src_bytes) return MOE_ERR_INVALID_ARG;   // overlap
  return cuda_status(moe::launch_pack_mx_scales(src, src_ld, dst, E, N, C, static_cast<cudaStream_t>(stream)));
}

int64_t moe_sf_offset(int64_t block, int64_t group, int64_t n_groups, int32_t row) {
  return moe::sf_fp8_offset(block, group, n_groups, row);
}

const char* moe_strerror(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MOE_ERR_BUFFER_TOO_SMALL: return "buffer too small";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_EXPERT_ID: return "expert id outside [-1, E_global)";
    case MOE_ERR_MASKED_OVERFLOW: return "masked expert received more than max_m rows";
    case MOE_ERR_TIMEOUT: return "bounded wait inside a kernel timed out";
    case MOE_ERR_DTYPE_MISMATCH: return "weights contradict the declared dtype";
  }
  return "unknown status";
}

}  // extern "C"
