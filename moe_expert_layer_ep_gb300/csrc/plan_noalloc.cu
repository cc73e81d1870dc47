// moe_plan_layout_noalloc: the layout step for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine): code
// embedded in a host framework whose memory planner owns the whole device
// heap and hands it only the tensors it reads and writes, or code running
// where an allocation would synchronise the device or re-enter that
// framework's allocator.  Such a caller can pass its inputs and outputs but
// cannot provide the layout step's scratch workspace.  This entry point keeps
// that scratch (the per-chunk expert histograms and in-chunk ranks) in a
// fixed-size array that lives in the library's device image: every GPU that
// loads the library holds it until the process exits.
//
// The kernels are the ones moe_plan_layout launches; only the scratch
// pointers differ.  The first call on a device looks up the array's device
// address (cudaGetSymbolAddress, with that device current) and caches it, so
// make that first call before any stream capture.  The cached address
// belongs to the device's primary context and stays valid as long as that
// context is not reset (cudaDeviceReset) while the library is loaded.  All
// calls share the one array, which keeps the contents of the last call:
// every scratch word is written before it is read within a call, so nothing
// needs clearing, but calls whose kernels overlap on the GPU (different
// streams, no ordering) race on it.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int64_t kScratchWords = int64_t(1) << 18;  // 1 MiB of int32
constexpr int kMaxDevices = 256;

}  // namespace

static __device__ __align__(256) int32_t g_plan_scratch[kScratchWords];

namespace {

std::mutex g_scratch_mutex;
int32_t* g_scratch_addr[kMaxDevices] = {};

// Device address of g_plan_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from the
// runtime, once per device.
moe_status_t scratch_on_current_device(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" moe_status_t moe_plan_layout_noalloc(const moe_shape_t* s, const int32_t* topk_ids,
                                                const moe_plan_outputs_t* out, void* stream) {
  if (!s || !out) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->topk <= 0 || s->E_global <= 0 || s->E_local <= 0 || s->expert_start < 0 ||
      static_cast<int64_t>(s->E_local) + s->expert_start > s->E_global)
    return MOE_ERR_INVALID_ARG;
  if (s->block_e != 128 || s->E_local > moe::kMaxLocalExperts || s->topk > moe::kMaxTopk)
    return MOE_ERR_UNSUPPORTED;
  int layout = s->layout;
  if (layout == MOE_LAYOUT_AUTO) layout = moe_choose_layout(s->E_global, s->E_local);
  if (layout != MOE_LAYOUT_COMPACT && layout != MOE_LAYOUT_MASKED) return MOE_ERR_INVALID_ARG;
  const bool masked = layout == MOE_LAYOUT_MASKED;
  if (masked && s->max_m < (s->T > 0 ? s->T : 1)) return MOE_ERR_INVALID_ARG;
  // masked row offsets e * max_m + pos are int32 in the outputs
  if (masked && static_cast<int64_t>(s->E_local) * s->max_m >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;

  const int64_t A = s->T * s->topk;
  const int64_t chunks = (A + moe::kPlanChunk - 1) / moe::kPlanChunk;
  if (A >= (int64_t(1) << 31) || chunks * s->E_local + A > kScratchWords) return MOE_ERR_BUFFER_TOO_SMALL;
  const int64_t all_tokens = masked ? 0 : moe_compact_all_tokens(A, s->E_local, s->block_e);
  const int64_t blocks = masked ? s->E_local * ((s->max_m + 127) / 128) : all_tokens / 128;

  if (!out->status || !out->meta || !out->counts) return MOE_ERR_INVALID_ARG;
  if ((A > 0 && (!topk_ids || !out->src2dst)) || (blocks > 0 && !out->block_info)) return MOE_ERR_INVALID_ARG;
  if (!masked && (!out->padded || !out->start || (all_tokens > 0 && !out->m_indices))) return MOE_ERR_INVALID_ARG;
  if (masked && !out->masked_m) return MOE_ERR_INVALID_ARG;
  if ((topk_ids && !aligned(topk_ids, 16)) || (out->block_info && !aligned(out->block_info, 16)) ||
      !aligned(out->status, 4) || !aligned(out->meta, 4) || !aligned(out->counts, 4) ||
      (out->src2dst && !aligned(out->src2dst, 4)) || (out->padded && !aligned(out->padded, 4)) ||
      (out->start && !aligned(out->start, 4)) || (out->masked_m && !aligned(out->masked_m, 4)) ||
      (out->m_indices && !aligned(out->m_indices, 4)))
    return MOE_ERR_MISALIGNED;

  int32_t* scratch = nullptr;
  moe_status_t st = scratch_on_current_device(&scratch);
  if (st != MOE_OK) return st;

  moe::PlanArgs p;
  memset(&p, 0, sizeof(p));
  p.topk_ids = topk_ids;
  p.A = A;
  p.E_global = s->E_global;
  p.E_local = s->E_local;
  p.expert_start = s->expert_start;
  p.masked = masked;
  p.max_m = s->max_m;
  p.all_tokens = all_tokens;
  p.blocks_per_expert = static_cast<int32_t>((s->max_m + 127) / 128);
  p.chunks = static_cast<int32_t>(chunks);
  p.status = out->status;
  p.meta = out->meta;
  p.counts = out->counts;
  p.padded = out->padded;
  p.start = out->start;
  p.masked_m = out->masked_m;
  p.m_indices = out->m_indices;
  p.src2dst = out->src2dst;
  p.block_info = out->block_info;
  p.chunk_hist = scratch;                           // [E_local, chunks]
  p.chunk_rank = scratch + chunks * s->E_local;     // [A]
  return moe::launch_plan(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
