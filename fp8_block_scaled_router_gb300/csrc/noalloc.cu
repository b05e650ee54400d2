// noalloc.cu -- moe_fp8_forward_noalloc: the few-row forward (gate/up with in-kernel hidden
// quantisation, then down fused with the combine) using a fixed scratch area compiled into
// the library instead of a caller-provided workspace.
//
// Why it exists: some callers cannot allocate device memory at the point where they run
// the layer -- code that runs while a memory pool is locked or being resized, callbacks
// that must not enter the allocator, or integrations that own no device allocator at all.
// For those callers the intermediate activation (FP8 codes + per-128 scales) lives in a
// file-scope __device__ array of kNoAllocScratchBytes (1 MiB) that every GPU which loads
// this library keeps until the process exits.
//
// Set-up: the first call in each CUDA context (with that context current) looks up the
// array's device address with cudaGetSymbolAddress and caches it under (device, context);
// make that first call before any stream capture. Host code never passes the array's
// host-side symbol to a kernel.
// Sharing: every call on a device uses the same array and leaves its contents behind; calls
// whose GPU work overlaps (different streams, no ordering between them) race on it. The
// status word at the start of the array is cleared on every call (an asynchronous memset
// on the caller's stream); no other part of the array needs to start at zero.
#include <cudaTypedefs.h>

#include <mutex>

#include "launch.h"


using namespace moe;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kMaxContexts = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address per (device, context) seen so far.
struct ScratchEntry {
  int dev;
  CUcontext ctx;
  void* ptr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_used = 0;

PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

// Layout inside the scratch array: header (256 B), act [R][I], act_scale [R][I/128].
size_t noalloc_bytes(int64_t R, int I) {
  return 256 + align256((size_t)(R * I)) + (size_t)(R * (I / 128)) * 4;
}

bool ok16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_fp8_forward_noalloc(const void* hidden, const int32_t* topk_ids,
                                                const float* topk_w, int32_t M, const uint8_t* w13,
                                                const float* w13_scale, const uint8_t* w2,
                                                const float* w2_scale, void* out,
                                                const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (!shape) return MOE_ERR_INVALID_ARG;
  if (moe_fp8_workspace_bytes(shape) == 0) return MOE_ERR_UNSUPPORTED;
  if (M < 0 || M > shape->max_tokens) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {hidden, topk_ids, topk_w, w13, w13_scale, w2, w2_scale, out};
  for (const void* p : ptrs)
    if (!p || !ok16(p)) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  const int H = shape->hidden, I = shape->inter, E = shape->num_experts, K = shape->top_k;
  const int64_t R = (int64_t)M * K;
  // limits: the few-row path only, and the activation must fit the scratch array
  if (!pair_capable(R) || noalloc_bytes(R, I) > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MOE_ERR_LAUNCH;
  void* base = nullptr;
  {
    CUcontext ctx = nullptr;
    auto get_ctx = ctx_get_current();
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return MOE_ERR_LAUNCH;
    if (!ctx) {  // no context current yet: the runtime's first symbol lookup creates the primary one
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || get_ctx(&ctx) != CUDA_SUCCESS || !ctx)
        return MOE_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    for (int i = 0; i < g_scratch_used; ++i)
      if (g_scratch[i].dev == dev && g_scratch[i].ctx == ctx) base = g_scratch[i].ptr;
    if (!base) {
      if (g_scratch_used == kMaxContexts) return MOE_ERR_LAUNCH;
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_LAUNCH;
      g_scratch[g_scratch_used++] = ScratchEntry{dev, ctx, p};
      base = p;
    }
  }
  char* b = static_cast<char*>(base);
  WsPtrs ws{};
  ws.hdr = reinterpret_cast<Header*>(b);
  ws.act = reinterpret_cast<uint8_t*>(b + 256);
  ws.act_scale = reinterpret_cast<float*>(b + 256 + align256((size_t)(R * I)));
  if (cudaMemsetAsync(ws.hdr, 0, sizeof(Header), stream) != cudaSuccess) return MOE_ERR_LAUNCH;
  if (launch_pair_gateup(w13, w13_scale, topk_ids, static_cast<const uint16_t*>(hidden), M, H, I, E, K, ws,
                         stream, w2, w2_scale) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  if (launch_pair_down(w2, w2_scale, topk_ids, topk_w, static_cast<uint16_t*>(out), M, H, I, E, K, ws,
                       stream) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  return MOE_OK;
}
