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
// Set-up: the first call on each device (with that device current) looks up the array's
// device address with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture. Host code never passes the array's host-side symbol to a kernel.
// Sharing: every call on a device uses the same array and leaves its contents behind; calls
// whose GPU work overlaps (different streams, no ordering between them) race on it. The
// status word at the start of the array is cleared on every call (an asynchronous memset
// on the caller's stream); no other part of the array needs to start at zero.
#include <mutex>

#include "common.cuh"

namespace moe {
cudaError_t launch_pair_gateup(const uint8_t* w13, const float* s13, const int32_t* ids,
                               const uint16_t* hidden, int M, int H, int I, int E, int K,
                               const WsPtrs& ws, cudaStream_t st, const uint8_t* w2 = nullptr,
                               const float* s2w = nullptr);
cudaError_t launch_pair_down(const uint8_t* w2, const float* s2w, const int32_t* ids, const float* topk_w,
                             uint16_t* out, int M, int H, int I, int E, int K, const WsPtrs& ws,
                             cudaStream_t st);
}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev[kMaxDevices] = {};

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
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_LAUNCH;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_dev[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_LAUNCH;
      g_scratch_dev[dev] = p;
    }
    base = g_scratch_dev[dev];
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
