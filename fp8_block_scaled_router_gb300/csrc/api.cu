// api.cu -- the C ABI (include/moe_fp8.h): host-side validation, workspace layout and the
// launch sequence. No call allocates, frees or reads device memory; only the host-buffer
// call with pageable (not page-locked) buffers blocks, in the driver's staged copies.
//
// Sources: "NetraRuntime/netra-kernel" README (stable C ABI that launches on a
// caller-provided stream; exact profile guards, unsupported contracts are refused) and
// older kernel-lab README "Design" (dispatch without allocation, synchronisation,
// filesystem access, environment parsing or symbol lookup); docs/compiler/architecture.md
// (caller-local kernel arguments so concurrent calls cannot mix pointers).
#include <cstdint>

#include <cmath>

#include "launch.h"


using namespace moe;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Device address of page-locked (pinned or registered) host memory, or null for any other
// pointer (pageable host memory, device memory, unknown).
const void* device_view(const void* host) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The compiled contract set.
bool shape_supported(const moe_fp8_shape_t* s) {
  if (!s) return false;
  const int H = s->hidden, I = s->inter, E = s->num_experts, K = s->top_k;
  if (H < 256 || H > 8192 || H % 256) return false;
  if (I < 128 || I > 4096 || I % 128) return false;
  if (!(E == 8 || E == 16 || E == 32 || E == 64 || E == 128 || E == 256)) return false;
  if (K < 1 || K > 16 || K > E) return false;
  if (s->max_tokens < 1 || s->max_tokens > (1 << 20) / K) return false;
  return true;
}

moe_status_t check_common(const moe_fp8_shape_t* s, int32_t M) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(s)) return MOE_ERR_UNSUPPORTED;
  if (M < 0 || M > s->max_tokens) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t check_ws(void* ws, size_t bytes, const moe_fp8_shape_t* s, Layout* L) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  *L = make_layout(*s);
  if (bytes < L->total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t launched(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH; }

// The RMSNorm arguments: gamma a 16-byte aligned device pointer, eps finite and > 0 (eps = 0
// would turn an all-zero row into 0 * inf = NaN).
moe_status_t check_norm(const void* norm_weight, float eps, Norm* nm) {
  if (!norm_weight || !aligned16(norm_weight)) return MOE_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || !std::isfinite(eps)) return MOE_ERR_INVALID_ARG;
  *nm = Norm{static_cast<const uint16_t*>(norm_weight), eps};
  return MOE_OK;
}

moe_status_t route_impl(const void* hidden, Norm nm, const void* router_w, const float* bias, int32_t M,
                        const moe_fp8_shape_t* shape, int32_t renormalize, int32_t* topk_ids, float* topk_w,
                        cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!hidden || !router_w || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(router_w) || !aligned16(topk_ids) || !aligned16(topk_w) ||
      (bias && !aligned16(bias)))
    return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  return launched(launch_route(static_cast<const uint16_t*>(hidden), nm, static_cast<const uint16_t*>(router_w), bias,
                               M, shape->hidden, shape->num_experts, shape->top_k, renormalize ? 1 : 0, topk_ids,
                               topk_w, stream));
}

moe_status_t forward_impl(const void* hidden, Norm nm, const int32_t* topk_ids, const float* topk_w, int32_t M,
                          const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                          void* out, void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                          cudaStream_t stream);

}  // namespace

extern "C" {

const char* moe_fp8_version(void) { return "moe_fp8 0.1.0 (sm_103a)"; }

size_t moe_fp8_workspace_bytes(const moe_fp8_shape_t* shape) {
  if (!shape_supported(shape)) return 0;
  return make_layout(*shape).total;
}

moe_status_t moe_fp8_workspace_init(void* workspace, size_t workspace_bytes,
                                    const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (!shape) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  // the status word and the single-launch path's arrival tickets (contiguous)
  return launched(cudaMemsetAsync(static_cast<char*>(workspace) + L.header, 0, L.qa - L.header, stream));
}

moe_status_t moe_route(const void* hidden, const void* router_w, const float* bias, int32_t M,
                       const moe_fp8_shape_t* shape, int32_t renormalize, int32_t* topk_ids,
                       float* topk_w, cudaStream_t stream) {
  return route_impl(hidden, Norm{nullptr, 0.0f}, router_w, bias, M, shape, renormalize, topk_ids, topk_w, stream);
}

moe_status_t moe_norm_route(const void* hidden, const void* norm_weight, float eps, const void* router_w,
                            const float* bias, int32_t M, const moe_fp8_shape_t* shape, int32_t renormalize,
                            int32_t* topk_ids, float* topk_w, cudaStream_t stream) {
  Norm nm;
  if (moe_status_t st = check_norm(norm_weight, eps, &nm)) return st;
  return route_impl(hidden, nm, router_w, bias, M, shape, renormalize, topk_ids, topk_w, stream);
}

moe_status_t moe_rmsnorm(const void* hidden, const void* norm_weight, float eps, int32_t M, void* out,
                         const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  Norm nm;
  if (moe_status_t st = check_norm(norm_weight, eps, &nm)) return st;
  if (!hidden || !out || !aligned16(hidden) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  return launched(launch_rmsnorm(static_cast<const uint16_t*>(hidden), nm, M, shape->hidden,
                                 static_cast<uint16_t*>(out), stream));
}

moe_status_t moe_fp8_prepare(const void* hidden, const int32_t* topk_ids, int32_t M,
                             void* workspace, size_t workspace_bytes,
                             const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!hidden || !topk_ids || !aligned16(hidden) || !aligned16(topk_ids)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const WsPtrs ws = ws_ptrs(workspace, L);
  const int64_t R = (int64_t)M * shape->top_k;
  if (use_pair_mode(R))
    return launched(launch_prep(static_cast<const uint16_t*>(hidden), topk_ids, M, shape->hidden,
                                shape->num_experts, shape->top_k, ws, stream));
  return launched(launch_sort_gather(static_cast<const uint16_t*>(hidden), Norm{nullptr, 0.0f}, topk_ids, M, shape->hidden,
                                     shape->num_experts, shape->top_k, ws, stream));
}

moe_status_t moe_fp8_gate_up(const uint8_t* w13, const float* w13_scale, int32_t M,
                             void* workspace, size_t workspace_bytes,
                             const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!w13 || !w13_scale || !aligned16(w13) || !aligned16(w13_scale)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const WsPtrs ws = ws_ptrs(workspace, L);
  const int64_t R = (int64_t)M * shape->top_k;
  if (use_pair_mode(R))
    return launched(launch_pair_gateup(w13, w13_scale, ws.pair_expert, nullptr, M, shape->hidden,
                                       shape->inter, shape->num_experts, shape->top_k, ws, stream));
  if (use_group_mode(R))
    return launched(launch_gpair_gateup(false, w13, w13_scale, R, shape->hidden, shape->inter, shape->num_experts,
                                        L.max_groups, ws, stream));
  return launched(launch_grouped_gateup(w13, w13_scale, R, shape->hidden, shape->inter, shape->num_experts,
                                        max_tiles_for(R, shape->num_experts, kTileRows), ws, stream));
}

moe_status_t moe_fp8_down(const uint8_t* w2, const float* w2_scale, int32_t M, void* workspace,
                          size_t workspace_bytes, const moe_fp8_shape_t* shape,
                          cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!w2 || !w2_scale || !aligned16(w2) || !aligned16(w2_scale)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const WsPtrs ws = ws_ptrs(workspace, L);
  const int64_t R = (int64_t)M * shape->top_k;
  if (use_pair_mode(R))
    return launched(launch_pair_down(w2, w2_scale, ws.pair_expert, nullptr, nullptr, M, shape->hidden,
                                     shape->inter, shape->num_experts, shape->top_k, ws, stream));
  if (use_group_mode(R))
    return launched(launch_gpair_down(false, w2, w2_scale, R, shape->hidden, shape->inter, shape->num_experts,
                                      L.max_groups, ws, stream));
  return launched(launch_grouped_down(w2, w2_scale, R, shape->hidden, shape->inter, shape->num_experts,
                                      max_tiles_for(R, shape->num_experts, kTileRows), ws, stream));
}

moe_status_t moe_fp8_combine(const float* topk_w, int32_t M, void* out, void* workspace,
                             size_t workspace_bytes, const moe_fp8_shape_t* shape,
                             cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!topk_w || !out || !aligned16(topk_w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const WsPtrs ws = ws_ptrs(workspace, L);
  return launched(launch_combine(topk_w, M, shape->hidden, shape->top_k, static_cast<uint16_t*>(out),
                                 ws, stream));
}

}  // extern "C"

namespace {
moe_status_t forward_impl(const void* hidden, Norm nm, const int32_t* topk_ids, const float* topk_w, int32_t M,
                          const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                          void* out, void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                          cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!hidden || !topk_ids || !topk_w || !w13 || !w13_scale || !w2 || !w2_scale || !out)
    return MOE_ERR_INVALID_ARG;
  for (const void* p : {hidden, (const void*)topk_ids, (const void*)topk_w, (const void*)w13,
                        (const void*)w13_scale, (const void*)w2, (const void*)w2_scale, (const void*)out})
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const int H = shape->hidden, I = shape->inter, E = shape->num_experts, K = shape->top_k;
  const WsPtrs ws = ws_ptrs(workspace, L);
  const int64_t R = (int64_t)M * K;
  if (use_pair_mode(R)) {
    // few routed rows: two launches -- gate/up quantises its own hidden row (through the
    // norm, if any) and prefetches the routed experts' down weights into L2, down is fused
    // with the combine (same arithmetic as the four stage calls)
    if (moe_status_t st = launched(launch_pair_gateup(w13, w13_scale, topk_ids, static_cast<const uint16_t*>(hidden),
                                                      M, H, I, E, K, ws, stream, w2, w2_scale, nm)))
      return st;
    return launched(launch_pair_down(w2, w2_scale, topk_ids, topk_w, static_cast<uint16_t*>(out), M, H, I, E, K,
                                     ws, stream));
  }
  // more routed rows: quantise (through the norm, if any) and sort by expert; then the
  // expert-grouped pair kernels (groups of up to 16 rows) or, for many rows, the two tile
  // GEMMs over 128-row tiles; the slot-order combine
  if (moe_status_t st = launched(launch_sort_gather(static_cast<const uint16_t*>(hidden), nm, topk_ids, M, H, E, K,
                                                    ws, stream)))
    return st;
  if (use_group_mode(R)) {
    if (moe_status_t st = launched(launch_gpair_gateup(false, w13, w13_scale, R, H, I, E, L.max_groups, ws, stream)))
      return st;
    if (moe_status_t st = launched(launch_gpair_down(false, w2, w2_scale, R, H, I, E, L.max_groups, ws, stream)))
      return st;
  } else {
    const int64_t tiles = max_tiles_for(R, E, kTileRows);
    if (moe_status_t st = launched(launch_grouped_gateup(w13, w13_scale, R, H, I, E, tiles, ws, stream))) return st;
    if (moe_status_t st = launched(launch_grouped_down(w2, w2_scale, R, H, I, E, tiles, ws, stream))) return st;
  }
  return launched(launch_combine(topk_w, M, H, K, static_cast<uint16_t*>(out), ws, stream));
}
}  // namespace

extern "C" {

moe_status_t moe_fp8_forward(const void* hidden, const int32_t* topk_ids, const float* topk_w,
                             int32_t M, const uint8_t* w13, const float* w13_scale,
                             const uint8_t* w2, const float* w2_scale, void* out,
                             void* workspace, size_t workspace_bytes,
                             const moe_fp8_shape_t* shape, cudaStream_t stream) {
  return forward_impl(hidden, Norm{nullptr, 0.0f}, topk_ids, topk_w, M, w13, w13_scale, w2, w2_scale, out, workspace,
                      workspace_bytes, shape, stream);
}

moe_status_t moe_fp8_norm_forward(const void* hidden, const void* norm_weight, float eps, const int32_t* topk_ids,
                                  const float* topk_w, int32_t M, const uint8_t* w13, const float* w13_scale,
                                  const uint8_t* w2, const float* w2_scale, void* out, void* workspace,
                                  size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream) {
  Norm nm;
  if (moe_status_t st = check_norm(norm_weight, eps, &nm)) return st;
  return forward_impl(hidden, nm, topk_ids, topk_w, M, w13, w13_scale, w2, w2_scale, out, workspace, workspace_bytes,
                      shape, stream);
}

moe_status_t moe_fp8_forward_partials(const void* hidden, const int32_t* topk_ids, int32_t M, const uint8_t* w13,
                                      const float* w13_scale, const uint8_t* w2, const float* w2_scale, float* y_out,
                                      void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                      cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, (const void*)topk_ids, (const void*)w13, (const void*)w13_scale, (const void*)w2,
                        (const void*)w2_scale, (const void*)y_out})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  if (moe_status_t st = moe_fp8_prepare(hidden, topk_ids, M, workspace, workspace_bytes, shape, stream)) return st;
  if (moe_status_t st = moe_fp8_gate_up(w13, w13_scale, M, workspace, workspace_bytes, shape, stream)) return st;
  if (moe_status_t st = moe_fp8_down(w2, w2_scale, M, workspace, workspace_bytes, shape, stream)) return st;
  return launched(launch_gather_pairs(ws_ptrs(workspace, L), M * shape->top_k, shape->hidden, y_out, stream));
}

moe_status_t moe_fp8_combine_pairs(const float* y, const int32_t* topk_ids, const float* topk_w, int32_t M, void* out,
                                   const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {(const void*)y, (const void*)topk_ids, (const void*)topk_w, (const void*)out})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  return launched(launch_combine_pairs(y, topk_ids, topk_w, M, shape->hidden, shape->top_k, shape->num_experts,
                                       static_cast<uint16_t*>(out), stream));
}

moe_status_t moe_mxfp4_forward(const void* hidden, const int32_t* topk_ids, const float* topk_w, int32_t M,
                               const uint8_t* w13q, const uint8_t* w13_scale, const uint8_t* w2q,
                               const uint8_t* w2_scale, void* out, void* workspace, size_t workspace_bytes,
                               const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, (const void*)topk_ids, (const void*)topk_w, (const void*)w13q,
                        (const void*)w13_scale, (const void*)w2q, (const void*)w2_scale, (const void*)out})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (!aligned32(w13q) || !aligned32(w2q)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const int H = shape->hidden, I = shape->inter, E = shape->num_experts, K = shape->top_k;
  const WsPtrs ws = ws_ptrs(workspace, L);
  const int64_t R = (int64_t)M * K;
  if (use_pair_mode(R)) {  // one unit per routed pair: gate/up, then down fused with the combine
    if (moe_status_t st = launched(launch_mx_gateup(w13q, w13_scale, topk_ids, static_cast<const uint16_t*>(hidden),
                                                    M, H, I, E, K, ws, stream)))
      return st;
    return launched(launch_mx_down_combine(w2q, w2_scale, topk_ids, topk_w, static_cast<uint16_t*>(out), M, H, I, E,
                                           K, ws, stream));
  }
  // more rows: quantise and sort by expert, the expert-grouped pair kernels, the combine
  if (moe_status_t st = launched(launch_sort_gather(static_cast<const uint16_t*>(hidden), Norm{nullptr, 0.0f}, topk_ids,
                                                    M, H, E, K, ws, stream)))
    return st;
  if (moe_status_t st = launched(launch_gpair_gateup(true, w13q, w13_scale, R, H, I, E, L.max_groups, ws, stream)))
    return st;
  if (moe_status_t st = launched(launch_gpair_down(true, w2q, w2_scale, R, H, I, E, L.max_groups, ws, stream)))
    return st;
  return launched(launch_combine(topk_w, M, H, K, static_cast<uint16_t*>(out), ws, stream));
}

moe_status_t moe_mxfp4_gate_up_direct(const void* hidden, const int32_t* topk_ids, int32_t M, const uint8_t* w13q,
                                      const uint8_t* w13_scale, void* workspace, size_t workspace_bytes,
                                      const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, (const void*)topk_ids, (const void*)w13q, (const void*)w13_scale})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (!aligned32(w13q)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  if (!pair_capable((int64_t)M * shape->top_k)) return MOE_ERR_UNSUPPORTED;
  return launched(launch_mx_gateup(w13q, w13_scale, topk_ids, static_cast<const uint16_t*>(hidden), M, shape->hidden,
                                   shape->inter, shape->num_experts, shape->top_k, ws_ptrs(workspace, L), stream));
}

moe_status_t moe_mxfp4_down_combine(const int32_t* topk_ids, const float* topk_w, int32_t M, const uint8_t* w2q,
                                    const uint8_t* w2_scale, void* out, void* workspace, size_t workspace_bytes,
                                    const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {(const void*)topk_ids, (const void*)topk_w, (const void*)w2q, (const void*)w2_scale,
                        (const void*)out})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (!aligned32(w2q)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  if (!pair_capable((int64_t)M * shape->top_k)) return MOE_ERR_UNSUPPORTED;
  return launched(launch_mx_down_combine(w2q, w2_scale, topk_ids, topk_w, static_cast<uint16_t*>(out), M,
                                         shape->hidden, shape->inter, shape->num_experts, shape->top_k,
                                         ws_ptrs(workspace, L), stream));
}

moe_status_t moe_mxfp4_gate_up(const uint8_t* w13q, const uint8_t* w13_scale, int32_t M, void* workspace,
                               size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!w13q || !w13_scale || !aligned32(w13q) || !aligned16(w13_scale)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const int64_t R = (int64_t)M * shape->top_k;
  if (use_pair_mode(R)) return MOE_ERR_UNSUPPORTED;  // the workspace holds no sort at so few rows
  return launched(launch_gpair_gateup(true, w13q, w13_scale, R, shape->hidden, shape->inter, shape->num_experts,
                                      L.max_groups, ws_ptrs(workspace, L), stream));
}

moe_status_t moe_mxfp4_down(const uint8_t* w2q, const uint8_t* w2_scale, int32_t M, void* workspace,
                            size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!w2q || !w2_scale || !aligned32(w2q) || !aligned16(w2_scale)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  const int64_t R = (int64_t)M * shape->top_k;
  if (use_pair_mode(R)) return MOE_ERR_UNSUPPORTED;
  return launched(launch_gpair_down(true, w2q, w2_scale, R, shape->hidden, shape->inter, shape->num_experts,
                                    L.max_groups, ws_ptrs(workspace, L), stream));
}

moe_status_t moe_mxfp4_route_forward(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                     int32_t renormalize, const uint8_t* w13q, const uint8_t* w13_scale,
                                     const uint8_t* w2q, const uint8_t* w2_scale, void* out, int32_t* topk_ids,
                                     float* topk_w, void* workspace, size_t workspace_bytes,
                                     const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, router_w, (const void*)w13q, (const void*)w13_scale, (const void*)w2q,
                        (const void*)w2_scale, (const void*)out, (const void*)topk_ids, (const void*)topk_w})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  if (!aligned32(w13q) || !aligned32(w2q)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  if (moe_status_t st = moe_route(hidden, router_w, bias, M, shape, renormalize, topk_ids, topk_w, stream)) return st;
  return moe_mxfp4_forward(hidden, topk_ids, topk_w, M, w13q, w13_scale, w2q, w2_scale, out, workspace,
                           workspace_bytes, shape, stream);
}

moe_status_t moe_fp8_gate_up_direct(const void* hidden, const int32_t* topk_ids, int32_t M,
                                    const uint8_t* w13, const float* w13_scale, void* workspace,
                                    size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                    cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, (const void*)topk_ids, (const void*)w13, (const void*)w13_scale})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  if (!pair_capable((int64_t)M * shape->top_k)) return MOE_ERR_UNSUPPORTED;
  const WsPtrs ws = ws_ptrs(workspace, L);
  return launched(launch_pair_gateup(w13, w13_scale, topk_ids, static_cast<const uint16_t*>(hidden), M,
                                     shape->hidden, shape->inter, shape->num_experts, shape->top_k, ws,
                                     stream));
}

moe_status_t moe_fp8_gate_up_prefetch(const void* hidden, const int32_t* topk_ids, int32_t M, const uint8_t* w13,
                                      const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                      void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                      cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, (const void*)topk_ids, (const void*)w13, (const void*)w13_scale, (const void*)w2,
                        (const void*)w2_scale})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  if (!pair_capable((int64_t)M * shape->top_k)) return MOE_ERR_UNSUPPORTED;
  const WsPtrs ws = ws_ptrs(workspace, L);
  return launched(launch_pair_gateup(w13, w13_scale, topk_ids, static_cast<const uint16_t*>(hidden), M, shape->hidden,
                                     shape->inter, shape->num_experts, shape->top_k, ws, stream, w2, w2_scale));
}

moe_status_t moe_fp8_down_combine(const int32_t* topk_ids, const float* topk_w, int32_t M,
                                  const uint8_t* w2, const float* w2_scale, void* out, void* workspace,
                                  size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                  cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {(const void*)topk_ids, (const void*)topk_w, (const void*)w2, (const void*)w2_scale,
                        (const void*)out})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  if (!pair_capable((int64_t)M * shape->top_k)) return MOE_ERR_UNSUPPORTED;
  const WsPtrs ws = ws_ptrs(workspace, L);
  return launched(launch_pair_down(w2, w2_scale, topk_ids, topk_w, static_cast<uint16_t*>(out), M,
                                   shape->hidden, shape->inter, shape->num_experts, shape->top_k, ws,
                                   stream));
}

moe_status_t moe_fp8_workspace_view(void* workspace, size_t workspace_bytes,
                                    const moe_fp8_shape_t* shape, moe_fp8_ws_view_t* view) {
  if (!shape || !view) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  const WsPtrs ws = ws_ptrs(workspace, L);
  view->qa = ws.qa;
  view->sa = ws.sa;
  view->row_src = ws.row_src;
  view->perm_row = ws.perm_row;
  view->act = ws.act;
  view->act_scale = ws.act_scale;
  view->y = ws.y;
  view->expert_offsets = ws.offsets;
  view->topk_ids = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + L.ids_stage);
  view->topk_w = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.wts_stage);
  view->tickets = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + L.tickets);
  return MOE_OK;
}

namespace {
moe_status_t check_route_forward(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                 const uint8_t* w13, const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                 void* out, int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
                                 const moe_fp8_shape_t* shape, Layout* L) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, router_w, (const void*)w13, (const void*)w13_scale, (const void*)w2,
                        (const void*)w2_scale, (const void*)out, (const void*)topk_ids, (const void*)topk_w})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  return check_ws(workspace, workspace_bytes, shape, L);
}
}  // namespace

moe_status_t moe_fp8_route_forward(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                   int32_t renormalize, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                   const float* w2_scale, void* out, int32_t* topk_ids, float* topk_w,
                                   void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                   cudaStream_t stream) {
  Layout L;
  if (moe_status_t st = check_route_forward(hidden, router_w, bias, M, w13, w13_scale, w2, w2_scale, out, topk_ids,
                                            topk_w, workspace, workspace_bytes, shape, &L))
    return st;
  if (M == 0) return MOE_OK;
  if (moe_status_t st = moe_route(hidden, router_w, bias, M, shape, renormalize, topk_ids, topk_w, stream)) return st;
  return moe_fp8_forward(hidden, topk_ids, topk_w, M, w13, w13_scale, w2, w2_scale, out, workspace,
                         workspace_bytes, shape, stream);
}

moe_status_t moe_fp8_norm_route_forward(const void* hidden, const void* norm_weight, float eps, const void* router_w,
                                        const float* bias, int32_t M, int32_t renormalize, const uint8_t* w13,
                                        const float* w13_scale, const uint8_t* w2, const float* w2_scale, void* out,
                                        int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
                                        const moe_fp8_shape_t* shape, cudaStream_t stream) {
  Norm nm;
  if (moe_status_t st = check_norm(norm_weight, eps, &nm)) return st;
  Layout L;
  if (moe_status_t st = check_route_forward(hidden, router_w, bias, M, w13, w13_scale, w2, w2_scale, out, topk_ids,
                                            topk_w, workspace, workspace_bytes, shape, &L))
    return st;
  if (M == 0) return MOE_OK;
  if (moe_status_t st = route_impl(hidden, nm, router_w, bias, M, shape, renormalize, topk_ids, topk_w, stream))
    return st;
  return forward_impl(hidden, nm, topk_ids, topk_w, M, w13, w13_scale, w2, w2_scale, out, workspace, workspace_bytes,
                      shape, stream);
}

moe_status_t moe_fp8_verify_produce(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                    int32_t renormalize, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, int32_t* topk_ids, float* topk_w, void* workspace,
                                    size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, router_w, (const void*)w13, (const void*)w13_scale, (const void*)w2,
                        (const void*)w2_scale, (const void*)topk_ids, (const void*)topk_w})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (!verify_profile(M, shape->hidden, shape->inter, shape->num_experts, shape->top_k)) return MOE_ERR_UNSUPPORTED;
  // routing, then the 96 routed rows quantised and sorted by expert, gate/up with SiLU and
  // the requantisation, and the down partials y (FP32, the sort's rows), by the expert-grouped
  // kernels; the reducer sums them in slot order through the sort's permutation
  const int H = shape->hidden, I = shape->inter, E = shape->num_experts, K = shape->top_k;
  const WsPtrs ws = ws_ptrs(workspace, L);
  const int64_t R = (int64_t)M * K;
  if (moe_status_t st = route_impl(hidden, Norm{nullptr, 0.0f}, router_w, bias, M, shape, renormalize, topk_ids,
                                   topk_w, stream))
    return st;
  if (moe_status_t st = launched(launch_sort_gather(static_cast<const uint16_t*>(hidden), Norm{nullptr, 0.0f},
                                                    topk_ids, M, H, E, K, ws, stream)))
    return st;
  if (moe_status_t st = launched(launch_gpair_gateup(false, w13, w13_scale, R, H, I, E, L.max_groups, ws, stream)))
    return st;
  return launched(launch_gpair_down(false, w2, w2_scale, R, H, I, E, L.max_groups, ws, stream));
}

moe_status_t moe_fp8_verify_produce_one_launch(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                               int32_t renormalize, const uint8_t* w13, const float* w13_scale,
                                               const uint8_t* w2, const float* w2_scale, int32_t* topk_ids,
                                               float* topk_w, void* workspace, size_t workspace_bytes,
                                               const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  for (const void* p : {hidden, router_w, (const void*)w13, (const void*)w13_scale, (const void*)w2,
                        (const void*)w2_scale, (const void*)topk_ids, (const void*)topk_w})
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (!verify_profile(M, shape->hidden, shape->inter, shape->num_experts, shape->top_k)) return MOE_ERR_UNSUPPORTED;
  if (!verify_capable()) return MOE_ERR_UNSUPPORTED;
  return launched(launch_verify_produce(static_cast<const uint16_t*>(hidden), static_cast<const uint16_t*>(router_w),
                                        bias, renormalize ? 1 : 0, topk_ids, topk_w, w13, w13_scale, w2, w2_scale,
                                        ws_ptrs(workspace, L), stream));
}

moe_status_t moe_fp8_verify_reduce(const float* topk_w, int32_t M, void* out, void* workspace, size_t workspace_bytes,
                                   const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!topk_w || !out || !aligned16(topk_w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (!verify_profile(M, shape->hidden, shape->inter, shape->num_experts, shape->top_k)) return MOE_ERR_UNSUPPORTED;
  return launched(launch_combine(topk_w, M, shape->hidden, shape->top_k, static_cast<uint16_t*>(out),
                                 ws_ptrs(workspace, L), stream));
}

moe_status_t moe_fp8_route_forward_one_launch(const void* hidden, const void* router_w, const float* bias,
                                              int32_t M, int32_t renormalize, const uint8_t* w13,
                                              const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                              void* out, int32_t* topk_ids, float* topk_w, void* workspace,
                                              size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                              cudaStream_t stream) {
  Layout L;
  if (moe_status_t st = check_route_forward(hidden, router_w, bias, M, w13, w13_scale, w2, w2_scale, out, topk_ids,
                                            topk_w, workspace, workspace_bytes, shape, &L))
    return st;
  if (M == 0) return MOE_OK;
  const int H = shape->hidden, I = shape->inter, E = shape->num_experts, K = shape->top_k;
  if (!fused_capable(M, H, I, E, K)) return MOE_ERR_UNSUPPORTED;
  return launched(launch_fused(true, static_cast<const uint16_t*>(hidden), static_cast<const uint16_t*>(router_w), bias,
                               renormalize ? 1 : 0, topk_ids, topk_w, w13, w13_scale, w2, w2_scale,
                               static_cast<uint16_t*>(out), M, H, I, E, K, ws_ptrs(workspace, L),
                               reinterpret_cast<float*>(static_cast<char*>(workspace) + L.yt),
                               reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + L.tickets), stream));
}

moe_status_t moe_fp8_route_forward_host(const void* host_hidden, void* host_out, int32_t M,
                                        const void* router_w, const float* bias, int32_t renormalize,
                                        const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                        const float* w2_scale, void* workspace, size_t workspace_bytes,
                                        const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!host_hidden || !host_out) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  char* b = static_cast<char*>(workspace);
  int32_t* ids = reinterpret_cast<int32_t*>(b + L.ids_stage);
  float* wts = reinterpret_cast<float*>(b + L.wts_stage);
  const size_t bytes = (size_t)M * shape->hidden * 2;
  // Page-locked host buffers are device-addressable: the kernels read hidden from and write
  // out to them directly, with no copies (one fewer round trip per direction). Pageable
  // buffers go through device copies in the workspace.
  const void* hid = device_view(host_hidden);
  void* out = const_cast<void*>(device_view(host_out));
  const bool copy_in = hid == nullptr, copy_out = out == nullptr;
  if (copy_in) {
    hid = b + L.hid_stage;
    if (cudaMemcpyAsync(const_cast<void*>(hid), host_hidden, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return MOE_ERR_LAUNCH;
  }
  if (copy_out) out = b + L.out_stage;
  if (!aligned16(hid) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (moe_status_t st = moe_fp8_route_forward(hid, router_w, bias, M, renormalize, w13, w13_scale, w2, w2_scale, out,
                                              ids, wts, workspace, workspace_bytes, shape, stream))
    return st;
  if (copy_out) return launched(cudaMemcpyAsync(host_out, out, bytes, cudaMemcpyDeviceToHost, stream));
  return MOE_OK;
}

moe_status_t moe_fp8_route_forward_pinned(const void* host_hidden, void* host_out, int32_t M,
                                          const void* router_w, const float* bias, int32_t renormalize,
                                          const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                          const float* w2_scale, void* workspace, size_t workspace_bytes,
                                          const moe_fp8_shape_t* shape, cudaStream_t stream) {
  if (moe_status_t st = check_common(shape, M)) return st;
  if (!host_hidden || !host_out || !aligned16(host_hidden) || !aligned16(host_out)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  if (M == 0) return MOE_OK;
  char* b = static_cast<char*>(workspace);
  int32_t* ids = reinterpret_cast<int32_t*>(b + L.ids_stage);
  float* wts = reinterpret_cast<float*>(b + L.wts_stage);
  // page-locked host memory under unified addressing: the host pointers are device-usable
  return moe_fp8_route_forward(host_hidden, router_w, bias, M, renormalize, w13, w13_scale, w2, w2_scale, host_out,
                               ids, wts, workspace, workspace_bytes, shape, stream);
}

moe_status_t moe_fp8_selftest_wait(void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                   uint32_t limit_us, cudaStream_t stream) {
  if (!shape) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED;
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (moe_status_t st = check_ws(workspace, workspace_bytes, shape, &L)) return st;
  return launched(launch_wait_selftest(ws_ptrs(workspace, L).hdr, limit_us, stream));
}

moe_status_t moe_fp8_read_status(const void* workspace, uint32_t* host_dst, cudaStream_t stream) {
  if (!workspace || !host_dst || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  return launched(cudaMemcpyAsync(host_dst, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
}

}  // extern "C"
