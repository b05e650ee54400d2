// launch.h -- the kernels' host-side launchers (internal to the library; the C ABI in
// api.cu and noalloc.cu calls these). Every launcher enqueues on `st` and returns the launch
// error, if any; none allocates, synchronises or reads device memory.
#pragma once

#include "common.cuh"

namespace moe {

// route.cu: top-k routing of M tokens (norm: an RMSNorm in front, gamma null for none)
cudaError_t launch_route(const uint16_t* hidden, Norm nm, const uint16_t* router_w, const float* bias, int M,
                         int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st);
// norm.cu: y = RMSNorm(hidden) as BF16 [M][H]
cudaError_t launch_rmsnorm(const uint16_t* hidden, Norm nm, int M, int H, uint16_t* y, cudaStream_t st);
// prep.cu: hidden codes + the pair-mode identity permutation (few routed rows), or the
// counting sort and the gather of codes into expert order (many routed rows)
cudaError_t launch_prep(const uint16_t* hidden, const int32_t* ids, int M, int H, int E, int K,
                        const WsPtrs& ws, cudaStream_t st);
cudaError_t launch_sort_gather(const uint16_t* hidden, Norm nm, const int32_t* ids, int M, int H, int E, int K,
                               const WsPtrs& ws, cudaStream_t st);
// tc_grouped.cu: the expert-sorted tile GEMMs
cudaError_t launch_grouped_gateup(const uint8_t* w13, const float* s13, int64_t R, int H, int I, int E,
                                  int64_t max_tiles, const WsPtrs& ws, cudaStream_t st);
cudaError_t launch_grouped_down(const uint8_t* w2, const float* s2w, int64_t R, int H, int I, int E,
                                int64_t max_tiles, const WsPtrs& ws, cudaStream_t st);
// tc_pair.cu: one unit per routed pair. gate/up quantises hidden itself when hidden is set
// (then w2/s2w, if set, are prefetched into L2 and nm applies), else reads the workspace codes
cudaError_t launch_pair_gateup(const uint8_t* w13, const float* s13, const int32_t* ids,
                               const uint16_t* hidden, int M, int H, int I, int E, int K,
                               const WsPtrs& ws, cudaStream_t st, const uint8_t* w2 = nullptr,
                               const float* s2w = nullptr, Norm nm = Norm{nullptr, 0.0f});
cudaError_t launch_pair_down(const uint8_t* w2, const float* s2w, const int32_t* ids, const float* topk_w,
                             uint16_t* out, int M, int H, int I, int E, int K, const WsPtrs& ws,
                             cudaStream_t st);
// mx_pair.cu: the pair kernels with MXFP4 weights (packed E2M1 codes, UE8M0 scales per 32)
cudaError_t launch_mx_gateup(const uint8_t* w13q, const uint8_t* w13s, const int32_t* ids, const uint16_t* hidden,
                             int M, int H, int I, int E, int K, const WsPtrs& ws, cudaStream_t st);
cudaError_t launch_mx_down_combine(const uint8_t* w2q, const uint8_t* w2s, const int32_t* ids, const float* topk_w,
                                   uint16_t* out, int M, int H, int I, int E, int K, const WsPtrs& ws,
                                   cudaStream_t st);
// gpair.cu: expert-grouped pair kernels over the sort's groups of up to kGroupRows rows
// (FP8 or MXFP4 weights; scales FP32 or UE8M0)
cudaError_t launch_gpair_gateup(bool mx, const uint8_t* w13, const void* s13, int64_t R, int H, int I, int E,
                                int64_t max_groups, const WsPtrs& ws, cudaStream_t st);
cudaError_t launch_gpair_down(bool mx, const uint8_t* w2, const void* s2, int64_t R, int H, int I, int E,
                              int64_t max_groups, const WsPtrs& ws, cudaStream_t st);
// combine.cu: out = slot-order combine of y (workspace rows through perm_row, or given rows in
// pair order with skipped pairs named by their ids), and the sorted y gathered into pair order
cudaError_t launch_combine(const float* topk_w, int M, int H, int K, uint16_t* out, const WsPtrs& ws,
                           cudaStream_t st);
cudaError_t launch_combine_pairs(const float* y, const int32_t* ids, const float* topk_w, int M, int H, int K, int E,
                                 uint16_t* out, cudaStream_t st);
cudaError_t launch_gather_pairs(const WsPtrs& ws, int R, int H, float* y_out, cudaStream_t st);
// selftest.cu: a bounded wait that runs out
cudaError_t launch_wait_selftest(Header* hdr, uint32_t limit_us, cudaStream_t st);
// fused.cu: the single-launch layer for a few routed pairs
bool fused_capable(int M, int H, int I, int E, int K);
cudaError_t launch_fused(bool route, const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                         int renorm, int32_t* ids, float* wts, const uint8_t* w13, const float* s13,
                         const uint8_t* w2, const float* s2w, uint16_t* out, int M, int H, int I, int E, int K,
                         const WsPtrs& ws, float* yt, uint32_t* tickets, cudaStream_t st);

// verify.cu: the verify_m12 profile's producer (routing, gate/up, SiLU and quantisation,
// down partials y in pair order, identity permutation) -- the reducer is launch_combine
bool verify_profile(int M, int H, int I, int E, int K);
bool verify_capable();
cudaError_t launch_verify_produce(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int renorm,
                                  int32_t* ids, float* wts, const uint8_t* w13, const float* s13, const uint8_t* w2,
                                  const float* s2w, const WsPtrs& ws, cudaStream_t st);

}  // namespace moe
