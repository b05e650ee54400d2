// combine.cu -- top-k weighted combine (the route reducer).
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (the route
// reducer is its own operation with its own reduction order); "Inferact/amd-kernels"
// README (expert partials are summed in a fixed order, never with atomic adds).
//
// out[t][h] = bf16_rn( sum over slots j ascending of w[t][j] * y[perm_row[t][j]][h] ),
// FP32 multiply then add, from 0; skipped pairs (perm_row < 0) contribute nothing.
// One thread owns 8 consecutive columns: two 128-bit loads of y per slot, one 128-bit
// store of 8 BF16 values.
#include "common.cuh"
#include "launch.h"

namespace moe {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ topk_w, int M,
                                                      int H, int K, uint16_t* __restrict__ out,
                                                      WsPtrs ws) {
  const int t = blockIdx.x;
  const int h = (blockIdx.y * 256 + threadIdx.x) * 8;
  // y and perm_row come from the kernels before this one on the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (t >= M || h >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  // four slots at a time: their indices and weights first, then all their row loads, so
  // the dependent loads of different slots overlap; the adds stay in slot order
  for (int j0 = 0; j0 < K; j0 += 4) {
    int pj[4];
    float wj[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      pj[u] = j0 + u < K ? ws.perm_row[t * K + j0 + u] : -1;
      wj[u] = j0 + u < K ? topk_w[t * K + j0 + u] : 0.0f;
    }
    float4 ya[4], yb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (pj[u] >= 0) {
        ya[u] = *reinterpret_cast<const float4*>(ws.y + (size_t)pj[u] * H + h);
        yb[u] = *reinterpret_cast<const float4*>(ws.y + (size_t)pj[u] * H + h + 4);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (pj[u] < 0) continue;
      const float y[8] = {ya[u].x, ya[u].y, ya[u].z, ya[u].w, yb[u].x, yb[u].y, yb[u].z, yb[u].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(wj[u], y[i]));
    }
  }
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat16 a = __float2bfloat16_rn(acc[2 * i]);
    const __nv_bfloat16 b = __float2bfloat16_rn(acc[2 * i + 1]);
    packed[i] = (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
  }
  *reinterpret_cast<uint4*>(out + (size_t)t * H + h) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

cudaError_t launch_combine(const float* topk_w, int M, int H, int K, uint16_t* out, const WsPtrs& ws,
                           cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, (unsigned)((H + 2047) / 2048), 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, topk_w, M, H, K, out, ws);
}

}  // namespace moe
