// combine.cu -- top-k weighted combine (the route reducer).
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (the route
// reducer is its own operation with its own reduction order); "Inferact/amd-kernels"
// README (expert partials are summed in a fixed order, never with atomic adds).
//
// out[t][h] = bf16_rn( sum over slots j ascending of w[t][j] * y[perm_row[t][j]][h] ),
// FP32 multiply then add, from 0; skipped pairs (perm_row < 0) contribute nothing. With no
// permutation the rows of y are in pair order (row t*K + j) and a pair is skipped when its
// expert id is outside [0, E) (the partials of an expert-parallel layer, gathered back).
// One thread owns 8 consecutive columns: two 128-bit loads of y per slot, one 128-bit
// store of 8 BF16 values.
#include "common.cuh"
#include "launch.h"

namespace moe {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ topk_w, int M,
                                                      int H, int K, uint16_t* __restrict__ out,
                                                      const float* __restrict__ y,
                                                      const int32_t* __restrict__ perm_row,
                                                      const int32_t* __restrict__ ids, int E) {
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
      if (j0 + u >= K) {
        pj[u] = -1;
      } else if (perm_row != nullptr) {
        pj[u] = perm_row[t * K + j0 + u];
      } else {
        const int e = ids[t * K + j0 + u];
        pj[u] = e >= 0 && e < E ? t * K + j0 + u : -1;
      }
      wj[u] = j0 + u < K ? topk_w[t * K + j0 + u] : 0.0f;
    }
    float4 ya[4], yb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (pj[u] >= 0) {
        ya[u] = *reinterpret_cast<const float4*>(y + (size_t)pj[u] * H + h);
        yb[u] = *reinterpret_cast<const float4*>(y + (size_t)pj[u] * H + h + 4);
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

namespace {
cudaError_t combine_launch(const float* topk_w, int M, int H, int K, uint16_t* out, const float* y,
                           const int32_t* perm_row, const int32_t* ids, int E, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, (unsigned)((H + 2047) / 2048), 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, topk_w, M, H, K, out, y, perm_row, ids, E);
}
}  // namespace

cudaError_t launch_combine(const float* topk_w, int M, int H, int K, uint16_t* out, const WsPtrs& ws,
                           cudaStream_t st) {
  return combine_launch(topk_w, M, H, K, out, ws.y, ws.perm_row, nullptr, 0, st);
}

cudaError_t launch_combine_pairs(const float* y, const int32_t* ids, const float* topk_w, int M, int H, int K, int E,
                                 uint16_t* out, cudaStream_t st) {
  return combine_launch(topk_w, M, H, K, out, y, nullptr, ids, E, st);
}

// y_out[p] = y[perm_row[p]] (FP32 rows of H), or zeros for a skipped pair (perm_row < 0): the
// expert-sorted down output back in pair order. One CTA of 256 threads per pair row, 16-byte
// loads and stores.
__global__ void __launch_bounds__(256) gather_pairs_kernel(const float* __restrict__ y, const int32_t* __restrict__ perm_row,
                                                           int R, int H, float* __restrict__ y_out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int p = blockIdx.x;
  if (p >= R) return;
  const int src = perm_row[p];
  const float4* s = reinterpret_cast<const float4*>(y + (size_t)(src < 0 ? 0 : src) * H);
  float4* d = reinterpret_cast<float4*>(y_out + (size_t)p * H);
  for (int i = threadIdx.x; i < H / 4; i += 256) d[i] = src < 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : s[i];
}

cudaError_t launch_gather_pairs(const WsPtrs& ws, int R, int H, float* y_out, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)R, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_pairs_kernel, (const float*)ws.y, (const int32_t*)ws.perm_row, R, H, y_out);
}

}  // namespace moe
