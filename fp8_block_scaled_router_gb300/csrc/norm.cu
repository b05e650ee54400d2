// norm.cu -- the RMSNorm in front of the layer, written out as BF16 rows.
//
// Source: older kernel-lab README, repository layout (gfx950 normalisation and quantisation
// fusions) and the Qwen3.6 RMSNorm patch listed beside it. The pages name the operation but
// not its epsilon or weight convention; this library takes y = bf16((x * r) * gamma) with
// r = 1 / sqrt(mean(x^2) + eps) and both eps and gamma from the caller (common.cuh gives the
// exact FP32 order). The router and the hidden quantisers apply the same transform on the
// fly (they never read this kernel's output); this kernel serves callers that also need y
// itself (a shared expert, the residual path).
//
// One warp per row: r from row_rms_scale, then 16-byte loads of x and gamma and 16-byte
// stores of y. HBM-bound: 2 * H bytes read and 2 * H written per row (gamma stays in L1/L2).
#include "device.h"
#include "launch.h"

namespace moe {

__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* __restrict__ x, const Norm nm, int M, int H,
                                                      uint16_t* __restrict__ y) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t nwarps = (int64_t)gridDim.x * 8;
  for (int64_t t = (int64_t)blockIdx.x * 8 + warp; t < M; t += nwarps) {
    const uint16_t* xr = x + t * H;
    const float r = row_rms_scale(xr, H, nm.eps, lane);
    for (int k8 = lane * 8; k8 < H; k8 += 256) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xr + k8);
      const uint4 gv = *reinterpret_cast<const uint4*>(nm.gamma + k8);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        o[u] = (uint32_t)norm_bits(xw[u] & 0xFFFF, r, gw[u] & 0xFFFF) |
               ((uint32_t)norm_bits(xw[u] >> 16, r, gw[u] >> 16) << 16);
      *reinterpret_cast<uint4*>(y + t * H + k8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_rmsnorm(const uint16_t* hidden, Norm nm, int M, int H, uint16_t* y, cudaStream_t st) {
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  int64_t blocks = ((int64_t)M + 7) / 8;
  if (blocks > 8 * (int64_t)d.sms) blocks = 8 * (int64_t)d.sms;  // 8 CTAs of 8 warps per SM, grid-stride
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, hidden, nm, M, H, y);
}

}  // namespace moe
