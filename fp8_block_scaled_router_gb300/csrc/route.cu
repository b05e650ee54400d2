// route.cu -- router: BF16 logits in a fixed chunk order, softmax and top-k.
//
// Source: "NetraRuntime/netra-kernel" README, capability table (BF16 routing) and the
// prefill-pair build section (the routed MoE producer starts with a routing stage).
//
// GB300 design. A thread-block cluster of CL CTAs covers one block of TB tokens; CTA r of
// the cluster owns 128-wide hidden chunks [r*nC, (r+1)*nC) and computes, for every token of
// the block and every expert, one FP32 fma chain per chunk (k ascending, from 0). The chunk
// partials stay in each CTA's shared memory; after a cluster barrier CTA 0 reads them over
// distributed shared memory and sums them in ascending chunk order, so the logits -- and
// hence the top-k ids -- do not depend on the launch shape. No workspace, no atomics and
// no spin-waits: the only synchronisation is the hardware cluster barrier.
#include <cooperative_groups.h>

#include <climits>
#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace moe {

struct RouteSmem {
  int TB, nC, E;
  size_t xs, ws, part, logits, total;
};

__host__ __device__ inline RouteSmem route_smem(int TB, int nC, int E) {
  RouteSmem s{TB, nC, E, 0, 0, 0, 0, 0};
  size_t o = 0;
  s.xs = o;     o += (size_t)TB * 128 * 4;
  s.ws = o;     o += (size_t)128 * E * 2;
  s.part = o;   o += (size_t)nC * TB * E * 4;
  s.logits = o; o += (size_t)TB * E * 4;
  s.total = o;
  return s;
}

// TPT tokens per thread; each thread owns 4 consecutive experts.
template <int TPT>
__global__ void __launch_bounds__(256) route_kernel(const uint16_t* __restrict__ hidden,
                                                    const uint16_t* __restrict__ router_w,
                                                    const float* __restrict__ bias, int M, int H,
                                                    int E, int K, int renorm, int nC,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ wts) {
  extern __shared__ __align__(16) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int EG = E / 4, TG = 256 / EG, TB = TG * TPT;
  const RouteSmem L = route_smem(TB, nC, E);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  uint16_t* wsm = reinterpret_cast<uint16_t*>(smem + L.ws);
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* logits = reinterpret_cast<float*>(smem + L.logits);

  const int tid = threadIdx.x;
  const int eg = tid % EG, tg = tid / EG;
  const int tok0 = blockIdx.y * TB;

  for (int cl = 0; cl < nC; ++cl) {
    const int c = rank * nC + cl;
    // stage the chunk: hidden [TB][128] as float, router rows [128][E]
    for (int i = tid; i < TB * 32; i += 256) {
      const int t = i / 32, k4 = (i % 32) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tok0 + t < M) {
        const uint2 raw = *reinterpret_cast<const uint2*>(hidden + (size_t)(tok0 + t) * H + c * 128 + k4);
        v = make_float4(bf16_bits_to_float(raw.x & 0xFFFF), bf16_bits_to_float(raw.x >> 16),
                        bf16_bits_to_float(raw.y & 0xFFFF), bf16_bits_to_float(raw.y >> 16));
      }
      *reinterpret_cast<float4*>(xs + t * 128 + k4) = v;
    }
    const uint4* wsrc = reinterpret_cast<const uint4*>(router_w + (size_t)c * 128 * E);
    for (int i = tid; i < 128 * E / 8; i += 256) reinterpret_cast<uint4*>(wsm)[i] = wsrc[i];
    __syncthreads();

    if (tg < TG) {
      float acc[TPT][4];
#pragma unroll
      for (int t = 0; t < TPT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;
#pragma unroll 4
      for (int k = 0; k < 128; ++k) {
        const uint2 w4 = *reinterpret_cast<const uint2*>(wsm + k * E + 4 * eg);
        const float w0 = bf16_bits_to_float(w4.x & 0xFFFF), w1 = bf16_bits_to_float(w4.x >> 16);
        const float w2 = bf16_bits_to_float(w4.y & 0xFFFF), w3 = bf16_bits_to_float(w4.y >> 16);
#pragma unroll
        for (int t = 0; t < TPT; ++t) {
          const float x = xs[(tg * TPT + t) * 128 + k];
          acc[t][0] = __fmaf_rn(x, w0, acc[t][0]);
          acc[t][1] = __fmaf_rn(x, w1, acc[t][1]);
          acc[t][2] = __fmaf_rn(x, w2, acc[t][2]);
          acc[t][3] = __fmaf_rn(x, w3, acc[t][3]);
        }
      }
#pragma unroll
      for (int t = 0; t < TPT; ++t)
        *reinterpret_cast<float4*>(part + ((size_t)cl * TB + tg * TPT + t) * E + 4 * eg) =
            make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
    }
    __syncthreads();
  }

  cluster.sync();  // every CTA's chunk partials are complete and visible cluster-wide
  if (rank == 0) {
    for (int i = tid; i < TB * E; i += 256) {
      const int t = i / E, e = i % E;
      float l = 0.0f;
      for (int r = 0; r < CL; ++r) {
        const float* pr = cluster.map_shared_rank(part, r);
        for (int cl = 0; cl < nC; ++cl) l = __fadd_rn(l, pr[((size_t)cl * TB + t) * E + e]);
      }
      if (bias != nullptr) l = __fadd_rn(l, bias[e]);
      logits[t * E + e] = l;
    }
  }
  cluster.sync();  // CTA 0 is done reading the other CTAs' shared memory
  if (rank != 0) return;
  __syncthreads();

  // top-k: one warp per token; lane holds experts lane, lane+32, ...
  const int warp = tid / 32, lane = tid % 32;
  constexpr int kMaxPerLane = 8;  // E <= 256
  for (int t = warp; t < TB; t += 8) {
    if (tok0 + t >= M) break;
    float v[kMaxPerLane];
    bool taken[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? logits[t * E + e] : -INFINITY;
      taken[i] = !(e < E);
    }
    float sel_v[16];
    int sel_i[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= K) break;
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if (!taken[i] && (v[i] > bv || (v[i] == bv && e < bi))) { bv = v[i]; bi = e; }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (lane + 32 * i == bi) taken[i] = true;
      sel_v[j] = bv;
      sel_i[j] = bi;
    }
    const float lmax = sel_v[0];
    float den = 0.0f;
    if (renorm) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j >= K) break;
        den = __fadd_rn(den, expf(__fsub_rn(sel_v[j], lmax)));
      }
    } else {
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (lane + 32 * i < E) den = __fadd_rn(den, expf(__fsub_rn(v[i], lmax)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, off));
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= K) break;
      if (lane == j) {
        const size_t o = (size_t)(tok0 + t) * K + j;
        ids[o] = sel_i[j] == INT_MAX ? -1 : sel_i[j];
        wts[o] = __fdiv_rn(expf(__fsub_rn(sel_v[j], lmax)), den);
      }
    }
  }
}

template <int TPT>
static cudaError_t launch_route_t(const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                                  int M, int H, int E, int K, int renorm, int32_t* ids, float* wts,
                                  cudaStream_t st) {
  const int nchunks = H / 128;
  int CL = 1;
  for (int c = 8; c >= 1; --c)
    if (nchunks % c == 0) { CL = c; break; }
  const int nC = nchunks / CL;
  const int TB = (256 / (E / 4)) * TPT;
  const RouteSmem L = route_smem(TB, nC, E);
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(route_kernel<TPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, (M + TB - 1) / TB, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel<TPT>, hidden, router_w, bias, M, H, E, K, renorm, nC,
                            ids, wts);
}

size_t route_smem_bytes(int M, int H, int E) {
  const int TPT = (M >= 256 && E >= 64) ? 4 : 1;
  const int nchunks = H / 128;
  int CL = 1;
  for (int c = 8; c >= 1; --c)
    if (nchunks % c == 0) { CL = c; break; }
  return route_smem((256 / (E / 4)) * TPT, nchunks / CL, E).total;
}

cudaError_t launch_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int M,
                         int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st) {
  if (M >= 256 && E >= 64)
    return launch_route_t<4>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  return launch_route_t<1>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
}

}  // namespace moe
