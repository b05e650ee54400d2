// route.cu -- router: BF16 logits in a fixed chunk order, softmax and top-k.
//
// Source: "NetraRuntime/netra-kernel" README, capability table (BF16 routing) and the
// prefill-pair build section (the routed MoE producer starts with a routing stage).
//
// GB300 design. A thread-block cluster of CL CTAs covers one block of TB tokens; CTA r
// owns experts [r*EC, (r+1)*EC). Its threads compute, for every token of the block, one
// FP32 fma chain per (expert, 128-wide hidden chunk) over the chunk's k ascending from 0,
// then sum the chunk partials in ascending chunk order -- so each logit is formed inside
// one CTA in the contract order and the top-k ids do not depend on the launch shape. The
// CTA stores its logits straight into CTA 0's shared memory (distributed shared memory
// stores: no round trips), one cluster barrier later CTA 0 holds all E logits of every
// token and a warp per token selects the top K (ties to the lower expert index) and forms
// the softmax weights. No workspace, no atomics, no spin-waits.
#include <cooperative_groups.h>

#include <climits>
#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kRouteThreads = 256;
constexpr int kRouteChunksPerRound = 16;  // hidden chunks staged in shared memory at once

struct RouteSmem {
  size_t ws, xs, part, logits, total;
};

// ws: router slab [16 chunks * 128 rows][EC] bf16; xs: hidden [TB][16*128] bf16;
// part: chunk partials [nchunks][TB][EC] f32; logits: [TB][E] f32 (filled on CTA 0).
__host__ __device__ inline RouteSmem route_smem(int TB, int EC, int E, int nchunks) {
  RouteSmem s{};
  size_t o = 0;
  s.ws = o;     o += (size_t)kRouteChunksPerRound * 128 * EC * 2;
  s.xs = o;     o += (size_t)TB * kRouteChunksPerRound * 128 * 2;
  s.part = o;   o += (size_t)nchunks * TB * EC * 4;
  s.logits = o; o += (size_t)TB * E * 4;
  s.total = o;
  return s;
}

template <int TB>
__global__ void __launch_bounds__(kRouteThreads)
    route_kernel(const uint16_t* __restrict__ hidden, const uint16_t* __restrict__ router_w,
                 const float* __restrict__ bias, int M, int H, int E, int K, int renorm,
                 int32_t* __restrict__ ids, float* __restrict__ wts) {
  extern __shared__ __align__(16) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int EC = E / CL;
  const int nchunks = H / 128;
  const RouteSmem L = route_smem(TB, EC, E, nchunks);
  uint16_t* wsm = reinterpret_cast<uint16_t*>(smem + L.ws);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* logits = reinterpret_cast<float*>(smem + L.logits);
  const int tid = threadIdx.x;
  const int tok0 = blockIdx.y * TB;
  const int e0 = rank * EC;

  // inputs may be written by the previous kernel in the stream (programmatic launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  // thread <-> (expert el, chunk lane cgl); chunks cgl, cgl + TPE, ... of each round.
  // Consecutive lanes take consecutive experts (one 2-byte router value each).
  const int TPE = kRouteThreads / EC;
  const int el = tid % EC, cgl = tid / EC;
  for (int c0 = 0; c0 < nchunks; c0 += kRouteChunksPerRound) {
    const int nc = min(kRouteChunksPerRound, nchunks - c0);
    // stage router rows [c0*128, (c0+nc)*128) x experts [e0, e0+EC) and the hidden chunk
    const int segs = EC * 2 / 16;  // 16-byte pieces per router row slice
    const int n16 = nc * 128 * segs;
    for (int i0 = tid; i0 < n16; i0 += kRouteThreads * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kRouteThreads;
        if (i < n16)
          v[u] = *reinterpret_cast<const uint4*>(router_w + (size_t)(c0 * 128 + i / segs) * E + e0 +
                                                 (i % segs) * 8);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * kRouteThreads < n16) reinterpret_cast<uint4*>(wsm)[i0 + u * kRouteThreads] = v[u];
    }
    for (int i = tid; i < TB * nc * 16; i += kRouteThreads) {
      const int t = i / (nc * 16), k8 = (i % (nc * 16)) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (tok0 + t < M) v = *reinterpret_cast<const uint4*>(hidden + (size_t)(tok0 + t) * H + c0 * 128 + k8);
      *reinterpret_cast<uint4*>(xs + t * kRouteChunksPerRound * 128 + k8) = v;
    }
    __syncthreads();
    {
      for (int cc = cgl; cc < nc; cc += TPE) {
        float acc[TB];
#pragma unroll
        for (int t = 0; t < TB; ++t) acc[t] = 0.0f;
#pragma unroll 8
        for (int k = 0; k < 128; ++k) {
          const float w = bf16_bits_to_float(wsm[(cc * 128 + k) * EC + el]);
#pragma unroll
          for (int t = 0; t < TB; ++t)
            acc[t] = __fmaf_rn(bf16_bits_to_float(xs[t * kRouteChunksPerRound * 128 + cc * 128 + k]), w, acc[t]);
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) part[((size_t)(c0 + cc) * TB + t) * EC + el] = acc[t];
      }
    }
    __syncthreads();
  }
  // logits of this CTA's experts, chunk partials summed in ascending chunk order, pushed
  // into CTA 0's shared memory
  float* logits0 = cluster.map_shared_rank(logits, 0);
  for (int i = tid; i < TB * EC; i += kRouteThreads) {
    const int t = i / EC, e = i % EC;
    float l = 0.0f;
    for (int c = 0; c < nchunks; ++c) l = __fadd_rn(l, part[((size_t)c * TB + t) * EC + e]);
    if (bias != nullptr) l = __fadd_rn(l, bias[e0 + e]);
    logits0[t * E + e0 + e] = l;
  }
  cluster.sync();  // all logits are in CTA 0's shared memory
  if (rank != 0) return;

  // top-k: one warp per token; lane holds experts lane, lane+32, ...
  const int warp = tid / 32, lane = tid % 32;
  constexpr int kMaxPerLane = 8;  // E <= 256
  for (int t = warp; t < TB; t += kRouteThreads / 32) {
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

namespace {

// CL CTAs per cluster, E/CL >= 8 experts each (a 16-byte router row slice); 16-CTA
// clusters (a non-portable size) for E >= 128 spread the router weights over more SMs
int route_cluster(int E) { return E >= 128 ? 16 : E / 8; }

template <int TB>
cudaError_t launch_route_t(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int M,
                           int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st) {
  const int CL = route_cluster(E);
  const RouteSmem L = route_smem(TB, E / CL, E, H / 128);
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(route_kernel<TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(route_kernel<TB>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, (M + TB - 1) / TB, 1);
  cfg.blockDim = dim3(kRouteThreads, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, route_kernel<TB>, hidden, router_w, bias, M, H, E, K, renorm, ids, wts);
}

}  // namespace

cudaError_t launch_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int M,
                         int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st) {
  if (M <= 2) return launch_route_t<1>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  if (M <= 32) return launch_route_t<2>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  return launch_route_t<8>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
}

}  // namespace moe
