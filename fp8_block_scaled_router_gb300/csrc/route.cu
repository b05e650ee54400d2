// route.cu -- router: BF16 logits in a fixed chunk order, softmax and top-k.
//
// Source: "NetraRuntime/netra-kernel" README, capability table (BF16 routing) and the
// prefill-pair build section (the routed MoE producer starts with a routing stage).
//
// GB300 design. A thread-block cluster of CL CTAs covers one block of TB tokens; CTA r
// owns the 128-wide hidden chunks [r*CPC, (r+1)*CPC) for every expert, so it reads whole,
// contiguous rows of the router matrix. Thread e forms, for each token of the block and each
// of its chunks, the FP32 fma chain over the chunk's k ascending from 0 (the token values of
// one k are one 16-byte shared-memory load). The chunk partials are stored straight into
// CTA 0's shared memory (distributed shared memory stores); after one cluster barrier CTA 0
// adds them in ascending chunk order, adds the bias, and selects the top K by rank: expert
// e takes slot #{e' : l[e'] > l[e] or (l[e'] == l[e] and e' < e)} when that is below K
// (ties to the lower index). Weights: softmax over the K selected logits (renormalised) or
// over all E. No workspace, no atomics, no spin-waits.
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kRouteThreads = 256;
constexpr int kRouteMaxCluster = 16;

struct RouteSmem {
  size_t ws, xs, part, logits, sel, bias, total;
};

// ws: router rows [CPC*128][E] bf16; xs: hidden [CPC*128][TB] bf16 (token-minor);
// part (CTA 0): chunk partials [nchunks][TB][E] f32; logits [TB][E] f32;
// sel: selected logits [TB][16] f32 + ids [TB][16] i32.
__host__ __device__ inline RouteSmem route_smem(int TB, int CPC, int E, int nchunks) {
  RouteSmem s{};
  size_t o = 0;
  s.ws = o;     o += (size_t)CPC * 128 * E * 2;
  s.xs = o;     o += (size_t)CPC * 128 * TB * 2;
  o = (o + 15) & ~size_t(15);
  s.part = o;   o += (size_t)nchunks * TB * E * 4;
  s.logits = o; o += (size_t)TB * E * 4;
  s.sel = o;    o += (size_t)TB * 16 * 8;
  s.bias = o;   o += (size_t)E * 4;
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
  const int nchunks = H / 128;
  const int CPC = nchunks / CL;
  const RouteSmem L = route_smem(TB, CPC, E, nchunks);
  uint16_t* wsm = reinterpret_cast<uint16_t*>(smem + L.ws);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* logits = reinterpret_cast<float*>(smem + L.logits);
  float* sel_v = reinterpret_cast<float*>(smem + L.sel);
  int* sel_i = reinterpret_cast<int*>(sel_v + TB * 16);
  float* bias_s = reinterpret_cast<float*>(smem + L.bias);
  const int tid = threadIdx.x;
  const int tok0 = blockIdx.y * TB;
  const int c0 = rank * CPC;

  // The router rows [c0*128, (c0+CPC)*128) (contiguous) and the bias are layer parameters:
  // they are staged while the previous kernel of the stream finishes (programmatic launch);
  // the hidden rows, which it may have written, only after the grid dependency resolves.
  {
    const uint4* src = reinterpret_cast<const uint4*>(router_w + (size_t)c0 * 128 * E);
    uint4* dst = reinterpret_cast<uint4*>(wsm);
    const int n16 = CPC * 128 * E / 8;
    for (int i0 = tid; i0 < n16; i0 += kRouteThreads * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * kRouteThreads < n16) v[u] = src[i0 + u * kRouteThreads];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * kRouteThreads < n16) dst[i0 + u * kRouteThreads] = v[u];
    }
    if (rank == 0)
      for (int e = tid; e < E; e += kRouteThreads) bias_s[e] = bias != nullptr ? bias[e] : 0.0f;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  {
    for (int i = tid; i < TB * CPC * 128; i += kRouteThreads) {
      const int t = i / (CPC * 128), k = i % (CPC * 128);
      xs[k * TB + t] = tok0 + t < M ? hidden[(size_t)(tok0 + t) * H + c0 * 128 + k] : (uint16_t)0;
    }
  }
  __syncthreads();

  float* part0 = cluster.map_shared_rank(part, 0);
  for (int e = tid; e < E; e += kRouteThreads) {
    for (int cl = 0; cl < CPC; ++cl) {
      float acc[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[t] = 0.0f;
      const uint16_t* wcol = wsm + (size_t)cl * 128 * E + e;
      const uint16_t* xk = xs + (size_t)cl * 128 * TB;
#pragma unroll 16
      for (int k = 0; k < 128; ++k) {
        const float w = bf16_bits_to_float(wcol[k * E]);
        uint32_t xw[(TB + 1) / 2];
        if constexpr (TB == 8) {
          const uint4 q = *reinterpret_cast<const uint4*>(xk + k * TB);
          xw[0] = q.x; xw[1] = q.y; xw[2] = q.z; xw[3] = q.w;
        } else if constexpr (TB == 2) {
          xw[0] = *reinterpret_cast<const uint32_t*>(xk + k * TB);
        } else {
          xw[0] = xk[k * TB];
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          const uint16_t b = (uint16_t)((t & 1) ? (xw[t / 2] >> 16) : (xw[t / 2] & 0xFFFF));
          acc[t] = __fmaf_rn(bf16_bits_to_float(b), w, acc[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < TB; ++t) part0[((size_t)(c0 + cl) * TB + t) * E + e] = acc[t];
    }
  }
  cluster.sync();  // CTA 0 holds every chunk partial
  if (rank != 0) return;

  for (int i = tid; i < TB * E; i += kRouteThreads) {
    const int t = i / E, e = i % E;
    const float* pc = part + (size_t)t * E + e;
    const size_t cstride = (size_t)TB * E;
    float l = 0.0f;
#pragma unroll 8
    for (int c = 0; c < nchunks; ++c) l = __fadd_rn(l, pc[c * cstride]);
    if (bias != nullptr) l = __fadd_rn(l, bias_s[e]);
    logits[t * E + e] = l;
  }
  __syncthreads();
  // rank selection: expert e goes to slot rank(e) if rank(e) < K (four independent counts
  // over 16-byte loads of the token's logits)
  for (int i = tid; i < TB * E; i += kRouteThreads) {
    const int t = i / E, e = i % E;
    const float4* lt4 = reinterpret_cast<const float4*>(logits + t * E);
    const float v = logits[t * E + e];
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll 8
    for (int q = 0; q < E / 4; ++q) {
      const float4 w = lt4[q];
      const int e2 = 4 * q;
      r0 += (w.x > v) || (w.x == v && e2 < e);
      r1 += (w.y > v) || (w.y == v && e2 + 1 < e);
      r2 += (w.z > v) || (w.z == v && e2 + 2 < e);
      r3 += (w.w > v) || (w.w == v && e2 + 3 < e);
    }
    const int rk = r0 + r1 + r2 + r3;
    if (rk < K) {
      sel_v[t * 16 + rk] = v;
      sel_i[t * 16 + rk] = e;
    }
  }
  __syncthreads();
  // weights: one warp per token
  const int warp = tid / 32, lane = tid % 32;
  for (int t = warp; t < TB; t += kRouteThreads / 32) {
    if (tok0 + t >= M) break;
    const float lmax = sel_v[t * 16];
    float den = 0.0f;
    if (renorm) {
      for (int j = 0; j < K; ++j) den = __fadd_rn(den, expf(__fsub_rn(sel_v[t * 16 + j], lmax)));
    } else {
      for (int e = lane; e < E; e += 32) den = __fadd_rn(den, expf(__fsub_rn(logits[t * E + e], lmax)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, off));
    }
    if (lane < K) {
      const size_t o = (size_t)(tok0 + t) * K + lane;
      ids[o] = sel_i[t * 16 + lane];
      wts[o] = __fdiv_rn(expf(__fsub_rn(sel_v[t * 16 + lane], lmax)), den);
    }
  }
}

// ---------------------------------------------------------------------------------------
// Many tokens: one CTA per block of kBigTB tokens covers all E experts over the whole hidden
// dimension, so every logit's chunk chains and their ascending chunk sum stay inside one
// thread. The router's 128-row chunks (128 * E * 2 contiguous bytes) stream through a
// two-slot shared-memory ring with bulk asynchronous copies; thread (e, token group) holds
// kBigTB/2 chain accumulators and the running logits of its tokens.
// ---------------------------------------------------------------------------------------
constexpr int kBigTB = 16;

__host__ __device__ inline size_t route_big_smem(int E) {
  return 16 + (size_t)2 * 128 * E * 2 + (size_t)2 * 128 * kBigTB * 4 + (size_t)kBigTB * E * 4 +
         (size_t)kBigTB * 16 * 8 + 64;
}

__global__ void __launch_bounds__(256)
    route_big_kernel(const uint16_t* __restrict__ hidden, const uint16_t* __restrict__ router_w,
                     const float* __restrict__ bias, int M, int H, int E, int K, int renorm,
                     int32_t* __restrict__ ids, float* __restrict__ wts) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);                 // [2] ring barriers
  uint16_t* wring = reinterpret_cast<uint16_t*>(smem + 16);          // [2][128][E]
  float* xring = reinterpret_cast<float*>(wring + (size_t)2 * 128 * E);  // [2][128][kBigTB] f32
  float* logits = xring + (size_t)2 * 128 * kBigTB;                  // [kBigTB][E]
  float* sel_v = logits + kBigTB * E;                                // [kBigTB][16]
  int* sel_i = reinterpret_cast<int*>(sel_v + kBigTB * 16);          // [kBigTB][16]
  const int tid = threadIdx.x;
  const int tok0 = blockIdx.x * kBigTB;
  const int nchunks = H / 128;
  const uint32_t wbytes = 128u * (uint32_t)E * 2u;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (tid == 0) {
    for (int b = 0; b < 2; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&bar[b])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto issue = [&](int c) {  // router chunk c -> slot c & 1 (thread 0)
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar[c & 1]);
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(wring + (size_t)(c & 1) * 128 * E);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(wbytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
                 "l"(router_w + (size_t)c * 128 * E), "r"(wbytes), "r"(b)
                 : "memory");
  };
  if (tid == 0) {
    issue(0);
    if (nchunks > 1) issue(1);
  }
  // thread <-> expert e, token group g (tokens g*8 .. g*8+7)
  const int e = tid % E, g = tid / E;
  const int ngroups = 256 / E;  // >= 2 for E <= 128
  constexpr int kTPG = kBigTB / 2;
  float logit[kTPG];
#pragma unroll
  for (int t = 0; t < kTPG; ++t) logit[t] = 0.0f;
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    // this chunk's hidden values, token-minor: xring[slot][k][t]
    float* xs = xring + (size_t)(c & 1) * 128 * kBigTB;
    for (int i = tid; i < 128 * kBigTB; i += 256) {
      const int t = i / 128, k = i % 128;
      xs[k * kBigTB + t] = tok0 + t < M ? bf16_bits_to_float(hidden[(size_t)(tok0 + t) * H + c * 128 + k]) : 0.0f;
    }
    __syncthreads();
    {  // bounded wait for the router chunk
      const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar[c & 1]);
      const uint32_t par = (c >> 1) & 1;
      uint32_t done = 0;
      const uint64_t t0 = globaltimer_ns();
      while (ok) {
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(b), "r"(par) : "memory");
        if (done) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) ok = false;
      }
    }
    if (g < 2 && ok) {
      const uint16_t* wcol = wring + (size_t)(c & 1) * 128 * E + e;
      const float* xk = xs + g * kTPG;
      float acc[kTPG];
#pragma unroll
      for (int t = 0; t < kTPG; ++t) acc[t] = 0.0f;
#pragma unroll 8
      for (int k = 0; k < 128; ++k) {
        const float w = bf16_bits_to_float(wcol[k * E]);
        const float4 x0 = *reinterpret_cast<const float4*>(xk + k * kBigTB);
        const float4 x1 = *reinterpret_cast<const float4*>(xk + k * kBigTB + 4);
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int t = 0; t < kTPG; ++t) acc[t] = __fmaf_rn(xv[t], w, acc[t]);
      }
#pragma unroll
      for (int t = 0; t < kTPG; ++t) logit[t] = __fadd_rn(logit[t], acc[t]);
    }
    __syncthreads();  // slot c & 1 is free again
    if (tid == 0 && c + 2 < nchunks) issue(c + 2);
  }
  (void)ngroups;
  // a router chunk that never arrived (bounded wait ran out): the block's tokens get id -1,
  // which the expert FFN skips and reports as MOE_STATUS_BAD_EXPERT_ID
  ok = __syncthreads_and(ok);
  if (!ok) {
    for (int i = tid; i < kBigTB * K; i += 256)
      if (tok0 + i / K < M) {
        ids[(size_t)tok0 * K + i] = -1;
        wts[(size_t)tok0 * K + i] = 0.0f;
      }
    return;
  }
  if (g < 2) {
#pragma unroll
    for (int t = 0; t < kTPG; ++t) {
      float l = logit[t];
      if (bias != nullptr) l = __fadd_rn(l, bias[e]);
      logits[(g * kTPG + t) * E + e] = l;
    }
  }
  __syncthreads();
  for (int i = tid; i < kBigTB * E; i += 256) {  // rank selection, ties to the lower index
    const int t = i / E, ee = i % E;
    const float* lt = logits + t * E;
    const float v = lt[ee];
    int rk = 0;
    for (int e2 = 0; e2 < E; ++e2) {
      const float v2 = lt[e2];
      rk += (v2 > v) || (v2 == v && e2 < ee);
    }
    if (rk < K) {
      sel_v[t * 16 + rk] = v;
      sel_i[t * 16 + rk] = ee;
    }
  }
  __syncthreads();
  const int warp = tid / 32, lane = tid % 32;
  for (int t = warp; t < kBigTB; t += 8) {
    if (tok0 + t >= M) break;
    const float lmax = sel_v[t * 16];
    float den = 0.0f;
    if (renorm) {
      for (int j = 0; j < K; ++j) den = __fadd_rn(den, expf(__fsub_rn(sel_v[t * 16 + j], lmax)));
    } else {
      for (int ee = lane; ee < E; ee += 32) den = __fadd_rn(den, expf(__fsub_rn(logits[t * E + ee], lmax)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, off));
    }
    if (lane < K) {
      const size_t o = (size_t)(tok0 + t) * K + lane;
      ids[o] = sel_i[t * 16 + lane];
      wts[o] = __fdiv_rn(expf(__fsub_rn(sel_v[t * 16 + lane], lmax)), den);
    }
  }
}

namespace {

// CL CTAs per cluster (<= 16, a divisor of the chunk count): one 128-row chunk per CTA
// whenever the chunk count allows
int route_cluster(int nchunks) {
  for (int c = kRouteMaxCluster; c >= 1; --c)
    if (nchunks % c == 0) return c;
  return 1;
}

template <int TB>
cudaError_t launch_route_t(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int M,
                           int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st) {
  const int nchunks = H / 128;
  const int CL = route_cluster(nchunks);
  const RouteSmem L = route_smem(TB, nchunks / CL, E, nchunks);
  if (L.total > 227 * 1024) return cudaErrorInvalidConfiguration;
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

// Tokens per cluster: 1 for a token or two, 8 (one 16-byte load of token values per k)
// when there are many and CTA 0's chunk partials [nchunks][8][E] still fit.
cudaError_t launch_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int M,
                         int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st) {
  const int nchunks = H / 128;
  if (M >= 512 && E <= 128) {
    static std::once_flag once;
    std::call_once(once, [] {
      cudaFuncSetAttribute(route_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M + kBigTB - 1) / kBigTB), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = route_big_smem(E);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_big_kernel, hidden, router_w, bias, M, H, E, K, renorm, ids, wts);
  }
  if (M >= 16 && route_smem(8, nchunks / route_cluster(nchunks), E, nchunks).total <= 227 * 1024)
    return launch_route_t<8>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  if (M >= 4 && route_smem(2, nchunks / route_cluster(nchunks), E, nchunks).total <= 227 * 1024)
    return launch_route_t<2>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  return launch_route_t<1>(hidden, router_w, bias, M, H, E, K, renorm, ids, wts, st);
}

}  // namespace moe
