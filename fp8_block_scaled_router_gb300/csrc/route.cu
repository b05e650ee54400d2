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
// With an RMSNorm in front (Norm::gamma set), the router reads y = bf16((x*r)*gamma) in place
// of x: each CTA first forms r of its tokens (one warp per token, common.cuh's
// row_rms_scale) and converts the hidden values as it stages them.
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "device.h"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kRouteThreads = 256;
constexpr int kRouteMaxCluster = 16;

struct RouteSmem {
  size_t ws, xs, part, logits, sel, bias, rs, total;
};

// ws: router rows [CPC*128][E] bf16 (or one chunk [128][E] at a time when they do not fit);
// xs: hidden [CPC*128][TB] bf16 (token-minor);
// part (CTA 0): chunk partials [nchunks][TB][E] f32; logits [TB][E] f32;
// sel: selected logits [TB][16] f32 + ids [TB][16] i32; rs: RMSNorm r [TB] f32.
// (All shared memory is dynamic: the kernel's dynamic limit is set to the device's opt-in
// maximum, which leaves no room for static shared variables.)
// stage_all: all CPC router chunks of the CTA are held in shared memory (staged before the
// grid dependency); otherwise one chunk at a time streams through it.
__host__ __device__ inline RouteSmem route_smem(int TB, int CPC, int E, int nchunks, bool stage_all) {
  RouteSmem s{};
  size_t o = 0;
  s.ws = o;     o += (size_t)(stage_all ? CPC : 1) * 128 * E * 2;
  s.xs = o;     o += (size_t)CPC * 128 * TB * 2;
  o = (o + 15) & ~size_t(15);
  s.part = o;   o += (size_t)nchunks * TB * E * 4;
  s.logits = o; o += (size_t)TB * E * 4;
  s.sel = o;    o += (size_t)TB * 16 * 8;
  s.bias = o;   o += (size_t)E * 4;
  s.rs = o;     o += (size_t)TB * 4;  // RMSNorm: r of each token
  s.total = o;
  return s;
}

// STREAM: the CTA's router chunks do not fit in shared memory together and stream through it
// one at a time (a separate instantiation, so the common path keeps its register budget).
template <int TB, bool STREAM>
__global__ void __launch_bounds__(kRouteThreads)
    route_kernel(const uint16_t* __restrict__ hidden, const Norm nm, const uint16_t* __restrict__ router_w,
                 const float* __restrict__ bias, int M, int H, int E, int K, int renorm,
                 int32_t* __restrict__ ids, float* __restrict__ wts) {
  constexpr bool stage_all = !STREAM;
  extern __shared__ __align__(16) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int nchunks = H / 128;
  const int CPC = nchunks / CL;
  const RouteSmem L = route_smem(TB, CPC, E, nchunks, stage_all);
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
  if constexpr (STREAM) {
    if (rank == 0)
      for (int e = tid; e < E; e += kRouteThreads) bias_s[e] = bias != nullptr ? bias[e] : 0.0f;
  } else {
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
  if (nm.gamma != nullptr) {
    float* rs = reinterpret_cast<float*>(smem + L.rs);
    const int w = tid / 32;  // TB <= 8 warps: warp t forms r of token t
    if (w < TB && tok0 + w < M) {
      const float r = row_rms_scale(hidden + (size_t)(tok0 + w) * H, H, nm.eps, tid % 32);
      if (tid % 32 == 0) rs[w] = r;
    }
    __syncthreads();
    for (int i = tid; i < TB * CPC * 128; i += kRouteThreads) {
      const int t = i / (CPC * 128), k = i % (CPC * 128);
      xs[k * TB + t] = tok0 + t < M ? norm_bits(hidden[(size_t)(tok0 + t) * H + c0 * 128 + k], rs[t], nm.gamma[c0 * 128 + k])
                                    : (uint16_t)0;
    }
  } else {
    for (int i = tid; i < TB * CPC * 128; i += kRouteThreads) {
      const int t = i / (CPC * 128), k = i % (CPC * 128);
      xs[k * TB + t] = tok0 + t < M ? hidden[(size_t)(tok0 + t) * H + c0 * 128 + k] : (uint16_t)0;
    }
  }
  __syncthreads();

  float* part0 = cluster.map_shared_rank(part, 0);
  // one chunk's fma chains over the plain [128][E] layout at w (k ascending, from 0)
  auto plain_chains = [&](const uint16_t* w, const uint16_t* xk, int e, float (&acc)[TB]) {
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = 0.0f;
    const uint16_t* wcol = w + e;
#pragma unroll 16
    for (int k = 0; k < 128; ++k) {
      const float wv = bf16_bits_to_float(wcol[k * E]);
      uint32_t xw[(TB + 1) / 2];
      if constexpr (TB == 8) {
        const uint4 q = *reinterpret_cast<const uint4*>(xk + k * TB);
        xw[0] = q.x; xw[1] = q.y; xw[2] = q.z; xw[3] = q.w;
      } else if constexpr (TB == 4) {
        const uint2 q = *reinterpret_cast<const uint2*>(xk + k * TB);
        xw[0] = q.x; xw[1] = q.y;
      } else if constexpr (TB == 2) {
        xw[0] = *reinterpret_cast<const uint32_t*>(xk + k * TB);
      } else {
        xw[0] = xk[k * TB];
      }
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const uint16_t b = (uint16_t)((t & 1) ? (xw[t / 2] >> 16) : (xw[t / 2] & 0xFFFF));
        acc[t] = __fmaf_rn(bf16_bits_to_float(b), wv, acc[t]);
      }
    }
  };
  if constexpr (STREAM) {
    // chunks streamed through one staging buffer: stage chunk cl, then every expert's chains
    for (int cl = 0; cl < CPC; ++cl) {
      if (cl > 0) __syncthreads();  // the previous chunk's readers are done
      const uint4* src = reinterpret_cast<const uint4*>(router_w + (size_t)(c0 + cl) * 128 * E);
      uint4* dst = reinterpret_cast<uint4*>(wsm);
      for (int i = tid; i < 128 * E / 8; i += kRouteThreads) dst[i] = src[i];
      __syncthreads();
      for (int e = tid; e < E; e += kRouteThreads) {
        float acc[TB];
        plain_chains(wsm, xs + (size_t)cl * 128 * TB, e, acc);
#pragma unroll
        for (int t = 0; t < TB; ++t) part0[((size_t)(c0 + cl) * TB + t) * E + e] = acc[t];
      }
    }
  } else {
  for (int e = tid; e < E; e += kRouteThreads) {
    for (int cl = 0; cl < CPC; ++cl) {
      float acc[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[t] = 0.0f;
      const uint16_t* xk = xs + (size_t)cl * 128 * TB;
      const uint16_t* wcol = wsm + (size_t)cl * 128 * E + e;
#pragma unroll 16
      for (int k = 0; k < 128; ++k) {
        const float w = bf16_bits_to_float(wcol[k * E]);
        uint32_t xw[(TB + 1) / 2];
        if constexpr (TB == 8) {
          const uint4 q = *reinterpret_cast<const uint4*>(xk + k * TB);
          xw[0] = q.x; xw[1] = q.y; xw[2] = q.z; xw[3] = q.w;
        } else if constexpr (TB == 4) {
          const uint2 q = *reinterpret_cast<const uint2*>(xk + k * TB);
          xw[0] = q.x; xw[1] = q.y;
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
// Many tokens (E = 32 * EPT experts, EPT in {1, 2, 4}): one CTA per kBigTok = 32 tokens
// covers all experts over the whole hidden dimension, so every logit's chunk chains and
// their ascending chunk sum stay inside the CTA. Thread (lane, warp) owns experts
// lane*EPT .. lane*EPT+EPT-1 of the 8 tokens of group (warp % 4): 8*EPT independent fma
// chains, one 8*EPT-byte router load and two broadcast 16-byte hidden loads per k. Warps
// 0-3 take the even chunks, warps 4-7 the odd ones; after each pair of chunks the odd
// partials pass through shared memory and warps 0-3 add them to the running logits in chunk
// order ((l + acc_2p) + acc_2p+1). The router's chunks (128 * E * 2 contiguous bytes) stream
// four ahead through a shared-memory ring with bulk asynchronous copies; the next pair's
// hidden values are prefetched into registers while the current pair is computed.
// Top-k: one warp per token, K rounds of a warp argmax over 64-bit keys (order-preserving
// bits of the logit, then the complement of the expert index: the larger logit wins, ties
// go to the lower index).
// With an RMSNorm in front, the CTA first forms r of its 32 tokens (four per warp) and the
// hidden values become y = bf16((x*r)*gamma) as they are written to the ring.
// ---------------------------------------------------------------------------------------
constexpr int kBigTok = 32;
// packed FP32x2 (sm_100 family): two IEEE round-to-nearest fmas per instruction,
// bit-identical to two __fmaf_rn
__device__ __forceinline__ uint64_t rt_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
  return r;
}
__device__ __forceinline__ void rt_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t rt_fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
constexpr int kBigSlots = 4;

__host__ __device__ inline size_t route_big_smem(int E) {
  return 64 + (size_t)kBigSlots * 128 * E * 2 + (size_t)2 * 128 * kBigTok * 4 + (size_t)128 * 8 * (E / 32) * 4 +
         (size_t)kBigTok * E * 4 + (size_t)kBigTok * 4;
}

__device__ __forceinline__ uint64_t logit_key(float v, int e) {
  uint32_t u = __float_as_uint(v);
  if (v == 0.0f) u = 0u;  // -0 and +0 are one value
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
}

template <int EPT>
__global__ void __launch_bounds__(256, 1)
    route_big_kernel(const uint16_t* __restrict__ hidden, const Norm nm, const uint16_t* __restrict__ router_w,
                     const float* __restrict__ bias, int M, int H, int K, int renorm,
                     int32_t* __restrict__ ids, float* __restrict__ wts) {
  constexpr int E = 32 * EPT;
  constexpr int NA = 8 * EPT;  // accumulators per thread
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);                         // [kBigSlots]
  uint16_t* wring = reinterpret_cast<uint16_t*>(smem + 64);                  // [slots][128][E]
  float* xring = reinterpret_cast<float*>(wring + (size_t)kBigSlots * 128 * E);  // [2][128][32]
  float* xch = xring + 2 * 128 * kBigTok;                                    // [NA][128]
  float* logits = xch + NA * 128;                                            // [32][E]
  float* rs = logits + kBigTok * E;                                          // [32] RMSNorm r
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int grp = warp & 3, par = warp >> 2;
  const int tok0 = blockIdx.x * kBigTok;
  const int nchunks = H / 128, npairs = nchunks / 2;
  constexpr uint32_t wbytes = 128u * E * 2u;

  // layer parameters first (router chunks, bias), while the previous kernel finishes
  auto issue = [&](int c) {
    const int slot = c % kBigSlots;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar[slot]);
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(wring + (size_t)slot * 128 * E);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(wbytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
                 "l"(router_w + (size_t)c * 128 * E), "r"(wbytes), "r"(b)
                 : "memory");
  };
  if (tid == 0) {
    for (int b = 0; b < kBigSlots; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&bar[b])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int c = 0; c < kBigSlots && c < nchunks; ++c) issue(c);
  }
  float bias_r[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) bias_r[j] = bias != nullptr ? bias[lane * EPT + j] : 0.0f;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  const bool normed = nm.gamma != nullptr;
  if (normed) {
    for (int t = warp; t < kBigTok; t += 8) {
      const float r = tok0 + t < M ? row_rms_scale(hidden + (size_t)(tok0 + t) * H, H, nm.eps, lane) : 0.0f;
      if (lane == 0) rs[t] = r;
    }
    __syncthreads();
  }

  // hidden values of one pair of chunks: 2 x 128 x 32 BF16, four 16-byte loads per thread;
  // element (cc, k, t) lands at xring[cc][k][t] as FP32 (with the norm weights beside them)
  uint4 xr[4], gr[4];
  auto load_pair = [&](int p) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int idx = j * 256 + tid, t = idx & 31, g8 = idx >> 5;
      const int cc = g8 >> 4, k8 = (g8 & 15) * 8;
      xr[j] = tok0 + t < M ? *reinterpret_cast<const uint4*>(hidden + (size_t)(tok0 + t) * H + (2 * p + cc) * 128 + k8)
                           : make_uint4(0, 0, 0, 0);
      if (normed) gr[j] = *reinterpret_cast<const uint4*>(nm.gamma + (2 * p + cc) * 128 + k8);
    }
  };
  auto store_pair = [&]() {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int idx = j * 256 + tid, t = idx & 31, g8 = idx >> 5;
      const int cc = g8 >> 4, k8 = (g8 & 15) * 8;
      const uint32_t w4[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
      const uint32_t g4[4] = {gr[j].x, gr[j].y, gr[j].z, gr[j].w};
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint16_t xb = (uint16_t)((u & 1) ? (w4[u / 2] >> 16) : (w4[u / 2] & 0xFFFF));
        const uint16_t gb = (uint16_t)((u & 1) ? (g4[u / 2] >> 16) : (g4[u / 2] & 0xFFFF));
        xring[((size_t)cc * 128 + k8 + u) * kBigTok + t] = normed ? norm_value(xb, rs[t], gb) : bf16_bits_to_float(xb);
      }
    }
  };
  load_pair(0);
  store_pair();
  __syncthreads();

  float logit[NA];
#pragma unroll
  for (int i = 0; i < NA; ++i) logit[i] = 0.0f;
  bool ok = true;
  for (int p = 0; p < npairs; ++p) {
    if (p + 1 < npairs) load_pair(p + 1);
    const int c = 2 * p + par, slot = c % kBigSlots;
    {  // bounded wait for this warp's router chunk
      const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar[slot]);
      const uint32_t ph = (uint32_t)(c / kBigSlots) & 1u;
      uint32_t done = 0;
      const uint64_t t0 = globaltimer_ns();
      while (ok) {
        asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                     : "=r"(done) : "r"(b), "r"(ph) : "memory");
        if (done) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) ok = false;
      }
    }
    // chains of tokens (2u, 2u + 1) of expert j as one FP32 pair: acc2[j * 4 + u]
    uint64_t acc2[NA / 2];
#pragma unroll
    for (int i = 0; i < NA / 2; ++i) acc2[i] = 0ull;
    if (ok) {
      const uint16_t* wk = wring + (size_t)slot * 128 * E + lane * EPT;
      const float* xk = xring + (size_t)par * 128 * kBigTok + grp * 8;
#pragma unroll 4
      for (int k = 0; k < 128; ++k) {
        float w[EPT];
        if constexpr (EPT == 4) {
          const uint2 q = *reinterpret_cast<const uint2*>(wk + k * E);
          w[0] = bf16_bits_to_float(q.x & 0xFFFF); w[1] = bf16_bits_to_float(q.x >> 16);
          w[2] = bf16_bits_to_float(q.y & 0xFFFF); w[3] = bf16_bits_to_float(q.y >> 16);
        } else if constexpr (EPT == 2) {
          const uint32_t q = *reinterpret_cast<const uint32_t*>(wk + k * E);
          w[0] = bf16_bits_to_float(q & 0xFFFF); w[1] = bf16_bits_to_float(q >> 16);
        } else {
          w[0] = bf16_bits_to_float(wk[k * E]);
        }
        const float4 x0 = *reinterpret_cast<const float4*>(xk + k * kBigTok);
        const float4 x1 = *reinterpret_cast<const float4*>(xk + k * kBigTok + 4);
        const uint64_t xp[4] = {rt_pack(x0.x, x0.y), rt_pack(x0.z, x0.w), rt_pack(x1.x, x1.y), rt_pack(x1.z, x1.w)};
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
          const uint64_t wj = rt_pack(w[j], w[j]);
#pragma unroll
          for (int u = 0; u < 4; ++u) acc2[j * 4 + u] = rt_fma2(xp[u], wj, acc2[j * 4 + u]);
        }
      }
    }
    float acc[NA];
#pragma unroll
    for (int i = 0; i < NA / 2; ++i) rt_unpack(acc2[i], acc[2 * i], acc[2 * i + 1]);
    if (par == 1) {
#pragma unroll
      for (int i = 0; i < NA; ++i) xch[i * 128 + grp * 32 + lane] = acc[i];
    }
    __syncthreads();
    if (par == 0) {
#pragma unroll
      for (int i = 0; i < NA; ++i) logit[i] = __fadd_rn(__fadd_rn(logit[i], acc[i]), xch[i * 128 + grp * 32 + lane]);
    }
    __syncthreads();  // the pair's ring slots, hidden values and exchange buffer are free
    if (tid == 0) {
      if (2 * p + kBigSlots < nchunks) issue(2 * p + kBigSlots);
      if (2 * p + 1 + kBigSlots < nchunks) issue(2 * p + 1 + kBigSlots);
    }
    if (p + 1 < npairs) {
      store_pair();
      __syncthreads();
    }
  }
  // a router chunk that never arrived (bounded wait ran out): the block's tokens get id -1,
  // which the expert FFN skips and reports as MOE_STATUS_BAD_EXPERT_ID
  ok = __syncthreads_and(ok);
  if (!ok) {
    for (int i = tid; i < kBigTok * K; i += 256)
      if (tok0 + i / K < M) {
        ids[(size_t)tok0 * K + i] = -1;
        wts[(size_t)tok0 * K + i] = 0.0f;
      }
    return;
  }
  if (par == 0) {
#pragma unroll
    for (int j = 0; j < EPT; ++j)
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        float l = logit[j * 8 + t];
        if (bias != nullptr) l = __fadd_rn(l, bias_r[j]);
        logits[(grp * 8 + t) * E + lane * EPT + j] = l;
      }
  }
  __syncthreads();
  // top-k per token: warp `warp` takes tokens warp, warp + 8, ...
  for (int t = warp; t < kBigTok; t += 8) {
    if (tok0 + t >= M) break;
    const float* lt = logits + t * E;
    uint64_t key[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) key[j] = logit_key(lt[lane * EPT + j], lane * EPT + j);
    int my_e = -1;   // lane r < K: the expert of slot r
    float my_v = 0.0f;
    for (int r = 0; r < K; ++r) {
      uint64_t best = key[0];
#pragma unroll
      for (int j = 1; j < EPT; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
      }
      const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
#pragma unroll
      for (int j = 0; j < EPT; ++j)
        if (lane * EPT + j == e) key[j] = 0;  // taken
      if (lane == r) {
        my_e = e;
        my_v = lt[e];
      }
    }
    const float lmax = __shfl_sync(0xffffffffu, my_v, 0);
    float den = 0.0f;
    if (renorm) {
      for (int j = 0; j < K; ++j) den = __fadd_rn(den, expf(__fsub_rn(__shfl_sync(0xffffffffu, my_v, j), lmax)));
    } else {
#pragma unroll
      for (int j = 0; j < EPT; ++j) den = __fadd_rn(den, expf(__fsub_rn(lt[lane * EPT + j], lmax)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, off));
    }
    if (lane < K) {
      const size_t o = (size_t)(tok0 + t) * K + lane;
      ids[o] = my_e;
      wts[o] = __fdiv_rn(expf(__fsub_rn(my_v, lmax)), den);
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
cudaError_t launch_route_t(const uint16_t* hidden, Norm nm, const uint16_t* router_w, const float* bias, int M,
                           int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st) {
  const int nchunks = H / 128;
  const int CL = route_cluster(nchunks);
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  bool stream = false;
  RouteSmem L = route_smem(TB, nchunks / CL, E, nchunks, true);
  if (L.total > d.smem_optin) {  // the CTA's router chunks do not all fit: stream them
    stream = true;
    L = route_smem(TB, nchunks / CL, E, nchunks, false);
  }
  if (L.total > d.smem_optin) return cudaErrorInvalidConfiguration;
  static PerDeviceOnce once;
  once_per_device(once, [&] {
    cudaFuncSetAttribute(route_kernel<TB, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
    cudaFuncSetAttribute(route_kernel<TB, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncSetAttribute(route_kernel<TB, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
    cudaFuncSetAttribute(route_kernel<TB, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  if (stream)
    return cudaLaunchKernelEx(&cfg, route_kernel<TB, true>, hidden, nm, router_w, bias, M, H, E, K, renorm, ids, wts);
  return cudaLaunchKernelEx(&cfg, route_kernel<TB, false>, hidden, nm, router_w, bias, M, H, E, K, renorm, ids, wts);
}

}  // namespace

// Tokens per cluster: 1 for a token or two, 8 (one 16-byte load of token values per k)
// when there are many and CTA 0's chunk partials [nchunks][8][E] still fit, else 4 or 2
// (the wide hidden sizes: 48 chunks of partials for 8 tokens do not fit).
cudaError_t launch_route(const uint16_t* hidden, Norm nm, const uint16_t* router_w, const float* bias, int M,
                         int H, int E, int K, int renorm, int32_t* ids, float* wts, cudaStream_t st) {
  const int nchunks = H / 128;
  if (M >= 512 && (E == 32 || E == 64 || E == 128) && nchunks % 2 == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M + kBigTok - 1) / kBigTok), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = route_big_smem(E);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static PerDeviceOnce once;
    once_per_device(once, [] {
      const int bytes = (int)route_big_smem(128);
      cudaFuncSetAttribute(route_big_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      cudaFuncSetAttribute(route_big_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      cudaFuncSetAttribute(route_big_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    });
    auto go = [&](auto kern) { return cudaLaunchKernelEx(&cfg, kern, hidden, nm, router_w, bias, M, H, K, renorm, ids, wts); };
    if (E == 128) return go(route_big_kernel<4>);
    if (E == 64) return go(route_big_kernel<2>);
    return go(route_big_kernel<1>);
  }
  const size_t optin = device_info().smem_optin;
  if (M >= 16 && route_smem(8, nchunks / route_cluster(nchunks), E, nchunks, true).total <= optin)
    return launch_route_t<8>(hidden, nm, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  // 4 tokens per cluster only when 2 would need more than one wave of resident CTAs (wide
  // hidden sizes: the CTA's router chunks fill an SM's shared memory): half the clusters, each
  // CTA staging the same router rows
  const int CL = route_cluster(nchunks);
  const size_t smem2 = route_smem(2, nchunks / CL, E, nchunks, true).total;
  const int64_t per_sm2 = (int64_t)(device_info().smem_per_sm / (smem2 + 1024));
  const int64_t resident2 = (int64_t)device_info().sms * per_sm2 * 9 / 10;
  if (M >= 8 && (int64_t)((M + 1) / 2) * CL > resident2 &&
      route_smem(4, nchunks / CL, E, nchunks, true).total <= optin)
    return launch_route_t<4>(hidden, nm, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  if (M >= 4 && route_smem(2, nchunks / route_cluster(nchunks), E, nchunks, true).total <= optin)
    return launch_route_t<2>(hidden, nm, router_w, bias, M, H, E, K, renorm, ids, wts, st);
  return launch_route_t<1>(hidden, nm, router_w, bias, M, H, E, K, renorm, ids, wts, st);
}

}  // namespace moe
