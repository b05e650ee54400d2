// fused.cu -- the whole layer for a few routed pairs in one launch: routing (softmax and
// top-k over BF16 logits), the hidden quantisation, gate/up on tcgen05, SiLU(gate)*up with
// the FP8 requantisation, down on tcgen05, and the slot-order combine.
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (one producer
// made of semantic routing, gate/up, SiLU and quantisation, down-partial and metadata
// stages, and a route reducer with its own fixed reduction order); docs/compiler/
// architecture.md, accepted M=1 MoE objects (gate/up, SiLU+quant, down/reduce);
// "Inferact/amd-kernels" README (split-K and expert partials summed in a fixed order --
// by the last CTA or inside the next kernel -- never with atomic adds).
//
// Shape of the work. One thread-block cluster of 16 CTAs per routed (token, slot) pair;
// the clusters never wait on one another. Inside a cluster CTA r owns
//   * routing: the 128-wide hidden chunks c = r, r+16, ... of every expert (the fma chain
//     of each chunk, k ascending from 0); the chunk partials go to every CTA of the
//     cluster (distributed shared memory), and each CTA then adds them in chunk order,
//     adds the bias, and picks the top K by rank (ties to the lower expert) -- the same
//     arithmetic as the router kernel, so the ids and weights are bit-identical to it;
//   * gate/up: K blocks kb = r, r+16, ... of every 128-row output unit u (128 gate rows +
//     the matching 128 up rows). Swap-AB MMAs (the weight tile is the M=128 operand, the
//     token's FP8 hidden row the first of N=16 B rows) put one weight row per TMEM lane;
//     the epilogue forms each promoted term t_kb = P_kb * (sa_kb * sw_kb) and stores it into
//     the unit's owner CTA (u mod 16), which sums the terms in kb order from 0, applies
//     silu(g) * u, requantises the 128 values (scale = amax/448) and sends the codes and the
//     scale to every CTA of the cluster;
//   * down: output blocks hb = r, r+16, ... of 128 rows, all K blocks of the activation
//     locally (the promotion chain kb ascending from 0 in registers);
//   * combine: y goes to the workspace; the last of the token's K pairs to finish a block
//     (an arrival ticket per token and block -- a counter, never a value sum) adds
//     w_j * y_j over j ascending in FP32 (multiply then add, from 0) and writes BF16.
// All weight tiles of a CTA (gate/up first, then down) stream through one TMA ring as soon
// as the expert is known; the down tiles wait in the ring for the activation.
// Warp roles: 0 TMA, 1 TMEM + MMA issue, 2-5 epilogue (TMEM lane quadrant = warp % 4),
// all eight warps for the routing chains and the hidden quantisation.
// Cross-CTA signalling: distributed-shared-memory stores followed by one release-arrive per
// destination on an mbarrier of that CTA (acquired at cluster scope by its readers); every
// wait is bounded and reports MOE_STATUS_WAIT_TIMEOUT.
#include <cudaTypedefs.h>

#include <algorithm>

#include "device.h"
#include "tc.cuh"

namespace moe {

constexpr int kFusedCL = 16;
constexpr int kFusedThreads = 256;
constexpr int kFusedTile = 128 * 128;  // one 128 x 128 FP8 weight tile
constexpr int kFusedMaxStages = 8;
constexpr int kFusedTmemCols = 128;    // four 32-column accumulator buffers
constexpr int kFusedMaxTokens = 16;
constexpr int kRouterRow = 136;        // transposed router row: 128 weights + 8 of padding

struct FusedParams {
  int M, H, I, E, K;
  int renorm;
  int nst;                    // ring stages
  const uint16_t* hidden;     // BF16 [M][H]
  const uint16_t* router_w;   // BF16 [H][E] (routing mode)
  const float* bias;          // [E] or null (routing mode)
  int32_t* ids;               // [M][K]: written (routing mode) or read
  float* wts;                 // [M][K]
  const float* s13;           // [E][2I/128][H/128]
  const float* s2w;           // [E][H/128][I/128]
  uint16_t* out;              // BF16 [M][H]
  uint8_t* qa;                // workspace views: hidden codes [M][H], scales [M][H/128]
  float* sa;
  uint8_t* act;               // activation codes [R][I] and scales [R][I/128], pair order
  float* act_scale;
  float* y;                   // down output [R][H] FP32, pair order
  uint32_t* tickets;          // [M][H/128] arrival counters, zero between calls
  Header* hdr;
};

struct FusedSmem {
  size_t ring, hid, actpart, terms, xs, own, logits, sel, sc, bars, total;
  int nkh, cpc, nki, nu, nhb;
};

__host__ __device__ inline size_t fused_align(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ring: stages of one weight tile (before the expert is known: the CTA's router chunks,
// transposed); hid: the CTA's hidden B tiles (2 KB each, row 0 = codes); actpart: the
// activation B tiles (one 1 KB row group per K block of I, +1 KB for the last tile's upper
// rows; rows 1..15 of a tile are never read into an output column that is used); terms: the split-K
// terms of the unit this CTA owns [nkh][256] f32; xs: hidden values f32 [M][cpc][128]; own:
// this CTA's chunk partials [cpc][M][E] f32 (read by the others); logits [M][E]; sel: [M][16]
// f32 + [M][16] i32; sc: scales, weights and ids.
__host__ __device__ inline FusedSmem fused_smem(int nst, int M, int H, int I, int E, int K) {
  FusedSmem s{};
  s.nkh = H / 128;
  s.cpc = (s.nkh + kFusedCL - 1) / kFusedCL;
  s.nki = I / 128;
  s.nu = I / 128;
  s.nhb = H / 128;
  size_t o = 0;
  s.ring = o;    o += (size_t)nst * kFusedTile;
  s.hid = o;     o += (size_t)s.cpc * 2048;
  s.actpart = o; o += (size_t)(s.nki + 1) * 1024;
  s.terms = o;   o += (size_t)s.nkh * 256 * 4;
  s.xs = o;      o += (size_t)M * s.cpc * 128 * 4;
  s.own = o;     o += (size_t)s.cpc * M * E * 4;
  s.logits = o;  o += (size_t)M * E * 4;
  s.sel = o;     o += (size_t)M * 16 * 8;
  s.sc = o;      o += 128 + (size_t)(2 * s.nu * s.cpc + s.cpc * s.nki + s.cpc + s.nki + E + 8) * 4 + (size_t)M * K * 8;
  o = fused_align(o, 16);
  s.bars = o;    o += (size_t)(2 * nst + 13) * 8 + 16;
  s.total = o + 1024;  // alignment slack of the dynamic shared memory base
  return s;
}

template <bool ROUTE>
__global__ void __launch_bounds__(kFusedThreads, 2)
    fused_kernel(const __grid_constant__ CUtensorMap tm13, const __grid_constant__ CUtensorMap tm2,
                 const FusedParams p) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int M = p.M, H = p.H, I = p.I, E = p.E, K = p.K, NS = p.nst;
  const FusedSmem L = fused_smem(NS, M, H, I, E, K);
  const int nkh = L.nkh, cpc = L.cpc, nki = L.nki, nu = L.nu, nhb = L.nhb;
  unsigned char* ring = base + L.ring;
  unsigned char* hid = base + L.hid;
  unsigned char* acttile = base + L.actpart;
  float* terms = reinterpret_cast<float*>(base + L.terms);
  float* xs = reinterpret_cast<float*>(base + L.xs);
  float* own = reinterpret_cast<float*>(base + L.own);
  float* logits = reinterpret_cast<float*>(base + L.logits);
  float* sel_v = reinterpret_cast<float*>(base + L.sel);
  int* sel_i = reinterpret_cast<int*>(sel_v + M * 16);
  uint8_t* code_s = base + L.sc;                           // [128] the owner's codes (16-byte aligned)
  float* sw13_s = reinterpret_cast<float*>(code_s + 128);  // [cpc][2][nu]
  float* sw2_s = sw13_s + 2 * nu * cpc;                    // [cpc][nki]
  float* sa_s = sw2_s + cpc * nki;                         // [cpc]
  float* s2_s = sa_s + cpc;                                // [nki]
  float* bias_s = s2_s + nki;                              // [E]
  float* red = bias_s + E;                                 // [4] warp maxima, [4] flags
  int* flag_s = reinterpret_cast<int*>(red + 4);
  float* twt = red + 8;                                    // [M][K]
  int* tid_s = reinterpret_cast<int*>(twt + M * K);        // [M][K]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + NS;
  uint64_t* accf = bars + 2 * NS;
  uint64_t* acce = accf + 4;
  uint64_t* part_full = acce + 4;  // every routing CTA's partials are here
  uint64_t* terms_full = part_full + 1;  // all 16 CTAs' terms for the owned unit
  uint64_t* act_full = terms_full + 1;   // every unit's activation codes are here
  uint64_t* hid_ready = act_full + 1;    // this CTA's hidden B tiles and scales are written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(hid_ready + 1);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int rank = (int)tc::cluster_rank();
  const int route = (int)tc::cluster_id_x();  // one cluster per routed pair
  const int t_r = route / K, s_r = route % K;
  const int n_mine = rank < nkh ? (nkh - 1 - rank) / kFusedCL + 1 : 0;  // my hidden chunks / K blocks
  const int h_mine = rank < nhb ? (nhb - 1 - rank) / kFusedCL + 1 : 0;  // my 128-row down blocks
  const int n_rt = nkh < kFusedCL ? nkh : kFusedCL;                     // CTAs with routing chunks

  // ---- set-up that reads no dynamic input: barriers, TMEM, the router rows (parameters)
  if (tid == 0) {
    tc::prefetch_tmap(&tm13);
    tc::prefetch_tmap(&tm2);
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 4; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 4);
    }
    tc::mbar_init(part_full, n_rt);
    tc::mbar_init(terms_full, kFusedCL);
    tc::mbar_init(act_full, nu);
    tc::mbar_init(hid_ready, 1);
    tc::fence_mbar_init();
  }
  if (ROUTE) {
    // this CTA's router chunks, transposed to [chunk][expert][k] (rows padded to 136 values so
    // that 16-byte loads of consecutive experts' rows spread over the banks): each routing
    // thread then reads its expert's 128 weights of a chunk as sixteen 16-byte loads
    uint16_t* wt = reinterpret_cast<uint16_t*>(ring);
    const int n8 = 128 * E / 8;  // 8-value groups of one chunk
    for (int cl = 0; cl < n_mine; ++cl) {
      const uint4* src = reinterpret_cast<const uint4*>(p.router_w + (size_t)(rank + kFusedCL * cl) * 128 * E);
      uint16_t* dst = wt + (size_t)cl * E * kRouterRow;
      for (int i = tid; i < n8; i += kFusedThreads) {  // consecutive threads: consecutive k
        const int k = i % 128, e0 = (i / 128) * 8;
        const uint4 v = src[(size_t)k * (E / 8) + e0 / 8];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[(size_t)(e0 + j) * kRouterRow + k] = (uint16_t)((j & 1) ? (w[j / 2] >> 16) : (w[j / 2] & 0xFFFF));
      }
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kFusedTmemCols);
    tc::tmem_relinquish();
  }
  for (int i = tid; i < cpc * 2048 / 16; i += kFusedThreads)  // hidden B tiles: rows 1..15 zero
    reinterpret_cast<uint4*>(hid)[i] = make_uint4(0, 0, 0, 0);
  if (ROUTE)
    for (int e = tid; e < E; e += kFusedThreads) bias_s[e] = p.bias != nullptr ? p.bias[e] : 0.0f;
  tc::cluster_arrive();  // every CTA's barriers are initialised before anyone signals them

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- hidden values of this CTA's chunks (all tokens when routing, else the pair's token)
  {
    const int t0 = ROUTE ? 0 : t_r, t1 = ROUTE ? M : t_r + 1;
    const int per_tok = n_mine * 32;  // 4 values per item
    for (int i = tid; i < (t1 - t0) * per_tok; i += kFusedThreads) {
      const int t = t0 + i / per_tok, r2 = i % per_tok, cl = r2 / 32, k4 = (r2 % 32) * 4;
      const uint2 raw =
          *reinterpret_cast<const uint2*>(p.hidden + (size_t)t * H + (size_t)(rank + kFusedCL * cl) * 128 + k4);
      float* d = xs + ((size_t)t * cpc + cl) * 128 + k4;
      d[0] = bf16_bits_to_float(raw.x & 0xFFFF);
      d[1] = bf16_bits_to_float(raw.x >> 16);
      d[2] = bf16_bits_to_float(raw.y & 0xFFFF);
      d[3] = bf16_bits_to_float(raw.y >> 16);
    }
  }
  bool ok = true;
  tc::fence_before_sync();  // the TMEM allocation's address, for every warp
  __syncthreads();
  tc::fence_after_sync();
  tc::cluster_wait();

  if (ROUTE) {
    // ---- routing: chunk chains, every chunk's partials gathered, chunk-order sums, rank top-k
    const uint16_t* wt = reinterpret_cast<const uint16_t*>(ring);
    for (int e = tid; e < E; e += kFusedThreads) {
      for (int cl = 0; cl < n_mine; ++cl) {
        const uint4* wrow = reinterpret_cast<const uint4*>(wt + ((size_t)cl * E + e) * kRouterRow);
        for (int t = 0; t < M; ++t) {
          const float4* x4 = reinterpret_cast<const float4*>(xs + ((size_t)t * cpc + cl) * 128);
          float acc = 0.0f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {  // k = 8j .. 8j+7, ascending
            const uint4 w8 = wrow[j];
            const float4 xa = x4[2 * j], xb = x4[2 * j + 1];
            acc = __fmaf_rn(xa.x, bf16_bits_to_float(w8.x & 0xFFFF), acc);
            acc = __fmaf_rn(xa.y, bf16_bits_to_float(w8.x >> 16), acc);
            acc = __fmaf_rn(xa.z, bf16_bits_to_float(w8.y & 0xFFFF), acc);
            acc = __fmaf_rn(xa.w, bf16_bits_to_float(w8.y >> 16), acc);
            acc = __fmaf_rn(xb.x, bf16_bits_to_float(w8.z & 0xFFFF), acc);
            acc = __fmaf_rn(xb.y, bf16_bits_to_float(w8.z >> 16), acc);
            acc = __fmaf_rn(xb.z, bf16_bits_to_float(w8.w & 0xFFFF), acc);
            acc = __fmaf_rn(xb.w, bf16_bits_to_float(w8.w >> 16), acc);
          }
          own[((size_t)cl * M + t) * E + e] = acc;
        }
      }
    }
    __syncthreads();
    // one release-arrive per destination CTA, in parallel; then every CTA pulls every chunk's
    // partials (chunk c lives in CTA c mod 16) as 16-byte loads
    if (n_mine > 0 && tid < kFusedCL) tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(part_full), tid));
    if (!tc::mbar_wait_cluster(part_full, 0)) ok = false;
    // logit = the chunk partials added in chunk order (chunk c read from CTA c mod 16), + bias
    for (int i = tid; i < M * E; i += kFusedThreads) {
      const int t = i / E, e = i % E;
      const uint32_t la = tc::smem_u32(own + (size_t)t * E + e);
      float l = 0.0f;
#pragma unroll 16
      for (int c = 0; c < nkh; ++c)
        l = __fadd_rn(l, tc::ld_cluster_f32(tc::mapa(la + (uint32_t)((c / kFusedCL) * M * E * 4), (uint32_t)(c % kFusedCL))));
      if (p.bias != nullptr) l = __fadd_rn(l, bias_s[e]);
      logits[t * E + e] = l;
    }
    __syncthreads();
    for (int i = tid; i < M * E; i += kFusedThreads) {
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
    for (int t = warp; t < M; t += kFusedThreads / 32) {
      const float lmax = sel_v[t * 16];
      float den = 0.0f;
      if (p.renorm) {
        for (int j = 0; j < K; ++j) den = __fadd_rn(den, expf(__fsub_rn(sel_v[t * 16 + j], lmax)));
      } else {
        for (int e = lane; e < E; e += 32) den = __fadd_rn(den, expf(__fsub_rn(logits[t * E + e], lmax)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, off));
      }
      if (lane < K) {
        const float w = __fdiv_rn(expf(__fsub_rn(sel_v[t * 16 + lane], lmax)), den);
        twt[t * K + lane] = w;
        tid_s[t * K + lane] = sel_i[t * 16 + lane];
        if (route == 0 && rank == 0) {
          p.ids[t * K + lane] = sel_i[t * 16 + lane];
          p.wts[t * K + lane] = w;
        }
      }
    }
  } else {
    for (int i = tid; i < M * K; i += kFusedThreads) {
      tid_s[i] = p.ids[i];
      twt[i] = p.wts[i];
    }
  }
  __syncthreads();

  const int e = tid_s[t_r * K + s_r];
  const bool valid = e >= 0 && e < E;
  if (!valid && rank == 0 && tid == 0) set_status(p.hdr, MOE_STATUS_BAD_EXPERT_ID);

  const uint32_t tmem = *tmem_slot;  // written by the allocation, before the first block barrier
  const int n_gu = n_mine * nu;           // gate/up pieces (each two tiles)
  const int n_dn = h_mine * nki;          // down pieces (one tile each)

  if (valid && warp == 0) {
    // ---- TMA: gate/up tiles (kb-major, then unit; gate then up), then the down tiles
    const int n_loads = 2 * n_gu + n_dn;
    auto tile = [&](int n, int& x, int& y, const CUtensorMap*& m) {
      if (n < 2 * n_gu) {
        const int pc = n / 2, cl = pc / nu, u = pc % nu, gu = n % 2;
        x = (rank + kFusedCL * cl) * 128;
        y = e * 2 * I + gu * I + u * 128;
        m = &tm13;
      } else {
        const int dn = n - 2 * n_gu, hl = dn / nki, kb2 = dn % nki;
        x = kb2 * 128;
        y = e * H + (rank + kFusedCL * hl) * 128;
        m = &tm2;
      }
    };
    auto load = [&](int n) {  // one tile into its ring stage, after the stage is free
      const int s = n % NS;
      if (!tc::mbar_wait(&empty[s], ((n / NS) & 1) ^ 1)) return false;
      int x, y;
      const CUtensorMap* m;
      tile(n, x, y, m);
      tc::mbar_arrive_expect_tx(&full[s], kFusedTile);
      tc::tma_load_2d(ring + (size_t)s * kFusedTile, m, &full[s], x, y);
      return true;
    };
    const int first = n_loads < NS ? n_loads : NS;
    if (lane == 0) {
      tc::fence_proxy_async_smem();  // the routing reads of the ring precede these writes
      for (int n = 0; n < first && ok; ++n) ok = load(n);
    }
    __syncwarp();
    // the rest of this CTA's tiles into L2 at once, one per lane: the weight stream runs at
    // the memory's pace, not at the pace at which ring stages free up (the down tiles wait in
    // the ring for the activation)
    for (int n = first + lane; n < n_loads; n += 32) {
      int x, y;
      const CUtensorMap* m;
      tile(n, x, y, m);
      tc::tma_prefetch_2d(m, x, y);
    }
    if (lane == 0)
      for (int n = first; n < n_loads && ok; ++n) ok = load(n);
  } else if (valid && warp == 1) {
    // ---- MMA issue: gate/up pieces into 32-column buffers (gate 0..15, up 16..31), then
    // the down pieces once every unit's activation codes have arrived
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3(128, 16);
      if (n_gu > 0 && !tc::mbar_wait(hid_ready, 0)) ok = false;
      for (int pc = 0; pc < n_gu + n_dn && ok; ++pc) {
        const int buf = pc & 3;
        if (pc == n_gu) {
          if (!tc::mbar_wait_cluster(act_full, 0)) { ok = false; break; }
          tc::fence_proxy_async_smem();  // codes written by other CTAs, read by the tensor core
        }
        int s0, s1 = -1;
        if (pc < n_gu) {
          s0 = (2 * pc) % NS;
          s1 = (2 * pc + 1) % NS;
          if (!tc::mbar_wait(&full[s0], ((2 * pc) / NS) & 1) || !tc::mbar_wait(&full[s1], ((2 * pc + 1) / NS) & 1)) {
            ok = false;
            break;
          }
        } else {
          const int n = 2 * n_gu + (pc - n_gu);
          s0 = n % NS;
          if (!tc::mbar_wait(&full[s0], (n / NS) & 1)) { ok = false; break; }
        }
        if (!tc::mbar_wait(&acce[buf], ((pc >> 2) & 1) ^ 1)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t d = tmem + buf * 32;
        if (pc < n_gu) {
          const int cl = pc / nu;
          const uint64_t db = tc::sdesc_sw128(tc::smem_u32(hid + (size_t)cl * 2048));
          const uint64_t dg = tc::sdesc_sw128(tc::smem_u32(ring + (size_t)s0 * kFusedTile));
          const uint64_t du = tc::sdesc_sw128(tc::smem_u32(ring + (size_t)s1 * kFusedTile));
#pragma unroll
          for (int k = 0; k < 4; ++k) tc::mma_e4m3(d, dg + 2 * k, db + 2 * k, idesc, k > 0);
#pragma unroll
          for (int k = 0; k < 4; ++k) tc::mma_e4m3(d + 16, du + 2 * k, db + 2 * k, idesc, k > 0);
          tc::mma_commit(&empty[s0]);
          tc::mma_commit(&empty[s1]);
        } else {
          const int kb2 = (pc - n_gu) % nki;
          const uint64_t db = tc::sdesc_sw128(tc::smem_u32(acttile + (size_t)kb2 * 1024));
          const uint64_t dw = tc::sdesc_sw128(tc::smem_u32(ring + (size_t)s0 * kFusedTile));
#pragma unroll
          for (int k = 0; k < 4; ++k) tc::mma_e4m3(d, dw + 2 * k, db + 2 * k, idesc, k > 0);
          tc::mma_commit(&empty[s0]);
        }
        tc::mma_commit(&accf[buf]);
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ---- epilogue: thread <-> weight row (warp % 4) * 32 + lane of the 128-row tile
    const int q = warp & 3, row = q * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    if (valid) {
      // the block scales of this CTA's tiles (off the weight stream's critical path)
      for (int i = row; i < n_mine * 2 * nu; i += 128) {
        const int cl = i / (2 * nu), gu = (i / nu) % 2, u = i % nu;
        const int kb = rank + kFusedCL * cl;
        sw13_s[i] = p.s13[((size_t)e * (2 * nu) + gu * nu + u) * nkh + kb];
      }
      for (int i = row; i < h_mine * nki; i += 128) {
        const int hl = i / nki, kb2 = i % nki;
        const int hb = rank + kFusedCL * hl;
        sw2_s[i] = p.s2w[((size_t)e * nhb + hb) * nki + kb2];
      }
      tc::named_bar(1, 128);
      if (n_gu > 0 && ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(hid_ready, 0));  // sa_s
      for (int pc = 0; pc < n_gu; ++pc) {
        const int buf = pc & 3, cl = pc / nu, u = pc % nu;
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&accf[buf], (pc >> 2) & 1));
        tc::fence_after_sync();
        float pg = 0.0f, pu = 0.0f;
        if (ok) tc::tmem_ld1x2(tl + buf * 32, tl + buf * 32 + 16, pg, pu);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[buf]);
        const float a = sa_s[cl];
        const float tg = __fmul_rn(pg, __fmul_rn(a, sw13_s[(cl * 2 + 0) * nu + u]));
        const float tu = __fmul_rn(pu, __fmul_rn(a, sw13_s[(cl * 2 + 1) * nu + u]));
        const int kb = rank + kFusedCL * cl;
        const uint32_t la = tc::smem_u32(terms + (size_t)kb * 256 + row);
        const uint32_t owner = (uint32_t)(u % kFusedCL);
        tc::st_cluster_f32(tc::mapa(la, owner), tg);
        tc::st_cluster_f32(tc::mapa(la + 512, owner), tu);
      }
      tc::named_bar(1, 128);
      if (warp == 2 && lane < nu) tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(terms_full), (uint32_t)lane));

      if (rank < nu) {
        // ---- owner of unit `rank`: the promotion chain over kb ascending, SiLU*up, the
        // activation's 128-value quantisation, the codes and scale to every CTA
        const int u = rank;
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait_cluster(terms_full, 0));
        float g = 0.0f, uu = 0.0f;
        for (int kb = 0; kb < nkh; ++kb) {
          g = __fadd_rn(g, terms[kb * 256 + row]);
          uu = __fadd_rn(uu, terms[kb * 256 + 128 + row]);
        }
        const float act = silu_mul(g, uu);
        float m = fabsf(act);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) red[q] = m;
        tc::named_bar(1, 128);
        const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        const float s2 = quant_scale(amax);
        const uint8_t code = (uint8_t)(e4m3x2_encode(__fdiv_rn(act, s2), 0.0f) & 0xFF);
        code_s[row] = code;
        p.act[(size_t)route * I + u * 128 + row] = code;
        if (row == 0) p.act_scale[(size_t)route * nu + u] = s2;
        tc::named_bar(1, 128);
        {  // 8 x 16 bytes of codes to each of the 16 CTAs: one 16-byte store per thread
          const int d = row / 8, c16 = row % 8;
          const uint4 v = reinterpret_cast<const uint4*>(code_s)[c16];
          tc::st_cluster_v4(tc::mapa(tc::smem_u32(acttile + (size_t)u * 1024 + c16 * 16), d), v);
          if (row < kFusedCL) tc::st_cluster_f32(tc::mapa(tc::smem_u32(s2_s + u), row), s2);
        }
        tc::named_bar(1, 128);
        if (warp == 2 && lane < kFusedCL) tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(act_full), (uint32_t)lane));
      }

      // ---- down: chain over kb ascending per 128-row block, then y and the combine
      if (h_mine > 0 && ok) ok = __all_sync(0xffffffffu, tc::mbar_wait_cluster(act_full, 0));
      for (int hl = 0; hl < h_mine; ++hl) {
        float y = 0.0f;
        for (int kb2 = 0; kb2 < nki; ++kb2) {
          const int pc = n_gu + hl * nki + kb2, buf = pc & 3;
          if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&accf[buf], (pc >> 2) & 1));
          tc::fence_after_sync();
          float pd = 0.0f;
          if (ok) pd = tc::tmem_ld1(tl + buf * 32);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&acce[buf]);
          y = __fadd_rn(y, __fmul_rn(pd, __fmul_rn(s2_s[kb2], sw2_s[hl * nki + kb2])));
        }
        const int hb = rank + kFusedCL * hl, h = hb * 128 + row;
        p.y[(size_t)route * H + h] = y;
        __threadfence();
        tc::named_bar(1, 128);
        if (row == 0) flag_s[0] = (int)atomicAdd(&p.tickets[(size_t)t_r * nhb + hb], 1u) == K - 1;
        tc::named_bar(1, 128);
        if (flag_s[0]) {  // the last of the token's pairs for this block: the combine
          __threadfence();
          float acc = 0.0f;
          for (int j = 0; j < K; ++j) {
            const int ej = tid_s[t_r * K + j];
            if (ej < 0 || ej >= E) continue;
            const float yj = j == s_r ? y : __ldcg(p.y + (size_t)(t_r * K + j) * H + h);
            acc = __fadd_rn(acc, __fmul_rn(twt[t_r * K + j], yj));
          }
          p.out[(size_t)t_r * H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
          if (row == 0) p.tickets[(size_t)t_r * nhb + hb] = 0u;
        }
        tc::named_bar(1, 128);
      }
    } else {
      // a skipped pair: no loads and no exchange; its tickets still count, so the token's
      // last pair combines the valid ones
      for (int hl = 0; hl < h_mine; ++hl) {
        const int hb = rank + kFusedCL * hl;
        if (row == 0) flag_s[0] = (int)atomicAdd(&p.tickets[(size_t)t_r * nhb + hb], 1u) == K - 1;
        tc::named_bar(1, 128);
        if (flag_s[0]) {
          __threadfence();
          const int h = hb * 128 + row;
          float acc = 0.0f;
          for (int j = 0; j < K; ++j) {
            const int ej = tid_s[t_r * K + j];
            if (ej < 0 || ej >= E) continue;
            acc = __fadd_rn(acc, __fmul_rn(twt[t_r * K + j], __ldcg(p.y + (size_t)(t_r * K + j) * H + h)));
          }
          p.out[(size_t)t_r * H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
          if (row == 0) p.tickets[(size_t)t_r * nhb + hb] = 0u;
        }
        tc::named_bar(1, 128);
      }
    }
  } else if (warp >= 6) {
    // ---- helpers: the pair's hidden row, quantised per 128 columns into this CTA's B tiles
    // (row 0) and, once per token, into the workspace view
    for (int cl = warp - 6; cl < n_mine; cl += 2) {
      const int kb = rank + kFusedCL * cl;
      const float* v = xs + ((size_t)t_r * cpc + cl) * 128 + lane * 4;
      const float x0 = v[0], x1 = v[1], x2 = v[2], x3 = v[3];
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sc = quant_scale(amax);
      const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
      const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
      reinterpret_cast<uint32_t*>(hid + (size_t)cl * 2048)[lane] = lo | (hi << 16);
      if (lane == 0) sa_s[cl] = sc;
      if (s_r == 0) {  // one copy of the token's codes, for the workspace view
        reinterpret_cast<uint32_t*>(p.qa + (size_t)t_r * H + (size_t)kb * 128)[lane] = lo | (hi << 16);
        if (lane == 0) p.sa[(size_t)t_r * nkh + kb] = sc;
      }
    }
    tc::fence_proxy_async_smem();  // generic writes of the B tiles before the tensor core reads them
    tc::named_bar(2, 64);
    if (warp == 6 && lane == 0) tc::mbar_arrive(hid_ready);
  }
  if (!ok) set_status(p.hdr, MOE_STATUS_WAIT_TIMEOUT);
  // no CTA leaves while another may still store into its shared memory
  tc::fence_before_sync();
  tc::cluster_arrive();
  tc::cluster_wait();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kFusedTmemCols);
  }
}

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);

namespace {

struct FusedPlan {
  int nst;
  size_t smem;
};

// Deepest ring (4..8 stages of one tile) whose CTA keeps the launch's clusters resident: two
// CTAs per SM (so that up to 14 clusters of 16 are resident at once) when there are more
// routed pairs than one-CTA-per-SM clusters fit, otherwise up to the per-block limit. The
// router chunks of a CTA are staged in the ring, so it must hold them.
FusedPlan plan_fused(const DeviceInfo& d, int M, int H, int I, int E, int K) {
  const int R = M * K;
  const int nkh = H / 128, cpc = (nkh + kFusedCL - 1) / kFusedCL;
  const size_t two_per_sm = d.smem_per_sm / 2 - 1024;
  const size_t limit = R > 7 ? two_per_sm : d.smem_optin;
  for (int nst = kFusedMaxStages; nst >= 4; --nst) {
    if ((size_t)nst * kFusedTile < (size_t)cpc * E * kRouterRow * 2) break;
    const size_t smem = fused_smem(nst, M, H, I, E, K).total;
    if (smem <= limit) return FusedPlan{nst, smem};
  }
  return FusedPlan{0, 0};
}

}  // namespace

// Whether the fused launch covers this call (host arithmetic only).
bool fused_capable(int M, int H, int I, int E, int K) {
  if (M < 1 || M > kFusedMaxTokens || (int64_t)M * K > kFusedCL) return false;
  if (E > kFusedThreads || E % 4 || I / 128 > kFusedCL || H / 128 > 4 * kFusedCL) return false;
  const DeviceInfo d = device_info();
  if (d.sms == 0) return false;
  return plan_fused(d, M, H, I, E, K).nst > 0;
}

// route: ids/wts are outputs (routing in the kernel); otherwise inputs.
cudaError_t launch_fused(bool route, const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                         int renorm, int32_t* ids, float* wts, const uint8_t* w13, const float* s13,
                         const uint8_t* w2, const float* s2w, uint16_t* out, int M, int H, int I, int E, int K,
                         const WsPtrs& ws, uint32_t* tickets, cudaStream_t st) {
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  const FusedPlan pl = plan_fused(d, M, H, I, E, K);
  if (pl.nst == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap t13, t2;
  if (!make_tmap_u8(&t13, w13, (uint64_t)H, (uint64_t)E * 2 * I, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&t2, w2, (uint64_t)I, (uint64_t)E * H, 128)) return cudaErrorInvalidValue;
  static PerDeviceOnce once;
  once_per_device(once, [&] {
    for (auto k : {fused_kernel<true>, fused_kernel<false>}) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
      cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
  });
  FusedParams prm{};
  prm.M = M; prm.H = H; prm.I = I; prm.E = E; prm.K = K;
  prm.renorm = renorm;
  prm.nst = pl.nst;
  prm.hidden = hidden; prm.router_w = router_w; prm.bias = bias;
  prm.ids = ids; prm.wts = wts;
  prm.s13 = s13; prm.s2w = s2w; prm.out = out;
  prm.qa = ws.qa; prm.sa = ws.sa; prm.act = ws.act; prm.act_scale = ws.act_scale; prm.y = ws.y;
  prm.tickets = tickets;
  prm.hdr = ws.hdr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(kFusedCL * M * K), 1, 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFusedCL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (route) return cudaLaunchKernelEx(&cfg, fused_kernel<true>, t13, t2, prm);
  return cudaLaunchKernelEx(&cfg, fused_kernel<false>, t13, t2, prm);
}

}  // namespace moe
