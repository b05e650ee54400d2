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
// Work unit: (routed pair j, 128-wide block u of the activation). A unit's gate/up is the
// 128 gate rows and the 128 matching up rows of output block u over all K blocks of the
// hidden row; its SiLU*up and requantisation give the activation block u (128 FP8 codes and
// one scale); its down part is the K block u of the down projection for every output row:
// the promoted terms t_u[h] = P_u[h] * (s2_u * sw2[h/128][u]). The units are spread over as
// many 16-CTA clusters as are resident at once with one CTA per SM (the clusters never wait
// on one another). Inside a cluster CTA r owns
//   * routing: the 128-wide hidden chunks c = r, r+16, ... of every expert (the fma chain
//     of each chunk, k ascending from 0); every CTA receives all chunk partials (copied
//     into its shared memory by their CTAs), adds them in chunk order, adds the bias and picks the top
//     K by rank (ties to the lower expert) -- the router kernel's arithmetic, so the ids and
//     weights are bit-identical to it; every cluster routes for itself;
//   * gate/up: K blocks kb = r, r+16, ... of each of its units. Swap-AB MMAs (the weight
//     tile is the M=128 operand, the token's FP8 hidden row the first of N=16 B rows) put one
//     weight row per TMEM lane; the epilogue forms each promoted term P_kb * (sa_kb * sw_kb)
//     and stores it into the unit's owner CTA, whose helper warps add the terms in kb order
//     from 0, apply silu(g) * u, requantise the 128 values (scale = amax/448) and send the
//     codes and the scale to every CTA of the cluster;
//   * down: output rows hb*128 .. +127 for hb = r, r+16, ...; each term goes to the
//     workspace, and the last of a token's K * (I/128) terms of a block to arrive (an arrival
//     ticket per token and block -- a counter, never a value sum) forms
//     y_j = sum over u ascending of t_u (from 0) for each slot j, and
//     out = bf16(sum over j ascending of w_j * y_j), FP32 multiply then add, from 0:
//     exactly the down and combine chains of the contract.
// The weight tiles of a CTA stream through one deep TMA ring in a fixed order: every unit's
// gate/up tiles, then the down tiles, which wait in the ring for their unit's activation
// (so a unit's activation exchange never holds up the gate/up of the units after it).
// Warp roles: 0 TMA, 1 TMEM + MMA issue, 2-5 epilogue (TMEM lane quadrant = warp % 4),
// 6-7 helpers (hidden quantisation, then the owner's SiLU and requantisation); all eight
// warps route.
// Cross-CTA signalling: distributed-shared-memory stores followed by one release-arrive per
// destination on an mbarrier of that CTA (acquired at cluster scope by its readers); every
// wait is bounded and reports MOE_STATUS_WAIT_TIMEOUT.
#include <cudaTypedefs.h>

#include <algorithm>

#include "device.h"
#include "launch.h"
#include "tc.cuh"

namespace moe {

constexpr int kFusedCL = 16;
constexpr int kFusedThreads = 256;
constexpr int kFusedTile = 128 * 128;  // one 128 x 128 FP8 weight tile
constexpr int kFusedMaxStages = 12;
constexpr int kFusedTmemCols = 256;    // gate/up: 4 x 32 columns; down: 8 x 16 columns
constexpr int kFusedMaxUnits = 16;     // units per cluster (one owner CTA each)
constexpr int kFusedMaxTokens = 16;
constexpr int kFusedLag = kFusedMaxUnits;  // a unit's down pieces follow every gate/up piece

struct FusedParams {
  int M, H, I, E, K;
  int renorm;
  int nst;                    // ring stages
  int nc;                     // clusters
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
  float* yt;                  // down terms [M][H][K * I/128 padded to 4] FP32
  uint32_t* tickets;          // [M][H/128] arrival counters, zero between calls
  Header* hdr;
};

struct FusedSmem {
  size_t ring, hid, act, terms, tstage, astage, part, xs, own, logits, sel, seq, sc, bars, total;
  int nkh, cpc, nhb, hpc;
};

__host__ __device__ inline size_t fused_align(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ring: stages of one weight tile (before the experts are known: the CTA's router chunks
// [chunk][k][expert]); hid: hidden B tiles [M][cpc] (2 KB each, row 0 =
// codes); act: activation B tiles, one 1 KB row group per unit (+1 KB for the last tile's
// upper rows; rows 1..15 of a tile are never read into an output column that is used, and
// row 1 carries the unit's activation scale in its first 4 bytes);
// terms: the split-K terms of the unit this CTA owns [nkh][256] f32 (copied in by every CTA);
// tstage: this CTA's terms [U][cpc][256] f32, staged for the copies; astage: the owner's
// activation codes and scale [U][144 B], staged for the copies; part: every chunk's routing
// partials [nkh][M][E] f32 (copied in by every CTA); xs: hidden values f32 [M][cpc][128];
// own: this CTA's chunk partials [cpc][M][E] f32, staged for the copies; logits
// [M][E]; sel: [M][16] f32 + [M][16] i32; seq: the CTA's piece order; sc: scales, weights,
// ids.
__host__ __device__ inline FusedSmem fused_smem(int nst, int M, int H, int I, int E, int K, int U) {
  FusedSmem s{};
  s.nkh = H / 128;
  s.cpc = (s.nkh + kFusedCL - 1) / kFusedCL;
  s.nhb = H / 128;
  s.hpc = (s.nhb + kFusedCL - 1) / kFusedCL;
  (void)I;
  size_t o = 0;
  s.ring = o;    o += (size_t)nst * kFusedTile;
  s.hid = o;     o += (size_t)M * s.cpc * 2048;
  s.act = o;     o += (size_t)(U + 1) * 1024;
  s.terms = o;   o += (size_t)s.nkh * 256 * 4;
  s.tstage = o;  o += (size_t)U * s.cpc * 256 * 4;
  s.astage = o;  o += (size_t)U * 144;
  s.part = o;    o += (size_t)s.nkh * M * E * 4;
  s.xs = o;      o += (size_t)M * s.cpc * 128 * 4;
  s.own = o;     o += (size_t)s.cpc * M * E * 4;
  s.logits = o;  o += (size_t)M * E * 4;
  s.sel = o;     o += (size_t)M * 16 * 8;
  s.seq = o;     o += fused_align((size_t)U * (s.cpc + s.hpc) * 4, 16);
  s.sc = o;      o += 128 + (size_t)(U * s.cpc * 2 + U * s.hpc + M * s.cpc + U + E + 8) * 4 + (size_t)M * K * 8;
  o = fused_align(o, 16);
  s.bars = o;    o += (size_t)(2 * nst + 28 + 2 * U) * 8 + 16;
  s.total = o + 1024;  // alignment slack of the dynamic shared memory base
  return s;
}

// A piece of a CTA's work: the gate/up of one unit for one K block (two tiles) or the down
// of one unit for one 128-row output block (one tile). Pieces of a unit whose expert id is
// invalid issue no loads or MMAs; its down pieces still count their arrival tickets.
struct Piece {
  int down, i, idx;
};
__device__ __forceinline__ Piece piece_of(int code) { return Piece{(code >> 15) & 1, (code >> 8) & 127, code & 255}; }

// tm13: w13 as [2E][I][H] (z = 2e gate, 2e + 1 up), box 128 bytes x 128 rows x 2: one
// instruction loads a unit's gate and up tiles of one K block (32 KB, gate then up);
// tm2: w2 as [E*H][I], box 128 bytes x 128 rows.
template <bool ROUTE>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tm13, const __grid_constant__ CUtensorMap tm2,
                 const FusedParams p) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int M = p.M, H = p.H, I = p.I, E = p.E, K = p.K, NS = p.nst;
  const int nu = I / 128;
  const int KNp = (K * nu + 3) & ~3;  // a row's down terms in the workspace, padded to 16 bytes
  const int cid = (int)tc::cluster_id_x();
  const int RU = M * K * nu;                                  // units of the launch
  const int U = cid < RU ? (RU - 1 - cid) / p.nc + 1 : 0;     // units of this cluster: cid + i * nc
  const int Umax = (RU + p.nc - 1) / p.nc;                    // the layout uses the largest count
  const FusedSmem L = fused_smem(NS, M, H, I, E, K, Umax);
  const int nkh = L.nkh, cpc = L.cpc, nhb = L.nhb, hpc = L.hpc;
  unsigned char* ring = base + L.ring;
  unsigned char* hid = base + L.hid;
  unsigned char* acttile = base + L.act;
  float* terms = reinterpret_cast<float*>(base + L.terms);
  float* tstage = reinterpret_cast<float*>(base + L.tstage);
  unsigned char* astage = base + L.astage;
  float* part = reinterpret_cast<float*>(base + L.part);
  float* xs = reinterpret_cast<float*>(base + L.xs);
  float* own = reinterpret_cast<float*>(base + L.own);
  float* logits = reinterpret_cast<float*>(base + L.logits);
  float* sel_v = reinterpret_cast<float*>(base + L.sel);
  int* sel_i = reinterpret_cast<int*>(sel_v + M * 16);
  int* seq = reinterpret_cast<int*>(base + L.seq);
  uint8_t* code_s = base + L.sc;                           // [128] the owner's codes (16-byte aligned)
  float* sw13_s = reinterpret_cast<float*>(code_s + 128);  // [U][cpc][2]
  float* sw2_s = sw13_s + Umax * cpc * 2;                  // [U][hpc]
  float* sa_s = sw2_s + Umax * hpc;                        // [M][cpc]
  float* s2_s = sa_s + M * cpc;                            // [U]
  float* bias_s = s2_s + Umax;                             // [E]
  float* red = bias_s + E;                                 // [2] warp maxima, [4] flags
  int* flag_s = reinterpret_cast<int*>(red + 4);
  float* twt = red + 8;                                    // [M][K]
  int* tid_s = reinterpret_cast<int*>(twt + M * K);        // [M][K]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + NS;
  uint64_t* accf = bars + 2 * NS;  // gate/up accumulators [4]
  uint64_t* acce = accf + 4;
  uint64_t* accf2 = acce + 4;      // down accumulators [8]
  uint64_t* acce2 = accf2 + 8;
  uint64_t* part_full = acce2 + 8;         // every chunk's routing partials are here
  uint64_t* hid_ready = part_full + 1;     // this CTA's hidden B tiles and scales are written
  uint64_t* terms_full = hid_ready + 1;    // [U] every K block's terms of the unit are here
  uint64_t* act_full = terms_full + Umax;  // [U] the unit's activation codes are here
  uint64_t* rbar = act_full + Umax;        // this CTA's router chunks have landed
  uint64_t* drainb = rbar + 1;             // every MMA this CTA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drainb + 1);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int rank = (int)tc::cluster_rank();
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
    for (int b = 0; b < 8; ++b) {
      tc::mbar_init(&accf2[b], 1);
      tc::mbar_init(&acce2[b], 4);
    }
    tc::mbar_init(part_full, 1);
    tc::mbar_init(hid_ready, 1);
    tc::mbar_init(rbar, 1);
    tc::mbar_init(drainb, 1);
    for (int i = 0; i < Umax; ++i) {
      tc::mbar_init(&terms_full[i], 1);
      tc::mbar_init(&act_full[i], 1);
    }
    // the bytes each exchange copies into this CTA: every chunk's routing partials, every
    // K block's terms of the units it owns, each unit's activation codes and scale
    if (ROUTE) tc::mbar_arrive_expect_tx(part_full, (uint32_t)(nkh * M * E * 4));
    for (int i = 0; i < U; ++i) {
      if (i % kFusedCL == rank) tc::mbar_arrive_expect_tx(&terms_full[i], (uint32_t)(nkh * 1024));
      tc::mbar_arrive_expect_tx(&act_full[i], 144u);
    }
    tc::fence_mbar_init();
  }
  if (ROUTE) {
    // this CTA's router chunks [chunk][k][expert] (contiguous rows of the router matrix) by
    // bulk asynchronous copies, and the bias: layer parameters, read before the dependency
    if (tid == 0 && n_mine > 0) {
      const uint32_t chunk = 128u * (uint32_t)E * 2u;
      tc::mbar_arrive_expect_tx(rbar, chunk * (uint32_t)n_mine);
      for (int cl = 0; cl < n_mine; ++cl)
        tc::bulk_load(ring + (size_t)cl * chunk, p.router_w + (size_t)(rank + kFusedCL * cl) * 128 * E, chunk, rbar);
    }
    for (int e = tid; e < E; e += kFusedThreads) bias_s[e] = p.bias != nullptr ? p.bias[e] : 0.0f;
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kFusedTmemCols);
    tc::tmem_relinquish();
  }
  // this CTA's piece order: unit i's gate/up pieces, and after the gate/up pieces of unit
  // i + lag the down pieces of unit i; bit 15 = down, bits 8..14 = unit, 0..7 = index
  for (int i = tid; i < U + kFusedLag; i += kFusedThreads) {
    const int d = i - kFusedLag;
    int o = (i < U ? i : U) * n_mine + (d > 0 ? (d < U ? d : U) : 0) * h_mine;
    if (i < U)
      for (int c = 0; c < n_mine; ++c) seq[o++] = (i << 8) | c;
    if (d >= 0 && d < U)
      for (int c = 0; c < h_mine; ++c) seq[o++] = (1 << 15) | (d << 8) | c;
  }
  for (int i = tid; i < M * cpc * 2048 / 16; i += kFusedThreads)  // hidden B tiles: rows 1..15 zero
    reinterpret_cast<uint4*>(hid)[i] = make_uint4(0, 0, 0, 0);
  tc::cluster_arrive();  // every CTA's barriers are initialised before anyone signals them

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- hidden values of this CTA's chunks, every token
  {
    const int per_tok = n_mine * 32;  // 4 values per item
    for (int i = tid; i < M * per_tok; i += kFusedThreads) {
      const int t = i / per_tok, r2 = i % per_tok, cl = r2 / 32, k4 = (r2 % 32) * 4;
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
    // thread e2 runs the chains of experts 2*e2 and 2*e2+1 as one packed FP32x2 fma per k
    // (two IEEE fmas, bit-identical to separate ones): one 4-byte load gives both weights
    if (n_mine > 0 && !tc::mbar_wait(rbar, 0)) ok = false;
    const uint32_t* wr2 = reinterpret_cast<const uint32_t*>(ring);
    for (int e2 = tid; e2 < E / 2; e2 += kFusedThreads) {
      for (int cl = 0; cl < n_mine; ++cl) {
        const uint32_t* wcol = wr2 + (size_t)cl * 128 * (E / 2) + e2;
        for (int t = 0; t < M; ++t) {
          const float* xk = xs + ((size_t)t * cpc + cl) * 128;
          uint64_t acc = 0ull;
#pragma unroll 16
          for (int k = 0; k < 128; ++k) {
            const uint32_t w = wcol[(size_t)k * (E / 2)];
            const uint64_t w2 = tc::f2pack(w << 16, w & 0xFFFF0000u);  // bf16 -> f32: (expert 2e2, 2e2+1)
            const uint32_t xb = __float_as_uint(xk[k]);
            acc = tc::f2fma(tc::f2pack(xb, xb), w2, acc);
          }
          float a0, a1;
          tc::f2unpack(acc, a0, a1);
          own[((size_t)cl * M + t) * E + 2 * e2] = a0;
          own[((size_t)cl * M + t) * E + 2 * e2 + 1] = a1;
        }
      }
    }
    tc::fence_proxy_async_smem();  // the partials are read by the copies below
    __syncthreads();
    // each chunk's partials to every CTA of the cluster, one copy per (chunk, destination)
    if (tid < n_mine * kFusedCL) {
      const int cl = tid / kFusedCL, d = tid % kFusedCL, c = rank + kFusedCL * cl;
      tc::bulk_copy_cluster(tc::mapa(tc::smem_u32(part + (size_t)c * M * E), (uint32_t)d), own + (size_t)cl * M * E,
                            (uint32_t)(M * E * 4), tc::mapa(tc::smem_u32(part_full), (uint32_t)d));
    }
    if (!tc::mbar_wait(part_full, 0)) ok = false;
    for (int i = tid; i < M * E; i += kFusedThreads) {
      const int t = i / E, e = i % E;
      float l = 0.0f;
#pragma unroll 16
      for (int c = 0; c < nkh; ++c) l = __fadd_rn(l, part[((size_t)c * M + t) * E + e]);  // chunk order
      if (p.bias != nullptr) l = __fadd_rn(l, bias_s[e]);
      logits[t * E + e] = l;
    }
    __syncthreads();
    // rank of each expert: two adjacent threads count the larger logits (ties: lower index)
    // in one half of the experts each, and add their counts
    for (int i0 = 0; i0 < M * E; i0 += kFusedThreads / 2) {
      const int i = i0 + tid / 2, half = tid & 1;
      const bool live = i < M * E;
      const int t = live ? i / E : 0, e = live ? i % E : 0;
      const float4* lt4 = reinterpret_cast<const float4*>(logits + t * E) + half * (E / 8);
      const float v = logits[t * E + e];
      int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll 8
      for (int q = 0; q < E / 8; ++q) {
        const float4 w = lt4[q];
        const int e2 = 4 * q + half * (E / 2);
        r0 += (w.x > v) || (w.x == v && e2 < e);
        r1 += (w.y > v) || (w.y == v && e2 + 1 < e);
        r2 += (w.z > v) || (w.z == v && e2 + 2 < e);
        r3 += (w.w > v) || (w.w == v && e2 + 3 < e);
      }
      int rk = r0 + r1 + r2 + r3;
      rk += __shfl_xor_sync(0xffffffffu, rk, 1);
      if (live && half == 0 && rk < K) {
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
        if (cid == 0 && rank == 0) {
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

  auto unit_expert = [&](int i) {
    const int ej = tid_s[(cid + i * p.nc) / nu];
    return (ej >= 0 && ej < E) ? ej : -1;
  };
  const int n_seq = U * (n_mine + h_mine);
  if (rank == 0 && tid < U && unit_expert(tid) < 0) set_status(p.hdr, MOE_STATUS_BAD_EXPERT_ID);
  const uint32_t tmem = *tmem_slot;  // written by the allocation, before the first block barrier

  if (warp == 0) {
    // ---- TMA: the tiles of the pieces with a valid expert, in piece order

    // lane 0 issues the ring's loads in piece order (the first NS stages at once). A gate/up
    // piece takes an aligned pair of stages (s, s + 1) loaded by one 3-D box whose bytes
    // complete on full[s]; full[s + 1] gets a plain arrival so that every stage's phases
    // advance alike. All gate/up pieces come first, so their pairs start at even tile counts.
    if (lane == 0) {
      tc::fence_proxy_async_smem();  // the routing reads of the ring precede these writes
      int n = 0;
      for (int k = 0; k < n_seq && ok; ++k) {
        const Piece pc = piece_of(seq[k]);
        const int e = unit_expert(pc.i);
        if (e < 0) continue;
        const int u = (cid + pc.i * p.nc) % nu;
        const int s = n % NS;
        if (!pc.down) {
          if (!tc::mbar_wait(&empty[s], ((n / NS) & 1) ^ 1) ||
              !tc::mbar_wait(&empty[s + 1], (((n + 1) / NS) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&full[s], 2 * kFusedTile);
          tc::mbar_arrive(&full[s + 1]);
          tc::tma_load_3d(ring + (size_t)s * kFusedTile, &tm13, &full[s], (rank + kFusedCL * pc.idx) * 128, u * 128,
                          2 * e);
          n += 2;
        } else {
          if (!tc::mbar_wait(&empty[s], ((n / NS) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&full[s], kFusedTile);
          tc::tma_load_2d(ring + (size_t)s * kFusedTile, &tm2, &full[s], u * 128, e * H + (rank + kFusedCL * pc.idx) * 128);
          n += 1;
        }
      }
      // no load is still writing when the CTA leaves: the last phase of each stage issued has
      // completed (a no-op unless a wait gave up)
      for (int j = n - 1; j >= 0 && j >= n - NS; --j)
        if (!tc::mbar_wait(&full[j % NS], (j / NS) & 1)) ok = false;
    }
  } else if (warp == 1) {
    // ---- MMA issue in piece order: gate/up into 32-column buffers (gate 0..15, up 16..31),
    // down into 16-column buffers once the unit's activation codes have arrived
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3(128, 16);
      if (n_mine > 0 && !tc::mbar_wait(hid_ready, 0)) ok = false;
      int n = 0, ng = 0, nd = 0;
      for (int k = 0; k < n_seq && ok; ++k) {
        const Piece pc = piece_of(seq[k]);
        if (unit_expert(pc.i) < 0) continue;
        const int j = (cid + pc.i * p.nc) / nu;
        if (!pc.down) {
          const int s0 = n % NS, s1 = (n + 1) % NS, buf = ng & 3;
          if (!tc::mbar_wait(&full[s0], (n / NS) & 1) || !tc::mbar_wait(&full[s1], ((n + 1) / NS) & 1) ||
              !tc::mbar_wait(&acce[buf], ((ng >> 2) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t d = tmem + buf * 32;
          const uint64_t db = tc::sdesc_sw128(tc::smem_u32(hid + ((size_t)(j / K) * cpc + pc.idx) * 2048));
          const uint64_t dg = tc::sdesc_sw128(tc::smem_u32(ring + (size_t)s0 * kFusedTile));
          const uint64_t du = tc::sdesc_sw128(tc::smem_u32(ring + (size_t)s1 * kFusedTile));
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::mma_e4m3(d, dg + 2 * q, db + 2 * q, idesc, q > 0);
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::mma_e4m3(d + 16, du + 2 * q, db + 2 * q, idesc, q > 0);
          tc::mma_commit(&empty[s0]);
          tc::mma_commit(&empty[s1]);
          tc::mma_commit(&accf[buf]);
          n += 2;
          ++ng;
        } else {
          const int s0 = n % NS, buf = nd & 7;
          if (pc.idx == 0 && !tc::mbar_wait(&act_full[pc.i], 0)) {  // the codes, copied in by the owner
            ok = false;
            break;
          }
          if (!tc::mbar_wait(&full[s0], (n / NS) & 1) || !tc::mbar_wait(&acce2[buf], ((nd >> 3) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t d = tmem + 128 + buf * 16;
          const uint64_t db = tc::sdesc_sw128(tc::smem_u32(acttile + (size_t)pc.i * 1024));
          const uint64_t dw = tc::sdesc_sw128(tc::smem_u32(ring + (size_t)s0 * kFusedTile));
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::mma_e4m3(d, dw + 2 * q, db + 2 * q, idesc, q > 0);
          tc::mma_commit(&empty[s0]);
          tc::mma_commit(&accf2[buf]);
          n += 1;
          ++nd;
        }
      }
      // every arrival the MMAs owe this CTA's barriers has landed before the CTA can leave
      tc::mma_commit(drainb);
      if (!tc::mbar_wait(drainb, 0)) ok = false;
    }
  } else if (warp < 6) {
    // ---- epilogue: thread <-> weight row (warp % 4) * 32 + lane of the 128-row tile
    const int q = warp & 3, row = q * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    // the block scales of this CTA's tiles (off the weight stream's critical path)
    for (int x = row; x < U * n_mine * 2; x += 128) {
      const int i = x / (n_mine * 2), cl = (x / 2) % n_mine, gu = x % 2;
      const int u = (cid + i * p.nc) % nu, e = unit_expert(i);
      const int kb = rank + kFusedCL * cl;
      sw13_s[(i * cpc + cl) * 2 + gu] = e < 0 ? 0.0f : p.s13[((size_t)e * (2 * nu) + gu * nu + u) * nkh + kb];
    }
    for (int x = row; x < U * h_mine; x += 128) {
      const int i = x / h_mine, hl = x % h_mine;
      const int u = (cid + i * p.nc) % nu, e = unit_expert(i);
      const int hb = rank + kFusedCL * hl;
      sw2_s[i * hpc + hl] = e < 0 ? 0.0f : p.s2w[((size_t)e * nhb + hb) * nu + u];
    }
    tc::named_bar(1, 128);
    if (n_mine > 0 && ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(hid_ready, 0));  // sa_s
    int ng = 0, nd = 0;
    for (int k = 0; k < n_seq; ++k) {
      const Piece pc = piece_of(seq[k]);
      const int w = cid + pc.i * p.nc, j = w / nu, u = w % nu, t = j / K;
      const bool real = unit_expert(pc.i) >= 0;
      if (!pc.down) {
        if (!real) continue;
        const int buf = ng & 3;
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&accf[buf], (ng >> 2) & 1));
        tc::fence_after_sync();
        float pg = 0.0f, pu = 0.0f;
        if (ok) tc::tmem_ld1x2(tl + buf * 32, tl + buf * 32 + 16, pg, pu);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[buf]);
        ++ng;
        const float a = sa_s[t * cpc + pc.idx];
        const float tg = __fmul_rn(pg, __fmul_rn(a, sw13_s[(pc.i * cpc + pc.idx) * 2 + 0]));
        const float tu = __fmul_rn(pu, __fmul_rn(a, sw13_s[(pc.i * cpc + pc.idx) * 2 + 1]));
        const int kb = rank + kFusedCL * pc.idx;
        float* st = tstage + ((size_t)pc.i * cpc + pc.idx) * 256;
        st[row] = tg;
        st[128 + row] = tu;
        tc::fence_proxy_async_smem();  // read by the copy
        tc::named_bar(1, 128);
        if (warp == 2 && lane == 0) {  // the piece's 256 terms into the owner's K block kb
          const uint32_t owner = (uint32_t)(pc.i % kFusedCL);
          tc::bulk_copy_cluster(tc::mapa(tc::smem_u32(terms + (size_t)kb * 256), owner), st, 1024u,
                                tc::mapa(tc::smem_u32(&terms_full[pc.i]), owner));
        }
      } else {
        // a term of the down chain: t_u[h] for this unit's K block u, to the workspace
        if (!real) continue;
        const int hb = rank + kFusedCL * pc.idx, h = hb * 128 + row;
        const int buf = nd & 7;
        if (pc.idx == 0 && ok)  // the unit's scale, copied in by its owner
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&act_full[pc.i], 0));
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&accf2[buf], (nd >> 3) & 1));
        tc::fence_after_sync();
        float pd = 0.0f;
        if (ok) pd = tc::tmem_ld1(tl + 128 + buf * 16);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce2[buf]);
        ++nd;
        const float s2u = *reinterpret_cast<const float*>(acttile + (size_t)pc.i * 1024 + 128);
        p.yt[((size_t)t * H + h) * KNp + (j % K) * nu + u] = __fmul_rn(pd, __fmul_rn(s2u, sw2_s[pc.i * hpc + pc.idx]));
      }
    }
    // arrival tickets: one add per (token, 128-row block) of this CTA, counting its units of
    // that token (skipped pairs' units too); the add that completes K * (I/128) arrivals is the
    // last, and its CTA sums the terms and combines the slots
    __threadfence();
    tc::named_bar(1, 128);
    for (int t = 0; t < M; ++t) {
      int n_t = 0;  // units of token t in this cluster
      for (int i = 0; i < U; ++i) n_t += ((cid + i * p.nc) / nu) / K == t;
      if (n_t == 0) continue;
      for (int hl = 0; hl < h_mine; ++hl) {
        const int hb = rank + kFusedCL * hl, h = hb * 128 + row;
        if (row == 0)
          flag_s[0] = (int)atomicAdd(&p.tickets[(size_t)t * nhb + hb], (uint32_t)n_t) + n_t == K * nu;
        tc::named_bar(1, 128);
        if (flag_s[0]) {
          __threadfence();
          // the row's terms, contiguous in (slot, K block) order; 32 of them in flight, then the
          // chains: y over the K blocks ascending, acc over the slots ascending
          const float4* y4 = reinterpret_cast<const float4*>(p.yt + ((size_t)t * H + h) * KNp);
          float acc = 0.0f, y = 0.0f;
          int jj = 0, uu = 0;
          for (int f0 = 0; f0 < K * nu; f0 += 32) {
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (f0 + 4 * q < K * nu) v[q] = __ldcg(y4 + f0 / 4 + q);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              if (f0 + q < K * nu) {
                const float4 w4 = v[q / 4];
                const float val = (q & 3) == 0 ? w4.x : (q & 3) == 1 ? w4.y : (q & 3) == 2 ? w4.z : w4.w;
                const int ej = tid_s[t * K + jj];
                const bool valid_j = ej >= 0 && ej < E;  // a skipped pair contributes nothing
                if (valid_j) y = __fadd_rn(y, val);
                if (++uu == nu) {
                  if (valid_j) acc = __fadd_rn(acc, __fmul_rn(twt[t * K + jj], y));
                  y = 0.0f;
                  uu = 0;
                  ++jj;
                }
              }
            }
          }
          p.out[(size_t)t * H + h] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
          if (row == 0) p.tickets[(size_t)t * nhb + hb] = 0u;
        }
        tc::named_bar(1, 128);
      }
    }
  } else {
    // ---- helpers: the hidden rows quantised per 128 columns into this CTA's B tiles (row 0),
    // and once per token into the workspace view ...
    const int ht = tid - 192;  // 0..63
    for (int x = warp - 6; x < M * n_mine; x += 2) {
      const int t = x / n_mine, cl = x % n_mine, kb = rank + kFusedCL * cl;
      const float* v = xs + ((size_t)t * cpc + cl) * 128 + lane * 4;
      const float x0 = v[0], x1 = v[1], x2 = v[2], x3 = v[3];
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sc = quant_scale(amax);
      const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
      const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
      reinterpret_cast<uint32_t*>(hid + ((size_t)t * cpc + cl) * 2048)[lane] = lo | (hi << 16);
      if (lane == 0) sa_s[t * cpc + cl] = sc;
      if (cid == 0) {
        reinterpret_cast<uint32_t*>(p.qa + (size_t)t * H + (size_t)kb * 128)[lane] = lo | (hi << 16);
        if (lane == 0) p.sa[(size_t)t * nkh + kb] = sc;
      }
    }
    tc::fence_proxy_async_smem();  // generic writes of the B tiles before the tensor core reads them
    tc::named_bar(2, 64);
    if (ht == 0) tc::mbar_arrive(hid_ready);
    // ... then, for the units this CTA owns (unit i is owned by CTA i mod 16): the terms
    // added in kb order from 0, silu(g) * u, the 128-value requantisation, and the codes
    // and the scale to every CTA of the cluster
    for (int i = rank; i < U; i += kFusedCL) {
      if (unit_expert(i) < 0) continue;
      const int w = cid + i * p.nc, j = w / nu, u = w % nu;
      if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&terms_full[i], 0));
      float act[2];
      float m = 0.0f;
#pragma unroll
      for (int r2 = 0; r2 < 2; ++r2) {
        const int rw = ht + 64 * r2;
        float g = 0.0f, uu = 0.0f;
        for (int kb = 0; kb < nkh; ++kb) {
          g = __fadd_rn(g, terms[kb * 256 + rw]);
          uu = __fadd_rn(uu, terms[kb * 256 + 128 + rw]);
        }
        act[r2] = silu_mul(g, uu);
        m = fmaxf(m, fabsf(act[r2]));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[warp - 6] = m;
      tc::named_bar(2, 64);
      const float amax = fmaxf(red[0], red[1]);
      const float s2 = quant_scale(amax);
      unsigned char* ast = astage + (size_t)i * 144;  // codes [128], then the scale
#pragma unroll
      for (int r2 = 0; r2 < 2; ++r2) {
        const uint8_t code = (uint8_t)(e4m3x2_encode(__fdiv_rn(act[r2], s2), 0.0f) & 0xFF);
        ast[ht + 64 * r2] = code;
        p.act[(size_t)j * I + u * 128 + ht + 64 * r2] = code;
      }
      if (ht == 0) {
        *reinterpret_cast<float*>(ast + 128) = s2;
        p.act_scale[(size_t)j * nu + u] = s2;
      }
      tc::fence_proxy_async_smem();  // read by the copies
      tc::named_bar(2, 64);
      if (ht < kFusedCL)  // codes and scale into row 0 and 1 of unit i's B tile of every CTA
        tc::bulk_copy_cluster(tc::mapa(tc::smem_u32(acttile + (size_t)i * 1024), (uint32_t)ht), ast, 144u,
                              tc::mapa(tc::smem_u32(&act_full[i]), (uint32_t)ht));
      tc::named_bar(2, 64);  // red is rewritten by the next owned unit
    }
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
bool make_tmap_u8_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                     uint64_t s2, uint32_t b1, uint32_t b2);

namespace {

struct FusedPlan {
  int nst, nc;
  size_t smem;
};

struct PlanKey {
  int dev, M, H, I, E, K;
};

// The deepest ring (4..12 stages of one tile) that fits one CTA per SM with the units' other
// buffers, and one cluster fewer than the 16-CTA clusters resident at once with that
// footprint (more than half of an SM's shared memory, so that no two CTAs of the launch share
// an SM), capped at the unit count. The occupancy query runs once per device and shape;
// plans are cached.
FusedPlan plan_fused(const DeviceInfo& d, int M, int H, int I, int E, int K) {
  static std::mutex mu;
  static PlanKey keys[64];
  static FusedPlan plans[64];
  static int used = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (keys[i].dev == d.ordinal && keys[i].M == M && keys[i].H == H && keys[i].I == I && keys[i].E == E &&
          keys[i].K == K)
        return plans[i];
  }
  FusedPlan best{0, 0, 0};
  const int RU = M * K * (I / 128);
  const int nkh = H / 128, cpc = (nkh + kFusedCL - 1) / kFusedCL;
  const size_t one_per_sm = d.smem_per_sm / 2 + 1024;
  // clusters resident at once with one CTA per SM (any footprint above half an SM gives the
  // same count)
  int nc = 0;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kFusedCL * 64, 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = one_per_sm;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = kFusedCL;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&nc, fused_kernel<true>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      nc = 0;
    }
  }
  // one cluster fewer than fit: the next launch's clusters (programmatic dependent launch)
  // then find a free GPC more often than when every GPC is taken
  if (nc > 1) --nc;
  nc = std::min(nc, RU);
  const int U = nc > 0 ? (RU + nc - 1) / nc : 0;
  for (int nst = kFusedMaxStages; nc > 0 && U <= kFusedMaxUnits && nst >= 4; nst -= 2) {  // even: gate/up pairs
    if ((size_t)nst * kFusedTile < (size_t)cpc * 128 * E * 2) break;
    const size_t smem = std::max(fused_smem(nst, M, H, I, E, K, U).total, one_per_sm);
    if (smem <= d.smem_optin) {
      best = FusedPlan{nst, nc, smem};
      break;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  if (used < 64) {
    keys[used] = PlanKey{d.ordinal, M, H, I, E, K};
    plans[used] = best;
    ++used;
  }
  return best;
}

void set_fused_attrs(const DeviceInfo& d) {
  static PerDeviceOnce once;
  once_per_device(once, [&] {
    cudaFuncSetAttribute(fused_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
    cudaFuncSetAttribute(fused_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
}

}  // namespace

// Whether the fused launch covers this call (host arithmetic and cached device queries).
bool fused_capable(int M, int H, int I, int E, int K) {
  if (M < 1 || M > kFusedMaxTokens || (int64_t)M * K > kFusedCL) return false;
  if (E > kFusedThreads || E % 8 || I / 128 > kFusedCL || H / 128 > 4 * kFusedCL) return false;
  if ((H / 128 + kFusedCL - 1) / kFusedCL * M > 8) return false;  // hidden B tiles per CTA
  const DeviceInfo d = device_info();
  if (d.sms == 0) return false;
  set_fused_attrs(d);
  return plan_fused(d, M, H, I, E, K).nst > 0;
}

// Routing and the layer as one launch: ids/wts receive the routing. yt: [M][H][K * (I/128)
// rounded up to 4] f32.
cudaError_t launch_fused(bool route, const uint16_t* hidden, const uint16_t* router_w, const float* bias,
                         int renorm, int32_t* ids, float* wts, const uint8_t* w13, const float* s13,
                         const uint8_t* w2, const float* s2w, uint16_t* out, int M, int H, int I, int E, int K,
                         const WsPtrs& ws, float* yt, uint32_t* tickets, cudaStream_t st) {
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  set_fused_attrs(d);
  const FusedPlan pl = plan_fused(d, M, H, I, E, K);
  if (pl.nst == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap t13, t2;
  if (!make_tmap_u8_3d(&t13, w13, (uint64_t)H, (uint64_t)I, (uint64_t)E * 2, (uint64_t)H, (uint64_t)I * H, 128, 2))
    return cudaErrorInvalidValue;
  if (!make_tmap_u8(&t2, w2, (uint64_t)I, (uint64_t)E * H, 128)) return cudaErrorInvalidValue;
  FusedParams prm{};
  prm.M = M; prm.H = H; prm.I = I; prm.E = E; prm.K = K;
  prm.renorm = renorm;
  prm.nst = pl.nst;
  prm.nc = pl.nc;
  prm.hidden = hidden; prm.router_w = router_w; prm.bias = bias;
  prm.ids = ids; prm.wts = wts;
  prm.s13 = s13; prm.s2w = s2w; prm.out = out;
  prm.qa = ws.qa; prm.sa = ws.sa; prm.act = ws.act; prm.act_scale = ws.act_scale;
  prm.yt = yt;
  prm.tickets = tickets;
  prm.hdr = ws.hdr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(kFusedCL * pl.nc), 1, 1);
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
  if (!route) return cudaErrorInvalidValue;  // the kernel's given-routing form is not built
  return cudaLaunchKernelEx(&cfg, fused_kernel<true>, t13, t2, prm);
}

}  // namespace moe
