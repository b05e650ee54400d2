// mx_pair.cu -- the few-row expert GEMMs with MXFP4 weights (E2M1 codes, one UE8M0 scale per
// 32 K elements) on tcgen05: one unit per routed (token, slot) pair.
//
// Sources: "Inferact/amd-kernels" README (the MoE shape token mxfp4_h6144_i768_e128_top4;
// split-K and expert partials summed in a fixed order, never with atomics); the older
// kernel-lab README (gfx1151 MXFP4 targets, validated against FP64 dequantised references);
// docs/compiler/architecture.md (accepted M=1 MoE objects: gate/up, SiLU+quant, down/reduce).
//
// Arithmetic (the MXFP4 contract of this library): for each 128-wide K block kb (the
// activation's quantisation group) T_kb = sum over its four 32-wide sub-blocks s ascending
// of P_s * 2^(e_s - 127) (FP32, from 0; P_s = the tensor core's FP32 sum of the 32 products),
// term_kb = T_kb * sa_kb, and the chain acc = acc + term_kb over kb ascending from 0 -- then
// SiLU*up and the E4M3 requantisation (gate/up) or the slot-order combine (down), exactly as
// for FP8 weights.
//
// GB300 design: the pair kernels of the FP8 path with the weight tile in E2M1. The tensor
// map reads the packed codes (64 bytes per weight row and K block) and the TMA unit writes
// them in the tensor core's padded 4-bit layout (each 16 codes in the low 8 bytes of a 16-byte
// chunk, 128-byte swizzle), so a tile has the FP8 tile's footprint and descriptors, while
// the load reads (and its barrier counts) the 64 packed bytes per row: half an FP8 tile. The MMA is kind::f8f6f4 with A = E2M1 (weights) and
// B = E4M3 (the pair's activation row): every E2M1 value is an E4M3 value and every product
// is exact in FP32. One 128x16x32 MMA per 32-wide sub-block writes its own accumulator (four
// per K block and weight tile); the epilogue reads the four sums of its row, scales each by
// the row's UE8M0 factor and adds them in sub-block order. The per-row scale bytes are loaded
// four K blocks ahead of their use. Warp roles: 0 TMA, 1 TMEM + MMA, 2-5 epilogue (TMEM lane
// quadrant = warp % 4); in the gate/up launch warps 1-5 first quantise the hidden row. Split-K
// over a cluster and the down launch's fused combine are those of the FP8 pair kernels
// (distributed-shared-memory stores between cluster barriers). Shared memory is padded so
// that no more CTAs of one launch share an SM than its 512 TMEM columns hold.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "device.h"
#include "launch.h"
#include "pair_plan.h"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace moe {

struct MxParams {
  int H, I, K, E;
  int nkb, nkb_cta, ncb;  // K blocks total / per CTA; 128-row output blocks per unit
  int nst;
  const int32_t* ids;     // [R]
  const uint8_t* wscale;  // UE8M0 [E][N][Kd/32] of the weight rows (N = 2I for gate/up, H for down)
  const float* a_scale;   // down: act_scale [R][I/128]
  const uint16_t* hidden; // gate/up: BF16 [M][H]
  const float* topk_w;    // down
  uint16_t* out;          // down: BF16 [M][H]
  uint8_t* act_out;       // gate/up: [R][I]
  float* act_scale_out;   // gate/up: [R][I/128]
  uint8_t* qa_out;        // gate/up: the hidden codes [M][H] and scales [M][H/128] (slot 0's
  float* sa_out;          //   CTAs of the first output block write them)
  Header* hdr;
};

// kind::f8f6f4 instruction descriptor with A = E2M1 (type code 5), B = E4M3, D = FP32
__host__ __device__ constexpr uint32_t idesc_e2m1_e4m3(int M, int N) { return tc::idesc_e4m3(M, N) | (5u << 7); }

__device__ __forceinline__ float ue8m0(uint32_t e) {
  return e == 255u ? __uint_as_float(0x7FC00000u) : e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// column 0 of the eight sub-block accumulators (gate 0..3 at +0, +16, +32, +48; up 0..3 at
// +64 ..) of this warp's lane quadrant, one wait
__device__ __forceinline__ void tmem_ld_sub8(uint32_t t, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%8];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%1}, [%9];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%2}, [%10];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%3}, [%11];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%4}, [%12];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%5}, [%13];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%6}, [%14];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%7}, [%15];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(t), "r"(t + 16), "r"(t + 32), "r"(t + 48), "r"(t + 64), "r"(t + 80), "r"(t + 96), "r"(t + 112)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_sub4(uint32_t t, float (&v)[4]) {
  uint32_t r[4];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%4];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%1}, [%5];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%2}, [%6];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%3}, [%7];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(t), "r"(t + 16), "r"(t + 32), "r"(t + 48)
      : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// T = sum over the four sub-blocks ascending of P_j * 2^(e_j - 127), from 0 (e: four bytes)
__device__ __forceinline__ float mx_block_sum(const float* p, uint32_t e4) {
  float t = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) t = __fadd_rn(t, __fmul_rn(p[j], ue8m0((e4 >> (8 * j)) & 0xFFu)));
  return t;
}

// tmA: the packed codes as 4-bit elements [rows][Kd] (box 128 codes x 128 rows, padded 4-bit
// layout, 128-byte swizzle); tmB (down): the activation codes [R][I] (box 128 bytes x 16
// rows, 128-byte swizzle).
template <bool GATEUP>
__global__ void __launch_bounds__(kMxThreads, 2)
    mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const MxParams p) {
  using C = MxCfg<GATEUP>;
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int nst = p.nst;
  const MxSmem SL = mx_smem<GATEUP>(nst, p.nkb_cta, p.K);
  unsigned char* stages = base + SL.stages;
  float* xterm = reinterpret_cast<float*>(stages);  // split-K terms, after CTA 0's MMAs
  uint8_t* bq = base + SL.bq;
  float* sas = reinterpret_cast<float*>(base + SL.sas);
  float* comb = reinterpret_cast<float*>(base + SL.comb);
  float* cwt = reinterpret_cast<float*>(base + SL.cw);  // [16] combine weights
  int* cid = reinterpret_cast<int*>(cwt + 16);           // [16] their expert ids
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + SL.bars);
  uint64_t* full = bars;                      // [kMaxStages] the stage's tiles landed
  uint64_t* empty = bars + kMaxStages;        // [kMaxStages] the stage's MMAs are done
  uint64_t* accf = bars + 2 * kMaxStages;     // [2]
  uint64_t* acce = accf + 2;                  // [2]
  uint64_t* drainb = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drainb + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 1);  // [4] warp maxima
  int* e_sh = reinterpret_cast<int*>(red + 4);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int S = (int)cluster.num_blocks();
  const bool clustered = S > 1;
  const int split = GATEUP ? S : 1;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    if (!GATEUP) tc::prefetch_tmap(&tmB);
    for (int s = 0; s < nst; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 4);
    }
    tc::mbar_init(drainb, 1);
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  // down: every CTA of the cluster has started before any writes a peer's shared memory
  if (!GATEUP && clustered) tc::cluster_arrive();
  // B tile rows 1..15 stay zero (row 0, the first 128 bytes, is the quantisers' alone)
  if (GATEUP)
    for (int i = threadIdx.x; i < nst * (C::kBBytes / 16 - 8); i += kMxThreads) {
      const int s = i / (C::kBBytes / 16 - 8), c = 8 + i % (C::kBBytes / 16 - 8);
      reinterpret_cast<uint4*>(stages + s * C::kStageBytes + C::kATiles * C::kABytes)[c] = make_uint4(0, 0, 0, 0);
    }
  const int unit = blockIdx.y;
  int pr, cb, tok;
  if (!GATEUP) {
    tok = unit / p.ncb;
    cb = unit % p.ncb;
    pr = tok * p.K + rank;
  } else {
    pr = unit / p.ncb;
    cb = unit % p.ncb;
    tok = pr / p.K;
  }
  const int kb0 = GATEUP ? rank * p.nkb_cta : 0;
  const int npre = min(nst, p.nkb_cta);
  const int nrows_e = GATEUP ? 2 * p.I : p.H;  // weight rows per expert

  // down: the ids, weights and down weights are complete before this grid can start (the
  // gate/up launch waited for whatever wrote them): the packed weight tiles stream in now,
  // the activation tiles after the grid dependency
  if (!GATEUP && warp == 0) {
    const int e = p.ids[pr];
    if (lane == 0) *e_sh = e;
    if (e >= 0 && e < p.E && lane < npre) {  // one lane per stage: the weight tile, then the B tile
      tc::mbar_arrive_expect_tx(&full[lane], C::kATx + C::kBBytes);
      tc::tma_load_2d(stages + lane * C::kStageBytes, &tmA, &full[lane], (kb0 + lane) * 128, e * nrows_e + cb * 128);
    }
  }
  if (!GATEUP && rank == 0 && warp == 1 && lane < p.K) {
    cwt[lane] = p.topk_w[tok * p.K + lane];
    cid[lane] = p.ids[tok * p.K + lane];
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  if (!GATEUP && warp == 0) {
    if (lane == 0) {
      const int e = *e_sh;
      if (e >= 0 && e < p.E)
        for (int i = 0; i < npre; ++i)
          tc::tma_load_2d(stages + i * C::kStageBytes + C::kABytes, &tmB, &full[i], (kb0 + i) * 128, pr);
    }
  } else if (warp == 0) {
    const int e = p.ids[pr];
    if (lane == 0) *e_sh = e;
    if (e >= 0 && e < p.E && lane < npre) {  // one lane per stage: the gate and up tiles
      unsigned char* st = stages + lane * C::kStageBytes;
      tc::mbar_arrive_expect_tx(&full[lane], C::kATiles * C::kATx);
      const int x = (kb0 + lane) * 128;
      tc::tma_load_2d(st, &tmA, &full[lane], x, e * nrows_e + cb * 128);
      tc::tma_load_2d(st + C::kABytes, &tmA, &full[lane], x, e * nrows_e + p.I + cb * 128);
    }
  } else if (GATEUP) {
    // warps 1..5 quantise the pair's hidden row for this CTA's K blocks: row 0 of the stage
    // B tiles for the first stages, the rest into bq
    for (int i = warp - 1; i < p.nkb_cta; i += kMxThreads / 32 - 1) {
      const uint2 raw = *reinterpret_cast<const uint2*>(p.hidden + (size_t)tok * p.H + (kb0 + i) * 128 + lane * 4);
      const float x0 = bf16_bits_to_float(raw.x & 0xFFFF), x1 = bf16_bits_to_float(raw.x >> 16);
      const float x2 = bf16_bits_to_float(raw.y & 0xFFFF), x3 = bf16_bits_to_float(raw.y >> 16);
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sc = quant_scale(amax);
      const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
      const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
      uint8_t* dst = i < nst ? stages + i * C::kStageBytes + C::kATiles * C::kABytes : bq + i * 128;
      reinterpret_cast<uint32_t*>(dst)[lane] = lo | (hi << 16);
      if (lane == 0) sas[i] = sc;
      if (p.qa_out != nullptr && cb == 0 && pr % p.K == 0) {
        reinterpret_cast<uint32_t*>(p.qa_out + (size_t)tok * p.H + (kb0 + i) * 128)[lane] = lo | (hi << 16);
        if (lane == 0) p.sa_out[(size_t)tok * p.nkb + kb0 + i] = sc;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else {
    for (int i = threadIdx.x - 32; i < p.nkb_cta; i += kMxThreads - 32)
      sas[i] = p.a_scale[(size_t)pr * p.nkb + kb0 + i];
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const int e = *e_sh;
  const bool valid = e >= 0 && e < p.E;
  if (GATEUP && !valid && cb == 0 && rank == 0 && threadIdx.x == 0) set_status(p.hdr, MOE_STATUS_BAD_EXPERT_ID);
  const uint32_t tmem = *tmem_slot;
  if (GATEUP && !valid) {  // the whole cluster shares the unit and leaves together
    if (warp == 1) tc::tmem_dealloc(tmem, C::kTmemCols);
    return;
  }

  bool ok = true;
  float chain0 = 0.0f, chain1 = 0.0f;
  float term0[kMaxSplitTerms], term1[kMaxSplitTerms];
  if (valid && warp == 0) {
    int issued = npre;
    for (int i = npre; i < p.nkb_cta; ++i) {
      const int s = i % nst;
      const uint32_t ph = (i / nst) & 1;
      bool w_ok = true;
      if (lane == 0) w_ok = tc::mbar_wait(&empty[s], ph ^ 1);
      if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) { ok = false; break; }
      unsigned char* st = stages + s * C::kStageBytes;
      if (GATEUP) {
        if (lane < 8)
          reinterpret_cast<uint4*>(st + C::kATiles * C::kABytes)[lane] = reinterpret_cast<const uint4*>(bq + i * 128)[lane];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      if (lane == 0) {
        const int x = (kb0 + i) * 128;
        tc::mbar_arrive_expect_tx(&full[s], GATEUP ? C::kATiles * C::kATx : C::kATx + C::kBBytes);
        tc::tma_load_2d(st, &tmA, &full[s], x, e * nrows_e + cb * 128);
        if (GATEUP) tc::tma_load_2d(st + C::kABytes, &tmA, &full[s], x, e * nrows_e + p.I + cb * 128);
        if (!GATEUP) tc::tma_load_2d(st + C::kABytes, &tmB, &full[s], x, pr);
      }
      issued = i + 1;
    }
    // no load is still writing when the CTA leaves (a no-op unless a wait gave up)
    if (lane == 0)
      for (int i = issued - 1; i >= 0 && i >= issued - nst; --i)
        if (!tc::mbar_wait(&full[i % nst], (i / nst) & 1)) ok = false;
  } else if (valid && warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e2m1_e4m3(128, kPairN);
      for (int i = 0; i < p.nkb_cta; ++i) {
        const int s = i % nst;
        const uint32_t ph = (i / nst) & 1;
        const int buf = i & 1;
        if (!tc::mbar_wait(&full[s], ph)) { ok = false; break; }
        if (!tc::mbar_wait(&acce[buf], ((i >> 1) & 1) ^ 1)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t sa = tc::smem_u32(stages + s * C::kStageBytes);
        const uint64_t da0 = tc::sdesc_sw128(sa);
        const uint64_t da1 = tc::sdesc_sw128(sa + C::kABytes);
        const uint64_t db = tc::sdesc_sw128(sa + C::kATiles * C::kABytes);
        const uint32_t d = tmem + buf * C::kAccCols;
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // one 32-wide sub-block per MMA, each into its own sums
          tc::mma_e4m3(d + j * kPairN, da0 + 2 * j, db + 2 * j, idesc, 0);
          if (GATEUP) tc::mma_e4m3(d + 64 + j * kPairN, da1 + 2 * j, db + 2 * j, idesc, 0);
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&accf[buf]);
      }
      // every arrival the MMAs owe this CTA's barriers has landed before the CTA can leave
      tc::mma_commit(drainb);
      if (!tc::mbar_wait(drainb, 0)) ok = false;
    }
  } else if (valid && warp >= 2) {
    // epilogue: thread <-> weight row (warp % 4) * 32 + lane of the 128-row tile; the row's
    // four scale bytes of K block i (one 32-bit load per tile) are loaded kAhead blocks early
    constexpr int kAhead = 4;
    const int q = warp & 3, r = q * 32 + lane;
    const int nsub = p.nkb * 4;
    const uint8_t* sc0 = p.wscale + ((size_t)e * nrows_e + cb * 128 + r) * nsub + kb0 * 4;  // gate (or down) row
    const uint8_t* sc1 = p.wscale + ((size_t)e * nrows_e + p.I + cb * 128 + r) * nsub + kb0 * 4;  // up row
    const int n = p.nkb_cta;
    uint32_t ea[kAhead], eb[kAhead];
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      ea[j] = j < n ? *reinterpret_cast<const uint32_t*>(sc0 + 4 * j) : 0u;
      eb[j] = (GATEUP && j < n) ? *reinterpret_cast<const uint32_t*>(sc1 + 4 * j) : 0u;
    }
    for (int i0 = 0; i0 < n && ok; i0 += kAhead) {
#pragma unroll
      for (int j = 0; j < kAhead; ++j) {
        const int i = i0 + j;
        if (i >= n || !ok) break;
        const uint32_t e0 = ea[j], e1 = eb[j];
        if (i + kAhead < n) {
          ea[j] = *reinterpret_cast<const uint32_t*>(sc0 + 4 * (i + kAhead));
          if (GATEUP) eb[j] = *reinterpret_cast<const uint32_t*>(sc1 + 4 * (i + kAhead));
        }
        const int buf = i & 1;
        if (!tc::mbar_wait(&accf[buf], (i >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * C::kAccCols;
        float v[8];
        if (GATEUP) {
          tmem_ld_sub8(ta, v);
        } else {
          float v4[4];
          tmem_ld_sub4(ta, v4);
#pragma unroll
          for (int k = 0; k < 4; ++k) v[k] = v4[k];
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[buf]);
        const float a = sas[i];
        const float t0 = __fmul_rn(mx_block_sum(v, e0), a);
        const float t1 = GATEUP ? __fmul_rn(mx_block_sum(v + 4, e1), a) : 0.0f;
        if (split == 1) {
          chain0 = __fadd_rn(chain0, t0);
          if (GATEUP) chain1 = __fadd_rn(chain1, t1);
        } else {
#pragma unroll
          for (int k = 0; k < kMaxSplitTerms; ++k)
            if (k == i) { term0[k] = t0; term1[k] = t1; }
        }
      }
    }
  }

  // ---- cross-CTA exchange (as in the FP8 pair kernels): terms or combine rows into CTA 0
  __syncwarp();
  if (clustered) {
    if (GATEUP) cluster.sync();
    else tc::cluster_wait();
    if (warp >= 2) {
      const int r = (warp & 3) * 32 + lane;
      if (!GATEUP) {
        cluster.map_shared_rank(comb, 0)[rank * 128 + r] = chain0;
      } else {
        float* x0 = cluster.map_shared_rank(xterm, 0);
#pragma unroll
        for (int j = 0; j < kMaxSplitTerms; ++j) {
          if (j < p.nkb_cta) {
            x0[(kb0 + j) * 128 + r] = term0[j];
            x0[(p.nkb + kb0 + j) * 128 + r] = term1[j];
          }
        }
      }
    }
    cluster.sync();
  } else if (!GATEUP && warp >= 2) {
    comb[(warp & 3) * 32 + lane] = chain0;
  }
  if (!ok) set_status(p.hdr, MOE_STATUS_WAIT_TIMEOUT);

  if (rank == 0 && warp >= 2) {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    float g = chain0, u = chain1;
    if (split > 1) {
      g = 0.0f;
      u = 0.0f;
      for (int kb = 0; kb < p.nkb; ++kb) {
        g = __fadd_rn(g, xterm[kb * 128 + r]);
        u = __fadd_rn(u, xterm[(p.nkb + kb) * 128 + r]);
      }
    }
    if (GATEUP) {
      const float act = silu_mul(g, u);
      float m = fabsf(act);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[q] = m;
      tc::named_bar(1, 128);
      const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
      const float s2 = quant_scale(amax);
      const uint16_t code = e4m3x2_encode(__fdiv_rn(act, s2), 0.0f);
      p.act_out[(size_t)pr * p.I + cb * 128 + r] = (uint8_t)(code & 0xFF);
      if (r == 0) p.act_scale_out[(size_t)pr * (p.I / 128) + cb] = s2;
    } else {
      float acc = 0.0f;
      for (int j = 0; j < p.K; ++j) {
        const int ej = cid[j];
        if (ej < 0 || ej >= p.E) continue;
        acc = __fadd_rn(acc, __fmul_rn(cwt[j], comb[j * 128 + r]));
      }
      p.out[(size_t)tok * p.H + cb * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------------------ host side
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
bool make_tmap_e2m1(CUtensorMap* m, const void* base, uint64_t codes, uint64_t rows);

namespace {

template <bool GATEUP>
void set_mx_attrs(const DeviceInfo& d) {
  static PerDeviceOnce once;
  once_per_device(once, [&] {
    cudaFuncSetAttribute(mx_pair_kernel<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
    cudaFuncSetAttribute(mx_pair_kernel<GATEUP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
}

template <bool GATEUP>
cudaError_t launch_mx(const CUtensorMap& tA, const CUtensorMap& tB, MxParams prm, int cluster_x, int64_t units,
                      cudaStream_t st) {
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  const PlanDevice dv{d.sms, d.smem_per_sm, d.smem_optin};
  const size_t smem = mx_request<GATEUP>(dv, prm.nst, prm.nkb_cta, prm.K);
  if (smem > d.smem_optin) return cudaErrorInvalidConfiguration;
  set_mx_attrs<GATEUP>(d);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_x, (unsigned)units, 1);
  cfg.blockDim = dim3(kMxThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mx_pair_kernel<GATEUP>, tA, tB, prm);
}

}  // namespace

// MXFP4 gate/up for R = M*K pairs, the hidden row quantised inside the kernel: act [R][I] and
// act_scale [R][I/128] in pair order (the K split and the stages from plan_mx).
cudaError_t launch_mx_gateup(const uint8_t* w13q, const uint8_t* w13s, const int32_t* ids, const uint16_t* hidden,
                             int M, int H, int I, int E, int K, const WsPtrs& ws, cudaStream_t st) {
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  CUtensorMap tA;
  if (!make_tmap_e2m1(&tA, w13q, (uint64_t)H, (uint64_t)E * 2 * I)) return cudaErrorInvalidValue;
  MxParams prm{};
  prm.H = H; prm.I = I; prm.K = K; prm.E = E;
  prm.nkb = H / 128;
  prm.ncb = I / 128;
  prm.ids = ids;
  prm.wscale = w13s;
  prm.hidden = hidden;
  prm.act_out = ws.act;
  prm.act_scale_out = ws.act_scale;
  prm.qa_out = ws.qa;
  prm.sa_out = ws.sa;
  prm.hdr = ws.hdr;
  const int64_t units = (int64_t)M * K * prm.ncb;
  const PairPlan pl = plan_mx<true>(PlanDevice{d.sms, d.smem_per_sm, d.smem_optin}, prm.nkb, units, K);
  prm.nkb_cta = prm.nkb / pl.split;
  prm.nst = pl.nst;
  return launch_mx<true>(tA, tA, prm, pl.split, units, st);  // B is written by the kernel
}

// MXFP4 down fused with the combine: a cluster of K CTAs (one per slot) per token and
// 128-column output block; out BF16 [M][H].
cudaError_t launch_mx_down_combine(const uint8_t* w2q, const uint8_t* w2s, const int32_t* ids, const float* topk_w,
                                   uint16_t* out, int M, int H, int I, int E, int K, const WsPtrs& ws,
                                   cudaStream_t st) {
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  CUtensorMap tA, tB;
  const int R = M * K;
  if (!make_tmap_e2m1(&tA, w2q, (uint64_t)I, (uint64_t)E * H)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tB, ws.act, (uint64_t)I, (uint64_t)R, kPairN)) return cudaErrorInvalidValue;
  MxParams prm{};
  prm.H = H; prm.I = I; prm.K = K; prm.E = E;
  prm.nkb = I / 128;
  prm.ncb = H / 128;
  prm.ids = ids;
  prm.wscale = w2s;
  prm.a_scale = ws.act_scale;
  prm.topk_w = topk_w;
  prm.out = out;
  prm.hdr = ws.hdr;
  prm.nkb_cta = prm.nkb;
  const int64_t units = (int64_t)M * prm.ncb;
  prm.nst = plan_mx<false>(PlanDevice{d.sms, d.smem_per_sm, d.smem_optin}, prm.nkb, units, K).nst;
  return launch_mx<false>(tA, tB, prm, K, units, st);
}

}  // namespace moe
