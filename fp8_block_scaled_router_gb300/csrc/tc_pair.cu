// tc_pair.cu -- block-scaled expert GEMMs on tcgen05 for few routed rows (decode, verify,
// wide-expert sweeps): one unit per routed (token, slot) pair.
//
// Sources: docs/compiler/architecture.md, accepted M=1 MoE objects (gate/up, SiLU+quant,
// down/reduce; FP8 activation plus activation-scale intermediates); "NetraRuntime/
// netra-kernel" older lab README, supported-targets table (FP8 E4M3 weights with 128x128
// FP32 block scales); netra-kernel README, prefill-pair section (a route reducer with its
// own fixed reduction order); "Inferact/amd-kernels" README (split-K and expert partials
// summed in a fixed order -- by the last CTA or inside the next kernel -- never with
// atomics).
//
// Shape of the work. A unit is (pair p, 128-row block of the output). The 128 weight rows
// are the MMA's M operand; the pair's FP8 activation row is the first of N=16 B rows (the
// other rows are zero or neighbours' rows and are ignored), so D = W_tile * x^T lands in
// TMEM with one weight row per lane. Each CTA streams its 128-wide K blocks with TMA
// (128-byte swizzle) through a ring of stages, issues four 128x16x32 FP8 MMAs per block
// into a fresh accumulator (double-buffered in TMEM), and its epilogue warps read the block
// sum P back with tcgen05.ld and form the promoted term t_kb = P * (sa_kb * sw_kb). The
// promotion chain acc = acc + t_kb runs over kb ascending in FP32 from 0 -- in registers
// when one CTA owns all K blocks, otherwise CTA 0 of the cluster runs it over every CTA's
// terms.
//
// Latency plan (one dependent chain per launch, so every step is taken as early as it can
// be): warp 0 loads the expert id and issues the TMA loads of the first stages straight
// after the grid dependency resolves, while the other warps quantise the hidden row (or load
// the activation scales) and stage the weight scales. The split-K terms and the combine
// rows cross the cluster as plain distributed-shared-memory stores between hardware cluster
// barriers (measured faster here than point-to-point mbarrier signalling between CTAs).
//
// Modes:
//   kGateUpWs     gate/up, B rows from the prepared hidden codes in the workspace (TMA)
//   kGateUpFused  gate/up, each CTA quantises its pair's hidden row for its own K blocks
//                 (scale = amax/448 per 128 columns, RNE saturating E4M3) into the B tile
//   kDownY        down, y[p][cb*128 + r] in FP32 to the workspace
//   kDownCombine  down fused with the combine: a cluster of K CTAs computes the K pairs of
//                 one token for one 128-column block; CTA 0 adds w_j * y_j over j
//                 ascending (FP32 multiply then add, from 0) and writes BF16 out.
// gate/up epilogue: act = silu(g) * u per row, block amax over the 128 rows (warp max +
// shared memory), scale = amax/448, RNE saturating E4M3 codes into act [p][I] and the
// scale into act_scale [p][I/128]. A gate/up launch may also be given the down weights:
// each CTA then prefetches its share of its expert's w2 block into L2, so the down launch
// reads them from L2.
// Warp roles: warp 0 feeds the stages (TMA), warp 1 owns TMEM and issues MMAs, warps 2..5
// are the epilogue (TMEM lane quadrant = warp % 4). Every kernel waits on the previous
// kernel of the stream (griddepcontrol.wait) before touching global memory and then
// releases its dependents, so consecutive launches overlap their launch latency.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "device.h"
#include "pair_plan.h"
#include "launch.h"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace moe {

struct PairParams {
  int H, I, K, E;
  int nkb, nkb_cta, ncb;   // K blocks total / per CTA; 128-row output blocks per unit
  int nst;                 // pipeline stages (<= kMaxStages)
  const int32_t* ids;      // [R] expert of each pair (raw top-k ids or the workspace copy)
  const float* w_scale;    // s13 [E][2I/128][H/128] or s2w [E][H/128][I/128]
  const float* a_scale;    // sa [M][H/128] (kGateUpWs) or act_scale [R][I/128] (down)
  const uint16_t* hidden;  // BF16 [M][H] (kGateUpFused)
  const float* topk_w;     // [R] (kDownCombine)
  uint16_t* out;           // BF16 [M][H] (kDownCombine)
  uint8_t* act_out;        // [R][I]
  float* act_scale_out;    // [R][I/128]
  float* y_out;            // [R][H]
  Header* hdr;
  const uint8_t* pf_w2;    // gate/up: w2 [E][H][I] to prefetch into L2, or null
  const float* pf_s2;      // gate/up: its scales [E][H/128][I/128]
  uint8_t* qa_out;         // kGateUpFused: the hidden codes it quantised [M][H] (slot 0's
  float* sa_out;           //   CTAs of the first output block write them), scales [M][H/128]
  Norm nm;                 // kGateUpFused: RMSNorm in front (gamma null: none)
};

template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 3)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const PairParams p) {
  using C = PairCfg<MODE>;
  constexpr bool kGateUp = C::kGateUp;
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int nst = p.nst;
  const PairSmem<MODE> SL = pair_smem<MODE>(nst, p.nkb_cta, p.K);
  unsigned char* stages = base + SL.stages;
  float* xterm = reinterpret_cast<float*>(stages);  // split-K terms, after CTA 0's MMAs
  uint8_t* bq = base + SL.bq;
  float* sas = reinterpret_cast<float*>(base + SL.sas);
  float* sws = reinterpret_cast<float*>(base + SL.sws);
  float* comb = reinterpret_cast<float*>(base + SL.comb);
  float* cwt = reinterpret_cast<float*>(base + SL.cw);  // [16] combine weights
  int* cid = reinterpret_cast<int*>(cwt + 16);           // [16] their expert ids
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + SL.bars);
  uint64_t* full = bars;                      // [kMaxStages]
  uint64_t* empty = bars + kMaxStages;        // [kMaxStages]
  uint64_t* accf = bars + 2 * kMaxStages;     // [2]
  uint64_t* acce = accf + 2;                  // [2]
  uint64_t* drainb = acce + 2;                // every MMA this CTA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drainb + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 1);  // [4] warp maxima
  int* e_sh = reinterpret_cast<int*>(red + 4);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int S = (int)cluster.num_blocks();
  const bool clustered = S > 1;
  const int split = MODE == kDownCombine ? 1 : S;  // CTAs sharing one unit's K blocks
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // set-up that touches no global memory overlaps the previous kernel's tail
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    if (MODE != kGateUpFused) tc::prefetch_tmap(&tmB);
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
  if (MODE == kGateUpFused) {  // B tile rows 1..15 stay zero (row 0, the first 128 bytes, is the quantisers')
    for (int i = threadIdx.x; i < nst * (C::kBBytes / 16 - 8); i += kPairThreads) {
      const int s = i / (C::kBBytes / 16 - 8), c = 8 + i % (C::kBBytes / 16 - 8);
      reinterpret_cast<uint4*>(stages + s * C::kStageBytes + C::kTxA)[c] = make_uint4(0, 0, 0, 0);
    }
  }
  const int unit = blockIdx.y;
  int pr, cb, tok;
  if (MODE == kDownCombine) {
    tok = unit / p.ncb;
    cb = unit % p.ncb;
    pr = tok * p.K + rank;
  } else {
    pr = unit / p.ncb;
    cb = unit % p.ncb;
    tok = pr / p.K;
  }
  const int kb0 = MODE == kDownCombine ? 0 : rank * p.nkb_cta;
  const int brow = MODE == kGateUpWs ? tok : pr;  // B row (qa row or act row)
  const int npre = min(nst, p.nkb_cta);           // stages issued before the block barrier
  // Down fused with the combine runs right after the gate/up launch, which itself waited
  // for whatever wrote the top-k ids and weights: those, and the down weights, are complete
  // before this grid can start, so the weight tiles stream in while gate/up finishes; only
  // the activation rows (gate/up's output) wait for the grid dependency.
  constexpr bool kEarly = MODE == kDownCombine;
  if (kEarly && warp == 0) {
    // one lane per stage issues its load: several issuers keep more of a CTA's tiles moving
    const int e = p.ids[pr];
    if (lane == 0) *e_sh = e;
    if (e >= 0 && e < p.E && lane < npre) {
      tc::mbar_arrive_expect_tx(&full[lane], C::kTxA + C::kBBytes);
      tc::tma_load_2d(stages + lane * C::kStageBytes, &tmA, &full[lane], (kb0 + lane) * 128, e * p.H + cb * 128);
    }
  }
  if (kEarly && rank == 0 && warp == 1 && lane < p.K) {
    cwt[lane] = p.topk_w[tok * p.K + lane];
    cid[lane] = p.ids[tok * p.K + lane];
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  if (kEarly && warp == 0) {
    if (lane == 0) {
      const int e = *e_sh;
      if (e >= 0 && e < p.E)
        for (int i = 0; i < npre; ++i)
          tc::tma_load_2d(stages + i * C::kStageBytes + C::kTxA, &tmB, &full[i], (kb0 + i) * 128, brow);
    }
  } else if (warp == 0) {
    // the expert id, then the first stages' loads: the first bytes are in flight before the
    // rest of the prologue runs
    const int e = p.ids[pr];
    if (lane == 0) *e_sh = e;
    if (e >= 0 && e < p.E && lane < npre) {  // one lane per stage issues its loads
      const int i = lane;
      const int ya = kGateUp ? e * 2 * p.I + cb * 128 : e * p.H + cb * 128;
      const int yb = e * 2 * p.I + p.I + cb * 128;
      unsigned char* st = stages + i * C::kStageBytes;
      const int x = (kb0 + i) * 128;
      tc::mbar_arrive_expect_tx(&full[i], MODE == kGateUpFused ? C::kTxA : C::kTxA + C::kBBytes);
      tc::tma_load_2d(st, &tmA, &full[i], x, ya);
      if (kGateUp) tc::tma_load_2d(st + C::kABytes, &tmA, &full[i], x, yb);
      if (MODE != kGateUpFused) tc::tma_load_2d(st + C::kTxA, &tmB, &full[i], x, brow);
    }
  } else if (MODE == kGateUpFused) {
    // warps 1..5 quantise the pair's hidden row for this CTA's K blocks straight into the
    // stage B tiles (row 0; unswizzled in the first 8-row group), the rest into bq. With an
    // RMSNorm in front each of these warps first forms the row's r itself (the whole row,
    // from L2) and quantises y = bf16((x*r)*gamma).
    const bool normed = p.nm.gamma != nullptr;
    const float r = normed ? row_rms_scale(p.hidden + (size_t)tok * p.H, p.H, p.nm.eps, lane) : 0.0f;
    for (int i = warp - 1; i < p.nkb_cta; i += kPairThreads / 32 - 1) {
      const uint2 raw = *reinterpret_cast<const uint2*>(p.hidden + (size_t)tok * p.H + (kb0 + i) * 128 + lane * 4);
      float x0 = bf16_bits_to_float(raw.x & 0xFFFF), x1 = bf16_bits_to_float(raw.x >> 16);
      float x2 = bf16_bits_to_float(raw.y & 0xFFFF), x3 = bf16_bits_to_float(raw.y >> 16);
      if (normed) {
        const uint2 g = *reinterpret_cast<const uint2*>(p.nm.gamma + (kb0 + i) * 128 + lane * 4);
        x0 = norm_value(raw.x & 0xFFFF, r, g.x & 0xFFFF);
        x1 = norm_value(raw.x >> 16, r, g.x >> 16);
        x2 = norm_value(raw.y & 0xFFFF, r, g.y & 0xFFFF);
        x3 = norm_value(raw.y >> 16, r, g.y >> 16);
      }
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sc = quant_scale(amax);
      const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
      const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
      uint8_t* dst = i < nst ? stages + i * C::kStageBytes + C::kTxA : bq + i * 128;
      reinterpret_cast<uint32_t*>(dst)[lane] = lo | (hi << 16);
      if (lane == 0) sas[i] = sc;
      if (p.qa_out != nullptr && cb == 0 && pr % p.K == 0) {  // one copy of the token's codes (view)
        reinterpret_cast<uint32_t*>(p.qa_out + (size_t)tok * p.H + (kb0 + i) * 128)[lane] = lo | (hi << 16);
        if (lane == 0) p.sa_out[(size_t)tok * p.nkb + kb0 + i] = sc;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else {
    for (int i = threadIdx.x - 32; i < p.nkb_cta; i += kPairThreads - 32)
      sas[i] = p.a_scale[(size_t)brow * p.nkb + kb0 + i];
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const int e = *e_sh;
  const bool valid = e >= 0 && e < p.E;
  if (MODE == kGateUpFused && !valid && cb == 0 && rank == 0 && threadIdx.x == 0)
    set_status(p.hdr, MOE_STATUS_BAD_EXPERT_ID);
  const uint32_t tmem = *tmem_slot;
  // a skipped pair (not kDownCombine): the whole cluster shares the unit and leaves together
  if (MODE != kDownCombine && !valid) {
    if (warp == 1) tc::tmem_dealloc(tmem, C::kTmemCols);
    return;
  }

  bool ok = true;
  float chain0 = 0.0f, chain1 = 0.0f;
  float term0[kMaxSplitTerms], term1[kMaxSplitTerms];
  if (valid && warp == 0) {
    int issued = npre;  // stages with loads issued (the first npre in the prologue)
    const int ya = kGateUp ? e * 2 * p.I + cb * 128 : e * p.H + cb * 128;
    const int yb = e * 2 * p.I + p.I + cb * 128;
    for (int i = npre; i < p.nkb_cta; ++i) {
      const int s = i % nst;
      const uint32_t ph = (i / nst) & 1;
      bool w_ok = true;
      if (lane == 0) w_ok = tc::mbar_wait(&empty[s], ph ^ 1);
      if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) { ok = false; break; }
      unsigned char* st = stages + s * C::kStageBytes;
      if (MODE == kGateUpFused) {
        if (lane < 8)
          reinterpret_cast<uint4*>(st + C::kTxA)[lane] = reinterpret_cast<const uint4*>(bq + i * 128)[lane];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      if (lane == 0) {
        const int x = (kb0 + i) * 128;
        tc::mbar_arrive_expect_tx(&full[s], MODE == kGateUpFused ? C::kTxA : C::kTxA + C::kBBytes);
        tc::tma_load_2d(st, &tmA, &full[s], x, ya);
        if (kGateUp) tc::tma_load_2d(st + C::kABytes, &tmA, &full[s], x, yb);
        if (MODE != kGateUpFused) tc::tma_load_2d(st + C::kTxA, &tmB, &full[s], x, brow);
      }
      issued = i + 1;
    }
    // no load is still writing when the CTA leaves: the last load issued into each stage has
    // landed (a no-op unless a wait gave up)
    if (lane == 0)
      for (int i = issued - 1; i >= 0 && i >= issued - nst; --i)
        if (!tc::mbar_wait(&full[i % nst], (i / nst) & 1)) ok = false;
  } else if (valid && warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3(128, kPairN);
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
        const uint64_t db = tc::sdesc_sw128(sa + C::kTxA);
        const uint32_t d = tmem + buf * C::kAccCols;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tc::mma_e4m3(d, da0 + 2 * k, db + 2 * k, idesc, k > 0);
          if (kGateUp) tc::mma_e4m3(d + kPairN, da1 + 2 * k, db + 2 * k, idesc, k > 0);
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&accf[buf]);
      }
      // every arrival the MMAs owe this CTA's barriers has landed before the CTA can leave
      tc::mma_commit(drainb);
      if (!tc::mbar_wait(drainb, 0)) ok = false;
      if (kGateUp && ok && p.pf_w2 != nullptr) {
        // every weight byte of this CTA has landed: spend the idle memory time of the
        // epilogue on this CTA's share of the expert's down weights (and, once per pair,
        // their scales)
        const size_t wbytes = (size_t)p.H * p.I;
        const int parts = p.ncb * S, part = cb * S + rank;
        const size_t chunk = ((wbytes + parts - 1) / parts + 15) & ~size_t(15);
        const size_t off = (size_t)part * chunk;
        if (off < wbytes)
          tc::prefetch_l2_bulk(p.pf_w2 + (size_t)e * wbytes + off, (uint32_t)min(chunk, wbytes - off));
        if (part == 0) {
          const size_t sb = (size_t)(p.H / 128) * (p.I / 128) * 4;
          const char* s0 = reinterpret_cast<const char*>(p.pf_s2) + (size_t)e * sb;
          for (size_t o = 0; o < sb; o += 128) tc::prefetch_l2_line(s0 + o);
        }
      }
    }
  } else if (valid) {
    // epilogue: thread <-> weight row (warp % 4) * 32 + lane of the 128-row tile; the
    // block's weight scales are staged first, while the loads are in flight
    const int q = warp & 3;
    {
      const float* sw0 = p.w_scale + ((size_t)e * (kGateUp ? 2 * p.I / 128 : p.H / 128) + cb) * p.nkb;
      const float* sw1 = p.w_scale + ((size_t)e * (2 * p.I / 128) + p.I / 128 + cb) * p.nkb;
      for (int i = threadIdx.x - 64; i < p.nkb_cta; i += 128) {
        sws[i] = sw0[kb0 + i];
        if (kGateUp) sws[p.nkb_cta + i] = sw1[kb0 + i];
      }
      tc::named_bar(1, 128);
    }
    for (int i = 0; i < p.nkb_cta; ++i) {
      const int buf = i & 1;
      if (!tc::mbar_wait(&accf[buf], (i >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * C::kAccCols;
      float v0[16], v1[16];
      tc::tmem_ld16x2(ta, kGateUp ? ta + kPairN : ta, v0, v1);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acce[buf]);
      const float a = sas[i];
      const float t0 = __fmul_rn(v0[0], __fmul_rn(a, sws[i]));
      const float t1 = kGateUp ? __fmul_rn(v1[0], __fmul_rn(a, sws[p.nkb_cta + i])) : 0.0f;
      if (split == 1) {  // the whole chain is local: kb ascending
        chain0 = __fadd_rn(chain0, t0);
        if (kGateUp) chain1 = __fadd_rn(chain1, t1);
      } else {           // kept until CTA 0's stage buffers are free (<= kMaxSplitTerms)
#pragma unroll
        for (int j = 0; j < kMaxSplitTerms; ++j)
          if (j == i) { term0[j] = t0; term1[j] = t1; }
      }
    }
  }

  // ---- cross-CTA exchange: every CTA stores its terms (or its combine row) into CTA 0's
  // shared memory between two cluster barriers -- the first one guarantees that CTA 0's own
  // MMAs, and with them every read of its stage buffers, are complete
  if (clustered) {
    if (MODE != kDownCombine) cluster.sync();
    if (warp >= 2) {
      const int r = (warp & 3) * 32 + lane;
      if (MODE == kDownCombine) {
        cluster.map_shared_rank(comb, 0)[rank * 128 + r] = chain0;
      } else {
        float* x0 = cluster.map_shared_rank(xterm, 0);
#pragma unroll
        for (int j = 0; j < kMaxSplitTerms; ++j) {
          if (j < p.nkb_cta) {
            x0[(kb0 + j) * 128 + r] = term0[j];
            if (kGateUp) x0[(p.nkb + kb0 + j) * 128 + r] = term1[j];
          }
        }
      }
    }
    cluster.sync();
  } else if (MODE == kDownCombine && warp >= 2) {
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
        if (kGateUp) u = __fadd_rn(u, xterm[(p.nkb + kb) * 128 + r]);
      }
    }
    if (kGateUp) {
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
    } else if (MODE == kDownY) {
      p.y_out[(size_t)pr * p.H + cb * 128 + r] = g;
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
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

// 2-D u8 tensor [rows][inner] (row stride = inner bytes), box = 128 bytes x box_rows,
// 128-byte swizzle, out-of-range rows read as zero.
// Tensor maps depend only on (base, inner, rows, box_rows): the last few encodings of each
// host thread are kept, so a call sequence that reuses its weights and workspace encodes
// them once (the encode is a driver call on the launch path).
namespace {
struct TmapEntry {
  const void* base;
  uint64_t inner, rows;
  uint32_t box_rows;
  CUtensorMap map;
};
constexpr int kTmapCache = 32;
thread_local TmapEntry g_tmap_cache[kTmapCache];
thread_local int g_tmap_used = 0, g_tmap_next = 0;
}  // namespace

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  for (int i = 0; i < g_tmap_used; ++i) {
    const TmapEntry& c = g_tmap_cache[i];
    if (c.base == base && c.inner == inner && c.rows == rows && c.box_rows == box_rows) {
      *m = c.map;
      return true;
    }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  TmapEntry& c = g_tmap_cache[g_tmap_next];
  c = TmapEntry{base, inner, rows, box_rows, *m};
  g_tmap_next = (g_tmap_next + 1) % kTmapCache;
  if (g_tmap_used < kTmapCache) ++g_tmap_used;
  return true;
}

// 2-D tensor of packed 4-bit codes [rows][codes] (two per byte, row stride codes / 2 bytes),
// box 128 codes x 128 rows, written to shared memory in the tensor core's padded 4-bit layout
// (the 8 bytes of each 16 codes in the low half of a 16-byte chunk) with the 128-byte swizzle:
// a box occupies 128 x 128 bytes, like an FP8 tile. Needs a 32-byte aligned base, codes a
// multiple of 128 and a row stride that is a multiple of 32 bytes.
bool make_tmap_e2m1(CUtensorMap* m, const void* base, uint64_t codes, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {codes, rows};
  cuuint64_t strides[1] = {codes / 2};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D FP32 tensor [rows][inner] (row stride inner * 4 bytes), box box_inner x box_rows
// elements, no swizzle (for stores of row-major shared-memory tiles).
bool make_tmap_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                   uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D u8 tensor [d2][d1][d0] (strides s1, s2 bytes), box 128 bytes x b1 x b2, 128-byte
// swizzle; the box lands in shared memory as b2 blocks of b1 rows.
bool make_tmap_u8_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                     uint64_t s2, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {128, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int MODE>
void set_pair_attrs(const DeviceInfo& d) {
  static PerDeviceOnce once;
  once_per_device(once, [&] {
    cudaFuncSetAttribute(pair_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
    cudaFuncSetAttribute(pair_gemm_kernel<MODE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
}

PlanDevice plan_device(const DeviceInfo& d) { return PlanDevice{d.sms, d.smem_per_sm, d.smem_optin}; }

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& tA, const CUtensorMap& tB, PairParams prm, int cluster_x,
                        int64_t units, cudaStream_t st) {
  const PairSmem<MODE> SL = pair_smem<MODE>(prm.nst, prm.nkb_cta, prm.K);
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  if (SL.total > d.smem_optin) return cudaErrorInvalidConfiguration;
  set_pair_attrs<MODE>(d);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_x, (unsigned)units, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = SL.total;
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
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<MODE>, tA, tB, prm);
}

PairParams base_params(int M, int H, int I, int E, int K, const WsPtrs& ws) {
  PairParams prm{};
  prm.H = H; prm.I = I; prm.K = K; prm.E = E;
  prm.act_out = ws.act; prm.act_scale_out = ws.act_scale; prm.y_out = ws.y; prm.hdr = ws.hdr;
  (void)M;
  return prm;
}

}  // namespace

// gate/up for R = M*K pairs: act [R][I] + act_scale [R][I/128] in pair order. fused: the
// hidden row is quantised inside the kernel (ids = raw top-k ids); otherwise B comes from
// the prepared codes ws.qa / ws.sa and ids = ws.pair_expert. w2 / s2w (optional): the down
// weights the next launch will read; each routed expert's block is prefetched into L2.
cudaError_t launch_pair_gateup(const uint8_t* w13, const float* s13, const int32_t* ids,
                               const uint16_t* hidden, int M, int H, int I, int E, int K,
                               const WsPtrs& ws, cudaStream_t st, const uint8_t* w2, const float* s2w, Norm nm) {
  CUtensorMap tA, tB;
  if (!make_tmap_u8(&tA, w13, (uint64_t)H, (uint64_t)E * 2 * I, 128)) return cudaErrorInvalidValue;
  PairParams prm = base_params(M, H, I, E, K, ws);
  prm.nkb = H / 128;
  prm.ncb = I / 128;
  prm.ids = ids;
  prm.w_scale = s13;
  prm.a_scale = ws.sa;
  prm.hidden = hidden;
  prm.pf_w2 = w2;
  prm.pf_s2 = s2w;
  prm.nm = nm;
  const int64_t units = (int64_t)M * K * prm.ncb;
  prm.qa_out = ws.qa;
  prm.sa_out = ws.sa;
  const PlanDevice dv = plan_device(device_info());
  const PairPlan pl = hidden ? plan_pair<kGateUpFused>(dv, prm.nkb, units, K, true)
                             : plan_pair<kGateUpWs>(dv, prm.nkb, units, K, true);
  prm.nkb_cta = prm.nkb / pl.split;
  prm.nst = pl.nst;
  if (hidden) {
    tB = tA;  // unused: the B tile is written by the kernel
    return launch_pair<kGateUpFused>(tA, tB, prm, pl.split, units, st);
  }
  if (!make_tmap_u8(&tB, ws.qa, (uint64_t)H, (uint64_t)M, kPairN)) return cudaErrorInvalidValue;
  return launch_pair<kGateUpWs>(tA, tB, prm, pl.split, units, st);
}

// down for R pairs. combine: fused with the top-k combine into out (cluster of K CTAs per
// token and 128-column block); otherwise y [R][H] in pair order.
cudaError_t launch_pair_down(const uint8_t* w2, const float* s2w, const int32_t* ids, const float* topk_w,
                             uint16_t* out, int M, int H, int I, int E, int K, const WsPtrs& ws,
                             cudaStream_t st) {
  CUtensorMap tA, tB;
  const int R = M * K;
  if (!make_tmap_u8(&tA, w2, (uint64_t)I, (uint64_t)E * H, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tB, ws.act, (uint64_t)I, (uint64_t)R, kPairN)) return cudaErrorInvalidValue;
  PairParams prm = base_params(M, H, I, E, K, ws);
  prm.nkb = I / 128;
  prm.ncb = H / 128;
  prm.ids = ids;
  prm.w_scale = s2w;
  prm.a_scale = ws.act_scale;
  if (out) {
    prm.topk_w = topk_w;
    prm.out = out;
    prm.nkb_cta = prm.nkb;
    prm.nst = plan_pair<kDownCombine>(plan_device(device_info()), prm.nkb, (int64_t)M * prm.ncb, K, false, K).nst;
    return launch_pair<kDownCombine>(tA, tB, prm, K, (int64_t)M * prm.ncb, st);
  }
  const int64_t units = (int64_t)R * prm.ncb;
  const PairPlan pl = plan_pair<kDownY>(plan_device(device_info()), prm.nkb, units, K, true);
  prm.nkb_cta = prm.nkb / pl.split;
  prm.nst = pl.nst;
  return launch_pair<kDownY>(tA, tB, prm, pl.split, units, st);
}

}  // namespace moe
