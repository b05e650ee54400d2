// pair_plan.h -- shapes, shared-memory layout and the launch planner of the few-row pair
// kernels (tc_pair.cu). Plain C++17: the CUDA build includes it, and a CPU test compiles
// it with a host compiler to check the planner at several device sizes.
//
// A pair unit is (routed pair, 128-row output block). Its K blocks may be split over a
// cluster of S CTAs; the planner picks S and the pipeline depth so that every CTA of the
// launch is resident at once, for the device it is given (SM count and shared memory per
// SM come from the device, never from constants).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <algorithm>

#ifndef __CUDACC__
#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#endif

namespace moe {

constexpr int kPairN = 16;  // B rows per MMA (row 0 is the unit's pair)
constexpr int kMaxSplitTerms = 8;  // K blocks per CTA when a unit's K blocks are split
constexpr int kPairThreads = 192;
constexpr int kMaxStages = 8;

enum PairMode { kGateUpWs = 0, kGateUpFused = 1, kDownY = 2, kDownCombine = 3 };

template <int MODE>
struct PairCfg {
  static constexpr bool kGateUp = MODE == kGateUpWs || MODE == kGateUpFused;
  static constexpr int kATiles = kGateUp ? 2 : 1;
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = kPairN * 128;
  static constexpr int kStageBytes = ((kATiles * kABytes + kBBytes + 1023) / 1024) * 1024;
  static constexpr uint32_t kTxA = kATiles * kABytes;
  static constexpr int kAccCols = kATiles * kPairN;  // one K block's accumulators
  static constexpr int kTmemCols = 2 * kAccCols < 32 ? 32 : 2 * kAccCols;
};

// Split-K terms [kATiles][nkb][128] f32 arrive in CTA 0's stage buffers once its own MMAs
// are complete (the planner keeps kATiles * nkb * 512 bytes within them); the combine rows
// [K][128] f32 have a region of their own.
template <int MODE>
struct PairSmem {
  size_t stages, bq, sas, sws, comb, cw, bars, total;
};

template <int MODE>
__host__ __device__ inline PairSmem<MODE> pair_smem(int nst, int nkb_cta, int K) {
  using C = PairCfg<MODE>;
  PairSmem<MODE> s{};
  size_t o = 0;
  s.stages = o; o += (size_t)nst * C::kStageBytes;
  s.bq = o;   o += MODE == kGateUpFused ? (size_t)nkb_cta * 128 : 0;  // hidden codes past the stages
  s.sas = o;  o += (size_t)nkb_cta * 4;                               // activation scales
  s.sws = o;  o += (size_t)C::kATiles * nkb_cta * 4;                  // weight scales
  o = (o + 15) & ~size_t(15);
  s.comb = o; o += MODE == kDownCombine ? (size_t)K * 512 : 0;        // combine rows
  s.cw = o;   o += MODE == kDownCombine ? 16 * 8 : 0;                 // combine weights + ids
  s.bars = o; o += 256;
  s.total = o + 1024;  // + alignment slack of the dynamic shared memory base
  return s;
}

struct PairPlan {
  int split, nst;
};

// The device a plan is made for.
struct PlanDevice {
  int sms;              // multiprocessors
  size_t smem_per_sm;   // shared memory per multiprocessor
  size_t smem_optin;    // largest dynamic shared memory per block
};

// CTAs of `smem` bytes resident at once in clusters of `cluster`: SMs x CTAs per SM, less a
// tenth for clusters that a GPC cannot place whole. Clusters of two or more CTAs at one CTA
// per SM are counted as not fitting (a GPC's SM count is not a multiple of the cluster).
inline int64_t resident_ctas(const PlanDevice& d, int cluster, size_t smem) {
  const int64_t per_sm = (int64_t)(d.smem_per_sm / (smem + 1024));
  if (per_sm == 0 || (cluster > 1 && per_sm < 2)) return 0;
  return cluster > 1 ? (int64_t)d.sms * per_sm * 9 / 10 : (int64_t)d.sms * per_sm;
}

// The largest K split S (a divisor of nkb, S <= 8) whose units * S CTAs are all resident at
// once, with the most pipeline stages (<= the CTA's K blocks, <= kMaxStages) that keep them
// resident; `fixed_cluster` (down fused with the combine) is the cluster size when the mode
// fixes it. When nothing fits one wave: no split, 2 stages for gate/up and 4 for down.
template <int MODE>
inline PairPlan plan_pair(const PlanDevice& d, int nkb, int64_t units, int K, bool allow_split,
                          int fixed_cluster = 0) {
  using C = PairCfg<MODE>;
  PairPlan best{1, std::min(nkb, C::kGateUp ? 2 : 4)};
  for (int s = 1; s <= (allow_split ? 8 : 1); ++s) {
    if (nkb % s) continue;
    const int per = nkb / s;
    if (s > 1 && per > kMaxSplitTerms) continue;
    const int cluster = fixed_cluster ? fixed_cluster : s;
    int chosen = 0;
    for (int n = std::min(per, kMaxStages); n >= std::min(per, 2); --n) {
      // split-K terms land in CTA 0's stage buffers
      if (s > 1 && (size_t)C::kATiles * nkb * 512 > (size_t)n * C::kStageBytes) break;
      const size_t smem = pair_smem<MODE>(n, per, K).total;
      if (smem > d.smem_optin) continue;
      if (units * cluster <= resident_ctas(d, cluster, smem)) {
        chosen = n;
        break;
      }
    }
    if (chosen) best = {s, chosen};
  }
  return best;
}

// ---- MXFP4 weights (mx_pair.cu): TMA expands each K block's packed E2M1 codes (64 bytes
// per weight row) into the tensor core's padded 4-bit layout (16 codes in the low half of
// each 16-byte chunk), so an operand tile has the FP8 tile's 128 x 128-byte footprint; one
// accumulator per 32-wide sub-block (four per K block and tile).
constexpr int kMxThreads = 192;  // TMA, MMA, 4 epilogue warps

template <bool GATEUP>
struct MxCfg {
  static constexpr int kATiles = GATEUP ? 2 : 1;
  static constexpr int kABytes = 128 * 128;  // one weight tile in shared memory (128-byte swizzle)
  static constexpr int kATx = 128 * 64;      // the bytes its load counts: the packed codes read
  static constexpr int kBBytes = kPairN * 128;
  static constexpr int kStageBytes = ((kATiles * kABytes + kBBytes + 1023) / 1024) * 1024;
  static constexpr int kAccCols = kATiles * 4 * kPairN;
  static constexpr int kTmemCols = 2 * kAccCols;
  static constexpr int kMaxCtasPerSm = 512 / kTmemCols;  // TMEM columns of one SM
};

struct MxSmem {
  size_t stages, bq, sas, comb, cw, bars, total;
};

template <bool GATEUP>
__host__ __device__ inline MxSmem mx_smem(int nst, int nkb_cta, int K) {
  using C = MxCfg<GATEUP>;
  MxSmem s{};
  size_t o = 0;
  s.stages = o; o += (size_t)nst * C::kStageBytes;
  s.bq = o;     o += GATEUP ? (size_t)nkb_cta * 128 : 0;  // hidden codes past the stages
  s.sas = o;    o += (size_t)nkb_cta * 4;                 // activation scales
  o = (o + 15) & ~size_t(15);
  s.comb = o;   o += GATEUP ? 0 : (size_t)K * 512;        // combine rows
  s.cw = o;     o += GATEUP ? 0 : 16 * 8;                 // combine weights + ids
  s.bars = o;   o += 512;
  s.total = o + 1024;
  return s;
}

// Dynamic shared memory a launch requests: the layout, raised so that no more CTAs of the
// launch share an SM than its TMEM columns hold.
template <bool GATEUP>
inline size_t mx_request(const PlanDevice& d, int nst, int nkb_cta, int K) {
  using C = MxCfg<GATEUP>;
  return std::max(mx_smem<GATEUP>(nst, nkb_cta, K).total, d.smem_per_sm / (C::kMaxCtasPerSm + 1) + 1);
}

// As plan_pair: gate/up may split its K blocks over a cluster (split-K terms land in CTA 0's
// stages); down is fused with the combine, a cluster of K CTAs with every K block each.
template <bool GATEUP>
inline PairPlan plan_mx(const PlanDevice& d, int nkb, int64_t units, int K) {
  using C = MxCfg<GATEUP>;
  PairPlan best{1, std::min(nkb, 2)};
  for (int s = 1; s <= (GATEUP ? 8 : 1); ++s) {
    if (nkb % s) continue;
    const int per = nkb / s;
    if (s > 1 && per > kMaxSplitTerms) continue;
    const int cluster = GATEUP ? s : K;
    int chosen = 0;
    for (int n = std::min(per, kMaxStages); n >= std::min(per, 2); --n) {
      if (s > 1 && (size_t)C::kATiles * nkb * 512 > (size_t)n * C::kStageBytes) break;
      const size_t smem = mx_request<GATEUP>(d, n, per, K);
      if (smem > d.smem_optin) continue;
      if (units * cluster <= resident_ctas(d, cluster, smem)) {
        chosen = n;
        break;
      }
    }
    if (chosen) best = {s, chosen};
  }
  return best;
}

}  // namespace moe
