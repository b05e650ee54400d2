// gpair.cu -- expert-grouped pair GEMMs on tcgen05 for tens to a few hundred routed rows:
// each expert's weights stream once for all the rows routed to it.
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (a producer whose
// gate/up, SiLU and quantisation and down-partial stages are followed by a separate route
// reducer with its own reduction order); "Inferact/amd-kernels" README (the token count is a
// runtime argument of the wide-expert MoE kernels; expert partials summed in a fixed order,
// never with atomics); older kernel-lab README, supported targets (FP8 E4M3 weights with
// 128x128 FP32 block scales; MXFP4).
//
// Shape of the work. After the counting sort (prep.cu) the routed rows sit in expert order
// and the sort's group list cuts each expert's rows into groups of up to 16. A unit is
// (group, 128-row block of the output): the 128 weight rows are the MMA's M operand and the
// group's rows its N = 16 operand (rows past the group's end are computed and ignored), so
// D = W_tile * X^T lands in TMEM with one weight row per lane and one routed row per column.
// The weights of an expert with n routed rows are read ceil(n / 16) times instead of n times
// (the pair kernels) or once per 128 rows with most of a 128-row tile empty (the grouped
// GEMM). Per 128-wide K block, per routed row b:
//   FP8 weights    term = P_kb[b] * (sa[b][kb] * sw_kb)
//   MXFP4 weights  T = sum over the four 32-wide sub-blocks s ascending of P_s[b] * 2^(e_s - 127)
//                  (FP32 from 0), term = T * sa[b][kb]
// and the chain acc[b] = acc[b] + term over kb ascending from 0 -- the pair kernels'
// arithmetic, so each routed row's result is theirs. gate/up then forms act = silu(g) * u and
// requantises each routed row's 128 values (scale = amax/448, the max over the unit's 128
// weight rows) into act / act_scale at the row's sorted position; down writes y in FP32 at
// the sorted position, and the slot-order combine (combine.cu) reduces it.
// Warp roles: 0 TMA (weight tiles and the group's 16 B rows), 1 TMEM + MMA, 2-5 epilogue (TMEM
// lane quadrant = warp % 4). MXFP4 weight tiles are written by TMA in the tensor core's
// padded 4-bit layout (kind::f8f6f4, A = E2M1), one accumulator per 32-wide sub-block.
// Every wait is bounded and reports MOE_STATUS_WAIT_TIMEOUT. The kernels are persistent (three
// CTAs per SM, two for the MXFP4 gate/up) and deal the (group, output block) items
// round-robin, so the load stays even for any group count the sort produces.
#include <cudaTypedefs.h>

#include <algorithm>

#include "device.h"
#include "launch.h"
#include "pair_plan.h"
#include "tc.cuh"

namespace moe {

constexpr int kGpThreads = 192;

template <bool MX, bool GATEUP>
struct GpCfg {
  static constexpr int kATiles = GATEUP ? 2 : 1;
  static constexpr int kABytes = 128 * 128;
  static constexpr int kATx = MX ? 128 * 64 : 128 * 128;  // bytes a weight tile's load reads
  static constexpr int kBBytes = kGroupRows * 128;
  static constexpr int kStageBytes = ((kATiles * kABytes + kBBytes + 1023) / 1024) * 1024;
  static constexpr int kSubs = MX ? 4 : 1;                 // accumulators per K block and tile
  static constexpr int kAccCols = kATiles * kSubs * kGroupRows;
  static constexpr int kTmemCols = 2 * kAccCols < 32 ? 32 : 2 * kAccCols;
  static constexpr int kMaxCtasPerSm = 512 / kTmemCols;
  // CTAs per SM the launch plans for (and the register budget it is compiled to): three,
  // except for the MXFP4 gate/up, whose 256 TMEM columns allow two
  static constexpr int kCtasPerSm = kMaxCtasPerSm >= 3 ? 3 : 2;
};

struct GpParams {
  int H, I, E;
  int nkb, ncb, nst;
  int sms;                // multiprocessors of the device
  const Tile* groups;
  const Header* hdr_ro;
  const void* w_scale;    // FP8: FP32 [E][N/128][Kd/128]; MXFP4: UE8M0 [E][N][Kd/32]
  const float* a_scale;   // gate/up: sa_p [R][H/128]; down: act_scale [R][I/128] (sorted rows)
  uint8_t* act_out;       // gate/up: [R][I]
  float* act_scale_out;   // gate/up: [R][I/128]
  float* y_out;           // down: [R][H]
  Header* hdr;
};

struct GpSmem {
  size_t stages, bars, total;
};
template <bool MX, bool GATEUP>
__host__ __device__ inline GpSmem gp_smem(int nst) {
  using C = GpCfg<MX, GATEUP>;
  GpSmem s{};
  size_t o = 0;
  s.stages = o; o += (size_t)nst * C::kStageBytes;
  s.bars = o;   o += 512;  // barriers, the TMEM address, the row maxima [4][16]
  s.total = o + 1024;
  return s;
}

__host__ __device__ constexpr uint32_t gp_idesc(bool mx) {
  return tc::idesc_e4m3(128, kGroupRows) | (mx ? (5u << 7) : 0u);
}

__device__ __forceinline__ float gp_ue8m0(uint32_t e) {
  return e == 255u ? __uint_as_float(0x7FC00000u) : e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// NC (4, 8 or 16) consecutive accumulator columns of this warp's lane quadrant, from one or
// two TMEM addresses, one wait
template <int NC>
__device__ __forceinline__ void gp_ld(uint32_t t, float (&v)[16]) {
  uint32_t r[16];
  if constexpr (NC == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\ttcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(t)
                 : "memory");
  } else if constexpr (NC == 8) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\ttcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(t)
        : "memory");
  } else {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(t)
        : "memory");
  }
#pragma unroll
  for (int i = 0; i < NC; ++i) v[i] = __uint_as_float(r[i]);
}
template <int NC>
__device__ __forceinline__ void gp_ld2(uint32_t t0, uint32_t t1, float (&a)[16], float (&b)[16]) {
  uint32_t r[32];
  if constexpr (NC == 4) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%8];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%9];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19])
        : "r"(t0), "r"(t1)
        : "memory");
  } else if constexpr (NC == 8) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
        : "r"(t0), "r"(t1)
        : "memory");
  } else {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
        "[%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t0), "r"(t1)
        : "memory");
  }
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[16 + i]);
  }
}

// One K block of the epilogue for the routed-row columns [0, NC) of a group (NC >= its rows):
// read the block's sums from TMEM, release the buffer, promote into the chains (FP32 pairs).
template <bool MX, bool GATEUP, int NC>
__device__ __forceinline__ void gp_promote(uint32_t ta, uint64_t* acce_buf, int lane, const uint64_t (&sa2)[8],
                                           uint32_t e0, uint32_t e1, float s0, float s1, uint64_t (&ch0)[8],
                                           uint64_t (&ch1)[8]) {
  constexpr int kP = NC / 2;
  if (MX) {
    // T = sum over the sub-blocks j ascending of P_j * 2^(e_j - 127), from 0
    uint64_t T0[kP], T1[kP];
#pragma unroll
    for (int c = 0; c < kP; ++c) T0[c] = T1[c] = 0ull;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float v0[16], v1[16];
      if (GATEUP) {
        gp_ld2<NC>(ta + j * kGroupRows, ta + 4 * kGroupRows + j * kGroupRows, v0, v1);
      } else {
        gp_ld<NC>(ta + j * kGroupRows, v0);
      }
      const uint32_t f0 = __float_as_uint(gp_ue8m0((e0 >> (8 * j)) & 0xFFu));
      const uint32_t f1 = GATEUP ? __float_as_uint(gp_ue8m0((e1 >> (8 * j)) & 0xFFu)) : 0u;
      const uint64_t f0x2 = tc::f2pack(f0, f0), f1x2 = tc::f2pack(f1, f1);
#pragma unroll
      for (int c = 0; c < kP; ++c) {
        T0[c] = tc::f2add(T0[c], tc::f2mul(tc::f2pack(__float_as_uint(v0[2 * c]), __float_as_uint(v0[2 * c + 1])), f0x2));
        if (GATEUP)
          T1[c] = tc::f2add(T1[c], tc::f2mul(tc::f2pack(__float_as_uint(v1[2 * c]), __float_as_uint(v1[2 * c + 1])), f1x2));
      }
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(acce_buf);
#pragma unroll
    for (int c = 0; c < kP; ++c) {
      ch0[c] = tc::f2add(ch0[c], tc::f2mul(T0[c], sa2[c]));
      if (GATEUP) ch1[c] = tc::f2add(ch1[c], tc::f2mul(T1[c], sa2[c]));
    }
  } else {
    float v0[16], v1[16];
    if (GATEUP) {
      gp_ld2<NC>(ta, ta + kGroupRows, v0, v1);
    } else {
      gp_ld<NC>(ta, v0);
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(acce_buf);
    // term = P * (sa * sw): the scale product first, then the multiply and the add
    const uint64_t s0x2 = tc::f2pack(__float_as_uint(s0), __float_as_uint(s0));
    const uint64_t s1x2 = tc::f2pack(__float_as_uint(s1), __float_as_uint(s1));
#pragma unroll
    for (int c = 0; c < kP; ++c) {
      ch0[c] = tc::f2add(ch0[c], tc::f2mul(tc::f2pack(__float_as_uint(v0[2 * c]), __float_as_uint(v0[2 * c + 1])),
                                           tc::f2mul(sa2[c], s0x2)));
      if (GATEUP)
        ch1[c] = tc::f2add(ch1[c], tc::f2mul(tc::f2pack(__float_as_uint(v1[2 * c]), __float_as_uint(v1[2 * c + 1])),
                                             tc::f2mul(sa2[c], s1x2)));
    }
  }
}

// tmA: weight tiles (FP8: u8 [rows][Kd], box 128 x 128, 128-byte swizzle; MXFP4: the packed
// codes as 4-bit elements, padded layout); tmB: the sorted routed rows (gate/up: xp [R][H],
// down: act [R][I]), box 128 bytes x 16 rows, 128-byte swizzle.
// Persistent: the work items are (group, output block) pairs, n_groups * ncb of them (the
// group count comes from the sort); CTA c takes items c, c + G, c + 2G, ... (G = the grid),
// so every CTA gets the same number of items, give or take one, whatever the group count.
// Every role walks the same (item, K block) steps through one ring and one TMEM double
// buffer; the epilogue finishes an item (SiLU and requantisation, or the y stores) as its
// last K block is promoted.
template <bool MX, bool GATEUP>
__global__ void __launch_bounds__(kGpThreads, GpCfg<MX, GATEUP>::kCtasPerSm)
    gpair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GpParams p) {
  using C = GpCfg<MX, GATEUP>;
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int nst = p.nst, nkb = p.nkb;
  const GpSmem SL = gp_smem<MX, GATEUP>(nst);
  unsigned char* stages = base + SL.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + SL.bars);
  uint64_t* full = bars;                   // [kMaxStages]
  uint64_t* empty = bars + kMaxStages;     // [kMaxStages]
  uint64_t* accf = bars + 2 * kMaxStages;  // [2]
  uint64_t* acce = accf + 2;               // [2]
  uint64_t* drainb = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drainb + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 1);  // [4][16] warp maxima per routed row
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
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
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int n_items = (int)*reinterpret_cast<volatile const uint32_t*>(&p.hdr_ro->n_groups) * p.ncb;
  // the CTAs that take items: all the items at once if the grid holds them; for up to two
  // rounds of the grid, two or three per SM, whichever needs fewer rounds x CTAs per SM (the
  // items cost the same and an SM's bandwidth is shared by its CTAs); for more, the whole grid
  // (the last round's share is small and more CTAs hide more latency); the rest leave at once
  int G = (int)gridDim.x;
  if (n_items <= G) {
    G = n_items;
  } else if (G > 2 * p.sms && n_items <= 2 * G) {
    const int g2 = 2 * p.sms;
    const long long c2 = (long long)((n_items + g2 - 1) / g2) * g2, c3 = (long long)((n_items + G - 1) / G) * G;
    if (c2 < c3) G = g2;
  }
  if ((int)blockIdx.x >= G) return;
  const int my_items = (n_items - (int)blockIdx.x + G - 1) / G;
  const int total = my_items * nkb;  // (item, K block) steps
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  const int nrows_e = GATEUP ? 2 * p.I : p.H;
  const int npre = min(nst, total);
  // item j of this CTA: group u / ncb, output block u % ncb (u = blockIdx.x + j * G)
  auto item = [&](int j, Tile& gr, int& cb) {
    const int u = (int)blockIdx.x + j * G;
    gr = p.groups[u / p.ncb];
    cb = u % p.ncb;
  };
  auto load_step = [&](int i, int s, const Tile& gr, int cb) {
    unsigned char* st = stages + s * C::kStageBytes;
    const int x = (i % nkb) * 128;  // 128 codes (MXFP4) or bytes per K block
    tc::mbar_arrive_expect_tx(&full[s], C::kATiles * C::kATx + C::kBBytes);
    tc::tma_load_2d(st, &tmA, &full[s], x, gr.expert * nrows_e + cb * 128);
    if (GATEUP) tc::tma_load_2d(st + C::kABytes, &tmA, &full[s], x, gr.expert * nrows_e + p.I + cb * 128);
    tc::tma_load_2d(st + C::kATiles * C::kABytes, &tmB, &full[s], x, gr.row0);
  };

  if (warp == 0 && lane < npre) {  // one lane per stage for the first stages
    Tile gr;
    int cb;
    item(lane / nkb, gr, cb);
    load_step(lane, lane, gr, cb);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (warp == 0) {
    int issued = npre;
    Tile gr{};
    int cb = 0, cur = -1;
    for (int i = npre; i < total; ++i) {
      const int s = i % nst;
      const uint32_t ph = (i / nst) & 1;
      bool w_ok = true;
      if (lane == 0) w_ok = tc::mbar_wait(&empty[s], ph ^ 1);
      if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) { ok = false; break; }
      if (i / nkb != cur) {
        cur = i / nkb;
        item(cur, gr, cb);
      }
      if (lane == 0) load_step(i, s, gr, cb);
      issued = i + 1;
    }
    // no load is still writing when the CTA leaves (a no-op unless a wait gave up)
    if (lane == 0)
      for (int i = issued - 1; i >= 0 && i >= issued - nst; --i)
        if (!tc::mbar_wait(&full[i % nst], (i / nst) & 1)) ok = false;
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = gp_idesc(MX);
      for (int i = 0; i < total; ++i) {
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
        if (MX) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // one 32-wide sub-block per MMA, each into its own sums
            tc::mma_e4m3(d + j * kGroupRows, da0 + 2 * j, db + 2 * j, idesc, 0);
            if (GATEUP) tc::mma_e4m3(d + 4 * kGroupRows + j * kGroupRows, da1 + 2 * j, db + 2 * j, idesc, 0);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc::mma_e4m3(d, da0 + 2 * k, db + 2 * k, idesc, k > 0);
            if (GATEUP) tc::mma_e4m3(d + kGroupRows, da1 + 2 * k, db + 2 * k, idesc, k > 0);
          }
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&accf[buf]);
      }
      tc::mma_commit(drainb);
      if (!tc::mbar_wait(drainb, 0)) ok = false;
    }
  } else {
    // epilogue: thread <-> weight row r = (warp % 4) * 32 + lane of the 128-row tile
    const int q = warp & 3, r = q * 32 + lane;
    const int nsub = nkb * 4;
    const uint8_t* es = static_cast<const uint8_t*>(p.w_scale);
    const float* fs = static_cast<const float*>(p.w_scale);
    Tile gr{};
    int cb = 0;
    // the chains as FP32 pairs (routed rows 2c, 2c + 1): gate (or down) and up; every packed
    // operation is two IEEE round-to-nearest operations, bit-identical to the scalar ones
    constexpr int kP = kGroupRows / 2;
    uint64_t ch0[kP], ch1[kP];
#pragma unroll
    for (int c = 0; c < kP; ++c) ch0[c] = ch1[c] = 0ull;
    for (int i = 0; i < total; ++i) {
      const int buf = i & 1, kb = i % nkb;
      if (kb == 0) item(i / nkb, gr, cb);
      const int e = gr.expert, n = gr.nrows;
      // this step's scales, loaded before the accumulator wait that covers their latency:
      // the routed rows' activation scales (rows past n read 0: their columns are ignored)
      // and the weight scales (FP8: the block's; MXFP4: the row's four sub-block bytes)
      uint64_t sa2[kP];
#pragma unroll
      for (int c = 0; c < kP; ++c) {
        const float lo = 2 * c < n ? __ldg(p.a_scale + (size_t)(gr.row0 + 2 * c) * nkb + kb) : 0.0f;
        const float hi = 2 * c + 1 < n ? __ldg(p.a_scale + (size_t)(gr.row0 + 2 * c + 1) * nkb + kb) : 0.0f;
        sa2[c] = tc::f2pack(__float_as_uint(lo), __float_as_uint(hi));
      }
      uint32_t e0 = 0, e1 = 0;
      float s0 = 0.0f, s1 = 0.0f;
      if (MX) {
        const size_t row = (size_t)e * nrows_e + cb * 128 + r;
        e0 = __ldg(reinterpret_cast<const uint32_t*>(es + row * nsub + kb * 4));
        if (GATEUP) e1 = __ldg(reinterpret_cast<const uint32_t*>(es + (row + p.I) * nsub + kb * 4));
      } else {
        s0 = __ldg(fs + ((size_t)e * (nrows_e / 128) + cb) * nkb + kb);
        if (GATEUP) s1 = __ldg(fs + ((size_t)e * (nrows_e / 128) + p.I / 128 + cb) * nkb + kb);
      }
      if (ok && !tc::mbar_wait(&accf[buf], (i >> 1) & 1)) ok = false;
      tc::fence_after_sync();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * C::kAccCols;
      // only the group's rows' columns are read (a uniform branch: n is the group's)
      if (n <= 4)
        gp_promote<MX, GATEUP, 4>(ta, &acce[buf], lane, sa2, e0, e1, s0, s1, ch0, ch1);
      else if (n <= 8)
        gp_promote<MX, GATEUP, 8>(ta, &acce[buf], lane, sa2, e0, e1, s0, s1, ch0, ch1);
      else
        gp_promote<MX, GATEUP, 16>(ta, &acce[buf], lane, sa2, e0, e1, s0, s1, ch0, ch1);
      if (kb != nkb - 1) continue;
      // ---- item complete: group gr, output block cb
      const int row0 = gr.row0;
      float g0[kGroupRows], g1[kGroupRows];
#pragma unroll
      for (int c = 0; c < kP; ++c) {
        tc::f2unpack(ch0[c], g0[2 * c], g0[2 * c + 1]);
        tc::f2unpack(ch1[c], g1[2 * c], g1[2 * c + 1]);
      }
      if (GATEUP) {
        // act = silu(g) * u per routed row; its scale over the 128 rows of this block
        float act[kGroupRows];
#pragma unroll
        for (int b = 0; b < kGroupRows; ++b) {
          act[b] = silu_mul(g0[b], g1[b]);
          float m = fabsf(act[b]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
          if (lane == 0) red[q * kGroupRows + b] = m;
        }
        tc::named_bar(1, 128);
#pragma unroll
        for (int b = 0; b < kGroupRows; ++b) {
          if (b < n) {
            const float amax =
                fmaxf(fmaxf(red[b], red[kGroupRows + b]), fmaxf(red[2 * kGroupRows + b], red[3 * kGroupRows + b]));
            const float s2 = quant_scale(amax);
            const uint16_t code = e4m3x2_encode(__fdiv_rn(act[b], s2), 0.0f);
            p.act_out[(size_t)(row0 + b) * p.I + cb * 128 + r] = (uint8_t)(code & 0xFF);
            if (r == 0) p.act_scale_out[(size_t)(row0 + b) * (p.I / 128) + cb] = s2;
          }
        }
        tc::named_bar(1, 128);  // red is rewritten by the next item
      } else {
#pragma unroll
        for (int b = 0; b < kGroupRows; ++b)
          if (b < n) p.y_out[(size_t)(row0 + b) * p.H + cb * 128 + r] = g0[b];
      }
#pragma unroll
      for (int c = 0; c < kP; ++c) ch0[c] = ch1[c] = 0ull;
    }
  }
  if (!ok) set_status(p.hdr, MOE_STATUS_WAIT_TIMEOUT);
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

template <bool MX, bool GATEUP>
void set_gp_attrs(const DeviceInfo& d) {
  static PerDeviceOnce once;
  once_per_device(once, [&] {
    cudaFuncSetAttribute(gpair_kernel<MX, GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem_optin);
  });
}

// The launch plan (persistent): three CTAs per SM where their TMEM columns fit and a ring of
// at least two stages does too (more CTAs split a small item count finer), else two; the
// deepest ring (<= kMaxStages) at that count; shared memory raised so that the CTAs on an SM
// never need more TMEM columns than it has. The grid never exceeds the host's bound on the
// work items.
template <bool MX, bool GATEUP>
cudaError_t launch_gp(const CUtensorMap& tA, const CUtensorMap& tB, GpParams prm, int64_t max_groups,
                      cudaStream_t st) {
  using C = GpCfg<MX, GATEUP>;
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  auto stages_for = [&](int cps) {
    int n = kMaxStages;
    for (; n > 1; --n)
      if ((gp_smem<MX, GATEUP>(n).total + 1024) * cps <= d.smem_per_sm) break;
    return n;
  };
  int cps = 2;
  if (C::kCtasPerSm >= 3 && stages_for(3) >= 2) cps = 3;
  prm.nst = stages_for(cps);
  prm.sms = d.sms;
  const size_t smem = std::max(gp_smem<MX, GATEUP>(prm.nst).total, d.smem_per_sm / (C::kMaxCtasPerSm + 1) + 1);
  if (smem > d.smem_optin) return cudaErrorInvalidConfiguration;
  set_gp_attrs<MX, GATEUP>(d);
  const int64_t grid = std::min<int64_t>((int64_t)cps * d.sms, max_groups * prm.ncb);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kGpThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gpair_kernel<MX, GATEUP>, tA, tB, prm);
}

bool weight_map(bool mx, CUtensorMap* m, const uint8_t* w, uint64_t kd, uint64_t rows) {
  return mx ? make_tmap_e2m1(m, w, kd, rows) : make_tmap_u8(m, w, kd, rows, 128);
}

}  // namespace

// gate/up over the sort's groups: act / act_scale at the sorted rows (R = routed rows placed
// by the sort, max_groups = the host's bound on the group count).
cudaError_t launch_gpair_gateup(bool mx, const uint8_t* w13, const void* s13, int64_t R, int H, int I, int E,
                                int64_t max_groups, const WsPtrs& ws, cudaStream_t st) {
  CUtensorMap tA, tB;
  if (!weight_map(mx, &tA, w13, (uint64_t)H, (uint64_t)E * 2 * I)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tB, ws.xp, (uint64_t)H, (uint64_t)R, kGroupRows)) return cudaErrorInvalidValue;
  GpParams prm{};
  prm.H = H; prm.I = I; prm.E = E;
  prm.nkb = H / 128;
  prm.ncb = I / 128;
  prm.groups = ws.groups;
  prm.hdr_ro = ws.hdr;
  prm.w_scale = s13;
  prm.a_scale = ws.sa_p;
  prm.act_out = ws.act;
  prm.act_scale_out = ws.act_scale;
  prm.hdr = ws.hdr;
  return mx ? launch_gp<true, true>(tA, tB, prm, max_groups, st) : launch_gp<false, true>(tA, tB, prm, max_groups, st);
}

// down over the sort's groups: y [R][H] FP32 at the sorted rows.
cudaError_t launch_gpair_down(bool mx, const uint8_t* w2, const void* s2, int64_t R, int H, int I, int E,
                              int64_t max_groups, const WsPtrs& ws, cudaStream_t st) {
  CUtensorMap tA, tB;
  if (!weight_map(mx, &tA, w2, (uint64_t)I, (uint64_t)E * H)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tB, ws.act, (uint64_t)I, (uint64_t)R, kGroupRows)) return cudaErrorInvalidValue;
  GpParams prm{};
  prm.H = H; prm.I = I; prm.E = E;
  prm.nkb = I / 128;
  prm.ncb = H / 128;
  prm.groups = ws.groups;
  prm.hdr_ro = ws.hdr;
  prm.w_scale = s2;
  prm.a_scale = ws.act_scale;
  prm.y_out = ws.y;
  prm.hdr = ws.hdr;
  return mx ? launch_gp<true, false>(tA, tB, prm, max_groups, st) : launch_gp<false, false>(tA, tB, prm, max_groups, st);
}

}  // namespace moe
