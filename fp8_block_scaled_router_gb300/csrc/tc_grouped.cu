// tc_grouped.cu -- block-scaled grouped expert GEMMs on tcgen05 for many routed rows
// (prefill): expert-sorted tiles of up to 128 routed rows.
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (the routed MoE
// producer: gate/up, SiLU and quantisation, down-partial); older lab README, supported
// targets (FP8 E4M3 weights with 128x128 FP32 block scales); docs/compiler/architecture.md
// (FP8 activation and activation-scale intermediates between gate/up and down).
//
// Persistent: one CTA per SM walks the (tile, 256-wide output block) units. A = the tile's 128 activation rows (FP8,
// expert-sorted: the gathered hidden codes for gate/up, the activation codes for down),
// B = 256 weight rows of the tile's expert -- for gate/up the 128 gate rows of an output
// block and the matching 128 up rows, interleaved in groups of 64 (two boxes of a 3-D view
// of w13: 64 rows x {gate, up}), for down 256 rows of w2 (one box). Per 128-wide K block
// three lanes of the TMA warp load A (16 KB) and B (32 KB) -- few, tall boxes stream
// faster per issue than many short ones -- into a four-stage ring (128-byte swizzle), the
// MMA warp issues four 128x256x32 FP8 MMAs into a fresh accumulator (double-buffered:
// per K block: two 128x128x32 halves into four 128-column TMEM buffers, so the tensor
// core runs up to two K blocks ahead of the epilogue), and sixteen epilogue warps promote
// the block sums into FP32 chains
//   acc = fma(P_kb, sa[row][kb] * sw[block][kb], acc)     kb ascending, from 0,
// (one rounding per step: the multiply-add is fused here, which the parity window covers;
// two adjacent columns per packed fma.rn.f32x2);
// thread = (accumulator row, 64 of the 256 columns).
// gate/up epilogue: act = silu(g) * u (split-argument base-2 exponential and the fast
// division, a few ulp for every g) for the thread's columns, the row's amax over 128
// columns (the partner warps' parts via shared memory), scale = amax/448, RNE saturating
// E4M3 codes of act * (448/amax) -> act [row][I] and
// act_scale [row][I/128]. down epilogue: y [row][H] FP32 in 32-byte stores.
// Rows of a tile past its length are computed on zero/neighbour rows and never stored.
#include <cudaTypedefs.h>

#include <mutex>

#include "device.h"
#include "launch.h"
#include "tc.cuh"

namespace moe {

constexpr int kGrpEpiWarps = 16;
constexpr int kGrpThreads = 32 * (2 + kGrpEpiWarps);  // warp 0 TMA, warp 1 MMA + TMEM, 2.. epilogue
constexpr int kGrpStages = 4;
constexpr int kGrpABytes = 128 * 128;
constexpr int kGrpBBytes = 256 * 128;
constexpr int kGrpStageBytes = kGrpABytes + kGrpBBytes;
constexpr int kGrpTmemCols = 512;

struct GrpParams {
  int H, I, E;
  int nkb;                 // K blocks
  int nnb;                 // 256-wide output blocks per tile
  const Tile* tiles;
  const float* w_scale;    // s13 [E][2I/128][H/128] or s2w [E][H/128][I/128]
  const float* a_scale;    // sa_p [R][H/128] (gate/up) or act_scale [R][I/128] (down)
  uint8_t* act_out;        // [R][I]
  float* act_scale_out;    // [R][I/128]
  float* y_out;            // [R][H]
  Header* hdr;
};

// stages, barriers, then gate/up: the row-amax exchange [128][4] f32; down: 16 per-warp
// staging tiles of 32 rows x 16 FP32 for the y stores
__host__ __device__ constexpr size_t grp_smem_bytes(bool gateup) {
  return 1024 + (size_t)kGrpStages * kGrpStageBytes + 256 + (gateup ? 128 * 4 * 4 : kGrpEpiWarps * 32 * 16 * 4);
}

template <bool GATEUP>
__global__ void __launch_bounds__(kGrpThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmY, const GrpParams p) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kGrpStages * kGrpStageBytes);
  uint64_t* full = bars;                      // [kGrpStages]
  uint64_t* empty = bars + kGrpStages;        // [kGrpStages]
  uint64_t* accf = bars + 2 * kGrpStages;     // [4]
  uint64_t* acce = bars + 2 * kGrpStages + 4; // [4]
  uint64_t* drainb = bars + 2 * kGrpStages + 8;  // every MMA this CTA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kGrpStages + 9);
  float* red = reinterpret_cast<float*>(base + kGrpStages * kGrpStageBytes + 256);  // [128][4]
  float* ystage = red;  // down: [16 warps][32 rows][16] f32
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
    for (int s = 0; s < kGrpStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 4; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], kGrpEpiWarps / 2);
    }
    tc::mbar_init(drainb, 1);
    tc::fence_mbar_init();
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  // persistent: CTA b takes units b, b + gridDim.x, ... (a unit = one tile x one 256-wide
  // output block); every role walks the same (unit, K block) sequence, so the stage ring
  // and the TMEM double buffer run on across unit boundaries
  const int n_units = (int)*reinterpret_cast<volatile const uint32_t*>(&p.hdr->n_tiles) * p.nnb;
  if ((int)blockIdx.x >= n_units) return;

  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kGrpTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int nkb = p.nkb;

  bool ok = true;
  if (warp == 0) {
    int it = 0, last = -1;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int nb = u % p.nnb;
      const Tile tl = p.tiles[u / p.nnb];
      // B rows in shared memory: gate/up [gate 0-63 | up 0-63 | gate 64-127 | up 64-127]
      // of the output block (each 128-row half = matching gate and up rows), down
      // [w2 rows nb*256 .. +256]
      const int yd = tl.expert * p.H + nb * 256;
      for (int i = 0; i < nkb; ++i, ++it) {
        const int s = it % kGrpStages;
        const uint32_t ph = (it / kGrpStages) & 1;
        bool w_ok = true;
        if (lane == 0) w_ok = tc::mbar_wait(&empty[s], ph ^ 1);
        if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) { ok = false; break; }
        unsigned char* st = stages + s * kGrpStageBytes;
        last = it;
        if (lane == 0) tc::mbar_arrive_expect_tx(&full[s], kGrpStageBytes);
        __syncwarp();
        const int x = i * 128;
        if (lane == 0) tc::tma_load_2d(st, &tmA, &full[s], x, tl.row0);
        if (GATEUP) {
          if (lane == 1 || lane == 2) {
            const int h = lane - 1;  // rows nb*128 + h*64 .. +64 of gate (z = 2e) and up (2e+1)
            tc::tma_load_3d(st + kGrpABytes + h * 128 * 128, &tmB, &full[s], x, nb * 128 + h * 64, 2 * tl.expert);
          }
        } else if (lane == 1) {
          tc::tma_load_2d(st + kGrpABytes, &tmB, &full[s], x, yd);
        }
      }
    }
    // no load is still writing when the CTA leaves (a no-op unless a wait gave up)
    if (lane == 0 && last >= 0 && !tc::mbar_wait(&full[last % kGrpStages], (last / kGrpStages) & 1)) ok = false;
  } else if (warp == 1) {
    if (lane == 0) {
      // per K block two 128x128 halves into TMEM buffers (2*it + h) % 4 (128 columns each),
      // so the MMAs run up to two K blocks ahead of the epilogue
      constexpr uint32_t idesc = tc::idesc_e4m3(128, 128);
      int it = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        for (int i = 0; i < nkb; ++i, ++it) {
          const int s = it % kGrpStages;
          const uint32_t ph = (it / kGrpStages) & 1;
          if (!tc::mbar_wait(&full[s], ph)) { ok = false; break; }
          const uint32_t sa = tc::smem_u32(stages + s * kGrpStageBytes);
          const uint64_t da = tc::sdesc_sw128(sa);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int slot = 2 * it + h;
            const int buf = slot & 3;
            if (!tc::mbar_wait(&acce[buf], ((slot >> 2) & 1) ^ 1)) { ok = false; break; }
            tc::fence_after_sync();
            const uint64_t db = tc::sdesc_sw128(sa + kGrpABytes + h * 128 * 128);
            const uint32_t d = tmem + buf * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k) tc::mma_e4m3(d, da + 2 * k, db + 2 * k, idesc, k > 0);
            // the stage is read once both halves are issued: released before the last
            // accumulator, whose arrival the epilogue waits for
            if (h == 1) tc::mma_commit(&empty[s]);
            tc::mma_commit(&accf[buf]);
          }
          if (!ok) break;
        }
      }
      // every arrival the MMAs owe this CTA's barriers has landed before the CTA can leave
      tc::mma_commit(drainb);
      if (!tc::mbar_wait(drainb, 0)) ok = false;
    }
  } else {
    // epilogue: 8 warps per MMA half hh; thread = (accumulator row, 64 of the half's 128
    // columns): gate/up -> 32 gate + 32 up chains (act columns hh*64 + sub*32 .. +32),
    // down -> 64 output columns of w2 block nb*2 + hh
    const int q = warp & 3;               // TMEM lane quadrant (hardware: warp % 4)
    const int ew = warp - 2;
    const int hh = ew >> 3;               // MMA half
    const int sub = (ew >> 2) & 1;        // which 64 of the half's 128 columns
    const int row = q * 32 + lane;
    const int slot4 = hh * 2 + sub;       // column quarter of the row's 256 outputs
    constexpr int kEpiThreads = 32 * kGrpEpiWarps;
    // every epilogue warp walks every unit (the named barriers below need all of them);
    // after a wait has run out the remaining waits are skipped, so the kernel still ends
    int it = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const int nb = u % p.nnb;
      const Tile tl = p.tiles[u / p.nnb];
      const int e = tl.expert, row0 = tl.row0;
      const bool live = row < tl.nrows;
      const float* sarow = p.a_scale + (size_t)(row0 + (live ? row : 0)) * nkb;
      const float* sw0 = GATEUP ? p.w_scale + ((size_t)e * (2 * p.I / 128) + nb) * nkb
                                : p.w_scale + ((size_t)e * (p.H / 128) + nb * 2 + hh) * nkb;
      const float* sw1 = GATEUP ? p.w_scale + ((size_t)e * (2 * p.I / 128) + p.I / 128 + nb) * nkb : sw0;
      // within the half's 128 accumulator columns: gate/up [gate 64 | up 64], down [128]
      const uint32_t c0 = GATEUP ? sub * 32 : sub * 64;
      const uint32_t c1 = GATEUP ? 64 + sub * 32 : sub * 64 + 32;
      // promoted chains as FP32 pairs (adjacent columns share a scale): [0,16) the run at
      // c0, [16,32) the run at c1; fma.rn.f32x2 is two IEEE fmas, bit-identical to fmaf
      uint64_t acc2[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) acc2[c] = 0ull;
      for (int i = 0; i < nkb; ++i, ++it) {
        // block i's scales, loaded before the accumulator wait that covers their latency
        const float a = live ? sarow[i] : 0.0f, s0 = sw0[i], s1 = sw1[i];
        const int slot = 2 * it + hh;
        const int buf = slot & 3;
        if (ok && !tc::mbar_wait(&accf[buf], (slot >> 2) & 1)) ok = false;
        tc::fence_after_sync();
        const uint32_t sc0 = __float_as_uint(__fmul_rn(a, s0)), sc1 = __float_as_uint(__fmul_rn(a, s1));
        const uint64_t sc0x2 = tc::f2pack(sc0, sc0), sc1x2 = tc::f2pack(sc1, sc1);
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * 128;
        uint32_t P[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tc::tmem_ld16x2u(ta + c0 + h * 16, ta + c1 + h * 16, P);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            acc2[h * 8 + c] = tc::f2fma(tc::f2pack(P[2 * c], P[2 * c + 1]), sc0x2, acc2[h * 8 + c]);
            acc2[16 + h * 8 + c] = tc::f2fma(tc::f2pack(P[16 + 2 * c], P[16 + 2 * c + 1]), sc1x2, acc2[16 + h * 8 + c]);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[buf]);
      }
      float acc[64];  // [0,32) run at c0, [32,64) run at c1
#pragma unroll
      for (int c = 0; c < 32; ++c) tc::f2unpack(acc2[c], acc[2 * c], acc[2 * c + 1]);
      if (GATEUP) {
        // act = silu(g) * u for 32 columns; row amax over the 128 columns of the block
        float act[32];
        float amax = 0.0f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          act[c] = silu_mul_fast(acc[c], acc[32 + c]);
          amax = fmaxf(amax, fabsf(act[c]));
        }
        red[row * 4 + slot4] = amax;
        tc::named_bar(1, kEpiThreads);
        amax = fmaxf(fmaxf(red[row * 4], red[row * 4 + 1]), fmaxf(red[row * 4 + 2], red[row * 4 + 3]));
        tc::named_bar(1, kEpiThreads);  // red is rewritten by the next unit
        const float s2 = quant_scale(amax);
        // codes = RNE_E4M3(act * (448 / amax)): one reciprocal per row instead of 32
        // divisions; within one ulp of act / s2 before rounding to E4M3
        const float inv = amax == 0.0f ? 1.0f : __fdiv_rn(448.0f, amax);
        if (live) {
          uint8_t* dst = p.act_out + (size_t)(row0 + row) * p.I + nb * 128 + slot4 * 32;
          uint32_t w8[8];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const int c = q4 * 4;
            const uint32_t lo = e4m3x2_encode(__fmul_rn(act[c], inv), __fmul_rn(act[c + 1], inv));
            const uint32_t hi = e4m3x2_encode(__fmul_rn(act[c + 2], inv), __fmul_rn(act[c + 3], inv));
            w8[q4] = lo | (hi << 16);
          }
          // the row's 32 codes in one 32-byte store (a whole L2 sector)
          asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(w8[0]), "r"(w8[1]),
                       "r"(w8[2]), "r"(w8[3]), "r"(w8[4]), "r"(w8[5]), "r"(w8[6]), "r"(w8[7])
                       : "memory");
          if (slot4 == 0) p.act_scale_out[(size_t)(row0 + row) * (p.I / 128) + nb] = s2;
        }
      } else if (q * 32 + 32 <= tl.nrows) {
        // all 32 rows of this warp belong to the tile: four 32 x 16 pieces through shared
        // memory, each written by one TMA store (whole rows of 64 bytes per request)
        float* stw = ystage + (ew * 32) * 16;
        for (int ch = 0; ch < 4; ++ch) {
          if (lane == 0) tc::bulk_wait_read_all();  // the previous piece has left shared memory
          __syncwarp();
          float4* d4 = reinterpret_cast<float4*>(stw + lane * 16);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            d4[c4] = make_float4(acc[ch * 16 + 4 * c4], acc[ch * 16 + 4 * c4 + 1], acc[ch * 16 + 4 * c4 + 2],
                                 acc[ch * 16 + 4 * c4 + 3]);
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tc::tma_store_2d(&tmY, stw, nb * 256 + slot4 * 64 + ch * 16, row0 + q * 32);
            tc::bulk_commit();
          }
        }
      } else if (live) {
        // a warp straddling the tile's end (the next rows belong to another tile): 32-byte
        // stores of the live rows, each one filling a whole L2 sector
        float* dst = p.y_out + (size_t)(row0 + row) * p.H + nb * 256 + slot4 * 64;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 8 * c8), "f"(acc[8 * c8]),
                       "f"(acc[8 * c8 + 1]), "f"(acc[8 * c8 + 2]), "f"(acc[8 * c8 + 3]), "f"(acc[8 * c8 + 4]),
                       "f"(acc[8 * c8 + 5]), "f"(acc[8 * c8 + 6]), "f"(acc[8 * c8 + 7])
                       : "memory");
      }
    }
  }
  if (!ok) set_status(p.hdr, MOE_STATUS_WAIT_TIMEOUT);
  if (!GATEUP && warp >= 2 && lane == 0) tc::bulk_wait_all();  // this warp's y stores are done
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kGrpTmemCols);
  }
}

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
bool make_tmap_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                   uint32_t box_rows);
bool make_tmap_u8_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                     uint64_t s2, uint32_t b1, uint32_t b2);

namespace {

template <bool GATEUP>
cudaError_t launch_grouped(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tY,
                           const GrpParams& prm, int64_t max_tiles, cudaStream_t st) {
  static PerDeviceOnce once;
  once_per_device(once, [] {
    cudaFuncSetAttribute(grouped_gemm_kernel<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)grp_smem_bytes(GATEUP));
  });
  const int num_sms = device_info().sms;
  if (num_sms == 0) return cudaErrorInvalidDevice;
  const int64_t units = max_tiles * prm.nnb;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units < num_sms ? units : num_sms), 1, 1);
  cfg.blockDim = dim3(kGrpThreads, 1, 1);
  cfg.dynamicSmemBytes = grp_smem_bytes(GATEUP);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<GATEUP>, tA, tB, tY, prm);
}

}  // namespace

// gate/up over the expert tiles: A = gathered hidden codes xp [R][H] with scales sa_p.
cudaError_t launch_grouped_gateup(const uint8_t* w13, const float* s13, int64_t R, int H, int I, int E,
                                  int64_t max_tiles, const WsPtrs& ws, cudaStream_t st) {
  CUtensorMap tA, tB;
  if (!make_tmap_u8(&tA, ws.xp, (uint64_t)H, (uint64_t)R, 128)) return cudaErrorInvalidValue;
  // w13 viewed as [2E][I][H] (z = 2e gate, 2e + 1 up); a box is 64 rows of gate then the same
  // 64 rows of up
  if (!make_tmap_u8_3d(&tB, w13, (uint64_t)H, (uint64_t)I, (uint64_t)E * 2, (uint64_t)H, (uint64_t)I * H, 64, 2))
    return cudaErrorInvalidValue;
  GrpParams prm{};
  prm.H = H; prm.I = I; prm.E = E;
  prm.nkb = H / 128;
  prm.nnb = I / 128;
  prm.tiles = ws.tiles;
  prm.w_scale = s13;
  prm.a_scale = ws.sa_p;
  prm.act_out = ws.act;
  prm.act_scale_out = ws.act_scale;
  prm.y_out = ws.y;
  prm.hdr = ws.hdr;
  return launch_grouped<true>(tA, tB, tA, prm, max_tiles, st);  // no y stores
}

// down over the expert tiles: A = activation codes act [R][I], y [R][H] (H % 256 == 0).
cudaError_t launch_grouped_down(const uint8_t* w2, const float* s2w, int64_t R, int H, int I, int E,
                                int64_t max_tiles, const WsPtrs& ws, cudaStream_t st) {
  CUtensorMap tA, tB, tY;
  if (!make_tmap_u8(&tA, ws.act, (uint64_t)I, (uint64_t)R, 128)) return cudaErrorInvalidValue;
  // y [R][H] FP32 written in 32-row x 16-column pieces
  if (!make_tmap_f32(&tY, ws.y, (uint64_t)H, (uint64_t)R, 16, 32)) return cudaErrorInvalidValue;
  // one 256-row box per stage: the w2 rows of the 256-wide output block
  if (!make_tmap_u8(&tB, w2, (uint64_t)I, (uint64_t)E * H, 256)) return cudaErrorInvalidValue;
  GrpParams prm{};
  prm.H = H; prm.I = I; prm.E = E;
  prm.nkb = I / 128;
  prm.nnb = H / 256;
  prm.tiles = ws.tiles;
  prm.w_scale = s2w;
  prm.a_scale = ws.act_scale;
  prm.act_out = ws.act;
  prm.act_scale_out = ws.act_scale;
  prm.y_out = ws.y;
  prm.hdr = ws.hdr;
  return launch_grouped<false>(tA, tB, tY, prm, max_tiles, st);
}

}  // namespace moe
