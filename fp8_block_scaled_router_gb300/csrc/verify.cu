// verify.cu -- the speculative-verify layer as two operations: a producer launch (routing,
// gate/up, SiLU(gate)*up with the FP8 requantisation, and the down partials of every routed
// pair) and a separate route reducer (the slot-order combine), both behind an exact batch
// guard.
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (a producer
// composed of semantic routing, gate/up, SiLU and quantisation, down-partial and metadata
// stages; the route reducer a separate fixed operation with its own ABI, launch geometry and
// reduction order; the verify_m12 profiles) and the compiler notes on profiles (a kernel
// whose grid depends on the batch takes an exact batch guard, e.g. verify_m12_b1).
//
// The profile compiled here: 12 tokens (one verify step of one request) through the
// h2048 / i768 / e128 / top-8 layer. The grid, the tile shapes and the shared-memory plan
// depend on those numbers; any other call is refused on the host.
//
// GB300 design. The launch is as many 16-CTA clusters as are resident at once with one CTA
// per SM; the clusters never wait on one another. Inside a cluster:
//   * routing: CTA r owns hidden chunk r (128 columns) of every expert and runs the chunk's
//     FP32 fma chains (k ascending from 0) for all 12 tokens; token t's 16 chunk partials
//     are copied into CTA t, which adds them in chunk order, adds the bias, ranks the top 8
//     (ties to the lower expert) and forms the softmax weights -- the router kernel's
//     arithmetic, so ids and weights are those of moe_route -- and copies the route to
//     every CTA of the cluster. Every cluster routes for itself.
//   * metadata: the distinct routed experts in ascending order, and for each of them the
//     slot each token gave it (or none). Cluster c takes distinct experts c, c + nc, ...
//   * gate/up: units (expert, 128-column block cb of the activation) dealt round-robin to
//     the 16 CTAs. A unit reads its 128 gate and 128 up weight rows over all 16 K blocks
//     once; the B operand is every token's hidden row (12 of the 16 MMA columns), so one
//     read of the weights serves every token routed to the expert. The epilogue promotes
//     each K block's sums (P_kb * (sa_kb * sw_kb), multiply then add, kb ascending from 0),
//     applies silu(g) * u, requantises each routed token's 128 values (scale = amax/448) and
//     writes the codes and scale of that pair (row t*8 + slot) to the workspace.
//   * down: CTA r runs output block r (128 rows) of every expert of the cluster, each as soon
//     as the expert's 6 activation blocks are written (the CTA of each block arrives,
//     releasing at cluster scope, on that expert's mbarrier in every CTA): B = the routed
//     tokens' activation rows, gathered from the workspace into shared memory; y = sum over
//     the 6 K blocks ascending of P_kb * (s2_kb * sw2_kb); each routed pair's y goes to the
//     workspace. A CTA that finishes its gate/up units early starts on the down blocks of
//     the experts already complete.
// The reducer then forms out[t] = bf16(sum over slots ascending of w[t][j] * y[t*8 + j]).
// The arithmetic is that of the few-row pair kernels (moe_fp8_gate_up_direct +
// moe_fp8_down_combine), so outputs are bitwise theirs.
//
// Teardown: the MMA lane's last commit goes to a drain barrier that it waits for, and each TMA
// lane waits for its last load, so no asynchronous arrival or write can reach this CTA's shared
// memory after it has left (or land in the next CTA to get the SM).
// Warp roles: 0 TMA (four issuing lanes, one per ring slot), 1 TMEM + MMA issue,
// 2-5 epilogue (TMEM lane quadrant = warp % 4), 6-7 down B-tile builders; all eight warps
// quantise the hidden rows and route. Every wait is bounded and reports
// MOE_STATUS_WAIT_TIMEOUT.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "device.h"
#include "launch.h"
#include "tc.cuh"

namespace moe {

constexpr int kVM = 12, kVH = 2048, kVI = 768, kVE = 128, kVK = 8;  // the verify_m12 profile
constexpr int kVR = kVM * kVK;                                     // routed pairs
constexpr int kVCL = 16;                                           // CTAs per cluster
constexpr int kVThreads = 256;
constexpr int kVNkh = kVH / 128;  // hidden K blocks (one router chunk per CTA)
constexpr int kVNu = kVI / 128;   // activation blocks
constexpr int kVNhb = kVH / 128;  // down output blocks (one per CTA)
constexpr int kVSlots = 4;        // ring slots of two 16 KB tiles
constexpr int kVTile = 128 * 128;
constexpr int kVMaxGU = 8;        // gate/up units per CTA
constexpr int kVMaxDn = 16;       // experts per cluster (down units per CTA)
constexpr int kVTmemCols = 512;   // gate/up: 8 x 32 columns; down: 8 x 16 columns from 256
static_assert(kVNkh == kVCL && kVNhb == kVCL, "one router chunk and one down block per CTA");
static_assert(kVE == 128 && kVK == 8, "routing staging assumes 128 experts and 8 slots");

struct VerifyParams {
  int renorm;
  int nc;                    // clusters
  const uint16_t* hidden;    // BF16 [12][2048]
  const uint16_t* router_w;  // BF16 [2048][128]
  const float* bias;         // [128] or null
  int32_t* ids;              // [12][8] out
  float* wts;                // [12][8] out
  const float* s13;          // [E][2I/128][H/128]
  const float* s2w;          // [E][H/128][I/128]
  WsPtrs ws;                 // qa, sa, act, act_scale, y, perm_row, row_src, pair_expert, hdr
};

// Shared memory (offsets from the 1024-aligned base).
//   ring     kVSlots x 32 KB (two weight tiles per slot; before the weights: the CTA's router
//            chunk in [0, 32 KB) and the 12 hidden rows (BF16) in [32 KB, 80 KB))
//   hid      16 x 2 KB hidden B tiles (row t = token t's codes of K block kb, rows 12..15 0)
//   acttile  2 x 6 x 2 KB down B tiles (one expert's activation rows), aliased before the
//            down phase by own (12 x 128 f32 chain partials of chunk r, staged for the copies)
//   part     16 x 128 f32 (token t's chunk partials, owner CTA t)
//   misc     logits, selection, routes, bias, scales, metadata
constexpr size_t kVoRing = 0;
constexpr size_t kVoHid = kVoRing + (size_t)kVSlots * 2 * kVTile;
constexpr size_t kVoAct = kVoHid + (size_t)kVNkh * 2048;
constexpr size_t kVoHs = kVoRing + (size_t)2 * kVTile;  // the hidden rows, in ring slot 1
constexpr size_t kVoOwn = kVoAct;
constexpr size_t kVoPart = kVoAct + (size_t)2 * kVNu * 2048;
constexpr size_t kVoLogits = kVoPart + (size_t)kVCL * 128 * 4;
constexpr size_t kVoSel = kVoLogits + 128 * 4;            // sel_v [16] f32, sel_i [16] i32
constexpr size_t kVoRst = kVoSel + 32 * 4;                // the owner's route: 8 ids, 8 weights
constexpr size_t kVoRoutes = kVoRst + 16 * 4;             // [12][16]: ids, weights (bits)
constexpr size_t kVoBias = kVoRoutes + (size_t)kVM * 16 * 4;
constexpr size_t kVoSa = kVoBias + 128 * 4;               // [12][16] hidden scales
constexpr size_t kVoSw13 = kVoSa + (size_t)kVM * kVNkh * 4;   // [kVMaxGU][16][2]
constexpr size_t kVoSw2 = kVoSw13 + (size_t)kVMaxGU * kVNkh * 2 * 4;  // [kVMaxDn][8]
constexpr size_t kVoAsc = kVoSw2 + (size_t)kVMaxDn * 8 * 4;   // [2][12][8] activation scales
constexpr size_t kVoRed = kVoAsc + (size_t)2 * kVM * 8 * 4;   // [4][16] warp maxima
constexpr size_t kVoUsed = kVoRed + 4 * 16 * 4;               // [128] i32
constexpr size_t kVoDist = kVoUsed + 128 * 4;                 // [128] i32 distinct experts
constexpr size_t kVoE2l = kVoDist + 128 * 4;                  // [128] i32 expert -> local index
constexpr size_t kVoWcnt = kVoE2l + 128 * 4;                  // [4] i32 + n_dist
constexpr size_t kVoSlot = kVoWcnt + 8 * 4;                   // [96][12] i8 slot of token t
constexpr size_t kVoBars = (kVoSlot + (size_t)kVR * kVM + 15) & ~size_t(15);
constexpr int kVNumBars = 2 * kVSlots + 16 + 16 + 4 + kVMaxDn + 2 + 2 + 1;
constexpr size_t kVSmem = kVoBars + (size_t)kVNumBars * 8 + 16 + 1024;  // + alignment slack
static_assert(kVoOwn + (size_t)kVM * 128 * 4 <= kVoPart, "own fits in the down tiles");
static_assert(kVoHs + (size_t)kVM * kVH * 2 <= kVoHid, "the hidden rows fit in the ring");

// Byte offset of 16-byte chunk c of row r in a K-major tile of 128-byte rows with the
// 128-byte swizzle (8-row atoms of 1024 bytes; chunk c of row r sits at c ^ (r % 8)).
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// tm13: w13 as [2E][I][H] (z = 2e gate, 2e + 1 up), box 128 bytes x 128 rows x 2; tm2: w2 as
// [E*H][I], box 128 bytes x 128 rows.
__global__ void __launch_bounds__(kVThreads, 1)
    verify_kernel(const __grid_constant__ CUtensorMap tm13, const __grid_constant__ CUtensorMap tm2,
                  const VerifyParams p) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* ring = base + kVoRing;
  unsigned char* hid = base + kVoHid;
  unsigned char* acttile = base + kVoAct;
  const uint16_t* hs = reinterpret_cast<const uint16_t*>(base + kVoHs);
  float* own = reinterpret_cast<float*>(base + kVoOwn);
  float* part = reinterpret_cast<float*>(base + kVoPart);
  float* logits = reinterpret_cast<float*>(base + kVoLogits);
  float* sel_v = reinterpret_cast<float*>(base + kVoSel);
  int* sel_i = reinterpret_cast<int*>(sel_v + 16);
  uint32_t* rst = reinterpret_cast<uint32_t*>(base + kVoRst);
  uint32_t* routes = reinterpret_cast<uint32_t*>(base + kVoRoutes);
  float* bias_s = reinterpret_cast<float*>(base + kVoBias);
  float* sa_s = reinterpret_cast<float*>(base + kVoSa);
  float* sw13_s = reinterpret_cast<float*>(base + kVoSw13);
  float* sw2_s = reinterpret_cast<float*>(base + kVoSw2);
  float* asc_s = reinterpret_cast<float*>(base + kVoAsc);
  float* red = reinterpret_cast<float*>(base + kVoRed);
  int* used = reinterpret_cast<int*>(base + kVoUsed);
  int* dist = reinterpret_cast<int*>(base + kVoDist);
  int* e2l = reinterpret_cast<int*>(base + kVoE2l);
  int* wcnt = reinterpret_cast<int*>(base + kVoWcnt);
  int8_t* tslot = reinterpret_cast<int8_t*>(base + kVoSlot);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kVoBars);
  uint64_t* fullp = bars;                  // [kVSlots] a slot's two tiles have landed
  uint64_t* emptyp = bars + kVSlots;       // [kVSlots] the MMAs reading a slot are done
  uint64_t* accf = bars + 2 * kVSlots;     // [8] gate/up TMEM buffer written
  uint64_t* acce = accf + 8;               // [8] gate/up TMEM buffer read (4 warps)
  uint64_t* accf2 = acce + 8;              // [8] down TMEM buffer written
  uint64_t* acce2 = accf2 + 8;             // [8] down TMEM buffer read
  uint64_t* rbar = acce2 + 8;              // this CTA's router chunk has landed
  uint64_t* hbar = rbar + 1;               // the hidden rows have landed
  uint64_t* part_full = hbar + 1;          // token rank's 16 chunk partials are here
  uint64_t* routes_full = part_full + 1;   // all 12 routes are here
  uint64_t* eready = routes_full + 1;      // [kVMaxDn] all 6 activation blocks of expert ie are written
  uint64_t* act_ready = eready + kVMaxDn;  // [2] an expert's down B tiles and scales are built
  uint64_t* act_free = act_ready + 2;      // [2] ... and no longer read (MMA + epilogue)
  uint64_t* drainb = act_free + 2;         // every MMA this CTA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(act_free + 3);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int rank = (int)tc::cluster_rank();
  const int cid = (int)tc::cluster_id_x();
  bool ok = true;

  // ---- set-up: barriers, TMEM, this CTA's router chunk and the bias (parameters)
  if (tid == 0) {
    tc::prefetch_tmap(&tm13);
    tc::prefetch_tmap(&tm2);
    for (int s = 0; s < kVSlots; ++s) {
      tc::mbar_init(&fullp[s], 1);
      tc::mbar_init(&emptyp[s], 1);
    }
    for (int b = 0; b < 8; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 4);
      tc::mbar_init(&accf2[b], 1);
      tc::mbar_init(&acce2[b], 4);
    }
    tc::mbar_init(rbar, 1);
    tc::mbar_init(hbar, 1);
    tc::mbar_init(part_full, 1);
    tc::mbar_init(routes_full, 1);
    for (int i = 0; i < kVMaxDn; ++i) tc::mbar_init(&eready[i], kVNu);  // one arrival per gate/up unit
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&act_ready[b], 1);
      tc::mbar_init(&act_free[b], 2);
    }
    tc::mbar_init(drainb, 1);
    // the bytes the exchanges copy into this CTA: token rank's chunk partials (owners) and
    // every token's route
    if (rank < kVM) tc::mbar_arrive_expect_tx(part_full, (uint32_t)(kVCL * 128 * 4));
    tc::mbar_arrive_expect_tx(routes_full, (uint32_t)(kVM * 64));
    tc::fence_mbar_init();
    const uint32_t chunk = 128u * kVE * 2u;
    tc::mbar_arrive_expect_tx(rbar, chunk);
    tc::bulk_load(ring, p.router_w + (size_t)rank * 128 * kVE, chunk, rbar);
    constexpr uint32_t hbytes = (uint32_t)kVM * kVH * 2u;
    tc::mbar_arrive_expect_tx(hbar, hbytes);
    tc::bulk_load(base + kVoHs, p.hidden, hbytes, hbar);
  }
  for (int e = tid; e < kVE; e += kVThreads) bias_s[e] = p.bias != nullptr ? p.bias[e] : 0.0f;
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kVTmemCols);
    tc::tmem_relinquish();
  }
  // rows 12..15 of the hidden B tiles are zero: the last 512 bytes of each 2 KB tile
  for (int i = tid; i < kVNkh * 32; i += kVThreads)
    reinterpret_cast<uint4*>(hid + (size_t)(i / 32) * 2048 + 1536)[i % 32] = make_uint4(0, 0, 0, 0);
  tc::cluster_arrive();  // every CTA's barriers are initialised before anyone signals them

  // ---- the hidden rows (one bulk copy into the ring): codes per 128 columns into the B tiles
  // (row t of tile kb) and the scales. Warp w takes the (token, K block) groups w, w + 8, ...
  if (!tc::mbar_wait(hbar, 0)) ok = false;
  for (int g = warp; g < kVM * kVNkh; g += 8) {
    const int t = g / kVNkh, kb = g % kVNkh;
    const uint2 raw = *reinterpret_cast<const uint2*>(hs + t * kVH + kb * 128 + lane * 4);
    const float x0 = bf16_bits_to_float(raw.x & 0xFFFF), x1 = bf16_bits_to_float(raw.x >> 16);
    const float x2 = bf16_bits_to_float(raw.y & 0xFFFF), x3 = bf16_bits_to_float(raw.y >> 16);
    float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = quant_scale(amax);
    const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
    const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
    const uint32_t codes = lo | (hi << 16);
    *reinterpret_cast<uint32_t*>(hid + (size_t)kb * 2048 + sw128_off(t, lane >> 2) + (lane & 3) * 4) = codes;
    if (lane == 0) sa_s[t * kVNkh + kb] = sc;
    if (cid == 0 && rank == 0) {  // the workspace view of the hidden codes and scales
      reinterpret_cast<uint32_t*>(p.ws.qa + (size_t)t * kVH + kb * 128)[lane] = codes;
      if (lane == 0) p.ws.sa[t * kVNkh + kb] = sc;
    }
  }
  tc::fence_proxy_async_smem();  // generic writes of the B tiles before the tensor core reads them
  tc::fence_before_sync();       // the TMEM allocation's address, for every warp
  __syncthreads();
  tc::fence_after_sync();
  tc::cluster_wait();

  // ---- routing. Thread (e2, tq) runs the chains of experts 2*e2, 2*e2 + 1 for tokens tq,
  // tq + 4, tq + 8 over this CTA's chunk: one packed FP32x2 fma per token and k (two IEEE
  // fmas, bit-identical to separate ones)
  if (!tc::mbar_wait(rbar, 0)) ok = false;
  {
    const uint32_t* wr2 = reinterpret_cast<const uint32_t*>(ring);
    const int e2 = tid & 63, tq = tid >> 6;
    uint64_t acc[3] = {0ull, 0ull, 0ull};
#pragma unroll 8
    for (int k = 0; k < 128; ++k) {
      const uint32_t w = wr2[k * (kVE / 2) + e2];
      const uint64_t wp = tc::f2pack(w << 16, w & 0xFFFF0000u);  // bf16 -> f32: (expert 2e2, 2e2+1)
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const uint32_t xb = (uint32_t)hs[(tq + 4 * q) * kVH + rank * 128 + k] << 16;  // bf16 -> f32
        acc[q] = tc::f2fma(tc::f2pack(xb, xb), wp, acc[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      float a0, a1;
      tc::f2unpack(acc[q], a0, a1);
      own[(tq + 4 * q) * 128 + 2 * e2] = a0;
      own[(tq + 4 * q) * 128 + 2 * e2 + 1] = a1;
    }
  }
  tc::fence_proxy_async_smem();  // the partials are read by the copies below
  __syncthreads();
  if (tid < kVM)  // token tid's partials of chunk `rank` into CTA tid's slot `rank`
    tc::bulk_copy_cluster(tc::mapa(tc::smem_u32(part + (size_t)rank * 128), (uint32_t)tid), own + tid * 128, 512u,
                          tc::mapa(tc::smem_u32(part_full), (uint32_t)tid));
  if (rank < kVM) {
    // owner of token t = rank: chunk-order sums, bias, rank top-8, softmax weights
    const int t = rank;
    if (!tc::mbar_wait(part_full, 0)) ok = false;
    if (tid < kVE) {
      float l = 0.0f;
#pragma unroll
      for (int c = 0; c < kVNkh; ++c) l = __fadd_rn(l, part[c * 128 + tid]);
      if (p.bias != nullptr) l = __fadd_rn(l, bias_s[tid]);
      logits[tid] = l;
    }
    __syncthreads();
    {  // expert e = tid / 2: two threads count the larger logits (ties: lower index) in
       // one half of the experts each
      const int e = tid >> 1, half = tid & 1;
      const float v = logits[e];
      const float4* lt4 = reinterpret_cast<const float4*>(logits) + half * (kVE / 8);
      int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll 8
      for (int q = 0; q < kVE / 8; ++q) {
        const float4 w = lt4[q];
        const int ee = 4 * q + half * (kVE / 2);
        r0 += (w.x > v) || (w.x == v && ee < e);
        r1 += (w.y > v) || (w.y == v && ee + 1 < e);
        r2 += (w.z > v) || (w.z == v && ee + 2 < e);
        r3 += (w.w > v) || (w.w == v && ee + 3 < e);
      }
      int rk = r0 + r1 + r2 + r3;
      rk += __shfl_xor_sync(0xffffffffu, rk, 1);
      if (half == 0 && rk < kVK) {
        sel_v[rk] = v;
        sel_i[rk] = e;
      }
    }
    __syncthreads();
    if (warp == 0) {
      const float lmax = sel_v[0];
      float den = 0.0f;
      if (p.renorm) {
        for (int j = 0; j < kVK; ++j) den = __fadd_rn(den, expf(__fsub_rn(sel_v[j], lmax)));
      } else {
        for (int e = lane; e < kVE; e += 32) den = __fadd_rn(den, expf(__fsub_rn(logits[e], lmax)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, off));
      }
      if (lane < kVK) {
        const float w = __fdiv_rn(expf(__fsub_rn(sel_v[lane], lmax)), den);
        rst[lane] = (uint32_t)sel_i[lane];
        rst[kVK + lane] = __float_as_uint(w);
        if (cid == 0) {
          p.ids[t * kVK + lane] = sel_i[lane];
          p.wts[t * kVK + lane] = w;
        }
      }
      tc::fence_proxy_async_smem();  // read by the copies
      __syncwarp();
      if (lane < kVCL)  // the route into slot t of every CTA
        tc::bulk_copy_cluster(tc::mapa(tc::smem_u32(routes + t * 16), (uint32_t)lane), rst, 64u,
                              tc::mapa(tc::smem_u32(routes_full), (uint32_t)lane));
    }
  }
  if (!tc::mbar_wait(routes_full, 0)) ok = false;

  // ---- metadata: distinct experts ascending, their local index, each token's slot
  if (tid < kVE) used[tid] = 0;
  for (int i = tid; i < kVR * kVM / 4; i += kVThreads) reinterpret_cast<uint32_t*>(tslot)[i] = 0xFFFFFFFFu;
  __syncthreads();
  if (tid < kVR) used[routes[(tid / kVK) * 16 + tid % kVK]] = 1;  // ids are in [0, E)
  __syncthreads();
  if (tid < kVE) {
    const unsigned b = __ballot_sync(0xffffffffu, used[tid] != 0);
    if (lane == 0) wcnt[warp] = __popc(b);
  }
  __syncthreads();
  if (tid < kVE) {
    const unsigned b = __ballot_sync(0xffffffffu, used[tid] != 0);
    int pre = __popc(b & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) pre += wcnt[w];
    e2l[tid] = used[tid] ? pre : -1;
    if (used[tid]) dist[pre] = tid;
    if (tid == 0) wcnt[4] = wcnt[0] + wcnt[1] + wcnt[2] + wcnt[3];
  }
  __syncthreads();
  if (tid < kVR) {
    const int t = tid / kVK, j = tid % kVK;
    tslot[e2l[routes[t * 16 + j]] * kVM + t] = (int8_t)j;
    if (cid == 0 && rank == 0) {  // identity pair order for the reducer and the workspace views
      p.ws.perm_row[tid] = tid;
      p.ws.row_src[tid] = tid;
      p.ws.pair_expert[tid] = (int)routes[t * 16 + j];
    }
  }
  __syncthreads();
  const int n_dist = wcnt[4];
  const int ne = n_dist > cid ? (n_dist - 1 - cid) / p.nc + 1 : 0;  // this cluster's experts
  const int n_gu_all = ne * kVNu;
  const int n_gu = n_gu_all > rank ? (n_gu_all - 1 - rank) / kVCL + 1 : 0;  // my gate/up units
  const int n_pieces = n_gu * kVNkh + ne * (kVNu / 2);
  auto gu_unit = [&](int n, int& el, int& e, int& cb) {
    const int g = rank + kVCL * n;
    el = cid + (g / kVNu) * p.nc;
    e = dist[el];
    cb = g % kVNu;
  };
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA: lane L issues the pieces k = L, L + 4, ... into ring slot L: a gate/up piece is
    // one 3-D box (gate and up tiles of one K block), a down piece two 2-D boxes (two K blocks)
    if (lane < kVSlots) {
      tc::fence_proxy_async_smem();  // the routing reads of the ring precede these writes
      int last_use = -1;
      for (int k = lane; k < n_pieces && ok; k += kVSlots) {
        const int s = k % kVSlots, use = k / kVSlots;
        if (!tc::mbar_wait(&emptyp[s], (use & 1) ^ 1)) {
          ok = false;
          break;
        }
        unsigned char* dst = ring + (size_t)s * 2 * kVTile;
        last_use = use;
        tc::mbar_arrive_expect_tx(&fullp[s], 2 * kVTile);
        if (k < n_gu * kVNkh) {
          int el, e, cb;
          gu_unit(k / kVNkh, el, e, cb);
          tc::tma_load_3d(dst, &tm13, &fullp[s], (k % kVNkh) * 128, cb * 128, 2 * e);
        } else {
          const int kd = k - n_gu * kVNkh, ie = kd / (kVNu / 2), kb = 2 * (kd % (kVNu / 2));
          const int e = dist[cid + ie * p.nc];
          const int y = e * kVH + rank * 128;
          tc::tma_load_2d(dst, &tm2, &fullp[s], kb * 128, y);
          tc::tma_load_2d(dst + kVTile, &tm2, &fullp[s], (kb + 1) * 128, y);
        }
      }
      // no load of this lane is still writing when the CTA leaves (a no-op unless a wait gave up)
      if (last_use >= 0 && !tc::mbar_wait(&fullp[lane], last_use & 1)) ok = false;
    }
  } else if (warp == 1) {
    // ---- MMA issue in piece order: swap-AB 128 x 16 x 32 steps; gate/up into 32-column
    // buffers (gate 0..15, up 16..31), down into 16-column buffers from column 256
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3(128, 16);
      int ng = 0, nd = 0;
      for (int k = 0; k < n_pieces && ok; ++k) {
        const int s = k % kVSlots, use = k / kVSlots;
        const unsigned char* a = ring + (size_t)s * 2 * kVTile;
        if (k < n_gu * kVNkh) {
          const int kb = k % kVNkh, buf = ng & 7;
          if (!tc::mbar_wait(&fullp[s], use & 1) || !tc::mbar_wait(&acce[buf], ((ng >> 3) & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t d = tmem + buf * 32;
          const uint64_t db = tc::sdesc_sw128(tc::smem_u32(hid + (size_t)kb * 2048));
          const uint64_t dg = tc::sdesc_sw128(tc::smem_u32(a));
          const uint64_t du = tc::sdesc_sw128(tc::smem_u32(a + kVTile));
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::mma_e4m3(d, dg + 2 * q, db + 2 * q, idesc, q > 0);
#pragma unroll
          for (int q = 0; q < 4; ++q) tc::mma_e4m3(d + 16, du + 2 * q, db + 2 * q, idesc, q > 0);
          tc::mma_commit(&emptyp[s]);
          tc::mma_commit(&accf[buf]);
          ++ng;
        } else {
          const int kd = k - n_gu * kVNkh, ie = kd / (kVNu / 2), kp = kd % (kVNu / 2), ab = ie & 1;
          if (kp == 0 && !tc::mbar_wait(&act_ready[ab], (ie >> 1) & 1)) {
            ok = false;
            break;
          }
          if (!tc::mbar_wait(&fullp[s], use & 1)) {
            ok = false;
            break;
          }
          for (int h = 0; h < 2 && ok; ++h) {
            const int kb = 2 * kp + h, buf = nd & 7;
            if (!tc::mbar_wait(&acce2[buf], ((nd >> 3) & 1) ^ 1)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t d = tmem + 256 + buf * 16;
            const uint64_t db = tc::sdesc_sw128(tc::smem_u32(acttile + ((size_t)ab * kVNu + kb) * 2048));
            const uint64_t dw = tc::sdesc_sw128(tc::smem_u32(a + (size_t)h * kVTile));
#pragma unroll
            for (int q = 0; q < 4; ++q) tc::mma_e4m3(d, dw + 2 * q, db + 2 * q, idesc, q > 0);
            if (h == 1) {  // the slot and the expert's B tiles are read: released before the last
                           // accumulator, whose arrival the epilogue waits for
              tc::mma_commit(&emptyp[s]);
              if (kp == kVNu / 2 - 1) tc::mma_commit(&act_free[ab]);
            }
            tc::mma_commit(&accf2[buf]);
            ++nd;
          }
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
    for (int x = row; x < n_gu * kVNkh * 2; x += 128) {  // gate/up block scales of my units
      const int n = x / (kVNkh * 2), kb = (x / 2) % kVNkh, gu = x % 2;
      int el, e, cb;
      gu_unit(n, el, e, cb);
      sw13_s[x] = p.s13[((size_t)e * (2 * kVNu) + gu * kVNu + cb) * kVNkh + kb];
    }
    for (int x = row; x < ne * kVNu; x += 128) {  // down block scales of output block `rank`
      const int ie = x / kVNu, kb = x % kVNu;
      sw2_s[ie * 8 + kb] = p.s2w[((size_t)dist[cid + ie * p.nc] * kVNhb + rank) * kVNu + kb];
    }
    tc::named_bar(1, 128);
    int ng = 0, nd = 0;
    for (int n = 0; n < n_gu; ++n) {
      int el, e, cb;
      gu_unit(n, el, e, cb);
      float g[kVM], u[kVM];
#pragma unroll
      for (int t = 0; t < kVM; ++t) g[t] = u[t] = 0.0f;
      for (int kb = 0; kb < kVNkh; ++kb) {
        const int buf = ng & 7;
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&accf[buf], (ng >> 3) & 1));
        tc::fence_after_sync();
        float pg[16], pu[16];
        if (ok) {
          tc::tmem_ld16x2(tl + buf * 32, tl + buf * 32 + 16, pg, pu);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) pg[t] = pu[t] = 0.0f;
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[buf]);
        ++ng;
        const float swg = sw13_s[(n * kVNkh + kb) * 2], swu = sw13_s[(n * kVNkh + kb) * 2 + 1];
#pragma unroll
        for (int t = 0; t < kVM; ++t) {
          const float a = sa_s[t * kVNkh + kb];
          g[t] = __fadd_rn(g[t], __fmul_rn(pg[t], __fmul_rn(a, swg)));
          u[t] = __fadd_rn(u[t], __fmul_rn(pu[t], __fmul_rn(a, swu)));
        }
      }
      // silu(g) * u, then each routed token's 128 values requantised (amax over the 4 warps)
      float act[kVM];
#pragma unroll
      for (int t = 0; t < kVM; ++t) {
        act[t] = silu_mul(g[t], u[t]);
        float m = fabsf(act[t]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) red[q * 16 + t] = m;
      }
      tc::named_bar(1, 128);
#pragma unroll
      for (int t = 0; t < kVM; ++t) {
        const int j = tslot[el * kVM + t];
        if (j < 0) continue;
        const float amax = fmaxf(fmaxf(red[t], red[16 + t]), fmaxf(red[32 + t], red[48 + t]));
        const float s2 = quant_scale(amax);
        const int pr = t * kVK + j;
        p.ws.act[(size_t)pr * kVI + cb * 128 + row] = (uint8_t)(e4m3x2_encode(__fdiv_rn(act[t], s2), 0.0f) & 0xFF);
        if (row == 0) p.ws.act_scale[pr * kVNu + cb] = s2;
      }
      // every CTA of the cluster learns that this block of expert ie is written (red is
      // rewritten by the next unit only after this barrier too)
      __threadfence();
      tc::named_bar(1, 128);
      if (row < kVCL)
        tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(&eready[(rank + kVCL * n) / kVNu]), (uint32_t)row));
    }
    for (int ie = 0; ie < ne; ++ie) {
      const int el = cid + ie * p.nc, ab = ie & 1;
      if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&act_ready[ab], (ie >> 1) & 1));
      float y[kVM];
#pragma unroll
      for (int t = 0; t < kVM; ++t) y[t] = 0.0f;
      for (int kb = 0; kb < kVNu; ++kb) {
        const int buf = nd & 7;
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&accf2[buf], (nd >> 3) & 1));
        tc::fence_after_sync();
        float pd[16];
        if (ok) {
          tc::tmem_ld16(tl + 256 + buf * 16, pd);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) pd[t] = 0.0f;
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce2[buf]);
        ++nd;
        const float sw = sw2_s[ie * 8 + kb];
#pragma unroll
        for (int t = 0; t < kVM; ++t)
          y[t] = __fadd_rn(y[t], __fmul_rn(pd[t], __fmul_rn(asc_s[(ab * kVM + t) * 8 + kb], sw)));
      }
#pragma unroll
      for (int t = 0; t < kVM; ++t) {
        const int j = tslot[el * kVM + t];
        if (j >= 0) p.ws.y[(size_t)(t * kVK + j) * kVH + rank * 128 + row] = y[t];
      }
      tc::named_bar(1, 128);  // the expert's scales are no longer read
      if (row == 0) tc::mbar_arrive(&act_free[ab]);
    }
  } else {
    // ---- down B tiles: once the 6 activation blocks of expert ie are written (by whichever
    // CTAs of the cluster ran them), its routed activation rows (row t = token t's pair, other
    // rows 0) and scales; all loads of an expert are issued before its stores
    const int ht = tid - 192;  // 0..63
    constexpr int kPer = 16 * kVNu * 8 / 64;  // 16-byte chunks per thread and expert
    for (int ie = 0; ie < ne; ++ie) {
      const int el = cid + ie * p.nc, ab = ie & 1;
      if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait_cluster(&eready[ie], 0));
      if (ie >= 2 && ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&act_free[ab], ((ie - 2) >> 1) & 1));
      unsigned char* tiles = acttile + (size_t)ab * kVNu * 2048;
      uint4 v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {  // (row, K block, 16-byte chunk)
        const int x = ht + 64 * i, r = x / (kVNu * 8), kb = (x / 8) % kVNu, c = x % 8;
        const int j = r < kVM ? tslot[el * kVM + r] : -1;
        v[i] = make_uint4(0, 0, 0, 0);
        if (j >= 0) v[i] = __ldcg(reinterpret_cast<const uint4*>(p.ws.act + (size_t)(r * kVK + j) * kVI + kb * 128) + c);
      }
      float sv[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int x = ht + 64 * i, t = x / kVNu, kb = x % kVNu;
        const int j = x < kVM * kVNu ? tslot[el * kVM + t] : -1;
        sv[i] = j >= 0 ? __ldcg(p.ws.act_scale + (t * kVK + j) * kVNu + kb) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int x = ht + 64 * i, r = x / (kVNu * 8), kb = (x / 8) % kVNu, c = x % 8;
        *reinterpret_cast<uint4*>(tiles + (size_t)kb * 2048 + sw128_off(r, c)) = v[i];
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int x = ht + 64 * i, t = x / kVNu, kb = x % kVNu;
        if (x < kVM * kVNu) asc_s[(ab * kVM + t) * 8 + kb] = sv[i];
      }
      tc::fence_proxy_async_smem();  // generic writes of the B tiles before the tensor core reads them
      tc::named_bar(2, 64);
      if (ht == 0) tc::mbar_arrive(&act_ready[ab]);
    }
  }
  if (!ok) set_status(p.ws.hdr, MOE_STATUS_WAIT_TIMEOUT);
  __syncwarp();  // the cluster barrier below is warp-aligned: reconverge the role warps first
  // no CTA leaves while another may still signal it or copy into its shared memory
  tc::fence_before_sync();
  tc::cluster_arrive();
  tc::cluster_wait();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kVTmemCols);
  }
}

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
bool make_tmap_u8_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                     uint64_t s2, uint32_t b1, uint32_t b2);

namespace {

// Clusters resident at once with one CTA per SM (the occupancy query runs once per device).
int verify_clusters(const DeviceInfo& d) {
  static std::mutex mu;
  static int dev_of[64];
  static int nc_of[64];
  static int used = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (dev_of[i] == d.ordinal) return nc_of[i];
  int nc = 0;
  if (kVSmem <= d.smem_optin && kVSmem > d.smem_per_sm / 2) {
    cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVSmem);
    cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kVCL * 64, 1, 1);
    cfg.blockDim = dim3(kVThreads, 1, 1);
    cfg.dynamicSmemBytes = kVSmem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = kVCL;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&nc, verify_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      nc = 0;
    }
  }
  // every cluster must hold the experts it is dealt: at most kVMaxDn experts and kVMaxGU
  // gate/up units per CTA for up to 96 distinct experts
  const int need = (kVR + kVMaxDn - 1) / kVMaxDn;
  if (nc < need || ((kVR + nc - 1) / nc * kVNu + kVCL - 1) / kVCL > kVMaxGU) nc = 0;
  if (used < 64) {
    dev_of[used] = d.ordinal;
    nc_of[used] = nc;
    ++used;
  }
  return nc;
}

}  // namespace

bool verify_profile(int M, int H, int I, int E, int K) {
  return M == kVM && H == kVH && I == kVI && E == kVE && K == kVK;
}

bool verify_capable() {
  const DeviceInfo d = device_info();
  return d.sms > 0 && verify_clusters(d) > 0;
}

cudaError_t launch_verify_produce(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int renorm,
                                  int32_t* ids, float* wts, const uint8_t* w13, const float* s13, const uint8_t* w2,
                                  const float* s2w, const WsPtrs& ws, cudaStream_t st) {
  const DeviceInfo d = device_info();
  if (d.sms == 0) return cudaErrorInvalidDevice;
  const int nc = verify_clusters(d);
  if (nc == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap t13, t2;
  if (!make_tmap_u8_3d(&t13, w13, (uint64_t)kVH, (uint64_t)kVI, (uint64_t)kVE * 2, (uint64_t)kVH,
                       (uint64_t)kVI * kVH, 128, 2))
    return cudaErrorInvalidValue;
  if (!make_tmap_u8(&t2, w2, (uint64_t)kVI, (uint64_t)kVE * kVH, 128)) return cudaErrorInvalidValue;
  VerifyParams prm{};
  prm.renorm = renorm;
  prm.nc = nc;
  prm.hidden = hidden;
  prm.router_w = router_w;
  prm.bias = bias;
  prm.ids = ids;
  prm.wts = wts;
  prm.s13 = s13;
  prm.s2w = s2w;
  prm.ws = ws;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(kVCL * nc), 1, 1);
  cfg.blockDim = dim3(kVThreads, 1, 1);
  cfg.dynamicSmemBytes = kVSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kVCL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_kernel, t13, t2, prm);
}

}  // namespace moe
