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
// when one CTA owns all K blocks, otherwise every CTA of the cluster stores its terms into
// CTA 0's shared memory and CTA 0 runs the chain after one cluster barrier.
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
// scale into act_scale [p][I/128].
// Warp roles: warp 0 feeds the stages (TMA), warp 1 owns TMEM and issues MMAs, warps 2..5
// are the epilogue (TMEM lane quadrant = warp % 4). Every kernel waits on the previous
// kernel of the stream (griddepcontrol.wait) before touching global memory and then
// releases its dependents, so consecutive launches overlap their launch latency.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tc.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kPairN = 16;  // B rows per MMA (row 0 is the unit's pair)
constexpr int kMaxSplitTerms = 8;  // K blocks per CTA when a unit's K blocks are split
constexpr int kPairThreads = 192;

enum PairMode { kGateUpWs = 0, kGateUpFused = 1, kDownY = 2, kDownCombine = 3 };

template <int MODE>
struct PairCfg {
  static constexpr bool kGateUp = MODE == kGateUpWs || MODE == kGateUpFused;
  static constexpr int kATiles = kGateUp ? 2 : 1;
  static constexpr int kStages = kGateUp ? 2 : 4;
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = kPairN * 128;
  static constexpr int kStageBytes = ((kATiles * kABytes + kBBytes + 1023) / 1024) * 1024;
  static constexpr uint32_t kTxA = kATiles * kABytes;
  static constexpr int kAccCols = kATiles * kPairN;  // one K block's accumulators
  static constexpr int kTmemCols = 2 * kAccCols < 32 ? 32 : 2 * kAccCols;
};

struct PairParams {
  int H, I, K, E;
  int nkb, nkb_cta, ncb;   // K blocks total / per CTA; 128-row output blocks per unit
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
};

// Split-K terms [kATiles][nkb][128] f32 and combine rows [K][128] f32 are gathered in CTA
// 0's stage buffers once every CTA of the cluster has drained its pipeline, so they need
// no shared memory of their own (the host keeps kATiles * nkb * 512 and K * 512 bytes within
// the stage buffers).
template <int MODE>
struct PairSmem {
  size_t stages, bq, sas, bars, total;
};

template <int MODE>
__host__ __device__ inline PairSmem<MODE> pair_smem(int nkb, int nkb_cta, int K) {
  using C = PairCfg<MODE>;
  PairSmem<MODE> s{};
  (void)nkb;
  (void)K;
  size_t o = 0;
  s.stages = o; o += (size_t)C::kStages * C::kStageBytes;
  s.bq = o;  o += MODE == kGateUpFused ? (size_t)nkb_cta * 128 : 0;  // hidden codes
  s.sas = o; o += (size_t)nkb_cta * 4;                             // hidden scales
  o = (o + 15) & ~size_t(15);
  s.bars = o; o += 256;
  s.total = o + 1024;  // + alignment slack of the dynamic shared memory base
  return s;
}

template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 3)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const PairParams p) {
  using C = PairCfg<MODE>;
  constexpr bool kGateUp = C::kGateUp;
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const PairSmem<MODE> SL = pair_smem<MODE>(p.nkb, p.nkb_cta, p.K);
  unsigned char* stages = base + SL.stages;
  float* xterm = reinterpret_cast<float*>(stages);  // reused after the pipeline drains
  uint8_t* bq = base + SL.bq;
  float* sas = reinterpret_cast<float*>(base + SL.sas);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + SL.bars);
  uint64_t* full = bars;                        // [kStages]
  uint64_t* empty = bars + C::kStages;          // [kStages]
  uint64_t* accf = bars + 2 * C::kStages;       // [2]
  uint64_t* acce = bars + 2 * C::kStages + 2;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 4);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);  // [4] warp maxima

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int S = (int)cluster.num_blocks();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // set-up that touches no global memory overlaps the previous kernel's tail
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    if (MODE != kGateUpFused) tc::prefetch_tmap(&tmB);
    for (int s = 0; s < C::kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 4);
    }
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

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
  const int split = MODE == kDownCombine ? 1 : S;  // CTAs sharing one unit's K blocks
  const int kb0 = MODE == kDownCombine ? 0 : rank * p.nkb_cta;
  const int brow = MODE == kGateUpWs ? tok : pr;  // B row (qa row or act row)
  if (MODE == kGateUpFused) {
    // zero the B tiles (rows 1..15 stay zero) and quantise the pair's hidden row for this
    // CTA's K blocks (warp w takes blocks w, w+6, ...); independent of the expert id, so
    // these loads overlap the id load below
    for (int i = threadIdx.x; i < C::kStages * (C::kBBytes / 16); i += kPairThreads) {
      const int s = i / (C::kBBytes / 16), c = i % (C::kBBytes / 16);
      reinterpret_cast<uint4*>(stages + s * C::kStageBytes + C::kTxA)[c] = make_uint4(0, 0, 0, 0);
    }
    for (int i = warp; i < p.nkb_cta; i += kPairThreads / 32) {
      const uint2 raw = *reinterpret_cast<const uint2*>(p.hidden + (size_t)tok * p.H + (kb0 + i) * 128 + lane * 4);
      const float x0 = bf16_bits_to_float(raw.x & 0xFFFF), x1 = bf16_bits_to_float(raw.x >> 16);
      const float x2 = bf16_bits_to_float(raw.y & 0xFFFF), x3 = bf16_bits_to_float(raw.y >> 16);
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sc = quant_scale(amax);
      const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
      const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, sc), __fdiv_rn(x3, sc));
      reinterpret_cast<uint32_t*>(bq + i * 128)[lane] = lo | (hi << 16);
      if (lane == 0) sas[i] = sc;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else {
    for (int i = threadIdx.x; i < p.nkb_cta; i += kPairThreads) sas[i] = p.a_scale[(size_t)brow * p.nkb + kb0 + i];
  }
  const int e = p.ids[pr];
  const bool valid = e >= 0 && e < p.E;
  if (MODE == kGateUpFused && !valid && cb == 0 && rank == 0 && threadIdx.x == 0)
    set_status(p.hdr, MOE_STATUS_BAD_EXPERT_ID);
  // a skipped pair (not kDownCombine): the whole cluster shares the unit and leaves together
  const bool skip_unit = MODE != kDownCombine && !valid;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (skip_unit) {
    if (warp == 1) tc::tmem_dealloc(tmem, C::kTmemCols);
    return;
  }

  bool ok = true;
  float chain0 = 0.0f, chain1 = 0.0f;
  float term0[kMaxSplitTerms], term1[kMaxSplitTerms];
  if (valid && warp == 0) {
    const int yA0 = kGateUp ? e * 2 * p.I + cb * 128 : e * p.H + cb * 128;
    const int yA1 = e * 2 * p.I + p.I + cb * 128;
    for (int i = 0; i < p.nkb_cta; ++i) {
      const int s = i % C::kStages;
      const uint32_t ph = (i / C::kStages) & 1;
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
        tc::tma_load_2d(st, &tmA, &full[s], x, yA0);
        if (kGateUp) tc::tma_load_2d(st + C::kABytes, &tmA, &full[s], x, yA1);
        if (MODE != kGateUpFused) tc::tma_load_2d(st + C::kTxA, &tmB, &full[s], x, brow);
      }
    }
  } else if (valid && warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3(128, kPairN);
      for (int i = 0; i < p.nkb_cta; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
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
    }
  } else if (valid) {
    // epilogue: thread <-> weight row (warp % 4) * 32 + lane of the 128-row tile
    const int q = warp & 3;
    const float* sw0 = p.w_scale + ((size_t)e * (kGateUp ? 2 * p.I / 128 : p.H / 128) + cb) * p.nkb;
    const float* sw1 = p.w_scale + ((size_t)e * (2 * p.I / 128) + p.I / 128 + cb) * p.nkb;
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
      const int kb = kb0 + i;
      const float a = sas[i];
      const float t0 = __fmul_rn(v0[0], __fmul_rn(a, sw0[kb]));
      const float t1 = kGateUp ? __fmul_rn(v1[0], __fmul_rn(a, sw1[kb])) : 0.0f;
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
  if (!ok) set_status(p.hdr, MOE_STATUS_WAIT_TIMEOUT);
  __syncthreads();
  if (split > 1 || MODE == kDownCombine) {
    cluster.sync();  // every CTA's pipeline has drained: CTA 0's stage buffers are free
    if (valid && warp >= 2) {
      const int r = (warp & 3) * 32 + lane;
      float* x0 = cluster.map_shared_rank(xterm, 0);
      if (MODE == kDownCombine) {
        x0[rank * 128 + r] = chain0;
      } else {
#pragma unroll
        for (int j = 0; j < kMaxSplitTerms; ++j) {
          if (j < p.nkb_cta) {
            x0[(kb0 + j) * 128 + r] = term0[j];
            if (kGateUp) x0[(p.nkb + kb0 + j) * 128 + r] = term1[j];
          }
        }
      }
    }
    cluster.sync();  // CTA 0 holds every term / row
  }

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
        const int ej = p.ids[tok * p.K + j];
        if (ej < 0 || ej >= p.E) continue;
        acc = __fadd_rn(acc, __fmul_rn(p.topk_w[tok * p.K + j], xterm[j * 128 + r]));
      }
      p.out[(size_t)tok * p.H + cb * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    }
  }
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
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

constexpr int kNumSMs = 152;
constexpr size_t kSmemPerSM = 228 * 1024;

// Largest divisor S of nkb (S <= 8, the cluster size) such that units * S CTAs fit in one
// wave at the occupancy their shared memory allows; at least 1.
template <int MODE>
int pick_split(int nkb, int64_t units, int K) {
  int best = 1;
  for (int s = 1; s <= 8; ++s) {
    if (nkb % s) continue;
    if (s > 1 && (nkb / s > kMaxSplitTerms ||
                  (size_t)PairCfg<MODE>::kATiles * nkb * 512 > (size_t)PairCfg<MODE>::kStages * PairCfg<MODE>::kStageBytes))
      continue;
    const size_t smem = pair_smem<MODE>(nkb, nkb / s, K).total + 1024;
    const int64_t wave = (int64_t)kNumSMs * (int64_t)(kSmemPerSM / smem);
    if (units * s <= wave) best = s;
  }
  return best;
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& tA, const CUtensorMap& tB, PairParams prm, int cluster_x,
                        int64_t units, cudaStream_t st) {
  const PairSmem<MODE> SL = pair_smem<MODE>(prm.nkb, prm.nkb_cta, prm.K);
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(pair_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(pair_gemm_kernel<MODE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
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
// the prepared codes ws.qa / ws.sa and ids = ws.pair_expert.
cudaError_t launch_pair_gateup(const uint8_t* w13, const float* s13, const int32_t* ids,
                               const uint16_t* hidden, int M, int H, int I, int E, int K,
                               const WsPtrs& ws, cudaStream_t st) {
  CUtensorMap tA, tB;
  if (!make_tmap_u8(&tA, w13, (uint64_t)H, (uint64_t)E * 2 * I, 128)) return cudaErrorInvalidValue;
  PairParams prm = base_params(M, H, I, E, K, ws);
  prm.nkb = H / 128;
  prm.ncb = I / 128;
  prm.ids = ids;
  prm.w_scale = s13;
  prm.a_scale = ws.sa;
  prm.hidden = hidden;
  const int64_t units = (int64_t)M * K * prm.ncb;
  const int S = hidden ? pick_split<kGateUpFused>(prm.nkb, units, K) : pick_split<kGateUpWs>(prm.nkb, units, K);
  prm.nkb_cta = prm.nkb / S;
  if (hidden) {
    tB = tA;  // unused: the B tile is written by the kernel
    return launch_pair<kGateUpFused>(tA, tB, prm, S, units, st);
  }
  if (!make_tmap_u8(&tB, ws.qa, (uint64_t)H, (uint64_t)M, kPairN)) return cudaErrorInvalidValue;
  return launch_pair<kGateUpWs>(tA, tB, prm, S, units, st);
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
    return launch_pair<kDownCombine>(tA, tB, prm, K, (int64_t)M * prm.ncb, st);
  }
  const int64_t units = (int64_t)R * prm.ncb;
  const int S = pick_split<kDownY>(prm.nkb, units, K);
  prm.nkb_cta = prm.nkb / S;
  return launch_pair<kDownY>(tA, tB, prm, S, units, st);
}

}  // namespace moe
