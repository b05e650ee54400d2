// tc_pair.cu -- block-scaled expert GEMMs on tcgen05 for few routed rows (decode, verify,
// wide-expert sweeps): one unit per routed (token, slot) pair.
//
// Sources: docs/compiler/architecture.md, accepted M=1 MoE objects (gate/up, SiLU+quant,
// down/reduce; FP8 activation plus activation-scale intermediates); "NetraRuntime/
// netra-kernel" older lab README, supported-targets table (FP8 E4M3 weights with 128x128
// FP32 block scales); "Inferact/amd-kernels" README (split-K partials summed in a fixed
// order, never with atomics).
//
// Shape of the work. A unit is (pair p, 128-row block of the output). The 128 weight rows
// are the MMA's M operand; the pair's quantised activation row is the first of N=16 B rows
// (the other rows are neighbours' rows and are ignored), so D = W_tile * x^T lands in
// TMEM with one weight row per lane. A thread-block cluster of S CTAs splits the unit's
// 128-wide K blocks; each CTA streams its blocks with TMA (128-byte swizzle) through a
// two-stage ring, issues four 128x16x32 FP8 MMAs per block into a fresh accumulator
// (double-buffered in TMEM), and its epilogue warps read the block sum P back with
// tcgen05.ld and form the promoted term t_kb = P * (sa_kb * sw_kb). CTA 0 then reads every
// CTA's terms over distributed shared memory and adds them in ascending kb order, FP32,
// from 0 -- exactly the promotion chain of the block-scaled GEMM.
//   gate/up: A tiles are gate rows [cb*128, +128) and up rows [I + cb*128, +128) of w13[e];
//            CTA 0 forms act = silu(g) * u per row, the block amax over the 128 rows
//            (warp max + shared memory), scale = amax/448 and RNE saturating E4M3 codes.
//   down:    A tile is rows [cb*128, +128) of w2[e]; CTA 0 writes y[p][cb*128 + r].
// Warp roles: warp 0 issues TMA, warp 1 owns TMEM and issues MMAs, warps 2..5 are the
// epilogue (TMEM lane quadrant = warp % 4).
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tc.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kPairN = 16;        // B rows per MMA (only row 0 is the unit's pair)
constexpr int kPairStages = 2;
constexpr int kPairThreads = 192;

template <bool GATEUP>
struct PairCfg {
  static constexpr int kATiles = GATEUP ? 2 : 1;
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = kPairN * 128;
  static constexpr int kStageBytes = ((kATiles * kABytes + kBBytes + 1023) / 1024) * 1024;
  static constexpr uint32_t kTx = kATiles * kABytes + kBBytes;
  static constexpr int kAccCols = kATiles * kPairN;       // one K block's accumulators
  static constexpr int kTmemCols = 2 * kAccCols < 32 ? 32 : 2 * kAccCols;
};

struct PairParams {
  int H, I, K;
  int nkb, nkb_cta, ncb;   // K blocks total / per CTA; output 128-row blocks per unit
  int tok_rows;            // rows of the B matrix (M for gate/up, R for down)
  const int32_t* ids;      // [R]
  int E;
  const float* w_scale;    // s13 [E][2I/128][H/128] or s2w [E][H/128][I/128]
  const float* a_scale;    // sa [M][H/128] (gate/up) or act_scale [R][I/128] (down)
  uint8_t* act_out;        // [R][I]
  float* act_scale_out;    // [R][I/128]
  float* y_out;            // [R][H]
  Header* hdr;
};

__host__ __device__ inline size_t pair_smem_bytes(int stage_bytes, int nkb_cta, int S) {
  // 1024 alignment slack + stages + exchange terms (2 x nkb_cta x 128 floats, split K
  // only) + barriers
  return 1024 + (size_t)kPairStages * stage_bytes + (S > 1 ? (size_t)2 * nkb_cta * 128 * 4 : 0) + 256;
}

template <bool GATEUP>
__global__ void __launch_bounds__(kPairThreads)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const PairParams p) {
  using C = PairCfg<GATEUP>;
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int S = (int)cluster.num_blocks();
  float* xterm = reinterpret_cast<float*>(base + kPairStages * C::kStageBytes);  // [2][nkb_cta][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(xterm + (S > 1 ? 2 * p.nkb_cta * 128 : 0));
  uint64_t* full = bars;                         // [kPairStages]
  uint64_t* empty = bars + kPairStages;          // [kPairStages]
  uint64_t* accf = bars + 2 * kPairStages;       // [2]
  uint64_t* acce = bars + 2 * kPairStages + 2;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kPairStages + 4);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);  // [4] warp maxima

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int unit = blockIdx.y;
  const int pr = unit / p.ncb, cb = unit % p.ncb;
  const int e = p.ids[pr];
  if (e < 0 || e >= p.E) return;  // skipped pair: the whole cluster leaves together
  const int kb0 = rank * p.nkb_cta;
  const int brow = GATEUP ? pr / p.K : pr;

  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
    for (int s = 0; s < kPairStages; ++s) {
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
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  float chain_g = 0.0f, chain_u = 0.0f;
  if (warp == 0) {
    if (lane == 0) {
      const int yA0 = GATEUP ? e * 2 * p.I + cb * 128 : e * p.H + cb * 128;
      const int yA1 = e * 2 * p.I + p.I + cb * 128;
      for (int i = 0; i < p.nkb_cta && ok; ++i) {
        const int s = i % kPairStages;
        const uint32_t ph = (i / kPairStages) & 1;
        if (!tc::mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
        unsigned char* st = stages + s * C::kStageBytes;
        tc::mbar_arrive_expect_tx(&full[s], C::kTx);
        const int x = (kb0 + i) * 128;
        tc::tma_load_2d(st, &tmA, &full[s], x, yA0);
        if (GATEUP) tc::tma_load_2d(st + C::kABytes, &tmA, &full[s], x, yA1);
        tc::tma_load_2d(st + C::kATiles * C::kABytes, &tmB, &full[s], x, brow);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3(128, kPairN);
      for (int i = 0; i < p.nkb_cta && ok; ++i) {
        const int s = i % kPairStages;
        const uint32_t ph = (i / kPairStages) & 1;
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
        for (int k = 0; k < 4; ++k) {
          tc::mma_e4m3(d, da0 + 2 * k, db + 2 * k, idesc, k > 0);
          if (GATEUP) tc::mma_e4m3(d + kPairN, da1 + 2 * k, db + 2 * k, idesc, k > 0);
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&accf[buf]);
      }
    }
  } else {
    // epilogue: thread <-> weight row r of the 128-row tile
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int nkh = p.nkb;  // K blocks of the weight rows' scale grid
    const float* sw0 = p.w_scale + ((size_t)e * (GATEUP ? 2 * p.I / 128 : p.H / 128) + cb) * nkh;
    const float* sw1 = p.w_scale + ((size_t)e * (2 * p.I / 128) + p.I / 128 + cb) * nkh;
    const float* sa = p.a_scale + (size_t)brow * p.nkb;
    for (int i = 0; i < p.nkb_cta; ++i) {
      const int buf = i & 1;
      if (!tc::mbar_wait(&accf[buf], (i >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * C::kAccCols;
      float v0[16], v1[16];
      tc::tmem_ld16(ta, v0);
      if (GATEUP) tc::tmem_ld16(ta + kPairN, v1);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acce[buf]);
      const int kb = kb0 + i;
      const float a = sa[kb];
      const float tg = __fmul_rn(v0[0], __fmul_rn(a, sw0[kb]));
      const float tu = GATEUP ? __fmul_rn(v1[0], __fmul_rn(a, sw1[kb])) : 0.0f;
      if (S == 1) {  // the whole chain is local: kb ascending
        chain_g = __fadd_rn(chain_g, tg);
        if (GATEUP) chain_u = __fadd_rn(chain_u, tu);
      } else {
        xterm[i * 128 + r] = tg;
        if (GATEUP) xterm[(p.nkb_cta + i) * 128 + r] = tu;
      }
    }
  }
  if (!ok) set_status(p.hdr, MOE_STATUS_WAIT_TIMEOUT);
  __syncthreads();
  if (S > 1) cluster.sync();  // every CTA's promoted terms are in its shared memory

  if (rank == 0 && warp >= 2) {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    float g = chain_g, u = chain_u;
    if (S > 1) {
      g = 0.0f;
      u = 0.0f;
      for (int kb = 0; kb < p.nkb; ++kb) {
        const float* src = cluster.map_shared_rank(xterm, kb / p.nkb_cta);
        const int i = kb % p.nkb_cta;
        g = __fadd_rn(g, src[i * 128 + r]);
        if (GATEUP) u = __fadd_rn(u, src[(p.nkb_cta + i) * 128 + r]);
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
      p.y_out[(size_t)pr * p.H + cb * 128 + r] = g;
    }
  }
  if (S > 1) cluster.sync();  // CTA 0 has finished reading the other CTAs' terms
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

// Largest divisor S of nkb (S <= 8, cluster size) such that units * S fits one wave of
// three CTAs per SM; at least 1.
int pick_split(int nkb, int64_t units) {
  const int64_t wave = 3 * 152;
  int best = 1;
  for (int s = 1; s <= 8; ++s)
    if (nkb % s == 0 && units * s <= wave) best = s;
  return best;
}

template <bool GATEUP>
cudaError_t launch_pair(const CUtensorMap& tA, const CUtensorMap& tB, PairParams prm, int64_t units,
                        cudaStream_t st) {
  using C = PairCfg<GATEUP>;
  const int S = pick_split(prm.nkb, units);
  prm.nkb_cta = prm.nkb / S;
  const size_t smem = pair_smem_bytes(C::kStageBytes, prm.nkb_cta, S);
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(pair_gemm_kernel<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(pair_gemm_kernel<GATEUP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, (unsigned)units, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<GATEUP>, tA, tB, prm);
}

}  // namespace

// gate/up for R = M*K pairs: act [R][I] + act_scale [R][I/128] in pair order.
cudaError_t launch_pair_gateup(const uint8_t* w13, const float* s13, const int32_t* ids, int M, int H,
                               int I, int E, int K, const WsPtrs& ws, cudaStream_t st) {
  CUtensorMap tA, tB;
  if (!make_tmap_u8(&tA, w13, (uint64_t)H, (uint64_t)E * 2 * I, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tB, ws.qa, (uint64_t)H, (uint64_t)M, kPairN)) return cudaErrorInvalidValue;
  PairParams prm{};
  prm.H = H; prm.I = I; prm.K = K; prm.E = E;
  prm.nkb = H / 128; prm.ncb = I / 128; prm.tok_rows = M;
  prm.ids = ids; prm.w_scale = s13; prm.a_scale = ws.sa;
  prm.act_out = ws.act; prm.act_scale_out = ws.act_scale; prm.y_out = ws.y; prm.hdr = ws.hdr;
  return launch_pair<true>(tA, tB, prm, (int64_t)M * K * prm.ncb, st);
}

// down for R pairs: y [R][H] in pair order.
cudaError_t launch_pair_down(const uint8_t* w2, const float* s2w, const int32_t* ids, int M, int H, int I,
                             int E, int K, const WsPtrs& ws, cudaStream_t st) {
  CUtensorMap tA, tB;
  const int R = M * K;
  if (!make_tmap_u8(&tA, w2, (uint64_t)I, (uint64_t)E * H, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tB, ws.act, (uint64_t)I, (uint64_t)R, kPairN)) return cudaErrorInvalidValue;
  PairParams prm{};
  prm.H = H; prm.I = I; prm.K = K; prm.E = E;
  prm.nkb = I / 128; prm.ncb = H / 128; prm.tok_rows = R;
  prm.ids = ids; prm.w_scale = s2w; prm.a_scale = ws.act_scale;
  prm.act_out = ws.act; prm.act_scale_out = ws.act_scale; prm.y_out = ws.y; prm.hdr = ws.hdr;
  return launch_pair<false>(tA, tB, prm, (int64_t)R * prm.ncb, st);
}

}  // namespace moe
