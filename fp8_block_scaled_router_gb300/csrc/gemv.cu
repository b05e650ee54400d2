// gemv.cu -- block-scaled grouped GEMV on CUDA cores (expert-sorted tiles of <= 16 rows).
//
// Sources: docs/compiler/architecture.md, accepted M=1 MoE objects (gate/up, SiLU+quant,
// down/reduce); "NetraRuntime/netra-kernel" older lab README, supported-targets table
// (FP8 E4M3 weights with 128x128 block scales).
//
// Each CTA owns 32 weight rows of one expert and one tile of routed rows (tokens). For a
// K chunk of four 128-blocks, 256 threads (row r, block kbl, half) form 64-term FP32 dot
// products for every routed row of the tile; the two halves are added (lo + hi) to give
// the block sum P. Threads (r, m) then advance the promotion chain
//   acc = acc + P * (sa[kb] * sw[kb])      kb ascending, FP32 mul and add, from 0
// so the chain has the same order as the block-scaled GEMM's definition.
// gate/up: a cluster of 8 CTAs covers one 128-column activation block (16 gate + 16 up
// rows each); SiLU(g)*u stays in shared memory, the 8 local amax values are exchanged over
// distributed shared memory, and each CTA writes its 16 FP8 codes (scale = amax/448).
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kRows = 32;     // weight rows per CTA
constexpr int kChunk = 512;   // K bytes per chunk (four 128-blocks)

template <int TM>
struct GemvShared {
  float hs[TM][kChunk];               // activation chunk, decoded
  float part[2][4][kRows][TM];        // half-block dot products
  float chain[kRows][TM];             // promotion chains
  const uint8_t* wrow[kRows];
  const float* wsc[kRows];
  const uint8_t* arow[TM];
  const float* asc[TM];
};

template <int TM>
__device__ void scaled_rows_tile(GemvShared<TM>& sh, int nrows, int Kdim) {
  const int tid = threadIdx.x;
  for (int i = tid; i < kRows * TM; i += blockDim.x) (&sh.chain[0][0])[i] = 0.0f;
  for (int k0 = 0; k0 < Kdim; k0 += kChunk) {
    const int ckb = min(4, (Kdim - k0) / 128);
    // decode the activation chunk: TM rows x ckb*128 codes
    for (int i = tid; i < nrows * (ckb * 128 / 16); i += blockDim.x) {
      const int m = i / (ckb * 8), c16 = i % (ckb * 8);
      const uint4 raw = *reinterpret_cast<const uint4*>(sh.arow[m] + k0 + c16 * 16);
      const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
      float* dst = &sh.hs[m][c16 * 16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 a = e4m3x2_decode((uint16_t)(wv[q] & 0xFFFF));
        const float2 b = e4m3x2_decode((uint16_t)(wv[q] >> 16));
        *reinterpret_cast<float4*>(dst + q * 4) = make_float4(a.x, a.y, b.x, b.y);
      }
    }
    __syncthreads();
    {
      const int r = tid & 31, kbl = (tid >> 5) & 3, half = tid >> 7;
      if (kbl < ckb) {
        const uint8_t* wp = sh.wrow[r] + k0 + kbl * 128 + half * 64;
        float acc[TM];
#pragma unroll
        for (int m = 0; m < TM; ++m) acc[m] = 0.0f;
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(wp + piece * 16));
          const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
          float w[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 a = e4m3x2_decode((uint16_t)(wv[q] & 0xFFFF));
            const float2 b = e4m3x2_decode((uint16_t)(wv[q] >> 16));
            w[4 * q] = a.x; w[4 * q + 1] = a.y; w[4 * q + 2] = b.x; w[4 * q + 3] = b.y;
          }
          const int kk = kbl * 128 + half * 64 + piece * 16;
#pragma unroll
          for (int m = 0; m < TM; ++m) {
            if (m < nrows) {
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 h = *reinterpret_cast<const float4*>(&sh.hs[m][kk + i]);
                acc[m] = __fmaf_rn(w[i], h.x, acc[m]);
                acc[m] = __fmaf_rn(w[i + 1], h.y, acc[m]);
                acc[m] = __fmaf_rn(w[i + 2], h.z, acc[m]);
                acc[m] = __fmaf_rn(w[i + 3], h.w, acc[m]);
              }
            }
          }
        }
#pragma unroll
        for (int m = 0; m < TM; ++m)
          if (m < nrows) sh.part[half][kbl][r][m] = acc[m];
      }
    }
    __syncthreads();
    for (int i = tid; i < kRows * nrows; i += blockDim.x) {
      const int r = i & 31, m = i >> 5;
      float c = sh.chain[r][m];
      for (int kbl = 0; kbl < ckb; ++kbl) {
        const int kb = k0 / 128 + kbl;
        const float p = __fadd_rn(sh.part[0][kbl][r][m], sh.part[1][kbl][r][m]);
        const float sc = __fmul_rn(sh.asc[m][kb], sh.wsc[r][kb]);
        c = __fadd_rn(c, __fmul_rn(p, sc));
      }
      sh.chain[r][m] = c;
    }
    __syncthreads();
  }
}

template <int TM>
__global__ void __cluster_dims__(8, 1, 1) __launch_bounds__(256)
    gateup_gemv_kernel(const uint8_t* __restrict__ w13, const float* __restrict__ s13, int H,
                       int I, int K, WsPtrs ws) {
  extern __shared__ __align__(16) unsigned char dsm[];
  GemvShared<TM>& sh = *reinterpret_cast<GemvShared<TM>*>(dsm);
  __shared__ float actv[TM][16];
  __shared__ float amax_loc[TM];
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned tile_idx = blockIdx.y;
  if (tile_idx >= ws.hdr->n_tiles) return;  // uniform over the cluster (same tile)
  const int q = (int)cluster.block_rank(), cb = blockIdx.x / 8;
  const Tile tl = ws.tiles[tile_idx];
  const int e = tl.expert, row0 = tl.row0, nrows = tl.nrows;
  const int tid = threadIdx.x;
  const int nkh = H / 128;
  if (tid < kRows) {
    const int n = (tid < 16 ? 0 : I) + cb * 128 + q * 16 + (tid & 15);
    sh.wrow[tid] = w13 + ((size_t)e * 2 * I + n) * H;
    sh.wsc[tid] = s13 + ((size_t)e * (2 * I / 128) + n / 128) * nkh;
  } else if (tid >= 64 && tid < 64 + TM) {
    const int m = tid - 64;
    if (m < nrows) {
      const int t = ws.row_src[row0 + m] / K;
      sh.arow[m] = ws.qa + (size_t)t * H;
      sh.asc[m] = ws.sa + (size_t)t * nkh;
    }
  }
  __syncthreads();
  scaled_rows_tile<TM>(sh, nrows, H);
  for (int i = tid; i < 16 * nrows; i += blockDim.x) {
    const int c = i & 15, m = i >> 4;
    actv[m][c] = silu_mul(sh.chain[c][m], sh.chain[16 + c][m]);
  }
  __syncthreads();
  if (tid < nrows) {
    float a = 0.0f;
    for (int c = 0; c < 16; ++c) a = fmaxf(a, fabsf(actv[tid][c]));
    amax_loc[tid] = a;
  }
  cluster.sync();
  for (int i = tid; i < 16 * nrows; i += blockDim.x) {
    const int c = i & 15, m = i >> 4;
    float a = 0.0f;
    for (int r = 0; r < 8; ++r) a = fmaxf(a, cluster.map_shared_rank(amax_loc, r)[m]);
    const float s = quant_scale(a);
    const float2 v = make_float2(__fdiv_rn(actv[m][c], s), 0.0f);
    ws.act[(size_t)(row0 + m) * I + cb * 128 + q * 16 + c] =
        (uint8_t)(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3) & 0xFF);
    if (q == 0 && c == 0) ws.act_scale[(size_t)(row0 + m) * (I / 128) + cb] = s;
  }
  cluster.sync();  // no CTA leaves while another may still read its amax_loc
}

template <int TM>
__global__ void __launch_bounds__(256)
    down_gemv_kernel(const uint8_t* __restrict__ w2, const float* __restrict__ s2w, int H, int I,
                     WsPtrs ws) {
  extern __shared__ __align__(16) unsigned char dsm[];
  GemvShared<TM>& sh = *reinterpret_cast<GemvShared<TM>*>(dsm);
  const unsigned tile_idx = blockIdx.y;
  if (tile_idx >= ws.hdr->n_tiles) return;
  const Tile tl = ws.tiles[tile_idx];
  const int e = tl.expert, row0 = tl.row0, nrows = tl.nrows;
  const int tid = threadIdx.x;
  const int h0 = blockIdx.x * kRows;
  const int nki = I / 128;
  if (tid < kRows) {
    const int h = h0 + tid;
    sh.wrow[tid] = w2 + ((size_t)e * H + h) * I;
    sh.wsc[tid] = s2w + ((size_t)e * (H / 128) + h / 128) * nki;
  } else if (tid >= 64 && tid < 64 + TM) {
    const int m = tid - 64;
    if (m < nrows) {
      sh.arow[m] = ws.act + (size_t)(row0 + m) * I;
      sh.asc[m] = ws.act_scale + (size_t)(row0 + m) * nki;
    }
  }
  __syncthreads();
  scaled_rows_tile<TM>(sh, nrows, I);
  for (int i = tid; i < kRows * nrows; i += blockDim.x) {
    const int r = i & 31, m = i >> 5;
    ws.y[(size_t)(row0 + m) * H + h0 + r] = sh.chain[r][m];
  }
}

cudaError_t launch_gateup_gemv(const uint8_t* w13, const float* s13, int H, int I, int K,
                               int64_t max_tiles, const WsPtrs& ws, cudaStream_t st) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(gateup_gemv_kernel<kTileRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(GemvShared<kTileRows>));
  });
  dim3 grid(8 * (I / 128), (unsigned)max_tiles);
  gateup_gemv_kernel<kTileRows><<<grid, 256, sizeof(GemvShared<kTileRows>), st>>>(w13, s13, H, I, K, ws);
  return cudaGetLastError();
}

cudaError_t launch_down_gemv(const uint8_t* w2, const float* s2w, int H, int I, int64_t max_tiles,
                             const WsPtrs& ws, cudaStream_t st) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(down_gemv_kernel<kTileRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(GemvShared<kTileRows>));
  });
  dim3 grid(H / kRows, (unsigned)max_tiles);
  down_gemv_kernel<kTileRows><<<grid, 256, sizeof(GemvShared<kTileRows>), st>>>(w2, s2w, H, I, ws);
  return cudaGetLastError();
}

}  // namespace moe
