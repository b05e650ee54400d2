// common.cuh -- device helpers and the workspace layout shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_fp8.h"

namespace moe {

constexpr int kBlock = 128;  // block-scale grid: 128x128 for weights, 1x128 for activations

// --------------------------------------------------------------------------------------
// Workspace layout (caller-owned, sized for max_tokens). Every region starts on a 256-byte
// boundary. R = max_tokens * K routed rows.
// --------------------------------------------------------------------------------------
struct Header {             // first 256 bytes
  uint32_t status;          // MOE_STATUS_* bits, cleared by moe_fp8_workspace_init
  uint32_t n_tiles;         // tiles written by the last prepare
  uint32_t n_groups;        // groups of up to kGroupRows rows written by the last prepare
  uint32_t pad[61];
};

struct Tile {               // a run of up to `tile_rows` expert-sorted rows of one expert
  int32_t expert;
  int32_t row0;
  int32_t nrows;
  int32_t pad;
};

struct Layout {
  size_t header, tickets, qa, sa, offsets, row_src, perm_row, pair_expert, blk_counts, tiles, groups, xp, sa_p,
      act, act_scale, y, yt;
  size_t hid_stage, out_stage, ids_stage, wts_stage;  // host-buffer calls: device copies
  size_t total;
  int64_t R, max_tiles, max_groups;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Tokens per call that the single-launch path takes (its arrival tickets, one per token and
// 128-column block, sit right after the header and are cleared with it).
constexpr int kTicketTokens = 16;

// Routed rows per tile of the grouped GEMMs (the MMA's M).
constexpr int kTileRows = 128;

// Routed rows per group of the expert-grouped pair kernels (the MMA's N).
constexpr int kGroupRows = 16;

// Routed pairs per block of the multi-block counting sort.
constexpr int kSortBlock = 256;

// Pair mode: every (token, slot) pair is its own GEMM unit -- no sort, but the weights of
// an expert chosen by several pairs are re-read once per pair. The pair kernels take up to
// kPairMaxRows routed rows (M*K); the layer uses them up to kPairPreferRows, above which
// sorting the rows into expert tiles (each expert's weights read once per 128 rows) was
// measured faster on every shape tried (h2048/i768/e128/top8 and h6144/i768/e128/top4).
constexpr int kPairMaxRows = 256;
constexpr int kPairPreferRows = 64;
inline bool pair_capable(int64_t R) { return R <= kPairMaxRows; }
inline bool use_pair_mode(int64_t R) { return R <= kPairPreferRows; }

// Above kPairPreferRows and up to kGroupMaxRows routed rows the layer sorts the rows and runs
// the expert-grouped pair kernels (each expert's weights read once per 16 of its rows);
// above that, the grouped GEMM over 128-row tiles.
constexpr int kGroupMaxRows = 256;
inline bool use_group_mode(int64_t R) { return R > kPairPreferRows && R <= kGroupMaxRows; }

inline int64_t max_tiles_for(int64_t R, int E, int tile_rows) {
  // sum over experts of ceil(n_e / tile_rows) <= R / tile_rows + (non-empty experts)
  return R / tile_rows + (R < E ? R : E) + 1;
}

inline Layout make_layout(const moe_fp8_shape_t& s) {
  Layout L{};
  const int64_t H = s.hidden, I = s.inter, E = s.num_experts, K = s.top_k, Mx = s.max_tokens;
  L.R = Mx * K;
  L.max_tiles = max_tiles_for(L.R, (int)E, kTileRows);
  L.max_groups = max_tiles_for(L.R, (int)E, kGroupRows);
  size_t o = 0;
  L.header = o;    o = align256(o + sizeof(Header));
  L.tickets = o;   o = align256(o + (size_t)(Mx < kTicketTokens ? Mx : kTicketTokens) * (H / kBlock) * 4);
  L.qa = o;        o = align256(o + (size_t)(Mx * H));
  L.sa = o;        o = align256(o + (size_t)(Mx * (H / kBlock)) * 4);
  L.offsets = o;   o = align256(o + (size_t)(E + 1) * 4);
  L.row_src = o;   o = align256(o + (size_t)L.R * 4);
  L.perm_row = o;  o = align256(o + (size_t)L.R * 4);
  L.pair_expert = o; o = align256(o + (size_t)L.R * 4);
  L.blk_counts = o; o = align256(o + (size_t)((L.R + kSortBlock - 1) / kSortBlock) * E * 4);
  L.tiles = o;     o = align256(o + (size_t)L.max_tiles * sizeof(Tile));
  L.groups = o;    o = align256(o + (size_t)L.max_groups * sizeof(Tile));
  L.xp = o;        o = align256(o + (size_t)(L.R * H));
  L.sa_p = o;      o = align256(o + (size_t)(L.R * (H / kBlock)) * 4);
  L.act = o;       o = align256(o + (size_t)(L.R * I));
  L.act_scale = o; o = align256(o + (size_t)(L.R * (I / kBlock)) * 4);
  L.y = o;         o = align256(o + (size_t)(L.R * H) * 4);
  // the single-launch path's down terms: per token and output row, its pairs' K blocks
  L.yt = o;        o = align256(o + (size_t)(Mx < kTicketTokens ? Mx : kTicketTokens) * H * ((K * (I / kBlock) + 3) & ~3) * 4);
  L.hid_stage = o; o = align256(o + (size_t)(Mx * H) * 2);
  L.out_stage = o; o = align256(o + (size_t)(Mx * H) * 2);
  L.ids_stage = o; o = align256(o + (size_t)L.R * 4);
  L.wts_stage = o; o = align256(o + (size_t)L.R * 4);
  L.total = o;
  return L;
}

// Device pointers into one workspace.
struct WsPtrs {
  Header* hdr;
  uint8_t* qa;
  float* sa;
  int32_t* offsets;
  int32_t* row_src;
  int32_t* perm_row;
  int32_t* pair_expert;  // [R] expert of each routed pair, -1 if skipped (pair mode)
  int32_t* blk_counts;   // [R/kSortBlock][E] per-block expert histograms (sorted mode)
  Tile* tiles;
  Tile* groups;     // runs of up to kGroupRows expert-sorted rows of one expert
  uint8_t* xp;      // [R][H] hidden codes gathered into expert-sorted row order
  float* sa_p;      // [R][H/128] their scales
  uint8_t* act;
  float* act_scale;
  float* y;
};

inline WsPtrs ws_ptrs(void* ws, const Layout& L) {
  char* b = static_cast<char*>(ws);
  return WsPtrs{reinterpret_cast<Header*>(b + L.header), reinterpret_cast<uint8_t*>(b + L.qa),
                reinterpret_cast<float*>(b + L.sa), reinterpret_cast<int32_t*>(b + L.offsets),
                reinterpret_cast<int32_t*>(b + L.row_src), reinterpret_cast<int32_t*>(b + L.perm_row),
                reinterpret_cast<int32_t*>(b + L.pair_expert), reinterpret_cast<int32_t*>(b + L.blk_counts),
                reinterpret_cast<Tile*>(b + L.tiles), reinterpret_cast<Tile*>(b + L.groups),
                reinterpret_cast<uint8_t*>(b + L.xp), reinterpret_cast<float*>(b + L.sa_p),
                reinterpret_cast<uint8_t*>(b + L.act),
                reinterpret_cast<float*>(b + L.act_scale), reinterpret_cast<float*>(b + L.y)};
}

// --------------------------------------------------------------------------------------
// Numeric helpers (device).
// --------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Per-128 quantiser scale: amax / 448 with IEEE division; 1.0 for an all-zero group.
__device__ __forceinline__ float quant_scale(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Round-to-nearest-even, saturating E4M3 encode of two values (low byte = a).
__device__ __forceinline__ uint16_t e4m3x2_encode(float a, float b) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// exp(-g) from the hardware base-2 exponential with a split argument, accurate to a few
// ulp for every g. -g*log2(e) is carried as an unevaluated sum hi + lo: hi = fl(-g * L2E_HI),
// lo = its exact rounding error (one fma, the TwoProduct of Dekker / Ogita-Rump-Oishi) plus
// -g * L2E_LO, the product with the low part of log2(e) (Cody-Waite style argument
// splitting). Then exp(-g) = 2^hi * 2^lo with 2^lo = 1 + lo*ln2 to first order (|lo| is a
// few ulp of hi). A single rounded product -g*log2(e) would instead lose about |g| ulp.
__device__ __forceinline__ float exp_neg_split(float g) {
  constexpr float kL2eHi = 1.4426950216293335f;    // float32 nearest to log2(e)
  constexpr float kL2eLo = 1.925963033500011e-08f; // log2(e) - kL2eHi
  constexpr float kLn2 = 0.6931471805599453f;
  const float x = -g;
  const float hi = __fmul_rn(x, kL2eHi);
  const float lo = __fadd_rn(__fmaf_rn(x, kL2eHi, -hi), __fmul_rn(x, kL2eLo));
  float p;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(hi));
  return __fmaf_rn(p, __fmul_rn(lo, kLn2), p);
}

// silu(g) * u with the split-argument exponential and the fast division intrinsic: within a
// few ulp of silu_mul for every g (for the many-row epilogue, where the tail of each 128-row
// tile is on the tensor core's critical path). For g below about -88 the exponential
// overflows to +inf and the quotient is -0, as in silu_mul.
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
  return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, exp_neg_split(g))), u);
}

// --------------------------------------------------------------------------------------
// RMSNorm in front of the layer (optional input transform of the hidden rows):
//   y[k] = bf16_rn((x[k] * r) * gamma[k]),   r = 1 / sqrt(ss / H + eps),
// ss = the sum of x[k]^2 formed as the router forms a logit: an FP32 fma chain over each
// 128-wide chunk (k ascending, from 0), the chunk partials added in ascending chunk order.
// Each step is one correctly rounded FP32 operation. Every kernel that reads y computes r
// itself with row_rms_scale, so the router and the quantisers see the same bits.
// --------------------------------------------------------------------------------------
struct Norm {
  const uint16_t* gamma;  // BF16 [H]; nullptr: no normalisation (y = x)
  float eps;
};

// r of the BF16 row x[0, H) (H a multiple of 128, at most 64 chunks; x 16-byte aligned),
// computed by one whole warp; every lane returns it. Lane c (and c + 32) runs chunk c's chain.
__device__ __forceinline__ float row_rms_scale(const uint16_t* __restrict__ x, int H, float eps, int lane) {
  const int nch = H / 128;
  float part0 = 0.0f, part1 = 0.0f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int c = lane + 32 * half;
    if (c < nch) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)c * 128);
      uint4 v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = src[q];
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a = bf16_bits_to_float((uint16_t)(w4[u] & 0xFFFF));
          const float b = bf16_bits_to_float((uint16_t)(w4[u] >> 16));
          acc = __fmaf_rn(a, a, acc);
          acc = __fmaf_rn(b, b, acc);
        }
      }
      if (half == 0) part0 = acc; else part1 = acc;
    }
  }
  float ss = 0.0f;
  for (int c = 0; c < nch; ++c) ss = __fadd_rn(ss, __shfl_sync(0xffffffffu, c < 32 ? part0 : part1, c & 31));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
}

// y of one element (BF16 bits in, BF16 value out as FP32)
__device__ __forceinline__ float norm_value(uint16_t x, float r, uint16_t g) {
  const float v = __fmul_rn(__fmul_rn(bf16_bits_to_float(x), r), bf16_bits_to_float(g));
  return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ uint16_t norm_bits(uint16_t x, float r, uint16_t g) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__fmul_rn(bf16_bits_to_float(x), r), bf16_bits_to_float(g))));
}

__device__ __forceinline__ void set_status(Header* hdr, uint32_t bits) {
  atomicOr(&hdr->status, bits);  // a flag word, never a value accumulation
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound on any device wait (a wait that runs out sets MOE_STATUS_WAIT_TIMEOUT). The
// kernels' waits are for their own copies, MMAs and cluster peers, which take microseconds;
// the bound only has to outlast a time slice of another context on a shared GPU.
constexpr uint64_t kWaitLimitNs = 100000000ull;  // 100 ms

}  // namespace moe
