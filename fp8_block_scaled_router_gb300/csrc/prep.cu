// prep.cu -- hidden-state quantisation and the token -> expert permutation.
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (the producer's
// metadata stage, which lays routed rows out per expert); older kernel-lab README,
// repository layout (MoE "activation packing"); the per-token-per-128 FP8 activation
// format of docs/compiler/architecture.md (FP8 activation plus activation-scale tensors).
//
// One launch. Block 0 (1024 threads) runs a stable counting sort of the R = M*K (token,
// slot) pairs by expert: a shared-memory histogram, an exclusive scan, then a scatter in
// rounds of 1024 pairs where each pair's position is its expert's base + the pairs of the
// same expert in earlier warps of the round (per-warp counts) + its rank inside its warp
// (__match_any_sync). Within an expert, rows therefore keep ascending flat pair order
// t*K + j. It also cuts each expert's rows into tiles of at most kTileRows rows.
// Blocks 1.. quantise hidden: one warp per (token, 128-column group), amax by a warp max
// reduction, scale = amax/448, RNE saturating E4M3 codes.
#include "common.cuh"

namespace moe {

constexpr int kPrepThreads = 1024;
constexpr int kMaxExperts = 256;

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const uint16_t* __restrict__ hidden,
                                                            const int32_t* __restrict__ ids, int M,
                                                            int H, int E, int K, int pair_mode,
                                                            WsPtrs ws) {
  const int tid = threadIdx.x;
  if (blockIdx.x > 0) {
    // ---- quantise hidden: warp per (token, 128-group) ----
    const int warp = tid / 32, lane = tid % 32;
    const int ngroups_row = H / 128;
    const int64_t ngroups = (int64_t)M * ngroups_row;
    const int64_t nwarps = (int64_t)(gridDim.x - 1) * (kPrepThreads / 32);
    for (int64_t gidx = (int64_t)(blockIdx.x - 1) * (kPrepThreads / 32) + warp; gidx < ngroups;
         gidx += nwarps) {
      const int64_t t = gidx / ngroups_row;
      const int g = (int)(gidx % ngroups_row);
      const uint2 raw = *reinterpret_cast<const uint2*>(hidden + t * H + g * 128 + lane * 4);
      const float x0 = bf16_bits_to_float(raw.x & 0xFFFF), x1 = bf16_bits_to_float(raw.x >> 16);
      const float x2 = bf16_bits_to_float(raw.y & 0xFFFF), x3 = bf16_bits_to_float(raw.y >> 16);
      float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float s = quant_scale(amax);
      const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
      const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, s), __fdiv_rn(x3, s));
      *reinterpret_cast<uint32_t*>(ws.qa + t * H + g * 128 + lane * 4) = lo | (hi << 16);
      if (lane == 0) ws.sa[t * ngroups_row + g] = s;
    }
    return;
  }

  if (pair_mode) {
    // ---- block 0, pair mode: each routed pair is its own unit (identity permutation) ----
    __shared__ int bad_pair;
    if (tid == 0) bad_pair = 0;
    __syncthreads();
    for (int i = tid; i < M * K; i += kPrepThreads) {
      const int e = ids[i];
      const bool valid = e >= 0 && e < E;
      ws.pair_expert[i] = valid ? e : -1;
      ws.perm_row[i] = valid ? i : -1;
      ws.row_src[i] = i;
      if (!valid) bad_pair = 1;
    }
    __syncthreads();
    if (tid == 0) {
      ws.hdr->n_tiles = 0;
      if (bad_pair) set_status(ws.hdr, MOE_STATUS_BAD_EXPERT_ID);
    }
    return;
  }

  // ---- block 0: stable counting sort of the routed pairs by expert ----
  __shared__ int cnt[kMaxExperts];
  __shared__ int base[kMaxExperts + 1];
  __shared__ int tile_base[kMaxExperts + 1];
  __shared__ int wcnt[kPrepThreads / 32][kMaxExperts];
  __shared__ int bad;
  const int R = M * K;
  const int warp = tid / 32, lane = tid % 32;
  for (int e = tid; e < E; e += kPrepThreads) cnt[e] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int i = tid; i < R; i += kPrepThreads) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // integer count: order-independent
    else bad = 1;
  }
  __syncthreads();
  if (tid == 0) {
    // E <= 256: a serial scan is a few hundred cycles, off the critical path of the quant blocks
    int acc = 0, tacc = 0;
    for (int e = 0; e < E; ++e) {
      base[e] = acc;
      tile_base[e] = tacc;
      acc += cnt[e];
      tacc += (cnt[e] + kTileRows - 1) / kTileRows;
    }
    base[E] = acc;
    tile_base[E] = tacc;
    ws.hdr->n_tiles = (uint32_t)tacc;
    if (bad) set_status(ws.hdr, MOE_STATUS_BAD_EXPERT_ID);
  }
  __syncthreads();
  for (int e = tid; e <= E; e += kPrepThreads) ws.offsets[e] = base[e];
  for (int e = tid; e < E; e += kPrepThreads) {
    const int n = cnt[e];
    for (int j = 0, tb = tile_base[e]; j < n; j += kTileRows, ++tb)
      ws.tiles[tb] = Tile{e, base[e] + j, min(kTileRows, n - j), 0};
  }
  for (int r0 = 0; r0 < R; r0 += kPrepThreads) {
    for (int i = tid; i < (kPrepThreads / 32) * E; i += kPrepThreads) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int i = r0 + tid;
    const int e = i < R ? ids[i] : -1;
    const bool valid = i < R && e >= 0 && e < E;
    const unsigned mask = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int rank = __popc(mask & ((1u << lane) - 1u));
    if (valid && rank == 0) wcnt[warp][e] = __popc(mask);
    __syncthreads();
    if (i < R) {
      if (valid) {
        int pos = base[e] + rank;
        for (int w = 0; w < warp; ++w) pos += wcnt[w][e];
        ws.row_src[pos] = i;
        ws.perm_row[i] = pos;
      } else {
        ws.perm_row[i] = -1;
      }
    }
    __syncthreads();
    for (int e2 = tid; e2 < E; e2 += kPrepThreads) {
      int s = 0;
      for (int w = 0; w < kPrepThreads / 32; ++w) s += wcnt[w][e2];
      base[e2] += s;
    }
    __syncthreads();
  }
}

// Gather the hidden codes and scales of every routed row into expert-sorted order (the A
// operand rows of the grouped GEMM): xp[r] = qa[row_src[r] / K], sa_p[r] = sa[row_src[r] / K].
// One warp per sorted row; rows past the valid count (skipped pairs) are left untouched.
__global__ void __launch_bounds__(256) gather_kernel(int R, int H, int E, int K, WsPtrs ws) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int r = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (r >= R || r >= ws.offsets[E]) return;
  const int t = ws.row_src[r] / K;
  const uint4* src = reinterpret_cast<const uint4*>(ws.qa + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(ws.xp + (size_t)r * H);
  for (int i = lane; i < H / 16; i += 32) dst[i] = src[i];
  for (int i = lane; i < H / 128; i += 32) ws.sa_p[(size_t)r * (H / 128) + i] = ws.sa[(size_t)t * (H / 128) + i];
}

cudaError_t launch_gather(int R, int H, int E, int K, const WsPtrs& ws, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((R + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_kernel, R, H, E, K, ws);
}

cudaError_t launch_prep(const uint16_t* hidden, const int32_t* ids, int M, int H, int E, int K,
                        const WsPtrs& ws, cudaStream_t st) {
  const int pair_mode = use_pair_mode((int64_t)M * K) ? 1 : 0;
  const int64_t groups = (int64_t)M * (H / 128);
  int64_t qblocks = (groups + (kPrepThreads / 32) - 1) / (kPrepThreads / 32);
  if (qblocks > 4 * 152) qblocks = 4 * 152;
  prep_kernel<<<(unsigned)(1 + qblocks), kPrepThreads, 0, st>>>(hidden, ids, M, H, E, K, pair_mode, ws);
  return cudaGetLastError();
}

}  // namespace moe
