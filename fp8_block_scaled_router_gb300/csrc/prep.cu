// prep.cu -- hidden-state quantisation and the token -> expert permutation.
//
// Sources: "NetraRuntime/netra-kernel" README, prefill-pair build section (the producer's
// metadata stage, which lays routed rows out per expert); older kernel-lab README,
// repository layout (MoE "activation packing"); the per-token-per-128 FP8 activation
// format of docs/compiler/architecture.md (FP8 activation plus activation-scale tensors).
//
// Quantisation: one warp per (token, 128-column group), amax by a warp max reduction,
// scale = amax/448 (IEEE division; 1.0 for an all-zero group), RNE saturating E4M3 codes.
// With an RMSNorm in front (many-row path), one warp per token forms r and quantises the
// token's y = bf16((x*r)*gamma) group by group.
// Few routed rows (pair mode): block 0 records each pair's expert (-1 if out of range) and
// the identity permutation. Routed rows sorted by expert: up to one sort block of pairs, one
// launch that sorts, quantises and gathers (sort_small_kernel); more, the two-launch counting
// sort and the gather below.
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "device.h"

namespace moe {

constexpr int kPrepThreads = 1024;
constexpr int kMaxExperts = 256;

// One warp quantises one 128-column group: lane l holds columns 4l..4l+3 (x0..x3) and gets
// their four codes (one 32-bit word, column 4l in the low byte); every lane gets the scale.
__device__ __forceinline__ uint32_t quant_group(float x0, float x1, float x2, float x3, float& s) {
  float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  s = quant_scale(amax);
  const uint32_t lo = e4m3x2_encode(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
  const uint32_t hi = e4m3x2_encode(__fdiv_rn(x2, s), __fdiv_rn(x3, s));
  return lo | (hi << 16);
}

__device__ __forceinline__ void quant_group_store(float x0, float x1, float x2, float x3, int lane, uint8_t* qdst,
                                                  float* sdst) {
  float s;
  const uint32_t w = quant_group(x0, x1, x2, x3, s);
  reinterpret_cast<uint32_t*>(qdst)[lane] = w;
  if (lane == 0) *sdst = s;
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const uint16_t* __restrict__ hidden,
                                                            const int32_t* __restrict__ ids, int M,
                                                            int H, int E, int K, WsPtrs ws) {
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
      quant_group_store(bf16_bits_to_float(raw.x & 0xFFFF), bf16_bits_to_float(raw.x >> 16),
                        bf16_bits_to_float(raw.y & 0xFFFF), bf16_bits_to_float(raw.y >> 16), lane,
                        ws.qa + t * H + g * 128, ws.sa + t * ngroups_row + g);
    }
    return;
  }

  {
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
}

// ---------------------------------------------------------------------------------------
// Many routed rows: a counting sort over blocks of kSortBlock pairs in two launches.
//   count:   blocks [0, NB) histogram their pairs by expert into blk_counts[b][E]; the
//            remaining blocks quantise hidden (as above).
//   scatter: block b forms, for every expert, tot[e] = sum over all blocks and
//            pre[e] = sum over blocks before b, the exclusive scan base[e] over experts, and
//            places its pairs at base[e] + pre[e] + (earlier pairs of e in this block), so
//            rows keep ascending flat pair order t*K + j within each expert. Block 0 also
//            writes the expert offsets, the 128-row tile list and the 16-row group list.
//   gather:  each warp copies up to four placed rows' hidden codes (H bytes) and scales
//            into xp / sa_p -- thousands of independent 16-byte copies in flight.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) count_quant_kernel(const uint16_t* __restrict__ hidden, const Norm nm,
                                                          const int32_t* __restrict__ ids, int M, int H,
                                                          int E, int K, int nblk, WsPtrs ws) {
  const int tid = threadIdx.x;
  const int R = M * K;
  if ((int)blockIdx.x < nblk) {
    __shared__ int hist[kMaxExperts];
    __shared__ int bad;
    for (int e = tid; e < E; e += 256) hist[e] = 0;
    if (tid == 0) bad = 0;
    __syncthreads();
    const int i = blockIdx.x * kSortBlock + tid;
    if (i < R) {
      const int e = ids[i];
      if (e >= 0 && e < E) atomicAdd(&hist[e], 1);  // integer count: order-independent
      else bad = 1;
    }
    __syncthreads();
    for (int e = tid; e < E; e += 256) ws.blk_counts[(size_t)blockIdx.x * E + e] = hist[e];
    if (tid == 0 && bad) set_status(ws.hdr, MOE_STATUS_BAD_EXPERT_ID);
    return;
  }
  const int warp = tid / 32, lane = tid % 32;
  const int ngroups_row = H / 128;
  const int64_t nwarps = (int64_t)(gridDim.x - nblk) * 8;
  if (nm.gamma != nullptr) {
    // RMSNorm in front: one warp per row forms r, then quantises y = bf16((x*r)*gamma)
    for (int64_t t = (int64_t)(blockIdx.x - nblk) * 8 + warp; t < M; t += nwarps) {
      const uint16_t* xr = hidden + t * H;
      const float r = row_rms_scale(xr, H, nm.eps, lane);
      for (int g = 0; g < ngroups_row; ++g) {
        const uint2 raw = *reinterpret_cast<const uint2*>(xr + g * 128 + lane * 4);
        const uint2 gm = *reinterpret_cast<const uint2*>(nm.gamma + g * 128 + lane * 4);
        quant_group_store(norm_value(raw.x & 0xFFFF, r, gm.x & 0xFFFF), norm_value(raw.x >> 16, r, gm.x >> 16),
                          norm_value(raw.y & 0xFFFF, r, gm.y & 0xFFFF), norm_value(raw.y >> 16, r, gm.y >> 16),
                          lane, ws.qa + t * H + g * 128, ws.sa + t * ngroups_row + g);
      }
    }
    return;
  }
  // four groups per warp and pass, their loads issued before the first reduction
  const int64_t ngroups = (int64_t)M * ngroups_row;
  for (int64_t g0 = (int64_t)(blockIdx.x - nblk) * 8 + warp; g0 < ngroups; g0 += 4 * nwarps) {
    uint2 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t gidx = g0 + u * nwarps;
      if (gidx < ngroups)
        raw[u] = *reinterpret_cast<const uint2*>(hidden + (gidx / ngroups_row) * H + (gidx % ngroups_row) * 128 +
                                                 lane * 4);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t gidx = g0 + u * nwarps;  // the same for every lane of the warp
      if (gidx >= ngroups) break;
      const int64_t t = gidx / ngroups_row;
      const int g = (int)(gidx % ngroups_row);
      quant_group_store(bf16_bits_to_float(raw[u].x & 0xFFFF), bf16_bits_to_float(raw[u].x >> 16),
                        bf16_bits_to_float(raw[u].y & 0xFFFF), bf16_bits_to_float(raw[u].y >> 16), lane,
                        ws.qa + t * H + g * 128, ws.sa + t * ngroups_row + g);
    }
  }
}

// Exclusive prefix sum of v over the 256 threads of the block in thread order (warp
// shuffles, then the 8 warp totals); `total` receives the sum. wsum: 8 ints of shared memory.
__device__ __forceinline__ int scan256(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int base = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int t = wsum[w];
    base += w < warp ? t : 0;
    total += t;
  }
  __syncthreads();  // wsum is rewritten by the next scan
  return base + x - v;
}

__global__ void __launch_bounds__(256) scatter_kernel(const int32_t* __restrict__ ids, int M, int H,
                                                             int E, int K, int nblk, WsPtrs ws) {
  __shared__ int start[kMaxExperts];
  __shared__ int wsum[8];
  __shared__ int wcnt[8][kMaxExperts];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int R = M * K;
  const int b = blockIdx.x;
  (void)lane;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  // per expert: total over all blocks and the count in blocks before this one. Thread
  // (g, q) sums experts 4q .. 4q+3 over blocks g, g + ng, ... with 16-byte loads (E is a
  // multiple of 4 and a histogram row E * 4 bytes), so few load rounds are in flight
  __shared__ int4 part_tot[256], part_pre[256];
  {
    const int nq = E / 4, q = tid % nq, g = tid / nq, ng = 256 / nq;
    const int4* bc = reinterpret_cast<const int4*>(ws.blk_counts);
    int4 t_ = make_int4(0, 0, 0, 0), p_ = make_int4(0, 0, 0, 0);
#pragma unroll 8
    for (int bb = g; bb < nblk; bb += ng) {
      const int4 c = bc[(size_t)bb * nq + q];
      t_.x += c.x; t_.y += c.y; t_.z += c.z; t_.w += c.w;
      if (bb < b) { p_.x += c.x; p_.y += c.y; p_.z += c.z; p_.w += c.w; }
    }
    part_tot[tid] = t_;
    part_pre[tid] = p_;
  }
  __syncthreads();
  int tot = 0, pre = 0;
  if (tid < E) {
    const int nq = E / 4, q = tid / 4, comp = tid % 4;
    const int* pt = reinterpret_cast<const int*>(part_tot);
    const int* pp = reinterpret_cast<const int*>(part_pre);
    for (int g = 0; g < 256 / nq; ++g) {
      tot += pt[(g * nq + q) * 4 + comp];
      pre += pp[(g * nq + q) * 4 + comp];
    }
  }
  // exclusive scan of tot over experts
  int placed = 0;
  const int base_e = scan256(tid < E ? tot : 0, wsum, placed);
  if (tid < E) start[tid] = base_e + pre;
  if (b == 0) {
    if (tid < E) ws.offsets[tid] = base_e;
    if (tid == 0) ws.offsets[E] = placed;
  }
  // per-warp counts of each expert in this block (stable order: warp, then lane)
  for (int i = tid; i < 8 * E; i += 256) wcnt[i / E][i % E] = 0;
  __syncthreads();
  const int i = b * kSortBlock + tid;
  const int e = i < R ? ids[i] : -1;
  const bool valid = i < R && e >= 0 && e < E;
  const unsigned mask = __match_any_sync(0xffffffffu, valid ? e : -1);
  const int rank = __popc(mask & ((1u << lane) - 1u));
  if (valid && rank == 0) wcnt[warp][e] = __popc(mask);
  __syncthreads();
  int pos = -1;
  if (valid) {
    pos = start[e] + rank;
    for (int w = 0; w < warp; ++w) pos += wcnt[w][e];
    ws.row_src[pos] = i;
  }
  if (i < R) ws.perm_row[i] = pos;
  // block 0: the 128-row tile list (expert counts are the totals)
  if (b == 0) {
    int n_tiles = 0;
    int tb = scan256(tid < E ? (tot + kTileRows - 1) / kTileRows : 0, wsum, n_tiles);
    if (tid < E)
      for (int j = 0; j < tot; j += kTileRows, ++tb) ws.tiles[tb] = Tile{tid, base_e + j, min(kTileRows, tot - j), 0};
    if (tid == 0) ws.hdr->n_tiles = (uint32_t)n_tiles;
    // and the list of groups of up to kGroupRows rows (the expert-grouped pair kernels' units)
    int n_groups = 0;
    int gb = scan256(tid < E ? (tot + kGroupRows - 1) / kGroupRows : 0, wsum, n_groups);
    if (tid < E)
      for (int j = 0; j < tot; j += kGroupRows, ++gb) ws.groups[gb] = Tile{tid, base_e + j, min(kGroupRows, tot - j), 0};
    if (tid == 0) ws.hdr->n_groups = (uint32_t)n_groups;
  }
}

// ---------------------------------------------------------------------------------------
// Few routed pairs (R <= kSortBlock, one sort block): the sort, the hidden quantisation and
// the gather in one launch. Every block repeats the counting sort of the R pairs in shared
// memory -- the arithmetic of the two-launch sort with a single block, so the positions are
// the same -- and block 0 writes its results (offsets, row_src, perm_row, the tile and group
// lists, the invalid-id status). Each warp then quantises (token, 128-column group) units
// (with an RMSNorm in front: whole tokens) and writes the codes and scale to qa / sa and to
// each of the token's placed rows in xp / sa_p. No block waits for another.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) sort_small_kernel(const uint16_t* __restrict__ hidden, const Norm nm,
                                                         const int32_t* __restrict__ ids, int M, int H, int E, int K,
                                                         WsPtrs ws) {
  __shared__ int start[kMaxExperts];
  __shared__ int wsum[8];
  __shared__ int wcnt[8][kMaxExperts];
  __shared__ int s_pos[kSortBlock];
  __shared__ int bad;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int R = M * K;
  const int nsc = H / 128;
  const int64_t nwarps = (int64_t)gridDim.x * 8;
  const int64_t w0 = (int64_t)blockIdx.x * 8 + warp;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  // the warp's first group of hidden values is on its way while the block sorts
  const bool normed = nm.gamma != nullptr;
  const int64_t ngroups = (int64_t)M * nsc;
  uint2 raw0 = make_uint2(0, 0);
  if (!normed && w0 < ngroups)
    raw0 = *reinterpret_cast<const uint2*>(hidden + (w0 / nsc) * H + (w0 % nsc) * 128 + lane * 4);

  for (int j = tid; j < 8 * E; j += 256) wcnt[j / E][j % E] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  const int i = tid;
  const int e = i < R ? ids[i] : -1;
  const bool valid = i < R && e >= 0 && e < E;
  if (i < R && !valid) bad = 1;
  const unsigned mask = __match_any_sync(0xffffffffu, valid ? e : -1);
  const int rank = __popc(mask & ((1u << lane) - 1u));
  if (valid && rank == 0) wcnt[warp][e] = __popc(mask);
  __syncthreads();
  int tot = 0;
  if (tid < E)
    for (int w = 0; w < 8; ++w) tot += wcnt[w][tid];
  int placed = 0;
  const int base_e = scan256(tid < E ? tot : 0, wsum, placed);
  if (tid < E) start[tid] = base_e;
  __syncthreads();
  int pos = -1;
  if (valid) {
    pos = start[e] + rank;
    for (int w = 0; w < warp; ++w) pos += wcnt[w][e];
  }
  s_pos[tid] = pos;
  if (blockIdx.x == 0) {
    if (valid) ws.row_src[pos] = i;
    if (i < R) ws.perm_row[i] = pos;
    if (tid < E) ws.offsets[tid] = base_e;
    if (tid == 0) ws.offsets[E] = placed;
    if (tid == 0 && bad) set_status(ws.hdr, MOE_STATUS_BAD_EXPERT_ID);
    int n_tiles = 0;
    int tb = scan256(tid < E ? (tot + kTileRows - 1) / kTileRows : 0, wsum, n_tiles);
    if (tid < E)
      for (int j = 0; j < tot; j += kTileRows, ++tb) ws.tiles[tb] = Tile{tid, base_e + j, min(kTileRows, tot - j), 0};
    if (tid == 0) ws.hdr->n_tiles = (uint32_t)n_tiles;
    int n_groups = 0;
    int gb = scan256(tid < E ? (tot + kGroupRows - 1) / kGroupRows : 0, wsum, n_groups);
    if (tid < E)
      for (int j = 0; j < tot; j += kGroupRows, ++gb) ws.groups[gb] = Tile{tid, base_e + j, min(kGroupRows, tot - j), 0};
    if (tid == 0) ws.hdr->n_groups = (uint32_t)n_groups;
  }
  __syncthreads();  // s_pos is complete

  // codes and scale of group g of token t, to qa / sa and to the token's placed rows
  auto store = [&](int64_t t, int g, uint32_t word, float sc) {
    reinterpret_cast<uint32_t*>(ws.qa + t * H + g * 128)[lane] = word;
    if (lane == 0) ws.sa[t * nsc + g] = sc;
    for (int j = 0; j < K; ++j) {
      const int p = s_pos[t * K + j];
      if (p < 0) continue;
      reinterpret_cast<uint32_t*>(ws.xp + (size_t)p * H + g * 128)[lane] = word;
      if (lane == 0) ws.sa_p[(size_t)p * nsc + g] = sc;
    }
  };
  if (normed) {
    for (int64_t t = w0; t < M; t += nwarps) {
      const uint16_t* xr = hidden + t * H;
      const float r = row_rms_scale(xr, H, nm.eps, lane);
      for (int g = 0; g < nsc; ++g) {
        const uint2 raw = *reinterpret_cast<const uint2*>(xr + g * 128 + lane * 4);
        const uint2 gm = *reinterpret_cast<const uint2*>(nm.gamma + g * 128 + lane * 4);
        float sc;
        const uint32_t word = quant_group(norm_value(raw.x & 0xFFFF, r, gm.x & 0xFFFF), norm_value(raw.x >> 16, r, gm.x >> 16),
                                          norm_value(raw.y & 0xFFFF, r, gm.y & 0xFFFF), norm_value(raw.y >> 16, r, gm.y >> 16),
                                          sc);
        store(t, g, word, sc);
      }
    }
    return;
  }
  for (int64_t gidx = w0; gidx < ngroups; gidx += nwarps) {
    const uint2 raw = gidx == w0 ? raw0
                                 : *reinterpret_cast<const uint2*>(hidden + (gidx / nsc) * H + (gidx % nsc) * 128 +
                                                                   lane * 4);
    float sc;
    const uint32_t word = quant_group(bf16_bits_to_float(raw.x & 0xFFFF), bf16_bits_to_float(raw.x >> 16),
                                      bf16_bits_to_float(raw.y & 0xFFFF), bf16_bits_to_float(raw.y >> 16), sc);
    store(gidx / nsc, (int)(gidx % nsc), word, sc);
  }
}

// xp[p] = qa[row_src[p] / K], sa_p[p] = sa[row_src[p] / K]: each warp copies rpw consecutive
// placed rows (rpw * H / 16 <= 512 16-byte pieces, at most 16 per lane, all loaded before the
// first store). Only the first offsets[E] rows are placed (pairs with an invalid id are not);
// row_src past them is not written by this call and is never read.
__global__ void __launch_bounds__(256) gather_rows_kernel(int R, int H, int E, int K, int rpw, WsPtrs ws) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int p0 = (blockIdx.x * 8 + warp) * rpw;
  const int placed = min(R, ws.offsets[E]);
  if (p0 >= placed) return;
  const int nr = min(rpw, placed - p0);
  const int n16 = H / 16;
  // lane r < nr holds the source token of row p0 + r
  const int my_tok = lane < nr ? ws.row_src[p0 + lane] / K : 0;
  uint4 v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int idx = lane + 32 * j, r = idx / n16;
    const int t = __shfl_sync(0xffffffffu, my_tok, r & 31);
    if (r < nr) v[j] = reinterpret_cast<const uint4*>(ws.qa + (size_t)t * H)[idx % n16];
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int idx = lane + 32 * j, r = idx / n16;
    if (r < nr) reinterpret_cast<uint4*>(ws.xp + (size_t)(p0 + r) * H)[idx % n16] = v[j];
  }
  const int nsc = H / 128;  // <= 64
  for (int r = 0; r < nr; ++r) {
    const int t = __shfl_sync(0xffffffffu, my_tok, r);
    for (int c = lane; c < nsc; c += 32) ws.sa_p[(size_t)(p0 + r) * nsc + c] = ws.sa[(size_t)t * nsc + c];
  }
}

cudaError_t launch_sort_gather(const uint16_t* hidden, Norm nm, const int32_t* ids, int M, int H, int E, int K,
                               const WsPtrs& ws, cudaStream_t st) {
  const int R = M * K;
  const int nblk = (R + kSortBlock - 1) / kSortBlock;
  const int64_t groups = (int64_t)M * (H / 128);
  const int sms = device_info().sms > 0 ? device_info().sms : 1;
  if (nblk == 1) {
    // one launch: a warp per hidden group (per token with an RMSNorm), at most 2 CTAs per SM
    int64_t blocks = nm.gamma != nullptr ? (M + 7) / 8 : (groups + 7) / 8;
    blocks = std::max<int64_t>(1, std::min<int64_t>(blocks, 2 * (int64_t)sms));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sort_small_kernel, hidden, nm, ids, M, H, E, K, ws);
  }
  int64_t qblocks = (groups + 7) / 8;
  const int64_t cap8 = 8 * (int64_t)sms;  // 8 CTAs per SM
  if (qblocks > cap8) qblocks = cap8;
  count_quant_kernel<<<(unsigned)(nblk + qblocks), 256, 0, st>>>(hidden, nm, ids, M, H, E, K, nblk, ws);
  if (cudaError_t e = cudaGetLastError()) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nblk, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaError_t e = cudaLaunchKernelEx(&cfg, scatter_kernel, ids, M, H, E, K, nblk, ws)) return e;
  // rows per warp: as many as 16 pieces of 16 bytes per lane hold, at most 4
  const int rpw = std::max(1, std::min(4, 512 / (H / 16)));
  cfg.gridDim = dim3((unsigned)((R + 8 * rpw - 1) / (8 * rpw)), 1, 1);  // R rows at most
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, R, H, E, K, rpw, ws);
}

cudaError_t launch_prep(const uint16_t* hidden, const int32_t* ids, int M, int H, int E, int K,
                        const WsPtrs& ws, cudaStream_t st) {
  const int64_t groups = (int64_t)M * (H / 128);
  int64_t qblocks = (groups + (kPrepThreads / 32) - 1) / (kPrepThreads / 32);
  const int64_t cap4 = 4 * (int64_t)(device_info().sms > 0 ? device_info().sms : 1);  // 4 CTAs per SM
  if (qblocks > cap4) qblocks = cap4;
  prep_kernel<<<(unsigned)(1 + qblocks), kPrepThreads, 0, st>>>(hidden, ids, M, H, E, K, ws);
  return cudaGetLastError();
}

}  // namespace moe
